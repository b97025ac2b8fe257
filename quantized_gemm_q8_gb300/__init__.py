"""GB300 (sm_103a) hot path of one LLaDA-style diffusion-LLM denoising step.

Thin Python binding over the C ABI in include/dllm.h (libdllm.so, built in-tree by
``quantized_gemm_q8_gb300.build``). The functions here only marshal arguments: device
memory and streams come from PyTorch, every step of the path runs in the library's CUDA
kernels, and there is no CPU fallback - a missing library raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# DLLM_CHECKED=1 loads the bounds-checked build (every kernel access checked against its
# buffer; slower, for tests and debugging) in place of the regular library.
CHECKED = os.environ.get("DLLM_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "libdllm_checked.so" if CHECKED else "libdllm.so")

Q4_K = 12
Q6_K = 14
QK = 256

OK, E_INVAL, E_SHAPE, E_ALIGN, E_TYPE, E_WORKSPACE, E_CUDA, E_TIMEOUT, E_DEVICE, E_BOUNDS = range(10)


class DllmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[dllm status {code}] {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None

P, I64, I32, SZ, F32, INT = C.c_void_p, C.c_int64, C.c_int32, C.c_size_t, C.c_float, C.c_int
U64, U32 = C.c_uint64, C.c_uint32
_SIGS = {
    "dllm_last_error": ([], C.c_char_p),
    "dllm_version": ([], INT),
    "dllm_check": ([P], INT),
    "dllm_packed_bytes": ([INT, I64, I64], SZ),
    "dllm_pack_weights": ([INT, P, I64, I64, P, SZ, P], INT),
    "dllm_act_rows": ([I64], I64),
    "dllm_act_bytes": ([I64, I64], SZ),
    "dllm_quantize_act": ([P, I64, I64, I64, P, F32, P, P, P, P, SZ, P], INT),
    "dllm_qgemm_workspace_bytes": ([INT, I64, I64, I64], SZ),
    "dllm_qgemm": ([INT, P, I64, I64, P, I64, P, I64, INT, P, SZ, P], INT),
    "dllm_pack_act": ([P, P, P, I64, I64, P, SZ, P], INT),
    "dllm_qgemm_plain_workspace_bytes": ([INT, I64, I64, I64], SZ),
    "dllm_qgemm_q4k": ([P, P, P, I64, I64, P, I64, P, I64, INT, P, SZ, P], INT),
    "dllm_qgemm_q6k": ([P, P, P, I64, I64, P, I64, P, I64, INT, P, SZ, P], INT),
    "dllm_qgemm_intsums": ([INT, P, I64, I64, P, I64, P, P], INT),
    "dllm_selftest_timeout": ([I64, P], INT),
    "dllm_step_graph_host": ([P, P, P, I64, P, I32, I32, P, P], INT),
    "dllm_bounds_checked": ([], INT),
    "dllm_selftest_bounds": ([P, I32, I32, P], INT),
    "dllm_lmhead_workspace_bytes": ([I64, I64, I64], SZ),
    "dllm_lmhead_masked_select": ([P, I64, I64, I64, P, F32, P, I64, P, I32, I32, I32, I32, P, P, P, P, P, P, SZ, P],
                                  INT),
    "dllm_lmhead_select": ([P, I64, I64, I64, P, F32, P, I64, P, I32, I32, I32, I32, I32, F32, U64, U32, P, P, P, P,
                            P, P, SZ, P], INT),
    "dllm_step_workspace_bytes": ([P, I64, INT], SZ),
    "dllm_step_linear_stream": ([P, P, I64, P, INT, P, SZ, P], INT),
    "dllm_denoise_workspace_bytes": ([P, I64, I32], SZ),
    "dllm_denoise_step": ([P, P, I64, I32, I32, I32, P, P, P, P, P, SZ, P], INT),
    "dllm_kv_cache_bytes": ([P, I64], SZ),
    "dllm_denoise_cached_workspace_bytes": ([P, I64, I32], SZ),
    "dllm_denoise_step_cached": ([P, P, I64, I32, I32, I32, I32, P, SZ, P, P, P, P, P, SZ, P], INT),
    "dllm_launch_count": ([], C.c_longlong),
    "dllm_qgemm_partials_bytes": ([INT, I64, I64, I64], SZ),
    "dllm_qgemm_partials": ([INT, P, I64, I64, P, I64, P, SZ, P, P], INT),
    "dllm_qgemm_noalloc": ([INT, P, I64, I64, P, I64, P, I64, INT, P], INT),
    "dllm_step_taps": ([P, P, I64, P, INT, P, P, SZ, P], INT),
    "dllm_peak_mma_i8": ([I64, P, P, P], INT),
    "dllm_transfer_counts": ([I64, I64, P], INT),
    "dllm_schedule": ([I64, I64, I64, I64, P, P, P], INT),
}


def lib():
    """The loaded C library (raises if it was not built: there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; "
                                   "g.build()'` (this package has no CPU fallback)")
            l = C.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                f = getattr(l, name)
                f.argtypes = args
                f.restype = res
            _lib = l
    return _lib


def last_error() -> str:
    return lib().dllm_last_error().decode()


def _ok(rc: int):
    if rc != OK:
        raise DllmError(rc, last_error())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def check(stream=None):
    """Synchronize the stream and raise if a kernel recorded a device-side timeout."""
    _ok(lib().dllm_check(_stream(stream)))


# --- weights -------------------------------------------------------------------------------

def packed_bytes(type_id: int, n: int, k: int) -> int:
    return int(lib().dllm_packed_bytes(type_id, n, k))


def pack_weights(type_id: int, blocks: torch.Tensor, n: int, k: int, stream=None) -> torch.Tensor:
    """GGUF block bytes (uint8 CUDA tensor, n x k/256 blocks) -> packed uint8 CUDA tensor."""
    nbytes = packed_bytes(type_id, n, k)
    if nbytes == 0:
        raise DllmError(E_SHAPE, f"bad packed shape type={type_id} n={n} k={k}")
    out = torch.empty(nbytes, dtype=torch.uint8, device=blocks.device)
    _ok(lib().dllm_pack_weights(type_id, _ptr(blocks), n, k, _ptr(out), nbytes, _stream(stream)))
    return out


# --- activations ---------------------------------------------------------------------------

def act_rows(rows: int) -> int:
    return int(lib().dllm_act_rows(rows))


def act_bytes(rows: int, k: int) -> int:
    return int(lib().dllm_act_bytes(rows, k))


def quantize_act(x: torch.Tensor, norm_w: torch.Tensor | None = None, eps: float = 1e-5,
                 plain: bool = True, operand: bool = True, act: torch.Tensor | None = None, stream=None):
    """Q8_K-quantize f32 rows of x (optionally RMSNorm-ed). Returns dict(q, d, bsum, act)."""
    rows, k = x.shape
    dev = x.device
    out = {"q": None, "d": None, "bsum": None, "act": None}
    if plain:
        out["q"] = torch.empty((rows, k), dtype=torch.int8, device=dev)
        out["d"] = torch.empty((rows, k // QK), dtype=torch.float32, device=dev)
        out["bsum"] = torch.empty((rows, k // 16), dtype=torch.int16, device=dev)
    nb = 0
    if operand:
        nb = act_bytes(rows, k)
        out["act"] = act if act is not None else torch.empty(nb, dtype=torch.uint8, device=dev)
    _ok(lib().dllm_quantize_act(_ptr(x), rows, k, x.stride(0), _ptr(norm_w), eps, _ptr(out["q"]),
                                _ptr(out["d"]), _ptr(out["bsum"]), _ptr(out["act"]), nb, _stream(stream)))
    return out


# --- GEMM ----------------------------------------------------------------------------------

def qgemm_workspace_bytes(type_id: int, m: int, n: int, k: int) -> int:
    return int(lib().dllm_qgemm_workspace_bytes(type_id, m, n, k))


def qgemm(type_id: int, act: torch.Tensor, m: int, k: int, w_packed: torch.Tensor, n: int,
          y: torch.Tensor | None = None, accumulate: bool = False, ws: torch.Tensor | None = None,
          stream=None) -> torch.Tensor:
    """y[m, n] (+)= Q8_K activations x decoded Q4_K/Q6_K weights^T (f32)."""
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=act.device)
    wsb = qgemm_workspace_bytes(type_id, m, n, k)
    if wsb and ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device=act.device)
    _ok(lib().dllm_qgemm(type_id, _ptr(act), m, k, _ptr(w_packed), n, _ptr(y), y.stride(0), int(accumulate),
                         _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
    return y


def pack_act(q: torch.Tensor, d: torch.Tensor, bsum: torch.Tensor, act: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """Operand form of plain Q8_K arrays (q int8 [rows, k], d f32 [rows, k/256], bsum int16)."""
    rows, k = q.shape
    nb = act_bytes(rows, k)
    if act is None:
        act = torch.empty(nb, dtype=torch.uint8, device=q.device)
    _ok(lib().dllm_pack_act(_ptr(q), _ptr(d), _ptr(bsum), rows, k, _ptr(act), act.numel(), _stream(stream)))
    return act


def qgemm_plain(type_id: int, q: torch.Tensor, d: torch.Tensor, bsum: torch.Tensor, w_packed: torch.Tensor, n: int,
                y: torch.Tensor | None = None, accumulate: bool = False, ws: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """y[m, n] (+)= plain Q8_K activations x decoded weights^T (dllm_qgemm_q4k / dllm_qgemm_q6k)."""
    m, k = q.shape
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=q.device)
    nb = int(lib().dllm_qgemm_plain_workspace_bytes(type_id, m, n, k))
    if ws is None:
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    fn = lib().dllm_qgemm_q4k if type_id == Q4_K else lib().dllm_qgemm_q6k
    _ok(fn(_ptr(q), _ptr(d), _ptr(bsum), m, k, _ptr(w_packed), n, _ptr(y), y.stride(0), int(accumulate), _ptr(ws),
           ws.numel(), _stream(stream)))
    return y


def qgemm_intsums(type_id: int, act: torch.Tensor, m: int, k: int, w_packed: torch.Tensor, n: int,
                  stream=None) -> torch.Tensor:
    """Exact per-super-block integer sums int32 [2, k/256, m, n] (test hook)."""
    sums = torch.zeros((2, k // QK, m, n), dtype=torch.int32, device=act.device)
    _ok(lib().dllm_qgemm_intsums(type_id, _ptr(act), m, k, _ptr(w_packed), n, _ptr(sums), _stream(stream)))
    return sums


def qgemm_noalloc(type_id: int, act: torch.Tensor, m: int, k: int, w_packed: torch.Tensor, n: int,
                  y: torch.Tensor, accumulate: bool = False, stream=None) -> torch.Tensor:
    """Same result as qgemm without any workspace: for callers that cannot allocate device
    memory at call time; the library keeps the split-K partials in its own fixed 32 MiB array
    (m * n * 4 bytes at most). Calls must not overlap on the GPU."""
    _ok(lib().dllm_qgemm_noalloc(type_id, _ptr(act), m, k, _ptr(w_packed), n, _ptr(y), y.stride(0), int(accumulate),
                                 _stream(stream)))
    return y


def launch_count() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(lib().dllm_launch_count())


def qgemm_partials(type_id: int, act: torch.Tensor, m: int, k: int, w_packed: torch.Tensor, n: int,
                   partials: torch.Tensor | None = None, stream=None):
    """The GEMM kernel alone: split partials f32 [splits, m, n] (sum = qgemm result)."""
    nb = int(lib().dllm_qgemm_partials_bytes(type_id, m, n, k))
    if partials is None:
        partials = torch.empty(nb // 4, dtype=torch.float32, device=act.device)
    sp = C.c_int32(0)
    _ok(lib().dllm_qgemm_partials(type_id, _ptr(act), m, k, _ptr(w_packed), n, _ptr(partials), partials.numel() * 4,
                                  C.byref(sp), _stream(stream)))
    return partials, sp.value


def peak_mma_i8_tops(iters: int = 20000, reps: int = 3, stream=None) -> float:
    """Measured dense rate of mma.sync int8 (m16n8k32) on this GPU, TOPS (best of reps)."""
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops = C.c_double(0.0)
    s = torch.cuda.current_stream() if stream is None else stream
    _ok(lib().dllm_peak_mma_i8(100, _ptr(sink), None, _stream(s)))  # warm-up
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        _ok(lib().dllm_peak_mma_i8(iters, _ptr(sink), C.byref(ops), _stream(s)))
        e1.record(s)
        s.synchronize()
        best = max(best, ops.value / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    return best


def selftest_timeout(limit_cycles: int, stream=None):
    _ok(lib().dllm_selftest_timeout(limit_cycles, _stream(stream)))


def bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().dllm_bounds_checked())


def selftest_bounds(buf: torch.Tensor, n_write: int, n_declared: int, stream=None):
    """buf[i] = i for i < n_write, each store checked against the first n_declared floats."""
    assert buf.dtype == torch.float32 and buf.is_cuda and buf.numel() >= n_write
    _ok(lib().dllm_selftest_bounds(_ptr(buf), n_write, n_declared, _stream(stream)))


# --- transfer schedule (host only) -----------------------------------------------------------

def transfer_counts(masked: int, steps: int) -> list:
    """Tokens committed at each of a block's `steps` steps for `masked` masked positions."""
    arr = (C.c_int32 * max(steps, 1))()
    _ok(lib().dllm_transfer_counts(masked, steps, arr))
    return [int(v) for v in arr[:steps]]


def schedule(prompt_len: int, gen_len: int, block_len: int, steps: int) -> list:
    """[(block_begin, block_end, k)] for each step of the whole generation."""
    n = max(steps, 1)
    b0, b1, k = (C.c_int32 * n)(), (C.c_int32 * n)(), (C.c_int32 * n)()
    _ok(lib().dllm_schedule(prompt_len, gen_len, block_len, steps, b0, b1, k))
    return [(int(b0[s]), int(b1[s]), int(k[s])) for s in range(steps)]


# --- LM head + commit --------------------------------------------------------------------------

def lmhead_workspace_bytes(rows: int, vocab: int, d: int) -> int:
    return int(lib().dllm_lmhead_workspace_bytes(rows, vocab, d))


CONF_PMAX = 0         # confidence = softmax probability of the argmax token (LLaDA)
CONF_NEG_ENTROPY = 1  # confidence = -entropy of the row's softmax (Dream's entropy ranking)


def lmhead_masked_select(hidden: torch.Tensor, canvas: torch.Tensor, mask_id: int, block_begin: int,
                         block_end: int, k_commit: int, out_norm_w: torch.Tensor, w_out_packed: torch.Tensor,
                         vocab: int, eps: float = 1e-5, ws: torch.Tensor | None = None, stream=None) -> dict:
    """Masked-rows-only LM head + softmax confidence + top-k commit; updates `canvas` in place.
    Returns dict(pos, id, conf [k_commit], row_id, row_conf [block rows])."""
    return lmhead_select(hidden, canvas, mask_id, block_begin, block_end, k_commit, out_norm_w, w_out_packed, vocab,
                         CONF_PMAX, eps, ws, stream)


def lmhead_select(hidden: torch.Tensor, canvas: torch.Tensor, mask_id: int, block_begin: int, block_end: int,
                  k_commit: int, out_norm_w: torch.Tensor, w_out_packed: torch.Tensor, vocab: int,
                  conf_kind: int = CONF_PMAX, eps: float = 1e-5, ws: torch.Tensor | None = None, stream=None,
                  temperature: float = 0.0, seed: int = 0, step: int = 0) -> dict:
    """lmhead_masked_select with the confidence chosen by conf_kind (CONF_PMAX, CONF_NEG_ENTROPY)
    and, for temperature > 0, Gumbel-max draws keyed by (seed, step, position, token)."""
    L, d = hidden.shape
    R = block_end - block_begin
    dev = hidden.device
    out = {
        "pos": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
        "id": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
        "conf": torch.empty(max(k_commit, 1), dtype=torch.float32, device=dev),
        "row_id": torch.empty(R, dtype=torch.int32, device=dev),
        "row_conf": torch.empty(R, dtype=torch.float32, device=dev),
    }
    nb = lmhead_workspace_bytes(R, vocab, d)
    if ws is None:
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    _ok(lib().dllm_lmhead_select(_ptr(hidden), L, d, hidden.stride(0), _ptr(out_norm_w), eps, _ptr(w_out_packed),
                                 vocab, _ptr(canvas), mask_id, block_begin, block_end, k_commit, conf_kind,
                                 temperature, seed, step, _ptr(out["pos"]), _ptr(out["id"]), _ptr(out["conf"]), _ptr(out["row_id"]),
                                 _ptr(out["row_conf"]), _ptr(ws), ws.numel(), _stream(stream)))
    for key in ("pos", "id", "conf"):
        out[key] = out[key][:k_commit]
    return out


# --- model, layer stream and denoising step ------------------------------------------------------

STREAM_LINEAR = 0
STREAM_FULL = 1


class _Layer(C.Structure):
    _fields_ = [("wqk", P), ("wv", P), ("wo", P), ("wgu", P), ("wdown", P), ("attn_norm", P), ("ffn_norm", P)]


class _Model(C.Structure):
    _fields_ = [("n_layers", I32), ("d_model", I32), ("n_heads", I32), ("head_dim", I32), ("d_ff", I32),
                ("vocab", I32), ("mask_id", I32), ("eps", F32), ("rope_theta", F32), ("layers", C.POINTER(_Layer)),
                ("tok_embd", P), ("out_norm", P), ("w_out", P)]


class DeviceModel:
    """Device copy of a LLaDA-shaped model: packed projections, norms, token table, head.

    `layers` is a list of dicts of GGUF block arrays (numpy, as from synth.layer_weights);
    `tok_embd` the Q4_K token table blocks; `head` a dict(w_out=Q6_K blocks, out_norm=f32).
    The device tensors are kept alive by this object; `.ref` is the C struct pointer."""

    def __init__(self, dims: dict, layers, tok_embd=None, head=None, device="cuda", n_layers: int | None = None):
        import numpy as np

        self.dims = dict(dims)
        self._keep = []
        d, f = dims["d_model"], dims["d_ff"]
        if n_layers is None:
            n_layers = len(layers)

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
            self._keep.append(t)
            return t

        def packed(type_id, blocks, n, k):
            t = pack_weights(type_id, dev(blocks.reshape(-1)), n, k)
            self._keep.append(t)
            return t

        arr = (_Layer * n_layers)()
        for i, lw in enumerate(layers):
            wqk = packed(Q4_K, np.concatenate([lw["wq"], lw["wk"]], axis=0), 2 * d, d)
            wv = packed(Q6_K, lw["wv"], d, d)
            wo = packed(Q4_K, lw["wo"], d, d)
            wgu = packed(Q4_K, np.concatenate([lw["wgate"], lw["wup"]], axis=0), 2 * f, d)
            wdn = packed(Q6_K, lw["wdown"], d, f)
            an, fn = dev(lw["attn_norm"]), dev(lw["ffn_norm"])
            arr[i] = _Layer(wqk.data_ptr(), wv.data_ptr(), wo.data_ptr(), wgu.data_ptr(), wdn.data_ptr(),
                            an.data_ptr(), fn.data_ptr())
            torch.cuda.synchronize()
        self._layers = arr
        te = dev(tok_embd.reshape(-1)).data_ptr() if tok_embd is not None else None
        on = wout = None
        self.w_out_packed = self.out_norm = None
        if head is not None:
            self.out_norm = dev(head["out_norm"])
            self.w_out_packed = packed(Q6_K, head["w_out"], dims["vocab"], d)
            on, wout = self.out_norm.data_ptr(), self.w_out_packed.data_ptr()
        self.struct = _Model(n_layers, d, dims["n_heads"], dims["head_dim"], f, dims["vocab"], dims["mask_id"],
                             dims["eps"], dims["rope_theta"], arr, te, on, wout)
        self.ref = C.byref(self.struct)
        torch.cuda.synchronize()


def step_workspace_bytes(model: DeviceModel, L: int, flags: int) -> int:
    return int(lib().dllm_step_workspace_bytes(model.ref, L, flags))


def step_linear_stream(model: DeviceModel, x: torch.Tensor, flags: int = STREAM_LINEAR,
                       canvas: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """Run the layer stream; x (f32 [L, d]) is updated in place (filled from the canvas when FULL)."""
    L = x.shape[0]
    nb = step_workspace_bytes(model, L, flags)
    if ws is None:
        ws = torch.empty(nb + 1024, dtype=torch.uint8, device=x.device)
    wsp = (ws.data_ptr() + 1023) // 1024 * 1024
    _ok(lib().dllm_step_linear_stream(model.ref, _ptr(canvas), L, _ptr(x), flags, C.c_void_p(wsp),
                                      ws.numel() - (wsp - ws.data_ptr()), _stream(stream)))
    return x


class _Taps(C.Structure):
    _fields_ = [("layer", I32), ("x_in", P), ("act_attn", P), ("q", P), ("k", P), ("v", P), ("attn", P), ("act_o", P),
                ("x_mid", P), ("act_ffn", P), ("h", P), ("act_down", P), ("x_out", P)]


TAP_NAMES = ("x_in", "act_attn", "q", "k", "v", "attn", "act_o", "x_mid", "act_ffn", "h", "act_down", "x_out")


def step_taps(model: DeviceModel, x: torch.Tensor, flags: int, layer: int, canvas: torch.Tensor | None = None,
              names=TAP_NAMES, stream=None) -> dict:
    """step_linear_stream that also captures layer `layer`'s intermediates (test hook). Returns
    a dict of device tensors: f32 [L, d] / [L, d_ff] for x_in, q, k, v, attn, x_mid, h, x_out,
    and uint8 operand-form buffers for act_attn, act_o, act_ffn, act_down."""
    L = x.shape[0]
    d, f = model.dims["d_model"], model.dims["d_ff"]
    dev = x.device
    out = {}
    for nm in names:
        if nm.startswith("act_"):
            out[nm] = torch.zeros(act_bytes(L, f if nm == "act_down" else d), dtype=torch.uint8, device=dev)
        else:
            out[nm] = torch.zeros((L, f if nm == "h" else d), dtype=torch.float32, device=dev)
    taps = _Taps(layer, *[out[nm].data_ptr() if nm in out else None for nm in TAP_NAMES])
    nb = step_workspace_bytes(model, L, flags)
    ws = torch.empty(nb + 1024, dtype=torch.uint8, device=dev)
    wsp = (ws.data_ptr() + 1023) // 1024 * 1024
    _ok(lib().dllm_step_taps(model.ref, _ptr(canvas), L, _ptr(x), flags, C.byref(taps), C.c_void_p(wsp),
                             ws.numel() - (wsp - ws.data_ptr()), _stream(stream)))
    return out


def denoise_workspace_bytes(model: DeviceModel, L: int, block_rows: int) -> int:
    return int(lib().dllm_denoise_workspace_bytes(model.ref, L, block_rows))


def denoise_step(model: DeviceModel, canvas: torch.Tensor, block_begin: int, block_end: int, k_commit: int,
                 hidden_out: torch.Tensor | None = None, ws: torch.Tensor | None = None, out: dict | None = None,
                 stream=None) -> dict:
    """One full denoising step (forward + masked LM head + commit); canvas updated in place."""
    L = canvas.shape[0]
    dev = canvas.device
    if out is None:
        out = {"pos": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
               "id": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
               "conf": torch.empty(max(k_commit, 1), dtype=torch.float32, device=dev)}
    nb = denoise_workspace_bytes(model, L, block_end - block_begin)
    if ws is None:
        ws = torch.empty(nb + 1024, dtype=torch.uint8, device=dev)
    wsp = (ws.data_ptr() + 1023) // 1024 * 1024
    _ok(lib().dllm_denoise_step(model.ref, _ptr(canvas), L, block_begin, block_end, k_commit, _ptr(out["pos"]),
                                _ptr(out["id"]), _ptr(out["conf"]), _ptr(hidden_out), C.c_void_p(wsp),
                                ws.numel() - (wsp - ws.data_ptr()), _stream(stream)))
    return out


def kv_cache_bytes(model: DeviceModel, L: int) -> int:
    return int(lib().dllm_kv_cache_bytes(model.ref, L))


def denoise_cached_workspace_bytes(model: DeviceModel, L: int, block_rows: int) -> int:
    return int(lib().dllm_denoise_cached_workspace_bytes(model.ref, L, block_rows))


def denoise_step_cached(model: DeviceModel, canvas: torch.Tensor, block_begin: int, block_end: int, k_commit: int,
                        refresh: bool, kv_cache: torch.Tensor, hidden_out: torch.Tensor | None = None,
                        ws: torch.Tensor | None = None, out: dict | None = None, stream=None) -> dict:
    """One denoising step with the inter-step K/V cache: refresh=True runs the full step and fills
    kv_cache; refresh=False recomputes only the block's rows against the cached K/V."""
    L = canvas.shape[0]
    dev = canvas.device
    if out is None:
        out = {"pos": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
               "id": torch.empty(max(k_commit, 1), dtype=torch.int32, device=dev),
               "conf": torch.empty(max(k_commit, 1), dtype=torch.float32, device=dev)}
    nb = denoise_cached_workspace_bytes(model, L, block_end - block_begin)
    if ws is None:
        ws = torch.empty(nb + 1024, dtype=torch.uint8, device=dev)
    wsp = (ws.data_ptr() + 1023) // 1024 * 1024
    _ok(lib().dllm_denoise_step_cached(model.ref, _ptr(canvas), L, block_begin, block_end, k_commit, int(refresh),
                                       _ptr(kv_cache), kv_cache.numel() * kv_cache.element_size(), _ptr(out["pos"]),
                                       _ptr(out["id"]), _ptr(out["conf"]), _ptr(hidden_out), C.c_void_p(wsp),
                                       ws.numel() - (wsp - ws.data_ptr()), _stream(stream)))
    return out


def model_from_seed(dims: dict, seed: int, device="cuda") -> DeviceModel:
    """Seeded synthetic LLaDA-shaped model (generated, uploaded and packed one layer at a time)."""
    from . import synth

    gen = (synth.layer_weights(seed, i, dims) for i in range(dims["n_layers"]))
    return DeviceModel(dims, gen, synth.embed_weights(seed, dims), synth.head_weights(seed, dims), device,
                       n_layers=dims["n_layers"])


class StepGraphs:
    """One CUDA graph per kind of denoising step (forward + masked LM head + commit), all on the
    same device canvas and output buffers. A kind is (block_begin, block_end, k_commit), e.g. the
    distinct entries of `schedule(...)`; replay(i) runs kind i. Workspace and outputs are
    allocated once, before capture."""

    def __init__(self, model: DeviceModel, canvas: torch.Tensor, kinds: list):
        self.model, self.canvas, self.kinds = model, canvas, list(kinds)
        dev = canvas.device
        L = canvas.shape[0]
        rows = max(b1 - b0 for b0, b1, _ in self.kinds)
        kmax = max(max(k for _, _, k in self.kinds), 1)
        nb = denoise_workspace_bytes(model, L, rows)
        self.ws = torch.empty(nb + 1024, dtype=torch.uint8, device=dev)
        self.kmax = kmax
        self.pos_id = torch.empty(2 * kmax, dtype=torch.int32, device=dev)  # positions, then ids
        self.out = {"pos": self.pos_id[:kmax], "id": self.pos_id[kmax:],
                    "conf": torch.empty(kmax, dtype=torch.float32, device=dev)}
        self.stream = torch.cuda.Stream(device=dev)
        self.graphs = []
        self.launches_per_step = []
        saved = canvas.clone()
        with torch.cuda.stream(self.stream):
            for b0, b1, k in self.kinds:  # warm the library (attributes, tensor-map entry point) once
                denoise_step(model, canvas, b0, b1, k, ws=self.ws, out=self.out, stream=self.stream)
        self.stream.synchronize()
        check(self.stream)
        for b0, b1, k in self.kinds:
            g = torch.cuda.CUDAGraph()
            n0 = launch_count()
            with torch.cuda.graph(g, stream=self.stream):
                denoise_step(model, canvas, b0, b1, k, ws=self.ws, out=self.out, stream=self.stream)
            self.launches_per_step.append(launch_count() - n0)
            self.graphs.append(g)
        canvas.copy_(saved)
        torch.cuda.synchronize()

    def replay(self, kind_index: int):
        """Replay on self.stream (a graph replays on the caller's current stream)."""
        with torch.cuda.stream(self.stream):
            self.graphs[kind_index].replay()

    def step_host(self, kind_index: int, canvas_host: torch.Tensor, out_host: torch.Tensor):
        """One step from host buffers through dllm_step_graph_host: the host canvas (pinned int32
        [L]) goes in, graph kind_index runs, its commits come back into out_host (pinned int32
        [2 * kmax]: positions, then ids) and are applied to canvas_host."""
        k = self.kinds[kind_index][2]
        exec_ = self.graphs[kind_index].raw_cuda_graph_exec()
        _ok(lib().dllm_step_graph_host(C.c_void_p(exec_), _ptr(canvas_host), _ptr(self.canvas), self.canvas.shape[0],
                                       _ptr(self.pos_id), self.kmax, k, _ptr(out_host), _stream(self.stream)))


class CachedStepGraphs:
    """Two CUDA graphs per kind of step (block_begin, block_end, k_commit) for the inter-step K/V
    cache: the refreshing step (full forward, cache filled) and the cached step (block rows
    only); replay(kind, refresh). One cache, workspace and output set, allocated before capture."""

    def __init__(self, model: DeviceModel, canvas: torch.Tensor, kinds: list):
        self.model, self.canvas, self.kinds = model, canvas, list(kinds)
        dev = canvas.device
        L = canvas.shape[0]
        rows = max(b1 - b0 for b0, b1, _ in self.kinds)
        kmax = max(max(k for _, _, k in self.kinds), 1)
        nb = denoise_cached_workspace_bytes(model, L, rows)
        self.ws = torch.empty(nb + 1024, dtype=torch.uint8, device=dev)
        self.kv = torch.empty(kv_cache_bytes(model, L) // 4, dtype=torch.float32, device=dev)
        self.out = {"pos": torch.empty(kmax, dtype=torch.int32, device=dev),
                    "id": torch.empty(kmax, dtype=torch.int32, device=dev),
                    "conf": torch.empty(kmax, dtype=torch.float32, device=dev)}
        self.stream = torch.cuda.Stream(device=dev)
        self.graphs = {}
        saved = canvas.clone()

        def step(b0, b1, k, refresh):
            denoise_step_cached(model, canvas, b0, b1, k, refresh, self.kv, ws=self.ws, out=self.out,
                                stream=self.stream)

        with torch.cuda.stream(self.stream):
            for b0, b1, k in self.kinds:  # warm the library once; the refresh fills the cache first
                step(b0, b1, k, True)
                step(b0, b1, k, False)
        self.stream.synchronize()
        check(self.stream)
        for i, (b0, b1, k) in enumerate(self.kinds):
            for refresh in (True, False):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    step(b0, b1, k, refresh)
                self.graphs[(i, refresh)] = g
        canvas.copy_(saved)
        torch.cuda.synchronize()

    def replay(self, kind_index: int, refresh: bool):
        with torch.cuda.stream(self.stream):
            self.graphs[(kind_index, refresh)].replay()
