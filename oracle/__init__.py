"""CPU oracle for the diffusion-LLM denoising-step hot path (test infrastructure).

ONLY the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It shares no code with the CUDA library: the
arithmetic lives in ``orc.c`` (plain C, f64, OpenMP over output rows) and the
compositions below chain those primitives in the order the pages give:

* mojo-dllm "Technical Specification", section 11 (the order inside one LLaDA
  layer: normalize, project to Q/K/V, rotate Q and K, attend over every
  position, project the attention output and add it to the stream, normalize
  again, run the gated MLP and add its output) and "Development plan", "Model facts" (eps 1e-5,
  NORM RoPE with theta 500000, SwiGLU 12288, untied output);
* "Development plan", "Compute design": every projection consumes Q8_K
  activations (quantized per token, decisions in f32) and decoded Q4_K/Q6_K
  weights; the output head is evaluated for the masked rows of the active
  block and nowhere else;
* "Technical Specification", section 12: confidence, top-k select, scatter.

Readings where the pages are silent:
* the final RMSNorm (``out_norm``) is applied to the masked rows before the
  LM head;
* the "linear stream" workload has no attention: the O projection consumes
  the V projection's output;
* confidence = softmax probability of the argmax token; ties in the argmax go
  to the lowest token id, ties in top-k to the lowest position;
* the entropy confidence (README, "Each model's own sampler": Dream's entropy
  ranking) is minus the natural-log entropy of the row's softmax;
* temperature sampling (specification section 14: temperature, categorical
  sampling, deterministic PRNG) is the Gumbel-max draw with noise from
  counter-based SplitMix64 keyed by (seed, step, position, token); the draw's
  confidence is its probability under the untempered softmax;
* the inter-step K/V cache (README status table, "--dual-cache"; specification
  section 23) refreshes every layer's K and V on a block's first step and then
  recomputes only the block's rows against them.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orc.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

TYPE_Q4_K = 12
TYPE_Q6_K = 14
QK = 256
BLOCK_BYTES = {TYPE_Q4_K: 144, TYPE_Q6_K: 210}


def build(force: bool = False) -> str:
    """Compile orc.c into liborc.so (plain gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_LIB)
            P, I64, I32, D = C.c_void_p, C.c_int64, C.c_int32, C.c_double
            sig = {
                "orc_num_threads": ([], C.c_int),
                "orc_dequant": ([C.c_int, P, I64, P], C.c_int),
                "orc_quantize_q8k": ([P, I64, I64, I64, P, P, P], None),
                "orc_rmsnorm": ([P, I64, I64, P, D, P], None),
                "orc_qgemm_rows": ([C.c_int, P, I64, I64, P, P, I64, P, I64, P], C.c_int),
                "orc_qgemm_intsums": ([C.c_int, P, I64, I64, P, I64, P, P], C.c_int),
                "orc_block_scales": ([C.c_int, P, I64, P, P], C.c_int),
                "orc_q4k_fields": ([P, P, P, P], None),
                "orc_q6k_fields": ([P, P, P], None),
                "orc_rope": ([P, I64, I64, I64, D], None),
                "orc_attention": ([P, P, P, I64, I64, I64, P], None),
                "orc_swiglu": ([P, P, I64, P], None),
                "orc_embed_q4k": ([P, I64, I64, P, I64, P], C.c_int),
                "orc_row_confidence": ([P, I64, I64, P, P, P, P], None),
                "orc_row_neg_entropy": ([P, I64, I64, P], None),
                "orc_splitmix64_at": ([C.c_uint64, C.c_uint64], C.c_uint64),
                "orc_row_sample": ([P, I64, I64, C.c_double, C.c_uint64, C.c_uint32, P, P, P, P], None),
                "orc_commit_topk": ([P, I64, I32, I64, I64, P, P, I64, P, P], C.c_int),
                "orc_transfer_counts": ([I64, I64, P], None),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().orc_num_threads())


# --- formats ---------------------------------------------------------------------------------

def dequant(type_id: int, blocks: np.ndarray) -> np.ndarray:
    """Exact decoded weights (f64). blocks [..., nb, bytes] -> [..., nb*256]."""
    b = _c(blocks, np.uint8)
    bb = BLOCK_BYTES[type_id]
    nb = b.size // bb
    out = np.empty(nb * QK, dtype=np.float64)
    rc = _load().orc_dequant(type_id, _p(b), nb, _p(out))
    if rc:
        raise ValueError(f"orc_dequant failed ({rc})")
    return out.reshape(*b.shape[:-2], b.shape[-2] * QK) if b.ndim >= 2 else out


def q4k_fields(block: np.ndarray):
    """(scales[8], mins[8], quants[256]) of one Q4_K block."""
    b = _c(block, np.uint8)
    sc = np.zeros(8, np.int32)
    mn = np.zeros(8, np.int32)
    q = np.zeros(256, np.uint8)
    _load().orc_q4k_fields(_p(b), _p(sc), _p(mn), _p(q))
    return sc, mn, q


def q6k_fields(block: np.ndarray):
    """(scales[16], quants[256] in [0,63]) of one Q6_K block."""
    b = _c(block, np.uint8)
    sc = np.zeros(16, np.int32)
    q = np.zeros(256, np.uint8)
    _load().orc_q6k_fields(_p(b), _p(sc), _p(q))
    return sc, q


def quantize_q8k(x: np.ndarray):
    """Q8_K codes of f32 rows: (q int8 [r,k], d f32 [r,k/256], bsum int16 [r,k/16])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    if k % QK:
        raise ValueError("k must be a multiple of 256")
    q = np.empty((rows, k), np.int8)
    d = np.empty((rows, k // QK), np.float32)
    bs = np.empty((rows, k // 16), np.int16)
    _load().orc_quantize_q8k(_p(x), rows, k, k, _p(q), _p(d), _p(bs))
    return q, d, bs


def rmsnorm(x: np.ndarray, w=None, eps: float = 1e-5) -> np.ndarray:
    x = _c(x, np.float64)
    rows, k = x.shape
    out = np.empty_like(x)
    wp = None if w is None else _c(w, np.float32)
    _load().orc_rmsnorm(_p(x), rows, k, None if wp is None else _p(wp), float(eps), _p(out))
    return out


def quantize_act(x: np.ndarray, norm_w=None, eps: float = 1e-5):
    """Activation quantization as the path does it: optional RMSNorm (f64), then the
    normalized values rounded to f32 and quantized to Q8_K with f32 decisions."""
    if norm_w is not None:
        x = rmsnorm(np.asarray(x, np.float64), norm_w, eps)
    return quantize_q8k(np.asarray(x, np.float32))


def qgemm(type_id: int, wblocks: np.ndarray, q: np.ndarray, d: np.ndarray, rows=None) -> np.ndarray:
    """y[m][n] = sum_k W[n][k] * d[m][k/256] * q[m][k] in f64 (rows: subset of n)."""
    w = _c(wblocks, np.uint8)
    n, nsb = w.shape[0], w.shape[1]
    k = nsb * QK
    q = _c(q, np.int8)
    d = _c(d, np.float32)
    m = q.shape[0]
    if rows is None:
        sel, nsel = None, n
    else:
        sel = _c(rows, np.int64)
        nsel = sel.size
    y = np.empty((m, nsel), np.float64)
    rc = _load().orc_qgemm_rows(type_id, _p(w), n, k, _p(q), _p(d), m,
                                None if sel is None else _p(sel), nsel, _p(y))
    if rc:
        raise RuntimeError(f"orc_qgemm_rows failed ({rc})")
    return y


def intsums(type_id: int, wblocks: np.ndarray, q: np.ndarray):
    """Integer sums U, J [m][n][nsb] (int64) of the unified decoded form."""
    w = _c(wblocks, np.uint8)
    n, nsb = w.shape[0], w.shape[1]
    q = _c(q, np.int8)
    m = q.shape[0]
    U = np.empty((m, n, nsb), np.int64)
    J = np.empty((m, n, nsb), np.int64)
    rc = _load().orc_qgemm_intsums(type_id, _p(w), n, nsb * QK, _p(q), m, _p(U), _p(J))
    if rc:
        raise RuntimeError("orc_qgemm_intsums failed")
    return U, J


def block_scales(type_id: int, wblocks: np.ndarray):
    """Per-block (c0, c1) with block value = c0*U - c1*J (shape [n, nsb])."""
    w = _c(wblocks, np.uint8)
    nb = w.size // BLOCK_BYTES[type_id]
    c0 = np.empty(nb, np.float64)
    c1 = np.empty(nb, np.float64)
    _load().orc_block_scales(type_id, _p(w), nb, _p(c0), _p(c1))
    return c0.reshape(w.shape[:-1]), c1.reshape(w.shape[:-1])


# --- layer maths -----------------------------------------------------------------------------

def rope(x: np.ndarray, n_heads: int, head_dim: int, theta: float) -> np.ndarray:
    out = _c(x, np.float64).copy()
    _load().orc_rope(_p(out), out.shape[0], n_heads, head_dim, float(theta))
    return out


def attention(q, k, v, n_heads: int, head_dim: int) -> np.ndarray:
    q, k, v = (_c(a, np.float64) for a in (q, k, v))
    o = np.empty_like(q)
    _load().orc_attention(_p(q), _p(k), _p(v), q.shape[0], n_heads, head_dim, _p(o))
    return o


def swiglu(g, u) -> np.ndarray:
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    h = np.empty_like(g)
    _load().orc_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def embed(table_blocks: np.ndarray, ids: np.ndarray) -> np.ndarray:
    t = _c(table_blocks, np.uint8)
    vocab, nsb = t.shape[0], t.shape[1]
    ids = _c(ids, np.int32)
    x = np.empty((ids.size, nsb * QK), np.float64)
    if _load().orc_embed_q4k(_p(t), vocab, nsb * QK, _p(ids), ids.size, _p(x)):
        raise ValueError("token id out of range")
    return x


def row_confidence(logits: np.ndarray):
    """(argmax id int32, softmax confidence f64, top1 logit, top2 logit) per row."""
    l = _c(logits, np.float64)
    r, v = l.shape
    ids = np.empty(r, np.int32)
    conf = np.empty(r, np.float64)
    t1 = np.empty(r, np.float64)
    t2 = np.empty(r, np.float64)
    _load().orc_row_confidence(_p(l), r, v, _p(ids), _p(conf), _p(t1), _p(t2))
    return ids, conf, t1, t2


def row_neg_entropy(logits: np.ndarray) -> np.ndarray:
    """Minus the entropy (natural log) of each row's softmax, f64: the entropy-ranking confidence."""
    l = _c(logits, np.float64)
    r, v = l.shape
    out = np.empty(r, np.float64)
    _load().orc_row_neg_entropy(_p(l), r, v, _p(out))
    return out


def splitmix64_at(seed: int, counter: int) -> int:
    """Output number `counter` (from 0) of the SplitMix64 stream started at `seed`."""
    return int(_load().orc_splitmix64_at(seed & 0xFFFFFFFFFFFFFFFF, counter & 0xFFFFFFFFFFFFFFFF))


def row_sample(logits: np.ndarray, temperature: float, seed: int, step: int, pos) -> tuple:
    """Gumbel-max draws from softmax(logits / temperature) per row (row r at canvas position
    pos[r]): (id int32, probability of the id under softmax(logits) f64, perturbed-score gap)."""
    l = _c(logits, np.float64)
    r, v = l.shape
    p = _c(np.asarray(pos, np.int64).reshape(r), np.int64)
    ids = np.empty(r, np.int32)
    conf = np.empty(r, np.float64)
    gap = np.empty(r, np.float64)
    _load().orc_row_sample(_p(l), r, v, float(temperature), seed & 0xFFFFFFFFFFFFFFFF, step, _p(p), _p(ids),
                           _p(conf), _p(gap))
    return ids, conf, gap


def commit_topk(canvas: np.ndarray, mask_id: int, b0: int, b1: int, conf_by_pos, ids_by_pos, k: int):
    """Commit in place; returns (positions, ids) in selection order."""
    cv = np.ascontiguousarray(canvas, np.int32)
    conf = _c(conf_by_pos, np.float64)
    ids = _c(ids_by_pos, np.int32)
    pos = np.zeros(max(k, 1), np.int32)
    tid = np.zeros(max(k, 1), np.int32)
    n = _load().orc_commit_topk(_p(cv), cv.size, int(mask_id), int(b0), int(b1), _p(conf), _p(ids),
                                int(k), _p(pos), _p(tid))
    if n < 0:
        raise ValueError("bad block range")
    canvas[...] = cv
    return pos[:n].copy(), tid[:n].copy()


def transfer_counts(masked: int, steps: int) -> np.ndarray:
    out = np.empty(steps, np.int64)
    _load().orc_transfer_counts(int(masked), int(steps), _p(out))
    return out


# --- compositions ----------------------------------------------------------------------------

def linear(type_id, wblocks, x, norm_w=None, eps=1e-5, rows=None):
    """One quantized projection of activation rows x (optionally RMSNorm-ed first)."""
    q, d, _ = quantize_act(x, norm_w, eps)
    return qgemm(type_id, wblocks, q, d, rows)


def layer(lw: dict, x, dims: dict, attention_on: bool, with_qk: bool = True):
    """One LLaDA layer on residual rows x (f64 out).

    attention_on=False is the "linear stream" workload: Q and K are projected
    (and returned) but unused, and the O projection consumes V's output.
    Returns (x_out, extras) where extras holds the intermediate f64 tensors.
    """
    eps, nh, hd = dims["eps"], dims["n_heads"], dims["head_dim"]
    x = np.asarray(x, np.float64)
    q1, d1, _ = quantize_act(x, lw["attn_norm"], eps)
    ex = {}
    if with_qk or attention_on:
        ex["q"] = qgemm(TYPE_Q4_K, lw["wq"], q1, d1)
        ex["k"] = qgemm(TYPE_Q4_K, lw["wk"], q1, d1)
    ex["v"] = qgemm(TYPE_Q6_K, lw["wv"], q1, d1)
    if attention_on:
        ex["q_rope"] = rope(ex["q"], nh, hd, dims["rope_theta"])
        ex["k_rope"] = rope(ex["k"], nh, hd, dims["rope_theta"])
        o = attention(ex["q_rope"], ex["k_rope"], ex["v"], nh, hd)
    else:
        o = ex["v"]
    ex["attn_out"] = o
    q2, d2, _ = quantize_act(o)
    x = x + qgemm(TYPE_Q4_K, lw["wo"], q2, d2)
    ex["x_mid"] = x
    q3, d3, _ = quantize_act(x, lw["ffn_norm"], eps)
    g = qgemm(TYPE_Q4_K, lw["wgate"], q3, d3)
    u = qgemm(TYPE_Q4_K, lw["wup"], q3, d3)
    h = swiglu(g, u)
    ex["h"] = h
    q4, d4, _ = quantize_act(h)
    x = x + qgemm(TYPE_Q6_K, lw["wdown"], q4, d4)
    return x, ex


def layer_block(lw: dict, xb, dims: dict, k_cache: np.ndarray, v_cache: np.ndarray, b0: int):
    """One LLaDA layer on the block rows xb (canvas positions b0 .. b0 + R - 1) of a cached step
    (the inter-step K/V cache, "--dual-cache"): the block's Q, K, V are projected as in `layer`,
    RoPE uses the rows' canvas positions, the fresh K (after RoPE) and V overwrite the block's rows
    of k_cache / v_cache ([L][d], in place), and the block's queries attend to all L cached rows.
    Everything after the attention is `layer` on the block rows. Returns the block's x_out."""
    eps, nh, hd = dims["eps"], dims["n_heads"], dims["head_dim"]
    xb = np.asarray(xb, np.float64)
    L, R = k_cache.shape[0], xb.shape[0]
    q1, d1, _ = quantize_act(xb, lw["attn_norm"], eps)
    q = qgemm(TYPE_Q4_K, lw["wq"], q1, d1)
    k = qgemm(TYPE_Q4_K, lw["wk"], q1, d1)
    v = qgemm(TYPE_Q6_K, lw["wv"], q1, d1)

    def at_positions(a):  # rows placed at their canvas positions, so RoPE rotates by position
        full = np.zeros((L, a.shape[1]))
        full[b0:b0 + R] = a
        return full

    q_full = rope(at_positions(q), nh, hd, dims["rope_theta"])
    k_cache[b0:b0 + R] = rope(at_positions(k), nh, hd, dims["rope_theta"])[b0:b0 + R]
    v_cache[b0:b0 + R] = v
    o = attention(q_full, k_cache, v_cache, nh, hd)[b0:b0 + R]  # only the block's query rows are kept
    q2, d2, _ = quantize_act(o)
    x = xb + qgemm(TYPE_Q4_K, lw["wo"], q2, d2)
    q3, d3, _ = quantize_act(x, lw["ffn_norm"], eps)
    h = swiglu(qgemm(TYPE_Q4_K, lw["wgate"], q3, d3), qgemm(TYPE_Q4_K, lw["wup"], q3, d3))
    q4, d4, _ = quantize_act(h)
    return x + qgemm(TYPE_Q6_K, lw["wdown"], q4, d4)


def forward_cached(lws, table, canvas, dims: dict, b0: int, b1: int, refresh: bool, cache: list):
    """The residual stream of a cached step: refresh runs every layer on all rows and stores each
    layer's (K after RoPE, V) in `cache` (a list, filled in place); otherwise only rows [b0, b1)
    run, through layer_block. Returns x [L][d] (rows outside the block are zero for a cached step)."""
    if refresh:
        x = embed(table, canvas)
        cache.clear()
        for lw in lws:
            x, ex = layer(lw, x, dims, attention_on=True)
            cache.append((ex["k_rope"].copy(), ex["v"].copy()))
        return x
    xb = embed(table, np.asarray(canvas)[b0:b1])
    for lw, (kc, vc) in zip(lws, cache):
        xb = layer_block(lw, xb, dims, kc, vc, b0)
    x = np.zeros((np.asarray(canvas).size, xb.shape[1]))
    x[b0:b1] = xb
    return x


def lmhead_logits(hidden_rows, out_norm, w_out, eps=1e-5):
    """Logits (f64) of the given hidden rows: RMSNorm -> Q8_K -> Q6_K head."""
    q, d, _ = quantize_act(hidden_rows, out_norm, eps)
    return qgemm(TYPE_Q6_K, w_out, q, d)


CONF_PMAX, CONF_NEG_ENTROPY = 0, 1


def lmhead_commit(hidden, canvas, mask_id, b0, b1, k, out_norm, w_out, eps=1e-5, conf_kind=CONF_PMAX,
                  temperature=0.0, seed=0, step=0):
    """Masked-rows-only LM head + confidence + top-k commit (canvas updated in place). The
    committed token is the argmax (temperature 0) or a Gumbel-max draw from
    softmax(logits / temperature) keyed by (seed, step, position, token). The confidence is
    that token's probability under softmax(logits) (CONF_PMAX, LLaDA) or minus the softmax
    entropy (CONF_NEG_ENTROPY, Dream's ranking).

    Returns dict(pos, id, conf, rows, ids_rows, conf_rows, top1, top2[, sample_gap])."""
    rows = np.array([p for p in range(b0, b1) if canvas[p] == mask_id], dtype=np.int64)
    res = dict(rows=rows)
    L = canvas.size
    conf_pos = np.full(L, -np.inf)
    ids_pos = np.zeros(L, np.int32)
    if rows.size:
        logits = lmhead_logits(np.asarray(hidden, np.float64)[rows], out_norm, w_out, eps)
        ids, conf, t1, t2 = row_confidence(logits)
        if temperature > 0:
            ids, conf, gap = row_sample(logits, temperature, seed, step, rows)
            res.update(sample_gap=gap)
        if conf_kind == CONF_NEG_ENTROPY:
            conf = row_neg_entropy(logits)
        conf_pos[rows] = conf
        ids_pos[rows] = ids
        res.update(ids_rows=ids, conf_rows=conf, top1=t1, top2=t2)
    pos, tid = commit_topk(canvas, mask_id, b0, b1, conf_pos, ids_pos, k)
    res.update(pos=pos, id=tid, conf=conf_pos[pos] if pos.size else np.zeros(0))
    return res
