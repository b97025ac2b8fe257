"""Stage-isolated GPU parity of one layer (the Development plan's correctness ladder: RMSNorm,
RoPE, softmax, attention, one transformer layer), every stage against the f64 oracle run on the
GPU's own input to that stage.

dllm_step_taps copies out the layer's intermediates. For each stage the oracle recomputes the
stage from the GPU's tapped input and the stage's output is held to the GEMM bar on EVERY row:
max |y - y_ref| <= 2e-3 x ||y_ref row||_2. Quantizations of an f32 input the GPU also used
(attention output, SwiGLU output) must give bit-identical codes and scales; the two RMSNorm +
Q8_K stages start from the same f32 rows but normalize in f32 (GPU) against f64 (oracle), so a
value that lands on a rounding tie may take the neighbouring code: at most one code step, on
fewer than 1e-3 of the values.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_gemm_q8_gb300 as dl
from quantized_gemm_q8_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-3
SMALL = dict(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ff=1024, vocab=1000, mask_id=997, eps=1e-5,
             rope_theta=500000.0)


def unpack_act(buf: np.ndarray, rows: int, k: int):
    """Operand form (dllm_quantize_act's `act`) -> (codes int8 [rows][k], scales f32 [rows][k/256])."""
    lp = dl.act_rows(rows)
    nsb = k // 256
    a_bytes = lp * k * 2
    off_j = -(-a_bytes // 1024) * 1024
    off_d = -(-(off_j + nsb * lp * 32) // 1024) * 1024
    A = buf[:a_bytes].view(np.float16).reshape(k // 64, lp, 16, 4)[:, :rows]
    A = A[..., [0, 2, 1, 3]]  # within each group of 4 the operand holds k-positions (0, 2, 1, 3)
    q = A.transpose(1, 0, 2, 3).reshape(rows, k).astype(np.int8)
    d = buf[off_d:off_d + nsb * lp * 4].view(np.float32).reshape(nsb, lp)[:, :rows].T.copy()
    return q, d


def _row_errs(y, ref):
    den = np.linalg.norm(ref, axis=1)
    den[den == 0] = 1.0
    return np.max(np.abs(np.asarray(y, np.float64) - ref), axis=1) / den


def _every_row(y, ref, label, log):
    e = _row_errs(y, ref)
    log.append(f"{label}: max row error {e.max():.2e}")
    assert e.max() <= TOL, (label, float(e.max()), np.argsort(e)[-5:])


def _codes_exact(q_gpu, d_gpu, x_f32, label, log):
    q, d, _ = orc.quantize_q8k(np.asarray(x_f32, np.float32))
    np.testing.assert_array_equal(q_gpu, q, err_msg=label)
    np.testing.assert_array_equal(d_gpu, d, err_msg=label)
    log.append(f"{label}: codes and scales bit-exact")


def _codes_near(q_gpu, d_gpu, x_f32, norm_w, eps, label, log):
    q, d, _ = orc.quantize_act(np.asarray(x_f32, np.float32), norm_w, eps)
    diff = np.abs(q_gpu.astype(np.int32) - q.astype(np.int32))
    frac = float((diff > 0).mean())
    log.append(f"{label}: {int((diff > 0).sum())} of {diff.size} codes one step apart (rounding ties)")
    assert diff.max() <= 1 and frac < 1e-3, (label, int(diff.max()), frac)
    np.testing.assert_allclose(d_gpu, d, rtol=2e-6, err_msg=label)


def _layers(seed, dims, n):
    lws = [synth.layer_weights(seed, i, dims) for i in range(n)]
    for i, lw in enumerate(lws):  # non-trivial norm weights
        lw["attn_norm"] = (1.0 + 0.2 * synth.activations(seed + 100 + i, 1, dims["d_model"])[0]).astype(np.float32)
        lw["ffn_norm"] = (1.0 + 0.2 * synth.activations(seed + 200 + i, 1, dims["d_model"])[0]).astype(np.float32)
    return lws


def _check_layer(dims, lws, li, x, flags, canvas=None):
    L, d, f = x.shape[0], dims["d_model"], dims["d_ff"]
    nh, hd, eps = dims["n_heads"], dims["head_dim"], dims["eps"]
    lw = lws[li]
    table = synth.embed_weights(11, dims) if canvas is not None else None
    model = dl.DeviceModel(dims, lws, table)
    gx = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    names = dl.TAP_NAMES if flags == dl.STREAM_FULL else tuple(n for n in dl.TAP_NAMES if n not in ("q", "k", "v"))
    t = dl.step_taps(model, gx, flags, li, canvas=None if canvas is None else torch.from_numpy(canvas).cuda(),
                     names=names)
    dl.check()
    T = {k: v.cpu().numpy() for k, v in t.items()}
    log = []
    x_in = T["x_in"].astype(np.float64)
    # 1. RMSNorm (attn_norm) + Q8_K
    q1, d1 = unpack_act(T["act_attn"], L, d)
    _codes_near(q1, d1, T["x_in"], lw["attn_norm"], eps, "attn RMSNorm + Q8_K", log)
    # 2. Q, K (+ RoPE, 1/sqrt(hd)) and V projections from the GPU's codes
    v_ref = orc.qgemm(orc.TYPE_Q6_K, lw["wv"], q1, d1)
    if flags == dl.STREAM_FULL:
        q_ref = orc.rope(orc.qgemm(orc.TYPE_Q4_K, lw["wq"], q1, d1), nh, hd, dims["rope_theta"]) / np.sqrt(hd)
        k_ref = orc.rope(orc.qgemm(orc.TYPE_Q4_K, lw["wk"], q1, d1), nh, hd, dims["rope_theta"])
        _every_row(T["q"], q_ref, "Q projection + RoPE", log)
        _every_row(T["k"], k_ref, "K projection + RoPE", log)
        _every_row(T["v"], v_ref, "V projection", log)
        # 3. attention (softmax(q k^T / sqrt(hd)) v) on the GPU's Q, K, V
        att_ref = orc.attention(T["q"].astype(np.float64) * np.sqrt(hd), T["k"], T["v"], nh, hd)
        _every_row(T["attn"], att_ref, "attention", log)
    else:
        _every_row(T["attn"], v_ref, "V projection (linear stream)", log)
    # 4. Q8_K of the attention output: same f32 input on both sides
    q2, d2 = unpack_act(T["act_o"], L, d)
    _codes_exact(q2, d2, T["attn"], "attention output Q8_K", log)
    # 5. O projection + residual
    _every_row(T["x_mid"], x_in + orc.qgemm(orc.TYPE_Q4_K, lw["wo"], q2, d2), "O projection + residual", log)
    # 6. RMSNorm (ffn_norm) + Q8_K
    q3, d3 = unpack_act(T["act_ffn"], L, d)
    _codes_near(q3, d3, T["x_mid"], lw["ffn_norm"], eps, "ffn RMSNorm + Q8_K", log)
    # 7. gate | up + SwiGLU
    h_ref = orc.swiglu(orc.qgemm(orc.TYPE_Q4_K, lw["wgate"], q3, d3), orc.qgemm(orc.TYPE_Q4_K, lw["wup"], q3, d3))
    _every_row(T["h"], h_ref, "gate|up + SwiGLU", log)
    # 8. Q8_K of the SwiGLU output: same f32 input
    q4, d4 = unpack_act(T["act_down"], L, f)
    _codes_exact(q4, d4, T["h"], "SwiGLU output Q8_K", log)
    # 9. down projection + residual
    _every_row(T["x_out"], T["x_mid"].astype(np.float64) + orc.qgemm(orc.TYPE_Q6_K, lw["wdown"], q4, d4),
               "down projection + residual", log)
    print("\n  " + "\n  ".join(log))


@pytest.mark.parametrize("L", [129, 160, 200])
def test_stages_full_layer_small(L):
    # 129: a second 128-query tile of one row; 160: the largest tensor-core attention canvas;
    # 200: the chunked f32 attention and its multi-chunk merge. Layer 1, so that the layer's input
    # is a real residual stream (the embedding through layer 0)
    dims = SMALL
    lws = _layers(51 + L, dims, 2)
    canvas = synth.canvas(51 + L, prompt_len=8, gen_len=L - 8, mask_id=dims["mask_id"], prompt_max=990)
    _check_layer(dims, lws, 1, np.zeros((L, dims["d_model"]), np.float32), dl.STREAM_FULL, canvas)


def test_stages_full_layer_llada_shapes():
    dims = dict(synth.LLADA, n_layers=1)
    lws = _layers(synth.config_seed(4), dims, 1)
    canvas = synth.canvas(synth.config_seed(4))
    _check_layer(dims, lws, 0, np.zeros((148, dims["d_model"]), np.float32), dl.STREAM_FULL, canvas)


def test_stages_linear_stream_llada_shapes():
    dims = dict(synth.LLADA, n_layers=1)
    lws = _layers(synth.config_seed(2), dims, 1)
    x = synth.activations(synth.config_seed(2) + 1, 148, dims["d_model"])
    _check_layer(dims, lws, 0, x, dl.STREAM_LINEAR)
