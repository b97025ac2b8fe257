"""Closed-form pins of the oracle's layer maths and compositions (CPU only).

Each pin takes the oracle module as an argument, so that the same check runs on the real oracle
and, in test_oracle_mutations.py, on copies with one planted mistake, where it must fail.

What they fix, from the pages:
  * RoPE (Development plan, "Model facts": NORM / adjacent-pair RoPE; Technical Specification
    section 11): pair i of a head rotates by position * theta^(-2i / head_dim);
  * attention (Technical Specification sections 11 and 11.1): softmax(q k^T / sqrt(head_dim)) v;
  * the layer order (Technical Specification section 11): RMSNorm (attn_norm) -> Q, K, V ->
    RoPE -> attention -> O -> residual add; RMSNorm (ffn_norm) -> gate, up -> silu(gate) * up
    -> down -> residual add; every projection consumes Q8_K codes of its input (Development
    plan, "Compute design");
  * the LM head (README, "How it works"; Development plan, "Model facts": untied output, F32
    norms): the output norm, then the head, then softmax confidence and top-k commit.

The layer pins use weights whose decoded values are known by construction (zero blocks,
identity and permutation matrices built with the independent encoders) and a one-token canvas,
where attention returns V exactly. Their expected values are written from the layer order
above, using only oracle parts that other tests pin on their own (Q8_K quantization,
RMSNorm, decode).
"""
import math

import numpy as np

from _encoders import encode_q4k, encode_q6k

D = 256
DIMS = dict(n_layers=1, d_model=D, n_heads=2, head_dim=128, d_ff=D, vocab=D, mask_id=D - 1, eps=1e-5,
            rope_theta=500000.0)
TYPE_Q4_K, TYPE_Q6_K = 12, 14

# Code pattern of one super-block: every integer in [-127, 127] once (37 is prime to 255), with
# a single +127 (index 254).
PATTERN = np.array([(i * 37) % 255 - 127 for i in range(D)], np.int64)
# Norm weights: powers of two, so that x = PATTERN / w is exact and RMSNorm(x) * w is
# proportional to PATTERN.
POW2 = np.array([2.0 ** ((i % 4) - 1) for i in range(D)], np.float32)


def q4k_matrix(n, k, col_of_row, d_bits=0x3C00):
    """Q4_K [n][k/256] blocks with w[r][col_of_row[r]] = d and every other weight 0
    (scale 1 and quant 1 at that column, mins 0, dmin 0)."""
    nsb = k // 256
    out = np.zeros((n, nsb, 144), np.uint8)
    for r in range(n):
        c = int(col_of_row[r])
        b, i = divmod(c, 256)
        sc = [0] * 8
        sc[i // 32] = 1
        q = [0] * 256
        q[i] = 1
        for bb in range(nsb):
            out[r, bb] = encode_q4k(d_bits if bb == b else 0, 0, sc if bb == b else [0] * 8, [0] * 8,
                                    q if bb == b else [0] * 256)
    return out


def q6k_matrix(n, k, col_of_row, d_bits=0x3C00):
    """Q6_K [n][k/256] blocks with w[r][col_of_row[r]] = d and every other weight 0
    (quants 32 everywhere except 33 at that column, group scales 1)."""
    nsb = k // 256
    out = np.zeros((n, nsb, 210), np.uint8)
    for r in range(n):
        c = int(col_of_row[r])
        b, i = divmod(c, 256)
        for bb in range(nsb):
            q = [32] * 256
            if bb == b:
                q[i] = 33
            out[r, bb] = encode_q6k(d_bits, [1] * 16, q)
    return out


def zero_matrix(type_id, n, k):
    return np.zeros((n, k // 256, 144 if type_id == TYPE_Q4_K else 210), np.uint8)


def perm(n, a, b):
    return np.array([(a * r + b) % n for r in range(n)], np.int64)


def _layer_weights(**over):
    from quantized_gemm_q8_gb300 import synth

    lw = synth.layer_weights(5, 0, DIMS)  # random Q, K (and whatever is not overridden)
    lw.update(over)
    return lw


def pin_rope_frequency(orc):
    # theta 16, head_dim 8: pair i rotates by position * 16^(-2i/8) = position * 2^-i
    hd, L = 8, 3
    x = np.zeros((L, hd))
    x[:, 0::2] = 1.0  # every pair is the unit vector (1, 0)
    r = orc.rope(x, 1, hd, 16.0)
    for p in range(L):
        for i in range(hd // 2):
            a = p * 2.0 ** (-i)
            assert abs(r[p, 2 * i] - math.cos(a)) < 1e-14 and abs(r[p, 2 * i + 1] - math.sin(a)) < 1e-14, \
                (p, i, r[p, 2 * i:2 * i + 2], a)


def pin_attention_scale(orc):
    # one head of 16 dims, two keys: scores 0 and (2 * 2 ln 3) / sqrt(16) = ln 3, so the second
    # key's weight is 3 / (3 + 1) = 0.75, and every output value is 0.75 * 1 + 0.25 * 0
    hd, L = 16, 2
    q = np.zeros((L, hd))
    q[:, 0] = 2.0
    k = np.zeros((L, hd))
    k[1, 0] = 2.0 * math.log(3.0)
    v = np.zeros((L, hd))
    v[1, :] = 1.0
    o = orc.attention(q, k, v, 1, hd)
    np.testing.assert_allclose(o, np.full((L, hd), 0.75), rtol=1e-14, atol=0)


def pin_layer_residuals(orc):
    # O and down are zero matrices: both residual adds return their input, so x_out == x
    # exactly, with and without attention
    from quantized_gemm_q8_gb300 import synth

    lw = _layer_weights(wo=zero_matrix(TYPE_Q4_K, D, D), wdown=zero_matrix(TYPE_Q6_K, D, D))
    x = synth.activations(77, 5, D).astype(np.float64)
    for att in (True, False):
        out, _ = orc.layer(lw, x, DIMS, attention_on=att)
        np.testing.assert_array_equal(out, x)


def pin_layer_attention_half(orc):
    # one token (attention over one key returns V exactly); attn_norm = POW2 and x = PATTERN /
    # POW2, so the codes of RMSNorm(x) * attn_norm are PATTERN; V a permutation, O the identity,
    # gate zero (silu(0) * up = 0, so the FFN adds exactly 0):
    #   x_out = x + d2 * PATTERN[pv],  (q2, d2) = Q8_K(d1 * PATTERN[pv]),  (q1, d1) = Q8_K(RMSNorm(x) * w)
    pv = perm(D, 5, 3)
    lw = _layer_weights(wv=q6k_matrix(D, D, pv), wo=q4k_matrix(D, D, np.arange(D)),
                        wgate=zero_matrix(TYPE_Q4_K, D, D))
    lw["attn_norm"] = POW2.copy()
    lw["ffn_norm"] = np.ones(D, np.float32)
    x = (PATTERN / POW2.astype(np.float64))[None, :]
    q1, d1, _ = orc.quantize_act(x, POW2, DIMS["eps"])
    assert np.array_equal(q1[0], PATTERN)
    v = float(d1[0, 0]) * PATTERN[pv].astype(np.float64)
    q2, d2, _ = orc.quantize_q8k(v[None, :].astype(np.float32))
    assert np.array_equal(q2[0], PATTERN[pv])
    want = x[0] + float(d2[0, 0]) * PATTERN[pv]
    out, ex = orc.layer(lw, x, DIMS, attention_on=True)
    np.testing.assert_array_equal(ex["x_mid"][0], want)
    np.testing.assert_array_equal(out[0], want)


def pin_layer_ffn_half(orc):
    # V zero (the attention adds exactly 0, so x_mid = x); ffn_norm = POW2 and x = PATTERN / POW2,
    # so the codes of RMSNorm(x) * ffn_norm are PATTERN with scale d3; gate = 2 I, up = I, down a
    # permutation:  a = d3 * PATTERN,  h = silu(2a) * a,  x_out = x + d4 * q4[pd], (q4, d4) = Q8_K(h)
    pd = perm(D, 7, 11)
    lw = _layer_weights(wv=zero_matrix(TYPE_Q6_K, D, D), wgate=q4k_matrix(D, D, np.arange(D), d_bits=0x4000),
                        wup=q4k_matrix(D, D, np.arange(D)), wdown=q6k_matrix(D, D, pd))
    lw["attn_norm"] = np.ones(D, np.float32)
    lw["ffn_norm"] = POW2.copy()
    x = (PATTERN / POW2.astype(np.float64))[None, :]
    q3, d3, _ = orc.quantize_act(x, POW2, DIMS["eps"])
    assert np.array_equal(q3[0], PATTERN)
    a = float(d3[0, 0]) * PATTERN.astype(np.float64)
    h = np.array([2.0 * t / (1.0 + math.exp(-2.0 * t)) * t for t in a])
    q4, d4, _ = orc.quantize_q8k(h[None, :].astype(np.float32))
    want = x[0] + float(d4[0, 0]) * q4[0][pd].astype(np.float64)
    for att in (True, False):
        out, ex = orc.layer(lw, x, DIMS, attention_on=att)
        np.testing.assert_array_equal(ex["x_mid"][0], x[0])
        np.testing.assert_allclose(out[0], want, rtol=1e-13, atol=0)


def pin_head_out_norm(orc):
    # vocab = d = 256, W_out = identity (Q6_K). Row r's hidden state is PATTERN_r / POW2 with
    # out_norm = POW2, so its logits are d_r * PATTERN_r: the argmax is the +127 entry and
    # p_max = 1 / sum_v exp(d_r (PATTERN_r[v] - 127)). Without the out_norm weights the codes
    # (and the argmax) would differ. Canvas [mask, mask, 5], block [0, 3), one commit: the row
    # with the larger p_max commits its argmax.
    second = np.roll(PATTERN, 100)
    second = np.where(np.abs(second) < 100, second // 3, second)  # a different confidence
    rows = [PATTERN, second]
    hid = np.stack([r / POW2.astype(np.float64) for r in rows])
    w_out = q6k_matrix(D, D, np.arange(D))
    mask = DIMS["mask_id"]
    want_ids, want_conf = [], []
    for r in range(2):
        q, d, _ = orc.quantize_act(hid[r:r + 1], POW2, DIMS["eps"])
        assert np.array_equal(q[0], rows[r])
        logits = float(d[0, 0]) * rows[r].astype(np.float64)
        want_ids.append(int(np.argmax(rows[r])))
        want_conf.append(1.0 / np.sum(np.exp(logits - logits.max())))
    assert want_ids[0] != want_ids[1] and abs(want_conf[0] - want_conf[1]) > 1e-3 * max(want_conf)
    canvas = np.array([mask, mask, 5], np.int32)
    res = orc.lmhead_commit(hid, canvas, mask, 0, 3, 1, POW2, w_out, DIMS["eps"])
    assert res["ids_rows"].tolist() == want_ids
    np.testing.assert_allclose(res["conf_rows"], want_conf, rtol=1e-13, atol=0)
    first = int(np.argmax(want_conf))
    assert res["pos"].tolist() == [first] and res["id"].tolist() == [want_ids[first]]
    assert canvas.tolist() == [want_ids[0] if first == 0 else mask, want_ids[1] if first == 1 else mask, 5]


PINS = {
    "rope_frequency": pin_rope_frequency,
    "attention_scale": pin_attention_scale,
    "layer_residuals": pin_layer_residuals,
    "layer_attention_half": pin_layer_attention_half,
    "layer_ffn_half": pin_layer_ffn_half,
    "head_out_norm": pin_head_out_norm,
}
