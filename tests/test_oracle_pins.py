"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each check ties the oracle to something other than itself: hand-worked block
bytes (tests/golden), an independent encoder that packs known fields into
the GGUF bytes, numpy's own f16 decoding, exact rational arithmetic,
closed forms and invariants of the method.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
from quantized_gemm_q8_gb300 import synth

from _encoders import encode_q4k, encode_q6k, f16_bits, f16_val  # noqa: F401

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


def q4k_expected(d_bits, dmin_bits, sc, mn, q):
    d, dmin = f16_val(d_bits), f16_val(dmin_bits)
    return np.array([d * sc[i // 32] * q[i] - dmin * mn[i // 32] for i in range(256)])


def q6k_expected(d_bits, sc, q):
    d = f16_val(d_bits)
    return np.array([d * sc[8 * (i // 128) + (i % 128) // 16] * (int(q[i]) - 32) for i in range(256)])


# ---- Q4_K -------------------------------------------------------------------------------------

def test_q4k_scales_handworked():
    g = _golden("q4k_scales_handworked.txt")
    blk = np.zeros(144, np.uint8)
    blk[4:16] = [int(b, 16) for b in g["scales_bytes"]]
    sc, mn, _ = orc.q4k_fields(blk)
    assert sc.tolist() == [int(v) for v in g["scale"]]
    assert mn.tolist() == [int(v) for v in g["min"]]


def test_q4k_closed_form_block():
    # d = 1, dmin = 0.5, scale_j = j+1, min_j = 2j, q_i = i mod 16  ->  w_i = (j+1)(i%16) - j
    sc = [j + 1 for j in range(8)]
    mn = [2 * j for j in range(8)]
    q = [i % 16 for i in range(256)]
    blk = encode_q4k(0x3C00, 0x3800, sc, mn, q)
    w = orc.dequant(orc.TYPE_Q4_K, blk[None, None, :])[0]
    want = np.array([(i // 32 + 1) * (i % 16) - (i // 32) for i in range(256)], np.float64)
    np.testing.assert_array_equal(w, want)


@pytest.mark.parametrize("j", range(8))
def test_q4k_single_subblock_high_bits(j):
    # scale = min = 63 in sub-block j only: exercises the 2 high bits packed for j >= 4
    sc = [0] * 8
    mn = [0] * 8
    sc[j], mn[j] = 63, 63
    q = [15] * 256
    blk = encode_q4k(0x3C00, 0x3C00, sc, mn, q)
    w = orc.dequant(orc.TYPE_Q4_K, blk[None, None, :])[0]
    want = np.zeros(256)
    want[32 * j:32 * j + 32] = 63 * 15 - 63
    np.testing.assert_array_equal(w, want)


def test_q4k_random_fields_roundtrip():
    rng = np.random.default_rng(7)
    for _ in range(20):
        sc = rng.integers(0, 64, 8).tolist()
        mn = rng.integers(0, 64, 8).tolist()
        q = rng.integers(0, 16, 256).tolist()
        db, mb = int(rng.integers(0x0400, 0x7800)), int(rng.integers(0x0001, 0x7800))
        blk = encode_q4k(db, mb, sc, mn, q)
        s2, m2, q2 = orc.q4k_fields(blk)
        assert s2.tolist() == sc and m2.tolist() == mn and q2.tolist() == q
        w = orc.dequant(orc.TYPE_Q4_K, blk[None, None, :])[0]
        np.testing.assert_array_equal(w, q4k_expected(db, mb, sc, mn, q))


def test_f16_subnormal_and_sign():
    # d = smallest subnormal 2^-24, dmin = -2.0 (sign bit)
    sc = [1] * 8
    mn = [1] * 8
    q = [1] * 256
    blk = encode_q4k(0x0001, f16_bits(-2.0), sc, mn, q)
    w = orc.dequant(orc.TYPE_Q4_K, blk[None, None, :])[0]
    np.testing.assert_array_equal(w, np.full(256, 2.0 ** -24 + 2.0))


# ---- Q6_K -------------------------------------------------------------------------------------

def test_q6k_handworked():
    g = _golden("q6k_handworked.txt")
    blk = np.zeros(210, np.uint8)
    for item in g["bytes"]:
        name, val = item.split("=")
        off = int(name[2:]) + (128 if name.startswith("qh") else 0)
        blk[off] = int(val, 16)
    blk[192:208] = np.array([int(v) for v in g["scales"]], np.int8).view(np.uint8)
    blk[208:210] = np.array([0x3C00], np.uint16).view(np.uint8)
    w = orc.dequant(orc.TYPE_Q6_K, blk[None, None, :])[0]
    for item in g["expect"]:
        i, v = item.split(":")
        assert w[int(i)] == float(v), (i, w[int(i)], v)


def test_q6k_random_fields_roundtrip():
    rng = np.random.default_rng(11)
    for it in range(20):
        sc = rng.integers(-128, 128, 16).tolist()
        if it == 0:
            sc[3] = -128
        q = rng.integers(0, 64, 256).tolist()
        db = int(rng.integers(0x0400, 0x7800))
        blk = encode_q6k(db, sc, q)
        s2, q2 = orc.q6k_fields(blk)
        assert s2.tolist() == sc and q2.tolist() == q
        w = orc.dequant(orc.TYPE_Q6_K, blk[None, None, :])[0]
        np.testing.assert_array_equal(w, q6k_expected(db, sc, q))


def test_q6k_t_patterns():
    # q values that set each t slot's nibble choice and high bits distinctly
    q = [(i * 37 + (i // 32)) % 64 for i in range(256)]
    sc = [1] * 16
    blk = encode_q6k(0x3C00, sc, q)
    w = orc.dequant(orc.TYPE_Q6_K, blk[None, None, :])[0]
    np.testing.assert_array_equal(w, np.array(q, np.float64) - 32)


# ---- Q8_K -------------------------------------------------------------------------------------

def test_q8k_zero_block():
    q, d, bs = orc.quantize_q8k(np.zeros((1, 256), np.float32))
    assert not q.any() and d[0, 0] == 0.0 and not bs.any()


def test_q8k_spike_and_extremes():
    x = np.zeros((2, 256), np.float32)
    x[0, 7] = 5.0
    x[1, 0], x[1, 1] = 3.0, -3.0
    q, d, bs = orc.quantize_q8k(x)
    assert q[0, 7] == 127 and np.count_nonzero(q[0]) == 1
    assert d[0, 0] == np.float32(5.0) / np.float32(127.0)
    assert q[1, 0] == 127 and q[1, 1] == -127
    assert bs[0, 0] == 127 and bs[1, 0] == 0


def test_q8k_round_half_even():
    # amax = 127 -> iscale = 1 exactly, so the codes are rint(x) with ties to even
    x = np.zeros((1, 256), np.float32)
    vals = [127.0, 2.5, 3.5, -2.5, -0.5, 126.5, -126.5, 0.49999997]
    x[0, :len(vals)] = vals
    q, d, _ = orc.quantize_q8k(x)
    assert q[0, :len(vals)].tolist() == [127, 2, 4, -2, 0, 126, -126, 0]
    assert d[0, 0] == np.float32(1.0)


def test_q8k_error_bound_and_bsums():
    x = synth.activations(3, 8, 1024)
    q, d, bs = orc.quantize_q8k(x)
    recon = q.reshape(8, 4, 256).astype(np.float64) * d[:, :, None].astype(np.float64)
    err = np.abs(recon - x.reshape(8, 4, 256))
    assert np.all(err <= d[:, :, None] * (0.5 + 1e-6) + 1e-12)
    np.testing.assert_array_equal(bs, q.reshape(8, 64, 16).astype(np.int64).sum(-1))
    amax = np.abs(x.reshape(8, 4, 256)).max(-1)
    assert np.all(np.abs(q.reshape(8, 4, 256)).max(-1) == 127)
    np.testing.assert_array_equal(d, (amax / np.float32(127.0)).astype(np.float32))


# ---- GEMM -------------------------------------------------------------------------------------

@pytest.mark.parametrize("t", [orc.TYPE_Q4_K, orc.TYPE_Q6_K])
def test_qgemm_equals_dequant_then_dot(t):
    n, k, m = 37, 768, 5
    w = synth.blocks(t, 101 + t, n, k)
    x = synth.activations(202 + t, m, k)
    q, d, _ = orc.quantize_q8k(x)
    y = orc.qgemm(t, w, q, d)
    W = orc.dequant(t, w).reshape(n, k)
    A = q.astype(np.float64) * np.repeat(d.astype(np.float64), 256, axis=1)
    ref = A @ W.T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * (np.abs(A) @ np.abs(W).T).max())
    rows = np.array([36, 0, 5])
    np.testing.assert_array_equal(orc.qgemm(t, w, q, d, rows=rows), y[:, rows])


@pytest.mark.parametrize("t", [orc.TYPE_Q4_K, orc.TYPE_Q6_K])
def test_intsums_compose_to_gemm(t):
    n, k, m = 19, 1024, 4
    w = synth.blocks(t, 303 + t, n, k)
    x = synth.activations(404 + t, m, k)
    q, d, _ = orc.quantize_q8k(x)
    U, J = orc.intsums(t, w, q)
    c0, c1 = orc.block_scales(t, w)
    y_int = (d.astype(np.float64)[:, None, :] * (c0[None] * U - c1[None] * J)).sum(-1)
    y = orc.qgemm(t, w, q, d)
    np.testing.assert_allclose(y_int, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_q4k_intsums_brute_force():
    rng = np.random.default_rng(5)
    for m, n, k in [(1, 1, 256), (2, 3, 512), (3, 2, 256)]:
        fields, wb = [], []
        for _ in range(n):
            row = []
            for _ in range(k // 256):
                sc = rng.integers(0, 64, 8).tolist()
                mn = rng.integers(0, 64, 8).tolist()
                q = rng.integers(0, 16, 256).tolist()
                db, mb = int(rng.integers(0x0400, 0x3C00)), int(rng.integers(0x0400, 0x3C00))
                row.append(encode_q4k(db, mb, sc, mn, q))
                fields.append((db, mb, sc, mn, q))
            wb.append(np.stack(row))
        wb = np.stack(wb)
        a = rng.integers(-127, 128, (m, k)).astype(np.int8)
        da = rng.uniform(0.001, 0.1, (m, k // 256)).astype(np.float32)
        U, J = orc.intsums(orc.TYPE_Q4_K, wb, a)
        y = orc.qgemm(orc.TYPE_Q4_K, wb, a, da)
        for mm in range(m):
            for nn in range(n):
                tot = Fraction(0)
                for b in range(k // 256):
                    db, mb, sc, mn, q = fields[nn * (k // 256) + b]
                    u = sum(sc[i // 32] * q[i] * int(a[mm, 256 * b + i]) for i in range(256))
                    jj = sum(mn[i // 32] * int(a[mm, 256 * b + i]) for i in range(256))
                    assert U[mm, nn, b] == u and J[mm, nn, b] == jj
                    tot += Fraction(float(da[mm, b])) * (Fraction(f16_val(db)) * u - Fraction(f16_val(mb)) * jj)
                assert abs(Fraction(y[mm, nn]) - tot) <= abs(tot) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 18)


def test_q6k_intsums_brute_force():
    rng = np.random.default_rng(6)
    m, n, k = 2, 2, 512
    fields, wb = [], []
    for _ in range(n):
        row = []
        for _ in range(k // 256):
            sc = rng.integers(-128, 128, 16).tolist()
            q = rng.integers(0, 64, 256).tolist()
            db = int(rng.integers(0x0400, 0x3C00))
            row.append(encode_q6k(db, sc, q))
            fields.append((db, sc, q))
        wb.append(np.stack(row))
    wb = np.stack(wb)
    a = rng.integers(-127, 128, (m, k)).astype(np.int8)
    da = rng.uniform(0.001, 0.1, (m, k // 256)).astype(np.float32)
    U, J = orc.intsums(orc.TYPE_Q6_K, wb, a)
    y = orc.qgemm(orc.TYPE_Q6_K, wb, a, da)
    for mm in range(m):
        for nn in range(n):
            tot = Fraction(0)
            for b in range(k // 256):
                db, sc, q = fields[nn * (k // 256) + b]
                g = lambda i: 8 * (i // 128) + (i % 128) // 16
                u = sum(sc[g(i)] * q[i] * int(a[mm, 256 * b + i]) for i in range(256))
                jj = sum(sc[g(i)] * int(a[mm, 256 * b + i]) for i in range(256))
                assert U[mm, nn, b] == u and J[mm, nn, b] == jj
                tot += Fraction(float(da[mm, b])) * Fraction(f16_val(db)) * (u - 32 * jj)
            assert abs(Fraction(y[mm, nn]) - tot) <= abs(tot) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 18)


# ---- layer maths ------------------------------------------------------------------------------

def test_rmsnorm_constant_vector():
    x = np.full((2, 512), -3.0)
    w = np.linspace(0.5, 1.5, 512).astype(np.float32)
    out = orc.rmsnorm(x, w, 1e-5)
    np.testing.assert_allclose(out, np.tile(-3.0 / math.sqrt(9.0 + 1e-5) * w.astype(np.float64), (2, 1)), rtol=1e-14)


def test_rope_identities():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 2 * 8))
    # theta -> infinity: only pair 0 rotates (angle = position)
    r = orc.rope(x, 2, 8, 1e300)
    for p in range(6):
        for h in range(2):
            v, o = x[p, 8 * h:8 * h + 8], r[p, 8 * h:8 * h + 8]
            c, s = math.cos(p), math.sin(p)
            assert abs(o[0] - (v[0] * c - v[1] * s)) < 1e-14 and abs(o[1] - (v[0] * s + v[1] * c)) < 1e-14
            np.testing.assert_allclose(o[2:], v[2:], rtol=0, atol=1e-15)
    # theta = 1: every pair rotates by the position; norms preserved
    r1 = orc.rope(x, 2, 8, 1.0)
    np.testing.assert_allclose(np.linalg.norm(r1, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    p = 3
    c, s = math.cos(p), math.sin(p)
    np.testing.assert_allclose(r1[p, 2], x[p, 2] * c - x[p, 3] * s, rtol=1e-13)
    np.testing.assert_array_equal(orc.rope(x, 2, 8, 500000.0)[0], x[0])  # position 0 untouched


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    L, nh, hd = 7, 2, 8
    q = rng.standard_normal((L, nh * hd))
    k = np.tile(rng.standard_normal((1, nh * hd)), (L, 1))  # identical keys
    v = rng.standard_normal((L, nh * hd))
    o = orc.attention(q, k, v, nh, hd)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (L, 1)), rtol=1e-13)
    # one dominant key per head: output = that key's value row
    k2 = np.zeros((L, nh * hd))
    k2[4] = 1e3 * q[0]
    o2 = orc.attention(q, k2, v, nh, hd)
    np.testing.assert_allclose(o2[0], v[4], rtol=1e-10)


def test_swiglu_values():
    g = np.array([0.0, 1.0, -1.0, 40.0])
    u = np.array([3.0, 2.0, 2.0, 0.5])
    h = orc.swiglu(g, u)
    np.testing.assert_allclose(h, [0.0, 2.0 / (1 + math.exp(-1)), -2.0 / (1 + math.e), 20.0], rtol=1e-15)


def test_embed_is_row_decode():
    t = synth.q4k_blocks(9, 50, 512)
    ids = np.array([3, 49, 0, 3], np.int32)
    x = orc.embed(t, ids)
    W = orc.dequant(orc.TYPE_Q4_K, t).reshape(50, 512)
    np.testing.assert_array_equal(x, W[ids])
    with pytest.raises(ValueError):
        orc.embed(t, np.array([50], np.int32))


# ---- confidence and commit --------------------------------------------------------------------

def test_commit_tiny_handworked():
    g = _golden("commit_tiny.txt")
    logits = np.array([[float(v) for v in g[f"logits{i}"]] for i in range(4)])
    ids, conf, t1, t2 = orc.row_confidence(logits)
    assert ids.tolist() == [2, 0, 0, 6]
    np.testing.assert_allclose(conf[[0, 1, 3]], [math.e ** 2 / (math.e ** 2 + 7), 0.125,
                                                 math.e ** 5 / (2 * math.e ** 5 + 6)], rtol=1e-14)
    assert t1[3] == t2[3] == 5.0
    for k, key in [(2, "k2"), (3, "k3")]:
        canvas = np.array([int(v) for v in g["canvas"]], np.int32)
        conf_pos = conf.copy()
        pos, tid = orc.commit_topk(canvas, 7, 0, 4, conf_pos, ids, k)
        assert pos.tolist() == [int(v) for v in g[f"{key}_pos"]]
        assert canvas.tolist() == [int(v) for v in g[f"{key}_canvas"]]
    canvas = np.array([7, 7, 7, 7], np.int32)
    pos, _ = orc.commit_topk(canvas, 7, 0, 4, np.array([0.3, 0.3, 0.1, 0.3]), np.zeros(4, np.int32), 2)
    assert pos.tolist() == [0, 1]  # equal confidence -> lowest positions first


def test_neg_entropy_closed_forms():
    # uniform over V tokens: H = log V; two equal logits far above the rest: H = log 2; one
    # logit 60 above 999 others: H = 999 e^-60 (60 + 1) to first order (below 1e-20)
    V = 1000
    ne = orc.row_neg_entropy(np.vstack([np.full(V, 0.37), np.r_[[3.0, 3.0], np.full(V - 2, -1e4)],
                                        np.r_[[60.0], np.zeros(V - 1)]]))
    np.testing.assert_allclose(ne[:2], [-math.log(V), -math.log(2.0)], rtol=1e-13)
    assert -1e-20 < ne[2] <= 0.0


def test_neg_entropy_matches_library_and_is_shift_invariant():
    scipy_special = pytest.importorskip("scipy.special")
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(7)
    logits = rng.normal(0.0, 3.0, size=(5, 777))
    ref = -scipy_stats.entropy(scipy_special.softmax(logits, axis=1), axis=1)  # natural log
    ne = orc.row_neg_entropy(logits)
    np.testing.assert_allclose(ne, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.row_neg_entropy(logits + 123.5), ne, rtol=1e-12, atol=1e-12)
    assert np.all(ne <= 0.0) and np.all(ne >= -math.log(777) - 1e-12)


def test_entropy_ranking_commit_order():
    # the entropy ranking commits the most peaked rows first: one-hot-like < 2-way < 4-way
    V = 16
    rows = np.full((4, V), -1e4)
    rows[0, :4] = 0.0          # uniform over 4
    rows[1, 5] = 0.0           # one token
    rows[2, [1, 9]] = 0.0      # uniform over 2
    rows[3, :] = 0.0           # uniform over 16
    ids, _, _, _ = orc.row_confidence(rows)
    conf = orc.row_neg_entropy(rows)
    canvas = np.array([7, 7, 7, 7], np.int32)
    pos, tid = orc.commit_topk(canvas, 7, 0, 4, conf, ids, 3)
    assert pos.tolist() == [1, 2, 0] and tid.tolist() == [5, 1, 0]
    assert canvas.tolist() == [0, 5, 1, 7]


def test_splitmix64_published_first_output():
    g = _golden("splitmix64.txt")
    assert orc.splitmix64_at(int(g["seed"][0]), 0) == int(g["first_output"][0], 16)


def test_splitmix64_counter_form_is_the_stream():
    # output c of the stream = output 0 of the stream started c increments later
    gamma = 0x9E3779B97F4A7C15
    for seed, c in [(0, 1), (12345, 7), (2**63 + 5, 1000)]:
        assert orc.splitmix64_at(seed, c) == orc.splitmix64_at((seed + c * gamma) % 2**64, 0)
    outs = {orc.splitmix64_at(99, c) for c in range(4096)}
    assert len(outs) == 4096  # a bijective finalizer over distinct states


def test_gumbel_max_draws_follow_softmax_over_temperature():
    # 40000 draws (one per canvas position) from V = 5 logits at T = 0.7: the frequencies match
    # softmax(l / T) (chi-square, 4 degrees of freedom, far below the 1e-4 critical value 23.5)
    l = np.array([0.0, 1.0, -0.5, 2.0, 0.3])
    n, T = 40000, 0.7
    ids, conf, _ = orc.row_sample(np.tile(l, (n, 1)), T, 2024, 5, np.arange(n))
    p = np.exp(l / T) / np.exp(l / T).sum()
    cnt = np.bincount(ids, minlength=5)
    chi2 = float(((cnt - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 23.5, (cnt, n * p, chi2)
    # the confidence is the drawn token's probability under the untempered softmax
    np.testing.assert_allclose(conf, (np.exp(l) / np.exp(l).sum())[ids], rtol=1e-13)


def test_gumbel_max_limits():
    rng = np.random.default_rng(3)
    logits = rng.normal(0.0, 1.0, size=(64, 50))
    # T -> 0: the draw is the argmax (logit gaps / T dwarf the noise)
    ids0 = orc.row_confidence(logits)[0]
    ids, _, _ = orc.row_sample(logits, 1e-7, 7, 0, np.arange(64))
    assert np.array_equal(ids, ids0)
    # equal logits: every token is drawn, each with probability 1 / V
    ids, conf, _ = orc.row_sample(np.zeros((20000, 4)), 1.3, 11, 2, np.arange(20000))
    np.testing.assert_allclose(conf, 0.25, rtol=1e-15)
    assert np.all(np.abs(np.bincount(ids, minlength=4) / 20000 - 0.25) < 0.02)
    # the draw depends on (seed, step, position) and on nothing else
    a, _, _ = orc.row_sample(logits, 0.9, 5, 1, np.arange(64))
    b, _, _ = orc.row_sample(logits, 0.9, 5, 1, np.arange(64))
    c, _, _ = orc.row_sample(logits, 0.9, 5, 2, np.arange(64))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


TINY = dict(n_layers=2, d_model=256, n_heads=2, head_dim=128, d_ff=512, vocab=300, mask_id=297, eps=1e-5,
            rope_theta=500000.0)


def _tiny_model(seed):
    lws = [synth.layer_weights(seed, i, TINY) for i in range(TINY["n_layers"])]
    for i, lw in enumerate(lws):  # norm weights away from 1 so that every norm matters
        lw["attn_norm"] = (1.0 + 0.2 * synth.activations(seed + 10 + i, 1, TINY["d_model"])[0]).astype(np.float32)
        lw["ffn_norm"] = (1.0 + 0.2 * synth.activations(seed + 20 + i, 1, TINY["d_model"])[0]).astype(np.float32)
    table = synth.embed_weights(seed, TINY)
    canvas = synth.canvas(seed, prompt_len=8, gen_len=16, mask_id=TINY["mask_id"], prompt_max=290)
    return lws, table, canvas


def test_cached_step_right_after_refresh_equals_the_full_forward():
    # nothing has changed since the refresh, so the cached K/V equal the fresh ones and the block
    # rows of the cached step reproduce the uncached forward (to rounding)
    lws, table, canvas = _tiny_model(71)
    cache = []
    x_full = orc.forward_cached(lws, table, canvas, TINY, 8, 16, True, cache)
    x_blk = orc.forward_cached(lws, table, canvas, TINY, 8, 16, False, cache)
    np.testing.assert_allclose(x_blk[8:16], x_full[8:16], rtol=1e-12, atol=1e-12)
    assert np.all(x_blk[:8] == 0) and np.all(x_blk[16:] == 0)


def test_cached_step_sees_the_block_but_not_stale_rows():
    lws, table, canvas = _tiny_model(72)
    cache = []
    orc.forward_cached(lws, table, canvas, TINY, 8, 16, True, cache)
    # a token outside the block changes after the refresh: the cached step cannot see it
    outside = canvas.copy()
    outside[20] = 5
    a = orc.forward_cached(lws, table, canvas, TINY, 8, 16, False, [(k.copy(), v.copy()) for k, v in cache])
    b = orc.forward_cached(lws, table, outside, TINY, 8, 16, False, [(k.copy(), v.copy()) for k, v in cache])
    np.testing.assert_array_equal(a[8:16], b[8:16])
    fresh = orc.forward_cached(lws, table, outside, TINY, 8, 16, True, [])
    assert np.abs(fresh[8:16] - a[8:16]).max() > 1e-6  # the uncached step does see it
    # a token inside the block changes: the cached step recomputes the block and sees it
    inside = canvas.copy()
    inside[10] = 5
    c = orc.forward_cached(lws, table, inside, TINY, 8, 16, False, [(k.copy(), v.copy()) for k, v in cache])
    assert np.abs(c[8:16] - a[8:16]).max() > 1e-6


def test_commit_invariants_random():
    rng = np.random.default_rng(3)
    L, mask = 148, 126336
    for trial in range(20):
        canvas = rng.integers(0, 1000, L).astype(np.int32)
        masked = rng.random(L) < 0.6
        canvas[masked] = mask
        b0 = 20 + 32 * (trial % 4)
        b1 = b0 + 32
        conf = rng.random(L)
        ids = rng.integers(0, 126464, L).astype(np.int32)
        before = canvas.copy()
        k = int(rng.integers(1, 8))
        pos, tid = orc.commit_topk(canvas, mask, b0, b1, conf, ids, k)
        cand = [p for p in range(b0, b1) if before[p] == mask]
        assert len(pos) == min(k, len(cand))
        assert all(b0 <= p < b1 and before[p] == mask for p in pos)
        assert len(set(pos.tolist())) == len(pos)
        rest = [p for p in cand if p not in set(pos.tolist())]
        if rest and len(pos):
            assert conf[pos].min() >= conf[rest].max()
        np.testing.assert_array_equal(canvas[pos], ids[pos])
        untouched = np.ones(L, bool)
        untouched[pos] = False
        np.testing.assert_array_equal(canvas[untouched], before[untouched])


def test_transfer_counts():
    assert orc.transfer_counts(32, 8).tolist() == [4] * 8
    assert orc.transfer_counts(10, 4).tolist() == [3, 3, 2, 2]
    assert orc.transfer_counts(3, 5).tolist() == [1, 1, 1, 0, 0]
    for masked, steps in [(128, 32), (37, 8), (1, 1)]:
        c = orc.transfer_counts(masked, steps)
        assert c.sum() == masked and c.max() - c.min() <= 1 and np.all(np.diff(c) <= 0)


def test_generator_is_deterministic_and_in_range():
    a = synth.q4k_blocks(5, 3, 512)
    b = synth.q4k_blocks(5, 3, 512)
    np.testing.assert_array_equal(a, b)
    d = a[..., 0:2].copy().view(np.uint16).ravel()
    assert np.all((d >> 10) == 1)  # f16 exponent field 1 -> [2^-14, 2^-13)
    x = synth.activations(1, 64, 1024)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    cv = synth.canvas(1)
    assert cv.size == 148 and np.all(cv[20:] == 126336) and np.all(cv[:20] < 126000)
