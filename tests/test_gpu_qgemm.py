"""GPU parity of Q8_K quantization and the tcgen05 Q4_K / Q6_K GEMMs against the CPU oracle.

Bars: quantized codes, scales and integer sums bit-exact; GEMM outputs within
2e-3 x the L2 norm of the oracle's output row (the stated tolerance; the integer path
makes the real error ~1e-6 of it). Inputs come from the seeded generator only.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import quantized_gemm_q8_gb300 as dl
from quantized_gemm_q8_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dl.lib()
    torch.cuda.set_device(0)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _packed(t, blocks, n, k):
    return dl.pack_weights(t, _dev(blocks.reshape(-1)), n, k)


def _row_rel_err(y, ref):
    y = np.asarray(y, np.float64)
    den = np.linalg.norm(ref, axis=1, keepdims=True)
    den[den == 0] = 1.0
    return float(np.max(np.abs(y - ref) / den))


# ---- quantization ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,k", [(1, 256), (5, 4096), (148, 4096), (37, 12288), (200, 512)])
def test_quantize_bitexact(rows, k):
    x = synth.activations(1000 + rows + k, rows, k)
    x[0, :256] = 0.0  # an all-zero super-block
    q, d, bs = orc.quantize_q8k(x)
    g = dl.quantize_act(_dev(x), operand=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g["q"].cpu().numpy(), q)
    np.testing.assert_array_equal(g["d"].cpu().numpy(), d)
    np.testing.assert_array_equal(g["bsum"].cpu().numpy(), bs)


def test_quantize_with_rmsnorm():
    rows, k = 148, 4096
    x = synth.activations(77, rows, k) * 3.0
    w = (1.0 + 0.25 * synth.activations(78, 1, k)[0]).astype(np.float32)
    q, d, _ = orc.quantize_act(x, w, 1e-5)
    g = dl.quantize_act(_dev(x), _dev(w), 1e-5)
    gq = g["q"].cpu().numpy().astype(np.int32)
    diff = np.abs(gq - q.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3  # f32 vs f64 normalization: rare ties only
    np.testing.assert_allclose(g["d"].cpu().numpy(), d, rtol=2e-6)


def test_act_operand_layout():
    rows, k = 37, 768
    x = synth.activations(5, rows, k)
    q, d, bs = orc.quantize_q8k(x)
    g = dl.quantize_act(_dev(x))
    torch.cuda.synchronize()
    lp = dl.act_rows(rows)
    buf = g["act"].cpu().numpy()
    nsb = k // 256
    a_bytes = lp * k * 2
    off_j = -(-a_bytes // 1024) * 1024
    off_d = -(-(off_j + nsb * lp * 32) // 1024) * 1024
    A = buf[:a_bytes].view(np.float16).reshape(k // 64, lp, 64).astype(np.float32)
    perm = np.array([0, 2, 1, 3])
    for sbq in range(k // 64):
        for s in range(64):
            kk = 64 * sbq + 4 * (s // 4) + perm[s % 4]
            np.testing.assert_array_equal(A[sbq, :rows, s], q[:, kk].astype(np.float32))
    assert not A[:, rows:, :].any()
    Jp = buf[off_j:off_j + nsb * lp * 32].view(np.float16).reshape(nsb, lp // 8, 2, 8, 8).astype(np.float32)
    Jt = Jp.transpose(0, 1, 3, 2, 4).reshape(nsb, lp, 16)
    np.testing.assert_array_equal(Jt[:, :rows, :], bs.reshape(rows, nsb, 16).transpose(1, 0, 2).astype(np.float32))
    D = buf[off_d:off_d + nsb * lp * 4].view(np.float32).reshape(nsb, lp)
    np.testing.assert_array_equal(D[:, :rows], d.T)
    assert not D[:, rows:].any()


# ---- GEMM -----------------------------------------------------------------------------------

def _case(t, m, n, k, seed):
    w = synth.blocks(t, seed, n, k)
    x = synth.activations(seed + 1, m, k)
    return w, x


def _gemm_check(t, m, n, k, seed, accumulate=False):
    w, x = _case(t, m, n, k, seed)
    q, d, _ = orc.quantize_q8k(x)
    ref = orc.qgemm(t, w, q, d)
    pk = _packed(t, w, n, k)
    g = dl.quantize_act(_dev(x), plain=False)
    y0 = None
    if accumulate:
        y0 = synth.activations(seed + 2, m, n)
        y = _dev(y0)
        dl.qgemm(t, g["act"], m, k, pk, n, y=y, accumulate=True)
        ref = ref + y0
    else:
        y = dl.qgemm(t, g["act"], m, k, pk, n)
    dl.check()
    err = _row_rel_err(y.cpu().numpy(), ref)
    assert err <= TOL, err
    return err


@pytest.mark.parametrize("t", [dl.Q4_K, dl.Q6_K])
@pytest.mark.parametrize("m,n,k", [(16, 4096, 4096), (1, 128, 256), (37, 300, 1024), (148, 512, 4096),
                                   (160, 256, 512), (200, 384, 1024), (32, 1024, 12288), (64, 200, 2048)])
def test_qgemm_parity(t, m, n, k):
    err = _gemm_check(t, m, n, k, 3000 + m + n + k + t)
    assert err < 1e-5  # integer-exact path: only f32 epilogue rounding remains


@pytest.mark.parametrize("t", [dl.Q4_K, dl.Q6_K])
def test_qgemm_accumulate(t):
    _gemm_check(t, 148, 256, 4096, 99 + t, accumulate=True)


@pytest.mark.parametrize("t", [dl.Q4_K, dl.Q6_K])
@pytest.mark.parametrize("m,n,k", [(16, 256, 512), (40, 300, 768), (148, 128, 256)])
def test_qgemm_intsums_bitexact(t, m, n, k):
    w, x = _case(t, m, n, k, 500 + m + n + t)
    q, d, _ = orc.quantize_q8k(x)
    U, J = orc.intsums(t, w, q)  # [m][n][nsb]
    pk = _packed(t, w, n, k)
    g = dl.quantize_act(_dev(x), plain=False)
    s = dl.qgemm_intsums(t, g["act"], m, k, pk, n)
    dl.check()
    s = s.cpu().numpy().astype(np.int64).transpose(0, 2, 3, 1)  # [2][m][n][nsb]
    if t == dl.Q4_K:
        np.testing.assert_array_equal(s[0], U)
        np.testing.assert_array_equal(s[1], J)
    else:  # tensor cores hold I_hi, I_lo with 16*I_hi + I_lo = U - 32*J (signed q-32 form)
        np.testing.assert_array_equal(16 * s[0] + s[1], U - 32 * J)


def test_qgemm_adversarial_extremes():
    # all-max weights and activations: the Q6_K sums stay exact at their worst case
    t, m, n, k = dl.Q6_K, 16, 128, 512
    w = synth.q6k_blocks(1, n, k)
    w[..., :192] = 0xFF  # q = 63 everywhere (ql, qh all ones)
    w[..., 192:208] = 0x80  # scale -128
    x = np.full((m, k), 1.0, np.float32)
    q, d, _ = orc.quantize_q8k(x)
    U, J = orc.intsums(t, w, q)
    pk = _packed(t, w, n, k)
    g = dl.quantize_act(_dev(x), plain=False)
    s = dl.qgemm_intsums(t, g["act"], m, k, pk, n).cpu().numpy().astype(np.int64).transpose(0, 2, 3, 1)
    np.testing.assert_array_equal(16 * s[0] + s[1], U - 32 * J)


# ---- plain Q8_K input (the boundary's (q, d, bsum) form) ----------------------------------------

@pytest.mark.parametrize("rows,k", [(37, 768), (148, 4096), (1, 256)])
def test_pack_act_equals_quantize_operand(rows, k):
    x = synth.activations(900 + rows, rows, k)
    x[0, :256] = 0.0
    nb = dl.act_bytes(rows, k)
    a1 = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    g = dl.quantize_act(_dev(x), act=a1)
    a2 = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    dl.pack_act(g["q"], g["d"], g["bsum"], act=a2)
    dl.check()
    assert torch.equal(a1, a2)


@pytest.mark.parametrize("t", [dl.Q4_K, dl.Q6_K])
@pytest.mark.parametrize("m,n,k", [(148, 512, 4096), (37, 300, 1024)])
def test_qgemm_plain_q8k_input(t, m, n, k):
    w, x = _case(t, m, n, k, 7000 + m + t)
    q, d, bs = orc.quantize_q8k(x)  # the oracle's Q8_K blocks are the input
    ref = orc.qgemm(t, w, q, d)
    pk = _packed(t, w, n, k)
    y = dl.qgemm_plain(t, _dev(q), _dev(d), _dev(bs), pk, n)
    g = dl.quantize_act(_dev(x), plain=False)
    y2 = dl.qgemm(t, g["act"], m, k, pk, n)
    dl.check()
    assert torch.equal(y, y2)  # the same operand, the same kernel
    assert _row_rel_err(y.cpu().numpy(), ref) <= 1e-5
    acc0 = synth.activations(7001 + m, m, n)
    ya = _dev(acc0)
    dl.qgemm_plain(t, _dev(q), _dev(d), _dev(bs), pk, n, y=ya, accumulate=True)
    dl.check()
    assert _row_rel_err(ya.cpu().numpy(), ref + acc0) <= 1e-5


def test_pack_act_reports_inconsistent_sums():
    x = synth.activations(950, 8, 512)
    q, d, bs = orc.quantize_q8k(x)
    bs[3, 17] += 1
    dl.pack_act(_dev(q), _dev(d), _dev(bs))
    with pytest.raises(dl.DllmError) as e:
        dl.check()
    assert e.value.code == dl.E_INVAL and "bsum" in str(e.value)
    dl.check()


def _q4k_fields_block(d_bits, dmin_bits, sc, mn, q):
    from _encoders import encode_q4k
    return encode_q4k(d_bits, dmin_bits, sc, mn, q)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_qgemm_q4k_adversarial_extremes(sign):
    # scale 63, min 63, quant 15 everywhere and activations of one sign (codes +-127): the
    # pages' integer sum I = 63 * 15 * 127 * 256 per super-block exceeds 2^24; the kernel's
    # re-centred chain keeps its partial sums below it, and the sums and outputs stay exact
    t, m, n, k = dl.Q4_K, 16, 128, 512
    blk = _q4k_fields_block(0x3C00, 0x3C00, [63] * 8, [63] * 8, [15] * 256)
    w = np.tile(blk, (n, k // 256, 1))
    x = np.full((m, k), sign, np.float32)
    q, d, _ = orc.quantize_q8k(x)
    assert np.all(q == int(127 * sign))
    U, J = orc.intsums(t, w, q)
    assert abs(int(U[0, 0, 0])) == 63 * 15 * 127 * 256 > 2 ** 24
    pk = _packed(t, w, n, k)
    g = dl.quantize_act(_dev(x), plain=False)
    s = dl.qgemm_intsums(t, g["act"], m, k, pk, n).cpu().numpy().astype(np.int64).transpose(0, 2, 3, 1)
    np.testing.assert_array_equal(s[0], U)
    np.testing.assert_array_equal(s[1], J)
    y = dl.qgemm(t, g["act"], m, k, pk, n)
    dl.check()
    ref = orc.qgemm(t, w, q, d)
    assert _row_rel_err(y.cpu().numpy(), ref) <= 1e-6


def _fold_case():
    """Random Q4_K matrix with hand-set super-block scales that take every branch of the
    kernel's min-term fold: d = 0 (the min term alone), dmin / d = 1024 and 512 and 2^16 (the
    A operand scaled by 2^-k, k = 2, 1, 8), and an all-zero block."""
    n, k = 256, 1024
    w = synth.q4k_blocks(71, n, k)

    def set_dd(row, sb, d_bits, dmin_bits):
        w[row, sb, 0:2] = np.array([d_bits], np.uint16).view(np.uint8)
        w[row, sb, 2:4] = np.array([dmin_bits], np.uint16).view(np.uint8)

    for sb in range(k // 256):
        set_dd(0, sb, 0x0000, 0x3C00)    # d = 0, dmin = 1
        set_dd(1, sb, 0x1400, 0x3C00)    # d = 2^-10, dmin = 1: k = 2
        set_dd(2, sb, 0x2400, 0x4800)    # d = 2^-6, dmin = 8: k = 1
        set_dd(129, sb, 0x0010, 0x2C00)  # d = 2^-20 (subnormal), dmin = 2^-4: k = 8
    w[3, 1] = 0                          # an all-zero block
    set_dd(130, 2, 0x0000, 0x0000)       # d = dmin = 0 with non-zero quants
    return w, n, k


def test_qgemm_q4k_fold_branches():
    w, n, k = _fold_case()
    m = 24
    x = synth.activations(72, m, k)
    q, d, _ = orc.quantize_q8k(x)
    ref = orc.qgemm(dl.Q4_K, w, q, d)
    pk = _packed(dl.Q4_K, w, n, k)
    g = dl.quantize_act(_dev(x), plain=False)
    y = dl.qgemm(dl.Q4_K, g["act"], m, k, pk, n)
    dl.check()
    err = np.abs(y.cpu().numpy() - ref) / np.linalg.norm(ref, axis=1, keepdims=True)
    assert err.max() <= 1e-5, (err.max(), np.unravel_index(np.argmax(err), err.shape))
    U, J = orc.intsums(dl.Q4_K, w, q)
    s = dl.qgemm_intsums(dl.Q4_K, g["act"], m, k, pk, n).cpu().numpy().astype(np.int64).transpose(0, 2, 3, 1)
    dl.check()
    np.testing.assert_array_equal(s[0], U)
    np.testing.assert_array_equal(s[1], J)


def test_qgemm_q4k_unfoldable_block_is_reported():
    # |dmin / d| = 2^24 > 4e6: no f16 shift can carry the min term; the kernel records it in the
    # device error word (no fault) and dllm_check reports DLLM_E_INVAL; the context stays usable
    n, k, m = 128, 512, 8
    w = synth.q4k_blocks(73, n, k)
    w[5, 1, 0:2] = np.array([0x0001], np.uint16).view(np.uint8)  # d = 2^-24
    w[5, 1, 2:4] = np.array([0x3C00], np.uint16).view(np.uint8)  # dmin = 1
    pk = _packed(dl.Q4_K, w, n, k)
    g = dl.quantize_act(_dev(synth.activations(74, m, k)), plain=False)
    dl.qgemm(dl.Q4_K, g["act"], m, k, pk, n)
    with pytest.raises(dl.DllmError) as e:
        dl.check()
    assert e.value.code == dl.E_INVAL and "4e6" in str(e.value)
    dl.check()  # the error word was cleared
    _gemm_check(dl.Q4_K, 16, 128, 256, 4243)


# ---- boundary errors ------------------------------------------------------------------------

def test_errors_are_reported_without_launch():
    x = torch.zeros((4, 256), device="cuda")
    g = dl.quantize_act(x)
    pk = _packed(dl.Q4_K, synth.q4k_blocks(1, 128, 256), 128, 256)
    y = torch.empty((4, 128), device="cuda")
    L = dl.lib()
    s = dl._stream()
    assert L.dllm_qgemm(13, dl._ptr(g["act"]), 4, 256, dl._ptr(pk), 128, dl._ptr(y), 128, 0, None, 0, s) == dl.E_TYPE
    assert "Q4_K" in dl.last_error()
    assert L.dllm_qgemm(12, dl._ptr(g["act"]), 4, 300, dl._ptr(pk), 128, dl._ptr(y), 128, 0, None, 0, s) == dl.E_SHAPE
    host = np.zeros(1 << 16, np.uint8)
    assert L.dllm_qgemm(12, host.ctypes.data_as(dl.C.c_void_p), 4, 256, dl._ptr(pk), 128, dl._ptr(y), 128, 0,
                        None, 0, s) == dl.E_INVAL
    assert L.dllm_quantize_act(dl._ptr(x), 4, 256, 256, None, 1e-5, None, None, None, dl._ptr(g["act"]), 16,
                               s) == dl.E_WORKSPACE
    m, n, k = 148, 1024, 12288
    need = dl.qgemm_workspace_bytes(dl.Q6_K, m, n, k)
    assert need > 0  # this shape is split along k
    xa = torch.zeros((m, k), device="cuda")
    ga = dl.quantize_act(xa, plain=False)
    pk6 = torch.zeros(dl.packed_bytes(dl.Q6_K, n, k), dtype=torch.uint8, device="cuda")
    y2 = torch.empty((m, n), device="cuda")
    assert L.dllm_qgemm(14, dl._ptr(ga["act"]), m, k, dl._ptr(pk6), n, dl._ptr(y2), n, 0, None, 0, s) == dl.E_WORKSPACE
    dl.check()


def test_device_timeout_is_reported_and_context_survives():
    dl.selftest_timeout(200000)
    with pytest.raises(dl.DllmError) as e:
        dl.check()
    assert e.value.code == dl.E_TIMEOUT and "selftest" in str(e.value)
    dl.check()  # the error word was cleared
    _gemm_check(dl.Q4_K, 16, 128, 256, 4242)  # the context still runs kernels


def test_peak_mma_i8_runs():
    # the benchmark's second roofline: a short measurement of mma.sync int8 gives a finite rate
    tops = dl.peak_mma_i8_tops(iters=2000, reps=1)
    dl.check()
    assert 1.0 < tops < 1e5, tops


def test_concurrent_host_threads_match_sequential_results():
    # four host threads, each with its own stream and buffers, quantize and multiply at the same
    # time (ctypes releases the interpreter lock during each call, so the library's host code runs
    # concurrently); every result is bit-identical to the same call made alone
    import threading
    cases = [(dl.Q4_K, 148, 512, 1024), (dl.Q6_K, 37, 768, 2048), (dl.Q4_K, 16, 1024, 512), (dl.Q6_K, 160, 256, 4096)]
    prep, ref = [], []
    for i, (t, m, n, k) in enumerate(cases):
        w, x = _case(t, m, n, k, 7100 + i)
        pk, xd = _packed(t, w, n, k), _dev(x)
        prep.append((t, m, n, k, pk, xd))
        ref.append(dl.qgemm(t, dl.quantize_act(xd, plain=False)["act"], m, k, pk, n))
    torch.cuda.synchronize()
    dl.check()
    out, errs = [None] * len(cases), []

    def work(i):
        try:
            torch.cuda.set_device(0)
            t, m, n, k, pk, xd = prep[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(10):
                    y = dl.qgemm(t, dl.quantize_act(xd, plain=False, stream=s)["act"], m, k, pk, n, stream=s)
            s.synchronize()
            out[i] = y
        except Exception as e:  # reported by the main thread
            errs.append(repr(e))

    ths = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert not errs, errs
    dl.check()
    for i in range(len(cases)):
        assert torch.equal(out[i], ref[i]), cases[i]
