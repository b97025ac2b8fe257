"""The allocation-free GEMM entry point (dllm_qgemm_noalloc) against the workspace one.

It exists for callers that cannot allocate device memory at call time (a server that reserves
all memory at start-up, a plugin interface without a scratch buffer, a loop that must not call
cudaMalloc). It must give the same result as dllm_qgemm, within the GEMM tolerance used by the
other tests, on consecutive calls that reuse its fixed scratch array with different shapes.
This file is collected last so that a failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
import quantized_gemm_q8_gb300 as dl
from quantized_gemm_q8_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _case(t, m, n, k, seed):
    w = synth.blocks(t, seed, n, k)
    x = synth.activations(seed + 1, m, k)
    pk = dl.pack_weights(t, torch.from_numpy(w.reshape(-1)).cuda(), n, k)
    act = dl.quantize_act(torch.from_numpy(x).cuda(), plain=False)["act"]
    return w, x, pk, act


def _noalloc_c(t, act, m, k, pk, n, y, accumulate=0):
    """Call the entry point through the C ABI directly."""
    L = dl.lib()
    rc = L.dllm_qgemm_noalloc(t, ctypes.c_void_p(act.data_ptr()), m, k, ctypes.c_void_p(pk.data_ptr()), n,
                              ctypes.c_void_p(y.data_ptr()), y.stride(0), accumulate,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dl.last_error()


def _rel(a, b):
    den = np.linalg.norm(b, axis=1, keepdims=True)
    den[den == 0] = 1.0
    return float(np.max(np.abs(np.asarray(a, np.float64) - b) / den))


def test_noalloc_matches_workspace_gemm_on_two_calls_in_a_row():
    torch.cuda.set_device(0)
    cases = [(dl.Q4_K, 148, 8192, 4096, 7001), (dl.Q6_K, 37, 300, 1024, 7002)]
    prepared = [_case(*c) for c in cases]
    for (t, m, n, k, seed), (w, x, pk, act) in zip(cases, prepared):  # two consecutive calls
        y_na = torch.full((m, n), float("nan"), device="cuda")
        _noalloc_c(t, act, m, k, pk, n, y_na)
        y_ws = dl.qgemm(t, act, m, k, pk, n)
        dl.check()
        a, b = y_na.cpu().numpy(), y_ws.cpu().numpy()
        assert np.isfinite(a).all()
        assert _rel(a, b.astype(np.float64)) <= TOL
        q, d, _ = orc.quantize_q8k(x)
        assert _rel(a, orc.qgemm(t, w, q, d)) <= TOL


def test_noalloc_accumulate_and_size_limit():
    torch.cuda.set_device(0)
    t, m, n, k = dl.Q4_K, 16, 4096, 4096
    w, x, pk, act = _case(t, m, n, k, 7003)
    y0 = torch.from_numpy(synth.activations(7004, m, n)).cuda()
    y = y0.clone()
    _noalloc_c(t, act, m, k, pk, n, y, accumulate=1)
    ref = dl.qgemm(t, act, m, k, pk, n) + y0
    dl.check()
    assert _rel(y.cpu().numpy(), ref.cpu().numpy().astype(np.float64)) <= TOL
    # an output larger than the fixed 32 MiB array is refused with a clear error, nothing launched
    big_m, big_n = 4096, 4096
    yb = torch.empty(1, device="cuda")
    rc = dl.lib().dllm_qgemm_noalloc(t, ctypes.c_void_p(act.data_ptr()), big_m, k, ctypes.c_void_p(pk.data_ptr()),
                                     big_n, ctypes.c_void_p(yb.data_ptr()), big_n, 0,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dl.E_SHAPE and "scratch" in dl.last_error()


@pytest.mark.parametrize("accumulate", [0, 1])
def test_noalloc_single_split_fallback(accumulate):
    # the workspace plan splits k four ways (partials above the 32 MiB array) while the output
    # itself fits: the entry point falls back to one split, written straight into the array
    torch.cuda.set_device(0)
    t, m, n, k = dl.Q6_K, 148, 40960, 12288
    limit = 32 << 20
    assert dl.qgemm_workspace_bytes(t, m, n, k) > limit >= m * n * 4  # the branch under test
    w = synth.blocks(t, 7005, n, k)
    x = synth.activations(7006, m, k)
    pk = dl.pack_weights(t, torch.from_numpy(w.reshape(-1)).cuda(), n, k)
    act = dl.quantize_act(torch.from_numpy(x).cuda(), plain=False)["act"]
    y0 = synth.activations(7007, m, n) if accumulate else np.zeros((m, n), np.float32)
    y = torch.from_numpy(y0).cuda()
    _noalloc_c(t, act, m, k, pk, n, y, accumulate=accumulate)
    ref_ws = dl.qgemm(t, act, m, k, pk, n)
    dl.check()
    got = y.cpu().numpy().astype(np.float64) - (y0 if accumulate else 0.0)
    assert _rel(got, ref_ws.cpu().numpy().astype(np.float64)) <= 1e-5
    rows = np.array([0, 1, 127, 128, 20000, n - 1])  # weight rows checked against the oracle
    q, d, _ = orc.quantize_q8k(x)
    assert _rel(got[:, rows], orc.qgemm(t, w, q, d, rows=rows)) <= TOL
