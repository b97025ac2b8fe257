"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every call that
include/dllm.h declares (no compute calls: this runs on CPU)."""
import ctypes
import os
import re

import quantized_gemm_q8_gb300 as dl
from quantized_gemm_q8_gb300 import build as dlbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"DLLM_API\s+[\w\s\*]+?\b(dllm_\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    dlbuild.build()
    lib = ctypes.CDLL(dl.LIB_PATH)
    names = _declared()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_checked_library_exports_every_declared_symbol_and_says_so():
    # the bounds-checked twin is built by the same build() and has the same ABI
    dlbuild.build()
    names = _declared()
    chk = ctypes.CDLL(dlbuild.LIB_CHECKED)
    missing = [n for n in names if not hasattr(chk, n)]
    assert not missing, missing
    chk.dllm_bounds_checked.restype = ctypes.c_int
    reg = ctypes.CDLL(dlbuild.LIB)
    reg.dllm_bounds_checked.restype = ctypes.c_int
    assert chk.dllm_bounds_checked() == 1 and reg.dllm_bounds_checked() == 0


def test_binding_covers_declared_symbols():
    names = set(_declared())
    assert names <= set(dl._SIGS), sorted(names - set(dl._SIGS))


def test_host_only_calls():
    dlbuild.build()
    L = dl.lib()
    assert L.dllm_version() >= 100
    assert L.dllm_packed_bytes(12, 4096, 4096) == 4096 * 16 * 144
    assert L.dllm_packed_bytes(14, 126464, 4096) == 126464 * 16 * 210
    assert L.dllm_packed_bytes(13, 128, 256) == 0
    assert L.dllm_act_rows(148) == 160 and L.dllm_act_rows(16) == 32 and L.dllm_act_rows(512) == 512
    assert L.dllm_act_bytes(148, 4096) >= 160 * 4096 * 2
    assert L.dllm_act_bytes(148, 300) == 0


def test_host_only_size_queries_of_the_cache_and_the_head():
    # size queries read only the model's dimensions: no device is touched
    dlbuild.build()
    L = dl.lib()
    m = dl._Model(n_layers=32, d_model=4096, n_heads=32, head_dim=128, d_ff=12288, vocab=126464, mask_id=126336,
                  eps=1e-5, rope_theta=500000.0)
    ref = ctypes.byref(m)
    assert L.dllm_kv_cache_bytes(ref, 148) == 32 * 2 * 148 * 4096 * 4  # f32 K and V per layer
    assert L.dllm_kv_cache_bytes(ref, 0) == 0
    blk = L.dllm_denoise_cached_workspace_bytes(ref, 148, 32)
    assert blk >= L.dllm_denoise_workspace_bytes(ref, 148, 32) > 0
    assert L.dllm_denoise_cached_workspace_bytes(ref, 148, 149) == 0  # more block rows than the canvas
    # the head's workspace holds, per row and tile quadrant, the softmax, entropy and draw partials
    P = (126464 + 127) // 128 * 4
    assert L.dllm_lmhead_workspace_bytes(32, 126464, 4096) >= 7 * P * 32 * 4
    assert L.dllm_lmhead_workspace_bytes(161, 126464, 4096) == 0
