"""The bounds-checked build (libdllm_checked.so: the same sources with DLLM_BOUNDS_CHECK, every
global-memory access of every kernel checked against the extent of its buffer, the extents
computed on the host from each call's shapes).

1. The check works: a store outside its declared span is skipped and reported as DLLM_E_BOUNDS
   with its source site, and the context stays usable. The span is declared smaller than the
   real buffer, so no store ever leaves real memory: nothing can fault.
2. The library's kernels stay inside their buffers: the GPU parity tests that reach every kernel
   (quantization and packing, the GEMM in every token tile and mode, the split-K reduction, the
   LM head with its merge, sampling and entropy, the tensor-core and chunked attention and their
   merge, the row kernels, RoPE and embedding, the cached step, the allocation-free entry point)
   run against the checked library in a child process and must all pass; any access outside a
   buffer would make its dllm_check fail.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

import quantized_gemm_q8_gb300 as dl

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child(code_or_args, timeout):
    env = dict(os.environ, DLLM_CHECKED="1")
    cmd = [sys.executable] + (["-c", code_or_args] if isinstance(code_or_args, str) else code_or_args)
    return subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=timeout)


def test_loaded_library_matches_the_request():
    # in the child runs below DLLM_CHECKED=1 loads the checked build; here (the regular run) not
    assert dl.bounds_checked() == dl.CHECKED


def test_selftest_bounds_regular_build_writes_everything():
    if dl.CHECKED:
        pytest.skip("runs against the regular build")
    torch.cuda.set_device(0)
    buf = torch.full((512,), -1.0, device="cuda")
    dl.selftest_bounds(buf, 512, 200)  # the regular build performs every store
    dl.check()
    assert torch.equal(buf.cpu(), torch.arange(512, dtype=torch.float32))


def test_checked_build_skips_and_reports_an_access_outside_its_buffer():
    code = r"""
import torch
import quantized_gemm_q8_gb300 as dl
assert dl.CHECKED and dl.bounds_checked()
torch.cuda.set_device(0)
buf = torch.full((512,), -1.0, device="cuda")
dl.selftest_bounds(buf, 512, 200)
try:
    dl.check()
    raise SystemExit("no bounds error reported")
except dl.DllmError as e:
    assert e.code == dl.E_BOUNDS, e
    assert "api.cu:" in str(e), e
host = buf.cpu()
assert torch.equal(host[:200], torch.arange(200, dtype=torch.float32)), "in-span stores performed"
assert bool((host[200:] == -1.0).all()), "out-of-span stores skipped"
dl.selftest_bounds(buf, 512, 512)  # the context is still usable and the error word was cleared
dl.check()
assert torch.equal(buf.cpu(), torch.arange(512, dtype=torch.float32))
print("CHECKED-OK")
"""
    r = _child(code, 600)
    assert r.returncode == 0 and "CHECKED-OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_gpu_suite_under_the_checked_build():
    if dl.CHECKED:
        pytest.skip("the parent run starts the checked child")
    sel = ["tests/test_gpu_qgemm.py", "tests/test_gpu_stages.py", "tests/test_gpu_lmhead.py",
           "tests/test_gpu_layer.py", "tests/test_zz_no_alloc.py", "tests/test_gpu_checked_build.py"]
    # every kernel is reached by this selection; the long full-size comparisons are left to the
    # regular run (the checked kernels take longer)
    keep = ("not llada_head and not full_depth and not two_layers_first_block and not gpu_suite_under "
            "and not llada_shapes_two_layers and not linear_stream_sweep and not whole_protocol")
    r = _child(["-m", "pytest", *sel, "-m", "gpu", "-q", "-x", "-k", keep], 3000)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and "failed" not in r.stdout, tail
    assert int(m.group(1)) >= 70, tail  # the selection above runs 76 tests (one skips under the checked build)
    print("\n" + r.stdout.strip().splitlines()[-1])
