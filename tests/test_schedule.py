"""The product's transfer schedule (host-only C-ABI calls, CPU) against the oracle's transfer
counts and the pages' benchmark protocol (128 generated tokens, blocks of 32, 32 steps, 4
commits per step)."""
import pytest

import oracle as orc
import quantized_gemm_q8_gb300 as dl
from quantized_gemm_q8_gb300 import build as dlbuild


@pytest.mark.parametrize("masked,steps", [(128, 32), (37, 8), (10, 4), (32, 8), (3, 5), (0, 4), (1, 1), (31, 8)])
def test_transfer_counts_match_the_oracle(masked, steps):
    dlbuild.build()
    assert dl.transfer_counts(masked, steps) == orc.transfer_counts(masked, steps).tolist()


def test_schedule_of_the_benchmark_protocol():
    dlbuild.build()
    sch = dl.schedule(20, 128, 32, 32)
    assert len(sch) == 32
    for s, (b0, b1, k) in enumerate(sch):
        assert (b0, b1, k) == (20 + 32 * (s // 8), 20 + 32 * (s // 8 + 1), 4)
    # uneven: 3 blocks of 5 over 6 steps, 2 steps per block commit 3 then 2
    assert dl.schedule(0, 15, 5, 6) == [(0, 5, 3), (0, 5, 2), (5, 10, 3), (5, 10, 2), (10, 15, 3), (10, 15, 2)]
    # every block ends fully committed
    for prompt, gen, blk, steps in [(20, 128, 32, 32), (7, 96, 32, 12), (0, 40, 8, 20)]:
        sch = dl.schedule(prompt, gen, blk, steps)
        per_block = {}
        for b0, b1, k in sch:
            per_block[b0] = per_block.get(b0, 0) + k
        assert per_block == {prompt + blk * b: blk for b in range(gen // blk)}


@pytest.mark.parametrize("args", [(20, 128, 30, 32), (20, 128, 32, 30), (20, 0, 32, 32), (-1, 128, 32, 32)])
def test_schedule_rejects_bad_shapes(args):
    dlbuild.build()
    with pytest.raises(dl.DllmError) as e:
        dl.schedule(*args)
    assert e.value.code == dl.E_INVAL and "dllm_schedule" in str(e.value)


def test_transfer_counts_rejects_bad_arguments():
    dlbuild.build()
    for masked, steps in [(-1, 4), (4, 0)]:
        with pytest.raises(dl.DllmError) as e:
            dl.transfer_counts(masked, steps)
        assert e.value.code == dl.E_INVAL
