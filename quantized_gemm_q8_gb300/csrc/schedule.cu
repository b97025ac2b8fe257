// Transfer schedule of the diffusion loop (host only): how many masked positions each step
// commits. mojo-dllm Development plan, "Benchmark protocol": 128 generated tokens in blocks of
// 32 over 32 steps, 4 commits per step, with the transfer counts checked against the
// reference generator; Technical Specification, section 13 "Scheduler Interface" (select the
// positions to commit at each step, then update the canvas) and section 12 (the loop).
#include "internal.h"

using namespace dllm;

extern "C" {

DLLM_API int dllm_transfer_counts(int64_t masked, int64_t steps, int32_t* counts) {
  if (masked < 0 || masked > (int64_t)1 << 30 || steps <= 0 || steps > (1 << 20))
    return fail(DLLM_E_INVAL, "dllm_transfer_counts: masked=%lld must be in [0, 2^30] and steps=%lld in [1, 2^20]",
                (long long)masked, (long long)steps);
  if (!counts) return fail(DLLM_E_INVAL, "dllm_transfer_counts: counts is NULL");
  // every step commits the floor share; the remainder goes one by one to the earliest steps
  const int64_t base = masked / steps, extra = masked % steps;
  for (int64_t s = 0; s < steps; ++s) counts[s] = (int32_t)(base + (s < extra ? 1 : 0));
  return DLLM_OK;
}

DLLM_API int dllm_schedule(int64_t prompt_len, int64_t gen_len, int64_t block_len, int64_t steps, int32_t* block_begin,
                           int32_t* block_end, int32_t* k) {
  if (prompt_len < 0 || gen_len <= 0 || block_len <= 0 || steps <= 0 || prompt_len + gen_len > (int64_t)1 << 30 ||
      steps > (1 << 20))
    return fail(DLLM_E_INVAL,
                "dllm_schedule: prompt_len=%lld must be >= 0 and gen_len=%lld, block_len=%lld, steps=%lld > 0",
                (long long)prompt_len, (long long)gen_len, (long long)block_len, (long long)steps);
  if (gen_len % block_len)
    return fail(DLLM_E_INVAL, "dllm_schedule: gen_len=%lld is not a multiple of block_len=%lld", (long long)gen_len,
                (long long)block_len);
  const int64_t blocks = gen_len / block_len;
  if (steps % blocks)
    return fail(DLLM_E_INVAL, "dllm_schedule: steps=%lld is not a multiple of the %lld blocks", (long long)steps,
                (long long)blocks);
  if (!block_begin || !block_end || !k) return fail(DLLM_E_INVAL, "dllm_schedule: an output array is NULL");
  const int64_t per_block = steps / blocks;
  for (int64_t b = 0; b < blocks; ++b) {
    // every position of a block is masked when the block starts
    int rc = dllm_transfer_counts(block_len, per_block, k + b * per_block);
    if (rc) return rc;
    for (int64_t s = 0; s < per_block; ++s) {
      block_begin[b * per_block + s] = (int32_t)(prompt_len + b * block_len);
      block_end[b * per_block + s] = (int32_t)(prompt_len + (b + 1) * block_len);
    }
  }
  return DLLM_OK;
}

}  // extern "C"
