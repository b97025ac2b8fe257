// Measured peak of the legacy int8 tensor path on this GPU: mma.sync m16n8k32, s8 x s8 -> s32
// (the form an int8 GEMM takes where tcgen05 has no int8 kind). Benchmark hook: one launch of
// `iters` iterations per warp, eight independent accumulator chains per warp so that the issue
// of one mma never waits for the previous one's result; every CTA has 8 warps and the grid is
// four CTAs per SM. Work per launch: grid * 8 warps * iters * 8 mma * 2 * 16 * 8 * 32 ops.
#include "internal.h"

#define DLLM_FILE 4  // bounds-check sites of this file

namespace dllm {
namespace {

constexpr int PK_WARPS = 8, PK_CHAINS = 8;

__global__ void __launch_bounds__(PK_WARPS * 32) mma_i8_peak_kernel(long long iters, int* sink, Bounds bd) {
  const uint32_t t = threadIdx.x * 2654435761u + blockIdx.x;
  const uint32_t a0 = t, a1 = t ^ 0x5A5A5A5Au, a2 = t * 3u, a3 = ~t, b0 = t >> 3, b1 = t * 7u;
  int acc[PK_CHAINS][4];
#pragma unroll
  for (int c = 0; c < PK_CHAINS; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0;
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < PK_CHAINS; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};\n"
          : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < PK_CHAINS; ++c) s += acc[c][0] + acc[c][1] + acc[c][2] + acc[c][3];
  if (s == 0x7fffffff) STB(bd, 0, sink, s);  // keeps the chains live; practically never true
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" DLLM_API int dllm_peak_mma_i8(int64_t iters, int32_t* sink, double* ops_per_launch, dllm_stream_t stream) {
  if (iters <= 0 || iters > ((int64_t)1 << 30))
    return fail(DLLM_E_INVAL, "dllm_peak_mma_i8: iters=%lld must be in [1, 2^30]", (long long)iters);
  int rc = check_device();
  if (rc) return rc;
  if (!device_ptr(sink)) return fail(DLLM_E_INVAL, "dllm_peak_mma_i8: sink is NULL or not a device pointer");
  const int grid = 4 * num_sms();
  mma_i8_peak_kernel<<<grid, PK_WARPS * 32, 0, (cudaStream_t)stream>>>((long long)iters, sink,
                                                                       make_bounds({{sink, sizeof(int)}}));
  note_launch();
  if (ops_per_launch) *ops_per_launch = (double)grid * PK_WARPS * (double)iters * PK_CHAINS * 2.0 * 16 * 8 * 32;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch mma_i8_peak");
}
