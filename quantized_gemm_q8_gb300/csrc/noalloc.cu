// Allocation-free variant of the quantized GEMM.
//
// Some callers cannot hand this library a device workspace and cannot allocate one at call
// time: an inference server that reserves all device memory at start-up and forbids later
// allocations, a host framework whose plugin interface passes inputs and outputs but no
// scratch buffer, or a latency-critical loop that must not call cudaMalloc because that call
// can synchronize the device and stall every other stream. dllm_qgemm_noalloc serves them: it
// keeps the split-K partial sums in a fixed array that the library itself holds in device
// memory, so the caller only passes the activations, the packed weights and the output.
//
// The array is a file-scope device variable of kNoallocScratchBytes (32 MiB). Every GPU that
// loads the library holds it until the process exits. Host code cannot use the array's name as
// a device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; that first call should come
// before any stream capture. All calls share the array and it keeps the previous call's
// contents; the GEMM writes every partial it later reads, so nothing needs clearing. Calls
// that overlap on the GPU (on different streams, or from different host threads without
// ordering) race on the array and must not be issued that way. The cached address belongs to
// the device's context at the time of the first call: after cudaDeviceReset (or any teardown
// of that context) it is stale, so a process that resets a device must not call this entry
// point on that device again.
#include <mutex>

#include "internal.h"
#include "qgemm.cuh"

namespace dllm {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DLLM_E_DEVICE, "dllm_qgemm_noalloc: device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return DLLM_OK;
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" DLLM_API int dllm_qgemm_noalloc(int type, const void* act, int64_t m, int64_t k, const void* w_packed,
                                           int64_t n, float* y, int64_t ldy, int accumulate, dllm_stream_t stream) {
  DLLM_RANGE();
  if (type != DLLM_Q4_K && type != DLLM_Q6_K)
    return fail(DLLM_E_TYPE, "dllm_qgemm_noalloc: unsupported block type %d: the GEMM kernels take Q4_K (12) or Q6_K (14)",
                type);
  if (m <= 0 || m > 65536 || n <= 0 || n > (1 << 24) || k <= 0 || k % QK || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "dllm_qgemm_noalloc: bad shape m=%lld n=%lld k=%lld (k must be a positive multiple of 256)",
                (long long)m, (long long)n, (long long)k);
  if (accumulate != 0 && accumulate != 1) return fail(DLLM_E_INVAL, "dllm_qgemm_noalloc: accumulate must be 0 or 1");
  int rc = check_device();
  if (rc) return rc;
  if (!device_ptr(act) || !device_ptr(w_packed) || !device_ptr(y))
    return fail(DLLM_E_INVAL, "dllm_qgemm_noalloc: act, w_packed and y must be device pointers");
  if ((reinterpret_cast<uintptr_t>(act) & 255) || (reinterpret_cast<uintptr_t>(w_packed) & 255))
    return fail(DLLM_E_ALIGN, "dllm_qgemm_noalloc: act and w_packed must be 256-byte aligned");
  if (ldy < n) return fail(DLLM_E_SHAPE, "dllm_qgemm_noalloc: ldy=%lld < n=%lld", (long long)ldy, (long long)n);
  const size_t one = (size_t)m * n * sizeof(float);
  if (one > kNoallocScratchBytes)
    return fail(DLLM_E_SHAPE,
                "dllm_qgemm_noalloc: m*n = %lld outputs need %zu bytes of scratch, above the fixed %zu-byte array; "
                "use dllm_qgemm with a workspace for this shape",
                (long long)(m * n), one, kNoallocScratchBytes);
  float* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  // the plan's split count, reduced to 1 when its partials would not fit the array
  QgemmPlan P = plan_qgemm(type, m, n, k);
  if ((size_t)P.splits * one > kNoallocScratchBytes) P = plan_single_split(type, m, n, k);
  cudaStream_t s = (cudaStream_t)stream;
  GemmLaunch g{type, act, m, k, w_packed, n, scratch, n, 0, scratch, 0, nullptr, nullptr, nullptr, nullptr};
  if ((rc = launch_gemm(g, P, s))) return rc;
  return launch_reduce_splits(scratch, P.splits, m * n, m, n, y, ldy, accumulate, s);
}
