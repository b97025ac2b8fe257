// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <initializer_list>
#include <string>

#include "bounds.cuh"
#include "dllm.h"

namespace dllm {

// An NVTX range over one C-ABI call, named after the call (NVTX v3 is header-only: with no
// profiler attached a range costs a few nanoseconds).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define DLLM_RANGE() ::dllm::NvtxRange dllm_nvtx_range_(__func__)

struct QgemmParams;

// Status helpers: record an actionable message for dllm_last_error() and return the code.
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);

// Device properties of the current device (cached per device).
int num_sms();
int check_device();  // DLLM_OK if the current device is sm_103
int* err_word();     // device address of the current device's error word (nullptr on failure)
int* site_word();    // device address of the first failing bounds-check site (checked build)

// One buffer of a launch for the bounds-checked build: `bytes` bytes from p (a null p is an
// empty span). make_bounds lays the spans out in order (span i = the i-th); in the regular
// build it returns the empty Bounds and the spans are not used.
struct Span {
  const void* p;
  size_t bytes;
};
Bounds make_bounds(std::initializer_list<Span> spans);
// Bytes covered by `rows` rows of `cols` elements of `esize` bytes with a row stride of `ld`
// elements: the extent of a strided matrix (0 when empty).
inline size_t strided_bytes(int64_t rows, int64_t cols, int64_t ld, size_t esize) {
  return rows <= 0 || cols <= 0 ? 0 : ((size_t)(rows - 1) * (size_t)ld + (size_t)cols) * esize;
}

// Activation operand layout ("act" buffer of dllm_quantize_act).
struct ActLayout {
  int64_t rows, k, lpad, nsb;
  size_t off_a, off_j, off_d, bytes;
};
ActLayout act_layout(int64_t rows, int64_t k);
int64_t act_rows_padded(int64_t rows);

// Tensor map over the A-plane of an act buffer (3-D: 64 x lpad x k/64, f16, 128-byte swizzle,
// box 64 x nt x 1).
int make_act_tmap(CUtensorMap* map, const void* act_a, int64_t lpad, int64_t k, int nt);
int make_planes_tmap(CUtensorMap* map, const void* base, int64_t planes, int64_t rows, int64_t cols, int box_rows);

// GEMM launch plan.
struct QgemmPlan {
  int nt, lpad, tiles_n, tiles_m, splits, sbps, units, grid, nsb;
  size_t ws_bytes;
};
QgemmPlan plan_qgemm(int type, int64_t m, int64_t n, int64_t k);

QgemmPlan plan_single_split(int type, int64_t m, int64_t n, int64_t k);

// One GEMM launch (no argument validation; callers validate). When P.splits > 1 the kernel
// writes split partials [splits][m][n] to `partial`, otherwise y (mode 0) or the LM-head
// softmax partials (mode 1).
// Launch with programmatic stream serialization: the kernel may start while its predecessor
// drains; it synchronizes with griddep_wait() before touching the predecessor's data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct GemmLaunch {
  int type;
  const void* act;
  int64_t m, k;
  const void* w;
  int64_t n;
  float* y;
  int64_t ldy;
  int accumulate;
  float* partial;
  int mode;
  float* pmax;
  int* parg;
  float* psum;
  int32_t* dbg;
  int dbg_mode;
  float* pent;  // mode 1: optional entropy partials
  // mode 1: Gumbel-max sampling when inv_temp > 0 (partials pscore / pidx / plogit)
  float inv_temp;
  unsigned long long seed;
  int step, pos0;
  float* pscore;
  int* pidx;
  float* plogit;
};
int launch_gemm(const GemmLaunch& g, const QgemmPlan& P, cudaStream_t stream);
size_t packed_blob_bytes(int type, int64_t n, int64_t k);
bool device_ptr(const void* p);
size_t align_up(size_t x, size_t a);

// Launch the tcgen05 GEMM kernel instantiated for (type, nt) (defined in qgemm_q4k.cu /
// qgemm_q6k.cu). Returns DLLM_OK or a status.
int launch_qgemm_q4k(int nt, const CUtensorMap& map, const QgemmParams& p, int grid, cudaStream_t s);
int launch_qgemm_q6k(int nt, const CUtensorMap& map, const QgemmParams& p, int grid, cudaStream_t s);
int launch_qgemm_q6k_sample(int nt, const CUtensorMap& map, const QgemmParams& p, int grid, cudaStream_t s);

// y (+)= the sum of `splits` split-K partials P[splits][m][n] (stride elements apart), summed in
// split order (deterministic); one launch on `stream`. Returns DLLM_OK or a status.
int launch_reduce_splits(const float* P, int splits, int64_t stride, int64_t m, int64_t n, float* y, int64_t ldy,
                         int accumulate, cudaStream_t stream);

// Quantize rows of x into the operand form (internal, no validation).
int quantize_rows(const float* x, int64_t rows, int64_t k, int64_t ldx, const float* norm_w, float eps, void* act,
                  cudaStream_t stream);

// Count of kernel launches issued by this library (for benchmark bookkeeping).
void note_launch();

constexpr long long kDefaultTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz

}  // namespace dllm
