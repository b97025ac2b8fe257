// C ABI of the library (include/dllm.h): status handling, weight packing, Q8_K activation
// quantization, GEMM planning / dispatch, split-K reduction and test hooks.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "qgemm.cuh"
#include "quant.cuh"

#define DLLM_FILE 1  // bounds-check sites of this file

namespace dllm {

__device__ int g_err_word = 0;
__device__ int g_bounds_site = 0;  // checked build: DLLM_SITE_AT of the first failing check

// Per-device caches of symbol addresses and attributes: atomic, so that host threads calling
// the library concurrently may fill them at the same time (each writes the same value).
template <typename Sym>
static int* symbol_address(const Sym& sym, std::atomic<int*>* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, sym) != cudaSuccess) return nullptr;
    p = static_cast<int*>(a);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

int* err_word() {
  static std::atomic<int*> cache[64];
  return symbol_address(g_err_word, cache);
}

int* site_word() {
  static std::atomic<int*> cache[64];
  return symbol_address(g_bounds_site, cache);
}

void set_quant_bounds(QuantOut& o, int64_t rows, int64_t k) {
  const int64_t nsb = k / QK, lp = o.lpad;
  o.bd = make_bounds({{o.q, (size_t)(rows * k)},
                      {o.d, (size_t)(rows * nsb * 4)},
                      {o.bsum, (size_t)(rows * (k / 16) * 2)},
                      {o.act_a, (size_t)(lp * k * 2)},
                      {o.act_j, (size_t)(nsb * lp * 32)},
                      {o.act_d, (size_t)(nsb * lp * 4)},
                      {o.vtap, (size_t)(rows * k * 4)}});
}

Bounds make_bounds(std::initializer_list<Span> spans) {
  Bounds b{};
#ifdef DLLM_BOUNDS_CHECK
  int i = 0;
  for (const Span& s : spans) {
    if (i < kMaxSpans) {
      b.lo[i] = reinterpret_cast<unsigned long long>(s.p);
      b.hi[i] = b.lo[i] + (s.p ? s.bytes : 0);
    }
    ++i;
  }
  b.err = err_word();
  b.site = site_word();
#else
  (void)spans;
#endif
  return b;
}

static thread_local char g_msg[1024] = "";
static std::atomic<long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }


int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DLLM_E_CUDA, "%s failed: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

static int cached_attr(cudaDeviceAttr attr, std::atomic<int>* cache, int dflt) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return dflt;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) return dflt;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int num_sms() {
  static std::atomic<int> cache[64];
  return cached_attr(cudaDevAttrMultiProcessorCount, cache, 152);
}

int check_device() {
  static std::atomic<int> major_c[64], minor_c[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = cached_attr(cudaDevAttrComputeCapabilityMajor, major_c, 0);
  int minor = cached_attr(cudaDevAttrComputeCapabilityMinor, minor_c, 0);
  if (major != 10 || minor != 3)
    return fail(DLLM_E_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, major,
                minor);
  return DLLM_OK;
}

static bool is_device_ptr(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool device_ptr(const void* p) { return is_device_ptr(p); }

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define CHECK_DEV(ptr, name)                                                                      \
  do {                                                                                            \
    if (!is_device_ptr(ptr)) return fail(DLLM_E_INVAL, "%s: %s is NULL or not a device pointer", \
                                         __func__, name);                                         \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool device_ptr(const void* p);

// ---------------------------------------------------------------------------------------------
// Activation operand layout
// ---------------------------------------------------------------------------------------------
int64_t act_rows_padded(int64_t rows) {
  if (rows <= 32) return 32;
  if (rows <= 64) return 64;
  if (rows <= 128) return 128;
  if (rows <= 160) return 160;
  return (rows + 127) / 128 * 128;
}

ActLayout act_layout(int64_t rows, int64_t k) {
  ActLayout L;
  L.rows = rows;
  L.k = k;
  L.lpad = act_rows_padded(rows);
  L.nsb = k / QK;
  L.off_a = 0;
  L.off_j = align_up((size_t)L.lpad * k * 2, 1024);
  L.off_d = align_up(L.off_j + (size_t)L.nsb * L.lpad * 32, 1024);
  L.bytes = align_up(L.off_d + (size_t)L.nsb * L.lpad * 4, 1024);
  return L;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_act_tmap(CUtensorMap* map, const void* act_a, int64_t lpad, int64_t k, int nt) {
  auto enc = get_encode();
  if (!enc) return fail(DLLM_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {64, (cuuint64_t)lpad, (cuuint64_t)(k / 64)};
  cuuint64_t strides[2] = {128, (cuuint64_t)lpad * 128};
  cuuint32_t box[3] = {64, (cuuint32_t)nt, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(act_a), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DLLM_E_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return DLLM_OK;
}

// Tensor map over f16 planes [planes][rows][cols] (row-major), boxes of 64 columns x box_rows
// rows of one plane, 128-byte swizzle (the K-major operand layout of the tensor cores); rows past
// `rows` read as zeros.
int make_planes_tmap(CUtensorMap* map, const void* base, int64_t planes, int64_t rows, int64_t cols, int box_rows) {
  auto enc = get_encode();
  if (!enc) return fail(DLLM_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(rows * cols * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DLLM_E_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return DLLM_OK;
}

// ---------------------------------------------------------------------------------------------
// Weight packing (GGUF AoS blocks -> tile-major blobs + scale plane)
// ---------------------------------------------------------------------------------------------
static int block_bytes(int type) { return type == DLLM_Q4_K ? 144 : type == DLLM_Q6_K ? 210 : 0; }

// Spans (bounds-checked build): 0 the source blocks, 1 the blob, 2 the scale plane.
__global__ void pack_q4k_kernel(const uint8_t* __restrict__ src, int n, int nsb, uint8_t* __restrict__ blob,
                                uint8_t* __restrict__ dd, Bounds bd) {
  const int ts = blockIdx.x;  // tile * nsb + sb
  const int tile = ts / nsb, sb = ts % nsb, r = threadIdx.x;
  const int64_t grow = (int64_t)tile * BM + r;
  const bool valid = grow < n;
  const uint8_t* b = src + (grow * nsb + sb) * 144;
  uint8_t* o = blob + (size_t)ts * Q4K_BLOB;
  const uint4 z4 = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int h = 0; h < 8; ++h)
    STB(bd, 1, reinterpret_cast<uint4*>(o + h * 2048 + r * 16),
        valid ? LDB(bd, 0, reinterpret_cast<const uint4*>(b + 16 + 16 * h), z4) : z4);
#pragma unroll
  for (int w = 0; w < 3; ++w)
    STB(bd, 1, reinterpret_cast<uint32_t*>(o + 16384 + w * 512 + r * 4),
        valid ? LDB(bd, 0, reinterpret_cast<const uint32_t*>(b + 4 + 4 * w), 0u) : 0u);
  STB(bd, 2, reinterpret_cast<uint32_t*>(dd + (size_t)ts * Q4K_DD + r * 4),
      valid ? LDB(bd, 0, reinterpret_cast<const uint32_t*>(b), 0u) : 0u);
}

__global__ void pack_q6k_kernel(const uint8_t* __restrict__ src, int n, int nsb, uint8_t* __restrict__ blob,
                                uint8_t* __restrict__ dd, Bounds bd) {
  const int ts = blockIdx.x;
  const int tile = ts / nsb, sb = ts % nsb, r = threadIdx.x;
  const int64_t grow = (int64_t)tile * BM + r;
  const bool valid = grow < n;
  const uint8_t* b = src + (grow * nsb + sb) * 210;
  uint8_t* o = blob + (size_t)ts * Q6K_BLOB;
  const uint8_t z = 0;
  for (int i = 0; i < 128; ++i) STB(bd, 1, o + (i >> 4) * 2048 + r * 16 + (i & 15), valid ? LDB(bd, 0, b + i, z) : z);
  for (int i = 0; i < 64; ++i)
    STB(bd, 1, o + 16384 + (i >> 4) * 2048 + r * 16 + (i & 15), valid ? LDB(bd, 0, b + 128 + i, z) : z);
  for (int i = 0; i < 16; ++i) STB(bd, 1, o + 24576 + r * 16 + i, valid ? LDB(bd, 0, b + 192 + i, z) : z);
  uint8_t* d = dd + (size_t)ts * Q6K_DD + r * 2;
  STB(bd, 2, d, valid ? LDB(bd, 0, b + 208, z) : z);
  STB(bd, 2, d + 1, valid ? LDB(bd, 0, b + 209, z) : z);
}

struct Packed {
  size_t blob_bytes, dd_bytes;
};
static Packed packed_sizes(int type, int64_t n, int64_t k);
size_t packed_blob_bytes(int type, int64_t n, int64_t k) { return packed_sizes(type, n, k).blob_bytes; }
static Packed packed_sizes(int type, int64_t n, int64_t k) {
  const int64_t tiles = (n + BM - 1) / BM, nsb = k / QK;
  Packed p;
  p.blob_bytes = (size_t)tiles * nsb * (type == DLLM_Q4_K ? Q4K_BLOB : Q6K_BLOB);
  p.dd_bytes = (size_t)tiles * nsb * (type == DLLM_Q4_K ? Q4K_DD : Q6K_DD);
  return p;
}

// ---------------------------------------------------------------------------------------------
// Q8_K activation quantization (+ optional RMSNorm), writing the plain arrays and/or the
// tensor-core operand planes.
// ---------------------------------------------------------------------------------------------
// Spans (bounds-checked build): 0 x, 1 norm_w; the outputs carry their own (QuantOut::bd).
__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ x, int rows, int64_t k,
                                                           int64_t ldx, const float* __restrict__ norm_w, float eps,
                                                           QuantOut o, Bounds bd) {
  __shared__ float red[8];
  griddep_wait();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = (int)(k / QK);
  // super-blocks of this CTA: all of the row (RMSNorm needs its sum of squares), or without a
  // norm one per warp along gridDim.y
  const int sbw = blockIdx.y * 8 + warp, sbstep = 8 * gridDim.y;
  if (row >= rows) {  // padding rows of the operand planes
    float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int sb = sbw; sb < nsb; sb += sbstep) q8k_emit(z, row, rows, sb, k, o);
    return;
  }
  const float* xr = x + (int64_t)row * ldx;
  float rstd = 1.f;
  if (norm_w) {
    float ss = 0.f;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = threadIdx.x * 4; i < k; i += blockDim.x * 4) {
      const float4 v = LDB(bd, 0, reinterpret_cast<const float4*>(xr + i), z4);
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
    ss = block_sum(ss, red);
    rstd = 1.0f / sqrtf(ss / (float)k + eps);
  }
  for (int sb = sbw; sb < nsb; sb += sbstep) {
    const int64_t base = (int64_t)sb * QK + 8 * lane;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 a = LDB(bd, 0, reinterpret_cast<const float4*>(xr + base), z4);
    const float4 b = LDB(bd, 0, reinterpret_cast<const float4*>(xr + base + 4), z4);
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (norm_w) {
      const float4 wa = LDB(bd, 1, reinterpret_cast<const float4*>(norm_w + base), z4);
      const float4 wb = LDB(bd, 1, reinterpret_cast<const float4*>(norm_w + base + 4), z4);
      const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (v[i] * rstd) * w[i];
    }
    q8k_emit(v, row, rows, sb, k, o);
  }
  griddep_launch();
}

// Plain Q8_K arrays -> the operand form: warp (blockIdx.y * 8 + w) of row blockIdx.x copies
// super-block sb (lane = codes 8*lane .. 8*lane+7); padding rows are written as zeros. Each lane
// pair checks that its group's 16-sum matches the codes and records ERR_BSUM if not.
// Spans (bounds-checked build): 0 q, 1 d, 2 bsum.
__global__ void __launch_bounds__(256) pack_act_kernel(const int8_t* __restrict__ q, const float* __restrict__ d,
                                                       const int16_t* __restrict__ bsum, int rows, int64_t k,
                                                       QuantOut o, int* err, Bounds bd) {
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const int sb = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int64_t nsb = k / QK;
  if (sb >= nsb) return;
  int qi[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int s16 = 0;
  float dsc = 0.f;
  if (row < rows) {
    const uint2 w = LDB(bd, 0, reinterpret_cast<const uint2*>(q + (int64_t)row * k + (int64_t)sb * QK + 8 * lane),
                        make_uint2(0u, 0u));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qi[i] = (int)(int8_t)(w.x >> (8 * i));
      qi[4 + i] = (int)(int8_t)(w.y >> (8 * i));
    }
    s16 = LDB(bd, 2, bsum + (int64_t)row * (k / 16) + (int64_t)sb * 16 + (lane >> 1), (int16_t)0);
    dsc = LDB(bd, 1, d + (int64_t)row * nsb + sb, 0.f);
    int s8 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s8 += qi[i];
    if (s8 + __shfl_xor_sync(0xffffffffu, s8, 1) != s16 && (lane & 1) == 0) atomicOr(err, ERR_BSUM);
  }
  QuantOut a = o;
  a.q = nullptr;
  a.d = nullptr;
  a.bsum = nullptr;
  q8k_store(qi, s16, dsc, row, rows, sb, k, a);
}

// y (+)= sum of split partials, fixed order.
// Spans (bounds-checked build): 0 P, 1 y.
__global__ void reduce_splits_kernel(const float* __restrict__ P, int splits, int64_t stride, int m, int n,
                                     float* __restrict__ y, int64_t ldy, int accumulate, Bounds bd) {
  const int64_t total = (int64_t)m * n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n, c = i % n;
    float s = 0.f;
    for (int sp = 0; sp < splits; ++sp) s += LDB(bd, 0, P + sp * stride + i, 0.f);
    float* o = y + r * ldy + c;
    STB(bd, 1, o, accumulate ? LDB(bd, 1, (const float*)o, 0.f) + s : s);
  }
}

__global__ void selftest_timeout_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the bounded wait must run out
    if (!mbar_wait(b, 0, &abort_flag, limit)) atomicOr(&g_err_word, ERR_TIMEOUT_SELFTEST);
    mbar_arrive(b);  // complete the phase so the barrier is left consistent
  }
}

// buf[i] = i for i < n, each store checked against span 0 (dllm_selftest_bounds).
__global__ void selftest_bounds_kernel(float* buf, int n, Bounds bd) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) STB(bd, 0, buf + i, (float)i);
}

// ---------------------------------------------------------------------------------------------
// LM head: merge of the per-(tile, quadrant) softmax partials and top-k commit
// ---------------------------------------------------------------------------------------------
struct SoftPart {
  float m;  // max logit
  int a;    // its token id (lowest on ties)
  float s;  // sum exp(logit - m)
  float t;  // sum exp(logit - m) (logit - m), for the entropy
};

__device__ __forceinline__ SoftPart soft_merge(SoftPart x, SoftPart y) {
  if (y.m > x.m || (y.m == x.m && y.a < x.a)) {
    const SoftPart t = x;
    x = y;
    y = t;
  }
  // x has the larger max (or the lower id at equal max); y's sums move to x's max:
  // exp(l - x.m) = f exp(l - y.m) and l - x.m = (l - y.m) + (y.m - x.m), f = exp(y.m - x.m)
  if (y.s != 0.f) {
    const float f = expf(y.m - x.m);
    x.t = x.t + f * (y.t + (y.m - x.m) * y.s);
    x.s = x.s + y.s * f;
  }
  return x;
}

// One Gumbel-max partial: best perturbed score, its token id (lowest on ties), its logit.
struct SampPart {
  float sc;
  int a;
  float l;
};
__device__ __forceinline__ SampPart samp_merge(SampPart x, SampPart y) {
  return (y.sc > x.sc || (y.sc == x.sc && y.a < x.a)) ? y : x;
}

// Merge and commit, one launch: CTA r (256 threads) merges row r's P partials (contiguous,
// [R][P]) into the argmax id and the row's confidence, and stores them; the CTA that
// finishes last (a counter, zeroed before the launch) picks the k masked positions of the
// block with the highest confidence (ties: lowest position) and scatters their ids into the
// canvas. Confidence: kind 0 p_max = 1 / sum exp(l - l_max); kind 1 the negative entropy
// -H = sum p log p = t / s - log s with s = sum exp(l - l_max), t = sum exp(l - l_max)(l - l_max)
// (pent holds the t partials; unused for kind 0). With sampling (pscore non-null) the row's
// token is the Gumbel-max draw instead of the argmax, and kind 0 is its probability
// exp(l_draw - l_max) / s.
// Spans (bounds-checked build), in LmSpan order.
enum LmSpan : int { LS_PMAX = 0, LS_PARG, LS_PSUM, LS_PENT, LS_PSCORE, LS_PIDX, LS_PLOGIT, LS_CANVAS, LS_OPOS, LS_OID,
                    LS_OCONF, LS_RID, LS_RCONF, LS_CONF, LS_ID, LS_DONE };
__global__ void __launch_bounds__(256) lmhead_merge_commit_kernel(
    const float* __restrict__ pmax, const int* __restrict__ parg, const float* __restrict__ psum,
    const float* __restrict__ pent, const float* __restrict__ pscore, const int* __restrict__ pidx,
    const float* __restrict__ plogit, int kind, int P, int R, int32_t* canvas, int32_t mask_id, int b0, int k,
    int32_t* out_pos, int32_t* out_id, float* out_conf, int32_t* row_id, float* row_conf, float* conf_ws, int* id_ws,
    unsigned int* done, Bounds bd) {
  __shared__ SoftPart red[8];
  __shared__ SampPart sred[8];
  __shared__ bool last;
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  SoftPart acc{-INFINITY, 0x7fffffff, 0.f, 0.f};
  SampPart sacc{-INFINITY, 0x7fffffff, 0.f};
  const bool sample = pscore != nullptr;
  const size_t base = (size_t)r * P;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    acc = soft_merge(acc, SoftPart{LDB(bd, LS_PMAX, pmax + base + i, -INFINITY), LDB(bd, LS_PARG, parg + base + i, 0),
                                   LDB(bd, LS_PSUM, psum + base + i, 0.f),
                                   kind ? LDB(bd, LS_PENT, pent + base + i, 0.f) : 0.f});
    if (sample)
      sacc = samp_merge(sacc, SampPart{LDB(bd, LS_PSCORE, pscore + base + i, -INFINITY),
                                       LDB(bd, LS_PIDX, pidx + base + i, 0), LDB(bd, LS_PLOGIT, plogit + base + i, 0.f)});
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    SoftPart o{__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.a, off),
               __shfl_xor_sync(0xffffffffu, acc.s, off), __shfl_xor_sync(0xffffffffu, acc.t, off)};
    acc = soft_merge(acc, o);
    SampPart so{__shfl_xor_sync(0xffffffffu, sacc.sc, off), __shfl_xor_sync(0xffffffffu, sacc.a, off),
                __shfl_xor_sync(0xffffffffu, sacc.l, off)};
    sacc = samp_merge(sacc, so);
  }
  if (lane == 0) {
    red[warp] = acc;
    sred[warp] = sacc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) {
      acc = soft_merge(acc, red[w]);
      sacc = samp_merge(sacc, sred[w]);
    }
    if (sample) acc.a = sacc.a;  // the committed token is the draw
    const float c = kind ? acc.t / acc.s - logf(acc.s) : (sample ? expf(sacc.l - acc.m) : 1.0f) / acc.s;
    STB(bd, LS_CONF, conf_ws + r, c);
    STB(bd, LS_ID, id_ws + r, acc.a);
    if (row_id) STB(bd, LS_RID, row_id + r, acc.a);
    if (row_conf) STB(bd, LS_RCONF, row_conf + r, c);
    __threadfence();
    last = BOK(bd, LS_DONE, done, 4) && atomicAdd(done, 1u) == (unsigned)(R - 1);
  }
  __syncthreads();
  if (!last || warp != 0) return;
  __threadfence();
  for (int step = 0; step < k; ++step) {
    float best = -INFINITY;  // below every confidence (p_max > 0, -entropy >= -log vocab)
    int bp = 0x7fffffff;
    for (int q = lane; q < R; q += 32) {
      const volatile float* cv = conf_ws;
      const float cq = BOK(bd, LS_CONF, cv + q, 4) ? cv[q] : -INFINITY;
      if (LDB(bd, LS_CANVAS, (const int32_t*)canvas + b0 + q, ~mask_id) == mask_id &&
          (cq > best || (cq == best && q < bp))) {
        bool taken = false;
        for (int s2 = 0; s2 < step; ++s2) taken |= LDB(bd, LS_OPOS, (const int32_t*)out_pos + s2, -1) == b0 + q;
        if (!taken) {
          best = cq;
          bp = q;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int op = __shfl_xor_sync(0xffffffffu, bp, off);
      if (ob > best || (ob == best && op < bp)) {
        best = ob;
        bp = op;
      }
    }
    if (lane == 0) {
      const volatile int* iv = id_ws;
      if (bp != 0x7fffffff) {
        STB(bd, LS_OPOS, out_pos + step, b0 + bp);
        STB(bd, LS_OID, out_id + step, BOK(bd, LS_ID, iv + bp, 4) ? iv[bp] : -1);
        if (out_conf) STB(bd, LS_OCONF, out_conf + step, best);
      } else {
        STB(bd, LS_OPOS, out_pos + step, -1);
        STB(bd, LS_OID, out_id + step, -1);
        if (out_conf) STB(bd, LS_OCONF, out_conf + step, 0.f);
      }
    }
    __syncwarp();
    __threadfence_block();
  }
  if (lane == 0) {
    for (int step = 0; step < k; ++step) {
      const int32_t pos = LDB(bd, LS_OPOS, (const int32_t*)out_pos + step, -1);
      if (pos >= 0) STB(bd, LS_CANVAS, canvas + pos, LDB(bd, LS_OID, (const int32_t*)out_id + step, 0));
    }
  }
}

struct LmheadWs {
  size_t act, pmax, parg, psum, pent, pscore, pidx, plogit, conf, id, done, bytes;
  int P;
};
static LmheadWs lmhead_ws(int64_t R, int64_t vocab, int64_t d) {
  LmheadWs w;
  const int64_t tiles = (vocab + BM - 1) / BM;
  w.P = (int)(tiles * 4);
  w.act = 0;
  w.pmax = align_up(act_layout(R, d).bytes, 256);
  w.parg = w.pmax + align_up((size_t)w.P * R * 4, 256);
  w.psum = w.parg + align_up((size_t)w.P * R * 4, 256);
  w.pent = w.psum + align_up((size_t)w.P * R * 4, 256);
  w.pscore = w.pent + align_up((size_t)w.P * R * 4, 256);
  w.pidx = w.pscore + align_up((size_t)w.P * R * 4, 256);
  w.plogit = w.pidx + align_up((size_t)w.P * R * 4, 256);
  w.conf = w.plogit + align_up((size_t)w.P * R * 4, 256);
  w.id = w.conf + align_up((size_t)R * 4, 256);
  w.done = w.id + align_up((size_t)R * 4, 256);
  w.bytes = w.done + 256;
  return w;
}

// ---------------------------------------------------------------------------------------------
// GEMM plan
// ---------------------------------------------------------------------------------------------
QgemmPlan plan_qgemm(int type, int64_t m, int64_t n, int64_t k) {
  QgemmPlan P{};
  P.lpad = (int)act_rows_padded(m);
  P.nt = P.lpad <= 160 ? P.lpad : 128;
  P.tiles_n = (int)((n + BM - 1) / BM);
  P.tiles_m = P.lpad / P.nt;
  P.nsb = (int)(k / QK);
  const int nsm = num_sms();
  const double w = type == DLLM_Q6_K ? 2.0 : 1.0625;  // MMA work per super-block
  const double c_unit = 1.5;                           // fill + epilogue store, in super-block units
  double best = 1e30;
  for (int s = 1; s <= std::min(P.nsb, 32); ++s) {
    const int sbps = (P.nsb + s - 1) / s;
    const int sp = (P.nsb + sbps - 1) / sbps;
    const long long units = (long long)P.tiles_n * P.tiles_m * sp;
    const int grid = (int)std::min<long long>(units, nsm);
    const long long waves = (units + grid - 1) / grid;
    const double cost = waves * (sbps * w + c_unit) + (sp > 1 ? 0.02 * sp : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      P.splits = sp;
      P.sbps = sbps;
      P.units = (int)units;
      P.grid = grid;
    }
  }
  P.ws_bytes = P.splits > 1 ? align_up((size_t)P.splits * m * n * 4, 256) : 0;
  return P;
}


// Quantize `rows` rows of x into the operand form at `act` (no validation).
int quantize_rows(const float* x, int64_t rows, int64_t k, int64_t ldx, const float* norm_w, float eps, void* act,
                  cudaStream_t stream) {
  ActLayout L = act_layout(rows, k);
  uint8_t* base = static_cast<uint8_t*>(act);
  QuantOut o{nullptr, nullptr, nullptr, reinterpret_cast<__half*>(base + L.off_a), base + L.off_j,
             reinterpret_cast<float*>(base + L.off_d), (int)L.lpad};
  set_quant_bounds(o, rows, k);
  const dim3 grid((unsigned)L.lpad, norm_w ? 1u : (unsigned)((k / QK + 7) / 8));
  cudaError_t e = launch_pdl(quantize_act_kernel, grid, dim3(256), 0, stream, x, (int)rows, k, ldx, norm_w, eps, o,
                             make_bounds({{x, strided_bytes(rows, k, ldx, 4)}, {norm_w, (size_t)k * 4}}));
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch quantize_act");
}
}  // namespace dllm

using namespace dllm;

extern "C" {

DLLM_API const char* dllm_last_error(void) { return g_msg; }

DLLM_API int dllm_version(void) { return 100; }

DLLM_API int dllm_check(dllm_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int w = 0;
  e = cudaMemcpyFromSymbol(&w, g_err_word, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (w) {
    int z = 0;
    cudaMemcpyToSymbol(g_err_word, &z, sizeof(int));
    if (w & ERR_BOUNDS) {
      int site = 0;
      cudaMemcpyFromSymbol(&site, g_bounds_site, sizeof(int));
      cudaMemcpyToSymbol(g_bounds_site, &z, sizeof(int));
      static const char* const files[] = {"?", "api.cu", "layer.cu", "noalloc.cu", "peak.cu", "?", "?", "?", "?",
                                          "qgemm.cuh", "quant.cuh"};
      const int f = site / 100000;
      return fail(DLLM_E_BOUNDS,
                  "bounds-checked build: a kernel access outside its buffer was skipped (first at %s:%d); the "
                  "outputs of that launch are not valid%s",
                  f >= 0 && f <= 10 ? files[f] : "?", site % 100000,
                  (w & ~ERR_BOUNDS) ? " (other error bits were set too; a skipped copy can make waits run out)" : "");
    }
    if ((w & ~(ERR_RANGE | ERR_BSUM)) == 0)
      return fail(DLLM_E_INVAL, "%s%s",
                  (w & ERR_RANGE) ? "a Q4_K super-block has |dmin / d| above 4e6: its min term cannot be folded into "
                                    "the f16 tensor-core operands (the outputs of that launch are not valid). "
                                  : "",
                  (w & ERR_BSUM) ? "plain Q8_K input to dllm_pack_act has a 16-value sum (bsum) that does not match "
                                   "its codes (the operand and the GEMM outputs made from it are not valid). "
                                 : "");
    return fail(DLLM_E_TIMEOUT, "device-side bounded wait ran out (roles: %s%s%s%s%s%s)",
                (w & ERR_TIMEOUT_PRODUCER) ? "producer " : "", (w & ERR_TIMEOUT_DECODE) ? "decode " : "",
                (w & ERR_TIMEOUT_MMA) ? "mma " : "", (w & ERR_TIMEOUT_EPILOGUE) ? "epilogue " : "",
                (w & ERR_TIMEOUT_SELFTEST) ? "selftest " : "", (w & ERR_TIMEOUT_OTHER) ? "other " : "");
  }
  return DLLM_OK;
}

DLLM_API size_t dllm_packed_bytes(int type, int64_t n, int64_t k) {
  if (!block_bytes(type) || n <= 0 || k <= 0 || k % QK) return 0;
  Packed p = packed_sizes(type, n, k);
  return p.blob_bytes + p.dd_bytes;
}

DLLM_API int dllm_pack_weights(int type, const void* blocks, int64_t n, int64_t k, void* packed,
                               size_t packed_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  if (!block_bytes(type))
    return fail(DLLM_E_TYPE, "dllm_pack_weights: unsupported block type %d: the GEMM kernels take Q4_K (12) or Q6_K (14)",
                type);
  if (n <= 0 || k <= 0 || k % QK || n > (1 << 24) || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "dllm_pack_weights: bad shape n=%lld k=%lld (k must be a positive multiple of 256)",
                (long long)n, (long long)k);
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(blocks, "blocks");
  CHECK_DEV(packed, "packed");
  if (!aligned(packed, 256)) return fail(DLLM_E_ALIGN, "dllm_pack_weights: packed must be 256-byte aligned");
  if (type == DLLM_Q4_K && !aligned(blocks, 16))
    return fail(DLLM_E_ALIGN, "dllm_pack_weights: Q4_K blocks must be 16-byte aligned");
  if (type == DLLM_Q6_K && !aligned(blocks, 2))
    return fail(DLLM_E_ALIGN, "dllm_pack_weights: Q6_K blocks must be 2-byte aligned");
  const size_t need = dllm_packed_bytes(type, n, k);
  if (packed_bytes < need)
    return fail(DLLM_E_WORKSPACE, "dllm_pack_weights: packed buffer has %zu bytes, needs %zu", packed_bytes, need);
  Packed ps = packed_sizes(type, n, k);
  const int nsb = (int)(k / QK), tiles = (int)((n + BM - 1) / BM);
  uint8_t* blob = static_cast<uint8_t*>(packed);
  uint8_t* dd = blob + ps.blob_bytes;
  const uint8_t* src = static_cast<const uint8_t*>(blocks);
  const Bounds bd = make_bounds({{src, (size_t)n * nsb * block_bytes(type)}, {blob, ps.blob_bytes}, {dd, ps.dd_bytes}});
  if (type == DLLM_Q4_K)
    pack_q4k_kernel<<<tiles * nsb, BM, 0, (cudaStream_t)stream>>>(src, (int)n, nsb, blob, dd, bd);
  else
    pack_q6k_kernel<<<tiles * nsb, BM, 0, (cudaStream_t)stream>>>(src, (int)n, nsb, blob, dd, bd);
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch pack kernel");
}

DLLM_API int64_t dllm_act_rows(int64_t rows) { return rows > 0 ? act_rows_padded(rows) : 0; }

DLLM_API size_t dllm_act_bytes(int64_t rows, int64_t k) {
  if (rows <= 0 || k <= 0 || k % QK) return 0;
  return act_layout(rows, k).bytes;
}

DLLM_API int dllm_quantize_act(const float* x, int64_t rows, int64_t k, int64_t ldx, const float* norm_w, float eps,
                               int8_t* q, float* d, int16_t* bsum, void* act, size_t act_bytes,
                               dllm_stream_t stream) {
  DLLM_RANGE();
  if (rows <= 0 || rows > 65536 || k <= 0 || k % QK || k > (1 << 20) || ldx < k)
    return fail(DLLM_E_SHAPE, "dllm_quantize_act: bad shape rows=%lld k=%lld ldx=%lld (k %% 256 == 0, ldx >= k)",
                (long long)rows, (long long)k, (long long)ldx);
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(x, "x");
  if (!aligned(x, 16) || ldx % 4) return fail(DLLM_E_ALIGN, "dllm_quantize_act: x must be 16-byte aligned, ldx %% 4 == 0");
  if (norm_w) {
    CHECK_DEV(norm_w, "norm_w");
    if (!aligned(norm_w, 16)) return fail(DLLM_E_ALIGN, "dllm_quantize_act: norm_w must be 16-byte aligned");
  }
  if (q) {
    CHECK_DEV(q, "q");
    if (!aligned(q, 8)) return fail(DLLM_E_ALIGN, "dllm_quantize_act: q must be 8-byte aligned");
  }
  if (d) CHECK_DEV(d, "d");
  if (bsum) CHECK_DEV(bsum, "bsum");
  QuantOut o{q, d, bsum, nullptr, nullptr, nullptr, 0};
  int grid = (int)rows;
  if (act) {
    CHECK_DEV(act, "act");
    if (!aligned(act, 256)) return fail(DLLM_E_ALIGN, "dllm_quantize_act: act must be 256-byte aligned");
    ActLayout L = act_layout(rows, k);
    if (act_bytes < L.bytes)
      return fail(DLLM_E_WORKSPACE, "dllm_quantize_act: act buffer has %zu bytes, needs %zu", act_bytes, L.bytes);
    uint8_t* base = static_cast<uint8_t*>(act);
    o.act_a = reinterpret_cast<__half*>(base + L.off_a);
    o.act_j = base + L.off_j;
    o.act_d = reinterpret_cast<float*>(base + L.off_d);
    o.lpad = (int)L.lpad;
    grid = (int)L.lpad;
  }
  set_quant_bounds(o, rows, k);
  quantize_act_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
      x, (int)rows, k, ldx, norm_w, eps, o, make_bounds({{x, strided_bytes(rows, k, ldx, 4)}, {norm_w, (size_t)k * 4}}));
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch quantize_act");
}

DLLM_API size_t dllm_qgemm_workspace_bytes(int type, int64_t m, int64_t n, int64_t k) {
  if (!block_bytes(type) || m <= 0 || n <= 0 || k <= 0 || k % QK) return 0;
  return plan_qgemm(type, m, n, k).ws_bytes;
}

}  // extern "C"

namespace dllm {

int launch_gemm(const GemmLaunch& g, const QgemmPlan& P, cudaStream_t stream) {
  ActLayout L = act_layout(g.m, g.k);
  const uint8_t* abase = static_cast<const uint8_t*>(g.act);
  CUtensorMap map;
  int rc = make_act_tmap(&map, abase + L.off_a, L.lpad, g.k, P.nt);
  if (rc) return rc;
  Packed ps = packed_sizes(g.type, g.n, g.k);
  QgemmParams prm{};
  prm.wblob = static_cast<const uint8_t*>(g.w);
  prm.wdd = prm.wblob + ps.blob_bytes;
  prm.act_j = abase + L.off_j;
  prm.act_d = reinterpret_cast<const float*>(abase + L.off_d);
  prm.nsb = P.nsb;
  prm.n = (int)g.n;
  prm.m = (int)g.m;
  prm.lpad = P.lpad;
  prm.tiles_n = P.tiles_n;
  prm.tiles_m = P.tiles_m;
  prm.splits = P.splits;
  prm.sbps = P.sbps;
  prm.units = P.units;
  if (P.splits > 1) {
    prm.y = g.partial;
    prm.ldy = g.n;
    prm.split_stride = g.m * g.n;
    prm.accumulate = 0;
  } else {
    prm.y = g.y;
    prm.ldy = g.ldy;
    prm.split_stride = 0;
    prm.accumulate = g.accumulate;
  }
  prm.mode = g.mode;
  prm.pmax = g.pmax;
  prm.parg = g.parg;
  prm.psum = g.psum;
  prm.pent = g.pent;
  prm.inv_temp = g.inv_temp;
  prm.seed = g.seed;
  prm.step = g.step;
  prm.pos0 = g.pos0;
  prm.pscore = g.pscore;
  prm.pidx = g.pidx;
  prm.plogit = g.plogit;
  prm.dbg = g.dbg;
  prm.dbg_mode = g.dbg_mode;
  prm.timeout = kDefaultTimeoutCycles;
  prm.err = err_word();
  if (!prm.err) return fail(DLLM_E_CUDA, "cannot resolve the device error word");
  {
    const size_t ys = P.splits > 1 ? (size_t)P.splits * g.m * g.n * 4 : strided_bytes(g.m, g.n, g.ldy, 4);
    const size_t pb = (size_t)g.m * P.tiles_n * 4 * 4;  // LM-head partials: [m][tiles_n * 4]
    prm.bd = make_bounds({{prm.wblob, ps.blob_bytes},
                          {prm.wdd, ps.dd_bytes},
                          {prm.act_j, (size_t)P.nsb * L.lpad * 32},
                          {prm.act_d, (size_t)P.nsb * L.lpad * 4},
                          {prm.y, ys},
                          {g.dbg, (size_t)P.nsb * g.m * g.n * 4},
                          {g.pmax, pb},
                          {g.parg, pb},
                          {g.psum, pb},
                          {g.pent, pb},
                          {g.pscore, pb},
                          {g.pidx, pb},
                          {g.plogit, pb}});
  }
  return g.type == DLLM_Q4_K ? launch_qgemm_q4k(P.nt, map, prm, P.grid, stream)
                             : launch_qgemm_q6k(P.nt, map, prm, P.grid, stream);
}

QgemmPlan plan_single_split(int type, int64_t m, int64_t n, int64_t k) {
  QgemmPlan P = plan_qgemm(type, m, n, k);
  P.splits = 1;
  P.sbps = P.nsb;
  P.units = P.tiles_n * P.tiles_m;
  P.grid = std::min(P.units, num_sms());
  P.ws_bytes = 0;
  return P;
}

static int qgemm_common(const char* fn, int type, const void* act, int64_t m, int64_t k, const void* w_packed,
                        int64_t n, float* y, int64_t ldy, int accumulate, void* ws, size_t ws_bytes,
                        int32_t* dbg, cudaStream_t stream) {
  if (!block_bytes(type))
    return fail(DLLM_E_TYPE, "%s: unsupported block type %d: the GEMM kernels take Q4_K (12) or Q6_K (14)", fn,
                type);
  if (m <= 0 || m > 65536 || n <= 0 || n > (1 << 24) || k <= 0 || k % QK || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "%s: bad shape m=%lld n=%lld k=%lld (k must be a positive multiple of 256)", fn,
                (long long)m, (long long)n, (long long)k);
  if (accumulate != 0 && accumulate != 1) return fail(DLLM_E_INVAL, "%s: accumulate must be 0 or 1", fn);
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(act, "act");
  CHECK_DEV(w_packed, "w_packed");
  if (!aligned(act, 256) || !aligned(w_packed, 256))
    return fail(DLLM_E_ALIGN, "%s: act and w_packed must be 256-byte aligned", fn);
  if (y) {
    CHECK_DEV(y, "y");
    if (ldy < n) return fail(DLLM_E_SHAPE, "%s: ldy=%lld < n=%lld", fn, (long long)ldy, (long long)n);
  }
  QgemmPlan P = dbg ? plan_single_split(type, m, n, k) : plan_qgemm(type, m, n, k);
  if (P.splits > 1) {
    if (!ws || ws_bytes < P.ws_bytes)
      return fail(DLLM_E_WORKSPACE, "%s: workspace has %zu bytes, needs %zu (dllm_qgemm_workspace_bytes)", fn,
                  ws ? ws_bytes : (size_t)0, P.ws_bytes);
    CHECK_DEV(ws, "ws");
  }
  GemmLaunch g{type, act, m, k, w_packed, n, y, ldy, accumulate, static_cast<float*>(ws), 0, nullptr, nullptr, nullptr,
               nullptr, 0};
  if (dbg) {
    // the integer sums: one launch per isolated part, each writing its own plane; Q4_K's plane 0
    // is I' (re-centred quants) and a third launch adds the offset part 8 * sum scale * bsum
    const int parts = type == DLLM_Q4_K ? 3 : 2;
    for (int part = 0; part < parts; ++part) {
      g.dbg = dbg + (size_t)(part == 1) * P.nsb * m * n;
      g.dbg_mode = part + 1;
      if ((rc = launch_gemm(g, P, stream))) return rc;
    }
    return DLLM_OK;
  }
  rc = launch_gemm(g, P, stream);
  if (rc) return rc;
  if (P.splits > 1 && y) return launch_reduce_splits(static_cast<float*>(ws), P.splits, m * n, m, n, y, ldy, accumulate, stream);
  return DLLM_OK;
}

int launch_reduce_splits(const float* P, int splits, int64_t stride, int64_t m, int64_t n, float* y, int64_t ldy,
                         int accumulate, cudaStream_t stream) {
  const int64_t total = m * n;
  const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4 * num_sms());
  reduce_splits_kernel<<<blocks, 256, 0, stream>>>(
      P, splits, stride, (int)m, (int)n, y, ldy, accumulate,
      make_bounds({{P, (size_t)splits * stride * 4}, {y, strided_bytes(m, n, ldy, 4)}}));
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch reduce_splits");
}

}  // namespace dllm

extern "C" {

DLLM_API int dllm_qgemm(int type, const void* act, int64_t m, int64_t k, const void* w_packed, int64_t n, float* y,
                        int64_t ldy, int accumulate, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  if (!y) return fail(DLLM_E_INVAL, "dllm_qgemm: y is NULL");
  return qgemm_common("dllm_qgemm", type, act, m, k, w_packed, n, y, ldy, accumulate, ws, ws_bytes, nullptr,
                      (cudaStream_t)stream);
}

DLLM_API int dllm_pack_act(const int8_t* q, const float* d, const int16_t* bsum, int64_t rows, int64_t k, void* act,
                           size_t act_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  if (rows <= 0 || rows > 65536 || k <= 0 || k % QK || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "dllm_pack_act: bad shape rows=%lld k=%lld (k must be a positive multiple of 256)",
                (long long)rows, (long long)k);
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(q, "q");
  CHECK_DEV(d, "d");
  CHECK_DEV(bsum, "bsum");
  CHECK_DEV(act, "act");
  if (!aligned(q, 8) || !aligned(d, 4) || !aligned(bsum, 2))
    return fail(DLLM_E_ALIGN, "dllm_pack_act: q must be 8-byte, d 4-byte and bsum 2-byte aligned");
  if (!aligned(act, 256)) return fail(DLLM_E_ALIGN, "dllm_pack_act: act must be 256-byte aligned");
  const ActLayout L = act_layout(rows, k);
  if (act_bytes < L.bytes)
    return fail(DLLM_E_WORKSPACE, "dllm_pack_act: act buffer has %zu bytes, needs %zu (dllm_act_bytes)", act_bytes,
                L.bytes);
  int* err = err_word();
  if (!err) return fail(DLLM_E_CUDA, "cannot resolve the device error word");
  uint8_t* base = static_cast<uint8_t*>(act);
  QuantOut o{nullptr, nullptr, nullptr, reinterpret_cast<__half*>(base + L.off_a), base + L.off_j,
             reinterpret_cast<float*>(base + L.off_d), (int)L.lpad};
  set_quant_bounds(o, rows, k);
  const dim3 grid((unsigned)L.lpad, (unsigned)((k / QK + 7) / 8));
  cudaError_t e = launch_pdl(pack_act_kernel, grid, dim3(256), 0, (cudaStream_t)stream, q, d, bsum, (int)rows, k, o,
                             err,
                             make_bounds({{q, (size_t)(rows * k)},
                                          {d, (size_t)(rows * (k / QK) * 4)},
                                          {bsum, (size_t)(rows * (k / 16) * 2)}}));
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch pack_act");
}

DLLM_API size_t dllm_qgemm_plain_workspace_bytes(int type, int64_t m, int64_t n, int64_t k) {
  if (!block_bytes(type) || m <= 0 || m > 65536 || n <= 0 || k <= 0 || k % QK) return 0;
  return align_up(act_layout(m, k).bytes, 256) + plan_qgemm(type, m, n, k).ws_bytes;
}

}  // extern "C"

namespace dllm {
// The GEMM on plain Q8_K arrays: the operand form is built at the start of ws, the split-K
// partials follow it.
static int qgemm_plain(const char* fn, int type, const int8_t* q, const float* d, const int16_t* bsum, int64_t m,
                       int64_t k, const void* w_packed, int64_t n, float* y, int64_t ldy, int accumulate, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  if (!y) return fail(DLLM_E_INVAL, "%s: y is NULL", fn);
  if (m <= 0 || m > 65536 || n <= 0 || n > (1 << 24) || k <= 0 || k % QK || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "%s: bad shape m=%lld n=%lld k=%lld (k must be a positive multiple of 256)", fn,
                (long long)m, (long long)n, (long long)k);
  const size_t need = dllm_qgemm_plain_workspace_bytes(type, m, n, k);
  if (!ws || ws_bytes < need)
    return fail(DLLM_E_WORKSPACE, "%s: workspace has %zu bytes, needs %zu (dllm_qgemm_plain_workspace_bytes)", fn,
                ws ? ws_bytes : (size_t)0, need);
  if (!aligned(ws, 256)) return fail(DLLM_E_ALIGN, "%s: ws must be 256-byte aligned", fn);
  const size_t act_b = align_up(act_layout(m, k).bytes, 256);
  int rc = dllm_pack_act(q, d, bsum, m, k, ws, act_b, (dllm_stream_t)stream);
  if (rc) return rc;
  return qgemm_common(fn, type, ws, m, k, w_packed, n, y, ldy, accumulate, static_cast<uint8_t*>(ws) + act_b,
                      ws_bytes - act_b, nullptr, stream);
}
}  // namespace dllm

extern "C" {

DLLM_API int dllm_qgemm_q4k(const int8_t* q, const float* d, const int16_t* bsum, int64_t m, int64_t k,
                            const void* w_packed, int64_t n, float* y, int64_t ldy, int accumulate, void* ws,
                            size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  return qgemm_plain("dllm_qgemm_q4k", DLLM_Q4_K, q, d, bsum, m, k, w_packed, n, y, ldy, accumulate, ws, ws_bytes,
                     (cudaStream_t)stream);
}

DLLM_API int dllm_qgemm_q6k(const int8_t* q, const float* d, const int16_t* bsum, int64_t m, int64_t k,
                            const void* w_packed, int64_t n, float* y, int64_t ldy, int accumulate, void* ws,
                            size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  return qgemm_plain("dllm_qgemm_q6k", DLLM_Q6_K, q, d, bsum, m, k, w_packed, n, y, ldy, accumulate, ws, ws_bytes,
                     (cudaStream_t)stream);
}

DLLM_API int dllm_qgemm_intsums(int type, const void* act, int64_t m, int64_t k, const void* w_packed, int64_t n,
                                int32_t* sums, dllm_stream_t stream) {
  DLLM_RANGE();
  if (!is_device_ptr(sums)) return fail(DLLM_E_INVAL, "dllm_qgemm_intsums: sums is NULL or not a device pointer");
  return qgemm_common("dllm_qgemm_intsums", type, act, m, k, w_packed, n, nullptr, n, 0, nullptr, 0, sums,
                      (cudaStream_t)stream);
}

DLLM_API int dllm_step_graph_host(void* graph_exec, int32_t* canvas_host, int32_t* canvas, int64_t L,
                                  const int32_t* out, int32_t out_stride, int32_t k_commit, int32_t* out_host,
                                  dllm_stream_t stream) {
  DLLM_RANGE();
  if (!graph_exec || !canvas_host || !out_host || L <= 0 || L > (1 << 24) || k_commit < 0 || out_stride < k_commit)
    return fail(DLLM_E_INVAL,
                "dllm_step_graph_host: graph_exec, canvas_host and out_host must be set, L in [1, 2^24], "
                "0 <= k_commit <= out_stride");
  CHECK_DEV(canvas, "canvas");
  CHECK_DEV(out, "out");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(canvas, canvas_host, (size_t)L * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(graph_exec), s);
  if (e == cudaSuccess && k_commit > 0) {
    e = cudaMemcpyAsync(out_host, out, (size_t)k_commit * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(out_host + k_commit, out + out_stride, (size_t)k_commit * 4, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "dllm_step_graph_host");
  for (int32_t i = 0; i < k_commit; ++i) {
    const int32_t pos = out_host[i];
    if (pos >= 0 && pos < L) canvas_host[pos] = out_host[k_commit + i];
  }
  return DLLM_OK;
}

DLLM_API int dllm_bounds_checked(void) {
#ifdef DLLM_BOUNDS_CHECK
  return 1;
#else
  return 0;
#endif
}

DLLM_API int dllm_selftest_bounds(float* buf, int32_t n_write, int32_t n_declared, dllm_stream_t stream) {
  if (n_write <= 0 || n_write > (1 << 20) || n_declared < 0 || n_declared > n_write)
    return fail(DLLM_E_INVAL, "dllm_selftest_bounds: need 0 < n_write <= 2^20 and 0 <= n_declared <= n_write");
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(buf, "buf");
  selftest_bounds_kernel<<<(n_write + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
      buf, n_write, make_bounds({{buf, (size_t)n_declared * 4}}));
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch selftest_bounds");
}

DLLM_API int dllm_selftest_timeout(int64_t limit_cycles, dllm_stream_t stream) {
  if (limit_cycles <= 0 || limit_cycles > (int64_t)1 << 34)
    return fail(DLLM_E_INVAL, "dllm_selftest_timeout: limit_cycles out of range");
  int rc = check_device();
  if (rc) return rc;
  selftest_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)limit_cycles);
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch selftest_timeout");
}


DLLM_API size_t dllm_lmhead_workspace_bytes(int64_t rows, int64_t vocab, int64_t d) {
  if (rows <= 0 || rows > 160 || vocab <= 0 || d <= 0 || d % QK) return 0;
  return lmhead_ws(rows, vocab, d).bytes;
}

DLLM_API int dllm_lmhead_select(const float* hidden, int64_t L, int64_t d, int64_t ldh, const float* out_norm_w,
                                float eps, const void* w_out_packed, int64_t vocab, int32_t* canvas, int32_t mask_id,
                                int32_t block_begin, int32_t block_end, int32_t k_commit, int32_t conf_kind,
                                float temperature, uint64_t seed, uint32_t step, int32_t* out_pos, int32_t* out_id,
                                float* out_conf, int32_t* row_id, float* row_conf, void* ws, size_t ws_bytes,
                                dllm_stream_t stream) {
  DLLM_RANGE();
  const int64_t R = (int64_t)block_end - block_begin;
  if (L <= 0 || d <= 0 || d % QK || d > (1 << 20) || ldh < d || vocab <= 0 || vocab > (1 << 24))
    return fail(DLLM_E_SHAPE, "dllm_lmhead_select: bad shape L=%lld d=%lld ldh=%lld vocab=%lld", (long long)L,
                (long long)d, (long long)ldh, (long long)vocab);
  if (block_begin < 0 || block_end > L || R <= 0 || R > 160)
    return fail(DLLM_E_INVAL, "dllm_lmhead_select: block [%d, %d) must lie in [0, L=%lld) and hold 1..160 positions",
                block_begin, block_end, (long long)L);
  if (k_commit < 0 || k_commit > R)
    return fail(DLLM_E_INVAL, "dllm_lmhead_select: k_commit=%d must be in [0, %lld]", k_commit, (long long)R);
  if (conf_kind != DLLM_CONF_PMAX && conf_kind != DLLM_CONF_NEG_ENTROPY)
    return fail(DLLM_E_INVAL, "dllm_lmhead_select: conf_kind=%d must be DLLM_CONF_PMAX (0) or DLLM_CONF_NEG_ENTROPY (1)",
                conf_kind);
  if (!std::isfinite(temperature) || temperature < 0.f)
    return fail(DLLM_E_INVAL, "dllm_lmhead_select: temperature must be finite and >= 0 (0 = greedy)");
  if (temperature > 0.f && (L > 65536 || step >= (1u << 24)))
    return fail(DLLM_E_INVAL, "dllm_lmhead_select: sampling needs L <= 65536 and step < 2^24 (the noise counter)");
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(hidden, "hidden");
  CHECK_DEV(w_out_packed, "w_out_packed");
  CHECK_DEV(canvas, "canvas");
  if (k_commit > 0) {
    CHECK_DEV(out_pos, "out_pos");
    CHECK_DEV(out_id, "out_id");
  }
  if (out_conf) CHECK_DEV(out_conf, "out_conf");
  if (row_id) CHECK_DEV(row_id, "row_id");
  if (row_conf) CHECK_DEV(row_conf, "row_conf");
  CHECK_DEV(out_norm_w, "out_norm_w");
  if (!aligned(out_norm_w, 16)) return fail(DLLM_E_ALIGN, "dllm_lmhead_select: out_norm_w must be 16-byte aligned");
  if (!aligned(hidden, 16) || ldh % 4 || !aligned(w_out_packed, 256))
    return fail(DLLM_E_ALIGN, "dllm_lmhead_select: hidden 16-byte aligned with ldh %% 4 == 0, w_out_packed 256-byte aligned");
  const LmheadWs W = lmhead_ws(R, vocab, d);
  if (!ws || ws_bytes < W.bytes)
    return fail(DLLM_E_WORKSPACE, "dllm_lmhead_select: workspace has %zu bytes, needs %zu", ws ? ws_bytes : (size_t)0,
                W.bytes);
  CHECK_DEV(ws, "ws");
  if (!aligned(ws, 256)) return fail(DLLM_E_ALIGN, "dllm_lmhead_select: ws must be 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = static_cast<uint8_t*>(ws);
  // 1) RMSNorm + Q8_K of the block's rows (contiguous in the residual stream)
  rc = quantize_rows(hidden + (int64_t)block_begin * ldh, R, d, ldh, out_norm_w, eps, base + W.act, s);
  if (rc) return rc;
  // 2) Q6_K head GEMM with the softmax-partial epilogue (one split: logits complete per tile)
  QgemmPlan P = plan_single_split(DLLM_Q6_K, R, vocab, d);
  GemmLaunch g{DLLM_Q6_K, base + W.act, R, d, w_out_packed, vocab, nullptr, 0, 0, nullptr, 1,
               reinterpret_cast<float*>(base + W.pmax), reinterpret_cast<int*>(base + W.parg),
               reinterpret_cast<float*>(base + W.psum), nullptr};
  g.pent = conf_kind == DLLM_CONF_NEG_ENTROPY ? reinterpret_cast<float*>(base + W.pent) : nullptr;
  const bool sample = temperature > 0.f;
  g.inv_temp = sample ? 1.0f / temperature : 0.f;
  g.seed = seed;
  g.step = (int)step;
  g.pos0 = block_begin;
  g.pscore = sample ? reinterpret_cast<float*>(base + W.pscore) : nullptr;
  g.pidx = sample ? reinterpret_cast<int*>(base + W.pidx) : nullptr;
  g.plogit = sample ? reinterpret_cast<float*>(base + W.plogit) : nullptr;
  rc = launch_gemm(g, P, s);
  if (rc) return rc;
  // 3) merge, confidence, top-k commit
  unsigned int* done = reinterpret_cast<unsigned int*>(base + W.done);
  cudaError_t e = cudaMemsetAsync(done, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return cuda_fail(e, "zero the merge counter");
  e = launch_pdl(lmhead_merge_commit_kernel, dim3((unsigned)R), dim3(256), 0, s,
                 reinterpret_cast<const float*>(base + W.pmax), reinterpret_cast<const int*>(base + W.parg),
                 reinterpret_cast<const float*>(base + W.psum), reinterpret_cast<const float*>(base + W.pent),
                 g.pscore, g.pidx, g.plogit, (int)conf_kind, W.P, (int)R, canvas, mask_id, (int)block_begin,
                 (int)k_commit, out_pos, out_id, out_conf, row_id, row_conf, reinterpret_cast<float*>(base + W.conf),
                 reinterpret_cast<int*>(base + W.id), done,
                 make_bounds({{base + W.pmax, (size_t)W.P * R * 4},
                              {base + W.parg, (size_t)W.P * R * 4},
                              {base + W.psum, (size_t)W.P * R * 4},
                              {base + W.pent, (size_t)W.P * R * 4},
                              {g.pscore, (size_t)W.P * R * 4},
                              {g.pidx, (size_t)W.P * R * 4},
                              {g.plogit, (size_t)W.P * R * 4},
                              {canvas, (size_t)L * 4},
                              {out_pos, (size_t)k_commit * 4},
                              {out_id, (size_t)k_commit * 4},
                              {out_conf, (size_t)k_commit * 4},
                              {row_id, (size_t)R * 4},
                              {row_conf, (size_t)R * 4},
                              {base + W.conf, (size_t)R * 4},
                              {base + W.id, (size_t)R * 4},
                              {done, 4}}));
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch lmhead_merge_commit");
}


DLLM_API int dllm_lmhead_masked_select(const float* hidden, int64_t L, int64_t d, int64_t ldh, const float* out_norm_w,
                                       float eps, const void* w_out_packed, int64_t vocab, int32_t* canvas,
                                       int32_t mask_id, int32_t block_begin, int32_t block_end, int32_t k_commit,
                                       int32_t* out_pos, int32_t* out_id, float* out_conf, int32_t* row_id,
                                       float* row_conf, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  return dllm_lmhead_select(hidden, L, d, ldh, out_norm_w, eps, w_out_packed, vocab, canvas, mask_id, block_begin,
                            block_end, k_commit, DLLM_CONF_PMAX, 0.f, 0, 0, out_pos, out_id, out_conf, row_id,
                            row_conf, ws, ws_bytes, stream);
}


DLLM_API long long dllm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

DLLM_API size_t dllm_qgemm_partials_bytes(int type, int64_t m, int64_t n, int64_t k) {
  if (!block_bytes(type) || m <= 0 || n <= 0 || k <= 0 || k % QK) return 0;
  const QgemmPlan P = plan_qgemm(type, m, n, k);
  return align_up((size_t)P.splits * m * n * 4, 256);
}

DLLM_API int dllm_qgemm_partials(int type, const void* act, int64_t m, int64_t k, const void* w_packed, int64_t n,
                                 float* partials, size_t partials_bytes, int32_t* splits, dllm_stream_t stream) {
  DLLM_RANGE();
  if (!block_bytes(type))
    return fail(DLLM_E_TYPE, "dllm_qgemm_partials: unsupported block type %d", type);
  if (m <= 0 || m > 65536 || n <= 0 || n > (1 << 24) || k <= 0 || k % QK || k > (1 << 20))
    return fail(DLLM_E_SHAPE, "dllm_qgemm_partials: bad shape m=%lld n=%lld k=%lld", (long long)m, (long long)n,
                (long long)k);
  int rc = check_device();
  if (rc) return rc;
  CHECK_DEV(act, "act");
  CHECK_DEV(w_packed, "w_packed");
  CHECK_DEV(partials, "partials");
  if (!aligned(act, 256) || !aligned(w_packed, 256))
    return fail(DLLM_E_ALIGN, "dllm_qgemm_partials: act and w_packed must be 256-byte aligned");
  const QgemmPlan P = plan_qgemm(type, m, n, k);
  if (partials_bytes < (size_t)P.splits * m * n * 4)
    return fail(DLLM_E_WORKSPACE, "dllm_qgemm_partials: buffer has %zu bytes, needs %zu", partials_bytes,
                (size_t)P.splits * m * n * 4);
  if (splits) *splits = P.splits;
  GemmLaunch g{type, act, m, k, w_packed, n, partials, n, 0, partials, 0, nullptr, nullptr, nullptr, nullptr};
  return launch_gemm(g, P, (cudaStream_t)stream);
}

}  // extern "C"
