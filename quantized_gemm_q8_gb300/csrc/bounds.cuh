// Bounds-checked build. Compiled with -DDLLM_BOUNDS_CHECK (libdllm_checked.so, built beside
// the regular library), every global-memory access of the library's kernels first checks that
// it lies inside the buffer it targets. The buffers' extents are computed on the host from the
// call's shapes (the same sizes the C ABI documents) and travel with the launch as a Bounds
// value, one span per buffer. An access outside its span is skipped, ERR_BOUNDS is set in the
// device error word and the first failing site (file and line) is recorded; dllm_check then
// reports DLLM_E_BOUNDS with that site. Tensor-map (TMA) copies are checked by the hardware
// against the map's own extents and need no span. In the regular build Bounds is empty and
// every check is the constant true, so the kernels compile to the same code as without it.
#pragma once
#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace dllm {

constexpr int kMaxSpans = 16;

struct Bounds {
#ifdef DLLM_BOUNDS_CHECK
  unsigned long long lo[kMaxSpans], hi[kMaxSpans];  // span i = bytes [lo[i], hi[i])
  int* err;                                         // device error word
  int* site;                                        // first failing site (0: none yet)
#else
  char unused;
#endif
};

// Site of a check: a file number (each source file defines its own) and the source line.
#define DLLM_SITE_AT(file) ((file) * 100000 + __LINE__)

// True when bytes [p, p + bytes) lie inside span `span` of b. Otherwise records the failure and
// returns false; the caller skips the access.
__device__ __forceinline__ bool in_bounds(const Bounds& b, int span, const volatile void* p, size_t bytes, int site) {
#ifdef DLLM_BOUNDS_CHECK
  const unsigned long long a = reinterpret_cast<unsigned long long>(const_cast<const void*>(p));
  if (span >= 0 && span < kMaxSpans && a >= b.lo[span] && a + bytes <= b.hi[span] && a + bytes >= a) return true;
  atomicOr(b.err, ERR_BOUNDS);
  atomicCAS(b.site, 0, site);
  return false;
#else
  (void)b;
  (void)span;
  (void)p;
  (void)bytes;
  (void)site;
  return true;
#endif
}
#define BOK_AT(file, b, span, p, bytes) ::dllm::in_bounds((b), (span), (p), (bytes), DLLM_SITE_AT(file))

// Guarded global loads and stores of T (a scalar or a 16/8-byte vector): a load outside the
// span yields `dflt`, a store outside it is dropped.
template <typename T>
__device__ __forceinline__ T ld_chk(const Bounds& b, int span, const T* p, T dflt, int site) {
  return in_bounds(b, span, p, sizeof(T), site) ? *p : dflt;
}
template <typename T>
__device__ __forceinline__ void st_chk(const Bounds& b, int span, T* p, T v, int site) {
  if (in_bounds(b, span, p, sizeof(T), site)) *p = v;
}
#define LDB_AT(file, b, span, p, dflt) ::dllm::ld_chk((b), (span), (p), (dflt), DLLM_SITE_AT(file))
#define STB_AT(file, b, span, p, v) ::dllm::st_chk((b), (span), (p), (v), DLLM_SITE_AT(file))
// File numbers of the sites (dllm_check names the file): api.cu 1, layer.cu 2, peak.cu 4,
// qgemm.cuh 9, quant.cuh 10. A .cu file defines DLLM_FILE for its own checks.
#define BOK(b, span, p, bytes) BOK_AT(DLLM_FILE, b, span, p, bytes)
#define LDB(b, span, p, dflt) LDB_AT(DLLM_FILE, b, span, p, dflt)
#define STB(b, span, p, v) STB_AT(DLLM_FILE, b, span, p, v)

}  // namespace dllm
