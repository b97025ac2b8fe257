// LLaDA layer stream and full denoising step (mojo-dllm Technical Specification, section 11,
// the order inside a layer: normalize, Q/K/V projections, rotate Q and K, attention over all
// positions, O projection added to the stream, normalize, gated MLP added; Development plan, "Model facts": eps 1e-5, NORM RoPE theta 500000,
// 32 x 128 MHA non-causal, SwiGLU FFN, untied output). Every projection is the tcgen05
// quantized GEMM; the glue between them is fused into row kernels that consume the GEMMs'
// split-K partials directly (fixed summation order), so no intermediate takes an extra pass.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "qgemm.cuh"
#include "quant.cuh"

#define DLLM_FILE 2  // bounds-check sites of this file

namespace dllm {

// ---------------------------------------------------------------------------------------------
// RoPE table: cs[p][i] = (cos, sin) of p * theta^(-2i/hd), computed in f64 once per step.
// ---------------------------------------------------------------------------------------------
// Span (bounds-checked build): 0 cs.
__global__ void rope_table_kernel(float2* cs, int L, int half, double theta, int hd, Bounds bd) {
  griddep_wait();
  griddep_launch();
  const int p = blockIdx.x, i = threadIdx.x;
  if (p < L && i < half) {
    const double ang = (double)p * pow(theta, -2.0 * (double)i / (double)hd);
    double s, c;
    sincos(ang, &s, &c);
    STB(bd, 0, cs + p * half + i, make_float2((float)c, (float)s));
  }
}

// Token embedding: x[p] = decoded Q4_K row ids[p] of the GGUF table (AoS blocks), f32.
// w = d * scale * q - dmin * min is formed with one fused multiply-add.
// Spans (bounds-checked build): 0 the table, 1 ids, 2 x.
__global__ void embed_q4k_kernel(const uint8_t* __restrict__ table, int nsb, const int32_t* __restrict__ ids,
                                 float* __restrict__ x, int d, Bounds bd) {
  griddep_wait();
  griddep_launch();
  const int p = blockIdx.x;
  const int64_t row = LDB(bd, 1, ids + p, 0);
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    const uint8_t* blk = table + (row * nsb + k / QK) * 144;
    if (!BOK(bd, 0, blk, 144)) continue;
    const int i = k % QK, j = i / 32;
    const uint8_t* sc = blk + 4;
    int scale, mn;
    if (j < 4) {
      scale = sc[j] & 63;
      mn = sc[j + 4] & 63;
    } else {
      scale = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
      mn = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
    const uint8_t b = blk[16 + 32 * (i / 64) + (i % 32)];
    const int q = ((i % 64) < 32) ? (b & 15) : (b >> 4);
    const float dd = __half2float(*reinterpret_cast<const __half*>(blk));
    const float dm = __half2float(*reinterpret_cast<const __half*>(blk + 2));
    STB(bd, 2, x + (int64_t)p * d + k, fmaf(dd, (float)(scale * q), -dm * (float)mn));
  }
}

// x = hi + lo for a pair of f32 values, packed as two f16x2 words
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x, y);
  const __half2 l = __floats2half2_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Q, K, V of one layer from the split-K partials of the Q|K and V projections: the splits are
// summed in split order, RoPE rotates adjacent pairs of Q and K within each head (position =
// pos0 + row), Q is also scaled by 1/sqrt(hd). Out: QKV [L][3d] f32 (Q, K, V side by side), or,
// when `planes` is set (the tensor-core attention), six f16 planes [Qhi, Qlo, Khi, Klo, Vhi,
// Vlo][L][d] with x = hi + lo. With kcache / vcache set, K (after RoPE) and V also go to rows
// pos0 + row of those [*][d] caches. All partial loads of a thread are issued together.
__global__ void __launch_bounds__(256) qkv_reduce_rope_kernel(const float* __restrict__ Pqk, int Sqk,
                                                              const float* __restrict__ Pv, int Sv,
                                                              const float2* __restrict__ cs, int L, int d, int hd,
                                                              float qscale, float* __restrict__ QKV,
                                                              __half* __restrict__ planes, int pos0,
                                                              float* __restrict__ kcache, float* __restrict__ vcache,
                                                              Bounds bd) {
  griddep_wait();
  griddep_launch();
  // one thread per 4 consecutive columns (two RoPE pairs): 16-byte partial loads
  const int64_t nquad = (int64_t)L * (3 * d / 4);
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= nquad) return;
  const int p = (int)(i / (3 * d / 4)), c = 4 * (int)(i % (3 * d / 4));  // row, column in [Q | K | V]
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < 2 * d) {
    const float* src = Pqk + (int64_t)p * 2 * d + c;
    const int64_t st = (int64_t)L * 2 * d;
#pragma unroll 4
    for (int sp = 0; sp < Sqk; ++sp) {
      const float4 v = LDB(bd, 0, reinterpret_cast<const float4*>(src + sp * st), make_float4(0.f, 0.f, 0.f, 0.f));
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    const int64_t rp = (int64_t)(pos0 + p) * (hd / 2) + (c % hd) / 2;
    const float2 r0 = LDB(bd, 2, cs + rp, make_float2(1.f, 0.f)), r1 = LDB(bd, 2, cs + rp + 1, make_float2(1.f, 0.f));
    const float sc = c < d ? qscale : 1.f;
    a = make_float4((a.x * r0.x - a.y * r0.y) * sc, (a.x * r0.y + a.y * r0.x) * sc, (a.z * r1.x - a.w * r1.y) * sc,
                    (a.z * r1.y + a.w * r1.x) * sc);
  } else {
    const float* src = Pv + (int64_t)p * d + (c - 2 * d);
    const int64_t st = (int64_t)L * d;
#pragma unroll 4
    for (int sp = 0; sp < Sv; ++sp) {
      const float4 v = LDB(bd, 1, reinterpret_cast<const float4*>(src + sp * st), make_float4(0.f, 0.f, 0.f, 0.f));
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
  }
  if (kcache && c >= d) {
    float* dst = (c < 2 * d ? kcache : vcache) + (int64_t)(pos0 + p) * d + (c % d);
    STB(bd, c < 2 * d ? 4 : 5, reinterpret_cast<float4*>(dst), a);
  }
  if (planes) {
    const int which = c / d, col = c % d;
    uint32_t h0, l0, h1, l1;
    split2(a.x, a.y, h0, l0);
    split2(a.z, a.w, h1, l1);
    STB(bd, 3, reinterpret_cast<uint2*>(planes + ((int64_t)(2 * which) * L + p) * d + col), make_uint2(h0, h1));
    STB(bd, 3, reinterpret_cast<uint2*>(planes + ((int64_t)(2 * which + 1) * L + p) * d + col), make_uint2(l0, l1));
  } else {
    STB(bd, 3, reinterpret_cast<float4*>(QKV + (int64_t)p * 3 * d + c), a);
  }
}

// Non-causal multi-head attention O = softmax(q k^T) v per head, f32, split over chunks of 32
// keys (flash-decoding style): Lq query rows (q pre-scaled, row stride ldq) against Lk key and
// value rows (row stride ldkv); for self-attention on the reduced QKV ([L][3d]) q = QKV,
// k = QKV + d, v = QKV + 2d. CTA (head, 16 queries, chunk c) writes for each query the chunk's
// max score m_c, sum l_c = sum exp(s - m_c) and unnormalized a_c = sum exp(s - m_c) v;
// attn_merge_quant_kernel combines the chunks. Small
// CTAs (4 warps, 43 KB shared) let five share an SM. Warp w owns queries 4w..4w+3; lane = key
// of the chunk for the scores (k rows padded to 132 floats: a quarter-warp's float4 loads of 8
// keys hit distinct banks; q read as broadcast float4, query pairs as f32x2), and dims
// 4*lane..4*lane+3 for the PV product (probabilities through shared memory).
constexpr int ATT_QB = 16, ATT_KC = 32, ATT_HD = 128, ATT_KP = ATT_HD + 4, ATT_THREADS = 128;
constexpr int ATT_SMEM = (ATT_KC * ATT_KP + ATT_KC * ATT_HD + ATT_QB * ATT_HD + ATT_QB * ATT_KC) * 4;

__device__ __forceinline__ void fma2f(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n mov.b64 rc, {%0,%1};\n"
      " fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0,%1}, rc;\n}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

struct AttPart {
  float* acc;  // [nchunk][Lq][d]   unnormalized chunk sums a_c
  float* ml;   // [nchunk][Lq][heads][2]   (m_c, l_c)
};

__global__ void __launch_bounds__(ATT_THREADS) attention_partial_kernel(const float* __restrict__ Qm, int64_t ldq,
                                                                       const float* __restrict__ Km,
                                                                       const float* __restrict__ Vm, int64_t ldkv,
                                                                       AttPart part, int Lq, int Lk, int d,
                                                                       int heads, Bounds bd) {
  extern __shared__ float4 att_smem4[];
  float* Ks = reinterpret_cast<float*>(att_smem4);  // [KC][KP]
  float* Vs = Ks + ATT_KC * ATT_KP;                 // [KC][HD]
  float* Qs = Vs + ATT_KC * ATT_HD;                 // [QB][HD]
  float* Ps = Qs + ATT_QB * ATT_HD;                 // [QB][KC]
  griddep_wait();
  const int h = blockIdx.x, q0 = blockIdx.y * ATT_QB, c = blockIdx.z, k0 = c * ATT_KC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int HV = ATT_HD / 4;  // float4 per head row
  {
    constexpr int RQ = ATT_QB * HV / ATT_THREADS, RK = ATT_KC * HV / ATT_THREADS;
    float4 qv[RQ], kv[RK], vv[RK];
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int i = threadIdx.x + ATT_THREADS * r, p = q0 + i / HV;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      qv[r] = p < Lq ? LDB(bd, 0, reinterpret_cast<const float4*>(Qm + p * ldq + h * ATT_HD + 4 * (i % HV)), z4) : z4;
    }
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      const int i = threadIdx.x + ATT_THREADS * r, p = k0 + i / HV;
      const int64_t off = p * ldkv + h * ATT_HD + 4 * (i % HV);
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      kv[r] = p < Lk ? LDB(bd, 1, reinterpret_cast<const float4*>(Km + off), z4) : z4;
      vv[r] = p < Lk ? LDB(bd, 2, reinterpret_cast<const float4*>(Vm + off), z4) : z4;
    }
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int i = threadIdx.x + ATT_THREADS * r;
      *reinterpret_cast<float4*>(Qs + (i / HV) * ATT_HD + 4 * (i % HV)) = qv[r];
    }
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      const int i = threadIdx.x + ATT_THREADS * r;
      *reinterpret_cast<float4*>(Ks + (i / HV) * ATT_KP + 4 * (i % HV)) = kv[r];
      *reinterpret_cast<float4*>(Vs + (i / HV) * ATT_HD + 4 * (i % HV)) = vv[r];
    }
  }
  __syncthreads();
  // scores of 4 queries x key `lane`, as two f32x2 pairs of queries
  const float* qw = Qs + warp * 4 * ATT_HD;
  const float* kr = Ks + lane * ATT_KP;
  float s01[2] = {0.f, 0.f}, s23[2] = {0.f, 0.f};
#pragma unroll 4
  for (int e = 0; e < ATT_HD; e += 4) {
    const float4 k = *reinterpret_cast<const float4*>(kr + e);
    const float4 a0 = *reinterpret_cast<const float4*>(qw + e);
    const float4 a1 = *reinterpret_cast<const float4*>(qw + ATT_HD + e);
    const float4 a2 = *reinterpret_cast<const float4*>(qw + 2 * ATT_HD + e);
    const float4 a3 = *reinterpret_cast<const float4*>(qw + 3 * ATT_HD + e);
    fma2f(s01[0], s01[1], a0.x, a1.x, k.x, k.x);
    fma2f(s23[0], s23[1], a2.x, a3.x, k.x, k.x);
    fma2f(s01[0], s01[1], a0.y, a1.y, k.y, k.y);
    fma2f(s23[0], s23[1], a2.y, a3.y, k.y, k.y);
    fma2f(s01[0], s01[1], a0.z, a1.z, k.z, k.z);
    fma2f(s23[0], s23[1], a2.z, a3.z, k.z, k.z);
    fma2f(s01[0], s01[1], a0.w, a1.w, k.w, k.w);
    fma2f(s23[0], s23[1], a2.w, a3.w, k.w, k.w);
  }
  const bool valid = k0 + lane < Lk;
  const float sc[4] = {s01[0], s01[1], s23[0], s23[1]};
  float* pw = Ps + warp * 4 * ATT_KC;
  float mq[4], lq[4];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    const float sv = valid ? sc[qq] : -INFINITY;
    float mx = sv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float pr = expf(sv - mx);  // the chunk's key k0 is always valid, so mx is finite
    float ps = pr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    mq[qq] = mx;
    lq[qq] = ps;
    pw[qq * ATT_KC + lane] = pr;
  }
  __syncwarp();
  float acc[4][4];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[qq][i] = 0.f;
#pragma unroll 2
  for (int j = 0; j < ATT_KC; j += 4) {  // keys past Lk have p = 0 and zero V rows
    float4 pj[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) pj[qq] = *reinterpret_cast<const float4*>(pw + qq * ATT_KC + j);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float4 vv = *reinterpret_cast<const float4*>(Vs + (j + t) * ATT_HD + lane * 4);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const float pv = t == 0 ? pj[qq].x : t == 1 ? pj[qq].y : t == 2 ? pj[qq].z : pj[qq].w;
        fma2f(acc[qq][0], acc[qq][1], pv, pv, vv.x, vv.y);
        fma2f(acc[qq][2], acc[qq][3], pv, pv, vv.z, vv.w);
      }
    }
  }
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    const int qi = q0 + warp * 4 + qq;
    if (qi < Lq) {
      STB(bd, 3, reinterpret_cast<float4*>(part.acc + ((int64_t)c * Lq + qi) * d + h * ATT_HD + lane * 4),
          make_float4(acc[qq][0], acc[qq][1], acc[qq][2], acc[qq][3]));
      if (lane == 0)
        STB(bd, 4, reinterpret_cast<float2*>(part.ml + (((int64_t)c * Lq + qi) * heads + h) * 2),
            make_float2(mq[qq], lq[qq]));
    }
  }
  griddep_launch();
}

// Tensor-core attention for canvases of up to TA_KEYS tokens. CTA (head, 128 queries, chunk of
// TA_KC keys), 8 warps; warp w serves TMEM lane quarter w % 4 (query rows 32 (w % 4) ..) and
// half w / 4 of the chunk's keys. Splitting the keys in two chunks halves each CTA's work and
// doubles the CTAs (128 at L = 148); attn_merge_quant_kernel combines the chunks.
// Operands are f16 head/tail pairs x = hi + lo (qkv_reduce_rope_kernel writes the planes):
//   Q, K    by TMA (128-byte swizzle, the K-major layout of the GEMM's activation operand),
//           keys past L read as zeros;
//   V^T     by a register transpose of the V planes into the no-swizzle K-major layout
//           (core matrices of 8 rows x 16 bytes, 128 bytes apart along K, 8-row groups SBO apart).
// One thread of warp 0 issues S = Q K^T (24 MMAs: M 128, N 80, K 16 x 8, terms hi*hi + hi*lo +
// lo*hi) into TMEM as soon as Q and K land, while warps 1-7 stage V^T; each row's softmax over the chunk is exact (the two column halves meet through
// shared memory); P goes back as head/tail planes over Q and K; O = P V (15 MMAs: M 128, N 128,
// K 16 x 5) and each row is written unnormalized with its chunk's (m, l). The three-term
// products carry each product to ~2^-22 relative, far below the f32 accumulation's own
// rounding. Values must stay inside the f16 range.
constexpr int TA_M = 128, TA_KC = 80, TA_KEYS = 2 * TA_KC, TA_HD = 128, TA_THREADS = 256, TA_BOXR = 16;
constexpr int TA_ATOM_Q = TA_M * 128;                 // one 64-dim swizzled atom column of Q rows
constexpr int TA_ATOM_K = TA_KC * 128;                // ... of K rows
constexpr int TA_SBO_P = (TA_KC / 8) * 128;           // 8-row group stride of P (K = keys)
constexpr int TA_SBO_V = (TA_KC / 8) * 128 + 16;      // ... of V^T, padded: spreads the staging stores
constexpr int TA_VPL = (TA_HD / 8) * TA_SBO_V;        // one V^T plane
constexpr int TA_PPL = (TA_M / 8) * TA_SBO_P;         // one P plane
// Q[hl][atom] at (2 hl + atom) TA_ATOM_Q; K[hl][atom] after them; V^T hi, lo last
constexpr int TA_OFF_Q = 0, TA_OFF_K = 4 * TA_ATOM_Q, TA_OFF_VH = TA_OFF_K + 4 * TA_ATOM_K;
constexpr int TA_OFF_VL = TA_OFF_VH + TA_VPL;
constexpr int TA_OFF_PH = 0, TA_OFF_PL = TA_PPL;      // P overwrites Q and K once S is complete
constexpr int TA_OFF_RED = TA_OFF_VL + TA_VPL;        // row max / sum exchange, after V^T: the O
                                                      // staging below overwrites Q, K and P
constexpr int TA_OP = TA_HD + 4;                      // padded O row (floats) for the write-back
constexpr int TA_SMEM = TA_OFF_RED + 2 * 2 * TA_M * 4 + 1024;  // + slack to align the base to 1024
constexpr uint32_t TA_TX = (4 * TA_M + 4 * TA_KC) * 128;  // TMA bytes of Q and K
static_assert(2 * TA_PPL <= TA_OFF_VH, "P fits over Q and K");
static_assert(TA_M * TA_OP * 4 <= TA_OFF_VH, "O staging fits over Q, K and P");
static_assert(TA_ATOM_Q % 1024 == 0 && TA_ATOM_K % 1024 == 0, "swizzle atoms 1024-byte aligned");
static_assert(TA_SMEM + 64 <= 232448, "shared memory budget");
static_assert(TA_KC % 16 == 0 && TA_KC % TA_BOXR == 0 && (TA_KC / 2) % 8 == 0, "chunk shape");
constexpr int TA_COLS = 256;                          // S at columns [0, 80), O at [80, 208)

__global__ void __launch_bounds__(TA_THREADS, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap qk_map, const __half* __restrict__ planes, AttPart part,
                        int L, int d, int heads, int* err, Bounds bd) {
  extern __shared__ uint8_t ta_raw[];
  __shared__ uint64_t ta_bar[3];
  __shared__ uint32_t ta_tmem;
  // 1024-byte aligned base (the swizzled operands), by offset from the shared array
  uint8_t* ta_smem = ta_raw + ((1024u - (smem_u32(ta_raw) & 1023u)) & 1023u);
  float(*ta_red)[2][TA_M] = reinterpret_cast<float(*)[2][TA_M]>(ta_smem + TA_OFF_RED);  // [max|sum][half][row]
  const int h = blockIdx.x, q0 = blockIdx.y * TA_M, kb = blockIdx.z * TA_KC;  // keys [kb, kb + TA_KC)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, ch = warp >> 2, row = 32 * qd + lane;
  const uint32_t sbase = smem_u32(ta_smem);
  const uint32_t bar_in = smem_u32(&ta_bar[0]), bar_s = smem_u32(&ta_bar[1]), bar_o = smem_u32(&ta_bar[2]);
  if (threadIdx.x == 0) {
    mbar_init(bar_in, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_barrier_init();
    prefetch_tensormap(&qk_map);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&ta_tmem), TA_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // the planes are the preceding kernel's output
  if (threadIdx.x == 0) {
    // Q (planes 0, 1) rows q0.., K (planes 2, 3) rows kb..: boxes of 64 dims x TA_BOXR rows
    mbar_expect_tx(bar_in, TA_TX);
#pragma unroll 1
    for (int hl = 0; hl < 2; ++hl)
#pragma unroll 1
      for (int a = 0; a < 2; ++a) {
        for (int b = 0; b < TA_M / TA_BOXR; ++b)
          tma_g2s_3d(sbase + TA_OFF_Q + (2 * hl + a) * TA_ATOM_Q + b * TA_BOXR * 128, &qk_map, h * TA_HD + 64 * a,
                     q0 + b * TA_BOXR, hl, bar_in);
        for (int b = 0; b < TA_KC / TA_BOXR; ++b)
          tma_g2s_3d(sbase + TA_OFF_K + (2 * hl + a) * TA_ATOM_K + b * TA_BOXR * 128, &qk_map, h * TA_HD + 64 * a,
                     kb + b * TA_BOXR, 2 + hl, bar_in);
      }
  }
  const uint32_t tmem = ta_tmem;
  volatile int never = 0;
  bool ok = true;
  if (warp == 0) {
    // S = Q K^T as soon as Q and K have landed, while warps 1-7 stage V^T
    if (lane == 0) {
      ok = mbar_wait(bar_in, 0, &never, kDefaultTimeoutCycles);
      tc_fence_after();
      constexpr uint32_t IDS = idesc_f16(TA_M, TA_KC);
#pragma unroll 1
      for (int kk = 0; kk < TA_HD / 16 && ok; ++kk) {
        const int a = kk >> 2;
        const uint32_t ko = (uint32_t)(kk & 3) * 32;  // K advance inside the 128-byte swizzled row
        const uint64_t qh = desc_sw128(sbase + TA_OFF_Q + (0 + a) * TA_ATOM_Q + ko);
        const uint64_t ql = desc_sw128(sbase + TA_OFF_Q + (2 + a) * TA_ATOM_Q + ko);
        const uint64_t kh = desc_sw128(sbase + TA_OFF_K + (0 + a) * TA_ATOM_K + ko);
        const uint64_t kl = desc_sw128(sbase + TA_OFF_K + (2 + a) * TA_ATOM_K + ko);
        mma_f16(tmem, qh, kh, IDS, kk > 0);
        mma_f16(tmem, qh, kl, IDS, 1);
        mma_f16(tmem, ql, kh, IDS, 1);
      }
      mma_commit(bar_s);  // arrives even when the inputs timed out, so the waits below end
    }
  } else {
    // V^T (rows = dims, K = the chunk's keys) by a register transpose of the V planes: item =
    // (key pair, block of 8 dims), all of a thread's loads in flight, then (key, key + 1) pairs
    // per 4-byte store; warps 1-7
    constexpr int NST = TA_THREADS - 32;
    const int tid = threadIdx.x - 32;
    const int64_t pl = (int64_t)L * d;
    constexpr int NIT = (TA_KC / 2) * (TA_HD / 8), PER = (NIT + NST - 1) / NST;
    uint4 vh[PER][2], vl[PER][2];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + u * NST;
      const int k0 = 2 * (i / (TA_HD / 8)), nb = i % (TA_HD / 8);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        vh[u][e] = vl[u][e] = make_uint4(0u, 0u, 0u, 0u);
        if (i < NIT && kb + k0 + e < L) {
          const __half* src = planes + (int64_t)(kb + k0 + e) * d + h * TA_HD + 8 * nb;
          vh[u][e] = LDB(bd, 0, reinterpret_cast<const uint4*>(src + 4 * pl), vh[u][e]);
          vl[u][e] = LDB(bd, 0, reinterpret_cast<const uint4*>(src + 5 * pl), vl[u][e]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + u * NST;
      if (i >= NIT) break;
      const int k0 = 2 * (i / (TA_HD / 8)), nb = i % (TA_HD / 8);
      const uint32_t* h0 = reinterpret_cast<const uint32_t*>(&vh[u][0]);
      const uint32_t* h1 = reinterpret_cast<const uint32_t*>(&vh[u][1]);
      const uint32_t* l0 = reinterpret_cast<const uint32_t*>(&vl[u][0]);
      const uint32_t* l1 = reinterpret_cast<const uint32_t*>(&vl[u][1]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {  // dim 8 nb + e: key k0 in the low half, k0 + 1 in the high half
        const int sh = 16 * (e & 1);
        const uint32_t hw = ((h0[e >> 1] >> sh) & 0xFFFFu) | (((h1[e >> 1] >> sh) & 0xFFFFu) << 16);
        const uint32_t lw = ((l0[e >> 1] >> sh) & 0xFFFFu) | (((l1[e >> 1] >> sh) & 0xFFFFu) << 16);
        const int o = nb * TA_SBO_V + (k0 >> 3) * 128 + e * 16 + (k0 & 7) * 2;
        *reinterpret_cast<uint32_t*>(ta_smem + TA_OFF_VH + o) = hw;
        *reinterpret_cast<uint32_t*>(ta_smem + TA_OFF_VL + o) = lw;
      }
    }
    fence_proxy_async();  // V^T is read by the tensor core
  }
  __syncthreads();
  griddep_launch();
  // this thread's row, its half of the chunk's columns of S: keys kb + [HK ch, HK ch + HK)
  ok = __all_sync(0xffffffffu, mbar_wait(bar_s, 0, &never, kDefaultTimeoutCycles));
  tc_fence_after();
  const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
  constexpr int HK = TA_KC / 2;
  float m = -INFINITY, l = 0.f;
  {
    uint32_t sv[HK];
#pragma unroll
    for (int c = 0; c < HK / 8; ++c) tmem_ld8(trow + HK * ch + 8 * c, *reinterpret_cast<uint32_t(*)[8]>(sv + 8 * c));
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < HK; ++k)
      if (kb + HK * ch + k < L) m = fmaxf(m, __uint_as_float(sv[k]));
    ta_red[0][ch][row] = m;
    __syncthreads();
    m = fmaxf(ta_red[0][0][row], ta_red[0][1][row]);  // the chunk's first key is real, so m is finite
    // p = e^(s - m) as 2^((s - m) log2 e) (exp2f: 2 ulp)
    constexpr float LOG2E = 1.4426950408889634f;
    const float ml2 = m * LOG2E;
#pragma unroll
    for (int c = 0; c < HK / 8; ++c) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = HK * ch + 8 * c + e;
        pv[e] = kb + k < L ? exp2f(fmaf(__uint_as_float(sv[8 * c + e]), LOG2E, -ml2)) : 0.f;
        l += pv[e];
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split2(pv[2 * e], pv[2 * e + 1], hi[e], lo[e]);
      const int o = (row >> 3) * TA_SBO_P + (HK / 8 * ch + c) * 128 + (row & 7) * 16;
      *reinterpret_cast<uint4*>(ta_smem + TA_OFF_PH + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ta_smem + TA_OFF_PL + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    ta_red[1][ch][row] = l;
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  l = ta_red[1][0][row] + ta_red[1][1][row];
  if (threadIdx.x == 0) {
    constexpr uint32_t IDO = idesc_f16(TA_M, TA_HD);
#pragma unroll 1
    for (int kk = 0; kk < TA_KC / 16 && ok; ++kk) {
      const uint32_t ko = (uint32_t)kk * 256;
      const uint64_t ph = desc_noswz(sbase + TA_OFF_PH + ko, 128, TA_SBO_P);
      const uint64_t pl = desc_noswz(sbase + TA_OFF_PL + ko, 128, TA_SBO_P);
      const uint64_t vh = desc_noswz(sbase + TA_OFF_VH + ko, 128, TA_SBO_V);
      const uint64_t vl = desc_noswz(sbase + TA_OFF_VL + ko, 128, TA_SBO_V);
      mma_f16(tmem + TA_KC, ph, vh, IDO, kk > 0);
      mma_f16(tmem + TA_KC, ph, vl, IDO, 1);
      mma_f16(tmem + TA_KC, pl, vh, IDO, 1);
    }
    mma_commit(bar_o);
  }
  ok = ok && __all_sync(0xffffffffu, mbar_wait(bar_o, 0, &never, kDefaultTimeoutCycles));
  tc_fence_after();
  // O through shared memory (rows padded to TA_OP floats, over the finished Q, K and P), then out
  // row-contiguously into chunk blockIdx.z: this thread's row, its half of the dims; all lanes
  // load from TMEM
  const int q = q0 + row;
  const int64_t cofs = (int64_t)blockIdx.z * L;  // the chunk's first row in the partial arrays
  {
    float* os = reinterpret_cast<float*>(ta_smem);
    uint32_t ov[TA_HD / 2];
#pragma unroll
    for (int c = 0; c < TA_HD / 32; ++c)
      tmem_ld16(trow + TA_KC + (TA_HD / 2) * ch + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(ov + 16 * c));
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < TA_HD / 2; e += 4)
      *reinterpret_cast<uint4*>(os + row * TA_OP + (TA_HD / 2) * ch + e) = make_uint4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
    if (ok && ch == 0 && q < L)
      STB(bd, 2, reinterpret_cast<float2*>(part.ml + ((cofs + q) * heads + h) * 2), make_float2(m, l));
    __syncthreads();
    if (ok) {
      float* dst = part.acc + (cofs + q0) * d + h * TA_HD;
#pragma unroll 4
      for (int i = threadIdx.x; i < TA_M * (TA_HD / 4); i += TA_THREADS) {
        const int r = i / (TA_HD / 4), c4 = i % (TA_HD / 4);
        if (q0 + r < L)
          STB(bd, 1, reinterpret_cast<float4*>(dst + (int64_t)r * d + 4 * c4),
              *reinterpret_cast<const float4*>(os + r * TA_OP + 4 * c4));
      }
    }
  }
  if (!ok && threadIdx.x == 0) atomicOr(err, ERR_TIMEOUT_OTHER);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TA_COLS);
  }
}

// Merge the key chunks of the attention and quantize the output to Q8_K in one pass: warp
// (blockIdx.y * 8 + w) of row blockIdx.x handles super-block sb (dims 256 sb .. = two heads);
// lane's 8 dims belong to head 2 sb + lane / 16. O = sum_c e^(m_c - M) a_c / sum_c e^(m_c - M) l_c.
// Spans (bounds-checked build): 0 part.acc, 1 part.ml; the output carries its own.
__global__ void __launch_bounds__(256) attn_merge_quant_kernel(AttPart part, int nchunk, int L, int d, int heads,
                                                               QuantOut o, WPrefetch pf, Bounds bd) {
  if (threadIdx.x == 0 && blockIdx.y == 0) prefetch_weights(pf);
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const int sb = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nsb = d / QK;
  if (sb >= nsb) return;
  float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (row < L) {
    const int dim = sb * QK + 8 * lane, h = dim / ATT_HD;
    float M = -INFINITY;
    for (int c = 0; c < nchunk; ++c)
      M = fmaxf(M, LDB(bd, 1, (const float*)part.ml + (((int64_t)c * L + row) * heads + h) * 2, -INFINITY));
    float den = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      const float2 ml = LDB(bd, 1, reinterpret_cast<const float2*>(part.ml + (((int64_t)c * L + row) * heads + h) * 2),
                            make_float2(-INFINITY, 0.f));
      const float w = expf(ml.x - M);
      den = fmaf(w, ml.y, den);
      const float* ac = part.acc + ((int64_t)c * L + row) * d + dim;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 a0 = LDB(bd, 0, reinterpret_cast<const float4*>(ac), z4);
      const float4 a1 = LDB(bd, 0, reinterpret_cast<const float4*>(ac + 4), z4);
      v[0] = fmaf(w, a0.x, v[0]); v[1] = fmaf(w, a0.y, v[1]); v[2] = fmaf(w, a0.z, v[2]); v[3] = fmaf(w, a0.w, v[3]);
      v[4] = fmaf(w, a1.x, v[4]); v[5] = fmaf(w, a1.y, v[5]); v[6] = fmaf(w, a1.z, v[6]); v[7] = fmaf(w, a1.w, v[7]);
    }
    const float inv = 1.0f / den;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= inv;
  }
  q8k_emit(v, row, L, sb, d, o);  // padding rows quantize zeros
}

// Fused row kernels: the source of each row is built from split partials, then quantized.
enum RowMode : int {
  ROW_RESID_NORM_QUANT = 0,  // x += sum_s P; act = Q8_K(RMSNorm(x) * w)
  ROW_SUM_QUANT = 1,         // act = Q8_K(sum_s P)
  ROW_SWIGLU_QUANT = 2,      // act = Q8_K(silu(sum_s G) * sum_s U), G|U side by side in P
  ROW_RESID_ONLY = 3,        // x += sum_s P
};

struct RowArgs {
  float* x;
  const float* P;
  int S;
  int64_t pstride;
  int ldp;
  const float* norm_w;
  float eps;
  int rows, k;
  QuantOut o;
  WPrefetch pf0, pf1;  // the next GEMMs' first weights, prefetched into L2 (optional)
  Bounds bd;           // bounds-checked build: spans 0 x, 1 P, 2 norm_w
};

// Residual modes (RESID_NORM_QUANT, RESID_ONLY): one CTA per row, warp w holding super-blocks
// w, w + nwarp, ... (up to RR_J of them) in registers from the residual add through the
// quantization, lane = 8 consecutive values; RMSNorm needs the row's sum of squares, one block
// reduction. Each thread's partial loads are issued together.
constexpr int RR_WARPS = 16, RR_J = 4;  // rows of up to RR_WARPS * RR_J * 256 = 16384 values
template <int MODE>
__global__ void __launch_bounds__(RR_WARPS * 32) row_resid_kernel(RowArgs a) {
  __shared__ float red[RR_WARPS];
  if (threadIdx.x == 0) {
    prefetch_weights(a.pf0);
    prefetch_weights(a.pf1);
  }
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int nsb = a.k / QK;
  if (row >= a.rows) {  // padding rows of the operand planes
    if (MODE != ROW_RESID_ONLY) {
      float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int sb = warp; sb < nsb; sb += nwarp) q8k_emit(z, row, a.rows, sb, a.k, a.o);
    }
    return;
  }
  const float* Pr = a.P + (int64_t)row * a.ldp;
  float* xr = a.x + (int64_t)row * a.k;
  float v[RR_J][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < RR_J; ++j) {
    const int sb = warp + j * nwarp;
    if (sb < nsb) {
      const int base = sb * QK + 8 * lane;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 x0 = LDB(a.bd, 0, reinterpret_cast<const float4*>(xr + base), z4);
      float4 x1 = LDB(a.bd, 0, reinterpret_cast<const float4*>(xr + base + 4), z4);
#pragma unroll 4
      for (int sp = 0; sp < a.S; ++sp) {
        const float4 p0 = LDB(a.bd, 1, reinterpret_cast<const float4*>(Pr + sp * a.pstride + base), z4);
        const float4 p1 = LDB(a.bd, 1, reinterpret_cast<const float4*>(Pr + sp * a.pstride + base + 4), z4);
        x0.x += p0.x; x0.y += p0.y; x0.z += p0.z; x0.w += p0.w;
        x1.x += p1.x; x1.y += p1.y; x1.z += p1.z; x1.w += p1.w;
      }
      STB(a.bd, 0, reinterpret_cast<float4*>(xr + base), x0);
      STB(a.bd, 0, reinterpret_cast<float4*>(xr + base + 4), x1);
      v[j][0] = x0.x; v[j][1] = x0.y; v[j][2] = x0.z; v[j][3] = x0.w;
      v[j][4] = x1.x; v[j][5] = x1.y; v[j][6] = x1.z; v[j][7] = x1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[j][i], v[j][i], ss);
    }
  }
  if constexpr (MODE != ROW_RESID_ONLY) {  // RMSNorm + Q8_K of the updated row
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nwarp; ++w) tot += red[w];
    const float rstd = 1.0f / sqrtf(tot / (float)a.k + a.eps);
#pragma unroll
    for (int j = 0; j < RR_J; ++j) {
      const int sb = warp + j * nwarp;
      if (sb < nsb) {
        const int base = sb * QK + 8 * lane;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 w0 = LDB(a.bd, 2, reinterpret_cast<const float4*>(a.norm_w + base), z4);
        const float4 w1 = LDB(a.bd, 2, reinterpret_cast<const float4*>(a.norm_w + base + 4), z4);
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[j][i] = v[j][i] * rstd * w[i];
        q8k_emit(v[j], row, a.rows, sb, a.k, a.o);
      }
    }
  }
}

// Per-super-block modes (SUM_QUANT, SWIGLU_QUANT): warp (blockIdx.y * 8 + w) of row blockIdx.x
// builds and quantizes one super-block; each lane's partial loads are issued together.
template <int MODE>
__global__ void __launch_bounds__(256) row_sb_kernel(RowArgs a) {
  if (threadIdx.x == 0 && blockIdx.y == 0) {
    prefetch_weights(a.pf0);
    prefetch_weights(a.pf1);
  }
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const int sb = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nsb = a.k / QK;
  if (sb >= nsb) return;
  float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (row < a.rows) {
    const int base = sb * QK + 8 * lane;
    const float* ps = a.P + (int64_t)row * a.ldp + base;
    float u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = 0; s < a.S; ++s, ps += a.pstride) {
      const float4 p0 = LDB(a.bd, 1, reinterpret_cast<const float4*>(ps), z4);
      const float4 p1 = LDB(a.bd, 1, reinterpret_cast<const float4*>(ps + 4), z4);
      v[0] += p0.x; v[1] += p0.y; v[2] += p0.z; v[3] += p0.w;
      v[4] += p1.x; v[5] += p1.y; v[6] += p1.z; v[7] += p1.w;
      if (MODE == ROW_SWIGLU_QUANT) {
        const float4 q0 = LDB(a.bd, 1, reinterpret_cast<const float4*>(ps + a.k), z4);
        const float4 q1 = LDB(a.bd, 1, reinterpret_cast<const float4*>(ps + a.k + 4), z4);
        u[0] += q0.x; u[1] += q0.y; u[2] += q0.z; u[3] += q0.w;
        u[4] += q1.x; u[5] += q1.y; u[6] += q1.z; u[7] += q1.w;
      }
    }
    if (MODE == ROW_SWIGLU_QUANT) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = v[i] / (1.0f + expf(-v[i])) * u[i];
    }
  }
  q8k_emit(v, row, a.rows, sb, a.k, a.o);  // padding rows quantize zeros
}

static QuantOut quant_out(void* act, int64_t rows, int64_t k, float* vtap = nullptr) {
  ActLayout L = act_layout(rows, k);
  uint8_t* base = static_cast<uint8_t*>(act);
  QuantOut o{nullptr, nullptr, nullptr, reinterpret_cast<__half*>(base + L.off_a), base + L.off_j,
             reinterpret_cast<float*>(base + L.off_d), (int)L.lpad, vtap};
  set_quant_bounds(o, rows, k);
  return o;
}

// The first-wave weights of a GEMM launch with plan P (see WPrefetch): as many super-blocks per
// unit as the kernel's weight ring holds (3 Q4_K, 6 Q6_K), at most the unit's own.
static WPrefetch wprefetch(int type, const void* w, const QgemmPlan& P) {
  WPrefetch f{};
  f.wblob = static_cast<const uint8_t*>(w);
  f.tiles_n = P.tiles_n;
  f.tiles_m = P.tiles_m;
  f.nsb = P.nsb;
  f.sbps = P.sbps;
  f.units = std::min(P.units, P.grid);
  f.w_bytes = type == DLLM_Q4_K ? Q4K_BLOB : Q6K_BLOB;
  f.ahead = std::min(P.sbps, type == DLLM_Q4_K ? 3 : 6);
  f.bd = make_bounds({{w, (size_t)P.tiles_n * P.nsb * f.w_bytes}});
  return f;
}

template <int MODE>
static int run_row(float* x, const float* P, int S, int64_t pstride, int ldp, const float* w, float eps, int rows,
                   int k, void* act, cudaStream_t s, float* vtap = nullptr, WPrefetch pf0 = {}, WPrefetch pf1 = {}) {
  RowArgs a{x, P, S, pstride, ldp, w, eps, rows, k, act ? quant_out(act, rows, k, vtap) : QuantOut{}, pf0, pf1,
            make_bounds({{x, (size_t)rows * k * 4}, {P, (size_t)S * pstride * 4}, {w, (size_t)k * 4}})};
  cudaError_t e;
  if (MODE == ROW_RESID_NORM_QUANT || MODE == ROW_RESID_ONLY) {
    const int grid = MODE == ROW_RESID_ONLY ? rows : (int)act_rows_padded(rows);
    const int warps = std::min(RR_WARPS, k / QK);  // k <= RR_WARPS * RR_J * 256: each warp holds <= RR_J
    e = launch_pdl(row_resid_kernel<MODE>, dim3(grid), dim3(32 * warps), 0, s, a);
  } else {
    const dim3 grid((unsigned)act_rows_padded(rows), (unsigned)((k / QK + 7) / 8));
    e = launch_pdl(row_sb_kernel<MODE>, grid, dim3(256), 0, s, a);
  }
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "launch row kernel");
}

// Test taps: Q, K, V of a layer as f32 [L][d] each, from the f16 head/tail planes of the
// tensor-core attention (x = hi + lo) or from the f32 [L][3d] rows of the chunked one.
// Spans (bounds-checked build): 0 planes, 1 QKV, 2 q, 3 k, 4 v.
__global__ void tap_qkv_kernel(const __half* __restrict__ planes, const float* __restrict__ QKV, int L, int d,
                               float* __restrict__ q, float* __restrict__ k, float* __restrict__ v, Bounds bd) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= (int64_t)L * 3 * d) return;
  const int which = (int)(i / ((int64_t)L * d));
  const int64_t r = i % ((int64_t)L * d), p = r / d, c = r % d;
  float val;
  const __half hz = __float2half(0.f);
  if (planes)
    val = __half2float(LDB(bd, 0, planes + (2 * which * (int64_t)L + p) * d + c, hz)) +
          __half2float(LDB(bd, 0, planes + ((2 * which + 1) * (int64_t)L + p) * d + c, hz));
  else
    val = LDB(bd, 1, QKV + p * 3 * d + which * d + c, 0.f);
  float* dst = which == 0 ? q : (which == 1 ? k : v);
  if (dst) STB(bd, 2 + which, dst + r, val);
}

static int tap_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (!dst) return DLLM_OK;
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? DLLM_OK : cuda_fail(e, "cudaMemcpyAsync (tap)");
}

// ---------------------------------------------------------------------------------------------
// Step workspace layout
// ---------------------------------------------------------------------------------------------
struct StepPlan {
  QgemmPlan qk, v, o, gu, dn;
  size_t x, act_d, act_ff, pqk, pv, po, pgu, pdn, qkv, att, attml, rope, lm, bytes;
};

// L rows run through the layers; Lk (0: L) is the canvas length, i.e. the attention's keys, the
// RoPE positions and the hidden-state rows (Lk > L: the block rows of a cached step).
static StepPlan step_plan(const dllm_model* m, int64_t L, int flags, bool lmhead, int64_t Lk = 0) {
  const int64_t d = m->d_model, f = m->d_ff;
  if (Lk <= 0) Lk = L;
  StepPlan S{};
  S.qk = plan_qgemm(DLLM_Q4_K, L, 2 * d, d);
  S.v = plan_qgemm(DLLM_Q6_K, L, d, d);
  S.o = plan_qgemm(DLLM_Q4_K, L, d, d);
  S.gu = plan_qgemm(DLLM_Q4_K, L, 2 * f, d);
  S.dn = plan_qgemm(DLLM_Q6_K, L, d, f);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  const bool full = flags & DLLM_STREAM_FULL;
  S.x = take(lmhead ? (size_t)Lk * d * 4 : 0);
  S.act_d = take(act_layout(L, d).bytes);
  S.act_ff = take(act_layout(L, f).bytes);
  // The split-K partials of Q|K, O, gate|up and down share one region: each is read by the row
  // kernel right after its GEMM and is dead before the next of them is written (each kernel
  // waits for its predecessor before it writes), so the GEMMs keep storing into lines that are
  // already in L2 instead of allocating fresh ones. V's partials are read together with Q|K's.
  {
    const size_t r1 = std::max(std::max((size_t)S.qk.splits * L * 2 * d * 4, (size_t)S.o.splits * L * d * 4),
                               std::max((size_t)S.gu.splits * L * 2 * f * 4, (size_t)S.dn.splits * L * d * 4));
    S.pqk = take(r1);
    S.po = S.pgu = S.pdn = S.pqk;
  }
  S.pv = take((size_t)S.v.splits * L * d * 4);
  S.qkv = take(full ? (size_t)L * 3 * d * 4 : 0);
  S.att = take(full ? (size_t)((Lk + 31) / 32) * L * d * 4 : 0);
  S.attml = take(full ? (size_t)((Lk + 31) / 32) * L * m->n_heads * 8 : 0);
  S.rope = take(full ? (size_t)Lk * (m->head_dim / 2) * 8 : 0);
  S.lm = 0;
  S.bytes = off;
  return S;
}

static int check_model(const dllm_model* m, int64_t L, const char* fn) {
  if (!m) return fail(DLLM_E_INVAL, "%s: model is NULL", fn);
  if (m->n_layers <= 0 || m->d_model <= 0 || m->d_model % QK || m->d_model > RR_WARPS * RR_J * QK || m->d_ff <= 0 ||
      m->d_ff % QK ||
      m->head_dim != ATT_HD || m->n_heads * m->head_dim != m->d_model || m->vocab <= 0)
    return fail(DLLM_E_SHAPE,
                "%s: unsupported model shape (d_model %% 256 == 0 and <= 16384, d_ff %% 256 == 0, head_dim == 128, "
                "n_heads * head_dim == d_model): d=%d d_ff=%d heads=%d head_dim=%d",
                fn, m->d_model, m->d_ff, m->n_heads, m->head_dim);
  if (L <= 0 || L > 8192) return fail(DLLM_E_SHAPE, "%s: L=%lld must be in [1, 8192]", fn, (long long)L);
  if (!m->layers) return fail(DLLM_E_INVAL, "%s: model->layers is NULL", fn);
  for (int i = 0; i < m->n_layers; ++i) {
    const dllm_layer& y = m->layers[i];
    const void* ps[7] = {y.wqk, y.wv, y.wo, y.wgu, y.wdown, y.attn_norm, y.ffn_norm};
    for (const void* p : ps)
      if (!device_ptr(p)) return fail(DLLM_E_INVAL, "%s: layer %d has a NULL or non-device weight pointer", fn, i);
  }
  return DLLM_OK;
}

static int gemm(int type, const void* act, int64_t m, int64_t k, const void* w, int64_t n, float* out,
                const QgemmPlan& P, cudaStream_t s) {
  GemmLaunch g{type, act, m, k, w, n, out, n, 0, out, 0, nullptr, nullptr, nullptr, nullptr};
  return launch_gemm(g, P, s);
}

// The forward pass over all layers; x is [L][d] (input for the linear stream, output always).
// kv (optional, full stream only): per layer K (after RoPE) then V of every row, [layers][2][L][d].
// taps (optional, tests): the intermediates of layer taps->layer are copied out as they appear.
static int forward(const dllm_model* m, const int32_t* canvas, int64_t L, float* x, int flags, uint8_t* ws,
                   const StepPlan& S, cudaStream_t s, float* kv = nullptr, const dllm_taps* taps = nullptr) {
  const int d = m->d_model, f = m->d_ff, hd = m->head_dim;
  const bool full = flags & DLLM_STREAM_FULL;
  float* Pqk = reinterpret_cast<float*>(ws + S.pqk);
  float* Pv = reinterpret_cast<float*>(ws + S.pv);
  float* Po = reinterpret_cast<float*>(ws + S.po);
  float* Pgu = reinterpret_cast<float*>(ws + S.pgu);
  float* Pdn = reinterpret_cast<float*>(ws + S.pdn);
  void* actd = ws + S.act_d;
  void* actf = ws + S.act_ff;
  int rc;
  const size_t rope_bytes = (size_t)L * (hd / 2) * 8, table_bytes = (size_t)m->vocab * (d / QK) * 144;
  if (full) {
    cudaError_t e = launch_pdl(rope_table_kernel, dim3((unsigned)L), dim3(hd / 2), 0, s,
                               reinterpret_cast<float2*>(ws + S.rope), (int)L, hd / 2, (double)m->rope_theta, hd,
                               make_bounds({{ws + S.rope, rope_bytes}}));
    note_launch();
    if (e == cudaSuccess)
      e = launch_pdl(embed_q4k_kernel, dim3((unsigned)L), dim3(256), 0, s, static_cast<const uint8_t*>(m->tok_embd),
                     d / QK, canvas, x, d,
                     make_bounds({{m->tok_embd, table_bytes}, {canvas, (size_t)L * 4}, {x, (size_t)L * d * 4}}));
    note_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch embedding");
  }
  // layer 0 input: RMSNorm + quantize of x
  if ((rc = quantize_rows(x, L, d, d, m->layers[0].attn_norm, m->eps, actd, s))) return rc;
  const size_t act_d_bytes = act_layout(L, d).bytes, act_f_bytes = act_layout(L, f).bytes;
  for (int li = 0; li < m->n_layers; ++li) {
    const dllm_layer& Ly = m->layers[li];
    const dllm_taps* tp = (taps && taps->layer == li) ? taps : nullptr;
    if (tp && (rc = tap_copy(tp->x_in, x, (size_t)L * d * 4, s))) return rc;
    if (tp && (rc = tap_copy(tp->act_attn, actd, act_d_bytes, s))) return rc;
    if ((rc = gemm(DLLM_Q4_K, actd, L, d, Ly.wqk, 2 * d, Pqk, S.qk, s))) return rc;
    if ((rc = gemm(DLLM_Q6_K, actd, L, d, Ly.wv, d, Pv, S.v, s))) return rc;
    if (full) {
      // Q, K, V: f32 rows for the chunked attention, or (short canvases) the f16 head/tail planes
      // of the tensor-core attention, in the same bytes
      const bool tc_att = L <= TA_KEYS;
      float* QKV = reinterpret_cast<float*>(ws + S.qkv);
      __half* planes = tc_att ? reinterpret_cast<__half*>(ws + S.qkv) : nullptr;
      const int64_t nquad = L * (3 * d / 4);
      float* kc = kv ? kv + (int64_t)li * 2 * L * d : nullptr;
      cudaError_t e = launch_pdl(qkv_reduce_rope_kernel, dim3((unsigned)((nquad + 255) / 256)), dim3(256), 0, s,
                                 (const float*)Pqk, S.qk.splits, (const float*)Pv, S.v.splits,
                                 reinterpret_cast<const float2*>(ws + S.rope), (int)L, d, hd, 1.0f / sqrtf((float)hd),
                                 QKV, planes, 0, kc, kc ? kc + L * d : nullptr,
                                 make_bounds({{Pqk, (size_t)S.qk.splits * L * 2 * d * 4},
                                              {Pv, (size_t)S.v.splits * L * d * 4},
                                              {ws + S.rope, rope_bytes},
                                              {ws + S.qkv, (size_t)L * 3 * d * 4},
                                              {kc, (size_t)L * d * 4},
                                              {kc ? kc + L * d : nullptr, (size_t)L * d * 4}}));
      note_launch();
      if (e != cudaSuccess) return cuda_fail(e, "launch qkv reduce");
      if (tp && (tp->q || tp->k || tp->v)) {
        const int64_t n3 = L * 3 * d;
        tap_qkv_kernel<<<(unsigned)((n3 + 255) / 256), 256, 0, s>>>(
            planes, tc_att ? nullptr : QKV, (int)L, d, tp->q, tp->k, tp->v,
            make_bounds({{planes, (size_t)L * 3 * d * 4}, {QKV, (size_t)L * 3 * d * 4}, {tp->q, (size_t)L * d * 4},
                         {tp->k, (size_t)L * d * 4}, {tp->v, (size_t)L * d * 4}}));
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch tap_qkv");
      }
      const AttPart ap{reinterpret_cast<float*>(ws + S.att), reinterpret_cast<float*>(ws + S.attml)};
      const size_t att_bytes = (size_t)((L + 31) / 32) * L * d * 4, ml_bytes = (size_t)((L + 31) / 32) * L * m->n_heads * 8;
      int nchunk = 1;
      if (tc_att) {  // whole rows per CTA on the tensor cores
        int* err = err_word();
        if (!err) return fail(DLLM_E_CUDA, "cannot resolve the device error word");
        CUtensorMap qk_map;
        if ((rc = make_planes_tmap(&qk_map, planes, 6, L, d, TA_BOXR))) return rc;
        e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TA_SMEM);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
        nchunk = (int)((L + TA_KC - 1) / TA_KC);
        const dim3 ag(m->n_heads, (unsigned)((L + TA_M - 1) / TA_M), (unsigned)nchunk);
        e = launch_pdl(attention_tc_kernel, ag, dim3(TA_THREADS), TA_SMEM, s, qk_map, (const __half*)planes, ap,
                       (int)L, d, m->n_heads, err,
                       make_bounds({{planes, (size_t)L * 3 * d * 4}, {ap.acc, att_bytes}, {ap.ml, ml_bytes}}));
      } else {  // longer canvases: chunks of 32 keys, merged below
        nchunk = (int)((L + ATT_KC - 1) / ATT_KC);
        e = cudaFuncSetAttribute(attention_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
        const dim3 ag(m->n_heads, (unsigned)((L + ATT_QB - 1) / ATT_QB), (unsigned)nchunk);
        const Span qkv{QKV, (size_t)L * 3 * d * 4};
        e = launch_pdl(attention_partial_kernel, ag, dim3(ATT_THREADS), ATT_SMEM, s, (const float*)QKV,
                       (int64_t)3 * d, (const float*)(QKV + d), (const float*)(QKV + 2 * d), (int64_t)3 * d, ap,
                       (int)L, (int)L, d, m->n_heads,
                       make_bounds({qkv, qkv, qkv, {ap.acc, att_bytes}, {ap.ml, ml_bytes}}));
      }
      note_launch();
      const dim3 mg((unsigned)act_rows_padded(L), (unsigned)((d / QK + 7) / 8));
      if (e == cudaSuccess)
        e = launch_pdl(attn_merge_quant_kernel, mg, dim3(256), 0, s, ap, nchunk, (int)L, d, m->n_heads,
                       quant_out(actd, L, d, tp ? tp->attn : nullptr), wprefetch(DLLM_Q4_K, Ly.wo, S.o),
                       make_bounds({{ap.acc, att_bytes}, {ap.ml, ml_bytes}}));
      note_launch();
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "launch attention");
    } else {
      // linear stream: the O projection consumes the V projection's output
      if ((rc = run_row<ROW_SUM_QUANT>(nullptr, Pv, S.v.splits, L * d, d, nullptr, 0.f, (int)L, d, actd, s,
                                       tp ? tp->attn : nullptr, wprefetch(DLLM_Q4_K, Ly.wo, S.o))))
        return rc;
    }
    if (tp && (rc = tap_copy(tp->act_o, actd, act_d_bytes, s))) return rc;
    if ((rc = gemm(DLLM_Q4_K, actd, L, d, Ly.wo, d, Po, S.o, s))) return rc;
    if ((rc = run_row<ROW_RESID_NORM_QUANT>(x, Po, S.o.splits, L * d, d, Ly.ffn_norm, m->eps, (int)L, d, actd, s,
                                            nullptr, wprefetch(DLLM_Q4_K, Ly.wgu, S.gu))))
      return rc;
    if (tp && (rc = tap_copy(tp->x_mid, x, (size_t)L * d * 4, s))) return rc;
    if (tp && (rc = tap_copy(tp->act_ffn, actd, act_d_bytes, s))) return rc;
    if ((rc = gemm(DLLM_Q4_K, actd, L, d, Ly.wgu, 2 * f, Pgu, S.gu, s))) return rc;
    if ((rc = run_row<ROW_SWIGLU_QUANT>(nullptr, Pgu, S.gu.splits, L * 2 * f, 2 * f, nullptr, 0.f, (int)L, f, actf,
                                        s, tp ? tp->h : nullptr, wprefetch(DLLM_Q6_K, Ly.wdown, S.dn))))
      return rc;
    if (tp && (rc = tap_copy(tp->act_down, actf, act_f_bytes, s))) return rc;
    if ((rc = gemm(DLLM_Q6_K, actf, L, f, Ly.wdown, d, Pdn, S.dn, s))) return rc;
    if (li + 1 < m->n_layers) {
      const dllm_layer& Ln = m->layers[li + 1];
      if ((rc = run_row<ROW_RESID_NORM_QUANT>(x, Pdn, S.dn.splits, L * d, d, Ln.attn_norm, m->eps, (int)L, d, actd,
                                              s, nullptr, wprefetch(DLLM_Q4_K, Ln.wqk, S.qk),
                                              wprefetch(DLLM_Q6_K, Ln.wv, S.v))))
        return rc;
    } else {
      if ((rc = run_row<ROW_RESID_ONLY>(x, Pdn, S.dn.splits, L * d, d, nullptr, 0.f, (int)L, d, nullptr, s)))
        return rc;
    }
    if (tp && (rc = tap_copy(tp->x_out, x, (size_t)L * d * 4, s))) return rc;
  }
  return DLLM_OK;
}

// The forward pass of a cached step over the block rows only (LLaDA's inter-step K/V cache,
// "--dual-cache"): rows [b0, b0 + R) of the canvas (length L) run through every layer; their
// queries attend to all L keys and values, which come from kv ([layers][2][L][d], K after
// RoPE, then V) written by the last refreshing step, with the block's own rows overwritten by
// their fresh K and V. x is [L][d]; only rows [b0, b0 + R) are computed. Not exact: the cached
// rows outside the block do not see the block's new tokens until the next refresh.
static int forward_block(const dllm_model* m, const int32_t* canvas, int64_t L, int64_t b0, int64_t R, float* x,
                         float* kv, uint8_t* ws, const StepPlan& S, cudaStream_t s) {
  const int d = m->d_model, f = m->d_ff, hd = m->head_dim;
  float* Pqk = reinterpret_cast<float*>(ws + S.pqk);
  float* Pv = reinterpret_cast<float*>(ws + S.pv);
  float* Po = reinterpret_cast<float*>(ws + S.po);
  float* Pgu = reinterpret_cast<float*>(ws + S.pgu);
  float* Pdn = reinterpret_cast<float*>(ws + S.pdn);
  void* actd = ws + S.act_d;
  void* actf = ws + S.act_ff;
  float* xb = x + b0 * d;
  int rc;
  const size_t rope_bytes = (size_t)L * (hd / 2) * 8, table_bytes = (size_t)m->vocab * (d / QK) * 144;
  cudaError_t e = launch_pdl(rope_table_kernel, dim3((unsigned)L), dim3(hd / 2), 0, s,
                             reinterpret_cast<float2*>(ws + S.rope), (int)L, hd / 2, (double)m->rope_theta, hd,
                             make_bounds({{ws + S.rope, rope_bytes}}));
  note_launch();
  if (e == cudaSuccess)
    e = launch_pdl(embed_q4k_kernel, dim3((unsigned)R), dim3(256), 0, s, static_cast<const uint8_t*>(m->tok_embd),
                   d / QK, canvas + b0, xb, d,
                   make_bounds({{m->tok_embd, table_bytes}, {canvas + b0, (size_t)R * 4}, {xb, (size_t)R * d * 4}}));
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch embedding");
  if ((rc = quantize_rows(xb, R, d, d, m->layers[0].attn_norm, m->eps, actd, s))) return rc;
  const int nchunk = (int)((L + ATT_KC - 1) / ATT_KC);
  e = cudaFuncSetAttribute(attention_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
  for (int li = 0; li < m->n_layers; ++li) {
    const dllm_layer& Ly = m->layers[li];
    float* kc = kv + (int64_t)li * 2 * L * d;
    float* vc = kc + L * d;
    if ((rc = gemm(DLLM_Q4_K, actd, R, d, Ly.wqk, 2 * d, Pqk, S.qk, s))) return rc;
    if ((rc = gemm(DLLM_Q6_K, actd, R, d, Ly.wv, d, Pv, S.v, s))) return rc;
    float* QKV = reinterpret_cast<float*>(ws + S.qkv);
    const int64_t nquad = R * (3 * d / 4);
    e = launch_pdl(qkv_reduce_rope_kernel, dim3((unsigned)((nquad + 255) / 256)), dim3(256), 0, s, (const float*)Pqk,
                   S.qk.splits, (const float*)Pv, S.v.splits, reinterpret_cast<const float2*>(ws + S.rope), (int)R, d,
                   hd, 1.0f / sqrtf((float)hd), QKV, (__half*)nullptr, (int)b0, kc, vc,
                   make_bounds({{Pqk, (size_t)S.qk.splits * R * 2 * d * 4},
                                {Pv, (size_t)S.v.splits * R * d * 4},
                                {ws + S.rope, rope_bytes},
                                {QKV, (size_t)R * 3 * d * 4},
                                {kc, (size_t)L * d * 4},
                                {vc, (size_t)L * d * 4}}));
    note_launch();
    if (e != cudaSuccess) return cuda_fail(e, "launch qkv reduce");
    const AttPart ap{reinterpret_cast<float*>(ws + S.att), reinterpret_cast<float*>(ws + S.attml)};
    const size_t att_bytes = (size_t)nchunk * R * d * 4, ml_bytes = (size_t)nchunk * R * m->n_heads * 8;
    const dim3 ag(m->n_heads, (unsigned)((R + ATT_QB - 1) / ATT_QB), (unsigned)nchunk);
    e = launch_pdl(attention_partial_kernel, ag, dim3(ATT_THREADS), ATT_SMEM, s, (const float*)QKV, (int64_t)3 * d,
                   (const float*)kc, (const float*)vc, (int64_t)d, ap, (int)R, (int)L, d, m->n_heads,
                   make_bounds({{QKV, (size_t)R * 3 * d * 4},
                                {kc, (size_t)L * d * 4},
                                {vc, (size_t)L * d * 4},
                                {ap.acc, att_bytes},
                                {ap.ml, ml_bytes}}));
    note_launch();
    const dim3 mg((unsigned)act_rows_padded(R), (unsigned)((d / QK + 7) / 8));
    if (e == cudaSuccess)
      e = launch_pdl(attn_merge_quant_kernel, mg, dim3(256), 0, s, ap, nchunk, (int)R, d, m->n_heads,
                     quant_out(actd, R, d), wprefetch(DLLM_Q4_K, Ly.wo, S.o),
                     make_bounds({{ap.acc, att_bytes}, {ap.ml, ml_bytes}}));
    note_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch attention");
    if ((rc = gemm(DLLM_Q4_K, actd, R, d, Ly.wo, d, Po, S.o, s))) return rc;
    if ((rc = run_row<ROW_RESID_NORM_QUANT>(xb, Po, S.o.splits, R * d, d, Ly.ffn_norm, m->eps, (int)R, d, actd, s)))
      return rc;
    if ((rc = gemm(DLLM_Q4_K, actd, R, d, Ly.wgu, 2 * f, Pgu, S.gu, s))) return rc;
    if ((rc = run_row<ROW_SWIGLU_QUANT>(nullptr, Pgu, S.gu.splits, R * 2 * f, 2 * f, nullptr, 0.f, (int)R, f, actf,
                                        s)))
      return rc;
    if ((rc = gemm(DLLM_Q6_K, actf, R, f, Ly.wdown, d, Pdn, S.dn, s))) return rc;
    if (li + 1 < m->n_layers) {
      if ((rc = run_row<ROW_RESID_NORM_QUANT>(xb, Pdn, S.dn.splits, R * d, d, m->layers[li + 1].attn_norm, m->eps,
                                              (int)R, d, actd, s)))
        return rc;
    } else {
      if ((rc = run_row<ROW_RESID_ONLY>(xb, Pdn, S.dn.splits, R * d, d, nullptr, 0.f, (int)R, d, nullptr, s)))
        return rc;
    }
  }
  return DLLM_OK;
}

}  // namespace dllm

using namespace dllm;

extern "C" {

DLLM_API size_t dllm_step_workspace_bytes(const dllm_model* m, int64_t L, int flags) {
  if (!m || L <= 0 || m->d_model <= 0 || m->d_ff <= 0) return 0;
  return step_plan(m, L, flags, false).bytes;
}

DLLM_API int dllm_step_linear_stream(const dllm_model* m, const int32_t* canvas, int64_t L, float* x, int flags,
                                     void* ws, size_t ws_bytes, dllm_stream_t stream) {
  return dllm_step_taps(m, canvas, L, x, flags, nullptr, ws, ws_bytes, stream);
}

DLLM_API int dllm_step_taps(const dllm_model* m, const int32_t* canvas, int64_t L, float* x, int flags,
                            const dllm_taps* taps, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  int rc = check_model(m, L, "dllm_step_linear_stream");
  if (rc) return rc;
  if (flags != DLLM_STREAM_LINEAR && flags != DLLM_STREAM_FULL)
    return fail(DLLM_E_INVAL, "dllm_step_linear_stream: flags must be DLLM_STREAM_LINEAR or DLLM_STREAM_FULL");
  if ((rc = check_device())) return rc;
  if (!device_ptr(x)) return fail(DLLM_E_INVAL, "dllm_step_linear_stream: x is NULL or not a device pointer");
  if (flags == DLLM_STREAM_FULL) {
    if (!device_ptr(canvas)) return fail(DLLM_E_INVAL, "dllm_step_linear_stream: canvas is NULL or not a device pointer");
    if (!device_ptr(m->tok_embd)) return fail(DLLM_E_INVAL, "dllm_step_linear_stream: model->tok_embd is not a device pointer");
  }
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0)
    return fail(DLLM_E_ALIGN, "dllm_step_linear_stream: x must be 16-byte aligned");
  const StepPlan S = step_plan(m, L, flags, false);
  if (!ws || ws_bytes < S.bytes || !device_ptr(ws))
    return fail(DLLM_E_WORKSPACE, "dllm_step_linear_stream: workspace has %zu bytes, needs %zu", ws ? ws_bytes : (size_t)0,
                S.bytes);
  if ((reinterpret_cast<uintptr_t>(ws) & 1023) != 0)
    return fail(DLLM_E_ALIGN, "dllm_step_linear_stream: ws must be 1024-byte aligned");
  if (taps) {
    if (taps->layer < 0 || taps->layer >= m->n_layers)
      return fail(DLLM_E_INVAL, "dllm_step_taps: taps->layer=%d is not a layer of the model", taps->layer);
    const void* ps[] = {taps->x_in, taps->act_attn, taps->q, taps->k, taps->v, taps->attn, taps->act_o,
                        taps->x_mid, taps->act_ffn, taps->h, taps->act_down, taps->x_out};
    for (const void* p : ps)
      if (p && !device_ptr(p)) return fail(DLLM_E_INVAL, "dllm_step_taps: a tap pointer is not a device pointer");
    const float* f4[] = {taps->attn, taps->h};
    for (const float* p : f4)
      if (p && (reinterpret_cast<uintptr_t>(p) & 15))
        return fail(DLLM_E_ALIGN, "dllm_step_taps: the attn and h taps must be 16-byte aligned");
    if (flags != DLLM_STREAM_FULL && (taps->q || taps->k || taps->v))
      return fail(DLLM_E_INVAL, "dllm_step_taps: the q, k, v taps need DLLM_STREAM_FULL");
  }
  return forward(m, canvas, L, x, flags, static_cast<uint8_t*>(ws), S, (cudaStream_t)stream, nullptr, taps);
}

DLLM_API size_t dllm_denoise_workspace_bytes(const dllm_model* m, int64_t L, int32_t block_rows) {
  if (!m || L <= 0 || block_rows <= 0 || m->d_model <= 0) return 0;
  const StepPlan S = step_plan(m, L, DLLM_STREAM_FULL, true);
  return align_up(S.bytes, 1024) + dllm_lmhead_workspace_bytes(block_rows, m->vocab, m->d_model);
}

DLLM_API int dllm_denoise_step(const dllm_model* m, int32_t* canvas, int64_t L, int32_t block_begin, int32_t block_end,
                               int32_t k_commit, int32_t* out_pos, int32_t* out_id, float* out_conf,
                               float* hidden_out, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  int rc = check_model(m, L, "dllm_denoise_step");
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  if (!device_ptr(canvas) || !device_ptr(m->tok_embd) || !device_ptr(m->w_out) || !device_ptr(m->out_norm))
    return fail(DLLM_E_INVAL, "dllm_denoise_step: canvas / tok_embd / w_out / out_norm must be device pointers");
  const StepPlan S = step_plan(m, L, DLLM_STREAM_FULL, true);
  const size_t need = dllm_denoise_workspace_bytes(m, L, block_end - block_begin);
  if (block_end - block_begin <= 0 || need == 0)
    return fail(DLLM_E_INVAL, "dllm_denoise_step: empty block [%d, %d)", block_begin, block_end);
  if (!ws || ws_bytes < need || !device_ptr(ws))
    return fail(DLLM_E_WORKSPACE, "dllm_denoise_step: workspace has %zu bytes, needs %zu", ws ? ws_bytes : (size_t)0,
                need);
  if ((reinterpret_cast<uintptr_t>(ws) & 1023) != 0)
    return fail(DLLM_E_ALIGN, "dllm_denoise_step: ws must be 1024-byte aligned");
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* x = hidden_out ? hidden_out : reinterpret_cast<float*>(base + S.x);
  if (hidden_out && !device_ptr(hidden_out))
    return fail(DLLM_E_INVAL, "dllm_denoise_step: hidden_out is not a device pointer");
  cudaStream_t s = (cudaStream_t)stream;
  if ((rc = forward(m, canvas, L, x, DLLM_STREAM_FULL, base, S, s))) return rc;
  const size_t lm_off = align_up(S.bytes, 1024);
  return dllm_lmhead_masked_select(x, L, m->d_model, m->d_model, m->out_norm, m->eps, m->w_out, m->vocab, canvas,
                                   m->mask_id, block_begin, block_end, k_commit, out_pos, out_id, out_conf, nullptr,
                                   nullptr, base + lm_off, ws_bytes - lm_off, stream);
}

DLLM_API size_t dllm_kv_cache_bytes(const dllm_model* m, int64_t L) {
  if (!m || L <= 0 || m->d_model <= 0 || m->n_layers <= 0) return 0;
  return (size_t)m->n_layers * 2 * (size_t)L * m->d_model * 4;
}

DLLM_API size_t dllm_denoise_cached_workspace_bytes(const dllm_model* m, int64_t L, int32_t block_rows) {
  if (!m || L <= 0 || block_rows <= 0 || block_rows > L || m->d_model <= 0 || m->d_ff <= 0) return 0;
  const StepPlan F = step_plan(m, L, DLLM_STREAM_FULL, true);
  const StepPlan B = step_plan(m, block_rows, DLLM_STREAM_FULL, true, L);
  return align_up(std::max(F.bytes, B.bytes), 1024) + dllm_lmhead_workspace_bytes(block_rows, m->vocab, m->d_model);
}

DLLM_API int dllm_denoise_step_cached(const dllm_model* m, int32_t* canvas, int64_t L, int32_t block_begin,
                                      int32_t block_end, int32_t k_commit, int32_t refresh, float* kv_cache,
                                      size_t kv_bytes, int32_t* out_pos, int32_t* out_id, float* out_conf,
                                      float* hidden_out, void* ws, size_t ws_bytes, dllm_stream_t stream) {
  DLLM_RANGE();
  int rc = check_model(m, L, "dllm_denoise_step_cached");
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  if (!device_ptr(canvas) || !device_ptr(m->tok_embd) || !device_ptr(m->w_out) || !device_ptr(m->out_norm))
    return fail(DLLM_E_INVAL, "dllm_denoise_step_cached: canvas / tok_embd / w_out / out_norm must be device pointers");
  if (refresh != 0 && refresh != 1) return fail(DLLM_E_INVAL, "dllm_denoise_step_cached: refresh must be 0 or 1");
  const int64_t R = (int64_t)block_end - block_begin;
  if (block_begin < 0 || block_end > L || R <= 0 || R > 160)
    return fail(DLLM_E_INVAL, "dllm_denoise_step_cached: block [%d, %d) must lie in [0, L=%lld) and hold 1..160 rows",
                block_begin, block_end, (long long)L);
  const size_t kv_need = dllm_kv_cache_bytes(m, L);
  if (!kv_cache || kv_bytes < kv_need || !device_ptr(kv_cache))
    return fail(DLLM_E_WORKSPACE, "dllm_denoise_step_cached: kv_cache has %zu bytes, needs %zu (dllm_kv_cache_bytes)",
                kv_cache ? kv_bytes : (size_t)0, kv_need);
  if ((reinterpret_cast<uintptr_t>(kv_cache) & 15) != 0)
    return fail(DLLM_E_ALIGN, "dllm_denoise_step_cached: kv_cache must be 16-byte aligned");
  const size_t need = dllm_denoise_cached_workspace_bytes(m, L, (int32_t)R);
  if (!ws || ws_bytes < need || !device_ptr(ws))
    return fail(DLLM_E_WORKSPACE, "dllm_denoise_step_cached: workspace has %zu bytes, needs %zu",
                ws ? ws_bytes : (size_t)0, need);
  if ((reinterpret_cast<uintptr_t>(ws) & 1023) != 0)
    return fail(DLLM_E_ALIGN, "dllm_denoise_step_cached: ws must be 1024-byte aligned");
  if (hidden_out && (!device_ptr(hidden_out) || (reinterpret_cast<uintptr_t>(hidden_out) & 15) != 0))
    return fail(DLLM_E_INVAL, "dllm_denoise_step_cached: hidden_out must be a 16-byte aligned device pointer");
  uint8_t* base = static_cast<uint8_t*>(ws);
  const StepPlan F = step_plan(m, L, DLLM_STREAM_FULL, true);
  const StepPlan B = step_plan(m, R, DLLM_STREAM_FULL, true, L);
  float* x = hidden_out ? hidden_out : reinterpret_cast<float*>(base + F.x);  // F.x == B.x == 0
  cudaStream_t s = (cudaStream_t)stream;
  if (refresh)
    rc = forward(m, canvas, L, x, DLLM_STREAM_FULL, base, F, s, kv_cache);
  else
    rc = forward_block(m, canvas, L, block_begin, R, x, kv_cache, base, B, s);
  if (rc) return rc;
  const size_t lm_off = align_up(std::max(F.bytes, B.bytes), 1024);
  return dllm_lmhead_masked_select(x, L, m->d_model, m->d_model, m->out_norm, m->eps, m->w_out, m->vocab, canvas,
                                   m->mask_id, block_begin, block_end, k_commit, out_pos, out_id, out_conf, nullptr,
                                   nullptr, base + lm_off, ws_bytes - lm_off, stream);
}

}  // extern "C"
