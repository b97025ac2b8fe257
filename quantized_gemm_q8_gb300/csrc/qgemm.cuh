// Quantized GEMM y = A(Q8_K activations) x W(Q4_K | Q6_K)^T on the sm_103a tensor cores.
//
// Method (mojo-dllm "Development plan", "Compute design"): activations are Q8_K (int8 codes,
// one f32 scale per 256, int sums per 16); each weight super-block is decoded to small
// integers plus a per-16 scale and per-16 offset; the integer inner product of a
// super-block runs to its end before the f32 scales apply. Here every such integer sum is
// computed EXACTLY by tcgen05.mma kind::f16: the small integers are carried in f16 operands
// (exactly representable) and accumulated in f32 tensor memory (exact below 2^24).
//
// Tile: 128 weight rows (MMA M = TMEM lanes) x NT tokens (MMA N). The weights are operand A
// and live in TENSOR MEMORY: decode threads (one per weight row = TMEM lane) turn the packed
// quants into f16 integers in registers and store them with tcgen05.st; the activations are
// operand B in shared memory (TMA, 128-byte swizzle). Keeping A out of shared memory halves
// the shared-memory traffic per MMA, which bounds an M=128, N<=160 tile otherwise.
//
// Per super-block sb two accumulator "parts" are produced into TMEM slots of NT columns:
//   Q4_K: part 0 = I = sum_k (scale_j * q4_k) * a_k           (16 MMAs, K = 256)
//         part 1 = J = sum_g min_{g/2} * bsum16_g               (1 MMA, K = 16, A from smem)
//         y += d_a * (d * I - dmin * J)
//   Q6_K: the int8 group scale s = 16 * s_hi + s_lo (s_lo in [0,15]) so that both products
//         s_hi * (q-32) and s_lo * (q-32) are exact f16 integers:
//         part 0 = I_hi = sum s_hi (q-32) a,  part 1 = I_lo = sum s_lo (q-32) a   (16+16 MMAs)
//         y += d_a * d * (16 * I_hi + I_lo)
// The epilogue folds part p as y += (c_p * P) * d_a with c = (d, -dmin) or (16 d, d); it
// drains a whole part into registers at once and frees the slot before the arithmetic.
//
// Warp roles (896 threads, 7 warpgroups): warps 0-15 epilogue (warp w reads TMEM lanes
// 32*(w%4).. and quarter w/4 of the NT columns), warps 16-23 decode (two threads per weight
// row = TMEM lane, one per half of each K-quarter), warp 24 producer (one thread issues bulk /
// tensor copies), warp 25 MMA issuer (one thread) + TMEM owner, warps 26-27 idle. setmaxnreg
// re-splits the 72-per-thread launch allocation: 88 epilogue, 56 decode, 40 control
// (512*88 + 256*56 + 128*40 = 896*72).
//
// Rings (mbarrier-synchronized, every wait bounded):
//   W  raw packed super-block of the 128 rows, smem (bulk copy)       producer -> decode
//   X  per-super-block extras, smem: d/dmin plane, d_a, J operands    producer,decode -> MMA,epi
//   B  activation quarter tile NT x 64 f16, smem, 128-byte swizzle    producer -> MMA
//   A  decoded weight quarter 128 x 64 f16 (Q6_K: hi and lo), TMEM    decode -> MMA
//   S  accumulator slots, TMEM                                        MMA -> epilogue
// K order inside each aligned group of 4 is (0,2,1,3) on both operands (the order in which
// the nibble-to-f16 trick below produces weights); the activation operand is stored that way.
#pragma once
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace dllm {

constexpr int QK = 256;
constexpr int BM = 128;
constexpr int TYPE_Q4K = 12;
constexpr int TYPE_Q6K = 14;
constexpr int Q4K_BLOB = 17920;  // 128 rows x (128 B quants + 12 B scales)
constexpr int Q6K_BLOB = 26624;  // 128 rows x (128 B ql + 64 B qh + 16 B scales)
constexpr int Q4K_DD = 512;      // 128 rows x (f16 d, f16 dmin)
constexpr int Q6K_DD = 256;      // 128 rows x f16 d
constexpr int QG_THREADS = 896;
constexpr int QG_EPI_WARPS = 16, QG_DEC_WARP0 = 16, QG_DEC_WARPS = 8, QG_PROD_WARP = 24, QG_MMA_WARP = 25;
constexpr int QG_REGS_LAUNCH = 72;  // 65536 / 896 rounded down to a multiple of 8
constexpr int QG_REGS_EPI = 88, QG_REGS_DEC = 56, QG_REGS_CTL = 40;
static_assert(512 * QG_REGS_EPI + 256 * QG_REGS_DEC + 128 * QG_REGS_CTL <= QG_THREADS * QG_REGS_LAUNCH,
              "register split");
constexpr int SMEM_LIMIT = 232448;
constexpr int TMEM_COLS = 512;

__host__ __device__ constexpr int al128(int x) { return (x + 127) & ~127; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int TYPE, int NT>
struct QCfg {
  static constexpr bool Q4 = TYPE == TYPE_Q4K;
  static constexpr int NC = NT / 4;  // columns per epilogue thread
  static constexpr int W_BYTES = Q4 ? Q4K_BLOB : Q6K_BLOB;
  static constexpr int DD_BYTES = Q4 ? Q4K_DD : Q6K_DD;
  // K-stage ring: one stage = QPS K-quarters (64 each) of both operands, 8 MMAs per stage:
  // Q4_K two quarters (one MMA chain), Q6_K one quarter (hi and lo chains).
  static constexpr int QPS = Q4 ? 2 : 1;
  static constexpr int SPS = 4 / QPS;  // stages per super-block
  // TMEM: accumulator slots, then the A operand of each stage (64 columns per stage)
  static constexpr int NSLOT = NT >= 128 ? 2 : 4;
  static constexpr int ACOL = NSLOT * NT;
  static constexpr int ASTG = 64;
  static constexpr int K_STAGES = cmin(6, (TMEM_COLS - ACOL) / ASTG);
  // shared memory
  static constexpr int X_STAGES = 3;
  static constexpr int X_DD = 0;
  static constexpr int X_DA = al128(DD_BYTES);
  static constexpr int X_BJ = X_DA + al128(NT * 4);
  static constexpr int X_AJ = X_BJ + (Q4 ? NT * 32 : 0);
  static constexpr int X_BYTES = al128(X_AJ + (Q4 ? 4096 : 0));
  static constexpr int X_TX = DD_BYTES + NT * 4 + (Q4 ? NT * 32 : 0);
  static constexpr int B_QUARTER = NT * 128;
  static constexpr int B_STAGE = QPS * B_QUARTER;
  static constexpr int SM_AVAIL = SMEM_LIMIT - 2048 - K_STAGES * B_STAGE - X_STAGES * X_BYTES;
  static constexpr int W_STAGES = cmin(6, SM_AVAIL / W_BYTES);
  static constexpr int OFF_B = 0;
  static constexpr int OFF_W = OFF_B + K_STAGES * B_STAGE;
  static constexpr int OFF_X = OFF_W + W_STAGES * W_BYTES;
  static constexpr int OFF_BAR = OFF_X + X_STAGES * X_BYTES;
  // barrier indices
  static constexpr int BK_FULL = 0, BK_EMPTY = BK_FULL + K_STAGES;
  static constexpr int BW_FULL = BK_EMPTY + K_STAGES, BW_EMPTY = BW_FULL + W_STAGES;
  static constexpr int BX_FULL = BW_EMPTY + W_STAGES, BX_EMPTY = BX_FULL + X_STAGES;
  static constexpr int BS_FULL = BX_EMPTY + X_STAGES, BS_EMPTY = BS_FULL + NSLOT;
  static constexpr int B_DONE = BS_EMPTY + NSLOT;
  static constexpr int NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
  static_assert(W_STAGES >= 2 && K_STAGES >= 2, "ring depth");
  static_assert(NT % 32 == 0 && NT >= 32 && NT <= 160, "token tile");
  static_assert(OFF_W % 16 == 0 && OFF_X % 128 == 0, "alignment");
};

struct QgemmParams {
  const uint8_t* wblob;  // packed blobs [tiles_n][nsb]
  const uint8_t* wdd;    // packed scale plane [tiles_n][nsb][128]
  const uint8_t* act_j;  // activation J plane
  const float* act_d;    // activation D plane
  int nsb, n, m, lpad;
  int tiles_n, tiles_m, splits, sbps, units;
  float* y;  // may be null (debug sums only)
  long long ldy, split_stride;
  int accumulate;
  int32_t* dbg;  // [2][nsb][m][n] or null
  int* err;      // device error word
  // mode 1 (LM head): instead of y, per (weight tile, TMEM lane quadrant, token) softmax
  // partials over the 32 weight rows of the quadrant: max logit, its row (lowest on ties),
  // and sum_rows exp(logit - max); layout [tiles_n * 4][m].
  int mode;
  float* pmax;
  int* parg;
  float* psum;
#ifdef DLLM_TRACE
  unsigned long long* trace;  // per-role clock64 stamps of CTA 0 (trace builds only)
#endif
  long long timeout;
};

#ifdef DLLM_TRACE
#define QTRACE(cond, slot, idx)                                                             \
  do {                                                                                      \
    if ((cond) && blockIdx.x == 0 && (idx) < 256) p.trace[(slot) * 256 + (idx)] = clock64(); \
  } while (0)
#else
#define QTRACE(cond, slot, idx) \
  do {                          \
  } while (0)
#endif

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t hfma2u(uint32_t v, __half2 m, __half2 a) {
  return h2u(__hfma2(u2h(v), m, a));
}

// Packed f32x2 arithmetic (sm_100+): d = a * b and d = a * b + d on register pairs.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n"
      " mul.rn.f32x2 rc, ra, rb;\n mov.b64 {%0,%1}, rc;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n mov.b64 rc, {%0,%1};\n"
      " fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0,%1}, rc;\n}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Q4_K: decode K-quarter q of row t (its 32 quant bytes: low nibbles = sub-block 2q, high
// nibbles = sub-block 2q+1) into 32 words = 64 f16 values scale*q4, in TMEM column order
// (word 4c + i = 16-byte chunk c, chunks 0-3 low nibbles, 4-7 high nibbles). The value is
// produced exactly: the nibble is OR-ed into the f16 pattern 0x6400 (= 1024 + q, or 1024 + 16q
// for a high nibble) and one fused multiply-add with (scale, -1024*scale) [or (scale/16,
// -64*scale)] returns scale*q (an integer <= 945). Inside a chunk the k order is
// (0,2,1,3, 4,6,5,7), the order in which the two nibble lanes of a 32-bit word come out.
__device__ __forceinline__ void decode_q4k_quarter(const uint8_t* W, int t, int q, __half2 mlo, __half2 alo,
                                                   __half2 mhi, __half2 ahi, uint32_t (&o)[2][16]) {
  const uint4 v0 = *reinterpret_cast<const uint4*>(W + (2 * q) * 2048 + t * 16);
  const uint4 v1 = *reinterpret_cast<const uint4*>(W + (2 * q + 1) * 2048 + t * 16);
  const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = x[2 * c], w1 = x[2 * c + 1];
    const uint32_t w0s = w0 >> 8, w1s = w1 >> 8;
    o[0][4 * c + 0] = hfma2u((w0 & 0x000F000Fu) | 0x64006400u, mlo, alo);
    o[0][4 * c + 1] = hfma2u((w0s & 0x000F000Fu) | 0x64006400u, mlo, alo);
    o[0][4 * c + 2] = hfma2u((w1 & 0x000F000Fu) | 0x64006400u, mlo, alo);
    o[0][4 * c + 3] = hfma2u((w1s & 0x000F000Fu) | 0x64006400u, mlo, alo);
    o[1][4 * c + 0] = hfma2u((w0 & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    o[1][4 * c + 1] = hfma2u((w0s & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    o[1][4 * c + 2] = hfma2u((w1 & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    o[1][4 * c + 3] = hfma2u((w1s & 0x00F000F0u) | 0x64006400u, mhi, ahi);
  }
}

// Q4_K, one half of a K-quarter: h = 0 the low nibbles (chunks 0-3), h = 1 the high nibbles
// (chunks 4-7) of the quarter's 32 quant bytes, as 16 words; (mul, add) as above for the
// half's sub-block.
__device__ __forceinline__ void decode_q4k_half(const uint8_t* W, int t, int q, int h, __half2 mul, __half2 add,
                                                uint32_t (&o)[16]) {
  const uint4 v0 = *reinterpret_cast<const uint4*>(W + (2 * q) * 2048 + t * 16);
  const uint4 v1 = *reinterpret_cast<const uint4*>(W + (2 * q + 1) * 2048 + t * 16);
  const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  const uint32_t mask = h ? 0x00F000F0u : 0x000F000Fu;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = x[2 * c], w1 = x[2 * c + 1];
    o[4 * c + 0] = hfma2u((w0 & mask) | 0x64006400u, mul, add);
    o[4 * c + 1] = hfma2u(((w0 >> 8) & mask) | 0x64006400u, mul, add);
    o[4 * c + 2] = hfma2u((w1 & mask) | 0x64006400u, mul, add);
    o[4 * c + 3] = hfma2u(((w1 >> 8) & mask) | 0x64006400u, mul, add);
  }
}

// Q6_K: decode half tt of K-quarter q (half-block hq = q/2, t-slot 2(q%2)+tt) of row t into
// 16 words of the hi operand (value s_hi*(q6-32)) and 16 words of the lo operand (value
// s_lo*(q6-32)); both exact f16 integers (the int8 group scale s = 16*s_hi + s_lo, s_lo in
// [0,15]). Even quarters take the low ql nibble and the f16 pattern 1024 + q6 (qh bits at 4-5),
// odd quarters the high nibble and 1024 + 16*q6 (qh bits at 8-9) with the scale divided by 16.
__device__ __forceinline__ void decode_q6k_half(const uint8_t* W, int t, int q, int tt, const int8_t* sc,
                                                uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  const int hq = q >> 1, odd = q & 1;
  uint32_t ql[8], qh[8];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(W + (4 * hq + 2 * tt + i) * 2048 + t * 16);
    ql[4 * i] = v.x;
    ql[4 * i + 1] = v.y;
    ql[4 * i + 2] = v.z;
    ql[4 * i + 3] = v.w;
    const uint4 u = *reinterpret_cast<const uint4*>(W + 16384 + (2 * hq + i) * 2048 + t * 16);
    qh[4 * i] = u.x;
    qh[4 * i + 1] = u.y;
    qh[4 * i + 2] = u.z;
    qh[4 * i + 3] = u.w;
  }
  const uint32_t nmask = odd ? 0x00F000F0u : 0x000F000Fu;
  const uint32_t hmask = odd ? 0x03000300u : 0x00300030u;
  const float fm = odd ? 0.0625f : 1.0f;
  const float fa = odd ? -96.0f : -1056.0f;
  const int tslot = 2 * odd + tt;
  const int shift = tt ? 2 : 4;
#pragma unroll
  for (int cp = 0; cp < 4; ++cp) {
    const int s = sc[8 * hq + 2 * tslot + (cp >> 1)];
    const int s_hi = s >> 4, s_lo = s & 15;
    const __half2 mH = __float2half2_rn((float)s_hi * fm), aH = __float2half2_rn((float)s_hi * fa);
    const __half2 mL = __float2half2_rn((float)s_lo * fm), aL = __float2half2_rn((float)s_lo * fa);
    const uint32_t X0 = ql[2 * cp], X1 = ql[2 * cp + 1];
    const uint32_t H0 = qh[2 * cp], H1 = qh[2 * cp + 1];
    const uint32_t v0 = (X0 & nmask) | ((H0 << shift) & hmask) | 0x64006400u;
    const uint32_t v1 = ((X0 >> 8) & nmask) | (((H0 >> 8) << shift) & hmask) | 0x64006400u;
    const uint32_t v2 = (X1 & nmask) | ((H1 << shift) & hmask) | 0x64006400u;
    const uint32_t v3 = ((X1 >> 8) & nmask) | (((H1 >> 8) << shift) & hmask) | 0x64006400u;
    hi[4 * cp + 0] = hfma2u(v0, mH, aH);
    hi[4 * cp + 1] = hfma2u(v1, mH, aH);
    hi[4 * cp + 2] = hfma2u(v2, mH, aH);
    hi[4 * cp + 3] = hfma2u(v3, mH, aH);
    lo[4 * cp + 0] = hfma2u(v0, mL, aL);
    lo[4 * cp + 1] = hfma2u(v1, mL, aL);
    lo[4 * cp + 2] = hfma2u(v2, mL, aL);
    lo[4 * cp + 3] = hfma2u(v3, mL, aL);
  }
}

__device__ __forceinline__ void unit_coords(const QgemmParams& p, int u, int& tn, int& tm, int& sp, int& sb0,
                                            int& sb1) {
  tn = u % p.tiles_n;
  const int r = u / p.tiles_n;
  tm = r % p.tiles_m;
  sp = r / p.tiles_m;
  sb0 = sp * p.sbps;
  sb1 = min(p.nsb, sb0 + p.sbps);
}

template <int TYPE, int NT>
__global__ void __launch_bounds__(QG_THREADS, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmap, const QgemmParams p) {
  using C = QCfg<TYPE, NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  auto BAR = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  const long long lim = p.timeout;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::K_STAGES; ++i) {
      mbar_init(BAR(C::BK_FULL + i), 1 + QG_DEC_WARPS);  // producer (with the B bytes) + decode warps
      mbar_init(BAR(C::BK_EMPTY + i), 1);
    }
    for (int i = 0; i < C::W_STAGES; ++i) {
      mbar_init(BAR(C::BW_FULL + i), 1);
      mbar_init(BAR(C::BW_EMPTY + i), QG_DEC_WARPS);
    }
    for (int i = 0; i < C::X_STAGES; ++i) {
      mbar_init(BAR(C::BX_FULL + i), C::Q4 ? 1 + QG_DEC_WARPS : 1);
      mbar_init(BAR(C::BX_EMPTY + i), C::Q4 ? QG_EPI_WARPS + 1 : QG_EPI_WARPS);
    }
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(BAR(C::BS_FULL + i), 1);
      mbar_init(BAR(C::BS_EMPTY + i), QG_EPI_WARPS);
    }
    mbar_init(BAR(C::B_DONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == QG_MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= QG_PROD_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_CTL));
    if (warp == QG_PROD_WARP && lane == 0) {
      // ---------------------------------------------------------- producer (one thread)
      prefetch_tensormap(&tmap);
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int tn, tm, sp, sb0, sb1;
        unit_coords(p, u, tn, tm, sp, sb0, sb1);
        const uint8_t* blob = p.wblob + (size_t)tn * p.nsb * C::W_BYTES;
        const uint8_t* dd = p.wdd + (size_t)tn * p.nsb * C::DD_BYTES;
        const int tok0 = tm * NT;
        for (int sb = sb0; sb < sb1; ++sb, ++it) {
          const int w = it % C::W_STAGES;
          if (!(ok = mbar_wait(BAR(C::BW_EMPTY + w), ((it / C::W_STAGES) & 1) ^ 1, abort_flag, lim))) break;
          mbar_expect_tx(BAR(C::BW_FULL + w), C::W_BYTES);
          bulk_g2s(sbase + C::OFF_W + w * C::W_BYTES, blob + (size_t)sb * C::W_BYTES, C::W_BYTES,
                   BAR(C::BW_FULL + w));
          QTRACE(true, 1, it);
          const int x = it % C::X_STAGES;
          if (!(ok = mbar_wait(BAR(C::BX_EMPTY + x), ((it / C::X_STAGES) & 1) ^ 1, abort_flag, lim))) break;
          const uint32_t xs = sbase + C::OFF_X + x * C::X_BYTES;
          mbar_expect_tx(BAR(C::BX_FULL + x), C::X_TX);
          bulk_g2s(xs + C::X_DD, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES, BAR(C::BX_FULL + x));
          bulk_g2s(xs + C::X_DA, p.act_d + (size_t)sb * p.lpad + tok0, NT * 4, BAR(C::BX_FULL + x));
          if (C::Q4)
            bulk_g2s(xs + C::X_BJ, p.act_j + ((size_t)sb * p.lpad + tok0) * 32, NT * 32, BAR(C::BX_FULL + x));
          for (int st = 0; st < C::SPS; ++st) {
            const int j = C::SPS * it + st, b = j % C::K_STAGES;
            if (!(ok = mbar_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim))) break;
            mbar_expect_tx(BAR(C::BK_FULL + b), C::B_STAGE);
#pragma unroll
            for (int qq = 0; qq < C::QPS; ++qq)
              tma_g2s_3d(sbase + C::OFF_B + b * C::B_STAGE + qq * C::B_QUARTER, &tmap, 0, tok0,
                         sb * 4 + st * C::QPS + qq, BAR(C::BK_FULL + b));
            QTRACE(true, 0, j);
          }
          if (!ok) break;
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        // copies already issued land within microseconds; hold the CTA (bounded, ~1 ms) so none
        // of them can write into shared memory after it exits
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
      }
    } else if (warp == QG_MMA_WARP && lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      constexpr uint32_t IDESC = idesc_f16(BM, NT);
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int tn, tm, sp, sb0, sb1;
        unit_coords(p, u, tn, tm, sp, sb0, sb1);
        for (int sb = sb0; sb < sb1; ++sb, ++it) {
          const int c0 = 2 * it, c1 = 2 * it + 1;
          const int s0 = c0 % C::NSLOT, s1 = c1 % C::NSLOT;
          if (!(ok = mbar_wait(BAR(C::BS_EMPTY + s0), ((c0 / C::NSLOT) & 1) ^ 1, abort_flag, lim))) break;
          tc_fence_after();
          for (int st = 0; st < C::SPS; ++st) {
            const int j = C::SPS * it + st, b = j % C::K_STAGES;
            if (!(ok = mbar_wait(BAR(C::BK_FULL + b), (j / C::K_STAGES) & 1, abort_flag, lim))) break;
            QTRACE(true, 2, j);
            tc_fence_after();
            const uint32_t acol = tmem + C::ACOL + b * C::ASTG;
            const uint32_t bst = sbase + C::OFF_B + b * C::B_STAGE;
#pragma unroll
            for (int qq = 0; qq < C::QPS; ++qq) {
              const int q = st * C::QPS + qq;
              const uint32_t baddr = bst + qq * C::B_QUARTER;
              const uint32_t aq = acol + qq * 32;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ts(tmem + s0 * NT, aq + kk * 8, desc_sw128(baddr + kk * 32), IDESC, (q | kk) != 0);
              if (q == 3) mma_commit(BAR(C::BS_FULL + s0));
              if (!C::Q4) {
                if (q == 0) {
                  if (!(ok = mbar_wait(BAR(C::BS_EMPTY + s1), ((c1 / C::NSLOT) & 1) ^ 1, abort_flag, lim))) break;
                  tc_fence_after();
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f16_ts(tmem + s1 * NT, aq + 32 + kk * 8, desc_sw128(baddr + kk * 32), IDESC, (q | kk) != 0);
                if (q == 3) mma_commit(BAR(C::BS_FULL + s1));
              }
            }
            if (!ok) break;
            mma_commit(BAR(C::BK_EMPTY + b));
          }
          if (!ok) break;
          if (C::Q4) {
            const int x = it % C::X_STAGES;
            if (!(ok = mbar_wait(BAR(C::BX_FULL + x), (it / C::X_STAGES) & 1, abort_flag, lim))) break;
            if (!(ok = mbar_wait(BAR(C::BS_EMPTY + s1), ((c1 / C::NSLOT) & 1) ^ 1, abort_flag, lim))) break;
            tc_fence_after();
            const uint32_t xs = sbase + C::OFF_X + x * C::X_BYTES;
            mma_f16(tmem + s1 * NT, desc_noswz(xs + C::X_AJ, 128, 256), desc_noswz(xs + C::X_BJ, 128, 256), IDESC,
                    0);
            mma_commit(BAR(C::BS_FULL + s1));
            mma_commit(BAR(C::BX_EMPTY + x));
          }
        }
      }
      if (!ok) atomicOr(p.err, ERR_TIMEOUT_MMA);
      // all issued MMAs complete before the tensor memory is released
      mma_commit(BAR(C::B_DONE));
      volatile int never = 0;
      mbar_wait(BAR(C::B_DONE), 0, &never, lim);
    }
  } else if (warp >= QG_DEC_WARP0) {
    // ------------------------------------------------------------ decode (thread = row = lane)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_DEC));
    const int d = threadIdx.x - 32 * QG_DEC_WARP0;
    const int t = d & 127, h = d >> 7;  // weight row (= TMEM lane, warp % 4 == t / 32), half
    const uint32_t tlane = tmem + ((uint32_t)(t & ~31) << 16) + C::ACOL;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      int tn, tm, sp, sb0, sb1;
      unit_coords(p, u, tn, tm, sp, sb0, sb1);
      for (int sb = sb0; sb < sb1; ++sb, ++it) {
        const int w = it % C::W_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::BW_FULL + w), (it / C::W_STAGES) & 1, abort_flag, lim));
        if (!ok) break;
        const uint8_t* W = smem + C::OFF_W + w * C::W_BYTES;
        if constexpr (C::Q4) {
          const uint32_t sw0 = *reinterpret_cast<const uint32_t*>(W + 16384 + t * 4);
          const uint32_t sw1 = *reinterpret_cast<const uint32_t*>(W + 16384 + 512 + t * 4);
          const uint32_t sw2 = *reinterpret_cast<const uint32_t*>(W + 16384 + 1024 + t * 4);
          // 6-bit fields: the bytes of *_lo4 are entries 0..3, of *_hi4 entries 4..7
          const uint32_t sc_lo4 = sw0 & 0x3F3F3F3Fu;
          const uint32_t mn_lo4 = sw1 & 0x3F3F3F3Fu;
          const uint32_t sc_hi4 = (sw2 & 0x0F0F0F0Fu) | ((sw0 >> 2) & 0x30303030u);
          const uint32_t mn_hi4 = ((sw2 >> 4) & 0x0F0F0F0Fu) | ((sw1 >> 2) & 0x30303030u);
          // J operand row t: (min_0, min_0, min_1, min_1, ..., min_7, min_7) in 8x16 B core
          // matrices (K-major, no swizzle), shared memory; half h writes core matrix h
          const int x = it % C::X_STAGES;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(BAR(C::BX_EMPTY + x), ((it / C::X_STAGES) & 1) ^ 1, abort_flag, lim));
          if (!ok) break;
          uint8_t* aj = smem + C::OFF_X + x * C::X_BYTES + C::X_AJ + (t >> 3) * 256 + (t & 7) * 16;
          {
            const uint32_t m4 = h ? mn_hi4 : mn_lo4;
            uint4 o;
            o.x = h2u(__float2half2_rn((float)(m4 & 0xFF)));
            o.y = h2u(__float2half2_rn((float)((m4 >> 8) & 0xFF)));
            o.z = h2u(__float2half2_rn((float)((m4 >> 16) & 0xFF)));
            o.w = h2u(__float2half2_rn((float)(m4 >> 24)));
            *reinterpret_cast<uint4*>(aj + h * 128) = o;
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::BX_FULL + x));
#pragma unroll 1
          for (int st = 0; st < 2; ++st) {
            // quarters 2st, 2st+1: sub-blocks 4st..4st+3, scales are the bytes of sc_lo4 / sc_hi4
            const uint32_t s4 = st ? sc_hi4 : sc_lo4;
            const int j = 2 * it + st, b = j % C::K_STAGES;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim));
            if (!ok) break;
            QTRACE(t == 0, 4, j);
            tc_fence_after();
            const uint32_t ta = tlane + b * C::ASTG;
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              // sub-block 2q + h of quarter q = 2st + qq
              const float sc = (float)((s4 >> (16 * qq + 8 * h)) & 0xFF);
              uint32_t o[16];
              decode_q4k_half(W, t, 2 * st + qq, h, __float2half2_rn(h ? sc * 0.0625f : sc),
                              __float2half2_rn(h ? -64.f * sc : -1024.f * sc), o);
              tmem_st16(ta + 32 * qq + 16 * h, o);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::BK_FULL + b));
            QTRACE(t == 0, 5, j);
          }
        } else {
          const uint4 scv = *reinterpret_cast<const uint4*>(W + 24576 + t * 16);
          const int8_t* sc = reinterpret_cast<const int8_t*>(&scv);
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            const int j = 4 * it + q, b = j % C::K_STAGES;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim));
            if (!ok) break;
            QTRACE(t == 0, 4, j);
            tc_fence_after();
            {
              uint32_t hi[16], lo[16];
              decode_q6k_half(W, t, q, h, sc, hi, lo);
              tmem_st16(tlane + b * C::ASTG + 16 * h, hi);
              tmem_st16(tlane + b * C::ASTG + 32 + 16 * h, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::BK_FULL + b));
            QTRACE(t == 0, 5, j);
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BW_EMPTY + w));
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, ERR_TIMEOUT_DECODE);
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-15)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_EPI));
    constexpr int NC = C::NC;
    constexpr int NCH = NC / 8;
    const int qd = warp & 3, hf = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t tlane = tmem + ((uint32_t)(32 * qd) << 16) + hf * NC;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      int tn, tm, sp, sb0, sb1;
      unit_coords(p, u, tn, tm, sp, sb0, sb1);
      const int grow = tn * BM + row;
      const int tokb = tm * NT + hf * NC;
      float acc[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) acc[i] = 0.f;
      for (int sb = sb0; sb < sb1; ++sb, ++it) {
        const int x = it % C::X_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::BX_FULL + x), (it / C::X_STAGES) & 1, abort_flag, lim));
        if (!ok) break;
        const uint8_t* X = smem + C::OFF_X + x * C::X_BYTES;
        float cf[2];
        if constexpr (C::Q4) {
          const __half2 dd = *reinterpret_cast<const __half2*>(X + C::X_DD + row * 4);
          cf[0] = __low2float(dd);
          cf[1] = -__high2float(dd);
        } else {
          const float dv = __half2float(*reinterpret_cast<const __half*>(X + C::X_DD + row * 2));
          cf[0] = 16.f * dv;
          cf[1] = dv;
        }
        const float4* da4 = reinterpret_cast<const float4*>(X + C::X_DA) + hf * (NC / 4);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int cnt = 2 * it + part, s = cnt % C::NSLOT;
          ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::BS_FULL + s), (cnt / C::NSLOT) & 1, abort_flag, lim));
          if (!ok) break;
          tc_fence_after();
          QTRACE(warp == 0 && lane == 0, 6, cnt);
          // drain the part in groups of up to 3 x 8 columns; the slot is freed as soon as the
          // last group is in registers, before its arithmetic
          const float cp = cf[part];
          constexpr int G = 3;
#pragma unroll
          for (int g0 = 0; g0 < NCH; g0 += G) {
            uint32_t r[G][8];
#pragma unroll
            for (int c = 0; c < G; ++c)
              if (g0 + c < NCH) tmem_ld8(tlane + s * NT + (g0 + c) * 8, r[c]);
            tmem_ld_wait();
            if (g0 + G >= NCH) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(BAR(C::BS_EMPTY + s));
              QTRACE(warp == 0 && lane == 0, 7, cnt);
            }
#pragma unroll
            for (int c = 0; c < G; ++c) {
              if (g0 + c >= NCH) break;
              const int ch = g0 + c;
#pragma unroll
              for (int j4 = 0; j4 < 2; ++j4) {
                const float4 dv = da4[ch * 2 + j4];
                const int b = ch * 8 + 4 * j4;
                float t0, t1, t2, t3;
                fmul2(t0, t1, __uint_as_float(r[c][4 * j4]), __uint_as_float(r[c][4 * j4 + 1]), cp, cp);
                fmul2(t2, t3, __uint_as_float(r[c][4 * j4 + 2]), __uint_as_float(r[c][4 * j4 + 3]), cp, cp);
                ffma2(acc[b], acc[b + 1], t0, t1, dv.x, dv.y);
                ffma2(acc[b + 2], acc[b + 3], t2, t3, dv.z, dv.w);
              }
              if (p.dbg != nullptr && grow < p.n) {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                  const int tok = tokb + ch * 8 + jj;
                  if (tok < p.m)
                    p.dbg[(((size_t)part * p.nsb + sb) * p.m + tok) * p.n + grow] = (int32_t)__uint_as_float(r[c][jj]);
                }
              }
            }
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BX_EMPTY + x));
      }
      if (!ok) break;
      if (p.mode == 1) {
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          float v = grow < p.n ? acc[j] : -INFINITY;
          int idx = grow;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, off);
            const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
            if (ov > v || (ov == v && oi < idx)) {
              v = ov;
              idx = oi;
            }
          }
          float e = grow < p.n ? expf(acc[j] - v) : 0.f;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
          const int tok = tokb + j;
          if (lane == 0 && tok < p.m) {
            const size_t o = ((size_t)tn * 4 + qd) * p.m + tok;
            p.pmax[o] = v;
            p.parg[o] = idx;
            p.psum[o] = e;
          }
        }
      } else if (p.y != nullptr && grow < p.n) {
        float* dst = p.y + (size_t)sp * p.split_stride + grow;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int tok = tokb + j;
          if (tok < p.m) {
            float* o = dst + (size_t)tok * p.ldy;
            *o = p.accumulate ? *o + acc[j] : acc[j];
          }
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, ERR_TIMEOUT_EPILOGUE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == QG_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace dllm
