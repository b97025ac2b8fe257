// Quantized GEMM y = A(Q8_K activations) x W(Q4_K | Q6_K)^T on the sm_103a tensor cores.
//
// Method (mojo-dllm "Development plan", "Compute design"): activations are Q8_K (int8 codes,
// one f32 scale per 256, int sums per 16); each weight super-block is decoded to small
// integers plus a per-16 scale and per-16 offset; the integer inner product of a
// super-block runs to its end before the f32 scales apply. Here every such integer sum is
// computed EXACTLY by tcgen05.mma kind::f16: the small integers are carried in f16 operands
// (exactly representable) and accumulated in f32 tensor memory (exact below 2^24).
//
// Tile: 128 weight rows (MMA M, = TMEM lanes) x NT tokens (MMA N), "swap-AB": the weight tile
// is operand A so each epilogue thread owns one output feature and its scalars.
//
// Per super-block sb two accumulator "parts" are produced, each into one TMEM slot of NT
// columns (slot ring of NSLOT):
//   Q4_K: part 0 = I = sum_k (scale_j * q4_k) * a_k           (16 MMAs, K = 256)
//         part 1 = J = sum_g min_{g/2} * bsum16_g               (1 MMA, K = 16)
//         y += d_a * (d * I - dmin * J)
//   Q6_K: the int8 group scale s = 16 * s_hi + s_lo (s_lo in [0,15]) so that both products
//         s_hi * (q-32) and s_lo * (q-32) are exact f16 integers:
//         part 0 = I_hi = sum s_hi (q-32) a,  part 1 = I_lo = sum s_lo (q-32) a   (16+16 MMAs)
//         y += d_a * d * (16 * I_hi + I_lo)
// The epilogue folds part p as y += (c_p * P) * d_a with c = (d, -dmin) or (16 d, d).
//
// Warp roles (448 threads): warps 0-7 epilogue (warp w reads TMEM lanes 32*(w%4).. and half
// w/4 of the NT columns), warps 8-11 decode (thread = weight row), warp 12 producer (one
// thread issues bulk / tensor copies), warp 13 MMA issuer (one thread) + TMEM owner.
//
// Shared-memory rings (all mbarrier-synchronized, every wait bounded):
//   W  raw packed super-block of the 128 rows (bulk copy)            producer -> decode
//   X  per-super-block extras: d/dmin plane, d_a, J operands          producer,decode -> MMA,epi
//   B  activation quarter tile NT x 64 f16, 128-byte swizzle (TMA)    producer -> MMA
//   A  decoded weight quarter tile 128 x 64 f16, 128-byte swizzle    decode -> MMA
// K-order inside each aligned group of 4 is (0,2,1,3) on both operands (the order in which
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
constexpr int QG_THREADS = 448;
constexpr int SMEM_LIMIT = 232448;

__host__ __device__ constexpr int al128(int x) { return (x + 127) & ~127; }

template <int TYPE, int NT>
struct QCfg {
  static constexpr bool Q4 = TYPE == TYPE_Q4K;
  static constexpr int NC = NT / 2;  // columns per epilogue thread
  static constexpr int W_BYTES = Q4 ? Q4K_BLOB : Q6K_BLOB;
  static constexpr int DD_BYTES = Q4 ? Q4K_DD : Q6K_DD;
  static constexpr int B_STAGE = NT * 128;
  static constexpr int A_STAGE = Q4 ? 16384 : 32768;
  static constexpr int NSLOT = NT > 128 ? 3 : 4;
  static constexpr int TMEM_COLS = NSLOT * NT <= 128 ? 128 : (NSLOT * NT <= 256 ? 256 : 512);
  static constexpr int B_STAGES = 4;
  static constexpr int A_STAGES = Q4 ? 4 : (NT <= 32 ? 3 : 2);
  static constexpr int W_STAGES = NT <= 64 ? 4 : 2;
  static constexpr int X_STAGES = 3;
  static constexpr int X_DD = 0;
  static constexpr int X_DA = al128(DD_BYTES);
  static constexpr int X_BJ = X_DA + al128(NT * 4);
  static constexpr int X_AJ = X_BJ + (Q4 ? NT * 32 : 0);
  static constexpr int X_BYTES = al128(X_AJ + (Q4 ? 4096 : 0));
  static constexpr int X_TX = DD_BYTES + NT * 4 + (Q4 ? NT * 32 : 0);
  static constexpr int OFF_B = 0;
  static constexpr int OFF_A = OFF_B + B_STAGES * B_STAGE;
  static constexpr int OFF_W = OFF_A + A_STAGES * A_STAGE;
  static constexpr int OFF_X = OFF_W + W_STAGES * W_BYTES;
  static constexpr int OFF_BAR = OFF_X + X_STAGES * X_BYTES;
  // barrier indices
  static constexpr int BB_FULL = 0, BB_EMPTY = BB_FULL + B_STAGES;
  static constexpr int BA_FULL = BB_EMPTY + B_STAGES, BA_EMPTY = BA_FULL + A_STAGES;
  static constexpr int BW_FULL = BA_EMPTY + A_STAGES, BW_EMPTY = BW_FULL + W_STAGES;
  static constexpr int BX_FULL = BW_EMPTY + W_STAGES, BX_EMPTY = BX_FULL + X_STAGES;
  static constexpr int BS_FULL = BX_EMPTY + X_STAGES, BS_EMPTY = BS_FULL + NSLOT;
  static constexpr int B_DONE = BS_EMPTY + NSLOT;
  static constexpr int NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
  static_assert(NT % 32 == 0 && NT >= 32 && NT <= 160, "token tile");
  static_assert(OFF_A % 1024 == 0 && OFF_W % 16 == 0 && OFF_X % 128 == 0, "alignment");
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
  long long timeout;
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t hfma2u(uint32_t v, __half2 m, __half2 a) {
  return h2u(__hfma2(u2h(v), m, a));
}

// Q4_K: decode K-quarter q (sub-blocks 2q [low nibbles] and 2q+1 [high nibbles]) of row t
// into the 128-byte swizzled row t of the A tile, weight value scale*q4 as exact f16.
// (1024 + q) is formed by OR-ing a nibble into the f16 pattern 0x6400; for the high nibble
// the pattern holds 1024 + 16q and the scale is divided by 16. One fused multiply-add then
// gives scale*q exactly (the exact result is an integer <= 945).
__device__ __forceinline__ void decode_q4k_quarter(const uint8_t* W, int t, int q, int sc_lo, int sc_hi,
                                                   uint8_t* Arow) {
  const uint4 v0 = *reinterpret_cast<const uint4*>(W + (2 * q) * 2048 + t * 16);
  const uint4 v1 = *reinterpret_cast<const uint4*>(W + (2 * q + 1) * 2048 + t * 16);
  const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  const __half2 mlo = __float2half2_rn((float)sc_lo), alo = __float2half2_rn(-1024.f * (float)sc_lo);
  const __half2 mhi = __float2half2_rn((float)sc_hi * 0.0625f), ahi = __float2half2_rn(-64.f * (float)sc_hi);
  const int sw = t & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = x[2 * c], w1 = x[2 * c + 1];
    const uint32_t w0s = w0 >> 8, w1s = w1 >> 8;
    uint4 lo, hi;
    lo.x = hfma2u((w0 & 0x000F000Fu) | 0x64006400u, mlo, alo);
    lo.y = hfma2u((w0s & 0x000F000Fu) | 0x64006400u, mlo, alo);
    lo.z = hfma2u((w1 & 0x000F000Fu) | 0x64006400u, mlo, alo);
    lo.w = hfma2u((w1s & 0x000F000Fu) | 0x64006400u, mlo, alo);
    hi.x = hfma2u((w0 & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    hi.y = hfma2u((w0s & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    hi.z = hfma2u((w1 & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    hi.w = hfma2u((w1s & 0x00F000F0u) | 0x64006400u, mhi, ahi);
    *reinterpret_cast<uint4*>(Arow + ((c ^ sw) << 4)) = lo;
    *reinterpret_cast<uint4*>(Arow + (((c + 4) ^ sw) << 4)) = hi;
  }
}

// Q6_K: decode K-quarter q (half h = q/2, t-slots 2(q%2), 2(q%2)+1) of row t into the hi
// tile (value s_hi*(q6-32)) and the lo tile (value s_lo*(q6-32)), both exact f16 integers.
// Even quarters use the low ql nibble and the f16 pattern 1024 + q6 (qh bits at 4-5);
// odd quarters the high nibble and 1024 + 16*q6 (qh bits at 8-9) with the scale / 16.
__device__ __forceinline__ void decode_q6k_quarter(const uint8_t* W, int t, int q, const int8_t* sc,
                                                   uint8_t* Ahi, uint8_t* Alo) {
  const int h = q >> 1, odd = q & 1;
  uint32_t ql[16], qh[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(W + (4 * h + i) * 2048 + t * 16);
    ql[4 * i] = v.x;
    ql[4 * i + 1] = v.y;
    ql[4 * i + 2] = v.z;
    ql[4 * i + 3] = v.w;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(W + 16384 + (2 * h + i) * 2048 + t * 16);
    qh[4 * i] = v.x;
    qh[4 * i + 1] = v.y;
    qh[4 * i + 2] = v.z;
    qh[4 * i + 3] = v.w;
  }
  const uint32_t nmask = odd ? 0x00F000F0u : 0x000F000Fu;
  const uint32_t hmask = odd ? 0x03000300u : 0x00300030u;
  const float fm = odd ? 0.0625f : 1.0f;
  const float fa = odd ? -96.0f : -1056.0f;
  const int sw = t & 7;
#pragma unroll
  for (int tt = 0; tt < 2; ++tt) {
    const int tslot = 2 * odd + tt;
    const int shift = tt ? 2 : 4;
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) {
      const int c = 4 * tt + cp;
      const int s = sc[8 * h + 2 * tslot + (cp >> 1)];
      const int s_hi = s >> 4, s_lo = s & 15;
      const __half2 mH = __float2half2_rn((float)s_hi * fm), aH = __float2half2_rn((float)s_hi * fa);
      const __half2 mL = __float2half2_rn((float)s_lo * fm), aL = __float2half2_rn((float)s_lo * fa);
      const uint32_t X0 = ql[8 * tt + 2 * cp], X1 = ql[8 * tt + 2 * cp + 1];
      const uint32_t H0 = qh[2 * cp], H1 = qh[2 * cp + 1];
      const uint32_t v0 = (X0 & nmask) | ((H0 << shift) & hmask) | 0x64006400u;
      const uint32_t v1 = ((X0 >> 8) & nmask) | (((H0 >> 8) << shift) & hmask) | 0x64006400u;
      const uint32_t v2 = (X1 & nmask) | ((H1 << shift) & hmask) | 0x64006400u;
      const uint32_t v3 = ((X1 >> 8) & nmask) | (((H1 >> 8) << shift) & hmask) | 0x64006400u;
      uint4 oh, ol;
      oh.x = hfma2u(v0, mH, aH);
      oh.y = hfma2u(v1, mH, aH);
      oh.z = hfma2u(v2, mH, aH);
      oh.w = hfma2u(v3, mH, aH);
      ol.x = hfma2u(v0, mL, aL);
      ol.y = hfma2u(v1, mL, aL);
      ol.z = hfma2u(v2, mL, aL);
      ol.w = hfma2u(v3, mL, aL);
      *reinterpret_cast<uint4*>(Ahi + ((c ^ sw) << 4)) = oh;
      *reinterpret_cast<uint4*>(Alo + ((c ^ sw) << 4)) = ol;
    }
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
    for (int i = 0; i < C::B_STAGES; ++i) {
      mbar_init(BAR(C::BB_FULL + i), 1);
      mbar_init(BAR(C::BB_EMPTY + i), 1);
    }
    for (int i = 0; i < C::A_STAGES; ++i) {
      mbar_init(BAR(C::BA_FULL + i), 4);
      mbar_init(BAR(C::BA_EMPTY + i), 1);
    }
    for (int i = 0; i < C::W_STAGES; ++i) {
      mbar_init(BAR(C::BW_FULL + i), 1);
      mbar_init(BAR(C::BW_EMPTY + i), 4);
    }
    for (int i = 0; i < C::X_STAGES; ++i) {
      mbar_init(BAR(C::BX_FULL + i), C::Q4 ? 5 : 1);
      mbar_init(BAR(C::BX_EMPTY + i), C::Q4 ? 9 : 8);
    }
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(BAR(C::BS_FULL + i), 1);
      mbar_init(BAR(C::BS_EMPTY + i), 8);
    }
    mbar_init(BAR(C::B_DONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------------ producer (one thread)
    if (lane == 0) {
      prefetch_tensormap(&tmap);
      int it = 0;
      int armed_b = 0, armed_w = 0, armed_x = 0;
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
          armed_w = it + 1;
          const int x = it % C::X_STAGES;
          if (!(ok = mbar_wait(BAR(C::BX_EMPTY + x), ((it / C::X_STAGES) & 1) ^ 1, abort_flag, lim))) break;
          const uint32_t xs = sbase + C::OFF_X + x * C::X_BYTES;
          mbar_expect_tx(BAR(C::BX_FULL + x), C::X_TX);
          bulk_g2s(xs + C::X_DD, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES, BAR(C::BX_FULL + x));
          bulk_g2s(xs + C::X_DA, p.act_d + (size_t)sb * p.lpad + tok0, NT * 4, BAR(C::BX_FULL + x));
          if (C::Q4)
            bulk_g2s(xs + C::X_BJ, p.act_j + ((size_t)sb * p.lpad + tok0) * 32, NT * 32, BAR(C::BX_FULL + x));
          armed_x = it + 1;
          for (int q = 0; q < 4; ++q) {
            const int j = 4 * it + q, b = j % C::B_STAGES;
            if (!(ok = mbar_wait(BAR(C::BB_EMPTY + b), ((j / C::B_STAGES) & 1) ^ 1, abort_flag, lim))) break;
            mbar_expect_tx(BAR(C::BB_FULL + b), C::B_STAGE);
            tma_g2s_3d(sbase + C::OFF_B + b * C::B_STAGE, &tmap, 0, tok0, sb * 4 + q, BAR(C::BB_FULL + b));
            armed_b = j + 1;
          }
          if (!ok) break;
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        // drain copies still in flight into this CTA's shared memory (bounded)
        volatile int never = 0;
        for (int j = max(0, armed_b - C::B_STAGES); j < armed_b; ++j)
          mbar_wait(BAR(C::BB_FULL + j % C::B_STAGES), (j / C::B_STAGES) & 1, &never, lim);
        for (int j = max(0, armed_w - C::W_STAGES); j < armed_w; ++j)
          mbar_wait(BAR(C::BW_FULL + j % C::W_STAGES), (j / C::W_STAGES) & 1, &never, lim);
        for (int j = max(0, armed_x - C::X_STAGES); j < armed_x; ++j)
          mbar_wait(BAR(C::BX_FULL + j % C::X_STAGES), (j / C::X_STAGES) & 1, &never, lim);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
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
          for (int q = 0; q < 4; ++q) {
            const int j = 4 * it + q, a = j % C::A_STAGES, b = j % C::B_STAGES;
            if (!(ok = mbar_wait(BAR(C::BA_FULL + a), (j / C::A_STAGES) & 1, abort_flag, lim))) break;
            if (!(ok = mbar_wait(BAR(C::BB_FULL + b), (j / C::B_STAGES) & 1, abort_flag, lim))) break;
            tc_fence_after();
            const uint32_t aaddr = sbase + C::OFF_A + a * C::A_STAGE;
            const uint32_t baddr = sbase + C::OFF_B + b * C::B_STAGE;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(tmem + s0 * NT, desc_sw128(aaddr + kk * 32), desc_sw128(baddr + kk * 32), IDESC,
                      (q | kk) != 0);
            if (q == 3) mma_commit(BAR(C::BS_FULL + s0));
            if (!C::Q4) {
              if (q == 0) {
                if (!(ok = mbar_wait(BAR(C::BS_EMPTY + s1), ((c1 / C::NSLOT) & 1) ^ 1, abort_flag, lim))) break;
                tc_fence_after();
              }
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16(tmem + s1 * NT, desc_sw128(aaddr + 16384 + kk * 32), desc_sw128(baddr + kk * 32), IDESC,
                        (q | kk) != 0);
              if (q == 3) mma_commit(BAR(C::BS_FULL + s1));
            }
            mma_commit(BAR(C::BA_EMPTY + a));
            mma_commit(BAR(C::BB_EMPTY + b));
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
  } else if (warp >= 8) {
    // ------------------------------------------------------------ decode (thread = row)
    const int t = threadIdx.x - 256;
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
          // 6-bit fields: bytes of sc_lo4 = scale 0..3, sc_hi4 = scale 4..7 (same for mins)
          const uint32_t sc_lo4 = sw0 & 0x3F3F3F3Fu;
          const uint32_t mn_lo4 = sw1 & 0x3F3F3F3Fu;
          const uint32_t sc_hi4 = (sw2 & 0x0F0F0F0Fu) | ((sw0 >> 2) & 0x30303030u);
          const uint32_t mn_hi4 = ((sw2 >> 4) & 0x0F0F0F0Fu) | ((sw1 >> 2) & 0x30303030u);
          // J operand row t: (min_0, min_0, min_1, min_1, ..., min_7, min_7) in 8x16 B core matrices
          const int x = it % C::X_STAGES;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(BAR(C::BX_EMPTY + x), ((it / C::X_STAGES) & 1) ^ 1, abort_flag, lim));
          if (!ok) break;
          uint8_t* aj = smem + C::OFF_X + x * C::X_BYTES + C::X_AJ + (t >> 3) * 256 + (t & 7) * 16;
#pragma unroll
          for (int ki = 0; ki < 2; ++ki) {
            const uint32_t m4 = ki ? mn_hi4 : mn_lo4;
            uint4 o;
            o.x = h2u(__float2half2_rn((float)(m4 & 0xFF)));
            o.y = h2u(__float2half2_rn((float)((m4 >> 8) & 0xFF)));
            o.z = h2u(__float2half2_rn((float)((m4 >> 16) & 0xFF)));
            o.w = h2u(__float2half2_rn((float)(m4 >> 24)));
            *reinterpret_cast<uint4*>(aj + ki * 128) = o;
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::BX_FULL + x));
          for (int q = 0; q < 4; ++q) {
            const int j = 4 * it + q, a = j % C::A_STAGES;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(BAR(C::BA_EMPTY + a), ((j / C::A_STAGES) & 1) ^ 1, abort_flag, lim));
            if (!ok) break;
            const uint32_t s4 = q < 2 ? sc_lo4 : sc_hi4;
            const int sh = (q & 1) * 16;
            decode_q4k_quarter(W, t, q, (s4 >> sh) & 0xFF, (s4 >> (sh + 8)) & 0xFF,
                               smem + C::OFF_A + a * C::A_STAGE + t * 128);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::BA_FULL + a));
          }
        } else {
          const uint4 scv = *reinterpret_cast<const uint4*>(W + 24576 + t * 16);
          const int8_t* sc = reinterpret_cast<const int8_t*>(&scv);
          for (int q = 0; q < 4; ++q) {
            const int j = 4 * it + q, a = j % C::A_STAGES;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(BAR(C::BA_EMPTY + a), ((j / C::A_STAGES) & 1) ^ 1, abort_flag, lim));
            if (!ok) break;
            uint8_t* At = smem + C::OFF_A + a * C::A_STAGE + t * 128;
            decode_q6k_quarter(W, t, q, sc, At, At + 16384);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::BA_FULL + a));
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BW_EMPTY + w));
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, ERR_TIMEOUT_DECODE);
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
    constexpr int NC = C::NC;
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
          const float cp = cf[part];
#pragma unroll
          for (int ch = 0; ch < NC / 16; ++ch) {
            uint32_t r[16];
            tmem_ld16(tlane + s * NT + ch * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 dv = da4[ch * 4 + j4];
              acc[ch * 16 + 4 * j4 + 0] = fmaf(__uint_as_float(r[4 * j4 + 0]) * cp, dv.x, acc[ch * 16 + 4 * j4 + 0]);
              acc[ch * 16 + 4 * j4 + 1] = fmaf(__uint_as_float(r[4 * j4 + 1]) * cp, dv.y, acc[ch * 16 + 4 * j4 + 1]);
              acc[ch * 16 + 4 * j4 + 2] = fmaf(__uint_as_float(r[4 * j4 + 2]) * cp, dv.z, acc[ch * 16 + 4 * j4 + 2]);
              acc[ch * 16 + 4 * j4 + 3] = fmaf(__uint_as_float(r[4 * j4 + 3]) * cp, dv.w, acc[ch * 16 + 4 * j4 + 3]);
            }
            if (p.dbg != nullptr && grow < p.n) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const int tok = tokb + ch * 16 + jj;
                if (tok < p.m)
                  p.dbg[(((size_t)part * p.nsb + sb) * p.m + tok) * p.n + grow] = (int32_t)__uint_as_float(r[jj]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::BS_EMPTY + s));
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BX_EMPTY + x));
      }
      if (!ok) break;
      if (p.y != nullptr && grow < p.n) {
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
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace dllm
