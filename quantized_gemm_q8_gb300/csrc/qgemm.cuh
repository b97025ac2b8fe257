// Quantized GEMM y = A(Q8_K activations) x W(Q4_K | Q6_K)^T on the sm_103a tensor cores.
//
// Method (mojo-dllm "Development plan", "Compute design"): the activations are Q8_K (8-bit
// codes, an f32 scale for every 256 and the integer sum of every 16); every weight
// super-block expands to small integers with a scale and an offset for each 16; within a
// super-block the integer products are summed completely before the f32 scales apply. Here every such integer sum is
// computed EXACTLY by tcgen05.mma kind::f16: the small integers are carried in f16 operands
// (exactly representable) and accumulated in f32 tensor memory (exact below 2^24).
//
// Tile: 128 weight rows (MMA M = TMEM lanes) x NT tokens (MMA N). The weights are operand A
// and live in TENSOR MEMORY: decode threads (one per weight row = TMEM lane) turn the packed
// quants into f16 integers in registers and store them with tcgen05.st; the activations are
// operand B in shared memory (TMA, 128-byte swizzle). Keeping A out of shared memory halves
// the shared-memory traffic per MMA, which bounds an M=128, N<=160 tile otherwise.
//
// Per super-block ONE accumulator part D is produced, in TMEM slot t & 1 (two slots of NT
// columns: the epilogue drains super-block t while the tensor core fills t + 1):
//   Q4_K: D = 2^-k * I' + sum_g c_g * bsum16_g,   I' = sum_k (scale_j * (q4_k - 8)) * a_k,
//         c_g = (8 * scale_{g/2} - min_{g/2} * (dmin / d)) * 2^-k,   y += d_a * (d * 2^k) * D
//         so that D = 2^-k (I - (dmin / d) J) with I = sum scale * q4 * a, J = sum min * bsum.
//         The 16 MMAs of I' read A = scale * (q4 - 8) * 2^-k from tensor memory (exact f16
//         values); the re-centred quants keep every partial sum of that integer chain within
//         63 * 8 * 127 * 256 < 2^24, so it is exact for every input. The offset and min term are
//         two more K = 16 MMAs from shared memory whose A operands are the f16 head and tail of
//         c_g (their sum carries c_g to 2^-22 relative) against the exact f16 activation
//         16-sums. k >= 0 is the smallest shift keeping 63 * |dmin / d| * 2^-k below 2^14 (k = 0
//         for any realistic block). A row with d = 0 uses D = -sum min * bsum and
//         y += d_a * dmin * D.
//   Q6_K: the int8 group scale s = 16 * s_hi + s_lo (s_lo in [0,15]); per K-quarter 4 MMAs
//         with A = s_hi * (q-32) (exact f16 integers) and 4 with A = s_lo * (q-32) / 16 (exact
//         f16 multiples of 1/16) accumulate D = sum s (q-32) a / 16;  y += d_a * (16 d) * D.
// Integer sums are exact while every partial sum stays below 2^24 in magnitude: always for
// Q4_K's I' chain, Q6_K's separate hi and lo sums and the debug parts below; Q6_K's combined
// sum stays below it on random data, and an all-extreme Q6_K block can exceed it and then
// rounds at 2^-24 relative. A debug mode runs the same kernel with one part isolated (Q4_K:
// I', J or 8 * sum scale * bsum; Q6_K: I_hi or I_lo) and writes the exact integers.
// The epilogue loads the part into registers in groups, frees the slot once the last group is
// loaded, and folds y += (f * D) * d_a.
//
// Warp roles (896 threads, 7 warpgroups): warps 0-15 epilogue (warp w reads TMEM lanes
// 32*(w%4).. and quarter w/4 of the NT columns), warps 16-23 decode, warp 24 activation
// producer, warp 25 MMA
// issuer (one thread) and TMEM owner, warp 26 weight producer, warp
// 27 idle. The decode warps form two groups of four (one thread per weight row = TMEM lane
// in each) that take alternate K-stages, so one group's tensor-memory stores drain while the
// other decodes; each group also writes half of the Q4_K min-operand rows. setmaxnreg re-splits the 72-per-thread launch allocation: 88 epilogue, 56 decode,
// 40 control (512*88 + 256*56 + 128*40 = 896*72).
//
// Rings (mbarrier-synchronized, every wait bounded):
//   W  raw packed super-block of the 128 rows (+ Q4_K d/dmin), smem   weight producer -> decode
//   E  per-super-block scales for the epilogue, smem: d/dmin, d_a    act. producer -> epilogue
//   J  Q4_K offset/min operands, smem: activation 16-sums (bulk        producer, decode -> MMA
//      copy) and the c head and tail rows; only an "empty" barrier:
//      the copy completes on the super-block's last K-stage barrier
//      and each decode group writes its rows before arriving on its
//      own K-stage, so the MMA's K-stage waits cover the J operands
//   K  K-stage: activation tile (smem, TMA, 128-byte swizzle) and     producer, decode -> MMA
//      decoded weights (TMEM), 64 TMEM columns
//   S  accumulator slots, TMEM                                        MMA -> epilogue
// K order inside each aligned group of 4 is (0,2,1,3) on both operands (the order in which
// the nibble-to-f16 trick below produces weights); the activation operand is stored that way.
#pragma once
#include <cuda_fp16.h>

#include "bounds.cuh"
#include "ptx.cuh"

namespace dllm {

#define QG_FILE 9  // bounds-check sites of this file

constexpr int QK = 256;
constexpr int BM = 128;
constexpr int TYPE_Q4K = 12;
constexpr int TYPE_Q6K = 14;
constexpr int Q4K_BLOB = 17920;  // 128 rows x (128 B quants + 12 B scales)
constexpr int Q6K_BLOB = 26624;  // 128 rows x (128 B ql + 64 B qh + 16 B scales)
constexpr int Q4K_DD = 512;      // 128 rows x (f16 d, f16 dmin)
constexpr int Q6K_DD = 256;      // 128 rows x f16 d
constexpr int QG_THREADS = 896;
constexpr int QG_EPI_WARPS = 16, QG_DEC_WARP0 = 16, QG_DEC_WARPS = 8, QG_PROD_WARP = 24, QG_MMA_WARP = 25,
              QG_WPROD_WARP = 26;
constexpr int QG_REGS_LAUNCH = 72;  // 65536 / 896 rounded down to a multiple of 8
constexpr int QG_REGS_EPI = 88, QG_REGS_DEC = 56, QG_REGS_CTL = 40;
static_assert(512 * QG_REGS_EPI + 256 * QG_REGS_DEC + 128 * QG_REGS_CTL <= QG_THREADS * QG_REGS_LAUNCH,
              "register split");
constexpr int SMEM_LIMIT = 232448;
// how each role waits on an mbarrier: the MMA issuer tests back to back (it is one thread and
// the tensor pipe's feeder); every other role suspends in mbarrier.try_wait (see mbar_wait)
constexpr bool QG_POLL = true, QG_SUSPEND = false;
constexpr int TMEM_COLS = 512;

__host__ __device__ constexpr int al128(int x) { return (x + 127) & ~127; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int TYPE, int NT>
struct QCfg {
  static constexpr bool Q4 = TYPE == TYPE_Q4K;
  static constexpr int NC = NT / 4;  // columns per epilogue thread
  static constexpr int W_BYTES = Q4 ? Q4K_BLOB : Q6K_BLOB;
  static constexpr int DD_BYTES = Q4 ? Q4K_DD : Q6K_DD;
  // a W slot: the blob, then (Q4_K) the super-block's d/dmin plane for the decode warps
  static constexpr int W_SLOT = W_BYTES + (Q4 ? DD_BYTES : 0);
  // K-stage ring: one stage = QPS K-quarters (64 each) of both operands, 8 MMAs per stage:
  // Q4_K two quarters (one MMA chain), Q6_K one quarter (hi and lo chains).
  static constexpr int QPS = Q4 ? 2 : 1;
  static constexpr int SPS = 4 / QPS;  // stages per super-block
  // TMEM: accumulator slots, then the A operand of each stage (64 columns per stage)
  static constexpr int NSLOT = 2;
  static constexpr int ACOL = NSLOT * NT;
  static constexpr int ASTG = 64;
  // Q4_K keeps an odd stage count: its J operands live in the slot of the super-block's last
  // stage, (2 it + 1) % K_STAGES, which then walks through every slot (see the J ring below)
  static constexpr int K_FIT = cmin(6, (TMEM_COLS - ACOL) / ASTG);
  static constexpr int K_STAGES = Q4 ? K_FIT - (K_FIT % 2 == 0 ? 1 : 0) : K_FIT;
  // shared memory: E ring (epilogue scales), J ring (Q4_K min operands)
  static constexpr int E_STAGES = 6;
  static constexpr int E_DD = 0;
  static constexpr int E_DA = al128(DD_BYTES);
  static constexpr int E_BYTES = al128(E_DA + NT * 4);
  static constexpr int E_TX = DD_BYTES + NT * 4;
  static constexpr int J_STAGES = Q4 ? K_STAGES : 0;
  static constexpr int J_BJ = 0;
  static constexpr int J_AJ = al128(NT * 32);
  static constexpr int J_BYTES = J_AJ + 8192;  // c head, then tail, 128 rows x 16 f16 each
  static constexpr int J_TX = NT * 32;
  static constexpr int B_QUARTER = NT * 128;
  static constexpr int B_STAGE = QPS * B_QUARTER;
  static constexpr int SM_AVAIL = SMEM_LIMIT - 2048 - K_STAGES * B_STAGE - E_STAGES * E_BYTES - J_STAGES * J_BYTES;
  static constexpr int W_STAGES = cmin(6, SM_AVAIL / W_SLOT);
  static constexpr int OFF_B = 0;
  static constexpr int OFF_W = OFF_B + K_STAGES * B_STAGE;
  static constexpr int OFF_E = OFF_W + W_STAGES * W_SLOT;
  static constexpr int OFF_J = OFF_E + E_STAGES * E_BYTES;
  static constexpr int OFF_BAR = OFF_J + J_STAGES * J_BYTES;
  // barrier indices
  static constexpr int BK_FULL = 0, BK_EMPTY = BK_FULL + K_STAGES;
  static constexpr int BW_FULL = BK_EMPTY + K_STAGES, BW_EMPTY = BW_FULL + W_STAGES;
  static constexpr int BE_FULL = BW_EMPTY + W_STAGES, BE_EMPTY = BE_FULL + E_STAGES;
  static constexpr int BS_FULL = BE_EMPTY + E_STAGES, BS_EMPTY = BS_FULL + NSLOT;
  static constexpr int B_DONE = BS_EMPTY + NSLOT;
  static constexpr int NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
  static_assert(W_STAGES >= 2 && K_STAGES >= 2, "ring depth");
  static_assert(NT % 32 == 0 && NT >= 32 && NT <= 160, "token tile");
  static_assert(OFF_W % 16 == 0 && OFF_E % 128 == 0 && OFF_J % 128 == 0, "alignment");
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
  int32_t* dbg;   // debug: exact integer sums of one part, [nsb][m][n]
  int dbg_mode;   // 0 off; 1 part 0 only (Q4_K I', Q6_K I_hi); 2 part 1 only (Q4_K J, Q6_K I_lo);
                  // 3 (Q4_K) the offset part 8 * sum scale * bsum, added to dbg (I = I' + it)
  int* err;      // device error word
  // mode 1 (LM head): instead of y, per (weight tile, TMEM lane quadrant, token) softmax
  // partials over the 32 weight rows of the quadrant: max logit, its row (lowest on ties),
  // sum_rows exp(logit - max) and (pent, optional) sum_rows exp(logit - max) (logit - max);
  // layout [m][tiles_n * 4].
  int mode;
  float* pmax;
  int* parg;
  float* psum;
  float* pent;
  // mode 1 sampling (inv_temp > 0): per partial also the Gumbel-max draw over its rows: the
  // best score l * inv_temp + g (g from the counter (step, pos0 + token, row), see
  // gumbel_noise), its row (lowest on ties) and that row's logit
  float inv_temp;
  unsigned long long seed;
  int step, pos0;
  float* pscore;
  int* pidx;
  float* plogit;
  long long timeout;
  Bounds bd;  // bounds-checked build: one span per buffer, indexed by QgSpan
};
enum QgSpan : int { QS_W = 0, QS_DD, QS_AJ, QS_AD, QS_Y, QS_DBG, QS_PMAX, QS_PARG, QS_PSUM, QS_PENT, QS_PSCORE,
                    QS_PIDX, QS_PLOGIT };


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

// Q4_K, one half of a K-quarter: h = 0 the low nibbles (chunks 0-3), h = 1 the high nibbles
// (chunks 4-7) of the quarter's 32 quant bytes, as 16 words. Each nibble lands in bits 4-7 of
// an f16 half with the exponent of 1024 (the low nibbles shifted up by 4), i.e. the half holds
// 1024 + 16 q; (mul, add) = (scale / 16, -72 scale) times the fold's 2^-k turn it into
// scale * (q - 8) * 2^-k with one exact fused multiply-add (72 * scale has at most 10
// significant bits, so the addend is an exact f16 value).
__device__ __forceinline__ void decode_q4k_half(const uint8_t* W, int t, int q, int h, __half2 mul, __half2 add,
                                                uint32_t (&o)[16]) {
  const uint4 v0 = *reinterpret_cast<const uint4*>(W + (2 * q) * 2048 + t * 16);
  const uint4 v1 = *reinterpret_cast<const uint4*>(W + (2 * q + 1) * 2048 + t * 16);
  const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  constexpr uint32_t mask = 0x00F000F0u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = x[2 * c], w1 = x[2 * c + 1];
    // bytes (0, 2) and (1, 3) of each word, their nibble in bits 4-7 of each half
    const uint32_t a0 = h ? w0 : w0 << 4, b0 = h ? w0 >> 8 : w0 >> 4;
    const uint32_t a1 = h ? w1 : w1 << 4, b1 = h ? w1 >> 8 : w1 >> 4;
    o[4 * c + 0] = hfma2u((a0 & mask) | 0x64006400u, mul, add);
    o[4 * c + 1] = hfma2u((b0 & mask) | 0x64006400u, mul, add);
    o[4 * c + 2] = hfma2u((a1 & mask) | 0x64006400u, mul, add);
    o[4 * c + 3] = hfma2u((b1 & mask) | 0x64006400u, mul, add);
  }
}

// Q6_K: piece ps (0 or 1) of half tt of K-quarter q (half-block hq = q/2, t-slot 2(q%2)+tt) of
// row t, from one 16-byte load of ql and one of qh: 8 words of the hi operand
// (hs * s_hi * (q6-32), exact f16 integers) and 8 of the lo operand (ls * s_lo * (q6-32) / 16,
// exact f16 multiples of 1/16), where the int8 group scale s = 16 * s_hi + s_lo, s_lo in [0,15],
// and hs, ls in {0, 1}; so hi + lo = s (q6-32) / 16 and the epilogue applies 16 d. Even
// quarters take the low ql nibble and the f16 pattern 1024 + q6 (qh bits at 4-5), odd quarters
// the high nibble and 1024 + 16*q6 (qh bits at 8-9) with the multiplier divided by 16; every
// operand is one exact fused multiply-add of the pattern.
__device__ __forceinline__ void decode_q6k_piece(const uint8_t* W, int t, int q, int tt, int ps, uint32_t sw,
                                                 float hs, float ls, uint32_t (&hi)[8], uint32_t (&lo)[8]) {
  const int hq = q >> 1, odd = q & 1;
  const uint4 v = *reinterpret_cast<const uint4*>(W + (4 * hq + 2 * tt + ps) * 2048 + t * 16);
  const uint4 u = *reinterpret_cast<const uint4*>(W + 16384 + (2 * hq + ps) * 2048 + t * 16);
  const uint32_t ql[4] = {v.x, v.y, v.z, v.w}, qh[4] = {u.x, u.y, u.z, u.w};
  const uint32_t nmask = odd ? 0x00F000F0u : 0x000F000Fu;
  const uint32_t hmask = odd ? 0x03000300u : 0x00300030u;
  const float fm = odd ? 0.0625f : 1.0f;
  const float fa = odd ? -96.0f : -1056.0f;
  const int shift = tt ? 2 : 4;
  // the row's int8 group scale: scale byte 8 hq + 2 (2 odd + tt) + ps = byte 2 tt + ps of the
  // quarter's scale word sw (its bytes 4q .. 4q + 3)
  const int s = (int)(int8_t)(sw >> (8 * (2 * tt + ps)));
  const float s_hi = hs == 0.f ? 0.f : (float)(s >> 4), s_lo = (float)(s & 15) * ls * 0.0625f;
  const __half2 mH = __float2half2_rn(s_hi * fm), aH = __float2half2_rn(s_hi * fa);
  const __half2 mL = __float2half2_rn(s_lo * fm), aL = __float2half2_rn(s_lo * fa);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t X0 = ql[2 * c], X1 = ql[2 * c + 1];
    const uint32_t H0 = qh[2 * c], H1 = qh[2 * c + 1];
    const uint32_t v0 = (X0 & nmask) | ((H0 << shift) & hmask) | 0x64006400u;
    const uint32_t v1 = ((X0 >> 8) & nmask) | (((H0 >> 8) << shift) & hmask) | 0x64006400u;
    const uint32_t v2 = (X1 & nmask) | ((H1 << shift) & hmask) | 0x64006400u;
    const uint32_t v3 = ((X1 >> 8) & nmask) | (((H1 >> 8) << shift) & hmask) | 0x64006400u;
    hi[4 * c + 0] = hfma2u(v0, mH, aH);
    hi[4 * c + 1] = hfma2u(v1, mH, aH);
    hi[4 * c + 2] = hfma2u(v2, mH, aH);
    hi[4 * c + 3] = hfma2u(v3, mH, aH);
    lo[4 * c + 0] = hfma2u(v0, mL, aL);
    lo[4 * c + 1] = hfma2u(v1, mL, aL);
    lo[4 * c + 2] = hfma2u(v2, mL, aL);
    lo[4 * c + 3] = hfma2u(v3, mL, aL);
  }
}

// Q4_K per-row fold of the min term into the scale-sum accumulator (see the top of the
// file): A scale 2^-k (0 when d = 0), min coefficient -(dmin/d) * 2^-k (-1 when d = 0) and the
// epilogue factor d * 2^k (dmin when d = 0), k the smallest shift >= 0 with
// 63 |dmin/d| 2^-k <= 2^14. The decode and epilogue warps evaluate the same function on the
// same f16 inputs, so both sides agree on k. Sets *bad when no k <= 14 suffices (|dmin/d|
// beyond 4e6; no real block comes near). The ratio takes the fast division (within 2 ulp):
// it only enters the min coefficient, which the J operand carries as an f16 head + tail pair
// anyway; every power of two is built from exponent bits, so the fold has no loop.
struct Q4Fold {
  float ascale, cmul, factor;
};
__device__ __forceinline__ Q4Fold q4k_fold(float d, float dmin, bool* bad) {
  Q4Fold f;
  if (d == 0.f) {
    f.ascale = 0.f;
    f.cmul = -1.f;
    f.factor = dmin;
    return f;
  }
  const float r = __fdividef(dmin, d);
  const float mag = 63.f * fabsf(r);
  const uint32_t mb = __float_as_uint(mag);
  // mag = 2^e (1 + frac): mag * 2^-k <= 2^14 first holds at k = e - 14 (frac = 0) or e - 13
  int k = mag <= 16384.f ? 0 : (int)(mb >> 23) - 141 + ((mb & 0x7FFFFFu) != 0u);
  if (k > 14) {  // also NaN / inf ratios
    k = 14;
    *bad = true;
  }
  f.ascale = __uint_as_float((uint32_t)(127 - k) << 23);
  f.cmul = -r * f.ascale;
  f.factor = d * __uint_as_float((uint32_t)(127 + k) << 23);
  return f;
}

// Gumbel noise of one (row, vocabulary entry) of a sampling step: counter-based SplitMix64
// (Steele, Lea and Flood, "Fast splittable pseudorandom number generators"): the output for
// counter c of the stream `seed` is mix(seed + (c + 1) * 0x9E3779B97F4A7C15). Counter
// c = step * 2^40 + position * 2^24 + vocabulary id; its top 23 bits give the uniform
// u = (bits + 1/2) / 2^23, exact in f32 and strictly inside (0, 1) (with 24 bits the top value
// would round to 1 and give infinite noise), and g = -log(-log u).
__device__ __forceinline__ float gumbel_noise(unsigned long long seed, unsigned long long c) {
  unsigned long long z = seed + (c + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  const float u = ((float)(z >> 41) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
  return -logf(-logf(u));
}

// The first super-blocks that each CTA of a GEMM launch streams from HBM: the kernel that runs
// before the GEMM prefetches them into L2 (its data lives in L2, so HBM is otherwise idle then),
// and the GEMM's first weight copies hit L2 instead of waiting for HBM. wblob = nullptr: none.
struct WPrefetch {
  const uint8_t* wblob;
  int tiles_n, tiles_m, nsb, sbps, units, w_bytes, ahead;
  Bounds bd;  // span 0: the blob
};
// One thread per CTA of the prefetching kernel: units blockIdx.x, blockIdx.x + gridDim.x, ...
// of the GEMM's first wave (units < f.units), `ahead` super-blocks each (contiguous in the
// tile's blob run).
__device__ __forceinline__ void prefetch_weights(const WPrefetch& f) {
  if (f.wblob == nullptr) return;
  for (int u = blockIdx.x; u < f.units; u += gridDim.x) {
    const int tn = u % f.tiles_n, sp = (u / f.tiles_n) / f.tiles_m;
    const int sb0 = sp * f.sbps, n = min(f.ahead, f.nsb - sb0);
    const uint8_t* src = f.wblob + ((size_t)tn * f.nsb + sb0) * f.w_bytes;
    if (n > 0 && BOK_AT(QG_FILE, f.bd, 0, src, (size_t)n * f.w_bytes)) bulk_prefetch_l2(src, (uint32_t)(n * f.w_bytes));
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

// SAMPLE: the LM-head epilogue also makes the Gumbel-max draws (mode 1 with inv_temp > 0); a
// separate instantiation, so the other kernels carry none of its code.
template <int TYPE, int NT, bool SAMPLE = false>
__global__ void __launch_bounds__(QG_THREADS, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmap, const QgemmParams p) {
  using C = QCfg<TYPE, NT>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by offset from the shared array (keeps shared-memory addressing)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  auto BAR = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  const long long lim = p.timeout;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::K_STAGES; ++i) {
      mbar_init(BAR(C::BK_FULL + i), 1 + QG_DEC_WARPS / 2);  // producer (with the B bytes) + a decode group
      mbar_init(BAR(C::BK_EMPTY + i), 1);
    }
    for (int i = 0; i < C::W_STAGES; ++i) {
      mbar_init(BAR(C::BW_FULL + i), 1);
      mbar_init(BAR(C::BW_EMPTY + i), QG_DEC_WARPS);
    }
    for (int i = 0; i < C::E_STAGES; ++i) {
      mbar_init(BAR(C::BE_FULL + i), 1);
      mbar_init(BAR(C::BE_EMPTY + i), QG_EPI_WARPS);
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
  // the next kernel of the stream may be scheduled now (its CTAs start as ours exit); only the
  // roles that read the preceding kernel's outputs or write ours wait for it below
  griddep_launch();

  if (warp >= QG_PROD_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_CTL));
    if (warp == QG_WPROD_WARP && lane == 0) {
      // ---------------------------------------------------------- weight producer (one thread):
      // raw packed super-blocks as far ahead as the W ring allows (HBM latency is hidden only
      // by depth, so this runs independently of the activation stages); each blob is read once
      // per step, so it is copied with an L2 evict-first policy
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int tn, tm, sp, sb0, sb1;
        unit_coords(p, u, tn, tm, sp, sb0, sb1);
        const uint8_t* blob = p.wblob + (size_t)tn * p.nsb * C::W_BYTES;
        const uint8_t* dd = p.wdd + (size_t)tn * p.nsb * C::DD_BYTES;
        for (int sb = sb0; sb < sb1; ++sb, ++it) {
          const int w = it % C::W_STAGES;
          if (!(ok = mbar_wait(BAR(C::BW_EMPTY + w), ((it / C::W_STAGES) & 1) ^ 1, abort_flag, lim, QG_SUSPEND))) break;
          const uint32_t ws = sbase + C::OFF_W + w * C::W_SLOT;
          mbar_expect_tx(BAR(C::BW_FULL + w), C::W_SLOT);
          // a copy outside its buffer (bounds-checked build) is not issued: its stage never
          // fills and the waits on it run out, so the launch ends with both errors set
          if (BOK_AT(QG_FILE, p.bd, QS_W, blob + (size_t)sb * C::W_BYTES, C::W_BYTES))
            bulk_g2s_once(ws, blob + (size_t)sb * C::W_BYTES, C::W_BYTES, BAR(C::BW_FULL + w));
          if (C::Q4 && BOK_AT(QG_FILE, p.bd, QS_DD, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES))
            bulk_g2s(ws + C::W_BYTES, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES, BAR(C::BW_FULL + w));
        }
      }
      if (!ok) {
        atomicOr(p.err, ERR_TIMEOUT_PRODUCER);
        const long long t0 = clock64();  // let issued copies land before the CTA can exit (~1 ms)
        while (clock64() - t0 < 2000000) {
        }
      }
    } else if (warp == QG_PROD_WARP && lane == 0) {
      // ---------------------------------------------------------- activation producer (one
      // thread): per super-block the epilogue scales (E), the Q4_K activation 16-sums (J), then
      // the activation operand stages through the tensor map
      prefetch_tensormap(&tmap);
      griddep_wait();  // the activations are the preceding kernel's output
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int tn, tm, sp, sb0, sb1;
        unit_coords(p, u, tn, tm, sp, sb0, sb1);
        const uint8_t* dd = p.wdd + (size_t)tn * p.nsb * C::DD_BYTES;
        const int tok0 = tm * NT;
        for (int sb = sb0; sb < sb1; ++sb, ++it) {
          const int e = it % C::E_STAGES;
          if (!(ok = mbar_wait(BAR(C::BE_EMPTY + e), ((it / C::E_STAGES) & 1) ^ 1, abort_flag, lim, QG_SUSPEND))) break;
          const uint32_t es = sbase + C::OFF_E + e * C::E_BYTES;
          mbar_expect_tx(BAR(C::BE_FULL + e), C::E_TX);
          if (BOK_AT(QG_FILE, p.bd, QS_DD, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES))
            bulk_g2s(es + C::E_DD, dd + (size_t)sb * C::DD_BYTES, C::DD_BYTES, BAR(C::BE_FULL + e));
          if (BOK_AT(QG_FILE, p.bd, QS_AD, p.act_d + (size_t)sb * p.lpad + tok0, NT * 4))
            bulk_g2s(es + C::E_DA, p.act_d + (size_t)sb * p.lpad + tok0, NT * 4, BAR(C::BE_FULL + e));
          for (int st = 0; st < C::SPS; ++st) {
            const int j = C::SPS * it + st, b = j % C::K_STAGES;
            if (!(ok = mbar_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim, QG_SUSPEND))) break;
            // Q4_K: the super-block's activation 16-sums go to J slot b of its last stage and ride
            // on that stage's barrier, so the MMA issuer's wait for the stage also covers the
            // offset/min operands (the decode groups write their coefficient rows before they
            // arrive on their own stages); the BK_EMPTY wait above also frees the J slot (below)
            const bool jcopy = C::Q4 && st == C::SPS - 1;
            const int jx = b;
            mbar_expect_tx(BAR(C::BK_FULL + b), C::B_STAGE + (jcopy ? C::J_TX : 0));
#pragma unroll
            for (int qq = 0; qq < C::QPS; ++qq)
              tma_g2s_3d(sbase + C::OFF_B + b * C::B_STAGE + qq * C::B_QUARTER, &tmap, 0, tok0,
                         sb * 4 + st * C::QPS + qq, BAR(C::BK_FULL + b));
            if (jcopy && BOK_AT(QG_FILE, p.bd, QS_AJ, p.act_j + ((size_t)sb * p.lpad + tok0) * 32, NT * 32))
              bulk_g2s(sbase + C::OFF_J + jx * C::J_BYTES + C::J_BJ, p.act_j + ((size_t)sb * p.lpad + tok0) * 32,
                       NT * 32, BAR(C::BK_FULL + b));
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
      // ---------------------------------------------------------- MMA issuer (one thread; a
      // warp-wide issue was measured to replay each MMA once per lane). Accumulator slot s (NT
      // columns at s * NT) is written only after the epilogue drained its previous contents;
      // se0/se1 count those waits.
      constexpr uint32_t IDESC = idesc_f16(BM, NT);
      int it = 0;
      uint32_t se0 = 0, se1 = 0;
      bool ok = true;
      auto wait_tc = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool r = mbar_wait(bar, parity, abort_flag, lim, QG_POLL);
        tc_fence_after();
        return r;
      };
      auto slot_free = [&](int s) -> bool {
        const uint32_t n = s ? se1++ : se0++;
        return wait_tc(BAR(C::BS_EMPTY + s), (n & 1) ^ 1);
      };
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        int tn, tm, sp, sb0, sb1;
        unit_coords(p, u, tn, tm, sp, sb0, sb1);
        for (int sb = sb0; sb < sb1; ++sb, ++it) {
          const int s = it & 1;
          if (!(ok = slot_free(s))) break;  // super-block it - 2 drained
          const uint32_t dslot = tmem + s * NT;
          if constexpr (C::Q4) {
            for (int st = 0; st < 2; ++st) {
              const int j = 2 * it + st, b = j % C::K_STAGES;
              if (!(ok = wait_tc(BAR(C::BK_FULL + b), (j / C::K_STAGES) & 1))) break;
              const uint32_t acol = tmem + C::ACOL + b * C::ASTG;
              const uint64_t bdesc = desc_sw128(sbase + C::OFF_B + b * C::B_STAGE);
#pragma unroll
              for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f16_ts(dslot, acol + qq * 32 + kk * 8, bdesc + (uint64_t)((qq * C::B_QUARTER + kk * 32) >> 4),
                                  IDESC, (st | qq | kk) != 0);
              if (st == 1) {
                // offset and min term: head and tail coefficients x activation 16-sums, in J slot
                // b (ready with this stage: see the activation producer); the stage's commit
                // below then also releases the J slot
                const uint32_t js = sbase + C::OFF_J + b * C::J_BYTES;
                const uint64_t bj = desc_noswz(js + C::J_BJ, 128, 256);
                mma_f16(dslot, desc_noswz(js + C::J_AJ, 128, 256), bj, IDESC, 1);
                mma_f16(dslot, desc_noswz(js + C::J_AJ + 4096, 128, 256), bj, IDESC, 1);
              }
              mma_commit(BAR(C::BK_EMPTY + b));
            }
            if (!ok) break;
          } else {
            for (int q = 0; q < 4; ++q) {
              const int j = 4 * it + q, b = j % C::K_STAGES;
              if (!(ok = wait_tc(BAR(C::BK_FULL + b), (j / C::K_STAGES) & 1))) break;
              const uint32_t acol = tmem + C::ACOL + b * C::ASTG;
              const uint64_t bdesc = desc_sw128(sbase + C::OFF_B + b * C::B_STAGE);
#pragma unroll
              for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f16_ts(dslot, acol + part * 32 + kk * 8, bdesc + (uint64_t)((kk * 32) >> 4), IDESC,
                                  (q | part | kk) != 0);
              mma_commit(BAR(C::BK_EMPTY + b));
            }
            if (!ok) break;
          }
          // Q4_K: the last stage's commit (its K-stage barrier) already tells the epilogue that
          // the super-block's part is complete (see the epilogue's wait)
          if constexpr (!C::Q4) mma_commit(BAR(C::BS_FULL + s));
        }
      }
      if (!ok) atomicOr(p.err, ERR_TIMEOUT_MMA);
      // all issued MMAs complete before the tensor memory is released
      mma_commit(BAR(C::B_DONE));
      volatile int never = 0;
      mbar_wait(BAR(C::B_DONE), 0, &never, lim);
    }
  } else if (warp >= QG_DEC_WARP0) {
    // ------------------------------------------------------------ decode: group g (warps 16-19 or
    // 20-23), thread = weight row = TMEM lane; group g decodes the stages j with j % 2 == g
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_DEC));
    const int g = (warp - QG_DEC_WARP0) >> 2;
    const int t = (warp & 3) * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(warp & 3) * 32 << 16) + C::ACOL;
    int it = 0;
    bool ok = true, bad = false;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      int tn, tm, sp, sb0, sb1;
      unit_coords(p, u, tn, tm, sp, sb0, sb1);
      for (int sb = sb0; sb < sb1; ++sb, ++it) {
        const int w = it % C::W_STAGES;
        if (!(ok = warp_wait(BAR(C::BW_FULL + w), (it / C::W_STAGES) & 1, abort_flag, lim, QG_SUSPEND))) break;
        const uint8_t* W = smem + C::OFF_W + w * C::W_SLOT;
        if constexpr (C::Q4) {
          // row t's fold of this super-block (see q4k_fold): the A operand carries scale * q * 2^-k
          const __half2 ddv = *reinterpret_cast<const __half2*>(W + C::W_BYTES + t * 4);
          const Q4Fold fo = q4k_fold(__low2float(ddv), __high2float(ddv), &bad);
          // A scale, and the J coefficients on 8 * scale and on min (debug modes isolate a part)
          const float ascale = p.dbg_mode == 0 ? fo.ascale : (p.dbg_mode == 1 ? 1.f : 0.f);
          const float jsc = p.dbg_mode == 0 ? fo.ascale : (p.dbg_mode == 3 ? 1.f : 0.f);
          const float jmn = p.dbg_mode == 0 ? fo.cmul : (p.dbg_mode == 2 ? -1.f : 0.f);
          // stage g = quarters 2g, 2g+1 = sub-blocks 4g..4g+3; 6-bit scales: bytes 0-3 of scale
          // word 0 are entries 0..3, entries 4..7 combine word 2's low nibbles and word 0's top bits
          const uint32_t sw0 = *reinterpret_cast<const uint32_t*>(W + 16384 + t * 4);
          const uint32_t s4 = g ? (((*reinterpret_cast<const uint32_t*>(W + 16384 + 1024 + t * 4)) & 0x0F0F0F0Fu) |
                                   ((sw0 >> 2) & 0x30303030u))
                                : (sw0 & 0x3F3F3F3Fu);
          const int j = 2 * it + g, b = j % C::K_STAGES;
          if (!(ok = warp_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim, QG_SUSPEND))) break;
          tc_fence_after();
          const uint32_t ta = tlane + b * C::ASTG;
          // f16 multipliers (scale * 2^-k / 16) and addends (-72 scale * 2^-k): exact, from one
          // integer-to-half conversion per sub-block
          const __half2 asc = __float2half2_rn(ascale);
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // sub-block 2q + h of quarter q = 2g + qq; value scale * (q4 - 8) * 2^-k
              const __half2 sc = __hmul2(__half2half2(__int2half_rn((s4 >> (16 * qq + 8 * h)) & 0xFF)), asc);
              const __half2 mul = __hmul2(sc, __float2half2_rn(0.0625f));
              const __half2 add = __hmul2(sc, __float2half2_rn(-72.f));
              uint32_t o[16];
              decode_q4k_half(W, t, 2 * g + qq, h, mul, add, o);
              tmem_st16(ta + 32 * qq + 16 * h, o);
            }
          }
          {
            // while the stores drain: row t's J operand (K-major 8x16 B core matrices, no
            // swizzle; K = 16 groups of 16 values, group k pairs with sub-block k/2) holds the f16
            // head and tail of c = jsc * 8 * scale + jmn * min; group g writes core matrix g
            // (sub-blocks 4g..4g+3)
            // J slot of the super-block's last stage. Its previous user is super-block it - K_STAGES
            // (2 it + 1 walks every slot mod an odd K_STAGES), whose J MMAs were issued before the
            // stage this group waited on above (2 it + g - K_STAGES > 2 (it - K_STAGES) + 1), and
            // MMAs complete in issue order: the slot is free
            const int jx = (2 * it + 1) % C::K_STAGES;
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(W + 16384 + 512 + t * 4);
            // 6-bit mins: entries 0..3 are the bytes of word 1, entries 4..7 combine word 2's
            // high nibbles with word 1's top bits
            const uint32_t m4 =
                g ? ((((*reinterpret_cast<const uint32_t*>(W + 16384 + 1024 + t * 4)) >> 4) & 0x0F0F0F0Fu) |
                     ((w1 >> 2) & 0x30303030u))
                  : (w1 & 0x3F3F3F3Fu);
            uint32_t hd[4], tl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float c = fmaf(jmn, (float)((m4 >> (8 * i)) & 0xFF), jsc * (float)(8 * ((s4 >> (8 * i)) & 0xFF)));
              const __half ch = __float2half_rn(c);
              const __half ct = __float2half_rn(c - __half2float(ch));
              hd[i] = h2u(__halves2half2(ch, ch));
              tl[i] = h2u(__halves2half2(ct, ct));
            }
            uint8_t* row = smem + C::OFF_J + jx * C::J_BYTES + C::J_AJ + (t >> 3) * 256 + (t & 7) * 16 + g * 128;
            *reinterpret_cast<uint4*>(row) = make_uint4(hd[0], hd[1], hd[2], hd[3]);
            *reinterpret_cast<uint4*>(row + 4096) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
            fence_proxy_async();
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::BK_FULL + b));
        } else {

          const float hs = p.dbg_mode == 2 ? 0.f : 1.f;
          const float ls = p.dbg_mode == 1 ? 0.f : 1.f;
#pragma unroll 1
          for (int q = g; q < 4; q += 2) {
            const int j = 4 * it + q, b = j % C::K_STAGES;
            if (!(ok = warp_wait(BAR(C::BK_EMPTY + b), ((j / C::K_STAGES) & 1) ^ 1, abort_flag, lim, QG_SUSPEND))) break;
            tc_fence_after();
            const uint32_t sw = *reinterpret_cast<const uint32_t*>(W + 24576 + t * 16 + 4 * q);  // quarter q's scales
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int ps = 0; ps < 2; ++ps) {
                uint32_t hi[8], lo[8];
                decode_q6k_piece(W, t, q, h, ps, sw, hs, ls, hi, lo);
                tmem_st8(tlane + b * C::ASTG + 16 * h + 8 * ps, hi);
                tmem_st8(tlane + b * C::ASTG + 32 + 16 * h + 8 * ps, lo);
              }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::BK_FULL + b));
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BW_EMPTY + w));
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, ERR_TIMEOUT_DECODE);
    if (bad) atomicOr(p.err, ERR_RANGE);  // the row's own thread: any lane may hold the bad block
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-15)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(QG_REGS_EPI));
    griddep_wait();  // outputs may be read (accumulate) or still in use by the preceding kernel
    constexpr int NC = C::NC;
    constexpr int NCH = NC / 8;
    const int qd = warp & 3, hf = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t tlane = tmem + ((uint32_t)(32 * qd) << 16) + hf * NC;
    int it = 0;
    uint32_t sf0 = 0, sf1 = 0;  // full phases consumed per accumulator slot
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      int tn, tm, sp, sb0, sb1;
      unit_coords(p, u, tn, tm, sp, sb0, sb1);
      const int grow = tn * BM + row;
      const int tokb = tm * NT + hf * NC;
      float acc[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) acc[i] = 0.f;
      // one accumulator part per super-block, in slot it & 1
      const int nsbu = sb1 - sb0, it0 = it;
#pragma unroll 1
      for (int i = 0; i < nsbu; ++i) {
        const int itp = it0 + i, sbp = sb0 + i;
        const int s = itp & 1;
        const int e = itp % C::E_STAGES;
        if (!(ok = warp_wait(BAR(C::BE_FULL + e), (itp / C::E_STAGES) & 1, abort_flag, lim, QG_SUSPEND))) break;
        const uint8_t* E = smem + C::OFF_E + e * C::E_BYTES;
        float cp;
        if constexpr (C::Q4) {
          const __half2 dd = *reinterpret_cast<const __half2*>(E + C::E_DD + row * 4);
          bool bad = false;
          cp = q4k_fold(__low2float(dd), __high2float(dd), &bad).factor;
        } else {
          cp = 16.f * __half2float(*reinterpret_cast<const __half*>(E + C::E_DD + row * 2));  // D = sum s (q-32) a / 16
        }
        const float4* da4 = reinterpret_cast<const float4*>(E + C::E_DA) + hf * (NC / 4);
        const uint32_t n = s ? sf1++ : sf0++;
        if constexpr (C::Q4) {
          // the commit after the super-block's last stage, j = 2 itp + 1, covers all its MMAs. That
          // K-stage barrier cannot complete another phase before this wait is satisfied: its next
          // use, stage j + K_STAGES (odd), belongs to super-block itp + 2 or later, whose MMAs wait
          // for this epilogue to free slot s. So its parity identifies the phase.
          const int j = 2 * itp + 1;
          if (!(ok = warp_wait(BAR(C::BK_EMPTY + j % C::K_STAGES), (j / C::K_STAGES) & 1, abort_flag, lim,
                               QG_SUSPEND)))
            break;
        } else {
          if (!(ok = warp_wait(BAR(C::BS_FULL + s), n & 1, abort_flag, lim, QG_SUSPEND))) break;
        }
        tc_fence_after();
        // drain in groups of up to 2 x 8 columns; the slot is freed as soon as the last group
        // is in registers, before its arithmetic
        constexpr int G = 2;
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
            if (p.dbg_mode != 0 && grow < p.n) {
              // the isolated part's exact integers (Q4_K J is accumulated negated; the Q4_K offset
              // part is added to the I' already written, giving I; Q6_K's lo part is held / 16)
              const float sgn = p.dbg_mode != 2 ? 1.f : (C::Q4 ? -1.f : 16.f);
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int tok = tokb + ch * 8 + jj;
                if (tok < p.m) {
                  int32_t* dst = p.dbg + ((size_t)sbp * p.m + tok) * p.n + grow;
                  const int32_t v = (int32_t)(sgn * __uint_as_float(r[c][jj]));
                  if (BOK_AT(QG_FILE, p.bd, QS_DBG, dst, 4)) *dst = p.dbg_mode == 3 ? *dst + v : v;
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BE_EMPTY + e));
      }
      if (!ok) break;
      it = it0 + nsbu;
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
          const float dl = acc[j] - v;
          float ex = grow < p.n ? expf(dl) : 0.f;
          float tx = grow < p.n ? ex * dl : 0.f;  // for the entropy: sum exp(l - max) (l - max)
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ex += __shfl_xor_sync(0xffffffffu, ex, off);
          if (p.pent != nullptr) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tx += __shfl_xor_sync(0xffffffffu, tx, off);
          }
          const int tok = tokb + j;
          if constexpr (SAMPLE) {
            // Gumbel-max draw: the best perturbed score of the quadrant's rows
            float sc = -INFINITY, sl = 0.f;
            int si = grow;
            if (grow < p.n) {
              const unsigned long long c = ((unsigned long long)p.step << 40) |
                                           ((unsigned long long)(p.pos0 + tok) << 24) | (unsigned long long)grow;
              sc = acc[j] * p.inv_temp + gumbel_noise(p.seed, c);
              sl = acc[j];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
              const float os = __shfl_xor_sync(0xffffffffu, sc, off);
              const int oi = __shfl_xor_sync(0xffffffffu, si, off);
              const float ol = __shfl_xor_sync(0xffffffffu, sl, off);
              if (os > sc || (os == sc && oi < si)) {
                sc = os;
                si = oi;
                sl = ol;
              }
            }
            if (lane == 0 && tok < p.m) {
              const size_t o = (size_t)tok * (p.tiles_n * 4) + tn * 4 + qd;
              STB_AT(QG_FILE, p.bd, QS_PSCORE, p.pscore + o, sc);
              STB_AT(QG_FILE, p.bd, QS_PIDX, p.pidx + o, si);
              STB_AT(QG_FILE, p.bd, QS_PLOGIT, p.plogit + o, sl);
            }
          }
          if (lane == 0 && tok < p.m) {
            const size_t o = (size_t)tok * (p.tiles_n * 4) + tn * 4 + qd;
            STB_AT(QG_FILE, p.bd, QS_PMAX, p.pmax + o, v);
            STB_AT(QG_FILE, p.bd, QS_PARG, p.parg + o, idx);
            STB_AT(QG_FILE, p.bd, QS_PSUM, p.psum + o, ex);
            if (p.pent != nullptr) STB_AT(QG_FILE, p.bd, QS_PENT, p.pent + o, tx);
          }
        }
      } else if (p.y != nullptr && grow < p.n) {
        // two uniform branches: a plain store must not wait for a read of the old value
        float* dst = p.y + (size_t)sp * p.split_stride + grow;
        if (p.accumulate) {
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const int tok = tokb + j;
            if (tok < p.m && BOK_AT(QG_FILE, p.bd, QS_Y, dst + (size_t)tok * p.ldy, 4)) dst[(size_t)tok * p.ldy] += acc[j];
          }
        } else {
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const int tok = tokb + j;
            if (tok < p.m) STB_AT(QG_FILE, p.bd, QS_Y, dst + (size_t)tok * p.ldy, acc[j]);
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
