// Q8_K quantization of one super-block held in registers (shared by the activation
// quantizer and the fused layer kernels). Rule (mojo-dllm "Development plan", "Compute
// design": 8-bit codes, an f32 scale for every 256, the integer sum of every 16):
// amax = max|x|, d = amax / 127,
// q = clamp(rint(x * (127 / amax)), -127, 127) with an f32 multiply and IEEE division;
// amax == 0 gives d = 0 and q = 0.
#pragma once
#include <cuda_fp16.h>

#include "bounds.cuh"
#include "qgemm.cuh"

namespace dllm {

#define QT_FILE 10  // bounds-check sites of this file

struct QuantOut {
  int8_t* q;
  float* d;
  int16_t* bsum;
  __half* act_a;
  uint8_t* act_j;
  float* act_d;
  int lpad;
  float* vtap;  // optional: the f32 values being quantized, [rows][k] (row stride k), for tests
  Bounds bd;    // bounds-checked build: spans QO_* (set_quant_bounds)
};
enum QoSpan : int { QO_Q = 0, QO_D, QO_BSUM, QO_A, QO_J, QO_AD, QO_VTAP };
// Host: the spans of o's outputs for `rows` rows of k values (the plain arrays, the operand
// planes of an act buffer with o.lpad padded rows, the tap); the regular build leaves bd empty.
void set_quant_bounds(QuantOut& o, int64_t rows, int64_t k);

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
  return s;
}

// Write one quantized super-block (lane holds codes k = 8*lane .. 8*lane+7, s16 the sum of
// its lane pair's 16 codes, dsc the scale) to every requested output of (row, sb).
__device__ __forceinline__ void q8k_store(const int (&qi)[8], int s16, float dsc, int row, int rows, int sb, int64_t k,
                                          const QuantOut& o) {
  const int lane = threadIdx.x & 31;
  const int64_t nsb = k / QK;
  const int g = lane >> 1;
  if (row < rows) {
    if (o.q) {
      uint32_t lo = (qi[0] & 0xFF) | ((qi[1] & 0xFF) << 8) | ((qi[2] & 0xFF) << 16) | ((uint32_t)(qi[3] & 0xFF) << 24);
      uint32_t hi = (qi[4] & 0xFF) | ((qi[5] & 0xFF) << 8) | ((qi[6] & 0xFF) << 16) | ((uint32_t)(qi[7] & 0xFF) << 24);
      STB_AT(QT_FILE, o.bd, QO_Q, reinterpret_cast<uint2*>(o.q + (int64_t)row * k + (int64_t)sb * QK + 8 * lane),
             make_uint2(lo, hi));
    }
    if (o.d && lane == 0) STB_AT(QT_FILE, o.bd, QO_D, o.d + (int64_t)row * nsb + sb, dsc);
    if (o.bsum && (lane & 1) == 0)
      STB_AT(QT_FILE, o.bd, QO_BSUM, o.bsum + (int64_t)row * (k / 16) + (int64_t)sb * 16 + g, (int16_t)s16);
  }
  if (o.act_a) {
    // A-plane [k/64][lpad][64]; quarter q = lane/8, 16-byte chunk c = lane%8, order (0,2,1,3)
    const int q = lane >> 3, c = lane & 7;
    __half2 h0 = __floats2half2_rn((float)qi[0], (float)qi[2]);
    __half2 h1 = __floats2half2_rn((float)qi[1], (float)qi[3]);
    __half2 h2 = __floats2half2_rn((float)qi[4], (float)qi[6]);
    __half2 h3 = __floats2half2_rn((float)qi[5], (float)qi[7]);
    uint4 pk = make_uint4(h2u(h0), h2u(h1), h2u(h2), h2u(h3));
    STB_AT(QT_FILE, o.bd, QO_A, reinterpret_cast<uint4*>(o.act_a + (((int64_t)sb * 4 + q) * o.lpad + row) * 64 + c * 8), pk);
    // J-plane [nsb][lpad/8][2][8][8]
    if ((lane & 1) == 0) {
      __half* j = reinterpret_cast<__half*>(o.act_j + ((int64_t)sb * o.lpad) * 32) + (row >> 3) * 128 +
                  (g >> 3) * 64 + (row & 7) * 8 + (g & 7);
      STB_AT(QT_FILE, o.bd, QO_J, j, __int2half_rn(s16));
    }
    if (lane == 0) STB_AT(QT_FILE, o.bd, QO_AD, o.act_d + (int64_t)sb * o.lpad + row, dsc);
  }
}

// Quantize one super-block held as 8 values per lane (lane covers k = 8*lane .. 8*lane+7)
// and write all requested outputs for (row, sb).
__device__ __forceinline__ void q8k_emit(float (&v)[8], int row, int rows, int sb, int64_t k, const QuantOut& o) {
  if (o.vtap && row < rows) {
    float* t = o.vtap + (int64_t)row * k + (int64_t)sb * QK + 8 * (threadIdx.x & 31);
    STB_AT(QT_FILE, o.bd, QO_VTAP, reinterpret_cast<float4*>(t), make_float4(v[0], v[1], v[2], v[3]));
    STB_AT(QT_FILE, o.bd, QO_VTAP, reinterpret_cast<float4*>(t + 4), make_float4(v[4], v[5], v[6], v[7]));
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  int qi[8];
  float dsc = 0.f;
  if (amax == 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) qi[i] = 0;
  } else {
    const float iscale = __fdiv_rn(127.f, amax);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float r = rintf(__fmul_rn(v[i], iscale));
      r = fminf(127.f, fmaxf(-127.f, r));
      qi[i] = (int)r;
    }
    dsc = __fdiv_rn(amax, 127.f);
  }
  int s8 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s8 += qi[i];
  const int s16 = s8 + __shfl_xor_sync(0xffffffffu, s8, 1);  // group of 16 = lane pair
  q8k_store(qi, s16, dsc, row, rows, sb, k, o);
}

}  // namespace dllm
