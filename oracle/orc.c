/*
 * CPU oracle for the LLaDA-style denoising-step hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header or table with the CUDA
 * library.
 *
 * Everything here is the plain definition of what the method computes:
 * weights are decoded to their exact real values (held in f64), dot products
 * are accumulated in f64 in natural k order, and all layer maths (RMSNorm,
 * RoPE, attention, SwiGLU, softmax) is f64. The one place where floating
 * point decides an integer, Q8_K activation quantization, takes its
 * decisions in f32, the precision the GPU kernel uses.
 *
 * Sources (mojo-dllm pages):
 *   - Development plan, "Corrections to the spec": the LLaDA-8B Q4_K_M file
 *     mixes Q4_K and Q6_K weight matrices, with its norms in F32.
 *   - Development plan, "Compute design": every token's activations are
 *     quantized as Q8_K (8-bit codes, an f32 scale for each 256 of them, the
 *     integer sum of each 16); every weight block expands to small unsigned
 *     integers with an integer scale and an f32 offset for each 16; the
 *     integer products are summed over the whole row before any scale.
 *   - Development plan, "Model facts": RMSNorm eps 1e-5, RoPE theta 500000
 *     (adjacent-pair / NORM form), 32 x 128 MHA, non-causal, SwiGLU FFN.
 *   - Technical specification, section 12 (diffusion loop) and section 14
 *     (sampling primitives): softmax confidence, entropy, top-k selection,
 *     scatter.
 *   - README, "Each model's own sampler": LLaDA ranks masked positions by
 *     the argmax token's probability, Dream by entropy.
 *   - Technical specification, section 30 (definition of done: a fixed seed
 *     gives the same run every time), section 14 (sampling) and the
 *     --seed / --temperature flags: temperature sampling from a seeded,
 *     deterministic generator (here counter-based SplitMix64).
 *   - README, "How it works": the output head is evaluated only for the
 *     masked positions of the active block.
 * The GGUF byte layouts of Q4_K / Q6_K are the public GGUF formats that the
 * pages name; they are spelled out at each decoder below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256
#define Q4K_BYTES 144
#define Q6K_BYTES 210
#define TYPE_Q4_K 12
#define TYPE_Q6_K 14

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* IEEE binary16 -> exact double. */
static double f16_to_f64(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------------------
 * Q4_K super-block (144 bytes, 256 weights):
 *   [0,2) f16 d, [2,4) f16 dmin, [4,16) 12 bytes of packed 6-bit scales and
 *   mins, [16,144) 128 bytes of 4-bit quants.
 * Sub-block j (0..7) holds 32 weights. For j < 4: scale = s[j] & 63,
 * min = s[j+4] & 63. For j >= 4: scale = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 * min = (s[j+4] >> 4) | ((s[j] >> 6) << 4).
 * Weight i: c = i / 64, l = i % 32; byte qs[32c + l]; low nibble when
 * (i % 64) < 32, high nibble otherwise; sub-block j = i / 32.
 * Value: w = d * scale_j * q - dmin * min_j.
 * ------------------------------------------------------------------------- */
void orc_q4k_fields(const uint8_t* blk, int* sc /*8*/, int* mn /*8*/, uint8_t* q /*256*/) {
  const uint8_t* s = blk + 4;
  const uint8_t* qs = blk + 16;
  for (int j = 0; j < 8; ++j) {
    if (j < 4) {
      sc[j] = s[j] & 63;
      mn[j] = s[j + 4] & 63;
    } else {
      sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
  }
  for (int i = 0; i < QK; ++i) {
    int c = i / 64, l = i % 32;
    uint8_t b = qs[32 * c + l];
    q[i] = ((i % 64) < 32) ? (b & 15) : (b >> 4);
  }
}

static void dequant_q4k_block(const uint8_t* blk, double* out) {
  int sc[8], mn[8];
  uint8_t q[QK];
  orc_q4k_fields(blk, sc, mn, q);
  double d = f16_to_f64(rd16(blk)), dmin = f16_to_f64(rd16(blk + 2));
  for (int i = 0; i < QK; ++i) out[i] = d * sc[i / 32] * q[i] - dmin * mn[i / 32];
}

/* ---------------------------------------------------------------------------
 * Q6_K super-block (210 bytes, 256 weights):
 *   [0,128) ql: low 4 bits, [128,192) qh: high 2 bits, [192,208) 16 int8
 *   scales, [208,210) f16 d.
 * Weight i: h = i / 128, t = (i % 128) / 32, l = i % 32.
 *   low 4 bits: byte ql[64h + l + 32*(t & 1)], low nibble if t < 2 else high;
 *   high 2 bits: (qh[32h + l] >> 2t) & 3;  q = low | high << 4 in [0, 63].
 *   Group of 16: scale = scales[8h + (i % 128) / 16].
 * Value: w = d * scale * (q - 32).
 * ------------------------------------------------------------------------- */
void orc_q6k_fields(const uint8_t* blk, int* sc /*16*/, uint8_t* q /*256*/) {
  const uint8_t* ql = blk;
  const uint8_t* qh = blk + 128;
  const int8_t* s = (const int8_t*)(blk + 192);
  for (int g = 0; g < 16; ++g) sc[g] = s[g];
  for (int i = 0; i < QK; ++i) {
    int h = i / 128, t = (i % 128) / 32, l = i % 32;
    uint8_t b = ql[64 * h + l + 32 * (t & 1)];
    int lo = (t < 2) ? (b & 15) : (b >> 4);
    int hi = (qh[32 * h + l] >> (2 * t)) & 3;
    q[i] = (uint8_t)(lo | (hi << 4));
  }
}

static void dequant_q6k_block(const uint8_t* blk, double* out) {
  int sc[16];
  uint8_t q[QK];
  orc_q6k_fields(blk, sc, q);
  double d = f16_to_f64(rd16(blk + 208));
  for (int i = 0; i < QK; ++i) {
    int g = 8 * (i / 128) + (i % 128) / 16;
    out[i] = d * sc[g] * ((int)q[i] - 32);
  }
}

static int block_bytes(int type) {
  return type == TYPE_Q4_K ? Q4K_BYTES : type == TYPE_Q6_K ? Q6K_BYTES : 0;
}

/* Decode `nblocks` consecutive super-blocks to f64 (256 values each). */
int orc_dequant(int type, const uint8_t* blocks, int64_t nblocks, double* out) {
  int bb = block_bytes(type);
  if (!bb) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    if (type == TYPE_Q4_K)
      dequant_q4k_block(blocks + b * bb, out + b * QK);
    else
      dequant_q6k_block(blocks + b * bb, out + b * QK);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Q8_K activation quantization, one row of k values at a time, per 256:
 *   amax = max |x|;  if amax == 0: d = 0, q = 0;
 *   else iscale = 127 / amax (f32 division), q = clamp(rint(x * iscale),
 *   -127, 127) with a single f32 multiply and round-half-even, d = amax / 127.
 *   bsum[g] = sum of the 16 codes of group g (exact integer).
 * Development plan, "Compute design", fixes the format (8-bit codes, a single
 * f32 scale for each 256 values, integer sums for each 16) but not the
 * rounding rule; the symmetric 127/amax rule above is this build's reading.
 * ------------------------------------------------------------------------- */
void orc_quantize_q8k(const float* x, int64_t rows, int64_t k, int64_t ldx,
                      int8_t* q, float* d, int16_t* bsum) {
  int64_t nsb = k / QK;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nsb; ++b) {
      const float* xb = x + r * ldx + b * QK;
      int8_t* qb = q + r * k + b * QK;
      float amax = 0.0f;
      for (int i = 0; i < QK; ++i) {
        float a = fabsf(xb[i]);
        if (a > amax) amax = a;
      }
      if (amax == 0.0f) {
        for (int i = 0; i < QK; ++i) qb[i] = 0;
        d[r * nsb + b] = 0.0f;
      } else {
        volatile float iscale = 127.0f / amax;
        for (int i = 0; i < QK; ++i) {
          volatile float v = xb[i] * iscale;
          float rv = rintf(v);
          if (rv > 127.0f) rv = 127.0f;
          if (rv < -127.0f) rv = -127.0f;
          qb[i] = (int8_t)rv;
        }
        d[r * nsb + b] = amax / 127.0f;
      }
      for (int g = 0; g < 16; ++g) {
        int s = 0;
        for (int i = 0; i < 16; ++i) s += qb[16 * g + i];
        bsum[r * (k / 16) + b * 16 + g] = (int16_t)s;
      }
    }
  }
}

/* RMSNorm (f64): out = x / sqrt(mean(x^2) + eps) * w.  w may be NULL (= 1). */
void orc_rmsnorm(const double* x, int64_t rows, int64_t k, const float* w, double eps, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + r * k;
    double ss = 0.0;
    for (int64_t i = 0; i < k; ++i) ss += xr[i] * xr[i];
    double rstd = 1.0 / sqrt(ss / (double)k + eps);
    for (int64_t i = 0; i < k; ++i) out[r * k + i] = xr[i] * rstd * (w ? (double)w[i] : 1.0);
  }
}

/* ---------------------------------------------------------------------------
 * Quantized GEMM, plain definition:
 *   y[m][nsel] = sum_k W[n][k] * (d[m][k/256] * q[m][k])
 * with W decoded exactly and the sum taken in f64 in k order. `rows` lists
 * the weight rows n to compute (NULL = all n rows, nsel = n).
 * ------------------------------------------------------------------------- */
int orc_qgemm_rows(int type, const uint8_t* wblocks, int64_t n, int64_t k,
                   const int8_t* q, const float* d, int64_t m,
                   const int64_t* rows, int64_t nsel, double* y) {
  int bb = block_bytes(type);
  if (!bb || k % QK) return -1;
  int64_t nsb = k / QK;
  if (!rows) nsel = n;
  double* at = (double*)malloc(sizeof(double) * (size_t)(k * m)); /* at[kk][mm] */
  if (!at) return -2;
  for (int64_t mm = 0; mm < m; ++mm)
    for (int64_t kk = 0; kk < k; ++kk) at[kk * m + mm] = (double)d[mm * nsb + kk / QK] * (double)q[mm * k + kk];
  int err = 0;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    double* acc = (double*)malloc(sizeof(double) * (size_t)m);
    if (!w || !acc) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int64_t s = 0; s < nsel; ++s) {
        int64_t nn = rows ? rows[s] : s;
        for (int64_t b = 0; b < nsb; ++b) {
          const uint8_t* blk = wblocks + (nn * nsb + b) * bb;
          if (type == TYPE_Q4_K)
            dequant_q4k_block(blk, w + b * QK);
          else
            dequant_q6k_block(blk, w + b * QK);
        }
        for (int64_t mm = 0; mm < m; ++mm) acc[mm] = 0.0;
        for (int64_t kk = 0; kk < k; ++kk) {
          double wv = w[kk];
          const double* a = at + kk * m;
          for (int64_t mm = 0; mm < m; ++mm) acc[mm] += wv * a[mm];
        }
        for (int64_t mm = 0; mm < m; ++mm) y[mm * nsel + s] = acc[mm];
      }
    }
    free(w);
    free(acc);
  }
  free(at);
  return err;
}

int orc_qgemm(int type, const uint8_t* wblocks, int64_t n, int64_t k,
              const int8_t* q, const float* d, int64_t m, double* y) {
  return orc_qgemm_rows(type, wblocks, n, k, q, d, m, NULL, n, y);
}

/* ---------------------------------------------------------------------------
 * The method's integer sums per (token m, weight row n, super-block sb), in
 * the unified decoded form "unsigned byte u, per-16 integer scale S, per-16
 * f32 offset O" (w = d * S_g * u - O_g):
 *   U = sum_g S_g * sum_{i in g} u_i * a_i           (the integer dot)
 *   J = sum_g T_g * bsum16_g                          (the offset's integer)
 * Q4_K: S_g = scale_{g/2}, u = q4, O_g = dmin * min_{g/2}, T_g = min_{g/2};
 *       block value = d * U - dmin * J.
 * Q6_K: S_g = scale_g (int8), u = q6 in [0,63], O_g = 32 * d * scale_g,
 *       T_g = scale_g;  block value = d * (U - 32 * J).
 * Output layout: U[m][n][nsb], J[m][n][nsb] (int64).
 * ------------------------------------------------------------------------- */
int orc_qgemm_intsums(int type, const uint8_t* wblocks, int64_t n, int64_t k,
                      const int8_t* q, int64_t m, int64_t* U, int64_t* J) {
  int bb = block_bytes(type);
  if (!bb || k % QK) return -1;
  int64_t nsb = k / QK;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t nn = 0; nn < n; ++nn) {
    for (int64_t b = 0; b < nsb; ++b) {
      const uint8_t* blk = wblocks + (nn * nsb + b) * bb;
      int S[16], T[16];
      uint8_t u[QK];
      if (type == TYPE_Q4_K) {
        int sc[8], mn[8];
        orc_q4k_fields(blk, sc, mn, u);
        for (int g = 0; g < 16; ++g) {
          S[g] = sc[g / 2];
          T[g] = mn[g / 2];
        }
      } else {
        orc_q6k_fields(blk, S, u);
        for (int g = 0; g < 16; ++g) T[g] = S[g];
      }
      for (int64_t mm = 0; mm < m; ++mm) {
        const int8_t* a = q + mm * k + b * QK;
        int64_t su = 0, sj = 0;
        for (int g = 0; g < 16; ++g) {
          int64_t dot = 0, bs = 0;
          for (int i = 0; i < 16; ++i) {
            dot += (int64_t)u[16 * g + i] * a[16 * g + i];
            bs += a[16 * g + i];
          }
          su += (int64_t)S[g] * dot;
          sj += (int64_t)T[g] * bs;
        }
        U[(mm * n + nn) * nsb + b] = su;
        J[(mm * n + nn) * nsb + b] = sj;
      }
    }
  }
  return 0;
}

/* Per-block f64 scale factors for composing y from the integer sums:
 * Q4_K: c0 = d, c1 = dmin (value = c0*U - c1*J); Q6_K: c0 = d, c1 = 32*d. */
int orc_block_scales(int type, const uint8_t* blocks, int64_t nblocks, double* c0, double* c1) {
  int bb = block_bytes(type);
  if (!bb) return -1;
  for (int64_t b = 0; b < nblocks; ++b) {
    const uint8_t* blk = blocks + b * bb;
    if (type == TYPE_Q4_K) {
      c0[b] = f16_to_f64(rd16(blk));
      c1[b] = f16_to_f64(rd16(blk + 2));
    } else {
      c0[b] = f16_to_f64(rd16(blk + 208));
      c1[b] = 32.0 * c0[b];
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * RoPE, adjacent-pair ("NORM") form, in place on x[L][nh*hd] (f64):
 * position of row p is p; pair i of each head rotates (x[2i], x[2i+1]) by
 * angle p * theta^(-2i/hd).
 * ------------------------------------------------------------------------- */
void orc_rope(double* x, int64_t L, int64_t nh, int64_t hd, double theta) {
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < L; ++p) {
    for (int64_t h = 0; h < nh; ++h) {
      double* v = x + p * nh * hd + h * hd;
      for (int64_t i = 0; i < hd / 2; ++i) {
        double ang = (double)p * pow(theta, -2.0 * (double)i / (double)hd);
        double c = cos(ang), s = sin(ang);
        double x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * c - x1 * s;
        v[2 * i + 1] = x0 * s + x1 * c;
      }
    }
  }
}

/* Non-causal multi-head attention (f64): o = softmax(q k^T / sqrt(hd)) v per head. */
void orc_attention(const double* q, const double* k, const double* v, int64_t L, int64_t nh,
                   int64_t hd, double* o) {
  int64_t dm = nh * hd;
  double scale = 1.0 / sqrt((double)hd);
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
#pragma omp for collapse(2) schedule(static)
    for (int64_t h = 0; h < nh; ++h) {
      for (int64_t i = 0; i < L; ++i) {
        double mx = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
          double acc = 0.0;
          for (int64_t e = 0; e < hd; ++e) acc += q[i * dm + h * hd + e] * k[j * dm + h * hd + e];
          s[j] = acc * scale;
          if (s[j] > mx) mx = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          s[j] = exp(s[j] - mx);
          den += s[j];
        }
        for (int64_t e = 0; e < hd; ++e) {
          double acc = 0.0;
          for (int64_t j = 0; j < L; ++j) acc += s[j] * v[j * dm + h * hd + e];
          o[i * dm + h * hd + e] = acc / den;
        }
      }
    }
    free(s);
  }
}

/* SwiGLU (f64): h = silu(g) * u, silu(g) = g / (1 + exp(-g)). */
void orc_swiglu(const double* g, const double* u, int64_t n, double* h) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* Token embedding: x[p] = decoded row ids[p] of a Q4_K table [vocab][d] (f64). */
int orc_embed_q4k(const uint8_t* table, int64_t vocab, int64_t d, const int32_t* ids, int64_t L,
                  double* x) {
  int64_t nsb = d / QK;
  for (int64_t p = 0; p < L; ++p)
    if (ids[p] < 0 || ids[p] >= vocab) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < L; ++p)
    for (int64_t b = 0; b < nsb; ++b)
      dequant_q4k_block(table + ((int64_t)ids[p] * nsb + b) * Q4K_BYTES, x + p * d + b * QK);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Softmax confidence over one row of logits (f64):
 *   id = argmax (lowest id on ties), conf = softmax(l)[id] = 1 / sum_v exp(l_v - l_max).
 * Also reports the runner-up logit for margin diagnostics.
 * ------------------------------------------------------------------------- */
void orc_row_confidence(const double* logits, int64_t rows, int64_t vocab,
                        int32_t* id, double* conf, double* top1, double* top2) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* l = logits + r * vocab;
    int64_t best = 0;
    double b1 = l[0], b2 = -INFINITY;
    for (int64_t v = 1; v < vocab; ++v) {
      if (l[v] > b1) {
        b2 = b1;
        b1 = l[v];
        best = v;
      } else if (l[v] > b2) {
        b2 = l[v];
      }
    }
    double den = 0.0;
    for (int64_t v = 0; v < vocab; ++v) den += exp(l[v] - b1);
    id[r] = (int32_t)best;
    conf[r] = 1.0 / den;
    if (top1) top1[r] = b1;
    if (top2) top2[r] = b2;
  }
}

/* ---------------------------------------------------------------------------
 * Entropy of the softmax of one row of logits (f64, natural log), straight
 * from its definition: p_v = exp(l_v) / sum_u exp(l_u) (computed with the row
 * maximum subtracted, which leaves p unchanged), H = -sum_v p_v log p_v, with
 * 0 log 0 = 0. neg_entropy[r] = -H is the confidence of the entropy ranking
 * (README, "Each model's own sampler": Dream's entropy ranking).
 * ------------------------------------------------------------------------- */
void orc_row_neg_entropy(const double* logits, int64_t rows, int64_t vocab, double* neg_entropy) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* l = logits + r * vocab;
    double mx = l[0];
    for (int64_t v = 1; v < vocab; ++v)
      if (l[v] > mx) mx = l[v];
    double den = 0.0;
    for (int64_t v = 0; v < vocab; ++v) den += exp(l[v] - mx);
    double h = 0.0;
    for (int64_t v = 0; v < vocab; ++v) {
      const double p = exp(l[v] - mx) / den;
      if (p > 0.0) h -= p * log(p);
    }
    neg_entropy[r] = -h;
  }
}

/* ---------------------------------------------------------------------------
 * Counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014): the generator adds the
 * golden-ratio increment 0x9E3779B97F4A7C15 to its state and returns the
 * state through a 64-bit finalizer (xor-shift 30, multiply by
 * 0xBF58476D1CE4E5B9, xor-shift 27, multiply by 0x94D049BB133111EB,
 * xor-shift 31). Output number c (from 0) of the stream started at `seed`
 * therefore depends on (seed, c) alone: mix(seed + (c + 1) * increment).
 * ------------------------------------------------------------------------- */
uint64_t orc_splitmix64_at(uint64_t seed, uint64_t c) {
  uint64_t z = seed + (c + 1) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* ---------------------------------------------------------------------------
 * Temperature sampling (specification, section 14: temperature, categorical
 * sampling, deterministic PRNG) by the Gumbel-max rule: the draw
 * argmax_v (l_v / T + g_v) with independent standard Gumbel g_v is
 * distributed as softmax(l / T). g_v = -log(-log u_v), u_v uniform in (0, 1)
 * from the top 23 bits of SplitMix64 output number
 * c = step * 2^40 + position * 2^24 + v: u = (bits + 1/2) / 2^23. Per row:
 * the drawn id (lowest on ties), its probability under the untempered
 * softmax, exp(l_id - l_max) / sum_v exp(l_v - l_max), and the gap between
 * the best and second-best perturbed scores (a diagnostic). f64 throughout.
 * ------------------------------------------------------------------------- */
void orc_row_sample(const double* logits, int64_t rows, int64_t vocab, double temperature, uint64_t seed,
                    uint32_t step, const int64_t* pos, int32_t* id, double* conf, double* gap) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* l = logits + r * vocab;
    int64_t best = -1;
    double s1 = -INFINITY, s2 = -INFINITY, mx = -INFINITY;
    for (int64_t v = 0; v < vocab; ++v) {
      const uint64_t c = ((uint64_t)step << 40) | ((uint64_t)pos[r] << 24) | (uint64_t)v;
      const double u = ((double)(orc_splitmix64_at(seed, c) >> 41) + 0.5) / 8388608.0;
      const double score = l[v] / temperature - log(-log(u));
      if (score > s1) {
        s2 = s1;
        s1 = score;
        best = v;
      } else if (score > s2) {
        s2 = score;
      }
      if (l[v] > mx) mx = l[v];
    }
    double den = 0.0;
    for (int64_t v = 0; v < vocab; ++v) den += exp(l[v] - mx);
    id[r] = (int32_t)best;
    conf[r] = exp(l[best] - mx) / den;
    gap[r] = s1 - s2;
  }
}

/* ---------------------------------------------------------------------------
 * Low-confidence commit (LLaDA, greedy): among positions p in [b0, b1) with
 * canvas[p] == mask_id, take the k with the highest confidence (ties: lowest
 * position), write their ids into the canvas. `conf`/`ids` are indexed by
 * position (only masked entries inside the block are read). Outputs the
 * chosen positions in selection order (descending confidence). Returns the
 * number committed (min(k, masked count)).
 * ------------------------------------------------------------------------- */
int orc_commit_topk(int32_t* canvas, int64_t L, int32_t mask_id, int64_t b0, int64_t b1,
                    const double* conf, const int32_t* ids, int64_t k,
                    int32_t* out_pos, int32_t* out_id) {
  if (b0 < 0 || b1 > L || b0 > b1) return -1;
  char* taken = (char*)calloc((size_t)(b1 - b0 + 1), 1);
  int n = 0;
  for (int64_t step = 0; step < k; ++step) {
    int64_t best = -1;
    for (int64_t p = b0; p < b1; ++p) {
      if (canvas[p] != mask_id || taken[p - b0]) continue;
      if (best < 0 || conf[p] > conf[best]) best = p;
    }
    if (best < 0) break;
    taken[best - b0] = 1;
    out_pos[n] = (int32_t)best;
    out_id[n] = ids[best];
    ++n;
  }
  for (int i = 0; i < n; ++i) canvas[out_pos[i]] = out_id[i];
  free(taken);
  return n;
}

/* Tokens committed at each of `steps` steps for `masked` masked positions:
 * floor(masked / steps) each, the remainder going to the earliest steps. */
void orc_transfer_counts(int64_t masked, int64_t steps, int64_t* counts) {
  int64_t base = masked / steps, rem = masked % steps;
  for (int64_t s = 0; s < steps; ++s) counts[s] = base + (s < rem ? 1 : 0);
}
