/*
 * CPU oracle for the fused SwiGLU up-projection.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm may load this library.  The CUDA library never links, includes or calls
 * it, and this file includes nothing from the CUDA side: its bf16 codec, its
 * silu and its loops are its own.
 *
 * What it computes (plain definitions, fp64 throughout):
 *
 *   "Tile-Level Activation Overlap for Efficient LLM Inference", technical
 *   summary, section "Enonce du probleme": Y = SiLU(A x W1) (.) (A x W2),
 *   two independent GEMMs followed by an element-wise product.  Here
 *   A = x [M, d], W1 = W_gate [d, d_ff], W2 = W_up [d, d_ff], Y = h [M, d_ff].
 *
 *   "1 . Anatomie d'un transformeur sur GPU", section 1.1 (the layer skeleton,
 *   "Wgate, Wup -> SwiGLU") and section 1.2 (each projection is a
 *   (bS x d).(d x d') GEMM; gate and up cost 2 bS d d_ff FLOP each).
 *
 *   "Ou part le temps d'un token", section "Un kernel pour les matrices
 *   etroites": the weight b is indexed (k)*cols + col, i.e. row-major
 *   [K, N] with N contiguous.  The same section states the comparison rule
 *   (tolerance scaled by |a|.|b|), which is why this oracle also returns the
 *   first-order sensitivity s of each output to accumulation error.
 *
 * Readings taken where the pages are silent:
 *   - SiLU(z) = z * sigma(z) = z / (1 + exp(-z))  (Swish with beta = 1).
 *   - SiLU applies to x.W_gate; x.W_up enters linearly.
 *   - g and u are never rounded; only h is rounded (round-to-nearest-even)
 *     to the output type.
 *
 * Every product of two bf16 (8-bit significand) or two f32 (24-bit) values is
 * exact in fp64 (53-bit significand); each sum runs over k in ascending order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2   /* operands already dequantized to fp64 (the FP8 path) */

/* ---- number formats ---------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE-754 binary32 value. */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static uint16_t f32_bits_hi(float f) {
  uint32_t w;
  memcpy(&w, &f, sizeof w);
  return (uint16_t)(w >> 16);
}

/*
 * Round an fp64 value straight to bf16, to nearest, ties to even (one
 * rounding: no intermediate f32).  bf16 keeps 8 significant bits with the
 * binary32 exponent range; below 2^-126 the spacing is fixed at 2^-133.
 */
uint16_t oracle_f64_to_bf16(double v) {
  if (isnan(v)) return (uint16_t)0x7FC0;
  uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int ex;
  frexp(a, &ex);          /* a = m * 2^ex, m in [0.5, 1): a in [2^(ex-1), 2^ex) */
  int e = ex - 1;         /* a in [2^e, 2^(e+1)) */
  int q = (e < -126) ? -133 : e - 7; /* exponent of one unit in the last place */
  double n = nearbyint(ldexp(a, -q)); /* exact scaling; default mode is RNE */
  double r = ldexp(n, q);
  const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (r > bf16_max) return (uint16_t)(sign | 0x7F80);
  /* r now has at most 8 significant bits inside the binary32 range, so the
     conversion to float is exact and the bf16 pattern is its upper half. */
  return (uint16_t)(sign | (f32_bits_hi((float)r) & 0x7FFF));
}

static double load_elem(const void* p, int64_t idx, int dtype) {
  if (dtype == ORACLE_BF16) return oracle_bf16_to_f64(((const uint16_t*)p)[idx]);
  if (dtype == ORACLE_F64) return ((const double*)p)[idx];
  return (double)((const float*)p)[idx];
}

static void store_elem(void* p, int64_t idx, int dtype, double v) {
  if (dtype == ORACLE_BF16)
    ((uint16_t*)p)[idx] = oracle_f64_to_bf16(v);
  else if (dtype == ORACLE_F64)
    ((double*)p)[idx] = v;
  else
    ((float*)p)[idx] = (float)v; /* C conversion: round to nearest even */
}

/* ---- activation -------------------------------------------------------- */

/* SiLU(z) = z * sigma(z) = z / (1 + e^-z).  For z -> -inf the quotient
   tends to -0 (e^-z overflows to +inf), never NaN. */
double oracle_silu64(double z) { return z / (1.0 + exp(-z)); }

/* ---- fused definition ---------------------------------------------------- */

typedef struct {
  const void *x, *wg, *wu;
  int64_t M, d, d_ff, j0, j1;
  int dtype;
  double *h64, *sens;
  void* h_out;
  int status;
} job_t;

/*
 * For one block of output columns [j0, j1): for every row i, accumulate
 * g = sum_k x[i,k] Wg[k,j] and u = sum_k x[i,k] Wu[k,j] with k ascending
 * (the k loop runs outside the j loop only so that W is read along its
 * contiguous rows; each element's sum still adds its terms in k order),
 * then h = silu(g) * u.
 *
 * s = 1.1 * G * |u| + |silu(g)| * U, with G = sum_k |x||Wg| and
 * U = sum_k |x||Wu|, bounds to first order how much h moves per unit of
 * relative accumulation error in g and u (|silu'| <= 1.0999 everywhere).
 */
static void* fused_block(void* arg) {
  job_t* jb = (job_t*)arg;
  int64_t n = jb->j1 - jb->j0;
  if (n <= 0) return NULL;
  double* acc = (double*)malloc((size_t)n * 4 * sizeof(double));
  if (!acc) { jb->status = 1; return NULL; }
  double *g = acc, *u = acc + n, *G = acc + 2 * n, *U = acc + 3 * n;
  for (int64_t i = 0; i < jb->M; ++i) {
    memset(acc, 0, (size_t)n * 4 * sizeof(double));
    for (int64_t k = 0; k < jb->d; ++k) {
      double xv = load_elem(jb->x, i * jb->d + k, jb->dtype);
      double ax = fabs(xv);
      int64_t row = k * jb->d_ff + jb->j0;
      for (int64_t t = 0; t < n; ++t) {
        double wgv = load_elem(jb->wg, row + t, jb->dtype);
        double wuv = load_elem(jb->wu, row + t, jb->dtype);
        g[t] += xv * wgv;
        u[t] += xv * wuv;
        G[t] += ax * fabs(wgv);
        U[t] += ax * fabs(wuv);
      }
    }
    for (int64_t t = 0; t < n; ++t) {
      double sg = oracle_silu64(g[t]);
      double hv = sg * u[t];
      int64_t o = i * jb->d_ff + jb->j0 + t;
      if (jb->h64) jb->h64[o] = hv;
      if (jb->sens) jb->sens[o] = 1.1 * G[t] * fabs(u[t]) + fabs(sg) * U[t];
      if (jb->h_out) store_elem(jb->h_out, o, jb->dtype, hv);
    }
  }
  free(acc);
  return NULL;
}

/*
 * h = silu(x . Wg) (.) (x . Wu) for all M x d_ff outputs.
 *   x [M, d], Wg/Wu [d, d_ff], row-major, element type `dtype` (0 f32, 1 bf16).
 *   h64  [M, d_ff] fp64 exact-input result (may be NULL)
 *   h_out [M, d_ff] in `dtype`, RNE of h64 (may be NULL)
 *   sens [M, d_ff] sensitivity s defined above (may be NULL)
 * Column blocks are split across `nthreads` POSIX threads; the arithmetic of
 * each output does not depend on the split.  Returns 0 on success.
 */
int oracle_swiglu_up(const void* x, const void* wg, const void* wu, int64_t M,
                     int64_t d, int64_t d_ff, int dtype, double* h64,
                     void* h_out, double* sens, int nthreads) {
  if (M < 0 || d < 0 || d_ff < 0) return 2;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return 2;
  if (M == 0 || d_ff == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > d_ff) nthreads = (int)d_ff;
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 1; }
  for (int t = 0; t < nthreads; ++t) {
    job_t* jb = &jobs[t];
    jb->x = x; jb->wg = wg; jb->wu = wu;
    jb->M = M; jb->d = d; jb->d_ff = d_ff; jb->dtype = dtype;
    jb->j0 = d_ff * t / nthreads;
    jb->j1 = d_ff * (t + 1) / nthreads;
    jb->h64 = h64; jb->sens = sens; jb->h_out = h_out;
  }
  int rc = 0;
  if (nthreads == 1) {
    fused_block(&jobs[0]);
  } else {
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
      if (pthread_create(&th[t], NULL, fused_block, &jobs[t]) != 0) { rc = 1; break; }
      ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  }
  for (int t = 0; t < nthreads; ++t) rc |= jobs[t].status;
  free(jobs);
  free(th);
  return rc;
}

/*
 * The same definition evaluated only at n chosen outputs (rows[t], cols[t]),
 * one k loop per output.  Used for full-size shapes, where every row of h is
 * independent of the others and each output needs only one row of x and one
 * column of each weight.
 */
int oracle_swiglu_up_at(const void* x, const void* wg, const void* wu, int64_t M,
                        int64_t d, int64_t d_ff, int dtype, const int64_t* rows,
                        const int64_t* cols, int64_t n, double* h64,
                        double* sens) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return 2;
  for (int64_t t = 0; t < n; ++t) {
    int64_t i = rows[t], j = cols[t];
    if (i < 0 || i >= M || j < 0 || j >= d_ff) return 2;
    double g = 0, u = 0, G = 0, U = 0;
    for (int64_t k = 0; k < d; ++k) {
      double xv = load_elem(x, i * d + k, dtype);
      double wgv = load_elem(wg, k * d_ff + j, dtype);
      double wuv = load_elem(wu, k * d_ff + j, dtype);
      g += xv * wgv;
      u += xv * wuv;
      G += fabs(xv) * fabs(wgv);
      U += fabs(xv) * fabs(wuv);
    }
    double sg = oracle_silu64(g);
    h64[t] = sg * u;
    if (sens) sens[t] = 1.1 * G * fabs(u) + fabs(sg) * U;
  }
  return 0;
}

/* ---- unfused composition (the pages' baseline, without its bf16 rounding) */

/* out[i, j] = sum_k a[i, k] * b[k, j], fp64, k ascending.  a [m, kd], b [kd, n]. */
int oracle_gemm64(const void* a, const void* b, int64_t m, int64_t kd, int64_t n,
                  int dtype, double* out) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 2;
  for (int64_t i = 0; i < m; ++i) {
    double* o = out + i * n;
    for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
    for (int64_t k = 0; k < kd; ++k) {
      double av = load_elem(a, i * kd + k, dtype);
      for (int64_t j = 0; j < n; ++j) o[j] += av * load_elem(b, k * n + j, dtype);
    }
  }
  return 0;
}

/* h[t] = silu(g[t]) * u[t] over n elements. */
void oracle_silu_mul64(const double* g, const double* u, int64_t n, double* h) {
  for (int64_t t = 0; t < n; ++t) h[t] = oracle_silu64(g[t]) * u[t];
}

/* Round n fp64 values to `dtype` (RNE), writing the raw output elements. */
int oracle_round_to_dtype(const double* v, int64_t n, int dtype, void* out) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 2;
  for (int64_t t = 0; t < n; ++t) store_elem(out, t, dtype, v[t]);
  return 0;
}

/* ---- down projection (the MLP's second GEMM, plus the residual) --------- */

/*
 * y = h . W_down (+ r): "1 . Anatomie d'un transformeur sur GPU", section 1.2
 * (W_down is a d_ff x d projection, 2 bS d d_ff FLOP) and section 1.6
 * (kernel #10 "GEMM down", kernel #11 the residual addition).
 *   h [M, K] (K = d_ff), wd [K, N] (N = d) row-major, r [M, N] or NULL.
 *   y64 [M, N] fp64 (k ascending, then + r), y_out rounded to `dtype`
 *   (may be NULL), sens [M, N] = sum_k |h||wd| + |r| (may be NULL): the
 *   first-order sensitivity of y to relative accumulation error.
 */
int oracle_down_proj(const void* h, const void* wd, const void* r, int64_t M, int64_t K,
                     int64_t N, int dtype, double* y64, void* y_out, double* sens) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return 2;
  if (M < 0 || K < 0 || N < 0) return 2;
  double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * 2 * sizeof(double));
  if (!acc) return 1;
  double* S = acc + N;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) acc[j] = S[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double hv = load_elem(h, i * K + k, dtype);
      double ah = fabs(hv);
      for (int64_t j = 0; j < N; ++j) {
        double wv = load_elem(wd, k * N + j, dtype);
        acc[j] += hv * wv;
        S[j] += ah * fabs(wv);
      }
    }
    for (int64_t j = 0; j < N; ++j) {
      double v = acc[j], s = S[j];
      if (r) {
        double rv = load_elem(r, i * N + j, dtype);
        v += rv;
        s += fabs(rv);
      }
      int64_t o = i * N + j;
      if (y64) y64[o] = v;
      if (sens) sens[o] = s;
      if (y_out) store_elem(y_out, o, dtype, v);
    }
  }
  free(acc);
  return 0;
}

/* ---- weight packing (step a0) ------------------------------------------- */

/*
 * "Tile-Level Activation Overlap for Efficient LLM Inference", Kernel-2:
 * the gate and up weight columns are interleaved once, before any GEMM, so
 * that one tile of the packed matrix holds matching gate and up columns.
 * The interleave unit here is a block of 64 columns.  With
 * P = ceil(d_ff / 64) * 64, packed row k (2P elements) is
 *     Wg[k, 0:64] | Wu[k, 0:64] | Wg[k, 64:128] | Wu[k, 64:128] | ...
 * and an element whose column j = 64 t + i is >= d_ff is zero.  The packing
 * is a copy of element bits: nothing is rounded.
 *   wg, wu  [d, d_ff] row-major, element type `dtype`
 *   packed  [d, 2P], same element type
 * Returns 0 on success.
 */
int oracle_pack(const void* wg, const void* wu, int64_t d, int64_t d_ff, int dtype,
                void* packed) {
  if (d < 0 || d_ff < 0) return 2;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return 2;
  const size_t es = dtype == ORACLE_BF16 ? 2 : 4;
  const int64_t tiles = (d_ff + 63) / 64, width = 2 * 64 * tiles;
  const unsigned char* g = (const unsigned char*)wg;
  const unsigned char* u = (const unsigned char*)wu;
  unsigned char* out = (unsigned char*)packed;
  for (int64_t k = 0; k < d; ++k) {
    for (int64_t t = 0; t < tiles; ++t) {
      for (int64_t i = 0; i < 64; ++i) {
        const int64_t j = 64 * t + i;
        unsigned char* dg = out + ((size_t)(k * width + 128 * t + i)) * es;
        unsigned char* du = out + ((size_t)(k * width + 128 * t + 64 + i)) * es;
        if (j < d_ff) {
          memcpy(dg, g + (size_t)(k * d_ff + j) * es, es);
          memcpy(du, u + (size_t)(k * d_ff + j) * es, es);
        } else {
          memset(dg, 0, es);
          memset(du, 0, es);
        }
      }
    }
  }
  return 0;
}

/* ---- FP8 (e4m3) weights and activations ---------------------------------- */

/*
 * The e4m3 format (the "FP8 E4M3" of the OCP 8-bit floating-point
 * specification, the type tcgen05 kind::f8f6f4 reads as E4M3): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits, no infinities.  Code
 * s.eeee.mmm is (-1)^s (1 + m/8) 2^(e-7) for e >= 1, (-1)^s (m/8) 2^-6 for
 * e = 0, and NaN for e = 15, m = 7; the largest finite magnitude is 448.
 */
double oracle_e4m3_decode(uint8_t c) {
  const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return sgn ? -v : v;
}

/* Round-half-to-even of a non-negative double that holds few bits (exact). */
static double rne_nonneg(double q) {
  const double n = floor(q), r = q - n;
  if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) != 0.0)) return n + 1.0;
  return n;
}

/*
 * f32 -> e4m3, round to nearest (ties to even), finite results saturated to
 * +-448 (values past the largest finite magnitude, which would round to the
 * NaN pattern or beyond, become +-448); NaN -> 0x7F.
 */
uint8_t oracle_e4m3_encode(float f) {
  if (isnan(f)) return 0x7F;
  const uint8_t sgn = signbit(f) ? 0x80 : 0x00;
  const double a = fabs((double)f);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; rounding up to 8 gives the
       smallest normal, code 0x08 */
    const double n = rne_nonneg(ldexp(a, 9));
    return (uint8_t)(sgn | (uint8_t)n);
  }
  int ex = 0;
  (void)frexp(a, &ex);          /* a = fr 2^ex, fr in [0.5, 1) */
  int E = ex - 1;                /* a in [2^E, 2^(E+1)) */
  double n = rne_nonneg((ldexp(a, -E) - 1.0) * 8.0);
  if (n == 8.0) { n = 0.0; ++E; }
  const int biased = E + 7;
  if (biased > 15 || (biased == 15 && n == 7.0)) return (uint8_t)(sgn | 0x7E);
  return (uint8_t)(sgn | (biased << 3) | (int)n);
}

/* amax -> (multiplier 448 / amax, dequantization scale amax / 448), both in
   f32 arithmetic; an all-zero vector gets 0 and 0. */
static void e4m3_scale(float amax, float* inv, float* scale) {
  *inv = amax > 0.0f ? 448.0f / amax : 0.0f;
  *scale = amax > 0.0f ? amax / 448.0f : 0.0f;
}

/*
 * Per-row e4m3 quantization of a bf16 [R, K] matrix (the activations x):
 * for each row, amax = max |a| (exact in f32), then every element's code is
 * e4m3(f32(a) * (448 / amax)) with the product rounded to f32 first, and the
 * row's dequantization scale is amax / 448 (f32).
 *   codes [R, K], scales [R]
 */
int oracle_quantize_rows_e4m3(const uint16_t* a, int64_t R, int64_t K, uint8_t* codes,
                              float* scales) {
  if (R < 0 || K < 0) return 2;
  for (int64_t r = 0; r < R; ++r) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = fabsf((float)oracle_bf16_to_f64(a[r * K + k]));
      if (v > amax) amax = v;
    }
    float inv, sc;
    e4m3_scale(amax, &inv, &sc);
    for (int64_t k = 0; k < K; ++k) {
      const float v = (float)oracle_bf16_to_f64(a[r * K + k]);
      const float q = v * inv;
      codes[r * K + k] = oracle_e4m3_encode(q);
    }
    scales[r] = sc;
  }
  return 0;
}

/*
 * Per-column e4m3 quantization of a bf16 [K, N] weight matrix, as the rows
 * above but over each column j, with the codes written transposed:
 *   codes_nk [N, K] (code of w[k, j] at j * K + k), scales [N]
 */
int oracle_quantize_cols_e4m3(const uint16_t* w, int64_t K, int64_t N, uint8_t* codes_nk,
                              float* scales) {
  if (K < 0 || N < 0) return 2;
  for (int64_t j = 0; j < N; ++j) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = fabsf((float)oracle_bf16_to_f64(w[k * N + j]));
      if (v > amax) amax = v;
    }
    float inv, sc;
    e4m3_scale(amax, &inv, &sc);
    for (int64_t k = 0; k < K; ++k) {
      const float v = (float)oracle_bf16_to_f64(w[k * N + j]);
      const float q = v * inv;
      codes_nk[j * K + k] = oracle_e4m3_encode(q);
    }
    scales[j] = sc;
  }
  return 0;
}

/* out[r, k] = decode(codes[r, k]) * scales[r], exactly (a 4-bit significand
   times a 24-bit one fits a double). */
int oracle_dequant_rows_e4m3(const uint8_t* codes, const float* scales, int64_t R, int64_t K,
                             double* out) {
  if (R < 0 || K < 0) return 2;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = oracle_e4m3_decode(codes[r * K + k]) * (double)scales[r];
  return 0;
}

