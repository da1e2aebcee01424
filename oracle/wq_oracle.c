/*
 * wq_oracle.c -- plain, slow CPU oracle for the group-wise symmetric
 * weight-only quantized GEMM  Y[M,N] = X[M,K] . dequant(Wq)[K,N].
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA library (w4a16_weight_only_wq_gb300/csrc); the packed
 * word layout is re-derived here from its written definition.
 *
 * What the method computes, and where it is stated:
 *  - "Quantize the Target, Quantize the Drafter" (arXiv 2607.04244 HTML),
 *    QAD paragraph: the student's weights are the dequantized weights
 *    s (.) Wq with frozen symmetric per-group scales s; packing paragraph:
 *    at packing time the updated weights are rounded back onto the same
 *    grid, giving new INT4 codes under the original scales.
 *  - same paper, drafter-PTQ paragraph: group-wise symmetric INT4 with a
 *    group size of 128.
 *  - "Qwen3.5-4B-DFlash-W8A16" model card, "What changed vs upstream" table:
 *    int8 weight-only, RTN, symmetric, group = 128, bf16 activations.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - RTN scale when none is supplied: s = bf16_rne(fp32(absmax) / qpos),
 *    qpos = 7 (INT4) or 127 (INT8); absmax == 0 gives s = 1.
 *  - code: q = clamp(rint(w / s), qmin, qmax), IEEE fp32 divide, rint =
 *    round half to even; [qmin,qmax] = [-8,7] (INT4) or [-128,127] (INT8).
 *  - bf16 weights are widened to fp32 exactly before the divide.
 *  - dequant w^ = fp32(s) * fp32(q) is exact in fp32 (<= 8 + 8 significant
 *    bits); the GEMM accumulates in fp64.
 *  - the MLP pair's intermediate (the pages name no activation): the
 *    up-projection rounded to bf16 (RNE, straight from fp64), then either
 *    kept or mapped through silu(h) = h / (1 + e^-h) in fp64 and rounded to
 *    bf16 again; the down-projection reads those bf16 values.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread.
 * Everything here is single-threaded and element-by-element, except
 * wqo_gemm_rows, which splits whole output rows over POSIX threads (the
 * arithmetic per row is unchanged).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 is the top half of an IEEE binary32 pattern. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a finite binary32 to bf16, ties to even (IEEE 754 RNE on the
   16 discarded bits). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

uint16_t wqo_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* Round a binary64 to bf16 directly (8 significant bits, ties to even, bf16
   subnormal spacing 2^-133), without passing through binary32. */
static uint16_t f64_to_bf16_rne(double x) {
  if (x == 0.0 || !isfinite(x)) return f32_to_bf16_rne((float)x);
  int e;
  frexp(x, &e);           /* |x| = m 2^e, m in [0.5, 1) */
  int q = e - 8;          /* exponent of the last kept bit */
  if (q < -133) q = -133;
  const double r = nearbyint(ldexp(x, -q));  /* default mode: ties to even */
  const float f = (float)ldexp(r, q);        /* exact: <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

void wqo_round_bf16_f64(const double* x, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = f64_to_bf16_rne(x[i]);
}

/* The MLP activation on bf16 values: silu(h) = h / (1 + e^-h) in fp64,
   rounded to bf16. */
void wqo_silu_bf16(const uint16_t* h, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) {
    const double v = (double)bf16_to_f32(h[i]);
    out[i] = f64_to_bf16_rne(v / (1.0 + exp(-v)));
  }
}
float wqo_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/* --------------------------------------------------------- code ranges -- */

static int qmin_of(int bits) { return bits == 4 ? -8 : -128; }
static int qmax_of(int bits) { return bits == 4 ? 7 : 127; }
static int qpos_of(int bits) { return bits == 4 ? 7 : 127; }

/* ------------------------------------------------------- quantization -- */

/* RTN scales: one per (group g, column n), s = bf16(absmax / qpos).
   W is fp32 [K,N] row-major; s_out is bf16 [K/group, N] row-major. */
void wqo_rtn_scales(const float* W, int64_t K, int64_t N, int group, int bits,
                    uint16_t* s_out) {
  int64_t G = K / group;
  for (int64_t g = 0; g < G; ++g) {
    for (int64_t n = 0; n < N; ++n) {
      float amax = 0.0f;
      for (int64_t kk = 0; kk < group; ++kk) {
        float a = fabsf(W[(g * group + kk) * N + n]);
        if (a > amax) amax = a;
      }
      float s = (amax == 0.0f) ? 1.0f : amax / (float)qpos_of(bits);
      s_out[g * N + n] = f32_to_bf16_rne(s);
    }
  }
}

/* Round every weight onto the grid of its group's scale:
   q = clamp(rint(w / s), qmin, qmax).  The clamp is applied to the rounded
   float before the integer conversion so that huge ratios cannot overflow. */
void wqo_quantize(const float* W, const uint16_t* s, int64_t K, int64_t N,
                  int group, int bits, int8_t* q_out) {
  float lo = (float)qmin_of(bits), hi = (float)qmax_of(bits);
  for (int64_t k = 0; k < K; ++k) {
    for (int64_t n = 0; n < N; ++n) {
      float sc = bf16_to_f32(s[(k / group) * N + n]);
      float r = rintf(W[k * N + n] / sc);
      if (r < lo) r = lo;
      if (r > hi) r = hi;
      q_out[k * N + n] = (int8_t)(int)r;
    }
  }
}

/* fp32 -> bf16 (RNE), element by element. */
void wqo_round_bf16(const float* W, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = f32_to_bf16_rne(W[i]);
}

/* bf16 weights: widen exactly to fp32, then as above. */
void wqo_widen_bf16(const uint16_t* Wh, int64_t count, float* W_out) {
  for (int64_t i = 0; i < count; ++i) W_out[i] = bf16_to_f32(Wh[i]);
}

/* ------------------------------------------------------ packed layout -- */
/*
 * The tile-interleaved word layout (group size 128, N % 64 == 0,
 * K % 128 == 0).  For the element (k, n):
 *   nt  = n / 64            64-column tile
 *   j8  = (n % 64) / 8      8-column slab inside the tile
 *   c   = n % 8             column inside the slab
 *   g   = k / 128           group
 *   kk  = k % 128
 *   kb  = kk / 32           32-deep block inside the group
 *   t4  = (kk % 32) / 8
 *   r   = kk % 8            position among the 8 consecutive k of (kb, t4)
 *   lane = 4*c + t4
 * INT4 (4 words per lane per (slab, group)):
 *   word  = kb,  nibble = r/2 + 4*(r%2),  stored value u = q + 8
 * INT8 (8 words per lane per (slab, group), stored as two halves of 4):
 *   word  = 2*kb + r/4,  byte = (r%4)/2 + 2*((r%4)%2),  u = q + 128
 * Linear word index:
 *   INT4: (((nt * (K/128) + g) * 8 + j8) * 32 + lane) * 4 + word
 *   INT8: ((((nt * (K/128) + g) * 8 + j8) * 2 + word/4) * 32 + lane) * 4
 *         + word%4
 */
static int64_t word_index(int64_t k, int64_t n, int64_t K, int bits,
                          int* shift_out) {
  int64_t nt = n / 64, j8 = (n % 64) / 8, c = n % 8;
  int64_t g = k / 128, kk = k % 128;
  int64_t kb = kk / 32, t4 = (kk % 32) / 8, r = kk % 8;
  int64_t lane = 4 * c + t4;
  int64_t slab = (nt * (K / 128) + g) * 8 + j8;
  if (bits == 4) {
    int64_t word = kb;
    *shift_out = (int)(4 * (r / 2 + 4 * (r % 2)));
    return (slab * 32 + lane) * 4 + word;
  }
  int64_t rr = r % 4;
  int64_t word = 2 * kb + r / 4;
  *shift_out = (int)(8 * (rr / 2 + 2 * (rr % 2)));
  return ((slab * 2 + word / 4) * 32 + lane) * 4 + word % 4;
}

int64_t wqo_packed_words(int bits, int64_t K, int64_t N) {
  return bits == 4 ? K * N / 8 : K * N / 4;
}

void wqo_pack(const int8_t* q, int64_t K, int64_t N, int bits,
              uint32_t* packed) {
  memset(packed, 0, (size_t)wqo_packed_words(bits, K, N) * 4);
  uint32_t mask = (bits == 4) ? 0xFu : 0xFFu;
  int off = (bits == 4) ? 8 : 128;
  for (int64_t k = 0; k < K; ++k) {
    for (int64_t n = 0; n < N; ++n) {
      int sh;
      int64_t w = word_index(k, n, K, bits, &sh);
      uint32_t u = (uint32_t)(q[k * N + n] + off) & mask;
      packed[w] |= u << sh;
    }
  }
}

void wqo_unpack(const uint32_t* packed, int64_t K, int64_t N, int bits,
                int8_t* q_out) {
  uint32_t mask = (bits == 4) ? 0xFu : 0xFFu;
  int off = (bits == 4) ? 8 : 128;
  for (int64_t k = 0; k < K; ++k) {
    for (int64_t n = 0; n < N; ++n) {
      int sh;
      int64_t w = word_index(k, n, K, bits, &sh);
      int u = (int)((packed[w] >> sh) & mask);
      q_out[k * N + n] = (int8_t)(u - off);
    }
  }
}

/* ------------------------------------------------- checkpoint import -- */

/* Read a layer stored output-channel-major with its codes packed along the
   input dimension (the serving checkpoint format of the pages' target, whose
   layout the pages do not print; this is the format's definition): word j
   of row n of `qweight` [N][K*bits/32] holds codes k = (32/bits)*j + p,
   p = 0 .. 32/bits-1, at bits [bits*p, bits*p + bits), offset-binary;
   `s_nk` is [N][K/group] bf16.  Writes canonical codes q [K,N] and scales
   s [K/group, N]. */
void wqo_import_nk(const uint32_t* qweight, const uint16_t* s_nk, int64_t K, int64_t N,
                   int group, int bits, int8_t* q, uint16_t* s) {
  int per = 32 / bits;
  int64_t row_words = K / per;
  uint32_t mask = bits == 4 ? 0xFu : 0xFFu;
  int off = bits == 4 ? 8 : 128;
  int64_t G = K / group;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < row_words; ++j) {
      uint32_t word = qweight[n * row_words + j];
      for (int p = 0; p < per; ++p) {
        int64_t k = (int64_t)per * j + p;
        int u = (int)((word >> (bits * p)) & mask);
        q[k * N + n] = (int8_t)(u - off);
      }
    }
    for (int64_t g = 0; g < G; ++g) s[g * N + n] = s_nk[n * G + g];
  }
}

/* ------------------------------------------------------------ dequant -- */

/* w^[k,n] = s[k/group, n] * q[k,n], exact in fp32. */
void wqo_dequant(const int8_t* q, const uint16_t* s, int64_t K, int64_t N,
                 int group, float* W_out) {
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n)
      W_out[k * N + n] =
          bf16_to_f32(s[(k / group) * N + n]) * (float)q[k * N + n];
}

/* --------------------------------------------------------------- GEMM -- */
/*
 * Y_ref[m,n] = sum_k X[m,k] * w^[k,n], every product and sum in fp64.
 * The weights come in packed form and are unpacked/dequantized with the
 * routines above; X is bf16 [M,K] row-major; Y is fp64 [R,N] for the R
 * requested rows (rows[i] is the row of X to use for output row i).
 */
typedef struct {
  const uint16_t* X;
  const float* What; /* dequantized [K,N] */
  const int64_t* rows;
  int64_t r0, r1, K, N;
  double* Y;
} gemm_job;

static void* gemm_worker(void* p) {
  gemm_job* j = (gemm_job*)p;
  for (int64_t i = j->r0; i < j->r1; ++i) {
    int64_t m = j->rows[i];
    double* y = j->Y + i * j->N;
    for (int64_t n = 0; n < j->N; ++n) y[n] = 0.0;
    for (int64_t k = 0; k < j->K; ++k) {
      double x = (double)bf16_to_f32(j->X[m * j->K + k]);
      const float* wrow = j->What + k * j->N;
      for (int64_t n = 0; n < j->N; ++n) y[n] += x * (double)wrow[n];
    }
  }
  return NULL;
}

/* Returns 0 on success, -1 on allocation failure. */
int wqo_gemm_rows(const uint16_t* X, const uint32_t* packed, const uint16_t* s,
                  const int64_t* rows, int64_t R, int64_t N, int64_t K,
                  int group, int bits, int nthreads, double* Y) {
  int8_t* q = (int8_t*)malloc((size_t)(K * N));
  float* What = (float*)malloc((size_t)(K * N) * sizeof(float));
  if (!q || !What) {
    free(q);
    free(What);
    return -1;
  }
  wqo_unpack(packed, K, N, bits, q);
  wqo_dequant(q, s, K, N, group, What);
  free(q);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > R) nthreads = (int)(R > 0 ? R : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  gemm_job* jobs = (gemm_job*)malloc(sizeof(gemm_job) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].X = X;
    jobs[t].What = What;
    jobs[t].rows = rows;
    jobs[t].r0 = R * t / nthreads;
    jobs[t].r1 = R * (t + 1) / nthreads;
    jobs[t].K = K;
    jobs[t].N = N;
    jobs[t].Y = Y;
    pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  free(What);
  return 0;
}

/* ------------------------------------------ drafter attention (SWA) -- */

/* The drafter's attention ("Quantize the Target, Quantize the Drafter",
   drafter-SWA paragraph): a block of B query tokens, the last B positions
   p_b = T - B + b of a sequence of T tokens whose keys and values are all
   cached (the cache is kept whole), attends bidirectionally with a window
   symmetric around each query: query b sees key j iff |j - p_b| <= W / 2.
   W == 0, or a sequence no longer than the window (T <= W), is full
   attention.  Q [B][Hq][D], K and V [Hkv][T][D], all bf16; query head h
   reads key/value head h / (Hq / Hkv).  Scores q.k / sqrt(D), a softmax
   over the visible keys and the weighted sum of values, all in fp64.
   O [B][Hq][D] fp64. */
void wqo_swa_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int B, int Hq,
                       int Hkv, int D, int64_t T, int64_t W, double* O) {
  const int group = Hq / Hkv;
  const int full = (W == 0 || T <= W);
  double* score = (double*)malloc((size_t)T * sizeof(double));
  if (!score) return;
  for (int b = 0; b < B; ++b) {
    const int64_t p = T - B + b;
    const int64_t lo = full ? 0 : (p - W / 2 < 0 ? 0 : p - W / 2);
    const int64_t hi = full ? T - 1 : (p + W / 2 > T - 1 ? T - 1 : p + W / 2);
    for (int h = 0; h < Hq; ++h) {
      const int kv = h / group;
      const uint16_t* q = Q + ((int64_t)b * Hq + h) * D;
      double mx = -INFINITY;
      for (int64_t j = lo; j <= hi; ++j) {
        const uint16_t* k = K + ((int64_t)kv * T + j) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)bf16_to_f32(q[d]) * (double)bf16_to_f32(k[d]);
        score[j] = acc / sqrt((double)D);
        if (score[j] > mx) mx = score[j];
      }
      double den = 0.0;
      for (int64_t j = lo; j <= hi; ++j) {
        score[j] = exp(score[j] - mx);
        den += score[j];
      }
      double* o = O + ((int64_t)b * Hq + h) * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int64_t j = lo; j <= hi; ++j) {
        const uint16_t* v = V + ((int64_t)kv * T + j) * D;
        for (int d = 0; d < D; ++d) o[d] += score[j] * (double)bf16_to_f32(v[d]);
      }
      for (int d = 0; d < D; ++d) o[d] /= den;
    }
  }
  free(score);
}

