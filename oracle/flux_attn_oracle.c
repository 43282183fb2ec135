/*
 * flux_attn_oracle.c -- plain fp64 CPU oracle for joint text/image attention
 * with per-head Q/K RMSNorm and multi-axis RoPE.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check of the package entry
 * file and the CPU-baseline / reference legs of bench.py load this library.
 * The CUDA path never calls, links or includes it, and it includes nothing
 * from the CUDA path.
 *
 * What it computes (sources are web pages; none prints a formula, so the
 * plainest reading is written out here):
 *   - "Speed up image generation with FLUX 3 Image Klein on NVIDIA Blackwell
 *     GPUs" (NVIDIA developer blog), section "FLUX 3 inference with TensorRT
 *     LLM VisualGen": text, noisy-target-image and optional reference-image
 *     token streams are processed separately and then merged by JOINT
 *     attention -- one bidirectional softmax attention over the concatenated
 *     sequence [txt | img | ref], no mask between streams.
 *   - same page, section "GEMM kernel optimisation": the QKV projection
 *     carries query/key normalisation and rotary position embedding (RoPE),
 *     so attention consumes RMSNorm'ed, rotated Q and K; V is untouched.
 *   - same page, section "Quantized and sparse attention": the FP8 variant
 *     runs Q.K and P.V with FP8 Q, K and V (qk_dtype fp8, v_dtype fp8).
 *   - same page, section "GEMM kernel optimisation": the QKV projection is
 *     one GEMM of the hidden states with the stacked Q, K, V weights, and its
 *     epilogue applies the query/key normalisation and RoPE (oracle_qkv_rows).
 *   - same page, section "Quantized and sparse attention": VC-Attention FP8
 *     takes a repair budget (vc_repair_budget 0.005 in its configuration):
 *     up to that share of the tokens, the worst quantised ones, get their
 *     quantisation residual corrected (oracle_vc_attention_rows, reading R7).
 *   - same page, section "Quantized and sparse attention": Sol-Attention
 *     (algorithm sol_attn, tau 1.0, disabled_until_timestep 0.96) runs
 *     block-sparse attention (oracle_sol_attention_rows, reading R8).
 *
 * Readings taken where the pages are silent:
 *   R1 RMSNorm over the head dimension d: y_i = x_i / sqrt(mean_j x_j^2 + eps) * w_i,
 *      one weight vector for Q and one for K, shared by all heads.
 *   R2 RoPE rotates ADJACENT pairs (x_{2j}, x_{2j+1}); the head dimension is cut
 *      into consecutive axis blocks of sizes axes[0..2]; in block a the pair j
 *      turns by angle pos_a * theta^(-2j/axes[a]).
 *   R3 Norm first, then RoPE.
 *   R4 Softmax scale 1/sqrt(d).
 *   R5 FP8: per (batch, head) and per tensor, scale = amax / 448 (1 when
 *      amax = 0); codes are E4M3 (finite, max 448) of the real x / scale,
 *      rounded to nearest, ties to even, saturating; attention then runs
 *      exactly on the dequantised values code * scale.
 *   R6 QKV projection: y = x W^T (+ b) with W [3 H d, D] (output features
 *      first, as a linear layer stores it); y splits into Q (features
 *      0 .. H d - 1), K (the next H d) and V (the last H d), head h owning
 *      features h d .. h d + d - 1 of its part; Q and K then get R1-R3, V
 *      nothing.
 *   R7 VC-Attention repair, per (batch, head), after the quantisation of R5:
 *      key token m has the quantisation error
 *        e_m = |k'_m - deq(k'_m)|^2 + |v_m - deq(v_m)|^2
 *      (squared Euclidean norms of its K' and V rows, in their own units);
 *      the R = ceil(rho N) tokens with the largest e_m (equal errors: the
 *      lower token index first) are repaired: their residual x - deq(x) is
 *      added back, i.e. they take part in the attention with their exact K'
 *      and V, every other key keeps its dequantised values, and every query
 *      keeps its dequantised Q'.  rho = 0 is plain FP8 attention.
 *   R8 Sol-Attention, per (batch, head): queries and keys are cut into blocks
 *      of 128 tokens (the last one ragged), nb blocks each.  A block's pooled
 *      vector is the mean of its normalised, rotated rows (q_bar_i, k_bar_j);
 *      query block i gives key block j the mass
 *        mu_ij = c_j exp(q_bar_i . k_bar_j / sqrt(d)) / sum_j' c_j' exp(q_bar_i . k_bar_j' / sqrt(d))
 *      (c_j = keys in block j: the pooled estimate of the softmax mass of the
 *      block), and keeps it when mu_ij >= tau / nb, i.e. at least tau times
 *      the mass of a uniform split; the block of largest mass (lowest index
 *      on ties) is always kept.  A query then attends, with the usual
 *      softmax, to the keys of its kept blocks only.  tau = 0 keeps every
 *      block (dense attention); the timestep gate of the configuration
 *      (dense while the timestep is above disabled_until_timestep) is the
 *      caller's choice of tau.
 *
 * Every loop below follows the definition directly: no tiling, no online
 * softmax, no reordering beyond summation order inside a dot product.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- inputs */

/* An input tensor is either bf16 bit patterns or plain doubles. */
typedef struct {
  const void* p;
  int is_bf16;
} src_t;

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double ld(const src_t* s, int64_t i) {
  if (s->is_bf16) return bf16_to_f64(((const uint16_t*)s->p)[i]);
  return ((const double*)s->p)[i];
}

/* ------------------------------------------------------------ E4M3 codec */

/* Decode one OCP E4M3 ("fn") code: 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, 0x7F / 0xFF are NaN. */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^-6 */
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Encode a double to E4M3: round to nearest, ties to even, saturate finite
 * values to +-448 (reading R5).  NaN maps to 0x7F. */
uint8_t oracle_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);    /* 1.75 * 2^8 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: a = q * 2^-9, q in [0, 8); q == 8 carries into the
     * smallest normal, whose code (e=1, m=0) is exactly 8. */
    double q = nearbyint(ldexp(a, 9));
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  double fr = frexp(a, &e2);                        /* a = fr * 2^e2, fr in [0.5, 1) */
  int e = e2 - 1;                                   /* a = (2 fr) * 2^e, 2fr in [1, 2) */
  double m = nearbyint((2.0 * fr - 1.0) * 8.0);     /* exact products, RNE */
  if (m == 8.0) { m = 0.0; e += 1; }
  int be = e + 7;
  if (be > 15 || (be == 15 && m == 7.0)) return (uint8_t)(sign | 0x7E);
  return (uint8_t)(sign | (be << 3) | (int)m);
}

/* ------------------------------------------------------ per-row prologue */

/* Reading R1: RMSNorm of one head row of length d. */
static void rmsnorm_row(double* y, const double* x, int d, const double* w, double eps) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / d + eps);
  for (int i = 0; i < d; ++i) y[i] = x[i] * inv * w[i];
}

/* Reading R2: multi-axis RoPE on one head row, in place. */
static void rope_row(double* y, int d, const int32_t* pos3, double theta, const int* axes) {
  int off = 0;
  for (int a = 0; a < 3; ++a) {
    int da = axes[a];
    for (int j = 0; j < da / 2; ++j) {
      double ang = (double)pos3[a] * pow(theta, -2.0 * j / da);
      double c = cos(ang), s = sin(ang);
      double x0 = y[off + 2 * j], x1 = y[off + 2 * j + 1];
      y[off + 2 * j] = x0 * c - x1 * s;
      y[off + 2 * j + 1] = x0 * s + x1 * c;
    }
    off += da;
  }
  (void)d;
}

static int check_axes(int d, const int* axes) {
  if (d <= 0) return -1;
  if (axes[0] < 0 || axes[1] < 0 || axes[2] < 0) return -1;
  if (axes[0] % 2 || axes[1] % 2 || axes[2] % 2) return -1;
  if (axes[0] + axes[1] + axes[2] != d) return -1;
  return 0;
}

/* Normalised + rotated rows for every token of head (b, h): out[N*d]. */
static void prologue_head(double* out, const src_t* x, int b, int h, int N, int H, int d,
                          const int32_t* pos, const double* w, double eps, double theta,
                          const int* axes, int nt) {
  int64_t n;
#pragma omp parallel for num_threads(nt) schedule(static)
  for (n = 0; n < N; ++n) {
    double row[1024];
    int64_t base = (((int64_t)b * N + n) * H + h) * d;
    for (int i = 0; i < d; ++i) row[i] = ld(x, base + i);
    rmsnorm_row(out + n * d, row, d, w, eps);
    rope_row(out + n * d, d, pos + 3 * n, theta, axes);
  }
}

static void plain_head(double* out, const src_t* x, int b, int h, int N, int H, int d, int nt) {
  int64_t n;
#pragma omp parallel for num_threads(nt) schedule(static)
  for (n = 0; n < N; ++n) {
    int64_t base = (((int64_t)b * N + n) * H + h) * d;
    for (int i = 0; i < d; ++i) out[n * d + i] = ld(x, base + i);
  }
}

/* Reading R5: per-tensor-per-head amax scale, quantise, dequantise in place.
 * The code is E4M3 of the real quotient x / scale = 448 x / amax, formed as
 * (448 x) / amax: rounding the scale first would move quotients that sit
 * exactly halfway between two codes off the tie.  codes (optional) receives
 * the E4M3 codes. Returns the scale. */
static double fp8_roundtrip(double* a, int64_t count, uint8_t* codes) {
  double amax = 0.0;
  for (int64_t i = 0; i < count; ++i) if (fabs(a[i]) > amax) amax = fabs(a[i]);
  double scale = amax > 0.0 ? amax / 448.0 : 1.0;
  for (int64_t i = 0; i < count; ++i) {
    uint8_t c = oracle_e4m3_encode(amax > 0.0 ? (448.0 * a[i]) / amax : a[i]);
    if (codes) codes[i] = c;
    a[i] = oracle_e4m3_decode(c) * scale;
  }
  return scale;
}

/* One output row: o = sum_m softmax_m(q.k_m / sqrt(d)) v_m (reading R4). */
static void attention_row(double* o, const double* qh, const double* kh, const double* vh,
                          int N, int d, double* srow) {
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int m = 0; m < N; ++m) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += qh[i] * kh[(int64_t)m * d + i];
    s *= inv_sqrt_d;
    srow[m] = s;
    if (s > mx) mx = s;
  }
  double l = 0.0;
  for (int m = 0; m < N; ++m) {
    srow[m] = exp(srow[m] - mx);
    l += srow[m];
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int m = 0; m < N; ++m) {
    double p = srow[m] / l;
    for (int i = 0; i < d; ++i) o[i] += p * vh[(int64_t)m * d + i];
  }
}

/* ---------------------------------------------- VC-Attention repair (R7) */

typedef struct {
  double e;
  int64_t m;
} vc_key_t;

/* Larger error first; equal errors: lower token index first. */
static int vc_key_cmp(const void* a, const void* b) {
  const vc_key_t* x = (const vc_key_t*)a;
  const vc_key_t* y = (const vc_key_t*)b;
  if (x->e > y->e) return -1;
  if (x->e < y->e) return 1;
  return (x->m > y->m) - (x->m < y->m);
}

static int i64_cmp(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* R = ceil(rho N), clamped to [0, N]. */
int64_t oracle_vc_repair_count(double rho, int64_t N) {
  double r = ceil(rho * (double)N);
  if (!(r > 0.0)) return 0;
  if (r > (double)N) return N;
  return (int64_t)r;
}

/* Errors e_m of every key token of one head and its repair set: kx, vx the
 * exact K' and V rows, kq, vq their dequantised values ([N*d] each).  err
 * receives e_m [N], sel the R selected token indices in ascending order.
 * Returns R, or -1 when memory runs out. */
static int64_t vc_select(const double* kx, const double* kq, const double* vx, const double* vq, int64_t N,
                         int d, double rho, int64_t* sel, double* err) {
  int64_t R = oracle_vc_repair_count(rho, N);
  vc_key_t* keys = (vc_key_t*)malloc(sizeof(vc_key_t) * (N > 0 ? N : 1));
  if (!keys) return -1;
  for (int64_t m = 0; m < N; ++m) {
    double e = 0.0;
    for (int i = 0; i < d; ++i) {
      double dk = kx[m * d + i] - kq[m * d + i];
      double dv = vx[m * d + i] - vq[m * d + i];
      e += dk * dk + dv * dv;
    }
    err[m] = e;
    keys[m].e = e;
    keys[m].m = m;
  }
  qsort(keys, (size_t)N, sizeof(vc_key_t), vc_key_cmp);
  for (int64_t r = 0; r < R; ++r) sel[r] = keys[r].m;
  qsort(sel, (size_t)R, sizeof(int64_t), i64_cmp);
  free(keys);
  return R;
}

/* ---------------------------------------------------- Sol-Attention (R8) */

/* Block mask of one head: keep[i * nb + j] = 1 when query block i keeps key
 * block j; mass[i * nb + j] = mu_ij.  qh, kh: the head's Q', K' [N * d]. */
static void sol_mask(const double* qh, const double* kh, int64_t N, int d, double tau, unsigned char* keep,
                     double* mass) {
  const int64_t bs = 128;
  const int64_t nb = (N + bs - 1) / bs;
  double* qb = (double*)calloc((size_t)(nb * d), sizeof(double));
  double* kb = (double*)calloc((size_t)(nb * d), sizeof(double));
  double* cnt = (double*)calloc((size_t)nb, sizeof(double));
  double* sc = (double*)malloc(sizeof(double) * (nb > 0 ? nb : 1));
  if (!qb || !kb || !cnt || !sc) {
    free(qb); free(kb); free(cnt); free(sc);
    for (int64_t i = 0; i < nb * nb; ++i) { keep[i] = 1; mass[i] = NAN; }
    return;
  }
  for (int64_t n = 0; n < N; ++n) {
    int64_t blk = n / bs;
    cnt[blk] += 1.0;
    for (int i = 0; i < d; ++i) {
      qb[blk * d + i] += qh[n * d + i];
      kb[blk * d + i] += kh[n * d + i];
    }
  }
  for (int64_t blk = 0; blk < nb; ++blk)
    for (int i = 0; i < d; ++i) {
      qb[blk * d + i] /= cnt[blk];
      kb[blk * d + i] /= cnt[blk];
    }
  const double scale = 1.0 / sqrt((double)d);
  for (int64_t i = 0; i < nb; ++i) {
    double mx = -INFINITY;
    for (int64_t j = 0; j < nb; ++j) {
      double s = 0.0;
      for (int t = 0; t < d; ++t) s += qb[i * d + t] * kb[j * d + t];
      sc[j] = s * scale + log(cnt[j]);
      if (sc[j] > mx) mx = sc[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < nb; ++j) z += exp(sc[j] - mx);
    int64_t best = 0;
    for (int64_t j = 0; j < nb; ++j) {
      mass[i * nb + j] = exp(sc[j] - mx) / z;
      if (mass[i * nb + j] > mass[i * nb + best]) best = j;
    }
    for (int64_t j = 0; j < nb; ++j)
      keep[i * nb + j] = (unsigned char)(mass[i * nb + j] >= tau / (double)nb || j == best);
  }
  free(qb); free(kb); free(cnt); free(sc);
}

/* One output row over the keys of the kept blocks of its query block. */
static void sol_attention_row(double* o, const double* qh, const double* kh, const double* vh, int64_t N, int d,
                              const unsigned char* keep_row, double* srow) {
  const double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int64_t m = 0; m < N; ++m) {
    if (!keep_row[m / 128]) continue;
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += qh[i] * kh[m * d + i];
    srow[m] = s * scale;
    if (srow[m] > mx) mx = srow[m];
  }
  double l = 0.0;
  for (int64_t m = 0; m < N; ++m) {
    if (!keep_row[m / 128]) continue;
    srow[m] = exp(srow[m] - mx);
    l += srow[m];
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int64_t m = 0; m < N; ++m) {
    if (!keep_row[m / 128]) continue;
    const double w = srow[m] / l;
    for (int i = 0; i < d; ++i) o[i] += w * vh[m * d + i];
  }
}

/* ------------------------------------------------------------ public API */

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int nthreads_or_max(int nt) { return nt > 0 ? nt : oracle_max_threads(); }

/* Q or K prologue for every row: x [B,N,H,d] (bf16 bits or doubles) ->
 * out [B,N,H,d] doubles. */
static int prologue_all(const src_t* x, int B, int N, int H, int d, const int32_t* pos,
                        const double* w, double eps, double theta, const int* axes,
                        double* out, int nt) {
  if (check_axes(d, axes) || d > 1024 || B < 0 || N < 0 || H < 0) return -1;
  nt = nthreads_or_max(nt);
  int64_t r, rows = (int64_t)B * N * H;
#pragma omp parallel for num_threads(nt) schedule(static)
  for (r = 0; r < rows; ++r) {
    double row[1024];
    int64_t n = (r / H) % N;
    for (int i = 0; i < d; ++i) row[i] = ld(x, r * d + i);
    rmsnorm_row(out + r * d, row, d, w, eps);
    rope_row(out + r * d, d, pos + 3 * n, theta, axes);
  }
  return 0;
}

int oracle_prologue_bf16(const uint16_t* x, int B, int N, int H, int d, const int32_t* pos,
                         const float* wf, double eps, double theta, const int* axes,
                         double* out, int nt) {
  double w[1024];
  if (d > 1024 || d <= 0) return -1;
  for (int i = 0; i < d; ++i) w[i] = (double)wf[i];
  src_t s = {x, 1};
  return prologue_all(&s, B, N, H, d, pos, w, eps, theta, axes, out, nt);
}

int oracle_prologue_f64(const double* x, int B, int N, int H, int d, const int32_t* pos,
                        const double* w, double eps, double theta, const int* axes,
                        double* out, int nt) {
  src_t s = {x, 0};
  return prologue_all(&s, B, N, H, d, pos, w, eps, theta, axes, out, nt);
}

/* Attention output for the requested query rows.
 *   rows: nrows triples (b, h, n); out: nrows x d doubles.
 * All rows of one (b, h) share the normalised K (and V) of that head, built
 * once per distinct head in order of first appearance. */
static int attention_rows(const src_t* q, const src_t* k, const src_t* v, int B, int N, int H,
                          int d, const int32_t* pos, const double* wq, const double* wk,
                          double eps, double theta, const int* axes, int fp8, double rho,
                          const int64_t* rows, int64_t nrows, double* out, int nt) {
  if (check_axes(d, axes) || d > 1024 || B <= 0 || N <= 0 || H <= 0) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t b = rows[3 * r], h = rows[3 * r + 1], n = rows[3 * r + 2];
    if (b < 0 || b >= B || h < 0 || h >= H || n < 0 || n >= N) return -2;
  }
  nt = nthreads_or_max(nt);
  int64_t nd = (int64_t)N * d;
  double* kh = (double*)malloc(sizeof(double) * nd);
  double* vh = (double*)malloc(sizeof(double) * nd);
  double* qh = (double*)malloc(sizeof(double) * nd);
  unsigned char* done = (unsigned char*)calloc((size_t)B * H, 1);
  int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (nrows > 0 ? nrows : 1));
  int vc = fp8 && rho > 0.0;
  double* kx = vc ? (double*)malloc(sizeof(double) * nd) : NULL;  /* exact K', V (R7) */
  double* vx = vc ? (double*)malloc(sizeof(double) * nd) : NULL;
  double* err = vc ? (double*)malloc(sizeof(double) * N) : NULL;
  int64_t* sel = vc ? (int64_t*)malloc(sizeof(int64_t) * N) : NULL;
  if (!kh || !vh || !qh || !done || !idx || (vc && (!kx || !vx || !err || !sel))) {
    free(kh); free(vh); free(qh); free(done); free(idx);
    free(kx); free(vx); free(err); free(sel);
    return -3;
  }
  for (int64_t r0 = 0; r0 < nrows; ++r0) {
    int b = (int)rows[3 * r0], h = (int)rows[3 * r0 + 1];
    if (done[(size_t)b * H + h]) continue;
    done[(size_t)b * H + h] = 1;
    /* the rows of this head */
    int64_t cnt = 0;
    for (int64_t r = r0; r < nrows; ++r)
      if (rows[3 * r] == b && rows[3 * r + 1] == h) idx[cnt++] = r;
    prologue_head(kh, k, b, h, N, H, d, pos, wk, eps, theta, axes, nt);
    plain_head(vh, v, b, h, N, H, d, nt);
    if (fp8) {
      prologue_head(qh, q, b, h, N, H, d, pos, wq, eps, theta, axes, nt);
      if (vc) {
        memcpy(kx, kh, sizeof(double) * nd);
        memcpy(vx, vh, sizeof(double) * nd);
      }
      fp8_roundtrip(qh, nd, NULL);
      fp8_roundtrip(kh, nd, NULL);
      fp8_roundtrip(vh, nd, NULL);
      if (vc) {
        /* R7: the selected tokens take part with their exact K' and V */
        int64_t R = vc_select(kx, kh, vx, vh, N, d, rho, sel, err);
        if (R < 0) {
          free(kh); free(vh); free(qh); free(done); free(idx);
          free(kx); free(vx); free(err); free(sel);
          return -3;
        }
        for (int64_t r = 0; r < R; ++r) {
          memcpy(kh + sel[r] * d, kx + sel[r] * d, sizeof(double) * d);
          memcpy(vh + sel[r] * d, vx + sel[r] * d, sizeof(double) * d);
        }
      }
    }
    int64_t t;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
    for (t = 0; t < cnt; ++t) {
      int64_t r = idx[t];
      int64_t n = rows[3 * r + 2];
      double qrow[1024], tmp[1024];
      double* srow = (double*)malloc(sizeof(double) * N);
      const double* qp;
      if (fp8) {
        qp = qh + n * d;
      } else {
        int64_t base = (((int64_t)b * N + n) * H + h) * d;
        for (int i = 0; i < d; ++i) tmp[i] = ld(q, base + i);
        rmsnorm_row(qrow, tmp, d, wq, eps);
        rope_row(qrow, d, pos + 3 * n, theta, axes);
        qp = qrow;
      }
      if (srow) attention_row(out + r * d, qp, kh, vh, N, d, srow);
      else for (int i = 0; i < d; ++i) out[r * d + i] = NAN;
      free(srow);
    }
  }
  free(kh); free(vh); free(qh); free(done); free(idx);
  free(kx); free(vx); free(err); free(sel);
  return 0;
}

int oracle_attention_rows_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               int B, int N, int H, int d, const int32_t* pos,
                               const float* wqf, const float* wkf, double eps, double theta,
                               const int* axes, int fp8, const int64_t* rows, int64_t nrows,
                               double* out, int nt) {
  double wq[1024], wk[1024];
  if (d > 1024 || d <= 0) return -1;
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  src_t sq = {q, 1}, sk = {k, 1}, sv = {v, 1};
  return attention_rows(&sq, &sk, &sv, B, N, H, d, pos, wq, wk, eps, theta, axes, fp8, 0.0,
                        rows, nrows, out, nt);
}

int oracle_attention_rows_f64(const double* q, const double* k, const double* v,
                              int B, int N, int H, int d, const int32_t* pos,
                              const double* wq, const double* wk, double eps, double theta,
                              const int* axes, int fp8, const int64_t* rows, int64_t nrows,
                              double* out, int nt) {
  src_t sq = {q, 0}, sk = {k, 0}, sv = {v, 0};
  return attention_rows(&sq, &sk, &sv, B, N, H, d, pos, wq, wk, eps, theta, axes, fp8, 0.0,
                        rows, nrows, out, nt);
}

/* VC-Attention FP8 (readings R5, R7): like oracle_attention_rows_bf16 with
 * fp8 = 1, the R = ceil(rho N) worst-quantised key tokens of every head
 * repaired. */
int oracle_vc_attention_rows_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  int B, int N, int H, int d, const int32_t* pos,
                                  const float* wqf, const float* wkf, double eps, double theta,
                                  const int* axes, double rho, const int64_t* rows, int64_t nrows,
                                  double* out, int nt) {
  double wq[1024], wk[1024];
  if (d > 1024 || d <= 0 || !(rho >= 0.0 && rho <= 1.0)) return -1;
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  src_t sq = {q, 1}, sk = {k, 1}, sv = {v, 1};
  return attention_rows(&sq, &sk, &sv, B, N, H, d, pos, wq, wk, eps, theta, axes, 1, rho,
                        rows, nrows, out, nt);
}

/* FP8 intermediates of one head (reading R5): E4M3 codes of the normalised,
 * rotated Q and K and of V, each [N*d] in token-major order, and the three
 * scales (q, k, v). */
int oracle_fp8_quantize_head_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  int B, int N, int H, int d, const int32_t* pos,
                                  const float* wqf, const float* wkf, double eps, double theta,
                                  const int* axes, int b, int h, uint8_t* q8, uint8_t* k8,
                                  uint8_t* v8, double* scales, int nt) {
  double wq[1024], wk[1024];
  if (check_axes(d, axes) || d > 1024 || b < 0 || b >= B || h < 0 || h >= H || N <= 0) return -1;
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  nt = nthreads_or_max(nt);
  int64_t nd = (int64_t)N * d;
  double* t = (double*)malloc(sizeof(double) * nd);
  if (!t) return -3;
  src_t sq = {q, 1}, sk = {k, 1}, sv = {v, 1};
  prologue_head(t, &sq, b, h, N, H, d, pos, wq, eps, theta, axes, nt);
  scales[0] = fp8_roundtrip(t, nd, q8);
  prologue_head(t, &sk, b, h, N, H, d, pos, wk, eps, theta, axes, nt);
  scales[1] = fp8_roundtrip(t, nd, k8);
  plain_head(t, &sv, b, h, N, H, d, nt);
  scales[2] = fp8_roundtrip(t, nd, v8);
  free(t);
  return 0;
}

/* Reading R7 for one head (b, h): the quantisation error e_m of every key
 * token (err, [N]) and the repaired tokens in ascending order (sel, room for
 * N).  Returns R, or a negative value on bad arguments. */
int64_t oracle_vc_select_head_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   int B, int N, int H, int d, const int32_t* pos,
                                   const float* wqf, const float* wkf, double eps, double theta,
                                   const int* axes, double rho, int b, int h, int64_t* sel,
                                   double* err, int nt) {
  double wk[1024];
  (void)q;
  (void)wqf;
  if (check_axes(d, axes) || d > 1024 || b < 0 || b >= B || h < 0 || h >= H || N <= 0 ||
      !(rho >= 0.0 && rho <= 1.0))
    return -1;
  for (int i = 0; i < d; ++i) wk[i] = wkf[i];
  nt = nthreads_or_max(nt);
  int64_t nd = (int64_t)N * d;
  double* kx = (double*)malloc(sizeof(double) * nd);
  double* kq = (double*)malloc(sizeof(double) * nd);
  double* vx = (double*)malloc(sizeof(double) * nd);
  double* vq = (double*)malloc(sizeof(double) * nd);
  int64_t R = -3;
  if (kx && kq && vx && vq) {
    src_t sk = {k, 1}, sv = {v, 1};
    prologue_head(kx, &sk, b, h, N, H, d, pos, wk, eps, theta, axes, nt);
    plain_head(vx, &sv, b, h, N, H, d, nt);
    memcpy(kq, kx, sizeof(double) * nd);
    memcpy(vq, vx, sizeof(double) * nd);
    fp8_roundtrip(kq, nd, NULL);
    fp8_roundtrip(vq, nd, NULL);
    R = vc_select(kx, kq, vx, vq, N, d, rho, sel, err);
    if (R < 0) R = -3;
  }
  free(kx); free(kq); free(vx); free(vq);
  return R;
}

/* Reading R6: the QKV projection of the requested token rows, then the
 * query/key normalisation and RoPE of each head.
 *   x      bf16 bits [M, D] (M = B * N token rows, row m = b * N + n)
 *   w      bf16 bits [3 H d, D];  bias  float [3 H d] or NULL
 *   rows   nrows token rows m;  out_q, out_k, out_v  [nrows, H, d] doubles
 * Token row m takes the position ids of n = m % N. */
int oracle_qkv_rows(const uint16_t* x, const uint16_t* w, const float* bias, int M, int D, int H, int d,
                    int N, const int32_t* pos, const float* wqf, const float* wkf, double eps,
                    double theta, const int* axes, const int64_t* rows, int64_t nrows, double* out_q,
                    double* out_k, double* out_v, int nt) {
  double wq[1024], wk[1024];
  if (check_axes(d, axes) || d > 1024 || M <= 0 || D <= 0 || H <= 0 || N <= 0 || M % N) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return -2;
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  nt = nthreads_or_max(nt);
  const int F = 3 * H * d;
  int64_t r;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
  for (r = 0; r < nrows; ++r) {
    const int64_t m = rows[r];
    const int64_t n = m % N;
    double* y = (double*)malloc(sizeof(double) * F);
    double* xr = (double*)malloc(sizeof(double) * D);
    if (!y || !xr) {
      free(y); free(xr);
      for (int i = 0; i < H * d; ++i) out_q[r * H * d + i] = out_k[r * H * d + i] = out_v[r * H * d + i] = NAN;
      continue;
    }
    for (int c = 0; c < D; ++c) xr[c] = bf16_to_f64(x[m * D + c]);
    for (int o = 0; o < F; ++o) {
      double acc = 0.0;
      for (int c = 0; c < D; ++c) acc += xr[c] * bf16_to_f64(w[(int64_t)o * D + c]);
      y[o] = acc + (bias ? (double)bias[o] : 0.0);
    }
    for (int h = 0; h < H; ++h) {
      double* q = out_q + (r * H + h) * d;
      double* k = out_k + (r * H + h) * d;
      double* v = out_v + (r * H + h) * d;
      rmsnorm_row(q, y + (int64_t)h * d, d, wq, eps);
      rope_row(q, d, pos + 3 * n, theta, axes);
      rmsnorm_row(k, y + (int64_t)(H + h) * d, d, wk, eps);
      rope_row(k, d, pos + 3 * n, theta, axes);
      for (int i = 0; i < d; ++i) v[i] = y[(int64_t)(2 * H + h) * d + i];
    }
    free(y);
    free(xr);
  }
  return 0;
}

/* Reading R8 for head (b, h): keep [nb * nb] (1 = query block i keeps key
 * block j) and mass [nb * nb] (mu_ij).  Returns nb, or a negative value on
 * bad arguments. */
int64_t oracle_sol_mask_bf16(const uint16_t* q, const uint16_t* k, int B, int N, int H, int d,
                             const int32_t* pos, const float* wqf, const float* wkf, double eps, double theta,
                             const int* axes, double tau, int b, int h, unsigned char* keep, double* mass,
                             int nt) {
  double wq[1024], wk[1024];
  if (check_axes(d, axes) || d > 1024 || b < 0 || b >= B || h < 0 || h >= H || N <= 0 || !(tau >= 0.0))
    return -1;
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  nt = nthreads_or_max(nt);
  int64_t nd = (int64_t)N * d;
  double* qh = (double*)malloc(sizeof(double) * nd);
  double* kh = (double*)malloc(sizeof(double) * nd);
  if (!qh || !kh) { free(qh); free(kh); return -3; }
  src_t sq = {q, 1}, sk = {k, 1};
  prologue_head(qh, &sq, b, h, N, H, d, pos, wq, eps, theta, axes, nt);
  prologue_head(kh, &sk, b, h, N, H, d, pos, wk, eps, theta, axes, nt);
  sol_mask(qh, kh, N, d, tau, keep, mass);
  free(qh); free(kh);
  return ((int64_t)N + 127) / 128;
}

/* Sol-Attention rows (readings R1-R4, R8): rows (b, h, n) as for
 * oracle_attention_rows_bf16, each over the keys of the blocks its query
 * block keeps. */
int oracle_sol_attention_rows_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int N, int H,
                                   int d, const int32_t* pos, const float* wqf, const float* wkf, double eps,
                                   double theta, const int* axes, double tau, const int64_t* rows, int64_t nrows,
                                   double* out, int nt) {
  double wq[1024], wk[1024];
  if (check_axes(d, axes) || d > 1024 || B <= 0 || N <= 0 || H <= 0 || !(tau >= 0.0)) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t b = rows[3 * r], h = rows[3 * r + 1], n = rows[3 * r + 2];
    if (b < 0 || b >= B || h < 0 || h >= H || n < 0 || n >= N) return -2;
  }
  for (int i = 0; i < d; ++i) { wq[i] = wqf[i]; wk[i] = wkf[i]; }
  nt = nthreads_or_max(nt);
  const int64_t nd = (int64_t)N * d, nb = ((int64_t)N + 127) / 128;
  double* qh = (double*)malloc(sizeof(double) * nd);
  double* kh = (double*)malloc(sizeof(double) * nd);
  double* vh = (double*)malloc(sizeof(double) * nd);
  unsigned char* keep = (unsigned char*)malloc((size_t)(nb * nb));
  double* mass = (double*)malloc(sizeof(double) * nb * nb);
  unsigned char* done = (unsigned char*)calloc((size_t)B * H, 1);
  if (!qh || !kh || !vh || !keep || !mass || !done) {
    free(qh); free(kh); free(vh); free(keep); free(mass); free(done);
    return -3;
  }
  src_t sq = {q, 1}, sk = {k, 1}, sv = {v, 1};
  for (int64_t r0 = 0; r0 < nrows; ++r0) {
    int b = (int)rows[3 * r0], h = (int)rows[3 * r0 + 1];
    if (done[(size_t)b * H + h]) continue;
    done[(size_t)b * H + h] = 1;
    prologue_head(qh, &sq, b, h, N, H, d, pos, wq, eps, theta, axes, nt);
    prologue_head(kh, &sk, b, h, N, H, d, pos, wk, eps, theta, axes, nt);
    plain_head(vh, &sv, b, h, N, H, d, nt);
    sol_mask(qh, kh, N, d, tau, keep, mass);
    int64_t t;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
    for (t = r0; t < nrows; ++t) {
      if (rows[3 * t] != b || rows[3 * t + 1] != h) continue;
      int64_t n = rows[3 * t + 2];
      double* srow = (double*)malloc(sizeof(double) * N);
      if (srow) sol_attention_row(out + t * d, qh + n * d, kh, vh, N, d, keep + (n / 128) * nb, srow);
      else for (int i = 0; i < d; ++i) out[t * d + i] = NAN;
      free(srow);
    }
  }
  free(qh); free(kh); free(vh); free(keep); free(mass); free(done);
  return 0;
}

/* Reading R5 on given values: the E4M3 codes of x[0 .. n) with the scale
 * amax / 448 of the whole array (1 when it is all zero), as the FP8 path
 * quantises one (batch, head) of Q', K' or V.  Returns the scale. */
double oracle_fp8_quantize_values(const double* x, int64_t n, uint8_t* codes) {
  double* t = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
  if (!t) return NAN;
  memcpy(t, x, sizeof(double) * n);
  double scale = fp8_roundtrip(t, n, codes);
  free(t);
  return scale;
}
