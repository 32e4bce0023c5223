/*
 * MosaicQuant W4A4 + block-sparse 4-bit residual linear: the ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Plain, slow, single-threaded C in float64 / int64, written so that each
 * step can be checked by eye against its definition.  Citations name the
 * page "MosaicQuant: Inlier-Outlier Disaggregation for Unified 4-Bit LLM
 * Quantization" (technical summary) and its sections:
 *   [Metodologia 1]  the decomposition W^ ~= Q(W^) + R, both parts 4-bit;
 *   [Metodologia 2]  block-wise residual budget, Hessian-guided Delta-score
 *                    (residual error weighted by the diagonal-Hessian
 *                    activation sensitivity of the input channels), top-K;
 *   [Metodologia 3]  ZipperEngine: the residual product is reduce-added to
 *                    the dense 4-bit product.
 * The pages fix no group size, scale format or rounding; this library reads
 * them as: symmetric INT4 codes in [-7, 7], one fp16 scale per 128 inputs
 * (per token for activations, per output row for weights), scale =
 * fp16_RNE(amax / 7), codes = clamp(RNE(v / scale), -7, 7); residual blocks
 * of 64 output rows x 128 inputs, one fp16 scale per block row.
 *
 * Every function below takes plain arrays; the Python wrapper in this folder
 * marshals numpy arrays.  Build: gcc -O2 -ffp-contract=off -shared -fPIC.
 * (-ffp-contract=off keeps a*b+c as two rounded operations, which the
 * Delta-score definition below relies on.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MQO_GROUP 128 /* inputs per scale group and per residual block column */
#define MQO_BROWS 64  /* output rows per residual block                        */
#define MQO_QMAX 7    /* symmetric INT4 code range [-7, 7]                     */

/* ------------------------------------------------------------------------ */
/* 16-bit floating point, from the IEEE 754 binary16 and bfloat16 formats.  */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double mqo_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
double mqo_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xFF;
  int m = b & 0x7F;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133); /* subnormal: m * 2^-133 */
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + m), e - 134); /* (1 + m/128) * 2^(e-127) */
  return sign ? -v : v;
}

/*
 * Round a double to the nearest binary16 value, ties to even; overflow goes
 * to infinity.  The double must carry the exact value to be rounded (every
 * caller below passes either an exact value or one whose rounding to 53 bits
 * cannot move it across a binary16 rounding boundary; see the scale rule).
 */
uint16_t mqo_double_to_half(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7E00;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  e -= 1;              /* 2^e <= a < 2^(e+1) */
  if (e < -14) e = -14; /* subnormal range shares the 2^-24 quantum */
  double quantum = ldexp(1.0, e - 10);
  double r = rint(a / quantum); /* exact division by a power of two; RNE */
  double res = r * quantum;
  if (res > 65504.0) return sign | 0x7C00;
  /* r lies in [0, 2048]; the encoding (e+14)*1024 + r covers subnormals,
   * normals and the carry into the next binade alike. */
  return sign | (uint16_t)((e + 14) * 1024 + (int)r);
}

/* Round a double to the nearest bfloat16 value, ties to even. */
uint16_t mqo_double_to_bf16(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7FC0;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  e -= 1;
  if (e < -126) e = -126;
  double quantum = ldexp(1.0, e - 7);
  double r = rint(a / quantum);
  double res = r * quantum;
  double maxv = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (res > maxv) return sign | 0x7F80;
  return sign | (uint16_t)((e + 126) * 128 + (int)r);
}

/* ------------------------------------------------------------------------ */
/* The symmetric INT4 quantizer Qz, used for activations, base weights and  */
/* residual blocks alike [Metodologia 1: "both components at 4 bit"].       */
/* ------------------------------------------------------------------------ */

/*
 * Scale rule: s = fp16_RNE(amax / 7), saturated to 65504 when it would
 * overflow.  amax/7 is formed in double: amax carries at most 12 significant
 * bits, so the exact quotient is either a short dyadic (7 | mantissa) or ends
 * in the period-3 expansion of k/7, whose bits never run constant across the
 * window between binary16's and double's rounding points; the double is
 * therefore on the same side of every binary16 tie as the exact quotient.
 */
uint16_t mqo_scale_from_amax(double amax) {
  uint16_t s = mqo_double_to_half(amax / 7.0);
  if ((s & 0x7FFF) == 0x7C00) s = (s & 0x8000) | 0x7BFF;
  return s;
}

/* RNE of a quotient to an integer code clamped to [-7, 7]. */
static int mqo_code(double v, double s) {
  double t = rint(v / s);
  if (t > MQO_QMAX) t = MQO_QMAX;
  if (t < -MQO_QMAX) t = -MQO_QMAX;
  return (int)t;
}

/* Qz(v[0..n-1]) -> one scale (fp16 bits) and n codes. */
void mqo_quantize_group(const double* v, int n, uint16_t* s_bits, int8_t* q) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  uint16_t sb = mqo_scale_from_amax(amax);
  double s = mqo_half_to_double(sb);
  for (int i = 0; i < n; ++i) q[i] = (s == 0.0) ? 0 : (int8_t)mqo_code(v[i], s);
  *s_bits = sb;
}

/* Two codes per byte: element 2j in the low nibble, 2j+1 in the high nibble,
 * each as a 4-bit two's complement number. */
void mqo_pack_nibbles(const int8_t* q, int64_t n, uint8_t* out) {
  for (int64_t j = 0; j < n / 2; ++j)
    out[j] = (uint8_t)((q[2 * j] & 0xF) | ((q[2 * j + 1] & 0xF) << 4));
}

/* Reverse of the above. */
void mqo_unpack_nibbles(const uint8_t* p, int64_t n, int8_t* q) {
  for (int64_t j = 0; j < n / 2; ++j) {
    int lo = p[j] & 0xF, hi = (p[j] >> 4) & 0xF;
    q[2 * j] = (int8_t)(lo >= 8 ? lo - 16 : lo);
    q[2 * j + 1] = (int8_t)(hi >= 8 ? hi - 16 : hi);
  }
}

/* ------------------------------------------------------------------------ */
/* Activation quantizer: per token m, per 128-input group g.                 */
/* ------------------------------------------------------------------------ */

/* x: [M, K] 16-bit floats (is_bf16 selects the format), row-major.
 * q_out: [M, K] int8 codes.  s_out: [M, K/128] fp16 scale bits. */
void mqo_quantize_act(const uint16_t* x, int is_bf16, int64_t M, int64_t K, int8_t* q_out,
                      uint16_t* s_out) {
  double v[MQO_GROUP];
  int64_t G = K / MQO_GROUP;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < G; ++g) {
      for (int i = 0; i < MQO_GROUP; ++i) {
        uint16_t b = x[m * K + g * MQO_GROUP + i];
        v[i] = is_bf16 ? mqo_bf16_to_double(b) : mqo_half_to_double(b);
      }
      mqo_quantize_group(v, MQO_GROUP, &s_out[m * G + g], &q_out[m * K + g * MQO_GROUP]);
    }
}

/* ------------------------------------------------------------------------ */
/* Dense 4-bit base Q(W^) and the residual R = W^ - Q(W^)  [Metodologia 1]. */
/* ------------------------------------------------------------------------ */

/* w: [N, K] fp16 bits.  qw: [N, K] codes.  sw: [N, K/128] scale bits.
 * r: [N, K] residual in double (exact: w and s*q share a fine enough grid). */
void mqo_base_quant(const uint16_t* w, int64_t N, int64_t K, int8_t* qw, uint16_t* sw, double* r) {
  double v[MQO_GROUP];
  int64_t G = K / MQO_GROUP;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      for (int i = 0; i < MQO_GROUP; ++i) v[i] = mqo_half_to_double(w[n * K + g * MQO_GROUP + i]);
      int8_t* q = &qw[n * K + g * MQO_GROUP];
      mqo_quantize_group(v, MQO_GROUP, &sw[n * G + g], q);
      double s = mqo_half_to_double(sw[n * G + g]);
      if (r)
        for (int i = 0; i < MQO_GROUP; ++i) r[n * K + g * MQO_GROUP + i] = v[i] - s * (double)q[i];
    }
}

/* ------------------------------------------------------------------------ */
/* Hessian-guided block selection  [Metodologia 2].                          */
/* ------------------------------------------------------------------------ */

/* Diagonal Hessian estimate of the input channels: h_k = mean_c xcal[c,k]^2,
 * summed over ascending c, then divided by C. */
void mqo_hessian_diag(const uint16_t* xcal, int is_bf16, int64_t C, int64_t K, double* h) {
  for (int64_t k = 0; k < K; ++k) {
    double acc = 0.0;
    for (int64_t c = 0; c < C; ++c) {
      uint16_t b = xcal[c * K + k];
      double x = is_bf16 ? mqo_bf16_to_double(b) : mqo_half_to_double(b);
      acc = acc + x * x;
    }
    h[k] = acc / (double)C;
  }
}

/* Delta-score of every 64x128 block b = (br, g), b = br*(K/128) + g:
 *   Delta_b = sum_{k in g, ascending} h_k * ( sum_{n in br, ascending} R[n,k]^2 ).
 * The residual error of the block weighted by the sensitivity of its input
 * channels.  delta: [(N/64) * (K/128)]. */
void mqo_delta_scores(const double* r, const double* h, int64_t N, int64_t K, double* delta) {
  int64_t G = K / MQO_GROUP, NB = N / MQO_BROWS;
  for (int64_t br = 0; br < NB; ++br)
    for (int64_t g = 0; g < G; ++g) {
      double d = 0.0;
      for (int64_t kk = 0; kk < MQO_GROUP; ++kk) {
        int64_t k = g * MQO_GROUP + kk;
        double col = 0.0;
        for (int64_t rr = 0; rr < MQO_BROWS; ++rr) {
          double e = r[(br * MQO_BROWS + rr) * K + k];
          col = col + e * e;
        }
        d = d + h[k] * col;
      }
      delta[br * G + g] = d;
    }
}

/* Number of residual blocks a budget buys: floor(budget * #blocks), the
 * product nudged by 1e-9 so that e.g. 0.29 * 100 counts as 29. */
int64_t mqo_num_selected(int64_t N, int64_t K, double budget) {
  int64_t nb = (N / MQO_BROWS) * (K / MQO_GROUP);
  if (!(budget > 0.0)) return 0;
  double t = floor(budget * (double)nb + 1e-9);
  if (t > (double)nb) t = (double)nb;
  return (int64_t)t;
}

static const double* g_sort_delta; /* comparator context (single-threaded) */

/* Larger Delta first; equal Deltas by ascending block index. */
static int mqo_cmp_blocks(const void* a, const void* b) {
  int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
  double di = g_sort_delta[i], dj = g_sort_delta[j];
  if (di > dj) return -1;
  if (di < dj) return 1;
  return (i < j) ? -1 : (i > j) ? 1 : 0;
}

/* Top-K blocks by Delta, as a CSR list over 64-row block rows:
 * row_ptr[N/64 + 1], col_idx[ksel] = group index, ascending within a row. */
void mqo_select_topk(const double* delta, int64_t N, int64_t K, int64_t ksel, int32_t* row_ptr,
                     int32_t* col_idx) {
  int64_t G = K / MQO_GROUP, NB = N / MQO_BROWS, nb = NB * G;
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nb > 0 ? nb : 1));
  unsigned char* chosen = (unsigned char*)calloc((size_t)(nb > 0 ? nb : 1), 1);
  for (int64_t i = 0; i < nb; ++i) order[i] = i;
  g_sort_delta = delta;
  qsort(order, (size_t)nb, sizeof(int64_t), mqo_cmp_blocks);
  for (int64_t i = 0; i < ksel; ++i) chosen[order[i]] = 1;
  int64_t pos = 0;
  for (int64_t br = 0; br < NB; ++br) {
    row_ptr[br] = (int32_t)pos;
    for (int64_t g = 0; g < G; ++g)
      if (chosen[br * G + g]) col_idx[pos++] = (int32_t)g;
  }
  row_ptr[NB] = (int32_t)pos;
  free(order);
  free(chosen);
}

/* ------------------------------------------------------------------------ */
/* Sparse 4-bit residual on the selected blocks  [Metodologia 1 and 2].      */
/* ------------------------------------------------------------------------ */

/* For CSR entry i (block row br, group g) and block row r (n = 64*br + r):
 * Qz over R[n, 128g .. 128g+127].  qr: [nnzb][64][128] codes,
 * sr: [nnzb][64] scale bits. */
void mqo_residual_quant(const double* r, int64_t N, int64_t K, const int32_t* row_ptr,
                        const int32_t* col_idx, int8_t* qr, uint16_t* sr) {
  int64_t NB = N / MQO_BROWS;
  for (int64_t br = 0; br < NB; ++br)
    for (int64_t i = row_ptr[br]; i < row_ptr[br + 1]; ++i) {
      int64_t g = col_idx[i];
      for (int64_t rr = 0; rr < MQO_BROWS; ++rr) {
        const double* v = &r[(br * MQO_BROWS + rr) * K + g * MQO_GROUP];
        mqo_quantize_group(v, MQO_GROUP, &sr[i * MQO_BROWS + rr],
                           &qr[(i * MQO_BROWS + rr) * MQO_GROUP]);
      }
    }
}

/* ------------------------------------------------------------------------ */
/* The linear Y = Q(X) (Q(W^) + R^)^T, group by group  [Metodologia 3].      */
/* ------------------------------------------------------------------------ */

/* Exact integer dot of two code vectors. */
static int64_t mqo_dot(const int8_t* a, const int8_t* b, int n) {
  int64_t s = 0;
  for (int i = 0; i < n; ++i) s += (int64_t)a[i] * (int64_t)b[i];
  return s;
}

/* Dense group dots D_w[m][n][g] = sum_{k in g} qx[m,k] * qw[n,k]. */
void mqo_group_dots(const int8_t* qx, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                    int64_t* dw) {
  int64_t G = K / MQO_GROUP;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t g = 0; g < G; ++g)
        dw[(m * N + n) * G + g] =
            mqo_dot(&qx[m * K + g * MQO_GROUP], &qw[n * K + g * MQO_GROUP], MQO_GROUP);
}

/* Residual group dots D_r[m][i][r] = sum_{k in g_i} qx[m,k] * qr[i][r][k]
 * for every CSR entry i (group g_i) and block row r. */
void mqo_residual_dots(const int8_t* qx, const int8_t* qr, const int32_t* col_idx, int64_t M,
                       int64_t K, int64_t nnzb, int64_t* dr) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t i = 0; i < nnzb; ++i)
      for (int64_t rr = 0; rr < MQO_BROWS; ++rr)
        dr[(m * nnzb + i) * MQO_BROWS + rr] = mqo_dot(
            &qx[m * K + (int64_t)col_idx[i] * MQO_GROUP], &qr[(i * MQO_BROWS + rr) * MQO_GROUP],
            MQO_GROUP);
}

/*
 * Output entries y[m][n] for a list of (m, n) pairs (pass every pair for the
 * full matrix):
 *   y = sum_{g ascending} sx[m,g] * ( sw[n,g] * D_w + [block (n/64, g) selected] * sr * D_r )
 * in double, and the absolute-term sum
 *   a = sum_g |sx*sw*D_w| + |sx*sr*D_r|
 * that bounds the rounding error of any other evaluation order.
 * sel_of: [(N/64) * (K/128)] CSR entry index of block (br, g), or -1.
 */
void mqo_linear_entries(const int8_t* qx, const uint16_t* sx, const int8_t* qw, const uint16_t* sw,
                        const int8_t* qr, const uint16_t* sr, const int64_t* sel_of, int64_t M,
                        int64_t N, int64_t K, const int64_t* ms, const int64_t* ns, int64_t count,
                        double* y, double* abs_sum) {
  int64_t G = K / MQO_GROUP;
  (void)M;
  (void)N;
  for (int64_t t = 0; t < count; ++t) {
    int64_t m = ms[t], n = ns[t];
    double acc = 0.0, aacc = 0.0;
    for (int64_t g = 0; g < G; ++g) {
      double xs = mqo_half_to_double(sx[m * G + g]);
      double ws = mqo_half_to_double(sw[n * G + g]);
      int64_t dw = mqo_dot(&qx[m * K + g * MQO_GROUP], &qw[n * K + g * MQO_GROUP], MQO_GROUP);
      double base = ws * (double)dw;
      double res = 0.0;
      int64_t i = sel_of ? sel_of[(n / MQO_BROWS) * G + g] : -1;
      if (i >= 0) {
        int64_t rr = n % MQO_BROWS;
        double rs = mqo_half_to_double(sr[i * MQO_BROWS + rr]);
        int64_t dr = mqo_dot(&qx[m * K + g * MQO_GROUP], &qr[(i * MQO_BROWS + rr) * MQO_GROUP],
                             MQO_GROUP);
        res = rs * (double)dr;
      }
      acc = acc + xs * (base + res);
      aacc = aacc + fabs(xs * base) + fabs(xs * res);
    }
    y[t] = acc;
    if (abs_sum) abs_sum[t] = aacc;
  }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the format conversions, for the Python wrapper.          */
/* ------------------------------------------------------------------------ */

void mqo_half_to_double_n(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mqo_half_to_double(h[i]);
}
void mqo_bf16_to_double_n(const uint16_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mqo_bf16_to_double(b[i]);
}
void mqo_double_to_half_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mqo_double_to_half(v[i]);
}
void mqo_double_to_bf16_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mqo_double_to_bf16(v[i]);
}
void mqo_scale_from_amax_n(const double* a, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mqo_scale_from_amax(a[i]);
}
