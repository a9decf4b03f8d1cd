/*
 * mla_oracle.c -- CPU fp64 oracle for single-token MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only tests/, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header, table or constant generator with the CUDA library.
 *
 * What it computes (plain definition, no blocking or reordering):
 *   For batch row b and head h, over the cached rows r in [kv_indptr[b], kv_indptr[b+1]):
 *     Khat_r = dequant(kv row r)                      (576 values, fp64)
 *     s_r    = (1/sqrt(576)) * sum_d q[b,h,d] * Khat_r[d]
 *     p_r    = exp(s_r - max_r s_r) / sum_r exp(s_r - max_r s_r)
 *     o[b,h] = sum_r p_r * Khat_r[0:512]             (V is the first 512 columns)
 *     lse    = max_r s_r + log(sum_r exp(s_r - max_r s_r))
 *   Source: amd-mixed-mla submission 599694, the `_bmm` path (batched q.K^T times
 *   sm_scale, fp32 softmax over the cached tokens, times V = first 512 columns), with
 *   the 16-head / 576-wide / 512-value geometry and sm_scale = 1/sqrt(576) stated in the
 *   module constants of all three submissions (727205, 700955, 599694).
 *
 * Decoders (tables built here from the bit-field definitions):
 *   e4m3 (OCP FP8 "fn" variant, max 448; amd-mixed-mla submission 727205 uses 448 as the
 *         fp8 range, and submission 599694's fp8 path dequantises as code * kv_scale):
 *         S.EEEE.MMM -> (-1)^S * 2^(E-7) * (1 + M/8) for E>0, (-1)^S * 2^-6 * M/8 for E=0,
 *         S.1111.111 -> NaN (there is no infinity).
 *   e2m1 (OCP MX FP4): S.EE.M -> (-1)^S * {0, 0.5, 1, 1.5, 2, 3, 4, 6}[EEM].
 *         In a packed byte, element 2i is the low nibble and element 2i+1 the high
 *         nibble (submission 700955, `mla_attn_v74` value loop: dim/2 selects the byte,
 *         dim&1 selects the high nibble; dim/32 selects the scale).
 *   e8m0: E -> 2^(E-127); E = 255 -> NaN.  Code 0 decodes to 2^-127 here (OCP); the
 *         pages flush it to 0 (submission 727205 `e8f`, submission 700955 `e8m0f`).  The
 *         synthetic quantiser never emits code 0 (it clamps an all-zero block to E = 127),
 *         and any block whose nibbles are all zero decodes to 0 under either reading.
 *   bf16: the top 16 bits of an IEEE binary32 value (exact in fp64).
 *
 * Empty range (kv_indptr[b] == kv_indptr[b+1]): o = 0, lse = -inf (submission 700955
 * writes po = 0 for an empty split and its combine then yields 0; submission 599694
 * clamps the sum so that an empty row gives 0).
 *
 * Log-sum-exp merge of partial results (the combine step; submission 700955
 * `reduce_lse_v71`, submission 599694 `_flash_fp8_split_s2`, submission 727205 `mla_rd`):
 *     m* = max_s lse_s,  w_s = exp(lse_s - m*),  o = sum_s w_s o_s / sum_s w_s,
 *     lse = m* + log(sum_s w_s); parts with lse = -inf carry no weight; all empty -> 0.
 *
 * Split planning (submission 727205 `mla_s1` and submission 599694 `_flash_fp8_split_s1`):
 *     chunk = ceil(ceil(L / ns) / BN) * BN,  split s covers [s*chunk, min((s+1)*chunk, L)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NH 16
#define ORACLE_D 576
#define ORACLE_DV 512
#define ORACLE_MX_BLOCK 32
#define ORACLE_MX_PACKED 288 /* bytes of nibbles per row */
#define ORACLE_MX_SCALES 18  /* e8m0 scales per row */

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8 = 1, ORACLE_KV_MXFP4 = 2 };

static double g_e4m3[256];
static double g_e2m1[16];
static double g_e8m0[256];
static int g_ready = 0;

static void build_tables(void) {
  if (g_ready) return;
  for (int c = 0; c < 256; ++c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
      v = NAN;
    else if (e == 0)
      v = ldexp((double)m / 8.0, -6);
    else
      v = ldexp(1.0 + (double)m / 8.0, e - 7);
    g_e4m3[c] = s ? -v : v;
  }
  for (int c = 0; c < 16; ++c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    g_e2m1[c] = s ? -v : v;
  }
  for (int c = 0; c < 256; ++c) g_e8m0[c] = (c == 255) ? NAN : ldexp(1.0, c - 127);
  g_ready = 1;
}

double mla_oracle_e4m3(int code) { build_tables(); return g_e4m3[code & 0xFF]; }
double mla_oracle_e2m1(int code) { build_tables(); return g_e2m1[code & 0xF]; }
double mla_oracle_e8m0(int code) { build_tables(); return g_e8m0[code & 0xFF]; }

double mla_oracle_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Dequantise cached row `row` into out[576].
 *   bf16 : kv = uint16 [T][576] (bf16 bits), scale unused.
 *   fp8  : kv = uint8  [T][576] e4m3 codes, scale = float* (one per-tensor value).
 *   mxfp4: kv = uint8  [T][288] packed e2m1, scale = uint8 [T][18] e8m0. */
void mla_oracle_dequant_row(int dtype, const void* kv, const void* scale, int64_t row, double* out) {
  build_tables();
  if (dtype == ORACLE_KV_BF16) {
    const uint16_t* k = (const uint16_t*)kv + row * ORACLE_D;
    for (int d = 0; d < ORACLE_D; ++d) out[d] = mla_oracle_bf16(k[d]);
  } else if (dtype == ORACLE_KV_FP8) {
    const uint8_t* k = (const uint8_t*)kv + row * ORACLE_D;
    double s = (double)(*(const float*)scale);
    for (int d = 0; d < ORACLE_D; ++d) out[d] = g_e4m3[k[d]] * s;
  } else {
    const uint8_t* k = (const uint8_t*)kv + row * ORACLE_MX_PACKED;
    const uint8_t* sc = (const uint8_t*)scale + row * ORACLE_MX_SCALES;
    for (int d = 0; d < ORACLE_D; ++d) {
      int byte = k[d / 2];
      int nib = (d & 1) ? (byte >> 4) : (byte & 0xF);
      out[d] = g_e2m1[nib] * g_e8m0[sc[d / ORACLE_MX_BLOCK]];
    }
  }
}

/* Attention of one batch row (q_b = 16 x 576 bf16 bits) over cached rows [r0, r1).
 * o[16][512] and lse[16] receive the normalised output and log-sum-exp (natural log).
 * Returns 0, or -1 on allocation failure. */
int mla_oracle_attend(const uint16_t* q_b, int dtype, const void* kv, const void* scale,
                      int64_t r0, int64_t r1, double* o, double* lse) {
  build_tables();
  const double sm_scale = 1.0 / sqrt((double)ORACLE_D);
  int64_t L = r1 - r0;
  for (int i = 0; i < ORACLE_NH * ORACLE_DV; ++i) o[i] = 0.0;
  if (L <= 0) {
    for (int h = 0; h < ORACLE_NH; ++h) lse[h] = -INFINITY;
    return 0;
  }
  double q[ORACLE_NH][ORACLE_D];
  for (int h = 0; h < ORACLE_NH; ++h)
    for (int d = 0; d < ORACLE_D; ++d) q[h][d] = mla_oracle_bf16(q_b[h * ORACLE_D + d]);
  double* s = (double*)malloc(sizeof(double) * (size_t)L * ORACLE_NH);
  if (!s) return -1;
  double k[ORACLE_D];
  /* logits s[r][h] */
  for (int64_t r = 0; r < L; ++r) {
    mla_oracle_dequant_row(dtype, kv, scale, r0 + r, k);
    for (int h = 0; h < ORACLE_NH; ++h) {
      double acc = 0.0;
      for (int d = 0; d < ORACLE_D; ++d) acc += q[h][d] * k[d];
      s[r * ORACLE_NH + h] = acc * sm_scale;
    }
  }
  double m[ORACLE_NH], z[ORACLE_NH];
  for (int h = 0; h < ORACLE_NH; ++h) {
    m[h] = -INFINITY;
    for (int64_t r = 0; r < L; ++r) m[h] = fmax(m[h], s[r * ORACLE_NH + h]);
    z[h] = 0.0;
    for (int64_t r = 0; r < L; ++r) z[h] += exp(s[r * ORACLE_NH + h] - m[h]);
  }
  /* o = sum_r p_r * V_r */
  for (int64_t r = 0; r < L; ++r) {
    mla_oracle_dequant_row(dtype, kv, scale, r0 + r, k);
    for (int h = 0; h < ORACLE_NH; ++h) {
      double p = exp(s[r * ORACLE_NH + h] - m[h]) / z[h];
      double* oh = o + h * ORACLE_DV;
      for (int d = 0; d < ORACLE_DV; ++d) oh[d] += p * k[d];
    }
  }
  for (int h = 0; h < ORACLE_NH; ++h) lse[h] = m[h] + log(z[h]);
  free(s);
  return 0;
}

/* Whole decode: q [batch][16][576] bf16 bits, kv_indptr [batch+1].
 * out [batch][16][512] fp64, lse [batch][16] (may be NULL).  nthreads <= 0: library default.
 * Returns 0, or -1 on failure. */
int mla_oracle_decode(const uint16_t* q, int dtype, const void* kv, const void* scale,
                      const int32_t* kv_indptr, int batch, double* out, double* lse, int nthreads) {
  build_tables();
  int fail = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
#endif
  for (int b = 0; b < batch; ++b) {
    double l16[ORACLE_NH];
    int rc = mla_oracle_attend(q + (size_t)b * ORACLE_NH * ORACLE_D, dtype, kv, scale, kv_indptr[b],
                               kv_indptr[b + 1], out + (size_t)b * ORACLE_NH * ORACLE_DV, l16);
    if (rc) fail |= 1;
    if (lse)
      for (int h = 0; h < ORACLE_NH; ++h) lse[b * ORACLE_NH + h] = l16[h];
  }
  (void)nthreads;
  return fail ? -1 : 0;
}

/* Log-sum-exp merge of ns partial results for one batch row:
 * o_s [ns][16][512] (each normalised over its own part), lse_s [ns][16].
 * out [16][512], lse_out [16] (may be NULL). */
void mla_oracle_combine(int ns, const double* o_s, const double* lse_s, double* out, double* lse_out) {
  for (int h = 0; h < ORACLE_NH; ++h) {
    double m = -INFINITY;
    for (int s = 0; s < ns; ++s) m = fmax(m, lse_s[s * ORACLE_NH + h]);
    double* oh = out + h * ORACLE_DV;
    for (int d = 0; d < ORACLE_DV; ++d) oh[d] = 0.0;
    if (m == -INFINITY) {
      if (lse_out) lse_out[h] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int s = 0; s < ns; ++s) {
      double l = lse_s[s * ORACLE_NH + h];
      if (l == -INFINITY) continue;
      double w = exp(l - m);
      wsum += w;
      const double* os = o_s + ((size_t)s * ORACLE_NH + h) * ORACLE_DV;
      for (int d = 0; d < ORACLE_DV; ++d) oh[d] += w * os[d];
    }
    for (int d = 0; d < ORACLE_DV; ++d) oh[d] /= wsum;
    if (lse_out) lse_out[h] = m + log(wsum);
  }
}

/* Token range [n0, n1) (relative to the sequence start) of split s when a sequence of
 * length L is cut into ns splits of `bn`-rounded chunks.  Splits past the end are empty. */
void mla_oracle_split_range(int64_t L, int ns, int bn, int s, int64_t* n0, int64_t* n1) {
  int64_t per = (L + ns - 1) / ns;
  int64_t chunk = ((per + bn - 1) / bn) * bn;
  int64_t a = (int64_t)s * chunk, b = a + chunk;
  if (a > L) a = L;
  if (b > L) b = L;
  *n0 = a;
  *n1 = b;
}

int mla_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
