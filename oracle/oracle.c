/*
 * oracle.c -- plain CPU oracle of the single-GPU MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file's library.
 * It shares no code with the GPU path (no header, table or helper in common).
 *
 * What it computes (flashinfer PR #4069 "SM90 push FP8 mega-MoE backend",
 * Description, the forward diagram: compact -> FC1 with SwiGLU + 1x128
 * quantization -> FC2 -> combine with FP32 route reduction), restricted to one
 * GPU, where dispatch is a local stable permute and combine a local reduce:
 *
 *   1. route    validate (expert id in [0,E) or -1, no duplicate active id
 *               per token, finite weight on active routes); counts[E];
 *               exclusive scan offsets[E+1]; stable counting sort of the
 *               active routes by expert keyed by flat route id r = t*K + k
 *               giving perm[pos] = r and inv[r] = pos (or -1 when masked).
 *   2. quant    1x128 activation quantisation: per row and 128-column block,
 *               s = the smallest power of two with amax <= 448*s (s = 1 when
 *               amax = 0; the exponent is kept in [-127, 127], the range of
 *               an E8M0 scale), q = E4M3FN round-to-nearest-even of v/s.
 *   3. gather   A[pos] = xq[perm[pos] / K], As[pos] = xs[perm[pos] / K].
 *   4. FC1      gu[pos, n] = BF16( sum_kb ( sum_{j in kb} dec(A)*dec(W1[e,n,j]) )
 *                                          * As[pos,kb] * W1s[e, n/128, kb] ),
 *               W1 rows [0, I) are the gate, [I, 2I) the up projection.
 *   5. SwiGLU   h = float( g / (1 + exp(-g)) * u ), g, u the bf16 gu values.
 *   6. requant  hq, hs = quant1x128(h) along I.
 *   7. FC2      y[pos, c] = BF16( sum_kb (sum_j dec(hq)*dec(W2[e,c,j])) * hs * W2s ).
 *   8. combine  out[t, c] = BF16( sum over active k, ascending, of
 *                                 w[t,k] * y[inv[t*K+k], c] ); no route -> +0.
 *
 * Exactness: every E4M3 value is a multiple of 2^-9 with magnitude <= 448, so
 * each product is a multiple of 2^-18 below 2^18 and every 128-term block sum
 * is a multiple of 2^-18 below 2^25: at most 43 significant bits, exact in
 * double in any order.  Scaling by powers of two is exact.  Only the final sum
 * over the H/128 (or I/128) block terms rounds, at 2^-53 relative, before the
 * one BF16 rounding.  Because block sums are exact, the compiler may evaluate
 * them in any order (the simd pragma); no result changes.
 *
 * Format 2 (per-tensor scales, the "per_tensor" mode of flashinfer PR #4688)
 * is defined beside its functions below.
 *
 * Format 1 (MXFP8, "32e4m3xe8m0" on flashinfer PR #4688 and the SM100 MXFP8
 * megakernels of PR #4069's kernel drops): E4M3 values with one power-of-two
 * scale per 32 consecutive elements along K -- activations 1x32 (steps 2 and
 * 6), each weight row 1x32 -- with the same scale rule per 32-block.  Steps
 * 4 and 7 then sum 32-wide exact block sums, each times its activation and
 * weight-row scales.  Format 0 is the DeepSeek 1x128 / 128x128 layout above.
 *
 * Readings where the pages are silent (listed with their reasons in the
 * design notes): E4M3 is the OCP E4M3FN variant (max 448, NaN 0x7F/0xFF, no
 * infinity); scales are powers of two; gate/up are rounded to BF16 before
 * SwiGLU and h stays float into the re-quantisation; y is BF16; the sort is
 * stable in flat route id; offsets are unpadded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_ERR_ROUTE_RANGE 0x1u
#define OR_ERR_ROUTE_DUP 0x2u
#define OR_ERR_ROUTE_NONFINITE 0x4u

/* ---------------------------------------------------------------------------
 * Number formats, from their definitions.
 * ------------------------------------------------------------------------- */

/* OCP FP8 E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is
 * no infinity, so the largest finite value is 1.75 * 2^8 = 448. */
double or_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int ef = (code >> 3) & 0xF;
  int m = code & 7;
  double v;
  if (ef == 15 && m == 7) return NAN;
  if (ef == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, ef - 7);
  return sign ? -v : v;
}

/* round a non-negative double to an integer, ties to even */
static double round_half_even(double q) {
  double f = floor(q);
  double d = q - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* nearest E4M3FN code to v (ties to even mantissa), saturating to +-448.
 * The sign is kept, so values that round to zero from below give 0x80. */
uint8_t or_e4m3_encode(double v) {
  uint8_t sign = (signbit(v) != 0) ? 0x80 : 0x00;
  double a = fabs(v);
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9 */
    double m = round_half_even(ldexp(a, 9)); /* 0..8; 8 is the smallest normal */
    return sign | (uint8_t)m;
  }
  int ex;
  frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1; /* a in [2^e, 2^(e+1)) */
  double m = round_half_even((ldexp(a, -e) - 1.0) * 8.0); /* 0..8 */
  if (m == 8.0) {
    m = 0.0;
    e += 1;
  }
  int ef = e + 7;
  if (ef > 15 || (ef == 15 && m == 7.0)) return sign | 0x7E;
  return sign | (uint8_t)((ef << 3) | (int)m);
}

/* BF16: 1 sign, 8 exponent bits (bias 127), 7 mantissa bits; subnormals are
 * multiples of 2^-133.  Round a double once, to nearest, ties to even. */
uint16_t or_bf16_round(double v) {
  uint16_t sign = (signbit(v) != 0) ? 0x8000 : 0x0000;
  double a = fabs(v);
  if (isnan(v)) return 0x7FC0;
  if (isinf(v)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);
  int e = ex - 1;              /* a in [2^e, 2^(e+1)) */
  if (e < -126) e = -126;      /* subnormal: fixed quantum 2^-133 */
  double m = round_half_even(ldexp(a, 7 - e)); /* significand in units of 2^(e-7) */
  if (m >= 256.0) {
    m = 128.0;
    e += 1;
  }
  if (e > 127) return sign | 0x7F80; /* overflow to infinity */
  if (m < 128.0) return sign | (uint16_t)m; /* subnormal (e == -126) */
  return sign | (uint16_t)(((e + 127) << 7) | ((int)m - 128));
}

double or_bf16_decode(uint16_t b) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)b << 16;
  return (double)c.f;
}

/* smallest e with amax <= 448 * 2^e, kept in [-127, 127]; amax = 0 gives 0 */
int or_pow2_scale_exp(double amax) {
  if (!(amax > 0.0)) return 0;
  int ex;
  frexp(amax / 448.0, &ex); /* first guess, corrected by exact comparisons */
  int e = ex;
  while (448.0 * ldexp(1.0, e) < amax) e++;
  while (e > -200 && 448.0 * ldexp(1.0, e - 1) >= amax) e--;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* ---------------------------------------------------------------------------
 * 1x128 quantisation of rows, and 128x128 quantisation of weight matrices.
 * ------------------------------------------------------------------------- */

/* v [rows, cols] (cols % bw == 0) -> q [rows, cols], s [rows, cols/bw]: one
 * scale per row and bw-wide block (bw = 128: 1x128; bw = 32: MXFP8 1x32) */
void or_quant_rows_bw(const double* v, int64_t rows, int64_t cols, int bw, uint8_t* q, float* s) {
  int64_t nb = cols / bw;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const double* src = v + r * cols + b * bw;
      double amax = 0.0;
      for (int j = 0; j < bw; ++j) amax = fmax(amax, fabs(src[j]));
      int e = or_pow2_scale_exp(amax);
      for (int j = 0; j < bw; ++j) q[r * cols + b * bw + j] = or_e4m3_encode(ldexp(src[j], -e));
      s[r * nb + b] = (float)ldexp(1.0, e);
    }
  }
}

void or_quant_rows(const double* v, int64_t rows, int64_t cols, uint8_t* q, float* s) {
  or_quant_rows_bw(v, rows, cols, 128, q, s);
}

/* bf16 rows -> 1 x bw quantisation */
void or_quant_rows_bf16_bw(const uint16_t* x, int64_t rows, int64_t cols, int bw, uint8_t* q,
                           float* s) {
  double* v = (double*)malloc(sizeof(double) * (size_t)(rows * cols));
  for (int64_t i = 0; i < rows * cols; ++i) v[i] = or_bf16_decode(x[i]);
  or_quant_rows_bw(v, rows, cols, bw, q, s);
  free(v);
}

void or_quant_rows_bf16(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, float* s) {
  or_quant_rows_bf16_bw(x, rows, cols, 128, q, s);
}

/* w [nmat, rows, cols] float -> q (same shape), s [nmat, rows/128, cols/128] */
void or_quant_weights(const float* w, int64_t nmat, int64_t rows, int64_t cols, uint8_t* q,
                      float* s) {
  int64_t rb = rows / 128, cb = cols / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < nmat; ++m) {
    for (int64_t bi = 0; bi < rb; ++bi) {
      for (int64_t bj = 0; bj < cb; ++bj) {
        double amax = 0.0;
        for (int64_t i = 0; i < 128; ++i)
          for (int64_t j = 0; j < 128; ++j)
            amax = fmax(amax, fabs((double)w[(m * rows + bi * 128 + i) * cols + bj * 128 + j]));
        int e = or_pow2_scale_exp(amax);
        for (int64_t i = 0; i < 128; ++i)
          for (int64_t j = 0; j < 128; ++j) {
            int64_t o = (m * rows + bi * 128 + i) * cols + bj * 128 + j;
            q[o] = or_e4m3_encode(ldexp((double)w[o], -e));
          }
        s[(m * rb + bi) * cb + bj] = (float)ldexp(1.0, e);
      }
    }
  }
}

/* MXFP8 weights: w [nmat, rows, cols] float -> q, s [nmat, rows, cols/32]:
 * every row quantised 1x32 along K */
void or_quant_weights_mx(const float* w, int64_t nmat, int64_t rows, int64_t cols, uint8_t* q,
                         float* s) {
  double* v = (double*)malloc(sizeof(double) * (size_t)(rows * cols));
  for (int64_t m = 0; m < nmat; ++m) {
    for (int64_t i = 0; i < rows * cols; ++i) v[i] = (double)w[m * rows * cols + i];
    or_quant_rows_bw(v, rows, cols, 32, q + m * rows * cols, s + m * rows * (cols / 32));
  }
  free(v);
}

/* ---------------------------------------------------------------------------
 * NVFP4 checkpoint weights (flashinfer PR #4069, Reviewer notes: NVFP4
 * checkpoints ride the FP8 backend unchanged through a one-time
 * requantization).  An NVFP4 matrix [rows, cols] holds E2M1 codes packed two
 * per byte along the columns (column 2b in the low nibble of byte b, column
 * 2b+1 in the high nibble), one E4M3 scale per 16 consecutive columns of a
 * row and one float scale per matrix:
 *   value = e2m1(code) * e4m3(block scale) * global,
 * rounded to float once (the first product is exact).  The requantization
 * is the 128x128 weight quantiser above applied to these float values.
 * ------------------------------------------------------------------------- */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent
 * field 0 is the subnormal m * 0.5.  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double or_e2m1_decode(uint8_t nibble) {
  const int sgn = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sgn ? -mag : mag;
}

/* codes [nmat, rows, cols/2], sblk [nmat, rows, cols/16] E4M3, g [nmat]
 * -> out float [nmat, rows, cols].  The double product is exact (at most 30
 * significant bits), so the one conversion to float is the only rounding. */
void or_dequant_nvfp4(const uint8_t* codes, const uint8_t* sblk, const float* g, int64_t nmat,
                      int64_t rows, int64_t cols, float* out) {
  for (int64_t m = 0; m < nmat; ++m)
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t c = 0; c < cols; ++c) {
        const int64_t row = m * rows + r;
        const uint8_t nib = (uint8_t)((codes[row * (cols / 2) + c / 2] >> (4 * (c & 1))) & 0xF);
        const double v = or_e2m1_decode(nib) * or_e4m3_decode(sblk[row * (cols / 16) + c / 16]) *
                         (double)g[m];
        out[row * cols + c] = (float)v;
      }
}

/* ---------------------------------------------------------------------------
 * Routing: validation, histogram, exclusive scan, stable scatter.
 * ------------------------------------------------------------------------- */

/* Returns the error bits.  Routes whose id is out of range are flagged and
 * then treated as masked; duplicates are flagged and kept. */
uint32_t or_route(int64_t T, int K, int E, const int32_t* idx, const float* w, int check,
                  int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv) {
  uint32_t err = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      int32_t id = idx[t * K + k];
      if (id == -1) continue;
      if (id < 0 || id >= E) {
        err |= OR_ERR_ROUTE_RANGE;
        continue;
      }
      if (check) {
        for (int k2 = 0; k2 < k; ++k2)
          if (idx[t * K + k2] == id) err |= OR_ERR_ROUTE_DUP;
        if (!isfinite(w[t * K + k])) err |= OR_ERR_ROUTE_NONFINITE;
      }
    }
  }
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t r = 0; r < T * K; ++r)
    if (idx[r] >= 0 && idx[r] < E) counts[idx[r]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int64_t r = 0; r < T * K; ++r) {
    int32_t id = idx[r];
    if (id >= 0 && id < E) {
      int32_t pos = offsets[id] + cursor[id]++;
      perm[pos] = (int32_t)r;
      inv[r] = pos;
    } else {
      inv[r] = -1;
    }
  }
  free(cursor);
  return err;
}

/* ---------------------------------------------------------------------------
 * One FP8 block-scaled row-times-matrix product.
 * Format 0: row a (len K, scales as[K/128]), matrix W [N, K] with block
 *   scales ws [N/128, K/128]:
 *   out[n] = BF16( sum_kb blocksum_128(kb) * as[kb] * ws[n/128, kb] ).
 * Format 1 (MXFP8): scales as[K/32] and ws [N, K/32]:
 *   out[n] = BF16( sum_b blocksum_32(b) * as[b] * ws[n, b] ).
 * ------------------------------------------------------------------------- */
static void fp8_row_matmul(int fmt, const double* a, const float* as, const double* Wd,
                           const float* ws, int64_t N, int64_t Kd, uint16_t* out) {
  const int bw = fmt == 1 ? 32 : 128;
  const int64_t nb = Kd / bw;
  for (int64_t n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
      const double* ar = a + b * bw;
      const double* wr = Wd + n * Kd + b * bw;
      double bs = 0.0;
#pragma omp simd reduction(+ : bs)
      for (int j = 0; j < bw; ++j) bs += ar[j] * wr[j];
      const double wsc = fmt == 1 ? (double)ws[n * nb + b] : (double)ws[(n / 128) * nb + b];
      acc += bs * (double)as[b] * wsc;
    }
    out[n] = or_bf16_round(acc);
  }
}

static void decode_e4m3_array(const uint8_t* q, int64_t n, double* out) {
  double table[256];
  for (int c = 0; c < 256; ++c) table[c] = or_e4m3_decode((uint8_t)c);
  for (int64_t i = 0; i < n; ++i) out[i] = table[q[i]];
}

/* SwiGLU of one bf16 gate/up pair, rounded once to float */
float or_swiglu(uint16_t g_bits, uint16_t u_bits) {
  double g = or_bf16_decode(g_bits), u = or_bf16_decode(u_bits);
  return (float)(g / (1.0 + exp(-g)) * u);
}

/* ---------------------------------------------------------------------------
 * The expert FFN of one sorted position: A row -> gu -> h -> hq/hs -> y.
 * Positions are processed expert by expert so each expert's weights are
 * decoded once.  `sel` (nullable) marks which positions to compute.
 * ------------------------------------------------------------------------- */
void or_expert_ffn_fmt(int fmt, int H, int I, int E, const int32_t* offsets, const uint8_t* A,
                       const float* As, const uint8_t* W1, const float* W1s, const uint8_t* W2,
                       const float* W2s, const uint8_t* sel, uint16_t* gu, uint8_t* hq, float* hs,
                       uint16_t* y) {
  const int bw = fmt == 1 ? 32 : 128;
  const int64_t HB = H / bw, IB = I / bw;  /* activation scales per row */
  /* weight scales per expert: [2I/128][H/128] and [H/128][I/128], or per row [2I][H/32], [H][I/32] */
  const int64_t w1s_per_e = fmt == 1 ? (int64_t)2 * I * HB : (int64_t)(2 * I / 128) * HB;
  const int64_t w2s_per_e = fmt == 1 ? (int64_t)H * IB : (int64_t)(H / 128) * IB;
  double* w1d = (double*)malloc(sizeof(double) * (size_t)(2 * I) * (size_t)H);
  double* w2d = (double*)malloc(sizeof(double) * (size_t)H * (size_t)I);
  for (int e = 0; e < E; ++e) {
    int64_t p0 = offsets[e], p1 = offsets[e + 1];
    int any = 0;
    for (int64_t p = p0; p < p1; ++p)
      if (!sel || sel[p]) any = 1;
    if (!any) continue;
    decode_e4m3_array(W1 + (int64_t)e * 2 * I * H, (int64_t)2 * I * H, w1d);
    decode_e4m3_array(W2 + (int64_t)e * H * I, (int64_t)H * I, w2d);
    const float* w1s = W1s + (int64_t)e * w1s_per_e;
    const float* w2s = W2s + (int64_t)e * w2s_per_e;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = p0; p < p1; ++p) {
      if (sel && !sel[p]) continue;
      double* a = (double*)malloc(sizeof(double) * (size_t)H);
      double* h = (double*)malloc(sizeof(double) * (size_t)I);
      double* hd = (double*)malloc(sizeof(double) * (size_t)I);
      uint16_t* gup = gu + p * 2 * I;
      decode_e4m3_array(A + p * H, H, a);
      fp8_row_matmul(fmt, a, As + p * HB, w1d, w1s, 2 * I, H, gup);
      for (int n = 0; n < I; ++n) h[n] = (double)or_swiglu(gup[n], gup[I + n]);
      or_quant_rows_bw(h, 1, I, bw, hq + p * I, hs + p * IB);
      decode_e4m3_array(hq + p * I, I, hd);
      fp8_row_matmul(fmt, hd, hs + p * IB, w2d, w2s, H, I, y + p * H);
      free(a);
      free(h);
      free(hd);
    }
  }
  free(w1d);
  free(w2d);
}

void or_expert_ffn(int H, int I, int E, const int32_t* offsets, const uint8_t* A, const float* As,
                   const uint8_t* W1, const float* W1s, const uint8_t* W2, const float* W2s,
                   const uint8_t* sel, uint16_t* gu, uint8_t* hq, float* hs, uint16_t* y) {
  or_expert_ffn_fmt(0, H, I, E, offsets, A, As, W1, W1s, W2, W2s, sel, gu, hq, hs, y);
}

/* combine: out[t, c] = BF16( sum_k active  w[t,k] * y[inv[t*K+k], c] ) */
void or_combine(int64_t T, int K, int H, const int32_t* inv, const float* w, const uint16_t* y,
                const uint8_t* tok_sel, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    if (tok_sel && !tok_sel[t]) continue;
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        int32_t p = inv[t * K + k];
        if (p < 0) continue;
        acc += (double)w[t * K + k] * or_bf16_decode(y[(int64_t)p * H + c]);
      }
      out[t * H + c] = or_bf16_round(acc);
    }
  }
}

/* ---------------------------------------------------------------------------
 * The whole forward.  Intermediate outputs are optional (nullable) except the
 * ones the caller needs; `tok_sel` (nullable) restricts the expert FFN and the
 * combine to the selected tokens (routing always covers every token).
 * Returns the route error bits; on error nothing past routing is computed.
 * ------------------------------------------------------------------------- */
uint32_t or_forward_fmt(int fmt, int64_t T, int H, int I, int E, int K, int check,
                        const uint16_t* x, const int32_t* idx, const float* w, const uint8_t* W1,
                        const float* W1s, const uint8_t* W2, const float* W2s,
                        const uint8_t* tok_sel, int32_t* counts, int32_t* offsets, int32_t* perm,
                        int32_t* inv, uint8_t* xq, float* xs, uint8_t* A, float* As, uint16_t* gu,
                        uint8_t* hq, float* hs, uint16_t* y, uint16_t* out) {
  uint32_t err = or_route(T, K, E, idx, w, check, counts, offsets, perm, inv);
  if (err) return err;
  const int bw = fmt == 1 ? 32 : 128;
  const int64_t R = offsets[E], HB = H / bw;
  or_quant_rows_bf16_bw(x, T, H, bw, xq, xs);
  uint8_t* sel = NULL;
  if (tok_sel) {
    sel = (uint8_t*)calloc((size_t)(R > 0 ? R : 1), 1);
    for (int64_t p = 0; p < R; ++p) sel[p] = tok_sel[perm[p] / K];
  }
  for (int64_t p = 0; p < R; ++p) {
    int64_t t = perm[p] / K;
    memcpy(A + p * H, xq + t * H, (size_t)H);
    memcpy(As + p * HB, xs + t * HB, sizeof(float) * (size_t)HB);
  }
  or_expert_ffn_fmt(fmt, H, I, E, offsets, A, As, W1, W1s, W2, W2s, sel, gu, hq, hs, y);
  or_combine(T, K, H, inv, w, y, tok_sel, out);
  free(sel);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Format 2: per-tensor FP8, the "per_tensor" scale mode of flashinfer PR #4688
 * (Description, the scale-mode-equalized comparison: per_tensor needs
 * offline-calibrated activation scales, blockwise needs none).  One FP32 scale
 * per expert weight matrix and one static, calibrated FP32 scale per
 * activation tensor (x, and the SwiGLU output h); no block scales.
 *
 *   quantise v with scale s:  q = E4M3_RNE_sat( float(v) * r ),  r = float(1 / s)
 *       (r is the float division 1/s rounded once; the float product is rounded
 *       once and then encoded; |v * r| >= 448 saturates to +-448)
 *   weight scale of a matrix: s = float(amax / 448), or 1 for an all-zero matrix
 *   FC1:  gu[pos, n] = BF16( (sum_j dec(A[pos,j]) * dec(W1[e,n,j])) * s_x * s_w1[e] )
 *   FC2:  y[pos, c]  = BF16( (sum_j dec(hq[pos,j]) * dec(W2[e,c,j])) * s_h * s_w2[e] )
 *
 * Every product of two E4M3 values is a multiple of 2^-18 below 2^18, so a sum
 * of up to 2^17 of them is an integer multiple of 2^-18 below 2^53 of those
 * units: exact in double.  The two float scales multiply exactly in double
 * (24-bit significands).  Only the final BF16 rounding rounds.  SwiGLU and
 * combine are as in format 0.
 * ------------------------------------------------------------------------- */

/* one quantisation step of format 2: float product, then the E4M3 encoder */
static uint8_t pt_encode(float v, float r) {
  const float p = v * r;
  return or_e4m3_encode((double)p);
}

/* scale of one weight matrix of n floats */
float or_pt_weight_scale(const float* w, int64_t n) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    const float a = fabsf(w[i]);
    if (a > amax) amax = a;
  }
  return amax > 0.0f ? amax / 448.0f : 1.0f;
}

/* w [nmat, rows, cols] float -> q (same shape), s [nmat] */
void or_quant_weights_pt(const float* w, int64_t nmat, int64_t rows, int64_t cols, uint8_t* q,
                         float* s) {
  const int64_t n = rows * cols;
  for (int64_t m = 0; m < nmat; ++m) {
    const float sc = or_pt_weight_scale(w + m * n, n);
    const float r = 1.0f / sc;
    s[m] = sc;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) q[m * n + i] = pt_encode(w[m * n + i], r);
  }
}

/* n float values (given as double, each exactly a float) with static scale s */
void or_quant_values_pt(const double* v, int64_t n, float s, uint8_t* q) {
  const float r = 1.0f / s;
  for (int64_t i = 0; i < n; ++i) q[i] = pt_encode((float)v[i], r);
}

/* exact sum_j dec(a[j]) * dec(w[j]) over n terms (decoded values) */
static double dot_exact(const double* a, const double* w, int64_t n) {
  double acc = 0.0;
#pragma omp simd reduction(+ : acc)
  for (int64_t j = 0; j < n; ++j) acc += a[j] * w[j];
  return acc;
}

/* The whole forward in format 2.  W1s / W2s are [E]; x_scale and h_scale the
 * static activation scales.  Outputs as or_forward_fmt, without the per-row
 * scale arrays (the block scales are all 1).  Returns the route error bits. */
uint32_t or_forward_pt(int64_t T, int H, int I, int E, int K, int check, const uint16_t* x,
                       const int32_t* idx, const float* w, const uint8_t* W1, const float* W1s,
                       const uint8_t* W2, const float* W2s, float x_scale, float h_scale,
                       const uint8_t* tok_sel, int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv, uint8_t* xq, uint8_t* A, uint16_t* gu, uint8_t* hq,
                       uint16_t* y, uint16_t* out) {
  uint32_t err = or_route(T, K, E, idx, w, check, counts, offsets, perm, inv);
  if (err) return err;
  const int64_t R = offsets[E];
  /* 1. quantise x with the static scale */
  {
    const float rx = 1.0f / x_scale;
    for (int64_t i = 0; i < T * (int64_t)H; ++i) xq[i] = pt_encode((float)or_bf16_decode(x[i]), rx);
  }
  /* 2. gather */
  for (int64_t p = 0; p < R; ++p) memcpy(A + p * H, xq + (int64_t)(perm[p] / K) * H, (size_t)H);
  /* 3. expert FFN, expert by expert */
  const float rh = 1.0f / h_scale;
  double* w1d = (double*)malloc(sizeof(double) * (size_t)(2 * I) * (size_t)H);
  double* w2d = (double*)malloc(sizeof(double) * (size_t)H * (size_t)I);
  for (int e = 0; e < E; ++e) {
    const int64_t p0 = offsets[e], p1 = offsets[e + 1];
    int any = 0;
    for (int64_t p = p0; p < p1; ++p)
      if (!tok_sel || tok_sel[perm[p] / K]) any = 1;
    if (!any) continue;
    decode_e4m3_array(W1 + (int64_t)e * 2 * I * H, (int64_t)2 * I * H, w1d);
    decode_e4m3_array(W2 + (int64_t)e * H * I, (int64_t)H * I, w2d);
    const double f1 = (double)x_scale * (double)W1s[e];
    const double f2 = (double)h_scale * (double)W2s[e];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = p0; p < p1; ++p) {
      if (tok_sel && !tok_sel[perm[p] / K]) continue;
      double* a = (double*)malloc(sizeof(double) * (size_t)H);
      double* hd = (double*)malloc(sizeof(double) * (size_t)I);
      uint16_t* gup = gu + p * 2 * I;
      decode_e4m3_array(A + p * H, H, a);
      for (int n = 0; n < 2 * I; ++n) gup[n] = or_bf16_round(dot_exact(a, w1d + (int64_t)n * H, H) * f1);
      for (int n = 0; n < I; ++n) hq[p * I + n] = pt_encode(or_swiglu(gup[n], gup[I + n]), rh);
      decode_e4m3_array(hq + p * I, I, hd);
      for (int c = 0; c < H; ++c)
        y[p * H + c] = or_bf16_round(dot_exact(hd, w2d + (int64_t)c * I, I) * f2);
      free(a);
      free(hd);
    }
  }
  free(w1d);
  free(w2d);
  or_combine(T, K, H, inv, w, y, tok_sel, out);
  return 0;
}

uint32_t or_forward(int64_t T, int H, int I, int E, int K, int check, const uint16_t* x,
                    const int32_t* idx, const float* w, const uint8_t* W1, const float* W1s,
                    const uint8_t* W2, const float* W2s, const uint8_t* tok_sel,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                    uint8_t* xq, float* xs, uint8_t* A, float* As, uint16_t* gu, uint8_t* hq,
                    float* hs, uint16_t* y, uint16_t* out) {
  return or_forward_fmt(0, T, H, I, E, K, check, x, idx, w, W1, W1s, W2, W2s, tok_sel, counts,
                        offsets, perm, inv, xq, xs, A, As, gu, hq, hs, y, out);
}
