/*
 * tq1_oracle.c -- plain, slow, CPU oracle for the TQ1_0 ternary mat-vec (and
 * its 2-bit sibling TQ2_0).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant generator with
 * the CUDA library.
 *
 * Sources ("the pages"):
 *   [P1] PrismML-Eng/llama.cpp issue #139, "CUDA: TQ1_0 mat-vec is load-bound
 *        by the per-32-element chunk contract", sections "Current behavior"
 *        (five trits per byte in base 3; chunk c of a 256-element block reads
 *        digit c of bytes qs[0..31]) and "Upstream state" (powers of three).
 *   [SPEC] the block layout fixed alongside the pages: qs[48] (5 trits per
 *        byte), qh[4] (4 trits per byte), fp16 d; 54 bytes per block.  Byte
 *        code b = ceil((sum_i t_i*3^(4-i)) * 256/243); digit k of a byte is
 *        ((uint8)(b*3^k) * 3) >> 8; digit 0/1/2 means -1/0/+1.  Q8_1: 32 int8
 *        values with an fp16 scale and an fp16 sum.
 *
 * Readings where the pages are silent:
 *   R1 element order after element 160 continues the P1 pattern over the
 *      remaining 16 qs bytes, then over the 4 qh bytes (see tq1_elem_pos).
 *   R2 field order qs @0, qh @48, d @52 (little-endian fp16).
 *   R3 weight quantisation: d = fp16(amax); t = amax ? clamp(round_half_away(
 *      w / amax), -1, 1) : 0 (fp32 IEEE divide).
 *   R4 Q8_1 quantisation: d = amax/127; q = d ? clamp(round_half_away(x / d),
 *      -127, 127) : 0; stored fp16(d) and fp16(d*sum(q)); all fp32, IEEE, no
 *      contraction (built with -ffp-contract=off).  A divide, not a multiply
 *      by 1/d: 1/d overflows for denormal d and 0*inf is NaN, whose integer
 *      conversion differs between CPUs.  The stored sum is metadata and is
 *      never used by the dot product below.
 *   R5 mat-vec-id: token t's activations are used for every one of its
 *      top_k slots; ids outside [0, n_experts) leave their output untouched.
 *   R6 TQ2_0, the 2-bit sibling format P1 "Upstream state" names without a
 *      layout: qs[64] holding four 2-bit codes per byte, then the fp16 d at
 *      byte 64; 66 bytes per 256-element block.  Code = trit + 1 (0/1/2 means
 *      -1/0/+1; the unused code 3 decodes to +2).  Element order continues
 *      P1's chunk pattern with four codes per byte: chunk c (elements 32c ..
 *      32c+31) reads code c % 4 (bits 2(c%4)..2(c%4)+1) of bytes qs[32(c/4)
 *      .. 32(c/4)+31].  Quantisation from fp32 as R3.  Parity of this layout
 *      is unpinned by the pages; the tests pin the arithmetic on it against
 *      the TQ1_0 oracle (same trits, same outputs).
 *
 * Every floating-point result of the dot product is computed in fp64: each
 * product d_w*d_a*I is exact in fp64 (11+11+13 significant bits), so the
 * oracle is exact up to the final fp64 summation rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_QK 256            /* weights per TQ1_0 block          */
#define ORC_BLOCK_BYTES 54    /* qs[48] + qh[4] + fp16 d          */
#define ORC_TQ2_BYTES 66      /* R6: qs[64] + fp16 d              */
#define ORC_QK8 32            /* activations per Q8_1 block       */
#define ORC_Q8_BYTES 36       /* fp16 d + fp16 s + int8 q[32]     */

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format definition. */
/* ------------------------------------------------------------------ */

/* Round a float to the nearest binary16 (ties to even), keeping subnormals,
 * overflowing to infinity.  Method: pick the binade exponent E (clamped at
 * the subnormal floor -14), express |f| in units of the binade's quantum
 * 2^(E-10) (exact in fp64), round that count to the nearest integer with
 * ties to even, and re-normalise if the rounding carried into the next
 * binade. */
uint16_t orc_f16_from_f32(float f) {
  const uint16_t sign = signbit(f) ? 0x8000u : 0u;
  if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
  if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
  const double a = fabs((double)f);
  if (a == 0.0) return sign;
  int e2 = 0;
  (void)frexp(a, &e2); /* a = fr * 2^e2, fr in [0.5, 1) */
  int E = e2 - 1;      /* floor(log2(a)) */
  if (E < -14) E = -14;
  const double quantum = ldexp(1.0, E - 10);
  double M = nearbyint(a / quantum); /* default mode: nearest, ties even */
  if (M >= 2048.0) {
    E += 1;
    M *= 0.5;
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  if (M < 1024.0) return (uint16_t)(sign | (uint16_t)M); /* subnormal */
  return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | ((int)M - 1024)));
}

float orc_f32_from_f16(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m + 1024), e - 25);
  return (float)(s ? -v : v);
}

/* ------------------------------------------------------------------ */
/* TQ1_0 byte code.                                                    */
/* ------------------------------------------------------------------ */

static const int orc_pow3[6] = {1, 3, 9, 27, 81, 243};

/* Element e (0..255) of a block lives in byte *byte_idx at base-3 digit
 * *digit.  P1 "Current behavior": chunk c (elements 32c..32c+31, c < 5)
 * reads digit c of qs[0..31].  R1: elements 160..239 follow the same
 * pattern over qs[32..47] in strides of 16, elements 240..255 over qh[0..3]
 * in strides of 4. */
void orc_tq1_elem_pos(int e, int* byte_idx, int* digit) {
  if (e < 160) {
    *byte_idx = e % 32;
    *digit = e / 32;
  } else if (e < 240) {
    *byte_idx = 32 + (e - 160) % 16;
    *digit = (e - 160) / 16;
  } else {
    *byte_idx = 48 + (e - 240) % 4;
    *digit = (e - 240) / 4;
  }
}

/* SPEC: byte holding trits u_0..u_4 (u in {0,1,2}, u_0 most significant). */
uint8_t orc_tq1_pack_byte(const int u[5]) {
  int v = 0;
  for (int i = 0; i < 5; ++i) v = v * 3 + u[i];
  return (uint8_t)((v * 256 + 242) / 243); /* integer ceil(v*256/243) */
}

/* SPEC: digit k (0..4) of a packed byte. */
int orc_tq1_digit(uint8_t b, int k) {
  const uint8_t m = (uint8_t)(b * orc_pow3[k]);
  return (m * 3) >> 8;
}

/* R3: quantise one 256-weight block to TQ1_0. */
static void orc_tq1_encode_block(const float* x, uint8_t* blk) {
  float amax = 0.0f;
  for (int i = 0; i < ORC_QK; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  const uint16_t d16 = orc_f16_from_f32(amax);
  int u[ORC_QK];
  for (int i = 0; i < ORC_QK; ++i) {
    float r = amax != 0.0f ? roundf(x[i] / amax) : 0.0f; /* roundf: halves away from zero */
    if (r > 1.0f) r = 1.0f;
    if (r < -1.0f) r = -1.0f;
    u[i] = (int)r + 1;
  }
  memset(blk, 0, ORC_BLOCK_BYTES);
  /* Gather the five (or four) digits of each byte by walking the element
   * order; digit 4 of the qh bytes stays 0 (R1/SPEC: 4 trits per qh byte). */
  int digits[52][5];
  memset(digits, 0, sizeof(digits));
  for (int e = 0; e < ORC_QK; ++e) {
    int bi, dg;
    orc_tq1_elem_pos(e, &bi, &dg);
    digits[bi][dg] = u[e];
  }
  for (int bi = 0; bi < 52; ++bi) blk[bi] = orc_tq1_pack_byte(digits[bi]);
  blk[52] = (uint8_t)(d16 & 0xFF);
  blk[53] = (uint8_t)(d16 >> 8);
}

/* w: fp32 [n][k], k % 256 == 0.  blocks: [n][k/256] x 54 bytes. */
void orc_tq1_encode_rows(const float* w, uint8_t* blocks, int64_t n, int64_t k) {
  const int64_t nb = k / ORC_QK;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t b = 0; b < nb; ++b)
      orc_tq1_encode_block(w + r * k + b * ORC_QK, blocks + (r * nb + b) * ORC_BLOCK_BYTES);
}

/* Decode to trits t in {-1,0,1} [n][k] and scales d [n][k/256]. */
void orc_tq1_decode_rows(const uint8_t* blocks, int8_t* trits, float* scales, int64_t n, int64_t k) {
  const int64_t nb = k / ORC_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * ORC_BLOCK_BYTES;
      for (int e = 0; e < ORC_QK; ++e) {
        int bi, dg;
        orc_tq1_elem_pos(e, &bi, &dg);
        trits[r * k + b * ORC_QK + e] = (int8_t)(orc_tq1_digit(blk[bi], dg) - 1);
      }
      scales[r * nb + b] = orc_f32_from_f16((uint16_t)(blk[52] | (blk[53] << 8)));
    }
  }
}

/* ------------------------------------------------------------------ */
/* TQ2_0 (R6).                                                         */
/* ------------------------------------------------------------------ */

/* Element e (0..255) of a TQ2_0 block lives in byte *byte_idx, 2-bit field
 * *field (bits 2*field .. 2*field+1). */
void orc_tq2_elem_pos(int e, int* byte_idx, int* field) {
  const int chunk = e / 32;
  *byte_idx = 32 * (chunk / 4) + e % 32;
  *field = chunk % 4;
}

/* Code (0..3) of element e; its value is code - 1. */
int orc_tq2_code(const uint8_t* blk, int e) {
  int bi, f;
  orc_tq2_elem_pos(e, &bi, &f);
  return (blk[bi] >> (2 * f)) & 3;
}

/* R6 + R3: quantise one 256-weight block to TQ2_0. */
static void orc_tq2_encode_block(const float* x, uint8_t* blk) {
  float amax = 0.0f;
  for (int i = 0; i < ORC_QK; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  const uint16_t d16 = orc_f16_from_f32(amax);
  memset(blk, 0, ORC_TQ2_BYTES);
  for (int e = 0; e < ORC_QK; ++e) {
    float r = amax != 0.0f ? roundf(x[e] / amax) : 0.0f; /* roundf: halves away from zero */
    if (r > 1.0f) r = 1.0f;
    if (r < -1.0f) r = -1.0f;
    int bi, f;
    orc_tq2_elem_pos(e, &bi, &f);
    blk[bi] = (uint8_t)(blk[bi] | (((int)r + 1) << (2 * f)));
  }
  blk[64] = (uint8_t)(d16 & 0xFF);
  blk[65] = (uint8_t)(d16 >> 8);
}

/* w: fp32 [n][k], k % 256 == 0.  blocks: [n][k/256] x 66 bytes. */
void orc_tq2_encode_rows(const float* w, uint8_t* blocks, int64_t n, int64_t k) {
  const int64_t nb = k / ORC_QK;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t b = 0; b < nb; ++b)
      orc_tq2_encode_block(w + r * k + b * ORC_QK, blocks + (r * nb + b) * ORC_TQ2_BYTES);
}

/* Decode to values (code - 1) [n][k] and scales d [n][k/256]. */
void orc_tq2_decode_rows(const uint8_t* blocks, int8_t* trits, float* scales, int64_t n, int64_t k) {
  const int64_t nb = k / ORC_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * ORC_TQ2_BYTES;
      for (int e = 0; e < ORC_QK; ++e) trits[r * k + b * ORC_QK + e] = (int8_t)(orc_tq2_code(blk, e) - 1);
      scales[r * nb + b] = orc_f32_from_f16((uint16_t)(blk[64] | (blk[65] << 8)));
    }
  }
}

/* ------------------------------------------------------------------ */
/* Q8_1 activations (R4).                                              */
/* ------------------------------------------------------------------ */

/* x: fp32 [t][k], k % 32 == 0.  out: [t][k/32] x 36 bytes:
 * fp16 d @0, fp16 s @2, int8 q[32] @4. */
void orc_q8_1_quantize(const float* x, uint8_t* out, int64_t t, int64_t k) {
  const int64_t nq = k / ORC_QK8;
  for (int64_t c = 0; c < t; ++c) {
    for (int64_t j = 0; j < nq; ++j) {
      const float* v = x + c * k + j * ORC_QK8;
      uint8_t* o = out + (c * nq + j) * ORC_Q8_BYTES;
      float amax = 0.0f;
      for (int i = 0; i < ORC_QK8; ++i) {
        const float a = fabsf(v[i]);
        if (a > amax) amax = a;
      }
      const float d = amax / 127.0f;
      int sum = 0;
      for (int i = 0; i < ORC_QK8; ++i) {
        float r = d != 0.0f ? roundf(v[i] / d) : 0.0f;
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        const int q = (int)r;
        sum += q;
        o[4 + i] = (uint8_t)(int8_t)q;
      }
      const uint16_t d16 = orc_f16_from_f32(d);
      const uint16_t s16 = orc_f16_from_f32(d * (float)sum);
      o[0] = (uint8_t)(d16 & 0xFF);
      o[1] = (uint8_t)(d16 >> 8);
      o[2] = (uint8_t)(s16 & 0xFF);
      o[3] = (uint8_t)(s16 >> 8);
    }
  }
}

static float orc_q8_scale(const uint8_t* blk) { return orc_f32_from_f16((uint16_t)(blk[0] | (blk[1] << 8))); }

/* ------------------------------------------------------------------ */
/* Dot products.                                                       */
/* ------------------------------------------------------------------ */

/* Weight formats of the dot products below: 1 = TQ1_0, 2 = TQ2_0 (R6). */
static int64_t orc_fmt_bytes(int fmt) { return fmt == 2 ? ORC_TQ2_BYTES : ORC_BLOCK_BYTES; }

/* Value (-1, 0, +1; +2 for TQ2_0's unused code) of element e of a block. */
static int orc_elem_value(int fmt, const uint8_t* wblk, int e) {
  if (fmt == 2) return orc_tq2_code(wblk, e) - 1;
  int bi, dg;
  orc_tq1_elem_pos(e, &bi, &dg);
  return orc_tq1_digit(wblk[bi], dg) - 1;
}

static double orc_block_scale(int fmt, const uint8_t* wblk) {
  const int at = fmt == 2 ? 64 : 52;
  return (double)orc_f32_from_f16((uint16_t)(wblk[at] | (wblk[at + 1] << 8)));
}

/* Integer partial of one row against one column over one 32-element chunk:
 * I = sum over the chunk of (digit - 1) * q.  Elements are visited in
 * natural order and each one's byte/digit is looked up (P1: the CPU walk). */
static int32_t orc_chunk_partial(int fmt, const uint8_t* wblk, const uint8_t* qblk, int chunk) {
  int32_t acc = 0;
  for (int i = 0; i < ORC_QK8; ++i)
    acc += orc_elem_value(fmt, wblk, chunk * ORC_QK8 + i) * (int)(int8_t)qblk[4 + i];
  return acc;
}

/* part[c][r][k/32] = integer per-32 partials (exact). */
static void orc_partials_fmt(int fmt, const uint8_t* blocks, const uint8_t* q8, int32_t* part, int64_t n, int64_t k,
                             int64_t t) {
  const int64_t nb = k / ORC_QK, nq = k / ORC_QK8, bb = orc_fmt_bytes(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t c = 0; c < t; ++c)
      for (int64_t b = 0; b < nb; ++b)
        for (int j = 0; j < 8; ++j)
          part[(c * n + r) * nq + b * 8 + j] =
              orc_chunk_partial(fmt, blocks + (r * nb + b) * bb, q8 + (c * nq + b * 8 + j) * ORC_Q8_BYTES, j);
}

/* y = sum_b d_w[b] * sum_j d_a[8b+j] * I_j   (fp64; natural order). */
static double orc_row_dot(int fmt, const uint8_t* wrow, const uint8_t* qcol, int64_t nb) {
  const int64_t bb = orc_fmt_bytes(fmt);
  double y = 0.0;
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* wblk = wrow + b * bb;
    const double dw = orc_block_scale(fmt, wblk);
    double acc = 0.0;
    for (int j = 0; j < 8; ++j) {
      const uint8_t* qblk = qcol + (b * 8 + j) * ORC_Q8_BYTES;
      acc += (double)orc_q8_scale(qblk) * (double)orc_chunk_partial(fmt, wblk, qblk, j);
    }
    y += dw * acc;
  }
  return y;
}

/* y[c][r] for all rows r < n and columns c < t. */
static void orc_f64_fmt(int fmt, const uint8_t* blocks, const uint8_t* q8, double* y, int64_t n, int64_t k,
                        int64_t t) {
  const int64_t nb = k / ORC_QK, nq = k / ORC_QK8, bb = orc_fmt_bytes(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int64_t c = 0; c < t; ++c)
      y[c * n + r] = orc_row_dot(fmt, blocks + r * nb * bb, q8 + c * nq * ORC_Q8_BYTES, nb);
}

/* Sampled rows: y[c][i] = row rows[i] against column c. */
static void orc_f64_rows_fmt(int fmt, const uint8_t* blocks, const uint8_t* q8, double* y, int64_t k, int64_t t,
                             const int64_t* rows, int64_t nrows) {
  const int64_t nb = k / ORC_QK, nq = k / ORC_QK8, bb = orc_fmt_bytes(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nrows; ++i)
    for (int64_t c = 0; c < t; ++c)
      y[c * nrows + i] = orc_row_dot(fmt, blocks + rows[i] * nb * bb, q8 + c * nq * ORC_Q8_BYTES, nb);
}

void orc_mmv_partials(const uint8_t* blocks, const uint8_t* q8, int32_t* part, int64_t n, int64_t k, int64_t t) {
  orc_partials_fmt(1, blocks, q8, part, n, k, t);
}

void orc_mmv_f64(const uint8_t* blocks, const uint8_t* q8, double* y, int64_t n, int64_t k, int64_t t) {
  orc_f64_fmt(1, blocks, q8, y, n, k, t);
}

void orc_mmv_f64_rows(const uint8_t* blocks, const uint8_t* q8, double* y, int64_t n, int64_t k, int64_t t,
                      const int64_t* rows, int64_t nrows) {
  (void)n;
  orc_f64_rows_fmt(1, blocks, q8, y, k, t, rows, nrows);
}

void orc_tq2_mmv_partials(const uint8_t* blocks, const uint8_t* q8, int32_t* part, int64_t n, int64_t k, int64_t t) {
  orc_partials_fmt(2, blocks, q8, part, n, k, t);
}

void orc_tq2_mmv_f64(const uint8_t* blocks, const uint8_t* q8, double* y, int64_t n, int64_t k, int64_t t) {
  orc_f64_fmt(2, blocks, q8, y, n, k, t);
}

void orc_tq2_mmv_f64_rows(const uint8_t* blocks, const uint8_t* q8, double* y, int64_t n, int64_t k, int64_t t,
                          const int64_t* rows, int64_t nrows) {
  (void)n;
  orc_f64_rows_fmt(2, blocks, q8, y, k, t, rows, nrows);
}

/* R5: y[c][s][r] = expert ids[c][s] (matrix at expert_blocks + e*n*nb*bytes)
 * against token c's activations; only the listed rows (all rows when rows is
 * NULL: y[c][s][r], else y[c][s][i] for row rows[i]). */
static void orc_mmv_id_fmt(int fmt, const uint8_t* expert_blocks, int64_t n_experts, const uint8_t* q8,
                           const int32_t* ids, double* y, int64_t n, int64_t k, int64_t t, int64_t top_k,
                           const int64_t* rows, int64_t nrows) {
  const int64_t nb = k / ORC_QK, nq = k / ORC_QK8, bb = orc_fmt_bytes(fmt);
  const int64_t ebytes = n * nb * bb;
  const int64_t m = rows ? nrows : n;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t c = 0; c < t; ++c) {
    for (int64_t s = 0; s < top_k; ++s) {
      const int32_t e = ids[c * top_k + s];
      if (e < 0 || e >= n_experts) continue;
      for (int64_t i = 0; i < m; ++i) {
        const int64_t r = rows ? rows[i] : i;
        y[(c * top_k + s) * m + i] =
            orc_row_dot(fmt, expert_blocks + e * ebytes + r * nb * bb, q8 + c * nq * ORC_Q8_BYTES, nb);
      }
    }
  }
}

void orc_mmv_id_f64(const uint8_t* expert_blocks, int64_t n_experts, const uint8_t* q8, const int32_t* ids,
                    double* y, int64_t n, int64_t k, int64_t t, int64_t top_k) {
  orc_mmv_id_fmt(1, expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, NULL, 0);
}

/* Sampled variant of mat-vec-id: only the listed rows of every slot. */
void orc_mmv_id_f64_rows(const uint8_t* expert_blocks, int64_t n_experts, const uint8_t* q8, const int32_t* ids,
                         double* y, int64_t n, int64_t k, int64_t t, int64_t top_k, const int64_t* rows,
                         int64_t nrows) {
  orc_mmv_id_fmt(1, expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, rows, nrows);
}

void orc_tq2_mmv_id_f64(const uint8_t* expert_blocks, int64_t n_experts, const uint8_t* q8, const int32_t* ids,
                        double* y, int64_t n, int64_t k, int64_t t, int64_t top_k) {
  orc_mmv_id_fmt(2, expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, NULL, 0);
}

/* Threads the dot products may use from now on (n >= 1). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
