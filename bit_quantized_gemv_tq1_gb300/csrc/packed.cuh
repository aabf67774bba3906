// packed.cuh -- the decode kernels' packed-digit machinery (TQ1_0 x Q8_1 for
// a few token columns), shared by the dense decode kernel and the
// expert-routed one.
//
// Packed digits: a block's 256 trits become 64 digit words (4 digits of 0..2
// per word, one per byte lane).  Four digit words that pair with the same
// activation word index w but belong to Q8_1 chunks j = s, s+1.. (slot s = j
// mod 4) share one register: bits 2s..2s+1 of every byte lane.  Masking slot
// s leaves 4^s * digit in each lane, which an unsigned-by-signed dp4a uses
// directly; the exact factor 4^s is folded into the chunk's fp32 scale and
// -sum(q) seed, so the per-chunk integer partial stays exact.
//
// Work unit ("task"): 4 rows x 8 consecutive 256-blocks; lane = (row r,
// block s).
#pragma once

#include "tq1_device.cuh"

namespace tq1 {
namespace packed {

constexpr int kRowsPerTask = 4;
constexpr int kLanesPerRow = 8;  // = blocks per task chunk

// Shared-memory bytes reserved per 4-row group: up to 15 bytes of alignment
// slack before the rows, the rows, and the decoder's over-read after them;
// a multiple of 16 so every group's bulk-copy destination is 16-byte aligned.
__host__ __device__ __forceinline__ uint32_t group_stride(uint32_t rowbytes) {
  return (kRowsPerTask * rowbytes + 32u + 15u) & ~15u;
}

// Activation record of one column over one 256-block (word-major so that the
// four activation words meeting one packed register are contiguous):
//   words 8w + j  (w, j < 8): int8x4 word w of Q8_1 chunk j
//   words 64 + j:  chunk j's fp32 scale divided by 4^(j mod 4)
//   words 72 + j:  kFloatBias - 4^(j mod 4) * sum of chunk j's int8 values
// The dp4a sums of a chunk start from word 72 + j, so they end as
// kFloatBias + 4^s * I with |4^s * I| <= 64 * 32 * 127 * 2 < 2^22: the bit
// pattern of the fp32 number 1.5 * 2^23 + 4^s * I, exactly.  One fp32
// subtraction then gives 4^s * I as a float (no integer-to-float conversion,
// which issues on a slow pipe).
constexpr int kPRec = 84;  // stride: 16-byte aligned; 8 consecutive records start 20 banks apart (mod 32: 8 distinct 4-bank groups)

struct Packed {
  uint32_t a[8];  // slots 0..3: chunks 0..3, activation word w
  uint32_t b[8];  // slots 0..3: chunks 4..7, activation word w
  float dw;
};

// P_k(b) = floor(b * 3^k / 256) for the four bytes of `x` and k = 1..ND, as
// u8x4 words (P[0] = 0).  b * 3^5 < 2^16, so bytes 0,2 and bytes 1,3 are
// multiplied in 16-bit lanes of two words without interacting and a byte
// permute gathers the high byte of every lane.  The first three powers are
// shift-and-add chains (integer ALU pipe), the last two multiplies (FMA-heavy
// pipe), which keeps the two integer pipes balanced.
template <int ND>
__device__ __forceinline__ void pow3_floors(uint32_t x, uint32_t (&P)[ND + 1]) {
  const uint32_t L0 = x & 0x00FF00FFu;
  const uint32_t H0 = __byte_perm(x, 0u, 0x4341u);
  uint32_t L = L0, H = H0;
  P[0] = 0;
#pragma unroll
  for (int k = 1; k <= ND; ++k) {
    if (k <= 3) {
      L = times3(L);
      H = times3(H);
    } else {
      L = L0 * pow3(k);
      H = H0 * pow3(k);
    }
    P[k] = __byte_perm(L, H, 0x7351u);
  }
}

// Expand the block at byte offset `off` (even) of shared memory `slab` into
// packed digits.  Element order (PrismML-Eng/llama.cpp issue #139, "Current
// behavior", continued over the last 16 qs bytes and the 4 qh bytes):
//   qs word w < 8,  digit j      -> chunk j,         word w
//   qs word 8 + i,  digit 0 / 1  -> chunk 5,         word i / 4 + i
//                   digit 2 / 3  -> chunk 6,         word i / 4 + i
//                   digit 4      -> chunk 7,         word i
//   qh word,        digit k      -> chunk 7,         word 4 + k
//
// The specification's digit k of byte b, ((uint8)(b*3^k)*3) >> 8, equals
// P_{k+1}(b) - 3 P_k(b) (the carry out of 3 * (b*3^k mod 256)).  A packed
// register sum_s 4^s * digit_s is therefore an integer combination of the
// u8x4 words P_k; every byte lane of the result lies in [0, 170], so the
// combination computed in wrapping 32-bit arithmetic has no carries or
// borrows between lanes and equals the packed register exactly.  For a qs
// word of the first 32 bytes, slots 0..3 hold digits 0..3:
//   d0 + 4 d1 + 16 d2 + 64 d3 = 64 P4 - 11 P1 - 44 P2 - 176 P3
// and digit 4 (slot 0 of the b register) is P5 - 3 P4.
__device__ __forceinline__ void expand_pack(const uint8_t* slab, uint32_t off, Packed& Q) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(slab + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;
  uint32_t w[14];
#pragma unroll
  for (int m = 0; m < 14; ++m) w[m] = p[m];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t P[6];
    pow3_floors<5>(__funnelshift_r(w[i], w[i + 1], sh), P);
    Q.a[i] = P[4] * 64u - P[1] * 11u - P[2] * 44u - P[3] * 176u;
    Q.b[i] = P[5] - 3u * P[4];
  }
  // qs word 8 + i: slots 1, 2, 3 of b[i] take digits 0, 2, 4; slots 1, 2 of
  // b[4 + i] take digits 1, 3.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t P[6];
    pow3_floors<5>(__funnelshift_r(w[8 + i], w[9 + i], sh), P);
    Q.b[i] += P[1] * 4u - P[2] * 48u + P[3] * 16u - P[4] * 192u + P[5] * 64u;
    Q.b[4 + i] += P[2] * 4u - P[1] * 12u - P[3] * 48u + P[4] * 16u;
  }
  // qh word: digit k goes to slot 3 of b[4 + k].
  {
    uint32_t P[5];
    pow3_floors<4>(__funnelshift_r(w[12], w[13], sh), P);
#pragma unroll
    for (int k = 0; k < 4; ++k) Q.b[4 + k] += P[k + 1] * 64u - P[k] * 192u;
  }
  Q.dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w[13] >> sh) & 0xFFFFu)));
}

// TQ2_0 block at byte offset `off` (even) of `slab`: its qs words already
// are packed-digit registers.  qs word i < 8 holds, in field f of byte lane
// m, element 32f + 4i + m (chunk f, activation word i): exactly register a[i];
// qs word 8 + i holds chunk 4 + f, word i: register b[i].  Reads 68 bytes
// from (off & ~3).
__device__ __forceinline__ void load_pack_tq2(const uint8_t* slab, uint32_t off, Packed& Q) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(slab + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;
  uint32_t w[17];
#pragma unroll
  for (int m = 0; m < 17; ++m) w[m] = p[m];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Q.a[i] = __funnelshift_r(w[i], w[i + 1], sh);
    Q.b[i] = __funnelshift_r(w[8 + i], w[9 + i], sh);
  }
  Q.dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w[16] >> sh) & 0xFFFFu)));
}

// Packed registers of one block of either weight format.
template <int FMT>
__device__ __forceinline__ void unit_pack(const uint8_t* slab, uint32_t off, Packed& Q) {
  if (FMT == kFmtTq2)
    load_pack_tq2(slab, off, Q);
  else
    expand_pack(slab, off, Q);
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The eight chunk sums of one packed block against one column record, as
// integers: I[j] = kFloatBias + 4^(j mod 4) * I_j, where I_j is chunk j's
// exact partial sum (trit * q) (the record's seed carries -4^s * sum q and the
// bias).  Both the fp32 mat-vec and the integer-partials debug mode start from
// these sums.
__device__ __forceinline__ void packed_sums(const Packed& P, const uint32_t* rec, int (&I)[8]) {
  const int4 s0 = *reinterpret_cast<const int4*>(rec + 72);
  const int4 s1 = *reinterpret_cast<const int4*>(rec + 76);
  I[0] = s0.x; I[1] = s0.y; I[2] = s0.z; I[3] = s0.w;
  I[4] = s1.x; I[5] = s1.y; I[6] = s1.z; I[7] = s1.w;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint4 qa = *reinterpret_cast<const uint4*>(rec + 8 * w);
    const uint4 qb = *reinterpret_cast<const uint4*>(rec + 8 * w + 4);
    I[0] = dp4a_us(P.a[w] & 0x03030303u, qa.x, I[0]);
    I[1] = dp4a_us(P.a[w] & 0x0C0C0C0Cu, qa.y, I[1]);
    I[2] = dp4a_us(P.a[w] & 0x30303030u, qa.z, I[2]);
    I[3] = dp4a_us(P.a[w] & 0xC0C0C0C0u, qa.w, I[3]);
    I[4] = dp4a_us(P.b[w] & 0x03030303u, qb.x, I[4]);
    I[5] = dp4a_us(P.b[w] & 0x0C0C0C0Cu, qb.y, I[5]);
    I[6] = dp4a_us(P.b[w] & 0x30303030u, qb.z, I[6]);
    I[7] = dp4a_us(P.b[w] & 0xC0C0C0C0u, qb.w, I[7]);
  }
}

// packed_sums for two blocks of the same block column (two rows) against one
// column record: every record word read from shared memory serves both rows,
// so a lane needs half the record bytes per row.  Each row's sums are exactly
// packed_sums'.
__device__ __forceinline__ void packed_sums2(const Packed& P, const Packed& Q, const uint32_t* rec, int (&I)[8],
                                             int (&J)[8]) {
  const int4 s0 = *reinterpret_cast<const int4*>(rec + 72);
  const int4 s1 = *reinterpret_cast<const int4*>(rec + 76);
  I[0] = s0.x; I[1] = s0.y; I[2] = s0.z; I[3] = s0.w;
  I[4] = s1.x; I[5] = s1.y; I[6] = s1.z; I[7] = s1.w;
#pragma unroll
  for (int j = 0; j < 8; ++j) J[j] = I[j];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint4 qa = *reinterpret_cast<const uint4*>(rec + 8 * w);
    const uint4 qb = *reinterpret_cast<const uint4*>(rec + 8 * w + 4);
    I[0] = dp4a_us(P.a[w] & 0x03030303u, qa.x, I[0]);
    J[0] = dp4a_us(Q.a[w] & 0x03030303u, qa.x, J[0]);
    I[1] = dp4a_us(P.a[w] & 0x0C0C0C0Cu, qa.y, I[1]);
    J[1] = dp4a_us(Q.a[w] & 0x0C0C0C0Cu, qa.y, J[1]);
    I[2] = dp4a_us(P.a[w] & 0x30303030u, qa.z, I[2]);
    J[2] = dp4a_us(Q.a[w] & 0x30303030u, qa.z, J[2]);
    I[3] = dp4a_us(P.a[w] & 0xC0C0C0C0u, qa.w, I[3]);
    J[3] = dp4a_us(Q.a[w] & 0xC0C0C0C0u, qa.w, J[3]);
    I[4] = dp4a_us(P.b[w] & 0x03030303u, qb.x, I[4]);
    J[4] = dp4a_us(Q.b[w] & 0x03030303u, qb.x, J[4]);
    I[5] = dp4a_us(P.b[w] & 0x0C0C0C0Cu, qb.y, I[5]);
    J[5] = dp4a_us(Q.b[w] & 0x0C0C0C0Cu, qb.y, J[5]);
    I[6] = dp4a_us(P.b[w] & 0x30303030u, qb.z, I[6]);
    J[6] = dp4a_us(Q.b[w] & 0x30303030u, qb.z, J[6]);
    I[7] = dp4a_us(P.b[w] & 0xC0C0C0C0u, qb.w, I[7]);
    J[7] = dp4a_us(Q.b[w] & 0xC0C0C0C0u, qb.w, J[7]);
  }
}

// d_w * sum_j d_a[j] * I_j from packed_sums' integers: kFloatBias + 4^s * I_j
// is the bit pattern of 1.5 * 2^23 + 4^s * I_j, one subtraction gives
// 4^s * I_j exactly, and the record's chunk scale is d_a / 4^s.
__device__ __forceinline__ float packed_scale(const int (&I)[8], const uint32_t* rec, float dw) {
  const float4 a0 = *reinterpret_cast<const float4*>(rec + 64);
  const float4 a1 = *reinterpret_cast<const float4*>(rec + 68);
  float s = a0.x * unbias(I[0]);
  s = fmaf(a0.y, unbias(I[1]), s);
  s = fmaf(a0.z, unbias(I[2]), s);
  s = fmaf(a0.w, unbias(I[3]), s);
  s = fmaf(a1.x, unbias(I[4]), s);
  s = fmaf(a1.y, unbias(I[5]), s);
  s = fmaf(a1.z, unbias(I[6]), s);
  s = fmaf(a1.w, unbias(I[7]), s);
  return s * dw;
}

// The exact partial I_j of chunk j from packed_sums' integer (4^s * I_j is a
// multiple of 4^s, so the arithmetic shift is exact).
__device__ __forceinline__ int packed_partial(int v, int j) { return (v - kFloatBias) >> (2 * (j & 3)); }

// Store a block's eight exact partials (int32, 16-byte aligned destination).
__device__ __forceinline__ void store_partials(int32_t* dst, const int (&I)[8]) {
  reinterpret_cast<int4*>(dst)[0] =
      make_int4(packed_partial(I[0], 0), packed_partial(I[1], 1), packed_partial(I[2], 2), packed_partial(I[3], 3));
  reinterpret_cast<int4*>(dst)[1] =
      make_int4(packed_partial(I[4], 4), packed_partial(I[5], 5), packed_partial(I[6], 6), packed_partial(I[7], 7));
}

// d_w * sum_j d_a[j] * I_j for one packed block against one column record.
__device__ __forceinline__ float packed_dot(const Packed& P, const uint32_t* rec) {
  int I[8];
  packed_sums(P, rec, I);
  return packed_scale(I, rec, P.dw);
}

// packed_dot for two rows of the same block column (one record read for both).
__device__ __forceinline__ void packed_dot2(const Packed& P, const Packed& Q, const uint32_t* rec, float& sp,
                                            float& sq) {
  int I[8], J[8];
  packed_sums2(P, Q, rec, I, J);
  sp = packed_scale(I, rec, P.dw);
  sq = packed_scale(J, rec, Q.dw);
}

// Quantise 32 fp32 activations (16-byte aligned, global) to one Q8_1 chunk
// and write it as chunk j of a record, with the same operations and rounding
// as q8_1_quantize_acts (d = amax / 127 with IEEE division, q =
// round-half-away(x / d) clamped to +-127, stored scale fp16(d)), so the
// record equals the one built from the quantised block.  Two lanes per chunk
// (lane pair 2p, 2p+1 of the warp; every lane of the warp calls this, `live`
// false for pairs without a chunk): lane half h takes values 16h .. 16h+15.
__device__ __forceinline__ void quantize_precord_half(const float* xs, uint32_t* rec, int j, int h, bool live) {
  float v[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = live ? __ldg(reinterpret_cast<const float4*>(xs + 16 * h) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
  float m = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[e]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  const float d = __fdiv_rn(m, 127.0f);
  int sum = 0;
  uint32_t words[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int q = 0;
      if (d != 0.0f) {
        float r = roundf(__fdiv_rn(v[4 * w + i], d));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q = static_cast<int>(r);
      }
      sum += q;
      word |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
    }
    words[w] = word;
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  if (!live) return;
#pragma unroll
  for (int w = 0; w < 4; ++w) rec[8 * (4 * h + w) + j] = words[w];
  if (h == 0) {
    const int slot = j & 3;
    const float dh = __half2float(__float2half_rn(d));
    rec[64 + j] = __float_as_uint(dh * __int_as_float((127 - 2 * slot) << 23));  // d / 4^slot, exact
    rec[72 + j] = static_cast<uint32_t>(kFloatBias - (sum << (2 * slot)));
  }
}

// Build one chunk (j) of one column's record from its Q8_1 block (global).
__device__ __forceinline__ void fill_precord_chunk(const uint8_t* blk, uint32_t* rec, int j) {
  const uint32_t* s = reinterpret_cast<const uint32_t*>(blk);
  const uint32_t ds = __ldg(s);
  int sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = __ldg(s + 1 + w);
    rec[8 * w + j] = q;
    sum = __dp4a(static_cast<int>(q), 0x01010101, sum);
  }
  const int slot = j & 3;
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(ds & 0xFFFFu)));
  rec[64 + j] = __float_as_uint(d * __int_as_float((127 - 2 * slot) << 23));  // d / 4^slot, exact
  rec[72 + j] = static_cast<uint32_t>(kFloatBias - (sum << (2 * slot)));
}

}  // namespace packed
}  // namespace tq1
