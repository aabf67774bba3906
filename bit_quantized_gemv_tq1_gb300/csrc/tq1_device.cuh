// tq1_device.cuh -- device-side building blocks of the TQ1_0 library (sm_103a).
//
// TQ1_0 block (PrismML-Eng/llama.cpp issue #139, "Current behavior", and the
// block specification that accompanies it): 256 ternary weights in 54 bytes,
// qs[48] holding five base-3 trits per byte, qh[4] holding four, then an fp16
// scale d.  Digit k of a byte b is ((uint8)(b*3^k) * 3) >> 8; digit 0/1/2
// means -1/0/+1.  Element e sits in
//   e <  160: byte qs[e % 32],            digit e / 32        (the page)
//   e <  240: byte qs[32 + (e-160) % 16], digit (e-160) / 16  (same pattern)
//   e >= 240: byte qh[(e-240) % 4],       digit (e-240) / 4   (same pattern)
// Q8_1 activation block: fp16 d, fp16 s, int8 q[32] (36 bytes).
//
// TQ2_0, the 2-bit sibling format the same page names ("Upstream state")
// without giving its layout; this library reads it as: 256 ternary weights
// in 66 bytes, qs[64] holding four 2-bit codes per byte (code = trit + 1),
// then an fp16 scale d.  Chunk c (elements 32c .. 32c+31) reads field c % 4
// (bits 2(c%4) .. 2(c%4)+1) of bytes qs[32(c/4) .. 32(c/4)+31], the page's
// chunk pattern with four codes per byte.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tq1 {

constexpr int kQK = 256;          // weights per TQ1_0 block
constexpr int kBlockBytes = 54;   // qs[48] + qh[4] + fp16 d
constexpr int kTq2BlockBytes = 66;  // TQ2_0: qs[64] + fp16 d

// Weight formats of the mat-vec kernels.
enum : int { kFmtTq1 = 0, kFmtTq2 = 1 };
template <int FMT>
__host__ __device__ constexpr int fmt_block_bytes() {
  return FMT == kFmtTq2 ? kTq2BlockBytes : kBlockBytes;
}
constexpr int kQK8 = 32;          // activations per Q8_1 block
constexpr int kQ8Bytes = 36;      // fp16 d + fp16 s + int8 q[32]

// Device status word: bit flags OR-ed by kernels (the word's address is a
// kernel argument), read and cleared by the host through tq1_sync_status().
enum : unsigned { kStatusTimeout = 1u, kStatusBadId = 2u };

__device__ __forceinline__ void raise_status(unsigned* st, unsigned bits) { atomicOr(st, bits); }

// ------------------------------------------------------------------ PTX --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after ~2 s of wall time
// and returning false, so that a lost transfer turns into an error code on
// the host (the caller raises kStatusTimeout) instead of a hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 63u) == 63u && global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One-dimensional bulk copy global -> shared, completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same without an L2 eviction hint (for small, re-read data).
__device__ __forceinline__ void bulk_g2s_nohint(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------- base-3 expansion --
// Powers of three packed into one word (PrismML-Eng/llama.cpp issue #139,
// "Upstream state": extract them with a shift and a mask rather than keep a
// constant array).  In unrolled code the extraction folds to an immediate.
constexpr uint64_t kPow3Packed = 1ull | (3ull << 8) | (9ull << 16) | (27ull << 24) | (81ull << 32) | (243ull << 40);
__host__ __device__ constexpr uint32_t pow3(int k) { return static_cast<uint32_t>((kPow3Packed >> (8 * k)) & 0xFFu); }

// Expand the four packed bytes of `x` into ND digit words: word k holds digit
// k of byte 0..3 in byte lanes 0..3 (values 0..2), ready for dp4a against the
// matching int8x4 activation word.
//
// Let P_k(b) = floor(b * 3^k / 256).  The spec's digit formula equals
// P_{k+1} - 3*P_k (the low byte of b*3^k times 3, shifted down by 8, is the
// carry out of 3*(b*3^k)).  b * 3^5 < 2^16, so two bytes computed in 16-bit
// lanes of one 32-bit multiply never interact; a byte permute gathers the
// high byte of each lane.  Per four bytes: 2 permutes to split, 2 multiplies
// and 1 permute per power, 1 multiply-add per digit.
//
// Multiplies and multiply-adds issue on the FMA-heavy pipe, which the dp4a
// instructions also use; the first three powers are therefore formed as
// shift-and-add chains (x*3 = (x << 1) + x), which issue on the integer ALU
// pipe, and the last two as multiplies.  This balances the two pipes
// (measured ~4% faster than five multiplies per lane pair).
__device__ __forceinline__ uint32_t times3(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .u32 t;\n\tshl.b32 t, %1, 1;\n\tadd.u32 %0, t, %1;\n\t}" : "=r"(r) : "r"(x));
  return r;
}

template <int ND>
__device__ __forceinline__ void expand_digits(uint32_t x, uint32_t (&u)[ND]) {
  uint32_t L[ND + 1], H[ND + 1];
  L[0] = __byte_perm(x, 0u, 0x4240u);  // bytes 0,2 in 16-bit lanes
  H[0] = __byte_perm(x, 0u, 0x4341u);  // bytes 1,3 in 16-bit lanes
#pragma unroll
  for (int k = 1; k <= ND; ++k) {
    if (k <= 3) {
      L[k] = times3(L[k - 1]);
      H[k] = times3(H[k - 1]);
    } else {
      L[k] = L[0] * pow3(k);
      H[k] = H[0] * pow3(k);
    }
  }
  uint32_t prev = 0;
#pragma unroll
  for (int k = 1; k <= ND; ++k) {
    const uint32_t p = __byte_perm(L[k], H[k], 0x7351u);  // P_k of bytes 0..3
    u[k - 1] = p - 3u * prev;
    prev = p;
  }
}

// All 256 digits of one block, as 65 dp4a-ready words, plus its scale.
//   a[w][j]: qs word w (0..7),  digit j -> Q8_1 chunk j, word w
//   b[w][j]: qs word 8+w (0..3), digit j -> chunk 5 + j/2, word 4*(j%2) + w
//            (digit 4 -> chunk 7, word w)
//   c[j]   : qh word,           digit j -> chunk 7, word 4 + j
struct BlockDigits {
  uint32_t a[8][5];
  uint32_t b[4][5];
  uint32_t c[4];
  float dw;
};

// Decode the block that starts at byte offset `off` (even) of shared memory
// region `base`.  Reads 56 bytes from (off & ~3).
__device__ __forceinline__ void decode_block(const uint8_t* base, uint32_t off, BlockDigits& D) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;  // 0 or 16
  uint32_t w[14];
#pragma unroll
  for (int m = 0; m < 14; ++m) w[m] = p[m];
#pragma unroll
  for (int i = 0; i < 8; ++i) expand_digits<5>(__funnelshift_r(w[i], w[i + 1], sh), D.a[i]);
#pragma unroll
  for (int i = 0; i < 4; ++i) expand_digits<5>(__funnelshift_r(w[8 + i], w[9 + i], sh), D.b[i]);
  expand_digits<4>(__funnelshift_r(w[12], w[13], sh), D.c);
  D.dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w[13] >> sh) & 0xFFFFu)));
}

// TQ2_0 block as 64 dp4a-ready words: d[c][w] holds the codes of chunk c,
// activation word w (byte lanes 0..3, values 0..3), plus the scale.
struct BlockDigits2 {
  uint32_t d[8][8];
  float dw;
};

// Decode the TQ2_0 block at byte offset `off` (even) of shared memory region
// `base`.  Reads 68 bytes from (off & ~3).
__device__ __forceinline__ void decode_block(const uint8_t* base, uint32_t off, BlockDigits2& D) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;  // 0 or 16
  uint32_t w[17];
#pragma unroll
  for (int m = 0; m < 17; ++m) w[m] = p[m];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t q = __funnelshift_r(w[i], w[i + 1], sh);
#pragma unroll
    for (int f = 0; f < 4; ++f) D.d[4 * (i >> 3) + f][i & 7] = (q >> (2 * f)) & 0x03030303u;
  }
  D.dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w[16] >> sh) & 0xFFFFu)));
}

// Integer dot products seeded with kFloatBias end as the bit pattern of the
// fp32 number 1.5 * 2^23 + I whenever |I| < 2^22 (every per-chunk partial
// here: at most 64 * 32 * 127 * 2); one fp32 subtraction of the bias then
// gives I exactly, without an integer-to-float conversion (a slow pipe).
constexpr int kFloatBias = 0x4B400000;  // bits of 12582912.0f = 1.5 * 2^23
constexpr float kFloatBiasValue = 12582912.0f;
__device__ __forceinline__ float unbias(int v) { return __fsub_rn(__int_as_float(v), kFloatBiasValue); }

// Activation record of one column over one 256-block, in shared memory:
//   words  0..63: the 8 Q8_1 chunks' int8 values (chunk j at words 8j..8j+7)
//   words 64..71: the 8 chunk scales as fp32
//   words 72..79: kFloatBias minus the sum of each chunk's int8 values
// Stride 100 words: 16-byte aligned and 4 banks apart for consecutive blocks.
constexpr int kRecWords = 100;

// Exact per-chunk integer partials I_j = sum (digit - 1) * q over the block,
// plus kFloatBias.  The -1 offset enters as the precomputed -sum(q)
// accumulator seed.
__device__ __forceinline__ void block_partials(const BlockDigits& D, const uint32_t* rec, int (&I)[8]) {
  const int4 s0 = *reinterpret_cast<const int4*>(rec + 72);
  const int4 s1 = *reinterpret_cast<const int4*>(rec + 76);
  I[0] = s0.x; I[1] = s0.y; I[2] = s0.z; I[3] = s0.w;
  I[4] = s1.x; I[5] = s1.y; I[6] = s1.z; I[7] = s1.w;
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(rec + 8 * j);
    const uint4 q1 = *reinterpret_cast<const uint4*>(rec + 8 * j + 4);
    int acc = I[j];
    acc = __dp4a(static_cast<int>(D.a[0][j]), static_cast<int>(q0.x), acc);
    acc = __dp4a(static_cast<int>(D.a[1][j]), static_cast<int>(q0.y), acc);
    acc = __dp4a(static_cast<int>(D.a[2][j]), static_cast<int>(q0.z), acc);
    acc = __dp4a(static_cast<int>(D.a[3][j]), static_cast<int>(q0.w), acc);
    acc = __dp4a(static_cast<int>(D.a[4][j]), static_cast<int>(q1.x), acc);
    acc = __dp4a(static_cast<int>(D.a[5][j]), static_cast<int>(q1.y), acc);
    acc = __dp4a(static_cast<int>(D.a[6][j]), static_cast<int>(q1.z), acc);
    acc = __dp4a(static_cast<int>(D.a[7][j]), static_cast<int>(q1.w), acc);
    I[j] = acc;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // chunks 5 and 6: digits 2h (words 0..3), 2h+1 (words 4..7)
    const uint4 q0 = *reinterpret_cast<const uint4*>(rec + 8 * (5 + h));
    const uint4 q1 = *reinterpret_cast<const uint4*>(rec + 8 * (5 + h) + 4);
    int acc = I[5 + h];
    acc = __dp4a(static_cast<int>(D.b[0][2 * h]), static_cast<int>(q0.x), acc);
    acc = __dp4a(static_cast<int>(D.b[1][2 * h]), static_cast<int>(q0.y), acc);
    acc = __dp4a(static_cast<int>(D.b[2][2 * h]), static_cast<int>(q0.z), acc);
    acc = __dp4a(static_cast<int>(D.b[3][2 * h]), static_cast<int>(q0.w), acc);
    acc = __dp4a(static_cast<int>(D.b[0][2 * h + 1]), static_cast<int>(q1.x), acc);
    acc = __dp4a(static_cast<int>(D.b[1][2 * h + 1]), static_cast<int>(q1.y), acc);
    acc = __dp4a(static_cast<int>(D.b[2][2 * h + 1]), static_cast<int>(q1.z), acc);
    acc = __dp4a(static_cast<int>(D.b[3][2 * h + 1]), static_cast<int>(q1.w), acc);
    I[5 + h] = acc;
  }
  {  // chunk 7: digit 4 of qs[32..47] (words 0..3), then the qh word's digits
    const uint4 q0 = *reinterpret_cast<const uint4*>(rec + 56);
    const uint4 q1 = *reinterpret_cast<const uint4*>(rec + 60);
    int acc = I[7];
    acc = __dp4a(static_cast<int>(D.b[0][4]), static_cast<int>(q0.x), acc);
    acc = __dp4a(static_cast<int>(D.b[1][4]), static_cast<int>(q0.y), acc);
    acc = __dp4a(static_cast<int>(D.b[2][4]), static_cast<int>(q0.z), acc);
    acc = __dp4a(static_cast<int>(D.b[3][4]), static_cast<int>(q0.w), acc);
    acc = __dp4a(static_cast<int>(D.c[0]), static_cast<int>(q1.x), acc);
    acc = __dp4a(static_cast<int>(D.c[1]), static_cast<int>(q1.y), acc);
    acc = __dp4a(static_cast<int>(D.c[2]), static_cast<int>(q1.z), acc);
    acc = __dp4a(static_cast<int>(D.c[3]), static_cast<int>(q1.w), acc);
    I[7] = acc;
  }
}

__device__ __forceinline__ void block_partials(const BlockDigits2& D, const uint32_t* rec, int (&I)[8]) {
  const int4 s0 = *reinterpret_cast<const int4*>(rec + 72);
  const int4 s1 = *reinterpret_cast<const int4*>(rec + 76);
  I[0] = s0.x; I[1] = s0.y; I[2] = s0.z; I[3] = s0.w;
  I[4] = s1.x; I[5] = s1.y; I[6] = s1.z; I[7] = s1.w;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(rec + 8 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(rec + 8 * c + 4);
    int acc = I[c];
    acc = __dp4a(static_cast<int>(D.d[c][0]), static_cast<int>(q0.x), acc);
    acc = __dp4a(static_cast<int>(D.d[c][1]), static_cast<int>(q0.y), acc);
    acc = __dp4a(static_cast<int>(D.d[c][2]), static_cast<int>(q0.z), acc);
    acc = __dp4a(static_cast<int>(D.d[c][3]), static_cast<int>(q0.w), acc);
    acc = __dp4a(static_cast<int>(D.d[c][4]), static_cast<int>(q1.x), acc);
    acc = __dp4a(static_cast<int>(D.d[c][5]), static_cast<int>(q1.y), acc);
    acc = __dp4a(static_cast<int>(D.d[c][6]), static_cast<int>(q1.z), acc);
    acc = __dp4a(static_cast<int>(D.d[c][7]), static_cast<int>(q1.w), acc);
    I[c] = acc;
  }
}

// Digit words of one block per weight format.
template <int FMT>
struct FmtDigits {
  using type = BlockDigits;
};
template <>
struct FmtDigits<kFmtTq2> {
  using type = BlockDigits2;
};

// d_w * sum_j d_a[j] * I_j for one block, fp32, fixed order.
template <class Digits>
__device__ __forceinline__ float block_dot(const Digits& D, const uint32_t* rec) {
  int I[8];
  block_partials(D, rec, I);
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
  return s * D.dw;
}

// Fill the activation record of one 256-block from eight Q8_1 blocks at `src`
// (global, 4-byte aligned).  `lane8` in 0..7 picks the chunk this thread
// handles; eight threads fill one record.
__device__ __forceinline__ void fill_record_chunk(const uint8_t* src, uint32_t* rec, int lane8) {
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src + lane8 * kQ8Bytes);
  const uint32_t ds = __ldg(s);
  int sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = __ldg(s + 1 + w);
    rec[8 * lane8 + w] = q;
    sum = __dp4a(static_cast<int>(q), 0x01010101, sum);
  }
  rec[64 + lane8] = __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(ds & 0xFFFFu))));
  rec[72 + lane8] = static_cast<uint32_t>(kFloatBias - sum);
}

}  // namespace tq1
