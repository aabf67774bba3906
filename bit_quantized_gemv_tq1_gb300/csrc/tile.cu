// tile.cu -- TQ1_0 x Q8_1 contraction on the 5th-generation tensor cores
// (tcgen05, operands and accumulators in tensor memory) for prefill-sized
// token counts (tens to thousands of columns).
//
// With many columns the contraction itself dominates: the tensor cores run
// it, and the weights' base-3 expansion (which does not grow with T) is
// shared by a 128-token tile.  sm_103a has no integer MMA kind, so
// the contraction runs in kind::f16 on operands that reproduce the method's
// products exactly (PrismML-Eng/llama.cpp issue #139 "Proposed approach":
// expand each packed byte once, reuse the activation fragment across rows and
// columns):
//
//   A[row][k] = fp16(d_w * trit)           exact: trit in {-1, 0, 1}, d_w is fp16
//   x[t][k]   = d_a * q * 2^-e_t           exact in fp32 (11 + 7 significant bits)
//   x = hi + lo, hi = fp16(x), lo = fp16(x - hi)   (lo exact unless subnormal)
//   y[t][row] = 2^e_t * (sum_k A*hi + sum_k A*lo)   fp32 accumulation in TMEM
//
// e_t is a per-token power of two that keeps 127 * max d_a below 2^14 (0 for
// ordinary activations).  Every product is exact; only the fp32 accumulation
// rounds.
//
// A call runs two kernels:
//  1. tile_prep_kernel turns the Q8_1 activations into the B operand once:
//     fp16 hi rows [t_pad][k], then lo rows [t_pad][k], and the per-token
//     scales 2^e_t, in the caller's workspace.  Padding tokens are zero.
//  2. tile_kernel: one tile = 128 weight rows (TMEM lanes) x 128 tokens; K
//     advances in stages of 64 (a quarter of a 256-block).  Each MMA is
//     M = 128, N = 256 (the hi rows of the 128 tokens, then their lo rows),
//     K = 16: the 256-column fp32 accumulator and two 128-column A block
//     slots fill the 512 columns of tensor memory.
//     * a weight producer thread brings, per 256-block, the packed weights of
//       all 128 rows into a shared-memory ring with one 2-D TMA copy (an
//       80-byte, 16-byte-aligned window around each row's 54-byte block;
//       rows past n arrive as zeros);
//     * a B producer warp copies each stage's hi and lo rows (128-byte
//       swizzled, K-major: the MMA's operand layout) with 2-D TMA into a ring
//       of three half-block slots (64 KB each; fewer, larger slots mean fewer
//       barrier waits and commits on the MMA thread);
//     * A warps 0-7: group g = w/4 expands quarters 2g and 2g+1 of every
//       block for rows 32*(w%4) .. +31 into fp16 +-d_w and stores them
//       straight into tensor memory (tcgen05.st; a warp may only reach its
//       own quarter of the TMEM lanes, which is exactly its rows), so the
//       16-bit A operand never touches shared memory.  Block j uses A slot
//       j % 2, so a slot is free only once block j - 2's MMAs are done: both
//       groups work on every block to halve the time from a slot's release
//       to the block being ready (measured: one group per block 77.6 us, both
//       75.3 us; four groups of one quarter each crowd the thread that issues
//       the MMAs: 94.2 us);
//     * epilogue warps 8-15 (two per TMEM lane quarter, 64 tokens each):
//       TMEM -> registers, release the accumulator, then scale and store y
//       while the next tile's MMAs run;
//     * warp 16: TMEM allocation; its lane 0 issues the MMAs (A from TMEM);
//     * warps 17 and 18: the weight and the activation copies.
//     A group reaches block j only after block j - 2's MMAs completed, which
//     needed both groups' arrivals for j - 2, and a raw-weight slot is
//     reloaded only after all A warps released it: no warp can run a phase
//     ahead on a shared barrier, so every mbarrier parity wait is answered by
//     the phase it waits for.
//     Why 128 tokens and N = 256 rather than 64 tokens and N = 128: the A
//     warps' integer work competes for issue slots with the thread that
//     feeds the (shallow) MMA queue, and an N = 256 MMA keeps the tensor pipe
//     busy twice as long per issue and per expanded weight (measured on the
//     prefill shape N=14336, K=4096, T=512: 110.8 -> 84.6 us per call).
// Persistent CTAs (at most one per SM) walk the tiles.  Every wait is
// bounded; the first timeout sets a shared abort flag that releases every
// other wait, the status word records it, and the CTA lets its issued copies
// and MMAs finish before it leaves.
//
// Requires the weight row stride (k/256 * 54 bytes) to be a multiple of 16
// (k a multiple of 2048): the launcher returns TQ1_ERR_UNSUPPORTED otherwise
// and the caller uses the dp4a kernels.
//
// TQ2_0 weights (66-byte blocks of 2-bit codes) run the same kernel: the
// 80-byte window still covers a block at any even offset (14 + 66 bytes), the
// row-stride rule is the same (k a multiple of 2048), and the expansion is a
// shift and mask per chunk word before the same byte permute to fp16.
#include <atomic>
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kTileRows = 128;  // weight rows per tile = TMEM lanes
constexpr int kStageK = 64;     // K per MMA stage (a quarter of a 256-block)
constexpr int kWinBytes = 80;   // raw weight window per row and block (16-byte aligned)
constexpr uint32_t kWRawBytes = kTileRows * kWinBytes;
constexpr int kGroups = 2;      // A warp groups: group g expands quarters 2g and 2g + 1 of every block
constexpr int kASlots = 2;      // tensor-memory A block slots (block j uses slot j % 2)
// Raw weight ring: one block per A slot.  Every A warp copies its row's raw
// weights to registers first and releases the slot at once, so the next copy
// has the block's expansion and the wait for a free A slot to land in (the
// shared memory goes to the B ring instead).
constexpr int kRW = kASlots;
constexpr int kAWarps = 4 * kGroups, kEWarps = 8;  // two epilogue warps per TMEM lane quarter
constexpr int kEWarp0 = kAWarps, kMWarp = kEWarp0 + kEWarps, kPWarpW = kMWarp + 1, kPWarpB = kMWarp + 2;
constexpr int kTThreads = (kPWarpB + 1) * 32;
constexpr int kPrepThreads = 256;
constexpr int kPrepHeld = 4;  // 8-value groups a prep thread keeps in registers (k <= 8192: one pass over q8)
constexpr int kBlockCols = 4 * 32;  // TMEM columns of one block of A (4 quarters x 32)

constexpr int TOK = 128;                               // tokens per tile
struct TileCfg {
  static constexpr int N = 2 * TOK;                      // B rows: hi of TOK tokens, then lo (MMA N = 256)
  static constexpr uint32_t kBTile = N * 128;            // bytes of one quarter (K = 64) of B
  static constexpr uint32_t kBSlot = 2 * kBTile;         // a B ring slot: half a block (K = 128)
  // A block slots live in tensor memory (one per A warp group, so a slot has
  // a single owner); B lives in shared memory as a ring of half-block slots
  // (a whole block of B is 128 KB).
  static constexpr int kRB = 3;
  static constexpr int kAccCols = N;                     // TMEM columns of the tile accumulator
  static constexpr int kA0 = kAccCols;                   // first TMEM column of the A slots
  static constexpr int kTmemCols = 512;
  static_assert(kA0 + kASlots * kBlockCols <= kTmemCols, "tensor memory budget");
  static constexpr uint32_t kOffW = kRB * kBSlot;
  static constexpr uint32_t kSmem = kOffW + kRW * kWRawBytes + 1024;
  static_assert(kSmem + 2048 <= 232448, "shared memory budget");
  // Instruction descriptor: D fp32, A and B fp16, K-major, N, M = 128.
  static constexpr uint32_t kIdesc =
      (1u << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) | ((static_cast<uint32_t>(kTileRows) >> 4) << 24);
  static constexpr int kChunk = 32;                      // TMEM columns per epilogue load
};

struct TileArgs {
  const float* scale;  // per-token 2^e_t (prep kernel output)
  float* y;
  const float* res;    // optional residual added to y (same layout), or nullptr
  unsigned* status;
  int n, k, t, t_pad;
  int tiles_m, tiles_n;
  int nblk;  // 256-blocks per weight row (k / 256)
};

// ------------------------------------------------------------- helpers --
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// mbarrier phase test in which a thread whose phase is not complete yet is
// suspended (for at most `hint_ns`) until it completes, instead of returning
// at once: waiting warps then take no issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait that also gives up as soon as another role has aborted.  The
// waiting thread sleeps in the barrier (suspend-time hint) rather than spin,
// so the warps doing the work keep the issue slots.
constexpr uint32_t kAbortPollNs = 20000;  // how often a sleeping waiter looks at the abort flag
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kAbortPollNs)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      return false;
    }
  }
}

// The same bounded wait, spinning: for the single thread that issues the
// MMAs, whose reaction time sets the pace of the whole pipeline.
__device__ __forceinline__ bool spin_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Lane 0 waits; the outcome is broadcast and the warp re-converges, which
// orders the other lanes' later accesses after the wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading offset (unused: K fits one atom row)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// D (TMEM) += A (TMEM: lane = row, two fp16 per column) * B (shared memory).
__device__ __forceinline__ void umma_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 2-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[NC]);

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// P_k = floor(b * 3^k / 256) of the four bytes held in 16-bit lanes lo
// (bytes 0, 2) and hi (bytes 1, 3); digit k = P_{k+1} - 3 P_k.
template <int K>
__device__ __forceinline__ uint32_t pk(uint32_t lo, uint32_t hi) {
  return __byte_perm(lo * pow3(K), hi * pow3(K), 0x7351u);
}

// Four fp16 values (digit - 1) * d_w from one digit word: a byte permute reads
// them from the table {-d_w, 0, +d_w}; the selector of a digit pair (D0, D1)
// is 34 * (D0 + 256 * D1) + 0x1010, both pairs from one multiply-add.
__device__ __forceinline__ void digits_to_f16(uint32_t D, uint32_t tlo, uint32_t thi, uint32_t& v0, uint32_t& v1) {
  const uint32_t sel = D * 34u + 0x10101010u;
  v0 = __byte_perm(tlo, thi, sel);
  v1 = __byte_perm(tlo, thi, sel >> 16);
}

// Expand quarter `Q` of one block row into its 64 K values (fp16 +-d_w),
// two per 32-bit word in K order: out[i] holds elements 2i, 2i+1 of the
// stage.  Element order (issue #139, "Current behavior", continued over
// qs[32..47] and qh): chunk j < 5 = digit j of qs words 0..7; chunk 5 / 6 =
// digits 0,1 / 2,3 of qs words 8..11 (word i -> chunk words i and 4 + i);
// chunk 7 = digit 4 of qs words 8..11, then the qh word's digits 0..3.  Stage
// quarter Q holds chunks 2Q and 2Q + 1: chunk word wd of chunk j lands at
// out[16 * (j - 2Q) + 2 * wd].
template <int Q>
__device__ __forceinline__ void expand_quarter(const uint32_t (&wv)[13], uint32_t tlo, uint32_t thi,
                                               uint32_t (&out)[32]) {
  auto put = [&](int j, int wd, uint32_t D) {
    digits_to_f16(D, tlo, thi, out[16 * (j - 2 * Q) + 2 * wd], out[16 * (j - 2 * Q) + 2 * wd + 1]);
  };
  auto split = [&](uint32_t x, uint32_t& lo, uint32_t& hi) {
    lo = __byte_perm(x, 0u, 0x4240u);
    hi = __byte_perm(x, 0u, 0x4341u);
  };
  if (Q == 0) {
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
      uint32_t l, h;
      split(wv[wd], l, h);
      const uint32_t p1 = pk<1>(l, h), p2 = pk<2>(l, h);
      put(0, wd, p1);
      put(1, wd, p2 - 3u * p1);
    }
  } else if (Q == 1) {
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
      uint32_t l, h;
      split(wv[wd], l, h);
      const uint32_t p2 = pk<2>(l, h), p3 = pk<3>(l, h), p4 = pk<4>(l, h);
      put(2, wd, p3 - 3u * p2);
      put(3, wd, p4 - 3u * p3);
    }
  } else if (Q == 2) {
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {  // chunk 4: digit 4 of qs words 0..7
      uint32_t l, h;
      split(wv[wd], l, h);
      put(4, wd, pk<5>(l, h) - 3u * pk<4>(l, h));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // chunk 5: digits 0 / 1 of qs words 8..11
      uint32_t l, h;
      split(wv[8 + i], l, h);
      const uint32_t p1 = pk<1>(l, h), p2 = pk<2>(l, h);
      put(5, i, p1);
      put(5, 4 + i, p2 - 3u * p1);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // chunks 6, 7: digits 2, 3, 4 of qs words 8..11
      uint32_t l, h;
      split(wv[8 + i], l, h);
      const uint32_t p2 = pk<2>(l, h), p3 = pk<3>(l, h), p4 = pk<4>(l, h), p5 = pk<5>(l, h);
      put(6, i, p3 - 3u * p2);
      put(6, 4 + i, p4 - 3u * p3);
      put(7, i, p5 - 3u * p4);
    }
    {  // chunk 7, words 4..7: the qh digits
      uint32_t l, h;
      split(wv[12], l, h);
      const uint32_t p1 = pk<1>(l, h), p2 = pk<2>(l, h), p3 = pk<3>(l, h), p4 = pk<4>(l, h);
      put(7, 4, p1);
      put(7, 5, p2 - 3u * p1);
      put(7, 6, p3 - 3u * p2);
      put(7, 7, p4 - 3u * p3);
    }
  }
}

// TQ2_0: quarter Q (chunks 2Q, 2Q + 1) from the block's 16 qs words; chunk j
// reads field j % 4 of qs words 8 * (j / 4) .. + 7.  Code 3 (never written by
// the encoder) selects bytes 6-7 of the table, which hold fp16(2 d_w).
template <int Q>
__device__ __forceinline__ void expand_quarter_tq2(const uint32_t (&wv)[16], uint32_t tlo, uint32_t thi,
                                                   uint32_t (&out)[32]) {
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = 2 * Q + jj;
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
      const uint32_t D = (wv[8 * (j >> 2) + wd] >> (2 * (j & 3))) & 0x03030303u;
      digits_to_f16(D, tlo, thi, out[16 * jj + 2 * wd], out[16 * jj + 2 * wd + 1]);
    }
  }
}

template <int J0>
__device__ __forceinline__ void realign_tq2(const uint32_t (&W)[20], uint32_t sh, uint32_t (&wv)[16], uint32_t& h) {
#pragma unroll
  for (int m = 0; m < 16; ++m) wv[m] = __funnelshift_r(W[J0 + m], W[J0 + m + 1], sh);
  h = (W[J0 + 16] >> sh) & 0xFFFFu;
}

// The 13 logical words of a block and its fp16 scale from the row's raw
// window W (20 words), where the block starts 4*J0 + sh/8 bytes in.
template <int J0>
__device__ __forceinline__ void realign(const uint32_t (&W)[20], uint32_t sh, uint32_t (&wv)[13], uint32_t& h) {
#pragma unroll
  for (int m = 0; m < 13; ++m) wv[m] = __funnelshift_r(W[J0 + m], W[J0 + m + 1], sh);
  h = (W[J0 + 13] >> sh) & 0xFFFFu;
}

// Eight int8 activations (two words) times fp16 d -> fp16 hi and lo parts.
__device__ __forceinline__ void acts_to_hilo(uint32_t q0, uint32_t q1, __half2 d2, uint4& hv, uint4& lv) {
  const __half2 c1152 = __float2half2_rn(1152.0f);
  uint32_t h[4], l[4];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    // int8 q -> exact fp16: bias to 0..255, place under the exponent of 1024
    // (0x64xx), subtract 1024 + 128.
    const uint32_t x = (u ? q1 : q0) ^ 0x80808080u;
    const uint32_t m01 = __byte_perm(x, 0x64646464u, 0x5150u);
    const uint32_t m23 = __byte_perm(x, 0x64646464u, 0x5352u);
    const __half2 v01 = __hsub2(*reinterpret_cast<const __half2*>(&m01), c1152);
    const __half2 v23 = __hsub2(*reinterpret_cast<const __half2*>(&m23), c1152);
    const __half2 h01 = __hmul2(v01, d2), h23 = __hmul2(v23, d2);
    const __half2 l01 = __hfma2(v01, d2, __hneg2(h01)), l23 = __hfma2(v23, d2, __hneg2(h23));
    h[2 * u] = *reinterpret_cast<const uint32_t*>(&h01);
    h[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&h23);
    l[2 * u] = *reinterpret_cast<const uint32_t*>(&l01);
    l[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&l23);
  }
  hv = make_uint4(h[0], h[1], h[2], h[3]);
  lv = make_uint4(l[0], l[1], l[2], l[3]);
}


}  // namespace

// Q8_1 activations -> B operand: fp16 hi rows [t_pad][k], lo rows
// [t_pad][k], per-token scale 2^e_t.  One CTA per (padded) token.
__global__ void __launch_bounds__(kPrepThreads) tile_prep_kernel(const uint8_t* q8, int t, int k, int t_pad,
                                                                 uint16_t* hilo, float* scale) {
  __shared__ float s_red[kPrepThreads / 32];
  __shared__ float s_inv;
  pdl_launch_dependents();
  pdl_wait();  // the activations may come from the previous kernel
  const int tok = blockIdx.x, tid = threadIdx.x;
  const int nq = k / kQK8;
  uint16_t* hrow = hilo + static_cast<size_t>(tok) * k;
  uint16_t* lrow = hilo + (static_cast<size_t>(t_pad) + tok) * k;
  if (tok >= t) {
    for (int i = tid; i < k / 8; i += kPrepThreads) {
      reinterpret_cast<uint4*>(hrow)[i] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(lrow)[i] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) scale[tok] = 1.0f;
    return;
  }
  const uint8_t* qr = q8 + static_cast<int64_t>(tok) * nq * kQ8Bytes;
  // A thread handles 8-value groups i = tid, tid + kPrepThreads, ... (group
  // i: block i / 4, words 1 + 2 (i % 4) and 2 + 2 (i % 4) of it), so that the
  // fp16 stores of consecutive lanes are consecutive 16-byte pieces.  Up to
  // kPrepHeld groups per thread are read once, into registers, before the
  // token's maximum scale is known; larger k reads them again afterwards.
  const int ng = k / 8;
  const bool held = ng <= kPrepHeld * kPrepThreads;
  uint32_t gq[kPrepHeld][2], gd[kPrepHeld];
  auto load_group = [&](int i, uint32_t& q0, uint32_t& q1, uint32_t& d) {
    const uint32_t* b = reinterpret_cast<const uint32_t*>(qr + (i >> 2) * kQ8Bytes);
    d = __ldg(b) & 0xFFFFu;
    q0 = __ldg(b + 1 + 2 * (i & 3));
    q1 = __ldg(b + 2 + 2 * (i & 3));
  };
  float m = 0.0f;
  if (held) {
#pragma unroll
    for (int r = 0; r < kPrepHeld; ++r) {
      const int i = tid + r * kPrepThreads;
      if (i < ng) {
        load_group(i, gq[r][0], gq[r][1], gd[r]);
        m = fmaxf(m, fabsf(__half2float(__ushort_as_half(static_cast<unsigned short>(gd[r])))));
      }
    }
  } else {
    for (int j = tid; j < nq; j += kPrepThreads)
      m = fmaxf(m, fabsf(__half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(qr + j * kQ8Bytes))))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) s_red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    float v = 0.0f;
    for (int w = 0; w < kPrepThreads / 32; ++w) v = fmaxf(v, s_red[w]);
    int ex = 0;
    (void)frexpf(v * 127.0f, &ex);  // 127 * max d < 2^ex
    const int e = max(0, ex - 14);
    scale[tok] = ldexpf(1.0f, e);
    s_inv = ldexpf(1.0f, -e);
  }
  __syncthreads();
  const float inv = s_inv;
  auto convert = [&](int i, uint32_t q0, uint32_t q1, uint32_t d16) {
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(d16))) * inv;
    uint4 hv, lv;
    acts_to_hilo(q0, q1, __float2half2_rn(d), hv, lv);
    reinterpret_cast<uint4*>(hrow)[i] = hv;
    reinterpret_cast<uint4*>(lrow)[i] = lv;
  };
  if (held) {
#pragma unroll
    for (int r = 0; r < kPrepHeld; ++r) {
      const int i = tid + r * kPrepThreads;
      if (i < ng) convert(i, gq[r][0], gq[r][1], gd[r]);
    }
  } else {
    for (int i = tid; i < ng; i += kPrepThreads) {
      uint32_t q0, q1, d;
      load_group(i, q0, q1, d);
      convert(i, q0, q1, d);
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kTThreads, 1)
    tile_kernel(const TileArgs a, const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmb) {
  using C = TileCfg;
  constexpr int kBB = fmt_block_bytes<FMT>();
  extern __shared__ __align__(1024) uint8_t tsmem_raw[];
  __shared__ __align__(8) uint64_t afull_bar[kASlots], aempty_bar[kASlots];
  __shared__ __align__(8) uint64_t bfull_bar[C::kRB], bempty_bar[C::kRB];
  __shared__ __align__(8) uint64_t wfull_bar[kRW], wempty_bar[kRW];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar;  // the tile accumulator: full, free
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    // Fetch both tensor-map descriptors now: the first copy through a map
    // otherwise waits for its descriptor.
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmb)) : "memory");
  }
  const uint32_t raw = smem_addr(tsmem_raw);
  uint8_t* sm = tsmem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_addr(sm);
  uint8_t* wraw = sm + C::kOffW;
  __shared__ float s_tscale[kEWarps][TOK];  // per-token scales, one copy per epilogue warp

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = a.nblk;  // blocks per tile
  const int ntiles = a.tiles_m * a.tiles_n;
  // Tile of this CTA's unit u (>= ntiles: no more units).  Block j of the
  // CTA (counted over all its units) is block j % nblk of unit j / nblk.
  // The grid stride passes through an empty asm so that the compiler keeps
  // the walk over units as written: given the stride it can see, it reshapes
  // the role loops around a closed-form unit count, and the prefill shape
  // (N=14336, K=4096, T=512) measured 116 instead of 110 us per call.
  int gstride = static_cast<int>(gridDim.x);
  asm("" : "+r"(gstride));
  auto unit_tile = [&](int u) -> int { return static_cast<int>(blockIdx.x) + u * gstride; };
  int nunits = 0;
  while (unit_tile(nunits) < ntiles) ++nunits;
  const uint32_t nall = static_cast<uint32_t>(nunits * nblk);  // blocks of this CTA
  // Block j of the CTA uses raw-weight slot (and A slot) j % 2, the slot's
  // use number j / 2.
  auto issue_weights = [&](uint32_t j, uint32_t ws) {
    const int bi = static_cast<int>(j % nblk);
    const int row0 = (unit_tile(static_cast<int>(j / nblk)) / a.tiles_n) * kTileRows;
    mbar_arrive_expect_tx(&wfull_bar[ws], kWRawBytes);
    tma_load_2d(wraw + ws * kWRawBytes, &tmw, (bi * kBB) & ~15, row0, &wfull_bar[ws]);
  };
  const uint32_t nfirst = nall < static_cast<uint32_t>(kRW) ? nall : static_cast<uint32_t>(kRW);

  if (tid == 0) {
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(&afull_bar[i], kAWarps);  // every A warp expands part of every block
      mbar_init(&aempty_bar[i], 1);
    }
    for (int i = 0; i < C::kRB; ++i) {
      mbar_init(&bfull_bar[i], 1);
      mbar_init(&bempty_bar[i], 1);
    }
    for (int i = 0; i < kRW; ++i) {
      mbar_init(&wfull_bar[i], 1);
      mbar_init(&wempty_bar[i], kAWarps);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&acce_bar, kEWarps);
    s_abort = 0;
    fence_mbar_init();
  }
  // The weights do not depend on the previous kernel: the first ring's worth
  // of copies goes out at once, one per lane of warp 0.
  if (warp == 0) {
    __syncwarp();
    const uint32_t j = static_cast<uint32_t>(lane);
    if (j < nfirst) issue_weights(j, j % kRW);
  }
  if (warp == kMWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();

  if (warp < kAWarps) {
    // ---------------------------------------------------------------- A --
    // Both groups work on every block j (A slot and raw-weight slot j % 2):
    // group g expands quarters 2g and 2g + 1, so a block is ready in half the
    // time one group would take (the two tensor-memory slots leave little
    // time between a slot's release and the block's MMAs).
    const int g = warp >> 2;
    const int quarter = warp & 3;  // TMEM lane quarter = rows 32*quarter ..
    const int rl = (quarter << 5) | lane;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + C::kA0 + static_cast<uint32_t>(64 * g);
    int bi = 0;  // j % nblk, advanced without a division
    for (uint32_t j = 0; j < nall; ++j, bi = bi + 1 == nblk ? 0 : bi + 1) {
      const uint32_t sl = j & 1u, ph = (j >> 1) & 1u;
      if (!warp_wait(&wfull_bar[sl], ph, abort_flag)) break;
      uint32_t W[20];
      const uint4* src = reinterpret_cast<const uint4*>(wraw + sl * kWRawBytes + rl * kWinBytes);
#pragma unroll
      for (int cc = 0; cc < 5; ++cc) {
        const uint4 v = src[cc];
        W[4 * cc] = v.x;
        W[4 * cc + 1] = v.y;
        W[4 * cc + 2] = v.z;
        W[4 * cc + 3] = v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty_bar[sl]);
      const uint32_t off = static_cast<uint32_t>(bi * kBB) & 15u;
      const uint32_t sh = (off & 2u) * 8u;
      const uint32_t tslot = tlane + sl * kBlockCols;
      uint32_t out[32];
      if (FMT == kFmtTq2) {
        uint32_t wv[16], h;
        switch (off >> 2) {
          case 0: realign_tq2<0>(W, sh, wv, h); break;
          case 1: realign_tq2<1>(W, sh, wv, h); break;
          case 2: realign_tq2<2>(W, sh, wv, h); break;
          default: realign_tq2<3>(W, sh, wv, h); break;
        }
        const uint32_t tlo = h ^ 0x8000u;  // bytes 0-1: -d_w, bytes 2-3: 0
        const uint32_t h2 = __half_as_ushort(__float2half_rn(2.0f * __half2float(__ushort_as_half(
                                static_cast<unsigned short>(h)))));
        const uint32_t thi = h | (h2 << 16);  // bytes 4-5: +d_w, bytes 6-7: +2 d_w
        if (!warp_wait(&aempty_bar[sl], ph ^ 1u, abort_flag)) break;
        tc_fence_after();
        if (g == 0) {
          expand_quarter_tq2<0>(wv, tlo, thi, out);
          tmem_st32(tslot + 0 * 32, out);
          expand_quarter_tq2<1>(wv, tlo, thi, out);
          tmem_st32(tslot + 1 * 32, out);
        } else {
          expand_quarter_tq2<2>(wv, tlo, thi, out);
          tmem_st32(tslot + 0 * 32, out);
          expand_quarter_tq2<3>(wv, tlo, thi, out);
          tmem_st32(tslot + 1 * 32, out);
        }
      } else {
        uint32_t wv[13], h;
        switch (off >> 2) {
          case 0: realign<0>(W, sh, wv, h); break;
          case 1: realign<1>(W, sh, wv, h); break;
          case 2: realign<2>(W, sh, wv, h); break;
          default: realign<3>(W, sh, wv, h); break;
        }
        const uint32_t tlo = h ^ 0x8000u;  // bytes 0-1: -d_w, bytes 2-3: 0
        const uint32_t thi = h;            // bytes 4-5: +d_w
        // The slot is free once the MMAs of the block two before are done.
        if (!warp_wait(&aempty_bar[sl], ph ^ 1u, abort_flag)) break;
        tc_fence_after();
        if (g == 0) {
          expand_quarter<0>(wv, tlo, thi, out);
          tmem_st32(tslot + 0 * 32, out);
          expand_quarter<1>(wv, tlo, thi, out);
          tmem_st32(tslot + 1 * 32, out);
        } else {
          expand_quarter<2>(wv, tlo, thi, out);
          tmem_st32(tslot + 0 * 32, out);
          expand_quarter<3>(wv, tlo, thi, out);
          tmem_st32(tslot + 1 * 32, out);
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull_bar[sl]);
    }
  } else if (warp < kMWarp) {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3;  // TMEM lane quarter this warp may read
    const int rl = quarter * 32 + lane;
    const int c_lo = ((warp - kEWarp0) >> 2) * (TOK / 2);  // this warp's half of the tile's tokens
    float* tsc = s_tscale[warp - kEWarp0];
    pdl_wait();  // the scales are written by the prep kernel
    for (int u = 0; u < nunits; ++u) {
      const int tile = unit_tile(u);
      const int row = (tile / a.tiles_n) * kTileRows + rl;
      const int tok0 = (tile % a.tiles_n) * TOK;
      const uint32_t aph = static_cast<uint32_t>(u) & 1u;
      // Scales of this tile's tokens, fetched while the MMAs run.
      __syncwarp();
      for (int tl = c_lo + lane; tl < c_lo + TOK / 2; tl += 32) tsc[tl] = __ldg(a.scale + tok0 + tl);
      __syncwarp();
      if (!warp_wait(&accf_bar, aph, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      // Read the warp's 64 tokens (hi + lo) out of tensor memory first and
      // release the accumulator, so the next tile's MMAs run while these
      // outputs are scaled and stored (all CTAs finish a tile at about the
      // same time, and the y writes of that moment are bandwidth-bound).
      float sum[2][C::kChunk];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t vh[C::kChunk], vl[C::kChunk];
        tmem_ld<C::kChunk>(tbase + c_lo + h * C::kChunk, vh);
        tmem_ld<C::kChunk>(tbase + TOK + c_lo + h * C::kChunk, vl);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int jj = 0; jj < C::kChunk; ++jj) sum[h][jj] = __uint_as_float(vh[jj]) + __uint_as_float(vl[jj]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int jj = 0; jj < C::kChunk; ++jj) {
          const int tl = c_lo + h * C::kChunk + jj, tok = tok0 + tl;
          const float v = sum[h][jj] * tsc[tl];
          if (row < a.n && tok < a.t) {
            const int64_t yi = static_cast<int64_t>(tok) * a.n + row;
            a.y[yi] = a.res ? v + a.res[yi] : v;
          }
        }
    }
  } else if (warp == kMWarp) {
    // -------------------------------------------------------------- MMA --
    if (lane == 0) {
      bool issued = false, ok = true;
      uint64_t* last_bar = nullptr;
      uint32_t last_ph = 0;
      // Everything but the waits is precomputed: the B descriptors of a slot
      // differ from the ring's first descriptor only in the address field
      // (address >> 4, 14 bits, no carry for shared-memory addresses).
      const uint64_t d0 = umma_desc_sw128(sbase);
      uint32_t ga = 0, pa = 0, rb = 0, pb = 0;  // A group slot, B ring slot and their phases
      for (int u = 0; u < nunits && ok; ++u) {
        const uint32_t aph = static_cast<uint32_t>(u) & 1u;
        if (!spin_wait_or_abort(&acce_bar, aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t dt = tmem;
        for (int bi = 0; bi < nblk && ok; ++bi) {
          if (!spin_wait_or_abort(&afull_bar[ga], pa, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t at = tmem + C::kA0 + ga * kBlockCols;
          for (int h = 0; h < 2; ++h) {
            if (!spin_wait_or_abort(&bfull_bar[rb], pb, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t db = d0 + ((rb * C::kBSlot) >> 4);
#pragma unroll
            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
              for (int ks = 0; ks < kStageK / 16; ++ks)
                umma_ts(dt, at + 32u * (2 * h + qq) + 8u * ks, db + ((qq * C::kBTile + 32u * ks) >> 4), C::kIdesc,
                        (bi > 0 || h > 0 || qq > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&bempty_bar[rb]);
            issued = true;
            last_bar = &bempty_bar[rb];
            last_ph = pb;
            if (++rb == C::kRB) { rb = 0; pb ^= 1u; }
          }
          // The A slot is released only after both halves' MMAs were issued
          // (on an abort, those issued so far).
          umma_commit(&aempty_bar[ga]);
          if (++ga == kASlots) { ga = 0; pa ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&accf_bar);
      }
      // After an abort, let the MMAs already issued finish (bounded) before
      // the tensor memory is released.
      if (*abort_flag && issued) (void)mbar_wait(last_bar, last_ph);
    }
  } else if (warp == kPWarpW) {
    // ---------------------------------------------------- weight copies --
    if (lane == 0) {
      int last_slot = -1;
      uint32_t last_ph = 0;
      for (uint32_t j = nfirst; j < nall; ++j) {
        const uint32_t ws = j % kRW;
        const uint32_t ph = (j / kRW) & 1u;
        if (!wait_or_abort(&wempty_bar[ws], ph ^ 1u, abort_flag)) break;
        issue_weights(j, ws);
        last_slot = static_cast<int>(ws);
        last_ph = ph;
      }
      // Copies still in flight must land before the CTA leaves.
      if (*abort_flag && last_slot >= 0) (void)mbar_wait(&wfull_bar[last_slot], last_ph);
      else if (*abort_flag && nfirst > 0) {
        for (uint32_t j = 0; j < nfirst; ++j)
          (void)mbar_wait(&wfull_bar[j % kRW], 0);
      }
    }
  } else {
    // ------------------------------------------------ activation copies --
    // Lane 0 waits for a free half-block slot and posts the byte count;
    // lanes 0-3 then issue the half's four copies (two quarters x hi and lo
    // rows) at once.
    pdl_wait();  // the B operand is written by the prep kernel
    int last_slot = -1;
    uint32_t last_ph = 0, rb = 0, pb = 0;
    int bi = 0, u = 0;
    int tok0 = nunits > 0 ? (unit_tile(0) % a.tiles_n) * TOK : 0;
    for (uint32_t j = 0; j < nall; ++j) {
      bool stop = false;
      for (int h = 0; h < 2; ++h) {
        int ok = 1;
        if (lane == 0) {
          ok = wait_or_abort(&bempty_bar[rb], pb ^ 1u, abort_flag) ? 1 : 0;
          if (ok) mbar_arrive_expect_tx(&bfull_bar[rb], C::kBSlot);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        if (lane < 4) {
          const int qq = lane >> 1, hl = lane & 1;
          tma_load_2d(sm + rb * C::kBSlot + qq * C::kBTile + hl * TOK * 128, &tmb, bi * kQK + (2 * h + qq) * kStageK,
                      hl * a.t_pad + tok0, &bfull_bar[rb]);
        }
        __syncwarp();
        last_slot = static_cast<int>(rb);
        last_ph = pb;
        if (++rb == C::kRB) { rb = 0; pb ^= 1u; }
      }
      if (stop) break;
      if (++bi == nblk) {
        bi = 0;
        if (++u < nunits) tok0 = (unit_tile(u) % a.tiles_n) * TOK;
      }
    }
    if (lane == 0 && *abort_flag && last_slot >= 0) (void)mbar_wait(&bfull_bar[last_slot], last_ph);
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) raise_status(a.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == kMWarp) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  }
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major 2-D map over `rows` x `row_elems` elements with a `box` window.
bool make_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t esize, const void* base, uint64_t row_elems,
              uint64_t rows, uint32_t box_x, uint32_t box_y, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * esize};
  const cuuint32_t box[2] = {box_x, box_y};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scratch of one call: fp16 hi and lo activation rows [t_pad][k] each, then
// the per-token scales [t_pad], rounded up to 256 bytes.
size_t tile_scratch_bytes(int64_t k, int64_t t) {
  const int64_t t_pad = ((t + TOK - 1) / TOK) * TOK;
  const size_t b = 2 * static_cast<size_t>(t_pad) * k * sizeof(uint16_t) + static_cast<size_t>(t_pad) * sizeof(float);
  return (b + 255) & ~size_t(255);
}

template <int FMT>
int launch_tile_fmt(const uint8_t* w, const uint8_t* q8, TileArgs a, int num_sms, cudaStream_t s, void* ws,
                    size_t ws_bytes) {
  using C = TileCfg;
  const DeviceInfo& di = device_info();
  static std::atomic<bool> configured[64];  // per device (racing threads configure twice: idempotent)
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (C::kSmem + 2048 > di.max_smem_optin) return TQ1_ERR_UNSUPPORTED;
  if (!configured[di.device].load(std::memory_order_acquire)) {
    if (!cuda_ok(cudaFuncSetAttribute(tile_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(C::kSmem))))
      return TQ1_ERR_CUDA;
    configured[di.device].store(true, std::memory_order_release);
  }
  a.tiles_m = (a.n + kTileRows - 1) / kTileRows;
  a.tiles_n = (a.t + TOK - 1) / TOK;
  a.t_pad = a.tiles_n * TOK;
  const int nb = a.k / kQK;
  const uint64_t rowbytes = static_cast<uint64_t>(nb) * fmt_block_bytes<FMT>();
  const size_t hilo_bytes = 2 * static_cast<size_t>(a.t_pad) * a.k * sizeof(uint16_t);
  if (ws == nullptr || ws_bytes < tile_scratch_bytes(a.k, a.t)) return TQ1_ERR_WORKSPACE;

  CUtensorMap tmw;
  if (!make_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, rowbytes, static_cast<uint64_t>(a.n), kWinBytes, kTileRows,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return TQ1_ERR_UNSUPPORTED;
  uint16_t* hilo = static_cast<uint16_t*>(ws);
  float* scale = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + hilo_bytes);
  a.scale = scale;
  int rc = TQ1_OK;
  CUtensorMap tmb;
  if (!make_map(&tmb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hilo, static_cast<uint64_t>(a.k),
                2 * static_cast<uint64_t>(a.t_pad), kStageK, TOK, CU_TENSOR_MAP_SWIZZLE_128B))
    rc = TQ1_ERR_UNSUPPORTED;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (rc == TQ1_OK) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.t_pad));
    cfg.blockDim = dim3(kPrepThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (!cuda_ok(cudaLaunchKernelEx(&cfg, tile_prep_kernel, q8, a.t, a.k, a.t_pad, hilo, scale))) rc = TQ1_ERR_CUDA;
  }
  if (rc == TQ1_OK) {
    const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(tiles, num_sms)));
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    a.nblk = nb;
    if (!cuda_ok(cudaLaunchKernelEx(&cfg, tile_kernel<FMT>, a, tmw, tmb))) rc = TQ1_ERR_CUDA;
  }
  return rc;
}

template <int FMT>
int launch_tile_checked(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t,
                        cudaStream_t s, unsigned* status, const float* res, void* ws, size_t ws_bytes) {
  if (n > (int64_t{1} << 30) || t > (int64_t{1} << 24) || k > (int64_t{1} << 30)) return TQ1_ERR_UNSUPPORTED;
  // The weight map's row stride must be a multiple of 16 bytes.
  if (((k / kQK) * fmt_block_bytes<FMT>()) % 16 != 0) return TQ1_ERR_UNSUPPORTED;
  const DeviceInfo& di = device_info();
  TileArgs a = {};
  a.y = y;
  a.res = res;
  a.status = status;
  a.n = static_cast<int>(n);
  a.k = static_cast<int>(k);
  a.t = static_cast<int>(t);
  return launch_tile_fmt<FMT>(w, q8, a, di.num_sms, s, ws, ws_bytes);
}

}  // namespace

int launch_tile(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, cudaStream_t s,
                unsigned* status, const float* res, int fmt, void* ws, size_t ws_bytes) {
  return fmt == kFmtTq2 ? launch_tile_checked<kFmtTq2>(w, q8, y, n, k, t, s, status, res, ws, ws_bytes)
                        : launch_tile_checked<kFmtTq1>(w, q8, y, n, k, t, s, status, res, ws, ws_bytes);
}

size_t tile_workspace_bytes(int64_t n, int64_t k, int64_t t, int fmt) {
  if (n < 1 || t < 1 || k < kQK || n > (int64_t{1} << 30) || t > (int64_t{1} << 24) || k > (int64_t{1} << 30)) return 0;
  if (((k / kQK) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes)) % 16 != 0) return 0;  // the dp4a/mma kernels
  return tile_scratch_bytes(k, t);
}

}  // namespace tq1
