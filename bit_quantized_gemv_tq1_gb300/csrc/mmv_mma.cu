// mmv_mma.cu -- TQ1_0 / TQ2_0 x Q8_1 mat-vec for up to 32 token columns on
// the warp-level tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation): the 8/16/24/32-column rungs of the ladder (from t = 6 on).
//
// Neroued/ninfer issue #293: one rung sized for the largest batch makes every
// small batch pay its price; rungs per column count do not.  Here a rung is
// the number of 8-token n-tiles (NT = 1..4) one mma covers, so a call pays for
// ceil(t / 8) tiles of tokens, never for 32.
//
// Exactness.  B holds the Q8_1 integers q (|q| <= 127: exact in fp16).  On the
// rung of one n-tile, A holds 1024 + digit (digit = trit + 1 in
// {0, 1, 2}; TQ2_0's code 0..3), an exact fp16 integer, and each chunk's
// accumulator starts at -1025 * sum(q) (the chunk's activations summed
// exactly when they are staged): the tensor core returns
// sum((1024 + digit) q) - 1025 sum(q) = sum((digit - 1) q) = I_j, the chunk's
// exact integer partial (PrismML-Eng/llama.cpp issue #139, "Current
// behavior": the per-32-block integer dot product); every product and partial
// sum on the way is an integer below 2^22 in magnitude, so the fp32
// accumulation is exact.  The epilogue sums d_a[j] * I_j over a block's chunks
// and adds that sum times d_w to the row's total.  On the rungs of two to
// four n-tiles (whose registers are fuller) A holds d_w * trit from a per-row
// table: each product is an exact multiple of d_w's last place and a chunk's
// sum (at most 4064 d_w) needs 23 bits, so the tensor core returns d_w * I_j
// from a zero accumulator and the epilogue adds d_a[j] * (d_w * I_j).  Either
// way in fp32, chunk by chunk, in a fixed order.  The partials mode (the debug entry points) takes I_j from the
// first form, or from the second with the unscaled table {-1, 0, +1}, and
// stores it as int32.
//
// Expansion (byte-major, each packed byte loaded once: issue #139, "Proposed
// approach").  A thread (group g = lane / 4, q = lane % 4) of a warp holds
// rows g and g + 8 of a 16-row M-tile.  The K order inside each 32-element
// chunk is chosen so that the thread's A fragments are exactly digit words of
// bytes it owns: for chunks 0..4 (digit j of qs[0..31]) it owns qs bytes
// 8q .. 8q+7; for chunks 5..7 the qs bytes 32 + 4q .. 32 + 4q + 3 (digits
// 0/1, 2/3, 4) and digit q of the four qh bytes.  A digit word (four digits
// 0..2 in byte lanes, P_{k+1} - 3 P_k with P_k = floor(b 3^k / 256) from
// 16-bit-lane multiplies and one byte permute) becomes two fp16x2 fragment
// registers by one byte permute each: in the first form the digit byte under
// byte 0x64 (the fp16 value 1024 + digit), in the second a pair of bytes of
// the row's table {-d_w, 0, +d_w}.
// The activations are staged in shared memory as fp16 in the same per-chunk
// slot order (chunks 5..7 of TQ1_0 permuted), so one 16-byte load gives a
// thread both k16 halves of its B fragment.
//
// Work split.  The matrix's M-tiles are divided into row groups; a row
// group's K range is split over a thread-block cluster of S CTAs (one K range
// each).  Inside a CTA the (M-tile, block) units are dealt to the warps in
// contiguous runs; a warp accumulates in registers while its M-tile does not
// change and flushes each run to shared memory; runs of one M-tile are summed
// in warp order, the CTAs' partial tiles in cluster-rank order through
// distributed shared memory.  No atomics: bitwise deterministic.  No scratch
// memory: everything lives in shared memory.
//
// Weights are requested from HBM (one 1-D bulk copy per row slice, TMA
// engine) before the dependency wait on the previous kernel; activations are
// staged after it.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kMmaWarps = 16;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaMaxSplit = 8;
constexpr size_t kMmaSmemBudget = 225 * 1024;
// The rung of one n-tile uses the biased operand form (no per-row table, no
// selector arithmetic: ~60 fewer integer operations per 16-row block; a seed
// per chunk and token in shared memory, a block sum per row and token in
// registers): 11.6 -> 9.9 us at t = 8, N=5120, K=6144.  At two to four
// n-tiles those registers pass the 128 a thread has and it measured no
// faster (two) or slower (four: 19.7 -> 24.4 us), so they keep the table form.
__host__ __device__ constexpr bool mma_biased(int nt) { return nt == 1; }

struct MmaArgs {
  const uint8_t* w;
  const uint8_t* q8;
  float* y;
  int32_t* part;     // partials mode: int32 [t][n][k/32]
  const float* res;  // optional residual (y's layout)
  unsigned* status;
  int64_t n;
  int t;             // token columns (<= 8 * NT)
  int nb;            // blocks per row
  int mt_total;      // 16-row M-tiles of the matrix
  int groups;        // row groups (clusters)
  int split;         // CTAs per cluster (K ranges)
  int mt_max;        // M-tiles of the largest row group
  int bc_max;        // blocks of the largest K range
  uint32_t slab_row; // shared-memory bytes per weight row
  uint32_t act_row;  // shared-memory bytes per token row of activations
  uint32_t off_da, off_slab, off_p, off_slot, off_recv, off_bar;
  int own_max;       // rows any rank of a cluster owns in the final sum
  int recv_alias;    // the receive buffer overlays the activations (a cluster barrier first)
  uint64_t pow3;     // the packed powers-of-three word (bytes 3^0 .. 3^5)
};

}  // namespace

// ------------------------------------------------------------ helpers --

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                        const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Two fp16 fragment halves from a digit word (digits d0..d3 in byte lanes,
// values 0..3) and a row's table: table bytes 2d, 2d+1 (t0: d = 0, 1; t1:
// d = 2, 3) hold the fp16 value of digit d.  The permute selector for the pair
// (d0, d1) has nibbles 2 d0, 2 d0 + 1, 2 d1, 2 d1 + 1, i.e. D * 0x22 +
// 0x10101010 in its low half (lanes never carry: 2 d + 1 <= 7); the pair
// (d2, d3) uses the high half.
// The high pair's selector, (D * 0x22) >> 16 + 0x1010, is the high word of
// D * (0x22 << 16) plus 0x1010: one multiply-high on the FMA pipe instead of a
// shift on the (busier) integer ALU pipe.  The permute is the PTX prmt in its
// default mode: every selector nibble here is at most 7, so the nibble's top
// bit (sign replication) is never set and no masking is needed.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ void digits_to_frag(uint32_t D, uint32_t t0, uint32_t t1, uint32_t& lo, uint32_t& hi) {
  lo = prmt(t0, t1, D * 0x22u + 0x10101010u);
  hi = prmt(t0, t1, __umulhi(D, 0x220000u) + 0x1010u);
}

// The biased form: the fp16 value 1024 + d has the bits 0x6400 + d, so the
// digit byte under byte 0x64 is that value.  lo = (1024 + d0, 1024 + d1),
// hi = (1024 + d2, 1024 + d3): selector nibbles 0..3 pick digit bytes, 4..7
// bytes of 0x64646464.
__device__ __forceinline__ void digits_to_frag_biased(uint32_t D, uint32_t& lo, uint32_t& hi) {
  lo = prmt(D, 0x64646464u, 0x5140u);
  hi = prmt(D, 0x64646464u, 0x7362u);
}

// acc[0..1] += s[0..1] * d[0..1] as one paired fp32 FMA (two fp32 lanes, each
// the same single rounding as fmaf).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float s0, float s1, float d0, float d1) {
  asm("{\n\t.reg .b64 ra, rs, rd;\n\t"
      "mov.b64 ra, {%0, %1};\n\t"
      "mov.b64 rs, {%2, %3};\n\t"
      "mov.b64 rd, {%4, %5};\n\t"
      "fma.rn.f32x2 ra, rs, rd, ra;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(s0), "f"(s1), "f"(d0), "f"(d1));
}

// Powers of three for the digit chains, extracted from the packed
// powers-of-three word the kernel receives as an argument: each multiply by
// 3^k is then one integer multiply-add (with the constants known at compile
// time the compiler turns some of them into longer shift-and-add chains).
struct Pow3 {
  uint32_t p[6];
  __device__ __forceinline__ explicit Pow3(uint64_t packed) {
#pragma unroll
    for (int k = 0; k < 6; ++k) p[k] = static_cast<uint32_t>((packed >> (8 * k)) & 0xFFu);
  }
};

// Digit chain of one packed word: L, H hold bytes 0,2 and 1,3 in 16-bit
// lanes; step k gives P_k = floor(b 3^k / 256) for the four bytes (u8x4) and
// the digit word P_k - 3 P_{k-1} (digit k-1 of every byte).
struct Chain {
  uint32_t L, H, P;
  __device__ __forceinline__ void init(uint32_t x) {
    L = x & 0x00FF00FFu;
    H = __byte_perm(x, 0u, 0x4341u);
    P = 0;
  }
  template <int K>
  __device__ __forceinline__ uint32_t next(const Pow3& pw) {
    const uint32_t Pk = __byte_perm(L * pw.p[K], H * pw.p[K], 0x7351u);
    const uint32_t d = Pk - 3u * P;
    P = Pk;
    return d;
  }
};

// Digit q of the four bytes of x (q = 0..3, runtime): P_{q+1} - 3 P_q.
__device__ __forceinline__ uint32_t digit_of_word(uint32_t x, uint32_t m_q, uint32_t m_q1) {
  const uint32_t L = x & 0x00FF00FFu;
  const uint32_t H = __byte_perm(x, 0u, 0x4341u);
  const uint32_t P0 = __byte_perm(L * m_q, H * m_q, 0x7351u);
  const uint32_t P1 = __byte_perm(L * m_q1, H * m_q1, 0x7351u);
  return P1 - 3u * P0;
}

// The fp16 table of a row from its scale's raw fp16 bits h: digit 0 -> -d
// (sign flipped), 1 -> 0, 2 -> +d, 3 -> 2d (an fp16 addition, exact unless it
// overflows; only TQ2_0's unused code 3 reads it).  Byte pairs 2 digit,
// 2 digit + 1 of (t0, t1).
__device__ __forceinline__ void scale_table(uint32_t h, uint32_t& t0, uint32_t& t1) {
  const __half d = __ushort_as_half(static_cast<unsigned short>(h));
  t0 = h ^ 0x8000u;
  t1 = h | (static_cast<uint32_t>(__half_as_ushort(__hadd(d, d))) << 16);
}

// Wait for phase `parity` of an mbarrier, letting the thread sleep inside
// each try (a suspend-time hint) instead of spinning, for at most ~2 s; false
// if the transfer never completed (the caller raises kStatusTimeout).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// int8x4 -> two fp16x2 (exact): bias to unsigned, place each byte in the low
// mantissa of 1024 (0x64xx), subtract 1152.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), off);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), off);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// ------------------------------------------------------------- kernel --

template <int NT, int FMT, bool PART, bool RES>
__global__ void __launch_bounds__(kMmaThreads, 1) mmv_mma_kernel(const MmaArgs a) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  constexpr int TP = 8 * NT;  // token slots
  constexpr bool kBiased = mma_biased(NT);  // 1024 + digit operands, seeded accumulators
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* act = smem;                                            // [TP][act_row] fp16 slots
  float* da = reinterpret_cast<float*>(smem + a.off_da);          // [bc * 8][TP] scales, or [bc * 8][TP / 2][4] scales and seeds
  uint8_t* slab = smem + a.off_slab;                              // [mt * 16][slab_row]
  float* P = reinterpret_cast<float*>(smem + a.off_p);            // [mt * 16][TP] CTA partial tile
  float* slot = reinterpret_cast<float*>(smem + a.off_slot);      // [warps][MP * 16][TP] continued runs
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.off_bar); // [mt] one per M-tile
  __shared__ int s_abort;
  __shared__ int s_cont[kMmaWarps];  // M-tile group a warp's first run continues, or -1

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.split;
  // This CTA's row group and K range, and the row bounds of the cluster
  // ranks' shares of the final sum: divisions done once, by thread 0.
  __shared__ int s_geo[5 + kMmaMaxSplit + 1];  // rank, M-tiles lo/hi, blocks lo/hi, owner row bounds
  if (tid == 0) {
    const int rank0 = S > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int grp = static_cast<int>(blockIdx.x) / S;
    const int lo = static_cast<int>((static_cast<int64_t>(a.mt_total) * grp) / a.groups);
    const int hi = static_cast<int>((static_cast<int64_t>(a.mt_total) * (grp + 1)) / a.groups);
    const int rws = static_cast<int>(std::min<int64_t>(a.n, static_cast<int64_t>(hi) * 16) - static_cast<int64_t>(lo) * 16);
    s_geo[0] = rank0;
    s_geo[1] = lo;
    s_geo[2] = hi;
    s_geo[3] = (a.nb * rank0) / S;
    s_geo[4] = (a.nb * (rank0 + 1)) / S;
    for (int r = 0; r <= S; ++r) s_geo[5 + r] = (rws * r) / S;
  }
  __syncthreads();
  const int rank = s_geo[0];
  const int mt_lo = s_geo[1], mt_hi = s_geo[2];
  const int mtc = mt_hi - mt_lo;
  const int64_t row0 = static_cast<int64_t>(mt_lo) * 16;
  const int rows = static_cast<int>(std::min<int64_t>(a.n, static_cast<int64_t>(mt_hi) * 16) - row0);
  const int b_lo = s_geo[3], b_hi = s_geo[4];
  const int bc = b_hi - b_lo;
  const uint32_t rowbytes = static_cast<uint32_t>(a.nb) * kBB;
  const uint32_t slice = static_cast<uint32_t>(bc) * kBB;

  // Weights: one mbarrier per M-tile, completed by its 16 row threads (rows
  // past the matrix arrive with no bytes); each row thread copies its row
  // slice from the 16-byte boundary at or below its start to the one at or
  // above its end (the extra bytes belong to neighbouring blocks and are
  // never read); only where that end would pass the end of the weight buffer
  // are the last bytes copied with plain loads.
  if (tid == 0) s_abort = 0;
  if (tid < mtc) {
    mbar_init(&bars[tid], 16);
    fence_mbar_init();
  }
  __syncthreads();
  {
    const uint64_t policy = l2_evict_first_policy();
    const uintptr_t wend = reinterpret_cast<uintptr_t>(a.w) + static_cast<uintptr_t>(a.n) * rowbytes;
    for (int r = tid; r < mtc * 16; r += kMmaThreads) {
      uint64_t* bar = &bars[r >> 4];
      if (r >= rows) {
        mbar_arrive_expect_tx(bar, 0);
        continue;
      }
      const uintptr_t src = reinterpret_cast<uintptr_t>(a.w) + (row0 + r) * rowbytes + static_cast<uint32_t>(b_lo) * kBB;
      const uintptr_t c0 = src & ~uintptr_t(15), end = src + slice;
      uintptr_t c1 = (end + 15) & ~uintptr_t(15);
      uint8_t* dst = slab + static_cast<uint32_t>(r) * a.slab_row;
      if (c1 > wend) {
        c1 = end & ~uintptr_t(15);
        for (uintptr_t i = c1; i < end; ++i) dst[i - c0] = __ldg(reinterpret_cast<const uint8_t*>(i));
      }
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(c1 - c0));
      if (c1 > c0) bulk_g2s(dst, reinterpret_cast<const void*>(c0), static_cast<uint32_t>(c1 - c0), bar, policy);
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // activations may come from the previous kernel

  // Activations of this K range: fp16 slots [token][block][chunk][slot], and
  // the chunk scales; token slots beyond t are zero.  Warp w stages tokens
  // w, w + 16, ...; its lanes take the token's Q8_1 blocks (chunks of the K
  // range) two at a time, both loaded before either is converted.
  for (int tok = warp; tok < TP; tok += kMmaWarps) {
    const bool live = tok < a.t;
    const uint8_t* src_tok = a.q8 + (static_cast<int64_t>(tok) * a.nb + b_lo) * 8 * kQ8Bytes;
    uint8_t* dst_tok = act + static_cast<uint32_t>(tok) * a.act_row;
    for (int c0 = lane; c0 < bc * 8; c0 += 64) {
      uint32_t wq[2][9];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = c0 + 32 * h;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(src_tok + c * kQ8Bytes);
#pragma unroll
        for (int e = 0; e < 9; ++e) wq[h][e] = (live && c < bc * 8) ? __ldg(src + e) : 0u;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = c0 + 32 * h;
        if (c >= bc * 8) break;
        const int j = c & 7;
        // Per chunk and token pair: d_a of tokens 2p, 2p + 1, and in the
        // biased form their seeds -1025 * sum(q) (exact: |sum(q)| <= 4064).
        float* dsl = kBiased ? da + (c * (TP / 2) + (tok >> 1)) * 4 + (tok & 1) : da + c * TP + tok;
        dsl[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(wq[h][0] & 0xFFFFu)));
        if constexpr (kBiased) {
          int sq = 0;
#pragma unroll
          for (int e = 1; e < 9; ++e) sq = __dp4a(static_cast<int>(wq[h][e]), 0x01010101, sq);
          dsl[2] = -1025.0f * static_cast<float>(sq);
        }
        uint8_t* dst = dst_tok + static_cast<uint32_t>(c) * 64;
        const bool perm = FMT != kFmtTq2 && j >= 5;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // slots 8q .. 8q+7: positions 8q .. 8q+7, or (permuted chunks)
          // 4q .. 4q+3 and 16+4q .. 16+4q+3.
          const uint32_t w0 = perm ? wq[h][1 + q] : wq[h][1 + 2 * q];
          const uint32_t w1 = perm ? wq[h][5 + q] : wq[h][2 + 2 * q];
          uint4 v;
          i8x4_to_f16x4(w0, v.x, v.y);
          i8x4_to_f16x4(w1, v.z, v.w);
          *reinterpret_cast<uint4*>(dst + 16 * q) = v;
        }
      }
    }
  }
  __syncthreads();

  // Units (group of MP M-tiles, block) dealt to warps in contiguous runs.
  // (Two M-tiles per unit, so that every activation fragment loaded from
  // shared memory serves 32 rows, measured slower at 16 columns on GB300:
  // 15.9 against 13.5 us per call.)
  constexpr int MP = 1;
  const int mgc = (mtc + MP - 1) / MP;  // M-tile groups
  const int U = mgc * bc;
  const int u0 = (U * warp) / kMmaWarps, u1 = (U * (warp + 1)) / kMmaWarps;
  const int g = lane >> 2, q = lane & 3;
  // 3^q and 3^(q+1) from the packed powers-of-three word (q is per thread).
  const Pow3 pw(a.pow3);
  const uint32_t m_q = static_cast<uint32_t>((a.pow3 >> (8 * q)) & 0xFFu);
  const uint32_t m_q1 = static_cast<uint32_t>((a.pow3 >> (8 * (q + 1))) & 0xFFu);
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  float acc[MP][NT][4];
#pragma unroll
  for (int i = 0; i < MP; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
  bool ok = true;
  int cur_m = -1, run = 0;

  // Store a finished run of M-tile group mg.  A run that starts at the
  // group's first block (every run but perhaps a warp's first) is the group's
  // head: it goes straight into the CTA's partial tile.  A warp's first run
  // that continues a group another warp started goes to the warp's slot; the
  // continued runs are added to the head in warp order afterwards.
  const bool cont0 = u0 < u1 && (u0 % bc) != 0;
  auto flush = [&](int mg) {
#pragma unroll
    for (int i = 0; i < MP; ++i) {
      const int m = mg * MP + i;
      float* dst = (run == 0 && cont0) ? slot + (warp * MP + i) * 16 * TP : P + m * 16 * TP;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * q;
        if (m < mtc) {
          dst[g * TP + tok] = acc[i][nt][0];
          dst[g * TP + tok + 1] = acc[i][nt][1];
          dst[(g + 8) * TP + tok] = acc[i][nt][2];
          dst[(g + 8) * TP + tok + 1] = acc[i][nt][3];
        }
        acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
      }
    }
  };

  // Slab offsets of this thread's rows (g and g + 8 of each M-tile of the
  // current group): where the row's first block of the K range lands (its
  // copy started at the 16-byte boundary below it).
  uint32_t base_r[MP][2];
  int mg = u0 < u1 ? u0 / bc : 0, b = u0 < u1 ? u0 - mg * bc : 0;
  for (int u = u0; u < u1 && ok; ++u, ++b) {
    if (b == bc) {
      b = 0;
      ++mg;
    }
    if (mg != cur_m) {
      if (cur_m >= 0) {
        flush(cur_m);
        ++run;
      }
      cur_m = mg;
      const uintptr_t k0 = reinterpret_cast<uintptr_t>(a.w) + static_cast<uint32_t>(b_lo) * kBB;
#pragma unroll
      for (int i = 0; i < MP; ++i) {
        const int m = mg * MP + i;
        if (m < mtc && !mbar_wait_sleep(&bars[m], 0)) ok = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = m * 16 + g + 8 * h;
          base_r[i][h] = static_cast<uint32_t>(r) * a.slab_row + static_cast<uint32_t>((k0 + (row0 + r) * rowbytes) & 15u);
        }
      }
      if (!ok) break;
    }
    // This thread's rows and their block bytes: table (zero: no row) and the
    // packed words of each of its 2 * MP rows.
    uint32_t tt[MP][2][2];  // second form: the rows' tables
    float dw[MP][2];        // first form: the rows' block scales (0 past the matrix)
    uint32_t wd[MP][2][4];
#pragma unroll
    for (int i = 0; i < MP; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = (mg * MP + i) * 16 + g + 8 * h;
        const uint32_t off = base_r[i][h] + static_cast<uint32_t>(b) * kBB;
        const uint32_t* pp = reinterpret_cast<const uint32_t*>(slab + (off & ~3u));
        const uint32_t sh = (off & 2u) * 8u;
        uint32_t dh;  // the block's fp16 scale, raw bits
        if (FMT == kFmtTq2) {
          // chunks 0..3: qs bytes 8q..8q+7; chunks 4..7: qs bytes 32+8q..32+8q+7
          wd[i][h][0] = __funnelshift_r(pp[2 * q], pp[2 * q + 1], sh);
          wd[i][h][1] = __funnelshift_r(pp[2 * q + 1], pp[2 * q + 2], sh);
          wd[i][h][2] = __funnelshift_r(pp[8 + 2 * q], pp[9 + 2 * q], sh);
          wd[i][h][3] = __funnelshift_r(pp[9 + 2 * q], pp[10 + 2 * q], sh);
          dh = (pp[16] >> sh) & 0xFFFFu;
        } else {
          // qs bytes 8q..8q+7 (chunks 0..4), qs bytes 32+4q..32+4q+3 (chunks
          // 5, 6 and half of 7), the qh word (the other half of chunk 7)
          wd[i][h][0] = __funnelshift_r(pp[2 * q], pp[2 * q + 1], sh);
          wd[i][h][1] = __funnelshift_r(pp[2 * q + 1], pp[2 * q + 2], sh);
          wd[i][h][2] = __funnelshift_r(pp[8 + q], pp[9 + q], sh);
          wd[i][h][3] = __funnelshift_r(pp[12], pp[13], sh);
          dh = (pp[13] >> sh) & 0xFFFFu;
        }
        if constexpr (kBiased) {
          dw[i][h] = r < rows ? __half2float(__ushort_as_half(static_cast<unsigned short>(dh))) : 0.0f;
        } else {
          tt[i][h][0] = tt[i][h][1] = 0;
          if (r < rows) scale_table(PART ? 0x3C00u : dh, tt[i][h][0], tt[i][h][1]);  // PART: the unscaled trits
        }
      }
    }

    // One chunk: B fragments from shared memory once per n-tile, then for
    // each M-tile of the group its A fragments from four digit words (rows
    // g and g+8, k16 halves 0 and 1), two MMAs, and the epilogue (or the
    // partials store).
    const uint8_t* abase = act + static_cast<uint32_t>(b * 256) * 2 + 16 * q + static_cast<uint32_t>(g) * a.act_row;
    // chunk scales (and seeds) of this block, tokens 2q, 2q+1
    const float* dab = kBiased ? da + (b * 8 * (TP / 2) + q) * 4 : da + b * 8 * TP + 2 * q;
    float au[MP][NT][4];  // biased form: this block's sum of d_a[j] * I_j per row and token
#pragma unroll
    for (int i = 0; i < MP; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) au[i][nt][0] = au[i][nt][1] = au[i][nt][2] = au[i][nt][3] = 0.f;
    auto chunk = [&](int j, const uint32_t (&dA0)[MP], const uint32_t (&dB0)[MP], const uint32_t (&dA1)[MP],
                     const uint32_t (&dB1)[MP]) {
      uint32_t f0[MP][4], f1[MP][4];
#pragma unroll
      for (int i = 0; i < MP; ++i) {
        if constexpr (kBiased) {
          digits_to_frag_biased(dA0[i], f0[i][0], f0[i][2]);
          digits_to_frag_biased(dB0[i], f0[i][1], f0[i][3]);
          digits_to_frag_biased(dA1[i], f1[i][0], f1[i][2]);
          digits_to_frag_biased(dB1[i], f1[i][1], f1[i][3]);
        } else {
          digits_to_frag(dA0[i], tt[i][0][0], tt[i][0][1], f0[i][0], f0[i][2]);
          digits_to_frag(dB0[i], tt[i][1][0], tt[i][1][1], f0[i][1], f0[i][3]);
          digits_to_frag(dA1[i], tt[i][0][0], tt[i][0][1], f1[i][0], f1[i][2]);
          digits_to_frag(dB1[i], tt[i][1][0], tt[i][1][1], f1[i][1], f1[i][3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 bf = *reinterpret_cast<const uint4*>(abase + static_cast<uint32_t>(nt * 8) * a.act_row + j * 64);
        const int tok = nt * 8 + 2 * q;
        // d_a of tokens 2q, 2q+1 and, in the biased form, their seeds
        float2 sc = make_float2(0.f, 0.f), sd = make_float2(0.f, 0.f);
        if constexpr (kBiased) {
          const float4 s4 = *reinterpret_cast<const float4*>(dab + (j * (TP / 2) + nt * 4) * 4);
          sc = make_float2(s4.x, s4.y);
          sd = make_float2(s4.z, s4.w);
        } else if constexpr (!PART) {
          sc = *reinterpret_cast<const float2*>(dab + j * TP + nt * 8);
        }
#pragma unroll
        for (int i = 0; i < MP; ++i) {
          float d[4];
          if constexpr (kBiased) {
            const float seed[4] = {sd.x, sd.y, sd.x, sd.y};
            mma_f16(d, f0[i], bf.x, bf.y, seed);
          } else {
            mma_f16(d, f0[i], bf.x, bf.y, zero4);
          }
          mma_f16(d, f1[i], bf.z, bf.w, d);
          if constexpr (PART) {
            const int ra = (mg * MP + i) * 16 + g, rb = ra + 8;
            const int64_t kc = static_cast<int64_t>(a.nb) * 8;
            const int64_t cidx = static_cast<int64_t>(b_lo + b) * 8 + j;
            if (tok < a.t) {
              if (ra < rows) a.part[(static_cast<int64_t>(tok) * a.n + row0 + ra) * kc + cidx] = __float2int_rn(d[0]);
              if (rb < rows) a.part[(static_cast<int64_t>(tok) * a.n + row0 + rb) * kc + cidx] = __float2int_rn(d[2]);
            }
            if (tok + 1 < a.t) {
              if (ra < rows)
                a.part[(static_cast<int64_t>(tok + 1) * a.n + row0 + ra) * kc + cidx] = __float2int_rn(d[1]);
              if (rb < rows)
                a.part[(static_cast<int64_t>(tok + 1) * a.n + row0 + rb) * kc + cidx] = __float2int_rn(d[3]);
            }
          } else if constexpr (kBiased) {
            ffma2(au[i][nt][0], au[i][nt][1], sc.x, sc.y, d[0], d[1]);
            ffma2(au[i][nt][2], au[i][nt][3], sc.x, sc.y, d[2], d[3]);
          } else {
            ffma2(acc[i][nt][0], acc[i][nt][1], sc.x, sc.y, d[0], d[1]);
            ffma2(acc[i][nt][2], acc[i][nt][3], sc.x, sc.y, d[2], d[3]);
          }
        }
      }
    };

    if constexpr (FMT == kFmtTq2) {
      // Chunk j: field j % 4 of words 0,1 (j < 4) or 2,3 (j >= 4).
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i0 = j < 4 ? 0 : 2;
        const int f = 2 * (j & 3);
        uint32_t xa0[MP], xb0[MP], xa1[MP], xb1[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
          xa0[i] = (wd[i][0][i0] >> f) & 0x03030303u;
          xb0[i] = (wd[i][1][i0] >> f) & 0x03030303u;
          xa1[i] = (wd[i][0][i0 + 1] >> f) & 0x03030303u;
          xb1[i] = (wd[i][1][i0 + 1] >> f) & 0x03030303u;
        }
        chunk(j, xa0, xb0, xa1, xb1);
      }
    } else {
      // Chunks 0..4: digit j of qs bytes 8q..8q+3 (k16 half 0) and 8q+4..8q+7
      // (half 1).
      Chain ca0[MP], ca1[MP], cb0[MP], cb1[MP];
#pragma unroll
      for (int i = 0; i < MP; ++i) {
        ca0[i].init(wd[i][0][0]);
        ca1[i].init(wd[i][0][1]);
        cb0[i].init(wd[i][1][0]);
        cb1[i].init(wd[i][1][1]);
      }
#define TQ1_MMA_CHUNK04(J, K)                                                                 \
  {                                                                                           \
    uint32_t xa0[MP], xb0[MP], xa1[MP], xb1[MP];                                              \
    _Pragma("unroll") for (int i = 0; i < MP; ++i) {                                          \
      xa0[i] = ca0[i].next<K>(pw);                                                            \
      xb0[i] = cb0[i].next<K>(pw);                                                            \
      xa1[i] = ca1[i].next<K>(pw);                                                            \
      xb1[i] = cb1[i].next<K>(pw);                                                            \
    }                                                                                         \
    chunk(J, xa0, xb0, xa1, xb1);                                                             \
  }
      TQ1_MMA_CHUNK04(0, 1)
      TQ1_MMA_CHUNK04(1, 2)
      TQ1_MMA_CHUNK04(2, 3)
      TQ1_MMA_CHUNK04(3, 4)
      TQ1_MMA_CHUNK04(4, 5)
#undef TQ1_MMA_CHUNK04
      // Chunks 5, 6: digits 0/1 and 2/3 of qs bytes 32+4q..32+4q+3; chunk 7:
      // digit 4 of those bytes and digit q of the qh bytes.
      Chain ea[MP], eb[MP];
#pragma unroll
      for (int i = 0; i < MP; ++i) {
        ea[i].init(wd[i][0][2]);
        eb[i].init(wd[i][1][2]);
      }
      {
        uint32_t xa0[MP], xb0[MP], xa1[MP], xb1[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
          xa0[i] = ea[i].next<1>(pw);
          xb0[i] = eb[i].next<1>(pw);
          xa1[i] = ea[i].next<2>(pw);
          xb1[i] = eb[i].next<2>(pw);
        }
        chunk(5, xa0, xb0, xa1, xb1);
      }
      {
        uint32_t xa0[MP], xb0[MP], xa1[MP], xb1[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
          xa0[i] = ea[i].next<3>(pw);
          xb0[i] = eb[i].next<3>(pw);
          xa1[i] = ea[i].next<4>(pw);
          xb1[i] = eb[i].next<4>(pw);
        }
        chunk(6, xa0, xb0, xa1, xb1);
      }
      {
        uint32_t xa0[MP], xb0[MP], xa1[MP], xb1[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
          xa0[i] = ea[i].next<5>(pw);
          xb0[i] = eb[i].next<5>(pw);
          xa1[i] = digit_of_word(wd[i][0][3], m_q, m_q1);
          xb1[i] = digit_of_word(wd[i][1][3], m_q, m_q1);
        }
        chunk(7, xa0, xb0, xa1, xb1);
      }
    }
    if constexpr (kBiased && !PART) {
#pragma unroll
      for (int i = 0; i < MP; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          ffma2(acc[i][nt][0], acc[i][nt][1], dw[i][0], dw[i][0], au[i][nt][0], au[i][nt][1]);
          ffma2(acc[i][nt][2], acc[i][nt][3], dw[i][1], dw[i][1], au[i][nt][2], au[i][nt][3]);
        }
    }
  }
  if (cur_m >= 0 && ok) flush(cur_m);
  if (lane == 0) s_cont[warp] = cont0 ? u0 / bc : -1;
  if (!ok) s_abort = 1;
  __syncthreads();
  const bool abort = s_abort != 0;

  if constexpr (!PART) {
    // Add the continued runs to their M-tile groups' heads, in warp order:
    // warp w continued group u0(w) / bc if its first unit is not the first
    // block of a group.  One warp per group.
    if (!abort) {
      for (int grp_i = warp; grp_i < mgc; grp_i += kMmaWarps) {
        bool any = false;
        for (int w = 0; w < kMmaWarps; ++w) any = any || s_cont[w] == grp_i;
        if (!any) continue;
        for (int e = lane; e < MP * 16 * TP; e += 32) {
          const int m = grp_i * MP + e / (16 * TP);
          if (m >= mtc) break;
          float v = P[grp_i * MP * 16 * TP + e];
          for (int w = 0; w < kMmaWarps; ++w)
            if (s_cont[w] == grp_i) v += slot[w * MP * 16 * TP + e];
          P[grp_i * MP * 16 * TP + e] = v;
        }
      }
    }
    // Cluster reduction: rank r owns rows [rows*r/S, rows*(r+1)/S) of the
    // group.  Every rank stores its partial rows into their owner's receive
    // buffer (slot = the sending rank; fire-and-forget distributed
    // shared-memory stores), one cluster barrier, then the owner sums the
    // slots in rank order.
    float* recv = reinterpret_cast<float*>(smem + a.off_recv);  // [S][own_max][TP]
    __syncthreads();  // the partial tile is complete
    if (S > 1) {
      // Where the receive buffer overlays the activations, no rank may
      // store into it before every rank is done with them.
      if (a.recv_alias) cluster_sync();
      if (!abort) {
        const uint32_t rbase = smem_addr(recv);
        for (int s = 0; s < S; ++s) {
          const int o_lo = s_geo[5 + s], o_hi = s_geo[6 + s];
          const int cnt = (o_hi - o_lo) * TP;  // floats, a multiple of 8
          for (int e = 4 * tid; e < cnt; e += 4 * kMmaThreads) {
            const float4 v = *reinterpret_cast<const float4*>(P + o_lo * TP + e);
            const uint32_t local = rbase + static_cast<uint32_t>((rank * a.own_max * TP + e) * 4);
            uint32_t remote;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(static_cast<uint32_t>(s)));
            asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y),
                         "f"(v.z), "f"(v.w)
                         : "memory");
          }
        }
      }
      cluster_sync();  // every rank's rows are in their owners' receive buffers
    }
    if (!abort) {
      const int o_lo = s_geo[5 + rank], o_hi = s_geo[6 + rank];
      for (int r = o_lo + warp; r < o_hi; r += kMmaWarps) {
        for (int tok = lane; tok < a.t; tok += 32) {
          float v = 0.0f;
          if (S > 1) {
            for (int s = 0; s < S; ++s) v += recv[(s * a.own_max + (r - o_lo)) * TP + tok];
          } else {
            v = P[r * TP + tok];
          }
          const int64_t yi = static_cast<int64_t>(tok) * a.n + row0 + r;
          a.y[yi] = RES ? v + a.res[yi] : v;
        }
      }
    }
  }
  if (abort && tid == 0) {
    raise_status(a.status, kStatusTimeout);
    for (int m = 0; m < mtc; ++m) (void)mbar_wait(&bars[m], 0);  // let copies land (bounded)
  }
}

// --------------------------------------------------------------- host --

namespace {

struct MmaLayout {
  uint32_t act_row, off_da, off_slab, off_p, off_slot, off_recv, off_bar;
  int own_max;
  bool recv_alias;
  size_t bytes;
};

// Shared-memory bytes per weight row: the slice of bc blocks, copied from up
// to 15 bytes before its start to up to 15 bytes past its end.
uint32_t mma_slab_row(int fmt, int nb, int split) {
  const int bc_max = (nb + split - 1) / split;
  const int kbb = fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes;
  return (static_cast<uint32_t>(bc_max) * kbb + 30u + 15u) & ~15u;
}

// Shared-memory layout of one CTA.  With `alias`, the cluster reduction's
// receive buffer overlays the activation area (dead once the units are done)
// instead of having its own.
MmaLayout mma_layout(int nt, int fmt, int nb, int split, int mt_max, bool alias = false) {
  const int tp = 8 * nt;
  const int bc_max = (nb + split - 1) / split;
  MmaLayout L{};
  L.act_row = static_cast<uint32_t>(bc_max) * 512u + 64u;  // 64 mod 128: conflict-free B loads
  L.own_max = (mt_max * 16 + split - 1) / split;
  const size_t recv_bytes = split > 1 ? static_cast<size_t>(split) * L.own_max * tp * 4 : 0;
  L.recv_alias = alias && split > 1;
  size_t off = static_cast<size_t>(tp) * L.act_row;
  L.off_da = static_cast<uint32_t>(off);
  off += static_cast<size_t>(bc_max) * 8 * tp * (mma_biased(nt) ? 8 : 4);  // d_a (and the seeds)
  if (L.recv_alias) off = std::max(off, recv_bytes);
  off = (off + 127) & ~size_t(127);
  L.off_slab = static_cast<uint32_t>(off);
  const uint32_t slab_row = mma_slab_row(fmt, nb, split);
  off += static_cast<size_t>(mt_max) * 16 * slab_row;
  off = (off + 15) & ~size_t(15);
  L.off_p = static_cast<uint32_t>(off);
  off += static_cast<size_t>(mt_max) * 16 * tp * 4;
  L.off_slot = static_cast<uint32_t>(off);
  off += static_cast<size_t>(kMmaWarps) * 16 * tp * 4;
  if (L.recv_alias) {
    L.off_recv = 0;
  } else {
    L.off_recv = static_cast<uint32_t>(off);
    off += recv_bytes;
  }
  L.off_bar = static_cast<uint32_t>(off);
  off += static_cast<size_t>(mt_max) * 8;
  L.bytes = off;
  return L;
}

template <int NT, int FMT, bool PART, bool RES>
bool configure_mma_kernel() {
  static std::atomic<bool> configured[64];
  const DeviceInfo& di = device_info();
  if (di.device < 0 || di.device >= 64) return false;
  if (!configured[di.device].load(std::memory_order_acquire)) {
    if (!cuda_ok(cudaFuncSetAttribute(mmv_mma_kernel<NT, FMT, PART, RES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kMmaSmemBudget))))
      return false;
    configured[di.device].store(true, std::memory_order_release);
  }
  return true;
}

template <int NT, int FMT, bool PART, bool RES>
int launch_mma_kernel(MmaArgs a, size_t smem, cudaStream_t s) {
  if (!configure_mma_kernel<NT, FMT, PART, RES>()) return TQ1_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.groups * a.split));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (a.split > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(a.split);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cuda_ok(cudaLaunchKernelEx(&cfg, mmv_mma_kernel<NT, FMT, PART, RES>, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

// Clusters of `split` CTAs of this instantiation with `smem` bytes of shared
// memory each that the GPU holds at once (CTAs for split 1), cached per
// device, split and 4 KiB of shared memory; 0 when none fit.
template <int NT, int FMT, bool PART, bool RES>
int resident_clusters(int split, size_t smem) {
  static std::mutex mu;
  constexpr int kClasses = static_cast<int>(kMmaSmemBudget / 4096) + 1;
  static int cache[64][kMmaMaxSplit + 1][kClasses];  // 0: not queried yet; -1: none fit
  const DeviceInfo& di = device_info();
  if (di.device < 0 || di.device >= 64 || split < 1 || split > kMmaMaxSplit) return 0;
  const int cls = static_cast<int>((smem + 4095) / 4096);
  if (cls >= kClasses) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[di.device][split][cls];
  if (c == 0) {
    int n = 0;
    const size_t bytes = std::min(static_cast<size_t>(cls) * 4096, kMmaSmemBudget);  // the class's largest size
    if (!configure_mma_kernel<NT, FMT, PART, RES>()) return 0;
    if (split == 1) {
      int per_sm = 0;
      if (!cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mmv_mma_kernel<NT, FMT, PART, RES>,
                                                                  kMmaThreads, bytes)))
        per_sm = 0;
      n = per_sm * di.num_sms;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(split * 64));
      cfg.blockDim = dim3(kMmaThreads);
      cfg.dynamicSmemBytes = bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(split);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (!cuda_ok(cudaOccupancyMaxActiveClusters(&n, mmv_mma_kernel<NT, FMT, PART, RES>, &cfg))) n = 0;
    }
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// Split (K ranges per cluster) and row groups for one call, then the launch.
// One wave of resident clusters; estimated cost per CTA, in thread
// instructions: its units (M-tile x block: ~340 for the expansion plus ~48 per
// n-tile, over 8 warps), staging its activations (~1.7 per token slot and
// block), and the cluster reduction.
template <int NT, int FMT, bool PART, bool RES>
int plan_and_launch(MmaArgs a, cudaStream_t s) {
  const DeviceInfo& di = device_info();
  constexpr int tp = 8 * NT;
  const int nb = a.nb;
  const int64_t mt_total = a.mt_total;
  int best_split = 0, best_groups = 0, best_mt = 0;
  bool best_alias = false;
  double best_cost = 1e300;
  for (int sp = 1; sp <= std::min(kMmaMaxSplit, nb); ++sp) {
    const int bc = (nb + sp - 1) / sp;
    for (int al = 0; al < (sp > 1 ? 2 : 1); ++al) {
      // Row groups: one wave of resident clusters, or (tall matrices whose
      // M-tiles per group would not fit) several waves.
      for (int waves = 1; waves <= 8; ++waves) {
        int64_t groups = std::max<int64_t>(1, std::min<int64_t>(mt_total, waves * (di.num_sms / sp)));
        int mt_max = 0, rc = 0;
        bool fits = false;
        for (int it = 0; it < 3; ++it) {  // groups -> shared memory -> resident clusters -> groups
          mt_max = static_cast<int>((mt_total + groups - 1) / groups);
          if (mt_max > kMmaThreads) break;
          const size_t bytes = mma_layout(NT, FMT, nb, sp, mt_max, al != 0).bytes;
          if (bytes > kMmaSmemBudget) break;
          rc = resident_clusters<NT, FMT, PART, RES>(sp, bytes);
          if (rc <= 0) break;
          if (static_cast<int64_t>(rc) * waves >= groups) {
            fits = true;
            break;
          }
          groups = std::min<int64_t>(mt_total, static_cast<int64_t>(rc) * waves);
        }
        if (!fits) continue;
        const int64_t nwaves = (groups + rc - 1) / rc;
        const double cta = bc * (mt_max * (340.0 + 48.0 * NT) / kMmaWarps + 1.7 * tp) +
                           (sp > 1 ? 16.0 * mt_max * 16.0 * tp / 256.0 : 0.0) + (al ? 150.0 : 0.0);
        const double cost = nwaves * cta;
        if (cost < best_cost) {
          best_cost = cost;
          best_split = sp;
          best_groups = static_cast<int>(groups);
          best_mt = mt_max;
          best_alias = al != 0;
        }
        break;  // more waves than needed only add cost
      }
    }
  }
  if (best_split == 0) return TQ1_ERR_UNSUPPORTED;
  const MmaLayout L = mma_layout(NT, FMT, nb, best_split, best_mt, best_alias);
  a.groups = best_groups;
  a.split = best_split;
  a.mt_max = best_mt;
  a.bc_max = (nb + best_split - 1) / best_split;
  a.slab_row = mma_slab_row(FMT, nb, best_split);
  a.act_row = L.act_row;
  a.off_da = L.off_da;
  a.off_slab = L.off_slab;
  a.off_p = L.off_p;
  a.off_slot = L.off_slot;
  a.off_recv = L.off_recv;
  a.off_bar = L.off_bar;
  a.own_max = L.own_max;
  a.recv_alias = L.recv_alias ? 1 : 0;
  a.pow3 = kPow3Packed;
  return launch_mma_kernel<NT, FMT, PART, RES>(a, L.bytes, s);
}

template <int NT>
int dispatch_mma(const MmaArgs& a, int fmt, cudaStream_t s) {
  if (fmt == kFmtTq2)
    return a.part ? plan_and_launch<NT, kFmtTq2, true, false>(a, s)
                  : (a.res ? plan_and_launch<NT, kFmtTq2, false, true>(a, s)
                           : plan_and_launch<NT, kFmtTq2, false, false>(a, s));
  return a.part ? plan_and_launch<NT, kFmtTq1, true, false>(a, s)
                : (a.res ? plan_and_launch<NT, kFmtTq1, false, true>(a, s)
                         : plan_and_launch<NT, kFmtTq1, false, false>(a, s));
}

}  // namespace

// 1 <= t <= 32 on the warp-level tensor cores (y, or the exact partials when
// `part` is given).  Returns TQ1_ERR_UNSUPPORTED (launching nothing) when no
// split fits the shared-memory budget.
int launch_mmv_mma(const uint8_t* w, const uint8_t* q8, float* y, int32_t* part, int64_t n, int64_t k, int64_t t,
                   cudaStream_t s, unsigned* status, const float* res, int fmt) {
  if (t < 1 || t > 32 || n < 1) return TQ1_ERR_UNSUPPORTED;
  const int64_t mt_total = (n + 15) / 16;
  if (mt_total > (int64_t{1} << 24)) return TQ1_ERR_UNSUPPORTED;
  MmaArgs a = {};
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.part = part;
  a.res = part ? nullptr : res;
  a.status = status;
  a.n = n;
  a.t = static_cast<int>(t);
  a.nb = static_cast<int>(k / kQK);
  a.mt_total = static_cast<int>(mt_total);
  switch ((t + 7) / 8) {
    case 1: return dispatch_mma<1>(a, fmt, s);
    case 2: return dispatch_mma<2>(a, fmt, s);
    case 3: return dispatch_mma<3>(a, fmt, s);
    default: return dispatch_mma<4>(a, fmt, s);
  }
}

}  // namespace tq1
