// prefill.cu -- dense TQ1_0 x Q8_1 contraction for t >= 256 token columns on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Prefill was the one place the pages' CUDA patch helped (PrismML-Eng/
// llama.cpp issue #139, "Measured impact": prompt processing improved once
// the ops left the CPU); at hundreds of columns the mat-vec is a dense
// contraction and belongs on the tensor cores.  sm_103a has no integer MMA
// kind, so the contraction runs in kind::f16 on operands that reproduce the
// method's products exactly:
//
//   A[row][k] = fp16(d_w * trit)           exact: trit in {-1, 0, 1}, d_w is fp16
//   x[t][k]   = d_a * q * 2^-e_t            exact in fp32 (11 + 7 significant bits)
//   x = hi + lo,  hi = fp16(x), lo = fp16(x - hi)   (lo exact unless subnormal)
//   y[t][row] = 2^e_t * (sum_k A*hi + sum_k A*lo)   fp32 accumulation in TMEM
//
// e_t is a per-token power of two that keeps 127 * max d_a below 2^14 (it is 0
// for ordinary activations).  Every product A*hi, A*lo is exact; only the fp32
// accumulation rounds.
//
// Structure (one CTA per SM, persistent over 128-row x 128-token tiles):
//  * warps 0-3: expand one weight row each (byte-major base-3 expansion, one
//    quarter of a 256-block per 64-wide K stage) into fp16 +-d_w values,
//    written straight into the 128B-swizzled K-major operand layout;
//  * warps 4-7: turn one token's two Q8_1 blocks per stage into fp16 hi/lo;
//  * thread 0 issues 2 x 4 tcgen05.mma (M=128, N=128, K=16; hi then lo) per
//    stage into one fp32 TMEM accumulator and commits them to the stage's
//    mbarrier; stages are double-buffered so expansion of stage s+1 overlaps
//    the MMAs of stage s;
//  * epilogue: tcgen05.ld of the 128 x 128 accumulator, scale by 2^e_t, store
//    y rows (consecutive lanes = consecutive output rows: coalesced).
// Every wait is bounded; a timeout sets the status word and the CTA leaves
// after letting its in-flight MMAs finish.
#include <algorithm>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kPThreads = 256;
constexpr int kTileM = 128;   // weight rows per tile (TMEM lanes)
constexpr int kTileN = 128;   // tokens per tile (TMEM columns)
constexpr int kStageK = 64;   // K per stage: one 128-byte swizzle atom of fp16
constexpr uint32_t kOpBytes = kTileM * kStageK * 2;  // 16 KB per operand tile
constexpr uint32_t kStageBytes = 3 * kOpBytes;       // A | B hi | B lo
// Two stages + alignment slack, padded past half of the SM's shared memory so
// that the persistent grid spreads one CTA per SM.
constexpr uint32_t kPrefillSmem = 120 * 1024;
static_assert(2 * kStageBytes + 1024 <= kPrefillSmem, "stage buffers exceed the shared-memory request");

// Shared-memory matrix descriptor for a K-major operand tile in the 128-byte
// swizzled layout: 8-row groups of 128-byte rows, groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading offset (unused: K fits one atom row)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A and B fp16, both K-major, N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((static_cast<uint32_t>(kTileN) >> 3) << 17) |
                            ((static_cast<uint32_t>(kTileM) >> 4) << 24);

// Byte offset of fp16 element (r, k) (k < 64) in a swizzled 128 x 64 tile.
__device__ __forceinline__ uint32_t sw_off(int r, int k) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 fp32 accumulator columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// P_k = floor(b * 3^k / 256) of the four bytes of x (see expand_digits).
template <int K>
__device__ __forceinline__ uint32_t pk(uint32_t lo, uint32_t hi) {
  return __byte_perm(lo * pow3(K), hi * pow3(K), 0x7351u);
}

// Four fp16 values (digit - 1) * d_w from one digit word: a byte permute
// reads them from the table {-d_w, 0, +d_w}; the selector of a digit pair
// (D0, D1) is 34 * (D0 + 256 * D1) + 0x1010, both pairs from one multiply-add.
__device__ __forceinline__ uint2 digits_to_f16(uint32_t D, uint32_t tlo, uint32_t thi) {
  const uint32_t sel = D * 34u + 0x10101010u;
  return make_uint2(__byte_perm(tlo, thi, sel), __byte_perm(tlo, thi, sel >> 16));
}

struct PrefArgs {
  const uint8_t* w;
  const uint8_t* q8;
  float* y;
  unsigned* status;
  int n, k, t;
  int tiles_m, tiles_n;
};

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const PrefArgs a) {
  extern __shared__ __align__(1024) uint8_t psmem_raw[];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ float s_scale[kTileN];
  __shared__ int s_abort;
  const uint32_t raw = smem_addr(psmem_raw);
  uint8_t* sm = psmem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_addr(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = a.k / kQK;
  const int nstages = a.k / kStageK;
  const int64_t rowbytes = static_cast<int64_t>(nb) * kBlockBytes;
  const int64_t q8row = static_cast<int64_t>(a.k / kQK8) * kQ8Bytes;
  const int ntiles = a.tiles_m * a.tiles_n;

  if (tid == 0) {
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                 "r"(kTileN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  pdl_launch_dependents();
  pdl_wait();

  uint32_t g = 0;  // CTA-global stage counter (selects the buffer and the barrier phase)
  bool ok = true;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int tm = tile / a.tiles_n, tn = tile - (tile / a.tiles_n) * a.tiles_n;
    const int row0 = tm * kTileM, tok0 = tn * kTileN;

    // Per-token power-of-two scale (B threads), shared with the epilogue.
    if (tid >= 128) {
      const int tl = tid - 128, tok = tok0 + tl;
      float e_scale = 1.0f;
      if (tok < a.t) {
        const uint8_t* qr = a.q8 + static_cast<int64_t>(tok) * q8row;
        float dm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int nq = a.k / kQK8;  // a multiple of 8
        for (int j = 0; j < nq; j += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dm[u] = fmaxf(dm[u], fabsf(__half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(
                                      qr + static_cast<int64_t>(j + u) * kQ8Bytes))))));
        }
        const float dmax = fmaxf(fmaxf(fmaxf(dm[0], dm[1]), fmaxf(dm[2], dm[3])), fmaxf(fmaxf(dm[4], dm[5]), fmaxf(dm[6], dm[7])));
        int ex = 0;
        (void)frexpf(dmax * 127.0f, &ex);  // 127 * dmax < 2^ex
        const int e = max(0, ex - 14);
        e_scale = ldexpf(1.0f, e);
      }
      s_scale[tl] = e_scale;
    }

    // Weight row (A threads): the current block's 14 words (realigned) and
    // the next block's raw words, fetched a block (four stages) ahead.
    const int arow = row0 + tid;  // valid for tid < 128
    uint32_t wv[14], wn[14];
    uint32_t tlo = 0, thi = 0;
    auto load_block = [&](int b, uint32_t (&dst)[14]) {
      const uint8_t* blk = a.w + static_cast<int64_t>(arow) * rowbytes + static_cast<int64_t>(b) * kBlockBytes;
      const uintptr_t addr = reinterpret_cast<uintptr_t>(blk);
      const uint32_t* p = reinterpret_cast<const uint32_t*>(addr & ~static_cast<uintptr_t>(3));
#pragma unroll
      for (int m = 0; m < 13; ++m) dst[m] = __ldg(p + m);
      // The last word: the block ends 2 bytes into it when the block is
      // 4-byte aligned, so read only the scale's 16 bits then (the final
      // block of the matrix ends at the end of the buffer).
      dst[13] = (addr & 3u) ? __ldg(p + 13) : static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(blk + 52)));
    };
    if (tid < 128 && arow < a.n) load_block(0, wn);

    // Token (B threads): the current stage's two Q8_1 blocks, fetched a stage
    // ahead.
    const int btok = tok0 + (tid - 128);  // valid for tid >= 128
    uint32_t qc[2][9], qn[2][9];
    auto load_q = [&](int st2, uint32_t (&dst)[2][9]) {
      const uint32_t* s = reinterpret_cast<const uint32_t*>(a.q8 + static_cast<int64_t>(btok) * q8row +
                                                            static_cast<int64_t>(2 * st2) * kQ8Bytes);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < 9; ++m) dst[h][m] = __ldg(s + 9 * h + m);
    };
    if (tid >= 128 && btok < a.t) load_q(0, qn);

    for (int st = 0; st < nstages && ok; ++st, ++g) {
      const uint32_t buf = g & 1u;
      uint8_t* sA = sm + buf * kStageBytes;
      uint8_t* sBh = sA + kOpBytes;
      uint8_t* sBl = sBh + kOpBytes;
      // Buffer reuse: the MMAs of stage g-2 read this buffer.
      if (g >= 2 && !mbar_wait(&mma_done[buf], ((g - 2) >> 1) & 1u)) ok = false;

      if (tid < 128) {
        // ---- A: one weight row, K elements [64 st, 64 st + 64) ----
        const int b = st >> 2, qtr = st & 3;
        if (arow < a.n) {
          if (qtr == 0) {
            const uint32_t sh = (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(
                                     a.w + static_cast<int64_t>(arow) * rowbytes + static_cast<int64_t>(b) * kBlockBytes)) &
                                 2u) * 8u;
            // Realign the 13 logical words; the scale follows.
#pragma unroll
            for (int m = 0; m < 13; ++m) wv[m] = __funnelshift_r(wn[m], wn[m + 1], sh);
            wv[13] = wn[13];
            if (b + 1 < nb) load_block(b + 1, wn);
            const uint32_t h = (wv[13] >> sh) & 0xFFFFu;
            tlo = h ^ 0x8000u;  // bytes 0-1: -d_w, bytes 2-3: 0
            thi = h;            // bytes 4-5: +d_w
          }
          // Digit words of this quarter, in element order: chunk j, word w
          // -> K offset 32 (j - 2 qtr) + 4 w within the stage.
          auto put = [&](int j, int wd, uint32_t D) {
            const uint2 v = digits_to_f16(D, tlo, thi);
            const int kk = 32 * (j - 2 * qtr) + 4 * wd;
            *reinterpret_cast<uint2*>(sA + sw_off(tid, kk)) = v;
          };
          if (qtr == 0) {
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {
              const uint32_t lo = __byte_perm(wv[wd], 0u, 0x4240u), hi = __byte_perm(wv[wd], 0u, 0x4341u);
              const uint32_t p1 = pk<1>(lo, hi), p2 = pk<2>(lo, hi);
              put(0, wd, p1);
              put(1, wd, p2 - 3u * p1);
            }
          } else if (qtr == 1) {
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {
              const uint32_t lo = __byte_perm(wv[wd], 0u, 0x4240u), hi = __byte_perm(wv[wd], 0u, 0x4341u);
              const uint32_t p2 = pk<2>(lo, hi), p3 = pk<3>(lo, hi), p4 = pk<4>(lo, hi);
              put(2, wd, p3 - 3u * p2);
              put(3, wd, p4 - 3u * p3);
            }
          } else if (qtr == 2) {
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {  // chunk 4: digit 4 of qs words 0..7
              const uint32_t lo = __byte_perm(wv[wd], 0u, 0x4240u), hi = __byte_perm(wv[wd], 0u, 0x4341u);
              put(4, wd, pk<5>(lo, hi) - 3u * pk<4>(lo, hi));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // chunk 5: digits 0 / 1 of qs words 8..11
              const uint32_t lo = __byte_perm(wv[8 + i], 0u, 0x4240u), hi = __byte_perm(wv[8 + i], 0u, 0x4341u);
              const uint32_t p1 = pk<1>(lo, hi), p2 = pk<2>(lo, hi);
              put(5, i, p1);
              put(5, 4 + i, p2 - 3u * p1);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // chunks 6, 7: digits 2, 3, 4 of qs words 8..11
              const uint32_t lo = __byte_perm(wv[8 + i], 0u, 0x4240u), hi = __byte_perm(wv[8 + i], 0u, 0x4341u);
              const uint32_t p2 = pk<2>(lo, hi), p3 = pk<3>(lo, hi), p4 = pk<4>(lo, hi), p5 = pk<5>(lo, hi);
              put(6, i, p3 - 3u * p2);
              put(6, 4 + i, p4 - 3u * p3);
              put(7, i, p5 - 3u * p4);
            }
            {  // chunk 7, words 4..7: the qh digits
              const uint32_t lo = __byte_perm(wv[12], 0u, 0x4240u), hi = __byte_perm(wv[12], 0u, 0x4341u);
              const uint32_t p1 = pk<1>(lo, hi), p2 = pk<2>(lo, hi), p3 = pk<3>(lo, hi), p4 = pk<4>(lo, hi);
              put(7, 4, p1);
              put(7, 5, p2 - 3u * p1);
              put(7, 6, p3 - 3u * p2);
              put(7, 7, p4 - 3u * p3);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(sA + sw_off(tid, 8 * c)) = make_uint4(0, 0, 0, 0);
        }
      } else {
        // ---- B: one token, Q8_1 blocks 2 st and 2 st + 1 -> fp16 hi / lo ----
        const int tl = tid - 128, tok = tok0 + tl;
        if (tok < a.t) {
          const float inv = 1.0f / s_scale[tl];  // exact: a power of two
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int m = 0; m < 9; ++m) qc[h][m] = qn[h][m];
          if (st + 1 < nstages) load_q(st + 1, qn);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(qc[h][0] & 0xFFFFu))) * inv;
            const __half2 d2 = __float2half2_rn(da);
            const __half2 c1152 = __float2half2_rn(1152.0f);
#pragma unroll
            for (int wq = 0; wq < 8; wq += 2) {
              uint32_t hv[4], lv[4];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                // int8 q -> exact fp16: bias to 0..255, place under the
                // exponent of 1024 (0x64xx), subtract 1024 + 128.
                const uint32_t x = qc[h][1 + wq + u] ^ 0x80808080u;
                const uint32_t m01 = __byte_perm(x, 0x64646464u, 0x5150u);
                const uint32_t m23 = __byte_perm(x, 0x64646464u, 0x5352u);
                const __half2 q01 = __hsub2(*reinterpret_cast<const __half2*>(&m01), c1152);
                const __half2 q23 = __hsub2(*reinterpret_cast<const __half2*>(&m23), c1152);
                const __half2 h01 = __hmul2(q01, d2), h23 = __hmul2(q23, d2);
                const __half2 l01 = __hfma2(q01, d2, __hneg2(h01)), l23 = __hfma2(q23, d2, __hneg2(h23));
                hv[2 * u] = *reinterpret_cast<const uint32_t*>(&h01);
                hv[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&h23);
                lv[2 * u] = *reinterpret_cast<const uint32_t*>(&l01);
                lv[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&l23);
              }
              const int kk = 32 * h + 4 * wq;  // 8 elements = one 16-byte chunk
              *reinterpret_cast<uint4*>(sBh + sw_off(tl, kk)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
              *reinterpret_cast<uint4*>(sBl + sw_off(tl, kk)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(sBh + sw_off(tl, 8 * c)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sBl + sw_off(tl, 8 * c)) = make_uint4(0, 0, 0, 0);
          }
        }
      }

      fence_proxy_async();  // operand stores -> visible to the tensor cores
      if (!ok) s_abort = 1;
      __syncthreads();
      if (s_abort) {
        ok = false;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
        const uint32_t a0 = sbase + buf * kStageBytes;
#pragma unroll
        for (int ks = 0; ks < kStageK / 16; ++ks) {
          const uint32_t off = static_cast<uint32_t>(ks) * 32u;
          umma_f16(tmem, umma_desc_sw128(a0 + off), umma_desc_sw128(a0 + kOpBytes + off), (st > 0 || ks > 0) ? 1u : 0u);
          umma_f16(tmem, umma_desc_sw128(a0 + off), umma_desc_sw128(a0 + 2 * kOpBytes + off), 1u);
        }
        umma_commit(&mma_done[buf]);
      }
    }
    if (!ok) break;

    // ---- epilogue: all MMAs of the tile are covered by the last commit ----
    const uint32_t glast = g - 1;
    if (!mbar_wait(&mma_done[glast & 1u], (glast >> 1) & 1u)) ok = false;
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int q4 = warp & 3;             // TMEM lane quarter of this warp
      const int c0 = (warp >> 2) * 64;     // warps 0-3: columns 0..63, warps 4-7: 64..127
      const int row = row0 + q4 * 32 + lane;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(c0 + 32 * half), v);
        if (row < a.n) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tcol = c0 + 32 * half + j;
            const int tok = tok0 + tcol;
            if (tok < a.t) a.y[static_cast<int64_t>(tok) * a.n + row] = __uint_as_float(v[j]) * s_scale[tcol];
          }
        }
      }
    }
    if (!ok) s_abort = 1;
    tc_fence_before();
    __syncthreads();  // accumulator and scales free for the next tile
    if (s_abort) {
      ok = false;
      break;
    }
  }
  if (!ok) {
    if (tid == 0) raise_status(a.status, kStatusTimeout);
    // Let issued MMAs finish (bounded) before the tensor memory is released.
    if (tid == 0 && g > 0) (void)mbar_wait(&mma_done[(g - 1) & 1u], ((g - 1) >> 1) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTileN));
}

int launch_prefill(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, void*, size_t,
                   cudaStream_t s, unsigned* status) {
  if (n > (int64_t{1} << 30) || t > (int64_t{1} << 30) || k > (int64_t{1} << 30)) return TQ1_ERR_UNSUPPORTED;
  const DeviceInfo& di = device_info();
  static bool configured[64] = {};
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (!configured[di.device]) {
    if (!cuda_ok(cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kPrefillSmem))))
      return TQ1_ERR_CUDA;
    configured[di.device] = true;
  }
  PrefArgs a = {};
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.status = status;
  a.n = static_cast<int>(n);
  a.k = static_cast<int>(k);
  a.t = static_cast<int>(t);
  a.tiles_m = static_cast<int>((n + kTileM - 1) / kTileM);
  a.tiles_n = static_cast<int>((t + kTileN - 1) / kTileN);
  const int64_t ntiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  const int grid = static_cast<int>(std::min<int64_t>(ntiles, di.num_sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPrefillSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, prefill_kernel, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

}  // namespace tq1
