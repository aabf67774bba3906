// mmv_small.cu -- TQ1_0 x Q8_1 mat-vec for 1, 2 and 4 token columns: the
// decode path, streamed at HBM rate.
//
// PrismML-Eng/llama.cpp issue #139, "Proposed approach" option 1: a kernel
// that consumes whole 256-element blocks and iterates over packed bytes, so
// each packed byte is loaded from HBM once and expanded to all of its digits
// in registers.  Activation words are reused across the four rows a warp
// handles at a time and across all of a CTA's rows (strata PR #1418,
// "Descricao": a column's Q8_1 fragment loaded once and reused across output
// rows).
//
// Work decomposition (one CTA per SM, two CTAs of consecutive calls
// co-resident so that a call's weight streaming overlaps its predecessor):
//  * the CTA owns rows [r0, r1) of the output, split evenly over the grid;
//  * a task is 4 rows x 8 consecutive 256-blocks; lane = (row r, block s);
//    each lane folds its block into fp32 partial sums, the 8 lanes of a row
//    combine them with shuffles, and per-(row, block-chunk) results are summed
//    in a fixed order at the end (no atomics: bitwise deterministic);
//  * the CTA's weight bytes move HBM -> shared memory with one 1-D bulk copy
//    per 4-row group (TMA engine), each completing on its own mbarrier, all
//    requested before the kernel waits on the previous kernel in the stream;
//  * a block is decoded a quarter at a time (4 words -> 20 digit words) so
//    that only 20 digit registers are live.
#include <algorithm>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kRowsPerTask = 4;
constexpr int kLanesPerRow = 8;  // = blocks per task chunk
constexpr int kMaxGroups = 64;   // row groups (mbarriers) per round

// Shared-memory bytes reserved per 4-row group: up to 15 bytes of alignment
// slack before the rows, the rows, and the decoder's over-read after them;
// a multiple of 16 so every group's bulk-copy destination is 16-byte aligned.
__host__ __device__ __forceinline__ uint32_t group_stride(uint32_t rowbytes) {
  return (kRowsPerTask * rowbytes + 32u + 15u) & ~15u;
}

template <int C>
struct SmallCfg;
template <>
struct SmallCfg<1> {
  static constexpr int kThreads = 512;
  static constexpr uint32_t kSlab = 96 * 1024;
};
template <>
struct SmallCfg<2> {
  static constexpr int kThreads = 512;
  static constexpr uint32_t kSlab = 80 * 1024;
};
template <>
struct SmallCfg<4> {
  static constexpr int kThreads = 256;
  static constexpr uint32_t kSlab = 64 * 1024;
};

struct SmallArgs {
  const uint8_t* w;
  const uint8_t* q8;
  float* y;
  unsigned* status;
  int64_t n;
  int t;          // active columns (<= C)
  int nb;         // blocks per row
  int rows_round; // rows per slab round (multiple of 4)
  int rows_cta;   // max rows of any CTA (partials sizing)
  int nkc;        // 8-block chunks per row
  uint32_t slab_bytes;  // shared memory for weight rows (rounds of rows_round rows)
  uint32_t nkc_magic;  // ceil(2^32 / nkc) for nkc > 1: task / nkc == umulhi(task, magic)
};

// Accumulate the exact chunk partials of four qs words (logical words
// q0..q0+3 of the block) into I, for one column's activation record.
//   group A (q0 = 0 or 4): digit j -> chunk j, words q0..q0+3
//   group B (q0 = 8):      digit k -> chunk 5 + k/2 (k < 4) or 7, half k%2
template <bool kGroupB>
__device__ __forceinline__ void quarter_dot(const uint32_t (&d)[4][5], const uint32_t* rec, int q0, int (&I)[8]) {
  if (!kGroupB) {
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      const uint4 q = *reinterpret_cast<const uint4*>(rec + 8 * j + q0);
      int acc = I[j];
      acc = __dp4a(static_cast<int>(d[0][j]), static_cast<int>(q.x), acc);
      acc = __dp4a(static_cast<int>(d[1][j]), static_cast<int>(q.y), acc);
      acc = __dp4a(static_cast<int>(d[2][j]), static_cast<int>(q.z), acc);
      acc = __dp4a(static_cast<int>(d[3][j]), static_cast<int>(q.w), acc);
      I[j] = acc;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int chunk = k < 4 ? 5 + (k >> 1) : 7;
      const int half = k < 4 ? (k & 1) : 0;
      const uint4 q = *reinterpret_cast<const uint4*>(rec + 8 * chunk + 4 * half);
      int acc = I[chunk];
      acc = __dp4a(static_cast<int>(d[0][k]), static_cast<int>(q.x), acc);
      acc = __dp4a(static_cast<int>(d[1][k]), static_cast<int>(q.y), acc);
      acc = __dp4a(static_cast<int>(d[2][k]), static_cast<int>(q.z), acc);
      acc = __dp4a(static_cast<int>(d[3][k]), static_cast<int>(q.w), acc);
      I[chunk] = acc;
    }
  }
}

// One lane's unit: the 256-block at byte offset `off` (even) of shared memory
// `slab`, against C activation records starting at `rec0` (stride recs).
// Adds d_w * sum_j d_a[j] * I_j to acc[c].
template <int C>
__device__ __forceinline__ void unit_dot(const uint8_t* slab, uint32_t off, const uint32_t* rec0, uint32_t rstride,
                                         int t, float (&acc)[C]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(slab + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;
  int I[C][8];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    if (c < t) {
      const int4 s0 = *reinterpret_cast<const int4*>(rec0 + c * rstride + 72);
      const int4 s1 = *reinterpret_cast<const int4*>(rec0 + c * rstride + 76);
      I[c][0] = s0.x; I[c][1] = s0.y; I[c][2] = s0.z; I[c][3] = s0.w;
      I[c][4] = s1.x; I[c][5] = s1.y; I[c][6] = s1.z; I[c][7] = s1.w;
    }
  }
  uint32_t wprev = p[0];
#pragma unroll
  for (int qtr = 0; qtr < 3; ++qtr) {
    uint32_t d[4][5];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t wn = p[4 * qtr + i + 1];
      expand_digits<5>(__funnelshift_r(wprev, wn, sh), d[i]);
      wprev = wn;
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
      if (c < t) {
        if (qtr < 2) quarter_dot<false>(d, rec0 + c * rstride, 4 * qtr, I[c]);
        else quarter_dot<true>(d, rec0 + c * rstride, 0, I[c]);
      }
    }
  }
  // qh word (4 digits) -> chunk 7, words 4..7; then the block scale.
  const uint32_t w13 = p[13];
  uint32_t dq[4];
  expand_digits<4>(__funnelshift_r(wprev, w13, sh), dq);
  const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w13 >> sh) & 0xFFFFu)));
#pragma unroll
  for (int c = 0; c < C; ++c) {
    if (c < t) {
      const uint32_t* rec = rec0 + c * rstride;
      const uint4 q = *reinterpret_cast<const uint4*>(rec + 60);
      int acc7 = I[c][7];
      acc7 = __dp4a(static_cast<int>(dq[0]), static_cast<int>(q.x), acc7);
      acc7 = __dp4a(static_cast<int>(dq[1]), static_cast<int>(q.y), acc7);
      acc7 = __dp4a(static_cast<int>(dq[2]), static_cast<int>(q.z), acc7);
      acc7 = __dp4a(static_cast<int>(dq[3]), static_cast<int>(q.w), acc7);
      I[c][7] = acc7;
      const float4 a0 = *reinterpret_cast<const float4*>(rec + 64);
      const float4 a1 = *reinterpret_cast<const float4*>(rec + 68);
      float s = a0.x * static_cast<float>(I[c][0]);
      s = fmaf(a0.y, static_cast<float>(I[c][1]), s);
      s = fmaf(a0.z, static_cast<float>(I[c][2]), s);
      s = fmaf(a0.w, static_cast<float>(I[c][3]), s);
      s = fmaf(a1.x, static_cast<float>(I[c][4]), s);
      s = fmaf(a1.y, static_cast<float>(I[c][5]), s);
      s = fmaf(a1.z, static_cast<float>(I[c][6]), s);
      s = fmaf(a1.w, static_cast<float>(I[c][7]), s);
      acc[c] = fmaf(dw, s, acc[c]);
    }
  }
}

}  // namespace

template <int C>
__global__ void __launch_bounds__(SmallCfg<C>::kThreads, 2) mmv_small_kernel(const SmallArgs a) {
  constexpr int kThreads = SmallCfg<C>::kThreads;
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb;
  const int nkc = a.nkc;  // 8-block chunks per row
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * kBlockBytes;
  const uint32_t gstride = group_stride(rowbytes);
  // Layout: slab | activation records | per-(row, chunk) partials | barriers
  uint8_t* slab = smem;
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + a.slab_bytes);
  const uint32_t rstride = static_cast<uint32_t>(nb) * kRecWords;  // words per column
  float* part = reinterpret_cast<float*>(recs + static_cast<size_t>(C) * rstride);
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + ((static_cast<size_t>(a.rows_cta) * nkc * C + 1) & ~size_t(1)));
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t r0 = (a.n * blockIdx.x) / gridDim.x;
  const int64_t r1 = (a.n * (blockIdx.x + 1)) / gridDim.x;
  const int rows = static_cast<int>(r1 - r0);
  const int nrounds = (rows + a.rows_round - 1) / a.rows_round;
  const uint64_t policy = l2_evict_first_policy();
  const uint8_t* wcta = a.w + r0 * rowbytes;
  const uint32_t wlow = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(wcta));

  // Issue round `rd`: one bulk copy per 4-row group, each on its mbarrier.
  // A group's bytes start on any even byte; the copy starts at the 16-byte
  // boundary below, and the tail past the last 16-byte boundary is copied
  // with plain loads before the arrive (release -> acquire via the barrier).
  auto issue_round = [&](int rd) {
    const int rs = rd * a.rows_round;
    const int rrows = min(a.rows_round, rows - rs);
    const int ngroups = (rrows + kRowsPerTask - 1) / kRowsPerTask;
    for (int g = 0; g < ngroups; ++g) {
      const int gr = rs + g * kRowsPerTask;
      const int grows = min(kRowsPerTask, rows - gr);
      const uint8_t* src = wcta + static_cast<int64_t>(gr) * rowbytes;
      const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
      const uint32_t total = delta + static_cast<uint32_t>(grows) * rowbytes;
      const uint32_t main = total & ~15u;
      uint8_t* dst = slab + static_cast<uint32_t>(g) * gstride;
      for (uint32_t i = main; i < total; ++i) dst[i] = __ldg(src - delta + i);
      mbar_arrive_expect_tx(&bars[g], main);
      if (main) bulk_g2s(dst, src - delta, main, &bars[g], policy);
    }
  };

  if (tid == 0) {
    s_abort = 0;
    for (int g = 0; g < kMaxGroups; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
    if (nrounds > 0) issue_round(0);  // weights: before waiting on the previous kernel
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  // Activations (written by earlier work in the stream): records with fp32
  // chunk scales and -sum(q), one Q8_1 block per thread.  (Measured faster
  // here than one bulk copy followed by a shared-memory repack.)
  {
    const int nchunks = a.t * nb * 8;
    for (int i = tid; i < nchunks; i += kThreads) {
      const int c = i / (nb * 8);
      const int rem = i - c * nb * 8;
      const int b = rem >> 3, j = rem & 7;
      fill_record_chunk(a.q8 + static_cast<int64_t>(i - j) * kQ8Bytes, recs + c * rstride + b * kRecWords, j);
    }
  }
  bool ok = true;
  __syncthreads();

  const int r = lane >> 3, s = lane & 7;
  for (int rd = 0; rd < nrounds && !s_abort; ++rd) {
    const int rs = rd * a.rows_round;
    const int rrows = min(a.rows_round, rows - rs);
    const int ngroups = (rrows + kRowsPerTask - 1) / kRowsPerTask;
    const int ntasks = ngroups * nkc;
    const uint32_t parity = static_cast<uint32_t>(rd & 1);
    // Warp w takes tasks w, w + warps, ...; each task's results land in
    // fixed slots.  (A shared work counter measured slower.)
    for (int task = tid >> 5; task < ntasks; task += kThreads / 32) {
      const int g = nkc == 1 ? task : static_cast<int>(__umulhi(static_cast<uint32_t>(task), a.nkc_magic));
      const int kc = task - g * nkc;
      if (!mbar_wait(&bars[g], parity)) {
        ok = false;
        break;
      }
      const int row = rs + g * kRowsPerTask + r;
      const int b = kc * kLanesPerRow + s;
      float acc[C];
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = 0.0f;
      if (row < rows && b < nb) {
        const uint32_t gbase = static_cast<uint32_t>(rs + g * kRowsPerTask) * rowbytes;
        const uint32_t off = static_cast<uint32_t>(g) * gstride + ((wlow + gbase) & 15u) +
                             static_cast<uint32_t>(r) * rowbytes + static_cast<uint32_t>(b) * kBlockBytes;
        unit_dot<C>(slab, off, recs + b * kRecWords, rstride, a.t, acc);
      }
#pragma unroll
      for (int c = 0; c < C; ++c) {
        float v = acc[c];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        acc[c] = v;
      }
      if (s == 0 && row < rows) {
#pragma unroll
        for (int c = 0; c < C; ++c) part[(static_cast<size_t>(row) * nkc + kc) * C + c] = acc[c];
      }
    }
    if (!ok) {
      raise_status(a.status, kStatusTimeout);
      s_abort = 1;
    }
    __syncthreads();  // slab free, all tasks of the round done
    if (s_abort) {
      // Let this round's copies that are still in flight land (bounded)
      // before the CTA gives its shared memory back.
      if (tid == 0)
        for (int g = 0; g < ngroups; ++g) (void)mbar_wait(&bars[g], parity);
      return;
    }
    if (tid == 0 && rd + 1 < nrounds) issue_round(rd + 1);
  }
  if (s_abort) {
    if (tid == 0) raise_status(a.status, kStatusTimeout);
    return;
  }

  // y[c][r0 + row] = sum over block chunks, in order.
  for (int i = tid; i < rows * a.t; i += kThreads) {
    const int c = i / rows, row = i - (i / rows) * rows;
    float v = 0.0f;
    for (int kc = 0; kc < nkc; ++kc) v += part[(static_cast<size_t>(row) * nkc + kc) * C + c];
    a.y[static_cast<int64_t>(c) * a.n + r0 + row] = v;
  }
}

template <int C>
static size_t small_smem(int nb, int rows_cta, uint32_t slab_bytes) {
  const int nkc = (nb + kLanesPerRow - 1) / kLanesPerRow;
  size_t b = slab_bytes;
  b += static_cast<size_t>(C) * nb * kRecWords * 4;
  b += ((static_cast<size_t>(rows_cta) * nkc * C + 1) & ~size_t(1)) * 4;
  b += kMaxGroups * 8;
  return b;
}

template <int C>
static int launch_small_rung(const SmallArgs& a, int grid, cudaStream_t s) {
  const DeviceInfo& di = device_info();
  const size_t bytes = small_smem<C>(a.nb, a.rows_cta, a.slab_bytes);
  static size_t max_dyn[64] = {};
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (max_dyn[di.device] == 0) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, mmv_small_kernel<C>))) return TQ1_ERR_CUDA;
    const size_t lim = di.max_smem_optin - fa.sharedSizeBytes;
    if (!cuda_ok(cudaFuncSetAttribute(mmv_small_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(lim))))
      return TQ1_ERR_CUDA;
    max_dyn[di.device] = lim;
  }
  if (bytes > max_dyn[di.device]) return TQ1_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(SmallCfg<C>::kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, mmv_small_kernel<C>, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

// Returns TQ1_ERR_UNSUPPORTED (launching nothing) when the shape does not
// fit this kernel's staging; the caller then uses the general kernel.
int launch_mmv_small(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, cudaStream_t s,
                     unsigned* status) {
  if (t < 1 || t > 4) return TQ1_ERR_UNSUPPORTED;
  const DeviceInfo& di = device_info();
  SmallArgs a = {};
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.status = status;
  a.n = n;
  a.t = static_cast<int>(t);
  a.nb = static_cast<int>(k / kQK);
  const int rung = t == 1 ? 1 : (t == 2 ? 2 : 4);
  const uint32_t slab = rung == 1 ? SmallCfg<1>::kSlab : (rung == 2 ? SmallCfg<2>::kSlab : SmallCfg<4>::kSlab);
  const uint32_t rowbytes = static_cast<uint32_t>(a.nb) * kBlockBytes;
  // Shared memory is sized to the CTA's rows (capped at the rung's slab
  // budget): two CTAs of consecutive calls must fit on one SM together.
  const int64_t grid = std::min<int64_t>(di.num_sms, n);
  a.rows_cta = static_cast<int>((n + grid - 1) / grid);
  const int groups_needed = (a.rows_cta + kRowsPerTask - 1) / kRowsPerTask;
  const int groups_fit = std::min<int>({kMaxGroups, static_cast<int>(slab / group_stride(rowbytes)), groups_needed});
  if (groups_fit < 1) return TQ1_ERR_UNSUPPORTED;
  a.rows_round = groups_fit * kRowsPerTask;
  a.slab_bytes = static_cast<uint32_t>(groups_fit) * group_stride(rowbytes);
  a.nkc = (a.nb + kLanesPerRow - 1) / kLanesPerRow;
  a.nkc_magic = a.nkc > 1 ? static_cast<uint32_t>(((uint64_t{1} << 32) + a.nkc - 1) / a.nkc) : 0u;
  if (static_cast<int64_t>(a.rows_round / kRowsPerTask) * a.nkc >= (int64_t{1} << 20)) return TQ1_ERR_UNSUPPORTED;
  switch (rung) {
    case 1: return launch_small_rung<1>(a, static_cast<int>(grid), s);
    case 2: return launch_small_rung<2>(a, static_cast<int>(grid), s);
    default: return launch_small_rung<4>(a, static_cast<int>(grid), s);
  }
}

}  // namespace tq1
