// mmv_small.cu -- TQ1_0 x Q8_1 mat-vec for 1, 2 and 4 token columns: the
// decode path.
//
// PrismML-Eng/llama.cpp issue #139, "Proposed approach" option 1: a kernel
// that consumes whole 256-element blocks and iterates over packed bytes, so
// each packed byte is loaded from HBM once and expanded to all of its digits
// in registers.  Activation words are reused across the four rows a warp
// handles at a time and across all rows of a CTA (strata PR #1418,
// "Descricao": a column's Q8_1 fragment loaded once and reused across output
// rows).
//
// Calls in a stream are dependent (a call's activations may come from the
// previous kernel), so each call's critical path is: the previous kernel
// retires -> activations are read -> dot products -> outputs.  The base-3
// expansion of the weights does not depend on the activations, so it is
// moved off that path:
//
//  1. Before waiting on the previous kernel (programmatic dependent launch),
//     the CTA requests its weight rows from HBM with one 1-D bulk copy (TMA
//     engine) per 4-row group, and each warp expands its first tasks' blocks
//     into packed digit registers while the previous call is still running.
//  2. After the wait, the activation records are staged once per CTA and the
//     dot products run on the pre-expanded digits.
//
// Packed digits: a block's 256 trits become 64 digit words (4 digits of 0..2
// per word, one per byte lane).  Four digit words that pair with the same
// activation word index w but belong to Q8_1 chunks j = s, s+1.. (slot s = j
// mod 4) share one register: bits 2s..2s+1 of every byte lane.  Masking slot
// s leaves 4^s * digit in each lane, which an unsigned-by-signed dp4a uses
// directly; the exact factor 4^s is folded into the chunk's fp32 scale and
// -sum(q) seed, so the per-chunk integer partial stays exact.
//
// Work decomposition: a task is 4 rows x 8 consecutive 256-blocks; lane =
// (row r, block s).  The 8 lanes of a row combine their fp32 partials with
// shuffles; per-(row, 8-block chunk) results are summed in a fixed order at
// the end (no atomics: bitwise deterministic).
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

// Per column count: threads per CTA, tasks pre-expanded per warp (held in
// registers across the wait), and the weight-slab budget.
template <int C>
struct SmallCfg;
template <>
struct SmallCfg<1> {
  static constexpr int kThreads = 512;
  static constexpr int kHeld = 2;
  static constexpr uint32_t kSlab = 96 * 1024;
};
template <>
struct SmallCfg<2> {
  static constexpr int kThreads = 256;
  static constexpr int kHeld = 4;
  static constexpr uint32_t kSlab = 80 * 1024;
};
template <>
struct SmallCfg<4> {
  static constexpr int kThreads = 256;
  static constexpr int kHeld = 4;
  static constexpr uint32_t kSlab = 64 * 1024;
};

struct SmallArgs {
  const uint8_t* w;
  const uint8_t* q8;
  float* y;
  unsigned* status;
  int64_t n;
  int t;                // active columns (<= C)
  int nb;               // blocks per row
  int rows_round;       // rows per slab round (multiple of 4)
  int rows_cta;         // max rows of any CTA (partials sizing)
  int nkc;              // 8-block chunks per row
  uint32_t slab_bytes;  // shared memory for weight rows (rounds of rows_round rows)
  uint32_t nkc_magic;   // ceil(2^32 / nkc) for nkc > 1: task / nkc == umulhi(task, magic)
};

// Activation record of one column over one 256-block (word-major so that the
// four activation words meeting one packed register are contiguous):
//   words 8w + j  (w, j < 8): int8x4 word w of Q8_1 chunk j
//   words 64 + j:  chunk j's fp32 scale divided by 4^(j mod 4)
//   words 72 + j:  -4^(j mod 4) * sum of chunk j's int8 values
constexpr int kPRec = 100;  // stride: 16-byte aligned, 4 banks apart

struct Packed {
  uint32_t a[8];  // slots 0..3: chunks 0..3, activation word w
  uint32_t b[8];  // slots 0..3: chunks 4..7, activation word w
  float dw;
};

// Expand the block at byte offset `off` (even) of shared memory `slab` into
// packed digits.  Element order (PrismML-Eng/llama.cpp issue #139, "Current
// behavior", continued over the last 16 qs bytes and the 4 qh bytes):
//   qs word w < 8,  digit j      -> chunk j,         word w
//   qs word 8 + i,  digit 0 / 1  -> chunk 5,         word i / 4 + i
//                   digit 2 / 3  -> chunk 6,         word i / 4 + i
//                   digit 4      -> chunk 7,         word i
//   qh word,        digit k      -> chunk 7,         word 4 + k
__device__ __forceinline__ void expand_pack(const uint8_t* slab, uint32_t off, Packed& P) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(slab + (off & ~3u));
  const uint32_t sh = (off & 2u) * 8u;
  uint32_t w[14];
#pragma unroll
  for (int m = 0; m < 14; ++m) w[m] = p[m];
  // Chunks 5..7 first (slots 1..3 of the b registers).
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t d[5];
    expand_digits<5>(__funnelshift_r(w[8 + i], w[9 + i], sh), d);
    P.b[i] = (d[0] << 2) | (d[2] << 4) | (d[4] << 6);
    P.b[4 + i] = (d[1] << 2) | (d[3] << 4);
  }
  {
    uint32_t d[4];
    expand_digits<4>(__funnelshift_r(w[12], w[13], sh), d);
#pragma unroll
    for (int k = 0; k < 4; ++k) P.b[4 + k] |= d[k] << 6;
  }
  // Chunks 0..4.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t d[5];
    expand_digits<5>(__funnelshift_r(w[i], w[i + 1], sh), d);
    P.a[i] = d[0] | (d[1] << 2) | (d[2] << 4) | (d[3] << 6);
    P.b[i] |= d[4];
  }
  P.dw = __half2float(__ushort_as_half(static_cast<unsigned short>((w[13] >> sh) & 0xFFFFu)));
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// d_w * sum_j d_a[j] * I_j for one packed block against one column record.
__device__ __forceinline__ float packed_dot(const Packed& P, const uint32_t* rec) {
  const int4 s0 = *reinterpret_cast<const int4*>(rec + 72);
  const int4 s1 = *reinterpret_cast<const int4*>(rec + 76);
  int I0 = s0.x, I1 = s0.y, I2 = s0.z, I3 = s0.w, I4 = s1.x, I5 = s1.y, I6 = s1.z, I7 = s1.w;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint4 qa = *reinterpret_cast<const uint4*>(rec + 8 * w);
    const uint4 qb = *reinterpret_cast<const uint4*>(rec + 8 * w + 4);
    I0 = dp4a_us(P.a[w] & 0x03030303u, qa.x, I0);
    I1 = dp4a_us(P.a[w] & 0x0C0C0C0Cu, qa.y, I1);
    I2 = dp4a_us(P.a[w] & 0x30303030u, qa.z, I2);
    I3 = dp4a_us(P.a[w] & 0xC0C0C0C0u, qa.w, I3);
    I4 = dp4a_us(P.b[w] & 0x03030303u, qb.x, I4);
    I5 = dp4a_us(P.b[w] & 0x0C0C0C0Cu, qb.y, I5);
    I6 = dp4a_us(P.b[w] & 0x30303030u, qb.z, I6);
    I7 = dp4a_us(P.b[w] & 0xC0C0C0C0u, qb.w, I7);
  }
  const float4 a0 = *reinterpret_cast<const float4*>(rec + 64);
  const float4 a1 = *reinterpret_cast<const float4*>(rec + 68);
  float s = a0.x * static_cast<float>(I0);
  s = fmaf(a0.y, static_cast<float>(I1), s);
  s = fmaf(a0.z, static_cast<float>(I2), s);
  s = fmaf(a0.w, static_cast<float>(I3), s);
  s = fmaf(a1.x, static_cast<float>(I4), s);
  s = fmaf(a1.y, static_cast<float>(I5), s);
  s = fmaf(a1.z, static_cast<float>(I6), s);
  s = fmaf(a1.w, static_cast<float>(I7), s);
  return s * P.dw;
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
  rec[72 + j] = static_cast<uint32_t>(-(sum << (2 * slot)));
}

}  // namespace

template <int C>
__global__ void __launch_bounds__(SmallCfg<C>::kThreads, 2) mmv_small_kernel(const SmallArgs a) {
  constexpr int kThreads = SmallCfg<C>::kThreads;
  constexpr int kWarps = kThreads / 32;
  constexpr int kHeld = SmallCfg<C>::kHeld;
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb;
  const int nkc = a.nkc;  // 8-block chunks per row
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * kBlockBytes;
  const uint32_t gstride = group_stride(rowbytes);
  // Layout: slab | activation records | per-(row, chunk) partials | barriers
  uint8_t* slab = smem;
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + a.slab_bytes);
  const uint32_t rstride = static_cast<uint32_t>(nb) * kPRec;  // words per column
  float* part = reinterpret_cast<float*>(recs + static_cast<size_t>(C) * rstride);
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + ((static_cast<size_t>(a.rows_cta) * nkc * C + 1) & ~size_t(1)));
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = lane >> 3, s = lane & 7;
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

  // Task `task` of round `rd`: its group, chunk and this lane's block offset.
  struct TaskPos {
    int g, kc, row;
    bool live;
    uint32_t off;
  };
  auto task_pos = [&](int rd, int task) {
    TaskPos T;
    const int rs = rd * a.rows_round;
    T.g = nkc == 1 ? task : static_cast<int>(__umulhi(static_cast<uint32_t>(task), a.nkc_magic));
    T.kc = task - T.g * nkc;
    T.row = rs + T.g * kRowsPerTask + r;
    const int b = T.kc * kLanesPerRow + s;
    T.live = T.row < rows && b < nb;
    const uint32_t gbase = static_cast<uint32_t>(rs + T.g * kRowsPerTask) * rowbytes;
    T.off = static_cast<uint32_t>(T.g) * gstride + ((wlow + gbase) & 15u) + static_cast<uint32_t>(r) * rowbytes +
            static_cast<uint32_t>(b) * kBlockBytes;
    return T;
  };

  if (tid == 0) {
    s_abort = 0;
    for (int g = 0; g < kMaxGroups; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
    if (nrounds > 0) issue_round(0);  // weights: before waiting on the previous kernel
  }
  __syncthreads();
  pdl_launch_dependents();

  // Phase 1 (overlaps the previous kernel): expand this warp's first tasks.
  const int ntasks0 = nrounds > 0 ? ((min(a.rows_round, rows) + kRowsPerTask - 1) / kRowsPerTask) * nkc : 0;
  Packed held[kHeld];
  bool ok = true;
#pragma unroll
  for (int h = 0; h < kHeld; ++h) {
    const int task = warp + h * kWarps;
    if (task < ntasks0) {
      const TaskPos T = task_pos(0, task);
      if (!mbar_wait(&bars[T.g], 0)) ok = false;
      if (ok && T.live) expand_pack(slab, T.off, held[h]);
    }
  }

  pdl_wait();

  // Phase 2: activation records of the C columns, then the dot products.
  {
    const int nchunks = a.t * nb * 8;
    for (int i = tid; i < nchunks; i += kThreads) {
      const int c = i / (nb * 8);
      const int rem = i - c * nb * 8;
      const int b = rem >> 3, j = rem & 7;
      fill_precord_chunk(a.q8 + static_cast<int64_t>(i) * kQ8Bytes, recs + c * rstride + b * kPRec, j);
    }
  }
  if (!ok) s_abort = 1;
  __syncthreads();

  // Reduce a task's per-lane partials over the row's 8 lanes and store them.
  auto finish_task = [&](const TaskPos& T, float (&acc)[C]) {
#pragma unroll
    for (int c = 0; c < C; ++c) {
      float v = acc[c];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      acc[c] = v;
    }
    if (s == 0 && T.row < rows) {
#pragma unroll
      for (int c = 0; c < C; ++c) part[(static_cast<size_t>(T.row) * nkc + T.kc) * C + c] = acc[c];
    }
  };
  auto dot_task = [&](const TaskPos& T, const Packed& P) {
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.0f;
    if (T.live) {
      const int b = T.kc * kLanesPerRow + s;
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (c < a.t) acc[c] = packed_dot(P, recs + c * rstride + b * kPRec);
    }
    finish_task(T, acc);
  };

  if (!s_abort) {
#pragma unroll
    for (int h = 0; h < kHeld; ++h) {
      const int task = warp + h * kWarps;
      if (task < ntasks0) dot_task(task_pos(0, task), held[h]);
    }
  }
  for (int rd = 0; rd < nrounds && !s_abort; ++rd) {
    const int rs = rd * a.rows_round;
    const int ngroups = (min(a.rows_round, rows - rs) + kRowsPerTask - 1) / kRowsPerTask;
    const int ntasks = ngroups * nkc;
    const uint32_t parity = static_cast<uint32_t>(rd & 1);
    // Tasks not expanded before the wait (warp w: w + k * warps).
    for (int task = warp + (rd == 0 ? kHeld * kWarps : 0); task < ntasks; task += kWarps) {
      const TaskPos T = task_pos(rd, task);
      if (!mbar_wait(&bars[T.g], parity)) {
        ok = false;
        break;
      }
      Packed P;
      if (T.live) expand_pack(slab, T.off, P);
      dot_task(T, P);
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
    if (tid == 0) {
      raise_status(a.status, kStatusTimeout);
      const int ngroups = (min(a.rows_round, rows) + kRowsPerTask - 1) / kRowsPerTask;
      for (int g = 0; g < ngroups; ++g) (void)mbar_wait(&bars[g], 0);
    }
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
  b += static_cast<size_t>(C) * nb * kPRec * 4;
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
