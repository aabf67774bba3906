// mmv_small.cu -- TQ1_0 x Q8_1 mat-vec for 1 to 8 token columns (rungs of 1,
// 2, 4 and 8 columns): the decode path.  The same kernel runs TQ2_0 weights,
// whose 2-bit codes are already in the packed-digit layout below (no
// expansion step).
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
//
// Partials mode (PART, the debug entry points): the same expansion and the
// same dp4a sums, but each lane stores its block's eight exact per-chunk
// integer partials I_j instead of scaling them (PrismML-Eng/llama.cpp issue
// #139, "Acceptance criteria": the kernel checked against a CPU reference).
#include <atomic>
#include <algorithm>

#include "../../include/tq1.h"
#include "packed.cuh"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

using namespace packed;

constexpr int kMaxGroups = 64;   // row groups (mbarriers) per round

// Per column count: threads per CTA, tasks pre-expanded per warp (held in
// registers across the wait), the weight-slab budget, and pair mode.
//
// Pair mode: a lane holds two rows of one block column and reads each
// activation-record word once for both.  With several columns the record
// reads bind: a lane needs a column's whole 320-byte record for every block
// it handles, shared memory delivers at most 128 bytes per cycle to an SM's
// lanes, and without pairing the four lanes of a task that handle the same
// block each read it (measured with ncu at N=5120, K=6144: ~2270 shared-memory
// wavefronts per SM for every added column, ~1.1 us at 2.07 GHz, against
// ~1390 warp instructions per sub-partition).  Measured per rung in the bench's
// chained-call setting: 8 columns 14.7 -> 12.8 us at t = 8, 2 columns 5.52 ->
// 5.36 us (TQ2_0 4.78 -> 4.40 us); slower at 1 column (3.52 -> 3.98 us: the
// records do not bind there), at 4 columns (t = 3: 6.95 -> 7.80 us) and for
// TQ2_0 at 8 columns (15.2 -> 19.4 us), which keep one row per lane.
template <int C>
struct SmallCfg;
template <>
struct SmallCfg<1> {
  static constexpr int kThreads = 448;  // 14 warps (measured: 3% faster than 16 at N=5120, K=6144)
  static constexpr int kHeld = 2;
  static constexpr uint32_t kSlab = 96 * 1024;
  static constexpr bool kPair = false;
};
template <>
struct SmallCfg<2> {
  static constexpr int kThreads = 448;
  static constexpr int kHeld = 2;
  static constexpr uint32_t kSlab = 80 * 1024;
  static constexpr bool kPair = true;
};
template <>
struct SmallCfg<4> {
  static constexpr int kThreads = 448;
  static constexpr int kHeld = 2;
  static constexpr uint32_t kSlab = 64 * 1024;
  static constexpr bool kPair = false;
};
template <>
struct SmallCfg<8> {
  static constexpr int kThreads = 448;
  static constexpr int kHeld = 2;
  static constexpr uint32_t kSlab = 48 * 1024;
  static constexpr bool kPair = true;
};

struct SmallArgs {
  const uint8_t* w;
  const uint8_t* q8;
  float* y;
  int32_t* part;        // PART: exact partials [t][n][k/32] (y unused)
  const float* res;     // optional residual added to y (same layout), or nullptr
  const float* x;       // fp32 activations [t][k] quantised in the prologue (F32IN), else unused
  unsigned* status;
  int64_t n;
  int t;                // active columns (<= C)
  int nb;               // blocks per row
  int rows_round;       // rows per slab round (multiple of 4)
  int rows_cta;         // max rows of any CTA (partials sizing)
  int nkc;              // 8-block chunks per row
  uint32_t slab_bytes;  // shared memory for weight rows (rounds of rows_round rows)
  uint32_t nkc_magic;   // ceil(2^32 / nkc) for nkc > 1: task / nkc == umulhi(task, magic)
  int inject_timeout;   // test hook: CTA 0 issues no copy for its first row group (its waits give up)
};

}  // namespace

template <int C, bool RES, bool F32IN, int FMT, bool PART = false>
__global__ void __launch_bounds__(SmallCfg<C>::kThreads, 2) mmv_small_kernel(const SmallArgs a) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  constexpr int kThreads = SmallCfg<C>::kThreads;
  constexpr int kWarps = kThreads / 32;
  constexpr int kHeld = SmallCfg<C>::kHeld;
  // Pair mode: half-warp hsel takes task (warp + hsel * warps) and lane
  // (r2, s) of it rows 2 r2 and 2 r2 + 1 at block s; otherwise the warp's 32
  // lanes take one task, lane (r, s) row r at block s.
  constexpr bool kPair = SmallCfg<C>::kPair && !(FMT == kFmtTq2 && C == 8);
  static_assert(!kPair || kHeld == 2, "pair mode holds the two rows of one task");
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb;
  const int nkc = a.nkc;  // 8-block chunks per row
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * kBB;
  const uint32_t gstride = group_stride(rowbytes);
  // Layout: slab | activation records | per-(row, chunk) partials | barriers
  uint8_t* slab = smem;
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + a.slab_bytes);
  const uint32_t rstride = static_cast<uint32_t>(nb) * kPRec;  // words per column
  float* part = reinterpret_cast<float*>(recs + static_cast<size_t>(C) * rstride);
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + ((static_cast<size_t>(a.rows_cta) * nkc * C + 1) & ~size_t(1)));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hsel = kPair ? lane >> 4 : 0;
  const int r = kPair ? ((lane >> 3) & 1) * 2 : lane >> 3, s = lane & 7;
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
      if (a.inject_timeout && blockIdx.x == 0 && rd == 0 && g == 0) continue;  // nothing completes this barrier
      for (uint32_t i = main; i < total; ++i) dst[i] = __ldg(src - delta + i);
      mbar_arrive_expect_tx(&bars[g], main);
      if (main) bulk_g2s(dst, src - delta, main, &bars[g], policy);
    }
  };

  // Task `task` of round `rd`: its group, chunk and this lane's block offset.
  struct TaskPos {
    int g, kc, row;
    bool live, live2;  // live2: pair mode's second row (row + 1, at off + rowbytes)
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
    T.live2 = kPair && T.row + 1 < rows && b < nb;
    const uint32_t gbase = static_cast<uint32_t>(rs + T.g * kRowsPerTask) * rowbytes;
    T.off = static_cast<uint32_t>(T.g) * gstride + ((wlow + gbase) & 15u) + static_cast<uint32_t>(r) * rowbytes +
            static_cast<uint32_t>(b) * kBB;
    return T;
  };

  if (tid == 0) {
    const int nbars = min(kMaxGroups, (a.rows_round + kRowsPerTask - 1) / kRowsPerTask);
    for (int g = 0; g < nbars; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
    if (nrounds > 0) issue_round(0);  // weights: before waiting on the previous kernel
  }
  __syncthreads();
  pdl_launch_dependents();

  // Phase 1 (overlaps the previous kernel): expand this warp's first tasks.
  const int ntasks0 = nrounds > 0 ? ((min(a.rows_round, rows) + kRowsPerTask - 1) / kRowsPerTask) * nkc : 0;
  Packed held[kHeld];
  bool ok = true;
  if constexpr (kPair) {
    const int task = warp + hsel * kWarps;
    if (task < ntasks0) {
      const TaskPos T = task_pos(0, task);
      if (!mbar_wait(&bars[T.g], 0)) ok = false;
      if (ok && T.live) unit_pack<FMT>(slab, T.off, held[0]);
      if (ok && T.live2)
        unit_pack<FMT>(slab, T.off + rowbytes, held[1]);
      else
        held[1] = Packed{};  // a missing second row contributes zeros
    }
  } else {
#pragma unroll
    for (int h = 0; h < kHeld; ++h) {
      const int task = warp + h * kWarps;
      if (task < ntasks0) {
        const TaskPos T = task_pos(0, task);
        if (!mbar_wait(&bars[T.g], 0)) ok = false;
        if (ok && T.live) unit_pack<FMT>(slab, T.off, held[h]);
      }
    }
  }

  pdl_wait();

  // Phase 2: activation records of the C columns, then the dot products.
  // A failed wait anywhere in the CTA aborts it; the vote rides on the
  // barrier that publishes the records (a flag in shared memory read after
  // the barrier measurably slowed the dot phase).
  {
    const int per_col = nb * 8, nchunks = a.t * per_col;
    if (F32IN) {
      // Q8_1 quantisation fused into the prologue: two lanes per 32-element
      // chunk of the fp32 activations (each CTA quantises the whole row);
      // whole warps iterate so the pair shuffles always have every lane.
      for (int base = warp * 32; base < 2 * nchunks; base += kThreads) {
        const int i2 = base + lane;
        const bool live = i2 < 2 * nchunks;
        const int i = live ? i2 >> 1 : 0;
        const int c = i / per_col, rem = i - c * per_col;
        quantize_precord_half(a.x + static_cast<int64_t>(i) * kQK8, recs + c * rstride + (rem >> 3) * kPRec, rem & 7,
                              i2 & 1, live);
      }
    } else {
      for (int i = tid; i < nchunks; i += kThreads) {
        const int c = i / per_col, rem = i - c * per_col;
        fill_precord_chunk(a.q8 + static_cast<int64_t>(i) * kQ8Bytes, recs + c * rstride + (rem >> 3) * kPRec,
                           rem & 7);
      }
    }
  }
  bool abort = __syncthreads_or(!ok) != 0;

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
  // Partials mode: this lane's block of row T.row (and of row T.row + 1 in
  // pair mode), column by column, straight to global memory.
  auto part_out = [&](int c, int row, int b) {
    return a.part + ((static_cast<int64_t>(c) * a.n + r0 + row) * nb + b) * 8;
  };
  auto dot_task = [&](const TaskPos& T, const Packed& P) {
    if constexpr (PART) {
      if (T.live) {
        const int b = T.kc * kLanesPerRow + s;
        for (int c = 0; c < a.t; ++c) {
          int I[8];
          packed_sums(P, recs + c * rstride + b * kPRec, I);
          store_partials(part_out(c, T.row, b), I);
        }
      }
    } else {
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
    }
  };
  // Pair mode: the two rows of this lane's task (valid: the lane's half-warp
  // has a task), column by column; every lane of the warp calls it (shuffles).
  auto dot_pair = [&](const TaskPos& T, bool valid, const Packed& A, const Packed& B) {
    const bool la = valid && T.live;  // the second row is zeros where it does not exist
    const int b = T.kc * kLanesPerRow + s;
    if constexpr (PART) {
      if (la) {
        for (int c = 0; c < a.t; ++c) {
          int I[8], J[8];
          packed_sums2(A, B, recs + c * rstride + b * kPRec, I, J);
          store_partials(part_out(c, T.row, b), I);
          if (T.live2) store_partials(part_out(c, T.row + 1, b), J);
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < C; ++c) {
        if (c < a.t) {
          float va = 0.0f, vb = 0.0f;
          const uint32_t* rec = recs + c * rstride + b * kPRec;
          if (la) packed_dot2(A, B, rec, va, vb);
          va += __shfl_xor_sync(0xffffffffu, va, 1);
          vb += __shfl_xor_sync(0xffffffffu, vb, 1);
          va += __shfl_xor_sync(0xffffffffu, va, 2);
          vb += __shfl_xor_sync(0xffffffffu, vb, 2);
          va += __shfl_xor_sync(0xffffffffu, va, 4);
          vb += __shfl_xor_sync(0xffffffffu, vb, 4);
          if (s == 0 && valid) {
            if (T.row < rows) part[(static_cast<size_t>(T.row) * nkc + T.kc) * C + c] = va;
            if (T.row + 1 < rows) part[(static_cast<size_t>(T.row + 1) * nkc + T.kc) * C + c] = vb;
          }
        }
      }
    }
  };

  if (!abort) {
    if constexpr (kPair) {
      if (warp < ntasks0) {  // warp-uniform; the lane's own task may not exist
        const int task = warp + hsel * kWarps;
        dot_pair(task_pos(0, task), task < ntasks0, held[0], held[1]);
      }
    } else {
#pragma unroll
      for (int h = 0; h < kHeld; ++h) {
        const int task = warp + h * kWarps;
        if (task < ntasks0) dot_task(task_pos(0, task), held[h]);
      }
    }
  }
  int rd = 0;
  for (; rd < nrounds && !abort; ++rd) {
    const int rs = rd * a.rows_round;
    const int ngroups = (min(a.rows_round, rows - rs) + kRowsPerTask - 1) / kRowsPerTask;
    const int ntasks = ngroups * nkc;
    const uint32_t parity = static_cast<uint32_t>(rd & 1);
    // Tasks not expanded before the wait (warp w: w + k * warps).
    if constexpr (kPair) {
      for (int base = warp + (rd == 0 ? 2 * kWarps : 0); base < ntasks; base += 2 * kWarps) {
        const int task = base + hsel * kWarps;
        const bool valid = task < ntasks;
        const TaskPos T = task_pos(rd, valid ? task : base);
        const bool landed = !valid || mbar_wait(&bars[T.g], parity);
        if (__any_sync(0xffffffffu, !landed)) {
          ok = false;
          break;
        }
        Packed P0, P1;
        if (valid && T.live) unit_pack<FMT>(slab, T.off, P0);
        if (valid && T.live2)
          unit_pack<FMT>(slab, T.off + rowbytes, P1);
        else
          P1 = Packed{};
        dot_pair(T, valid, P0, P1);
      }
    } else {
      for (int task = warp + (rd == 0 ? kHeld * kWarps : 0); task < ntasks; task += kWarps) {
        const TaskPos T = task_pos(rd, task);
        if (!mbar_wait(&bars[T.g], parity)) {
          ok = false;
          break;
        }
        Packed P;
        if (T.live) unit_pack<FMT>(slab, T.off, P);
        dot_task(T, P);
      }
    }
    abort = __syncthreads_or(!ok) != 0;  // slab free, all tasks of the round done
    if (abort) break;
    if (tid == 0 && rd + 1 < nrounds) issue_round(rd + 1);
  }
  if (abort) {
    // Let the copies of the round that failed (still in flight, perhaps)
    // land, bounded, before the CTA gives its shared memory back.
    if (tid == 0) {
      raise_status(a.status, kStatusTimeout);
      const int rdw = min(rd, nrounds - 1);
      const int ngroups = (min(a.rows_round, rows - rdw * a.rows_round) + kRowsPerTask - 1) / kRowsPerTask;
      for (int g = 0; g < ngroups; ++g) (void)mbar_wait(&bars[g], static_cast<uint32_t>(rdw & 1));
    }
    return;
  }

  if constexpr (!PART) {
    // y[c][r0 + row] = sum over block chunks, in order.
    for (int c = 0; c < a.t; ++c)
      for (int row = tid; row < rows; row += kThreads) {
        float v = 0.0f;
        for (int kc = 0; kc < nkc; ++kc) v += part[(static_cast<size_t>(row) * nkc + kc) * C + c];
        const int64_t yi = static_cast<int64_t>(c) * a.n + r0 + row;
        a.y[yi] = RES ? v + a.res[yi] : v;
      }
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

template <int C, bool RES, bool F32IN, int FMT, bool PART = false>
static int launch_small_rung(const SmallArgs& a, int grid, cudaStream_t s) {
  const DeviceInfo& di = device_info();
  const size_t bytes = small_smem<C>(a.nb, a.rows_cta, a.slab_bytes);
  static std::atomic<size_t> max_dyn[64];  // per device; 0 until configured (threads may race to configure: idempotent)
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (max_dyn[di.device].load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, mmv_small_kernel<C, RES, F32IN, FMT, PART>))) return TQ1_ERR_CUDA;
    const size_t lim = di.max_smem_optin - fa.sharedSizeBytes;
    if (!cuda_ok(cudaFuncSetAttribute(mmv_small_kernel<C, RES, F32IN, FMT, PART>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(lim))))
      return TQ1_ERR_CUDA;
    // Two CTAs of consecutive calls share an SM: ask for the largest
    // shared-memory carveout so the L1 split never limits residency.
    if (!cuda_ok(cudaFuncSetAttribute(mmv_small_kernel<C, RES, F32IN, FMT, PART>, cudaFuncAttributePreferredSharedMemoryCarveout, 100)))
      return TQ1_ERR_CUDA;
    max_dyn[di.device].store(lim, std::memory_order_release);
  }
  if (bytes > max_dyn[di.device].load(std::memory_order_acquire)) return TQ1_ERR_UNSUPPORTED;
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
  return cuda_ok(cudaLaunchKernelEx(&cfg, mmv_small_kernel<C, RES, F32IN, FMT, PART>, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

// Returns TQ1_ERR_UNSUPPORTED (launching nothing) when the shape does not
// fit this kernel's staging; the caller then uses the general kernel.
int launch_mmv_small(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, cudaStream_t s,
                     unsigned* status, const float* res, const float* x, int fmt, int inject_timeout, int32_t* part) {
  if (t < 1 || t > 8 || (x && t > 4) || (part && (x || res))) return TQ1_ERR_UNSUPPORTED;
  const DeviceInfo& di = device_info();
  SmallArgs a = {};
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.part = part;
  a.res = res;
  a.x = x;
  a.status = status;
  a.inject_timeout = inject_timeout;
  a.n = n;
  a.t = static_cast<int>(t);
  a.nb = static_cast<int>(k / kQK);
  const int rung = t == 1 ? 1 : (t == 2 ? 2 : (t <= 4 ? 4 : 8));
  const uint32_t slab = rung == 1   ? SmallCfg<1>::kSlab
                        : rung == 2 ? SmallCfg<2>::kSlab
                        : rung == 4 ? SmallCfg<4>::kSlab
                                    : SmallCfg<8>::kSlab;
  const uint32_t rowbytes = static_cast<uint32_t>(a.nb) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes);
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
  const int g = static_cast<int>(grid);
  if (part) {
    switch (rung) {
      case 1: return fmt == kFmtTq2 ? launch_small_rung<1, false, false, kFmtTq2, true>(a, g, s)
                                    : launch_small_rung<1, false, false, kFmtTq1, true>(a, g, s);
      case 2: return fmt == kFmtTq2 ? launch_small_rung<2, false, false, kFmtTq2, true>(a, g, s)
                                    : launch_small_rung<2, false, false, kFmtTq1, true>(a, g, s);
      case 4: return fmt == kFmtTq2 ? launch_small_rung<4, false, false, kFmtTq2, true>(a, g, s)
                                    : launch_small_rung<4, false, false, kFmtTq1, true>(a, g, s);
      default: return fmt == kFmtTq2 ? launch_small_rung<8, false, false, kFmtTq2, true>(a, g, s)
                                     : launch_small_rung<8, false, false, kFmtTq1, true>(a, g, s);
    }
  }
  if (fmt == kFmtTq2) {
    switch (rung) {
      case 1: return x ? launch_small_rung<1, false, true, kFmtTq2>(a, g, s)
                       : (res ? launch_small_rung<1, true, false, kFmtTq2>(a, g, s)
                              : launch_small_rung<1, false, false, kFmtTq2>(a, g, s));
      case 2: return x ? launch_small_rung<2, false, true, kFmtTq2>(a, g, s)
                       : (res ? launch_small_rung<2, true, false, kFmtTq2>(a, g, s)
                              : launch_small_rung<2, false, false, kFmtTq2>(a, g, s));
      case 4: return x ? launch_small_rung<4, false, true, kFmtTq2>(a, g, s)
                       : (res ? launch_small_rung<4, true, false, kFmtTq2>(a, g, s)
                              : launch_small_rung<4, false, false, kFmtTq2>(a, g, s));
      default: return res ? launch_small_rung<8, true, false, kFmtTq2>(a, g, s)
                          : launch_small_rung<8, false, false, kFmtTq2>(a, g, s);
    }
  }
  switch (rung) {
    case 1: return x ? launch_small_rung<1, false, true, kFmtTq1>(a, g, s)
                     : (res ? launch_small_rung<1, true, false, kFmtTq1>(a, g, s)
                            : launch_small_rung<1, false, false, kFmtTq1>(a, g, s));
    case 2: return x ? launch_small_rung<2, false, true, kFmtTq1>(a, g, s)
                     : (res ? launch_small_rung<2, true, false, kFmtTq1>(a, g, s)
                            : launch_small_rung<2, false, false, kFmtTq1>(a, g, s));
    case 4: return x ? launch_small_rung<4, false, true, kFmtTq1>(a, g, s)
                     : (res ? launch_small_rung<4, true, false, kFmtTq1>(a, g, s)
                            : launch_small_rung<4, false, false, kFmtTq1>(a, g, s));
    default: return res ? launch_small_rung<8, true, false, kFmtTq1>(a, g, s)
                        : launch_small_rung<8, false, false, kFmtTq1>(a, g, s);
  }
}

}  // namespace tq1
