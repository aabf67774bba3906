// moe_small.cu -- expert-routed TQ1_0 x Q8_1 mat-vec for decode batches
// (mul_mat_id): the packed-digit decode kernel applied to the experts the
// routing selected.
//
// AMD-Ecosystem/llama.cpp PR #76 ("Summary"): mul_mat_id compacts the ids
// into per-expert bounds and runs a grid over the compacted list, so each
// expert's weights are read once for all the tokens routed to it.  Here a
// task is (active expert, a chunk of up to kChunk of its (token, slot)
// pairs, a range of its rows); the routing table lays the tasks of each
// active expert out contiguously and records where they start.  For small
// routings every CTA builds that table itself in shared memory (the
// compaction kernel's steps; no second kernel ahead of this one), larger ones
// read it from the workspace the compaction kernel filled.  Persistent CTAs
// walk the tasks: per task they request the rows' packed weights with one
// 1-D bulk copy (TMA engine) per 4-row group, each group's copy issued by its
// own thread, stage the chunk's
// activation records, and run the decode kernel's expansion and dot products
// (packed 2-bit digits, masked dp4a) for every pair of the chunk, so each
// packed weight byte is expanded once per chunk.  Outputs go to
// y[pair][row]; sums run in a fixed order (bitwise deterministic).
//
// Both kernels have a partials mode (PART) for the debug entry points: the
// same expansion and dp4a sums, with each lane storing its block's eight exact
// per-chunk integer partials to part[pair][row][k/32] instead of scaling them.
#include <atomic>
#include <algorithm>

#include "../../include/tq1.h"
#include "packed.cuh"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

using namespace packed;

constexpr int kMThreads = 256;
constexpr int kMWarps = kMThreads / 32;
constexpr int kChunk = 4;        // pairs per task
constexpr int kMaxRows = 96;     // rows per task: task granularity (128-row tasks left some CTAs a whole extra task)
// Routings of up to this many pairs (those direct mode cannot stage) take
// tasks of at most 64 rows: with few pairs there are fewer tasks than the
// CTAs can hold, and the longest task sets the time (config 4 at T = 8, 64
// pairs: 19.1 -> 16.4 us; at T = 64, 512 pairs, 64-row tasks took 59.7
// against 57.4 us).
constexpr int64_t kFinePairs = 128;
constexpr int kFineRows = 64;
constexpr int kMaxGroupsM = kMaxRows / kRowsPerTask;
constexpr uint32_t kSlabBudget = 96 * 1024;
constexpr size_t kMoeSmemBudget = 112 * 1024;  // per CTA (two, or three for smaller tasks, per SM)

struct MoeArgs {
  const uint8_t* w;      // expert 0's first weight block
  const uint8_t* q8;     // Q8_1 activations [t][k/32]
  float* y;              // [t * top_k][n]
  int32_t* part;         // PART: exact partials [t * top_k][n][k/32] (y unused)
  unsigned* status;
  const int32_t* table;  // compacted routing table (layout in tq1_internal.h), or
  const int32_t* ids;    // the ids themselves ([t][top_k]): every CTA builds the table in shared memory
  int64_t n;
  int n_experts, top_k, nb, nkc;
  int act_div;           // activation row of a pair = pair / act_div (top_k, or 1: one row per pair)
  int rows;              // rows per task (multiple of 4)
  int row_blocks;        // row ranges per expert
  int64_t pairs;         // t * top_k
  uint32_t slab_bytes;
};

}  // namespace

template <int FMT, bool PART>
__global__ void __launch_bounds__(kMThreads, 3) moe_small_kernel(const MoeArgs a) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb, nkc = a.nkc;
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * kBB;
  const uint32_t gstride = group_stride(rowbytes);
  uint8_t* slab = smem;
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + a.slab_bytes);
  const uint32_t rstride = static_cast<uint32_t>(nb) * kPRec;  // words per pair record
  float* part = reinterpret_cast<float*>(recs + static_cast<size_t>(kChunk) * rstride);
  __shared__ __align__(8) uint64_t bars[kMaxGroupsM];
  __shared__ int s_abort;
  __shared__ int s_nact;
  __shared__ int s_pair[kChunk];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = lane >> 3, s = lane & 7;
  const int ngroups_max = a.rows / kRowsPerTask;
  if (tid == 0) {
    for (int g = 0; g < ngroups_max; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // the routing table is written by the compaction kernel

  const int32_t* bounds = a.table + 1;
  const int32_t* active = bounds + (a.n_experts + 1);
  const int32_t* plist = active + a.n_experts;
  const int32_t* tstart = plist + a.pairs;
  int n_active = 0;
  if (a.ids) {
    // Few routed pairs: every CTA builds the routing table itself, in shared
    // memory, with the compaction kernel's steps (counts, one warp's scans,
    // one warp's stable scatter), so there is no second kernel before this
    // one.  The table (same layout as the compaction's, without the count
    // word) follows the partials.
    const int ne = a.n_experts;
    int32_t* t_cnt = reinterpret_cast<int32_t*>(part + static_cast<size_t>(a.rows) * nkc * kChunk);
    int32_t* t_bounds = t_cnt + ne;
    int32_t* t_active = t_bounds + ne + 1;
    int32_t* t_tstart = t_active + ne;
    int32_t* t_plist = t_tstart + ne + 1;
    for (int i = tid; i < ne; i += kMThreads) t_cnt[i] = 0;
    __syncthreads();
    for (int64_t p = tid; p < a.pairs; p += kMThreads) {
      const int e = __ldg(a.ids + p);
      if (e >= 0 && e < ne) atomicAdd(&t_cnt[e], 1);
      else if (blockIdx.x == 0) raise_status(a.status, kStatusBadId);
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scans of the counts and the tasks, and the active list
      int running = 0, nact = 0, running_tasks = 0;
      for (int base = 0; base < ne; base += 32) {
        const int i = base + lane;
        const int v = i < ne ? t_cnt[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        if (i < ne) t_bounds[i] = running + incl - v;
        const uint32_t has = __ballot_sync(0xffffffffu, v > 0);
        const int nt = v > 0 ? ((v + kChunk - 1) / kChunk) * a.row_blocks : 0;
        int tincl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, tincl, o);
          if (lane >= o) tincl += u;
        }
        if (v > 0) {
          const int slot = nact + __popc(has & ((1u << lane) - 1u));
          t_active[slot] = i;
          t_tstart[slot] = running_tasks + tincl - nt;
        }
        nact += __popc(has);
        running += __shfl_sync(0xffffffffu, incl, 31);
        running_tasks += __shfl_sync(0xffffffffu, tincl, 31);
      }
      if (lane == 0) {
        t_bounds[ne] = running;
        t_tstart[nact] = running_tasks;
        s_nact = nact;
      }
    }
    __syncthreads();
    for (int i = tid; i < ne; i += kMThreads) t_cnt[i] = t_bounds[i];  // scatter cursors
    __syncthreads();
    if (warp == 0) {  // stable scatter of pair indices, 32 at a time, in order
      for (int64_t base = 0; base < a.pairs; base += 32) {
        const int64_t p = base + lane;
        int e = p < a.pairs ? __ldg(a.ids + p) : -1;
        if (e >= ne || e < -1) e = -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0) t_plist[t_cnt[e] + rank] = static_cast<int32_t>(p);
        __syncwarp();
        if (e >= 0 && rank == 0) t_cnt[e] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    bounds = t_bounds;
    active = t_active;
    plist = t_plist;
    tstart = t_tstart;
    n_active = s_nact;
  } else {
    n_active = a.table[0];
  }
  const int total = tstart[n_active];
  const uint64_t policy = l2_evict_first_policy();
  uint32_t iter = 0;  // tasks done by this CTA: every group barrier completes one phase per task

  for (int task = blockIdx.x; task < total; task += gridDim.x, ++iter) {
    // Active expert of this task: the last slot whose first task is <= task.
    int lo = 0, hi = n_active - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tstart[mid] <= task) lo = mid;
      else hi = mid - 1;
    }
    const int e = active[lo];
    const int local = task - tstart[lo];
    const int chunk = local / a.row_blocks, rb = local - (local / a.row_blocks) * a.row_blocks;
    const int cnt = bounds[e + 1] - bounds[e];
    const int pc = min(kChunk, cnt - chunk * kChunk);  // pairs of this task
    const int64_t r0 = static_cast<int64_t>(rb) * a.rows;
    const int rows = static_cast<int>(a.n - r0 < a.rows ? a.n - r0 : a.rows);
    const int ngroups = (rows + kRowsPerTask - 1) / kRowsPerTask;
    const uint8_t* wtask = a.w + (static_cast<int64_t>(e) * a.n + r0) * rowbytes;
    const uint32_t wlow = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(wtask));

    // One bulk copy per 4-row group (thread g issues group g's), from the
    // 16-byte boundary at or below the group; the bytes past the last 16-byte
    // boundary with plain loads.  Groups past this task's rows complete their
    // phase with no bytes, so every barrier advances once per task.
    for (int g = tid; g < ngroups_max; g += kMThreads) {
      if (g < ngroups) {
        const int grows = min(kRowsPerTask, rows - g * kRowsPerTask);
        const uint8_t* src = wtask + static_cast<int64_t>(g) * kRowsPerTask * rowbytes;
        const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
        const uint32_t tot = delta + static_cast<uint32_t>(grows) * rowbytes;
        const uint32_t main = tot & ~15u;
        uint8_t* dst = slab + static_cast<uint32_t>(g) * gstride;
        for (uint32_t i = main; i < tot; ++i) dst[i] = __ldg(src - delta + i);
        mbar_arrive_expect_tx(&bars[g], main);
        if (main) bulk_g2s(dst, src - delta, main, &bars[g], policy);
      } else {
        mbar_arrive_expect_tx(&bars[g], 0);
      }
    }
    if (tid < kChunk) s_pair[tid] = tid < pc ? plist[bounds[e] + chunk * kChunk + tid] : 0;
    // Activation records of the task's pairs (token = pair / top_k), each
    // thread reading its pair from the table (s_pair is read after the next
    // barrier only).
    {
      const int nchunks = pc * nb * 8;
      const int32_t* tpairs = plist + bounds[e] + chunk * kChunk;
      for (int i = tid; i < nchunks; i += kMThreads) {
        const int c = i / (nb * 8);
        const int rem = i - c * nb * 8;
        const int b = rem >> 3, j = rem & 7;
        const int64_t token = tpairs[c] / a.act_div;
        fill_precord_chunk(a.q8 + (token * nb * 8 + b * 8 + j) * kQ8Bytes, recs + c * rstride + b * kPRec, j);
      }
    }
    __syncthreads();

    // Warp tasks: 4 rows x 8 blocks; lane (row r, block s).
    const int wtasks = ngroups * nkc;
    bool ok = true;
    for (int wt = warp; wt < wtasks; wt += kMWarps) {
      const int g = wt / nkc, kc = wt - (wt / nkc) * nkc;
      const int row = g * kRowsPerTask + r;
      const int b = kc * kLanesPerRow + s;
      if (!mbar_wait(&bars[g], iter & 1u)) {
        ok = false;
        break;
      }
      float acc[kChunk] = {0.f, 0.f, 0.f, 0.f};
      if (row < rows && b < nb) {
        Packed P;
        const uint32_t off = static_cast<uint32_t>(g) * gstride + ((wlow + static_cast<uint32_t>(g) * kRowsPerTask * rowbytes) & 15u) +
                             static_cast<uint32_t>(r) * rowbytes + static_cast<uint32_t>(b) * kBB;
        unit_pack<FMT>(slab, off, P);
        if constexpr (PART) {
          for (int c = 0; c < pc; ++c) {
            int I[8];
            packed_sums(P, recs + c * rstride + b * kPRec, I);
            store_partials(a.part + ((static_cast<int64_t>(s_pair[c]) * a.n + r0 + row) * nb + b) * 8, I);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kChunk; ++c)
            if (c < pc) acc[c] = packed_dot(P, recs + c * rstride + b * kPRec);
        }
      }
      if constexpr (!PART) {
#pragma unroll
        for (int c = 0; c < kChunk; ++c) {
          float v = acc[c];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          acc[c] = v;
        }
        if (s == 0 && row < rows) {
#pragma unroll
          for (int c = 0; c < kChunk; ++c) part[(row * nkc + kc) * kChunk + c] = acc[c];
        }
      }
    }
    if (!ok) s_abort = 1;
    __syncthreads();
    if (s_abort) {
      if (tid == 0) {
        raise_status(a.status, kStatusTimeout);
        // Let this task's copies still in flight land (bounded).
        for (int g = 0; g < ngroups_max; ++g) (void)mbar_wait(&bars[g], iter & 1u);
      }
      return;
    }
    // y[pair][r0 + row]: sum over the 8-block chunks, in order.
    for (int i = tid; i < (PART ? 0 : rows * pc); i += kMThreads) {
      const int c = i / rows, row = i - (i / rows) * rows;
      float v = 0.0f;
      for (int kc = 0; kc < nkc; ++kc) v += part[(row * nkc + kc) * kChunk + c];
      a.y[static_cast<int64_t>(s_pair[c]) * a.n + r0 + row] = v;
    }
    __syncthreads();  // slab, records and partials free for the next task
  }
}

// ----------------------------------------------------------- direct mode --
// Few routed pairs (a decode step: t * top_k of a few tens): compacting the
// routing table costs a kernel and two dependent round trips through L2 on
// the critical path, for little weight reuse to gain.  Instead each CTA owns
// one (pair, row range): it reads the pair's expert id itself once the
// previous kernel has finished, requests that expert's rows, builds the
// token's activation records while they arrive, and writes y[pair][rows].
// A pair whose id is outside [0, n_experts) leaves its outputs untouched and
// raises kStatusBadId.
constexpr int kDThreads = 448;
constexpr int kDWarps = kDThreads / 32;
constexpr int kDMaxRows = 128;
constexpr int kDMaxGroups = kDMaxRows / kRowsPerTask;
constexpr size_t kDSmemBudget = 112 * 1024;  // two CTAs per SM

struct DirectArgs {
  const uint8_t* w;      // expert 0's first weight block
  const uint8_t* q8;     // Q8_1 activations [t][k/32]
  const int32_t* ids;    // [t][top_k]
  float* y;              // [t * top_k][n]
  int32_t* part;         // PART: exact partials [t * top_k][n][k/32] (y unused)
  unsigned* status;
  int64_t n;
  int n_experts, top_k, nb, nkc;
  int act_div;           // activation row of a pair = pair / act_div (top_k, or 1: one row per pair)
  int rows;              // rows per CTA (multiple of 4)
  int row_blocks;        // CTAs per pair
  uint32_t slab_bytes;
};

template <int FMT, bool PART>
__global__ void __launch_bounds__(kDThreads, 2) moe_direct_kernel(const DirectArgs a) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  extern __shared__ __align__(128) uint8_t smem[];
  const int nb = a.nb, nkc = a.nkc;
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * kBB;
  const uint32_t gstride = group_stride(rowbytes);
  uint8_t* slab = smem;
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + a.slab_bytes);
  float* part = reinterpret_cast<float*>(recs + static_cast<size_t>(nb) * kPRec);
  __shared__ __align__(8) uint64_t bars[kDMaxGroups];

  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = lane >> 3, s = lane & 7;
  const int pair = static_cast<int>(blockIdx.x) / a.row_blocks;
  const int rb = static_cast<int>(blockIdx.x) - pair * a.row_blocks;
  const int64_t r0 = static_cast<int64_t>(rb) * a.rows;
  const int rows = static_cast<int>(a.n - r0 < a.rows ? a.n - r0 : a.rows);
  const int ngroups = (rows + kRowsPerTask - 1) / kRowsPerTask;
  if (tid == 0) {
    for (int g = 0; g < ngroups; ++g) mbar_init(&bars[g], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the barriers are initialised before any thread arms one
  pdl_wait();  // ids and activations may come from the previous kernel
  const int e = __ldg(a.ids + pair);
  if (e < 0 || e >= a.n_experts) {
    if (tid == 0 && rb == 0) raise_status(a.status, kStatusBadId);
    return;  // no copy was issued
  }
  const uint8_t* wtask = a.w + (static_cast<int64_t>(e) * a.n + r0) * rowbytes;
  const uint32_t wlow = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(wtask));
  {  // one bulk copy per 4-row group, thread g issuing group g's
    const uint64_t policy = l2_evict_first_policy();
    for (int g = tid; g < ngroups; g += kDThreads) {
      const int grows = min(kRowsPerTask, rows - g * kRowsPerTask);
      const uint8_t* src = wtask + static_cast<int64_t>(g) * kRowsPerTask * rowbytes;
      const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
      const uint32_t tot = delta + static_cast<uint32_t>(grows) * rowbytes;
      const uint32_t main = tot & ~15u;
      uint8_t* dst = slab + static_cast<uint32_t>(g) * gstride;
      for (uint32_t i = main; i < tot; ++i) dst[i] = __ldg(src - delta + i);
      mbar_arrive_expect_tx(&bars[g], main);
      if (main) bulk_g2s(dst, src - delta, main, &bars[g], policy);
    }
  }
  // Activation records of the pair's token while the weights arrive.
  const int64_t token = pair / a.act_div;
  for (int i = tid; i < nb * 8; i += kDThreads)
    fill_precord_chunk(a.q8 + (token * nb * 8 + i) * kQ8Bytes, recs + (i >> 3) * kPRec, i & 7);
  __syncthreads();

  // Warp tasks: 4 rows x 8 blocks; lane (row r, block s).
  const int wtasks = ngroups * nkc;
  bool ok = true;
  for (int wt = warp; wt < wtasks; wt += kDWarps) {
    const int g = wt / nkc, kc = wt - (wt / nkc) * nkc;
    const int row = g * kRowsPerTask + r;
    const int b = kc * kLanesPerRow + s;
    if (!mbar_wait(&bars[g], 0)) {
      ok = false;
      break;
    }
    float v = 0.0f;
    if (row < rows && b < nb) {
      Packed P;
      const uint32_t off = static_cast<uint32_t>(g) * gstride +
                           ((wlow + static_cast<uint32_t>(g) * kRowsPerTask * rowbytes) & 15u) +
                           static_cast<uint32_t>(r) * rowbytes + static_cast<uint32_t>(b) * kBB;
      unit_pack<FMT>(slab, off, P);
      if constexpr (PART) {
        int I[8];
        packed_sums(P, recs + b * kPRec, I);
        store_partials(a.part + ((static_cast<int64_t>(pair) * a.n + r0 + row) * nb + b) * 8, I);
      } else {
        v = packed_dot(P, recs + b * kPRec);
      }
    }
    if (PART) continue;
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    if (s == 0 && row < rows) {
      if (nkc == 1) a.y[static_cast<int64_t>(pair) * a.n + r0 + row] = v;
      else part[row * nkc + kc] = v;
    }
  }
  const bool abort = __syncthreads_or(!ok) != 0;
  if (abort) {
    if (tid == 0) {
      raise_status(a.status, kStatusTimeout);
      for (int g = 0; g < ngroups; ++g) (void)mbar_wait(&bars[g], 0);  // let copies land (bounded)
    }
    return;
  }
  if (nkc > 1 && !PART) {
    for (int row = tid; row < rows; row += kDThreads) {
      float v = 0.0f;
      for (int kc = 0; kc < nkc; ++kc) v += part[row * nkc + kc];  // in order
      a.y[static_cast<int64_t>(pair) * a.n + r0 + row] = v;
    }
  }
}

// Rows per CTA so that pairs x row blocks is about one CTA per SM, within the
// shared-memory budget; false if even four rows do not fit.
bool moe_direct_plan(int64_t n, int64_t k, int64_t pairs, MoePlan* plan, int fmt) {
  const DeviceInfo& di = device_info();
  const int nb = static_cast<int>(k / kQK);
  const int nkc = (nb + kLanesPerRow - 1) / kLanesPerRow;
  const uint32_t gs = group_stride(static_cast<uint32_t>(nb) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes));
  // Two CTAs per SM (the kernel's residency): the fewest rows per CTA whose
  // CTAs all fit at once.  Measured on config 4 against one CTA per SM:
  // T = 1 4.8 -> 4.0 us, T = 2 7.1 -> 5.3, T = 3 9.3 -> 6.4, T = 4 9.6 -> 7.7
  // (a probe timing single graph replays).
  const int64_t slots = 2 * static_cast<int64_t>(std::max(1, di.num_sms));
  int64_t rows = (n * pairs + slots - 1) / slots;
  rows = ((std::max<int64_t>(rows, kRowsPerTask) + kRowsPerTask - 1) / kRowsPerTask) * kRowsPerTask;
  while (rows < kDMaxRows && pairs * ((n + rows - 1) / rows) > slots) rows += kRowsPerTask;
  rows = std::min<int64_t>(rows, kDMaxRows);
  auto smem_of = [&](int64_t r) {
    return static_cast<size_t>(r / kRowsPerTask) * gs + static_cast<size_t>(nb) * kPRec * 4 +
           static_cast<size_t>(r) * nkc * 4;
  };
  while (rows > kRowsPerTask && smem_of(rows) > kDSmemBudget) rows -= kRowsPerTask;
  if (smem_of(rows) > kDSmemBudget) return false;
  plan->chunk = 1;
  plan->rows = static_cast<int>(rows);
  plan->row_blocks = static_cast<int>((n + rows - 1) / rows);
  return pairs * plan->row_blocks < (int64_t{1} << 31);
}

int launch_moe_direct(const uint8_t* w, const uint8_t* q8, const int32_t* ids, float* y, int64_t n, int64_t k,
                      int64_t top_k, int64_t n_experts, int64_t pairs, const MoePlan& plan, cudaStream_t s,
                      unsigned* status, int act_div, int fmt, int32_t* part) {
  const DeviceInfo& di = device_info();
  DirectArgs a = {};
  a.part = part;
  a.act_div = act_div;
  a.w = w;
  a.q8 = q8;
  a.ids = ids;
  a.y = y;
  a.status = status;
  a.n = n;
  a.n_experts = static_cast<int>(n_experts);
  a.top_k = static_cast<int>(top_k);
  a.nb = static_cast<int>(k / kQK);
  a.nkc = (a.nb + kLanesPerRow - 1) / kLanesPerRow;
  a.rows = plan.rows;
  a.row_blocks = plan.row_blocks;
  const uint32_t rowbytes = static_cast<uint32_t>(a.nb) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes);
  a.slab_bytes = static_cast<uint32_t>(plan.rows / kRowsPerTask) * group_stride(rowbytes);
  const size_t smem = a.slab_bytes + static_cast<size_t>(a.nb) * kPRec * 4 + static_cast<size_t>(plan.rows) * a.nkc * 4;
  const int kv = (fmt == kFmtTq2 ? 1 : 0) + (part ? 2 : 0);
  auto kern = kv == 0   ? moe_direct_kernel<kFmtTq1, false>
              : kv == 1 ? moe_direct_kernel<kFmtTq2, false>
              : kv == 2 ? moe_direct_kernel<kFmtTq1, true>
                        : moe_direct_kernel<kFmtTq2, true>;
  static std::atomic<bool> configured[4][64];  // per kernel variant and device (racing threads configure twice: idempotent)
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (!configured[kv][di.device].load(std::memory_order_acquire)) {
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kDSmemBudget))))
      return TQ1_ERR_CUDA;
    configured[kv][di.device].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pairs * plan.row_blocks));
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, kern, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

// Rows per task and row blocks per expert: enough tasks for about two per
// CTA slot when every routed pair lands on its own expert, within the shared
// memory budget (two CTAs per SM).
bool moe_small_plan(int64_t n, int64_t k, int64_t pairs, int64_t n_experts, MoePlan* plan, int fmt) {
  const DeviceInfo& di = device_info();
  const int nb = static_cast<int>(k / kQK);
  const int nkc = (nb + kLanesPerRow - 1) / kLanesPerRow;
  const uint32_t rowbytes = static_cast<uint32_t>(nb) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes);
  const int64_t chunks = std::min<int64_t>(pairs, n_experts + pairs / kChunk);
  const int64_t want_tasks = 2 * static_cast<int64_t>(std::max(1, di.num_sms));
  int64_t rows = (n * std::max<int64_t>(chunks, 1) + want_tasks - 1) / want_tasks;
  rows = std::max<int64_t>(16, std::min<int64_t>(pairs <= kFinePairs ? kFineRows : kMaxRows, rows));
  const int64_t fit = kRowsPerTask * static_cast<int64_t>(kSlabBudget / group_stride(rowbytes));
  rows = std::min(rows, fit);
  rows = (rows / kRowsPerTask) * kRowsPerTask;
  if (rows < kRowsPerTask) return false;
  const size_t smem = static_cast<size_t>(rows / kRowsPerTask) * group_stride(rowbytes) +
                      static_cast<size_t>(kChunk) * nb * kPRec * 4 + static_cast<size_t>(rows) * nkc * kChunk * 4;
  if (smem > kMoeSmemBudget) return false;
  plan->chunk = kChunk;
  plan->rows = static_cast<int>(rows);
  plan->row_blocks = static_cast<int>((n + rows - 1) / rows);
  return true;
}

int launch_moe_small(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t top_k,
                     int64_t n_experts, int64_t pairs, const MoePlan& plan, const int32_t* ws, cudaStream_t s,
                     unsigned* status, int act_div, int fmt, int32_t* part, const int32_t* ids) {
  const DeviceInfo& di = device_info();
  MoeArgs a = {};
  a.ids = ids;
  a.part = part;
  a.act_div = act_div;
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.status = status;
  a.table = ws;
  a.n = n;
  a.n_experts = static_cast<int>(n_experts);
  a.top_k = static_cast<int>(top_k);
  a.nb = static_cast<int>(k / kQK);
  a.nkc = (a.nb + kLanesPerRow - 1) / kLanesPerRow;
  a.rows = plan.rows;
  a.row_blocks = plan.row_blocks;
  a.pairs = pairs;
  const uint32_t rowbytes = static_cast<uint32_t>(a.nb) * (fmt == kFmtTq2 ? kTq2BlockBytes : kBlockBytes);
  a.slab_bytes = static_cast<uint32_t>(plan.rows / kRowsPerTask) * group_stride(rowbytes);
  const size_t smem = a.slab_bytes + static_cast<size_t>(kChunk) * a.nb * kPRec * 4 +
                      static_cast<size_t>(plan.rows) * a.nkc * kChunk * 4 + (ids ? moe_table_smem(n_experts, pairs) : 0);
  if (smem > kMoeSmemBudget) return TQ1_ERR_UNSUPPORTED;
  const int kv = (fmt == kFmtTq2 ? 1 : 0) + (part ? 2 : 0);
  auto kern = kv == 0   ? moe_small_kernel<kFmtTq1, false>
              : kv == 1 ? moe_small_kernel<kFmtTq2, false>
              : kv == 2 ? moe_small_kernel<kFmtTq1, true>
                        : moe_small_kernel<kFmtTq2, true>;
  static std::atomic<bool> configured[4][64];  // per kernel variant and device (racing threads configure twice: idempotent)
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (!configured[kv][di.device].load(std::memory_order_acquire)) {
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kMoeSmemBudget))))
      return TQ1_ERR_CUDA;
    // Up to three CTAs share an SM: the largest shared-memory carveout.
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100)))
      return TQ1_ERR_CUDA;
    configured[kv][di.device].store(true, std::memory_order_release);
  }
  // Upper bound on the tasks: every pair on its own expert.
  const int64_t max_tasks = std::min<int64_t>(pairs, n_experts) * plan.row_blocks +
                            (pairs / kChunk) * plan.row_blocks;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(3 * di.num_sms, max_tasks));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, kern, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

}  // namespace tq1
