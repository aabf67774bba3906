// mmv.cu -- TQ1_0 x Q8_1 mat-vec for T <= 32 columns, its debug variant that
// exports the exact per-32 integer partials, and the expert-routed variant;
// the same kernel serves TQ2_0 weights (2-bit codes: the unit's digit words
// are its 16 qs words shifted and masked).
//
// Structure (PrismML-Eng/llama.cpp issue #139, "Proposed approach" option 1:
// a dedicated kernel that consumes whole 256-element blocks and iterates over
// packed bytes, so every packed byte is loaded once):
//
//  * Each CTA owns a contiguous range of output rows.  Its weight bytes are a
//    contiguous stream (row-major blocks), moved HBM -> shared memory by 1-D
//    bulk copies (TMA engine) through a ring of kStages pass buffers.  The
//    first buffers are requested before the kernel waits on its predecessor
//    in the stream (programmatic dependent launch), so weight streaming
//    overlaps the previous kernel's tail.
//  * A pass gives each of the 256 threads one (row, 256-block) unit.  The
//    thread expands the unit's 52 packed bytes into 65 dp4a-ready digit words
//    once (byte-major, see expand_digits) and then reuses them for every
//    column.
//  * Activations are staged once per CTA into per-(column, block) records:
//    int8 words, fp32 chunk scales and -sum(q) (the -1 trit offset enters as
//    the dp4a accumulator seed, so the per-32 integer partial stays exact).
//    Columns are reused across all rows of the CTA (activation reuse across
//    output rows: strata PR #1418 "Descricao").
//  * Per-unit fp32 results are summed per row in a fixed order (deterministic,
//    no atomics) and written once.
#include <atomic>
#include <algorithm>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

constexpr int kThreads = 256;
constexpr int kPassUnits = kThreads;
// Pass bytes (units x block bytes: 13824 for TQ1_0, 16896 for TQ2_0, both
// multiples of 16) and ring stage bytes (+ 16 alignment slack + over-read).
__host__ __device__ constexpr uint32_t pass_bytes(int bb) { return kPassUnits * static_cast<uint32_t>(bb); }
__host__ __device__ constexpr uint32_t stage_bytes(int bb) { return pass_bytes(bb) + 32; }
constexpr int kStages = 3;
constexpr size_t kActBudget = 96 * 1024;   // activation records per CTA
constexpr size_t kAccBudget = 16 * 1024;   // per-tile row accumulators

enum { kModeY = 0, kModePartials = 1, kModeMoe = 2 };

struct MmvArgs {
  const uint8_t* w;   // weight blocks (MoE: expert 0's first block)
  const uint8_t* q8;  // Q8_1 activations [t][k/32]
  float* y;
  const float* res;   // optional residual added to y (same layout), or nullptr
  int32_t* part;
  unsigned* status;
  int64_t n, k, t;
  int nb;             // k / 256
  int bb;             // bytes per weight block (format)
  int cc;             // columns per activation staging chunk
  int rt;             // rows per tile
  int top_k;
  int act_div;        // MoE: activation row of a pair = pair / act_div
  int64_t n_experts;
  const int32_t* table;  // MoE routing table (see tq1_internal.h)
};

struct Tile {
  const uint8_t* src;  // first weight byte of the tile
  int64_t row0;        // first row within its matrix
  int rows;
  int slot;            // MoE: index into the active-expert list, else -1
  int col0, ncols;     // columns [col0, col0 + ncols) of the tile's column list
};

// ---------------------------------------------------------- work planning --
struct Plan {
  int64_t v0, v1;  // this CTA's (virtual) row range
  int ntiles;
};

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ int64_t split_point(int64_t total, int64_t parts, int64_t i) {
  return (total * i) / parts;
}

template <int CMAX, int MODE>
__device__ Tile get_tile(const MmvArgs& a, const Plan& P, int idx) {
  Tile T;
  const int64_t rowbytes = static_cast<int64_t>(a.nb) * a.bb;
  if (MODE != kModeMoe) {
    const int64_t r = P.v0 + static_cast<int64_t>(idx) * a.rt;
    T.row0 = r;
    T.rows = static_cast<int>(min64(a.rt, P.v1 - r));
    T.src = a.w + r * rowbytes;
    T.slot = -1;
    T.col0 = 0;
    T.ncols = static_cast<int>(a.t);
    return T;
  }
  // MoE: virtual rows v = slot * n + r over the active experts, split into
  // row tiles, each crossed with column groups of at most CMAX tokens.
  const int32_t* bounds = a.table + 1;
  const int32_t* active = a.table + 1 + (a.n_experts + 1);
  int i = 0;
  for (int64_t slot = P.v0 / a.n; slot * a.n < P.v1; ++slot) {
    const int64_t rs = max64(P.v0 - slot * a.n, 0);
    const int64_t re = min64(P.v1 - slot * a.n, a.n);
    const int e = active[slot];
    const int cnt = bounds[e + 1] - bounds[e];
    const int ng = (cnt + CMAX - 1) / CMAX;
    const int nrt = static_cast<int>((re - rs + a.rt - 1) / a.rt);
    if (idx < i + nrt * ng) {
      const int rel = idx - i;
      const int rti = rel / ng, g = rel % ng;
      T.row0 = rs + static_cast<int64_t>(rti) * a.rt;
      T.rows = static_cast<int>(min64(a.rt, re - T.row0));
      T.src = a.w + (static_cast<int64_t>(e) * a.n + T.row0) * rowbytes;
      T.slot = static_cast<int>(slot);
      T.col0 = g * CMAX;
      T.ncols = min(CMAX, cnt - g * CMAX);
      return T;
    }
    i += nrt * ng;
  }
  T.rows = 0;
  return T;
}

template <int CMAX, int MODE>
__device__ int count_tiles(const MmvArgs& a, const Plan& P) {
  if (MODE != kModeMoe) return static_cast<int>((P.v1 - P.v0 + a.rt - 1) / a.rt);
  const int32_t* bounds = a.table + 1;
  const int32_t* active = a.table + 1 + (a.n_experts + 1);
  int total = 0;
  for (int64_t slot = P.v0 / a.n; slot * a.n < P.v1; ++slot) {
    const int64_t rs = max64(P.v0 - slot * a.n, 0);
    const int64_t re = min64(P.v1 - slot * a.n, a.n);
    const int e = active[slot];
    const int cnt = bounds[e + 1] - bounds[e];
    total += static_cast<int>((re - rs + a.rt - 1) / a.rt) * ((cnt + CMAX - 1) / CMAX);
  }
  return total;
}

// A cursor over the CTA's pass sequence: tile index, pass within the tile.
struct Cursor {
  int tile, pass, npass;
  Tile T;
};

template <int CMAX, int MODE>
__device__ __forceinline__ void cursor_load(const MmvArgs& a, const Plan& P, Cursor& c) {
  if (c.tile < P.ntiles) {
    c.T = get_tile<CMAX, MODE>(a, P, c.tile);
    c.npass = (c.T.rows * a.nb + kPassUnits - 1) / kPassUnits;
  } else {
    c.npass = 0;
  }
}

template <int CMAX, int MODE>
__device__ __forceinline__ void cursor_next(const MmvArgs& a, const Plan& P, Cursor& c) {
  if (++c.pass >= c.npass) {
    ++c.tile;
    c.pass = 0;
    cursor_load<CMAX, MODE>(a, P, c);
  }
}

// Issue pass (T, p) into ring stage `st`.  The source may start on any even
// byte: the copy starts at the 16-byte boundary below it, and the bytes past
// the last 16-byte boundary are moved with plain loads by this thread before
// it arrives on the barrier (release/acquire through the mbarrier).
__device__ __forceinline__ void issue_pass(const MmvArgs& a, const Tile& T, int p, uint8_t* stage, uint64_t* bar,
                                           uint64_t policy) {
  const int units = min(kPassUnits, T.rows * a.nb - p * kPassUnits);
  const uint8_t* src = T.src + static_cast<int64_t>(p) * pass_bytes(a.bb);
  const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
  const uint8_t* a0 = src - delta;
  const uint32_t total = delta + static_cast<uint32_t>(units) * static_cast<uint32_t>(a.bb);
  const uint32_t main = total & ~15u;
  for (uint32_t i = main; i < total; ++i) stage[i] = __ldg(a0 + i);
  mbar_arrive_expect_tx(bar, main);
  if (main) bulk_g2s(stage, a0, main, bar, policy);
}

template <int CMAX, int MODE, int FMT>
__global__ void __launch_bounds__(kThreads, 2) mmv_kernel(const MmvArgs a) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  constexpr uint32_t kStageBytes = stage_bytes(kBB);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint32_t* act = reinterpret_cast<uint32_t*>(ring + kStages * kStageBytes);
  float* partial = reinterpret_cast<float*>(act + static_cast<size_t>(a.cc) * a.nb * kRecWords);
  float* acc = partial + kPassUnits * a.cc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(acc + a.rt * CMAX + ((a.rt * CMAX) & 1));
  __shared__ const uint8_t* s_qrow[CMAX];
  __shared__ float* s_yrow[CMAX];
  __shared__ const float* s_rrow[CMAX];
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int nb = a.nb;
  const int64_t nq = static_cast<int64_t>(nb) * 8;  // Q8_1 blocks per column

  Plan P;
  if (MODE != kModeMoe) {
    P.v0 = split_point(a.n, gridDim.x, blockIdx.x);
    P.v1 = split_point(a.n, gridDim.x, blockIdx.x + 1);
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  const uint64_t policy = l2_evict_first_policy();
  Cursor prod;          // meaningful in thread 0 only
  uint32_t issued = 0;  // passes requested so far (thread 0)
  if (MODE != kModeMoe) {
    P.ntiles = count_tiles<CMAX, MODE>(a, P);
    if (tid == 0) {
      // Weights do not depend on the previous kernel: start streaming now.
      prod.tile = 0;
      prod.pass = 0;
      cursor_load<CMAX, MODE>(a, P, prod);
      for (int s = 0; s < kStages && prod.tile < P.ntiles; ++s) {
        issue_pass(a, prod.T, prod.pass, ring + s * kStageBytes, &bars[s], policy);
        cursor_next<CMAX, MODE>(a, P, prod);
        ++issued;
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  if (MODE == kModeMoe) {
    const int64_t n_active = a.table[0];
    const int64_t vtotal = n_active * a.n;
    P.v0 = split_point(vtotal, gridDim.x, blockIdx.x);
    P.v1 = split_point(vtotal, gridDim.x, blockIdx.x + 1);
    P.ntiles = P.v1 > P.v0 ? count_tiles<CMAX, MODE>(a, P) : 0;
    if (tid == 0) {
      prod.tile = 0;
      prod.pass = 0;
      cursor_load<CMAX, MODE>(a, P, prod);
      for (int s = 0; s < kStages && prod.tile < P.ntiles; ++s) {
        issue_pass(a, prod.T, prod.pass, ring + s * kStageBytes, &bars[s], policy);
        cursor_next<CMAX, MODE>(a, P, prod);
        ++issued;
      }
    }
  }

  Cursor cons;
  cons.tile = 0;
  cons.pass = 0;
  cursor_load<CMAX, MODE>(a, P, cons);
  int staged_slot = -2, staged_col = -1;  // which columns the records hold
  uint32_t q = 0;                         // CTA-global pass counter

  for (; cons.tile < P.ntiles; ++q) {
    const Tile& T = cons.T;
    const int p = cons.pass;
    const int st = static_cast<int>(q % kStages);
    uint8_t* stage = ring + st * kStageBytes;

    if (p == 0) {  // new tile: column pointers, zeroed accumulators
      if (tid < T.ncols) {
        int64_t token, orow;
        if (MODE == kModeMoe) {
          const int32_t* bounds = a.table + 1;
          const int32_t* active = bounds + (a.n_experts + 1);
          const int32_t* pairs = active + a.n_experts;
          const int e = active[T.slot];
          const int64_t pair = pairs[bounds[e] + T.col0 + tid];
          token = pair / a.act_div;
          orow = pair;
        } else {
          token = T.col0 + tid;
          orow = token;
        }
        s_qrow[tid] = a.q8 + token * nq * kQ8Bytes;
        s_yrow[tid] = (MODE == kModePartials) ? nullptr : a.y + orow * a.n + T.row0;
        s_rrow[tid] = (MODE == kModeY && a.res) ? a.res + orow * a.n + T.row0 : nullptr;
      }
      for (int i = tid; i < a.rt * CMAX; i += kThreads) acc[i] = 0.0f;
      __syncthreads();
    }

    // Wait for this pass's weights (bounded; a timeout aborts the CTA).
    if (!mbar_wait(&bars[st], (q / kStages) & 1u)) {
      raise_status(a.status, kStatusTimeout);
      s_abort = 1;
    }
    __syncthreads();
    if (s_abort) break;

    const int ubase = p * kPassUnits;
    const int units = T.rows * nb;
    const int u = ubase + tid;
    const bool valid = u < units;
    const uint32_t delta =
        static_cast<uint32_t>(reinterpret_cast<uintptr_t>(T.src + static_cast<int64_t>(p) * pass_bytes(kBB)) & 15u);
    typename FmtDigits<FMT>::type D;
    int b = 0, rloc = 0;
    if (valid) {
      decode_block(stage, delta + static_cast<uint32_t>(tid) * kBB, D);
      rloc = u / nb;
      b = u - rloc * nb;
    }

    for (int c0 = 0; c0 < T.ncols; c0 += a.cc) {
      const int ncc = min(a.cc, T.ncols - c0);
      const int key_col = T.col0 + c0;
      if (staged_slot != T.slot || staged_col != key_col || T.ncols > a.cc) {
        // (Re)stage activation records for columns [c0, c0 + ncc).
        if (!(staged_slot == -2)) __syncthreads();
        const int nrec8 = ncc * nb * 8;
        for (int i = tid; i < nrec8; i += kThreads) {
          const int c = i / (nb * 8);
          const int rem = i - c * nb * 8;
          const int bb = rem >> 3, j = rem & 7;
          fill_record_chunk(s_qrow[c0 + c] + static_cast<int64_t>(bb) * 8 * kQ8Bytes,
                            act + (static_cast<size_t>(c) * nb + bb) * kRecWords, j);
        }
        staged_slot = T.slot;
        staged_col = key_col;
        __syncthreads();
      }

      if (MODE == kModePartials) {
        if (valid) {
          for (int c = 0; c < ncc; ++c) {
            int I[8];
            block_partials(D, act + (static_cast<size_t>(c) * nb + b) * kRecWords, I);
            int4* dst = reinterpret_cast<int4*>(a.part + ((T.col0 + c0 + c) * a.n + T.row0 + rloc) * nq + b * 8);
            dst[0] = make_int4(I[0] - kFloatBias, I[1] - kFloatBias, I[2] - kFloatBias, I[3] - kFloatBias);
            dst[1] = make_int4(I[4] - kFloatBias, I[5] - kFloatBias, I[6] - kFloatBias, I[7] - kFloatBias);
          }
        }
      } else {
        if (valid) {
          for (int c = 0; c < ncc; ++c)
            partial[c * kPassUnits + tid] = block_dot(D, act + (static_cast<size_t>(c) * nb + b) * kRecWords);
        }
        __syncthreads();
        // Fixed-order per-row sums of this pass's units.
        const int uend = min(ubase + kPassUnits, units);
        const int rlo = ubase / nb, rhi = (uend - 1) / nb;
        const int tasks = (rhi - rlo + 1) * ncc;
        for (int task = tid; task < tasks; task += kThreads) {
          const int rr = rlo + task / ncc;
          const int c = task - (task / ncc) * ncc;
          const int ua = max(rr * nb, ubase), ub = min((rr + 1) * nb, uend);
          float s = 0.0f;
          for (int uu = ua; uu < ub; ++uu) s += partial[c * kPassUnits + (uu - ubase)];
          acc[rr * CMAX + c0 + c] += s;
        }
      }
    }
    __syncthreads();  // stage and partials free

    if (tid == 0 && prod.tile < P.ntiles) {
      issue_pass(a, prod.T, prod.pass, stage, &bars[st], policy);
      cursor_next<CMAX, MODE>(a, P, prod);
      ++issued;
    }

    const bool tile_done = (p + 1 == cons.npass);
    if (tile_done && MODE != kModePartials) {
      const int rows = T.rows;
      for (int task = tid; task < rows * T.ncols; task += kThreads) {
        const int c = task / rows;
        const int r = task - c * rows;
        s_yrow[c][r] = acc[r * CMAX + c] + (s_rrow[c] ? s_rrow[c][r] : 0.0f);
      }
      __syncthreads();
    }
    cursor_next<CMAX, MODE>(a, P, cons);
  }
  // After an abort, let copies still in flight land (bounded) before the
  // CTA's shared memory is released.
  if (tid == 0) {
    for (uint32_t j = q; j < issued; ++j) (void)mbar_wait(&bars[j % kStages], (j / kStages) & 1u);
  }
}

// ----------------------------------------------------------------- host ---
template <int CMAX, int MODE, int FMT>
static size_t smem_bytes(int cc, int nb, int rt) {
  size_t b = static_cast<size_t>(kStages) * stage_bytes(fmt_block_bytes<FMT>());
  b += static_cast<size_t>(cc) * nb * kRecWords * 4;
  b += static_cast<size_t>(kPassUnits) * cc * 4;
  b += static_cast<size_t>(rt) * CMAX * 4 + 4;
  b = (b + 7) & ~static_cast<size_t>(7);
  b += kStages * 8;
  return b;
}

template <int CMAX, int MODE, int FMT>
static int launch_rung(const MmvArgs& args0, int grid, cudaStream_t s) {
  MmvArgs a = args0;
  a.bb = fmt_block_bytes<FMT>();
  const size_t bytes = smem_bytes<CMAX, MODE, FMT>(a.cc, a.nb, a.rt);
  const DeviceInfo& di = device_info();
  if (bytes > di.max_smem_optin) return TQ1_ERR_UNSUPPORTED;
  // Allow the device's full opt-in shared memory (less the kernel's static
  // shared memory) once per device.
  static std::atomic<size_t> max_dyn[64];  // per device; 0 until configured (threads may race to configure: idempotent)
  if (di.device < 0 || di.device >= 64) return TQ1_ERR_CUDA;
  if (max_dyn[di.device].load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, mmv_kernel<CMAX, MODE, FMT>))) return TQ1_ERR_CUDA;
    const size_t lim = di.max_smem_optin - fa.sharedSizeBytes;
    if (!cuda_ok(cudaFuncSetAttribute(mmv_kernel<CMAX, MODE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(lim))))
      return TQ1_ERR_CUDA;
    max_dyn[di.device].store(lim, std::memory_order_release);
  }
  if (bytes > max_dyn[di.device].load(std::memory_order_acquire)) return TQ1_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, mmv_kernel<CMAX, MODE, FMT>, a)) ? TQ1_OK : TQ1_ERR_CUDA;
}

template <int MODE, int FMT>
static int dispatch_rung(int rung, const MmvArgs& a, int grid, cudaStream_t s) {
  switch (rung) {
    case 1: return launch_rung<1, MODE, FMT>(a, grid, s);
    case 2: return launch_rung<2, MODE, FMT>(a, grid, s);
    case 4: return launch_rung<4, MODE, FMT>(a, grid, s);
    case 8: return launch_rung<8, MODE, FMT>(a, grid, s);
    case 16: return launch_rung<16, MODE, FMT>(a, grid, s);
    default: return launch_rung<32, MODE, FMT>(a, grid, s);
  }
}

static int rung_for(int64_t t) {
  int r = 1;
  while (r < t) r *= 2;
  return r;
}

int launch_mmv(const uint8_t* w, const uint8_t* q8, float* y, int32_t* part, int64_t n, int64_t k, int64_t t,
               cudaStream_t s, unsigned* status, const float* res, int fmt) {
  const DeviceInfo& di = device_info();
  MmvArgs a = {};
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.res = res;
  a.part = part;
  a.status = status;
  a.n = n;
  a.k = k;
  a.t = t;
  a.nb = static_cast<int>(k / kQK);
  const size_t rec_col = static_cast<size_t>(a.nb) * kRecWords * 4;
  const int64_t cc = std::min<int64_t>(t, static_cast<int64_t>(kActBudget / rec_col));
  if (cc < 1) return TQ1_ERR_UNSUPPORTED;
  a.cc = static_cast<int>(cc);
  const int rung = rung_for(t);
  // One CTA per SM (or fewer for small problems: at least 64 units each).
  const int64_t units = n * a.nb;
  int64_t grid = std::min<int64_t>(di.num_sms, std::max<int64_t>(1, (units + 63) / 64));
  grid = std::min<int64_t>(grid, n);
  const int64_t rows_per_cta = (n + grid - 1) / grid;
  const int64_t rt_cap = std::max<int64_t>(1, static_cast<int64_t>(kAccBudget / (4 * rung)));
  a.rt = static_cast<int>(std::min<int64_t>(rows_per_cta, rt_cap));
  if (fmt == kFmtTq2)
    return part ? dispatch_rung<kModePartials, kFmtTq2>(rung, a, static_cast<int>(grid), s)
                : dispatch_rung<kModeY, kFmtTq2>(rung, a, static_cast<int>(grid), s);
  if (part) return dispatch_rung<kModePartials, kFmtTq1>(rung, a, static_cast<int>(grid), s);
  return dispatch_rung<kModeY, kFmtTq1>(rung, a, static_cast<int>(grid), s);
}

int launch_mmv_id(const uint8_t* w, int64_t n_experts, const uint8_t* q8, float* y, int64_t n, int64_t k,
                  int64_t t, int64_t top_k, const int32_t* ws, cudaStream_t s, unsigned* status, int act_div,
                  int fmt) {
  const DeviceInfo& di = device_info();
  MmvArgs a = {};
  a.act_div = act_div;
  a.w = w;
  a.q8 = q8;
  a.y = y;
  a.status = status;
  a.n = n;
  a.k = k;
  a.t = t;
  a.nb = static_cast<int>(k / kQK);
  a.top_k = static_cast<int>(top_k);
  a.n_experts = n_experts;
  a.table = ws;
  const size_t rec_col = static_cast<size_t>(a.nb) * kRecWords * 4;
  const int64_t cc = std::min<int64_t>(32, static_cast<int64_t>(kActBudget / rec_col));
  if (cc < 1) return TQ1_ERR_UNSUPPORTED;
  a.cc = static_cast<int>(cc);
  a.rt = static_cast<int>(kAccBudget / (4 * 32));
  return fmt == kFmtTq2 ? launch_rung<32, kModeMoe, kFmtTq2>(a, di.num_sms, s)
                        : launch_rung<32, kModeMoe, kFmtTq1>(a, di.num_sms, s);
}

}  // namespace tq1
