// moe.cu -- routing-table compaction for the expert-routed mat-vec.
//
// The MoE path (AMD-Ecosystem/llama.cpp PR #76, "Summary": ids tensor ->
// expert_bounds -> a grid over the compacted list) turns per-token expert ids
// into: per-expert bounds (exclusive prefix sum of the routed counts), the
// ascending list of experts that received at least one token, the (token,
// slot) pairs sorted by expert, stable within an expert, and each active
// expert's first task (an expert's pairs in chunks, times its row blocks).
// The mat-vec kernels then walk only the active experts.
#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

constexpr int kCompactThreads = 1024;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __launch_bounds__(kCompactThreads) moe_compact_kernel(const int32_t* __restrict__ ids, int64_t pairs,
                                                                       int n_experts, int chunk, int row_blocks,
                                                                       int32_t* __restrict__ ws, unsigned* status) {
  extern __shared__ int s_cnt[];  // n_experts counters, reused as scatter cursors
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* bounds = ws + 1;
  int32_t* active = ws + 1 + (n_experts + 1);
  int32_t* plist = active + n_experts;
  int32_t* tasks = plist + pairs;

  for (int i = tid; i < n_experts; i += kCompactThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int64_t p = tid; p < pairs; p += kCompactThreads) {
    const int e = ids[p];
    if (e >= 0 && e < n_experts) atomicAdd(&s_cnt[e], 1);
    else raise_status(status, kStatusBadId);
  }
  __syncthreads();

  if (warp == 0) {  // exclusive scans of the counts and the tasks, and the active list
    int running = 0, nact = 0, running_tasks = 0;
    for (int base = 0; base < n_experts; base += 32) {
      const int i = base + lane;
      const int v = i < n_experts ? s_cnt[i] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (i < n_experts) bounds[i] = running + incl - v;
      const uint32_t has = __ballot_sync(0xffffffffu, v > 0);
      // Tasks of an active expert: its pairs in chunks, times the row blocks.
      const int nt = v > 0 ? ((v + chunk - 1) / chunk) * row_blocks : 0;
      int tincl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, tincl, o);
        if (lane >= o) tincl += u;
      }
      if (v > 0) {
        const int slot = nact + __popc(has & lanemask_lt());
        active[slot] = i;
        tasks[slot] = running_tasks + tincl - nt;
      }
      nact += __popc(has);
      running += __shfl_sync(0xffffffffu, incl, 31);
      running_tasks += __shfl_sync(0xffffffffu, tincl, 31);
    }
    if (lane == 0) {
      bounds[n_experts] = running;
      tasks[nact] = running_tasks;
      ws[0] = nact;
    }
  }
  __syncthreads();
  for (int i = tid; i < n_experts; i += kCompactThreads) s_cnt[i] = bounds[i];
  __syncthreads();

  if (warp == 0) {  // stable scatter of pair indices, 32 at a time, in order
    for (int64_t base = 0; base < pairs; base += 32) {
      const int64_t p = base + lane;
      int e = p < pairs ? ids[p] : -1;
      if (e >= n_experts) e = -1;
      if (e < -1) e = -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lanemask_lt());
      if (e >= 0) plist[s_cnt[e] + rank] = static_cast<int32_t>(p);
      __syncwarp();
      if (e >= 0 && rank == 0) s_cnt[e] += __popc(peers);
      __syncwarp();
    }
  }
}

int launch_moe_compact(const int32_t* ids, int64_t t, int64_t top_k, int64_t n_experts, int chunk, int row_blocks,
                       int32_t* ws, cudaStream_t s, unsigned* status) {
  if (chunk < 1 || row_blocks < 1) return TQ1_ERR_UNSUPPORTED;
  const size_t smem = static_cast<size_t>(n_experts) * sizeof(int);
  if (smem > 48 * 1024) return TQ1_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kCompactThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, moe_compact_kernel, ids, t * top_k, static_cast<int>(n_experts),
                                             chunk, row_blocks, ws, status);
  return cuda_ok(err) ? TQ1_OK : TQ1_ERR_CUDA;
}

}  // namespace tq1
