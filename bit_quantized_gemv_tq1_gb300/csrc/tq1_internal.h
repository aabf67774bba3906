// tq1_internal.h -- host-side launchers shared between the library's
// translation units.  Not part of the public C ABI (include/tq1.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tq1 {

struct DeviceInfo {
  int device;
  int num_sms;
  size_t max_smem_optin;
};

// Cached per current device; first call per device queries the runtime.
const DeviceInfo& device_info();

// Record a failed CUDA runtime call for tq1_last_cuda_error(); returns
// err == cudaSuccess.
bool cuda_ok(cudaError_t err);

// Kernel launchers.  All return a TQ1_* status code and never synchronise.
int launch_quantize_rows(const float* w, uint8_t* blocks, int64_t n, int64_t k, cudaStream_t s);
int launch_quantize_rows_tq2(const float* w, uint8_t* blocks, int64_t n, int64_t k, cudaStream_t s);
int launch_quantize_acts(const float* x, uint8_t* q8, int64_t t, int64_t k, cudaStream_t s);

// y[c][r] (y != nullptr) or int32 partials part[c][r][k/32] (part != nullptr)
// for columns c < t <= 32.  `res` (optional, y's layout) is added to y.
// `fmt`: kFmtTq1 (TQ1_0 blocks) or kFmtTq2 (TQ2_0 blocks).
int launch_mmv(const uint8_t* w, const uint8_t* q8, float* y, int32_t* part, int64_t n, int64_t k, int64_t t,
               cudaStream_t s, unsigned* status, const float* res = nullptr, int fmt = 0);

// Decode-path kernel for 1 <= t <= 8 columns.  Returns TQ1_ERR_UNSUPPORTED
// without launching when the shape does not fit its staging.
// With `x` (fp32 activations [t][k]) the kernel quantises them to Q8_1 in its
// prologue and `q8` is unused.
// `inject_timeout` (test hook): CTA 0 issues no copy for its first row group,
// so its waits give up and the call reports a timeout.
// With `part` (int32 [t][n][k/32], y unused) the kernel stores its exact
// per-chunk integer partials instead of the fp32 outputs.
int launch_mmv_small(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, cudaStream_t s,
                     unsigned* status, const float* res = nullptr, const float* x = nullptr, int fmt = 0,
                     int inject_timeout = 0, int32_t* part = nullptr);

// 1 <= t <= 32 columns on the warp-level tensor cores (mma.sync, fp16
// operands exact, fp32 accumulation): y[c][r] (+ res), or the exact int32
// partials part[c][r][k/32] when `part` is given.  Returns TQ1_ERR_UNSUPPORTED
// (launching nothing) when the shape does not fit its shared memory.
int launch_mmv_mma(const uint8_t* w, const uint8_t* q8, float* y, int32_t* part, int64_t n, int64_t k, int64_t t,
                   cudaStream_t s, unsigned* status, const float* res = nullptr, int fmt = 0);

// Expert-routed mat-vec over a compacted routing table in `ws` (general
// dp4a kernel).
// `act_div`: the activation row of routed pair p is p / act_div (top_k: one
// row per token shared by its slots; 1: one row per (token, slot)).
int launch_mmv_id(const uint8_t* w, int64_t n_experts, const uint8_t* q8, float* y, int64_t n, int64_t k,
                  int64_t t, int64_t top_k, const int32_t* ws, cudaStream_t s, unsigned* status, int act_div,
                  int fmt = 0);

// y[c][r] for any t on the tensor cores (tcgen05): 128-row tiles, split-K
// over a thread-block cluster when the tiles alone cannot fill the GPU.
// `fmt`: kFmtTq1 or kFmtTq2 weight blocks.  `ws` (caller-owned device memory
// of at least tile_workspace_bytes(n, k, t, fmt) bytes) holds the exact fp16
// hi/lo split of the activations between the prep and tile kernels
// (TQ1_ERR_WORKSPACE when absent or too small).  Returns TQ1_ERR_UNSUPPORTED
// (launching nothing) for shapes the weight tensor map cannot describe.
int launch_tile(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t t, cudaStream_t s,
                unsigned* status, const float* res, int fmt, void* ws, size_t ws_bytes);
// Scratch bytes of launch_tile for this shape; 0 when the tile path cannot
// run it (row stride not a multiple of 16 bytes, or sizes out of range).
size_t tile_workspace_bytes(int64_t n, int64_t k, int64_t t, int fmt);

// Rows of TQ1_0 (fmt kFmtTq1) or TQ2_0 blocks to fp32 (f16 = false) or fp16
// values: out row i is source row row_ids[i] (row_ids == nullptr: row i).
int launch_dequant(const uint8_t* blocks, const int32_t* row_ids, int64_t n_out, void* out, int64_t n, int64_t k,
                   bool f16, cudaStream_t s, unsigned* status, int fmt = 0);

// Workspace layout of the routing table (int32 words):
//   [0]                   n_active
//   [1, 1+E+1)            expert bounds (exclusive prefix sum of counts)
//   [E+2, E+2+E)          active expert ids, ascending
//   [2E+2, 2E+2+P)        pair indices (token*top_k + slot) sorted by expert,
//                         stable within an expert
//   [2E+2+P, 3E+3+P)      task offsets of the active experts (exclusive
//                         prefix sum of ceil(count / chunk) * row_blocks;
//                         entry n_active holds the total)
inline size_t moe_ws_words(int64_t n_experts, int64_t pairs) {
  return 1 + (size_t)(n_experts + 1) + n_experts + pairs + (n_experts + 1);
}

// Routing-table compaction; `chunk` (pairs per task) and `row_blocks`
// (row ranges per expert) define the task offsets of the expert-routed
// decode kernel.
int launch_moe_compact(const int32_t* ids, int64_t t, int64_t top_k, int64_t n_experts, int chunk, int row_blocks,
                       int32_t* ws, cudaStream_t s, unsigned* status);

// Expert-routed decode kernel over the compacted table.  Returns
// TQ1_ERR_UNSUPPORTED (launching nothing) when the shape does not fit its
// staging; `plan` gives the chunk and row-block counts the compaction needs.
struct MoePlan {
  int chunk, rows, row_blocks;
};
bool moe_small_plan(int64_t n, int64_t k, int64_t pairs, int64_t n_experts, MoePlan* plan, int fmt = 0);

// Expert-routed mat-vec without a routing table, for few pairs: one CTA per
// (pair, row range) reads its expert id itself.  `plan` gives the rows per
// CTA and the row ranges per pair.
bool moe_direct_plan(int64_t n, int64_t k, int64_t pairs, MoePlan* plan, int fmt = 0);
// With `part` (int32 [pairs][n][k/32], y unused) both kernels store their
// exact per-chunk integer partials instead of the fp32 outputs.
int launch_moe_direct(const uint8_t* w, const uint8_t* q8, const int32_t* ids, float* y, int64_t n, int64_t k,
                      int64_t top_k, int64_t n_experts, int64_t pairs, const MoePlan& plan, cudaStream_t s,
                      unsigned* status, int act_div, int fmt = 0, int32_t* part = nullptr);
// With `ids` (and `ws` unused) every CTA builds the routing table itself in
// shared memory (moe_table_smem bytes; for few pairs and experts: at most
// kMoeTableSmemMax), so no compaction kernel runs before it.
int launch_moe_small(const uint8_t* w, const uint8_t* q8, float* y, int64_t n, int64_t k, int64_t top_k,
                     int64_t n_experts, int64_t pairs, const MoePlan& plan, const int32_t* ws, cudaStream_t s,
                     unsigned* status, int act_div, int fmt = 0, int32_t* part = nullptr,
                     const int32_t* ids = nullptr);
inline size_t moe_table_smem(int64_t n_experts, int64_t pairs) {
  return static_cast<size_t>(4 * n_experts + 2 + pairs) * sizeof(int32_t);
}
constexpr size_t kMoeTableSmemMax = 16 * 1024;

}  // namespace tq1
