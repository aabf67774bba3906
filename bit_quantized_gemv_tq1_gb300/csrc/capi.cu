// capi.cu -- the extern "C" entry points of libtq1 (declared in include/tq1.h):
// host-side argument checks, rung/route selection and launches.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

// Device status word of this library (see tq1_sync_status).  Kernels get its
// address as an argument.
static __device__ unsigned int g_tq1_status;

namespace tq1 {

namespace {
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxK = 62720;  // activation records of one column must fit the staging budget
// The mat-vec ladder (tq1_mmv and its variants), from the crossovers measured
// on GB300 at N=5120, K=6144 (us per call in a chain of dependent calls):
//   t <  kMmaMinT:   the dp4a decode kernel, rungs of 1/2/4/8 columns (its
//                    cost grows ~1.1-1.5 us per column: 9.4 us at t = 5,
//                    10.5 at 6, 11.7 at 7)
//   t >= kMmaMinT:   the warp-level tensor-core kernel, rungs of 8/16/24/32
//                    columns (~9.9 us for any t <= 8, 13.2 at 9-16, 19.6 at
//                    32), in slices of 32 columns above 32
//   t >= kTileMinT with a caller workspace (tq1_mmv_ws): the tcgen05 tile
//                    path (prefill)
// Shapes a kernel cannot stage fall through to the general dp4a kernel.
#ifndef TQ1_MMA_MIN_T
#define TQ1_MMA_MIN_T 6
#endif
#ifndef TQ1_TILE_MIN_T
#define TQ1_TILE_MIN_T 33
#endif
constexpr int64_t kMmaMinT = TQ1_MMA_MIN_T;
constexpr int64_t kTileMinT = TQ1_TILE_MIN_T;
// Routed pairs up to which tq1_mmv_id skips the routing table (each pair's
// rows are then read once per pair, not once per distinct expert; pairs of
// one expert read them at about the same time, mostly from L2).  Measured on
// 128 experts of 768 x 2048, Zipf top-8, direct against compacted mode (us,
// single graph replays): 40 pairs 8.9 / 13.1, 64 pairs 14.9 / 16.4, 128
// pairs 24.7 / 25.2, 256 pairs 44.6 / 36.8, 512 pairs 81.9 / 57.4.
constexpr int64_t kMoeDirectMaxPairs = 128;
std::mutex g_mu;
std::atomic<int> g_inject_timeout{0};  // one-shot test hook (tq1_debug_inject_wait_timeout)
DeviceInfo g_info[kMaxDevices];
unsigned* g_status_ptr[kMaxDevices];
std::atomic<bool> g_have[kMaxDevices];  // set (release) once g_info / g_status_ptr hold the device

thread_local char g_last_err[256] = "";

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int current_device() {
  int d = 0;
  if (!cuda_ok(cudaGetDevice(&d)) || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

bool ensure_device(int d) {
  if (g_have[d].load(std::memory_order_acquire)) return true;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_have[d].load(std::memory_order_relaxed)) return true;
  DeviceInfo di{};
  di.device = d;
  int v = 0;
  if (!cuda_ok(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d))) return false;
  di.num_sms = v;
  if (!cuda_ok(cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d))) return false;
  di.max_smem_optin = static_cast<size_t>(v);
  void* p = nullptr;
  if (!cuda_ok(cudaGetSymbolAddress(&p, g_tq1_status))) return false;
  g_info[d] = di;
  g_status_ptr[d] = static_cast<unsigned*>(p);
  g_have[d].store(true, std::memory_order_release);
  return true;
}

unsigned* status_ptr() {
  const int d = current_device();
  if (d < 0 || !ensure_device(d)) return nullptr;
  return g_status_ptr[d];
}

int check_mmv_shape(int64_t n, int64_t k, int64_t t) {
  if (n < 0 || t < 0 || k <= 0 || (k % kQK) != 0) return TQ1_ERR_SHAPE;
  return TQ1_OK;
}
}  // namespace

bool cuda_ok(cudaError_t err) {
  if (err == cudaSuccess) return true;
  snprintf(g_last_err, sizeof(g_last_err), "%s: %s", cudaGetErrorName(err), cudaGetErrorString(err));
  return false;
}

const DeviceInfo& device_info() {
  static DeviceInfo dummy{};
  const int d = current_device();
  if (d < 0 || !ensure_device(d)) return dummy;
  return g_info[d];
}

}  // namespace tq1

using namespace tq1;

extern "C" {

const char* tq1_status_string(int status) {
  switch (status) {
    case TQ1_OK: return "ok";
    case TQ1_ERR_NULL: return "null pointer argument";
    case TQ1_ERR_SHAPE: return "invalid shape (k must be a positive multiple of 256; n, t, top_k >= 0)";
    case TQ1_ERR_ALIGN: return "pointer not 16-byte aligned";
    case TQ1_ERR_UNSUPPORTED: return "shape beyond the kernels' limits";
    case TQ1_ERR_WORKSPACE: return "workspace too small";
    case TQ1_ERR_CUDA: return "CUDA runtime error";
    case TQ1_ERR_TIMEOUT: return "a kernel timed out waiting for a transfer";
    case TQ1_ERR_BAD_ID: return "routing id outside [0, n_experts)";
    default: return "unknown status";
  }
}

const char* tq1_version(void) { return "0.1.0"; }

void tq1_debug_inject_wait_timeout(void) { g_inject_timeout.store(1); }

const char* tq1_last_cuda_error(void) { return g_last_err; }

size_t tq1_blocks_bytes(int64_t n, int64_t k) {
  if (n < 0 || k < 0) return 0;
  return static_cast<size_t>(n) * static_cast<size_t>(k / kQK) * kBlockBytes;
}

size_t tq2_blocks_bytes(int64_t n, int64_t k) {
  if (n < 0 || k < 0) return 0;
  return static_cast<size_t>(n) * static_cast<size_t>(k / kQK) * kTq2BlockBytes;
}

size_t tq1_q8_1_bytes(int64_t t, int64_t k) {
  if (t < 0 || k < 0) return 0;
  return static_cast<size_t>(t) * static_cast<size_t>(k / kQK8) * kQ8Bytes;
}

static int quantize_rows_common(const float* w, void* blocks, int64_t n, int64_t k, void* stream, int fmt) {
  if (n < 0 || k <= 0 || (k % kQK) != 0) return TQ1_ERR_SHAPE;
  if (n == 0) return TQ1_OK;
  if (!w || !blocks) return TQ1_ERR_NULL;
  if (misaligned(w) || misaligned(blocks)) return TQ1_ERR_ALIGN;
  if (!status_ptr()) return TQ1_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return fmt == kFmtTq2 ? launch_quantize_rows_tq2(w, static_cast<uint8_t*>(blocks), n, k, s)
                        : launch_quantize_rows(w, static_cast<uint8_t*>(blocks), n, k, s);
}

int tq1_quantize_rows(const float* w, void* blocks, int64_t n, int64_t k, void* stream) {
  return quantize_rows_common(w, blocks, n, k, stream, kFmtTq1);
}

int tq2_quantize_rows(const float* w, void* blocks, int64_t n, int64_t k, void* stream) {
  return quantize_rows_common(w, blocks, n, k, stream, kFmtTq2);
}

int q8_1_quantize_acts(const float* x, void* q8, int64_t t, int64_t k, void* stream) {
  if (t < 0 || k <= 0 || (k % kQK8) != 0) return TQ1_ERR_SHAPE;
  if (t == 0) return TQ1_OK;
  if (!x || !q8) return TQ1_ERR_NULL;
  if (misaligned(x) || misaligned(q8)) return TQ1_ERR_ALIGN;
  if (!status_ptr()) return TQ1_ERR_CUDA;
  return launch_quantize_acts(x, static_cast<uint8_t*>(q8), t, k, static_cast<cudaStream_t>(stream));
}

// Workspace bytes the tile path needs for this call (0: the call runs the
// allocation-free kernels).
static size_t mmv_ws_bytes(int64_t n, int64_t k, int64_t t, int fmt) {
  if (n < 1 || t < kTileMinT || k <= 0 || (k % kQK) != 0 || k > kMaxK) return 0;
  return tile_workspace_bytes(n, k, t, fmt);
}

static int mmv_common(const void* blocks, const void* q8, float* y, int32_t* part, int64_t n, int64_t k,
                      int64_t t, void* stream, const float* res = nullptr, int fmt = kFmtTq1, void* ws = nullptr,
                      size_t ws_bytes = 0) {
  int rc = check_mmv_shape(n, k, t);
  if (rc != TQ1_OK) return rc;
  if (n == 0 || t == 0) return TQ1_OK;
  if (!blocks || !q8 || (!y && !part)) return TQ1_ERR_NULL;
  if (misaligned(blocks) || misaligned(q8) || (y && misaligned(y)) || (part && misaligned(part)) ||
      (res && misaligned(res)) || (ws && misaligned(ws)))
    return TQ1_ERR_ALIGN;
  const size_t need_ws = y && ws ? mmv_ws_bytes(n, k, t, fmt) : 0;
  if (need_ws && ws_bytes < need_ws) return TQ1_ERR_WORKSPACE;
  if (k > kMaxK) return TQ1_ERR_UNSUPPORTED;
  unsigned* st = status_ptr();
  if (!st) return TQ1_ERR_CUDA;
  // The test hook is consumed by this call whichever kernel runs; only the
  // decode kernel acts on it.
  const int inject = g_inject_timeout.exchange(0);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* w = static_cast<const uint8_t*>(blocks);
  const uint8_t* a = static_cast<const uint8_t*>(q8);
  const int64_t q8_row = (k / kQK8) * kQ8Bytes;
  if (need_ws) {
    rc = launch_tile(w, a, y, n, k, t, s, st, res, fmt, ws, ws_bytes);
    if (rc != TQ1_ERR_UNSUPPORTED) return rc;  // otherwise the kernels below
  }
  if (t < kMmaMinT && t <= 8) {
    // The decode kernel: fp32 outputs, or (debug entry) its exact partials.
    rc = launch_mmv_small(w, a, y, n, k, t, s, st, res, nullptr, fmt, y ? inject : 0, y ? nullptr : part);
    if (rc != TQ1_ERR_UNSUPPORTED) return rc;  // otherwise the general kernel below
  } else {
    // The warp-level tensor-core rungs, 32 columns at a time: fp32 outputs or
    // (debug entry) their exact partials.
    bool all = true;
    for (int64_t c0 = 0; c0 < t && all; c0 += 32) {
      const int64_t tc = t - c0 < 32 ? t - c0 : 32;
      rc = launch_mmv_mma(w, a + c0 * q8_row, y ? y + c0 * n : nullptr, part ? part + c0 * n * (k / kQK8) : nullptr,
                          n, k, tc, s, st, res ? res + c0 * n : nullptr, fmt);
      if (rc == TQ1_ERR_UNSUPPORTED && c0 == 0) all = false;  // shape too large: the general kernel below
      else if (rc != TQ1_OK) return rc;
    }
    if (all) return TQ1_OK;
  }
  for (int64_t c0 = 0; c0 < t; c0 += 32) {
    const int64_t tc = t - c0 < 32 ? t - c0 : 32;
    rc = launch_mmv(w, a + c0 * q8_row, y ? y + c0 * n : nullptr, part ? part + c0 * n * (k / kQK8) : nullptr, n,
                    k, tc, s, st, res ? res + c0 * n : nullptr, fmt);
    if (rc != TQ1_OK) return rc;
  }
  return TQ1_OK;
}

int tq1_mmv(const void* blocks, const void* q8, float* y, int64_t n, int64_t k, int64_t t, void* stream) {
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream);
}

int tq2_mmv(const void* blocks, const void* q8, float* y, int64_t n, int64_t k, int64_t t, void* stream) {
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream, nullptr, kFmtTq2);
}

int tq2_mmv_partials(const void* blocks, const void* q8, int32_t* part, int64_t n, int64_t k, int64_t t,
                     void* stream) {
  if (!part && n > 0 && t > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_common(blocks, q8, nullptr, part, n, k, t, stream, nullptr, kFmtTq2);
}

static int mmv_f32_common(const void* blocks, const float* x, float* y, int64_t n, int64_t k, int64_t t,
                          void* stream, int fmt) {
  int rc = check_mmv_shape(n, k, t);
  if (rc != TQ1_OK) return rc;
  if (n == 0 || t == 0) return TQ1_OK;
  if (!blocks || !x || !y) return TQ1_ERR_NULL;
  if (misaligned(blocks) || misaligned(x) || misaligned(y)) return TQ1_ERR_ALIGN;
  if (t > 4 || k > kMaxK) return TQ1_ERR_UNSUPPORTED;
  unsigned* st = status_ptr();
  if (!st) return TQ1_ERR_CUDA;
  return launch_mmv_small(static_cast<const uint8_t*>(blocks), nullptr, y, n, k, t, static_cast<cudaStream_t>(stream),
                          st, nullptr, x, fmt);
}

int tq1_mmv_f32(const void* blocks, const float* x, float* y, int64_t n, int64_t k, int64_t t, void* stream) {
  return mmv_f32_common(blocks, x, y, n, k, t, stream, kFmtTq1);
}

int tq2_mmv_f32(const void* blocks, const float* x, float* y, int64_t n, int64_t k, int64_t t, void* stream) {
  return mmv_f32_common(blocks, x, y, n, k, t, stream, kFmtTq2);
}

int tq1_mmv_add(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
                void* stream) {
  if (!res && n > 0 && t > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream, res);
}

int tq2_mmv_add(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
                void* stream) {
  if (!res && n > 0 && t > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream, res, kFmtTq2);
}

size_t tq1_mmv_workspace_size(int64_t n, int64_t k, int64_t t) {
  // The tile path's scratch does not depend on the weight format, nor does
  // whether it runs (both formats' row strides are multiples of 16 bytes for
  // the same k).
  return mmv_ws_bytes(n, k, t, kFmtTq1);
}

int tq1_mmv_ws(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
               void* ws, size_t ws_bytes, void* stream) {
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream, res, kFmtTq1, ws, ws_bytes);
}

int tq2_mmv_ws(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
               void* ws, size_t ws_bytes, void* stream) {
  return mmv_common(blocks, q8, y, nullptr, n, k, t, stream, res, kFmtTq2, ws, ws_bytes);
}

int tq1_mmv_partials(const void* blocks, const void* q8, int32_t* part, int64_t n, int64_t k, int64_t t,
                     void* stream) {
  if (!part && n > 0 && t > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_common(blocks, q8, nullptr, part, n, k, t, stream);
}

static int dequant_common(const void* blocks, const int32_t* row_ids, int64_t n_ids, void* out, int64_t n,
                          int64_t k, int out_f16, void* stream, int fmt) {
  if (n < 0 || n_ids < 0 || k <= 0 || (k % kQK) != 0) return TQ1_ERR_SHAPE;
  if (n_ids == 0) return TQ1_OK;
  if (!blocks || !out || (row_ids == nullptr && n_ids != n)) return TQ1_ERR_NULL;
  if (misaligned(blocks) || misaligned(out) || (row_ids && misaligned(row_ids))) return TQ1_ERR_ALIGN;
  if (n_ids > (int64_t{1} << 40) / k) return TQ1_ERR_UNSUPPORTED;
  unsigned* st = status_ptr();
  if (!st) return TQ1_ERR_CUDA;
  return launch_dequant(static_cast<const uint8_t*>(blocks), row_ids, n_ids, out, n, k, out_f16 != 0,
                        static_cast<cudaStream_t>(stream), st, fmt);
}

int tq1_dequantize_rows(const void* blocks, void* out, int64_t n, int64_t k, int out_f16, void* stream) {
  if (n < 0) return TQ1_ERR_SHAPE;
  return dequant_common(blocks, nullptr, n, out, n, k, out_f16, stream, kFmtTq1);
}

int tq1_get_rows(const void* blocks, const int32_t* row_ids, int64_t n_ids, void* out, int64_t n, int64_t k,
                 int out_f16, void* stream) {
  if (!row_ids && n_ids > 0 && n >= 0 && k > 0 && (k % kQK) == 0) return TQ1_ERR_NULL;
  return dequant_common(blocks, row_ids, n_ids, out, n, k, out_f16, stream, kFmtTq1);
}

int tq2_dequantize_rows(const void* blocks, void* out, int64_t n, int64_t k, int out_f16, void* stream) {
  if (n < 0) return TQ1_ERR_SHAPE;
  return dequant_common(blocks, nullptr, n, out, n, k, out_f16, stream, kFmtTq2);
}

int tq2_get_rows(const void* blocks, const int32_t* row_ids, int64_t n_ids, void* out, int64_t n, int64_t k,
                 int out_f16, void* stream) {
  if (!row_ids && n_ids > 0 && n >= 0 && k > 0 && (k % kQK) == 0) return TQ1_ERR_NULL;
  return dequant_common(blocks, row_ids, n_ids, out, n, k, out_f16, stream, kFmtTq2);
}

size_t tq1_mmv_id_workspace_size(int64_t n_experts, int64_t t, int64_t top_k) {
  if (n_experts < 0 || t < 0 || top_k < 0) return 0;
  const size_t words = moe_ws_words(n_experts, t * top_k);
  return (words * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

}  // extern "C"

static int mmv_id_common(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                         int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream,
                         bool per_slot, int fmt = kFmtTq1, int32_t* part = nullptr) {
  int rc = check_mmv_shape(n, k, t);
  if (rc != TQ1_OK) return rc;
  if (n_experts <= 0 || top_k < 0) return TQ1_ERR_SHAPE;
  if (n == 0 || t == 0 || top_k == 0) return TQ1_OK;
  if (!expert_blocks || !q8 || !ids || (!y && !part) || !ws) return TQ1_ERR_NULL;
  if (misaligned(expert_blocks) || misaligned(q8) || misaligned(ids) || (y && misaligned(y)) ||
      (part && misaligned(part)) || misaligned(ws))
    return TQ1_ERR_ALIGN;
  if (ws_bytes < tq1_mmv_id_workspace_size(n_experts, t, top_k)) return TQ1_ERR_WORKSPACE;
  if (k > kMaxK || n_experts > 12288 || t * top_k > (int64_t{1} << 30)) return TQ1_ERR_UNSUPPORTED;
  unsigned* st = status_ptr();
  if (!st) return TQ1_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* table = static_cast<int32_t*>(ws);
  const uint8_t* w = static_cast<const uint8_t*>(expert_blocks);
  const uint8_t* a = static_cast<const uint8_t*>(q8);
  const int act_div = per_slot ? 1 : static_cast<int>(top_k);
  MoePlan plan{};
  // A few pairs (decode): no routing table, each CTA reads its pair's id.
  if (t * top_k <= kMoeDirectMaxPairs && moe_direct_plan(n, k, t * top_k, &plan, fmt))
    return launch_moe_direct(w, a, ids, y, n, k, top_k, n_experts, t * top_k, plan, s, st, act_div, fmt, part);
  const bool small = moe_small_plan(n, k, t * top_k, n_experts, &plan, fmt);
  if (part && !small) return TQ1_ERR_UNSUPPORTED;  // partials come from the routed decode kernels only
  if (small && moe_table_smem(n_experts, t * top_k) <= kMoeTableSmemMax) {
    // Few pairs: the routed decode kernel builds the routing table itself.
    rc = launch_moe_small(w, a, y, n, k, top_k, n_experts, t * top_k, plan, nullptr, s, st, act_div, fmt, part, ids);
    if (rc != TQ1_ERR_UNSUPPORTED || part) return rc;
  }
  rc = launch_moe_compact(ids, t, top_k, n_experts, small ? plan.chunk : 1, small ? plan.row_blocks : 1, table, s,
                          st);
  if (rc != TQ1_OK) return rc;
  if (small) {
    rc = launch_moe_small(w, a, y, n, k, top_k, n_experts, t * top_k, plan, table, s, st, act_div, fmt, part);
    if (rc != TQ1_ERR_UNSUPPORTED || part) return rc;  // otherwise the general kernel below
  }
  return launch_mmv_id(w, n_experts, a, y, n, k, t, top_k, table, s, st, act_div, fmt);
}

extern "C" {

int tq1_mmv_id(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
               int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream) {
  return mmv_id_common(expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, ws, ws_bytes, stream, false);
}

int tq1_mmv_id_slots(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                     int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream) {
  return mmv_id_common(expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, ws, ws_bytes, stream, true);
}

int tq2_mmv_id(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
               int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream) {
  return mmv_id_common(expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, ws, ws_bytes, stream, false, kFmtTq2);
}

int tq2_mmv_id_slots(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                     int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream) {
  return mmv_id_common(expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, ws, ws_bytes, stream, true, kFmtTq2);
}

int tq1_mmv_id_partials(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids,
                        int32_t* part, int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!part && n > 0 && t > 0 && top_k > 0 && n_experts > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_id_common(expert_blocks, n_experts, q8, ids, nullptr, n, k, t, top_k, ws, ws_bytes, stream, false,
                       kFmtTq1, part);
}

int tq2_mmv_id_partials(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids,
                        int32_t* part, int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!part && n > 0 && t > 0 && top_k > 0 && n_experts > 0 && check_mmv_shape(n, k, t) == TQ1_OK) return TQ1_ERR_NULL;
  return mmv_id_common(expert_blocks, n_experts, q8, ids, nullptr, n, k, t, top_k, ws, ws_bytes, stream, false,
                       kFmtTq2, part);
}

int tq1_sync_status(void* stream) {
  unsigned* st = status_ptr();
  if (!st) return TQ1_ERR_CUDA;
  if (!cuda_ok(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)))) return TQ1_ERR_CUDA;
  unsigned v = 0;
  if (!cuda_ok(cudaMemcpy(&v, st, sizeof(v), cudaMemcpyDeviceToHost))) return TQ1_ERR_CUDA;
  const unsigned zero = 0;
  if (!cuda_ok(cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice))) return TQ1_ERR_CUDA;
  if (v & kStatusTimeout) return TQ1_ERR_TIMEOUT;
  if (v & kStatusBadId) return TQ1_ERR_BAD_ID;
  return TQ1_OK;
}

}  // extern "C"
