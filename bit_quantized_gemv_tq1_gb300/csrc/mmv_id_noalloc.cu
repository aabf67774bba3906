// mmv_id_noalloc.cu -- tq1_mmv_id_noalloc: the expert-routed mat-vec for
// callers that cannot allocate device memory.
//
// tq1_mmv_id needs a small device workspace for its routing table (expert
// bounds, active-expert list, token/slot pairs sorted by expert).  Some callers
// cannot provide one: code that runs inside a stream capture (cudaMalloc is not
// allowed there), engines that hand a kernel library a fixed memory budget and
// forbid device allocation after start-up, latency-critical loops where an
// allocation could block on the allocator or synchronise the device, and plain
// C / foreign-language callers that have no caching allocator to borrow a
// buffer from.  For them this entry point keeps the routing table in a
// fixed-size array that is part of the library image.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (about 76 KiB) until the process exits.  Its device address
// is looked up once per device, with that device current, on the first call;
// that first call should therefore be made before any stream capture begins.
// All calls on a device share the one array and it keeps the previous call's
// contents; the routing kernel rewrites every word it reads, so nothing has to
// be cleared between calls.  Calls whose kernels may overlap on the GPU (on
// different streams without ordering between them) race on the array and must
// not be issued.
#include <atomic>
#include <mutex>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace {

constexpr int64_t kMaxExperts = 1024;
constexpr int64_t kMaxPairs = 16384;  // tokens * top_k
// Routing-table words for the largest accepted call, rounded up to whole
// 256-byte units (the size tq1_mmv_id asks of its workspace).
constexpr size_t kWords =
    (1 + static_cast<size_t>(kMaxExperts + 1) + kMaxExperts + kMaxPairs + (kMaxExperts + 1) + 63) & ~size_t(63);
constexpr int kMaxDevices = 64;

std::mutex g_mu;
std::atomic<int32_t*> g_table[kMaxDevices];  // published (release) once looked up

}  // namespace

static __device__ __align__(256) int32_t g_route_table[kWords];

// Device address of g_route_table on the current device (looked up once per
// device, under a lock; later calls read the published address without it),
// or nullptr if the runtime call failed.
static int32_t* route_table_address() {
  int dev = 0;
  if (!tq1::cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= kMaxDevices) return nullptr;
  int32_t* known = g_table[dev].load(std::memory_order_acquire);
  if (known != nullptr) return known;
  std::lock_guard<std::mutex> lock(g_mu);
  known = g_table[dev].load(std::memory_order_relaxed);
  if (known == nullptr) {
    void* p = nullptr;
    if (!tq1::cuda_ok(cudaGetSymbolAddress(&p, g_route_table))) return nullptr;
    known = static_cast<int32_t*>(p);
    g_table[dev].store(known, std::memory_order_release);
  }
  return known;
}

extern "C" int tq1_mmv_id_noalloc(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids,
                                  float* y, int64_t n, int64_t k, int64_t t, int64_t top_k, void* stream) {
  if (n < 0 || t < 0 || top_k < 0 || k <= 0 || (k % tq1::kQK) != 0 || n_experts <= 0) return TQ1_ERR_SHAPE;
  if (n == 0 || t == 0 || top_k == 0) return TQ1_OK;
  if (n_experts > kMaxExperts || t > kMaxPairs || top_k > kMaxPairs || t * top_k > kMaxPairs) return TQ1_ERR_WORKSPACE;
  int32_t* table = route_table_address();
  if (table == nullptr) return TQ1_ERR_CUDA;
  return tq1_mmv_id(expert_blocks, n_experts, q8, ids, y, n, k, t, top_k, table, kWords * sizeof(int32_t), stream);
}
