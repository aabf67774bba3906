// dequant.cu -- TQ1_0 rows back to fp32 or fp16 values: whole-matrix
// dequantisation and row gathers (get_rows, e.g. an embedding lookup).
//
// The CPU reference walks a 256-block once and amortises each packed byte
// over its trits (PrismML-Eng/llama.cpp issue #139, "Current behavior"); the
// Vulkan backend of the same format ships dequant and get_rows shaders next
// to its mat-vec ("Upstream state").  Here every warp owns an equal range of
// (output row, 256-block) units, taken in segments of up to eight
// consecutive blocks (for get_rows, never across an output row): a segment's
// bytes (the 16-byte pieces covering them) are copied global -> shared memory
// by asynchronous copies, three segments in flight per warp, so the load
// latency is paid once per three segments rather than once per block.  Each
// lane then produces eight elements of each block as two groups of four:
// elements 8l .. 8l+7 for fp16 rows (one 16-byte store), 4l .. 4l+3 and
// 128+4l .. 128+4l+3 for fp32 rows (two 16-byte stores, each instruction of
// the warp writing 512 contiguous bytes).  A group of four is digit k of four
// consecutive packed bytes (element order of the block: e < 160 -> qs[e % 32]
// digit e/32; e < 240 -> qs[32 + (e-160) % 16] digit (e-160)/16; else
// qh[(e-240) % 4] digit (e-240)/4), expanded with the specification's digit
// formula ((uint8)(b*3^k)*3) >> 8.  The kernel is bound by the output bytes
// written to HBM.
//
// TQ2_0 blocks (2-bit codes, 66 bytes) take the same path: a group of four is
// field (e/32) % 4 of four consecutive bytes qs[32 * (e/128) + e % 32 ..];
// code 3 (never written by the encoder) gives +2d, the fourth entry of the
// value table.
#include <algorithm>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kDqThreads = 256;
constexpr int kDqWarps = kDqThreads / 32;
constexpr int kDqSeg = 8;       // 256-blocks per segment
constexpr int kDqDepth = 3;     // segments whose copies are in flight per warp
// Resident CTAs per SM the grid is sized for: fp32 rows 5, fp16 rows 4
// (measured at N=5120, K=6144: fp32 22.8 -> 21.9 us with 5, fp16 11.3 ->
// 11.7 us).
constexpr int dq_ctas_per_sm(bool f16) { return f16 ? 4 : 5; }
// A slot holds the 16-byte pieces covering one segment (a segment starts at
// an even byte offset, so at most 14 bytes before it share its first piece).
template <int FMT>
__host__ __device__ constexpr int dq_slot_bytes() {
  return (kDqSeg * fmt_block_bytes<FMT>() + 14 + 15) / 16 * 16;
}

// 16 bytes global -> shared, the last 16 - src_bytes of them zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_depth() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kDqDepth - 1) : "memory");
}

// One segment in flight: its first unit (= output row * blocks per row +
// block), how many blocks it writes (0: none, e.g. a bad row id) and where
// its bytes start within the slot.
struct DqSeg {
  int64_t u;
  int nbk;
  int delta;
  bool issued;  // a segment was taken from the range (written or skipped)
};

template <bool F16, int FMT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const uint8_t* __restrict__ blocks,
                                                             const int32_t* __restrict__ row_ids, int64_t n_out,
                                                             void* __restrict__ out, int64_t n, int nb,
                                                             unsigned* status) {
  constexpr int kBB = fmt_block_bytes<FMT>();
  constexpr int kSlot = dq_slot_bytes<FMT>();
  __shared__ __align__(16) uint8_t s_ring[kDqWarps][kDqDepth][kSlot];
  pdl_wait();  // blocks and row ids may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // This warp's units [u_next, u_end): an equal share of all of them.
  const int64_t units = n_out * nb;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kDqWarps;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kDqWarps + warp;
  int64_t u_next = units / nw * w + min(w, units % nw);
  const int64_t u_end = u_next + units / nw + (w < units % nw ? 1 : 0);
  const uint8_t* mat_end = blocks + n * nb * kBB;
  // The lane's eight elements are two groups of four, each digit k (TQ2_0:
  // field k) of four consecutive bytes at offset boff within the block.  The
  // fp16 rows take elements 8l .. 8l+7 (one 16-byte store per lane); the
  // fp32 rows 4l .. 4l+3 and 128+4l .. 128+4l+3, so that each 16-byte store
  // instruction of the warp writes 512 contiguous bytes.  A group of four
  // elements never straddles a chunk of the element order (see above).
  int boff[2], dig[2];
  if (F16) {
    if (FMT == kFmtTq2) {
      boff[0] = 32 * (lane >> 4) + 8 * (lane & 3);
      dig[0] = (lane >> 2) & 3;
    } else if (lane < 20) {
      boff[0] = 8 * (lane & 3);
      dig[0] = lane >> 2;
    } else if (lane < 30) {
      boff[0] = 32 + 8 * ((lane - 20) & 1);
      dig[0] = (lane - 20) >> 1;
    } else {
      boff[0] = 48;  // qh[0..3]
      dig[0] = 2 * (lane - 30);
    }
    const bool qh = FMT != kFmtTq2 && lane >= 30;  // qh[0..3] twice: digits dig and dig + 1
    boff[1] = qh ? boff[0] : boff[0] + 4;
    dig[1] = qh ? dig[0] + 1 : dig[0];
  } else {
    boff[0] = 4 * (lane & 7);  // element group l: chunk l / 8 of the first 128
    dig[0] = lane >> 3;
    if (FMT == kFmtTq2) {  // element group 32 + l: the same field of qs[32 ..]
      boff[1] = 32 + 4 * (lane & 7);
      dig[1] = lane >> 3;
    } else if (lane < 8) {  // elements 128 .. 159: digit 4 of qs[0..31]
      boff[1] = 4 * lane;
      dig[1] = 4;
    } else if (lane < 28) {  // elements 160 .. 239: qs[32..47]
      boff[1] = 32 + 4 * ((lane - 8) & 3);
      dig[1] = (lane - 8) >> 2;
    } else {  // elements 240 .. 255: qh[0..3]
      boff[1] = 48;
      dig[1] = lane - 28;
    }
  }
  // Per group: the multiplier 3^k of the digit formula, or the field's shift.
  uint32_t dmul[2];
#pragma unroll
  for (int g = 0; g < 2; ++g)
    dmul[g] = FMT == kFmtTq2 ? static_cast<uint32_t>(2 * dig[g])
                             : static_cast<uint32_t>((kPow3Packed >> (8 * dig[g])) & 0xFFu);

  // Take the next segment of the range and copy its bytes into `slot`, as
  // one commit group (empty when there is nothing to copy): when segment j
  // is processed, waiting until at most kDqDepth - 1 groups are pending
  // means its own copies have landed.  Warp-uniform.
  auto issue = [&](uint8_t* slot, DqSeg& S) {
    S.nbk = 0;
    S.issued = u_next < u_end;
    if (S.issued) {
      const int64_t u = u_next;
      int len = static_cast<int>(min(static_cast<int64_t>(kDqSeg), u_end - u));
      const uint8_t* src = blocks + u * kBB;
      bool ok = true;
      if (row_ids) {
        // A gathered row's blocks are contiguous only within that row.
        const int64_t i = u / nb;
        const int b = static_cast<int>(u - i * nb);
        len = min(len, nb - b);
        const int64_t srow = __ldg(row_ids + i);
        if (srow < 0 || srow >= n) {
          if (lane == 0 && b == 0) raise_status(status, kStatusBadId);
          ok = false;  // the output row is left untouched
        } else {
          src = blocks + (srow * nb + b) * kBB;
        }
      }
      u_next = u + len;
      if (ok) {
        S.u = u;
        S.nbk = len;
        const uint8_t* a0 = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15));
        S.delta = static_cast<int>(src - a0);
        const int np = (S.delta + len * kBB + 15) >> 4;
        for (int p = lane; p < np; p += 32) {
          const uint8_t* g = a0 + 16 * p;  // holds at least one byte of the segment, so g < mat_end
          const int64_t left = mat_end - g;
          cp_async16(slot + 16 * p, g, left < 16 ? static_cast<uint32_t>(left) : 16u);
        }
      }
    }
    cp_async_commit();
  };

  DqSeg T[kDqDepth];
#pragma unroll
  for (int d = 0; d < kDqDepth; ++d) issue(s_ring[warp][d], T[d]);

  for (bool more = true; more;) {
    more = false;
#pragma unroll
    for (int d = 0; d < kDqDepth; ++d) {
      more = more || T[d].issued;
      cp_async_wait_depth();  // this lane's copies of the segment in slot d have landed
      __syncwarp();           // ... and every other lane's
      const DqSeg& C = T[d];
      const uint8_t* base = s_ring[warp][d] + C.delta;
#pragma unroll 2
      for (int b = 0; b < C.nbk; ++b) {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(base + b * kBB);
        uint32_t dg[8];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint32_t h0 = h[(boff[g] >> 1)], h1 = h[(boff[g] >> 1) + 1];
          const uint32_t by[4] = {h0 & 0xFFu, h0 >> 8, h1 & 0xFFu, h1 >> 8};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dg[4 * g + i] = FMT == kFmtTq2 ? (by[i] >> dmul[g]) & 3u : (((by[i] * dmul[g]) & 0xFFu) * 3u) >> 8;
        }
        const int64_t e0 = (C.u + b) * kQK;  // unit index * 256: output row-major
        const uint32_t h16 = h[(kBB - 2) / 2];
        if (F16) {
          // fp16 values by byte permute from the table {-d, 0, +d, +2d}: a
          // digit pair (a, b) selects bytes 2a, 2a+1, 2b, 2b+1 (selector
          // 34 * (a + 256 b) + 0x1010).  TQ1_0 digits never reach the fourth.
          uint32_t thi = h16;
          if (FMT == kFmtTq2)
            thi |= static_cast<uint32_t>(__half_as_ushort(__float2half_rn(
                       2.0f * __half2float(__ushort_as_half(static_cast<unsigned short>(h16))))))
                   << 16;
          const uint32_t tlo = h16 ^ 0x8000u;
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = __byte_perm(tlo, thi, (dg[2 * i] | (dg[2 * i + 1] << 8)) * 34u + 0x1010u);
          __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + e0 + 8 * lane),
                 make_uint4(o[0], o[1], o[2], o[3]));
        } else {
          const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[i] = dg[i] == 1u ? 0.0f : (dg[i] == 2u ? dw : ((FMT == kFmtTq2 && dg[i] == 3u) ? 2.0f * dw : -dw));  // exact
          float* o = static_cast<float*>(out) + e0 + 4 * lane;
          __stcs(reinterpret_cast<float4*>(o), make_float4(v[0], v[1], v[2], v[3]));
          __stcs(reinterpret_cast<float4*>(o + 128), make_float4(v[4], v[5], v[6], v[7]));
        }
      }
      __syncwarp();  // every lane has read the slot before it is refilled
      issue(s_ring[warp][d], T[d]);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA
}

}  // namespace

int launch_dequant(const uint8_t* blocks, const int32_t* row_ids, int64_t n_out, void* out, int64_t n, int64_t k,
                   bool f16, cudaStream_t s, unsigned* status, int fmt) {
  const DeviceInfo& di = device_info();
  const int nb = static_cast<int>(k / kQK);
  const int64_t units = n_out * nb;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((units + kDqWarps * kDqSeg - 1) / (kDqWarps * kDqSeg),
                                                               static_cast<int64_t>(di.num_sms) * dq_ctas_per_sm(f16)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDqThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (fmt == kFmtTq2)
    e = f16 ? cudaLaunchKernelEx(&cfg, dequant_kernel<true, kFmtTq2>, blocks, row_ids, n_out, out, n, nb, status)
            : cudaLaunchKernelEx(&cfg, dequant_kernel<false, kFmtTq2>, blocks, row_ids, n_out, out, n, nb, status);
  else
    e = f16 ? cudaLaunchKernelEx(&cfg, dequant_kernel<true, kFmtTq1>, blocks, row_ids, n_out, out, n, nb, status)
            : cudaLaunchKernelEx(&cfg, dequant_kernel<false, kFmtTq1>, blocks, row_ids, n_out, out, n, nb, status);
  return cuda_ok(e) ? TQ1_OK : TQ1_ERR_CUDA;
}

}  // namespace tq1
