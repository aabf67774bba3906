// dequant.cu -- TQ1_0 rows back to fp32 or fp16 values: whole-matrix
// dequantisation and row gathers (get_rows, e.g. an embedding lookup).
//
// The CPU reference walks a 256-block once and amortises each packed byte
// over its trits (PrismML-Eng/llama.cpp issue #139, "Current behavior"); the
// Vulkan backend of the same format ships dequant and get_rows shaders next
// to its mat-vec ("Upstream state").  Here one warp owns one 256-block of one
// output row: lane l produces elements 8l .. 8l+7.  Those eight elements are
// digit k of eight consecutive packed bytes (element order of the block:
// e < 160 -> qs[e % 32] digit e/32; e < 240 -> qs[32 + (e-160) % 16] digit
// (e-160)/16; else qh[(e-240) % 4] digit (e-240)/4), so each lane reads its
// eight bytes once and expands them with the specification's digit formula
// ((uint8)(b*3^k)*3) >> 8.  Stores are 16-byte vectors, a warp writing one
// contiguous 1 KiB (fp32) or 512 B (fp16) span: the kernel is bound by the
// output bytes written to HBM.
//
// TQ2_0 blocks (2-bit codes, 66 bytes) take the same path: lane l's eight
// elements lie in chunk c = l / 4, so they are field c % 4 of the eight
// consecutive bytes qs[32 * (c / 4) + 8 * (l % 4) ..]; code 3 (never written
// by the encoder) gives +2d, the fourth entry of the value table.
#include <algorithm>

#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

namespace {

constexpr int kDqThreads = 256;
constexpr int kDqWarps = kDqThreads / 32;
constexpr int kDqUnits = 2;  // 256-blocks per warp whose loads are in flight together (4: fewer resident warps, slower)

__device__ __forceinline__ uint32_t digit_of(uint32_t b, uint32_t k) {
  const uint32_t p = static_cast<uint32_t>((kPow3Packed >> (8 * k)) & 0xFFu);
  return (((b * p) & 0xFFu) * 3u) >> 8;
}

template <bool F16, int FMT>
__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const uint8_t* __restrict__ blocks,
                                                             const int32_t* __restrict__ row_ids, int64_t n_out,
                                                             void* __restrict__ out, int64_t n, int nb,
                                                             unsigned* status) {
  pdl_wait();  // blocks and row ids may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int64_t units = n_out * nb;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * kDqWarps;
  constexpr int kBB = fmt_block_bytes<FMT>();
  // Byte offset of this lane's first byte within the block, and its digit(s)
  // (TQ2_0: its 2-bit field).
  int boff, dig;
  if (FMT == kFmtTq2) {
    boff = 32 * (lane >> 4) + 8 * (lane & 3);
    dig = (lane >> 2) & 3;
  } else if (lane < 20) {
    boff = 8 * (lane & 3);
    dig = lane >> 2;
  } else if (lane < 30) {
    boff = 32 + 8 * ((lane - 20) & 1);
    dig = (lane - 20) >> 1;
  } else {
    boff = 48;              // qh[0..3], digits 2 (lane - 30) and 2 (lane - 30) + 1
    dig = 2 * (lane - 30);
  }
  // The warp's units are u = first, first + wstride, ...; their (output row,
  // block) advance by the stride's quotient and remainder (one division per
  // warp instead of one per unit).
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kDqWarps + (threadIdx.x >> 5);
  const int64_t sq = wstride / nb;
  const int sr = static_cast<int>(wstride - sq * nb);
  int64_t crow = first / nb;  // the next unit's output row and block
  int cb = static_cast<int>(first - crow * nb);
  // kDqUnits units per iteration: their loads are in flight together.
  for (int64_t u0 = first; u0 < units; u0 += kDqUnits * wstride) {
    uint32_t hw[kDqUnits][5];  // per unit: 4 halfwords of the lane's bytes, the fp16 scale
    int64_t orow[kDqUnits];
    int bb[kDqUnits];
    bool live[kDqUnits];
#pragma unroll
    for (int x = 0; x < kDqUnits; ++x) {
      const int64_t u = u0 + x * wstride;
      live[x] = u < units;
      orow[x] = crow;
      bb[x] = cb;
      crow += sq;
      cb += sr;
      if (cb >= nb) {
        cb -= nb;
        ++crow;
      }
      int64_t srow = orow[x];
      if (live[x] && row_ids) {
        srow = __ldg(row_ids + orow[x]);
        if (srow < 0 || srow >= n) {
          if (lane == 0 && bb[x] == 0) raise_status(status, kStatusBadId);
          live[x] = false;  // the output row is left untouched
        }
      }
      if (live[x]) {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(blocks + (srow * nb + bb[x]) * kBB);
#pragma unroll
        for (int i = 0; i < 4; ++i) hw[x][i] = __ldg(h + (boff >> 1) + i);
        hw[x][4] = __ldg(h + (kBB - 2) / 2);
      }
    }
#pragma unroll
    for (int x = 0; x < kDqUnits; ++x) {
      if (!live[x]) continue;
      uint32_t by[8];
      if (FMT == kFmtTq2 || lane < 30) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          by[2 * i] = hw[x][i] & 0xFFu;
          by[2 * i + 1] = hw[x][i] >> 8;
        }
      } else {  // qh[0..3] twice: digits dig and dig + 1
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          by[2 * i] = by[2 * i + 4] = hw[x][i] & 0xFFu;
          by[2 * i + 1] = by[2 * i + 5] = hw[x][i] >> 8;
        }
      }
      uint32_t dg[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dg[i] = FMT == kFmtTq2 ? (by[i] >> (2 * dig)) & 3u
                               : digit_of(by[i], lane < 30 ? static_cast<uint32_t>(dig) : static_cast<uint32_t>(dig + (i >> 2)));
      const int64_t e0 = orow[x] * static_cast<int64_t>(nb) * kQK + static_cast<int64_t>(bb[x]) * kQK + 8 * lane;
      const uint32_t h16 = hw[x][4];
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
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + e0), make_uint4(o[0], o[1], o[2], o[3]));
      } else {
        const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = dg[i] == 1u ? 0.0f : (dg[i] == 2u ? dw : ((FMT == kFmtTq2 && dg[i] == 3u) ? 2.0f * dw : -dw));  // exact
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + e0);
        __stcs(o, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(o + 1, make_float4(v[4], v[5], v[6], v[7]));
      }
    }
  }
}

}  // namespace

int launch_dequant(const uint8_t* blocks, const int32_t* row_ids, int64_t n_out, void* out, int64_t n, int64_t k,
                   bool f16, cudaStream_t s, unsigned* status, int fmt) {
  const DeviceInfo& di = device_info();
  const int nb = static_cast<int>(k / kQK);
  const int64_t warps = n_out * nb;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((warps + kDqWarps - 1) / kDqWarps,
                                                               static_cast<int64_t>(di.num_sms) * 16));
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
