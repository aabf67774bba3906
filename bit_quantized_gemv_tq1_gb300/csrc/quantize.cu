// quantize.cu -- fp32 -> TQ1_0 (and TQ2_0) weight blocks and fp32 -> Q8_1
// activation blocks, bit-exact with the rounding readings of the library:
//   weights: d = fp16(amax); t = amax ? clamp(round_half_away(w / amax), -1, 1) : 0
//   activations: d = amax / 127; q = d ? clamp(round_half_away(x / d), -127, 127) : 0;
//                stored fp16(d), fp16(d * sum(q)), q[32]
// All arithmetic is IEEE fp32 with explicit round-to-nearest intrinsics so
// that no contraction or fast-math substitution can change a bit.
// Byte code and element order: PrismML-Eng/llama.cpp issue #139, "Current
// behavior", and the TQ1_0 block specification (qs[48], qh[4], fp16 d).
#include "../../include/tq1.h"
#include "tq1_device.cuh"
#include "tq1_internal.h"

namespace tq1 {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per 256-weight block.  Lane i (< 32) packs qs[i] from elements
// i + 32c (c < 5); lanes 0..15 also pack qs[32 + i] from 160 + i + 16c;
// lanes 16..19 pack qh[i - 16] from 240 + (i - 16) + 4c (c < 4).
__global__ void __launch_bounds__(kWarpsPerCta * 32) quantize_rows_kernel(const float* __restrict__ w,
                                                                          uint8_t* __restrict__ out,
                                                                          int64_t nblocks) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (blk < nblocks) {
    const float* x = w + blk * kQK;
    float va[5], vb[5];
#pragma unroll
    for (int c = 0; c < 5; ++c) va[c] = x[lane + 32 * c];
    const bool has_b = lane < 20;
#pragma unroll
    for (int c = 0; c < 5; ++c) {
      if (lane < 16) vb[c] = x[160 + lane + 16 * c];
      else if (lane < 20 && c < 4) vb[c] = x[240 + (lane - 16) + 4 * c];
      else vb[c] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int c = 0; c < 5; ++c) m = fmaxf(m, fmaxf(fabsf(va[c]), fabsf(vb[c])));
    const float amax = warp_max(m);
    auto trit = [amax](float v) -> int {
      if (amax == 0.0f) return 1;
      float r = roundf(__fdiv_rn(v, amax));  // roundf: halves away from zero
      r = fminf(fmaxf(r, -1.0f), 1.0f);
      return static_cast<int>(r) + 1;
    };
    uint8_t* o = out + blk * kBlockBytes;
    int v = 0;
#pragma unroll
    for (int c = 0; c < 5; ++c) v = v * 3 + trit(va[c]);
    o[lane] = static_cast<uint8_t>((v * 256 + 242) / 243);
    if (has_b) {
      int vv = 0;
      const int nd = lane < 16 ? 5 : 4;
#pragma unroll
      for (int c = 0; c < 5; ++c)
        if (c < nd) vv = vv * 3 + trit(vb[c]);
      if (nd == 4) vv *= 3;  // four trits: the fifth digit is 0
      o[lane < 16 ? 32 + lane : 48 + (lane - 16)] = static_cast<uint8_t>((vv * 256 + 242) / 243);
    }
    if (lane == 0) {  // fp16 scale: one 16-bit store (54 * blk + 52 is even)
      const __half_raw d16 = __float2half_rn(amax);
      *reinterpret_cast<unsigned short*>(o + 52) = d16.x;
    }
  }
  // Dependents may prefetch weights before waiting on this kernel: make the
  // blocks visible device-wide before this CTA retires.
  __threadfence();
}

// TQ2_0 (four 2-bit codes per byte, code = trit + 1; chunk c reads field
// c % 4 of bytes 32(c/4) .. 32(c/4)+31): one warp per 256-weight block, lane
// i packs qs[i] from elements i + 32f and qs[32 + i] from 128 + i + 32f
// (f < 4).  Same scale and rounding as the TQ1_0 encoder.
__global__ void __launch_bounds__(kWarpsPerCta * 32) quantize_rows_tq2_kernel(const float* __restrict__ w,
                                                                              uint8_t* __restrict__ out,
                                                                              int64_t nblocks) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (blk < nblocks) {
    const float* x = w + blk * kQK;
    float v[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int f = 0; f < 4; ++f) v[h][f] = x[128 * h + 32 * f + lane];
    float m = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int f = 0; f < 4; ++f) m = fmaxf(m, fabsf(v[h][f]));
    const float amax = warp_max(m);
    uint8_t* o = out + blk * kTq2BlockBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t byte = 0;
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        int code = 1;
        if (amax != 0.0f) {
          float r = roundf(__fdiv_rn(v[h][f], amax));  // roundf: halves away from zero
          r = fminf(fmaxf(r, -1.0f), 1.0f);
          code = static_cast<int>(r) + 1;
        }
        byte |= static_cast<uint32_t>(code) << (2 * f);
      }
      o[32 * h + lane] = static_cast<uint8_t>(byte);
    }
    if (lane == 0) {  // fp16 scale: one 16-bit store (66 * blk + 64 is even)
      const __half_raw d16 = __float2half_rn(amax);
      *reinterpret_cast<unsigned short*>(o + 64) = d16.x;
    }
  }
  __threadfence();
}

// One warp per Q8_1 block of 32 activations.  This kernel does not signal
// its dependents early: its grid spans several waves, and a dependent grid
// admitted while those waves are still being placed ends up unevenly spread
// over the SMs (measured: a following chain of one-CTA-per-SM mat-vec
// launches ran ~50% slower).  Dependents start as its CTAs retire.
__global__ void __launch_bounds__(kWarpsPerCta * 32) quantize_acts_kernel(const float* __restrict__ x,
                                                                          uint8_t* __restrict__ out,
                                                                          int64_t nblocks) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (blk >= nblocks) return;
  const float v = x[blk * kQK8 + lane];
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  int q = 0;
  if (d != 0.0f) {
    float r = roundf(__fdiv_rn(v, d));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    q = static_cast<int>(r);
  }
  const int sum = warp_sum(q);
  // Gather four int8 codes per 32-bit word: lane l < 8 writes word l.
  const uint32_t qb = static_cast<uint32_t>(q) & 0xFFu;
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) word |= __shfl_sync(0xffffffffu, qb, ((lane & 7) << 2) + i) << (8 * i);
  uint32_t* o = reinterpret_cast<uint32_t*>(out + blk * kQ8Bytes);
  if (lane < 8) o[1 + lane] = word;
  if (lane == 0) {
    const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
    const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, static_cast<float>(sum))));
    o[0] = d16 | (s16 << 16);
  }
}

static int launch_simple(void (*kern)(const float*, uint8_t*, int64_t), const float* in, uint8_t* out,
                         int64_t nblocks, cudaStream_t s) {
  if (nblocks == 0) return TQ1_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((nblocks + kWarpsPerCta - 1) / kWarpsPerCta));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&cfg, kern, in, out, nblocks)) ? TQ1_OK : TQ1_ERR_CUDA;
}

int launch_quantize_rows(const float* w, uint8_t* blocks, int64_t n, int64_t k, cudaStream_t s) {
  return launch_simple(quantize_rows_kernel, w, blocks, n * (k / kQK), s);
}

int launch_quantize_rows_tq2(const float* w, uint8_t* blocks, int64_t n, int64_t k, cudaStream_t s) {
  return launch_simple(quantize_rows_tq2_kernel, w, blocks, n * (k / kQK), s);
}

int launch_quantize_acts(const float* x, uint8_t* q8, int64_t t, int64_t k, cudaStream_t s) {
  return launch_simple(quantize_acts_kernel, x, q8, t * (k / kQK8), s);
}

}  // namespace tq1
