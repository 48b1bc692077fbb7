// prefill.cu -- the prefill (W8A8) path of the block-FP8 MoE layer.
//
// Activations are quantised per token per 128-column group with a dynamic
// scale (fp8-moe-gather page, "Affects": dynamic activation scales):
// scale = amax / 448 in IEEE fp32, code = e4m3(x / scale) rounded to
// nearest even and saturated to the largest finite value.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 values -> two e4m3 codes (lo -> low byte), RNE, saturating.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per (row, 128-column group): each lane holds 4 consecutive values.
__global__ void __launch_bounds__(256) act_quant_kernel(const uint16_t* __restrict__ x, int64_t ld, int R, int K,
                                                        uint8_t* __restrict__ codes, float* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int groups = K / 128;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (int64_t)R * groups) return;
  const int lane = threadIdx.x & 31;
  const int64_t r = wid / groups;
  const int gi = (int)(wid % groups);
  const uint2 raw = *reinterpret_cast<const uint2*>(x + r * ld + gi * 128 + lane * 4);
  float v[4] = {bf16_to_f32(raw.x & 0xFFFFu), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xFFFFu),
                bf16_to_f32(raw.y >> 16)};
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sc = __fdiv_rn(m, 448.0f);
  uint32_t packed = 0;
  if (sc != 0.f) {
    const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc));
    const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc));
    packed = (uint32_t)c01 | ((uint32_t)c23 << 16);
  }
  *reinterpret_cast<uint32_t*>(codes + r * K + gi * 128 + lane * 4) = packed;
  if (lane == 0) scales[r * groups + gi] = sc;
}

cudaError_t launch_act_quant(const uint16_t* x, int64_t ld, int R, int K, uint8_t* codes, float* scales,
                             cudaStream_t st, bool pdl) {
  const int64_t warps = (int64_t)R * (K / 128);
  if (warps == 0) return cudaSuccess;
  const int per_block = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + per_block - 1) / per_block));
  cfg.blockDim = dim3(32 * per_block);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, act_quant_kernel, x, ld, R, K, codes, scales);
}

cudaError_t launch_prefill(const LayerArgs& a, const RouteBufs& rb, const PrefillBufs& pb, uint32_t* status,
                           int device, cudaStream_t st, int* launches) {
  (void)a;
  (void)rb;
  (void)pb;
  (void)status;
  (void)device;
  (void)st;
  (void)launches;
  return cudaErrorNotSupported;
}

}  // namespace moe
