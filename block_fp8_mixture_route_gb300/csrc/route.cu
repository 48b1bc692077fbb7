// route.cu -- the standalone routing kernel (moe_fp8_block_route) and the
// e4m3 widening test kernel.
#include "route_dev.cuh"
namespace moe {

int route_threads(int E) {
  // per-warp counters take 4*E bytes per warp; keep them within ~192 KiB
  int nw = (int)((192 * 1024) / (4 * (size_t)E + 4));
  nw = nw < 1 ? 1 : (nw > 32 ? 32 : nw);
  return nw * 32;
}

size_t route_smem_bytes(int E, int nthreads) {
  return (size_t)(nthreads / 32) * E * 4 + (size_t)E * 4;
}

__global__ void route_kernel(const int32_t* __restrict__ ids, int S, int E, RouteBufs rb, uint32_t* status) {
  extern __shared__ int smem_route[];
  route_block(ids, S, E, rb, status, smem_route);
}

cudaError_t launch_route(const int32_t* ids, int S, int E, const RouteBufs& rb, uint32_t* status,
                         cudaStream_t st) {
  const int nt = route_threads(E);
  const size_t sm = route_smem_bytes(E, nt);
  cudaError_t err = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (err != cudaSuccess) return err;
  route_kernel<<<1, nt, sm, st>>>(ids, S, E, rb, status);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------
// e4m3 widening exactly as the decode kernels do it (for the unit test).
__global__ void widen_kernel(const uint8_t* __restrict__ codes, int64_t n, float* __restrict__ out) {
  const int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 2;
  if (i >= n) return;
  const uint16_t lo = codes[i];
  const uint16_t hi = (i + 1 < n) ? codes[i + 1] : 0;
  const float2 f = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(lo | (hi << 8))));
  out[i] = f.x;
  if (i + 1 < n) out[i + 1] = f.y;
}

cudaError_t launch_widen(const uint8_t* codes, int64_t n, float* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t pairs = (n + 1) / 2;
  const int nt = 256;
  widen_kernel<<<(unsigned)((pairs + nt - 1) / nt), nt, 0, st>>>(codes, n, out);
  return cudaGetLastError();
}

}  // namespace moe
