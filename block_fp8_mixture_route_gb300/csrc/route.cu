// route.cu -- the standalone routing kernels (moe_fp8_block_route and the
// prefill path) and the e4m3 widening test kernel.
//
// Small slot counts use one CTA (route_block).  Large ones use three
// kernels: per-CTA expert histograms of contiguous slot chunks, one CTA that
// turns them into per-(chunk, expert) bases and the expert-level lists, and
// a stable per-chunk placement.  Both produce identical lists.
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

int route_chunks(int S) {
  if (S <= kRouteSingleMax) return 1;
  const int g = (S + kRouteChunk - 1) / kRouteChunk;
  return g < kRouteMaxChunks ? g : kRouteMaxChunks;
}

__global__ void route_kernel(const int32_t* __restrict__ ids, int S, int E, RouteBufs rb, uint32_t* status) {
  extern __shared__ int smem_route[];
  route_block(ids, S, E, rb, status, smem_route);
}

// Histogram of chunk blockIdx.x: cnt[chunk][e].
__global__ void __launch_bounds__(256) route_count_kernel(const int32_t* __restrict__ ids, int S, int E, int chunk,
                                                          int32_t* __restrict__ cnt, uint32_t* status) {
  extern __shared__ int hist[];
  __shared__ int bad;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  const int s0 = min(S, (int)blockIdx.x * chunk), s1 = min(S, s0 + chunk);
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const int id = ids[s];
    if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
    else if (id >= E) bad = 1;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(int64_t)blockIdx.x * E + e] = hist[e];
  if (threadIdx.x == 0 && bad) raise_status(status, MOE_STATUS_BAD_ID);
}

// One CTA: chunk histograms cnt[c][e] -> cbase[c][e], the first output
// position of chunk c's slots of expert e, and the expert-level lists.  Two
// read-only passes over cnt (totals, then running prefixes) whose loads do
// not depend on earlier stores, so each thread keeps many in flight.
__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ cnt,
                                                          int32_t* __restrict__ cbase, int G, int S, int E,
                                                          RouteBufs rb) {
  extern __shared__ int eoff[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll 8
    for (int c = 0; c < G; ++c) run += __ldg(cnt + (int64_t)c * E + e);
    eoff[e] = run;
  }
  __syncthreads();
  route_expert_scan(eoff, E, S, rb);   // eoff[e] becomes expert e's first position
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = eoff[e];
#pragma unroll 8
    for (int c = 0; c < G; ++c) {
      const int v = __ldg(cnt + (int64_t)c * E + e);
      cbase[(int64_t)c * E + e] = run;
      run += v;
    }
  }
}

// Stable placement of chunk blockIdx.x from its per-expert bases.
__global__ void route_place_kernel(const int32_t* __restrict__ ids, int S, int E, int chunk,
                                   const int32_t* __restrict__ cbase, RouteBufs rb) {
  extern __shared__ int smem_place[];
  __shared__ int bad;
  pdl_wait();
  pdl_trigger();
  const int nw = blockDim.x >> 5;
  int* wcnt = smem_place;
  int* tot = smem_place + nw * E;
  const int s0 = min(S, (int)blockIdx.x * chunk), s1 = min(S, s0 + chunk);
  const int32_t* base = cbase + (int64_t)blockIdx.x * E;
  route_warp_counts(ids, s0, s1, E, wcnt, &bad);
  route_warp_prefix(wcnt, E, tot);
  route_warp_place(ids, s0, s1, E, wcnt, [&](int e) { return base[e]; }, rb);
}

template <typename K, typename... Args>
static cudaError_t launch_k(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_route(const int32_t* ids, int S, int E, const RouteBufs& rb, uint32_t* status,
                         int32_t* scratch, cudaStream_t st, int* launches) {
  const int G = scratch ? route_chunks(S) : 1;
  cudaError_t err;
  if (G <= 1) {
    // few slots: a CTA of about one warp per 32 slots keeps the per-warp
    // counters and the block-wide scans short
    int nt = route_threads(E);
    const int want = (S + 31) / 32 * 32;
    if (want < nt) nt = want < 128 ? 128 : want;
    const size_t sm = route_smem_bytes(E, nt);
    if ((err = set_max_smem((const void*)route_kernel, (int)sm)))
      return err;
    route_kernel<<<1, nt, sm, st>>>(ids, S, E, rb, status);
    if (launches) *launches += 1;
    return cudaGetLastError();
  }
  const int chunk = (S + G - 1) / G;
  if ((err = set_max_smem((const void*)route_count_kernel, E * 4)))
    return err;
  if ((err = set_max_smem((const void*)route_scan_kernel, E * 4))) return err;
  const int nt = route_threads(E);
  const size_t psm = route_smem_bytes(E, nt);
  if ((err = set_max_smem((const void*)route_place_kernel, (int)psm)))
    return err;
  if ((err = launch_k(route_count_kernel, dim3(G), dim3(256), (size_t)E * 4, st, false, ids, S, E, chunk, scratch,
                      status)))
    return err;
  int32_t* cbase = scratch + (int64_t)G * E;
  if ((err = launch_k(route_scan_kernel, dim3(1), dim3(1024), (size_t)E * 4, st, true, (const int32_t*)scratch,
                      cbase, G, S, E, rb)))
    return err;
  if ((err = launch_k(route_place_kernel, dim3(G), dim3(nt), psm, st, true, ids, S, E, chunk,
                      (const int32_t*)cbase, rb)))
    return err;
  if (launches) *launches += 3;
  return cudaSuccess;
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
