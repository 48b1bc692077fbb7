// route_dev.cuh -- the routing-list computation as a device function, used
// by the standalone route kernel and by the first kernel of each path.
//
// The gathered path reads only the g = min(E, T*k) routed experts
// (fp8-moe-gather page, sections Problem and The fix).  The routing lists
// tell the expert kernels which slots each routed expert serves: per-expert
// counts and offsets, the slots grouped by expert (stable in slot index),
// the inverse permutation and the ascending list of distinct routed experts
// padded with -1 to its static length g.
//
// One CTA.  Every warp owns a contiguous segment of slots.  Pass 1 counts
// each warp's slots per expert with __match_any_sync (one leader per group
// of equal ids); a per-expert prefix over warps plus a block scan over
// experts gives every (warp, expert) its first output position; pass 2
// walks the segments again and places each slot at
// offset[e] + warp_prefix[w][e] + (rank among equal ids in the 32-slot step),
// which keeps the grouping stable in the slot index.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the total to *total (all threads).
static __device__ int block_exclusive_scan(int v, int* red /*[33]*/, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < nw ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) red[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int base = w > 0 ? red[w - 1] : 0;
  *total = red[nw - 1];
  __syncthreads();
  return base + x - v;
}

// The route computation for one CTA (blockDim.x threads, a multiple of 32).
// Dynamic shared memory: route_smem_bytes(E, blockDim.x).
static __device__ void route_block(const int32_t* __restrict__ ids, int S, int E, RouteBufs rb, uint32_t* status,
                           int* smem) {
  __shared__ int red[33];
  __shared__ int bad;
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = nt >> 5;
  int* wcnt = smem;            // [nw][E]
  int* eoff = smem + nw * E;   // [E]
  for (int i = tid; i < nw * E; i += nt) wcnt[i] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();

  const int seg = (S + nw - 1) / nw;
  const int s0 = min(S, w * seg), s1 = min(S, s0 + seg);
  // pass 1: per-warp counts
  for (int base = s0; base < s1; base += 32) {
    const int s = base + lane;
    const int id = s < s1 ? ids[s] : -1;
    const bool valid = s < s1 && id >= 0 && id < E;
    if (s < s1 && id >= E) bad = 1;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid && lane == __ffs(peers) - 1) wcnt[w * E + id] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per expert: exclusive prefix over warps, total count
  for (int e = tid; e < E; e += nt) {
    int run = 0;
    for (int ww = 0; ww < nw; ++ww) {
      const int c = wcnt[ww * E + e];
      wcnt[ww * E + e] = run;
      run += c;
    }
    eoff[e] = run;
  }
  __syncthreads();
  // block scan over experts: counts -> offsets; distinct flags -> glist
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int lc = 0, ld = 0;
  for (int e = e0; e < e1; ++e) {
    lc += eoff[e];
    ld += eoff[e] > 0;
  }
  int lm = 0;
  for (int e = e0; e < e1; ++e) lm += (eoff[e] + 127) >> 7;
  int tot_c, tot_d, tot_m;
  int oc = block_exclusive_scan(lc, red, &tot_c);
  int od = block_exclusive_scan(ld, red, &tot_d);
  int om = block_exclusive_scan(lm, red, &tot_m);
  for (int e = e0; e < e1; ++e) {
    const int c = eoff[e];
    rb.counts[e] = c;
    rb.offsets[e] = oc;
    if (rb.mtp) rb.mtp[e] = om;
    om += (c + 127) >> 7;
    eoff[e] = oc;
    if (c > 0) {
      if (rb.meta) rb.meta[od] = make_int4(e, oc, c, 0);
      rb.glist[od++] = e;
    }
    oc += c;
  }
  const int g = min(E, S);
  for (int d = tot_d + tid; d < g; d += nt) rb.glist[d] = -1;
  if (tid == 0) {
    rb.offsets[E] = tot_c;
    *rb.nd = tot_d;
    if (rb.mtp) rb.mtp[E] = tot_m;
  }
  __syncthreads();
  // pass 2: stable placement
  for (int base = s0; base < s1; base += 32) {
    const int s = base + lane;
    const int id = s < s1 ? ids[s] : -1;
    const bool valid = s < s1 && id >= 0 && id < E;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid) {
      const int pos = eoff[id] + wcnt[w * E + id] + __popc(peers & lanemask_lt());
      rb.perm[pos] = s;
      rb.inv[s] = pos;
    } else if (s < s1) {
      rb.inv[s] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[w * E + id] += __popc(peers);
    __syncwarp();
  }
  for (int q = tot_c + tid; q < S; q += nt) rb.perm[q] = -1;
  if (tid == 0 && bad) raise_status(status, MOE_STATUS_BAD_ID);
}

}  // namespace moe
