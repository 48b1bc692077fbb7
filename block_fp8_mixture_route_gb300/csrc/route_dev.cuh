// route_dev.cuh -- the routing-list computation, as device functions used by
// the single-CTA route (small slot counts, fused into the decode path's
// first kernel) and by the three-kernel route for large slot counts.
//
// The gathered path reads only the g = min(E, T*k) routed experts
// (fp8-moe-gather page, sections Problem and The fix).  The routing lists
// tell the expert kernels which slots each routed expert serves: per-expert
// counts and offsets, the slots grouped by expert (stable in slot index),
// the inverse permutation, the ascending list of distinct routed experts
// padded with -1 to its static length g, one (expert, offset, count) record
// per distinct expert and the per-expert prefix of 128-row tiles.
//
// Stable placement: every warp owns a contiguous segment of slots.  Pass 1
// counts each warp's slots per expert with __match_any_sync (one leader per
// group of equal ids); a per-expert prefix over warps plus the expert's base
// gives every (warp, expert) its first output position; pass 2 walks the
// segments again and places each slot at
// base[e] + warp_prefix[w][e] + (rank among equal ids in the 32-slot step),
// which keeps the grouping stable in the slot index.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

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

// The same for four independent counters at once (one pass of barriers).
static __device__ int4 block_exclusive_scan4(int4 v, int4* red /*[33]*/, int4* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int4 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yx = __shfl_up_sync(0xffffffffu, x.x, o), yy = __shfl_up_sync(0xffffffffu, x.y, o);
    const int yz = __shfl_up_sync(0xffffffffu, x.z, o), yw = __shfl_up_sync(0xffffffffu, x.w, o);
    if (lane >= o) {
      x.x += yx;
      x.y += yy;
      x.z += yz;
      x.w += yw;
    }
  }
  if (lane == 31) red[w] = x;
  __syncthreads();
  if (w == 0) {
    int4 s = lane < nw ? red[lane] : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yx = __shfl_up_sync(0xffffffffu, s.x, o), yy = __shfl_up_sync(0xffffffffu, s.y, o);
      const int yz = __shfl_up_sync(0xffffffffu, s.z, o), yw = __shfl_up_sync(0xffffffffu, s.w, o);
      if (lane >= o) {
        s.x += yx;
        s.y += yy;
        s.z += yz;
        s.w += yw;
      }
    }
    if (lane < nw) red[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int4 b = w > 0 ? red[w - 1] : make_int4(0, 0, 0, 0);
  *total = red[nw - 1];
  __syncthreads();
  return make_int4(b.x + x.x - v.x, b.y + x.y - v.y, b.z + x.z - v.z, b.w + x.w - v.w);
}

// Pass 1 over slots [s0, s1) split into contiguous per-warp segments:
// wcnt[w][e] = slots of warp w routed to expert e.  Sets *bad if an id >= E
// is seen.  Ends with __syncthreads.
static __device__ void route_warp_counts(const int32_t* __restrict__ ids, int s0, int s1, int E, int* wcnt,
                                         int* bad) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = nt >> 5;
  for (int i = tid; i < nw * E; i += nt) wcnt[i] = 0;
  __syncthreads();
  const int seg = (s1 - s0 + nw - 1) / nw;
  const int a = min(s1, s0 + w * seg), b = min(s1, a + seg);
  for (int base = a; base < b; base += 32) {
    const int s = base + lane;
    const int id = s < b ? ids[s] : -1;
    const bool valid = s < b && id >= 0 && id < E;
    if (s < b && id >= E) *bad = 1;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid && lane == __ffs(peers) - 1) wcnt[w * E + id] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
}

// wcnt[w][e] -> exclusive prefix over warps; tot[e] = column totals.
// Ends with __syncthreads.
static __device__ void route_warp_prefix(int* wcnt, int E, int* tot) {
  const int nt = blockDim.x, nw = nt >> 5;
  for (int e = threadIdx.x; e < E; e += nt) {
    int run = 0;
    for (int ww = 0; ww < nw; ++ww) {
      const int c = wcnt[ww * E + e];
      wcnt[ww * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
}

// Pass 2: place every valid slot of [s0, s1) at base(e) + wcnt[w][e] + rank.
template <typename BaseF>
static __device__ void route_warp_place(const int32_t* __restrict__ ids, int s0, int s1, int E, int* wcnt,
                                        BaseF base_of, RouteBufs rb) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = nt >> 5;
  const int seg = (s1 - s0 + nw - 1) / nw;
  const int a = min(s1, s0 + w * seg), b = min(s1, a + seg);
  for (int base = a; base < b; base += 32) {
    const int s = base + lane;
    const int id = s < b ? ids[s] : -1;
    const bool valid = s < b && id >= 0 && id < E;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid) {
      const int pos = base_of(id) + wcnt[w * E + id] + __popc(peers & lanemask_lt());
      rb.perm[pos] = s;
      rb.inv[s] = pos;
    } else if (s < b) {
      rb.inv[s] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[w * E + id] += __popc(peers);
    __syncwarp();
  }
}

// Expert-level lists from per-expert counts in eoff[E] (shared memory):
// writes counts, offsets, glist (padded to min(E, S)), meta, n_distinct,
// and either mtp, mtp2 or (decode) the per-pass work list, and fills
// perm[offsets[E] .. S) with -1.  On return eoff[e] holds the offset of
// expert e.  Ends with __syncthreads.
static __device__ void route_expert_scan(int* eoff, int E, int S, RouteBufs rb) {
  __shared__ int4 red[33];
  const int nt = blockDim.x, tid = threadIdx.x;
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  // the third scanned quantity: 128-row tiles (prefill) or passes of spp
  // slots (decode work list); the fourth: pairs of 128-row tiles (prefill)
  const bool vl = rb.vmeta != nullptr;
  auto q3 = [&](int c) { return vl ? (c + rb.spp - 1) / rb.spp : (c + 127) >> 7; };
  auto q4 = [&](int c) { return vl ? 0 : (((c + 127) >> 7) + 1) >> 1; };
  int lc = 0, ld = 0, lm = 0, lp = 0;
  for (int e = e0; e < e1; ++e) {
    lc += eoff[e];
    ld += eoff[e] > 0;
    lm += q3(eoff[e]);
    lp += q4(eoff[e]);
  }
  int4 tot;
  const int4 ex = block_exclusive_scan4(make_int4(lc, ld, lm, lp), red, &tot);
  int oc = ex.x, od = ex.y, om = ex.z, op = ex.w;
  const int tot_c = tot.x, tot_d = tot.y, tot_m = tot.z, tot_p = tot.w;
  for (int e = e0; e < e1; ++e) {
    const int c = eoff[e];
    rb.counts[e] = c;
    rb.offsets[e] = oc;
    if (vl) {
      const int n = q3(c);
      for (int q = 0; q < n; ++q) rb.vmeta[om + q] = make_int4(e, oc + q * rb.spp, min(rb.spp, c - q * rb.spp), n);
    } else {
      if (rb.mtp) rb.mtp[e] = om;
      if (rb.mtp2) rb.mtp2[e] = op;
    }
    om += q3(c);
    op += q4(c);
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
    rb.nd[0] = tot_d;
    if (vl) {
      rb.nd[1] = tot_m;
    } else {
      if (rb.mtp) rb.mtp[E] = tot_m;
      if (rb.mtp2) rb.mtp2[E] = tot_p;
    }
  }
  for (int q = tot_c + tid; q < S; q += nt) rb.perm[q] = -1;
  __syncthreads();
}

// The whole route for one CTA (blockDim.x threads, a multiple of 32).
// Dynamic shared memory: route_smem_bytes(E, blockDim.x).
static __device__ void route_block(const int32_t* __restrict__ ids, int S, int E, RouteBufs rb, uint32_t* status,
                                   int* smem) {
  __shared__ int bad;
  const int nw = blockDim.x >> 5;
  int* wcnt = smem;            // [nw][E]
  int* eoff = smem + nw * E;   // [E]
  if (threadIdx.x == 0) bad = 0;
  route_warp_counts(ids, 0, S, E, wcnt, &bad);
  route_warp_prefix(wcnt, E, eoff);
  route_expert_scan(eoff, E, S, rb);
  route_warp_place(ids, 0, S, E, wcnt, [&](int e) { return eoff[e]; }, rb);
  if (threadIdx.x == 0 && bad) raise_status(status, MOE_STATUS_BAD_ID);
}

}  // namespace moe
