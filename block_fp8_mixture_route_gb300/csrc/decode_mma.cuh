// decode_mma.cuh -- device helpers of the decode (W8A16 / W8A8) kernels:
// e4m3 widening into m16n8k16 fragments, the f16 tensor-core MMA, shared
// memory vector loads, bounded warp waits and the routed-expert bitmap.
// Written for sm_103a (GB300).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 values -> two e4m3 codes (lo -> low byte), RNE, saturating.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ float4 lds_f4(const void* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}


// Bounded wait by lane 0 of a warp; its outcome is returned on all lanes.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Widen one 64-wide K chunk of two weight rows (tile rows g and g+8) into
// the A fragments of four m16n8k16 MMAs.  Physical element 16c + 4m + v of
// the chunk (c = lane % 4) plays logical k {2c, 2c+1, 2c+8, 2c+9}[v] of MMA
// m; the B fragment uses the same map, so the four MMAs together sum over
// exactly the chunk's 64 elements.
__device__ __forceinline__ void afrag(const uint4& wa, const uint4& wb, uint32_t (&A)[4][4]) {
  const uint32_t wa_[4] = {wa.x, wa.y, wa.z, wa.w};
  const uint32_t wb_[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    e4m3x4_to_f16x4(wa_[m], A[m][0], A[m][2]);
    e4m3x4_to_f16x4(wb_[m], A[m][1], A[m][3]);
  }
}

// One 64-wide K chunk: four MMAs on two independent accumulators (shorter
// dependency chains).
__device__ __forceinline__ void chunk_mma(float (&b0)[4], float (&b1)[4], const uint4& wa, const uint4& wb,
                                          const uint4& x0, const uint4& x1) {
  uint32_t A[4][4];
  afrag(wa, wb, A);
  mma_f16_16816(b0, A[0], x0.x, x0.y);
  mma_f16_16816(b1, A[1], x0.z, x0.w);
  mma_f16_16816(b0, A[2], x1.x, x1.y);
  mma_f16_16816(b1, A[3], x1.z, x1.w);
}

// The routed experts as a bitmap in shared memory (bit e set when some slot
// routes to expert e, 0 <= e < E), built by one warp from the ids alone: the
// same experts, in the same ascending order, as the routing lists, so a
// kernel can know its first experts before the routing lists exist.  Lane l
// keeps words 4l .. 4l+3 (E <= 4096) and the exclusive / inclusive counts of
// set bits before and through them.  Returns the number of routed experts.
struct ExpertBits {
  uint32_t w[4];
  int excl, incl;
};

__device__ __forceinline__ int expert_bits(const int32_t* __restrict__ ids, int S, int E, uint32_t* bits, int lane,
                                           ExpertBits& eb) {
  const int nwords = (E + 31) >> 5;
  for (int i = lane; i < 128; i += 32) bits[i] = 0;
  __syncwarp();
  for (int s = lane; s < S; s += 32) {
    const int id = __ldg(ids + s);
    if (id >= 0 && id < E) atomicOr(&bits[id >> 5], 1u << (id & 31));
  }
  __syncwarp();
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int wi = lane * 4 + j;
    eb.w[j] = wi < nwords ? bits[wi] : 0u;
    cnt += __popc(eb.w[j]);
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  eb.excl = incl - cnt;
  eb.incl = incl;
  return __shfl_sync(0xffffffffu, incl, 31);
}

// The d-th routed expert (0-based, ascending), on all lanes.
__device__ __forceinline__ int expert_select(const ExpertBits& eb, int d, int lane) {
  int e = -1;
  if (eb.excl <= d && d < eb.incl) {
    int r = d - eb.excl;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = __popc(eb.w[j]);
      if (e < 0 && r < c) {
        uint32_t v = eb.w[j];
        for (int q = 0; q < r; ++q) v &= v - 1;   // drop the r lowest set bits
        e = (lane * 4 + j) * 32 + __ffs(v) - 1;
      } else if (e < 0) {
        r -= c;
      }
    }
  }
  const uint32_t owner = __ballot_sync(0xffffffffu, e >= 0);
  return owner ? __shfl_sync(0xffffffffu, e, __ffs(owner) - 1) : -1;
}

}  // namespace moe
