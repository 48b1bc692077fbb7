// prefill.cu -- the prefill (W8A8) path of the block-FP8 MoE layer.
//
// Activations are quantised per token per 128-column group with a dynamic
// scale (fp8-moe-gather page, "Affects": dynamic activation scales): scale =
// amax / 448 in IEEE fp32, code = e4m3(x / scale) rounded to nearest even
// and saturated to the largest finite value.  Both projections then run as
// grouped FP8 GEMMs on the tcgen05 tensor cores (kind::f8f6f4, fp32
// accumulators in tensor memory), with h = silu(gate) * up fused into the
// first GEMM's epilogue and quantised the same way, per slot per 128 columns.
//
// Kernels, in stream order (chained with programmatic dependent launch):
//   route               routing lists + per-expert 128-row tile counts
//   act_quant_permute   e4m3 codes/scales of every token, written to each of
//                       its routed slots' rows (routed order), so that every
//                       GEMM operand tile is one contiguous tensor-map load
//   prefill_gemm<1>     per (expert, 128 slots, 128-row block of gate + the
//                       matching block of up): X[128 x H] W13^T -> silu*up ->
//                       e4m3 h codes + scales
//   prefill_gemm<2>     per (expert, 128 slots, 256 rows of the down
//                       projection): H[128 x I] W2^T * top-k weight -> bf16
//                       slot rows
//   prefill_combine     out[t] = sum_j slot[t*k + j] in j order
//
// Block-scale promotion: a tcgen05 MMA chain covers one 128-wide K block
// into a fresh TMEM accumulator; the epilogue warps read it back and add
// (activation scale of the row) * (weight scale of the column block) times
// it into fp32 registers.  Two TMEM accumulators alternate, so the tensor
// core computes block kb+1 while block kb is promoted.
#include "common.cuh"
#include "kernels.h"
#include "route_dev.cuh"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace moe {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 values -> two e4m3 codes (lo -> low byte), RNE, saturating.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise one 128-value group held 4 per lane by a warp: returns the
// packed codes of this lane's 4 values and the group scale (all lanes).
__device__ __forceinline__ uint32_t quant_group_warp(const float (&v)[4], float& sc) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  sc = __fdiv_rn(m, 448.0f);
  if (sc == 0.f) return 0u;
  const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc));
  const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc));
  return (uint32_t)c01 | ((uint32_t)c23 << 16);
}

// ---------------------------------------------------------- act quant ----
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
  const float v[4] = {bf16_to_f32(raw.x & 0xFFFFu), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xFFFFu),
                      bf16_to_f32(raw.y >> 16)};
  float sc;
  const uint32_t packed = quant_group_warp(v, sc);
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

struct PrefillArgs {
  LayerArgs a;
  RouteBufs rb;
  PrefillBufs pb;
  uint32_t* status;
};

// The same quantisation, with the codes and scale of token t written to the
// rows of all its routed slots (routed order: row inv[t*k + j]).  A warp
// covers four 128-column groups of one token; eight lanes per group, 16
// values per lane, 16-byte code stores.
__global__ void __launch_bounds__(256) act_quant_permute_kernel(PrefillArgs p) {
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  const int groups = a.H / 128;
  const int nq = (groups + 3) / 4;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (int64_t)a.T * nq) return;
  const int lane = threadIdx.x & 31;
  const int t = (int)(wid / nq);
  const int gi = (int)(wid % nq) * 4 + (lane >> 3);
  const bool valid = gi < groups;
  const int col = gi * 128 + (lane & 7) * 16;
  float v[16];
  float m = 0.f;
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(a.hidden + (int64_t)t * a.hidden_ld + col);
    const uint4 r0 = src[0], r1 = src[1];
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
      v[2 * i + 1] = bf16_to_f32(w[i] >> 16);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (!valid) return;
  const float sc = __fdiv_rn(m, 448.0f);
  uint32_t q[4] = {0u, 0u, 0u, 0u};
  if (sc != 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i], sc), __fdiv_rn(v[4 * i + 1], sc));
      const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i + 2], sc), __fdiv_rn(v[4 * i + 3], sc));
      q[i] = (uint32_t)c01 | ((uint32_t)c23 << 16);
    }
  }
  const uint4 qq = make_uint4(q[0], q[1], q[2], q[3]);
  for (int j = 0; j < a.k; ++j) {
    const int pos = p.rb.inv[t * a.k + j];
    if (pos < 0) continue;
    *reinterpret_cast<uint4*>(p.pb.xq + (int64_t)pos * a.H + col) = qq;
    if ((lane & 7) == 0) p.pb.xs[(int64_t)pos * groups + gi] = sc;
  }
}

// ---------------------------------------------------------- grouped GEMM --
namespace pf {
constexpr int BM = 128;            // rows (routed slots) per tile
constexpr int BN = 256;            // output columns per tile
constexpr int BK = 128;            // K block (bytes = e4m3 elements)
constexpr int NS = 4;              // shared-memory stages
constexpr int A_BYTES = BM * BK;   // 16 KiB
constexpr int B_BYTES = BN * BK;   // 32 KiB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int NEPI = 8;            // epilogue warps (two per TMEM lane quarter)
constexpr int THREADS = 32 * (2 + NEPI);
constexpr int BAR_OFF = NS * STAGE;
constexpr int XCH_OFF = BAR_OFF + 256;
constexpr int SMEM = 1024 + XCH_OFF + 2 * BM * 2 * 4;
constexpr uint32_t TMEM_COLS = 512;
}  // namespace pf

// Tile t -> (expert e, first routed row p0, valid rows, column block nb).
struct Tile {
  int e, p0, nvalid, nb;
};

__device__ __forceinline__ Tile tile_of(const PrefillArgs& p, long t, int NBT) {
  const int mi = (int)(t / NBT);
  Tile r;
  r.nb = (int)(t % NBT);
  const int* mtp = p.rb.mtp;
  int lo = 0, hi = p.a.E;   // mtp[lo] <= mi < mtp[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(mtp + mid) <= mi) lo = mid;
    else hi = mid;
  }
  r.e = lo;
  const int mt = mi - __ldg(mtp + lo);
  r.p0 = __ldg(p.rb.offsets + lo) + mt * pf::BM;
  r.nvalid = min(pf::BM, __ldg(p.rb.counts + lo) - mt * pf::BM);
  return r;
}

// 64 fp32 values times wt -> 64 bf16 (RNE), stored as 128 contiguous bytes.
__device__ __forceinline__ void store_bf16_row64(uint16_t* dst, const float (&v)[64], float wt) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * i + 2 * q] * wt, v[8 * i + 2 * q + 1] * wt);
      w[q] = *reinterpret_cast<uint32_t*>(&b);
    }
    d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// MODE 1: gate/up projection, silu(gate)*up, e4m3 h codes + scales.
// MODE 2: down projection times the slot's top-k weight -> bf16 slot rows.
template <int MODE>
// 10 warps: two SM sub-partitions hold three of them, so each thread may
// use at most 16384 / (3 * 32) -> 168 registers.
__global__ void __launch_bounds__(pf::THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        PrefillArgs p) {
  using namespace pf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + BAR_OFF);
  uint64_t* empty = full + NS;
  uint64_t* tfull = empty + NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* xfull = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull + 2);
  float* xch = reinterpret_cast<float*>(base + XCH_OFF);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NEPI);
      mbar_init(&xfull[i], NEPI);
    }
    fence_mbar_init();
    abort_flag = 0;
    tc::prefetch_tensormap(&tmA);
    tc::prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  const LayerArgs& a = p.a;
  const int K = MODE == 1 ? a.H : a.I;
  const int nkb = K / BK;
  const int NBT = MODE == 1 ? a.I / 128 : (a.H + BN - 1) / BN;
  const long total = (long)__ldg(p.rb.mtp + a.E) * NBT;

  if (warp == 0) {
    // -------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      long it = 0;
      bool ok = true;
      // L2 prefetch runs PD K blocks ahead of the shared-memory loads (across
      // tile boundaries), so the stage loads find their tiles in L2.
      constexpr int PD = 8;
      long pt = blockIdx.x;
      int pkb = 0;
      Tile ptl = pt < total ? tile_of(p, pt, NBT) : Tile{0, 0, 0, 0};
      auto prefetch_next = [&]() {
        if (pt >= total) return;
        tc::tma_prefetch_2d(&tmA, pkb * BK, ptl.p0);
        if (MODE == 1) {
          const int r0 = ptl.e * 2 * a.I + ptl.nb * 128;
          tc::tma_prefetch_2d(&tmB, pkb * BK, r0);
          tc::tma_prefetch_2d(&tmB, pkb * BK, r0 + a.I);
        } else {
          tc::tma_prefetch_2d(&tmB, pkb * BK, ptl.e * a.H + ptl.nb * BN);
        }
        if (++pkb == nkb) {
          pkb = 0;
          pt += gridDim.x;
          if (pt < total) ptl = tile_of(p, pt, NBT);
        }
      };
      for (int i = 0; i < PD; ++i) prefetch_next();
      for (long t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = tile_of(p, t, NBT);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          prefetch_next();
          const int s = (int)(it % NS);
          if (it >= NS && !mbar_wait(&empty[s], (uint32_t)((it / NS) - 1) & 1)) {
            ok = false;
            break;
          }
          uint8_t* st = base + s * STAGE;
          mbar_arrive_expect_tx(&full[s], STAGE);
          tc::tma_load_2d(st, &tmA, kb * BK, tl.p0, &full[s], pol_a);
          if (MODE == 1) {
            const int r0 = tl.e * 2 * a.I + tl.nb * 128;
            tc::tma_load_2d(st + A_BYTES, &tmB, kb * BK, r0, &full[s], pol_b);
            tc::tma_load_2d(st + A_BYTES + B_BYTES / 2, &tmB, kb * BK, r0 + a.I, &full[s], pol_b);
          } else {
            tc::tma_load_2d(st + A_BYTES, &tmB, kb * BK, tl.e * a.H + tl.nb * BN, &full[s], pol_b);
          }
        }
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok) {
        abort_flag = 1;
        raise_status(p.status, MOE_STATUS_TIMEOUT);
        for (long i = it > NS ? it - NS : 0; i < it; ++i) mbar_wait(&full[i % NS], (uint32_t)(i / NS) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, BN);
      long it = 0, j = 0;
      bool ok = true;
      for (long t = blockIdx.x; t < total && ok; t += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++it, ++j) {
          const int s = (int)(it % NS);
          const int buf = (int)(j & 1);
          if (!mbar_wait(&full[s], (uint32_t)(it / NS) & 1) ||
              (j >= 2 && !mbar_wait(&tempty[buf], (uint32_t)((j >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint8_t* st = base + s * STAGE;
          const uint32_t d = tmem + buf * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            tc::mma_f8(d, tc::sw128_desc(st + k * 32), tc::sw128_desc(st + A_BYTES + k * 32), idesc, k > 0);
          tc::commit(&empty[s]);
          tc::commit(&tfull[buf]);
        }
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok) {
        abort_flag = 1;
        raise_status(p.status, MOE_STATUS_TIMEOUT);
      }
      // the last commits must land before TMEM is released
      if (j > 0) mbar_wait(&tfull[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int eq = warp & 3;                 // TMEM lane quarter of this warp
    const int hf = (warp - 2) >> 2;          // which 64-column half of each 128-column block
    const int row = eq * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(eq * 32) << 16);
    long j = 0;
    int tcount = 0;
    for (long t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
      const Tile tl = tile_of(p, t, NBT);
      const bool rvalid = row < tl.nvalid;
      const int pos = tl.p0 + row;
      float acc0[64], acc1[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0.f;
      const uint16_t* ws0;
      const uint16_t* ws1;
      const float* as;
      bool has1 = true;
      if (MODE == 1) {
        ws0 = a.w13s + (int64_t)tl.e * a.s13_exp + (int64_t)tl.nb * a.s13_row;
        ws1 = a.w13s + (int64_t)tl.e * a.s13_exp + (int64_t)(a.I / 128 + tl.nb) * a.s13_row;
        as = p.pb.xs + (int64_t)pos * (a.H / 128);
      } else {
        const int b0 = tl.nb * 2;
        has1 = (b0 + 1) * 128 < a.H;
        ws0 = a.w2s + (int64_t)tl.e * a.s2_exp + (int64_t)b0 * a.s2_row;
        ws1 = has1 ? ws0 + a.s2_row : ws0;
        as = p.pb.hs + (int64_t)pos * (a.I / 128);
      }
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++j) {
        const float sa = rvalid ? __ldg(as + kb) : 0.f;
        const float f0 = sa * bf16_to_f32(__ldg(ws0 + kb));
        const float f1 = has1 ? sa * bf16_to_f32(__ldg(ws1 + kb)) : 0.f;
        const int buf = (int)(j & 1);
        if (!mbar_wait(&tfull[buf], (uint32_t)(j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t tb = trow + buf * BN + hf * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
          tc::tmem_ld16(tb + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc0[c * 16 + i] = fmaf(f0, v[i], acc0[c * 16 + i]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
          tc::tmem_ld16(tb + 128 + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc1[c * 16 + i] = fmaf(f1, v[i], acc1[c * 16 + i]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      if (!ok || *(volatile int*)&abort_flag) {
        abort_flag = 1;
        raise_status(p.status, MOE_STATUS_TIMEOUT);
        break;
      }
      if (MODE == 1) {
        // h = silu(gate) * up for this thread's 64 columns of the 128-block
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float g = acc0[i];
          const float h = g / (1.0f + expf(-g)) * acc1[i];
          acc0[i] = h;
          amax = fmaxf(amax, fabsf(h));
        }
        // the other half of the row's 128-group sits in warp (warp +- 4)
        const int xb = tcount & 1;
        xch[(xb * BM + row) * 2 + hf] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfull[xb]);
        if (!mbar_wait(&xfull[xb], (uint32_t)(tcount >> 1) & 1)) {
          abort_flag = 1;
          raise_status(p.status, MOE_STATUS_TIMEOUT);
          break;
        }
        amax = fmaxf(amax, xch[(xb * BM + row) * 2 + (1 - hf)]);
        const float sc = __fdiv_rn(amax, 448.0f);
        if (rvalid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t c01 = 0, c23 = 0;
            if (sc != 0.f) {
              c01 = f32x2_to_e4m3x2(__fdiv_rn(acc0[4 * i], sc), __fdiv_rn(acc0[4 * i + 1], sc));
              c23 = f32x2_to_e4m3x2(__fdiv_rn(acc0[4 * i + 2], sc), __fdiv_rn(acc0[4 * i + 3], sc));
            }
            w[i] = c01 | (c23 << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.pb.hq + (int64_t)pos * a.I + tl.nb * 128 + hf * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          if (hf == 0) p.pb.hs[(int64_t)pos * (a.I / 128) + tl.nb] = sc;
        }
      } else {
        if (rvalid) {
          const int s = p.rb.perm[pos];
          const float wt = a.wts[s];
          uint16_t* dst = p.pb.slots + (int64_t)s * a.H + tl.nb * BN + hf * 64;
          store_bf16_row64(dst, acc0, wt);
          if (has1) store_bf16_row64(dst + 128, acc1, wt);
        }
      }
    }
  }
  // ---------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------ combine ----
__global__ void __launch_bounds__(256) prefill_combine_kernel(PrefillArgs p) {
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  const int t = blockIdx.x;
  const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (n >= a.H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < a.k; ++j) {
    const int s = t * a.k + j;
    const int id = a.ids[s];
    if (id < 0 || id >= a.E) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(p.pb.slots + (int64_t)s * a.H + n);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16_to_f32(w[i] & 0xFFFFu);
      acc[2 * i + 1] += bf16_to_f32(w[i] >> 16);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(a.out + (int64_t)t * a.H + n) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ------------------------------------------------------------- launch ----
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Row-major uint8 matrix [rows, cols] (row pitch = cols bytes), boxes of
// 128 bytes x box_rows, 128-byte swizzle; rows past the end read as zero.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Kern, typename... Args>
static cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
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

cudaError_t launch_prefill(const LayerArgs& a, const RouteBufs& rb, const PrefillBufs& pb, int32_t* route_scratch,
                           uint32_t* status, int device, cudaStream_t st, int* launches) {
  PrefillArgs p{a, rb, pb, status};
  CUtensorMap mx, m13, mh, m2;
  if (!make_map(&mx, pb.xq, (uint64_t)a.S, (uint64_t)a.H, 128) ||
      !make_map(&m13, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, 128) ||
      !make_map(&mh, pb.hq, (uint64_t)a.S, (uint64_t)a.I, 128) ||
      !make_map(&m2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, pf::BN))
    return note_error(cudaErrorInvalidValue, "tensor map encode");
  cudaError_t err;
  if ((err = note_error(
           cudaFuncSetAttribute(prefill_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM),
           "prefill_gemm1 smem attribute")))
    return err;
  if ((err = note_error(
           cudaFuncSetAttribute(prefill_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM),
           "prefill_gemm2 smem attribute")))
    return err;
  const int sms = num_sms(device);
  const bool timed = stage_mark(st, 0);
  const bool pdl = !timed;
  int nl = 0;
  if ((err = launch_check(launch_route(a.ids, a.S, a.E, rb, status, route_scratch, st, &nl), st, "route")))
    return err;
  stage_mark(st, 1);
  const int64_t warps = (int64_t)a.T * ((a.H / 128 + 3) / 4);
  if ((err = launch_check(launch_ex(act_quant_permute_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, st,
                                    pdl, p),
                          st, "act_quant_permute")))
    return err;
  stage_mark(st, 2);
  if ((err = launch_check(launch_ex(prefill_gemm_kernel<1>, dim3(sms), dim3(pf::THREADS), pf::SMEM, st, pdl, mx,
                                    m13, p),
                          st, "prefill_gemm1")))
    return err;
  stage_mark(st, 3);
  if ((err = launch_check(launch_ex(prefill_gemm_kernel<2>, dim3(sms), dim3(pf::THREADS), pf::SMEM, st, pdl, mh,
                                    m2, p),
                          st, "prefill_gemm2")))
    return err;
  stage_mark(st, 4);
  if ((err = launch_check(launch_ex(prefill_combine_kernel, dim3(a.T, (a.H + 2047) / 2048), dim3(256), 0, st,
                                    pdl, p),
                          st, "prefill_combine")))
    return err;
  stage_mark(st, 5);
  *launches += 4 + nl;
  return cudaSuccess;
}

}  // namespace moe
