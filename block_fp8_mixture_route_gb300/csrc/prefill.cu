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
// Row layout: the routed slots of expert e occupy rows [128*mtp[e],
// 128*mtp[e] + count[e]) of every per-row buffer (mtp = exclusive prefix of
// ceil(count/128)), so a 128-row tile never spans two experts; the rows
// after count[e] up to the next multiple of 128 are padding whose contents
// are never read back.  pinv[s] is the row of slot s.
//
// Kernels, in stream order (chained with programmatic dependent launch):
//   route               routing lists + per-expert 128-row tile prefix
//   act_quant_permute   e4m3 codes of every token written to the rows of
//                       its routed slots, their scales K-block major
//                       (xsT[kb][row]); extra CTAs repack the bf16 weight
//                       block scales into fp32 records a tensor map can load
//   prefill_gemm<1>     tile = (128 rows, 128-column block nb of gate and
//                       the same block of up): silu*up -> e4m3 h + scales
//   prefill_gemm<2>     tile = (128 rows, 256 rows of the down projection)
//                       -> bf16 y rows
//   prefill_combine     out[t] = sum_j w[t,j] * y[pinv[t*k + j]] in j order
//
// Every operand, scale and output of the GEMMs moves by tensor-map copies
// (loads into a shared-memory ring, stores from a shared-memory staging
// tile): ordinary global loads and stores issued while bulk tensor traffic
// is in flight wait thousands of cycles on this part, so the GEMM kernels
// issue none after their prologue.
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

// Weight block scales as fp32 records of four, one per (expert, K block,
// output tile), so one 16-byte tensor-map load brings the column-block
// scales a tile needs for one K block:
//   wsc13[e][kb][p] = (scale of gate rows p*128.., of the first and of the
//                      last of up rows p*128.., 0)
//   wsc2 [e][kb][p] = (w2 scale of row block 2p, of row block 2p+1 or 0, 0, 0)
// The scale blocks of w13 are 128 rows of the stacked [gate; up] bank, so
// when I is not a multiple of 128 the up rows of one tile straddle two of
// them: up row i uses block (I + i) / 128.
__device__ void repack_weight_scales(const PrefillArgs& p, int64_t idx) {
  const LayerArgs& a = p.a;
  const int np1 = (a.I + 127) / 128, nk1 = (a.H + 127) / 128;
  const int np2 = (a.H + 255) / 256, nk2 = (a.I + 127) / 128, nrow2 = (a.H + 127) / 128;
  const int64_t n13 = (int64_t)a.E * nk1 * np1;
  const int64_t n2 = (int64_t)a.E * nk2 * np2;
  if (idx < n13) {
    const int pp = (int)(idx % np1);
    const int kb = (int)((idx / np1) % nk1);
    const int e = (int)(idx / ((int64_t)np1 * nk1));
    const uint16_t* s = a.w13s + (int64_t)e * a.s13_exp + kb;
    const int last = (2 * a.I + 127) / 128 - 1;   // last scale row of the stacked bank
    const int ua = (a.I + pp * 128) / 128, ub = min((a.I + pp * 128 + 127) / 128, last);
    const float g = bf16_to_f32(s[(int64_t)pp * a.s13_row]);
    const float u0 = bf16_to_f32(s[(int64_t)ua * a.s13_row]);
    const float u1 = bf16_to_f32(s[(int64_t)ub * a.s13_row]);
    reinterpret_cast<float4*>(p.pb.wsc13)[idx] = make_float4(g, u0, u1, 0.f);
    return;
  }
  idx -= n13;
  if (idx < n2) {
    const int pp = (int)(idx % np2);
    const int kb = (int)((idx / np2) % nk2);
    const int e = (int)(idx / ((int64_t)np2 * nk2));
    const uint16_t* s = a.w2s + (int64_t)e * a.s2_exp + kb;
    const float r0 = bf16_to_f32(s[(int64_t)(2 * pp) * a.s2_row]);
    const float r1 = 2 * pp + 1 < nrow2 ? bf16_to_f32(s[(int64_t)(2 * pp + 1) * a.s2_row]) : 0.f;
    reinterpret_cast<float4*>(p.pb.wsc2)[idx] = make_float4(r0, r1, 0.f, 0.f);
  }
}

// The activation quantisation of act_quant_kernel, with the codes of token
// t written to the rows of all its routed slots and the scales K-block
// major.  A warp covers four 128-column groups of one token; eight lanes
// per group, 16 values per lane, 16-byte code stores.  CTAs from qblocks on
// repack the weight scales instead (they read only the weights, so they do
// it before waiting for the route kernel).
__global__ void __launch_bounds__(256) act_quant_permute_kernel(PrefillArgs p, int qblocks) {
  if ((int)blockIdx.x >= qblocks) {
    repack_weight_scales(p, (int64_t)(blockIdx.x - qblocks) * blockDim.x + threadIdx.x);
    pdl_trigger();
    return;
  }
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  const int groups = (a.H + 127) / 128;   // the last one partial when H is not a multiple of 128
  const int nq = (groups + 3) / 4;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (int64_t)a.T * nq) return;
  const int lane = threadIdx.x & 31;
  const int t = (int)(wid / nq);
  const bool first = (wid % nq) == 0;
  const int gi = (int)(wid % nq) * 4 + (lane >> 3);
  const int col = gi * 128 + (lane & 7) * 16;
  const bool valid = gi < groups && col < a.H;   // H is a multiple of 16
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
    const int s = t * a.k + j;
    const int e = a.ids[s];
    if (e < 0 || e >= a.E) {
      if (first && lane == 0) p.pb.pinv[s] = -1;
      continue;
    }
    const int64_t row = (int64_t)p.rb.inv[s] - p.rb.offsets[e] + (int64_t)p.rb.mtp[e] * 128;
    *reinterpret_cast<uint4*>(p.pb.xq + row * a.H + col) = qq;
    if ((lane & 7) == 0) p.pb.xsT[(int64_t)gi * p.pb.rows + row] = sc;
    if (first && lane == 0) p.pb.pinv[s] = (int32_t)row;
  }
}

// ---------------------------------------------------------- grouped GEMM --
namespace pf {
constexpr int BM = 128;            // rows per tile
constexpr int BN = 256;            // accumulator columns per tile
constexpr int BK = 128;            // K block (bytes = e4m3 elements)
constexpr int A_BYTES = BM * BK;   // 16 KiB
constexpr int B_BYTES = BN * BK;   // 32 KiB
constexpr int STAGE = A_BYTES + B_BYTES;
// A stage of a launch whose tiles have at most 32 valid rows (no expert has
// more than 32 slots: every decode-size batch): the A tile's first 32 rows
// only, then B.  The MMA still reads 128 A rows; rows 32..127 come from the
// stage's B bytes and yield accumulator rows that lie in the expert's
// padding, which no epilogue warp finishes.
constexpr int A_SMALL = 32 * BK;   // 4 KiB
constexpr int STAGE_S = A_SMALL + B_BYTES;
constexpr int KG = 4;              // K blocks per scale group (one scale-ring entry)
constexpr int NSG = 6;             // scale-ring entries
constexpr int LEAD_G = 3;          // groups the scale loads run ahead of the operand loads
                                   // (NSG - LEAD_G >= 3: the epilogue is never more than
                                   // 2 accumulators + 5 stages, i.e. under 3 groups, behind)
constexpr int SA_BYTES = BM * KG * 4;   // activation scales of one group: [KG][BM] fp32
constexpr int SW_BYTES = KG * 16;       // weight scale records of one group: [KG][4] fp32
constexpr int NEPI = 8;            // epilogue warps (two per TMEM lane quarter)
constexpr int THREADS = 32 * (2 + NEPI);
constexpr int OUT1 = BM * 128;     // GEMM1 staging: 128 rows x 128 h codes (+ 128 fp32 scales)
constexpr int OUT2 = BM * 256 * 2; // GEMM2 staging: 128 rows x 256 bf16, pair-major (32 rows x four 64-column quarters)
constexpr uint32_t TMEM_COLS = 512;
constexpr int kSmemMax = 232448;   // opt-in shared memory per CTA
}  // namespace pf

// Stages of STAGE_S bytes that fit where ns stages of STAGE bytes lie.
__host__ __device__ inline int pf_small_stages(int ns) { return ns * pf::STAGE / pf::STAGE_S; }

// Shared-memory layout of prefill_gemm_kernel<mode> with ns stages (byte
// offsets from a 1024-aligned base; the same function on host and device).
// Every tensor-copy destination or source is 128-byte aligned.
struct PfLayout {
  uint32_t out, ring_a, ring_w, xch, bars, mtp, cnt, total;
};

__host__ __device__ inline PfLayout pf_layout(int mode, int ns, int E) {
  PfLayout L;
  uint32_t o = (uint32_t)ns * pf::STAGE;
  L.out = o;
  o += mode == 1 ? pf::OUT1 + 512 : pf::OUT2;
  L.ring_a = o;
  o += pf::NSG * pf::SA_BYTES;
  L.ring_w = o;
  o += pf::NSG * 128;
  L.xch = o;
  o += pf::BM * 2 * 4;
  L.bars = o;
  // barriers of the most stages a launch uses: the stages of STAGE_S bytes
  // in the ring, and in GEMM2 one more in the staging tile
  o += (2 * (pf_small_stages(ns) + (mode == 2)) + 2 * pf::NSG + 4) * 8 + 16;
  o = (o + 15u) & ~15u;
  L.mtp = o;
  o += 4u * (uint32_t)(E + 1);
  L.cnt = o;   // GEMM2: the experts' slot counts (rows of each expert's last tile)
  if (mode == 2) o += 4u * (uint32_t)E;
  L.total = o + 1024;   // slack for aligning the dynamic shared memory base
  return L;
}

// The tensor maps one GEMM uses: A rows (a: 128-row boxes; a32: 32-row
// boxes, for launches whose tiles have at most 32 valid rows), B rows
// (GEMM1: 3-D view of w13 so one load brings a gate block and the matching
// up block), A scales (K-block major), B scale records, and the output(s):
// GEMM1 h codes (o) and scales (os); GEMM2 y rows as 32-row boxes of four
// 64-column quarters (o: one pair of epilogue warps' rows) and as 8-row
// boxes of one quarter (os), for pairs with few valid rows.
struct PfMaps {
  CUtensorMap a, a32, b, sa, sw, o, os;
};

// Largest expert e with mtp[e] <= mi (the expert owning 128-row tile mi).
__device__ __forceinline__ int expert_of_tile(const int* mtp, int E, int mi) {
  int lo = 0, hi = E;   // mtp[lo] <= mi < mtp[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mtp[mid] <= mi) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Barrier of the two epilogue warps of TMEM lane quarter q (warps ew and
// ew ^ 4: named barrier 2 + q, 64 threads), and the same returning the OR
// of `v` over those 64 threads.
__device__ __forceinline__ void pair_sync(int q) { asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory"); }
__device__ __forceinline__ bool pair_sync_or(int q, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t"
      "setp.ne.u32 t, %2, 0;\n\t"
      "bar.red.or.pred p, %1, 64, t;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(2 + q), "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Two fp32 values in one 64-bit register (the first in the low half): the
// operand form of the paired fp32 instructions.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// acc = ff * {x0, x1} + acc on both halves with one paired FMA (each half
// rounded as fmaf would).
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t ff, uint32_t x0, uint32_t x1) {
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%2, %3};\n\tfma.rn.f32x2 %0, %1, t, %0;\n\t}"
      : "+l"(acc)
      : "l"(ff), "r"(x0), "r"(x1));
}

// 64 fp32 values (32 pairs) -> bf16 (RNE) into one 128-byte row of a
// 128-byte-swizzled staging box (16-byte chunk c of row r sits at chunk
// c ^ (r & 7)).
__device__ __forceinline__ void stage_bf16_row64(uint8_t* box, int row, const uint64_t (&v)[32]) {
  uint8_t* r = box + row * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f2lo(v[4 * c + q]), f2hi(v[4 * c + q]));
      w[q] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(r + ((c ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// A tile of a CTA pair (CTAs 2c and 2c + 1 of the grid, rank = the low bit).
// Pair tiles come in units of h = ceil(NBT / 2), one unit per 128-row M tile
// of the padded routed order (mtp[E] units in all):
//  - M tiles 2i and 2i+1 of an expert (same B): the two CTAs take one M tile
//    each and the same column block nb, so they read the same weight block
//    at about the same time and the second read finds it in L2.  The pair's
//    two units cover column blocks 0..h-1 and h..2h-1.
//  - the last M tile of an expert with an odd count (same A): both CTAs take
//    that M tile and adjacent column blocks 2w and 2w+1.
// Each CTA loads all of its own operands (its 128 A rows and its 256 B rows)
// with plain tensor-map loads into its own shared memory; nothing is written
// into the other CTA's shared memory.  A column block past NBT (odd NBT) is
// a phantom: it loads zeros past the tensors and multiplies like a real one
// but stores nothing.
struct PairTile {
  int mi, nb, e;
  bool real;
  bool ashared;   // the last, odd M tile of its expert (both CTAs take it)
};

__device__ __forceinline__ PairTile pair_tile(const int* mtp, int E, int NBT, int pt, uint32_t rank) {
  PairTile r;
  const int h = (NBT + 1) >> 1;
  const int mt = pt / h;   // unit = M tile of the padded order
  const int w = pt - mt * h;
  r.e = expert_of_tile(mtp, E, mt);
  const int j = mt - mtp[r.e];
  const int m = mtp[r.e + 1] - mtp[r.e];
  r.ashared = j >= (m & ~1);
  if (!r.ashared) {
    r.mi = mtp[r.e] + (j & ~1) + (int)rank;
    r.nb = (j & 1) * h + w;
  } else {
    r.mi = mtp[r.e] + j;
    r.nb = 2 * w + (int)rank;
  }
  r.real = r.nb < NBT;
  return r;
}

// Position in a ring of n entries: index and phase parity, advanced by one.
struct RingPos {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// MODE 1: gate/up projection, silu(gate)*up, e4m3 h codes + scales.
// MODE 2: down projection -> bf16 y rows.
// 10 warps per CTA: warp 0 issues tensor-map loads, warp 1 owns TMEM and
// issues the MMAs, warps 2..9 promote, finish and store.  CTA pair c (CTAs
// 2c and 2c + 1) takes pair tiles c, c + pairs, ... (pair_tile).  A stage
// holds a 128-row A tile (its first 32 rows when no expert has more than 32
// slots) and a 256-row B tile, both loaded by the CTA itself; it is free
// again once this CTA's MMAs have read it (one commit arrives on its empty
// barrier).
// BIAS: GEMM1 adds the optional MLP gate/up bias.  SPLIT: GEMM1 of a layer
// whose I is not a multiple of 128, where each up tile's columns take two
// weight scales (see repack_weight_scales).
template <int MODE, bool BIAS = false, bool SPLIT = false>
__global__ void __launch_bounds__(pf::THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ PfMaps m, PrefillArgs p, int ns) {
  using namespace pf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const LayerArgs& a = p.a;
  const int E = a.E;
  const PfLayout L = pf_layout(MODE, ns, E);
  // barriers of the most stages a launch can use: when no expert has more
  // than 32 slots (every decode-size batch) the ring holds stages of
  // STAGE_S bytes, and in GEMM2, where only the first pair of epilogue warps
  // then ever stages output rows, the other 48 KB of the staging tile serve
  // as one more stage
  const int nsb = pf_small_stages(ns) + (MODE == 2 ? 1 : 0);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.bars);
  uint64_t* empty = full + nsb;
  uint64_t* sfull = empty + nsb;
  uint64_t* sempty = sfull + NSG;
  uint64_t* tfull = sempty + NSG;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  float* ring_a = reinterpret_cast<float*>(base + L.ring_a);
  float* ring_w = reinterpret_cast<float*>(base + L.ring_w);
  float* xch = reinterpret_cast<float*>(base + L.xch);
  int* mtp_s = reinterpret_cast<int*>(base + L.mtp);
  int* cnt_s = reinterpret_cast<int*>(base + L.cnt);
  const uint32_t rank = blockIdx.x & 1u;
  uint8_t* outs = base + L.out;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nsb; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < NSG; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], NEPI);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NEPI);
    }
    fence_mbar_init();
    abort_flag = 0;
    tc::prefetch_tensormap(&m.a);
    tc::prefetch_tensormap(&m.a32);
    tc::prefetch_tensormap(&m.b);
    tc::prefetch_tensormap(&m.sa);
    tc::prefetch_tensormap(&m.sw);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  // GEMM1 waits for the activation codes before anything else.  GEMM2 can
  // start only once every GEMM1 CTA has passed that wait, so the route
  // kernel's tile tables are complete by then: GEMM2 reads them (through
  // L2) and prefetches its first tile's weights before waiting for the h
  // codes, and its CTAs placed on SMs that GEMM1 has already left stream
  // weights during GEMM1's last wave.
  if (MODE == 1) pdl_wait();
  auto ld_table = [](const int* q) { return MODE == 2 ? __ldcg(q) : __ldg(q); };
  // the tile tables, read once before any tensor-map traffic starts
  int over32 = 0;   // some expert has more than 32 slots
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    mtp_s[i] = ld_table(p.rb.mtp + i);
    if (MODE == 2 && i < E) {
      cnt_s[i] = ld_table(p.rb.counts + i);
      over32 |= cnt_s[i] > 32;
    } else if (i < E) {
      over32 |= ld_table(p.rb.counts + i) > 32;
    }
  }
  tc::fence_before_sync();
  over32 = __syncthreads_or(over32);
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // ring stages of this launch (the same in every CTA: all read the same
  // counts), their size, B's offset in a stage, and the shared memory of
  // stage i.  With at most 32 valid rows per tile the stages hold 32 A rows:
  // 5 stages of 32 KB of weights instead of 4 (GEMM1; GEMM2 4 + 1 instead
  // of 3 + 1)
  const bool small = !over32;
  const int nring = small ? pf_small_stages(ns) : ns;
  const int nse = nring + (MODE == 2 && small ? 1 : 0);
  const uint32_t sbytes = small ? STAGE_S : STAGE;
  const int boff = small ? A_SMALL : A_BYTES;
  auto stage_at = [&](int i) -> uint8_t* { return i < nring ? base + i * sbytes : outs + OUT2 / 4; };

  const int K = MODE == 1 ? a.H : a.I;
  const int nkb = (int)(((unsigned)K + BK - 1) / BK);   // a partial last K block reads zeros past K
  const int ngpt = (nkb + KG - 1) / KG;                 // scale groups per tile
  const int NBT = MODE == 1 ? (int)(((unsigned)a.I + 127) / 128) : (a.H + BN - 1) / BN;
  const int total = mtp_s[E] * ((NBT + 1) >> 1);   // pair tiles
  const int bx = (int)blockIdx.x >> 1, gx = (int)gridDim.x >> 1;   // pair index, pairs
  if (MODE == 2) {
    // the first tile's rows of the down projection, contiguous in w2 (a hint:
    // the ring's loads read them again)
    if (threadIdx.x == 0 && bx < total) {
      const PairTile tl = pair_tile(mtp_s, E, NBT, bx, rank);
      if (tl.real) {
        const int r0 = tl.nb * BN, nr = min(BN, a.H - r0);
        const uint8_t* src = a.w2 + ((int64_t)tl.e * a.H + r0) * a.I;
        for (int c = 0; c < nr; c += 32)
          prefetch_l2(src + (int64_t)c * a.I, (uint32_t)(min(32, nr - c) * a.I));
      }
    }
    pdl_wait();
  }
  pdl_trigger();

  if (warp == 0) {
    // -------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      // weights: evict-first when the batch routes at most 32 slots to every
      // expert (each weight block is then read by one CTA, once) so that L2
      // keeps the activation codes and outputs; the gate/up projection only
      // up to 64 experts (wide layer T = 1 / 4: 95 -> 90 / 260 -> 256 us; at
      // T = 16, 109 experts, it was slower), the down projection always
      // (T = 16: 781 -> 775 us)
      const uint64_t polb = over32 || (MODE == 1 && mtp_s[E] > 64) ? pol : l2_policy_evict_first();
      const int my_tiles = total > bx ? (total - bx + gx - 1) / gx : 0;
      const int n_groups = my_tiles * ngpt;
      int n_main = 0, n_g = 0;          // operand stages / scale groups issued
      RingPos sp, gp;
      bool ok = true;
      // scale group g of this CTA: tile g / ngpt of its list, K blocks
      // KG * (g % ngpt) ... ; issued up to LEAD_G groups ahead
      auto issue_groups = [&](int upto) -> bool {
        if (upto > n_groups) upto = n_groups;
        for (; n_g < upto; ++n_g, gp.next(NSG)) {
          if (n_g >= NSG && !mbar_wait(&sempty[gp.i], gp.ph ^ 1u)) return false;
          const int ti = n_g / ngpt, g = n_g - ti * ngpt;
          const PairTile tl = pair_tile(mtp_s, E, NBT, bx + ti * gx, rank);
          mbar_arrive_expect_tx(&sfull[gp.i], SA_BYTES + SW_BYTES);
          tc::tma_load_2d(ring_a + gp.i * (SA_BYTES / 4), &m.sa, tl.mi * BM, g * KG, &sfull[gp.i], pol);
          tc::tma_load_2d(ring_w + gp.i * 32, &m.sw, 4 * tl.nb, tl.e * nkb + g * KG, &sfull[gp.i], pol);
        }
        return true;
      };
      int ti = 0;
      for (int t = bx; t < total && ok; t += gx, ++ti) {
        const PairTile tl = pair_tile(mtp_s, E, NBT, t, rank);
        const int p0 = tl.mi * BM;
        for (int kb = 0; kb < nkb; ++kb, ++n_main, sp.next(nse)) {
          if (!issue_groups(ti * ngpt + kb / KG + 1 + LEAD_G)) {
            ok = false;
            break;
          }
          if (n_main >= nse && !mbar_wait(&empty[sp.i], sp.ph ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* st = stage_at(sp.i);
          // A: the tile's 128 rows, 16 KB (or its first 32, 4 KB); B: the
          // column block's 256 rows, 32 KB
          mbar_arrive_expect_tx(&full[sp.i], sbytes);
          tc::tma_load_2d(st, small ? &m.a32 : &m.a, kb * BK, p0, &full[sp.i], pol);
          if (MODE == 1) {   // gate block nb, then up block nb
            tc::tma_load_3d(st + boff, &m.b, kb * BK, tl.nb * 128, 2 * tl.e, &full[sp.i], polb);
            tc::tma_load_3d(st + boff + B_BYTES / 2, &m.b, kb * BK, tl.nb * 128, 2 * tl.e + 1, &full[sp.i],
                            polb);
          } else {           // rows nb * 256 .. + 255 of the expert's down projection
            tc::tma_load_2d(st + boff, &m.b, kb * BK, tl.e * a.H + tl.nb * BN, &full[sp.i], polb);
            tc::tma_load_2d(st + boff + B_BYTES / 2, &m.b, kb * BK, tl.e * a.H + tl.nb * BN + 128, &full[sp.i],
                            polb);
          }
        }
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok) {
        abort_flag = 1;
        raise_status(p.status, MOE_STATUS_TIMEOUT);
        // let the copies already issued land before the CTA goes away
        for (int i = n_main > nse ? n_main - nse : 0; i < n_main; ++i)
          mbar_wait(&full[i % nse], (uint32_t)(i / nse) & 1);
        for (int i = n_g > NSG ? n_g - NSG : 0; i < n_g; ++i) mbar_wait(&sfull[i % NSG], (uint32_t)(i / NSG) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, BN);
      int it = 0;
      RingPos sp;
      bool ok = true;
      for (int t = bx; t < total && ok; t += gx) {
        for (int kb = 0; kb < nkb; ++kb, ++it, sp.next(nse)) {
          const int buf = it & 1;
          if (!mbar_wait(&full[sp.i], sp.ph) ||
              (it >= 2 && !mbar_wait(&tempty[buf], (uint32_t)((it >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint8_t* st = stage_at(sp.i);
          const uint32_t d = tmem + buf * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            tc::mma_f8(d, tc::sw128_desc(st + k * 32), tc::sw128_desc(st + boff + k * 32), idesc, k > 0);
          tc::commit(&empty[sp.i]);
          tc::commit(&tfull[buf]);
        }
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok) {
        abort_flag = 1;
        raise_status(p.status, MOE_STATUS_TIMEOUT);
      }
      // the last commits must land before TMEM is released and the CTA goes away
      if (it > 0) mbar_wait(&tfull[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1);
      for (int i = it > nse ? it - nse : 0; i < it; ++i) mbar_wait(&empty[i % nse], (uint32_t)(i / nse) & 1);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int ew = warp - 2;
    const int eq = warp & 3;                 // TMEM lane quarter this warp may access
    const int hf = ew >> 2;                  // which 64-column half of each 128-column block
    const int row = eq * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(eq * 32) << 16);
    const bool pair_issuer = hf == 0 && lane == 0;   // one per lane quarter
    // first up column (within a tile) of the stacked bank's next scale block
    const int split = SPLIT ? 128 - a.I % 128 : 128;
    int it = 0;
    RingPos gp;
    bool ok = true;
    for (int t = bx; t < total; t += gx) {
      const PairTile tl = pair_tile(mtp_s, E, NBT, t, rank);
      const int nb = tl.nb;
      const int p0 = tl.mi * BM;
      const bool has1 = MODE == 1 || nb * BN + 128 < a.H;
      // optional MLP biases (GEMM1): lane l holds the gate and up biases of
      // this warp's column pair l, read at the tile start so that the loads
      // complete during the K loop
      float2 bg2 = make_float2(0.f, 0.f), bu2 = bg2;
      if (BIAS && nb * 128 + hf * 64 + 2 * lane < a.I) {   // columns past I keep h = 0
        const float* br = a.b13 + (int64_t)tl.e * a.b13_ld + nb * 128 + hf * 64 + 2 * lane;
        bg2 = __ldg(reinterpret_cast<const float2*>(br));
        bu2 = __ldg(reinterpret_cast<const float2*>(br + a.I));
      }
      // GEMM1: the expert's slot count (which of the tile's rows are not
      // padding), read now so that the load completes during the K loop
      const int cnt_e = MODE == 1 ? __ldg(p.rb.counts + tl.e) : cnt_s[tl.e];
      // rows of this pair of warps (lane quarter eq) before the expert's
      // padding: a pair with none skips its tile end (decode-size batches
      // have at most 8 valid rows per tile, all in quarter 0)
      const int pvalid = cnt_e - (tl.mi - mtp_s[tl.e]) * BM - eq * 32;
      const bool pany = tl.real && pvalid > 0;
      // this thread's 64 columns of each 128-column block, as 32 pairs
      uint64_t acc0[32], acc1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc0[i] = acc1[i] = 0ull;
      // promotion factors of the scale group's K blocks (g: gate / first 128
      // columns, u: up / next 128, ub: up past `split`), element 0 = the
      // current K block.  A group's factors are read together at its first K
      // block and its ring entry released at once: between two K blocks a
      // warp then touches shared memory only for the accumulator barrier,
      // each access there waiting behind the copies and MMA operand reads.
      float fg[KG], fu[KG], fub[KG];
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int sub = kb % KG;
        const int buf = it & 1;
        if (sub == 0) {
          if (*(volatile int*)&abort_flag) ok = false;
          ok = __all_sync(0xffffffffu, ok && mbar_wait(&sfull[gp.i], gp.ph));
#pragma unroll
          for (int j = 0; j < KG; ++j) {
            const float sa = ok ? ring_a[gp.i * (SA_BYTES / 4) + j * BM + row] : 0.f;
            const float4 w = ok ? reinterpret_cast<const float4*>(ring_w + gp.i * 32)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
            fg[j] = sa * w.x;
            fu[j] = sa * w.y;
            fub[j] = SPLIT ? sa * w.z : 0.f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[gp.i]);
          gp.next(NSG);
        } else {
#pragma unroll
          for (int j = 0; j + 1 < KG; ++j) {
            fg[j] = fg[j + 1];
            fu[j] = fu[j + 1];
            fub[j] = fub[j + 1];
          }
        }
        const float f0 = fg[0], f1 = fu[0], f1b = fub[0];
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&tfull[buf], (uint32_t)(it >> 1) & 1));
        if (ok) {
          tc::fence_after_sync();
          const uint32_t tb = trow + buf * BN + hf * 64;
          const uint64_t ff0 = f2pack(f0, f0), ff1 = f2pack(f1, f1);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tc::tmem_ld16x2_raw(tb + c * 16, tb + 128 + c * 16, r);
            // up columns from `split` on lie in the next scale block of the stacked bank
            const uint64_t ffu = SPLIT && hf * 64 + c * 16 >= split ? f2pack(f1b, f1b) : ff1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              ffma2(acc0[c * 8 + i], ff0, r[2 * i], r[2 * i + 1]);
              ffma2(acc1[c * 8 + i], ffu, r[16 + 2 * i], r[16 + 2 * i + 1]);
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      bool stop;
      if (MODE == 1) {
        if (pany) {
          // h = silu(gate) * up for this thread's 64 columns of the 128-block.
          // silu(g) = g / (1 + e^-g) with the fast exponential and division:
          // an IEEE division here takes its slow path whenever e^-g overflows
          // (every strongly negative gate value), which made this loop cost
          // more than the whole K loop of a tile.  h feeds a quantiser, and
          // both approximations are within a few fp32 ulps (a denominator
          // past 2^126 gives 0, the limit silu takes there anyway).
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float g0 = f2lo(acc0[i]), g1 = f2hi(acc0[i]);
            float u0 = f2lo(acc1[i]), u1 = f2hi(acc1[i]);
            if (BIAS) {
              g0 += __shfl_sync(0xffffffffu, bg2.x, i);
              g1 += __shfl_sync(0xffffffffu, bg2.y, i);
              u0 += __shfl_sync(0xffffffffu, bu2.x, i);
              u1 += __shfl_sync(0xffffffffu, bu2.y, i);
            }
            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            acc0[i] = f2pack(h0, h1);
            amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
          }
          // the other half of the row's 128-group is held by warp ew ^ 4: the
          // two warps of lane quarter eq exchange, stage and store their 32
          // rows by themselves (no barrier among all eight epilogue warps)
          xch[row * 2 + hf] = amax;
          if (pair_issuer) tc::bulk_wait_read0();   // the pair's previous stores have left its staging rows
          pair_sync(eq);
          amax = fmaxf(amax, xch[row * 2 + (1 - hf)]);
          const float sc = __fdiv_rn(amax, 448.0f);
          // code = e4m3(h * (1 / scale)): one IEEE reciprocal per group instead
          // of a division per value
          const float inv = sc != 0.f ? __frcp_rn(sc) : 0.f;
          uint8_t* orow = outs + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int b = 8 * i + 2 * u;   // pairs b, b + 1 = values 16 i + 4 u .. + 3
              const uint32_t c01 = f32x2_to_e4m3x2(f2lo(acc0[b]) * inv, f2hi(acc0[b]) * inv);
              const uint32_t c23 = f32x2_to_e4m3x2(f2lo(acc0[b + 1]) * inv, f2hi(acc0[b + 1]) * inv);
              w[u] = c01 | (c23 << 16);
            }
            const int c = hf * 4 + i;
            *reinterpret_cast<uint4*>(orow + ((c ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (hf == 0) reinterpret_cast<float*>(outs + OUT1)[row] = sc;
          tc::fence_proxy_async_smem();
        }
        stop = pair_sync_or(eq, !ok || *(volatile int*)&abort_flag);
        if (pair_issuer && !stop && pany) {
          tc::tma_store_2d(&m.o, outs + eq * 32 * 128, nb * 128, p0 + eq * 32);
          tc::tma_store_2d(&m.os, outs + OUT1 + eq * 32 * 4, p0 + eq * 32, nb);
          tc::bulk_commit();
        }
      } else {
        // staging tile pair-major: the 32 rows of lane quarter eq, then
        // column quarter q (output columns nb*256 + 64 q ..), 4 KB each, so
        // that the two warps of the quarter stage and store their rows by
        // themselves, one box of 32 rows x 256 columns (quarters past H are
        // clipped by the tensor map)
        uint8_t* pst = outs + eq * (OUT2 / 4);
        if (pany) {
          if (pair_issuer) tc::bulk_wait_read0();   // the pair's previous stores have left its staging rows
          pair_sync(eq);
          stage_bf16_row64(pst + hf * (OUT2 / 16), row & 31, acc0);
          if (has1) stage_bf16_row64(pst + (2 + hf) * (OUT2 / 16), row & 31, acc1);
          tc::fence_proxy_async_smem();
        }
        stop = pair_sync_or(eq, !ok || *(volatile int*)&abort_flag);
        if (pair_issuer && !stop && pany) {
          // rows past the expert's slots are padding no combine reads: a
          // pair whose rows are all padding stages and stores nothing, one
          // with at most 8 valid rows (the decode-size batches) stores one
          // 8-row box per quarter
          const int valid = pvalid;
          if (valid > 8) {
            tc::tma_store_3d(&m.o, pst, 0, p0 + eq * 32, nb * 4);
            tc::bulk_commit();
          } else if (valid > 0) {
            for (int q = 0; q < 4 && (nb * 4 + q) * 64 < a.H; ++q)
              tc::tma_store_3d(&m.os, pst + q * (OUT2 / 16), 0, p0 + eq * 32, nb * 4 + q);
            tc::bulk_commit();
          }
        }
      }
      if (stop) {
        if (lane == 0) {
          abort_flag = 1;
          raise_status(p.status, MOE_STATUS_TIMEOUT);
        }
        break;
      }
    }
    if (pair_issuer) tc::bulk_wait0();
  }
  // ---------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------ combine ----
template <bool BIAS>
__global__ void __launch_bounds__(256) prefill_combine_kernel(PrefillArgs p) {
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  const int t = blockIdx.x;
  const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (n >= a.H) return;
  // slots in chunks of 8: the chunk's rows and weights, then all its row
  // loads, then the sums in slot order (the loads are in flight together)
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    const int64_t s0 = (int64_t)t * a.k + j0;
    int row[8];
    float w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      row[q] = j0 + q < a.k ? p.pb.pinv[s0 + q] : -1;
      w[q] = j0 + q < a.k ? a.wts[s0 + q] : 0.f;
    }
    uint4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = row[q] >= 0 ? *reinterpret_cast<const uint4*>(p.pb.ys + (int64_t)row[q] * a.H + n) : make_uint4(0, 0, 0, 0);
    if (BIAS) {
      // optional down-projection bias: out += w[t,j] * (y + b2[e_j])
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (row[q] < 0) continue;
        const float* br = a.b2 + (int64_t)a.ids[s0 + q] * a.b2_ld + n;
        const float4 b0 = *reinterpret_cast<const float4*>(br), b1 = *reinterpret_cast<const float4*>(br + 4);
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(w[q], bf16_to_f32(u[i] & 0xFFFFu) + bb[2 * i], acc[2 * i]);
          acc[2 * i + 1] = fmaf(w[q], bf16_to_f32(u[i] >> 16) + bb[2 * i + 1], acc[2 * i + 1]);
        }
      }
      continue;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (row[q] < 0) continue;
      const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w[q], bf16_to_f32(u[i] & 0xFFFFu), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w[q], bf16_to_f32(u[i] >> 16), acc[2 * i + 1]);
      }
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

// ------------------------------------------------- activation code copy ----
// Token t's codes and scales as the GEMMs read them: from the row of one of
// its routed slots (slot t mod k, else the next valid one).  A token with no
// valid slot has no row and is left untouched.
__global__ void __launch_bounds__(128) prefill_act_codes_kernel(PrefillArgs p) {
  const LayerArgs& a = p.a;
  const int t = blockIdx.x;
  int64_t row = -1;
  for (int jj = 0; jj < a.k && row < 0; ++jj) row = p.pb.pinv[(int64_t)t * a.k + (t + jj) % a.k];
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(p.pb.xq + row * a.H);
  uint4* dst = reinterpret_cast<uint4*>(a.dbg_codes + (int64_t)t * a.H);
  for (int i = threadIdx.x; i < a.H / 16; i += blockDim.x) dst[i] = src[i];
  const int nkb = (a.H + 127) / 128;
  for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x)
    a.dbg_scales[(int64_t)t * nkb + kb] = p.pb.xsT[(int64_t)kb * p.pb.rows + row];
}

cudaError_t launch_prefill_act_codes(const LayerArgs& a, const PrefillBufs& pb, cudaStream_t st) {
  PrefillArgs p{a, RouteBufs{}, pb, nullptr};
  prefill_act_codes_kernel<<<a.T, 128, 0, st>>>(p);
  return cudaGetLastError();
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

// Row-major 2-D tensor [rows, cols] of `esize`-byte elements, rows `pitch`
// bytes apart, copied in boxes of box_cols x box_rows; parts of a box
// outside the tensor read as zero and are not written by stores.
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t rows,
                     uint64_t cols, uint64_t pitch, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  (void)esize;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// w13 [E, 2I, H] viewed as [2E][I][H] (x = K byte, y = row within a gate or
// up half, z = 2e for gate, 2e + 1 for up): a box of 128 x 128 x 1 is one
// 128-row block of expert e's gate (z = 2e) or up (z = 2e + 1) rows.
static bool make_map_w13(CUtensorMap* m, const void* base, int E, int I, int H) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)I, 2 * (cuuint64_t)E};
  const cuuint64_t strides[2] = {(cuuint64_t)H, (cuuint64_t)I * H};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ys [rows, H] bf16 viewed as [H/64][rows][64] (x = column within a 64-column
// quarter, y = row, z = quarter), stored from 128-byte-swizzled staging
// quarters of 32 rows: a box of 64 x 32 x 4 is 32 rows x 256 columns (four
// 4 KB quarters); a box of 64 x 8 x 1 is 8 rows of one quarter (one 1 KB
// swizzle atom).
static bool make_map_ys(CUtensorMap* m, const void* base, uint64_t rows, int H, uint32_t box_rows = 128,
                        uint32_t box_quarters = 4) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, rows, (cuuint64_t)(H / 64)};
  const cuuint64_t strides[2] = {2 * (cuuint64_t)H, 128};
  const cuuint32_t box[3] = {64, box_rows, box_quarters};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch `pairs` CTA pairs (2 * pairs CTAs; the pair of a CTA is its grid
// index with the low bit cleared).
template <typename Kern, typename... Args>
static cudaError_t launch_pairs(Kern kernel, int pairs, size_t smem, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(pf::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// CTA pairs that can be resident at once (the persistent grid), per device
// and GEMM.
template <typename Kern>
static int resident_pairs(Kern kernel, int device, int mode, size_t smem) {
  static std::mutex mu;
  static int cache[64][2][2];   // [device][mode - 1] -> {smem, pairs}
  std::lock_guard<std::mutex> lk(mu);
  int* c = cache[device & 63][mode - 1];
  if (c[0] == (int)smem && c[1] > 0) return c[1];
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, pf::THREADS, smem) != cudaSuccess) {
    cudaGetLastError();
    per_sm = 0;
  }
  c[0] = (int)smem;
  c[1] = per_sm * num_sms(device) / 2;
  return c[1];
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

// Stages that fit in shared memory for this GEMM (0 if even two do not).
static int pick_stages(int mode, int E) {
  for (int ns = 4; ns >= 2; --ns)
    if (pf_layout(mode, ns, E).total <= (uint32_t)pf::kSmemMax) return ns;
  return 0;
}

int64_t prefill_rows(int64_t S, int E) {
  const int64_t g = S < E ? S : E;
  const int64_t r = (S + 127 * g + 127) / 128 * 128;
  return r > 128 ? r : 128;
}

cudaError_t launch_prefill(const LayerArgs& a, const RouteBufs& rb, const PrefillBufs& pb, int32_t* route_scratch,
                           uint32_t* status, int device, cudaStream_t st, int* launches) {
  PrefillArgs p{a, rb, pb, status};
  const uint64_t R = (uint64_t)pb.rows;
  const uint64_t np1 = (a.I + 127) / 128, nk1 = (a.H + 127) / 128, np2 = (a.H + 255) / 256,
                 nk2 = (a.I + 127) / 128;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  PfMaps g1, g2;
  bool ok = make_map(&g1.a, U8, 1, pb.xq, R, a.H, a.H, 128, 128, true) &&
            make_map(&g1.a32, U8, 1, pb.xq, R, a.H, a.H, 128, 32, true) &&
            make_map_w13(&g1.b, a.w13, a.E, a.I, a.H) &&
            make_map(&g1.sa, F32, 4, pb.xsT, nk1, R, 4 * R, 128, pf::KG, false) &&
            make_map(&g1.sw, F32, 4, pb.wsc13, (uint64_t)a.E * nk1, 4 * np1, 16 * np1, 4, pf::KG, false) &&
            make_map(&g1.o, U8, 1, pb.hq, R, a.I, a.I, 128, 32, true) &&
            make_map(&g1.os, F32, 4, pb.hsT, nk2, R, 4 * R, 32, 1, false);
  ok = ok && make_map(&g2.b, U8, 1, a.w2, (uint64_t)a.E * a.H, a.I, a.I, 128, pf::BN / 2, true) &&
       make_map(&g2.sa, F32, 4, pb.hsT, nk2, R, 4 * R, 128, pf::KG, false) &&
       make_map(&g2.sw, F32, 4, pb.wsc2, (uint64_t)a.E * nk2, 4 * np2, 16 * np2, 4, pf::KG, false) &&
       make_map_ys(&g2.o, pb.ys, R, a.H, 32, 4) && make_map_ys(&g2.os, pb.ys, R, a.H, 8, 1);
  if (!ok) return note_error(cudaErrorInvalidValue, "tensor map encode");
  // GEMM2 reads the h codes in 128-row tiles, or 32-row ones when no tile
  // has more valid rows (GEMM1 stores them in 32-row boxes, one per pair of
  // epilogue warps)
  if (!make_map(&g2.a, U8, 1, pb.hq, R, a.I, a.I, 128, 128, true) ||
      !make_map(&g2.a32, U8, 1, pb.hq, R, a.I, a.I, 128, 32, true))
    return note_error(cudaErrorInvalidValue, "tensor map encode");
  const int ns1 = pick_stages(1, a.E), ns2 = pick_stages(2, a.E);
  if (!ns1 || !ns2) return note_error(cudaErrorNotSupported, "prefill shared memory");
  const int sm1 = (int)pf_layout(1, ns1, a.E).total, sm2 = (int)pf_layout(2, ns2, a.E).total;
  // the gate/up projection with the optional MLP bias compiled in or out
  const bool split = a.I % 128 != 0;
  auto gemm1 = a.b13 ? (split ? prefill_gemm_kernel<1, true, true> : prefill_gemm_kernel<1, true, false>)
                     : (split ? prefill_gemm_kernel<1, false, true> : prefill_gemm_kernel<1, false, false>);
  cudaError_t err;
  if ((err = note_error(
           set_max_smem((const void*)gemm1, sm1),
           "prefill_gemm1 smem attribute")))
    return err;
  if ((err = note_error(
           set_max_smem((const void*)prefill_gemm_kernel<2>, sm2),
           "prefill_gemm2 smem attribute")))
    return err;
  const int sms = num_sms(device);
  int cl1 = resident_pairs(gemm1, device, 1, (size_t)sm1);
  int cl2 = resident_pairs(prefill_gemm_kernel<2>, device, 2, (size_t)sm2);
  cl1 = cl1 < sms / 2 ? cl1 : sms / 2;
  cl2 = cl2 < sms / 2 ? cl2 : sms / 2;
  if (cl1 < 1 || cl2 < 1) return note_error(cudaErrorNotSupported, "prefill CTA pairs do not fit");
  const bool timed = stage_mark(st, 0);
  const bool pdl = !timed;
  int nl = 0;
  if ((err = launch_check(launch_route(a.ids, a.S, a.E, rb, status, route_scratch, st, &nl), st, "route")))
    return err;
  stage_mark(st, 1);
  const int64_t warps = (int64_t)a.T * (((a.H + 127) / 128 + 3) / 4);
  const int qblocks = (int)((warps + 7) / 8);
  const int64_t nrep = (int64_t)a.E * (nk1 * np1 + nk2 * np2);
  const int rblocks = (int)((nrep + 255) / 256);
  if ((err = launch_check(launch_ex(act_quant_permute_kernel, dim3((unsigned)(qblocks + rblocks)), dim3(256), 0,
                                    st, pdl, p, qblocks),
                          st, "act_quant_permute")))
    return err;
  stage_mark(st, 2);
  if ((err = launch_check(launch_pairs(gemm1, cl1, (size_t)sm1, st, pdl, g1, p, ns1), st,
                          "prefill_gemm1")))
    return err;
  stage_mark(st, 3);
  if ((err = launch_check(launch_pairs(prefill_gemm_kernel<2>, cl2, (size_t)sm2, st, pdl, g2, p, ns2), st,
                          "prefill_gemm2")))
    return err;
  stage_mark(st, 4);
  auto combine = a.b2 ? prefill_combine_kernel<true> : prefill_combine_kernel<false>;
  if ((err = launch_check(launch_ex(combine, dim3(a.T, (a.H + 2047) / 2048), dim3(256), 0, st, pdl, p), st,
                          "prefill_combine")))
    return err;
  stage_mark(st, 5);
  *launches += 4 + nl;
  return cudaSuccess;
}

}  // namespace moe
