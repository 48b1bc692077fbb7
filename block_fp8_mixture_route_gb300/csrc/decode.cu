// decode.cu -- the decode (W8A16) path of the block-FP8 MoE layer.
//
// With few tokens, only a handful of experts receive any slot, and the
// layer is bound by reading the routed experts' weights (fp8-moe-gather
// page, Problem).  This path reads only those experts (the gathered-expert
// combine, same page, The fix).  Their e4m3 rows are streamed from HBM into
// shared memory with large bulk (TMA) copies of whole rows, widened in
// registers (exact: FreeToken PR #662, PR body), and each bf16 block scale
// is applied once per 128-wide K block to an fp32 partial sum; h =
// silu(gate) * up stays fp32 for the down projection ("the down projection
// in fp32", fp8-moe-gather page, The fix).
//
// Kernels, in stream order (chained with programmatic dependent launch):
//   decode_prep    CTA 0: routing lists; CTAs 1..T: f16 copy of each token
//                  scaled by a power of two 2^-s_t (max |x_t| in [2^14, 2^15))
//   decode_gemm1   gate/up projection of every routed (expert, R-row-pair)
//                  unit with mma.sync m16n8k16 (f16 x f16 -> fp32), the four
//                  consumer warps splitting K; fused silu(gate)*up epilogue
//                  -> h fp32 [S, I] in routed order
//   decode_gemm2   down projection of every routed (expert, R2-row) unit
//                  with mma.sync on a two-term f16 split of the fp32 h
//                  (about 22 significant bits), times the slot's top-k
//                  weight -> ybuf fp32 [S, H] in slot order
//   decode_combine out[t] = sum_j ybuf[t*k + j] in j order -> bf16
//
// Work split: the units of all routed experts form one list; CTA c of G
// takes the contiguous range [c*U/G, (c+1)*U/G), so every SM streams the
// same number of weight bytes whatever the routing.  Within a CTA, units of
// one expert share that expert's activation rows (x or h), loaded once per
// (expert, pass of up to SPP slots).  Two groups of four consumer warps take
// alternate units (one group's latency hides behind the other's work); the
// four warps of a group split the unit's K blocks and one of them sums the
// partials.
//
// Copy sizes: one SM's bulk-copy engine needs copies of several KiB to move
// data near the HBM rate (small copies are dominated by a fixed cost per
// copy), so every weight copy here is a block of whole rows of 8-32 KiB.
#include "common.cuh"
#include "kernels.h"
#include "decode_mma.cuh"
#include "route_dev.cuh"

#include <algorithm>

namespace moe {

// Launch-time configuration of the two streaming kernels (host computed).
struct StreamCfg {
  int R;        // rows (GEMM1: row pairs) per unit before halving for balance
  int NS;       // ring stages
  int SB;       // bytes per ring stage
  int SPP;      // slots per pass
  int XB;       // bytes of one activation buffer
  int XP;       // activation row pitch in the buffer (bytes)
  int HBB;      // bytes of one converted-h buffer (GEMM2)
  int HP;       // converted-h row pitch (bytes)
  int V;        // floats per lane in the cross-warp reduction
  int red_off, abuf_off, hb_off, ring_off, smem;
};

struct DecodeArgs {
  LayerArgs a;
  RouteBufs rb;
  DecodeBufs db;
  uint32_t* status;
  StreamCfg c1, c2;
};

constexpr int kMaxNS = 12;
constexpr int kGroups = 2;             // consumer groups taking alternate units
constexpr int kGW = 4;                 // warps per group (they split K)
constexpr int kNWC = kGroups * kGW;    // consumer warps
constexpr int kThreads = 32 * (kNWC + 1);
constexpr int kSmemLimit = 232448;
// Weight copies issued before the wait for the previous kernel.  A bulk
// copy's issue blocks while the SM's copy engine is busy, so copies issued
// early also delay the activation (x or h) copy behind them, which the first
// unit needs as much as its weights: only the first two go out early.
constexpr int kPreIssue = 2;

// ------------------------------------------------------------- prep ----
// ACT8: W8A8 activations (per-group e4m3 codes and scales); W8A16 otherwise.
template <bool ACT8>
__global__ void __launch_bounds__(1024) decode_prep_kernel(DecodeArgs p) {
  extern __shared__ int smem_prep[];
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  if (blockIdx.x == 0) {
    route_block(a.ids, a.S, a.E, p.rb, p.status, smem_prep);
    return;
  }
  // token t: f16 copy scaled so that max |x_t| * 2^-s lands in [2^14, 2^15).
  // Each thread reads its chunks of 8 values once (16-byte loads; at least
  // 256 threads and H <= 8192 make at most 4 chunks) and keeps them for the
  // conversion.
  constexpr int kMaxChunks = 4;
  __shared__ float wmax[32];
  const int t = blockIdx.x - 1;
  const uint16_t* x = a.hidden + (int64_t)t * a.hidden_ld;
  float v[kMaxChunks][8];
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int i0 = (c * (int)blockDim.x + threadIdx.x) * 8;
    if (i0 < a.H) {
      const uint4 r = *reinterpret_cast<const uint4*>(x + i0);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[c][2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu);
        v[c][2 * j + 1] = bf16_bits_to_f32(w[j] >> 16);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[c][j]));
    }
  }
  if (ACT8) {
    // W8A8: per 128-column group (16 chunks, held by 16 consecutive
    // threads) scale = amax / 448 and code = e4m3_rne_satfinite(x / scale),
    // both IEEE fp32 divisions; the copy holds the codes' values (exact in
    // f16) and the scales go to xs.  No token-wide exponent: xexp = 0.
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int i0 = (c * (int)blockDim.x + threadIdx.x) * 8;
      const bool valid = i0 < a.H;
      float gm = 0.f;
      if (valid) {
#pragma unroll
        for (int j = 0; j < 8; ++j) gm = fmaxf(gm, fabsf(v[c][j]));
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      if (valid) {
        const float sc = __fdiv_rn(gm, 448.0f);
        uint32_t o4[4], q4[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint16_t q = sc != 0.f ? e4m3x2_from_f32(__fdiv_rn(v[c][2 * j], sc), __fdiv_rn(v[c][2 * j + 1], sc))
                                       : (uint16_t)0;
          o4[j] = e4m3x2_to_f16x2(q);
          q4[j >> 1] |= (uint32_t)q << (16 * (j & 1));
        }
        *reinterpret_cast<uint4*>(p.db.xh + (int64_t)t * a.H + i0) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        if ((threadIdx.x & 15) == 0) p.db.xs[(int64_t)t * ((a.H + 127) / 128) + i0 / 128] = sc;
        if (a.dbg_codes) {   // moe_fp8_block_forward_act_codes: the codes and scales as quantised here
          *reinterpret_cast<uint2*>(a.dbg_codes + (int64_t)t * a.H + i0) = make_uint2(q4[0], q4[1]);
          if ((threadIdx.x & 15) == 0) a.dbg_scales[(int64_t)t * ((a.H + 127) / 128) + i0 / 128] = sc;
        }
      }
    }
    if (threadIdx.x == 0) p.db.xexp[t] = 0;
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, wmax[i]);
  int s = 0;
  if (m > 0.f) {
    int ex;
    frexpf(m, &ex);      // m = f * 2^ex, f in [0.5, 1)
    s = (ex - 1) - 14;   // floor(log2 m) - 14
  }
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int i0 = (c * (int)blockDim.x + threadIdx.x) * 8;
    if (i0 < a.H) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(ldexpf(v[c][2 * j], -s), ldexpf(v[c][2 * j + 1], -s));
        o[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(p.db.xh + (int64_t)t * a.H + i0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (threadIdx.x == 0) p.db.xexp[t] = s;
}

// Shared-memory layout common to both streaming kernels.
struct Smem {
  uint64_t* full;     // [kMaxNS] ring stage landed (tx)
  uint64_t* empty;    // [kMaxNS] ring stage consumed (kGW arrivals: the consuming group)
  uint64_t* afull;    // [2] activation buffer landed (tx)
  uint64_t* aempty;   // [2] activation buffer released (kNWC arrivals)
  uint64_t* hbfull;   // [2] converted h written (kNWC arrivals)
  uint64_t* hbfree;   // [2] converted h released (kNWC arrivals)
  uint64_t* rfull;    // [kGroups][2] cross-warp partials written (kGW arrivals)
  uint64_t* rempty;   // [kGroups][2] cross-warp partials read (1 arrival)
  float* red;         // [kGroups][2][kGW][32][V]
  uint8_t* abuf;
  uint8_t* hb;
  uint8_t* ring;      // [NS][SB]
};

__device__ __forceinline__ Smem smem_layout(uint8_t* base, const StreamCfg& c) {
  Smem s;
  uint64_t* b = reinterpret_cast<uint64_t*>(base);
  s.full = b;
  s.empty = b + kMaxNS;
  s.afull = b + 2 * kMaxNS;
  s.aempty = s.afull + 2;
  s.hbfull = s.aempty + 2;
  s.hbfree = s.hbfull + 2;
  s.rfull = s.hbfree + 2;
  s.rempty = s.rfull + 2 * kGroups;
  s.red = reinterpret_cast<float*>(base + c.red_off);
  s.abuf = base + c.abuf_off;
  s.hb = base + c.hb_off;
  s.ring = base + c.ring_off;
  return s;
}

__device__ __forceinline__ void smem_init(const Smem& s, int NS) {
  for (int i = 0; i < NS; ++i) {
    mbar_init(&s.full[i], 1);
    mbar_init(&s.empty[i], kGW);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&s.afull[i], 1);
    mbar_init(&s.aempty[i], kNWC);
    mbar_init(&s.hbfull[i], kNWC);
    mbar_init(&s.hbfree[i], kNWC);
  }
  for (int i = 0; i < 2 * kGroups; ++i) {
    mbar_init(&s.rfull[i], kGW);
    mbar_init(&s.rempty[i], 1);
  }
  fence_mbar_init();
}

// The CTA's units, walked entry by entry of a work list and, within an
// entry, pass by pass (a pass covers up to SPP of the entry's slots), so
// that each (expert, pass) activation load is shared by all units of the
// segment.  The gate/up projection walks one entry per routed expert; the
// down projection a per-pass list (one entry per pass), so that an expert
// with many slots weighs in its split as its passes over the weights do.
// Producer and consumers walk the same sequence; ring stage m goes to
// consumer group m % 2.
struct Walk {
  long u, ue;          // next segment start, range end
  int upe;             // units per list entry
  const int4* list;    // the work list
  int d, e, off, ne;   // current entry: expert, first routed position, slots
  int ep;              // passes over this expert's weights in the whole list
  long seg_b, seg_e;   // current segment [seg_b, seg_e)
  int passes;
};

__device__ __forceinline__ bool walk_next_segment(const DecodeArgs& p, Walk& w, int SPP) {
  (void)p;   // the list is the walk's own
  if (w.u >= w.ue) return false;
  w.d = (int)(w.u / w.upe);
  w.seg_b = w.u;
  w.seg_e = min(w.ue, (long)(w.d + 1) * w.upe);
  const int4 m = __ldg(w.list + w.d);
  w.e = m.x;
  w.off = m.y;
  w.ne = m.z;
  w.ep = m.w;
  w.passes = (w.ne + SPP - 1) / SPP;
  w.u = w.seg_e;
  return true;
}

// Weight copies: evict-first for an expert read once; the default policy
// where the list reads it again (later passes, often on a neighbouring SM
// shortly after), so that the repeat can find it in L2.
__device__ __forceinline__ uint64_t weight_policy(const Walk& w, uint64_t once, uint64_t again) {
  return w.ep > 1 ? again : once;
}

// Rows per unit: halved only while there are fewer units than SMs (the
// count of routed experts D is only known on the device).  Larger units
// stream better than more SMs each holding small ones: requiring 6 units per
// SM instead made the decode workload 4% slower, and 25% slower at T=1.
__device__ __forceinline__ int balanced_rows(int R, int min_rows, int rows_total, int D, int G) {
  while (R > min_rows && (long)D * (rows_total / R) < (long)G) R >>= 1;
  return R;
}

// Cross-warp sum of a group's K-split partials through shared memory.
// Every warp of the group deposits V floats per lane; the group's first
// warp (the leader) waits for all of them and returns the totals in tot.
// Double-buffered by the group's unit parity; every wait is bounded.
// Returns false on a timeout.
template <int V>
__device__ __forceinline__ bool group_reduce(const Smem& S, int gr, int wq, int lane, int ml, const float (&part)[V],
                                             float (&tot)[V]) {
  const int rb = ml & 1;
  uint64_t* rf = &S.rfull[gr * 2 + rb];
  uint64_t* re = &S.rempty[gr * 2 + rb];
  if (ml >= 2 && !warp_wait(re, ((ml >> 1) - 1) & 1, lane)) return false;
  float* dst = S.red + (((gr * 2 + rb) * kGW + wq) * 32 + lane) * V;
#pragma unroll
  for (int i = 0; i < V; ++i) dst[i] = part[i];
  __syncwarp();
  if (lane == 0) mbar_arrive(rf);
  if (wq != 0) return true;
  if (!warp_wait(rf, (ml >> 1) & 1, lane)) return false;
#pragma unroll
  for (int i = 0; i < V; ++i) tot[i] = 0.f;
#pragma unroll
  for (int w = 0; w < kGW; ++w) {
    const float* src = S.red + (((gr * 2 + rb) * kGW + w) * 32 + lane) * V;
#pragma unroll
    for (int i = 0; i < V; ++i) tot[i] += src[i];
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(re);
  return true;
}

// GEMM1 unit, K slice of KW blocks per warp (sa[j][kk]: the activation
// scale of the lane's slot 2c + j in K block kb0 + kk, 1 in W8A16 mode, so
// that the products there are exact): the warp first copies all of
// its weight bytes of the unit from the ring stage into registers (16 bytes
// per lane per 64-wide chunk and row) and releases the stage at once, so the
// stage is held only for those loads, not for the MMAs.  The arrive has
// release semantics and so orders the shared-memory reads before the
// producer's next copy into the stage.
template <int KW, bool RAG>
__device__ __forceinline__ void gemm1_unit_regs(const uint8_t* arow, const uint8_t* brow, const uint8_t* xrow,
                                                int kb0, int K, bool has_w, bool has_x, float sgl, float sul,
                                                const float (&sa)[2][4], uint64_t* empty_bar, int lane,
                                                float (&acc)[4]) {
  uint4 wa[2 * KW], wb[2 * KW];
#pragma unroll
  for (int i = 0; i < 2 * KW; ++i) {
    const int kk = (kb0 + (i >> 1)) * 128 + (i & 1) * 64;
    const bool in = has_w && (!RAG || kk < K);   // RAG: a 64-wide chunk past K is zero
    wa[i] = in ? lds128(arow + kk) : make_uint4(0, 0, 0, 0);
    wb[i] = in ? lds128(brow + kk) : make_uint4(0, 0, 0, 0);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = (kb0 + j) * 128 + ch * 64;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (has_x && (!RAG || kk < K)) {
        x0 = lds128(xrow + 2 * kk);
        x1 = lds128(xrow + 2 * kk + 16);
      }
      chunk_mma(b0, b1, wa[2 * j + ch], wb[2 * j + ch], x0, x1);
    }
    const float sg = __shfl_sync(0xffffffffu, sgl, j);
    const float su = __shfl_sync(0xffffffffu, sul, j);
    acc[0] = fmaf(sg * sa[0][j], b0[0] + b1[0], acc[0]);
    acc[1] = fmaf(sg * sa[1][j], b0[1] + b1[1], acc[1]);
    acc[2] = fmaf(su * sa[0][j], b0[2] + b1[2], acc[2]);
    acc[3] = fmaf(su * sa[1][j], b0[3] + b1[3], acc[3]);
  }
}

#define MOE_FAIL()                              \
  do {                                          \
    abort_flag = 1;                             \
    raise_status(p.status, MOE_STATUS_TIMEOUT); \
    return;                                     \
  } while (0)

// ------------------------------------------------------------ GEMM1 ----
// Unit: routed expert e, row pairs [i0, i0+R) (R <= 8).  A ring stage holds
// the R gate rows and the R up rows, whole (two contiguous bulk copies of
// R*H bytes).  The m16 MMA tile takes gate rows as tile rows 0..R-1 and up
// rows as tile rows 8..8+R-1, so each lane ends with gate and up of the same
// row pair.  The four warps of a group split the unit's K blocks; the
// group's leader sums the partials and applies silu(gate)*up.
// ACT8: W8A8 (the activation rows are e4m3 code values with per-group
// scales); W8A16 otherwise.
template <bool ACT8, bool BIAS, bool RAG>
__global__ void __launch_bounds__(kThreads, 1) decode_gemm1_kernel(DecodeArgs p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamCfg& cfg = p.c1;
  const Smem S = smem_layout(smem, cfg);
  __shared__ int abort_flag;
  __shared__ uint32_t ebits[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    smem_init(S, cfg.NS);
    abort_flag = 0;
  }
  __syncthreads();
  pdl_trigger();

  // The producer finds the routed experts itself (from the ids, an input)
  // and starts the weight stream before the prep kernel has finished; the
  // consumers, which need its activation rows and routing lists, wait for it.
  const LayerArgs& a = p.a;
  ExpertBits eb;
  int D;
  if (warp == kNWC) {
    D = expert_bits(a.ids, a.S, a.E, ebits, lane, eb);
  } else {
    pdl_wait();
    D = *p.rb.nd;
  }
  const int R = balanced_rows(cfg.R, 1, a.I, D, gridDim.x);
  const int upe = a.I / R;
  const long U = (long)D * upe;
  Walk wk;
  wk.u = U * blockIdx.x / gridDim.x;
  wk.ue = U * (blockIdx.x + 1) / gridDim.x;
  wk.upe = upe;
  wk.list = p.rb.meta;   // one entry per routed expert, its passes inside
  const int NS = cfg.NS, SPP = cfg.SPP;
  const int rowb = R * a.H;   // bytes of R whole rows

  if (warp == kNWC) {
    // ------------------------------------------------ producer warp
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    int m = 0, gen = 0;
    bool ok = true;
    // weight copies of the first units (of the range's first expert) go out
    // before the wait for the prep kernel
    int pre = 0;
    if (wk.u < wk.ue) {
      const int d0 = (int)(wk.u / upe);
      const int e0 = expert_select(eb, d0, lane);
      const long n = min((long)kPreIssue, min(wk.ue, (long)(d0 + 1) * upe) - wk.u);
      if (lane == 0 && e0 >= 0)
        for (long i = 0; i < n; ++i) {
          if (i == a.dbg_drop_stage - 1) continue;   // failure-detection test: this stage never comes
          const int i0 = (int)((wk.u + i) % upe) * R;
          const uint8_t* gsrc = a.w13 + ((int64_t)e0 * 2 * a.I + i0) * a.H;
          mbar_arrive_expect_tx(&S.full[i], 2 * rowb);
          bulk_g2s(S.ring + i * cfg.SB, gsrc, rowb, &S.full[i], pol_w);
          bulk_g2s(S.ring + i * cfg.SB + rowb, gsrc + (int64_t)a.I * a.H, rowb, &S.full[i], pol_w);
        }
      pre = e0 >= 0 ? (int)n : 0;
    }
    pdl_wait();
    while (ok && walk_next_segment(p, wk, SPP)) {
      for (int pass = 0; pass < wk.passes && ok; ++pass, ++gen) {
        const int nx = min(SPP, wk.ne - pass * SPP);
        const int b = gen & 1;
        // activation rows of this pass (lane j: the token of slot j), issued
        // right after the pass's first weight copy, so that the routed-position
        // lookup is off the path to the first weight bytes
        const int tok = lane < nx ? p.rb.perm[wk.off + pass * SPP + lane] / a.k : 0;
        bool x_sent = false;
        auto send_x = [&]() {
          x_sent = true;
          if (gen >= 2) ok = warp_wait(&S.aempty[b], ((gen >> 1) - 1) & 1, lane);
          if (!ok) return;
          if (lane == 0) mbar_arrive_expect_tx(&S.afull[b], nx * 2 * a.H);
          __syncwarp();
          if (lane < nx)
            bulk_g2s(S.abuf + b * cfg.XB + lane * cfg.XP, p.db.xh + (int64_t)tok * a.H, 2 * a.H, &S.afull[b],
                     pol_x);
        };
        for (long u = wk.seg_b; u < wk.seg_e && ok; ++u, ++m) {
          const int slot = m % NS;
          if (m >= pre) {
          if (m >= NS) ok = warp_wait(&S.empty[slot], ((m / NS) - 1) & 1, lane);
          if (!ok) break;
          if (lane == 0 && m != a.dbg_drop_stage - 1) {   // (the failure-detection test drops one)
            const int i0 = (int)(u % upe) * R;
            const uint8_t* gsrc = a.w13 + ((int64_t)wk.e * 2 * a.I + i0) * a.H;
            mbar_arrive_expect_tx(&S.full[slot], 2 * rowb);
            bulk_g2s(S.ring + slot * cfg.SB, gsrc, rowb, &S.full[slot], pol_w);
            bulk_g2s(S.ring + slot * cfg.SB + rowb, gsrc + (int64_t)a.I * a.H, rowb, &S.full[slot], pol_w);
          }
          __syncwarp();
          }
          if (!x_sent) send_x();
        }
        if (!x_sent && ok) send_x();
        if (*(volatile int*)&abort_flag) ok = false;
      }
    }
    if (!ok && lane == 0) {
      abort_flag = 1;
      raise_status(p.status, MOE_STATUS_TIMEOUT);
      // let the copies already issued land before the CTA exits
      const int issued = max(m, pre);
      for (int mm = max(0, issued - NS); mm < issued; ++mm) mbar_wait(&S.full[mm % NS], (mm / NS) & 1);
      for (int gg = max(0, gen - 1); gg <= gen; ++gg) mbar_wait(&S.afull[gg & 1], (gg >> 1) & 1);
    }
    return;
  }

  // -------------------------------------------------- consumer warps
  const int gr = warp / kGW, wq = warp % kGW;
  const int g = lane >> 2, c = lane & 3;
  const int nkb = (a.H + 127) >> 7;   // RAG: the last K block is a single 64-wide chunk
  const int kb0 = wq * nkb / kGW, kb1 = (wq + 1) * nkb / kGW;
  const bool has_w = g < R;
  int m = 0, gen = 0;
  while (walk_next_segment(p, wk, SPP)) {
    for (int pass = 0; pass < wk.passes; ++pass, ++gen) {
      const int nx = min(SPP, wk.ne - pass * SPP);
      const int b = gen & 1;
      const bool has_x = g < nx;
      const uint8_t* xrow = S.abuf + b * cfg.XB + g * cfg.XP + c * 32;
      // epilogue data (group leaders): routed positions and token scales of slots 2c, 2c+1
      const int pos0 = wk.off + pass * SPP + 2 * c;
      int sx[2] = {0, 0};
      if (wq == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (2 * c + j < nx) sx[j] = p.db.xexp[p.rb.perm[pos0 + j] / a.k];
      }
      // W8A8: the activation group scales of slots 2c, 2c+1 over this warp's
      // K blocks (1 in W8A16 mode and for slots past the pass)
      float sa[2][4] = {{1.f, 1.f, 1.f, 1.f}, {1.f, 1.f, 1.f, 1.f}};
      int stok[2] = {-1, -1};
      if (ACT8) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (2 * c + j < nx) {
            stok[j] = p.rb.perm[pos0 + j] / a.k;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kb0 + kk < kb1) sa[j][kk] = p.db.xs[(int64_t)stok[j] * nkb + kb0 + kk];
          }
        }
      }
      // this warp's block scales of unit u (lane j: K block kb0 + j).  Loaded a
      // unit ahead: ordinary global loads wait thousands of cycles while the
      // weight stream is in flight, so each group fetches its next unit's
      // scales while it computes the current one.
      auto scales_of = [&](long u, float& g_, float& u_) {
        const int i0u = (int)(u % upe) * R;
        const uint16_t* gr_ = a.w13s + (int64_t)wk.e * a.s13_exp + (int64_t)(i0u / 128) * a.s13_row;
        const uint16_t* ur_ = a.w13s + (int64_t)wk.e * a.s13_exp + (int64_t)((a.I + i0u) / 128) * a.s13_row;
        g_ = kb0 + lane < kb1 ? bf16_bits_to_f32(__ldg(gr_ + kb0 + lane)) : 0.f;
        u_ = kb0 + lane < kb1 ? bf16_bits_to_f32(__ldg(ur_ + kb0 + lane)) : 0.f;
      };
      long next_u = wk.seg_b + ((gr - m) & 1);   // this group's first unit of the pass
      float next_g = 0.f, next_up = 0.f;
      if (next_u < wk.seg_e) scales_of(next_u, next_g, next_up);
      if (!warp_wait(&S.afull[b], (gen >> 1) & 1, lane)) MOE_FAIL();
      for (long u = wk.seg_b; u < wk.seg_e; ++u, ++m) {
        if ((m & 1) != gr) continue;   // the other group's unit
        const int i0 = (int)(u % upe) * R;
        // optional MLP biases of this lane's gate and up row, read now so the
        // loads complete while the unit computes
        float bgv = 0.f, buv = 0.f;
        if (BIAS && wq == 0 && has_w) {
          const float* br = a.b13 + (int64_t)wk.e * a.b13_ld + i0 + g;
          bgv = __ldg(br);
          buv = __ldg(br + a.I);
        }
        float sgl, sul;
        if (u == next_u) {
          sgl = next_g;
          sul = next_up;
        } else {
          scales_of(u, sgl, sul);
        }
        next_u = u + 2;
        if (next_u < wk.seg_e) scales_of(next_u, next_g, next_up);
        const int slot = m % NS;
        if (!warp_wait(&S.full[slot], (m / NS) & 1, lane)) MOE_FAIL();
        const uint8_t* st = S.ring + slot * cfg.SB;
        const uint8_t* arow = st + g * a.H + c * 16;
        const uint8_t* brow = arow + rowb;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int kw = kb1 - kb0;
        if (kw >= 1 && kw <= 4) {
          switch (kw) {
            case 1: gemm1_unit_regs<1, RAG>(arow, brow, xrow, kb0, a.H, has_w, has_x, sgl, sul, sa, &S.empty[slot], lane, acc); break;
            case 2: gemm1_unit_regs<2, RAG>(arow, brow, xrow, kb0, a.H, has_w, has_x, sgl, sul, sa, &S.empty[slot], lane, acc); break;
            case 3: gemm1_unit_regs<3, RAG>(arow, brow, xrow, kb0, a.H, has_w, has_x, sgl, sul, sa, &S.empty[slot], lane, acc); break;
            default: gemm1_unit_regs<4, RAG>(arow, brow, xrow, kb0, a.H, has_w, has_x, sgl, sul, sa, &S.empty[slot], lane, acc); break;
          }
        } else {
#pragma unroll 1
        for (int kb = kb0; kb < kb1; ++kb) {
          float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int kk = kb * 128 + ch * 64;
            uint4 wa = make_uint4(0, 0, 0, 0), wb = wa, x0 = wa, x1 = wa;
            const bool in = !RAG || kk < a.H;
            if (has_w && in) {
              wa = lds128(arow + kk);
              wb = lds128(brow + kk);
            }
            if (has_x && in) {
              x0 = lds128(xrow + 2 * kk);
              x1 = lds128(xrow + 2 * kk + 16);
            }
            chunk_mma(b0, b1, wa, wb, x0, x1);
          }
          // the 128-wide K block is complete: apply its scales once
          const float sg = __shfl_sync(0xffffffffu, sgl, kb - kb0);
          const float su = __shfl_sync(0xffffffffu, sul, kb - kb0);
          float a0 = 1.f, a1 = 1.f;
          if (ACT8) {
            if (stok[0] >= 0) a0 = __ldg(p.db.xs + (int64_t)stok[0] * nkb + kb);
            if (stok[1] >= 0) a1 = __ldg(p.db.xs + (int64_t)stok[1] * nkb + kb);
          }
          acc[0] = fmaf(sg * a0, b0[0] + b1[0], acc[0]);
          acc[1] = fmaf(sg * a1, b0[1] + b1[1], acc[1]);
          acc[2] = fmaf(su * a0, b0[2] + b1[2], acc[2]);
          acc[3] = fmaf(su * a1, b0[3] + b1[3], acc[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        }
        float tot[4];
        if (!group_reduce<4>(S, gr, wq, lane, m >> 1, acc, tot)) MOE_FAIL();
        if (wq == 0 && has_w) {
          // lane: gate/up of row pair i0+g for slots 2c, 2c+1
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (2 * c + j < nx) {
              float gv = ldexpf(tot[j], sx[j]);
              float uv = ldexpf(tot[2 + j], sx[j]);
              if (BIAS) {
                gv += bgv;
                uv += buv;
              }
              p.db.h[(int64_t)(pos0 + j) * a.I + i0 + g] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
          }
        }
        if (*(volatile int*)&abort_flag) return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.aempty[b]);
    }
  }
}

// ------------------------------------------------------------ GEMM2 ----
// Unit: routed expert e, output rows [n0, n0+R2) (R2 in {16, 32, 64}, so a
// unit lies in one 128-row scale block); MT = R2/16 m16 tiles.  A ring stage
// holds the R2 whole rows (one contiguous copy of R2*I bytes).
//
// The pass's fp32 h rows (up to 4 slots, consecutive in routed order) land
// in a raw buffer; the consumers turn each slot's row into two f16 terms
// with a per-slot power-of-two scale 2^-s (max |h| * 2^-s in [2^14, 2^15)):
// hi = f16(h * 2^-s), lo = f16(h * 2^-s - hi), which together carry about
// 22 significant bits.  They form the eight MMA columns [hi_0..hi_3,
// lo_0..lo_3]; y_slot = (C[:, slot] + C[:, 4 + slot]) * 2^s.  The four warps
// of a group split K; the leader sums the partials and writes y times the
// slot's top-k weight.
template <int MT, bool RAG>
__device__ void gemm2_unit_compute(const uint8_t* st, const uint8_t* hbrow, int I, int kb0, int kb1, int lane,
                                   bool has_b, float sl, float (&acc)[MT][4]) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb) {
    float b0[MT][4], b1[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) b0[t][i] = b1[t][i] = 0.f;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = kb * 128 + ch * 64;
      if (RAG && kk >= I) break;   // the last K block is a single 64-wide chunk
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (has_b) {
        x0 = lds128(hbrow + 2 * kk);
        x1 = lds128(hbrow + 2 * kk + 16);
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint8_t* ra = st + (t * 16 + g) * I + kk + c * 16;
        const uint4 wa = lds128(ra);
        const uint4 wb = lds128(ra + 8 * I);
        chunk_mma(b0[t], b1[t], wa, wb, x0, x1);
      }
    }
    const float s = __shfl_sync(0xffffffffu, sl, kb - kb0);
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][i] = fmaf(s, b0[t][i] + b1[t][i], acc[t][i]);
  }
}

// The same with the warp's weight bytes first copied into registers and the
// ring stage released before the MMAs (KW K blocks per warp, MT * KW <= 4).
template <int MT, int KW, bool RAG>
__device__ __forceinline__ void gemm2_unit_regs(const uint8_t* st, const uint8_t* hbrow, int I, int kb0, int lane,
                                                bool has_b, float sl, uint64_t* empty_bar, float (&acc)[MT][4]) {
  const int g = lane >> 2, c = lane & 3;
  uint4 wa[MT][2 * KW], wb[MT][2 * KW];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int i = 0; i < 2 * KW; ++i) {
      const int kk = (kb0 + (i >> 1)) * 128 + (i & 1) * 64;
      const bool in = !RAG || kk < I;   // RAG: a 64-wide chunk past K is zero
      const uint8_t* ra = st + (t * 16 + g) * I + kk + c * 16;
      wa[t][i] = in ? lds128(ra) : make_uint4(0, 0, 0, 0);
      wb[t][i] = in ? lds128(ra + 8 * I) : make_uint4(0, 0, 0, 0);
    }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    float b0[MT][4], b1[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) b0[t][i] = b1[t][i] = 0.f;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = (kb0 + j) * 128 + ch * 64;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (has_b && (!RAG || kk < I)) {
        x0 = lds128(hbrow + 2 * kk);
        x1 = lds128(hbrow + 2 * kk + 16);
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) chunk_mma(b0[t], b1[t], wa[t][2 * j + ch], wb[t][2 * j + ch], x0, x1);
    }
    const float s = __shfl_sync(0xffffffffu, sl, j);
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][i] = fmaf(s, b0[t][i] + b1[t][i], acc[t][i]);
  }
}

// ROWS: the four warps of a group take the unit's 16-row tiles (warp wq
// rows wq*16 ..) over the whole K, so there is no cross-warp sum and every
// warp writes its own rows (used when a unit of 64 rows fits a stage).
// Otherwise the warps split K and the group's first warp sums and writes.
template <int MT, bool ROWS, bool RAG>
__device__ void gemm2_consumers(const DecodeArgs& p, const Smem& S, Walk& wk, int R2, int upe, int warp, int lane,
                                int* abort_flag) {
  const LayerArgs& a = p.a;
  const StreamCfg& cfg = p.c2;
  const int NS = cfg.NS, SPP = cfg.SPP;
  const int gr = warp / kGW, wq = warp % kGW;
  const int g = lane >> 2, c = lane & 3;
  const int nkb = (a.I + 127) >> 7;   // RAG: the last K block is a single 64-wide chunk
  const int kb0 = ROWS ? 0 : wq * nkb / kGW, kb1 = ROWS ? nkb : (wq + 1) * nkb / kGW;
  const bool lead = ROWS || wq == 0;   // writes outputs
  // this warp's share of the h conversion
  const int ck0 = warp * a.I / kNWC, ck1 = (warp + 1) * a.I / kNWC;
  int m = 0, gen = 0;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_status(p.status, MOE_STATUS_TIMEOUT);
  };
  while (walk_next_segment(p, wk, SPP)) {
    for (int pass = 0; pass < wk.passes; ++pass, ++gen) {
      const int nh = min(SPP, wk.ne - pass * SPP);
      const int b = gen & 1;
      uint8_t* hb = S.hb + b * cfg.HBB;
      const uint8_t* hraw = S.abuf;
      // epilogue data (output-writing warps): slots 2c, 2c+1 (lanes with c < 2)
      int so[2] = {-1, -1};
      float wo[2] = {0.f, 0.f};
      if (lead && c < 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (2 * c + j < nh) {
            so[j] = p.rb.perm[wk.off + pass * SPP + 2 * c + j];
            wo[j] = a.wts[so[j]];
          }
        }
      }
      // this warp's block scales of unit u (lane j: K block kb0 + j), loaded a
      // unit ahead (see the GEMM1 consumers)
      auto scales_of = [&](long u) -> float {
        if (ROWS && wq * 16 >= R2) return 0.f;   // no rows for this warp in a narrow unit
        const int n0u = (int)(u % upe) * R2 + (ROWS ? wq * 16 : 0);
        const uint16_t* sr = a.w2s + (int64_t)wk.e * a.s2_exp + (int64_t)(n0u / 128) * a.s2_row;
        return kb0 + lane < kb1 ? bf16_bits_to_f32(__ldg(sr + kb0 + lane)) : 0.f;
      };
      long next_u = wk.seg_b + ((gr - m) & 1);   // this group's first unit of the pass
      float next_s = next_u < wk.seg_e ? scales_of(next_u) : 0.f;
      if (!warp_wait(&S.afull[0], gen & 1, lane)) return fail();
      // per-slot scale exponents from the row maxima (every warp computes them)
      int es[4] = {0, 0, 0, 0};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (s < nh) {
          float mx = 0.f;
          for (int k = lane * 4; k < a.I; k += 128) {
            const float4 v = lds_f4(hraw + (s * a.I + k) * 4);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (mx > 0.f) {
            int ex;
            frexpf(mx, &ex);
            es[s] = (ex - 1) - 14;
          }
        }
      }
      if (gen >= 2 && !warp_wait(&S.hbfree[b], ((gen >> 1) - 1) & 1, lane)) return fail();
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (s >= nh) break;
        for (int k = ck0 + 2 * lane; k < ck1; k += 64) {
          const float2 v = *reinterpret_cast<const float2*>(hraw + (s * a.I + k) * 4);
          const float v0 = ldexpf(v.x, -es[s]), v1 = ldexpf(v.y, -es[s]);
          const __half2 hi = __floats2half2_rn(v0, v1);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
          *reinterpret_cast<__half2*>(hb + s * cfg.HP + 2 * k) = hi;
          *reinterpret_cast<__half2*>(hb + (4 + s) * cfg.HP + 2 * k) = lo;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.aempty[0]);
        mbar_arrive(&S.hbfull[b]);
      }
      if (!warp_wait(&S.hbfull[b], (gen >> 1) & 1, lane)) return fail();
      const bool has_b = (g & 3) < nh;
      const uint8_t* hbrow = hb + g * cfg.HP + c * 32;
      int esl[2] = {0, 0};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int s = (2 * c + j) & 3;
        esl[j] = s == 0 ? es[0] : (s == 1 ? es[1] : (s == 2 ? es[2] : es[3]));
      }
      for (long u = wk.seg_b; u < wk.seg_e; ++u, ++m) {
        if ((m & 1) != gr) continue;
        const int n0 = (int)(u % upe) * R2 + (ROWS ? wq * 16 : 0);
        float sl;
        if (u == next_u) {
          sl = next_s;
        } else {
          sl = scales_of(u);
        }
        next_u = u + 2;
        if (next_u < wk.seg_e) next_s = scales_of(next_u);
        const int slot = m % NS;
        if (!warp_wait(&S.full[slot], (m / NS) & 1, lane)) return fail();
        if (ROWS && wq * 16 >= R2) {   // a unit narrower than four tiles: nothing for this warp
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.empty[slot]);
          continue;
        }
        float acc[MT][4];
        const int kw = kb1 - kb0;
        const uint8_t* st = S.ring + slot * cfg.SB + (ROWS ? wq * 16 * a.I : 0);
        bool done = true;
        if constexpr (MT == 1) {
          switch (kw) {
            case 1: gemm2_unit_regs<1, 1, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            case 2: gemm2_unit_regs<1, 2, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            case 3: gemm2_unit_regs<1, 3, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            case 4: gemm2_unit_regs<1, 4, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            default: done = false;
          }
        } else if constexpr (MT == 2) {
          switch (kw) {
            case 1: gemm2_unit_regs<2, 1, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            case 2: gemm2_unit_regs<2, 2, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc); break;
            default: done = false;
          }
        } else {
          if (kw == 1) gemm2_unit_regs<MT, 1, RAG>(st, hbrow, a.I, kb0, lane, has_b, sl, &S.empty[slot], acc);
          else done = false;
        }
        if (!done) {
          gemm2_unit_compute<MT, RAG>(st, hbrow, a.I, kb0, kb1, lane, has_b, sl, acc);
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.empty[slot]);
        }
        float part[MT * 4], tot[MT * 4];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) part[t * 4 + i] = acc[t][i];
        if constexpr (ROWS) {
#pragma unroll
          for (int i = 0; i < MT * 4; ++i) tot[i] = part[i];
        } else {
          if (!group_reduce<MT * 4>(S, gr, wq, lane, m >> 1, part, tot)) return fail();
        }
        if (lead) {
          // columns 2c, 2c+1: hi terms on lanes c < 2, lo terms on lanes c >= 2
#pragma unroll
          for (int i = 0; i < MT * 4; ++i) tot[i] += __shfl_xor_sync(0xffffffffu, tot[i], 2);
          if (c < 2) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                if (so[j] >= 0) {
                  const int n = n0 + t * 16 + g;
                  p.db.ybuf[(int64_t)so[j] * a.H + n] = ldexpf(tot[t * 4 + j], esl[j]) * wo[j];
                  p.db.ybuf[(int64_t)so[j] * a.H + n + 8] = ldexpf(tot[t * 4 + 2 + j], esl[j]) * wo[j];
                }
              }
            }
          }
        }
        if (*(volatile int*)abort_flag) return;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.hbfree[b]);
    }
  }
}

template <bool RAG>
__global__ void __launch_bounds__(kThreads, 1) decode_gemm2_kernel(DecodeArgs p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamCfg& cfg = p.c2;
  const Smem S = smem_layout(smem, cfg);
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    smem_init(S, cfg.NS);
    abort_flag = 0;
  }
  __syncthreads();
  pdl_trigger();

  // The routing lists come from the prep kernel, which had completed before
  // the kernel this one follows (GEMM1) released its dependents, so they can
  // be read before waiting for GEMM1; only h needs the wait.
  const LayerArgs& a = p.a;
  const int D = p.rb.nd[1];
  const int R2 = balanced_rows(cfg.R, 16, a.H, D, gridDim.x);
  const int upe = a.H / R2;
  const long U = (long)D * upe;
  Walk wk;
  wk.u = U * blockIdx.x / gridDim.x;
  wk.ue = U * (blockIdx.x + 1) / gridDim.x;
  wk.upe = upe;
  wk.list = p.rb.vmeta;
  const int NS = cfg.NS, SPP = cfg.SPP;
  const int tileb = R2 * a.I;

  if (warp == kNWC) {
    const uint64_t pol_once = l2_policy_evict_first();
    const uint64_t pol_again = l2_policy_evict_normal();
    const uint64_t pol_h = l2_policy_evict_last();
    int m = 0, gen = 0;
    bool ok = true;
    // weight copies of the first units (first pass of the first segment) go
    // out before the wait for GEMM1, so they overlap its tail
    int pre = 0;
    {
      Walk w0 = wk;
      if (walk_next_segment(p, w0, SPP)) {
        const uint64_t pol_w = weight_policy(w0, pol_once, pol_again);
        const long n = min((long)kPreIssue, w0.seg_e - w0.seg_b);
        if (lane == 0)
          for (long i = 0; i < n; ++i) {
            const int n0 = (int)((w0.seg_b + i) % upe) * R2;
            mbar_arrive_expect_tx(&S.full[i], tileb);
            bulk_g2s(S.ring + i * cfg.SB, a.w2 + ((int64_t)w0.e * a.H + n0) * a.I, tileb, &S.full[i], pol_w);
          }
        pre = (int)n;
      }
    }
    pdl_wait();
    while (ok && walk_next_segment(p, wk, SPP)) {
      const uint64_t pol_w = weight_policy(wk, pol_once, pol_again);
      for (int pass = 0; pass < wk.passes && ok; ++pass, ++gen) {
        const int nh = min(SPP, wk.ne - pass * SPP);
        // the raw h buffer is single: wait until every consumer has converted the previous pass
        if (gen >= 1) ok = warp_wait(&S.aempty[0], (gen - 1) & 1, lane);
        if (!ok) break;
        if (lane == 0) {
          // the pass's h rows are consecutive in routed order: one copy
          mbar_arrive_expect_tx(&S.afull[0], nh * 4 * a.I);
          bulk_g2s(S.abuf, p.db.h + (int64_t)(wk.off + pass * SPP) * a.I, nh * 4 * a.I, &S.afull[0], pol_h);
        }
        __syncwarp();
        for (long u = wk.seg_b; u < wk.seg_e && ok; ++u, ++m) {
          if (m < pre) continue;   // copied before the wait
          const int slot = m % NS;
          if (m >= NS) ok = warp_wait(&S.empty[slot], ((m / NS) - 1) & 1, lane);
          if (!ok) break;
          if (lane == 0) {
            const int n0 = (int)(u % upe) * R2;
            mbar_arrive_expect_tx(&S.full[slot], tileb);
            bulk_g2s(S.ring + slot * cfg.SB, a.w2 + ((int64_t)wk.e * a.H + n0) * a.I, tileb, &S.full[slot], pol_w);
          }
          __syncwarp();
        }
        if (*(volatile int*)&abort_flag) ok = false;
      }
    }
    if (!ok && lane == 0) {
      abort_flag = 1;
      raise_status(p.status, MOE_STATUS_TIMEOUT);
      const int issued = max(m, pre);
      for (int mm = max(0, issued - NS); mm < issued; ++mm) mbar_wait(&S.full[mm % NS], (mm / NS) & 1);
      if (gen > 0) mbar_wait(&S.afull[0], (gen - 1) & 1);
    }
    return;
  }
  pdl_wait();
  if (cfg.V == 0) {
    gemm2_consumers<1, true, RAG>(p, S, wk, R2, upe, warp, lane, &abort_flag);
  } else {
    switch (R2 / 16) {
      case 1: gemm2_consumers<1, false, RAG>(p, S, wk, R2, upe, warp, lane, &abort_flag); break;
      case 2: gemm2_consumers<2, false, RAG>(p, S, wk, R2, upe, warp, lane, &abort_flag); break;
      default: gemm2_consumers<4, false, RAG>(p, S, wk, R2, upe, warp, lane, &abort_flag); break;
    }
  }
}

// ---------------------------------------------------------- combine ----
template <bool BIAS>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs p) {
  pdl_wait();
  pdl_trigger();
  const LayerArgs& a = p.a;
  const int t = blockIdx.x;
  const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (n >= a.H) return;
  // slots in chunks of 8: the chunk's ids, then all its row loads, then the
  // sums in slot order (the loads are in flight together instead of one
  // dependent id + row pair after another)
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    const int64_t s0 = (int64_t)t * a.k + j0;
    bool use[8];
    int id[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      id[q] = j0 + q < a.k ? a.ids[s0 + q] : -1;
      use[q] = id[q] >= 0 && id[q] < a.E;
    }
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = use[q] ? *reinterpret_cast<const float4*>(p.db.ybuf + (s0 + q) * a.H + n) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (BIAS) {
      // optional down-projection bias: slot j adds w[t,j] * b2[e_j] after its
      // weighted y (the per-slot rows already hold w[t,j] * y)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!use[q]) continue;
        const float w = a.wts[s0 + q];
        const float4 bv = *reinterpret_cast<const float4*>(a.b2 + (int64_t)id[q] * a.b2_ld + n);
        acc.x += v[q].x;
        acc.y += v[q].y;
        acc.z += v[q].z;
        acc.w += v[q].w;
        acc.x = fmaf(w, bv.x, acc.x);
        acc.y = fmaf(w, bv.y, acc.y);
        acc.z = fmaf(w, bv.z, acc.z);
        acc.w = fmaf(w, bv.w, acc.w);
      }
      continue;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (!use[q]) continue;
      acc.x += v[q].x;
      acc.y += v[q].y;
      acc.z += v[q].z;
      acc.w += v[q].w;
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (int64_t)t * a.H + n) = pk;
}

// ----------------------------------------------------------- launch ----
template <typename K>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                              const DecodeArgs& args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

static inline int align128(int x) { return (x + 127) / 128 * 128; }

// Place the regions of one streaming kernel: barriers, reduction area,
// activation buffer(s), converted-h buffers, ring.
static bool place(StreamCfg& c, int nabuf) {
  c.red_off = 1024;
  c.abuf_off = align128(c.red_off + kGroups * 2 * kGW * 32 * c.V * 4);
  c.hb_off = c.abuf_off + nabuf * c.XB;
  c.ring_off = c.hb_off + 2 * c.HBB;
  c.smem = c.ring_off + c.NS * c.SB;
  return c.smem <= kSmemLimit;
}

// GEMM1: R row pairs per unit with R*H <= 16 KiB (whole-row copies of 8-16
// KiB keep the per-SM bulk-copy engine near its peak); as many ring stages
// as fit next to two activation buffers of up to 8 slots.
static bool config_gemm1(int H, StreamCfg& c) {
  c.R = H <= 2048 ? 8 : (H <= 4096 ? 4 : 2);
  c.SB = align128(2 * c.R * H);
  c.XP = 2 * H + 16;          // == 16 mod 128: conflict-free B fragment loads
  c.HBB = 0;
  c.HP = 0;
  c.V = 4;
  // bytes in flight per SM set the streaming rate, so the ring comes first:
  // the most stages that fit next to activation buffers of at least 4 slots
  for (c.NS = kMaxNS; c.NS >= 3; --c.NS)
    for (int spp = 8; spp >= 4; --spp) {
      c.SPP = spp;
      c.XB = align128(spp * c.XP);
      if (place(c, 2)) return true;
    }
  for (int spp = 3; spp >= 1; --spp) {
    c.SPP = spp;
    c.XB = align128(spp * c.XP);
    for (c.NS = kMaxNS; c.NS >= 3; --c.NS)
      if (place(c, 2)) return true;
  }
  return false;
}

// GEMM2: R2 rows per unit (16, 32 or 64) with R2*I near 16 KiB; a raw h
// buffer for 4 slots and two converted buffers of 8 f16 rows.
static bool config_gemm2(int H, int I, StreamCfg& c) {
  if (64 * I <= 32768 && H >= 64) {
    // row-split units: 64 rows (one 16-row tile per warp of a group), no
    // cross-warp reduction (V = 0 selects this form in the kernel)
    c.R = 64;
    c.V = 0;
  } else {
    c.R = 16;
    while (c.R < 64 && 2 * c.R * I <= 16384 && 2 * c.R <= H) c.R *= 2;
    c.V = 4 * (c.R / 16);
  }
  c.SB = align128(c.R * I);
  c.XP = 4 * I;
  c.HP = 2 * I + 16;          // == 16 mod 128: conflict-free B fragment loads
  c.HBB = align128(8 * c.HP);
  c.SPP = 4;
  c.XB = align128(c.SPP * c.XP);
  for (c.NS = kMaxNS; c.NS >= 2; --c.NS)
    if (place(c, 1)) return true;
  return false;
}

// Decode layer shapes: H and I multiples of 64 (a K dimension that is not a
// multiple of 128 ends in one 64-wide chunk) and at least 128.
static bool decode_shape(int H, int I) { return H % 64 == 0 && I % 64 == 0 && H >= 128 && I >= 128; }

int decode_unit_rows(int H) {
  StreamCfg c;
  return config_gemm1(H, c) ? c.R : 0;
}

int decode_ring_stages(int H, int I) {
  StreamCfg c1, c2;
  if (!decode_shape(H, I) || !config_gemm1(H, c1) || !config_gemm2(H, I, c2)) return 0;
  return c1.NS;
}

bool decode_supported(int H, int I) {
  StreamCfg c1, c2;
  return decode_shape(H, I) && config_gemm1(H, c1) && config_gemm2(H, I, c2);
}

cudaError_t launch_decode(const LayerArgs& a, const RouteBufs& rb, const DecodeBufs& db, uint32_t* status,
                          int device, cudaStream_t st, int* launches) {
  if (a.decode_kernel == MOE_DECODE_KERNEL_FUSED && db.counters && fused_decode_ok(a.T, a.k, a.H, a.I, a.E))
    return launch_decode_fused(a, db.h, db.ybuf, db.counters, status, device, st, launches);
  DecodeArgs p{a, rb, db, status, {}, {}};
  if (!config_gemm1(a.H, p.c1) || !config_gemm2(a.H, a.I, p.c2)) return cudaErrorNotSupported;
  if (!db.vmeta) return cudaErrorInvalidValue;
  // the prep kernel's route also writes the down projection's per-pass work list
  p.rb.vmeta = db.vmeta;
  p.rb.spp = p.c2.SPP;
  const int sms = num_sms(device);
  cudaError_t err;
  // few slots: a smaller CTA keeps the route's block-wide scans short; the
  // activation CTAs need one thread per 8 values of a row
  int nt = route_threads(a.E);
  const int want = (a.S + 31) / 32 * 32;
  if (want < nt) nt = want < 256 ? 256 : want;   // >= 256 threads: the activation CTAs rely on it
  const size_t rsm = route_smem_bytes(a.E, nt);
  auto prep = a.act8 ? decode_prep_kernel<true> : decode_prep_kernel<false>;
  if ((err = set_max_smem((const void*)prep, (int)rsm))) return err;
  // the gate/up projection for the activation format, with the optional
  // MLP bias compiled in or out
  // H or I not a multiple of 128 (both multiples of 64): the kernels' last
  // K block is one 64-wide chunk
  const bool rag = a.H % 128 != 0 || a.I % 128 != 0;
  auto gemm1 = rag ? (a.act8 ? (a.b13 ? decode_gemm1_kernel<true, true, true> : decode_gemm1_kernel<true, false, true>)
                             : (a.b13 ? decode_gemm1_kernel<false, true, true> : decode_gemm1_kernel<false, false, true>))
                   : (a.act8 ? (a.b13 ? decode_gemm1_kernel<true, true, false> : decode_gemm1_kernel<true, false, false>)
                             : (a.b13 ? decode_gemm1_kernel<false, true, false>
                                      : decode_gemm1_kernel<false, false, false>));
  auto gemm2 = rag ? decode_gemm2_kernel<true> : decode_gemm2_kernel<false>;
  auto combine = a.b2 ? decode_combine_kernel<true> : decode_combine_kernel<false>;
  if ((err = set_max_smem((const void*)gemm1, p.c1.smem))) return err;
  if ((err = set_max_smem((const void*)gemm2, p.c2.smem)))
    return err;
  // a shortened wait limit for this call (failure-detection test aid)
  if (a.dbg_wait_ns) {
    const uint64_t v = a.dbg_wait_ns;
    if ((err = note_error(cudaMemcpyToSymbolAsync(g_wait_limit_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, st),
                          "decode wait limit")))
      return err;
  }
  // prep: route (CTA 0) + f16 activations (CTAs 1..T)
  const bool timed = stage_mark(st, 0);
  const bool pdl = !timed;
  if ((err = launch_check(launch_pdl(prep, dim3(1 + a.T), dim3(nt), rsm, st, false, p), st,
                          "decode_prep")))
    return err;
  stage_mark(st, 1);
  if ((err = launch_check(launch_pdl(gemm1, dim3(sms), dim3(kThreads), p.c1.smem, st, pdl, p), st,
                          "decode_gemm1")))
    return err;
  stage_mark(st, 2);
  if ((err = launch_check(launch_pdl(gemm2, dim3(sms), dim3(kThreads), p.c2.smem, st, pdl, p), st,
                          "decode_gemm2")))
    return err;
  stage_mark(st, 3);
  if ((err = launch_check(launch_pdl(combine, dim3(a.T, (a.H + 1023) / 1024), dim3(256), 0, st, pdl, p),
                          st, "decode_combine")))
    return err;
  stage_mark(st, 4);
  *launches += 4;
  if (a.dbg_wait_ns) {
    const uint64_t v = kWaitTimeoutNs;
    if ((err = note_error(cudaMemcpyToSymbolAsync(g_wait_limit_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, st),
                          "decode wait limit")))
      return err;
  }
  return cudaSuccess;
}

}  // namespace moe
