// decode_fused.cu -- the decode path of the block-FP8 MoE layer as one
// persistent kernel.
//
// At decode sizes the layer is bound by reading the routed experts' e4m3
// weights (fp8-moe-gather page, Problem), and only the routed experts are
// read (same page, The fix).  A forward of a few microseconds of HBM traffic
// cannot afford a chain of kernels (each launch and drain costs several
// microseconds on this part), so every step runs in one launch of one CTA
// per SM:
//
//   routing     each CTA builds the routing lists of all slots in its own
//               shared memory (warp ballots and matches, identical in every
//               CTA), so no kernel and no global list precede the weights
//   gate/up     units of (routed expert, RU gate rows + the matching RU up
//               rows); CTA c takes units [c*U1/G, (c+1)*U1/G).  The
//               activation rows of a pass (up to SPP1 slots of one expert)
//               are copied raw (bf16) into shared memory and converted
//               there to f16 scaled by a power of two per token (W8A16) or
//               quantised per 128-column group (W8A8).  e4m3 weights are
//               widened exactly (FreeToken PR #662, PR body), multiplied on
//               mma.sync m16n8k16 with fp32 accumulation, and each bf16
//               block scale is applied once per 128-wide K block.  The
//               eight consumer warps split K; one of them (rotating) sums
//               the partials and writes h = silu(gate) * up in fp32.
//   hand-off    when a CTA has finished its gate/up units it adds, per
//               routed expert, the (unit, pass) count it completed to a
//               counter in global memory (after a fence: one per warp per
//               forward); a down-projection pass of that expert waits until
//               the counter is complete (acquire).  The down-projection
//               weights do not depend on h, so the ring streams them right
//               after the gate/up weights and only the h copies wait.
//   down        units of (routed expert, R2 rows of w2); h enters the MMA
//               as two f16 terms (hi + lo, about 22 significant bits) after
//               a per-slot power of two ("the down projection in fp32",
//               fp8-moe-gather page, The fix); y * topk_weight goes to a
//               per-slot fp32 buffer.
//   combine     once every CTA has counted its down units as done (one
//               grid-wide counter), each CTA sums a share of the output
//               rows: out[t] = sum_j ybuf[t*k + j] in slot order (fixed
//               order, no atomics on the data) -> bf16.
//
// Warp roles: warps 0-7 consume ring stages (each unit: every warp takes
// one K slice or row tile and deposits its partial sums in shared memory),
// warp 8 streams the weights (bulk copies of whole-row blocks of 16-64 KiB:
// smaller copies leave one SM's copy engine far below its rate), warp 9
// routes and prepares the activation rows, warp 10 finishes every unit
// (sums the partials, applies silu * up or the top-k weight and stores), so
// that no consumer ever waits for another unit's epilogue.  Every wait is bounded (MOE_STATUS_TIMEOUT); the last
// CTA to finish resets the global counters for the next forward.
#include "decode_mma.cuh"

#include <cstdlib>
#include <cstdio>
#include <cstring>

namespace moe {

namespace {

constexpr int kCons = 8;                 // consumer warps
constexpr int kProd = 8;                 // producer warp index
constexpr int kAct = 9;                  // activation warp index
constexpr int kFin = 10;                 // finisher warp index
constexpr int kFThreads = 32 * 11;
constexpr int kFSmemLimit = 232448 - 1024;   // dynamic shared memory (static arrays take the rest)

// Global counters of one forward, in the workspace (zero between forwards;
// the last CTA to finish clears them).
struct Counters {
  uint32_t* done;     // [1] CTAs finished
  uint32_t* d2;       // [1] CTAs whose down units are all written
  uint32_t* c1;       // [DMAX] per routed expert: gate/up (unit, pass) completions
};

struct FusedCfg {
  int RU, RT;          // gate/up row pairs per unit; MMA row tiles (ceil(RU / 8))
  int R2;              // down-projection rows per unit
  int NS, SB;          // ring stages, stage bytes
  int SPP1, SPP2;      // slots per gate/up pass (<= 8), per down pass (<= 4)
  int XP, HP;          // f16 activation row pitch, converted-h row pitch (bytes)
  int S, DMAX;         // slots, min(E, S)
  int o_ids, o_wts, o_perm, o_meta, o_words, o_wbase, o_cnt, o_red, o_xaux, o_act, o_ring, smem;
};

struct FusedArgs {
  LayerArgs a;
  float* h;            // fp32 [S, I], routed order
  float* ybuf;         // fp32 [S, H], slot order, times the slot's top-k weight
  Counters ctr;
  uint32_t* status;
  FusedCfg c;
};

// Barrier block at the start of dynamic shared memory.
struct FBars {
  uint64_t full[8], empty[8];   // ring
  uint64_t xfull[2], xempty[2]; // activation (x) buffers
  uint64_t hfull[2], hempty[2]; // converted-h buffers
  uint64_t rfull[2], rempty[2]; // cross-warp partial sums
  uint64_t route;               // routing lists ready
  uint64_t abar;                // the activation warp's own bulk copies
  int abort;                    // CTA-wide: a wait gave up
  int D;                        // routed experts
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Barrier among the eight consumer warps and the finisher (named barrier 1;
// warps 0-7 and 10).
__device__ __forceinline__ void finish_sync() { asm volatile("bar.sync 1, 288;" ::: "memory"); }

// Bounded spin until *p >= target (acquire).  False on timeout.
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target) {
  uint64_t t0 = 0;
#pragma unroll 1
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_gpu(p) >= target) return true;
    if ((i & 63u) == 0) {
      const uint64_t t = globaltimer_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > *(volatile uint64_t*)&g_wait_limit_ns) return false;
    }
    __nanosleep(64);
  }
}

// The units of one phase that CTA `cta` of `G` takes: [u0, u1) of D * upe.
struct Range {
  long u0, u1;
  int upe;
};

__device__ __forceinline__ Range cta_range(int D, int upe, int cta, int G) {
  const long U = (long)D * upe;
  Range r;
  r.u0 = U * cta / G;
  r.u1 = U * (cta + 1) / G;
  r.upe = upe;
  return r;
}

// Rows per unit, halved while fewer units than CTAs (small D), never below lo.
__device__ __forceinline__ int halve_rows(int R, int lo, int rows_total, int D, int G) {
  while (R > lo && (long)D * (rows_total / R) < (long)G) R >>= 1;
  return R;
}

// ------------------------------------------------------------ routing ----
// The routing lists in shared memory, built by one warp from the ids:
// meta[d] = {expert, first routed position, slot count} of the d-th routed
// expert (ascending), perm[p] = the slot at routed position p (grouped by
// expert, stable in the slot index).  Identical in every CTA.  Returns D.
__device__ int route_smem(const LayerArgs& a, const FusedCfg& c, uint8_t* sm, uint32_t* status, int lane) {
  int* ids = reinterpret_cast<int*>(sm + c.o_ids);
  int* perm = reinterpret_cast<int*>(sm + c.o_perm);
  int4* meta = reinterpret_cast<int4*>(sm + c.o_meta);
  uint32_t* words = reinterpret_cast<uint32_t*>(sm + c.o_words);
  int* wbase = reinterpret_cast<int*>(sm + c.o_wbase);
  int* cnt = reinterpret_cast<int*>(sm + c.o_cnt);
  const int S = a.S, E = a.E;
  for (int i = lane; i < 128; i += 32) words[i] = 0u;
  bool bad = false;
  float* wts = reinterpret_cast<float*>(sm + c.o_wts);
  for (int s = lane; s < S; s += 32) {
    const int id = a.ids[s];
    ids[s] = id;
    wts[s] = a.wts[s];
    bad |= id >= E;
  }
  __syncwarp();
  for (int s = lane; s < S; s += 32) {
    const int id = ids[s];
    if (id >= 0 && id < E) atomicOr(&words[id >> 5], 1u << (id & 31));
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) raise_status(status, MOE_STATUS_BAD_ID);
  __syncwarp();
  // exclusive prefix of the set bits over the 128 words (lane l: words 4l..4l+3)
  int pc[4], tot = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    pc[j] = __popc(words[4 * lane + j]);
    tot += pc[j];
  }
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - tot;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    wbase[4 * lane + j] = run;
    run += pc[j];
  }
  const int D = __shfl_sync(0xffffffffu, incl, 31);
  for (int d = lane; d < D; d += 32) cnt[d] = 0;
  __syncwarp();
  auto rank = [&](int id) { return wbase[id >> 5] + __popc(words[id >> 5] & ((1u << (id & 31)) - 1u)); };
  for (int s = lane; s < S; s += 32) {
    const int id = ids[s];
    if (id >= 0 && id < E) {
      const int d = rank(id);
      atomicAdd(&cnt[d], 1);
      meta[d].x = id;   // every slot of expert id writes the same value
    }
  }
  __syncwarp();
  // offsets: exclusive scan of the counts, 32 at a time with a carry
  int carry = 0;
  for (int d0 = 0; d0 < D; d0 += 32) {
    const int d = d0 + lane;
    const int v = d < D ? cnt[d] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (d < D) {
      meta[d].y = carry + x - v;
      meta[d].z = v;
      meta[d].w = 0;
    }
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  __syncwarp();
  for (int d = lane; d < D; d += 32) cnt[d] = 0;   // reused: slots placed so far
  __syncwarp();
  // stable placement, 32 slots at a time
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s = s0 + lane;
    const int id = s < S ? ids[s] : -1;
    const bool valid = id >= 0 && id < E;
    const int d = valid ? rank(id) : -1 - (s >= S);
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int before = __popc(peers & lanemask_lt());
    if (valid) perm[meta[d].y + cnt[d] + before] = s;
    __syncwarp();
    if (valid && before == 0) cnt[d] += __popc(peers);
    __syncwarp();
  }
  return D;
}

// --------------------------------------------------- activation rows ----
// One activation row in shared memory, converted in place from bf16.
// W8A16: max |x| of the row -> exponent s with max * 2^-s in [2^14, 2^15)
// (exact in f16 for every element >= max * 2^-31), f16(x * 2^-s); returns s.
__device__ int convert_row_w8a16(uint8_t* row, int H, int lane) {
  float m = 0.f;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 r = lds128(row + 2 * i);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(w[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(w[j] >> 16))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int s = 0;
  if (m > 0.f) {
    int ex;
    frexpf(m, &ex);
    s = (ex - 1) - 14;
  }
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 r = lds128(row + 2 * i);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t o4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(ldexpf(bf16_bits_to_f32(w[j] & 0xFFFFu), -s),
                                           ldexpf(bf16_bits_to_f32(w[j] >> 16), -s));
      o4[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(row + 2 * i) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
  __syncwarp();
  return s;
}

// W8A8: per 128-column group, amax, scale = amax / 448 and code =
// e4m3(x / scale) rounded to nearest even and saturated, both IEEE fp32
// divisions (the prefill rule, fp8-moe-gather page, "Affects": dynamic
// activation scales); the row then holds the f16 values of the codes and
// xs[kb] the group scales.  With `codes` (global), the code bytes and scales
// are also written there.
__device__ void quantize_row_w8a8(uint8_t* row, int H, float* xs, uint8_t* codes, float* scales, int lane) {
  for (int g = 0; g < H / 128; ++g) {
    uint8_t* grp = row + 2 * (g * 128 + lane * 4);
    const uint2 r = *reinterpret_cast<const uint2*>(grp);
    const float v[4] = {bf16_bits_to_f32(r.x & 0xFFFFu), bf16_bits_to_f32(r.x >> 16), bf16_bits_to_f32(r.y & 0xFFFFu),
                        bf16_bits_to_f32(r.y >> 16)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float sc = __fdiv_rn(m, 448.0f);
    uint16_t q01 = 0, q23 = 0;
    if (sc != 0.f) {
      q01 = e4m3x2_from_f32(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc));
      q23 = e4m3x2_from_f32(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc));
    }
    *reinterpret_cast<uint2*>(grp) = make_uint2(e4m3x2_to_f16x2(q01), e4m3x2_to_f16x2(q23));
    if (lane == 0) xs[g] = sc;
    if (codes) {
      *reinterpret_cast<uint32_t*>(codes + g * 128 + lane * 4) = (uint32_t)q01 | ((uint32_t)q23 << 16);
      if (lane == 0) scales[g] = sc;
    }
  }
  __syncwarp();
}


// ------------------------------------------------------- warp slices ----
// A warp's K slice of one 16-row MMA tile, KW 128-wide K blocks from K block
// kb0: rows g (p0) and g + 8 (p1) of the tile, 16 bytes per lane per 64-wide
// chunk (the fragment layout of afrag), copied out of the ring stage into
// registers so that the stage can be released before the MMAs.
template <int KW>
__device__ __forceinline__ void load_slice(const uint8_t* p0, const uint8_t* p1, int kb0, bool has,
                                           uint4 (&wa)[2 * KW], uint4 (&wb)[2 * KW]) {
#pragma unroll
  for (int i = 0; i < 2 * KW; ++i) {
    const int kk = (kb0 + (i >> 1)) * 128 + (i & 1) * 64;
    wa[i] = has ? lds128(p0 + kk) : make_uint4(0, 0, 0, 0);
    wb[i] = has ? lds128(p1 + kk) : make_uint4(0, 0, 0, 0);
  }
}

// The slice's MMAs against the activation columns at xrow (f16, 16 bytes per
// lane per 64-wide chunk, 32 per 128 bytes of K).  Each K block's partial is
// scaled once: rows g (C[0], C[1]) by slo, rows g + 8 (C[2], C[3]) by shi,
// times the column scales a0[j] (column 2c) and a1[j] (column 2c + 1); slo
// and shi of K block kb0 + j come from lane j.
template <int KW>
__device__ __forceinline__ void mma_slice(const uint4 (&wa)[2 * KW], const uint4 (&wb)[2 * KW], const uint8_t* xrow,
                                          int kb0, bool has_x, float slo, float shi, const float (&a0)[8],
                                          const float (&a1)[8], float (&acc)[4]) {
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = (kb0 + j) * 128 + ch * 64;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (has_x) {
        x0 = lds128(xrow + 2 * kk);
        x1 = lds128(xrow + 2 * kk + 16);
      }
      chunk_mma(b0, b1, wa[2 * j + ch], wb[2 * j + ch], x0, x1);
    }
    const float sl = __shfl_sync(0xffffffffu, slo, j);
    const float sh = __shfl_sync(0xffffffffu, shi, j);
    acc[0] = fmaf(sl * a0[j], b0[0] + b1[0], acc[0]);
    acc[1] = fmaf(sl * a1[j], b0[1] + b1[1], acc[1]);
    acc[2] = fmaf(sh * a0[j], b0[2] + b1[2], acc[2]);
    acc[3] = fmaf(sh * a1[j], b0[3] + b1[3], acc[3]);
  }
}

// The same reading the weights from the ring stage inside the loop (K
// slices too long for registers); any KW.  Column scales from shared memory
// (a0[j], a1[j]) or 1 where a0 / a1 is null.
__device__ __forceinline__ void mma_slice_smem(const uint8_t* p0, const uint8_t* p1, int kb0, int kw, bool has,
                                               const uint8_t* xrow, bool has_x, float slo, float shi,
                                               const float* a0, const float* a1, float (&acc)[4]) {
#pragma unroll 1
  for (int j = 0; j < kw; ++j) {
    float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = (kb0 + j) * 128 + ch * 64;
      uint4 wa = make_uint4(0, 0, 0, 0), wb = wa, x0 = wa, x1 = wa;
      if (has) {
        wa = lds128(p0 + kk);
        wb = lds128(p1 + kk);
      }
      if (has_x) {
        x0 = lds128(xrow + 2 * kk);
        x1 = lds128(xrow + 2 * kk + 16);
      }
      chunk_mma(b0, b1, wa, wb, x0, x1);
    }
    const float sl = __shfl_sync(0xffffffffu, slo, j);
    const float sh = __shfl_sync(0xffffffffu, shi, j);
    const float c0 = a0 ? a0[j] : 1.f, c1 = a1 ? a1[j] : 1.f;
    acc[0] = fmaf(sl * c0, b0[0] + b1[0], acc[0]);
    acc[1] = fmaf(sl * c1, b0[1] + b1[1], acc[1]);
    acc[2] = fmaf(sh * c0, b0[2] + b1[2], acc[2]);
    acc[3] = fmaf(sh * c1, b0[3] + b1[3], acc[3]);
  }
}

// One warp's block scales of a 128-row block (lane j: K block kb0 + j, for
// j < kw), kept while consecutive units stay in the block, with the next
// block of the same bank loaded ahead.  Ordinary loads issued while the
// SM's bulk copies stream take microseconds to return, so a unit must never
// wait on its own scale load.
struct ScaleCache {
  const uint16_t* cur_row = nullptr;   // scale row the current values belong to
  const uint16_t* nxt_row = nullptr;
  float cur = 0.f, nxt = 0.f;
  __device__ __forceinline__ float get(const uint16_t* row, const uint16_t* next_row, int kb0, int kw, int lane) {
    if (row != cur_row) {
      if (row == nxt_row) {
        cur = nxt;
      } else {
        cur = lane < kw ? bf16_bits_to_f32(__ldg(row + kb0 + lane)) : 0.f;
      }
      cur_row = row;
      nxt_row = next_row;
      if (next_row) nxt = lane < kw ? bf16_bits_to_f32(__ldg(next_row + kb0 + lane)) : 0.f;
    }
    return cur;
  }
};

// ------------------------------------------------------------ the kernel --
template <bool ACT8, bool BIAS>
__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(const __grid_constant__ FusedArgs p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint32_t ebits[128];
  const LayerArgs& a = p.a;
  const FusedCfg& c = p.c;
  FBars& B = *reinterpret_cast<FBars*>(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  int* ids_s = reinterpret_cast<int*>(sm + c.o_ids);
  int* perm_s = reinterpret_cast<int*>(sm + c.o_perm);
  const float* wts_s = reinterpret_cast<const float*>(sm + c.o_wts);
  const int4* meta_s = reinterpret_cast<const int4*>(sm + c.o_meta);
  float* red = reinterpret_cast<float*>(sm + c.o_red);
  uint8_t* act = sm + c.o_act;
  uint8_t* ring = sm + c.o_ring;
  // per x buffer: token exponents [SPP1] then W8A8 group scales [SPP1][nkb]
  const int nkb1 = a.H >> 7, nkb2 = a.I >> 7;
  int* xaux = reinterpret_cast<int*>(sm + c.o_xaux);
  auto xexp = [&](int b) { return xaux + b * (c.SPP1 * (1 + nkb1)); };
  auto xsc = [&](int b) { return reinterpret_cast<float*>(xaux + b * (c.SPP1 * (1 + nkb1)) + c.SPP1); };
  int* hexp = xaux + 2 * c.SPP1 * (1 + nkb1);   // [2][4] per-slot h exponents
  uint8_t* xbuf0 = act;
  uint8_t* hraw = act;                               // phase 2: raw h rows [SPP2][4I]
  uint8_t* hconv0 = act + c.SPP2 * 4 * a.I;          // phase 2: [2][8][HP]

  if (threadIdx.x == 0) {
    for (int i = 0; i < c.NS; ++i) {
      mbar_init(&B.full[i], 1);
      mbar_init(&B.empty[i], kCons);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.xfull[i], 1);
      mbar_init(&B.xempty[i], kCons + 1);
      mbar_init(&B.hfull[i], 1);
      mbar_init(&B.hempty[i], kCons + 1);
      mbar_init(&B.rfull[i], kCons);
      mbar_init(&B.rempty[i], 1);
    }
    mbar_init(&B.route, 1);
    mbar_init(&B.abar, 1);
    B.abort = 0;
    B.D = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // inputs may come from the kernel before this one in the stream
  pdl_wait();
  pdl_trigger();
  auto fail = [&]() {
    B.abort = 1;
    raise_status(p.status, MOE_STATUS_TIMEOUT);
  };
  auto aborted = [&]() { return *(volatile int*)&B.abort != 0; };

  if (warp == kProd) {
    // ============================================== weight producer ====
    ExpertBits eb;
    const int D = expert_bits(a.ids, a.S, a.E, ebits, lane, eb);
    const int RU = halve_rows(c.RU, 1, a.I, D, G);
    const int R2 = halve_rows(c.R2, 16, a.H, D, G);
    const Range r1 = cta_range(D, a.I / RU, cta, G), r2 = cta_range(D, a.H / R2, cta, G);
    const uint64_t pol = l2_policy_evict_first();
    const int rowb = RU * a.H, tileb = R2 * a.I;
    int m = 0, pre = 0;
    bool ok = true;
    auto issue1 = [&](int slot, int e, int i0) {
      const uint8_t* g = a.w13 + ((int64_t)e * 2 * a.I + i0) * a.H;
      mbar_arrive_expect_tx(&B.full[slot], 2 * rowb);
      bulk_g2s(ring + slot * c.SB, g, rowb, &B.full[slot], pol);
      bulk_g2s(ring + slot * c.SB + rowb, g + (int64_t)a.I * a.H, rowb, &B.full[slot], pol);
    };
    // the first stages (pass 0 of the first expert) go out before the routing lists exist
    if (r1.u0 < r1.u1) {
      const int d0 = (int)(r1.u0 / r1.upe);
      const int e0 = expert_select(eb, d0, lane);
      const long n = min((long)c.NS, min(r1.u1, (long)(d0 + 1) * r1.upe) - r1.u0);
      if (lane == 0)
        for (long i = 0; i < n; ++i) issue1((int)i, e0, (int)((r1.u0 + i) % r1.upe) * RU);
      pre = (int)n;
    }
    __syncwarp();
    ok = warp_wait(&B.route, 0, lane);
    // phase 1: gate/up units, pass by pass
    for (long u = r1.u0; ok && u < r1.u1;) {
      const int d = (int)(u / r1.upe);
      const long se = min(r1.u1, (long)(d + 1) * r1.upe);
      const int4 md = meta_s[d];
      const int passes = (md.z + c.SPP1 - 1) / c.SPP1;
      for (int ps = 0; ps < passes && ok; ++ps)
        for (long uu = u; uu < se && ok; ++uu, ++m) {
          if (m < pre) continue;
          const int slot = m % c.NS;
          if (m >= c.NS) ok = warp_wait(&B.empty[slot], ((m / c.NS) - 1) & 1, lane);
          if (ok && lane == 0) issue1(slot, md.x, (int)(uu % r1.upe) * RU);
          __syncwarp();
          if (aborted()) ok = false;
        }
      u = se;
    }
    // phase 2: down-projection units (no dependency on h)
    for (long u = r2.u0; ok && u < r2.u1;) {
      const int d = (int)(u / r2.upe);
      const long se = min(r2.u1, (long)(d + 1) * r2.upe);
      const int4 md = meta_s[d];
      const int passes = (md.z + c.SPP2 - 1) / c.SPP2;
      for (int ps = 0; ps < passes && ok; ++ps)
        for (long uu = u; uu < se && ok; ++uu, ++m) {
          const int slot = m % c.NS;
          if (m >= c.NS) ok = warp_wait(&B.empty[slot], ((m / c.NS) - 1) & 1, lane);
          if (ok && lane == 0) {
            const int n0 = (int)(uu % r2.upe) * R2;
            mbar_arrive_expect_tx(&B.full[slot], tileb);
            bulk_g2s(ring + slot * c.SB, a.w2 + ((int64_t)md.x * a.H + n0) * a.I, tileb, &B.full[slot], pol);
          }
          __syncwarp();
          if (aborted()) ok = false;
        }
      u = se;
    }
    if (!ok) {
      if (lane == 0) {
        fail();
        // copies already issued must land before the CTA exits
        const int issued = max(m, pre);
        for (int mm = max(0, issued - c.NS); mm < issued; ++mm) mbar_wait(&B.full[mm % c.NS], (mm / c.NS) & 1);
      }
      __syncwarp();
    }
  } else if (warp == kAct) {
    // ============================================ activation warp ====
    const int D = route_smem(a, c, sm, p.status, lane);
    if (lane == 0) B.D = D;
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.route);
    const int RU = halve_rows(c.RU, 1, a.I, D, G);
    const int R2 = halve_rows(c.R2, 16, a.H, D, G);
    const Range r1 = cta_range(D, a.I / RU, cta, G), r2 = cta_range(D, a.H / R2, cta, G);
    const uint64_t pol = l2_policy_evict_last();
    uint32_t aph = 0;   // phase of abar
    bool ok = true;
    // copy `n` rows of `bytes` each (row i from src(i)) into dst rows of pitch `pitch`, and wait
    auto copy_rows = [&](uint8_t* dst, int pitch, int n, int bytes, auto src) -> bool {
      fence_proxy_async();   // earlier generic accesses of these bytes come first
      if (lane == 0) mbar_arrive_expect_tx(&B.abar, (uint32_t)(n * bytes));
      __syncwarp();
      if (lane < n) bulk_g2s(dst + lane * pitch, src(lane), (uint32_t)bytes, &B.abar, pol);
      const bool r = warp_wait(&B.abar, aph, lane);
      aph ^= 1u;
      return r;
    };
    if (ACT8 && a.dbg_codes && cta == 0) {
      // the activation codes as the forward quantises them, for every token
      for (int t = 0; t < a.T && ok; ++t) {
        ok = copy_rows(xbuf0, c.XP, 1, 2 * a.H, [&](int) { return a.hidden + (int64_t)t * a.hidden_ld; });
        if (ok)
          quantize_row_w8a8(xbuf0, a.H, xsc(0), a.dbg_codes + (int64_t)t * a.H, a.dbg_scales + (int64_t)t * nkb1,
                            lane);
      }
    }
    // phase 1: the x rows of every gate/up pass
    int gx = 0;
    for (long u = r1.u0; ok && u < r1.u1;) {
      const int d = (int)(u / r1.upe);
      const long se = min(r1.u1, (long)(d + 1) * r1.upe);
      const int4 md = meta_s[d];
      const int passes = (md.z + c.SPP1 - 1) / c.SPP1;
      for (int ps = 0; ps < passes && ok; ++ps, ++gx) {
        const int b = gx & 1, nx = min(c.SPP1, md.z - ps * c.SPP1);
        if (gx >= 2) ok = warp_wait(&B.xempty[b], ((gx >> 1) - 1) & 1, lane);
        if (!ok) break;
        uint8_t* xb = xbuf0 + b * c.SPP1 * c.XP;
        const int pos0 = md.y + ps * c.SPP1;
        ok = copy_rows(xb, c.XP, nx, 2 * a.H,
                       [&](int i) { return a.hidden + (int64_t)(perm_s[pos0 + i] / a.k) * a.hidden_ld; });
        if (!ok) break;
        for (int i = 0; i < nx; ++i) {
          if (ACT8) {
            quantize_row_w8a8(xb + i * c.XP, a.H, xsc(b) + i * nkb1, nullptr, nullptr, lane);
            if (lane == 0) xexp(b)[i] = 0;
          } else {
            const int s = convert_row_w8a16(xb + i * c.XP, a.H, lane);
            if (lane == 0) xexp(b)[i] = s;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.xfull[b]);
        if (aborted()) ok = false;
      }
      u = se;
    }
    // the h buffers share the x buffers' bytes: wait until both are released
    for (int g = max(0, gx - 2); ok && g < gx; ++g) ok = warp_wait(&B.xempty[g & 1], (g >> 1) & 1, lane);
    // phase 2: the h rows of every down pass, once the expert's h is complete
    const int upe1 = a.I / RU;
    int gh = 0;
    for (long u = r2.u0; ok && u < r2.u1;) {
      const int d = (int)(u / r2.upe);
      const long se = min(r2.u1, (long)(d + 1) * r2.upe);
      const int4 md = meta_s[d];
      const int passes = (md.z + c.SPP2 - 1) / c.SPP2;
      const uint32_t target = (uint32_t)(upe1 * ((md.z + c.SPP1 - 1) / c.SPP1));
      if (lane == 0) ok = wait_counter(p.ctr.c1 + d, target);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int ps = 0; ps < passes && ok; ++ps, ++gh) {
        const int b = gh & 1, nh = min(c.SPP2, md.z - ps * c.SPP2);
        if (gh >= 2) ok = warp_wait(&B.hempty[b], ((gh >> 1) - 1) & 1, lane);
        if (!ok) break;
        const float* src = p.h + (int64_t)(md.y + ps * c.SPP2) * a.I;
        ok = copy_rows(hraw, 4 * a.I, 1, nh * 4 * a.I, [&](int) { return src; });
        if (!ok) break;
        uint8_t* hb = hconv0 + b * 8 * c.HP;
        for (int s = 0; s < nh; ++s) {
          const float* row = reinterpret_cast<const float*>(hraw + s * 4 * a.I);
          float mx = 0.f;
          for (int kk = lane * 4; kk < a.I; kk += 128) {
            const float4 v = lds_f4(row + kk);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          int es = 0;
          if (mx > 0.f) {
            int ex;
            frexpf(mx, &ex);
            es = (ex - 1) - 14;
          }
          for (int kk = lane * 2; kk < a.I; kk += 64) {
            const float2 v = *reinterpret_cast<const float2*>(row + kk);
            const float v0 = ldexpf(v.x, -es), v1 = ldexpf(v.y, -es);
            const __half2 hi = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            *reinterpret_cast<__half2*>(hb + s * c.HP + 2 * kk) = hi;
            *reinterpret_cast<__half2*>(hb + (4 + s) * c.HP + 2 * kk) = lo;
          }
          if (lane == 0) hexp[b * 4 + s] = es;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.hfull[b]);
        if (aborted()) ok = false;
      }
      u = se;
    }
    if (!ok && lane == 0) fail();
    __syncwarp();
  } else {
    // ======================================= consumers 0-7, finisher 10 ====
    const bool fin = warp == kFin;
    const int w = fin ? 0 : warp;
    const int g = lane >> 2, cq = lane & 3;
    bool ok = warp_wait(&B.route, 0, lane);
    const int D = ok ? *(volatile int*)&B.D : 0;
    const int RU = halve_rows(c.RU, 1, a.I, D, G);
    const int RT = (RU + 7) >> 3;
    const int R2 = halve_rows(c.R2, 16, a.H, D, G);
    const Range r1 = cta_range(D, a.I / RU, cta, G), r2 = cta_range(D, a.H / R2, cta, G);
    const int kb0 = w * nkb1 / kCons, kb1 = (w + 1) * nkb1 / kCons, kw = kb1 - kb0;
    int m = 0;   // ring stage sequence (as the producer's) = reduction step
    // Reduction steps, double-buffered: every consumer deposits 8 floats per
    // lane for step m and arrives on rfull[m & 1]; the finisher waits for all
    // eight, sums, finishes the unit and arrives on rempty[m & 1], which a
    // deposit two steps later waits for.  (Compile-time indexes only: the
    // partial sums stay in registers.)
    auto deposit = [&](const float (&part)[8]) -> bool {
      const int rb = m & 1;
      if (m >= 2 && !warp_wait(&B.rempty[rb], ((m >> 1) - 1) & 1, lane)) return false;
      float4* dst = reinterpret_cast<float4*>(red + ((rb * kCons + w) * 32 + lane) * 8);
      dst[0] = make_float4(part[0], part[1], part[2], part[3]);
      dst[1] = make_float4(part[4], part[5], part[6], part[7]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.rfull[rb]);
      return true;
    };
    // the finisher: the partials of step m from warps w0, w0 + stride, ... (nw of them)
    auto gather = [&](float (&tot)[8], int w0, int nw, int stride) {
      const int rb = m & 1;
#pragma unroll
      for (int i = 0; i < 8; ++i) tot[i] = 0.f;
      for (int j = 0; j < nw; ++j) {
        const float4* src = reinterpret_cast<const float4*>(red + ((rb * kCons + w0 + j * stride) * 32 + lane) * 8);
        const float4 x = src[0], y = src[1];
        tot[0] += x.x; tot[1] += x.y; tot[2] += x.z; tot[3] += x.w;
        tot[4] += y.x; tot[5] += y.y; tot[6] += y.z; tot[7] += y.w;
      }
    };

    // ---------------------------------------------- gate/up units
    ScaleCache scg, scu;   // this warp's gate and up block scales
    int gx = 0;
    for (long u = r1.u0; ok && u < r1.u1;) {
      const int d = (int)(u / r1.upe);
      const long se = min(r1.u1, (long)(d + 1) * r1.upe);
      const int4 md = meta_s[d];
      const int e = md.x;
      const int passes = (md.z + c.SPP1 - 1) / c.SPP1;
      for (int ps = 0; ps < passes && ok; ++ps, ++gx) {
        const int b = gx & 1, nx = min(c.SPP1, md.z - ps * c.SPP1);
        const int pos0 = md.y + ps * c.SPP1;
        if (!warp_wait(&B.xfull[b], (gx >> 1) & 1, lane)) {
          ok = false;
          break;
        }
        if (fin) {
          // ------------------------------------------ finisher, gate/up
          int sx[2] = {0, 0};
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (2 * cq + j < nx) sx[j] = xexp(b)[2 * cq + j];
          for (long uu = u; uu < se; ++uu, ++m) {
            const int i0 = (int)(uu % r1.upe) * RU;
            if (!warp_wait(&B.rfull[m & 1], (m >> 1) & 1, lane)) {
              ok = false;
              break;
            }
            float tot[8];
            gather(tot, 0, kCons, 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.rempty[m & 1]);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int r = t * 8 + g;
              if (t >= RT || r >= RU) continue;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                if (2 * cq + j >= nx) continue;
                float gv = ldexpf(tot[4 * t + j], sx[j]);
                float uv = ldexpf(tot[4 * t + 2 + j], sx[j]);
                if (BIAS && a.b13) {   // either bias may be absent
                  const float* br = a.b13 + (int64_t)e * a.b13_ld + i0 + r;
                  gv += __ldg(br);
                  uv += __ldg(br + a.I);
                }
                p.h[(int64_t)(pos0 + 2 * cq + j) * a.I + i0 + r] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
              }
            }
            if (aborted()) {
              ok = false;
              break;
            }
          }
        } else {
          // ------------------------------------------ consumer, gate/up
          const uint8_t* xrow = xbuf0 + b * c.SPP1 * c.XP + g * c.XP + cq * 32;
          const bool has_x = g < nx;
          // W8A8 activation scales of slots 2cq, 2cq + 1 over this warp's K blocks
          float sa[2][8];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              sa[j][kk] = (ACT8 && 2 * cq + j < nx && kk < kw) ? xsc(b)[(2 * cq + j) * nkb1 + kb0 + kk] : 1.f;
          for (long uu = u; uu < se; ++uu, ++m) {
            const int i0 = (int)(uu % r1.upe) * RU;
            // this warp's block scales (lane j: K block kb0 + j) of the unit's
            // gate and up rows; the up rows' 128-row block is I/128 blocks on
            const int rb = i0 >> 7, nrb = a.I >> 7;
            const uint16_t* sbase = a.w13s + (int64_t)e * a.s13_exp;
            const bool more = rb + 1 < nrb && (int)((se - 1) % r1.upe) * RU >= (rb + 1) * 128;
            const float sgl = scg.get(sbase + (int64_t)rb * a.s13_row,
                                      more ? sbase + (int64_t)(rb + 1) * a.s13_row : nullptr, kb0, kw, lane);
            const float sul = scu.get(sbase + (int64_t)(nrb + rb) * a.s13_row,
                                      more ? sbase + (int64_t)(nrb + rb + 1) * a.s13_row : nullptr, kb0, kw, lane);
            const int slot = m % c.NS;
            if (!warp_wait(&B.full[slot], (m / c.NS) & 1, lane)) {
              ok = false;
              break;
            }
            const uint8_t* st = ring + slot * c.SB;
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = 0.f;
            // W8A8 group scales of columns 2cq, 2cq + 1 in shared memory (smem path)
            const float* xs0 = ACT8 && 2 * cq < nx ? xsc(b) + (2 * cq) * nkb1 + kb0 : nullptr;
            const float* xs1 = ACT8 && 2 * cq + 1 < nx ? xsc(b) + (2 * cq + 1) * nkb1 + kb0 : nullptr;
            const uint8_t* ar0 = st + g * a.H + cq * 16;   // tile 0: gate row g, up row g
            const uint8_t* ar1 = ar0 + 8 * a.H;             // tile 1: gate row 8 + g
            const bool hw0 = g < RU, hw1 = 8 + g < RU;
            bool released = true;
            if (RT == 1 && kw == 2) {
              uint4 wa[4], wb[4];
              load_slice<2>(ar0, ar0 + RU * a.H, kb0, hw0, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
              mma_slice<2>(wa, wb, xrow, kb0, has_x, sgl, sul, sa[0], sa[1], acc);
              part[0] = acc[0]; part[1] = acc[1]; part[2] = acc[2]; part[3] = acc[3];
            } else if (RT == 1 && kw == 3) {
              uint4 wa[6], wb[6];
              load_slice<3>(ar0, ar0 + RU * a.H, kb0, hw0, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
              mma_slice<3>(wa, wb, xrow, kb0, has_x, sgl, sul, sa[0], sa[1], acc);
              part[0] = acc[0]; part[1] = acc[1]; part[2] = acc[2]; part[3] = acc[3];
            } else if (RT == 1 && kw == 1) {
              uint4 wa[2], wb[2];
              load_slice<1>(ar0, ar0 + RU * a.H, kb0, hw0, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
              mma_slice<1>(wa, wb, xrow, kb0, has_x, sgl, sul, sa[0], sa[1], acc);
              part[0] = acc[0]; part[1] = acc[1]; part[2] = acc[2]; part[3] = acc[3];
            } else if (RT == 2 && kw == 2) {
              uint4 wa0[4], wb0[4], wa1[4], wb1[4];
              load_slice<2>(ar0, ar0 + RU * a.H, kb0, hw0, wa0, wb0);
              load_slice<2>(ar1, ar1 + RU * a.H, kb0, hw1, wa1, wb1);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
              mma_slice<2>(wa0, wb0, xrow, kb0, has_x, sgl, sul, sa[0], sa[1], acc0);
              mma_slice<2>(wa1, wb1, xrow, kb0, has_x, sgl, sul, sa[0], sa[1], acc1);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                part[i] = acc0[i];
                part[4 + i] = acc1[i];
              }
            } else {
              released = false;
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (t >= RT) break;
                const uint8_t* arow = t ? ar1 : ar0;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                mma_slice_smem(arow, arow + RU * a.H, kb0, kw, t ? hw1 : hw0, xrow, has_x, sgl, sul, xs0, xs1, acc);
#pragma unroll
                for (int i = 0; i < 4; ++i) part[4 * t + i] = acc[i];
              }
            }
            if (!released) {
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
            }
            if (!deposit(part)) {
              ok = false;
              break;
            }
            if (aborted()) {
              ok = false;
              break;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.xempty[b]);
      }
      u = se;
    }

    // every h row the finisher wrote is visible before this CTA's counts are
    __threadfence();
    finish_sync();
    if (fin && !aborted()) {
      // per routed expert: the (unit, pass) count this CTA completed
      const int dlo = (int)(r1.u0 / r1.upe), dhi = r1.u1 > r1.u0 ? (int)((r1.u1 - 1) / r1.upe) : dlo - 1;
      for (int d = dlo + lane; d <= dhi; d += 32) {
        const long ua = max(r1.u0, (long)d * r1.upe), ub = min(r1.u1, (long)(d + 1) * r1.upe);
        const int passes = (meta_s[d].z + c.SPP1 - 1) / c.SPP1;
        atomicAdd(p.ctr.c1 + d, (uint32_t)((ub - ua) * passes));
      }
    }

    // ---------------------------------------------- down units
    ScaleCache sc2;   // this warp's down-projection block scales
    const float ones[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
    const int NT2 = R2 >> 4, KS2 = kCons / NT2;
    const int tt = w % NT2, ks = w / NT2;
    const int k2a = ks * nkb2 / KS2, k2b = (ks + 1) * nkb2 / KS2;
    int gh = 0;
    for (long u = r2.u0; ok && u < r2.u1;) {
      const int d = (int)(u / r2.upe);
      const long se = min(r2.u1, (long)(d + 1) * r2.upe);
      const int4 md = meta_s[d];
      const int e = md.x;
      const int passes = (md.z + c.SPP2 - 1) / c.SPP2;
      for (int ps = 0; ps < passes && ok; ++ps, ++gh) {
        const int b = gh & 1, nh = min(c.SPP2, md.z - ps * c.SPP2);
        const int pos0 = md.y + ps * c.SPP2;
        if (!warp_wait(&B.hfull[b], (gh >> 1) & 1, lane)) {
          ok = false;
          break;
        }
        if (fin) {
          // ------------------------------------------ finisher, down
          // output slots of this lane (lanes cq < 2: slots 2cq, 2cq + 1),
          // their top-k weights and h exponents
          int so[2] = {-1, -1}, es[2] = {0, 0};
          float wo[2] = {0.f, 0.f};
          if (cq < 2) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (2 * cq + j < nh) {
                so[j] = perm_s[pos0 + 2 * cq + j];
                wo[j] = wts_s[so[j]];
                es[j] = hexp[b * 4 + 2 * cq + j];
              }
          }
          for (long uu = u; uu < se; ++uu, ++m) {
            const int nb = (int)(uu % r2.upe) * R2;
            if (!warp_wait(&B.rfull[m & 1], (m >> 1) & 1, lane)) {
              ok = false;
              break;
            }
            for (int t2 = 0; t2 < NT2; ++t2) {
              float tot[8];
              gather(tot, t2, KS2, NT2);
              // columns 2cq, 2cq + 1: hi terms on lanes cq < 2, lo terms on lanes cq >= 2
#pragma unroll
              for (int i = 0; i < 4; ++i) tot[i] += __shfl_xor_sync(0xffffffffu, tot[i], 2);
              const int n0 = nb + t2 * 16;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                if (so[j] < 0) continue;
                float y0 = ldexpf(tot[j], es[j]) * wo[j];
                float y1 = ldexpf(tot[2 + j], es[j]) * wo[j];
                if (BIAS && a.b2) {
                  const float* br = a.b2 + (int64_t)e * a.b2_ld + n0 + g;
                  y0 = fmaf(wo[j], __ldg(br), y0);
                  y1 = fmaf(wo[j], __ldg(br + 8), y1);
                }
                p.ybuf[(int64_t)so[j] * a.H + n0 + g] = y0;
                p.ybuf[(int64_t)so[j] * a.H + n0 + g + 8] = y1;
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.rempty[m & 1]);
            if (aborted()) {
              ok = false;
              break;
            }
          }
        } else {
          // ------------------------------------------ consumer, down
          const uint8_t* hbrow = hconv0 + b * 8 * c.HP + g * c.HP + cq * 32;
          const bool has_b = (g & 3) < nh;
          for (long uu = u; uu < se; ++uu, ++m) {
            const int n0 = (int)(uu % r2.upe) * R2 + tt * 16;   // this warp's 16 rows
            const int rb = n0 >> 7;
            const uint16_t* sbase = a.w2s + (int64_t)e * a.s2_exp;
            const bool more = rb + 1 < (a.H >> 7) && (int)((se - 1) % r2.upe) * R2 + tt * 16 >= (rb + 1) * 128;
            const float sl = sc2.get(sbase + (int64_t)rb * a.s2_row,
                                     more ? sbase + (int64_t)(rb + 1) * a.s2_row : nullptr, k2a, k2b - k2a, lane);
            const int slot = m % c.NS;
            if (!warp_wait(&B.full[slot], (m / c.NS) & 1, lane)) {
              ok = false;
              break;
            }
            const uint8_t* st = ring + slot * c.SB + (tt * 16) * a.I + g * a.I + cq * 16;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const int kw2 = k2b - k2a;
            if (kw2 == 2) {
              uint4 wa[4], wb[4];
              load_slice<2>(st, st + 8 * a.I, k2a, true, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              mma_slice<2>(wa, wb, hbrow, k2a, has_b, sl, sl, ones, ones, acc);
            } else if (kw2 == 1) {
              uint4 wa[2], wb[2];
              load_slice<1>(st, st + 8 * a.I, k2a, true, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              mma_slice<1>(wa, wb, hbrow, k2a, has_b, sl, sl, ones, ones, acc);
            } else if (kw2 == 3) {
              uint4 wa[6], wb[6];
              load_slice<3>(st, st + 8 * a.I, k2a, true, wa, wb);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
              mma_slice<3>(wa, wb, hbrow, k2a, has_b, sl, sl, ones, ones, acc);
            } else {
              mma_slice_smem(st, st + 8 * a.I, k2a, kw2, true, hbrow, has_b, sl, sl, nullptr, nullptr, acc);
              __syncwarp();
              if (lane == 0) mbar_arrive(&B.empty[slot]);
            }
            const float part[8] = {acc[0], acc[1], acc[2], acc[3], 0.f, 0.f, 0.f, 0.f};
            if (!deposit(part)) {
              ok = false;
              break;
            }
            if (aborted()) {
              ok = false;
              break;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.hempty[b]);
      }
      u = se;
    }
    if (!ok && lane == 0) fail();
    __syncwarp();

    // ---------------------------------------------- combine
    // every ybuf row the finisher wrote is visible before this CTA counts itself done
    __threadfence();
    finish_sync();
    if (fin && lane == 0) {
      atomicAdd(p.ctr.d2, 1u);
      if (!aborted() && !wait_counter(p.ctr.d2, (uint32_t)G)) fail();
    }
    finish_sync();
    if (!aborted()) {
      // items (token, 64-row block); this CTA's share, one item per warp at a time
      const int nrb = a.H >> 6;
      const long N = (long)a.T * nrb;
      const int wi = fin ? kCons : w;
      for (long it = N * cta / G + wi; it < N * (cta + 1) / G; it += kCons + 1) {
        const int t = (int)(it / nrb);
        const int row = (int)(it % nrb) * 64 + 2 * lane;
        float s0 = 0.f, s1 = 0.f;
        for (int j = 0; j < a.k; ++j) {
          const int id = ids_s[t * a.k + j];
          if (id < 0 || id >= a.E) continue;
          const float2 v = __ldcg(reinterpret_cast<const float2*>(p.ybuf + ((int64_t)t * a.k + j) * a.H + row));
          s0 += v.x;
          s1 += v.y;
        }
        *reinterpret_cast<__nv_bfloat162*>(a.out + (int64_t)t * a.H + row) = __floats2bfloat162_rn(s0, s1);
      }
    }
  }

  // ------------------------------------------------------- teardown --
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(p.ctr.done, 1u);
    if (prev + 1 == (uint32_t)G) {
      // every CTA is past its last wait: clear the counters for the next forward
      __threadfence();
      const int D = B.D;
      for (int d = 0; d < D; ++d) p.ctr.c1[d] = 0u;
      *p.ctr.d2 = 0u;
      *p.ctr.done = 0u;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------- config ----
inline int al128(int x) { return (x + 127) / 128 * 128; }

bool place(FusedCfg& c, int H, int I) {
  int o = (int)((sizeof(FBars) + 127) / 128 * 128);
  c.o_ids = o;
  o += al128(4 * c.S);
  c.o_wts = o;
  o += al128(4 * c.S);
  c.o_perm = o;
  o += al128(4 * c.S);
  c.o_meta = o;
  o += al128(16 * c.DMAX);
  c.o_words = o;
  o += 512;
  c.o_wbase = o;
  o += 512;
  c.o_cnt = o;
  o += al128(4 * c.DMAX);
  c.o_red = o;
  o += 2 * kCons * 32 * 8 * 4;
  c.o_xaux = o;
  o += al128(4 * (2 * c.SPP1 * (1 + H / 128) + 8));
  c.o_act = o;
  const int xb = 2 * c.SPP1 * c.XP;
  const int hb = c.SPP2 * 4 * I + 2 * 8 * c.HP;
  o += al128(xb > hb ? xb : hb);
  c.o_ring = o;
  o += c.NS * c.SB;
  c.smem = o;
  return o <= kFSmemLimit;
}

// Candidate shapes, best first: gate/up units whose two copies are as large
// as possible up to 32 KiB each, down units of at least the same stage,
// at least 3 ring stages (about 100-200 KiB in flight per SM), then passes
// of as many slots as still fit.
bool choose_cfg(int H, int I, int S, int E, FusedCfg& c) {
  c.S = S;
  c.DMAX = S < E ? S : E;
  c.XP = 2 * H + 16;   // == 16 mod 128: conflict-free fragment loads
  c.HP = 2 * I + 16;
  const char* env = getenv("MOE_FP8_BLOCK_DECODE_CFG");   // tuning aid: "RU,R2,SPP1,NS"
  if (env) {
    int ru, r2, spp, ns;
    if (sscanf(env, "%d,%d,%d,%d", &ru, &r2, &spp, &ns) == 4 && ru >= 1 && ru <= 16 && I % ru == 0 &&
        (r2 == 16 || r2 == 32 || r2 == 64 || r2 == 128) && H % r2 == 0 && spp >= 1 && spp <= 8 && ns >= 2 &&
        ns <= 8) {
      c.RU = ru;
      c.RT = (ru + 7) / 8;
      c.R2 = r2;
      c.SPP1 = spp;
      c.SPP2 = 4;
      c.SB = al128(2 * ru * H > r2 * I ? 2 * ru * H : r2 * I);
      c.NS = ns;
      if (place(c, H, I)) return true;
    }
  }
  for (int ns_min = 3; ns_min >= 2; --ns_min)
    for (int ru = 16; ru >= 1; ru >>= 1) {
      if (I % ru || 128 % ru || (ru * H > 32768 && ru > 1)) continue;
      c.RU = ru;
      c.RT = (ru + 7) / 8;
      for (int r2 = 128; r2 >= 16; r2 >>= 1) {
        if (H % r2 || (r2 * I > 2 * ru * H && r2 > 16)) continue;
        c.R2 = r2;
        c.SB = al128(2 * ru * H > r2 * I ? 2 * ru * H : r2 * I);
        for (int spp = 8; spp >= 2; --spp) {
          c.SPP1 = spp;
          c.SPP2 = I <= 1024 ? 4 : 2;
          for (c.NS = 8; c.NS >= ns_min; --c.NS)
            if (place(c, H, I)) return true;
        }
        break;
      }
    }
  return false;
}

}  // namespace

// 32-bit counters the fused decode kernel keeps in global memory for S slots
// over E experts (zero before the first forward; every forward leaves them
// zero).
size_t fused_counter_words(int S, int E) { return (size_t)(2 + (S < E ? S : E)); }

bool fused_decode_ok(int T, int k, int H, int I, int E) {
  if (H % 128 || I % 128 || H > 8192 || I > 8192) return false;
  const int64_t S = (int64_t)T * k;
  if (S > kFusedMaxSlots || S < 1) return false;
  FusedCfg c;
  return choose_cfg(H, I, (int)S, E, c);
}

cudaError_t launch_decode_fused(const LayerArgs& a, float* h, float* ybuf, uint32_t* counters,
                                uint32_t* status, int device, cudaStream_t st, int* launches) {
  FusedArgs p;
  p.a = a;
  p.h = h;
  p.ybuf = ybuf;
  p.status = status;
  p.ctr.done = counters;
  p.ctr.d2 = counters + 1;
  p.ctr.c1 = counters + 2;
  if (!choose_cfg(a.H, a.I, a.S, a.E, p.c)) return cudaErrorNotSupported;
  auto kern = a.act8 ? (a.b13 || a.b2 ? decode_fused_kernel<true, true> : decode_fused_kernel<true, false>)
                     : (a.b13 || a.b2 ? decode_fused_kernel<false, true> : decode_fused_kernel<false, false>);
  cudaError_t err = set_max_smem((const void*)kern, p.c.smem);
  if (err != cudaSuccess) return note_error(err, "decode_fused smem attribute");
  const bool timed = stage_mark(st, 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms(device));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = p.c.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = timed ? 0 : 1;
  if ((err = launch_check(cudaLaunchKernelEx(&cfg, kern, p), st, "decode_fused"))) return err;
  stage_mark(st, 1);
  *launches += 1;
  return cudaSuccess;
}

}  // namespace moe
