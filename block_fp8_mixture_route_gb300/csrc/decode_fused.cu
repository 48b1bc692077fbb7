// decode_fused.cu -- the decode path of the block-FP8 MoE layer as one
// persistent kernel (moe_options.decode_kernel = MOE_DECODE_KERNEL_FUSED).
//
// At decode sizes the layer is bound by reading the routed experts' e4m3
// weights (fp8-moe-gather page, Problem), and only the routed experts are
// read (same page, The fix).  Every step runs in one launch of one CTA per
// SM:
//
//   routing     each CTA builds the routing lists of all slots in its own
//               shared memory (warp ballots and matches, identical in every
//               CTA); no kernel and no global list precede the weights
//   gate/up     items of (routed expert, 8 gate rows + the matching 8 up
//               rows, one K round of up to 16 128-wide K blocks); CTA c
//               takes the tiles [c*U1/G, (c+1)*U1/G) with all their K
//               rounds.  The activation rows of a pass (up to SPP1 slots of
//               one expert) are copied raw (bf16) into shared memory and
//               converted there to f16 scaled by a power of two per token
//               (W8A16) or quantised per 128-column group (W8A8).  Each of
//               the eight consumer warps takes two K blocks of an item: its
//               e4m3 weights come straight from memory into registers with
//               16-byte non-allocating vector loads, one item ahead (device
//               banks: after a bulk prefetch has brought them from HBM into
//               L2 eight items ahead); they are widened exactly (FreeToken PR #662,
//               PR body) and multiplied on mma.sync m16n8k16 with fp32
//               accumulation; each bf16 block scale is applied once per
//               128-wide K block.
//   hand-off    when a CTA has finished its gate/up tiles it adds, per routed
//               expert, the (tile, pass) count it completed to a counter in
//               global memory (after a fence); a down-projection pass of that
//               expert waits until the counter is complete (acquire).  The
//               down-projection weights do not depend on h, so their loads
//               are issued as soon as a warp's gate/up items are loaded.
//   down        items of (routed expert, 16 * NT2 rows of w2); h enters the
//               MMA as two f16 terms (hi + lo, about 22 significant bits)
//               after a per-slot power of two ("the down projection in
//               fp32", fp8-moe-gather page, The fix); y * topk_weight goes
//               to a per-slot fp32 buffer.
//   combine     once every CTA has counted its down items as done (one
//               grid-wide counter), each CTA sums a share of the output
//               rows: out[t] = sum_j ybuf[t*k + j] in slot order (fixed
//               order, no atomics on the data) -> bf16.
//
// Warp roles: warps 0-7 compute (each item: every warp deposits its partial
// sums in shared memory), warp 8 routes and prepares the activation and h
// rows, warp 9 finishes every item (sums the partials over the warps and
// the K rounds, applies silu * up or the top-k weight and stores), so that
// no compute warp waits for another item's epilogue.  The weights never
// pass through shared memory and every weight access is an ordinary load,
// so the same kernel streams banks that live in page-locked host memory
// (read over the host link; moe_fp8_block_forward_host_experts), where bulk
// copies and prefetches are not used.  Registers bound how far ahead the
// loads run (three warps share each SM sub-partition's register file).  Every wait is bounded
// (MOE_STATUS_TIMEOUT); the last CTA to finish resets the global counters
// for the next forward.
#include "decode_mma.cuh"

#include <cstdlib>
#include <cstdio>
#include <cstring>

namespace moe {

namespace {

constexpr int kCons = 8;                 // compute warps
constexpr int kAct = 8;                  // activation warp index
constexpr int kFin = 9;                  // finisher warp index
constexpr int kFThreads = 32 * 10;
constexpr int kPD = 2;                   // items whose weights a compute warp holds or has in flight
constexpr int kPF = 8;                   // items ahead whose weights are prefetched into L2
constexpr int kFSmemLimit = 232448 - 1024;   // dynamic shared memory (static arrays take the rest)

// Global counters of one forward, in the workspace (zero between forwards;
// the last CTA to finish clears them).
struct Counters {
  uint32_t* done;     // [1] CTAs finished
  uint32_t* d2;       // [1] CTAs whose down items are all written
  uint32_t* c1;       // [DMAX] per routed expert: gate/up (tile, pass) completions
};

struct FusedCfg {
  int NKR1;            // K rounds of a gate/up tile (16 K blocks each)
  int NT2, KS2;        // down: 16-row tiles per item, K splits per tile (2 K blocks each)
  int SPP1, SPP2;      // slots per gate/up pass (<= 8), per down pass (<= 4)
  int XP, HP;          // f16 activation row pitch, converted-h row pitch (bytes)
  int S, DMAX;         // slots, min(E, S)
  int o_ids, o_wts, o_perm, o_meta, o_words, o_wbase, o_cnt, o_red, o_xaux, o_act, smem;
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

// Barrier among the eight compute warps and the finisher (named barrier 1;
// warps 0-7 and 9).
__device__ __forceinline__ void finish_sync() { asm volatile("bar.sync 1, 288;" ::: "memory"); }

// 16 bytes of weights that are read once: not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

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

// The range of a phase's work that CTA `cta` of `G` takes: [u0, u1) of
// D * per (per = tiles or items per routed expert).
struct Range {
  long u0, u1;
};

__device__ __forceinline__ Range cta_range(int D, int per, int cta, int G) {
  const long U = (long)D * per;
  return Range{U * cta / G, U * (cta + 1) / G};
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


// ------------------------------------------------------------ the walk ----
// The sequence of items a CTA works through, identical for the compute
// warps (twice: one walk issues loads kPD items ahead of the other), the
// finisher and, by segments and passes, the activation warp.  Phase 1: for
// each routed expert d in the CTA's range of gate/up tiles, each pass of up
// to SPP1 of the expert's slots, each tile, each K round.  Phase 2: for each
// expert in the range of down row blocks, each pass of up to SPP2 slots,
// each row block.  gen counts the passes of the current phase.
struct Walker {
  const int4* meta;
  Range r1, r2;
  int tpe1, upe2, NKR1, SPP1, SPP2;
  int phase;   // 1, 2, or 0 when done
  long u, se, uu;
  int d, passes, pass, kr, gen;
  int4 md;

  __device__ __forceinline__ void seg_begin() {
    for (;;) {
      if (phase == 0) return;
      const long end = phase == 1 ? r1.u1 : r2.u1;
      if (u < end) {
        const int per = phase == 1 ? tpe1 : upe2;
        d = (int)(u / per);
        se = min(end, (long)(d + 1) * per);
        md = meta[d];
        const int spp = phase == 1 ? SPP1 : SPP2;
        passes = (md.z + spp - 1) / spp;
        pass = 0;
        uu = u;
        kr = 0;
        return;
      }
      if (phase == 1) {
        phase = 2;
        u = r2.u0;
        gen = 0;
      } else {
        phase = 0;
      }
    }
  }
  __device__ __forceinline__ void init(const int4* m, Range a, Range b, int t1, int u2, int nkr, int s1, int s2) {
    meta = m;
    r1 = a;
    r2 = b;
    tpe1 = t1;
    upe2 = u2;
    NKR1 = nkr;
    SPP1 = s1;
    SPP2 = s2;
    phase = 1;
    u = r1.u0;
    gen = 0;
    seg_begin();
  }
  __device__ __forceinline__ void next() {
    if (phase == 1 && ++kr < NKR1) return;
    kr = 0;
    if (++uu < se) return;
    ++gen;
    if (++pass < passes) {
      uu = u;
      return;
    }
    u = se;
    seg_begin();
  }
  __device__ __forceinline__ bool done() const { return phase == 0; }
  __device__ __forceinline__ int pos0() const { return md.y + pass * (phase == 1 ? SPP1 : SPP2); }
  __device__ __forceinline__ int nslots() const {
    const int spp = phase == 1 ? SPP1 : SPP2;
    return min(spp, md.z - pass * spp);
  }
};

// ------------------------------------------------------- warp slices ----
// The MMAs of one item's two K blocks (nvb of them valid) of one 16-row tile
// against 8 activation columns at col (f16, 32 bytes per lane per 64-wide
// chunk): weights wa (rows g) and wb (rows g + 8), 16 bytes per lane per
// chunk in the fragment order of afrag.  K block j's partial is scaled once:
// rows g by slo(j) * colscale, rows g + 8 by shi(j) * colscale, where
// slo(j), shi(j) come from lane j (slo) and lane j (shi).
__device__ __forceinline__ void mma_item(const uint4 (&wa)[4], const uint4 (&wb)[4], const uint8_t* col, int kb0,
                                         int nvb, bool has_col, float slo, float shi, const float (&c0)[2],
                                         const float (&c1)[2], float (&acc)[4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j >= nvb) break;
    float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      const int kk = (kb0 + j) * 128 + ch * 64;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (has_col) {
        x0 = lds128(col + 2 * kk);
        x1 = lds128(col + 2 * kk + 16);
      }
      chunk_mma(b0, b1, wa[2 * j + ch], wb[2 * j + ch], x0, x1);
    }
    const float sl = __shfl_sync(0xffffffffu, slo, j);
    const float sh = __shfl_sync(0xffffffffu, shi, j);
    acc[0] = fmaf(sl * c0[j], b0[0] + b1[0], acc[0]);
    acc[1] = fmaf(sl * c1[j], b0[1] + b1[1], acc[1]);
    acc[2] = fmaf(sh * c0[j], b0[2] + b1[2], acc[2]);
    acc[3] = fmaf(sh * c1[j], b0[3] + b1[3], acc[3]);
  }
}

// ------------------------------------------------------------ the kernel --
template <bool ACT8, bool BIAS>
__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(const __grid_constant__ FusedArgs p) {
  extern __shared__ __align__(1024) uint8_t sm[];
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
  const int nkb1 = a.H >> 7, nkb2 = a.I >> 7;
  // per x buffer: token exponents [SPP1] then W8A8 group scales [SPP1][nkb1]
  int* xaux = reinterpret_cast<int*>(sm + c.o_xaux);
  auto xexp = [&](int b) { return xaux + b * (c.SPP1 * (1 + nkb1)); };
  auto xsc = [&](int b) { return reinterpret_cast<float*>(xaux + b * (c.SPP1 * (1 + nkb1)) + c.SPP1); };
  int* hexp = xaux + 2 * c.SPP1 * (1 + nkb1);   // [2][4] per-slot h exponents
  uint8_t* xbuf0 = act;
  uint8_t* hraw = act;                               // phase 2: raw h rows [SPP2][4I]
  uint8_t* hconv0 = act + c.SPP2 * 4 * a.I;          // phase 2: [2][8][HP]

  if (threadIdx.x == 0) {
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
  const int tpe1 = a.I >> 3;                        // gate/up tiles of 8 row pairs per expert
  const int upe2 = a.H / (16 * c.NT2);              // down row blocks per expert

  if (warp == kAct) {
    // ============================================ activation warp ====
    const int D = route_smem(a, c, sm, p.status, lane);
    if (lane == 0) B.D = D;
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.route);
    const Range r1 = cta_range(D, tpe1, cta, G), r2 = cta_range(D, upe2, cta, G);
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
      const int d = (int)(u / tpe1);
      const long se = min(r1.u1, (long)(d + 1) * tpe1);
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
    int gh = 0;
    for (long u = r2.u0; ok && u < r2.u1;) {
      const int d = (int)(u / upe2);
      const long se = min(r2.u1, (long)(d + 1) * upe2);
      const int4 md = meta_s[d];
      const int passes = (md.z + c.SPP2 - 1) / c.SPP2;
      const uint32_t target = (uint32_t)(tpe1 * ((md.z + c.SPP1 - 1) / c.SPP1));
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
    // ================================== compute warps 0-7, finisher 9 ====
    const bool fin = warp == kFin;
    const int w = fin ? 0 : warp;
    const int g = lane >> 2, cq = lane & 3;
    bool ok = warp_wait(&B.route, 0, lane);
    const int D = ok ? *(volatile int*)&B.D : 0;
    const Range r1 = cta_range(D, tpe1, cta, G), r2 = cta_range(D, upe2, cta, G);
    const int NT2 = c.NT2, KS2 = c.KS2;
    const int tt = w % NT2, ks = w / NT2;   // this warp's down tile and K split
    // the buffer (x or h) of the pass the walk is in: wait for it when a pass
    // starts, release the previous one
    int cur_phase = 0, cur_gen = -1;
    auto enter_pass = [&](const Walker& W) -> bool {
      if (W.phase == cur_phase && W.gen == cur_gen) return true;
      if (cur_phase != 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(cur_phase == 1 ? &B.xempty[cur_gen & 1] : &B.hempty[cur_gen & 1]);
      }
      cur_phase = W.phase;
      cur_gen = W.gen;
      if (cur_phase == 0) return true;
      uint64_t* full = cur_phase == 1 ? &B.xfull[cur_gen & 1] : &B.hfull[cur_gen & 1];
      return warp_wait(full, (cur_gen >> 1) & 1, lane);
    };
    int m = 0;   // item sequence = reduction step (double-buffered)

    if (!fin) {
      // ------------------------------------------ compute warps
      // one item's weights for this warp: two K blocks of rows g and g + 8
      // of its 16-row tile, loaded straight from global memory, and the
      // block scales (gate/up: lanes 0, 1 gate, lanes 2, 3 up; down: lanes 0, 1)
      auto issue = [&](const Walker& L, uint4 (&wa)[4], uint4 (&wb)[4], float& sv) {
        const int e = L.md.x;
        if (L.phase == 1) {
          const int i0 = (int)(L.uu % tpe1) * 8;
          const int kbA = 16 * L.kr + 2 * w;
          const uint8_t* pa = a.w13 + ((int64_t)e * 2 * a.I + i0 + g) * a.H + cq * 16;
          const uint8_t* pb = pa + (int64_t)a.I * a.H;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kb = kbA + (i >> 1);
            const int kk = kb * 128 + (i & 1) * 64;
            wa[i] = kb < nkb1 ? ldg_stream(pa + kk) : make_uint4(0, 0, 0, 0);
            wb[i] = kb < nkb1 ? ldg_stream(pb + kk) : make_uint4(0, 0, 0, 0);
          }
          const int kb = kbA + (lane & 1);
          const int rb = lane < 2 ? (i0 >> 7) : ((a.I + i0) >> 7);
          sv = lane < 4 && kb < nkb1 ? bf16_bits_to_f32(__ldg(a.w13s + (int64_t)e * a.s13_exp + (int64_t)rb * a.s13_row + kb))
                                     : 0.f;
        } else {
          const int n0 = (int)(L.uu % upe2) * 16 * NT2 + tt * 16;
          const int kbA = 2 * ks;
          const uint8_t* pa = a.w2 + ((int64_t)e * a.H + n0 + g) * a.I + cq * 16;
          const uint8_t* pb = pa + 8 * (int64_t)a.I;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kb = kbA + (i >> 1);
            const int kk = kb * 128 + (i & 1) * 64;
            wa[i] = kb < nkb2 ? ldg_stream(pa + kk) : make_uint4(0, 0, 0, 0);
            wb[i] = kb < nkb2 ? ldg_stream(pb + kk) : make_uint4(0, 0, 0, 0);
          }
          const int kb = kbA + lane;
          sv = lane < 2 && kb < nkb2
                   ? bf16_bits_to_f32(__ldg(a.w2s + (int64_t)e * a.s2_exp + (int64_t)(n0 >> 7) * a.s2_row + kb))
                   : 0.f;
        }
      };
      // one item: the MMAs, then this warp's partial sums to the finisher
      auto compute = [&](const Walker& W, const uint4 (&wa)[4], const uint4 (&wb)[4], float sv) -> bool {
        if (!enter_pass(W)) return false;
        const int b = W.gen & 1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (W.phase == 1) {
          const int nx = W.nslots();
          const int kbA = 16 * W.kr + 2 * w;
          const int nvb = max(0, min(2, nkb1 - kbA));
          float c0[2] = {1.f, 1.f}, c1[2] = {1.f, 1.f};
          if (ACT8) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (kbA + j >= nkb1) break;
              if (2 * cq < nx) c0[j] = xsc(b)[(2 * cq) * nkb1 + kbA + j];
              if (2 * cq + 1 < nx) c1[j] = xsc(b)[(2 * cq + 1) * nkb1 + kbA + j];
            }
          }
          const float shi = __shfl_sync(0xffffffffu, sv, (lane & 1) + 2);
          mma_item(wa, wb, xbuf0 + b * c.SPP1 * c.XP + g * c.XP + cq * 32, kbA, nvb, g < nx, sv, shi, c0, c1, acc);
        } else {
          const int nh = W.nslots();
          const int kbA = 2 * ks;
          const int nvb = max(0, min(2, nkb2 - kbA));
          const float one[2] = {1.f, 1.f};
          mma_item(wa, wb, hconv0 + b * 8 * c.HP + g * c.HP + cq * 32, kbA, nvb, (g & 3) < nh, sv, sv, one, one,
                   acc);
        }
        const int rb = m & 1;
        if (m >= 2 && !warp_wait(&B.rempty[rb], ((m >> 1) - 1) & 1, lane)) return false;
        *reinterpret_cast<float4*>(red + ((rb * kCons + w) * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.rfull[rb]);
        ++m;
        return !aborted();
      };
      // warp 0, lane 0: bulk prefetches into L2, kPF items ahead of the loads
      // (a gate/up tile once, at its first K round of its first pass; a down
      // item's rows at its first pass); not for banks in host memory
      Walker P;
      P.init(meta_s, r1, r2, tpe1, upe2, c.NKR1, c.SPP1, c.SPP2);
      auto prefetch_next = [&]() {
        if (P.done()) return;
        if (!a.host_weights && w == 0 && lane == 0 && P.pass == 0) {
          const int e = P.md.x;
          if (P.phase == 1 && P.kr == 0) {
            const int i0 = (int)(P.uu % tpe1) * 8;
            const uint8_t* pa = a.w13 + ((int64_t)e * 2 * a.I + i0) * a.H;
            prefetch_l2(pa, (uint32_t)(8 * a.H));
            prefetch_l2(pa + (int64_t)a.I * a.H, (uint32_t)(8 * a.H));
          } else if (P.phase == 2) {
            const int nb = (int)(P.uu % upe2) * 16 * NT2;
            prefetch_l2(a.w2 + ((int64_t)e * a.H + nb) * a.I, (uint32_t)(16 * NT2 * a.I));
          }
        }
        P.next();
      };
      for (int j = 0; j < kPF; ++j) prefetch_next();
      Walker L, W;
      L.init(meta_s, r1, r2, tpe1, upe2, c.NKR1, c.SPP1, c.SPP2);
      W = L;
      uint4 wa[kPD][4], wb[kPD][4];
      float sv[kPD];
#pragma unroll
      for (int j = 0; j < kPD; ++j) {
        if (!L.done()) {
          issue(L, wa[j], wb[j], sv[j]);
          L.next();
        }
      }
      while (ok && !W.done()) {
#pragma unroll
        for (int j = 0; j < kPD; ++j) {
          if (!ok || W.done()) break;
          prefetch_next();
          ok = compute(W, wa[j], wb[j], sv[j]);
          W.next();
          if (!L.done()) {
            issue(L, wa[j], wb[j], sv[j]);
            L.next();
          }
        }
      }
      if (ok) enter_pass(W);   // release the last pass's buffer
    } else {
      // ------------------------------------------ finisher
      Walker W;
      W.init(meta_s, r1, r2, tpe1, upe2, c.NKR1, c.SPP1, c.SPP2);
      float tacc[4] = {0.f, 0.f, 0.f, 0.f};   // a gate/up tile's sums over its K rounds
      bool signalled = false;
      // after the last gate/up tile: this CTA's (tile, pass) counts per routed
      // expert, once its h rows are visible
      auto signal_h = [&]() {
        signalled = true;
        __threadfence();
        __syncwarp();
        if (aborted()) return;
        const int dlo = (int)(r1.u0 / tpe1), dhi = r1.u1 > r1.u0 ? (int)((r1.u1 - 1) / tpe1) : dlo - 1;
        for (int d = dlo + lane; d <= dhi; d += 32) {
          const long ua = max(r1.u0, (long)d * tpe1), ub = min(r1.u1, (long)(d + 1) * tpe1);
          const int passes = (meta_s[d].z + c.SPP1 - 1) / c.SPP1;
          atomicAdd(p.ctr.c1 + d, (uint32_t)((ub - ua) * passes));
        }
      };
      while (ok && !W.done()) {
        if (W.phase == 2 && !signalled) signal_h();
        if (!enter_pass(W)) {
          ok = false;
          break;
        }
        const int b = W.gen & 1;
        const int rb = m & 1;
        if (!warp_wait(&B.rfull[rb], (m >> 1) & 1, lane)) {
          ok = false;
          break;
        }
        const int e = W.md.x;
        const int pos0 = W.pos0(), ns = W.nslots();
        if (W.phase == 1) {
#pragma unroll 4
          for (int j = 0; j < kCons; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(red + ((rb * kCons + j) * 32 + lane) * 4);
            tacc[0] += v.x;
            tacc[1] += v.y;
            tacc[2] += v.z;
            tacc[3] += v.w;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.rempty[rb]);
          if (W.kr == c.NKR1 - 1) {
            const int i0 = (int)(W.uu % tpe1) * 8;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (2 * cq + j >= ns) continue;
              const int sx = xexp(b)[2 * cq + j];
              float gv = ldexpf(tacc[j], sx);
              float uv = ldexpf(tacc[2 + j], sx);
              if (BIAS && a.b13) {   // either bias may be absent
                const float* br = a.b13 + (int64_t)e * a.b13_ld + i0 + g;
                gv += __ldg(br);
                uv += __ldg(br + a.I);
              }
              p.h[(int64_t)(pos0 + 2 * cq + j) * a.I + i0 + g] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
            tacc[0] = tacc[1] = tacc[2] = tacc[3] = 0.f;
          }
        } else {
          // output slots of this lane (lanes cq < 2: slots 2cq, 2cq + 1)
          int so[2] = {-1, -1}, es[2] = {0, 0};
          float wo[2] = {0.f, 0.f};
          if (cq < 2) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (2 * cq + j < ns) {
                so[j] = perm_s[pos0 + 2 * cq + j];
                wo[j] = wts_s[so[j]];
                es[j] = hexp[b * 4 + 2 * cq + j];
              }
          }
          const int nb = (int)(W.uu % upe2) * 16 * NT2;
          for (int t2 = 0; t2 < NT2; ++t2) {
            float tot[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k2 = 0; k2 < KS2; ++k2) {
              const float4 v =
                  *reinterpret_cast<const float4*>(red + ((rb * kCons + t2 + k2 * NT2) * 32 + lane) * 4);
              tot[0] += v.x;
              tot[1] += v.y;
              tot[2] += v.z;
              tot[3] += v.w;
            }
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
          if (lane == 0) mbar_arrive(&B.rempty[rb]);
        }
        ++m;
        W.next();
        if (aborted()) ok = false;
      }
      if (ok) {
        if (!signalled) signal_h();
        enter_pass(W);   // release the last pass's buffer
      }
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
  o += 2 * kCons * 32 * 4 * 4;
  c.o_xaux = o;
  o += al128(4 * (2 * c.SPP1 * (1 + H / 128) + 8));
  c.o_act = o;
  const int xb = 2 * c.SPP1 * c.XP;
  const int hb = c.SPP2 * 4 * I + 2 * 8 * c.HP;
  o += al128(xb > hb ? xb : hb);
  c.smem = o;
  return o <= kFSmemLimit;
}

// K rounds of 16 blocks for the gate/up tiles; for the down items two K
// blocks per warp, as many 16-row tiles as the eight warps then cover
// (the down projection's K, I, up to 2048); passes of as many slots as fit.
bool choose_cfg(int H, int I, int S, int E, FusedCfg& c) {
  const int nkb2 = I / 128;
  if (nkb2 > 16) return false;
  c.S = S;
  c.DMAX = S < E ? S : E;
  c.XP = 2 * H + 16;   // == 16 mod 128: conflict-free fragment loads
  c.HP = 2 * I + 16;
  c.NKR1 = (H / 128 + 15) / 16;
  c.KS2 = 1;
  while (2 * c.KS2 < nkb2) c.KS2 <<= 1;
  c.NT2 = kCons / c.KS2;
  c.SPP2 = 4;
  for (int spp = 8; spp >= 1; --spp) {
    c.SPP1 = spp;
    if (place(c, H, I)) return true;
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
  if (a.dbg_wait_ns) {
    const uint64_t v = a.dbg_wait_ns;
    if ((err = note_error(cudaMemcpyToSymbolAsync(g_wait_limit_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, st),
                          "decode wait limit")))
      return err;
  }
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
  if (a.dbg_wait_ns) {
    const uint64_t v = kWaitTimeoutNs;
    if ((err = note_error(cudaMemcpyToSymbolAsync(g_wait_limit_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, st),
                          "decode wait limit")))
      return err;
  }
  return cudaSuccess;
}

}  // namespace moe
