// kernels.h -- host-side launchers of the CUDA kernels (internal to the
// library; the public interface is include/moe_fp8_block.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moe_fp8_block.h"

namespace moe {

// Arguments shared by the kernels of one forward call.  All pointers are
// device memory.  Scale banks are bf16 bit patterns.
struct LayerArgs {
  const uint16_t* hidden;      // bf16 [T, H], row stride hidden_ld
  int64_t hidden_ld;
  const int32_t* ids;          // [T, k]
  const float* wts;            // [T, k]
  const uint8_t* w13;          // e4m3 [E, 2I, H]
  const uint16_t* w13s;        // bf16 [E, 2I/128, s13_row], expert stride s13_exp
  int64_t s13_row, s13_exp;
  const uint8_t* w2;           // e4m3 [E, H, I]
  const uint16_t* w2s;         // bf16 [E, H/128, s2_row], expert stride s2_exp
  int64_t s2_row, s2_exp;
  uint16_t* out;               // bf16 [T, H]
  int T, k, H, I, E, S;        // S = T*k
  int act8 = 0;                // decode: 1 = e4m3 activations (W8A8), 0 = bf16 (W8A16)
  const float* b13 = nullptr;  // optional fp32 [E, 2I] MLP bias row [gate | up], expert stride b13_ld
  int64_t b13_ld = 0;
  const float* b2 = nullptr;   // optional fp32 [E, H] down-projection bias, expert stride b2_ld
  int64_t b2_ld = 0;
  // optional copies of the activation codes and group scales the path's own
  // quantiser produced (moe_fp8_block_forward_act_codes): e4m3 [T, H] and
  // fp32 [T, ceil(H/128)], both row-contiguous
  uint8_t* dbg_codes = nullptr;
  float* dbg_scales = nullptr;
  int decode_kernel = MOE_DECODE_KERNEL_CHAIN;   // moe_options.decode_kernel
  int host_weights = 0;        // w13, w2 and their scales are mapped page-locked host memory
  uint64_t dbg_wait_ns = 0;    // moe_options.debug_wait_timeout_us (0 = the default limit)
  int dbg_drop_stage = 0;      // moe_options.debug_drop_stage (0 = none)
};

// Routing lists produced by the route kernel (device int32 buffers).
struct RouteBufs {
  int32_t* counts;    // [E]
  int32_t* offsets;   // [E+1]
  int32_t* perm;      // [S]
  int32_t* inv;       // [S]
  int32_t* glist;     // [min(E,S)]
  int32_t* nd;        // [1]
  int4* meta = nullptr;     // [min(E,S)]: {expert, first routed position, slot count, 0} per
                            // distinct expert (optional)
  int32_t* mtp = nullptr;   // [E+1]: exclusive prefix of ceil(count/128) per expert (optional)
  int32_t* mtp2 = nullptr;  // [E+1]: exclusive prefix of ceil(ceil(count/128)/2), the pairs of
                            // 128-row tiles per expert (optional)
  // Per-pass work list of the decode down projection (optional; then nd
  // must have room for 2 ints and mtp/mtp2 are not written): the routed
  // experts split into passes of at most spp consecutive slots, one entry
  // {expert, first routed position, slot count, passes of that expert} per
  // pass, in ascending (expert, pass) order; nd[1] receives the entry count.
  int4* vmeta = nullptr;    // [S]
  int spp = 0;
};

// Scratch of the decode path.
struct DecodeBufs {
  uint16_t* xh;       // f16 [T, H]: activations scaled by 2^-xexp[t]
  int32_t* xexp;      // [T]
  float* xs;          // [T, H/128]: W8A8 activation group scales (decode_act e4m3)
  float* h;           // [S, I] in routed (perm) order
  float* ybuf;        // [S, H] in slot order, times the slot's top-k weight
  uint32_t* counters = nullptr;   // fused kernel: kFusedCounterWords words, zero between forwards
  int4* vmeta = nullptr;          // [S]: the down projection's per-pass work list (RouteBufs::vmeta)
};

// Scratch of the prefill path.  Per-row buffers hold `rows` rows in the
// expert-padded routed order: expert e's slots start at row 128*mtp[e].
struct PrefillBufs {
  uint8_t* xq;        // e4m3 [rows, H] activation codes of each routed slot's token
  float* xsT;         // [H/128, rows] their scales, K-block major
  uint8_t* hq;        // e4m3 [rows, I] h codes
  float* hsT;         // [I/128, rows] h scales, K-block major
  uint16_t* ys;       // bf16 [rows, H] down-projection output of each row (not yet weighted)
  int32_t* pinv;      // [S] row of each slot, -1 for a skipped slot
  float* wsc13;       // [E, H/128, I/128, 4] fp32 (gate, up, 0, 0) block scales
  float* wsc2;        // [E, I/128, ceil(H/256), 4] fp32 (row block 2p, 2p+1, 0, 0) block scales
  int64_t rows;       // row capacity, prefill_rows(S, E)
};

// Rows the expert-padded layout can need for S slots over E experts.
int64_t prefill_rows(int64_t S, int E);

int num_sms(int device);

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) on the
// current device, skipped when an earlier call there already allowed at
// least `bytes` (it costs host time on every forward otherwise).
// clear_smem_attributes forgets what was set (moe_fp8_block_release).
cudaError_t set_max_smem(const void* func, int bytes);
void clear_smem_attributes();

// Argument checks of moe_fp8_block_forward for other entry points: fills
// *args and, when T > 0, the current device (which must be sm_103).
int validate_forward(const moe_tensor* hidden, const moe_tensor* topk_ids, const moe_tensor* topk_weights,
                     const moe_tensor* w13, const moe_tensor* w13_scale, int64_t w13_scale_stride,
                     const moe_tensor* w2, const moe_tensor* w2_scale, int64_t w2_scale_stride,
                     const moe_tensor* out, LayerArgs* args, int* device);
// Text returned by moe_fp8_block_last_error_detail on this thread.
void set_error_detail(const char* text);
// What moe_fp8_block_last_path / moe_fp8_block_last_launches report for the
// last successful call on this thread.
void record_call(int path, int launches);

// Stage events of moe_fp8_block_set_stage_events (per host thread).
struct StageEvents {
  cudaEvent_t ev[16];
  int n = 0;
};
StageEvents& stage_events();
// Record stage event i on st if one was requested; returns true while stage
// events are active (the launchers then drop programmatic dependent launch).
bool stage_mark(cudaStream_t st, int i);

// Record a CUDA failure for moe_fp8_block_last_error_detail; with
// MOE_FP8_BLOCK_SYNC_CHECK=1 also synchronise and check after each launch.
cudaError_t note_error(cudaError_t e, const char* stage);
cudaError_t launch_check(cudaError_t launch_err, cudaStream_t st, const char* stage);

// Routing lists.  With `scratch` (2 * route_chunks(S) * E ints) large slot
// counts use the three-kernel route; without it one CTA does everything.
// Adds the number of launches to *launches (if given).
constexpr int kRouteSingleMax = 2048;    // slots one CTA handles
constexpr int kRouteChunk = 1024;        // slots per chunk of the three-kernel route
constexpr int kRouteMaxChunks = 512;
int route_chunks(int S);
cudaError_t launch_route(const int32_t* ids, int S, int E, const RouteBufs& rb, uint32_t* status,
                         int32_t* scratch, cudaStream_t st, int* launches);
cudaError_t launch_widen(const uint8_t* codes, int64_t n, float* out, cudaStream_t st);

// Whether the decode path can stage rows of this layer shape in shared memory.
bool decode_supported(int H, int I);
// Ring stages the decode gate/up stream gets for this shape (0 if unsupported).
int decode_ring_stages(int H, int I);
// Row pairs of one decode gate/up unit (ring stage) for hidden width H: 8
// while 8 whole rows of gate and of up fit 16 KiB each (H <= 2048).
int decode_unit_rows(int H);

// The fused decode kernel (one launch per forward) handles up to this many
// slots, when its shared-memory layout fits; larger slot counts take the
// chained kernels.  It keeps 2 + min(E, S) counters in global memory.
constexpr int kFusedMaxSlots = 4096;
constexpr int kFusedCounterWords = 2 + 4096;
bool fused_decode_ok(int T, int k, int H, int I, int E);
size_t fused_counter_words(int S, int E);
cudaError_t launch_decode_fused(const LayerArgs& a, float* h, float* ybuf, uint32_t* counters, uint32_t* status,
                                int device, cudaStream_t st, int* launches);

// Decode (W8A16) path: the fused kernel when it applies (and db.counters is
// set), else prep (route + f16 activations), GEMM1+silu*up, GEMM2, combine.
// Adds the number of launches to *launches.
cudaError_t launch_decode(const LayerArgs& a, const RouteBufs& rb, const DecodeBufs& db, uint32_t* status,
                          int device, cudaStream_t st, int* launches);

// Prefill (W8A8) path.
cudaError_t launch_act_quant(const uint16_t* x, int64_t ld, int R, int K, uint8_t* codes, float* scales,
                             cudaStream_t st, bool pdl);
cudaError_t launch_prefill(const LayerArgs& a, const RouteBufs& rb, const PrefillBufs& pb, int32_t* route_scratch,
                           uint32_t* status, int device, cudaStream_t st, int* launches);
// After a prefill forward on the same buffers: copy each token's activation
// codes and scales from the GEMM input rows of one of its routed slots (slot
// t mod k, else the next valid one) into a.dbg_codes / a.dbg_scales.
cudaError_t launch_prefill_act_codes(const LayerArgs& a, const PrefillBufs& pb, cudaStream_t st);

// Shared-memory bytes the route kernel needs for E experts with nthreads.
size_t route_smem_bytes(int E, int nthreads);
int route_threads(int E);

}  // namespace moe
