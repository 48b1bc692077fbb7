/*
 * moe_fp8_block.h -- C ABI of the block-FP8 mixture-of-experts layer forward
 * for NVIDIA GB300 (sm_103a).
 *
 * The layer (one call of moe_fp8_block_forward):
 *   for every token t and routed slot j (expert e = topk_ids[t,j]):
 *     [gate; up] = dequant(w13[e]) . x_t           (one fused projection)
 *     h          = silu(gate) * up
 *     y_{t,j}    = dequant(w2[e]) . h              (fp32 accumulation)
 *   out_t = sum_j topk_weights[t,j] * y_{t,j}      (fixed order, no atomics)
 * Only the g = min(E, T*k) routed experts are read ("gathered-expert FP8 MoE
 * combine", fp8-moe-gather page, sections Problem and The fix).
 *
 * Weight format (FreeToken PR #662, PR body): every expert bank is e4m3
 * (float8 e4m3fn bytes) row-major [rows, K], K contiguous per output row,
 * with a bf16 scale for each 128 x 128 block.  The scale bank's row stride may be
 * padded (same PR, commit "honor padded fp8 scale strides"), so it is passed
 * explicitly and never recomputed from K.  w13 stacks the gate and up
 * projections along the output rows: rows [0, I) gate, rows [I, 2I) up
 * (tpu-inference PR #3040, review of the bias DMA: gate half at
 * n_id*tile_n1, up half at out_n1 + n_id*tile_n1).
 *
 * Paths (chosen per call; the choice is readable through
 * moe_fp8_block_last_path):
 *   decode  (W8A16): with a caller gate ratio, taken while T*k <= E*ratio
 *     (fp8-moe-gather page, environment-variable table, where the ratio is
 *     0.4).  By default, from measurements of both paths on GB300: taken
 *     while T*k <= E, the layer's hidden rows leave the decode weight
 *     stream at least 4 shared-memory ring stages (H = 2048: yes; H = 7168:
 *     no, where the prefill path streams faster), and its units are whole
 *     8-row-pair blocks (H <= 2048) or the batch routes at most 8 slots
 *     (H = 2560 with hot experts: decode only at T*k = 8).  bf16
 *     activations, e4m3 weights widened in registers, fp32 accumulation and
 *     fp32 h.
 *   prefill (W8A8): activations quantised per token per 128 columns with a
 *     dynamic scale amax/448 (fp8-moe-gather page, "Affects": dynamic
 *     activation scales), grouped FP8 tensor-core GEMMs, h quantised the same
 *     way, fp32 accumulation.
 *
 * Conventions common to all entry points:
 *   - Every pointer is DEVICE memory unless the entry point says otherwise.
 *     The caller owns every buffer it passes; the library never frees them.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous unless stated otherwise.  No entry point
 *     that takes a stream synchronises it, except moe_fp8_block_device_status
 *     and moe_fp8_block_forward_hostio.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  All argument
 *     checks run on the host before anything is enqueued; on error nothing is
 *     enqueued and the output is untouched.  No C++ exception crosses the ABI.
 *   - Inputs are never modified.  `out` is fully overwritten.
 *   - The library keeps a workspace per (device, stream), grown on demand.
 *     Growth calls cudaMalloc, which is not allowed while the stream is being
 *     captured into a CUDA graph: call moe_fp8_block_reserve first with the
 *     largest sizes, then capture (growth during capture returns
 *     MOE_ERR_CAPTURE_GROW).  Calls on one stream are ordered by the stream;
 *     calls on different streams use different workspaces.
 */
#ifndef MOE_FP8_BLOCK_H
#define MOE_FP8_BLOCK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight-format / ABI identifier.  The Python binding refuses a library whose
 * moe_fp8_block_abi_version() differs, so a stale build fails loudly instead
 * of reading the banks with the wrong layout (FreeToken PR #662, PR body: the
 * weight-format ABI probe max_weight_format_id). */
#define MOE_FP8_BLOCK_ABI_VERSION 4

/* Element types of moe_tensor.dtype. */
typedef enum {
  MOE_BF16 = 1,  /* bfloat16 (2 bytes)                                   */
  MOE_F32 = 2,   /* IEEE binary32                                        */
  MOE_E4M3 = 3,  /* float8 e4m3fn byte (codes 0x7F/0xFF are NaN)         */
  MOE_I32 = 4    /* int32                                                */
} moe_dtype;

/* A strided view of a buffer.  Strides are in ELEMENTS, shape[i] >= 0. */
typedef struct {
  void* data;         /* device pointer (host pointer where stated)       */
  int32_t ndim;       /* 1..4                                             */
  int32_t dtype;      /* moe_dtype                                        */
  int64_t shape[4];
  int64_t stride[4];
} moe_tensor;

/* Return codes. */
enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,          /* a required pointer or descriptor is NULL         */
  MOE_ERR_DTYPE = -2,         /* wrong element type                               */
  MOE_ERR_SHAPE = -3,         /* inconsistent shapes; unsupported H or I          */
  MOE_ERR_ALIGN = -4,         /* a base pointer is not 16-byte aligned            */
  MOE_ERR_STRIDE = -5,        /* unsupported stride (see each argument)           */
  MOE_ERR_ALIAS = -6,         /* out overlaps an input                            */
  MOE_ERR_CAPTURE_GROW = -7,  /* workspace must grow while the stream is captured */
  MOE_ERR_CUDA = -8,          /* a CUDA runtime/driver call failed                */
  MOE_ERR_ARG = -9,           /* another invalid argument (sizes, options)        */
  MOE_ERR_DEVICE = -10        /* unsupported device (not compute capability 10.3) */
};

/* Paths, as reported by moe_fp8_block_last_path and forced by options. */
enum { MOE_PATH_NONE = 0, MOE_PATH_DECODE = 1, MOE_PATH_PREFILL = 2 };

/* Bits of the device status word (moe_fp8_block_device_status). */
enum {
  MOE_STATUS_BAD_ID = 1u,    /* a topk id >= E was seen; its slot was skipped   */
  MOE_STATUS_TIMEOUT = 2u    /* a bounded pipeline wait gave up; output invalid */
};

/* Activation formats of the decode path (moe_options.decode_act). */
enum {
  /* W8A16: the bf16 activations enter the up/gate projection as they are
   * (FreeToken PR #662, the CPU and GPU decode kernels). */
  MOE_DECODE_ACT_BF16 = 0,
  /* W8A8: each token is quantised per 128-column group to e4m3 with a
   * dynamic fp32 scale amax/448 (the prefill rule) and the up/gate
   * projection multiplies e4m3 by e4m3; h stays fp32 for the down projection
   * (the Gaudi path of the fp8-moe-gather page, "The fix"). */
  MOE_DECODE_ACT_E4M3 = 1
};

/* Kernels of the decode path (moe_options.decode_kernel). */
enum {
  /* Four chained launches: routing and activation prep, gate/up projection,
   * down projection, combine (programmatic dependent launch between them). */
  MOE_DECODE_KERNEL_CHAIN = 0,
  /* One persistent launch for the whole forward (routing in every CTA's
   * shared memory, per-expert hand-off of h between the projections, a
   * grid-wide count before the combine).  Slot counts it cannot stage in
   * shared memory fall back to the chain. */
  MOE_DECODE_KERNEL_FUSED = 1
};

/* Options of moe_fp8_block_forward_ex.  Zero-initialise, then set fields. */
typedef struct {
  float gate_ratio;   /* decode while T*k <= E*gate_ratio; <= 0 -> measured rule */
  int32_t force_path; /* MOE_PATH_NONE (gate decides), _DECODE or _PREFILL     */
  int32_t decode_act; /* MOE_DECODE_ACT_BF16 (default) or _E4M3; the prefill  */
                      /* path always quantises activations (and h)             */
  int32_t decode_kernel;         /* MOE_DECODE_KERNEL_CHAIN (default) or _FUSED */
  /* Failure-detection test aids of the decode path (0 = off).  Every
   * pipeline wait of the decode kernels gives up after a bounded time (1 s
   * by default) and raises MOE_STATUS_TIMEOUT; debug_wait_timeout_us
   * shortens that limit for this call (1..1000000 us).  debug_drop_stage = n
   * makes the gate/up weight producer of the chained decode kernels skip
   * its n-th ring stage (1-based): it neither copies the stage nor arrives
   * on the stage's barrier, so the consumers' wait for it runs out.  The
   * kernels then wind down (every copy already issued lands first) and the
   * call's output is invalid; moe_fp8_block_device_status reports
   * MOE_STATUS_TIMEOUT.  Calls on other streams that overlap a call with a
   * shortened limit may use it too. */
  int32_t debug_wait_timeout_us;
  int32_t debug_drop_stage;
  int32_t reserved[2];           /* must be zero                                */
} moe_options;

/*
 * moe_fp8_block_forward -- the layer forward.
 *
 *  hidden        bf16 [T, H], stride[1] == 1, stride[0] >= H.  T >= 0.
 *  topk_ids      int32 [T, k], contiguous.  An id < 0 skips its slot (it adds
 *                nothing); an id >= E skips its slot and sets
 *                MOE_STATUS_BAD_ID.  A token may name one expert twice: each
 *                slot counts.
 *  topk_weights  fp32 [T, k], contiguous; used as given (no renormalisation).
 *  w13           e4m3 [E, 2I, H], contiguous; rows [0,I) gate, [I,2I) up.
 *  w13_scale     bf16 [E, ceil(2I/128), >= ceil(H/128)]; stride[2] == 1,
 *                stride[1] == w13_scale_stride >= ceil(H/128),
 *                stride[0] >= ceil(2I/128) * w13_scale_stride.  The blocks
 *                are 128 rows of the stacked [gate; up] bank, so when I is
 *                not a multiple of 128 up row i uses block (I + i) / 128.
 *  w13_scale_stride  row stride of w13_scale in elements (read from the tensor
 *                by the caller; it may be padded).
 *  w2            e4m3 [E, H, I], contiguous.
 *  w2_scale      bf16 [E, ceil(H/128), >= ceil(I/128)]; stride rules as for
 *                w13_scale with w2_scale_stride >= ceil(I/128).
 *  out           bf16 [T, H], contiguous; must not overlap any input.
 *  stream        cudaStream_t.
 * H and I in [128, 8192], H a multiple of 64 and I of 16.  A layer whose
 * H or I is not a multiple of 128 ("ragged K", FreeToken PR #662, Tests:
 * the last 128-wide K block of a projection is partial) runs on the decode
 * path when both are multiples of 64 (its last K block is one 64-wide
 * chunk), else on the prefill path.  Forcing decode on a layer the decode
 * kernels do not take (such a ragged layer, or an I whose down-projection
 * staging outgrows their shared memory, above about 2560) returns
 * MOE_ERR_SHAPE; the single-kernel decode option and the host-resident
 * entry point take multiples of 128 only.  k in [1, 64];
 * E in [1, 4096]; T*k <= 2^24.  Every
 * base pointer must be 16-byte aligned.  T == 0 is a no-op returning MOE_OK.
 */
int moe_fp8_block_forward(const moe_tensor* hidden, const moe_tensor* topk_ids,
                          const moe_tensor* topk_weights, const moe_tensor* w13,
                          const moe_tensor* w13_scale, int64_t w13_scale_stride,
                          const moe_tensor* w2, const moe_tensor* w2_scale,
                          int64_t w2_scale_stride, moe_tensor* out, void* stream);

/* As moe_fp8_block_forward, with options (NULL = defaults). */
int moe_fp8_block_forward_ex(const moe_tensor* hidden, const moe_tensor* topk_ids,
                             const moe_tensor* topk_weights, const moe_tensor* w13,
                             const moe_tensor* w13_scale, int64_t w13_scale_stride,
                             const moe_tensor* w2, const moe_tensor* w2_scale,
                             int64_t w2_scale_stride, moe_tensor* out, void* stream,
                             const moe_options* opt);

/*
 * moe_fp8_block_forward_bias -- moe_fp8_block_forward_ex with MLP biases
 * (tpu-inference PR #3040, review of the bias DMA: the up/gate bias row is
 * laid out like the stacked weight rows, gate biases first and the up
 * biases at offset I; the down projection's bias has no such split):
 *     gate = Wg . x + w13_bias[e, 0:I]
 *     up   = Wu . x + w13_bias[e, I:2I]
 *     y    = W2 . silu(gate) * up + w2_bias[e]
 *     out_t = sum_j topk_weights[t,j] * y_{t,j}
 *  w13_bias  fp32 [E, 2I] or NULL (no gate/up bias).
 *  w2_bias   fp32 [E, H] or NULL (no down-projection bias).
 * Each bias: stride[1] == 1; expert stride stride[0] >= its row length and a
 * multiple of 4 elements (when E > 1); 16-byte aligned base; it must not
 * overlap `out` (MOE_ERR_ALIAS).  Other arguments, the options and the
 * return codes are those of moe_fp8_block_forward_ex.  With both biases
 * NULL the call is moe_fp8_block_forward_ex.
 */
int moe_fp8_block_forward_bias(const moe_tensor* hidden, const moe_tensor* topk_ids,
                               const moe_tensor* topk_weights, const moe_tensor* w13,
                               const moe_tensor* w13_scale, int64_t w13_scale_stride,
                               const moe_tensor* w2, const moe_tensor* w2_scale,
                               int64_t w2_scale_stride, const moe_tensor* w13_bias,
                               const moe_tensor* w2_bias, moe_tensor* out, void* stream,
                               const moe_options* opt);

/* As moe_fp8_block_forward_ex, but hidden, topk_ids, topk_weights and out
 * are HOST buffers; the weight banks stay device memory.  When all four are
 * page-locked (cudaHostAlloc, cudaHostRegister, torch pin_memory), 16-byte
 * aligned and `out` overlaps no input, the kernels read the inputs and write
 * the output in place, over the host link, with no staging copies.
 * Otherwise the inputs are copied to the workspace and the output back (a
 * pageable buffer copies synchronously).  Everything runs on `stream`; the
 * call returns after synchronising `stream`, with `out` filled. */
int moe_fp8_block_forward_hostio(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                 const moe_tensor* topk_weights, const moe_tensor* w13,
                                 const moe_tensor* w13_scale, int64_t w13_scale_stride,
                                 const moe_tensor* w2, const moe_tensor* w2_scale,
                                 int64_t w2_scale_stride, moe_tensor* out, void* stream,
                                 const moe_options* opt);

/*
 * moe_fp8_block_forward_host_experts -- the decode forward with the expert
 * banks held in HOST memory: the layer of moe_fp8_block_forward, where
 * w13, w13_scale, w2 and w2_scale (same shapes, strides and rules) are
 * page-locked host buffers (cudaHostAlloc, cudaHostRegister, torch
 * pin_memory) that the device can address, and hidden, topk_ids,
 * topk_weights and out stay device memory.  Serving block-fp8 experts
 * that do not fit, or are not kept, in device memory is the offload case of
 * FreeToken PR #662 (PR body: the cpu and hybrid backends); on GB300 the GPU
 * reads the host-resident banks itself over NVLink-C2C, with ordinary
 * 16-byte loads only (no bulk or tensor-map copies, no prefetches, of host
 * memory), so only the routed experts' weights cross the link.
 * The path is the single-launch decode kernel (W8A16, or W8A8 with
 * decode_act = MOE_DECODE_ACT_E4M3); options are those of
 * moe_fp8_block_forward_ex, and force_path = MOE_PATH_PREFILL is refused
 * (MOE_ERR_ARG).  Returns MOE_ERR_ARG when a bank is not page-locked host
 * memory, MOE_ERR_SHAPE when the layer or the slot count is outside what the
 * single-launch decode kernel handles (H and I multiples of 128, I <= 2048,
 * T*k <= 4096 within its shared-memory budget); otherwise as
 * moe_fp8_block_forward_ex.  Asynchronous on `stream`.
 */
int moe_fp8_block_forward_host_experts(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                       const moe_tensor* topk_weights, const moe_tensor* w13,
                                       const moe_tensor* w13_scale, int64_t w13_scale_stride,
                                       const moe_tensor* w2, const moe_tensor* w2_scale,
                                       int64_t w2_scale_stride, moe_tensor* out, void* stream,
                                       const moe_options* opt);

/* Size in bytes of the fixed device array behind
 * moe_fp8_block_forward_decode_noalloc. */
#define MOE_FP8_BLOCK_NOALLOC_BYTES (8u << 20)

/*
 * moe_fp8_block_forward_decode_noalloc -- the decode (W8A16) path of
 * moe_fp8_block_forward, for callers that cannot let the library allocate
 * device memory.  It has no counterpart in the pages this library follows;
 * it exists for deployments where every byte of device memory is planned up
 * front (a framework-owned pool, a fixed per-model budget) or where an
 * allocation inside a serving loop is unacceptable (cudaMalloc can
 * synchronise the device and can fail under memory pressure), so that the
 * per-stream workspace that moe_fp8_block_forward grows on demand is not an
 * option.
 *
 * Arguments, layouts and return codes are those of moe_fp8_block_forward;
 * the path is always decode.  The caller passes inputs and outputs as usual;
 * all scratch (routing lists, the f16 activation copy, h and the per-slot
 * outputs) lives in one statically allocated device array of
 * MOE_FP8_BLOCK_NOALLOC_BYTES bytes that every GPU using the library keeps
 * until the process exits.  A call needs about
 * 4*T*k*(H + I) + 2*T*H + 16*E + 32*T*k bytes of it; a larger call returns
 * MOE_ERR_ARG and moe_fp8_block_last_error_detail says how many bytes it
 * needed.  The entry point itself calls no cudaMalloc or cudaFree and no
 * allocating library routine.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current).  CUDA loads modules
 * lazily by default, so that first lookup may load the library's module and
 * commit the array's memory on the device, with the implicit synchronisation
 * a module load brings: make the first call (a warm-up call, or
 * moe_fp8_block_noalloc_status) before the serving loop starts and before
 * capturing the stream into a CUDA graph.  Later calls allocate nothing.
 * Every call on every stream of a device uses the same array: calls whose
 * kernels overlap on the GPU race and give wrong results, so serialise them
 * (one stream, or events).  Each call clears the array's status word first;
 * read it with moe_fp8_block_noalloc_status (moe_fp8_block_device_status
 * reads the per-stream workspaces of the other entry points, not this
 * array).  moe_fp8_block_last_path reports MOE_PATH_DECODE and
 * moe_fp8_block_last_launches the kernels launched, as for the regular
 * forward.
 */
int moe_fp8_block_forward_decode_noalloc(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                         const moe_tensor* topk_weights, const moe_tensor* w13,
                                         const moe_tensor* w13_scale, int64_t w13_scale_stride,
                                         const moe_tensor* w2, const moe_tensor* w2_scale,
                                         int64_t w2_scale_stride, moe_tensor* out, void* stream);

/*
 * moe_fp8_block_noalloc_status -- waits for `stream`, then returns in
 * *status and clears the status word of moe_fp8_block_forward_decode_noalloc's
 * array on the current device (the MOE_STATUS_* bits the kernels of the last
 * such call raised: out-of-range expert ids, a wait that ran out).  Reading
 * and clearing are ordered on `stream`; a call on another stream that still
 * runs may set bits afterwards.  Allocates nothing.
 *  status   host uint32, written (0 on any error)
 * Returns MOE_OK, MOE_ERR_NULL (status NULL) or MOE_ERR_CUDA.
 */
int moe_fp8_block_noalloc_status(void* stream, uint32_t* status);

/*
 * moe_fp8_block_forward_act_codes -- moe_fp8_block_forward_ex, plus a copy
 * of the e4m3 activation codes and fp32 group scales that the forward's own
 * quantiser produced in this call, for checking them code by code (the
 * dynamic per-token, per-128-column activation scales of the fp8-moe-gather
 * page, "Affects": scale = amax / 448, code = e4m3(x / scale) rounded to
 * nearest even and saturated).
 *  codes   device uint8 [T, H], row-contiguous, 16-byte aligned
 *  scales  device fp32 [T, ceil(H/128)], row-contiguous
 * Prefill path: the copy is taken from the rows the grouped GEMM reads,
 * those of one routed slot of each token (slot t mod k, else the next valid
 * one); a token without a valid slot has no such row and its entries are
 * left untouched.  Decode path: only with decode_act = MOE_DECODE_ACT_E4M3,
 * where the gate/up kernel quantises the activations itself and also writes
 * this copy; the W8A16 decode path quantises nothing (MOE_ERR_ARG).
 * Everything else, including the return codes, is moe_fp8_block_forward_ex.
 */
int moe_fp8_block_forward_act_codes(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                    const moe_tensor* topk_weights, const moe_tensor* w13,
                                    const moe_tensor* w13_scale, int64_t w13_scale_stride,
                                    const moe_tensor* w2, const moe_tensor* w2_scale,
                                    int64_t w2_scale_stride, moe_tensor* out, void* stream,
                                    const moe_options* opt, uint8_t* codes, float* scales);

/*
 * moe_fp8_block_route -- the routing lists of the gathered path, on their
 * own (the same kernel the forward runs).  For S = T*k slots s = t*k + j:
 *  counts   int32 [E]     slots per expert (valid ids only)
 *  offsets  int32 [E+1]   exclusive prefix sum of counts
 *  perm     int32 [S]     slot indices grouped by expert ascending, stable in
 *                         s; entries past offsets[E] are -1
 *  inv      int32 [S]     position of slot s in perm, or -1 when skipped
 *  glist    int32 [min(E,S)] distinct routed experts ascending, padded with -1
 *  n_distinct int32 [1]   number of distinct routed experts
 * (At most g = min(E, T*k) experts are read, the routed ones: fp8-moe-gather
 * page, The fix.)  All outputs are device int32 buffers of the
 * sizes above, contiguous.  Requires S <= 2^24.
 */
int moe_fp8_block_route(const moe_tensor* topk_ids, int32_t E, int32_t* counts,
                        int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* glist,
                        int32_t* n_distinct, void* stream);

/*
 * moe_fp8_block_act_quant -- the dynamic activation quantisation rule of the
 * prefill path as a standalone kernel (the forward itself quantises inside
 * its own kernels; moe_fp8_block_forward_act_codes returns those codes): for
 * each row r
 * of x (bf16 [R, K], stride[1] == 1, K a multiple of 128) and each 128-column
 * group c: amax = max |x|, scale = amax / 448 in IEEE fp32,
 * code = e4m3(x / scale) rounded to nearest even and saturated to +-448
 * (amax == 0 gives scale 0 and codes 0).
 *  codes   uint8 [R, K] contiguous (e4m3 bytes)
 *  scales  fp32 [R, K/128] contiguous
 */
int moe_fp8_block_act_quant(const moe_tensor* x, uint8_t* codes, float* scales, void* stream);

/*
 * moe_fp8_block_widen_e4m3 -- the in-register e4m3 widening used by the
 * decode kernels, applied to n bytes: out[i] = value of codes[i] as fp32
 * (exact for every finite code; FreeToken PR #662, PR body: e4m3 -> bf16 is
 * exact).  codes: device uint8 [n]; out: device fp32 [n].
 */
int moe_fp8_block_widen_e4m3(const uint8_t* codes, int64_t n, float* out, void* stream);

/* Pre-size the workspace of (current device, stream) for calls with up to
 * max_T tokens of the given layer shape, so that a later call can be
 * captured into a CUDA graph.  Synchronous with respect to the host. */
int moe_fp8_block_reserve(int64_t max_T, int32_t k, int64_t H, int64_t I, int32_t E,
                          void* stream);

/* Synchronise `stream`, then read and clear the device status word of the
 * (current device, stream) workspace into *status (MOE_STATUS_* bits). */
int moe_fp8_block_device_status(void* stream, uint32_t* status);

/* Path taken by the last successful forward call on this host thread:
 * MOE_PATH_DECODE, MOE_PATH_PREFILL, or MOE_PATH_NONE before any call. */
int moe_fp8_block_last_path(void);

/* Number of kernel launches the last successful forward call on this host
 * thread enqueued. */
int moe_fp8_block_last_launches(void);

/* The path the default gate (no caller ratio, no forced path) takes for a
 * forward call of T tokens, top_k = k, E experts, hidden width H and
 * intermediate width I: MOE_PATH_DECODE or MOE_PATH_PREFILL; the rule is
 * the one in "Paths" above.  Host only, needs no device.  Returns
 * MOE_ERR_ARG for T < 0, k outside 1..64 or E outside 1..4096, and
 * MOE_ERR_SHAPE for H, I that no path takes. */
int moe_fp8_block_default_path(int64_t T, int32_t k, int32_t E, int64_t H, int64_t I);

/* Profiling aid.  The next forward call on this host thread records
 * events[i] (cudaEvent_t, created by the caller) on its stream before its
 * i-th kernel launch and one more event after its last launch, for as many
 * events as given (n <= 16), then forgets them.  While events are recorded
 * the kernels are launched without programmatic dependent launch, so each
 * interval is one kernel's device time.  n == 0 clears. */
int moe_fp8_block_set_stage_events(void* const* events, int n);

/* MOE_FP8_BLOCK_ABI_VERSION of the built library. */
int moe_fp8_block_abi_version(void);

/* Text of the CUDA error behind the last MOE_ERR_CUDA returned on this host
 * thread, with the stage that raised it (empty string if none).  Setting
 * the environment variable MOE_FP8_BLOCK_SYNC_CHECK=1 makes every forward
 * synchronise after each kernel and report the first failing one here
 * (a debugging aid; it serialises the stream). */
const char* moe_fp8_block_last_error_detail(void);

/* Static description of a return code (never NULL). */
const char* moe_fp8_block_error_string(int code);

/* Free every workspace (all devices, all streams).  No call may be in flight. */
void moe_fp8_block_release(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_BLOCK_H */
