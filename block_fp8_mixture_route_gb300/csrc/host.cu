// host.cu -- the C ABI of include/moe_fp8_block.h: argument checks, the
// path gate, per-(device, stream) workspaces and kernel dispatch.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"
#include "moe_fp8_block.h"

namespace moe {

namespace {

thread_local int g_last_path = MOE_PATH_NONE;
thread_local int g_last_launches = 0;

std::mutex g_mu;

struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::map<int, int> g_sms;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
// bytes of the status word and the fused decode counters at the start of a workspace
const size_t kCountersEnd = align_up(16) + align_up(4 * (size_t)kFusedCounterWords);

// Byte layout of one workspace.
struct Layout {
  size_t status, fctr, counts, offsets, perm, inv, glist, nd, meta, mtp, mtp2, rcnt;
  size_t xh, xexp, xsd, h, ybuf, vmeta;           // decode
  size_t xq, xs, hq, hs, ys, pinv, wsc13, wsc2;  // prefill
  int64_t prows;
  size_t hid, tids, twts, outb;                   // host-io staging
  size_t total;
};

Layout make_layout(int64_t T, int k, int64_t H, int64_t I, int E, int path, bool hostio) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const int64_t S = T * k;
  const int64_t g = S < E ? S : E;
  L.status = take(16);
  L.fctr = take(4 * (size_t)kFusedCounterWords);   // same offset in every layout
  L.counts = take(4 * (size_t)E);
  L.offsets = take(4 * (size_t)(E + 1));
  L.perm = take(4 * (size_t)S);
  L.inv = take(4 * (size_t)S);
  L.glist = take(4 * (size_t)(g > 0 ? g : 1));
  L.nd = take(16);
  L.meta = take(16 * (size_t)(g > 0 ? g : 1));
  L.mtp = take(4 * (size_t)(E + 1));
  L.mtp2 = take(4 * (size_t)(E + 1));
  L.rcnt = take(8 * (size_t)route_chunks((int)S) * (size_t)E);   // chunk histograms + chunk bases
  if (path == MOE_PATH_DECODE) {
    L.xh = take(2 * (size_t)(T * H));
    L.xexp = take(4 * (size_t)T);
    L.h = take(4 * (size_t)(S * I));
    L.ybuf = take(4 * (size_t)(S * H));
    L.xsd = take(4 * (size_t)T * (size_t)((H + 127) / 128));
    L.vmeta = take(16 * (size_t)(S > 0 ? S : 1));
  } else if (path == MOE_PATH_PREFILL) {
    const int64_t R = prefill_rows(S, E);
    L.prows = R;
    L.xq = take((size_t)(R * H));
    L.xs = take(4 * (size_t)(R * ((H + 127) / 128)));
    L.hq = take((size_t)(R * I));
    L.hs = take(4 * (size_t)(R * ((I + 127) / 128)));
    L.ys = take(2 * (size_t)(R * H));
    L.pinv = take(4 * (size_t)S);
    L.wsc13 = take(16 * (size_t)E * (size_t)((H + 127) / 128) * (size_t)((I + 127) / 128));
    L.wsc2 = take(16 * (size_t)E * (size_t)((I + 127) / 128) * (size_t)((H + 255) / 256));
  }
  if (hostio) {
    L.hid = take(2 * (size_t)(T * H));
    L.tids = take(4 * (size_t)S);
    L.twts = take(4 * (size_t)S);
    L.outb = take(2 * (size_t)(T * H));
  }
  L.total = o;
  return L;
}

size_t layout_max(int64_t T, int k, int64_t H, int64_t I, int E, bool hostio) {
  size_t a = make_layout(T, k, H, I, E, MOE_PATH_DECODE, hostio).total;
  size_t b = make_layout(T, k, H, I, E, MOE_PATH_PREFILL, hostio).total;
  return a > b ? a : b;
}

// Return the workspace of (current device, stream) with at least `bytes`.
int get_workspace(cudaStream_t st, size_t bytes, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& ws = g_ws[std::make_pair(dev, st)];
  if (ws.bytes >= bytes && ws.base) {
    *out = ws.base;
    return MOE_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MOE_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_CAPTURE_GROW;
  if (ws.base) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    cudaFree(ws.base);
    ws.base = nullptr;
    ws.bytes = 0;
  }
  size_t want = bytes < (1u << 20) ? (1u << 20) : bytes;
  if (cudaMalloc(&ws.base, want) != cudaSuccess) {
    ws.base = nullptr;
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  // the status word and the fused decode kernel's counters must start cleared
  // (they sit at the same offsets in every layout, before any other buffer)
  if (cudaMemsetAsync(ws.base, 0, kCountersEnd, st) != cudaSuccess) return MOE_ERR_CUDA;
  ws.bytes = want;
  *out = ws.base;
  return MOE_OK;
}

// ------------------------------------------------------- descriptor checks
int elem_size(int dtype) {
  switch (dtype) {
    case MOE_BF16: return 2;
    case MOE_F32: return 4;
    case MOE_E4M3: return 1;
    case MOE_I32: return 4;
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tensor(const moe_tensor* t, int ndim, int dtype) {
  if (!t) return MOE_ERR_NULL;
  if (t->ndim != ndim) return MOE_ERR_SHAPE;
  if (t->dtype != dtype) return MOE_ERR_DTYPE;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return MOE_ERR_SHAPE;
  return MOE_OK;
}

bool contiguous(const moe_tensor* t) {
  int64_t s = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != s) return false;
    s *= t->shape[i];
  }
  return true;
}

// Byte extent [lo, hi) covered by a strided tensor (empty tensors: lo == hi).
std::pair<uintptr_t, uintptr_t> extent(const moe_tensor* t) {
  uintptr_t lo = reinterpret_cast<uintptr_t>(t->data);
  int64_t last = 0;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] == 0) return {lo, lo};
    last += (t->shape[i] - 1) * t->stride[i];
  }
  return {lo, lo + (uintptr_t)((last + 1) * elem_size(t->dtype))};
}

bool overlap(const moe_tensor* a, const moe_tensor* b) {
  auto x = extent(a), y = extent(b);
  if (x.first == x.second || y.first == y.second) return false;
  return x.first < y.second && y.first < x.second;
}

int check_scale_bank(const moe_tensor* s, int64_t E, int64_t rows, int64_t cols, int64_t row_stride) {
  int rc = check_tensor(s, 3, MOE_BF16);
  if (rc) return rc;
  if (s->shape[0] != E || s->shape[1] != rows || s->shape[2] < cols) return MOE_ERR_SHAPE;
  if (row_stride < cols || s->stride[2] != 1 || (rows > 1 && s->stride[1] != row_stride)) return MOE_ERR_STRIDE;
  if (E > 1 && s->stride[0] < rows * row_stride) return MOE_ERR_STRIDE;
  if (!s->data) return MOE_ERR_NULL;
  return MOE_OK;
}

struct Checked {
  LayerArgs a;
  int64_t T;
};

// Layer shapes the library runs.  Multiples of 128 take either path.  A
// ragged layer (H or I not a multiple of 128) runs on the prefill path,
// whose tensor-map loads zero-fill the partial last blocks; it needs H a
// multiple of 64 (the output is stored in 64-column quarters) and I a
// multiple of 16 (16-byte rows and box coordinates), both at least 128.
bool layer_shape_ok(int64_t H, int64_t I) {
  if (H < 128 || I < 128 || H > 8192 || I > 8192) return false;
  return H % 64 == 0 && I % 16 == 0;
}

// An optional MLP bias: fp32 [E, n], stride[1] == 1, expert stride
// stride[0] >= n and a multiple of 4 elements, 16-byte aligned base.
int check_bias(const moe_tensor* b, int64_t E, int64_t n) {
  int rc = check_tensor(b, 2, MOE_F32);
  if (rc) return rc;
  if (b->shape[0] != E || b->shape[1] != n) return MOE_ERR_SHAPE;
  if (b->stride[1] != 1 || (E > 1 && (b->stride[0] < n || b->stride[0] % 4 != 0))) return MOE_ERR_STRIDE;
  if (!b->data) return MOE_ERR_NULL;
  if (!aligned16(b->data)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

int check_forward(const moe_tensor* hidden, const moe_tensor* topk_ids, const moe_tensor* topk_weights,
                  const moe_tensor* w13, const moe_tensor* w13_scale, int64_t w13_scale_stride,
                  const moe_tensor* w2, const moe_tensor* w2_scale, int64_t w2_scale_stride,
                  const moe_tensor* out, bool host_io, Checked* c) {
  int rc;
  if ((rc = check_tensor(hidden, 2, MOE_BF16))) return rc;
  if ((rc = check_tensor(topk_ids, 2, MOE_I32))) return rc;
  if ((rc = check_tensor(topk_weights, 2, MOE_F32))) return rc;
  if ((rc = check_tensor(w13, 3, MOE_E4M3))) return rc;
  if ((rc = check_tensor(w2, 3, MOE_E4M3))) return rc;
  if ((rc = check_tensor(out, 2, MOE_BF16))) return rc;
  const int64_t T = hidden->shape[0], H = hidden->shape[1];
  const int64_t k = topk_ids->shape[1];
  const int64_t E = w13->shape[0];
  const int64_t I2 = w13->shape[1];
  if (topk_ids->shape[0] != T || topk_weights->shape[0] != T || topk_weights->shape[1] != k) return MOE_ERR_SHAPE;
  if (out->shape[0] != T || out->shape[1] != H) return MOE_ERR_SHAPE;
  if (k < 1 || k > 64 || E < 1 || E > 4096) return MOE_ERR_ARG;
  if (w13->shape[2] != H || I2 % 2 != 0) return MOE_ERR_SHAPE;
  const int64_t I = I2 / 2;
  if (!layer_shape_ok(H, I)) return MOE_ERR_SHAPE;
  if (w2->shape[0] != E || w2->shape[1] != H || w2->shape[2] != I) return MOE_ERR_SHAPE;
  if (H > 8192 || I > 8192) return MOE_ERR_SHAPE;
  if (T > (1 << 24) / k) return MOE_ERR_ARG;
  const int64_t hb = (H + 127) / 128, ib = (I + 127) / 128, i2b = (2 * I + 127) / 128;
  if ((rc = check_scale_bank(w13_scale, E, i2b, hb, w13_scale_stride))) return rc;
  if ((rc = check_scale_bank(w2_scale, E, hb, ib, w2_scale_stride))) return rc;
  if (!contiguous(w13) || !contiguous(w2)) return MOE_ERR_STRIDE;
  if (!contiguous(topk_ids) || !contiguous(topk_weights) || !contiguous(out)) return MOE_ERR_STRIDE;
  if (hidden->stride[1] != 1 || (T > 1 && hidden->stride[0] < H)) return MOE_ERR_STRIDE;
  if (host_io && T > 1 && hidden->stride[0] != H) return MOE_ERR_STRIDE;
  if (T > 0) {
    if (!hidden->data || !topk_ids->data || !topk_weights->data || !out->data) return MOE_ERR_NULL;
    if (!aligned16(hidden->data) || !aligned16(out->data)) return MOE_ERR_ALIGN;
    if (hidden->stride[0] % 8 != 0) return MOE_ERR_ALIGN;
    if (!aligned16(topk_ids->data) && !host_io) return MOE_ERR_ALIGN;
  }
  if (!w13->data || !w2->data) return MOE_ERR_NULL;
  if (!aligned16(w13->data) || !aligned16(w2->data)) return MOE_ERR_ALIGN;
  if (!host_io) {
    const moe_tensor* ins[] = {hidden, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale};
    for (const moe_tensor* t : ins)
      if (overlap(out, t)) return MOE_ERR_ALIAS;
  }
  LayerArgs& a = c->a;
  a.hidden = static_cast<const uint16_t*>(hidden->data);
  a.hidden_ld = T > 1 ? hidden->stride[0] : H;
  a.ids = static_cast<const int32_t*>(topk_ids->data);
  a.wts = static_cast<const float*>(topk_weights->data);
  a.w13 = static_cast<const uint8_t*>(w13->data);
  a.w13s = static_cast<const uint16_t*>(w13_scale->data);
  a.s13_row = w13_scale_stride;
  a.s13_exp = E > 1 ? w13_scale->stride[0] : i2b * w13_scale_stride;
  a.w2 = static_cast<const uint8_t*>(w2->data);
  a.w2s = static_cast<const uint16_t*>(w2_scale->data);
  a.s2_row = w2_scale_stride;
  a.s2_exp = E > 1 ? w2_scale->stride[0] : hb * w2_scale_stride;
  a.out = static_cast<uint16_t*>(out->data);
  a.T = (int)T;
  a.k = (int)k;
  a.H = (int)H;
  a.I = (int)I;
  a.E = (int)E;
  a.S = (int)(T * k);
  c->T = T;
  return MOE_OK;
}

int check_options(const moe_options* opt, float* ratio, int* force, LayerArgs* a) {
  *ratio = 0.f;   // the measured default gate (choose_path)
  *force = MOE_PATH_NONE;
  a->act8 = 0;
  if (!opt) return MOE_OK;
  for (int i = 0; i < 2; ++i)
    if (opt->reserved[i] != 0) return MOE_ERR_ARG;
  if (opt->force_path < MOE_PATH_NONE || opt->force_path > MOE_PATH_PREFILL) return MOE_ERR_ARG;
  if (opt->decode_act != MOE_DECODE_ACT_BF16 && opt->decode_act != MOE_DECODE_ACT_E4M3) return MOE_ERR_ARG;
  if (opt->decode_kernel != MOE_DECODE_KERNEL_CHAIN && opt->decode_kernel != MOE_DECODE_KERNEL_FUSED)
    return MOE_ERR_ARG;
  if (opt->debug_wait_timeout_us < 0 || opt->debug_wait_timeout_us > 1000000 || opt->debug_drop_stage < 0)
    return MOE_ERR_ARG;
  if (opt->gate_ratio > 0.f) *ratio = opt->gate_ratio;
  *force = opt->force_path;
  a->act8 = opt->decode_act == MOE_DECODE_ACT_E4M3;
  a->decode_kernel = opt->decode_kernel;
  a->dbg_wait_ns = 1000ull * (uint64_t)opt->debug_wait_timeout_us;
  a->dbg_drop_stage = opt->debug_drop_stage;
  return MOE_OK;
}

int device_ok(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
  int maj = 0, min = 0;
  if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (maj != 10 || min != 3) return MOE_ERR_DEVICE;
  return MOE_OK;
}

// Run the forward on device buffers already described by `a`.
int run_forward(const LayerArgs& a, float ratio, int force, cudaStream_t st, bool hostio, void* ws_base,
                const Layout& L, int dev) {
  char* w = static_cast<char*>(ws_base);
  uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status);
  RouteBufs rb;
  rb.counts = reinterpret_cast<int32_t*>(w + L.counts);
  rb.offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  rb.perm = reinterpret_cast<int32_t*>(w + L.perm);
  rb.inv = reinterpret_cast<int32_t*>(w + L.inv);
  rb.glist = reinterpret_cast<int32_t*>(w + L.glist);
  rb.nd = reinterpret_cast<int32_t*>(w + L.nd);
  rb.meta = reinterpret_cast<int4*>(w + L.meta);
  rb.mtp = reinterpret_cast<int32_t*>(w + L.mtp);
  rb.mtp2 = reinterpret_cast<int32_t*>(w + L.mtp2);
  (void)hostio;
  int path = force;
  if (path == MOE_PATH_NONE)
    path = ((double)a.T * a.k <= (double)a.E * ratio) ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
  int launches = 0;
  cudaError_t err;
  if (path == MOE_PATH_DECODE) {
    DecodeBufs db;
    db.xh = reinterpret_cast<uint16_t*>(w + L.xh);
    db.xexp = reinterpret_cast<int32_t*>(w + L.xexp);
    db.xs = reinterpret_cast<float*>(w + L.xsd);
    db.h = reinterpret_cast<float*>(w + L.h);
    db.ybuf = reinterpret_cast<float*>(w + L.ybuf);
    db.counters = reinterpret_cast<uint32_t*>(w + L.fctr);
    db.vmeta = reinterpret_cast<int4*>(w + L.vmeta);
    err = launch_decode(a, rb, db, status, dev, st, &launches);
  } else {
    PrefillBufs pb;
    pb.xq = reinterpret_cast<uint8_t*>(w + L.xq);
    pb.xsT = reinterpret_cast<float*>(w + L.xs);
    pb.hq = reinterpret_cast<uint8_t*>(w + L.hq);
    pb.hsT = reinterpret_cast<float*>(w + L.hs);
    pb.ys = reinterpret_cast<uint16_t*>(w + L.ys);
    pb.pinv = reinterpret_cast<int32_t*>(w + L.pinv);
    pb.wsc13 = reinterpret_cast<float*>(w + L.wsc13);
    pb.wsc2 = reinterpret_cast<float*>(w + L.wsc2);
    pb.rows = L.prows;
    err = launch_prefill(a, rb, pb, reinterpret_cast<int32_t*>(w + L.rcnt), status, dev, st, &launches);
    if (err == cudaSuccess && a.dbg_codes) {
      err = note_error(launch_prefill_act_codes(a, pb, st), "prefill_act_codes");
      ++launches;
    }
  }
  if (err == cudaErrorNotSupported) {
    cudaGetLastError();
    return MOE_ERR_ARG;
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  stage_events().n = 0;
  g_last_path = path;
  g_last_launches = launches;
  return MOE_OK;
}

// Gate.  With a caller ratio: decode while T*k <= E*ratio (the rule of the
// fp8-moe-gather page, environment-variable table).  Default, from sweeps of
// both paths on GB300 (median forward us, decode / prefill): decode while
// T*k <= E, the decode gate/up stream gets at least 4 ring stages, and its
// units are the full 8 row pairs (H <= 2048) or the batch routes at most 8
// slots.  E128 H2048 I512 (8 row pairs, 5 stages): decode faster at every
// T*k/E up to 1 (T=8 61 / 69, T=16 86 / 93).  E256 H2560 I640 with hot
// experts (4 row pairs, 8 stages): decode faster only at T=1 (37 / 42),
// prefill from T=2 on (T=8 94 / 76, T=32 441 / 105).  E256 H7168 I2048
// (3 stages: the 14 KB activation rows crowd the ring): prefill from
// T*k/E = 0.03 on.
int choose_path(const LayerArgs& a, float ratio, int force) {
  if (force != MOE_PATH_NONE) return force;
  if (ratio > 0.f) {
    const bool gathered = (double)a.T * a.k <= (double)a.E * ratio;
    return gathered && decode_supported(a.H, a.I) ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
  }
  const bool gathered = (double)a.T * a.k <= (double)a.E;
  const bool units = decode_unit_rows(a.H) >= 8 || (int64_t)a.T * a.k <= 8;
  return gathered && units && decode_ring_stages(a.H, a.I) >= 4 ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
}

// Device address of page-locked host memory that kernels can read and write
// in place (cudaHostAlloc / cudaHostRegister memory, mapped into the unified
// address space; on GB300 such accesses cross NVLink-C2C), or nullptr for
// pageable memory.
void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost) return nullptr;
  return at.devicePointer;
}

int forward_impl(const moe_tensor* hidden, const moe_tensor* topk_ids, const moe_tensor* topk_weights,
                 const moe_tensor* w13, const moe_tensor* w13_scale, int64_t w13_scale_stride,
                 const moe_tensor* w2, const moe_tensor* w2_scale, int64_t w2_scale_stride, moe_tensor* out,
                 void* stream, const moe_options* opt, bool hostio, const moe_tensor* w13_bias = nullptr,
                 const moe_tensor* w2_bias = nullptr, uint8_t* dbg_codes = nullptr, float* dbg_scales = nullptr) {
  Checked c{};
  int rc = check_forward(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                         w2_scale_stride, out, hostio, &c);
  if (rc) return rc;
  if (w13_bias) {
    if ((rc = check_bias(w13_bias, c.a.E, 2 * (int64_t)c.a.I))) return rc;
    if (overlap(out, w13_bias)) return MOE_ERR_ALIAS;
    c.a.b13 = static_cast<const float*>(w13_bias->data);
    c.a.b13_ld = c.a.E > 1 ? w13_bias->stride[0] : 2 * (int64_t)c.a.I;
  }
  if (w2_bias) {
    if ((rc = check_bias(w2_bias, c.a.E, c.a.H))) return rc;
    if (overlap(out, w2_bias)) return MOE_ERR_ALIAS;
    c.a.b2 = static_cast<const float*>(w2_bias->data);
    c.a.b2_ld = c.a.E > 1 ? w2_bias->stride[0] : c.a.H;
  }
  float ratio;
  int force;
  if ((rc = check_options(opt, &ratio, &force, &c.a))) return rc;
  const int act8 = c.a.act8;
  if (c.T == 0) {
    g_last_launches = 0;
    return MOE_OK;
  }
  int dev;
  if ((rc = device_ok(&dev))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LayerArgs a = c.a;
  const int path = choose_path(a, ratio, force);
  if (path == MOE_PATH_DECODE && !decode_supported(a.H, a.I)) return MOE_ERR_SHAPE;
  if (dbg_codes) {
    // only a path that quantises its activations has codes to copy
    if (path == MOE_PATH_DECODE && !act8) return MOE_ERR_ARG;
    a.dbg_codes = dbg_codes;
    a.dbg_scales = dbg_scales;
  }
  const Layout L = make_layout(c.T, a.k, a.H, a.I, a.E, path, hostio);
  void* ws = nullptr;
  if ((rc = get_workspace(st, L.total, &ws))) return rc;
  char* w = static_cast<char*>(ws);
  // Page-locked host buffers (all four, not overlapping the output) are
  // read and written in place by the kernels: no staging copies.
  bool in_place = false;
  if (hostio) {
    void* dh = mapped_host(hidden->data);
    void* di = mapped_host(topk_ids->data);
    void* dw = mapped_host(topk_weights->data);
    void* dout = mapped_host(out->data);
    in_place = dh && di && dw && dout && aligned16(dh) && aligned16(di) && aligned16(dw) && aligned16(dout) &&
               !overlap(out, hidden) && !overlap(out, topk_ids) && !overlap(out, topk_weights);
    if (in_place) {
      a.hidden = static_cast<const uint16_t*>(dh);
      a.hidden_ld = a.H;
      a.ids = static_cast<const int32_t*>(di);
      a.wts = static_cast<const float*>(dw);
      a.out = static_cast<uint16_t*>(dout);
    }
  }
  if (hostio && !in_place) {
    const size_t xb = 2 * (size_t)a.T * a.H, sb = 4 * (size_t)a.S;
    if (cudaMemcpyAsync(w + L.hid, hidden->data, xb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(w + L.tids, topk_ids->data, sb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(w + L.twts, topk_weights->data, sb, cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    a.hidden = reinterpret_cast<const uint16_t*>(w + L.hid);
    a.hidden_ld = a.H;
    a.ids = reinterpret_cast<const int32_t*>(w + L.tids);
    a.wts = reinterpret_cast<const float*>(w + L.twts);
    a.out = reinterpret_cast<uint16_t*>(w + L.outb);
  }
  rc = run_forward(a, ratio, path, st, hostio, ws, L, dev);
  if (rc) return rc;
  if (hostio) {
    if ((!in_place &&
         cudaMemcpyAsync(out->data, w + L.outb, 2 * (size_t)a.T * a.H, cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
        cudaStreamSynchronize(st) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

}  // namespace

static thread_local char g_err_detail[256] = "";

cudaError_t note_error(cudaError_t e, const char* stage) {
  if (e != cudaSuccess && e != cudaErrorNotSupported)
    snprintf(g_err_detail, sizeof(g_err_detail), "%s: %s (%s)", stage, cudaGetErrorName(e), cudaGetErrorString(e));
  return e;
}

static bool sync_check_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_FP8_BLOCK_SYNC_CHECK");
    return v && v[0] == '1';
  }();
  return on;
}

cudaError_t launch_check(cudaError_t launch_err, cudaStream_t st, const char* stage) {
  if (launch_err != cudaSuccess) return note_error(launch_err, stage);
  if (sync_check_enabled()) return note_error(cudaStreamSynchronize(st), stage);
  return cudaSuccess;
}

StageEvents& stage_events() {
  static thread_local StageEvents se;
  return se;
}

bool stage_mark(cudaStream_t st, int i) {
  StageEvents& se = stage_events();
  if (se.n == 0) return false;
  if (i < se.n) cudaEventRecord(se.ev[i], st);
  return true;
}

int validate_forward(const moe_tensor* hidden, const moe_tensor* topk_ids, const moe_tensor* topk_weights,
                     const moe_tensor* w13, const moe_tensor* w13_scale, int64_t w13_scale_stride,
                     const moe_tensor* w2, const moe_tensor* w2_scale, int64_t w2_scale_stride,
                     const moe_tensor* out, LayerArgs* args, int* device) {
  Checked c{};
  int rc = check_forward(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                         w2_scale_stride, out, false, &c);
  if (rc) return rc;
  *args = c.a;
  if (c.T == 0) return MOE_OK;
  return device_ok(device);
}

static std::mutex g_smem_mu;
static std::map<std::pair<int, const void*>, int> g_smem_set;

cudaError_t set_max_smem(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_smem_mu);
  int& cur = g_smem_set[{dev, func}];
  if (cur >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

void clear_smem_attributes() {
  std::lock_guard<std::mutex> lk(g_smem_mu);
  g_smem_set.clear();
}

void set_error_detail(const char* text) { snprintf(g_err_detail, sizeof(g_err_detail), "%s", text); }

void record_call(int path, int launches) {
  g_last_path = path;
  g_last_launches = launches;
}

int num_sms(int device) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sms.find(device);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
  if (n <= 0) n = 1;
  g_sms[device] = n;
  return n;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_fp8_block_forward(const moe_tensor* hidden, const moe_tensor* topk_ids, const moe_tensor* topk_weights,
                          const moe_tensor* w13, const moe_tensor* w13_scale, int64_t w13_scale_stride,
                          const moe_tensor* w2, const moe_tensor* w2_scale, int64_t w2_scale_stride,
                          moe_tensor* out, void* stream) {
  return forward_impl(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                      w2_scale_stride, out, stream, nullptr, false);
}

int moe_fp8_block_forward_ex(const moe_tensor* hidden, const moe_tensor* topk_ids,
                             const moe_tensor* topk_weights, const moe_tensor* w13,
                             const moe_tensor* w13_scale, int64_t w13_scale_stride, const moe_tensor* w2,
                             const moe_tensor* w2_scale, int64_t w2_scale_stride, moe_tensor* out,
                             void* stream, const moe_options* opt) {
  return forward_impl(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                      w2_scale_stride, out, stream, opt, false);
}

int moe_fp8_block_forward_bias(const moe_tensor* hidden, const moe_tensor* topk_ids,
                               const moe_tensor* topk_weights, const moe_tensor* w13,
                               const moe_tensor* w13_scale, int64_t w13_scale_stride, const moe_tensor* w2,
                               const moe_tensor* w2_scale, int64_t w2_scale_stride, const moe_tensor* w13_bias,
                               const moe_tensor* w2_bias, moe_tensor* out, void* stream, const moe_options* opt) {
  return forward_impl(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                      w2_scale_stride, out, stream, opt, false, w13_bias, w2_bias);
}

int moe_fp8_block_forward_hostio(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                 const moe_tensor* topk_weights, const moe_tensor* w13,
                                 const moe_tensor* w13_scale, int64_t w13_scale_stride, const moe_tensor* w2,
                                 const moe_tensor* w2_scale, int64_t w2_scale_stride, moe_tensor* out,
                                 void* stream, const moe_options* opt) {
  return forward_impl(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                      w2_scale_stride, out, stream, opt, true);
}

int moe_fp8_block_forward_host_experts(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                       const moe_tensor* topk_weights, const moe_tensor* w13,
                                       const moe_tensor* w13_scale, int64_t w13_scale_stride, const moe_tensor* w2,
                                       const moe_tensor* w2_scale, int64_t w2_scale_stride, moe_tensor* out,
                                       void* stream, const moe_options* opt) {
  Checked c{};
  int rc = check_forward(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                         w2_scale_stride, out, false, &c);
  if (rc) return rc;
  float ratio;
  int force;
  if ((rc = check_options(opt, &ratio, &force, &c.a))) return rc;
  if (force == MOE_PATH_PREFILL) return MOE_ERR_ARG;
  if (c.T == 0) {
    g_last_launches = 0;
    return MOE_OK;
  }
  int dev;
  if ((rc = device_ok(&dev))) return rc;
  LayerArgs a = c.a;
  if (!fused_decode_ok(a.T, a.k, a.H, a.I, a.E)) return MOE_ERR_SHAPE;
  // the banks must be page-locked host memory the device can address
  void* d13 = mapped_host(w13->data);
  void* d13s = mapped_host(w13_scale->data);
  void* d2 = mapped_host(w2->data);
  void* d2s = mapped_host(w2_scale->data);
  if (!d13 || !d13s || !d2 || !d2s) return MOE_ERR_ARG;
  if (!aligned16(d13) || !aligned16(d2)) return MOE_ERR_ALIGN;
  a.w13 = static_cast<const uint8_t*>(d13);
  a.w13s = static_cast<const uint16_t*>(d13s);
  a.w2 = static_cast<const uint8_t*>(d2);
  a.w2s = static_cast<const uint16_t*>(d2s);
  a.host_weights = 1;
  a.decode_kernel = MOE_DECODE_KERNEL_FUSED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = make_layout(c.T, a.k, a.H, a.I, a.E, MOE_PATH_DECODE, false);
  void* ws = nullptr;
  if ((rc = get_workspace(st, L.total, &ws))) return rc;
  return run_forward(a, ratio, MOE_PATH_DECODE, st, false, ws, L, dev);
}

int moe_fp8_block_forward_act_codes(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                    const moe_tensor* topk_weights, const moe_tensor* w13,
                                    const moe_tensor* w13_scale, int64_t w13_scale_stride, const moe_tensor* w2,
                                    const moe_tensor* w2_scale, int64_t w2_scale_stride, moe_tensor* out,
                                    void* stream, const moe_options* opt, uint8_t* codes, float* scales) {
  if (!codes || !scales) return MOE_ERR_NULL;
  if (!aligned16(codes)) return MOE_ERR_ALIGN;
  return forward_impl(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                      w2_scale_stride, out, stream, opt, false, nullptr, nullptr, codes, scales);
}

int moe_fp8_block_route(const moe_tensor* topk_ids, int32_t E, int32_t* counts, int32_t* offsets, int32_t* perm,
                        int32_t* inv, int32_t* glist, int32_t* n_distinct, void* stream) {
  int rc = check_tensor(topk_ids, 2, MOE_I32);
  if (rc) return rc;
  if (!contiguous(topk_ids)) return MOE_ERR_STRIDE;
  if (E < 1 || E > 4096) return MOE_ERR_ARG;
  const int64_t S = topk_ids->shape[0] * topk_ids->shape[1];
  if (S > (1 << 24)) return MOE_ERR_ARG;
  if (!counts || !offsets || !n_distinct || (S > 0 && (!perm || !inv || !glist || !topk_ids->data)))
    return MOE_ERR_NULL;
  int dev;
  if ((rc = device_ok(&dev))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const size_t scratch_bytes = 8 * (size_t)route_chunks((int)S) * (size_t)E;
  if ((rc = get_workspace(st, kCountersEnd + scratch_bytes, &ws))) return rc;
  RouteBufs rb{counts, offsets, perm, inv, glist, n_distinct, nullptr, nullptr};
  // after the status word and the decode counters, which other calls on this
  // stream rely on
  int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kCountersEnd);
  if (note_error(launch_route(static_cast<const int32_t*>(topk_ids->data), (int)S, E, rb,
                              static_cast<uint32_t*>(ws), scratch, st, nullptr),
                 "route") != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_fp8_block_act_quant(const moe_tensor* x, uint8_t* codes, float* scales, void* stream) {
  int rc = check_tensor(x, 2, MOE_BF16);
  if (rc) return rc;
  const int64_t R = x->shape[0], K = x->shape[1];
  if (K % 128 != 0 || R > (1 << 24) || K > (1 << 20)) return MOE_ERR_SHAPE;
  if (x->stride[1] != 1 || (R > 1 && x->stride[0] < K)) return MOE_ERR_STRIDE;
  if (R == 0 || K == 0) return MOE_OK;
  if (!x->data || !codes || !scales) return MOE_ERR_NULL;
  if (!aligned16(x->data) || !aligned16(codes) || (R > 1 && x->stride[0] % 8 != 0)) return MOE_ERR_ALIGN;
  int dev;
  if ((rc = device_ok(&dev))) return rc;
  if (launch_act_quant(static_cast<const uint16_t*>(x->data), R > 1 ? x->stride[0] : K, (int)R, (int)K, codes,
                       scales, static_cast<cudaStream_t>(stream), false) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_fp8_block_widen_e4m3(const uint8_t* codes, int64_t n, float* out, void* stream) {
  if (n < 0) return MOE_ERR_ARG;
  if (n == 0) return MOE_OK;
  if (!codes || !out) return MOE_ERR_NULL;
  int dev, rc;
  if ((rc = device_ok(&dev))) return rc;
  if (launch_widen(codes, n, out, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_fp8_block_reserve(int64_t max_T, int32_t k, int64_t H, int64_t I, int32_t E, void* stream) {
  if (max_T < 0 || k < 1 || k > 64 || E < 1 || E > 4096 || !layer_shape_ok(H, I))
    return MOE_ERR_ARG;
  int dev, rc;
  if ((rc = device_ok(&dev))) return rc;
  void* ws = nullptr;
  rc = get_workspace(static_cast<cudaStream_t>(stream), layout_max(max_T, k, H, I, E, true), &ws);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_fp8_block_device_status(void* stream, uint32_t* status) {
  if (!status) return MOE_ERR_NULL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_ws.find(std::make_pair(dev, st));
    if (it != g_ws.end()) base = it->second.base;
  }
  *status = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (!base) return MOE_OK;
  uint32_t v = 0;
  if (cudaMemcpy(&v, base, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(base, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

int moe_fp8_block_last_path(void) { return g_last_path; }

int moe_fp8_block_default_path(int64_t T, int32_t k, int32_t E, int64_t H, int64_t I) {
  if (T < 0 || k < 1 || k > 64 || E < 1 || E > 4096) return MOE_ERR_ARG;
  if (!layer_shape_ok(H, I) || H > 8192 || I > 8192) return MOE_ERR_SHAPE;
  LayerArgs a{};
  a.T = T;
  a.k = k;
  a.E = E;
  a.H = (int)H;
  a.I = (int)I;
  return choose_path(a, 0.f, MOE_PATH_NONE);
}

int moe_fp8_block_last_launches(void) { return g_last_launches; }

int moe_fp8_block_set_stage_events(void* const* events, int n) {
  if (n < 0 || n > 16 || (n > 0 && !events)) return MOE_ERR_ARG;
  StageEvents& se = stage_events();
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return MOE_ERR_NULL;
    se.ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  se.n = n;
  return MOE_OK;
}

int moe_fp8_block_abi_version(void) { return MOE_FP8_BLOCK_ABI_VERSION; }

const char* moe_fp8_block_last_error_detail(void) { return g_err_detail; }

const char* moe_fp8_block_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer or descriptor is NULL";
    case MOE_ERR_DTYPE: return "wrong element type";
    case MOE_ERR_SHAPE: return "inconsistent shapes, or H / I not supported by the requested path";
    case MOE_ERR_ALIGN: return "a base pointer or row stride is not 16-byte aligned";
    case MOE_ERR_STRIDE: return "unsupported stride";
    case MOE_ERR_ALIAS: return "out overlaps an input";
    case MOE_ERR_CAPTURE_GROW: return "workspace must grow while the stream is being captured; reserve first";
    case MOE_ERR_CUDA: return "a CUDA call failed";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
    default: return "unknown error code";
  }
}

void moe_fp8_block_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& kv : g_ws)
    if (kv.second.base) cudaFree(kv.second.base);
  g_ws.clear();
  clear_smem_attributes();
}

}  // extern "C"
