// noalloc.cu -- moe_fp8_block_forward_decode_noalloc: the decode path with
// all of its scratch in one fixed, statically allocated device array, for
// callers that must not allocate device memory during a call.
//
// Who needs it: inference servers and real-time pipelines that plan every
// byte of device memory up front (a framework-owned pool, a fixed memory
// budget per model) and hot loops where an allocation would be a problem in
// itself -- cudaMalloc can synchronise the device and may fail under memory
// pressure -- cannot let the library grow its own per-stream workspace on
// the first call with a new shape.  This entry point never allocates: it
// carves the routing lists, the f16 activation copy, h and the per-slot
// outputs out of g_noalloc_scratch.
#include <cstdio>
#include <map>
#include <mutex>

#include "kernels.h"
#include "moe_fp8_block.h"

namespace moe {

// The scratch: every GPU that loads the library keeps these bytes until the
// process exits.  Calls share it; nothing in it survives from one call to
// the next except what the next call overwrites.
constexpr size_t kNoAllocBytes = (size_t)MOE_FP8_BLOCK_NOALLOC_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

std::mutex g_na_mu;
std::map<int, void*> g_na_ptr;   // device -> device address of g_noalloc_scratch

// Device address of the scratch on `device` (which must be current).  In
// host code the array's name is only a host-side stand-in, so the address
// is looked up once per device.
cudaError_t scratch_address(int device, void** out) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  auto it = g_na_ptr.find(device);
  if (it != g_na_ptr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  g_na_ptr[device] = p;
  *out = p;
  return cudaSuccess;
}

inline size_t al(size_t x) { return (x + 255) / 256 * 256; }

struct NaLayout {
  size_t status, fctr, counts, offsets, perm, inv, glist, nd, meta, vmeta, xh, xexp, xs, h, ybuf, total;
};

NaLayout na_layout(int64_t T, int k, int64_t H, int64_t I, int E) {
  NaLayout L{};
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t at = o;
    o = al(o + b);
    return at;
  };
  const int64_t S = T * k;
  const int64_t g = S < E ? S : E;
  L.status = take(16);
  L.fctr = take(4 * (size_t)kFusedCounterWords);   // same offset in every call; kept zero between calls
  L.counts = take(4 * (size_t)E);
  L.offsets = take(4 * (size_t)(E + 1));
  L.perm = take(4 * (size_t)S);
  L.inv = take(4 * (size_t)S);
  L.glist = take(4 * (size_t)(g > 0 ? g : 1));
  L.nd = take(16);
  L.meta = take(16 * (size_t)(g > 0 ? g : 1));
  L.vmeta = take(16 * (size_t)(S > 0 ? S : 1));
  L.xh = take(2 * (size_t)(T * H));
  L.xexp = take(4 * (size_t)T);
  L.h = take(4 * (size_t)(S * I));
  L.ybuf = take(4 * (size_t)(S * H));
  L.xs = take(4 * (size_t)T * (size_t)((H + 127) / 128));
  L.total = o;
  return L;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_fp8_block_forward_decode_noalloc(const moe_tensor* hidden, const moe_tensor* topk_ids,
                                                    const moe_tensor* topk_weights, const moe_tensor* w13,
                                                    const moe_tensor* w13_scale, int64_t w13_scale_stride,
                                                    const moe_tensor* w2, const moe_tensor* w2_scale,
                                                    int64_t w2_scale_stride, moe_tensor* out, void* stream) {
  LayerArgs a;
  int dev = 0;
  int rc = validate_forward(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                            w2_scale_stride, out, &a, &dev);
  if (rc) return rc;
  if (a.T == 0) {
    record_call(MOE_PATH_NONE, 0);
    return MOE_OK;
  }
  if (!decode_supported(a.H, a.I)) return MOE_ERR_SHAPE;
  const NaLayout L = na_layout(a.T, a.k, a.H, a.I, a.E);
  if (L.total > kNoAllocBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "moe_fp8_block_forward_decode_noalloc: this call needs %zu bytes of scratch; the fixed array holds %zu",
             L.total, kNoAllocBytes);
    set_error_detail(msg);
    return MOE_ERR_ARG;
  }
  void* base = nullptr;
  if (note_error(scratch_address(dev, &base), "noalloc scratch address") != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(base);
  uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status);
  // the status word is the only thing the kernels accumulate into
  if (note_error(cudaMemsetAsync(status, 0, 16, st), "noalloc status clear") != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  RouteBufs rb{reinterpret_cast<int32_t*>(w + L.counts), reinterpret_cast<int32_t*>(w + L.offsets),
               reinterpret_cast<int32_t*>(w + L.perm),   reinterpret_cast<int32_t*>(w + L.inv),
               reinterpret_cast<int32_t*>(w + L.glist),  reinterpret_cast<int32_t*>(w + L.nd),
               reinterpret_cast<int4*>(w + L.meta),       nullptr};
  DecodeBufs db{reinterpret_cast<uint16_t*>(w + L.xh), reinterpret_cast<int32_t*>(w + L.xexp),
                reinterpret_cast<float*>(w + L.xs), reinterpret_cast<float*>(w + L.h),
                reinterpret_cast<float*>(w + L.ybuf), reinterpret_cast<uint32_t*>(w + L.fctr),
                reinterpret_cast<int4*>(w + L.vmeta)};
  int launches = 0;
  const cudaError_t e = launch_decode(a, rb, db, status, dev, st, &launches);
  if (e != cudaSuccess) {
    note_error(e, "noalloc decode");
    cudaGetLastError();
    return e == cudaErrorNotSupported ? MOE_ERR_SHAPE : MOE_ERR_CUDA;
  }
  record_call(MOE_PATH_DECODE, launches);
  return MOE_OK;
}

extern "C" int moe_fp8_block_noalloc_status(void* stream, uint32_t* status) {
  if (!status) return MOE_ERR_NULL;
  *status = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  void* base = nullptr;
  if (note_error(scratch_address(dev, &base), "noalloc scratch address") != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  // the status word sits at the start of the array (na_layout's first field)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, base, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(base, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  *status = v;
  return MOE_OK;
}
