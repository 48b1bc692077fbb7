"""Python entry points with the names of the C ABI, taking torch tensors.

torch supplies device memory and streams only; each function builds the C
descriptors and calls the CUDA library (include/moe_fp8_block.h).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import MoeOptions, MoeTensor, check

_DTYPES = {
    torch.bfloat16: _lib.MOE_BF16,
    torch.float32: _lib.MOE_F32,
    torch.uint8: _lib.MOE_E4M3,
    torch.float8_e4m3fn: _lib.MOE_E4M3,
    torch.int32: _lib.MOE_I32,
}


def desc(t: torch.Tensor) -> MoeTensor:
    """C descriptor of a tensor (pointer, dtype, shape, strides in elements)."""
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() < 1 or t.dim() > 4:
        raise ValueError("tensors must have 1..4 dimensions")
    d = MoeTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or None)
    d.ndim = t.dim()
    d.dtype = _DTYPES[t.dtype]
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _options(gate_ratio, force_path, decode_act=None, decode_kernel=None, debug_wait_timeout_us=0,
             debug_drop_stage=0) -> Optional[MoeOptions]:
    if (gate_ratio is None and force_path is None and decode_act is None and decode_kernel is None
            and not debug_wait_timeout_us and not debug_drop_stage):
        return None
    o = MoeOptions()
    dk = {None: 0, "chain": 0, "fused": 1}
    o.decode_kernel = dk[decode_kernel] if not isinstance(decode_kernel, int) else decode_kernel
    o.debug_wait_timeout_us = int(debug_wait_timeout_us)
    o.debug_drop_stage = int(debug_drop_stage)
    o.gate_ratio = float(gate_ratio) if gate_ratio is not None else 0.0
    fp = {None: 0, "auto": 0, "decode": 1, "prefill": 2}
    o.force_path = fp[force_path] if not isinstance(force_path, int) else force_path
    da = {None: 0, "bf16": 0, "e4m3": 1}
    o.decode_act = da[decode_act] if not isinstance(decode_act, int) else decode_act
    return o


def moe_fp8_block_forward(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                          w2_scale_stride, out=None, stream=None, gate_ratio=None, force_path=None,
                          decode_act=None, w13_bias=None, w2_bias=None, decode_kernel=None,
                          debug_wait_timeout_us=0, debug_drop_stage=0):
    """Layer forward on device tensors; returns `out` (bf16 [T, H]).
    decode_act: "bf16" (W8A16, default) or "e4m3" (W8A8) for the decode path.
    w13_bias (fp32 [E, 2I], [gate | up]) and w2_bias (fp32 [E, H]): optional
    MLP biases, passed to moe_fp8_block_forward_bias."""
    if w13_bias is not None or w2_bias is not None:
        return moe_fp8_block_forward_bias(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2,
                                          w2_scale, w2_scale_stride, w13_bias, w2_bias, out=out, stream=stream,
                                          gate_ratio=gate_ratio, force_path=force_path, decode_act=decode_act,
                                          decode_kernel=decode_kernel)
    lib = _lib.load()
    if out is None:
        out = torch.empty(hidden.shape, dtype=torch.bfloat16, device=hidden.device)
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    o = desc(out)
    P = ctypes.byref
    opt = _options(gate_ratio, force_path, decode_act, decode_kernel, debug_wait_timeout_us, debug_drop_stage)
    if opt is None:
        rc = lib.moe_fp8_block_forward(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                       int(w2_scale_stride), P(o), _stream(stream))
    else:
        rc = lib.moe_fp8_block_forward_ex(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                          int(w2_scale_stride), P(o), _stream(stream), P(opt))
    check(rc, "moe_fp8_block_forward")
    return out


def moe_fp8_block_forward_bias(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2, w2_scale,
                               w2_scale_stride, w13_bias=None, w2_bias=None, out=None, stream=None,
                               gate_ratio=None, force_path=None, decode_act=None, decode_kernel=None):
    """Layer forward with optional MLP biases (either may be None)."""
    lib = _lib.load()
    if out is None:
        out = torch.empty(hidden.shape, dtype=torch.bfloat16, device=hidden.device)
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    b13 = desc(w13_bias) if w13_bias is not None else None
    b2 = desc(w2_bias) if w2_bias is not None else None
    o = desc(out)
    P = ctypes.byref
    opt = _options(gate_ratio, force_path, decode_act, decode_kernel)
    rc = lib.moe_fp8_block_forward_bias(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                        int(w2_scale_stride), P(b13) if b13 is not None else None,
                                        P(b2) if b2 is not None else None, P(o), _stream(stream),
                                        P(opt) if opt is not None else None)
    check(rc, "moe_fp8_block_forward_bias")
    return out


def moe_fp8_block_forward_hostio(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2,
                                 w2_scale, w2_scale_stride, out=None, stream=None, gate_ratio=None,
                                 force_path=None, decode_act=None):
    """Layer forward with HOST hidden/ids/weights/out (pinned for async
    copies) and device weight banks; returns `out` once it is filled."""
    lib = _lib.load()
    if out is None:
        out = torch.empty(hidden.shape, dtype=torch.bfloat16, pin_memory=True)
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    o = desc(out)
    P = ctypes.byref
    opt = _options(gate_ratio, force_path, decode_act)
    rc = lib.moe_fp8_block_forward_hostio(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                          int(w2_scale_stride), P(o), _stream(stream),
                                          P(opt) if opt is not None else None)
    check(rc, "moe_fp8_block_forward_hostio")
    return out


def moe_fp8_block_forward_host_experts(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2,
                                       w2_scale, w2_scale_stride, out=None, stream=None, decode_act=None):
    """Decode forward with the expert banks (w13, w13_scale, w2, w2_scale)
    in page-locked host memory; activations, routing and output on the
    device.  Returns `out` (bf16 [T, H], device)."""
    lib = _lib.load()
    if out is None:
        out = torch.empty(hidden.shape, dtype=torch.bfloat16, device=hidden.device)
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    o = desc(out)
    P = ctypes.byref
    opt = _options(None, None, decode_act) or MoeOptions()
    rc = lib.moe_fp8_block_forward_host_experts(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                                int(w2_scale_stride), P(o), _stream(stream), P(opt))
    check(rc, "moe_fp8_block_forward_host_experts")
    return out


def moe_fp8_block_forward_decode_noalloc(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2,
                                         w2_scale, w2_scale_stride, out, stream=None):
    """The decode path without any device allocation (scratch in a fixed
    library-owned array); `out` must be supplied by the caller."""
    lib = _lib.load()
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    o = desc(out)
    P = ctypes.byref
    rc = lib.moe_fp8_block_forward_decode_noalloc(*[P(x) for x in args], int(w13_scale_stride),
                                                  *[P(x) for x in a2], int(w2_scale_stride), P(o), _stream(stream))
    check(rc, "moe_fp8_block_forward_decode_noalloc")
    return out


def moe_fp8_block_forward_act_codes(hidden, topk_ids, topk_weights, w13, w13_scale, w13_scale_stride, w2,
                                    w2_scale, w2_scale_stride, out=None, stream=None, gate_ratio=None,
                                    force_path=None, decode_act=None, decode_kernel=None):
    """Layer forward that also returns the activation codes and group scales
    its own quantiser produced: (out, codes uint8 [T, H], scales fp32
    [T, ceil(H/128)])."""
    lib = _lib.load()
    T, H = hidden.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    codes = torch.zeros((T, H), dtype=torch.uint8, device=hidden.device)
    scales = torch.zeros((T, (H + 127) // 128), dtype=torch.float32, device=hidden.device)
    args = [desc(hidden), desc(topk_ids), desc(topk_weights), desc(w13), desc(w13_scale)]
    a2 = [desc(w2), desc(w2_scale)]
    o = desc(out)
    P = ctypes.byref
    opt = _options(gate_ratio, force_path, decode_act, decode_kernel) or MoeOptions()
    rc = lib.moe_fp8_block_forward_act_codes(*[P(x) for x in args], int(w13_scale_stride), *[P(x) for x in a2],
                                             int(w2_scale_stride), P(o), _stream(stream), P(opt),
                                             codes.data_ptr(), scales.data_ptr())
    check(rc, "moe_fp8_block_forward_act_codes")
    return out, codes, scales


def moe_fp8_block_route(topk_ids: torch.Tensor, E: int, stream=None):
    """Routing lists (see the header): dict of int32 device tensors."""
    lib = _lib.load()
    S = topk_ids.numel()
    dev = topk_ids.device
    r = dict(
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm=torch.empty(max(S, 1), dtype=torch.int32, device=dev),
        inv=torch.empty(max(S, 1), dtype=torch.int32, device=dev),
        glist=torch.empty(max(min(E, S), 1), dtype=torch.int32, device=dev),
        n_distinct=torch.empty(1, dtype=torch.int32, device=dev),
    )
    rc = lib.moe_fp8_block_route(ctypes.byref(desc(topk_ids)), int(E), *[r[n].data_ptr() for n in
                                 ("counts", "offsets", "perm", "inv", "glist", "n_distinct")], _stream(stream))
    check(rc, "moe_fp8_block_route")
    r["perm"], r["inv"], r["glist"] = r["perm"][:S], r["inv"][:S], r["glist"][:min(E, S)]
    return r


def moe_fp8_block_act_quant(x: torch.Tensor, stream=None):
    """Per-row, per-128-column e4m3 quantisation: (codes uint8 [R,K], scales fp32 [R,K/128])."""
    lib = _lib.load()
    R, K = x.shape
    codes = torch.empty((R, K), dtype=torch.uint8, device=x.device)
    scales = torch.empty((R, max(K // 128, 1)), dtype=torch.float32, device=x.device)
    rc = lib.moe_fp8_block_act_quant(ctypes.byref(desc(x)), codes.data_ptr(), scales.data_ptr(), _stream(stream))
    check(rc, "moe_fp8_block_act_quant")
    return codes, scales[:, :K // 128]


def moe_fp8_block_widen_e4m3(codes: torch.Tensor, stream=None) -> torch.Tensor:
    lib = _lib.load()
    out = torch.empty(codes.shape, dtype=torch.float32, device=codes.device)
    rc = lib.moe_fp8_block_widen_e4m3(codes.data_ptr(), codes.numel(), out.data_ptr(), _stream(stream))
    check(rc, "moe_fp8_block_widen_e4m3")
    return out


def moe_fp8_block_reserve(max_T: int, k: int, H: int, I: int, E: int, stream=None):
    check(_lib.load().moe_fp8_block_reserve(max_T, k, H, I, E, _stream(stream)), "moe_fp8_block_reserve")


def moe_fp8_block_device_status(stream=None) -> int:
    v = ctypes.c_uint32(0)
    check(_lib.load().moe_fp8_block_device_status(_stream(stream), ctypes.byref(v)), "moe_fp8_block_device_status")
    return v.value


def moe_fp8_block_noalloc_status(stream=None) -> int:
    """Read and clear the status word of the allocation-free entry point."""
    v = ctypes.c_uint32(0)
    check(_lib.load().moe_fp8_block_noalloc_status(_stream(stream), ctypes.byref(v)), "moe_fp8_block_noalloc_status")
    return v.value


def moe_fp8_block_last_path() -> int:
    return _lib.load().moe_fp8_block_last_path()


def moe_fp8_block_default_path(T: int, k: int, E: int, H: int, I: int) -> int:
    """The path (1 decode, 2 prefill) the default gate takes for a call of
    this shape; raises on arguments no path takes.  Host only."""
    rc = _lib.load().moe_fp8_block_default_path(T, k, E, H, I)
    if rc < 0:
        check(rc, "moe_fp8_block_default_path")
    return rc


def moe_fp8_block_last_launches() -> int:
    return _lib.load().moe_fp8_block_last_launches()


def moe_fp8_block_abi_version() -> int:
    return _lib.load().moe_fp8_block_abi_version()


def moe_fp8_block_release():
    _lib.load().moe_fp8_block_release()


def forward_problem(prob: dict, out=None, stream=None, **kw):
    """Convenience: forward on a dict of tensors (the synthetic generator's
    layout); scale strides are read from the scale tensors."""
    return moe_fp8_block_forward(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                 prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"],
                                 prob["w2_scale"].stride(1), out=out, stream=stream, **kw)
