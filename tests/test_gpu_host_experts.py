"""Expert banks in host memory (the offload case of FreeToken PR #662, PR
body: block-fp8 experts served from the cpu and hybrid backends), read by the
GPU over the host link with ordinary loads: the decode forward must match
the float64 oracle, and the device-bank forward of the same kernel, on the
decode workloads; pageable banks and the prefill path are refused."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args

pytestmark = pytest.mark.gpu

_BANKS = {}


def banks(shape):
    key = (shape.E, shape.H, shape.I)
    if key not in _BANKS:
        _BANKS.clear()
        dev = syn.make_weights(shape, 0, "cuda")
        host = []
        for t in dev:
            h = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host.append(h)
        _BANKS[key] = (dev, host)
    return _BANKS[key]


def run(shape, T, routing="softmax", decode_act=None, step=0):
    dev, host = banks(shape)
    ids, w = syn.make_routing(T, shape.E, shape.k, 0, "cuda", routing, step=step)
    x = syn.make_hidden(T, shape.H, 0, "cuda", step)
    out = api.moe_fp8_block_forward_host_experts(x, ids, w, host[0], host[1], host[1].stride(1), host[2], host[3],
                                                 host[3].stride(1), decode_act=decode_act)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == 1
    prob = dict(hidden=x, topk_ids=ids, topk_weights=w, w13=dev[0], w13_scale=dev[1], w2=dev[2], w2_scale=dev[3])
    return out, prob


@pytest.mark.parametrize("T", [1, 4, 16])
def test_host_experts_small_layer(cuda_lib, T):
    out, prob = run(syn.DECODE_SMALL, T, step=T)
    args, _ = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy(), mo.forward(*args)) < TOL
    # the same kernel on the device-resident banks gives the same bits
    ref = api.forward_problem(prob, force_path="decode", decode_kernel="fused")
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_host_experts_padded_skewed(cuda_lib):
    out, prob = run(syn.PADDED_SKEWED, 8, routing="hot", step=3)
    args, _ = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy(), mo.forward(*args)) < TOL


def test_host_experts_w8a8(cuda_lib):
    out, prob = run(syn.DECODE_SMALL, 4, decode_act="e4m3", step=9)
    args, _ = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy(), mo.forward(*args, act="e4m3_x")) <= TOL


def test_host_experts_refuses_pageable_banks_and_prefill(cuda_lib):
    shape = syn.TINY
    dev = syn.make_weights(shape, 0, "cuda")
    pageable = [t.cpu() for t in dev]
    ids, w = syn.make_routing(2, shape.E, shape.k, 0, "cuda", "softmax")
    x = syn.make_hidden(2, shape.H, 0, "cuda")
    with pytest.raises(_lib.MoeError) as ei:
        api.moe_fp8_block_forward_host_experts(x, ids, w, pageable[0], pageable[1], pageable[1].stride(1),
                                               pageable[2], pageable[3], pageable[3].stride(1))
    assert ei.value.code == -9
    pinned = [t.pin_memory() for t in pageable]
    lib = _lib.load()
    import ctypes
    o = _lib.MoeOptions()
    o.force_path = 2
    d = [api.desc(t) for t in (x, ids, w, pinned[0], pinned[1], pinned[2], pinned[3])]
    out = torch.empty_like(x)
    P = ctypes.byref
    rc = lib.moe_fp8_block_forward_host_experts(P(d[0]), P(d[1]), P(d[2]), P(d[3]), P(d[4]), pinned[1].stride(1),
                                                P(d[5]), P(d[6]), pinned[3].stride(1), P(api.desc(out)), None, P(o))
    assert rc == -9
