"""The single-launch decode kernel (moe_options.decode_kernel = fused) against
the float64 oracle, on the decode workloads: routing in every CTA's shared
memory, the per-expert hand-off of h between the projections and the
grid-wide count before the combine must give the chained kernels' results
within the per-token tolerance, deterministically, with skipped and
out-of-range slots, padded scale strides, MLP biases and W8A8 activations."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args, oracle_biases

pytestmark = pytest.mark.gpu

_W = {}


def problem(shape, T, routing="softmax", step=0):
    key = (shape.E, shape.H, shape.I, shape.w13_scale_stride, shape.w2_scale_stride)
    if key not in _W:
        _W.clear()
        torch.cuda.empty_cache()
        _W[key] = syn.make_weights(shape, 0, "cuda")
    w13, w13s, w2, w2s = _W[key]
    ids, w = syn.make_routing(T, shape.E, shape.k, 0, "cuda", routing, step=step)
    return dict(hidden=syn.make_hidden(T, shape.H, 0, "cuda", step), topk_ids=ids, topk_weights=w, w13=w13,
                w13_scale=w13s, w2=w2, w2_scale=w2s)


def run(prob, tokens=None, decode_act=None, **kw):
    out = api.forward_problem(prob, force_path="decode", decode_kernel="fused", decode_act=decode_act, **kw)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == 1
    args, tok = oracle_args(prob, tokens)
    bias = {}
    if kw.get("w13_bias") is not None or kw.get("w2_bias") is not None:
        bias = oracle_biases(dict(prob, **{k: v for k, v in kw.items() if k.endswith("bias")}), tokens)
    ref = mo.forward(*args, act="e4m3_x" if decode_act == "e4m3" else "bf16", **bias)
    return check_per_token(out.float().cpu().numpy()[tok], ref), out


@pytest.mark.parametrize("T", [1, 2, 4, 16])
def test_fused_small_experts(cuda_lib, T):
    r, _ = run(problem(syn.DECODE_SMALL, T, step=T))
    assert r < TOL
    assert api.moe_fp8_block_last_launches() == 1


@pytest.mark.parametrize("T", [1, 8, 32])
def test_fused_padded_skewed(cuda_lib, T):
    r, _ = run(problem(syn.PADDED_SKEWED, T, routing="hot", step=T))
    assert r < TOL


def test_fused_tiny_all_expert(cuda_lib):
    prob = problem(syn.TINY, 4)
    out = api.forward_problem(prob, force_path="decode", decode_kernel="fused")
    torch.cuda.synchronize()
    args, _ = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy(), mo.forward(*args, mode="all")) < TOL


@pytest.mark.slow
def test_fused_wide_experts(cuda_lib):
    r, _ = run(problem(syn.DECODE_WIDE, 4, step=4), tokens=[0, 3])
    assert r < TOL


def test_fused_matches_chain_and_is_deterministic(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 16, step=3)
    a = api.forward_problem(prob, force_path="decode", decode_kernel="fused")
    b = api.forward_problem(prob, force_path="decode", decode_kernel="fused")
    c = api.forward_problem(prob, force_path="decode")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    d = (a.float() - c.float()).abs().amax(dim=1)
    assert torch.all(d <= 1e-2 * c.float().abs().amax(dim=1))


def test_fused_skipped_and_bad_ids(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 6, step=7)
    ids = prob["topk_ids"].clone()
    ids[0, 1] = -1
    ids[1, 0] = 128          # >= E: skipped and flagged
    ids[2, 1] = ids[2, 0]    # a duplicate expert inside one token
    ids[3, :] = -1           # a token with no valid slot: zero output
    prob["topk_ids"] = ids
    api.moe_fp8_block_device_status()
    r, out = run(prob)
    assert r < TOL
    assert api.moe_fp8_block_device_status() == 1
    assert torch.count_nonzero(out[3]).item() == 0


def test_fused_padded_equals_unpadded(cuda_lib):
    prob = problem(syn.PADDED_SKEWED, 8, routing="hot", step=2)
    unp = dict(prob)
    unp["w2_scale"] = prob["w2_scale"][..., :5].contiguous()
    a = api.forward_problem(prob, force_path="decode", decode_kernel="fused")
    b = api.forward_problem(unp, force_path="decode", decode_kernel="fused")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("which", ["both", "w13", "w2"])
def test_fused_bias(cuda_lib, which):
    shape = syn.DECODE_SMALL
    prob = problem(shape, 8, step=4)
    b13, b2 = syn.make_biases(shape, 0, "cuda")
    kw = {"w13_bias": b13 if which in ("both", "w13") else None, "w2_bias": b2 if which in ("both", "w2") else None}
    r, _ = run(prob, **kw)
    assert r < TOL


@pytest.mark.parametrize("T", [1, 4, 16])
def test_fused_w8a8_and_codes(cuda_lib, T):
    prob = problem(syn.DECODE_SMALL, T, step=T + 1)
    r, _ = run(prob, decode_act="e4m3")
    assert r <= TOL
    _, codes, scales = api.moe_fp8_block_forward_act_codes(
        prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"], prob["w13_scale"],
        prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1),
        force_path="decode", decode_act="e4m3", decode_kernel="fused")
    torch.cuda.synchronize()
    rc, rs = mo.quantize_per_128(prob["hidden"].float().cpu().numpy())
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_fused_graph_replay_new_routing(cuda_lib):
    shape = syn.DECODE_SMALL
    prob = problem(shape, 4, step=1)
    s = torch.cuda.Stream()
    api.moe_fp8_block_reserve(16, shape.k, shape.H, shape.I, shape.E, stream=s)
    out = torch.empty(4, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        api.forward_problem(prob, out=out, stream=s, force_path="decode", decode_kernel="fused")
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.forward_problem(prob, out=out, stream=s, force_path="decode", decode_kernel="fused")
    for step in range(2, 5):
        nxt = problem(shape, 4, step=step)
        for n in ("hidden", "topk_ids", "topk_weights"):
            prob[n].copy_(nxt[n])
        g.replay()
        torch.cuda.synchronize()
        args, _ = oracle_args(prob)
        assert check_per_token(out.float().cpu().numpy(), mo.forward(*args)) < TOL
