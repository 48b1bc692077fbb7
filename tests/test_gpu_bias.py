"""MLP biases on the GPU against the float64 oracle, through the C ABI
(moe_fp8_block_forward_bias): gate biases added to the gate half and up
biases to the up half before silu, the down-projection bias after the down
projection (tpu-inference PR #3040, review of the bias DMA), on the decode
(W8A16 and W8A8) and prefill paths.  The biases are drawn at the size of
the projections they are added to, so a dropped, misplaced or swapped bias
breaks the per-token tolerance (each test checks that it would)."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args, oracle_biases

pytestmark = pytest.mark.gpu

# standard deviations of gate/up and of y on these workloads (N(0,1) bf16
# activations, full-range e4m3 weights, scales 2^-8..2^-2): the biases match them
STD13, STD2 = 300.0, 1.0e7


def bias_problem(shape, T, routing="softmax", seed=0, which=("w13", "w2")):
    prob = syn.make_problem(shape, T, seed, "cuda", routing)
    b13, b2 = syn.make_biases(shape, seed, "cuda", STD13, STD2)
    prob["w13_bias"] = b13 if "w13" in which else None
    prob["w2_bias"] = b2 if "w2" in which else None
    return prob


def run(prob, path, tokens=None, decode_act=None):
    out = api.moe_fp8_block_forward(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                    prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"],
                                    prob["w2_scale"].stride(1), force_path=path, decode_act=decode_act,
                                    w13_bias=prob["w13_bias"], w2_bias=prob["w2_bias"])
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == (1 if path == "decode" else 2)
    args, tok = oracle_args(prob, tokens)
    b = oracle_biases(prob, tokens)
    act = ("e4m3_x" if decode_act == "e4m3" else "bf16") if path == "decode" else "e4m3"
    ref = mo.forward(*args, act=act, **b)
    got = out.float().cpu().numpy()[tok]
    r = check_per_token(got, ref)
    # the same check would fail without the biases, or with gate and up
    # biases exchanged: the comparison sees them
    plain = mo.forward(*args, act=act)
    assert np.max(np.abs(plain - ref) / np.max(np.abs(ref), axis=1, keepdims=True)) > TOL
    if "w13_bias" in b:
        I = prob["w13"].shape[1] // 2
        sw = dict(b)
        sw["w13_bias"] = np.concatenate([b["w13_bias"][:, I:], b["w13_bias"][:, :I]], axis=1)
        swapped = mo.forward(*args, act=act, **sw)
        assert np.max(np.abs(swapped - ref) / np.max(np.abs(ref), axis=1, keepdims=True)) > TOL
    return r, out


@pytest.mark.parametrize("T", [1, 4, 16])
def test_bias_decode_small_experts(cuda_lib, T):
    r, _ = run(bias_problem(syn.DECODE_SMALL, T), "decode")
    assert r < TOL


def test_bias_decode_padded_skewed(cuda_lib):
    r, _ = run(bias_problem(syn.PADDED_SKEWED, 8, routing="hot"), "decode")
    assert r < TOL


def test_bias_decode_w8a8(cuda_lib):
    r, _ = run(bias_problem(syn.DECODE_SMALL, 4), "decode", decode_act="e4m3")
    assert r < TOL


@pytest.mark.parametrize("T,tokens", [(64, None), (1024, [0, 333, 1023])])
def test_bias_prefill(cuda_lib, T, tokens):
    r, _ = run(bias_problem(syn.PREFILL, T), "prefill", tokens=tokens)
    assert r < TOL


def test_bias_prefill_padded_skewed(cuda_lib):
    r, _ = run(bias_problem(syn.PADDED_SKEWED, 32, routing="hot"), "prefill")
    assert r < TOL


@pytest.mark.parametrize("path", ["decode", "prefill"])
@pytest.mark.parametrize("which", [("w13",), ("w2",)])
def test_one_bias_only(cuda_lib, path, which):
    r, _ = run(bias_problem(syn.DECODE_SMALL, 8, which=which), path)
    assert r < TOL


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_zero_biases_equal_no_bias(cuda_lib, path):
    prob = syn.make_problem(syn.DECODE_SMALL, 8, 0, "cuda")
    E, H, I = syn.DECODE_SMALL.E, syn.DECODE_SMALL.H, syn.DECODE_SMALL.I
    base = api.forward_problem(prob, force_path=path)
    z = api.forward_problem(prob, force_path=path, w13_bias=torch.zeros(E, 2 * I, device="cuda"),
                            w2_bias=torch.zeros(E, H, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(base, z)


def test_padded_bias_expert_stride(cuda_lib):
    """Bias banks with a padded expert stride read only their first 2I / H
    columns: padding filled with NaN would show in the output."""
    shp = syn.DECODE_SMALL
    prob = bias_problem(shp, 4)
    b13 = torch.full((shp.E, 2 * shp.I + 4), float("nan"), device="cuda")
    b13[:, :2 * shp.I] = prob["w13_bias"]
    b2 = torch.full((shp.E, shp.H + 8), float("nan"), device="cuda")
    b2[:, :shp.H] = prob["w2_bias"]
    ref = api.moe_fp8_block_forward_bias(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                         prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"],
                                         prob["w2_scale"], prob["w2_scale"].stride(1), prob["w13_bias"],
                                         prob["w2_bias"])
    for path in ("decode", "prefill"):
        a = api.moe_fp8_block_forward_bias(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                           prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"],
                                           prob["w2_scale"], prob["w2_scale"].stride(1), b13[:, :2 * shp.I],
                                           b2[:, :shp.H], force_path=path)
        b = api.moe_fp8_block_forward_bias(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                           prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"],
                                           prob["w2_scale"], prob["w2_scale"].stride(1), prob["w13_bias"],
                                           prob["w2_bias"], force_path=path)
        torch.cuda.synchronize()
        assert torch.isfinite(a.float()).all()
        assert torch.equal(a, b)
    assert torch.isfinite(ref.float()).all()
