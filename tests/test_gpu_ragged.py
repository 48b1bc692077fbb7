"""Ragged layers on the GPU against the float64 oracle: H or I not a
multiple of 128 (the page's "ragged K" case of FreeToken PR #662, Tests), so
both projections have a partial last K block and, when I is ragged, the up
rows of a 128-row scale block of the stacked [gate; up] bank start inside
it.  These layers run on the prefill path; forcing decode is refused."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args, oracle_biases

pytestmark = pytest.mark.gpu

RAGGED_BOTH = syn.MoeShape(E=16, H=320, I=176, k=4)
RAGGED_H = syn.MoeShape(E=8, H=192, I=256, k=2, w2_scale_stride=3)
RAGGED_I = syn.MoeShape(E=8, H=256, I=144, k=2, w13_scale_stride=3)
# GPT-OSS-like widths: 2880 = 22.5 x 128
WIDE_RAGGED = syn.MoeShape(E=32, H=2880, I=2880, k=4)


def run(prob, tokens=None, force="prefill"):
    kw = {}
    if prob.get("w13_bias") is not None:
        kw = dict(w13_bias=prob["w13_bias"], w2_bias=prob["w2_bias"])
    out = api.moe_fp8_block_forward(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                    prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"],
                                    prob["w2_scale"].stride(1), force_path=force, **kw)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == 2
    args, tok = oracle_args(prob, tokens)
    ref = mo.forward(*args, act="e4m3", **oracle_biases(prob, tokens))
    return check_per_token(out.float().cpu().numpy()[tok], ref), out


@pytest.mark.parametrize("shape", [RAGGED_BOTH, RAGGED_H, RAGGED_I], ids=["both", "H", "I"])
@pytest.mark.parametrize("T", [1, 64])
def test_ragged_prefill(cuda_lib, shape, T):
    r, _ = run(syn.make_problem(shape, T, 0, "cuda"))
    assert r < TOL


def test_ragged_default_gate_takes_prefill(cuda_lib):
    prob = syn.make_problem(RAGGED_BOTH, 1, 0, "cuda")
    r, _ = run(prob, force=None)
    assert r < TOL


def test_ragged_forced_decode_is_refused(cuda_lib):
    prob = syn.make_problem(RAGGED_I, 2, 0, "cuda")
    with pytest.raises(_lib.MoeError) as e:
        api.forward_problem(prob, force_path="decode")
    assert e.value.code == -3
    with pytest.raises(_lib.MoeError) as e:
        out = torch.empty(2, RAGGED_I.H, dtype=torch.bfloat16, device="cuda")
        api.moe_fp8_block_forward_decode_noalloc(prob["hidden"], prob["topk_ids"], prob["topk_weights"],
                                                 prob["w13"], prob["w13_scale"], prob["w13_scale"].stride(1),
                                                 prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1), out)
    assert e.value.code == -3


def test_ragged_with_biases(cuda_lib):
    prob = syn.make_problem(RAGGED_BOTH, 48, 0, "cuda")
    prob["w13_bias"], prob["w2_bias"] = syn.make_biases(RAGGED_BOTH, 0, "cuda", 300.0, 1.0e7)
    r, _ = run(prob)
    assert r < TOL


@pytest.mark.slow
@pytest.mark.parametrize("bias", [False, True])
def test_wide_ragged_layer(cuda_lib, bias):
    """H = I = 2880, the GPT-OSS widths, with and without MLP biases (three
    sampled tokens of 512)."""
    prob = syn.make_problem(WIDE_RAGGED, 512, 0, "cuda")
    if bias:
        prob["w13_bias"], prob["w2_bias"] = syn.make_biases(WIDE_RAGGED, 0, "cuda", 300.0, 1.0e7)
    r, _ = run(prob, tokens=[0, 255, 511])
    assert r < TOL


def test_ragged_deterministic(cuda_lib):
    prob = syn.make_problem(RAGGED_BOTH, 200, 0, "cuda", routing="zipf")
    a = api.forward_problem(prob)
    b = api.forward_problem(prob)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
