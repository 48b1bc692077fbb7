"""Ragged layers on the GPU against the float64 oracle: H or I not a
multiple of 128 (the page's "ragged K" case of FreeToken PR #662, Tests), so
both projections have a partial last K block and, when I is ragged, the up
rows of a 128-row scale block of the stacked [gate; up] bank start inside
it.  The prefill path takes H a multiple of 64 and I of 16; the decode path
H and I multiples of 64 (its last K block is one 64-wide chunk), and
forcing decode on any other ragged layer is refused."""
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
# both ragged, multiples of 64: the decode path takes it
RAGGED_64 = syn.MoeShape(E=16, H=320, I=192, k=4, w13_scale_stride=4)
# GPT-OSS's hidden width with an intermediate width whose down-projection
# staging fits the decode kernels' shared memory (I = 2880 does not)
WIDE_RAGGED_DEC = syn.MoeShape(E=32, H=2880, I=1472, k=4)


def run(prob, tokens=None, force="prefill", decode_act=None, decode_kernel=None):
    kw = {}
    if prob.get("w13_bias") is not None:
        kw = dict(w13_bias=prob["w13_bias"], w2_bias=prob["w2_bias"])
    out = api.moe_fp8_block_forward(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                    prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"],
                                    prob["w2_scale"].stride(1), force_path=force, decode_act=decode_act,
                                    decode_kernel=decode_kernel, **kw)
    torch.cuda.synchronize()
    path = api.moe_fp8_block_last_path()
    if force is not None:
        assert path == (1 if force == "decode" else 2)
    args, tok = oracle_args(prob, tokens)
    act = "e4m3" if path == 2 else ("e4m3_x" if decode_act == "e4m3" else "bf16")
    ref = mo.forward(*args, act=act, **oracle_biases(prob, tokens))
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


@pytest.mark.parametrize("shape", [RAGGED_64, RAGGED_H], ids=["both64", "H"])
@pytest.mark.parametrize("T", [1, 4, 16])
def test_ragged_decode(cuda_lib, shape, T):
    r, _ = run(syn.make_problem(shape, T, 0, "cuda", step=T), force="decode")
    assert r < TOL


def test_ragged_decode_w8a8_and_biases(cuda_lib):
    r, _ = run(syn.make_problem(RAGGED_64, 4, 0, "cuda", step=5), force="decode", decode_act="e4m3")
    assert r <= TOL
    prob = syn.make_problem(RAGGED_64, 4, 0, "cuda", step=6)
    prob["w13_bias"], prob["w2_bias"] = syn.make_biases(RAGGED_64, 0, "cuda", 300.0, 1.0e7)
    r, _ = run(prob, force="decode")
    assert r < TOL


def test_ragged_decode_default_gate_and_fused_option(cuda_lib):
    """A small batch of a decode-able ragged layer takes decode by default;
    the single-kernel option does not take ragged layers and the call runs
    the chained kernels."""
    r, _ = run(syn.make_problem(RAGGED_64, 1, 0, "cuda", step=2), force=None)
    assert r < TOL and api.moe_fp8_block_last_path() == 1
    r, _ = run(syn.make_problem(RAGGED_64, 2, 0, "cuda", step=3), force="decode", decode_kernel="fused")
    assert r < TOL and api.moe_fp8_block_last_launches() == 4


@pytest.mark.slow
def test_wide_ragged_layer_decode(cuda_lib):
    """H = 2880, I = 1472 on the decode path: 23 K blocks of the gate/up
    projection split over the four warps of a group (more than a warp keeps
    in registers), the last one a single 64-wide chunk; 12 K blocks of the
    down projection, the last one a single chunk too."""
    r, _ = run(syn.make_problem(WIDE_RAGGED_DEC, 8, 0, "cuda", step=8), tokens=[0, 4, 7], force="decode")
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
