"""The prefill path's grouped GEMMs on the GPU against the float64 oracle,
at small layers whose experts hold several 128-row M tiles (a few hundred
routed slots per expert), every token checked.  The two CTAs of a pair take
M tiles 2i and 2i+1 of an expert where it has them, and both take an odd
last tile (adjacent column blocks); the cases cover both forms, experts with
no slots (Zipf routing), ragged H and I (partial K blocks, up tiles
straddling two scale blocks, a down-projection column block half past H)
and the MLP biases.  Tolerance and oracle as everywhere: FreeToken PR #662,
the commit adding the float64 parity reference (2e-2 per token)."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args, oracle_biases

pytestmark = pytest.mark.gpu

TILES_A = syn.MoeShape(E=4, H=512, I=384, k=2)                       # T=512: 1024 slots = 256 E
TILES_B = syn.MoeShape(E=8, H=1024, I=512, k=4, w2_scale_stride=9)   # T=1024: 4096 slots = 512 E
TILES_RAGGED = syn.MoeShape(E=4, H=320, I=176, k=2)                  # H, I ragged; GEMM2's last block half past H
TILES_H384 = syn.MoeShape(E=4, H=384, I=256, k=2)                    # H = 1.5 column blocks of 256


def run(prob, tokens=None):
    kw = {}
    if prob.get("w13_bias") is not None:
        kw = dict(w13_bias=prob["w13_bias"], w2_bias=prob["w2_bias"])
    out = api.moe_fp8_block_forward(prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"],
                                    prob["w13_scale"], prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"],
                                    prob["w2_scale"].stride(1), **kw)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == 2   # the default gate takes prefill at these slot counts
    args, tok = oracle_args(prob, tokens)
    ref = mo.forward(*args, act="e4m3", **oracle_biases(prob, tokens))
    return check_per_token(out.float().cpu().numpy()[tok], ref), out


def tile_counts(prob, E):
    rl = mo.route_lists(prob["topk_ids"].cpu().numpy(), E)
    return -(-rl["counts"].astype(np.int64) // 128)


@pytest.mark.parametrize("routing", ["softmax", "zipf"])
def test_prefill_tiles(cuda_lib, routing):
    prob = syn.make_problem(TILES_A, 512, 0, "cuda", routing=routing)
    r, _ = run(prob)
    assert r < TOL


def test_prefill_tiles_odd_and_empty_experts(cuda_lib):
    prob = syn.make_problem(TILES_B, 1024, 1, "cuda", routing="zipf")
    tiles = tile_counts(prob, TILES_B.E)
    assert (tiles % 2 == 1).any(), "the case needs an expert with an odd tile count"
    r, _ = run(prob)
    assert r < TOL


def test_prefill_tiles_odd_tile_counts_softmax(cuda_lib):
    prob = syn.make_problem(TILES_B, 1100, 2, "cuda")
    r, _ = run(prob)
    assert r < TOL


@pytest.mark.parametrize("shape", [TILES_RAGGED, TILES_H384], ids=["ragged", "H384"])
def test_prefill_tiles_partial_blocks(cuda_lib, shape):
    prob = syn.make_problem(shape, 512, 3, "cuda")
    r, _ = run(prob)
    assert r < TOL


def test_prefill_tiles_biases(cuda_lib):
    prob = syn.make_problem(TILES_RAGGED, 512, 4, "cuda", routing="zipf")
    b13, b2 = syn.make_biases(TILES_RAGGED, 4, "cuda")
    prob["w13_bias"], prob["w2_bias"] = b13, b2
    r, _ = run(prob)
    assert r < TOL


def test_prefill_tiles_deterministic(cuda_lib):
    prob = syn.make_problem(TILES_B, 1024, 5, "cuda", routing="zipf")
    _, a = run(prob)
    b = api.forward_problem(prob)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
