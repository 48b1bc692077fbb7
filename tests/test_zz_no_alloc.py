"""The allocation-free decode entry point, through the C ABI.

For callers that cannot let the library allocate device memory (a
pre-planned memory budget, or a serving loop where cudaMalloc's implicit
synchronisation and possible failure are not acceptable), the library
offers moe_fp8_block_forward_decode_noalloc, whose scratch is a fixed,
statically allocated device array.  Its output must match the float64
oracle and the regular forward on the same inputs -- on two calls in a row,
since every call reuses the same array -- its status word must be readable
through moe_fp8_block_noalloc_status, and a call too large for the array
must be refused with an error instead of running.

This file is collected last so that a failure here does not hide the
results of the other GPU tests."""
import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args

pytestmark = pytest.mark.gpu


def _problem(shape, T, step, weights):
    w13, w13s, w2, w2s = weights
    ids, w = syn.make_routing(T, shape.E, shape.k, 0, "cuda", "softmax", step=step)
    return dict(hidden=syn.make_hidden(T, shape.H, 0, "cuda", step), topk_ids=ids, topk_weights=w, w13=w13,
                w13_scale=w13s, w2=w2, w2_scale=w2s)


def _noalloc(prob, out):
    return api.moe_fp8_block_forward_decode_noalloc(
        prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"], prob["w13_scale"],
        prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1), out)


def test_noalloc_matches_oracle_and_forward_on_two_calls(cuda_lib):
    shape = syn.DECODE_SMALL
    weights = syn.make_weights(shape, 0, "cuda")
    api.moe_fp8_block_noalloc_status()           # first call on the device: looks the array up, clears status
    for T, step in ((16, 1), (4, 2)):          # two calls in a row on the shared scratch
        prob = _problem(shape, T, step, weights)
        out = torch.empty(T, shape.H, dtype=torch.bfloat16, device="cuda")
        _noalloc(prob, out)
        assert api.moe_fp8_block_last_path() == 1
        assert api.moe_fp8_block_last_launches() >= 1
        ref = api.forward_problem(prob, force_path="decode")
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        args, _ = oracle_args(prob)
        assert check_per_token(got, mo.forward(*args)) < TOL
        assert check_per_token(got, ref.float().cpu().numpy()) < TOL
        assert api.moe_fp8_block_noalloc_status() == 0


def test_noalloc_status_reports_bad_expert_ids(cuda_lib):
    shape = syn.DECODE_SMALL
    weights = syn.make_weights(shape, 0, "cuda")
    prob = _problem(shape, 4, 5, weights)
    ids = prob["topk_ids"].clone()
    ids[1, 2] = shape.E + 3                     # out of range: skipped and flagged
    prob["topk_ids"] = ids
    out = torch.empty(4, shape.H, dtype=torch.bfloat16, device="cuda")
    _noalloc(prob, out)
    assert api.moe_fp8_block_noalloc_status() & _lib.MOE_STATUS_BAD_ID
    assert api.moe_fp8_block_noalloc_status() == 0      # reading clears it
    args, tok = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy()[tok], mo.forward(*args)) < TOL


def test_noalloc_refuses_calls_too_large_for_its_array(cuda_lib):
    shape = syn.DECODE_WIDE
    small = syn.MoeShape(E=8, H=shape.H, I=shape.I, k=8)
    weights = syn.make_weights(small, 0, "cuda")
    prob = _problem(small, 256, 3, weights)   # 2048 slots x (7168 + 2048) x 4 B > 8 MiB
    out = torch.empty(256, small.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.MoeError) as ei:
        _noalloc(prob, out)
    assert ei.value.code == -9
    assert "needs" in _lib.load().moe_fp8_block_last_error_detail().decode()
