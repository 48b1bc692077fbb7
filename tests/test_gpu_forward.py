"""Layer parity on the GPU against the float64 oracle, through the C ABI:
max_i |gpu[t,i] - oracle[t,i]| <= 2e-2 * max_i |oracle[t,i]| for every token,
on the five workloads (sampled tokens where the full oracle is too slow),
plus routing edge cases, determinism, padding and CUDA-graph replay."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args

pytestmark = pytest.mark.gpu

_WEIGHTS = {}


def weights(shape: syn.MoeShape, seed=0):
    key = (shape.E, shape.H, shape.I, shape.w13_scale_stride, shape.w2_scale_stride, seed)
    if key not in _WEIGHTS:
        if len(_WEIGHTS) >= 2:
            _WEIGHTS.clear()
            torch.cuda.empty_cache()
        _WEIGHTS[key] = syn.make_weights(shape, seed, "cuda")
    return _WEIGHTS[key]


def problem(shape, T, routing="softmax", seed=0, step=0):
    w13, w13s, w2, w2s = weights(shape, seed)
    hidden = syn.make_hidden(T, shape.H, seed, "cuda", step)
    ids, w = syn.make_routing(T, shape.E, shape.k, seed, "cuda", routing, step=step)
    return dict(hidden=hidden, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)


def run_and_check(prob, path, tokens=None, mode="gathered"):
    out = api.forward_problem(prob, force_path=path)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == (1 if path == "decode" else 2)
    args, tok = oracle_args(prob, tokens)
    act = "bf16" if path == "decode" else "e4m3"
    ref = mo.forward(*args, mode=mode, act=act)
    got = out.float().cpu().numpy()[tok]
    return check_per_token(got, ref), out


# -------------------------------------------------------- decode (W8A16)
def test_tiny_decode_all_expert_oracle(cuda_lib):
    prob = problem(syn.TINY, 4)
    r, _ = run_and_check(prob, "decode", mode="all")
    assert r < 0.01


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_decode_small_experts(cuda_lib, T):
    r, _ = run_and_check(problem(syn.DECODE_SMALL, T), "decode")
    assert r < TOL


@pytest.mark.parametrize("T", [1, 8, 32])
def test_padded_skewed_decode(cuda_lib, T):
    r, _ = run_and_check(problem(syn.PADDED_SKEWED, T, routing="hot"), "decode")
    assert r < TOL


@pytest.mark.slow
@pytest.mark.parametrize("T,tokens", [(1, None), (4, None), (16, [0, 7, 15]), (64, [0, 31, 63])])
def test_decode_wide_experts(cuda_lib, T, tokens):
    r, _ = run_and_check(problem(syn.DECODE_WIDE, T), "decode", tokens=tokens)
    assert r < TOL


@pytest.mark.slow
@pytest.mark.parametrize("T,tokens", [(32, [0, 15, 31])])
def test_prefill_wide_experts(cuda_lib, T, tokens):
    """The prefill path on the wide-expert layer (H=7168, I=2048), where
    the default gate sends every token count."""
    r, _ = run_and_check(problem(syn.DECODE_WIDE, T), "prefill", tokens=tokens)
    assert r < TOL


def test_decode_status_and_skipped_slots(cuda_lib):
    prob = problem(syn.TINY, 4)
    ids = prob["topk_ids"].clone()
    ids[0, 1] = -1
    ids[1, 0] = 8          # >= E: skipped and flagged
    ids[2, 1] = ids[2, 0]  # duplicate expert inside a token
    prob["topk_ids"] = ids
    api.moe_fp8_block_device_status()
    r, _ = run_and_check(prob, "decode")
    assert api.moe_fp8_block_device_status() == 1


def test_decode_deterministic(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 16)
    a = api.forward_problem(prob, force_path="decode")
    b = api.forward_problem(prob, force_path="decode")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_decode_padded_equals_unpadded(cuda_lib):
    """Same logical scales in a padded and an unpadded bank give identical
    output (FreeToken PR #662, 'honor padded fp8 scale strides')."""
    prob = problem(syn.PADDED_SKEWED, 8, routing="hot")
    w2s = prob["w2_scale"]
    assert w2s.shape[2] == 6
    unp = dict(prob)
    unp["w2_scale"] = w2s[..., :5].contiguous()
    a = api.forward_problem(prob, force_path="decode")
    b = api.forward_problem(unp, force_path="decode")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_default_gate(cuda_lib):
    """Default gate: decode while T*k <= E on a layer whose decode stream
    keeps at least 4 ring stages (H = 2048)."""
    for T in (6, 16):
        api.forward_problem(problem(syn.DECODE_SMALL, T))
        assert api.moe_fp8_block_last_path() == 1


def test_gate_ratio_option(cuda_lib):
    """A caller ratio applies the page's rule: decode while T*k <= E*ratio."""
    prob = problem(syn.DECODE_SMALL, 7)   # 56 slots > 128 * 0.4
    api.forward_problem(prob, gate_ratio=0.4)
    assert api.moe_fp8_block_last_path() == 2
    api.forward_problem(problem(syn.DECODE_SMALL, 6), gate_ratio=0.4)
    assert api.moe_fp8_block_last_path() == 1


@pytest.mark.slow
def test_default_gate_wide_layer(cuda_lib):
    """H = 7168 leaves the decode stream 3 ring stages: prefill by default."""
    api.forward_problem(problem(syn.DECODE_WIDE, 3))
    assert api.moe_fp8_block_last_path() == 2


def test_graph_capture_replay_new_routing(cuda_lib):
    shape = syn.DECODE_SMALL
    prob = problem(shape, 4)
    s = torch.cuda.Stream()
    api.moe_fp8_block_reserve(16, shape.k, shape.H, shape.I, shape.E, stream=s)
    out = torch.empty(4, shape.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        api.forward_problem(prob, out=out, stream=s, force_path="decode")
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.forward_problem(prob, out=out, stream=s, force_path="decode")
    for step in range(1, 3):
        nxt = problem(shape, 4, step=step)
        prob["hidden"].copy_(nxt["hidden"])
        prob["topk_ids"].copy_(nxt["topk_ids"])
        prob["topk_weights"].copy_(nxt["topk_weights"])
        g.replay()
        torch.cuda.synchronize()
        args, tok = oracle_args(prob)
        ref = mo.forward(*args)
        check_per_token(out.float().cpu().numpy(), ref)


def test_hostio_matches_device(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 4)
    dev_out = api.forward_problem(prob, force_path="decode")
    torch.cuda.synchronize()
    h = prob["hidden"].cpu().pin_memory()
    i = prob["topk_ids"].cpu().pin_memory()
    w = prob["topk_weights"].cpu().pin_memory()
    out = api.moe_fp8_block_forward_hostio(h, i, w, prob["w13"], prob["w13_scale"], prob["w13_scale"].stride(1),
                                           prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1),
                                           force_path="decode")
    assert torch.equal(out, dev_out.cpu())


def test_empty_and_all_skipped(cuda_lib):
    prob = problem(syn.TINY, 0)
    out = api.forward_problem(prob)
    assert out.shape == (0, 256)
    prob = problem(syn.TINY, 3)
    prob["topk_ids"] = torch.full_like(prob["topk_ids"], -1)
    out = api.forward_problem(prob, force_path="decode")
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


# ------------------------------------------------------- prefill (W8A8)
def test_tiny_prefill_all_expert_oracle(cuda_lib):
    prob = problem(syn.TINY, 4)
    r, _ = run_and_check(prob, "prefill", mode="all")
    assert r < TOL


@pytest.mark.parametrize("T", [1, 7, 16])
def test_prefill_small_experts(cuda_lib, T):
    r, _ = run_and_check(problem(syn.DECODE_SMALL, T), "prefill")
    assert r < TOL


@pytest.mark.parametrize("T", [8, 32])
def test_prefill_padded_skewed(cuda_lib, T):
    r, _ = run_and_check(problem(syn.PADDED_SKEWED, T, routing="hot"), "prefill")
    assert r < TOL


@pytest.mark.parametrize("T,routing,tokens", [
    (1024, "softmax", None), (1024, "zipf", None),
    (4096, "softmax", [0, 1, 2047, 4095]), (4096, "zipf", [3, 100, 4000]),
    (16384, "zipf", [0, 8191, 16383]),
])
def test_prefill_grouped_gemm(cuda_lib, T, routing, tokens):
    r, _ = run_and_check(problem(syn.PREFILL, T, routing=routing), "prefill", tokens=tokens)
    assert r < TOL


def test_default_gate_prefill(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 17)   # 136 slots > E = 128
    api.forward_problem(prob)
    assert api.moe_fp8_block_last_path() == 2


def test_prefill_deterministic_and_padded(cuda_lib):
    prob = problem(syn.PADDED_SKEWED, 32, routing="hot")
    a = api.forward_problem(prob, force_path="prefill")
    b = api.forward_problem(prob, force_path="prefill")
    unp = dict(prob)
    unp["w2_scale"] = prob["w2_scale"][..., :5].contiguous()
    c = api.forward_problem(unp, force_path="prefill")
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_prefill_matches_decode_closely(cuda_lib):
    """Gathered W8A16 and W8A8 paths on the same inputs agree to the
    activation-quantisation error (the pages' VERIFY mode compares the two
    paths of one layer)."""
    prob = problem(syn.DECODE_SMALL, 8)
    d = api.forward_problem(prob, force_path="decode").float()
    p = api.forward_problem(prob, force_path="prefill").float()
    torch.cuda.synchronize()
    scale = d.abs().amax(dim=1)
    assert torch.all((d - p).abs().amax(dim=1) <= 0.1 * scale)


def test_prefill_status_and_skipped_slots(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 16)
    ids = prob["topk_ids"].clone()
    ids[0, 1] = -1
    ids[1, 0] = 128
    ids[2, 1] = ids[2, 0]
    prob["topk_ids"] = ids
    api.moe_fp8_block_device_status()
    r, _ = run_and_check(prob, "prefill")
    assert api.moe_fp8_block_device_status() == 1
