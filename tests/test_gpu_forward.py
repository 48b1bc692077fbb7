"""Layer parity on the GPU against the float64 oracle, through the C ABI:
max_i |gpu[t,i] - oracle[t,i]| <= 2e-2 * max_i |oracle[t,i]| for every token,
on the five workloads (sampled tokens where the full oracle is too slow),
plus routing edge cases, determinism, padding and CUDA-graph replay."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, diagnostics, synthetic as syn
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


def run_and_check(prob, path, tokens=None, mode="gathered", decode_act=None):
    out = api.forward_problem(prob, force_path=path, decode_act=decode_act)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == (1 if path == "decode" else 2)
    args, tok = oracle_args(prob, tokens)
    if path == "decode":
        act = "e4m3_x" if decode_act == "e4m3" else "bf16"
    else:
        act = "e4m3"
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
@pytest.mark.parametrize("T,tokens", [(1, None), (4, None), (16, [0, 5, 10, 15]), (64, [0, 21, 42, 63])])
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


def test_default_gate_unit_rows(cuda_lib):
    """Default gate on a layer whose decode gate/up units hold 4 row pairs
    (H = 2560, hot experts): decode only while the batch routes at most 8
    slots, the grouped GEMMs from there on (measured faster from T = 2)."""
    api.forward_problem(problem(syn.PADDED_SKEWED, 1, routing="hot"))
    assert api.moe_fp8_block_last_path() == 1
    api.forward_problem(problem(syn.PADDED_SKEWED, 8, routing="hot"))
    assert api.moe_fp8_block_last_path() == 2


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


def test_hostio_pageable_and_prefill(cuda_lib):
    """Host buffers: pageable ones are staged through the workspace, page-locked
    ones are read and written in place by the kernels; both give the device
    call's output, on the decode and the prefill path."""
    for shape, T, path in ((syn.DECODE_SMALL, 4, "decode"), (syn.PREFILL, 64, "prefill")):
        prob = problem(shape, T)
        dev_out = api.forward_problem(prob, force_path=path)
        torch.cuda.synchronize()
        for pinned in (False, True):
            h, i, w = (prob[n].cpu() for n in ("hidden", "topk_ids", "topk_weights"))
            out = torch.full((T, shape.H), float("nan"), dtype=torch.bfloat16)
            if pinned:
                h, i, w, out = h.pin_memory(), i.pin_memory(), w.pin_memory(), out.pin_memory()
            api.moe_fp8_block_forward_hostio(h, i, w, prob["w13"], prob["w13_scale"], prob["w13_scale"].stride(1),
                                             prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1), out=out,
                                             force_path=path)
            assert torch.equal(out, dev_out.cpu()), (path, pinned)


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


def tile_probe_tokens(ids: np.ndarray, E: int, n: int = 64, seed: int = 0):
    """Tokens that land on every form of the grouped GEMM's 128-row M tiles
    (rows in the routing lists' order, expert ascending, stable in the slot
    index): rows 0, 127, 128 and 255 of experts with two or more tiles (the
    form where the two CTAs of a pair take M tiles 2i and 2i+1), the first
    and last rows of the last tile of experts with an odd tile count (the
    form where both CTAs take that one tile), the last row of every expert
    (the ragged tail), then random tokens up to `n`, plus tokens 0 and T-1.
    Every checked token covers all column blocks, the last one included."""
    T, k = ids.shape
    rl = mo.route_lists(ids, E)
    off, perm = rl["offsets"], rl["perm"]
    pick = {0, T - 1}
    tiles = -(-rl["counts"].astype(np.int64) // 128)
    two = [e for e in range(E) if tiles[e] >= 2]
    odd = [e for e in range(E) if tiles[e] % 2 == 1]
    rng = np.random.default_rng(seed)
    for e in rng.permutation(two)[:6]:
        c = off[e + 1] - off[e]
        pick.update(int(perm[off[e] + r]) // k for r in (0, 127, 128, min(255, c - 1)))
    for e in rng.permutation(odd)[:6]:
        c = off[e + 1] - off[e]
        first = (tiles[e] - 1) * 128
        pick.update(int(perm[off[e] + r]) // k for r in (first, c - 1))
    for e in rng.permutation(E)[:8]:
        if off[e + 1] > off[e]:
            pick.add(int(perm[off[e + 1] - 1]) // k)
    rest = [t for t in rng.permutation(T) if t not in pick]
    pick.update(int(t) for t in rest[:max(0, n - len(pick))])
    return sorted(pick)


@pytest.mark.parametrize("T,routing", [(1024, "softmax"), (1024, "zipf")])
def test_prefill_grouped_gemm(cuda_lib, T, routing):
    r, _ = run_and_check(problem(syn.PREFILL, T, routing=routing), "prefill")
    assert r < TOL


@pytest.mark.slow
@pytest.mark.parametrize("T,routing", [(4096, "softmax"), (4096, "zipf"), (16384, "softmax"), (16384, "zipf")])
def test_prefill_grouped_gemm_full_size(cuda_lib, T, routing):
    """The prefill workload at full size (the bench's T = 4096 and 16384),
    checked on at least 64 tokens chosen to hit both pair-tile forms and
    the ragged tail of several experts."""
    prob = problem(syn.PREFILL, T, routing=routing)
    tokens = tile_probe_tokens(prob["topk_ids"].cpu().numpy(), syn.PREFILL.E, n=64, seed=T)
    assert len(tokens) >= 64
    r, _ = run_and_check(prob, "prefill", tokens=tokens)
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


# -------------------------------------------------------- decode (W8A8)
@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_w8a8_small_experts(cuda_lib, T):
    r, _ = run_and_check(problem(syn.DECODE_SMALL, T), "decode", decode_act="e4m3")
    assert r <= TOL


def test_decode_w8a8_padded_skewed(cuda_lib):
    r, _ = run_and_check(problem(syn.PADDED_SKEWED, 8, routing="hot"), "decode", decode_act="e4m3")
    assert r <= TOL


@pytest.mark.slow
def test_decode_w8a8_wide_experts(cuda_lib):
    # H = 7168: 14 K blocks per warp, the kernel's non-register path
    r, _ = run_and_check(problem(syn.DECODE_WIDE, 2), "decode", tokens=[0, 1], decode_act="e4m3")
    assert r <= TOL


def test_decode_w8a8_exact_grid_equals_w8a16(cuda_lib):
    """Activations on the e4m3 grid with a 448 code in every group quantise
    exactly, so W8A8 decode must give the W8A16 output up to summation
    order."""
    prob = problem(syn.DECODE_SMALL, 4)
    g = torch.Generator().manual_seed(3)
    finite = torch.tensor([b for b in range(256) if b not in (0x7F, 0xFF)], dtype=torch.uint8)
    codes = finite[torch.randint(0, len(finite), (4, syn.DECODE_SMALL.H), generator=g)]
    codes[:, ::128] = 0x7E
    prob["hidden"] = (codes.view(torch.float8_e4m3fn).to(torch.float32) * 2.0 ** -4).to(torch.bfloat16).cuda()
    a = api.forward_problem(prob, force_path="decode").float()
    b = api.forward_problem(prob, force_path="decode", decode_act="e4m3").float()
    torch.cuda.synchronize()
    scale = a.abs().amax(dim=1, keepdim=True)
    assert torch.all((a - b).abs() <= 1e-5 * scale)


def test_decode_ulp_verify(cuda_lib):
    """The W8A8-versus-W8A16 diagnostic runs, its statistics are consistent,
    and its per-token distance agrees with the oracle's own W8A8-versus-W8A16
    distance: each GPU mode is within the parity tolerance of its oracle, so
    the two distances differ by at most twice that tolerance."""
    prob = problem(syn.DECODE_SMALL, 8)
    st = diagnostics.decode_ulp_verify(prob)
    assert np.isfinite(st["max_ulp"]) and st["max_ulp"] >= st["mean_ulp"] >= 0.0
    assert 0.0 <= st["frac_over_2"] <= 1.0
    args, _ = oracle_args(prob)
    r16 = mo.forward(*args, act="bf16")
    r8 = mo.forward(*args, act="e4m3_x")
    oracle_rel = float(np.max(np.max(np.abs(r16 - r8), axis=1) / np.max(np.abs(r16), axis=1)))
    assert abs(st["max_rel_row"] - oracle_rel) <= 2 * TOL
