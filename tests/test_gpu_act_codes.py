"""The forward's own activation codes, bit for bit against the oracle.

The dynamic activation quantisation (fp8-moe-gather page, "Affects": scale =
amax / 448 per token per 128 columns, codes rounded to nearest even and
saturated) runs inside the forward's kernels: the prefill path's
quantise-and-permute kernel writes the codes into the rows the grouped GEMM
reads, and the W8A8 decode path's gate/up kernel quantises each token
itself.  moe_fp8_block_forward_act_codes returns the codes and scales those
kernels produced in the call, and they must equal oracle.quantize_per_128
exactly: every code byte and every scale bit."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args

pytestmark = pytest.mark.gpu

RAGGED_H = syn.MoeShape(E=16, H=320, I=176, k=4)   # last 128-column group holds 64 columns
EDGE = syn.MoeShape(E=8, H=384, I=128, k=2)

_W = {}


def weights(shape):
    key = (shape.E, shape.H, shape.I, shape.w13_scale_stride, shape.w2_scale_stride)
    if key not in _W:
        _W.clear()
        torch.cuda.empty_cache()
        _W[key] = syn.make_weights(shape, 0, "cuda")
    return _W[key]


def problem(shape, T, routing="softmax", hidden=None):
    w13, w13s, w2, w2s = weights(shape)
    x = syn.make_hidden(T, shape.H, 0, "cuda", step=T) if hidden is None else hidden.cuda()
    ids, w = syn.make_routing(T, shape.E, shape.k, 0, "cuda", routing, step=T)
    return dict(hidden=x, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)


def forward_codes(prob, path, decode_act=None):
    out, codes, scales = api.moe_fp8_block_forward_act_codes(
        prob["hidden"], prob["topk_ids"], prob["topk_weights"], prob["w13"], prob["w13_scale"],
        prob["w13_scale"].stride(1), prob["w2"], prob["w2_scale"], prob["w2_scale"].stride(1),
        force_path=path, decode_act=decode_act)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_last_path() == (1 if path == "decode" else 2)
    return out, codes.cpu().numpy(), scales.cpu().numpy()


def check_codes(prob, codes, scales):
    ids = prob["topk_ids"].cpu().numpy()
    E = prob["w13"].shape[0]
    routed = np.any((ids >= 0) & (ids < E), axis=1)   # a token with no valid slot has no GEMM row
    rc, rs = mo.quantize_per_128(prob["hidden"].float().cpu().numpy())
    assert np.array_equal(scales[routed].view(np.uint32), rs[routed].view(np.uint32))
    bad = np.nonzero(np.any(codes[routed] != rc[routed], axis=1))[0]
    assert bad.size == 0, f"tokens {bad[:8]} differ"
    return int(routed.sum())


@pytest.mark.parametrize("T,routing", [(1, "softmax"), (16, "softmax"), (1024, "zipf"), (16384, "softmax")])
def test_prefill_forward_act_codes(cuda_lib, T, routing):
    prob = problem(syn.PREFILL, T, routing)
    _, codes, scales = forward_codes(prob, "prefill")
    assert check_codes(prob, codes, scales) == T


def test_prefill_forward_act_codes_ragged_group(cuda_lib):
    prob = problem(RAGGED_H, 64)
    out, codes, scales = forward_codes(prob, "prefill")
    check_codes(prob, codes, scales)
    args, _ = oracle_args(prob)
    check_per_token(out.float().cpu().numpy(), mo.forward(*args, act="e4m3"))


def edge_hidden(T=8):
    """Groups that exercise the quantiser's special cases: all zero, all equal,
    one sign, amax far above the rest (a value that underflows to code 0 and
    one that lands in e4m3's subnormal range), and large magnitudes."""
    x = torch.zeros(T, EDGE.H, dtype=torch.float32)
    x[1, :128] = 3.0                                   # all equal: every code 0x7E
    x[2, 128:256] = -0.5                               # all equal, negative: 0xFE
    x[3] = torch.linspace(-1e4, 1e4, EDGE.H)
    x[3, 300] = 2.0 ** -120                            # far below amax / 2^17: code 0
    x[4, :128] = torch.linspace(0, 1, 128)
    x[4, 5] = 1e-5                                     # x / scale in e4m3's subnormal range
    x[5] = (torch.arange(EDGE.H) % 7 - 3).float() * 2.0 ** -20
    x[6, 256:] = -1e-30                                # a tiny, all-equal group
    x[7] = torch.randn(EDGE.H, generator=torch.Generator().manual_seed(5)) * 1e3
    return x.to(torch.bfloat16)


def test_prefill_forward_act_codes_edge_groups(cuda_lib):
    prob = problem(EDGE, 8, hidden=edge_hidden())
    _, codes, scales = forward_codes(prob, "prefill")
    assert check_codes(prob, codes, scales) == 8
    assert np.all(codes[1, :128] == 0x7E) and np.all(codes[2, 128:256] == 0xFE)
    assert scales[0, 0] == 0.0 and np.all(codes[0] == 0)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_w8a8_forward_act_codes(cuda_lib, T):
    prob = problem(syn.DECODE_SMALL, T)
    out, codes, scales = forward_codes(prob, "decode", decode_act="e4m3")
    assert check_codes(prob, codes, scales) == T
    args, _ = oracle_args(prob)
    r = check_per_token(out.float().cpu().numpy(), mo.forward(*args, act="e4m3_x"))
    assert r <= TOL


def test_decode_w8a8_forward_act_codes_edge_groups(cuda_lib):
    prob = problem(EDGE, 8, hidden=edge_hidden())
    _, codes, scales = forward_codes(prob, "decode", decode_act="e4m3")
    assert check_codes(prob, codes, scales) == 8


def test_w8a16_decode_has_no_codes(cuda_lib):
    prob = problem(syn.DECODE_SMALL, 2)
    with pytest.raises(_lib.MoeError) as ei:
        forward_codes(prob, "decode")
    assert ei.value.code == -9
