"""Pins for the float64 oracle: every check here ties the oracle to something
other than itself -- a number or rule the pages state, a closed form, a
library routine, an invariant or a brute-force evaluation on a tiny case.
CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from block_fp8_mixture_route_gb300 import synthetic as syn

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
FINITE = [b for b in range(256) if b not in (0x7F, 0xFF)]


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ e4m3 table --
def test_e4m3_table_matches_fp16_bit_trick():
    """(b&0x80)<<8 | (b&0x7F)<<7 read as fp16 is e4m3(b) * 2^-8 (FreeToken
    PR #662, 'Kernels'); holds for every finite code, subnormals included."""
    f = GOLDEN["fp16_bit_trick"]
    b = np.array(FINITE, dtype=np.uint16)
    h = ((b & 0x80) << f["sign_shift"]) | ((b & 0x7F) << f["magnitude_shift"])
    v = h.astype(np.uint16).view(np.float16).astype(np.float64) * 2.0 ** (-f["power_of_two"])
    t = mo.e4m3_table()[FINITE]
    assert np.array_equal(v, t)
    assert np.array_equal(np.signbit(v), np.signbit(t))


def test_e4m3_table_matches_torch_float8_cast():
    codes = torch.tensor(FINITE, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(mo.e4m3_table()[FINITE], ref)


def test_e4m3_widening_to_bf16_is_exact():
    """e4m3 -> bf16 is exact for every finite code (FreeToken PR #662, PR body)."""
    t = mo.e4m3_table()[FINITE]
    rt = torch.tensor(t).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(t, rt)


def test_e4m3_special_values_from_pages():
    t = mo.e4m3_table()
    span = GOLDEN["e4m3_span"]
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == span["smallest_subnormal"]
    assert np.nanmax(t) == span["largest_finite"] and t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.nanmin(np.abs(t[t != 0])) == span["smallest_subnormal"]
    for c in GOLDEN["e4m3_nan_codes"]["codes"]:
        assert math.isnan(t[c])
    sub = GOLDEN["e4m3_subnormal_rule"]
    for m in range(8):
        assert t[(sub["exponent_field"] << 3) | m] == m * sub["value_per_mantissa_unit"]
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0 and t[0x30] == 0.5 and t[0xB8] == -1.0
    assert np.sum(np.isnan(t)) == 2


# ------------------------------------------------------- e4m3 encoding ---
def test_encode_round_trips_every_finite_code():
    t = mo.e4m3_table()
    for b in FINITE:
        assert mo.e4m3_encode_rne_satfinite(np.float32(t[b]))[()] == b, hex(b)


def test_encode_midpoints_round_to_even():
    t = mo.e4m3_table()
    pos = sorted(set(t[b] for b in range(0x7F)))
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2         # representable in fp32
        c = mo.e4m3_encode_rne_satfinite(mid)[()]
        expect = mo.e4m3_encode_rne_satfinite(np.float32(lo))[()]
        if expect & 1:
            expect = mo.e4m3_encode_rne_satfinite(np.float32(hi))[()]
        assert c == expect and (c & 1) == 0


def test_encode_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(1)
    mag = torch.exp2(torch.empty(200000).uniform_(-12, 8.807, generator=g))
    x = (mag * torch.where(torch.rand(200000, generator=g) < 0.5, -1.0, 1.0)).float()
    x = x[x.abs() <= 448]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mo.e4m3_encode_rne_satfinite(x.numpy()), ref)


def test_encode_saturates_and_nan():
    enc = mo.e4m3_encode_rne_satfinite
    assert enc(np.float32(1e6))[()] == 0x7E and enc(np.float32(-1e6))[()] == 0xFE
    assert enc(np.float32(np.inf))[()] == 0x7E and enc(np.float32(-np.inf))[()] == 0xFE
    assert enc(np.float32(470.0))[()] == 0x7E
    assert enc(np.float32(np.nan))[()] == 0x7F
    assert enc(np.float32(-0.0))[()] == 0x80 and enc(np.float32(0.0))[()] == 0x00
    assert enc(np.float32(2.0 ** -11))[()] == 0x00          # below half the smallest subnormal
    assert enc(np.float32(-2.0 ** -10 * 1.01))[()] == 0x81  # just above half: rounds to -2^-9


# ------------------------------------------------ activation quantisation --
def test_quantize_amax_maps_to_448_and_scale_is_amax_over_448():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(16, 384, generator=g).to(torch.bfloat16).float().numpy()
    codes, scales = mo.quantize_per_128(x)
    for r in range(16):
        for gi in range(3):
            blk = x[r, gi * 128:(gi + 1) * 128]
            i = int(np.argmax(np.abs(blk)))
            assert codes[r, gi * 128 + i] == (0xFE if blk[i] < 0 else 0x7E)
            assert scales[r, gi] == np.float32(np.float32(np.abs(blk[i])) / np.float32(448.0))
            # every code equals torch's cast of the fp32 quotient (|q| <= 448 here)
            q = torch.from_numpy((blk / scales[r, gi]).astype(np.float32))
            q = q.clamp(-448, 448)
            assert np.array_equal(codes[r, gi * 128:(gi + 1) * 128],
                                  q.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_quantize_degenerate_groups():
    x = np.zeros((3, 256), dtype=np.float32)
    x[1, :128] = 3.0                   # all-equal group
    x[2, 128:] = -0.5
    codes, scales = mo.quantize_per_128(x)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert np.all(codes[1, :128] == 0x7E) and scales[1, 0] == np.float32(3.0 / 448)
    assert np.all(codes[1, 128:] == 0) and scales[1, 1] == 0
    assert np.all(codes[2, 128:] == 0xFE)


# ------------------------------------------------------- block dequant ---
def test_block_scale_applies_to_exactly_its_block():
    """Doubling one block's scale doubles exactly that 128x128 block; a
    transposed or mis-strided scale index fails on this non-square grid."""
    g = torch.Generator().manual_seed(3)
    codes = syn.finite_e4m3_codes((256, 384), g, "cpu").numpy()
    scales = torch.ones(2, 4, dtype=torch.bfloat16)            # padded stride 4 >= 3
    base = mo.dequant_bank(codes, bits(scales))
    for rb in range(2):
        for kb in range(3):
            s2 = scales.clone()
            s2[rb, kb] = 2.0
            d = mo.dequant_bank(codes, bits(s2)) - base
            blk = np.zeros_like(d, dtype=bool)
            blk[rb * 128:(rb + 1) * 128, kb * 128:(kb + 1) * 128] = True
            assert np.array_equal(d[blk], base[blk])
            assert np.all(d[~blk] == 0)
    # padding column is never read
    s3 = scales.clone()
    s3[:, 3] = float("nan")
    assert np.array_equal(mo.dequant_bank(codes, bits(s3)), base)


# --------------------------------------------------------- hand cases ----
def _const_problem(E, H, I, T, k, gate_code, up_code, w2_code, x_val, ids, wts, w2_codes_per_expert=None):
    w13 = np.zeros((E, 2 * I, H), dtype=np.uint8)
    w2 = np.zeros((E, H, I), dtype=np.uint8)
    for e in range(E):
        gc = gate_code[e] if isinstance(gate_code, (list, tuple)) else gate_code
        uc = up_code[e] if isinstance(up_code, (list, tuple)) else up_code
        dc = w2_code[e] if isinstance(w2_code, (list, tuple)) else w2_code
        w13[e, :I] = gc
        w13[e, I:] = uc
        w2[e] = dc
    one = bits(torch.ones(1, dtype=torch.bfloat16))[0]
    w13s = np.full((E, 2 * I // 128, H // 128), one, dtype=np.uint16)
    w2s = np.full((E, H // 128, I // 128), one, dtype=np.uint16)
    hidden = bits(torch.full((T, H), x_val, dtype=torch.bfloat16))
    return hidden, np.array(ids, dtype=np.int32), np.array(wts, dtype=np.float32), w13, w13s, w2, w2s


def silu(z):
    return z / (1.0 + math.exp(-z))


@pytest.mark.parametrize("gate_code,gval", [(0x38, 1.0), (0xB8, -1.0)])
def test_hand_case_constant_codes(gate_code, gval):
    """H=256, I=128, one expert, gate codes +-1.0, up codes 0.5, down codes
    1.0, scales 1, x = 2^-6: gate = +-4, up = 2, h = silu(+-4)*2,
    y = I*h on every output row."""
    H, I = 256, 128
    p = _const_problem(1, H, I, 1, 1, gate_code, 0x30, 0x38, 2.0 ** -6, [[0]], [[1.0]])
    out = mo.forward(*p, mode="gathered")
    g, u = gval * H * 2.0 ** -6, 0.5 * H * 2.0 ** -6
    expect = I * silu(g) * u
    assert np.allclose(out, expect, rtol=1e-14, atol=0)
    assert np.allclose(mo.forward(*p, mode="all"), expect, rtol=1e-14, atol=0)


def test_hand_case_combine_weights():
    """Two experts, k=2; expert 0 has down codes 1.0, expert 1 down codes 0.5;
    token 0 routes (1, 0) with weights (0.25, 0.75)."""
    H, I = 128, 128
    p = _const_problem(2, H, I, 1, 2, 0x38, 0x38, [0x38, 0x30], 2.0 ** -5, [[1, 0]], [[0.25, 0.75]])
    g = H * 2.0 ** -5                      # = 4 for both experts
    h = silu(g) * g
    expect = 0.75 * (I * h * 1.0) + 0.25 * (I * h * 0.5)
    assert np.allclose(mo.forward(*p), expect, rtol=1e-14, atol=0)
    assert np.allclose(mo.forward(*p, mode="all"), expect, rtol=1e-14, atol=0)


def test_hand_case_subnormal_only_codes():
    """All weight codes the smallest subnormal 2^-9 (0x01) or its negative
    (FreeToken PR #662, 'Tests': subnormal-only codes)."""
    H, I = 256, 128
    p = _const_problem(1, H, I, 1, 1, 0x01, 0x81, 0x01, 1.0, [[0]], [[1.0]])
    g = H * 2.0 ** -9
    u = -H * 2.0 ** -9
    expect = I * 2.0 ** -9 * silu(g) * u
    assert np.allclose(mo.forward(*p), expect, rtol=1e-14, atol=0)


def test_scale_power_of_two_scales_its_block_contribution():
    """Doubling the down-projection scale of block (nb, kb) changes only output
    rows of block nb, and there by exactly the contribution of K-block kb."""
    H, I = 256, 256
    prob = syn.make_problem(syn.MoeShape(E=1, H=H, I=I, k=1), T=2, seed=5)
    args = [prob[n] for n in ("hidden", "topk_ids", "topk_weights", "w13", "w13_scale", "w2", "w2_scale")]
    args = [bits(a) if a.dtype == torch.bfloat16 else a.numpy() for a in args]
    base = mo.forward(*args)
    w2s = args[6].copy()
    one = bits(torch.ones(1, dtype=torch.bfloat16))[0]
    w2s[...] = one
    args[6] = w2s
    base = mo.forward(*args)
    w2s2 = w2s.copy()
    w2s2[0, 1, 0] = bits(torch.full((1,), 2.0, dtype=torch.bfloat16))[0]
    args2 = list(args)
    args2[6] = w2s2
    out2 = mo.forward(*args2)
    assert np.array_equal(out2[:, :128], base[:, :128])
    w2s3 = w2s.copy()
    w2s3[0, 1, 0] = 0                      # zero the block instead: removes its contribution
    args3 = list(args)
    args3[6] = w2s3
    out3 = mo.forward(*args3)
    np.testing.assert_allclose(out2[:, 128:] - base[:, 128:], base[:, 128:] - out3[:, 128:], rtol=1e-12, atol=1e-12)
    assert not np.allclose(out2[:, 128:], base[:, 128:])


# ------------------------------------------------------- invariants ------
def _np_args(prob):
    out = []
    for n in ("hidden", "topk_ids", "topk_weights", "w13", "w13_scale", "w2", "w2_scale"):
        a = prob[n]
        out.append(bits(a) if a.dtype == torch.bfloat16 else a.numpy())
    return out


@pytest.mark.parametrize("act", ["bf16", "e4m3", "e4m3_x"])
def test_gathered_equals_all_expert(act):
    """The gathered path equals the all-expert op (fp8-moe-gather page, The
    fix / VERIFY mode) on the tiny 8-expert, 256-hidden problem."""
    prob = syn.make_problem(syn.TINY, T=4, seed=0)
    a = _np_args(prob)
    g = mo.forward(*a, mode="gathered", act=act)
    al = mo.forward(*a, mode="all", act=act)
    scale = np.max(np.abs(al), axis=1, keepdims=True)
    assert np.all(np.abs(g - al) <= 1e-12 * scale)
    # with MLP biases: an unrouted expert's masked y (which includes its b2)
    # must still add nothing
    b13, b2 = (b.numpy() for b in syn.make_biases(syn.TINY, seed=1, std13=30.0, std2=1e5))
    g = mo.forward(*a, mode="gathered", act=act, w13_bias=b13, w2_bias=b2)
    al = mo.forward(*a, mode="all", act=act, w13_bias=b13, w2_bias=b2)
    scale = np.max(np.abs(al), axis=1, keepdims=True)
    assert np.all(np.abs(g - al) <= 1e-12 * scale)


def test_padded_equals_unpadded_scales():
    """Padded scale banks (the page's own 20x5 -> stride 6 example) give
    bit-identical results (FreeToken PR #662, 'honor padded fp8 scale strides')."""
    f = GOLDEN["padded_scale_example"]
    assert f["rows"] * f["cols"] * 2 == f["bytes_unpadded"] and f["bytes_unpadded"] % 16 != 0
    assert (f["rows"] * f["padded_cols"] * 2) % 16 == 0
    shp_p = syn.MoeShape(E=2, H=f["H"], I=f["I"], k=1, w2_scale_stride=f["padded_cols"])
    shp_u = syn.MoeShape(E=2, H=f["H"], I=f["I"], k=1)
    pp = syn.make_problem(shp_p, T=2, seed=7)
    pu = syn.make_problem(shp_u, T=2, seed=7)
    assert tuple(pp["w2_scale"].shape) == (2, f["rows"], f["padded_cols"])
    assert tuple(pu["w2_scale"].shape) == (2, f["rows"], f["cols"])
    assert torch.equal(pp["w2_scale"][..., :f["cols"]], pu["w2_scale"])
    assert torch.isnan(pp["w2_scale"][..., f["cols"]:].float()).all()
    a_p, a_u = _np_args(pp), _np_args(pu)
    for act in ("bf16", "e4m3"):
        o_p = mo.forward(*a_p, act=act)
        o_u = mo.forward(*a_u, act=act)
        assert np.array_equal(o_p, o_u) and np.all(np.isfinite(o_p))


def test_expert_relabelling_invariance():
    prob = syn.make_problem(syn.TINY, T=4, seed=0)
    a = _np_args(prob)
    base = mo.forward(*a)
    perm = np.random.default_rng(0).permutation(8)        # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    b = list(a)
    b[1] = perm[a[1]].astype(np.int32)
    for i in (3, 4, 5, 6):
        b[i] = a[i][inv]
    out = mo.forward(*b)
    assert np.allclose(out, base, rtol=1e-12, atol=1e-12 * np.max(np.abs(base)))


def test_slot_order_invariance_and_negative_slot():
    prob = syn.make_problem(syn.TINY, T=4, seed=0)
    a = _np_args(prob)
    base = mo.forward(*a)
    b = list(a)
    b[1], b[2] = a[1][:, ::-1].copy(), a[2][:, ::-1].copy()
    assert np.allclose(mo.forward(*b), base, rtol=1e-12, atol=1e-12 * np.max(np.abs(base)))
    # a negative id skips its slot: same as weight 0
    c = list(a)
    c[1] = a[1].copy()
    c[1][0, 1] = -1
    d = list(a)
    d[2] = a[2].copy()
    d[2][0, 1] = 0.0
    assert np.allclose(mo.forward(*c), mo.forward(*d), rtol=1e-12, atol=0)


# ------------------------------------------------------- brute force -----
def _brute(hidden_u16, ids, wts, w13, w13s, w2, w2s, act, b13=None, b2=None):
    """Scalar float64 loops; e4m3 decoded through the fp16 bit trick and
    torch's float8 cast for the activation codes (independent of the oracle)."""
    def dec(b):
        h = np.array([((int(b) & 0x80) << 8) | ((int(b) & 0x7F) << 7)], dtype=np.uint16)
        return float(h.view(np.float16)[0]) * 256.0

    def bf(u):
        return float(np.array([int(u) << 16], dtype=np.uint32).view(np.float32)[0])

    def quant_row(v):                       # v: list of fp32 values, one 128-group
        amax = max(abs(z) for z in v)
        sc = float(np.float32(np.float32(amax) / np.float32(448.0)))
        if sc == 0:
            return [0.0] * len(v)
        q = torch.tensor([float(np.float32(np.float32(z) / np.float32(sc))) for z in v], dtype=torch.float32)
        q = q.clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float64).tolist()
        return [qq * sc for qq in q]

    T, H = hidden_u16.shape
    E, I2, _ = w13.shape
    I = I2 // 2
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        x = [bf(hidden_u16[t, c]) for c in range(H)]
        if act in ("e4m3", "e4m3_x"):
            x = sum((quant_row(x[c:c + 128]) for c in range(0, H, 128)), [])
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if e < 0 or e >= E:
                continue
            h = []
            for i in range(I):
                g = sum(dec(w13[e, i, c]) * bf(w13s[e, i // 128, c // 128]) * x[c] for c in range(H))
                u = sum(dec(w13[e, I + i, c]) * bf(w13s[e, (I + i) // 128, c // 128]) * x[c] for c in range(H))
                if b13 is not None:
                    g += float(b13[e, i])
                    u += float(b13[e, I + i])
                # e^-g past the double range is +inf, and g / inf the limit 0
                h.append(g / (1.0 + (math.exp(-g) if g > -709.0 else math.inf)) * u)
            if act == "e4m3":
                h = sum((quant_row([float(np.float32(z)) for z in h[c:c + 128]]) for c in range(0, I, 128)), [])
            for n in range(H):
                y = sum(dec(w2[e, n, i]) * bf(w2s[e, n // 128, i // 128]) * h[i] for i in range(I))
                if b2 is not None:
                    y += float(b2[e, n])
                out[t][n] += float(wts[t, j]) * y
    return np.array(out)


@pytest.mark.parametrize("act", ["bf16", "e4m3", "e4m3_x"])
def test_brute_force_tiny(act):
    shp = syn.MoeShape(E=3, H=128, I=128, k=2, w2_scale_stride=3)
    prob = syn.make_problem(shp, T=2, seed=11)
    a = _np_args(prob)
    a[1][1, 1] = -1                                   # one skipped slot
    ref = _brute(*a, act=act)
    got = mo.forward(*a, act=act)
    scale = np.max(np.abs(ref), axis=1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 1e-12 * scale)


@pytest.mark.parametrize("act", ["bf16", "e4m3"])
def test_brute_force_tiny_bias(act):
    """As test_brute_force_tiny, with gate/up and down-projection biases of
    the size of the projections they are added to."""
    shp = syn.MoeShape(E=3, H=128, I=128, k=2, w2_scale_stride=3)
    prob = syn.make_problem(shp, T=2, seed=12)
    a = _np_args(prob)
    b13, b2 = (b.numpy() for b in syn.make_biases(shp, seed=12, std13=30.0, std2=1e5))
    ref = _brute(*a, act=act, b13=b13, b2=b2)
    got = mo.forward(*a, act=act, w13_bias=b13, w2_bias=b2)
    scale = np.max(np.abs(ref), axis=1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 1e-12 * scale)
    # the biases matter at this size
    assert np.max(np.abs(mo.forward(*a, act=act) - ref) / scale) > 1e-2


@pytest.mark.parametrize("act", ["bf16", "e4m3"])
def test_brute_force_ragged(act):
    """Ragged K and N: H = 192 and I = 144 are not multiples of 128, so the
    last K block of both projections is partial, and the stacked [gate; up]
    bank's 128-row scale blocks straddle the gate/up boundary (up row i uses
    scale row (I + i) // 128); the brute force indexes the banks on its own."""
    shp = syn.MoeShape(E=2, H=192, I=144, k=2)
    prob = syn.make_problem(shp, T=2, seed=13)
    a = _np_args(prob)
    assert a[4].shape[1:] == (3, 2) and a[6].shape[1:] == (2, 2)
    b13, b2 = (b.numpy() for b in syn.make_biases(shp, seed=13, std13=30.0, std2=1e5))
    for bias in (False, True):
        kw = dict(b13=b13, b2=b2) if bias else {}
        ref = _brute(*a, act=act, **kw)
        got = mo.forward(*a, act=act, **({"w13_bias": b13, "w2_bias": b2} if bias else {}))
        scale = np.max(np.abs(ref), axis=1, keepdims=True)
        assert np.all(np.abs(got - ref) <= 1e-12 * scale)


def _pad_problem(a, H2, I2):
    """The problem's banks and activations zero-padded to H2 >= H columns and
    I2 >= I intermediate rows (gate and up padded separately); scale banks
    keep their values, extended by repeating each expert's last scale."""
    x, ids, wts, w13, w13s, w2, w2s = a
    E, I2x, H = w13.shape
    I = I2x // 2
    xp = np.zeros((x.shape[0], H2), dtype=np.uint16)
    xp[:, :H] = x
    w13p = np.zeros((E, 2 * I2, H2), dtype=np.uint8)
    w13p[:, :I, :H] = w13[:, :I]
    w13p[:, I2:I2 + I, :H] = w13[:, I:]
    w2p = np.zeros((E, H2, I2), dtype=np.uint8)
    w2p[:, :H, :I] = w2
    s13 = np.repeat(w13s[:, :1, :1], -(-2 * I2 // 128), axis=1).repeat(-(-H2 // 128), axis=2)
    s2 = np.repeat(w2s[:, :1, :1], -(-H2 // 128), axis=1).repeat(-(-I2 // 128), axis=2)
    return [xp, ids, wts, w13p, s13, w2p, s2]


def test_ragged_equals_zero_padding():
    """With one scale per expert (so the 128-row blocking cannot matter), a
    ragged layer (H = 320, I = 176) equals the same layer zero-padded to
    H = 384, I = 256: the padded activation columns and weight rows add
    nothing, in both activation modes; the padded outputs are exactly 0."""
    shp = syn.MoeShape(E=3, H=320, I=176, k=2)
    prob = syn.make_problem(shp, T=3, seed=14)
    a = _np_args(prob)
    a[4] = np.repeat(a[4][:, :1, :1], a[4].shape[1], axis=1).repeat(a[4].shape[2], axis=2)
    a[6] = np.repeat(a[6][:, :1, :1], a[6].shape[1], axis=1).repeat(a[6].shape[2], axis=2)
    p = _pad_problem(a, 384, 256)
    for act in ("bf16", "e4m3"):
        r = mo.forward(*a, act=act)
        q = mo.forward(*p, act=act)
        assert np.all(q[:, 320:] == 0)
        scale = np.max(np.abs(r), axis=1, keepdims=True)
        assert np.all(np.abs(q[:, :320] - r) <= 1e-12 * scale)


def test_bias_zero_weights_gives_weighted_down_bias():
    """With every weight code 0x00 (+0) both projections vanish, so y = b2
    exactly whatever the gate/up biases, and out_t = sum_j w[t,j] b2[ids[t,j]]
    (tpu-inference PR #3040, review of the bias DMA: the down projection's
    bias is added as it is, with no gate/up split)."""
    prob = syn.make_problem(syn.TINY, T=4, seed=2)
    a = _np_args(prob)
    a[1][3, 0] = -1                                   # a skipped slot adds nothing
    a[3] = np.zeros_like(a[3])
    a[5] = np.zeros_like(a[5])
    b13, b2 = (b.numpy() for b in syn.make_biases(syn.TINY, seed=2))
    got = mo.forward(*a, w13_bias=b13, w2_bias=b2)
    exp = np.zeros_like(got)
    for t in range(a[1].shape[0]):
        for j in range(a[1].shape[1]):
            e = int(a[1][t, j])
            if e >= 0:
                exp[t] += float(a[2][t, j]) * b2[e].astype(np.float64)
    assert np.all(np.abs(got - exp) <= 1e-14 * np.max(np.abs(exp)))


def test_bias_gate_up_split_closed_form():
    """One expert, H = 128, I = 256 (two 128-row gate blocks), w13 codes all
    0x00, gate biases ln 3, up bias of row i equal to i / 256, w2 codes all
    0x38 (1.0), unit scales.  Then gate = ln 3 and silu(ln 3) = (3/4) ln 3, so
    h_i = (3/4) ln 3 * i / 256 and y_n = (3/4) ln 3 * 127.5 + b2_n.  An up
    bias read from the gate half instead (the defect reviewed in
    tpu-inference PR #3040) would give (3/4) (ln 3)^2 * 256 + b2_n."""
    H, I = 128, 256
    one = np.uint16(0x3F80)                           # bf16 1.0
    w13 = np.zeros((1, 2 * I, H), dtype=np.uint8)
    w13s = np.full((1, 2 * I // 128, 1), one, dtype=np.uint16)
    w2 = np.full((1, H, I), 0x38, dtype=np.uint8)
    w2s = np.full((1, 1, 2), one, dtype=np.uint16)
    hidden = np.full((1, H), 0x3F80, dtype=np.uint16)
    ids = np.zeros((1, 1), dtype=np.int32)
    wts = np.ones((1, 1), dtype=np.float32)
    ln3 = np.float32(math.log(3.0))
    b13 = np.concatenate([np.full(I, ln3, dtype=np.float32), np.arange(I, dtype=np.float32) / np.float32(I)])[None]
    b2 = (np.arange(H, dtype=np.float32) - 64.0)[None] * np.float32(0.25)
    got = mo.forward(hidden, ids, wts, w13, w13s, w2, w2s, w13_bias=b13, w2_bias=b2)[0]
    exp = 0.75 * math.log(3.0) * 127.5 + b2[0].astype(np.float64)
    # fp32 rounding of ln 3 moves silu by about 1e-8 relative
    assert np.all(np.abs(got - exp) <= 1e-6 * np.max(np.abs(exp)))


def test_zero_biases_change_nothing():
    prob = syn.make_problem(syn.TINY, T=4, seed=0)
    a = _np_args(prob)
    z13 = np.zeros((syn.TINY.E, 2 * syn.TINY.I), dtype=np.float32)
    z2 = np.zeros((syn.TINY.E, syn.TINY.H), dtype=np.float32)
    for act in ("bf16", "e4m3"):
        assert np.array_equal(mo.forward(*a, act=act, w13_bias=z13, w2_bias=z2), mo.forward(*a, act=act))


def test_w8a8_decode_equals_w8a16_on_the_e4m3_grid():
    """Activations that are e4m3 codes times 2^-4, with a 448 (0x7E) code in
    every 128-group, quantise exactly (scale = 28 / 448 = 2^-4, x / scale =
    the code's value): the W8A8 decode mode must then equal W8A16 exactly,
    while the prefill W8A8 mode, which also quantises h, must not."""
    shp = syn.MoeShape(E=4, H=256, I=128, k=2)
    prob = syn.make_problem(shp, T=3, seed=5)
    g = torch.Generator().manual_seed(3)
    codes = torch.tensor(FINITE, dtype=torch.uint8)[torch.randint(0, len(FINITE), (3, 256), generator=g)]
    codes[:, ::128] = 0x7E
    x = (codes.view(torch.float8_e4m3fn).to(torch.float32) * 2.0 ** -4).to(torch.bfloat16)
    assert torch.equal(x.float(), codes.view(torch.float8_e4m3fn).to(torch.float32) * 2.0 ** -4)
    a = _np_args(prob)
    a[0] = bits(x)
    w8a16 = mo.forward(*a, act="bf16")
    w8a8_dec = mo.forward(*a, act="e4m3_x")
    w8a8_pf = mo.forward(*a, act="e4m3")
    assert np.array_equal(w8a8_dec, w8a16)
    assert not np.array_equal(w8a8_pf, w8a16)


# ------------------------------------------------------- routing lists ---
def test_route_lists_hand_example():
    ids = np.array([[2, 0], [2, -1], [5, 2]], dtype=np.int32)
    r = mo.route_lists(ids, E=4)
    assert r["counts"].tolist() == [1, 0, 3, 0]
    assert r["offsets"].tolist() == [0, 1, 1, 4, 4]
    assert r["perm"].tolist() == [1, 0, 2, 5, -1, -1]
    assert r["inv"].tolist() == [1, 0, 2, -1, -1, 3]
    assert r["glist"].tolist() == [0, 2, -1, -1]
    assert r["D"] == 2 and r["bad_id"]


def test_route_lists_are_a_stable_grouping():
    g = torch.Generator().manual_seed(4)
    ids = torch.randint(-2, 70, (300, 8), generator=g, dtype=torch.int32).numpy()
    r = mo.route_lists(ids, E=64)
    flat = ids.reshape(-1)
    nvalid = int(((flat >= 0) & (flat < 64)).sum())
    p = r["perm"][:nvalid]
    assert sorted(p.tolist()) == sorted(np.nonzero((flat >= 0) & (flat < 64))[0].tolist())
    keys = [(int(flat[s]), int(s)) for s in p]
    assert keys == sorted(keys)
    assert np.all(r["perm"][nvalid:] == -1)
    for s in range(flat.size):
        if r["inv"][s] >= 0:
            assert r["perm"][r["inv"][s]] == s
    assert r["glist"].size == min(64, flat.size)


def test_gate_rule_from_page():
    f = GOLDEN["gate"]
    assert f["default_ratio"] == 0.4
    assert mo.gate_takes_gathered_path(6, 8, 128) and not mo.gate_takes_gathered_path(7, 8, 128)
    assert mo.gate_takes_gathered_path(1, 8, 20) and not mo.gate_takes_gathered_path(1, 8, 19)
