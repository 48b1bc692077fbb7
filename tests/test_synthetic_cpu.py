"""The seeded input recipe (block_fp8_mixture_route_gb300/synthetic.py) on
the CPU: the workloads' shapes and scale strides, and the value
distributions the pages test on -- mixed-sign full-range e4m3 weights with
the NaN codes excluded, bf16 block scales log-uniform in [2^-8, 2^-2],
zero-mean N(0, 1) bf16 activations, softmax / hot / Zipf routing -- plus the
generator's determinism."""
import dataclasses
import math

import pytest
import torch

from block_fp8_mixture_route_gb300 import synthetic as syn


def test_splitmix64_published_outputs():
    # the first three outputs of SplitMix64 seeded with 0 (Steele, Lea and
    # Flood 2014; the state advances by the golden-ratio increment)
    golden = 0x9E3779B97F4A7C15
    outs = [syn.splitmix64((i * golden) & ((1 << 64) - 1)) for i in range(3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


@pytest.mark.parametrize("shape,w13,s13,w2,s2", [
    (syn.TINY, (8, 256, 256), (8, 2, 2), (8, 256, 128), (8, 2, 1)),
    (syn.DECODE_SMALL, (128, 1024, 2048), (128, 8, 16), (128, 2048, 512), (128, 16, 8)),
    (syn.PADDED_SKEWED, (256, 1280, 2560), (256, 10, 20), (256, 2560, 640), (256, 20, 6)),
    (syn.PREFILL, (128, 1024, 2048), (128, 8, 16), (128, 2048, 512), (128, 16, 8)),
])
def test_workload_shapes_and_scale_strides(shape, w13, s13, w2, s2):
    """Bank shapes of the workloads; a padded scale row holds the valid
    block scales, then NaN padding (20 x 5 scales padded to stride 6 in the
    skewed case, 4 padded to 8 in the small-expert and prefill cases)."""
    small = dataclasses.replace(shape, E=2)
    a, sa, b, sb = syn.make_weights(small, seed=0)
    assert tuple(a.shape) == (2,) + w13[1:] and a.dtype == torch.uint8
    assert tuple(b.shape) == (2,) + w2[1:] and b.dtype == torch.uint8
    assert tuple(sa.shape) == (2,) + s13[1:] and sa.dtype == torch.bfloat16
    assert tuple(sb.shape) == (2,) + s2[1:] and sb.dtype == torch.bfloat16
    valid2 = -(-shape.I // 128)
    assert not torch.isnan(sb[..., :valid2].float()).any()
    assert torch.isnan(sb[..., valid2:].float()).all()
    assert not torch.isnan(sa.float()).any()


def test_wide_expert_bank_shapes():
    a, sa, b, sb = syn.make_weights(dataclasses.replace(syn.DECODE_WIDE, E=1), seed=0)
    assert tuple(a.shape) == (1, 4096, 7168) and tuple(b.shape) == (1, 7168, 2048)
    assert tuple(sa.shape) == (1, 32, 56) and tuple(sb.shape) == (1, 56, 16)
    # 256 experts of these banks: about 11 GB of e4m3 weights
    assert 256 * (a[0].numel() + b[0].numel()) == 11_274_289_152


def test_weight_codes_are_the_finite_e4m3_codes_uniformly():
    a, _, b, _ = syn.make_weights(dataclasses.replace(syn.DECODE_SMALL, E=1), seed=3)
    codes = torch.cat([a.flatten(), b.flatten()]).to(torch.int64)
    counts = torch.bincount(codes, minlength=256)
    assert counts[0x7F] == 0 and counts[0xFF] == 0          # the two NaN codes never drawn
    finite = torch.cat([counts[:0x7F], counts[0x80:0xFF]])
    assert (finite > 0).all()                                # every finite code, both zeros and subnormals
    expect = codes.numel() / 254
    assert (finite.double() / expect - 1).abs().max() < 0.05   # ~12k draws a code: 5 % is > 5 sigma
    sign = (codes >> 7) & 1
    assert abs(sign.double().mean().item() - 0.5) < 0.01    # mixed sign
    subnormal = ((codes & 0x78) == 0) & ((codes & 0x07) != 0)
    assert abs(subnormal.double().mean().item() - 14 / 254) < 0.005


def test_block_scales_are_log_uniform_in_range():
    _, sa, _, sb = syn.make_weights(dataclasses.replace(syn.DECODE_SMALL, E=8), seed=5)
    v = torch.cat([sa.float().flatten(), sb.float()[..., :4].flatten()]).double()
    assert v.min() >= 2.0 ** -8 and v.max() <= 2.0 ** -2
    lg = torch.log2(v)
    # log2 uniform on [-8, -2]: mean -5, variance 36 / 12 = 3
    assert abs(lg.mean().item() + 5) < 0.15
    assert abs(lg.var().item() - 3) < 0.3
    # every value is a bf16 number (rounded, not truncated float32 bits)
    assert torch.equal(v.float().to(torch.bfloat16).double(), v)


def test_hidden_is_zero_mean_unit_normal_bf16():
    x = syn.make_hidden(512, 2048, seed=1)
    assert x.dtype == torch.bfloat16 and tuple(x.shape) == (512, 2048)
    f = x.double()
    assert abs(f.mean().item()) < 0.01
    assert abs(f.std().item() - 1) < 0.01
    # heavier-than-uniform tails, as a normal has: about 0.27 % beyond 3 sigma
    assert 0.0015 < (f.abs() > 3).double().mean().item() < 0.004


def _check_router_outputs(ids, w, T, E, k):
    assert ids.dtype == torch.int32 and w.dtype == torch.float32
    assert tuple(ids.shape) == (T, k) and tuple(w.shape) == (T, k)
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(r)) == k for r in ids.tolist())      # k distinct experts per token
    assert (w > 0).all()
    assert torch.allclose(w.sum(dim=1), torch.ones(T), atol=1e-6)


def test_softmax_routing():
    T, E, k = 2048, 128, 8
    ids, w = syn.make_routing(T, E, k, seed=0, kind="softmax")
    _check_router_outputs(ids, w, T, E, k)
    assert (w[:, :-1] >= w[:, 1:]).all()                     # top-k order
    # uniform logits: every expert gets about T*k/E slots
    cnt = torch.bincount(ids.flatten().long(), minlength=E).double()
    assert cnt.min() > 0.6 * T * k / E and cnt.max() < 1.4 * T * k / E


def test_hot_routing_skews_toward_sixteen_experts():
    T, E, k = 32, 256, 8
    ids, w = syn.make_routing(T, E, k, seed=0, kind="hot")
    _check_router_outputs(ids, w, T, E, k)
    big = syn.make_routing(4096, E, k, seed=0, kind="hot")[0]
    cnt = torch.bincount(big.flatten().long(), minlength=E)
    top16 = cnt.sort(descending=True).values[:16].sum().item()
    # +2 on 16 of 256 logits: those experts take far more than their 1/16 share
    assert top16 > 0.3 * big.numel()
    # the same 16 experts are hot at every batch size (a seeded set)
    hot_small = set(torch.bincount(ids.flatten().long(), minlength=E).sort(descending=True).indices[:4].tolist())
    hot_big = set(cnt.sort(descending=True).indices[:16].tolist())
    assert hot_small <= hot_big


def test_zipf_routing_follows_rank_power_law():
    T, E, k = 8192, 128, 8
    ids, w = syn.make_routing(T, E, k, seed=0, kind="zipf")
    _check_router_outputs(ids, w, T, E, k)
    cnt = torch.bincount(ids.flatten().long(), minlength=E).double().sort(descending=True).values
    # drawing k distinct experts flattens the head, but the order by rank
    # and a steep tail (p ~ rank^-1.1) remain
    assert cnt[0] > cnt[9] > cnt[49] > cnt[-1]
    assert cnt[0] / cnt[-1] > 20
    slope = (math.log(cnt[99].item()) - math.log(cnt[19].item())) / (math.log(100) - math.log(20))
    assert -1.4 < slope < -0.8


def test_inputs_are_deterministic_and_seed_sensitive():
    p0 = syn.make_problem(syn.TINY, T=4, seed=0)
    p0b = syn.make_problem(syn.TINY, T=4, seed=0)
    p1 = syn.make_problem(syn.TINY, T=4, seed=1)
    for key in p0:
        a, b = p0[key], p0b[key]
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), key
    assert not torch.equal(p0["w13"], p1["w13"])
    assert not torch.equal(p0["hidden"].float(), p1["hidden"].float())
    # one expert's banks do not depend on how many experts were drawn
    a2 = syn.make_weights(dataclasses.replace(syn.TINY, E=2), seed=0)
    a8 = syn.make_weights(syn.TINY, seed=0)
    assert torch.equal(a2[0], a8[0][:2]) and torch.equal(a2[2], a8[2][:2])
    assert torch.equal(a2[1].float(), a8[1][:2].float())
    # successive batch steps draw different activations and routing
    assert not torch.equal(syn.make_hidden(4, 256, 0, step=0).float(), syn.make_hidden(4, 256, 0, step=1).float())
