"""Seeded synthetic inputs for the block-FP8 MoE layer forward.

This module only draws inputs: e4m3 weight bytes, bf16 block scales, bf16
activations and router outputs (top-k ids and weights).  It holds none of
the layer's own arithmetic (no e4m3 decoding, no dequantisation, no GEMM,
no combine), so both the CUDA path and the float64 oracle can be fed from
it without sharing any computation.

Value distributions follow the workloads the pages test on:

* weights: uniform over the 254 finite e4m3 codes (0x7F and 0xFF, the two
  NaN codes, excluded; subnormals and both zeros included) -- "mixed-sign,
  full-range e4m3 weights" (FreeToken PR #662, commit "add float64 parity
  reference and an avx512f fp8 tier");
* block scales: one bf16 per 128x128 block, log-uniform in [2^-8, 2^-2],
  rounded to bf16 by round-to-nearest-even;
* activations: bf16 N(0, 1) ("zero-mean activations", same commit);
* routing: N(0, 1) router logits, softmax, top-k, renormalised fp32 weights
  (optionally +bias on a seeded set of hot experts), or k distinct experts
  drawn without replacement with p ~ rank^-s (Zipf) and weights from a
  renormalised softmax over the chosen k.

Every tensor is drawn from its own torch.Generator whose seed is a
splitmix64 hash of (seed, tensor id, expert), so one expert's bytes can be
regenerated without drawing the others.  bf16 tensors are returned as
torch.bfloat16; e4m3 codes as torch.uint8.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

_MASK64 = (1 << 64) - 1

# tensor ids for the per-tensor generator seeds
(_TID_W13, _TID_W13S, _TID_W2, _TID_W2S, _TID_X, _TID_LOGITS, _TID_HOT, _TID_ZIPF, _TID_B13,
 _TID_B2) = range(1, 11)


def splitmix64(x: int) -> int:
    """One step of the splitmix64 output function (Steele, Lea, Flood 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _gen(seed: int, tid: int, idx: int, device) -> torch.Generator:
    s = splitmix64(splitmix64(splitmix64(seed) ^ tid) ^ idx) & ((1 << 63) - 1)
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def finite_e4m3_codes(shape, gen: torch.Generator, device) -> torch.Tensor:
    """Bytes drawn uniformly from the 254 finite e4m3 codes (0x7F/0xFF excluded)."""
    idx = torch.randint(0, 254, shape, generator=gen, device=device, dtype=torch.int16)
    # indices 0..126 -> codes 0x00..0x7E, 127..253 -> codes 0x80..0xFE
    return (idx + (idx >= 127).to(torch.int16)).to(torch.uint8)


def log_uniform_bf16(shape, gen: torch.Generator, device, lo: float = -8.0, hi: float = -2.0) -> torch.Tensor:
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float64)
    return torch.exp2(lo + (hi - lo) * u).to(torch.float32).to(torch.bfloat16)


def bf16_normal(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclasses.dataclass
class MoeShape:
    E: int
    H: int
    I: int
    k: int
    w13_scale_stride: Optional[int] = None   # row stride of w13 scales (>= H/128)
    w2_scale_stride: Optional[int] = None    # row stride of w2 scales (>= I/128)
    w13_scale_estride: Optional[int] = None  # expert stride of w13 scales (>= (2I/128)*stride)
    w2_scale_estride: Optional[int] = None   # expert stride of w2 scales (>= (H/128)*stride)

    def strides(self):
        s13 = self.w13_scale_stride or -(-self.H // 128)
        s2 = self.w2_scale_stride or -(-self.I // 128)
        e13 = self.w13_scale_estride or -(-2 * self.I // 128) * s13
        e2 = self.w2_scale_estride or -(-self.H // 128) * s2
        return s13, s2, e13, e2


# The five workloads (tiny oracle case, decode small experts, padded-scale
# skewed case, decode wide experts, prefill grouped GEMM).
TINY = MoeShape(E=8, H=256, I=128, k=2)
DECODE_SMALL = MoeShape(E=128, H=2048, I=512, k=8, w2_scale_stride=8)
PADDED_SKEWED = MoeShape(E=256, H=2560, I=640, k=8, w2_scale_stride=6)
DECODE_WIDE = MoeShape(E=256, H=7168, I=2048, k=8)
PREFILL = MoeShape(E=128, H=2048, I=512, k=8, w2_scale_stride=8)


def _scale_bank(E, rows, cols, stride, estride, gen_seed, tid, device, pad_value=float("nan")):
    """[E, rows, stride] bf16 view over an [E*estride] buffer; valid block
    scales in [..., :cols], padding filled with `pad_value` (NaN by default,
    so a kernel that reads padding produces NaN)."""
    flat = torch.full((E * estride,), pad_value, dtype=torch.bfloat16, device=device)
    for e in range(E):
        g = _gen(gen_seed, tid, e, device)
        vals = log_uniform_bf16((rows, cols), g, device)
        blk = flat[e * estride: e * estride + rows * stride].view(rows, stride)
        blk[:, :cols] = vals
    return torch.as_strided(flat, (E, rows, stride), (estride, stride, 1))


def make_weights(shape: MoeShape, seed: int = 0, device="cpu", experts_per_draw: int = 1):
    """Weight banks: w13 e4m3 [E, 2I, H] (rows [0,I) gate, [I,2I) up),
    w13_scale bf16 [E, ceil(2I/128), stride13], w2 e4m3 [E, H, I],
    w2_scale bf16 [E, ceil(H/128), stride2]."""
    E, H, I = shape.E, shape.H, shape.I
    s13, s2, e13, e2 = shape.strides()
    w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I), dtype=torch.uint8, device=device)
    for e in range(E):
        w13[e] = finite_e4m3_codes((2 * I, H), _gen(seed, _TID_W13, e, device), device)
        w2[e] = finite_e4m3_codes((H, I), _gen(seed, _TID_W2, e, device), device)
    w13_scale = _scale_bank(E, -(-2 * I // 128), -(-H // 128), s13, e13, seed, _TID_W13S, device)
    w2_scale = _scale_bank(E, -(-H // 128), -(-I // 128), s2, e2, seed, _TID_W2S, device)
    return w13, w13_scale, w2, w2_scale


def make_biases(shape: MoeShape, seed: int = 0, device="cpu", std13: float = 1.0, std2: float = 1.0):
    """MLP biases, fp32 N(0, std^2): w13_bias [E, 2I] (gate biases in
    [0, I), up biases in [I, 2I)) and w2_bias [E, H]."""
    E, H, I = shape.E, shape.H, shape.I
    b13 = torch.empty((E, 2 * I), dtype=torch.float32, device=device)
    b2 = torch.empty((E, H), dtype=torch.float32, device=device)
    for e in range(E):
        b13[e] = torch.randn((2 * I,), generator=_gen(seed, _TID_B13, e, device), device=device) * std13
        b2[e] = torch.randn((H,), generator=_gen(seed, _TID_B2, e, device), device=device) * std2
    return b13, b2


def make_hidden(T: int, H: int, seed: int = 0, device="cpu", step: int = 0) -> torch.Tensor:
    return bf16_normal((T, H), _gen(seed, _TID_X, step, device), device)


def make_routing(T: int, E: int, k: int, seed: int = 0, device="cpu", kind: str = "softmax",
                 hot: int = 16, hot_bias: float = 2.0, zipf_s: float = 1.1, step: int = 0):
    """Router outputs: (topk_ids int32 [T,k], topk_weights fp32 [T,k]).

    kind = "softmax": N(0,1) logits -> softmax -> top-k -> renormalise.
    kind = "hot":     as softmax, with +hot_bias on `hot` experts picked by a
                      seeded permutation (some experts get many tokens, others none).
    kind = "zipf":    k distinct experts per token without replacement,
                      p ~ rank^-zipf_s (rank -> expert by a seeded permutation);
                      weights = renormalised softmax of N(0,1) logits over the k.
    """
    g = _gen(seed, _TID_LOGITS, step, device)
    if kind in ("softmax", "hot"):
        logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
        if kind == "hot":
            gp = _gen(seed, _TID_HOT, 0, "cpu")
            hot_ids = torch.randperm(E, generator=gp)[:hot].to(device)
            logits[:, hot_ids] += hot_bias
        probs = torch.softmax(logits, dim=-1)
        w, ids = torch.topk(probs, k, dim=-1)
        w = w / w.sum(dim=-1, keepdim=True)
        return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()
    if kind == "zipf":
        gp = _gen(seed, _TID_ZIPF, 0, "cpu")
        rank_to_expert = torch.randperm(E, generator=gp).to(device)
        p = torch.arange(1, E + 1, device=device, dtype=torch.float64) ** (-zipf_s)
        ranks = torch.multinomial(p.expand(T, E).float(), k, replacement=False, generator=g)
        ids = rank_to_expert[ranks]
        logits = torch.randn((T, k), generator=g, device=device, dtype=torch.float32)
        w = torch.softmax(logits, dim=-1)
        w = w / w.sum(dim=-1, keepdim=True)
        return ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()
    raise ValueError(f"unknown routing kind {kind!r}")


def make_problem(shape: MoeShape, T: int, seed: int = 0, device="cpu", routing: str = "softmax", step: int = 0):
    """All inputs of one forward call as a dict of tensors."""
    w13, w13_scale, w2, w2_scale = make_weights(shape, seed, device)
    hidden = make_hidden(T, shape.H, seed, device, step)
    ids, w = make_routing(T, shape.E, shape.k, seed, device, routing, step=step)
    return dict(hidden=hidden, topk_ids=ids, topk_weights=w, w13=w13, w13_scale=w13_scale,
                w2=w2, w2_scale=w2_scale)
