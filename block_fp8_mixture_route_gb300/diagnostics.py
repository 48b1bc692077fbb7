"""Diagnostics over outputs of the library's forward (not part of its path).

decode_ulp_verify compares the decode path's W8A8 mode with its W8A16 mode
on the same inputs, in steps of the e4m3 grid at the W8A16 value's
magnitude, the unit in which the fp8-moe-gather page's Gaudi path reports
its FP8 verification ("FP8-ULP").  The e4m3 step at magnitude v (2^e <= v <
2^(e+1)) is 2^(e-3): three mantissa bits.  Magnitudes below e4m3's smallest
normal, 2^-6, count with the step there.
"""
from __future__ import annotations

import torch

from . import api


def decode_ulp_verify(prob: dict, stream=None) -> dict:
    """Run the decode path in both activation formats on `prob` (the
    synthetic generator's dict of device tensors) and return the distance
    statistics: max and mean in e4m3 steps, the fraction of outputs more
    than 2 steps apart, and the largest per-token distance relative to the
    token's largest W8A16 output.  Outputs near zero (cancellation) sit
    many steps apart at their own tiny magnitude, so the step counts are a
    diagnostic, not a bound."""
    a = api.forward_problem(prob, stream=stream, force_path="decode").float()
    b = api.forward_problem(prob, stream=stream, force_path="decode", decode_act="e4m3").float()
    mag = a.abs().clamp_min(2.0 ** -6)
    step = torch.exp2(torch.floor(torch.log2(mag)) - 3)
    d = (a - b).abs() / step
    # the same distance relative to each token's largest W8A16 output (the
    # scale of the layer's parity rule)
    row = ((a - b).abs().amax(dim=1) / a.abs().amax(dim=1).clamp_min(torch.finfo(torch.float32).tiny)).max()
    return {"max_ulp": float(d.max()), "mean_ulp": float(d.mean()), "frac_over_2": float((d > 2).float().mean()),
            "max_rel_row": float(row)}
