"""Host copies of a problem's inputs, in the oracle's argument order.

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the
smoke check and the benchmark's CPU-baseline legs use it.  It copies and
relabels inputs (torch tensors to NumPy arrays); it holds none of the
layer's arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_args(prob: dict, tokens=None):
    """Host copies of a problem's tensors in the oracle's argument order.

    With `tokens`, only those tokens and the experts they route to are copied
    (expert ids relabelled densely, which leaves the layer unchanged);
    returns (args, token_index_array)."""
    ids = prob["topk_ids"].cpu().numpy()
    T = ids.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    E = prob["w13"].shape[0]
    sub_ids = ids[tok]
    if tokens is None and E <= 16:
        experts = np.arange(E)
    else:
        experts = np.unique(sub_ids[(sub_ids >= 0) & (sub_ids < E)])
    remap = np.full(E, -1, dtype=np.int64)
    remap[experts] = np.arange(len(experts))
    new_ids = np.where((sub_ids >= 0) & (sub_ids < E), remap[np.clip(sub_ids, 0, E - 1)], sub_ids)
    new_ids = np.where(sub_ids >= E, 10 ** 6, new_ids).astype(np.int32)
    idx = torch.as_tensor(experts, dtype=torch.long, device=prob["w13"].device)
    if len(experts) == 0:
        idx = torch.zeros(1, dtype=torch.long, device=prob["w13"].device)
    args = [
        bits(prob["hidden"][torch.as_tensor(tok, device=prob["hidden"].device)]),
        new_ids,
        prob["topk_weights"].cpu().numpy()[tok],
        prob["w13"].index_select(0, idx).cpu().numpy(),
        bits(prob["w13_scale"].index_select(0, idx)),
        prob["w2"].index_select(0, idx).cpu().numpy(),
        bits(prob["w2_scale"].index_select(0, idx)),
    ]
    return args, tok


def oracle_biases(prob: dict, tokens=None) -> dict:
    """The optional MLP biases of a problem (keys w13_bias, w2_bias) as host
    arrays, with the experts relabelled exactly as oracle_args does; an empty
    dict when the problem has none."""
    ids = prob["topk_ids"].cpu().numpy()
    tok = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    E = prob["w13"].shape[0]
    sub_ids = ids[tok]
    if tokens is None and E <= 16:
        experts = np.arange(E)
    else:
        experts = np.unique(sub_ids[(sub_ids >= 0) & (sub_ids < E)])
    if len(experts) == 0:
        experts = np.zeros(1, dtype=np.int64)
    out = {}
    for name in ("w13_bias", "w2_bias"):
        if prob.get(name) is not None:
            out[name] = prob[name].cpu().numpy()[experts]
    return out
