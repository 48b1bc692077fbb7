"""Shared test helpers: the per-token tolerance check, and the host copies
of inputs for the oracle (re-exported from oracle.host_inputs).  No
arithmetic of the layer lives here."""
from __future__ import annotations

import numpy as np

from oracle.host_inputs import bits, oracle_args, oracle_biases  # noqa: F401

# max_i |gpu[t,i] - oracle[t,i]| <= TOL * max_i |oracle[t,i]| for every token t
# (FreeToken PR #662, commit adding the float64 parity reference: 2e-2)
TOL = 2e-2


def check_per_token(got: np.ndarray, ref: np.ndarray, tol: float = TOL) -> float:
    """Assert the per-token tolerance; return the worst ratio err/(tol*max)."""
    err = np.max(np.abs(got - ref), axis=1)
    scale = np.max(np.abs(ref), axis=1)
    assert np.all(np.isfinite(got)), "non-finite output"
    bad = err > tol * scale
    assert not np.any(bad), f"tokens {np.nonzero(bad)[0][:8]} err {err[bad][:4]} scale {scale[bad][:4]}"
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(scale > 0, err / scale, 0.0)
    return float(np.max(r)) if r.size else 0.0
