"""Per-head relative Frobenius error with a floor for vanishing references.

err(X, X*) = ||X - X*||_F / ||X*||_F over the trailing `inner` axes, maxed
over all leading (head) axes.  Where ||X*||_F < 1e-30 (a transition product
that has underflowed below the fp32 range, e.g. a long gated segment) the
reference carries no relative scale: the check then asks ||X||_F <= 1e-28
and scores the head 0 if it holds, +inf otherwise.
"""
from __future__ import annotations

import numpy as np

TOL_BF16 = 5e-3   # bf16 inputs, fp32 state
TOL_F32 = 1e-5    # fp32 inputs
FLOOR_REF = 1e-30
FLOOR_OUT = 1e-28


def _np(x):
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def per_head_rel_err(x, ref, inner: int = 2) -> np.ndarray:
    x, ref = _np(x), _np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    lead = x.shape[:x.ndim - inner]
    xf = x.reshape(lead + (-1,))
    rf = ref.reshape(lead + (-1,))
    dn = np.sqrt(((xf - rf) ** 2).sum(-1))
    rn = np.sqrt((rf ** 2).sum(-1))
    xn = np.sqrt((xf ** 2).sum(-1))
    out = np.where(rn >= FLOOR_REF, dn / np.maximum(rn, FLOOR_REF),
                   np.where(xn <= FLOOR_OUT, 0.0, np.inf))
    if not np.all(np.isfinite(x)):
        out = np.where(np.isfinite(xf).all(-1), out, np.inf)
    return out


def max_rel_err(x, ref, inner: int = 2) -> float:
    e = per_head_rel_err(x, ref, inner)
    return float(e.max()) if e.size else 0.0
