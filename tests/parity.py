"""Error metric and oracle drivers shared by the GPU parity tests.

Error metric (max relative error, normalised by the reference's largest
magnitude, in fp64):

    err(X) = max_i max(0, |X_i - R_i| - rho(R_i)) / max_i |R_i|

where rho(x) = u * |x| is the rounding bound of storing x in X's own dtype
(u = 2^-8 for bfloat16, 2^-24 for float32).  Storing an exact result in bf16
moves it by up to 2^-8 relative, more than the 2e-3 budget, so the budget can
only bound the computation; ``plain`` (without rho) is reported beside it.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}
UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}


def err(x: torch.Tensor, ref: np.ndarray) -> tuple[float, float]:
    """(err, plain) of a device or host tensor against an fp64 reference."""
    xd = x.detach().to("cpu").double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert xd.shape == ref.shape, (xd.shape, ref.shape)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if scale == 0.0:
        d = float(np.max(np.abs(xd))) if xd.size else 0.0
        return d, d
    diff = np.abs(xd - ref)
    rho = UNIT_ROUNDOFF[x.dtype] * np.abs(ref)
    return float(np.max(np.maximum(diff - rho, 0.0)) / scale), float(np.max(diff) / scale)


# (test id, tensor name, err, plain, tol) of every comparison of the session;
# conftest prints the workload rows at the end of the run and can write them all
# to a JSON file (KDA_PARITY_LOG)
RECORDS: list[tuple[str, str, float, float, float]] = []


def assert_close(name, x, ref, tol):
    e, plain = err(x, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.append((test, name, e, plain, tol))
    assert e <= tol, "%s: err %.3e > %.1e (plain %.3e)" % (name, e, tol, plain)
    return e, plain


def oracle_prefill_windowed(inp, t0, t1, S0, cols=None, heads=None, window=16384):
    """Oracle over tokens [t0, t1) of a single dense sequence held on the
    device, streamed to the host in windows; optionally restricted to a set of
    state columns (exact: columns never mix) and heads.  Returns
    (o [t1-t0, H', C'], S [H', dk, C']) as fp64 arrays."""
    hs = slice(None) if heads is None else heads
    cs = slice(None) if cols is None else cols
    S = None if S0 is None else np.asarray(S0, dtype=np.float64)
    outs = []
    for a in range(t0, t1, window):
        b = min(t1, a + window)
        q = inp["q"][a:b, hs]
        k = inp["k"][a:b, hs]
        v = inp["v"][a:b, hs][..., cs]
        g = inp["g"][a:b, hs]
        beta = inp["beta"][a:b, hs]
        o, S_T, _ = oracle.prefill(q, k, v, g, beta, None if S is None else S[None],
                                   [0, b - a])
        S = S_T[0]
        outs.append(o)
    return np.concatenate(outs, axis=0), S
