"""Shared checks for the GPU-vs-oracle parity tests.

Index rule (the tolerance for sampled indices): a GPU index may differ from the oracle's
only when the oracle's target T = t*Z lies within 1e-4*Z of a boundary of the oracle's
interval [W_{i-1}, W_i); such mismatches must occur at a rate below 0.1% of points.
Every other index is bit-exact.

The rate is a property of the arithmetic, so it is asserted strictly on pooled samples of
100k+ points (test_boundary_mismatch_rate_pooled).  A single call of a few thousand
points only has to be consistent with it: at most the mean plus three standard
deviations of a Poisson count at that rate (8 of 2816 points, for example).
"""
import math

import numpy as np
import torch

import oracle

BOUNDARY_REL = 1e-4
MISMATCH_FRAC = 1e-3
EST_TOL = 1e-2          # estimator max-abs error, bf16 V with fp32 accumulation
DENSE_REL_L2 = 2e-3


def bf16_cpu(x):
    return x.detach().cpu()


def allowed_mismatches(n_pts: int) -> int:
    """Largest mismatch count of one call consistent with a rate of MISMATCH_FRAC."""
    lam = MISMATCH_FRAC * n_pts
    return int(lam + 3.0 * math.sqrt(lam) + 1.0)


def count_mismatches(gpu_idx, orc_idx, q, k, sl, S, mode, seed, pairs=None, W_cache=None):
    """(n_mismatch, n_points): indices that differ from the oracle's.  Raises on a
    mismatch away from a boundary."""
    g = np.asarray(gpu_idx)
    o = np.asarray(orc_idx)
    if pairs is None:
        pairs = [(b, h) for b in range(o.shape[0]) for h in range(o.shape[1])]
    n_pts = 0
    bad = []
    for b, h in pairs:
        n_pts += S
        diff = np.nonzero(g[b, h] != o[b, h])[0]
        if len(diff) == 0:
            continue
        if W_cache is not None and (b, h) in W_cache:
            W = W_cache[(b, h)]
        else:
            W, _ = oracle.cdf(q, k, sl, b, h)
            if W_cache is not None:
                W_cache[(b, h)] = W
        Z = W[-1]
        t = oracle.points(mode, S, seed, b, h)
        for s in diff:
            i = int(o[b, h, s])
            T = t[s] * Z
            lo = W[i - 1] if i > 0 else 0.0
            dist = min(abs(T - lo), abs(W[i] - T))
            assert dist <= BOUNDARY_REL * Z, (
                f"(b={b},h={h},s={s}) gpu {g[b, h, s]} vs oracle {i}: point {dist / Z:.3e} Z from a boundary")
            bad.append((b, h, s))
    return len(bad), n_pts


def check_indices(gpu_idx, orc_idx, q, k, sl, S, mode, seed, pairs=None):
    """Returns (n_mismatch, n_points).  Raises on a mismatch away from a boundary or on
    more boundary mismatches than a rate of MISMATCH_FRAC explains."""
    nm, n_pts = count_mismatches(gpu_idx, orc_idx, q, k, sl, S, mode, seed, pairs)
    assert nm <= allowed_mismatches(n_pts), f"{nm} boundary mismatches of {n_pts} points"
    return nm, n_pts


def check_estimator(gpu_out, gpu_idx, v, sl, orc_out, pairs=None):
    """The GPU output against the oracle's gather-sum of the GPU's own indices (pure
    estimator arithmetic), and against the oracle's output."""
    go = np.asarray(gpu_out, dtype=np.float64)
    gi = np.asarray(gpu_idx)
    ref = oracle.gather(v, sl, gi)
    if pairs is not None:
        sel = tuple(np.array(pairs).T)
        go, ref, oo = go[sel], ref[sel], np.asarray(orc_out)[sel]
    else:
        oo = np.asarray(orc_out)
    e1 = np.abs(go - ref).max()
    assert e1 <= EST_TOL, f"estimator arithmetic max-abs {e1}"
    return e1, np.abs(go - oo).max()


def check_dense(gpu_out, orc_out, pairs=None):
    go = np.asarray(gpu_out, dtype=np.float64)
    oo = np.asarray(orc_out)
    if pairs is not None:
        sel = tuple(np.array(pairs).T)
        go, oo = go[sel], oo[sel]
    rel = np.linalg.norm(go - oo) / max(np.linalg.norm(oo), 1e-300)
    assert rel <= DENSE_REL_L2, f"dense relative L2 {rel}"
    return rel
