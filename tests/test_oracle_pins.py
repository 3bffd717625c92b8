"""Pins for the fp64 oracle, checked against what the pages and the mathematics fix
rather than against the oracle's own formulas.

"Stochastic Sparse Attention for Memory-Bound Inference" (abstract) fixes three
properties of SANTA: the indices are drawn from the post-softmax distribution, the
estimator of the post-softmax value aggregation is unbiased, and the stratified and
systematic variants reduce variance.  The pages print no worked example, so the pins
are closed forms, exact expectations, brute-force enumeration, library routines
(numpy's Philox, torch's softmax, numpy's searchsorted) and invariants.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def exact_attention(q, k, v, seq_lens, scale=None):
    """Softmax attention in fp64 from torch library routines (an independent
    restatement of the dense definition)."""
    B, H_q, d = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    if scale is None:
        scale = float(np.float32(1.0 / math.sqrt(d)))
    out = torch.zeros(B, H_q, d, dtype=torch.float64)
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        for h in range(H_q):
            kk = k[b, h // G, :n].double()
            vv = v[b, h // G, :n].double()
            p = torch.softmax(scale * (kk @ q[b, h].double()), dim=0)
            out[b, h] = p @ vv
    return out


def probs(q, k, b, h, n, scale=None):
    d = q.shape[-1]
    G = q.shape[1] // k.shape[1]
    if scale is None:
        scale = float(np.float32(1.0 / math.sqrt(d)))
    return torch.softmax(scale * (k[b, h // G, :n].double() @ q[b, h].double()), 0).numpy()


def rand_case(B, H_q, H_kv, d, n, seed, qstd=1.0):
    g = torch.Generator().manual_seed(seed)
    q = bf16(qstd * torch.randn(B, H_q, d, generator=g))
    k = bf16(torch.randn(B, H_kv, n, d, generator=g))
    v = bf16(torch.randn(B, H_kv, n, d, generator=g))
    return q, k, v


# ----------------------------------------------------------------------------- Philox

def test_philox_matches_numpy_philox4x64():
    """Philox4x64-10 (Salmon et al., SC'11) against numpy's independent implementation:
    numpy's random_raw with counter c returns the block of counter c + 1."""
    rs = np.random.default_rng(123)
    for _ in range(200):
        key = rs.integers(0, 2**63, size=2, dtype=np.uint64) * np.uint64(2) + rs.integers(0, 2, size=2, dtype=np.uint64)
        ctr = rs.integers(0, 2**62, size=4, dtype=np.uint64)
        bg = np.random.Philox(key=key, counter=ctr)
        want = bg.random_raw(4)
        got = oracle.philox4x64_10([ctr[0] + np.uint64(1), ctr[1], ctr[2], ctr[3]], key)
        assert np.array_equal(want, got)
    # small counters/keys, as the sampler uses them
    for seed in (0, 1, 2**40 + 5):
        for b in range(3):
            bg = np.random.Philox(key=np.array([seed, 0], dtype=np.uint64),
                                  counter=np.array([0, b, 7, 2], dtype=np.uint64))
            assert np.array_equal(bg.random_raw(4), oracle.philox4x64_10([1, b, 7, 2], [seed, 0]))


# ----------------------------------------------------------------------------- points

def test_systematic_points_structure_and_uniformity():
    """Systematic sampling: one uniform u per (b, h); t_s = (u + s)/S.  The points are
    equally spaced by 1/S, lie in [0, 1), and u = S*t_0 is uniform (KS test)."""
    from scipy import stats
    us = []
    for seed in range(40):
        for b in range(5):
            for h in range(5):
                S = 64
                t = oracle.points("systematic", S, seed, b, h)
                assert np.all(np.diff(t) > 0) and t[0] >= 0 and t[-1] < 1
                assert np.allclose(np.diff(t), 1.0 / S, rtol=0, atol=1e-15)
                u = t[0] * S
                assert np.allclose(S * t - np.arange(S), u, rtol=0, atol=1e-12)
                us.append(u)
    assert stats.kstest(us, "uniform").pvalue > 1e-4


def test_stratified_points_structure_and_uniformity():
    """Stratified sampling: point s is uniform on its stratum [s/S, (s+1)/S), the strata
    draws are independent (KS on offsets, lag-1 correlation near zero)."""
    from scipy import stats
    offs = []
    for seed in range(20):
        for h in range(10):
            S = 100
            t = oracle.points("stratified", S, seed, 0, h)
            s = np.arange(S)
            assert np.all(t >= s / S) and np.all(t < (s + 1) / S)
            offs.append(S * t - s)
    offs = np.concatenate(offs)
    assert stats.kstest(offs, "uniform").pvalue > 1e-4
    r = np.corrcoef(offs[:-1], offs[1:])[0, 1]
    assert abs(r) < 4 / math.sqrt(len(offs))


def test_points_depend_on_seed_batch_and_head():
    a = oracle.points("systematic", 8, 0, 0, 0)
    assert not np.array_equal(a, oracle.points("systematic", 8, 1, 0, 0))
    assert not np.array_equal(a, oracle.points("systematic", 8, 0, 1, 0))
    assert not np.array_equal(a, oracle.points("systematic", 8, 0, 0, 1))
    assert np.array_equal(a, oracle.points("systematic", 8, 0, 0, 0))


# ----------------------------------------------------------------------------- dense

def test_dense_matches_torch_softmax_attention():
    q, k, v = rand_case(2, 4, 2, 16, 37, seed=3, qstd=2.0)
    sl = torch.tensor([37, 20], dtype=torch.int32)
    out, _ = oracle.decode(q, k, v, sl, 0, "dense")
    assert np.allclose(out, exact_attention(q, k, v, sl).numpy(), rtol=0, atol=1e-13)


def test_cdf_matches_library_cumsum_and_search_rule():
    """W is the running sum of exp(s - m) (torch fp64), and the sampled index of a point
    is numpy's searchsorted(W, t*Z, side='right') -- the half-open rule
    i = min{j : W_j > T}."""
    q, k, v = rand_case(1, 2, 1, 32, 300, seed=5, qstd=3.0)
    sl = torch.tensor([300], dtype=torch.int32)
    scale = float(np.float32(1 / math.sqrt(32)))
    for h in range(2):
        W, m = oracle.cdf(q, k, sl, 0, h)
        s = scale * (k[0, 0].double() @ q[0, h].double())
        assert abs(m - float(s.max())) < 1e-13
        want = torch.cumsum(torch.exp(s - s.max()), 0).numpy()
        assert np.allclose(W, want, rtol=1e-14, atol=0)
    for mode in ("systematic", "stratified", "iid"):
        _, idx, Z = oracle.decode(q, k, v, sl, 48, mode, seed=11, want_Z=True)
        for h in range(2):
            W, _ = oracle.cdf(q, k, sl, 0, h)
            t = oracle.points(mode, 48, 11, 0, h)
            want = np.minimum(np.searchsorted(W, t * Z[0, h], side="right"), 299)
            assert np.array_equal(idx[0, h], want)


# ----------------------------------------------------------------------------- exact expectation

def _systematic_expectation(q, k, v, sl, S):
    """E_u[o_hat(u)] for systematic sampling: o_hat is piecewise constant in u with
    breakpoints frac(S*C_j); sum the oracle's o_hat at each piece's midpoint weighted
    by the piece's length."""
    B, H_q, d = q.shape
    W, _ = oracle.cdf(q, k, sl, 0, 0)
    C = W / W[-1]
    br = np.unique(np.concatenate([[0.0, 1.0], np.mod(S * C, 1.0)]))
    br = br[(br >= 0) & (br <= 1)]
    E = np.zeros(d)
    for lo, hi in zip(br[:-1], br[1:]):
        if hi - lo <= 0:
            continue
        u = 0.5 * (lo + hi)
        t = ((u + np.arange(S)) / S).reshape(1, 1, S)
        out, _ = oracle.decode(q, k, v, sl, S, "systematic", t=t)
        E += (hi - lo) * out[0, 0]
    return E


@pytest.mark.parametrize("n,S,qstd,seed", [(8, 4, 2.0, 1), (50, 7, 3.0, 2), (256, 64, 3.0, 3),
                                           (200, 16, 0.5, 4), (31, 64, 4.0, 5)])
def test_systematic_exact_expectation_equals_attention(n, S, qstd, seed):
    """Unbiasedness (abstract: "an unbiased estimator of the post-softmax value
    aggregation"): the exact expectation over u equals softmax attention to 1e-12."""
    q, k, v = rand_case(1, 1, 1, 16, n, seed, qstd)
    sl = torch.tensor([n], dtype=torch.int32)
    E = _systematic_expectation(q, k, v, sl, S)
    assert np.max(np.abs(E - exact_attention(q, k, v, sl).numpy()[0, 0])) < 1e-12


@pytest.mark.parametrize("n,S,seed", [(8, 2, 1), (8, 4, 2), (60, 12, 3), (256, 64, 4)])
def test_stratified_exact_expectation_equals_attention(n, S, seed):
    """Stratified: E = (1/S) sum_s int_0^1 v_{I((s+u)/S)} du, integrated piecewise
    (breakpoints S*C_j - s) with the oracle's search at each piece's midpoint."""
    q, k, v = rand_case(1, 1, 1, 16, n, seed, 3.0)
    sl = torch.tensor([n], dtype=torch.int32)
    W, _ = oracle.cdf(q, k, sl, 0, 0)
    C = W / W[-1]
    pieces = []
    for s in range(S):
        u = S * C - s
        br = np.unique(np.concatenate([[0.0, 1.0], u[(u > 0) & (u < 1)]]))
        pieces.append([(lo, hi) for lo, hi in zip(br[:-1], br[1:]) if hi > lo])
    K = max(len(p) for p in pieces)
    vv = v[0, 0].double().numpy()
    E = np.zeros(16)
    for kk in range(K):
        t = np.zeros(S)
        wts = np.zeros(S)
        for s in range(S):
            if kk < len(pieces[s]):
                lo, hi = pieces[s][kk]
                t[s] = (s + 0.5 * (lo + hi)) / S
                wts[s] = hi - lo
            else:
                t[s] = (s + 0.5) / S
        # keep the points sorted as the sampler does (each stays in its stratum)
        _, idx = oracle.decode(q, k, v, sl, S, "stratified", t=t.reshape(1, 1, S))
        E += (wts[:, None] * vv[idx[0, 0]]).sum(0) / S
    assert np.max(np.abs(E - exact_attention(q, k, v, sl).numpy()[0, 0])) < 1e-12


# ----------------------------------------------------------------------------- degenerate / special

@pytest.mark.parametrize("mode", ["systematic", "stratified"])
def test_zero_query_with_S_equal_n_gives_mean_of_V(mode):
    """q = 0: every w_j = 1 exactly, W_j = j + 1, Z = n.  With S = n, T_s = u + s (or
    s + u_s), so i_s = s for every draw and o_hat = mean(V) exactly."""
    n = 64
    _, k, v = rand_case(2, 4, 2, 16, n, 9)
    q = bf16(torch.zeros(2, 4, 16))
    sl = torch.tensor([n, n], dtype=torch.int32)
    for seed in range(5):
        out, idx = oracle.decode(q, k, v, sl, n, mode, seed=seed)
        assert np.array_equal(idx, np.broadcast_to(np.arange(n, dtype=np.int32), idx.shape))
        for h in range(4):
            want = v[0, h // 2].double().mean(0).numpy()
            assert np.max(np.abs(out[0, h] - want)) < 1e-14


def test_near_uniform_query_recovers_mean_of_V():
    n = 128
    _, k, v = rand_case(1, 1, 1, 16, n, 4)
    q = bf16(1e-3 * torch.randn(1, 1, 16, generator=torch.Generator().manual_seed(1)))
    sl = torch.tensor([n], dtype=torch.int32)
    out, _ = oracle.decode(q, k, v, sl, n, "systematic", seed=3)
    assert np.max(np.abs(out[0, 0] - v[0, 0].double().mean(0).numpy())) < 5e-3


def test_tie_break_point_on_boundary_goes_to_next_key():
    """Golden case (tests/golden/tie_break.json): q = 0 makes W_j = j + 1 exactly; a
    point with T exactly on W_j selects key j + 1 (half-open intervals)."""
    with open(os.path.join(HERE, "golden", "tie_break.json")) as f:
        g = json.load(f)
    n, S = g["n"], g["S"]
    _, k, v = rand_case(1, 1, 1, 8, n, 0)
    q = bf16(torch.zeros(1, 1, 8))
    sl = torch.tensor([n], dtype=torch.int32)
    t = np.array(g["t"], dtype=np.float64).reshape(1, 1, S)
    _, idx = oracle.decode(q, k, v, sl, S, "systematic", t=t)
    assert idx[0, 0].tolist() == g["idx"]


def test_single_key_and_one_hot_and_single_sample():
    q, k, v = rand_case(1, 1, 1, 16, 40, 21, 1.0)
    # n = 1: every index is 0 and o_hat = v_0
    sl1 = torch.tensor([1], dtype=torch.int32)
    for mode in ("systematic", "stratified", "iid"):
        out, idx = oracle.decode(q, k, v, sl1, 8, mode, seed=2)
        assert np.all(idx == 0)
        assert np.array_equal(out[0, 0], v[0, 0, 0].double().numpy())
    # one-hot: key 17 scores ~+50 above the rest -> every index is 17
    k2 = k.clone()
    k2[0, 0, 17] = bf16(q[0, 0].float() * (60.0 * 4 / q[0, 0].float().norm() ** 2))
    sl = torch.tensor([40], dtype=torch.int32)
    for mode in ("systematic", "stratified", "iid"):
        out, idx = oracle.decode(q, k2, v, sl, 16, mode, seed=5)
        assert np.all(idx == 17)
    # S = 1: o_hat is a single V row
    out, idx = oracle.decode(q, k, v, sl, 1, "systematic", seed=7)
    assert np.array_equal(out[0, 0], v[0, 0, idx[0, 0, 0]].double().numpy())


def test_ragged_lengths_and_empty_sequence():
    q, k, v = rand_case(3, 2, 1, 16, 50, 8, 3.0)
    sl = torch.tensor([50, 13, 0], dtype=torch.int32)
    out, idx = oracle.decode(q, k, v, sl, 32, "systematic", seed=1)
    assert idx[1].max() < 13 and idx[1].min() >= 0
    assert np.all(idx[2] == -1) and np.all(out[2] == 0)
    dense, _ = oracle.decode(q, k, v, sl, 0, "dense")
    assert np.allclose(dense, exact_attention(q, k, v, sl).numpy(), atol=1e-13, rtol=0)
    assert np.all(dense[2] == 0)
    with pytest.raises(ValueError):
        oracle.decode(q, k, v, torch.tensor([51, 1, 1], dtype=torch.int32), 4, "systematic")


def test_gather_agrees_with_decode_and_rejects_bad_index():
    q, k, v = rand_case(2, 4, 2, 16, 70, 12, 3.0)
    sl = torch.tensor([70, 33], dtype=torch.int32)
    out, idx = oracle.decode(q, k, v, sl, 20, "stratified", seed=4)
    assert np.array_equal(oracle.gather(v, sl, idx), out)
    bad = idx.copy()
    bad[1, 0, 0] = 33
    with pytest.raises(ValueError):
        oracle.gather(v, sl, bad)


# ----------------------------------------------------------------------------- brute force, n = 8

def _n8_case():
    g = torch.Generator().manual_seed(77)
    q = bf16(2.0 * torch.randn(1, 1, 4, generator=g))
    k = bf16(torch.randn(1, 1, 8, 4, generator=g))
    v = bf16(torch.randn(1, 1, 8, 4, generator=g))
    return q, k, v


def _chi2_ok(counts: dict, probs: dict, N: int):
    from scipy import stats
    keys = sorted(probs)
    exp_ = np.array([probs[t] * N for t in keys])
    obs = np.array([counts.get(t, 0) for t in keys], dtype=float)
    # no draw may fall outside the exact support
    assert sum(counts.values()) == obs.sum() == N, "draw outside the exact support"
    big = exp_ >= 5
    o = np.append(obs[big], obs[~big].sum())
    e = np.append(exp_[big], exp_[~big].sum())
    if e[-1] == 0:
        o, e = o[:-1], e[:-1]
    chi2 = ((o - e) ** 2 / e).sum()
    return stats.chi2.sf(chi2, len(e) - 1)


def _draws(q, k, v, S, mode, N):
    """N independent draws in one call: N identical batch rows have distinct Philox
    counters (the counter carries the batch index)."""
    qq = q.expand(N, -1, -1).contiguous()
    kk = k.expand(N, -1, -1, -1).contiguous()
    vv = v.expand(N, -1, -1, -1).contiguous()
    sl = torch.full((N,), 8, dtype=torch.int32)
    out, idx = oracle.decode(qq, kk, vv, sl, S, mode, seed=2024)
    return out[:, 0], idx[:, 0]


@pytest.mark.parametrize("S", [2, 4])
def test_bruteforce_n8_stratified_tuple_distribution(S):
    """Enumerate all 8^S index tuples: under stratified sampling point s lands on key j
    with probability S*|[s/S,(s+1)/S) ∩ [C_{j-1},C_j)|, independently over s."""
    q, k, v = _n8_case()
    p = probs(q, k, 0, 0, 8)
    C = np.concatenate([[0.0], np.cumsum(p)])
    P = np.zeros((S, 8))
    for s in range(S):
        for j in range(8):
            P[s, j] = S * max(0.0, min((s + 1) / S, C[j + 1]) - max(s / S, C[j]))
    exact = {}
    for tup in np.ndindex(*([8] * S)):
        pr = np.prod([P[s, tup[s]] for s in range(S)])
        if pr > 0:
            exact[tup] = pr
    assert abs(sum(exact.values()) - 1) < 1e-12
    N = 100000
    _, idx = _draws(q, k, v, S, "stratified", N)
    counts = {}
    for row in map(tuple, idx):
        counts[row] = counts.get(row, 0) + 1
    assert _chi2_ok(counts, exact, N) > 1e-5
    # exact mean over the enumeration equals attention; exact variance ordering
    vv = v[0, 0].double().numpy()
    E = sum(pr * vv[list(t)].mean(0) for t, pr in exact.items())
    assert np.max(np.abs(E - exact_attention(q, k, v, torch.tensor([8])).numpy()[0, 0])) < 1e-12
    var_strat = sum(pr * (vv[list(t)].mean(0) - E) ** 2 for t, pr in exact.items())
    var_iid = (p[:, None] * (vv - E) ** 2).sum(0) / S
    assert np.all(var_strat <= var_iid + 1e-15)


def test_bruteforce_n8_systematic_tuple_distribution():
    """Systematic: the tuple is a function of u alone; enumerate the u-intervals
    between the breakpoints frac(S*C_j) to get its exact distribution."""
    q, k, v = _n8_case()
    S = 4
    p = probs(q, k, 0, 0, 8)
    C = np.cumsum(p)
    br = np.unique(np.concatenate([[0.0, 1.0], np.mod(S * C, 1.0)]))
    exact = {}
    for lo, hi in zip(br[:-1], br[1:]):
        if hi <= lo:
            continue
        u = 0.5 * (lo + hi)
        tup = tuple(int(min(np.searchsorted(C, (u + s) / S, side="right"), 7)) for s in range(S))
        exact[tup] = exact.get(tup, 0) + (hi - lo)
    N = 100000
    _, idx = _draws(q, k, v, S, "systematic", N)
    counts = {}
    for row in map(tuple, idx):
        counts[row] = counts.get(row, 0) + 1
    assert _chi2_ok(counts, exact, N) > 1e-5


def test_bruteforce_n8_iid_tuple_distribution():
    """i.i.d. draws, sorted: P(a <= b) = p_a p_b (2 if a != b)."""
    q, k, v = _n8_case()
    p = probs(q, k, 0, 0, 8)
    exact = {}
    for a in range(8):
        for b in range(a, 8):
            exact[(a, b)] = p[a] * p[b] * (1 if a == b else 2)
    N = 100000
    _, idx = _draws(q, k, v, 2, "iid", N)
    counts = {}
    for row in map(tuple, idx):
        counts[row] = counts.get(row, 0) + 1
    assert _chi2_ok(counts, exact, N) > 1e-5


# ----------------------------------------------------------------------------- Monte Carlo

@pytest.mark.parametrize("mode", ["systematic", "stratified", "iid"])
def test_oracle_monte_carlo_unbiased_and_variance(mode):
    """4096 independent draws: the mean lies within 4 standard errors of exact
    attention in every coordinate; stratified and systematic variance is below the
    i.i.d. closed form (1/S) * Var_p(v) on average."""
    N, n, d, S = 4096, 64, 8, 16
    g = torch.Generator().manual_seed(31)
    q = bf16(2.5 * torch.randn(1, 1, d, generator=g))
    k = bf16(torch.randn(1, 1, n, d, generator=g))
    v = bf16(torch.randn(1, 1, n, d, generator=g))
    qq, kk, vv = q.expand(N, -1, -1).contiguous(), k.expand(N, -1, -1, -1).contiguous(), v.expand(N, -1, -1, -1).contiguous()
    sl = torch.full((N,), n, dtype=torch.int32)
    out, _ = oracle.decode(qq, kk, vv, sl, S, mode, seed=99)
    o = exact_attention(q, k, v, torch.tensor([n])).numpy()[0, 0]
    mean = out[:, 0].mean(0)
    sd = out[:, 0].std(0, ddof=1)
    z = (mean - o) / (sd / math.sqrt(N))
    assert np.all(np.abs(z) < 4), z
    p = probs(q, k, 0, 0, n)
    var_iid = (p[:, None] * (v[0, 0].double().numpy() - o) ** 2).sum(0) / S
    ratio = (sd ** 2).mean() / var_iid.mean()
    if mode == "iid":
        assert 0.85 < ratio < 1.15
    else:
        assert ratio < 0.9


# ----------------------------------------------------------------------------- Bernoulli qK^T
#
# "Stochastic Sparse Attention for Memory-Bound Inference", abstract, last sentences:
# Bernoulli qK^T sampling sparsifies the score stage with stochastic ternary queries.
# Reading: q~_i in {-a, 0, +a}, a = max |q_i|, P(q~_i = sign(q_i) a) = |q_i| / a, one
# independent Bernoulli draw per feature, so E[q~] = q (and E[q~ . k] = q . k).

def _head(vals):
    return bf16(torch.tensor(vals, dtype=torch.float32)).reshape(1, 1, -1)


def test_ternary_query_value_set_and_special_cases():
    g = torch.Generator().manual_seed(5)
    q = bf16(3.0 * torch.randn(2, 3, 64, generator=g))
    q[0, 0, 7] = 0.0
    for seed in range(20):
        qt, nnz = oracle.ternary_query(q, seed)
        qf, qtf = q.float(), qt.float()
        a = qf.abs().amax(-1, keepdim=True)
        assert torch.all((qtf == 0) | (qtf.abs() == a)), "values outside {-a, 0, +a}"
        nz = qtf != 0
        assert torch.all(torch.sign(qtf[nz]) == torch.sign(qf[nz])), "sign flipped"
        assert qtf[0, 0, 7] == 0, "a zero feature was drawn"
        top = qf.abs() == a  # probability 1: always kept
        assert torch.equal(qtf[top], qf[top])
        assert np.array_equal(nnz, nz.sum(-1).numpy())
    # every |q_i| equal: every feature kept, q~ = q exactly; q = 0: q~ = 0
    q_eq = _head([0.5, -0.5, 0.5, 0.5, -0.5, -0.5, 0.5, -0.5])
    assert torch.equal(oracle.ternary_query(q_eq, 3)[0], q_eq)
    q0 = _head([0.0] * 8)
    qt0, nnz0 = oracle.ternary_query(q0, 3)
    assert torch.all(qt0.float() == 0) and nnz0.sum() == 0


def test_ternary_query_unbiased_keep_rates():
    """Over many seeds, feature i is kept with frequency |q_i|/a (binomial z-score) and the
    mean of q~_i is q_i (z-score against the sample standard error)."""
    g = torch.Generator().manual_seed(11)
    q = bf16(torch.randn(1, 2, 48, generator=g))
    N = 6000
    draws = np.stack([oracle.ternary_query(q, seed)[0].float().numpy() for seed in range(N)])
    qf = q.float().numpy()
    a = np.abs(qf).max(-1, keepdims=True)
    p = np.abs(qf) / a
    kept = (draws != 0).mean(0)
    se_p = np.sqrt(np.maximum(p * (1 - p), 1e-12) / N)
    zp = (kept - p) / se_p
    assert np.abs(zp[p < 1]).max() < 5.0, np.abs(zp).max()
    assert np.all(kept[p == 1] == 1.0)
    mean = draws.mean(0)
    se = draws.std(0, ddof=1) / np.sqrt(N)
    z = (mean - qf)[se > 0] / se[se > 0]
    assert np.abs(z).max() < 5.0 and abs(z.mean()) < 0.2


def test_ternary_query_features_independent_by_enumeration():
    """Six features (two Philox blocks): the 64 keep/drop patterns have probability
    prod p_i or (1 - p_i); the oracle's pattern histogram over 20000 seeds fits it (chi^2).
    A uniform shared across features, or words reused between blocks, would not."""
    import itertools
    q = _head([1.0, -0.5, 0.75, 0.25, -1.0 * 0.625, 0.375])
    qf = q.float().numpy()[0, 0]
    p = np.abs(qf) / np.abs(qf).max()
    N = 20000
    counts = {}
    for seed in range(N):
        pat = tuple((oracle.ternary_query(q, seed)[0].float().numpy()[0, 0] != 0).astype(int))
        counts[pat] = counts.get(pat, 0) + 1
    chi2, dof = 0.0, 0
    for pat in itertools.product((0, 1), repeat=6):
        pr = float(np.prod([p[i] if pat[i] else 1 - p[i] for i in range(6)]))
        if pr == 0:
            assert counts.get(pat, 0) == 0
            continue
        e = N * pr
        chi2 += (counts.get(pat, 0) - e) ** 2 / e
        dof += 1
    dof -= 1
    # chi^2 with dof degrees of freedom: mean dof, sd sqrt(2 dof); 6 sd is far out
    assert chi2 < dof + 6 * math.sqrt(2 * dof), (chi2, dof)


def test_ternary_draw_differs_across_heads_and_seeds():
    q = bf16(torch.randn(2, 4, 64, generator=torch.Generator().manual_seed(2)))
    q[:] = q[0, 0]  # every head the same query: only the counter separates the draws
    qt, _ = oracle.ternary_query(q, 9)
    flat = qt.float().reshape(8, 64)
    assert len({tuple(r.tolist()) for r in flat}) == 8
    assert not torch.equal(oracle.ternary_query(q, 10)[0], qt)


@pytest.mark.parametrize("mode", ["dense", "systematic", "stratified", "iid"])
def test_bernoulli_decode_scores_with_the_ternary_query(mode):
    """The Bernoulli step comes first: decoding q with it equals decoding its ternary draw
    without it, exactly (same seed for both draws)."""
    q, k, v = rand_case(2, 8, 2, 64, 300, seed=41, qstd=2.0)
    sl = [300, 170]
    S = 0 if mode == "dense" else 32
    o1, i1 = oracle.decode(q, k, v, sl, S, mode, seed=6, bernoulli=True)
    qt, _ = oracle.ternary_query(q, 6)
    o2, i2 = oracle.decode(qt, k, v, sl, S, mode, seed=6)
    assert np.array_equal(o1, o2)
    if mode != "dense":
        assert np.array_equal(i1, i2)
    # a query whose features all have the same magnitude is drawn unchanged
    q_eq = bf16(0.5 * torch.sign(torch.randn(2, 8, 64, generator=torch.Generator().manual_seed(8))))
    o3, i3 = oracle.decode(q_eq, k, v, sl, S, mode, seed=6, bernoulli=True)
    o4, i4 = oracle.decode(q_eq, k, v, sl, S, mode, seed=6)
    assert np.array_equal(o3, o4)
    if mode != "dense":
        assert np.array_equal(i3, i4)
