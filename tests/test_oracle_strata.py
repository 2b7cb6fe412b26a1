"""Pins of the oracle's other strata (CPU): the top-k + uniform hybrid and the
top-p stratum, which the SSA page names as special cases of its strata.  The
uniform hybrid is pinned against the SSA sampler on constant scores (where the
two coincide), against its selection frequencies and against its limits; the
top-p size against a brute-force restatement (Python sort on the C order key,
math.fsum masses)."""
import math

import numpy as np
import pytest


def test_uniform_hybrid_equals_ssa_on_constant_scores(oracle_mod):
    # constant estimates make every remainder term equal: SSA's p is the uniform p
    N, k, B = 1000, 30, 70.0
    s = np.full(N, 0.25, np.float32)
    for seed in (0, 9):
        i_u, p_u = oracle_mod.select_unit_uniform(s, k, B, seed, 0, 1)
        i_s, p_s, _, _ = oracle_mod.select_unit(s, k, B, seed, 0, 1)
        assert np.array_equal(i_u, i_s) and np.array_equal(p_u, p_s)


def test_uniform_hybrid_keeps_the_topk_and_draws_the_rest_with_one_p(oracle_mod):
    rng = np.random.default_rng(2)
    N, k, B = 300, 20, 30.0
    s = (rng.standard_normal(N) * 1.5).astype(np.float32)
    t_idx = set(oracle_mod.select_unit(s, k, 0.0, 0, 0, 0)[0].tolist())
    p_r = np.float32(B) / np.float32(N - k)
    trials = 3000
    hits = np.zeros(N)
    counts = []
    for seed in range(trials):
        idx, p = oracle_mod.select_unit_uniform(s, k, B, seed, 1, 0)
        assert t_idx <= set(idx.tolist())
        assert np.all(p[np.isin(idx, list(t_idx))] == 1.0) and np.all(p[~np.isin(idx, list(t_idx))] == p_r)
        assert np.all(np.diff(idx) > 0)
        hits[idx] += 1
        counts.append(idx.size)
    rest = np.array([j for j in range(N) if j not in t_idx])
    freq = hits[rest] / trials
    sd = math.sqrt(float(p_r) * (1 - float(p_r)) / trials)
    assert np.all(np.abs(freq - float(p_r)) <= 5 * sd)
    assert abs(np.mean(counts) - (k + (N - k) * float(p_r))) < 5 * math.sqrt((N - k) * float(p_r) / trials)


def test_uniform_hybrid_limits(oracle_mod):
    s = np.random.default_rng(3).standard_normal(500).astype(np.float32)
    t = oracle_mod.select_unit(s, 25, 0.0, 0, 0, 0)[0]
    idx, p = oracle_mod.select_unit_uniform(s, 25, 0.0, 4, 0, 0)      # B = 0: pure top-k
    assert np.array_equal(idx, t) and np.all(p == 1.0)
    idx, p = oracle_mod.select_unit_uniform(s, 25, math.inf, 4, 0, 0)  # B = inf: everything
    assert idx.tolist() == list(range(500)) and np.all(p == 1.0)
    idx, p = oracle_mod.select_unit_uniform(s, 600, 5.0, 4, 0, 0)     # k >= N: no remainder
    assert idx.tolist() == list(range(500))
    idx, p = oracle_mod.select_unit_uniform(s, 25, 1e9, 4, 0, 0)      # clipped: p = 1 on R
    assert idx.size == 500 and np.all(p == 1.0)


def _brute_top_p(oracle_mod, s, top_p):
    n = len(s)
    order = sorted(range(n), key=lambda i: (-oracle_mod.orderkey(float(s[i])), i))
    mx = max(float(v) for v in s)
    w = [math.exp(float(s[i]) - mx) for i in order]
    total = math.fsum(w)
    for kk in range(1, n + 1):
        if math.fsum(w[:kk]) / total >= top_p:
            return kk, abs(math.fsum(w[:kk]) / total - top_p)
    return n, 1.0


@pytest.mark.parametrize("seed", range(6))
def test_top_p_count_matches_brute_force(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(40):
        n = int(rng.integers(1, 13))
        s = (np.round(rng.standard_normal(n) * 3) / 2).astype(np.float32)   # many exact ties
        if rng.random() < 0.3:
            s[rng.integers(0, n)] = -0.0
        top_p = float(rng.uniform(0.01, 0.99))
        want, margin = _brute_top_p(oracle_mod, s, top_p)
        if margin < 1e-9:
            continue   # too close to a boundary for two summation orders to agree
        assert oracle_mod.top_p_count(s, top_p) == want, (s, top_p)


def test_top_p_extremes_and_monotonicity(oracle_mod):
    s = np.random.default_rng(7).standard_normal(200).astype(np.float32)
    assert oracle_mod.top_p_count(s, 0.0) == 0
    assert oracle_mod.top_p_count(s, 1e-12) == 1
    assert oracle_mod.top_p_count(s, 1.0) == 200
    ks = [oracle_mod.top_p_count(s, t) for t in np.linspace(0.01, 0.99, 50)]
    assert all(a <= b for a, b in zip(ks, ks[1:]))
    # one dominant token carries almost all the mass
    s2 = np.zeros(50, np.float32)
    s2[17] = 40.0
    assert oracle_mod.top_p_count(s2, 0.999) == 1


def test_top_p_stratum_is_the_topk_stratum_of_its_size(oracle_mod):
    s = (np.random.default_rng(8).standard_normal(400) * 2).astype(np.float32)
    kp = oracle_mod.top_p_count(s, 0.6)
    a = oracle_mod.select_unit_top_p(s, 0.6, 12.0, 5, 0, 1)
    b = oracle_mod.select_unit(s, kp, 12.0, 5, 0, 1)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_uniform_hybrid_is_unbiased_by_enumeration(oracle_mod):
    # with one p on R the corrected numerator and denominator are still exactly unbiased
    import itertools
    from test_oracle_attend import _bf16, _dense_sums
    rng = np.random.default_rng(21)
    N, d, G, k, B = 12, 16, 2, 3, 4.0
    qh = _bf16(rng.standard_normal((G, d)) * 0.7)
    K = _bf16(rng.standard_normal((N, d)))
    V = _bf16(rng.standard_normal((N, d)))
    s = rng.standard_normal(N).astype(np.float32)
    scale = 0.25
    T = sorted(oracle_mod.select_unit(s, k, 0.0, 0, 0, 0)[0].tolist())
    R = [j for j in range(N) if j not in T]
    p_r = float(np.float32(B) / np.float32(N - k))
    idx, p = oracle_mod.select_unit_uniform(s, k, B, 0, 0, 0)
    assert set(T) <= set(idx.tolist()) and np.all(p[~np.isin(idx, T)] == np.float32(p_r))
    num = np.zeros((G, d))
    den = np.zeros(G)
    for x in itertools.product([0, 1], repeat=len(R)):
        prob = 1.0
        S = list(T)
        for j, xi in zip(R, x):
            prob *= p_r if xi else 1.0 - p_r
            if xi:
                S.append(j)
        S.sort()
        pw = np.array([1.0 if j in T else p_r for j in S], np.float32)
        out, lse = oracle_mod.attend_unit(qh, K, V, np.array(S, np.int32), pw, scale)
        w = np.exp(lse.astype(np.float64))
        num += prob * w[:, None] * out.astype(np.float64)
        den += prob * w
    want_num, want_den = _dense_sums(qh, K, V, scale)
    assert np.allclose(den, want_den, rtol=2e-6)
    assert np.allclose(num, want_num, rtol=2e-5, atol=2e-5 * np.abs(want_num).max())


def test_top_p_shares_bracket_top_p(oracle_mod):
    """The stratum's edge: the share of one token fewer stays below top_p, the stratum's own reaches it."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        N = int(rng.integers(2, 300))
        s = (rng.standard_normal(N) * 2).astype(np.float32)
        top_p = float(rng.uniform(0.05, 0.95))
        k, before, at = oracle_mod.top_p_shares(s, top_p)
        assert k == oracle_mod.top_p_count(s, top_p)
        assert before < top_p <= at
