"""Pins for the oracle's stratified selection.

Stratified Sparse Attention news page, "How SSA splits the cache into
strata": top-k stratum read deterministically; the remainder sampled with
probability proportional to approximate attention; top-k and the top-k +
uniform hybrid are special cases ("The idea is close to classical stratified
sampling").
"""
import math

import numpy as np
import pytest


def _next_down(x: np.float32) -> np.float32:
    return np.nextafter(np.float32(x), np.float32(-np.inf), dtype=np.float32)


def _check_bucket_floor(oracle_mod, m, v):
    """m is the smallest binary32 value in v's 12-bit order-key bucket: same top 12 key
    bits as v, m <= v, and the next value down lies in another bucket; and v - m is at most
    |v| / 8 (a bucket spans an eighth of an octave; 2^-129 in the subnormal range)."""
    assert m <= v
    assert oracle_mod.orderkey(m) >> 20 == oracle_mod.orderkey(v) >> 20
    below = _next_down(m)
    assert not np.isfinite(below) or oracle_mod.orderkey(below) >> 20 != oracle_mod.orderkey(v) >> 20
    assert float(v) - float(m) <= max(abs(float(v)) / 8, 2.0 ** -129)


def _order(s):
    # brute force: descending value with -0 below +0, ties by ascending index
    key = [(-(float(v)), -math.copysign(1.0, float(v)) if v == 0 else 0.0, i) for i, v in enumerate(s)]
    return [k[2] for k in sorted(key)]


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 400))
    s = np.round(rng.standard_normal(N) * 3) / 2       # many exact ties
    s[rng.random(N) < 0.1] = 0.0
    s[rng.random(N) < 0.1] = -0.0
    s = s.astype(np.float32)
    for k in sorted({0, 1, N // 3, N - 1, N, N + 5}):
        if k < 0:
            continue
        idx, p, m, Z = oracle_mod.select_unit(s, k, 0.0, 0, 0, 0)
        want = sorted(_order(s)[:k])
        assert idx.tolist() == want
        assert np.all(p == 1.0)
        if 0 < N and k <= N:
            _check_bucket_floor(oracle_mod, m, s[_order(s)[max(k, 1) - 1]])


def test_budget_infinite_selects_everything(oracle_mod):
    s = np.random.default_rng(0).standard_normal(333).astype(np.float32)
    idx, p, m, Z = oracle_mod.select_unit(s, 17, math.inf, 5, 0, 0)
    assert idx.tolist() == list(range(333)) and np.all(p == 1.0)


def test_k_at_least_n_is_dense(oracle_mod):
    s = np.random.default_rng(1).standard_normal(50).astype(np.float32)
    idx, p, m, Z = oracle_mod.select_unit(s, 50, 10.0, 5, 0, 0)
    assert idx.tolist() == list(range(50)) and np.all(p == 1.0) and Z == 0.0


def test_k_zero_uses_the_maximum_as_reference(oracle_mod):
    s = np.random.default_rng(2).standard_normal(100).astype(np.float32)
    idx, p, m, Z, p_all = oracle_mod.select_unit(s, 0, 10.0, 5, 0, 0, want_p_all=True)
    _check_bucket_floor(oracle_mod, m, s.max())
    assert Z >= 1.0  # the arg-max term is exp(max - m) >= 1
    assert np.all(p_all < 1.0 + 1e-7)


@pytest.mark.parametrize("v", [0.25, 1.0, 1.7, 3.14159, -0.3, -2.5, 1e-30, -1e-30, 0.0, -0.0, 1e30, -1e30,
                               1.4e-45, -1.4e-45, 3.4e38, -3.4e38])
def test_bucket_floor_is_the_lower_edge_of_the_key_bucket(oracle_mod, v):
    v = np.float32(v)
    _check_bucket_floor(oracle_mod, oracle_mod.bucket_floor(v), v)
    # normal positive powers of two are their own bucket floor: their low key bits are zero
    if v >= 2.0 ** -126 and float(v) == 2.0 ** math.floor(math.log2(float(v))):
        assert oracle_mod.bucket_floor(v) == v


def test_p_does_not_depend_on_the_reference_point(oracle_mod):
    # p_j = B exp(s_j - m) / sum_R exp(s_l - m): shifting every score by a power of two that
    # moves m across buckets leaves p unchanged up to rounding
    rng = np.random.default_rng(8)
    s = (rng.standard_normal(3000) * 0.7).astype(np.float32)
    _, _, m1, _, p1 = oracle_mod.select_unit(s, 30, 60.0, 2, 0, 0, want_p_all=True)
    _, _, m2, _, p2 = oracle_mod.select_unit(s + np.float32(0.5), 30, 60.0, 2, 0, 0, want_p_all=True)
    assert np.allclose(p1, p2, rtol=2e-5, atol=1e-12)


def test_inclusion_probabilities_sum_to_budget(oracle_mod):
    # sum_R B e_j / Z = B when no p is clipped
    rng = np.random.default_rng(3)
    s = (rng.standard_normal(5000) * 0.3).astype(np.float32)
    k, B = 50, 40.0
    idx, p, m, Z, p_all = oracle_mod.select_unit(s, k, B, 1, 0, 0, want_p_all=True)
    top = set(_order(s)[:k])
    R = [j for j in range(s.size) if j not in top]
    assert np.all(p_all[list(top)] == 1.0)
    assert p_all[R].max() < 1.0
    assert abs(p_all[R].astype(np.float64).sum() - B) < 1e-4 * B
    # proportional to exp(s): the ratio of two p's is the ratio of their exponentials
    a, b = R[0], R[1]
    assert abs(p_all[a] / p_all[b] - math.exp(float(s[a]) - float(s[b]))) < 1e-5


def test_clipping_keeps_sum_below_budget(oracle_mod):
    s = np.zeros(100, np.float32)
    s[:5] = 10.0
    idx, p, m, Z, p_all = oracle_mod.select_unit(s, 0, 50.0, 1, 0, 0, want_p_all=True)
    assert np.all(p_all[:5] == 1.0)
    assert p_all.sum() <= 50.0 + 1e-4


def test_constant_scores_give_the_uniform_hybrid(oracle_mod):
    # constant estimates: T = first k indices, every other token has p = B/(N-k)
    N, k, B = 1000, 30, 70.0
    s = np.full(N, 0.25, np.float32)
    idx, p, m, Z, p_all = oracle_mod.select_unit(s, k, B, 9, 0, 0, want_p_all=True)
    assert np.all(p_all[:k] == 1.0)
    assert Z == np.float32(N - k)
    assert np.all(p_all[k:] == np.float32(B) / np.float32(N - k))
    assert set(range(k)) <= set(idx.tolist())


def test_budget_zero_is_pure_topk(oracle_mod):
    s = np.random.default_rng(4).standard_normal(777).astype(np.float32)
    idx, p, m, Z = oracle_mod.select_unit(s, 40, 0.0, 3, 0, 0)
    assert idx.tolist() == sorted(_order(s)[:40])


def test_selection_frequency_matches_p(oracle_mod):
    # Poisson sampling: token j is drawn with probability p_j, independently of the others
    rng = np.random.default_rng(5)
    N, k, B = 64, 4, 12.0
    s = (rng.standard_normal(N) * 1.2).astype(np.float32)
    _, _, _, _, p_all = oracle_mod.select_unit(s, k, B, 0, 0, 0, want_p_all=True)
    trials = 4000
    hits = np.zeros(N)
    counts = []
    for seed in range(trials):
        idx, _, _, _ = oracle_mod.select_unit(s, k, B, seed, 1, 2)
        hits[idx] += 1
        counts.append(idx.size)
    freq = hits / trials
    sd = np.sqrt(np.maximum(p_all * (1 - p_all), 1e-12) / trials)
    assert np.all(np.abs(freq - p_all) <= 5 * sd + 1e-9)
    assert abs(np.mean(counts) - p_all.astype(np.float64).sum()) < 5 * np.sqrt(p_all.sum() / trials) + 1e-6


def test_selection_is_deterministic_per_seed_and_unit(oracle_mod):
    s = np.random.default_rng(6).standard_normal(4000).astype(np.float32)
    a = oracle_mod.select_unit(s, 20, 100.0, 11, 0, 0)[0]
    b = oracle_mod.select_unit(s, 20, 100.0, 11, 0, 0)[0]
    c = oracle_mod.select_unit(s, 20, 100.0, 12, 0, 0)[0]
    d = oracle_mod.select_unit(s, 20, 100.0, 11, 0, 1)[0]
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_non_finite_scores_are_rejected(oracle_mod):
    s = np.zeros(10, np.float32)
    s[3] = np.nan
    with pytest.raises(FloatingPointError):
        oracle_mod.select_unit(s, 2, 1.0, 0, 0, 0)
    s[3] = np.inf
    with pytest.raises(FloatingPointError):
        oracle_mod.select_unit(s, 2, 1.0, 0, 0, 0)


def test_cap_overflow_is_reported(oracle_mod):
    s = np.zeros(10, np.float32)
    with pytest.raises(OverflowError):
        oracle_mod.select_unit(s, 5, 0.0, 0, 0, 0, cap=3)


def _pinned_score_cases():
    """The selection's pinned input families: ties, constant scores, k = 0, pure top-k, k = N - 1, a
    single token, signed zeros, clipping, scores spanning many octaves, needles."""
    rng = np.random.default_rng(11)
    for N, k, B, kind in [(3000, 40, 40.0, "ties"), (3000, 40, 40.0, "constant"), (2500, 0, 30.0, "normal"),
                          (2500, 25, 0.0, "normal"), (700, 699, 10.0, "normal"), (1, 0, 5.0, "normal"),
                          (513, 5, 5.0, "signed_zero"), (4097, 60, 1e6, "normal"), (2000, 30, 30.0, "wide"),
                          (20000, 200, 200.0, "normal"), (20000, 200, 200.0, "needles")]:
        if kind == "ties":
            s = np.round(rng.standard_normal(N) * 2) / 4
        elif kind == "constant":
            s = np.full(N, 0.375)
        elif kind == "signed_zero":
            s = np.where(rng.random(N) < 0.5, 0.0, -0.0)
            s[::7] = rng.standard_normal(s[::7].shape)
        elif kind == "wide":
            s = rng.standard_normal(N) * np.exp2(rng.integers(-20, 6, N))
        elif kind == "needles":
            s = rng.standard_normal(N) * 1.5
            s[rng.choice(N, 16, replace=False)] += 8
        else:
            s = rng.standard_normal(N) * 1.5
        yield kind, s.astype(np.float32), k, B


def test_reference_point_reading_changes_nothing_beyond_rounding(oracle_mod):
    """The reference point m is free ("How SSA splits the cache into strata" defines p only through the
    normalised estimate).  Selecting with m = the lower edge of the k-th score's 12-bit key bucket (the
    library's reading) and with m = the k-th score itself gives the same index sets (apart from tokens
    with |u - p| <= 1e-6), and p differs only by the roundings that depend on m: fl32(s_j - m) (at most
    2^-24 |s_j - m| absolute, i.e. that relative error in e_j), the exp and the binary32 product and
    quotient (2^-24 each), and Z, whose relative error is a weighted mean of its terms' and so at most
    the largest of them."""
    eps = 2.0 ** -24
    for kind, s, k, B in _pinned_score_cases():
        N = s.size
        for seed in range(3):
            ia, pa, ma, Za, pall_a = oracle_mod.select_unit(s, k, B, seed, 0, 1, want_p_all=True)
            ib, pb, mb, Zb, pall_b = oracle_mod.select_unit(s, k, B, seed, 0, 1, want_p_all=True, m_at_kth=True)
            assert ma <= mb, (kind, ma, mb)   # the bucket edge lies at or below the k-th score
            for j in set(ia.tolist()) ^ set(ib.tolist()):
                u = oracle_mod.uniform(seed, j, 1, 0)
                assert min(abs(u - float(pall_a[j])), abs(u - float(pall_b[j]))) <= 1e-6, (kind, j)
            top = set(_order(s)[:min(k, N)])
            R = np.array([j for j in range(N) if j not in top], np.int64)
            if R.size == 0 or B == 0.0:
                assert np.array_equal(pall_a, pall_b)
                continue
            da = np.abs(s.astype(np.float64) - float(ma))
            db = np.abs(s.astype(np.float64) - float(mb))
            zrel = eps * (da[R].max() + db[R].max() + 2)
            bound = pall_a.astype(np.float64) * (eps * (da + db + 6) + zrel)
            diff = np.abs(pall_a.astype(np.float64) - pall_b.astype(np.float64))
            assert np.all(diff <= bound + 1e-45), (kind, seed, float(np.max(diff / (bound + 1e-45))))
