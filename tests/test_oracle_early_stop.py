"""Pins for the oracle's attention with S2O-style early stopping.

"S2O: early stopping for sparse attention via online permutation", technical
summary, Method section 2: candidate blocks are processed in descending
estimated importance, the marginal gain each processed block contributes is
tracked, and the computation ends once that gain falls below a preset
threshold tau relative to the accumulated score.  Applied to one unit's
selected rows: rows ordered by the estimated score s (descending, ties by
list position), blocks of `block` rows, the gain of a block is its share of
the corrected softmax denominator, and the step stops after the first block
whose gain is below tau times the denominator so far, for every query head.

The pins: closed-form values on a hand-built case, the two limits (tau = 0
keeps every row, tau > 1 keeps only the first block) against the plain
corrected attention, invariance to the list's order, and that the number of
blocks never grows with tau.
"""
import math

import numpy as np
import pytest


def _bf16_exact(x):
    """Values that bf16 holds exactly, as raw patterns."""
    a = np.asarray(x, np.float32)
    bits = a.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _rand_bf16(rng, shape, scale=1.0):
    a = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _hand_case():
    # one head, d = 2: q = (1, 0), K rows give logits 2, 0, -5 (scale 1, p = 1); the estimated scores put the
    # rows in that order; V rows are the unit vectors and their sum
    q = _bf16_exact([[1.0, 0.0]])
    K = _bf16_exact([[2.0, 0.0], [0.0, 0.0], [-5.0, 0.0]])
    V = _bf16_exact([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    idx = np.array([0, 1, 2], np.int32)
    p = np.ones(3, np.float32)
    s = np.array([3.0, 2.0, 1.0], np.float32)
    return q, K, V, idx, p, s


def test_hand_built_case_closed_form(oracle_mod):
    q, K, V, idx, p, s = _hand_case()
    e2, e0, em5 = math.exp(2.0), 1.0, math.exp(-5.0)
    want_ratios = [1.0, e0 / (e2 + e0), em5 / (e2 + e0 + em5)]
    # tau = 0.2: block 1's gain 1 / (e^2 + 1) = 0.119 is below it -> blocks 0 and 1
    out, lse, used, ratios = oracle_mod.attend_unit_early_stop(q, K, V, idx, p, s, 1.0, 0.2, block=1)
    assert used == 2
    assert np.allclose(ratios, want_ratios, rtol=1e-6)
    w = np.array([e2, e0]) / (e2 + e0)
    assert np.allclose(out[0], [w[0], w[1]], rtol=1e-6)
    assert math.isclose(float(lse[0]), math.log(e2 + e0), rel_tol=1e-6)
    # tau = 0.01: block 1 (0.119) passes, block 2 (0.0008) stops after itself -> all three
    _, lse, used, _ = oracle_mod.attend_unit_early_stop(q, K, V, idx, p, s, 1.0, 0.01, block=1)
    assert used == 3 and math.isclose(float(lse[0]), math.log(e2 + e0 + em5), rel_tol=1e-6)
    # tau = 0.5 with blocks of two rows: block 0 = rows 0, 1; block 1 = row 2, gain e^-5 / (...) < 0.5
    _, _, used, ratios = oracle_mod.attend_unit_early_stop(q, K, V, idx, p, s, 1.0, 0.5, block=2)
    assert used == 2 and np.allclose(ratios, [1.0, em5 / (e2 + e0 + em5)], rtol=1e-6)


def test_inclusion_probability_enters_the_gain(oracle_mod):
    # row 1 kept with p = 0.25: its corrected logit is 0 - log 0.25 = log 4, so its gain is 4 / (e^2 + 4)
    q, K, V, idx, p, s = _hand_case()
    p = np.array([1.0, 0.25, 1.0], np.float32)
    e2 = math.exp(2.0)
    out, lse, used, ratios = oracle_mod.attend_unit_early_stop(q, K, V, idx, p, s, 1.0, 0.4, block=1)
    assert math.isclose(float(ratios[1]), 4.0 / (e2 + 4.0), rel_tol=1e-6)
    # block 1's gain 0.351 is below 0.4: blocks 0 and 1 are kept, weighted e^2 : 4
    assert used == 2
    assert np.allclose(out[0], [e2 / (e2 + 4.0), 4.0 / (e2 + 4.0)], rtol=1e-6)
    assert math.isclose(float(lse[0]), math.log(e2 + 4.0), rel_tol=1e-6)
    # with tau = 0.3 block 1 passes and block 2 (gain ~6e-4) ends the step after itself
    _, _, used, _ = oracle_mod.attend_unit_early_stop(q, K, V, idx, p, s, 1.0, 0.3, block=1)
    assert used == 3


@pytest.mark.parametrize("G,d,n,block", [(1, 64, 300, 128), (4, 128, 517, 128), (8, 64, 1000, 64), (2, 128, 128, 128)])
def test_limits_match_the_plain_corrected_attention(oracle_mod, G, d, n, block):
    rng = np.random.default_rng(G * 1000 + n)
    N = n + 50
    qh = _rand_bf16(rng, (G, d), 0.5)
    K = _rand_bf16(rng, (N, d))
    V = _rand_bf16(rng, (N, d))
    idx = np.sort(rng.choice(N, size=n, replace=False)).astype(np.int32)
    p = rng.uniform(0.05, 1.0, n).astype(np.float32)
    s = rng.standard_normal(n).astype(np.float32)
    scale = 1 / math.sqrt(d)
    # tau = 0: every block, the plain corrected attention over the whole list
    out0, lse0, used0, _ = oracle_mod.attend_unit_early_stop(qh, K, V, idx, p, s, scale, 0.0, block=block)
    ref_out, ref_lse = oracle_mod.attend_unit(qh, K, V, idx, p, scale)
    assert used0 == -(-n // block)
    assert np.allclose(out0, ref_out, rtol=1e-5, atol=1e-6) and np.allclose(lse0, ref_lse, rtol=1e-6, atol=1e-6)
    # tau > 1: the first block only (every gain ratio is at most 1), i.e. the block-many highest-s rows
    out1, lse1, used1, _ = oracle_mod.attend_unit_early_stop(qh, K, V, idx, p, s, scale, 1.5, block=block)
    top = np.lexsort((np.arange(n), -s.astype(np.float64)))[:block]
    ref_out, ref_lse = oracle_mod.attend_unit(qh, K, V, idx[top], p[top], scale)
    assert used1 == 1
    assert np.allclose(out1, ref_out, rtol=1e-5, atol=1e-6) and np.allclose(lse1, ref_lse, rtol=1e-6, atol=1e-6)
    # a forced block count is the plain attention over that many blocks of the order
    order = np.lexsort((np.arange(n), -s.astype(np.float64)))
    for fb in (1, 2, used0):
        o, l, u, _ = oracle_mod.attend_unit_early_stop(qh, K, V, idx, p, s, scale, 0.0, block=block, force_blocks=fb)
        rows = order[:fb * block]
        r_out, r_lse = oracle_mod.attend_unit(qh, K, V, idx[rows], p[rows], scale)
        assert u == min(fb, used0)   # a count past the last block is clamped
        assert np.allclose(o, r_out, rtol=1e-5, atol=1e-6) and np.allclose(l, r_lse, rtol=1e-6)


def test_list_order_does_not_matter_and_blocks_shrink_with_tau(oracle_mod):
    rng = np.random.default_rng(7)
    G, d, N, n = 4, 64, 2000, 700
    qh = _rand_bf16(rng, (G, d), 0.8)
    K = _rand_bf16(rng, (N, d))
    V = _rand_bf16(rng, (N, d))
    idx = np.sort(rng.choice(N, size=n, replace=False)).astype(np.int32)
    p = rng.uniform(0.1, 1.0, n).astype(np.float32)
    s = rng.standard_normal(n).astype(np.float32)   # distinct values: the order has no ties
    scale = 0.125
    perm = rng.permutation(n)
    prev = None
    for tau in (0.0, 1e-4, 1e-3, 1e-2, 0.05, 0.2, 1.0, 2.0):
        a = oracle_mod.attend_unit_early_stop(qh, K, V, idx, p, s, scale, tau, block=64)
        b = oracle_mod.attend_unit_early_stop(qh, K, V, idx[perm], p[perm], s[perm], scale, tau, block=64)
        assert a[2] == b[2] and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        if prev is not None:
            assert a[2] <= prev
        prev = a[2]
        # the stop is the first block whose ratio is below tau
        r = a[3]
        below = np.nonzero(r < tau)[0]
        assert a[2] == (int(below[0]) + 1 if below.size else r.size)


def test_empty_list(oracle_mod):
    qh = np.zeros((2, 64), np.uint16)
    K = np.zeros((4, 64), np.uint16)
    out, lse, used, ratios = oracle_mod.attend_unit_early_stop(qh, K, K, np.zeros(0, np.int32),
                                                               np.zeros(0, np.float32), np.zeros(0, np.float32),
                                                               0.1, 0.01)
    assert used == 0 and ratios.size == 0 and np.all(out == 0) and np.all(np.isneginf(lse))
