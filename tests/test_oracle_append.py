"""Pins of the oracle's append step (CPU).  The appended summary row is
checked against the C pack_summary (written separately), and building a
cache token by token must give the cache and summary packed at once."""
import numpy as np
import pytest


def _rand(rng, shape):
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def test_append_row_matches_pack_summary(oracle_mod):
    rng = np.random.default_rng(3)
    Bt, Hkv, N, d, d_sel = 2, 3, 37, 64, 16
    K, V = _rand(rng, (Bt, Hkv, N, d)), _rand(rng, (Bt, Hkv, N, d))
    sel = np.stack([np.sort(rng.choice(d, d_sel, replace=False)) for _ in range(Hkv)]).astype(np.int32)
    Ks = oracle_mod.pack_summary(K, sel, d_sel)
    k_new, v_new = _rand(rng, (Bt, Hkv, d)), _rand(rng, (Bt, Hkv, d))
    for pos in (0, 17, N - 1):
        K2, V2, Ks2 = oracle_mod.append(K, V, Ks, k_new, v_new, sel, pos)
        assert np.array_equal(K2[:, :, pos], k_new) and np.array_equal(V2[:, :, pos], v_new)
        other = np.arange(N) != pos
        assert np.array_equal(K2[:, :, other], K[:, :, other])
        assert np.array_equal(V2[:, :, other], V[:, :, other])
        assert np.array_equal(Ks2[:, :, other], Ks[:, :, other])
        assert np.array_equal(Ks2, oracle_mod.pack_summary(K2, sel, d_sel))


def test_cache_built_token_by_token(oracle_mod):
    rng = np.random.default_rng(5)
    Bt, Hkv, N, d, d_sel = 1, 2, 20, 128, 32
    K, V = _rand(rng, (Bt, Hkv, N, d)), _rand(rng, (Bt, Hkv, N, d))
    sel = np.stack([rng.permutation(d)[:d_sel] for _ in range(Hkv)]).astype(np.int32)   # any order
    K2, V2 = np.zeros_like(K), np.zeros_like(V)
    Ks2 = np.zeros((Bt, Hkv, N, d_sel), np.uint16)
    for i in range(N):
        K2, V2, Ks2 = oracle_mod.append(K2, V2, Ks2, K[:, :, i], V[:, :, i], sel, i)
    assert np.array_equal(K2, K) and np.array_equal(V2, V)
    assert np.array_equal(Ks2, oracle_mod.pack_summary(K, sel, d_sel))


def test_append_rejects_positions_outside_the_cache(oracle_mod):
    z = np.zeros((1, 1, 4, 64), np.uint16)
    zs = np.zeros((1, 1, 4, 16), np.uint16)
    row = np.zeros((1, 1, 64), np.uint16)
    sel = np.arange(16, dtype=np.int32)[None]
    for pos in (-1, 4):
        with pytest.raises(ValueError):
            oracle_mod.append(z, z, zs, row, row, sel, pos)
