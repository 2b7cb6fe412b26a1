"""Pins for the oracle's corrected sparse attention and the whole step.

Stratified Sparse Attention news page, "How SSA splits the cache into
strata": the correction for each token's inclusion probability recovers the
attention mass outside the chosen set -- with Poisson sampling, the weighted
numerator sum_S e^{l_i} V_i / p_i and denominator sum_S e^{l_i} / p_i are
unbiased for the dense sums.  FASA section 3, Stage 2: exact attention over
the selected rows.
"""
import itertools
import math

import numpy as np
import pytest
import torch


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dense_sums(qh, K, V, scale):
    logits = scale * (_val(K) @ _val(qh).T)          # [N][G]
    w = np.exp(logits)
    return (w.T @ _val(V)), w.sum(axis=0)            # [G][d], [G]


def test_dense_attention_matches_library_sdpa(oracle_mod):
    rng = np.random.default_rng(0)
    Bt, Hq, Hkv, d, N = 2, 8, 2, 64, 300
    q = _bf16(rng.standard_normal((Bt, Hq, d)))
    K = _bf16(rng.standard_normal((Bt, Hkv, N, d)))
    V = _bf16(rng.standard_normal((Bt, Hkv, N, d)))
    scale = 1 / math.sqrt(d)
    out, lse = oracle_mod.dense_attention(q, K, V, scale)
    G = Hq // Hkv
    qt = torch.from_numpy(_val(q)).view(Bt, Hkv, G, d)
    kt = torch.from_numpy(_val(K))
    vt = torch.from_numpy(_val(V))
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(np.float32(scale)))
    want_lse = torch.logsumexp(float(np.float32(scale)) * qt @ kt.transpose(-1, -2), dim=-1)
    assert np.allclose(out.reshape(Bt, Hkv, G, d), want.numpy(), atol=2e-6, rtol=2e-6)
    assert np.allclose(lse.reshape(Bt, Hkv, G), want_lse.numpy(), atol=2e-6, rtol=2e-6)


def test_horvitz_thompson_expectation_by_enumeration(oracle_mod):
    # every inclusion subset of R, weighted by its probability: E[num] and E[den] are the dense sums
    rng = np.random.default_rng(1)
    N, d, G, k, B = 12, 16, 2, 3, 4.0
    qh = _bf16(rng.standard_normal((G, d)) * 0.7)
    K = _bf16(rng.standard_normal((N, d)))
    V = _bf16(rng.standard_normal((N, d)))
    s = (rng.standard_normal(N)).astype(np.float32)
    scale = 0.25
    _, _, _, _, p_all = oracle_mod.select_unit(s, k, B, 0, 0, 0, want_p_all=True)
    order = sorted(range(N), key=lambda i: (-float(s[i]), i))
    T = sorted(order[:k])
    R = [j for j in range(N) if j not in T]
    assert np.all(p_all[T] == 1.0) and np.all((p_all[R] > 0) & (p_all[R] < 1))
    num = np.zeros((G, d))
    den = np.zeros(G)
    for x in itertools.product([0, 1], repeat=len(R)):
        prob = 1.0
        S = list(T)
        for j, xi in zip(R, x):
            prob *= float(p_all[j]) if xi else 1.0 - float(p_all[j])
            if xi:
                S.append(j)
        S.sort()
        out, lse = oracle_mod.attend_unit(qh, K, V, np.array(S, np.int32), p_all[S], scale)
        w = np.exp(lse.astype(np.float64))
        num += prob * w[:, None] * out.astype(np.float64)
        den += prob * w
    want_num, want_den = _dense_sums(qh, K, V, scale)
    assert np.allclose(den, want_den, rtol=2e-6)
    assert np.allclose(num, want_num, rtol=2e-5, atol=2e-5 * np.abs(want_num).max())


def _tiny_case(rng, N=256, d=32, G=2, d_sel=8):
    q = _bf16(rng.standard_normal((1, G, d)))
    K = _bf16(rng.standard_normal((1, 1, N, d)))
    V = _bf16(rng.standard_normal((1, 1, N, d)))
    sel = np.arange(d_sel, dtype=np.int32)[None]
    Ks = oracle_mod_pack(K, sel, d_sel)
    return q, K, V, Ks, sel


def oracle_mod_pack(K, sel, d_sel):
    import oracle
    return oracle.pack_summary(K, sel, d_sel)


def test_budget_covering_remainder_is_dense(oracle_mod):
    rng = np.random.default_rng(2)
    q, K, V, Ks, sel = _tiny_case(rng)
    scale = 1 / math.sqrt(32)
    r = oracle_mod.decode(q, K, V, Ks, sel, 10, math.inf, 0, scale)
    out, lse = oracle_mod.dense_attention(q, K, V, scale)
    assert r["count"][0, 0] == 256
    assert np.allclose(r["out"], out, atol=1e-6) and np.allclose(r["lse"], lse, atol=1e-6)


def test_budget_zero_is_softmax_over_topk(oracle_mod):
    rng = np.random.default_rng(3)
    q, K, V, Ks, sel = _tiny_case(rng)
    scale = 1 / math.sqrt(32)
    k = 20
    r = oracle_mod.decode(q, K, V, Ks, sel, k, 0.0, 0, scale)
    s = r["s_hat"][0, 0]
    T = sorted(sorted(range(s.size), key=lambda i: (-float(s[i]), i))[:k])
    logits = scale * (_val(K)[0, 0][T] @ _val(q)[0].T)           # [k][G]
    w = torch.softmax(torch.from_numpy(logits), dim=0).numpy()
    want = w.T @ _val(V)[0, 0][T]
    assert r["count"][0, 0] == k
    assert np.allclose(r["out"][0], want, atol=1e-6)


def test_zero_query_on_summary_is_uniform_hybrid(oracle_mod):
    # q zero on the summary channels: every estimate is 0, T = the first k tokens and
    # the remainder is sampled uniformly with p = B/(N-k)
    rng = np.random.default_rng(4)
    q, K, V, Ks, sel = _tiny_case(rng)
    qv = q.copy()
    qv[..., :8] = 0
    k, B = 16, 24.0
    r = oracle_mod.decode(qv, K, V, Ks, sel, k, B, 3, 0.2)
    assert np.all(r["s_hat"] == 0)
    n = int(r["count"][0, 0])
    idx, p = r["idx"][0, 0, :n], r["p"][0, 0, :n]
    assert set(range(k)) <= set(idx.tolist())
    assert np.all(p[idx >= k] == np.float32(B) / np.float32(256 - k))


def test_monte_carlo_average_converges_to_dense(oracle_mod):
    # 10^4 seeds: the averaged corrected numerator and denominator approach the dense sums
    rng = np.random.default_rng(5)
    N, d, G, d_sel = 128, 16, 2, 8
    q, K, V, Ks, sel = _tiny_case(rng, N=N, d=d, G=G, d_sel=d_sel)
    scale = 0.25
    k, B = 8, 16.0
    want_num, want_den = _dense_sums(q[0], K[0, 0], V[0, 0], scale)
    seeds = 10_000
    nums = np.zeros((seeds, G, d))
    dens = np.zeros((seeds, G))
    for sd in range(seeds):
        r = oracle_mod.decode(q, K, V, Ks, sel, k, B, sd, scale, want_lists=False)
        w = np.exp(r["lse"][0].astype(np.float64))
        nums[sd] = w[:, None] * r["out"][0]
        dens[sd] = w
    for est, want in ((dens, want_den), (nums, want_num)):
        mean = est.mean(axis=0)
        se = est.std(axis=0, ddof=1) / math.sqrt(seeds)
        z = np.abs(mean - want) / np.maximum(se, 1e-12)
        assert np.all(z < 4.5), z.max()
