"""Pins for the oracle's key summary and approximate score.

Score (FASA, section 3, Stage 1, restricted to the summary channels; GQA
group combined by max): s_i = fl32(scale * max_g sum_j q_g[S_ch[j]] Ks[i][j]).
"""
import numpy as np
import torch


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_pack_summary_is_channel_gather(oracle_mod):
    rng = np.random.default_rng(0)
    K = _bf16(rng.standard_normal((2, 3, 37, 64)))
    sel = np.stack([rng.choice(64, 16, replace=False) for _ in range(3)]).astype(np.int32)
    Ks = oracle_mod.pack_summary(K, sel, 16)
    for h in range(3):
        assert np.array_equal(Ks[:, h], K[:, h][:, :, sel[h]])


def test_score_one_hot_keys_closed_form(oracle_mod):
    # key i has a single non-zero summary channel c_i with value v_i: s_i = scale*max_g q_g[S[c_i]]*v_i
    rng = np.random.default_rng(1)
    Bt, Hq, Hkv, d, d_sel, N = 1, 4, 1, 64, 16, 50
    q = _bf16(rng.standard_normal((Bt, Hq, d)))
    sel = np.arange(3, 3 + d_sel, dtype=np.int32)[None]
    Ks = np.zeros((Bt, Hkv, N, d_sel), np.uint16)
    c = rng.integers(0, d_sel, N)
    v = _bf16(rng.standard_normal(N))
    Ks[0, 0, np.arange(N), c] = v
    scale = 0.125
    s = oracle_mod.score(q, Ks, sel, scale)
    qv = _val(q)[0]
    want = np.array([np.float32(scale * max(float(qv[g, sel[0, c[i]]]) * float(_val(v[i])) for g in range(Hq)))
                     for i in range(N)], np.float32)
    assert np.array_equal(s[0, 0], want)


def test_score_all_channels_equals_group_max_of_dense_logits(oracle_mod):
    # with S_ch = every channel the estimate is the exact logit, max over the group
    rng = np.random.default_rng(2)
    Bt, Hq, Hkv, d, N = 2, 8, 2, 32, 200
    G = Hq // Hkv
    q = _bf16(rng.standard_normal((Bt, Hq, d)))
    K = _bf16(rng.standard_normal((Bt, Hkv, N, d)))
    sel = np.tile(np.arange(d, dtype=np.int32), (Hkv, 1))
    Ks = oracle_mod.pack_summary(K, sel, d)
    scale = float(np.float32(1 / np.sqrt(d)))
    s = oracle_mod.score(q, Ks, sel, scale)
    qt = torch.from_numpy(_val(q).astype(np.float64)).view(Bt, Hkv, G, d)
    kt = torch.from_numpy(_val(K).astype(np.float64))
    logits = torch.matmul(qt, kt.transpose(-1, -2))          # [Bt][Hkv][G][N]
    want = (scale * logits.max(dim=2).values).to(torch.float32).numpy()
    assert np.array_equal(s, want)


def test_score_group_max_picks_the_right_head(oracle_mod):
    # two heads with opposite signs: the max is |.| for every key
    d, d_sel, N = 64, 16, 30
    rng = np.random.default_rng(3)
    base = rng.standard_normal(d)
    q = _bf16(np.stack([base, -base])[None])
    K = _bf16(rng.standard_normal((1, 1, N, d)))
    sel = np.arange(d_sel, dtype=np.int32)[None]
    Ks = oracle_mod.pack_summary(K, sel, d_sel)
    s = oracle_mod.score(q, Ks, sel, 1.0)
    dots = (_val(Ks)[0, 0].astype(np.float64) @ _val(q)[0, 0, :d_sel].astype(np.float64))
    assert np.array_equal(s[0, 0], np.abs(dots).astype(np.float32))
