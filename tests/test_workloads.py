"""The synthetic input recipe (CPU): the budget split the pages' numbers
follow, seeded determinism, and the structure the generator promises (summary
channels as whole RoPE pairs, outlier channels, sinks, needles, bf16 values)."""
import math

import torch

import workloads
from workloads.synthetic import _outlier_channels, budget_split

SMALL_ROPE = workloads.make_config("ministral8b_32k", batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=3000,
                                   top_k=30, budget=30.0, n_needles=8)


def test_budget_split_gives_the_printed_pairs():
    # total budget floor(N / 50), top-k the larger half: 328/327, 1311/1310, 10486/10485
    assert budget_split(32768, 50) == (328, 327.0)
    assert budget_split(131072, 50) == (1311, 1310.0)
    assert budget_split(1048576, 50) == (10486, 10485.0)
    for name, (k, B) in (("ministral8b_32k", (328, 327.0)), ("ministral8b_128k", (1311, 1310.0)),
                         ("ministral8b_1m", (10486, 10485.0)), ("27b_128k_10x", (6554, 6553.0)),
                         ("27b_128k_100x", (655, 655.0))):
        cfg = workloads.CONFIGS[name]
        assert (cfg.top_k, cfg.budget) == (k, B), name
    assert math.isinf(workloads.CONFIGS["27b_128k_dense"].budget)


def test_generation_is_seeded():
    a = workloads.generate(SMALL_ROPE, 3)
    b = workloads.generate(SMALL_ROPE, 3)
    c = workloads.generate(SMALL_ROPE, 4)
    for key in ("q", "K", "V", "sel_ch", "needles"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["K"], c["K"]) and not torch.equal(a["q"], c["q"])


def test_shapes_types_and_values():
    cfg = SMALL_ROPE
    w = workloads.generate(cfg, 0)
    assert w["q"].shape == (cfg.batch, cfg.n_q_heads, cfg.head_dim) and w["q"].dtype == torch.bfloat16
    assert w["K"].shape == (cfg.batch, cfg.n_kv_heads, cfg.ctx_len, cfg.head_dim) and w["K"].dtype == torch.bfloat16
    assert w["V"].shape == w["K"].shape and w["V"].dtype == torch.bfloat16
    assert w["sel_ch"].shape == (cfg.n_kv_heads, cfg.d_sel) and w["sel_ch"].dtype == torch.int32
    for t in (w["q"], w["K"], w["V"]):
        assert torch.isfinite(t.float()).all()
    v = w["V"].float()
    assert abs(float(v.mean())) < 0.02 and abs(float(v.std()) - 1.0) < 0.02


def test_summary_channels_are_whole_rope_pairs():
    cfg = SMALL_ROPE
    w = workloads.generate(cfg, 0)
    h = cfg.head_dim // 2
    for row in w["sel_ch"].tolist():
        assert row == sorted(row) and len(set(row)) == cfg.d_sel
        assert all(0 <= c < cfg.head_dim for c in row)
        low = [c for c in row if c < h]
        assert sorted(low + [c + h for c in low]) == row   # both channels of each chosen pair
    tiny = workloads.generate(workloads.CONFIGS["tiny"], 0)
    assert tiny["sel_ch"].tolist() == [list(range(16))]


def test_outlier_pairs_carry_the_energy_and_sinks_are_scaled():
    cfg = SMALL_ROPE
    K = workloads.generate(cfg, 1)["K"].float()
    h = cfg.head_dim // 2
    pair_energy = K[..., :h] ** 2 + K[..., h:] ** 2          # invariant under the RoPE rotation
    e = pair_energy.mean(dim=(0, 1, 2))
    out = [c for c in _outlier_channels(cfg.head_dim) if c < h]
    rest = [j for j in range(h) if j not in out]
    assert float(e[out].min()) > 20 * float(e[rest].max())    # x5 in amplitude: ~x25 in energy
    tiny = workloads.generate(workloads.CONFIGS["tiny"], 0)["K"].float()[0, 0]
    assert float(tiny[:4].pow(2).mean()) > 2.5 * float(tiny[4:].pow(2).mean())   # sinks x2 in amplitude


def test_needles_are_planted_where_promised():
    cfg = SMALL_ROPE
    w = workloads.generate(cfg, 2)
    nd = w["needles"]
    assert nd.shape == (cfg.batch, cfg.n_kv_heads, cfg.n_needles)
    for row in nd.reshape(-1, cfg.n_needles).tolist():
        assert row == sorted(row) and len(set(row)) == len(row) and 0 <= row[0] and row[-1] < cfg.ctx_len
    even = workloads.make_config("ministral8b_1m", batch=1, n_q_heads=8, n_kv_heads=1, ctx_len=4096,
                                 n_needles=8, top_k=40, budget=40.0)
    pos = workloads.generate(even, 0)["needles"][0, 0].tolist()
    assert pos == [int((j + 0.5) * 4096 / 8) for j in range(8)]
    tiny = workloads.generate(workloads.CONFIGS["tiny"], 0)["needles"][0, 0]
    assert int(tiny.min()) >= 4   # after the sinks


def test_to_paged_places_every_token_in_its_page():
    """The paged layout helper: token t of sequence b is slot t % page_size of page block_table[b][t // page_size]
    in every pool, each pool page belongs to at most one sequence, and the block-table entries past a
    sequence's pages hold an id outside the pool."""
    import torch
    import workloads
    g = torch.Generator().manual_seed(0)
    Bt, Hkv, N, d, ds = 3, 2, 300, 16, 8
    K = torch.randn((Bt, Hkv, N, d), generator=g).to(torch.bfloat16)
    V = torch.randn((Bt, Hkv, N, d), generator=g).to(torch.bfloat16)
    Ks = torch.randn((Bt, Hkv, N, ds), generator=g).to(torch.bfloat16)
    lens = [N, 37, 0]
    for ps in (16, 64, 512):
        pg = workloads.to_paged(K, V, Ks, lens, ps, seed=1)
        bt = pg["block_table"]
        num_pages = pg["K_pool"].shape[0]
        used = []
        for b, n in enumerate(lens):
            need = (n + ps - 1) // ps
            for t in range(n):
                page, slot = int(bt[b, t // ps]), t % ps
                assert torch.equal(pg["K_pool"][page, :, slot], K[b, :, t])
                assert torch.equal(pg["V_pool"][page, :, slot], V[b, :, t])
                assert torch.equal(pg["Ks_pool"][page, :, slot], Ks[b, :, t])
            used += [int(x) for x in bt[b, :need]]
            assert all(int(x) >= num_pages for x in bt[b, need:])
        assert len(used) == len(set(used)) and all(0 <= x < num_pages for x in used)
        assert pg["seq_lens"].tolist() == lens
