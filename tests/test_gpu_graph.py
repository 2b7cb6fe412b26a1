"""The decode step captured in a CUDA graph (the launch form a serving loop
uses: one replay per token, inputs updated in place) gives, bit for bit, what
the eager calls give, including when the query changes between replays."""
import pytest
import torch

import long_context_decode_subset_b300 as ssa
from test_gpu_stages import case

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.contiguous().view(torch.int32)


@pytest.mark.parametrize("name", ["tiny", "g4_d128"])
def test_decode_graph_replay_matches_eager(name):
    w = case(name)
    cfg = w["cfg"]
    q = w["q"].clone()
    K, V, Ks, sel = w["K"], w["V"], w["Ks"], w["sel_ch"]
    shape = ssa.shape_of(q, K, Ks)
    ws = ssa.workspace(shape, 0, DEV)
    Bt, Hq, d = q.shape
    out = torch.empty((Bt, Hq, d), dtype=torch.float32, device=DEV)
    lse = torch.empty((Bt, Hq), dtype=torch.float32, device=DEV)
    q2 = torch.roll(w["q"], shifts=1, dims=1).contiguous()   # another query, same shapes

    ref1 = ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 5, cfg.scale, ws=ws)
    ref2 = ssa.ssa_decode(q2, K, V, Ks, sel, cfg.top_k, cfg.budget, 5, cfg.scale, ws=ws)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up on the capture's stream kind
        ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 5, cfg.scale, out=out, lse=lse, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ssa.ssa_decode(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 5, cfg.scale, out=out, lse=lse, ws=ws)

    out.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref1[0])) and torch.equal(_bits(lse), _bits(ref1[1]))

    q.copy_(q2)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref2[0])) and torch.equal(_bits(lse), _bits(ref2[1]))

    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref2[0]))
    st, flags = ssa.ssa_get_device_status(ws)
    assert st == 0, hex(flags)


def test_paged_graph_replay_with_lengths_updated_in_place():
    """The paged step in a graph: the query and the sequence lengths change in place between replays (the
    serving loop's form: the block table and lengths live on the device), and every replay gives the eager
    result for its inputs."""
    import workloads
    w = case("g4_d128")
    cfg = w["cfg"]
    N = cfg.ctx_len
    pg = workloads.to_paged(w["K"], w["V"], w["Ks"], [N] * cfg.batch, 64, seed=2)
    q = w["q"].clone()
    args = (pg["K_pool"], pg["V_pool"], pg["Ks_pool"], pg["block_table"], pg["seq_lens"], w["sel_ch"], cfg.top_k,
            cfg.budget, 5, cfg.scale, N)
    shape = ssa.paged_shape(q, pg["K_pool"], pg["Ks_pool"], N)
    ws = ssa.workspace(shape, 0, DEV)
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device=DEV)
    lse = torch.empty((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=DEV)
    steps = [(q.clone(), [N, N]), (torch.roll(q, 1, dims=1).contiguous(), [N - 700, N]), (q.clone(), [1000, 17])]
    refs = []
    for qq, lens in steps:
        pg["seq_lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        refs.append(tuple(t.clone() for t in ssa.ssa_decode_paged(qq, *args)))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ssa.ssa_decode_paged(q, *args, out=out, lse=lse, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ssa.ssa_decode_paged(q, *args, out=out, lse=lse, ws=ws)
    for (qq, lens), (r_out, r_lse) in zip(steps, refs):
        q.copy_(qq)
        pg["seq_lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_bits(out), _bits(r_out)) and torch.equal(_bits(lse), _bits(r_lse)), lens


def test_early_stop_graph_replay_matches_eager():
    w = case("g4_d128")
    cfg = w["cfg"]
    q, K, V, Ks, sel = w["q"], w["K"], w["V"], w["Ks"], w["sel_ch"]
    ws = ssa.workspace(ssa.shape_of(q, K, Ks), 0, DEV)
    ref = ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 4, cfg.scale, 0.05)
    out = torch.empty_like(ref[0])
    lse = torch.empty_like(ref[1])
    blocks = torch.empty_like(ref[2])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 4, cfg.scale, 0.05, out=out, lse=lse,
                                  blocks=blocks, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ssa.ssa_decode_early_stop(q, K, V, Ks, sel, cfg.top_k, cfg.budget, 4, cfg.scale, 0.05, out=out, lse=lse,
                                  blocks=blocks, ws=ws)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref[0])) and torch.equal(_bits(lse), _bits(ref[1]))
    assert torch.equal(blocks, ref[2])
