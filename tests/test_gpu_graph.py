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
