"""Forward + backward captured into a CUDA graph and replayed.

The calls only enqueue work on the caller's stream, so a training step can
be captured once and replayed.  The backward's three kernels are launched
with programmatic stream serialization, which capture turns into
programmatic graph edges.  Replays must reproduce the eager results bit for
bit (every kernel is deterministic), through the one-tile forward (D = 128)
and the forward one CTA per pair of query tiles (D = 64, forced on these
small problems), with and without generated dropout.
"""
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw

pytestmark = pytest.mark.gpu

CASES = {
    "bnsd_d128_band": (dict(layout="BNSD", B=2, N=3, D=128, S_q=700, S_kv=700, scale=128 ** -0.5, sparse_mode=4,
                            pre_tokens=200, next_tokens=20), 0),
    "bnsd_d64_band_pairs": (dict(layout="BNSD", B=1, N=4, D=64, S_q=600, S_kv=600, scale=0.125, sparse_mode=4,
                                 pre_tokens=150, next_tokens=40), 1),
    "tnd_d64_gen_dropout_pairs": (dict(layout="TND", B=3, N=2, D=64, cu_seqlens_q=[300, 300, 750],
                                       cu_seqlens_kv=[300, 300, 750], scale=0.125, sparse_mode=4, pre_tokens=90,
                                       next_tokens=10, keep_prob=0.85, dropout_gen=1, dropout_seed=5,
                                       dropout_offset=2), 1),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    swa.lib()


@pytest.mark.parametrize("name", sorted(CASES))
def test_graph_replay_matches_eager(name):
    kw, pairs = CASES[name]
    geom = Geometry(**kw)
    inp = draw(geom, 4242)
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    p = swa.Params(geom)
    ws_f = torch.empty(swa.swa_forward_workspace_size(p), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(swa.swa_backward_workspace_size(p), dtype=torch.uint8, device=dev)
    swa.swa_debug_forward_pairs(pairs)
    try:
        # eager reference
        out, smax, ssum = swa.forward(geom, q, k, v, mask)
        dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum, mask)
        torch.cuda.synchronize()
        ref = (out, smax, ssum, dq, dk, dv)
        got = [torch.empty_like(t) for t in ref]

        def step(stream):
            swa.forward(geom, q, k, v, mask, got[0], got[1], got[2], ws_f, stream)
            swa.backward(geom, q, k, v, dy, got[0], got[1], got[2], mask, got[3], got[4], got[5], ws_b, stream)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # one call outside capture first
            step(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(torch.cuda.current_stream())
        for t in got:
            t.zero_()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    finally:
        swa.swa_debug_forward_pairs(0)
    swa.check_workspace(ws_f)
    swa.check_workspace(ws_b)
    for label, a, b in zip(("out", "softmax_max", "softmax_sum", "dq", "dk", "dv"), got, ref):
        assert torch.equal(a, b), (name, label)
