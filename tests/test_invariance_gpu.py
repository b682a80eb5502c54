"""Invariances of the CUDA path, checked bit for bit between two calls.

The oracle pins the same identities on the CPU (tests/test_oracle_pins.py);
here they hold for the kernels themselves, whose tile schedule, masking and
reduction order must not depend on how an equivalent problem is written:
- a BAND wider than the sequence in both directions is no mask;
- one TND sequence is the BNSD problem of the same length;
- a batch of two is two calls with a batch of one;
- query heads sharing a key/value head (N_kv < N) are the heads of a problem
  with that head repeated: identical forward and dQ, and dK / dV equal to the
  sums over the group up to the bf16 rounding of each head's result.
"""
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    swa.lib()


def run(geom, q, k, v, dy, mask=None):
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (q, k, v, dy))
    m = mask.to(dev) if mask is not None else None
    out, smax, ssum = swa.forward(geom, q, k, v, m)
    ws = torch.empty(swa.swa_backward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
    dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum, m, workspace=ws)
    swa.check_workspace(ws)
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in (("out", out), ("smax", smax), ("ssum", ssum), ("dq", dq), ("dk", dk), ("dv", dv))}


def same(a, b, names=("out", "smax", "ssum", "dq", "dk", "dv"), label=""):
    for n in names:
        assert torch.equal(a[n], b[n]), (label, n)


@pytest.mark.parametrize("D", [64, 128])
def test_wide_band_is_no_mask(D):
    S = 333
    base = dict(layout="BNSD", B=1, N=2, D=D, S_q=S, S_kv=S, scale=D ** -0.5)
    g0 = Geometry(**base, sparse_mode=0)
    g4 = Geometry(**base, sparse_mode=4, pre_tokens=S, next_tokens=S + 5)
    inp = draw(g0, 71)
    same(run(g0, inp.q, inp.k, inp.v, inp.dy), run(g4, inp.q, inp.k, inp.v, inp.dy), label=f"D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_tnd_sequence_is_bnsd(D):
    S, N = 517, 3
    gb = Geometry(layout="BNSD", B=1, N=N, D=D, S_q=S, S_kv=S, scale=D ** -0.5, sparse_mode=4, pre_tokens=200,
                  next_tokens=30)
    gt = Geometry(layout="TND", B=1, N=N, D=D, cu_seqlens_q=[S], cu_seqlens_kv=[S], scale=D ** -0.5, sparse_mode=4,
                  pre_tokens=200, next_tokens=30)
    inp = draw(gb, 72)
    rb = run(gb, inp.q, inp.k, inp.v, inp.dy)
    # [1, N, S, D] -> [S, N, D]; statistics [1, N, S] -> [S, N]
    t = lambda x: x[0].transpose(0, 1).contiguous()
    rt = run(gt, t(inp.q), t(inp.k), t(inp.v), t(inp.dy))
    for n in ("out", "dq", "dk", "dv"):
        assert torch.equal(t(rb[n]), rt[n]), n
    for n in ("smax", "ssum"):
        assert torch.equal(rb[n][0].transpose(0, 1), rt[n]), n


def test_batch_of_two_is_two_calls():
    kw = dict(layout="BNSD", N=2, D=128, S_q=300, S_kv=300, scale=0.09, sparse_mode=4, pre_tokens=120, next_tokens=7)
    g2 = Geometry(B=2, **kw)
    g1 = Geometry(B=1, **kw)
    inp = draw(g2, 73)
    r2 = run(g2, inp.q, inp.k, inp.v, inp.dy)
    for b in range(2):
        r1 = run(g1, inp.q[b:b + 1], inp.k[b:b + 1], inp.v[b:b + 1], inp.dy[b:b + 1])
        for n in r1:
            assert torch.equal(r2[n][b:b + 1], r1[n]), (b, n)


@pytest.mark.parametrize("D", [64, 128])
def test_grouped_heads_are_repeated_heads(D):
    N, N_kv, S = 4, 2, 290
    kw = dict(layout="BNSD", B=1, D=D, S_q=S, S_kv=S, scale=D ** -0.5, sparse_mode=4, pre_tokens=150, next_tokens=40)
    gg = Geometry(N=N, N_kv=N_kv, **kw)
    gr = Geometry(N=N, **kw)
    inp = draw(gg, 74)
    rg = run(gg, inp.q, inp.k, inp.v, inp.dy)
    group = N // N_kv
    rep = lambda x: x.repeat_interleave(group, dim=1)  # query head n reads key/value head n // group
    rr = run(gr, inp.q, rep(inp.k), rep(inp.v), inp.dy)
    same(rg, rr, names=("out", "smax", "ssum", "dq"))
    for n in ("dk", "dv"):
        per_head = rr[n].float().reshape(1, N_kv, group, S, D)
        summed = per_head.sum(dim=2)
        got = rg[n].float()
        # the grouped pass sums the heads in fp32 and rounds once; the
        # repeated problem rounds every head's result to bf16 first.  Their
        # difference is bounded by those roundings: half an ulp (2^-9
        # relative) of each head's value and of the grouped value, doubled
        # for margin
        tol = 2.0 ** -8 * (per_head.abs().sum(dim=2) + got.abs()) + 1e-6
        assert torch.all((got - summed).abs() <= tol), n
