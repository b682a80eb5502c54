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


PAIR_CASES = {
    "band": dict(layout="BNSD", B=2, N=2, D=64, S_q=700, S_kv=700, scale=0.125, sparse_mode=4, pre_tokens=300,
                 next_tokens=40),
    "mask_dropout": dict(layout="BNSD", B=1, N=3, D=64, S_q=520, S_kv=520, scale=0.125, sparse_mode=4, pre_tokens=256,
                         next_tokens=256, keep_prob=0.9),
    "gen_dropout_tnd": dict(layout="TND", B=3, N=2, D=64, cu_seqlens_q=[300, 300, 750], cu_seqlens_kv=[300, 300, 750],
                            scale=0.125, sparse_mode=4, pre_tokens=90, next_tokens=10, keep_prob=0.85, dropout_gen=1,
                            dropout_seed=5, dropout_offset=2),
}


@pytest.mark.parametrize("name", sorted(PAIR_CASES))
def test_pair_forward_is_one_tile_forward(name):
    """At D <= 64 the forward over pairs of query tiles computes every row
    with the same operations in the same order as one CTA per tile."""
    geom = Geometry(**PAIR_CASES[name])
    inp = draw(geom, 75)
    res = []
    for mode in (1, 2):  # always pairs, never pairs
        swa.swa_debug_forward_pairs(mode)
        try:
            res.append(run(geom, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask))
        finally:
            swa.swa_debug_forward_pairs(0)
    same(res[0], res[1], label=name)


@pytest.mark.parametrize("D", [64, 128])
def test_fp32_storage_of_bf16_values_is_the_bf16_path(D):
    """fp32 inputs are rounded to bf16 once and computed like bf16 inputs in
    fp32: inputs that already are bf16 values give the bf16 path's results,
    once the fp32 outputs are rounded to bf16 (round to nearest even)."""
    kw = dict(layout="BNSD", B=1, N=2, D=D, S_q=333, S_kv=333, scale=D ** -0.5, sparse_mode=4, pre_tokens=150,
              next_tokens=20, keep_prob=0.9)
    g16 = Geometry(**kw)
    g32 = Geometry(**kw, dtype="fp32")
    inp = draw(g16, 76)
    r16 = run(g16, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    f = lambda x: x.to(torch.float32)
    r32 = run(g32, f(inp.q), f(inp.k), f(inp.v), f(inp.dy), inp.drop_mask)
    for n in ("out", "dq", "dk", "dv"):
        assert r32[n].dtype == torch.float32
        assert torch.equal(r32[n].to(torch.bfloat16), r16[n]), n
    same(r16, r32, names=("smax", "ssum"))


def test_concurrent_calls_on_two_streams_match_serial_calls():
    """Two host threads, each with its own stream, call forward + backward
    at the same time (the binding's calls release the interpreter lock):
    each gets exactly the results of a serial call.  The library keeps no
    shared mutable state between calls beyond once-only kernel attributes."""
    import threading

    geoms = [Geometry(layout="BNSD", B=1, N=3, D=128, S_q=600, S_kv=600, scale=0.09, sparse_mode=4, pre_tokens=200,
                      next_tokens=10),
             Geometry(layout="TND", B=3, N=2, D=64, cu_seqlens_q=[300, 300, 750], cu_seqlens_kv=[300, 300, 750],
                      scale=0.125, sparse_mode=4, pre_tokens=90, next_tokens=10, keep_prob=0.85, dropout_gen=1,
                      dropout_seed=5, dropout_offset=2)]
    inputs = [draw(g, 77 + i) for i, g in enumerate(geoms)]
    serial = [run(inp.geom, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask) for inp in inputs]
    results = [[None] * 4 for _ in inputs]
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for rep in range(4):
                    inp = inputs[t]
                    results[t][rep] = run(inp.geom, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
        except Exception as e:  # surfaced below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(inputs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(len(inputs)):
        for rep in range(4):
            same(results[t][rep], serial[t], label=f"thread {t} call {rep}")
