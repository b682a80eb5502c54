"""swa_step_host: forward + backward on host tensors, the copies overlapped
with the computation in head groups.  Heads are independent, so its results
must equal one swa_forward + swa_backward on device copies bit for bit."""
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


CASES = {
    "bnsd_b2_gqa_band": (dict(layout="BNSD", B=2, N=8, N_kv=4, D=128, S_q=300, S_kv=300, scale=0.09, sparse_mode=4,
                              pre_tokens=100, next_tokens=20), (1, 2, 4)),
    "tnd_varlen_nomask_d64": (dict(layout="TND", B=3, N=4, D=64, cu_seqlens_q=[130, 130, 400],
                                   cu_seqlens_kv=[130, 130, 400], scale=0.125, sparse_mode=0), (1, 4)),
    "bnsd_fp32_d72": (dict(layout="BNSD", B=1, N=4, D=72, S_q=200, S_kv=260, scale=72 ** -0.5, sparse_mode=4,
                           pre_tokens=50, next_tokens=80, dtype="fp32"), (2,)),
    # 3 and 6 chunks of 12 heads: split end groups around full ones (units
    # of 1, 1, 2, 4, 2, 1, 1 and of 1, 1, 2, 2, 2, 2, 1, 1 heads)
    "bnsd_n12_tapered": (dict(layout="BNSD", B=1, N=12, D=64, S_q=256, S_kv=256, scale=0.125, sparse_mode=4,
                              pre_tokens=90, next_tokens=30), (3, 6)),
    "bnsd_gendrop": (dict(layout="BNSD", B=1, N=2, D=64, S_q=256, S_kv=256, scale=0.125, sparse_mode=4,
                          pre_tokens=64, next_tokens=0, keep_prob=0.8, dropout_gen=1, dropout_seed=9,
                          dropout_offset=1), (1,)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_host_equals_device_path(name):
    kw, chunk_list = CASES[name]
    geom = Geometry(**kw)
    inp = draw(geom, 77)
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    out, smax, ssum = swa.forward(geom, q, k, v)
    dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum)
    torch.cuda.synchronize()
    ref = [t.cpu() for t in (out, smax, ssum, dq, dk, dv)]
    hq, hk, hv, hdy = (t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.dy))
    for chunks in chunk_list:
        got = [torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in ref]
        buf = swa.step_host(geom, hq, hk, hv, hdy, *got, chunks=chunks)
        torch.cuda.synchronize()
        swa.check_step_host(geom, chunks, buf)
        for label, a, b in zip(("out", "softmax_max", "softmax_sum", "dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), (name, chunks, label)


def test_step_host_rejects_bad_chunks():
    geom = Geometry("BNSD", 1, 6, 64, S_q=128, S_kv=128, sparse_mode=0)
    with pytest.raises(swa.SwaError) as e:
        swa.swa_step_host_buffer_size(swa.Params(geom), 4)
    assert e.value.status == swa.SWA_ERR_PARAM_INVALID
    drop = Geometry("BNSD", 1, 4, 64, S_q=128, S_kv=128, sparse_mode=0, keep_prob=0.9, dropout_gen=1)
    with pytest.raises(swa.SwaError):
        swa.swa_step_host_buffer_size(swa.Params(drop), 2)
    assert swa.swa_step_host_buffer_size(swa.Params(drop), 1) > 0


def test_concurrent_host_steps_share_the_internal_streams():
    """Two host threads call swa_step_host at once, each on its own stream,
    host tensors and device buffer, three times in a row.  The calls share
    the context's internal streams and events (their enqueueing is
    serialised, their GPU work runs one after the other): every result is
    the serial call's, bit for bit, and repeated calls reuse the events."""
    import threading

    kws = [dict(layout="BNSD", B=1, N=8, D=128, S_q=300, S_kv=300, scale=0.09, sparse_mode=4, pre_tokens=100,
                next_tokens=20),
           dict(layout="TND", B=3, N=4, D=64, cu_seqlens_q=[130, 130, 400], cu_seqlens_kv=[130, 130, 400],
                scale=0.125, sparse_mode=0)]
    chunks = [4, 2]
    geoms = [Geometry(**kw) for kw in kws]
    inputs = [draw(g, 78 + i) for i, g in enumerate(geoms)]
    hosts = [tuple(t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.dy)) for inp in inputs]

    def outputs(g, inp):
        st = tuple(g.stat_shape())
        return [torch.full(inp.q.shape, float("nan"), dtype=inp.q.dtype).pin_memory(),
                torch.full(st, float("nan")).pin_memory(), torch.full(st, float("nan")).pin_memory(),
                torch.full(inp.q.shape, float("nan"), dtype=inp.q.dtype).pin_memory(),
                torch.full(inp.k.shape, float("nan"), dtype=inp.k.dtype).pin_memory(),
                torch.full(inp.v.shape, float("nan"), dtype=inp.v.dtype).pin_memory()]

    serial = []
    for g, inp, h, c in zip(geoms, inputs, hosts, chunks):
        got = outputs(g, inp)
        buf = swa.step_host(g, *h, *got, chunks=c)
        torch.cuda.synchronize()
        swa.check_step_host(g, c, buf)
        serial.append(got)
    results = [[None] * 3 for _ in geoms]
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            buf = None
            for rep in range(3):
                got = outputs(geoms[t], inputs[t])
                buf = swa.step_host(geoms[t], *hosts[t], *got, chunks=chunks[t], device_buffer=buf, stream=stream)
                stream.synchronize()
                swa.check_step_host(geoms[t], chunks[t], buf, stream)
                results[t][rep] = got
        except Exception as e:  # surfaced below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(geoms))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(len(geoms)):
        for rep in range(3):
            for a, b, n in zip(results[t][rep], serial[t], ("out", "softmax_max", "softmax_sum", "dq", "dk", "dv")):
                assert torch.equal(a, b), (t, rep, n)
