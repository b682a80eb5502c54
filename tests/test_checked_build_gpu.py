"""The bounds-checked build, libswa_checked.so (SWA_CHECKS = 1).

Its kernels test every global load and store against the extent of the
caller's tensor before making it; an access outside it is skipped and the
call's status word reports SWA_ERR_BOUNDS instead of a memory fault.  Two
things are checked here:
- on cases that reach every kernel variant (both layouts, one-tile and pair
  forward, the preprocess at exact and padded head dims, stored and generated dropout, each
  element type, GQA, the head-group host step and the no-alloc backward)
  the checked build finds no access outside its tensor and computes the
  release build's results bit for bit: the checks only skip, they change no
  arithmetic;
- with swa_debug_extent_slack taking 8 elements off every extent, in-range
  accesses at the tensors' ends count as outside and the status is
  SWA_ERR_BOUNDS, for the forward and for the backward, while the release
  build, which has no checks, ignores the hook;
- at the full size of each of the five workloads, and on the seeded random
  geometries of the parity sweep (tests/test_parity_random_gpu.py), the
  checked build records nothing and matches the release build bit for bit.
"""
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import WORKLOAD_ORDER, Geometry, draw, workload_geometry

pytestmark = pytest.mark.gpu

NAMES = ("out", "smax", "ssum", "dq", "dk", "dv")


@pytest.fixture(scope="module", autouse=True)
def libs():
    B.build()
    B.build(checked=True)
    return swa.lib(), swa.checked_lib()


def run(geom, inp):
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    fws = torch.empty(swa.swa_forward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
    out, smax, ssum = swa.forward(geom, q, k, v, mask, workspace=fws)
    swa.check_workspace(fws)
    bws = torch.empty(swa.swa_backward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
    dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum, mask, workspace=bws)
    swa.check_workspace(bws)
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in zip(NAMES, (out, smax, ssum, dq, dk, dv))}


CASES = {
    # D = 128: one-tile forward, wide preprocess
    "bnsd_d128_band": dict(layout="BNSD", B=2, N=2, D=128, S_q=390, S_kv=390, scale=0.088, sparse_mode=4,
                           pre_tokens=150, next_tokens=20),
    # D = 64 GQA with a stored mask over ragged sequences (one empty)
    "tnd_d64_gqa_mask": dict(layout="TND", B=4, N=4, N_kv=2, D=64, cu_seqlens_q=[200, 200, 531, 700],
                             cu_seqlens_kv=[150, 150, 600, 777], scale=0.125, sparse_mode=4, pre_tokens=96,
                             next_tokens=40, keep_prob=0.9),
    # D = 40: the preprocess with lanes past D idle, fp32 storage, generated dropout
    "bnsd_d40_fp32_gendrop": dict(layout="BNSD", B=1, N=3, D=40, S_q=333, S_kv=270, scale=40 ** -0.5,
                                  sparse_mode=0, keep_prob=0.85, dropout_gen=1, dropout_seed=3, dropout_offset=7,
                                  dtype="fp32"),
    # fp16, BAND with a negative edge
    "bnsd_d96_fp16": dict(layout="BNSD", B=1, N=2, D=96, S_q=300, S_kv=300, scale=96 ** -0.5, sparse_mode=4,
                          pre_tokens=-20, next_tokens=120, dtype="fp16"),
}


# every case as the host chooses its forward; the D <= 64 ones also with the pair forward forced
RUNS = [(n, 0) for n in sorted(CASES)] + [(n, 1) for n in sorted(CASES) if CASES[n]["D"] <= 64]


@pytest.mark.parametrize("name,pairs", RUNS)
def test_checked_build_matches_release_without_bounds_errors(name, pairs, libs):
    geom = Geometry(**CASES[name])
    inp = draw(geom, 81)
    res = []
    for library in libs:
        with swa.using(library):
            swa.swa_debug_forward_pairs(pairs)
            try:
                res.append(run(geom, inp))  # check_workspace raises on SWA_ERR_BOUNDS
            finally:
                swa.swa_debug_forward_pairs(0)
    for n in NAMES:
        assert torch.equal(res[0][n], res[1][n]), (name, pairs, n)


def test_checked_build_host_step_and_noalloc_match_release(libs):
    # no dropout: the host step in head groups takes neither a stored mask
    # nor, with more than one group, generated bits
    geom = Geometry(layout="BNSD", B=1, N=6, D=64, S_q=256, S_kv=256, scale=0.125, sparse_mode=4, pre_tokens=90,
                    next_tokens=30)
    inp = draw(geom, 82)
    dev = torch.device("cuda:0")
    hq, hk, hv, hdy = (t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.dy))
    res = []
    for library in libs:
        with swa.using(library):
            ref = run(geom, inp)
            got = [torch.full(ref[n].shape, float("nan"), dtype=ref[n].dtype).pin_memory() for n in NAMES]
            buf = swa.step_host(geom, hq, hk, hv, hdy, *got, chunks=3)
            torch.cuda.synchronize()
            swa.check_step_host(geom, 3, buf)
            t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "dy")}
            o, m, s = (ref[n].to(dev) for n in ("out", "smax", "ssum"))
            dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
            st = swa.swa_backward_noalloc(swa.Params(geom), t["q"].data_ptr(), t["k"].data_ptr(),
                                          t["v"].data_ptr(), t["dy"].data_ptr(), o.data_ptr(), m.data_ptr(),
                                          s.data_ptr(), None, dq.data_ptr(), dk.data_ptr(),
                                          dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
            assert st == swa.SWA_OK, swa.swa_last_error()
            torch.cuda.synchronize()
            res.append((ref, got, [x.cpu() for x in (dq, dk, dv)]))
    (ref0, host0, na0), (ref1, host1, na1) = res
    for n in NAMES:
        assert torch.equal(ref0[n], ref1[n]), n
    for a, b, n in zip(host0, host1, NAMES):
        assert torch.equal(a, b), ("host step", n)
    for a, b, n in zip(na0, na1, ("dq", "dk", "dv")):
        assert torch.equal(a, b), ("no-alloc", n)


def test_extent_slack_reports_bounds_errors_in_the_checked_build_only(libs):
    geom = Geometry(layout="BNSD", B=1, N=2, D=64, S_q=200, S_kv=200, scale=0.125, sparse_mode=4, pre_tokens=64,
                    next_tokens=16, keep_prob=0.9)
    inp = draw(geom, 83)
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask.to(dev)
    release, checked = libs
    clean = {}
    for library in libs:
        with swa.using(library):
            clean[id(library)] = run(geom, inp)
    # forward: the last row's last chunk of out and the last statistics fall outside the shortened extents
    with swa.using(checked):
        swa.swa_debug_extent_slack(8)
        try:
            fws = torch.empty(swa.swa_forward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
            swa.forward(geom, q, k, v, mask, workspace=fws)
            with pytest.raises(swa.SwaError) as e:
                swa.check_workspace(fws)
            assert e.value.status == swa.SWA_ERR_BOUNDS
            # backward on a clean forward: the preprocess's reads of the last row of dY and O fall outside
            swa.swa_debug_extent_slack(0)
            out, smax, ssum = swa.forward(geom, q, k, v, mask)
            swa.swa_debug_extent_slack(8)
            bws = torch.empty(swa.swa_backward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
            swa.backward(geom, q, k, v, dy, out, smax, ssum, mask, workspace=bws)
            with pytest.raises(swa.SwaError) as e:
                swa.check_workspace(bws)
            assert e.value.status == swa.SWA_ERR_BOUNDS
        finally:
            swa.swa_debug_extent_slack(0)
        # the next call without slack starts from a clear status word
        again = run(geom, inp)
    for n in NAMES:
        assert torch.equal(again[n], clean[id(checked)][n]), n
    # the release build has no checks: the hook changes nothing
    with swa.using(release):
        swa.swa_debug_extent_slack(8)
        try:
            got = run(geom, inp)
        finally:
            swa.swa_debug_extent_slack(0)
    for n in NAMES:
        assert torch.equal(got[n], clean[id(release)][n]), n


# ------------------------------------------------- full-size workloads -----
def _device_inputs(geom, seed, dev):
    """Seeded device tensors of geom's shapes (values do not matter here:
    every access the kernels make depends on the shapes alone)."""
    g = torch.Generator(dev).manual_seed(seed)
    q = torch.randn(geom.q_shape(), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn(geom.kv_shape(), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(geom.kv_shape(), generator=g, device=dev).to(torch.bfloat16)
    dy = torch.randn(geom.q_shape(), generator=g, device=dev).to(torch.bfloat16)
    mask = None
    if geom.keep_prob < 1.0 and not geom.dropout_gen:
        nbytes = (geom.mask_bits() + 7) // 8
        mask = torch.randint(0, 256, (nbytes,), generator=g, device=dev, dtype=torch.uint8)
    return q, k, v, dy, mask


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_full_size_workloads_stay_in_bounds(name, libs):
    """At each workload's full size (the largest offsets the kernels form),
    the checked build records no access outside its tensor and matches the
    release build bit for bit."""
    geom = workload_geometry(name)
    dev = torch.device("cuda:0")
    q, k, v, dy, mask = _device_inputs(geom, 91, dev)
    res = []
    for library in libs:
        with swa.using(library):
            fws = torch.empty(swa.swa_forward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
            out, smax, ssum = swa.forward(geom, q, k, v, mask, workspace=fws)
            swa.check_workspace(fws)
            bws = torch.empty(swa.swa_backward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
            dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum, mask, workspace=bws)
            swa.check_workspace(bws)
            res.append((out, smax, ssum, dq, dk, dv))
            del fws, bws
    for n, a, b in zip(NAMES, *res):
        assert torch.equal(a, b), (name, n)


# ------------------------------------------ the random geometries ------
def _random_kws():
    from tests.test_parity_random_gpu import EXTREME, N_CASES, extreme_geometry, random_geometry
    kws = [(f"random{s}", random_geometry(s)) for s in range(N_CASES)]
    kws += [(f"extreme{s}", extreme_geometry(s)) for s in range(16)]
    kws += sorted(EXTREME.items())
    return kws


_RANDOM = dict(_random_kws())


@pytest.mark.parametrize("name", list(_RANDOM))
def test_random_geometries_stay_in_bounds(name, libs):
    """The seeded random geometries of the parity sweep (empty and ragged
    TND sequences, GQA / MQA, every head dim, both masks and dropout forms,
    every element type, scales and key counts outside the workloads'
    regime): no bounds error in the checked build, the release build's bits."""
    geom = Geometry(**_RANDOM[name])
    inp = draw(geom, 97_000 + sum(map(ord, name)))
    res = []
    for library in libs:
        with swa.using(library):
            res.append(run(inp.geom, inp))
    for n in NAMES:
        assert torch.equal(res[0][n], res[1][n]), (name, n)
