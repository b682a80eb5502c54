"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports
every symbol include/swa.h declares, the ctypes mirror matches the C struct,
and every argument check returns its documented status code before any CUDA
work is enqueued."""
import ctypes
import os
import re
import subprocess

import pytest

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import WORKLOADS, Geometry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return swa.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "swa.h")).read()
    return sorted(set(re.findall(r"SWA_API\s+[\w\s\*]+?\b(swa_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert declared, "no declarations found"
    out = subprocess.run(["nm", "-D", "--defined-only", swa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (swa_\w+)", out))
    assert set(declared) == exported, (declared, exported)
    for name in declared:
        assert hasattr(lib, name)
    assert sorted(swa.exported_symbols()) == declared


def test_workload_geometry_is_the_drawn_geometry():
    """workload_geometry() gives the sequence lengths draw_workload() draws
    (checked on a head dim of 8, which leaves the length draw unchanged)."""
    from attention_swa_forward_gb300.workloads import WORKLOADS, draw, workload_geometry
    for name, w in WORKLOADS.items():
        g = workload_geometry(name)
        if w.lengths is None:
            assert g is w.geom
            continue
        small = Geometry(**{**w.geom.as_dict(), "D": 8})
        drawn = draw(small, w.seed, w.lengths, with_dy=False).geom
        assert g.cu_seqlens_q == drawn.cu_seqlens_q and g.cu_seqlens_kv == drawn.cu_seqlens_kv
        assert g.D == w.geom.D and g.B == w.lengths[0]


def test_checked_build_exports_the_same_symbols():
    """The bounds-checked build (SWA_CHECKS=1) compiles from the same sources
    and loads with the same C ABI; only its kernels differ."""
    path = B.build(checked=True)
    assert path == swa.CHECKED_LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    assert sorted(set(re.findall(r" T (swa_\w+)", out))) == _declared_symbols()
    checked = swa.checked_lib()
    assert checked is not swa.lib()
    with swa.using(checked):
        assert swa.lib() is checked
        p = swa.Params(Geometry("BNSD", 1, 2, 64, S_q=300, S_kv=300, sparse_mode=0))
        assert swa.swa_backward_workspace_size(p) > 0
    assert swa.lib() is not checked


def test_library_choice_is_per_thread_and_restored():
    """using() routes only the calling thread, nests, and restores the
    previous choice on exit, also when the body raises."""
    import threading

    release = swa.lib()
    B.build(checked=True)
    checked = swa.checked_lib()
    seen = []
    with swa.using(checked):
        t = threading.Thread(target=lambda: seen.append(swa.lib()))
        t.start()
        t.join()
        with swa.using(release):
            assert swa.lib() is release
        assert swa.lib() is checked
    assert seen == [release]
    with pytest.raises(RuntimeError):
        with swa.using(checked):
            raise RuntimeError("inside")
    assert swa.lib() is release


def test_ctypes_struct_matches_c_layout(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "swa.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(swa_params_t),"
        " offsetof(swa_params_t, B), offsetof(swa_params_t, cu_seqlens_q), offsetof(swa_params_t, scale),"
        " offsetof(swa_params_t, sparse_mode), offsetof(swa_params_t, keep_prob));"
        "printf(\"%zu %zu %zu\\n\", offsetof(swa_params_t, N_kv), offsetof(swa_params_t, dropout_seed),"
        " offsetof(swa_params_t, dtype));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    P = swa.SwaParams
    want = [ctypes.sizeof(P), P.B.offset, P.cu_seqlens_q.offset, P.scale.offset, P.sparse_mode.offset,
            P.keep_prob.offset, P.N_kv.offset, P.dropout_seed.offset, P.dtype.offset]
    assert got == want


def test_defaults_match_documented_attributes(lib):
    p = swa.SwaParams()
    lib.swa_params_default(ctypes.byref(p))
    assert p.scale == 1.0 and p.keep_prob == 1.0
    assert p.pre_tokens == 2147483647 and p.next_tokens == 2147483647
    assert p.sparse_mode == 0
    assert p.N_kv == 0  # N_kv = N


def _size(geom, backward=False):
    p = swa.Params(geom)
    n = ctypes.c_size_t(0)
    fn = swa.lib().swa_backward_workspace_size if backward else swa.lib().swa_forward_workspace_size
    return fn(p.ref(), ctypes.byref(n)), n.value


BASE = dict(layout="BNSD", B=1, N=2, D=128, S_q=256, S_kv=256, scale=0.1, sparse_mode=4, pre_tokens=64,
            next_tokens=0)


@pytest.mark.parametrize("change,status", [
    ({}, swa.SWA_OK),
    ({"sparse_mode": 1}, swa.SWA_ERR_PARAM_INVALID),
    ({"sparse_mode": 3}, swa.SWA_ERR_PARAM_INVALID),
    ({"keep_prob": 0.0}, swa.SWA_ERR_PARAM_INVALID),
    ({"keep_prob": 1.5}, swa.SWA_ERR_PARAM_INVALID),
    ({"keep_prob": float("nan")}, swa.SWA_ERR_PARAM_INVALID),
    ({"N": 0}, swa.SWA_ERR_PARAM_INVALID),
    ({"N": 257}, swa.SWA_ERR_PARAM_INVALID),
    ({"B": 0}, swa.SWA_ERR_PARAM_INVALID),
    # head dims: multiples of 8 up to 128 (computed on 64 or 128 columns)
    ({"D": 96}, swa.SWA_OK),
    ({"D": 72}, swa.SWA_OK),
    ({"D": 88}, swa.SWA_OK),
    ({"D": 8}, swa.SWA_OK),
    ({"D": 36}, swa.SWA_ERR_UNSUPPORTED),
    ({"D": 136}, swa.SWA_ERR_UNSUPPORTED),
    ({"D": 192}, swa.SWA_ERR_UNSUPPORTED),
    ({"D": 1000}, swa.SWA_ERR_PARAM_INVALID),
    ({"S_q": 0}, swa.SWA_ERR_PARAM_INVALID),
    ({"pre_tokens": -10, "next_tokens": 5}, swa.SWA_ERR_PARAM_INVALID),
    ({"pre_tokens": -10, "next_tokens": 5, "sparse_mode": 0}, swa.SWA_OK),
    ({"pre_tokens": -1, "next_tokens": 2}, swa.SWA_OK),
    ({"scale": float("inf")}, swa.SWA_ERR_PARAM_INVALID),
    ({"D": 64}, swa.SWA_OK),
    # grouped key/value heads: N must be a multiple of N_kv
    ({"N": 8, "N_kv": 2}, swa.SWA_OK),
    ({"N": 8, "N_kv": 1}, swa.SWA_OK),
    ({"N": 8, "N_kv": 8}, swa.SWA_OK),
    ({"N": 8, "N_kv": 3}, swa.SWA_ERR_PARAM_INVALID),
    ({"N": 4, "N_kv": 8}, swa.SWA_ERR_PARAM_INVALID),
    ({"N": 4, "N_kv": -2}, swa.SWA_ERR_PARAM_INVALID),
    # element types: bf16, fp16, and fp32 (computed on bf16 copies, fp32 outputs)
    ({"dtype": "fp16"}, swa.SWA_OK),
    ({"dtype": "fp32"}, swa.SWA_OK),
])
def test_parameter_checks(lib, change, status):
    st, _ = _size(Geometry(**{**BASE, **change}))
    assert st == status, swa.swa_last_error()
    if status != swa.SWA_OK:
        assert swa.swa_last_error()


@pytest.mark.parametrize("cu_q,cu_kv,status", [
    ([2, 5, 9], [2, 5, 9], swa.SWA_OK),
    ([2, 5, 9, 0, 0], [2, 5, 9, 0, 0], swa.SWA_OK),   # trailing zeros skip batches
    ([0, 5, 5, 9], [3, 3, 6, 9], swa.SWA_OK),         # length-0 sequences
    ([2, 5, 4], [2, 5, 9], swa.SWA_ERR_PARAM_INVALID),  # decreasing
    ([2, 5, 8], [2, 5, 9], swa.SWA_ERR_PARAM_INVALID),  # last != T
    ([2, 5, 9, 0, 3], [2, 5, 9, 0, 0], swa.SWA_ERR_PARAM_INVALID),  # non-zero after the tail
    ([2, 5, 0, 9], [2, 5, 0, 9], swa.SWA_ERR_PARAM_INVALID),  # tail before reaching T
])
def test_cumulative_lengths(lib, cu_q, cu_kv, status):
    g = Geometry("TND", len(cu_q), 2, 64, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, sparse_mode=0)
    p = swa.Params(g)
    p.c.T_q = 9  # the T the caller states
    p.c.T_kv = 9
    n = ctypes.c_size_t(0)
    assert swa.lib().swa_forward_workspace_size(p.ref(), ctypes.byref(n)) == status, swa.swa_last_error()


def test_null_params_and_pointers(lib):
    n = ctypes.c_size_t(0)
    assert lib.swa_forward_workspace_size(None, ctypes.byref(n)) == swa.SWA_ERR_PARAM_NULLPTR
    p = swa.Params(Geometry(**BASE))
    assert lib.swa_forward_workspace_size(p.ref(), None) == swa.SWA_ERR_PARAM_NULLPTR
    fake = 1 << 20  # never dereferenced: every check below fails first
    st = swa.swa_forward(p, None, fake, fake, None, fake, fake, fake, fake, 256, None)
    assert st == swa.SWA_ERR_PARAM_NULLPTR
    st = swa.swa_backward(p, fake, fake, fake, fake, fake, fake, fake, None, fake, None, fake, fake, 1 << 30, None)
    assert st == swa.SWA_ERR_PARAM_NULLPTR
    g = Geometry("TND", 1, 2, 64, cu_seqlens_q=[4], cu_seqlens_kv=[4])
    pt = swa.Params(g)
    pt.c.cu_seqlens_q = None
    assert lib.swa_forward_workspace_size(pt.ref(), ctypes.byref(n)) == swa.SWA_ERR_PARAM_NULLPTR


def test_dropout_mask_presence_and_alignment_and_workspace(lib):
    fake = 1 << 20
    p = swa.Params(Geometry(**{**BASE, "keep_prob": 0.9}))
    assert swa.swa_forward(p, fake, fake, fake, None, fake, fake, fake, fake, 256, None) == swa.SWA_ERR_PARAM_INVALID
    p1 = swa.Params(Geometry(**BASE))
    assert swa.swa_forward(p1, fake, fake, fake, fake, fake, fake, fake, fake, 256, None) == swa.SWA_ERR_PARAM_INVALID
    assert swa.swa_forward(p1, fake + 2, fake, fake, None, fake, fake, fake, fake, 256, None) == \
        swa.SWA_ERR_PARAM_INVALID
    assert swa.swa_forward(p1, fake, fake, fake, None, fake, fake, fake, None, 256, None) == swa.SWA_ERR_WORKSPACE
    assert swa.swa_forward(p1, fake, fake, fake, None, fake, fake, fake, fake, 128, None) == swa.SWA_ERR_WORKSPACE
    need = swa.swa_backward_workspace_size(p1)
    assert swa.swa_backward(p1, fake, fake, fake, fake, fake, fake, fake, None, fake, fake, fake, fake, need - 256,
                            None) == swa.SWA_ERR_WORKSPACE


def test_workspace_sizes_scale_with_rows(lib):
    g = WORKLOADS["bnsd_1x32x32768x128_band4096"].geom
    st_f, f = _size(g)
    st_b, b = _size(g, backward=True)
    assert st_f == swa.SWA_OK and st_b == swa.SWA_OK
    rows = g.B * g.S_q * g.N
    assert f == 256
    assert b >= 2 * rows * 4  # D + lse2 per query row and head
    assert b < 2 * rows * 4 + 4096


def test_fp32_workspace_holds_bf16_copies(lib):
    """fp32 inputs: the workspace also holds bf16 copies of q, k, v (forward)
    and of q, k, v, dy, out (backward), each 256-byte aligned."""
    g = Geometry("BNSD", 2, 4, 72, S_q=300, S_kv=200, N_kv=2, sparse_mode=0, dtype="fp32")
    st_f, f = _size(g)
    st_b, b = _size(g, backward=True)
    assert st_f == swa.SWA_OK and st_b == swa.SWA_OK
    r256 = lambda x: (x + 255) // 256 * 256
    qe, kve = 2 * 4 * 300 * 72, 2 * 2 * 200 * 72
    assert f == 256 + r256(2 * qe) + 2 * r256(2 * kve)
    stats = 2 * r256(2 * 4 * 300 * 4)
    assert b == 256 + stats + 3 * r256(2 * qe) + 2 * r256(2 * kve)
    g16 = Geometry(**{**g.as_dict(), "dtype": "bf16"})
    assert _size(g16)[1] == 256 and _size(g16, backward=True)[1] == 256 + stats


def test_step_host_rejects_bad_arguments_before_any_device_work(lib):
    """swa_step_host checks its arguments on the host and returns before it
    touches a stream (no GPU is needed to see these statuses)."""
    g = Geometry("BNSD", 1, 4, 64, S_q=128, S_kv=128, scale=0.125, sparse_mode=0)
    p = swa.Params(g)
    need = swa.swa_step_host_buffer_size(p, 2)
    fake, buf = 1 << 20, 1 << 24  # never dereferenced: every case fails its checks first
    L = swa.lib()
    args = lambda **kw: [kw.get(n, fake) for n in ("q", "k", "v", "dy", "out", "smax", "ssum", "dq", "dk", "dv")]
    call = lambda chunks, a, b, n: L.swa_step_host(p.ref(), chunks, *a, b, n, None)
    assert call(2, args(dq=None), buf, need) == swa.SWA_ERR_PARAM_NULLPTR
    assert call(2, args(q=None), buf, need) == swa.SWA_ERR_PARAM_NULLPTR
    assert call(2, args(), None, need) == swa.SWA_ERR_WORKSPACE
    assert call(2, args(), buf, need - 1) == swa.SWA_ERR_WORKSPACE
    assert call(2, args(), buf + 16, need) == swa.SWA_ERR_WORKSPACE  # not 256-byte aligned
    assert call(3, args(), buf, need) == swa.SWA_ERR_PARAM_INVALID  # 3 does not divide N = 4
    assert call(0, args(), buf, need) == swa.SWA_ERR_PARAM_INVALID


def test_step_host_buffer_sizes(lib):
    """swa_step_host's device buffer: per pipeline unit, compact copies of q,
    k, v, dy, out, dq, dk, dv and the statistics plus that unit's workspaces.
    A unit is a group of N / chunks heads, except at the ends: the first group
    is split in halves, its first half again, and so on while 2^l * chunks
    divides N and N_kv (at most three levels), and the last group the same way
    mirrored; the chunk count must divide N and N_kv, and dropout needs one
    chunk."""
    g = Geometry("BNSD", 2, 8, 64, S_q=256, S_kv=256, N_kv=4, sparse_mode=0)
    p = swa.Params(g)
    r256 = lambda x: (x + 255) // 256 * 256

    def unit_bytes(groups):  # one unit of a split into `groups` equal head groups
        qb, kb = 2 * (8 // groups) * 256 * 64 * 2, 2 * (4 // groups) * 256 * 64 * 2
        sb = 2 * (8 // groups) * 256 * 4
        sub = Geometry(**{**g.as_dict(), "N": 8 // groups, "N_kv": 4 // groups})
        fws, bws = _size(sub)[1], _size(sub, backward=True)[1]
        return 4 * r256(qb) + 4 * r256(kb) + 2 * r256(sb) + r256(fws) + r256(bws)

    # 1 chunk: one unit; 2 chunks: 2*2 = 4 divides N = 8 and N_kv = 4 (8 does
    # not divide N_kv), so one level: both groups halved, four units of the
    # 4-way split; 4 chunks: 8 does not divide N_kv, so four plain groups
    expect = {1: unit_bytes(1), 2: 4 * unit_bytes(4), 4: 4 * unit_bytes(4)}
    for chunks, want in expect.items():
        assert swa.swa_step_host_buffer_size(p, chunks) == want, chunks
    # three chunks of N = 12: 6 and 12 divide N, so two levels; units of
    # 1, 1, 2, 4, 2, 1, 1 heads (12-, 6-, 3-, 6- and 12-way splits)
    g3 = Geometry("BNSD", 1, 12, 64, S_q=128, S_kv=128, sparse_mode=0)

    def unit3(groups):
        qb = (12 // groups) * 128 * 64 * 2
        sb = (12 // groups) * 128 * 4
        sub = Geometry(**{**g3.as_dict(), "N": 12 // groups})
        fws, bws = _size(sub)[1], _size(sub, backward=True)[1]
        return 8 * r256(qb) + 2 * r256(sb) + r256(fws) + r256(bws)

    assert swa.swa_step_host_buffer_size(swa.Params(g3), 3) == 4 * unit3(12) + 2 * unit3(6) + unit3(3)
    n = ctypes.c_size_t(0)
    assert swa.lib().swa_step_host_buffer_size(p.ref(), 3, ctypes.byref(n)) == swa.SWA_ERR_PARAM_INVALID
    assert swa.lib().swa_step_host_buffer_size(p.ref(), 0, ctypes.byref(n)) == swa.SWA_ERR_PARAM_INVALID
    d = swa.Params(Geometry(**{**g.as_dict(), "keep_prob": 0.9}))  # a packed mask cannot be passed
    assert swa.lib().swa_step_host_buffer_size(d.ref(), 1, ctypes.byref(n)) == swa.SWA_ERR_PARAM_INVALID
