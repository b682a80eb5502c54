"""GPU parity: libswa's CUDA path against the fp64 CPU oracle, element by
element on seeded inputs, through the C ABI.

Gates (tests/helpers.py): relative L2 <= 5e-3 for out and <= 1e-2 for
dq / dk / dv; every element |got - ref| <= 2e-2 plus half an ulp of the
output type at |ref| (the storage rounding of the result; nothing for fp32
outputs); softmax_max / softmax_sum within 1e-3 relative (1e-6 absolute
below |ref| = 1e-3); and the set of visible (query, key) pairs identical to
the oracle's, in the forward and in both backward passes.

The five workloads at full size are compared on whole tensors: the two that
the oracle finishes in seconds in full (BNSD 2x16x4096x128 BAND(2047, 0) and
BNSD 4x16x2048x64 BAND(256, 256) with dropout), and complete heads of the
two long ones (heads are independent problems, so the oracle runs on one
head's slice): two heads of BNSD 1x32x32768x128 BAND(4096, 0) and two
(sequence, head) slices of the TND workload.
"""
import math

import numpy as np
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw, draw_workload, edge_probe_inputs
from oracle import swa_oracle as orc
from tests.helpers import (TOL_GRAD, TOL_OUT, check_stat, check_tensor, out_dtype, rel_l2, to_problem)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    orc.build()
    swa.lib()


def run_gpu(inp, backward=True):
    """Forward (+ backward) on cuda:0 through the binding; results as CPU tensors."""
    g = inp.geom
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    mask = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    out, smax, ssum = swa.forward(g, q, k, v, mask)
    res = {"out": out, "smax": smax, "ssum": ssum}
    if backward:
        dy = inp.dy.to(dev)
        need = swa.swa_backward_workspace_size(swa.Params(g))
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        dq, dk, dv = swa.backward(g, q, k, v, dy, out, smax, ssum, mask, workspace=ws)
        swa.check_workspace(ws)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return {k_: t.cpu() for k_, t in res.items()}


def as_np(res):
    return {k_: t.double().numpy() for k_, t in res.items()}


def check_forward(res, out, smax, ssum, label="", dtype="bf16"):
    check_tensor(label, "out", res["out"], out, dtype, TOL_OUT)
    check_stat(label, "softmax_max", res["smax"], smax)
    check_stat(label, "softmax_sum", res["ssum"], ssum)


def check_grads(res, dq, dk, dv, label="", dtype="bf16"):
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tensor(label, name, res[name], ref, dtype, TOL_GRAD)


# ----------------------------------------------------------- small cases --
# 600 short sequences: more work entries than one launch's table holds (512),
# so every pass runs as two launches
_CU600 = np.cumsum(np.random.default_rng(600).integers(1, 41, 600)).tolist()

SMALL = {
    "bnsd_nomask_d64_ragged": dict(layout="BNSD", B=2, N=2, D=64, S_q=300, S_kv=300, scale=0.125, sparse_mode=0),
    "bnsd_band_d128_ragged": dict(layout="BNSD", B=1, N=3, D=128, S_q=517, S_kv=517, scale=128 ** -0.5,
                                  sparse_mode=4, pre_tokens=200, next_tokens=0),
    "bnsd_symband_d64_dropout": dict(layout="BNSD", B=2, N=2, D=64, S_q=400, S_kv=400, scale=0.125, sparse_mode=4,
                                     pre_tokens=70, next_tokens=90, keep_prob=0.8),
    "bnsd_band_d128_dropout_ragged": dict(layout="BNSD", B=1, N=2, D=128, S_q=333, S_kv=333, scale=0.09,
                                          sparse_mode=4, pre_tokens=150, next_tokens=40, keep_prob=0.7),
    "bnsd_rect_band": dict(layout="BNSD", B=1, N=2, D=128, S_q=200, S_kv=450, scale=0.09, sparse_mode=4,
                           pre_tokens=30, next_tokens=200),
    "bnsd_rect_nomask_sq_gt_skv": dict(layout="BNSD", B=1, N=2, D=64, S_q=390, S_kv=130, scale=0.125, sparse_mode=0),
    "bnsd_empty_rows": dict(layout="BNSD", B=1, N=2, D=64, S_q=260, S_kv=260, scale=0.125, sparse_mode=4,
                            pre_tokens=-3, next_tokens=10),
    "bnsd_wide_band": dict(layout="BNSD", B=1, N=2, D=128, S_q=256, S_kv=256, scale=0.09, sparse_mode=4,
                           pre_tokens=2147483647, next_tokens=2147483647),
    "bnsd_zero_band": dict(layout="BNSD", B=1, N=2, D=64, S_q=200, S_kv=200, scale=0.125, sparse_mode=4,
                           pre_tokens=0, next_tokens=0),
    # a scale <= 0 takes the forward's scale-then-mask path on every tile (full ones included)
    "bnsd_band_negative_scale": dict(layout="BNSD", B=1, N=2, D=64, S_q=520, S_kv=520, scale=-0.125,
                                     sparse_mode=4, pre_tokens=300, next_tokens=0),
    "bnsd_nomask_zero_scale": dict(layout="BNSD", B=1, N=2, D=128, S_q=260, S_kv=260, scale=0.0, sparse_mode=0),
    "tnd_600_sequences_band": dict(layout="TND", B=600, N=2, D=64, cu_seqlens_q=_CU600, cu_seqlens_kv=_CU600,
                                   scale=0.125, sparse_mode=4, pre_tokens=7, next_tokens=3),
    "tnd_varlen_nomask": dict(layout="TND", B=5, N=2, D=128, cu_seqlens_q=[130, 130, 387, 388, 452],
                              cu_seqlens_kv=[130, 130, 387, 388, 452], scale=0.09, sparse_mode=0),
    "tnd_varlen_band_dropout_d64": dict(layout="TND", B=4, N=3, D=64, cu_seqlens_q=[200, 201, 460, 0],
                                        cu_seqlens_kv=[200, 201, 460, 0], scale=0.125, sparse_mode=4,
                                        pre_tokens=100, next_tokens=17, keep_prob=0.85),
    "tnd_rect": dict(layout="TND", B=3, N=2, D=128, cu_seqlens_q=[50, 300, 310], cu_seqlens_kv=[170, 180, 420],
                     scale=0.09, sparse_mode=4, pre_tokens=64, next_tokens=64),
    # grouped key/value heads (query head n reads key/value head n // (N / N_kv))
    "bnsd_gqa4_band_d128_ragged": dict(layout="BNSD", B=1, N=8, N_kv=2, D=128, S_q=517, S_kv=517,
                                       scale=128 ** -0.5, sparse_mode=4, pre_tokens=200, next_tokens=0),
    "bnsd_mqa_nomask_d64": dict(layout="BNSD", B=2, N=4, N_kv=1, D=64, S_q=300, S_kv=300, scale=0.125,
                                sparse_mode=0),
    "bnsd_gqa2_band_dropout_d64": dict(layout="BNSD", B=1, N=4, N_kv=2, D=64, S_q=333, S_kv=333, scale=0.125,
                                       sparse_mode=4, pre_tokens=150, next_tokens=40, keep_prob=0.8),
    "bnsd_gqa2_band_dropout_d128": dict(layout="BNSD", B=1, N=4, N_kv=2, D=128, S_q=290, S_kv=290, scale=0.09,
                                        sparse_mode=4, pre_tokens=100, next_tokens=30, keep_prob=0.75),
    # fp16 inputs (the MMAs run on fp16 operands, P and dS are rounded to fp16)
    "bnsd_band_d128_ragged_fp16": dict(layout="BNSD", B=1, N=3, D=128, S_q=517, S_kv=517, scale=128 ** -0.5,
                                       sparse_mode=4, pre_tokens=200, next_tokens=0, dtype="fp16"),
    "bnsd_nomask_d64_ragged_fp16": dict(layout="BNSD", B=2, N=2, D=64, S_q=300, S_kv=300, scale=0.125,
                                        sparse_mode=0, dtype="fp16"),
    "tnd_varlen_band_dropout_d64_fp16": dict(layout="TND", B=4, N=3, D=64, cu_seqlens_q=[200, 201, 460, 0],
                                             cu_seqlens_kv=[200, 201, 460, 0], scale=0.125, sparse_mode=4,
                                             pre_tokens=100, next_tokens=17, keep_prob=0.85, dtype="fp16"),
    "bnsd_gqa2_band_dropout_d128_fp16": dict(layout="BNSD", B=1, N=4, N_kv=2, D=128, S_q=290, S_kv=290, scale=0.09,
                                             sparse_mode=4, pre_tokens=100, next_tokens=30, keep_prob=0.75,
                                             dtype="fp16"),
    "tnd_gqa2_varlen_band_d128": dict(layout="TND", B=3, N=4, N_kv=2, D=128, cu_seqlens_q=[200, 200, 520],
                                      cu_seqlens_kv=[200, 200, 520], scale=0.09, sparse_mode=4, pre_tokens=100,
                                      next_tokens=20),
    # head dims other than 64 / 128: computed on 64 or 128 zero-padded columns
    "bnsd_band_d72_ragged": dict(layout="BNSD", B=1, N=3, D=72, S_q=333, S_kv=333, scale=72 ** -0.5,
                                 sparse_mode=4, pre_tokens=150, next_tokens=0),
    "bnsd_nomask_d88": dict(layout="BNSD", B=2, N=2, D=88, S_q=260, S_kv=260, scale=88 ** -0.5, sparse_mode=0),
    "tnd_varlen_band_dropout_d96": dict(layout="TND", B=3, N=2, D=96, cu_seqlens_q=[150, 150, 420],
                                        cu_seqlens_kv=[150, 150, 420], scale=96 ** -0.5, sparse_mode=4,
                                        pre_tokens=90, next_tokens=30, keep_prob=0.85),
    "bnsd_gqa2_band_d32": dict(layout="BNSD", B=1, N=4, N_kv=2, D=32, S_q=300, S_kv=300, scale=32 ** -0.5,
                               sparse_mode=4, pre_tokens=120, next_tokens=10),
    "bnsd_band_d8": dict(layout="BNSD", B=1, N=2, D=8, S_q=200, S_kv=200, scale=8 ** -0.5, sparse_mode=4,
                         pre_tokens=60, next_tokens=60),
    "bnsd_band_d120_fp16": dict(layout="BNSD", B=1, N=2, D=120, S_q=270, S_kv=270, scale=120 ** -0.5,
                                sparse_mode=4, pre_tokens=100, next_tokens=0, dtype="fp16"),
    "bnsd_rect_band_d40": dict(layout="BNSD", B=1, N=2, D=40, S_q=150, S_kv=330, scale=40 ** -0.5, sparse_mode=4,
                               pre_tokens=40, next_tokens=160),
    # fp32 inputs and outputs (the MMAs take bf16 copies of the inputs)
    "bnsd_band_d128_ragged_fp32": dict(layout="BNSD", B=1, N=3, D=128, S_q=517, S_kv=517, scale=128 ** -0.5,
                                       sparse_mode=4, pre_tokens=200, next_tokens=0, dtype="fp32"),
    "tnd_varlen_band_dropout_d64_fp32": dict(layout="TND", B=4, N=3, D=64, cu_seqlens_q=[200, 201, 460, 0],
                                             cu_seqlens_kv=[200, 201, 460, 0], scale=0.125, sparse_mode=4,
                                             pre_tokens=100, next_tokens=17, keep_prob=0.85, dtype="fp32"),
    "bnsd_gqa2_nomask_d72_fp32": dict(layout="BNSD", B=1, N=4, N_kv=2, D=72, S_q=290, S_kv=290, scale=72 ** -0.5,
                                      sparse_mode=0, dtype="fp32"),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    geom = Geometry(**SMALL[name])
    inp = draw(geom, 5000 + sum(map(ord, name)))
    pr = to_problem(geom)
    res = as_np(run_gpu(inp))
    dt = out_dtype(geom)
    if dt == "fp32":
        # fp32 inputs are computed on their bf16 roundings (include/swa.h):
        # every gate against the oracle on those operands; out and the
        # gradients also against the oracle on the exact fp32 inputs, where
        # the input rounding (2^-9 relative per operand) is added to the flat
        # element bound
        rq, rk, rv, rdy = (t.to(torch.bfloat16).to(torch.float32) for t in (inp.q, inp.k, inp.v, inp.dy))
        out, smax, ssum = orc.forward(pr, rq, rk, rv, inp.drop_mask)
        dq, dk, dv = orc.backward(pr, rq, rk, rv, rdy, inp.drop_mask)
        check_forward(res, out, smax, ssum, name, "fp32")
        check_grads(res, dq, dk, dv, name, "fp32")
        out_x, _, _ = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
        dq_x, dk_x, dv_x = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
        for tname, got, ref, tol in (("out", res["out"], out_x, TOL_OUT), ("dq", res["dq"], dq_x, TOL_GRAD),
                                     ("dk", res["dk"], dk_x, TOL_GRAD), ("dv", res["dv"], dv_x, TOL_GRAD)):
            assert rel_l2(got, ref) <= tol, (name, tname, "vs exact fp32 inputs")
            bound = 2e-2 + 2.0 ** -8 * np.abs(ref)
            assert np.all(np.abs(got - ref) <= bound), (name, tname, "vs exact fp32 inputs")
        return
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    check_forward(res, out, smax, ssum, name, dt)
    check_grads(res, dq, dk, dv, name, dt)


@pytest.mark.parametrize("name", sorted(n for n, kw in SMALL.items() if kw["D"] <= 64))
def test_small_parity_pair_forward(name):
    """The D <= 64 cases with the forward forced onto one CTA per pair of query
    tiles (the size rule picks that kernel only when the pairs fill every SM):
    every output, the gradients computed from its out and statistics
    included, against the oracle."""
    geom = Geometry(**SMALL[name])
    inp = draw(geom, 5000 + sum(map(ord, name)))
    pr = to_problem(geom)
    swa.swa_debug_forward_pairs(1)
    try:
        res = as_np(run_gpu(inp))
    finally:
        swa.swa_debug_forward_pairs(0)
    dt = out_dtype(geom)
    ops = (inp.q, inp.k, inp.v, inp.dy)
    if dt == "fp32":  # computed on the bf16 roundings of fp32 inputs
        ops = tuple(t.to(torch.bfloat16).to(torch.float32) for t in ops)
    out, smax, ssum = orc.forward(pr, *ops[:3], inp.drop_mask)
    dq, dk, dv = orc.backward(pr, *ops, inp.drop_mask)
    label = f"{name} (query tile pairs)"
    check_forward(res, out, smax, ssum, label, dt)
    check_grads(res, dq, dk, dv, label, dt)


def test_repeat_calls_are_deterministic_forward():
    geom = Geometry(**SMALL["bnsd_band_d128_ragged"])
    inp = draw(geom, 77)
    a = as_np(run_gpu(inp, backward=False))
    b = as_np(run_gpu(inp, backward=False))
    for k_ in a:
        assert np.array_equal(a[k_], b[k_])


def test_repeat_calls_are_deterministic_backward():
    # dQ, dK and dV accumulate in TMEM in a fixed order: no atomics, so two
    # runs agree bit for bit (grouped heads included)
    geom = Geometry(**SMALL["bnsd_gqa4_band_d128_ragged"])
    inp = draw(geom, 78)
    a = as_np(run_gpu(inp))
    b = as_np(run_gpu(inp))
    for k_ in a:
        assert np.array_equal(a[k_], b[k_]), k_


# ------------------------------------------------------ masked set, exact --
MASKSETS = {
    "band": dict(layout="BNSD", B=1, N=2, D=64, S_q=1000, S_kv=1000, sparse_mode=4, pre_tokens=300,
                 next_tokens=5),
    "band_negative_pre": dict(layout="BNSD", B=1, N=1, D=128, S_q=700, S_kv=700, sparse_mode=4, pre_tokens=-40,
                              next_tokens=300),
    "rect_band": dict(layout="BNSD", B=2, N=1, D=64, S_q=300, S_kv=900, sparse_mode=4, pre_tokens=10,
                      next_tokens=500),
    "long_band_4096": dict(layout="BNSD", B=1, N=1, D=128, S_q=32768, S_kv=32768, sparse_mode=4, pre_tokens=4096,
                           next_tokens=0),
    "tnd_band": dict(layout="TND", B=3, N=2, D=64, cu_seqlens_q=[300, 300, 1000], cu_seqlens_kv=[250, 260, 1100],
                     sparse_mode=4, pre_tokens=129, next_tokens=255),
    "nomask": dict(layout="BNSD", B=1, N=1, D=64, S_q=333, S_kv=555, sparse_mode=0),
    "gqa_band": dict(layout="BNSD", B=1, N=4, N_kv=2, D=64, S_q=600, S_kv=600, sparse_mode=4, pre_tokens=200,
                     next_tokens=70),
}


def _stat_probe(geom, which):
    """Inputs whose statistics expose the visible key range exactly.
    which = 'count': q = 0 -> softmax_sum_i = |V_i|.
    which = 'hi' / 'lo': s_ij = +j / -j -> softmax_max_i = max / -min visible j."""
    g = Geometry(**{**geom.as_dict(), "scale": 1.0, "keep_prob": 1.0})
    inp = draw(g, 9)
    q = torch.zeros_like(inp.q)
    k = torch.zeros_like(inp.k)
    if which != "count":
        sign = 1.0 if which == "hi" else -1.0
        q[..., 0] = sign
        q[..., 1] = sign * 256.0
        if g.layout == "BNSD":
            j = torch.arange(g.S_kv)
            k[..., 0] = (j % 256).float().to(torch.bfloat16)
            k[..., 1] = (j // 256).float().to(torch.bfloat16)
        else:
            start = 0
            for (lq, lk) in g.seq_lens():
                j = torch.arange(lk)
                k[start:start + lk, :, 0] = (j % 256).float()[:, None].to(torch.bfloat16)
                k[start:start + lk, :, 1] = (j // 256).float()[:, None].to(torch.bfloat16)
                start += lk
    inp.q, inp.k = q, k
    return g, inp


@pytest.mark.parametrize("name", sorted(MASKSETS))
def test_masked_set_exact_forward(name):
    geom = Geometry(**MASKSETS[name])
    pr = to_problem(geom)
    rows = np.arange(np.prod(geom.stat_shape()))
    lo, hi = orc.key_ranges(pr, rows)
    empty = lo > hi
    g, inp = _stat_probe(geom, "count")
    res = as_np(run_gpu(inp, backward=False))
    count = res["ssum"].reshape(-1)
    assert np.array_equal(count, np.where(empty, 0, hi - lo + 1).astype(np.float64))
    for which, ref in (("hi", hi), ("lo", -lo)):
        g, inp = _stat_probe(geom, which)
        res = as_np(run_gpu(inp, backward=False))
        m = res["smax"].reshape(-1)
        assert np.all(np.isneginf(m[empty]))
        got = m[~empty]
        assert np.all(np.abs(got - ref[~empty]) < 0.25), which
        assert np.array_equal(np.rint(got), ref[~empty].astype(np.float64)), which


@pytest.mark.parametrize("alpha", [-1.0, 1.0], ids=["left_edge", "right_edge"])
@pytest.mark.parametrize("name", sorted(MASKSETS))
def test_masked_set_exact_backward(name, alpha):
    """Both backward passes use exactly the oracle's visible pairs.

    The edge probe (workloads.edge_probe_inputs) puts half of each row's
    probability on the key at one edge of its window (alpha < 0: the
    leftmost visible key, alpha > 0: the rightmost), halving per key inward,
    with exact scores.  One pair too many at that edge then has twice the
    row's largest probability, and one pair too few drops half of the row's
    mass, so dV (key-major pass) and dQ (query-major pass) move far past the
    element gate on every row and key the error touches; tests/test_oracle_pins.py shows that on
    the oracle with windows moved by one pair at each edge."""
    geom = Geometry(**{**MASKSETS[name], "scale": math.log(2.0)})
    inp = draw(geom, 13)
    inp.q, inp.k, inp.v, inp.dy = edge_probe_inputs(geom, inp.k, inp.dy, alpha)
    pr = to_problem(geom)
    res = as_np(run_gpu(inp))
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy)
    label = f"edge probe {name} alpha={alpha:+g}"
    check_forward(res, out, smax, ssum, label)
    # dQ columns 0-1 and dK columns 0-3 carry the position code of k and q
    # (entries up to 255 and 32512): there the bf16 rounding of dS alone is
    # above the gate, and they add nothing about the window that columns 4+
    # do not show
    check_tensor(label, "dq[2:]", res["dq"][..., 2:], dq[..., 2:], "bf16", TOL_GRAD)
    check_tensor(label, "dk[4:]", res["dk"][..., 4:], dk[..., 4:], "bf16")
    check_tensor(label, "dv", res["dv"], dv, "bf16", TOL_GRAD)


# ------------------------------------------------- full-size workloads -----
def _invariants(geom, inp, res):
    """Whole-tensor properties of the exact gradients (no dropout, no empty
    rows), per head: sum_j dV_j = sum_i dY_i (rows of P sum to one) and
    sum_j dK_j = 0 (rows of dS sum to zero)."""
    if geom.keep_prob < 1.0:
        return
    if geom.layout == "BNSD":
        heads = [((b, n), (b, n)) for b in range(geom.B) for n in range(geom.N)]
        get_q = lambda t, h: t[h[0], h[1]]
        get_k = get_q
    else:
        heads, qs, ks = [], 0, 0
        for (lq, lk) in geom.seq_lens():
            if lq and lk:
                heads += [((qs, lq, n), (ks, lk, n)) for n in range(geom.N)]
            qs += lq
            ks += lk
        get_q = lambda t, h: t[h[0]:h[0] + h[1], h[2]]
        get_k = get_q
    for hq, hk in heads:
        s_dy = get_q(inp.dy, hq).double().sum(0).numpy()
        s_dv = get_k(res["dv"], hk).double().sum(0).numpy()
        assert np.linalg.norm(s_dv - s_dy) <= 1e-3 * np.linalg.norm(s_dy) + 0.05, "dV mass"
        dkh = get_k(res["dk"], hk).double()
        s_dk = dkh.sum(0).numpy()
        walk = float(torch.sqrt((dkh ** 2).sum()))  # size of a sum of unrelated rows
        assert np.linalg.norm(s_dk) <= 0.05 * walk + 1e-3, "dK rows of dS sum to zero"


@pytest.mark.parametrize("name", ["bnsd_2x16x4096x128_band2047", "bnsd_4x16x2048x64_band256_256_drop0.9",
                                  "bnsd_1x2x256x64_nomask"])
def test_workload_full_parity(name):
    """Every element of all six outputs against the oracle's full run."""
    inp = draw_workload(name)
    pr = to_problem(inp.geom)
    res = as_np(run_gpu(inp))
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    check_forward(res, out, smax, ssum, name)
    check_grads(res, dq, dk, dv, name)


def _head_slice(geom, inp, res, seq, n):
    """One complete (sequence, head) of a problem as a problem of its own:
    (sub-geometry, oracle inputs, GPU outputs of that slice as float64)."""
    if geom.layout == "BNSD":
        sub = Geometry(**{**geom.as_dict(), "B": 1, "N": 1})
        cut = lambda t: t[seq:seq + 1, n:n + 1].contiguous()
        cut_s = lambda t: t[seq:seq + 1, n:n + 1]
    else:
        lens = geom.seq_lens()
        start = sum(lq for lq, _ in lens[:seq])
        L = lens[seq][0]
        sub = Geometry(**{**geom.as_dict(), "B": 1, "N": 1, "cu_seqlens_q": [L], "cu_seqlens_kv": [L]})
        cut = lambda t: t[start:start + L, n:n + 1].contiguous()
        cut_s = cut
    tens = [cut(t) for t in (inp.q, inp.k, inp.v, inp.dy)]
    got = {k_: cut_s(res[k_]).double().numpy() for k_ in ("out", "dq", "dk", "dv", "smax", "ssum")}
    return sub, tens, got


@pytest.fixture(scope="module")
def long_runs():
    """The two long workloads, run once on the GPU (CPU copies of the outputs)."""
    runs = {}
    for name in ("bnsd_1x32x32768x128_band4096", "tnd_8xU512_8192_n32_d128_nomask"):
        inp = draw_workload(name)
        runs[name] = (inp, run_gpu(inp))
    return runs


def _long_slices(name, geom):
    if geom.layout == "BNSD":
        return [(0, 0), (0, geom.N - 1)]
    lens = [lq for lq, _ in geom.seq_lens()]
    return [(int(np.argmax(lens)), 0), (int(np.argmin(lens)), geom.N - 1)]


@pytest.mark.parametrize("name", ["bnsd_1x32x32768x128_band4096", "tnd_8xU512_8192_n32_d128_nomask"])
def test_workload_full_head_parity(name, long_runs):
    """Every element of complete heads (BNSD) or (sequence, head) slices (TND)
    against the oracle run on that slice alone, plus whole-tensor checks of
    every row: 1 <= softmax_sum <= |V_i| and the gradient invariants."""
    inp, res_t = long_runs[name]
    geom = inp.geom
    pr = to_problem(geom)
    for key in ("out", "dq", "dk", "dv", "smax", "ssum"):
        assert not torch.isnan(res_t[key]).any(), key
    rows_all = np.arange(int(np.prod(geom.stat_shape())))
    lo, hi = orc.key_ranges(pr, rows_all)
    ssum = res_t["ssum"].double().numpy().reshape(-1)
    ne = lo <= hi
    assert np.all(ssum[ne] >= 1.0 - 1e-4) and np.all(ssum[ne] <= (hi - lo + 1)[ne] * (1 + 1e-4))
    _invariants(geom, inp, res_t)
    for seq, n in _long_slices(name, geom):
        sub, (q, k, v, dy), got = _head_slice(geom, inp, res_t, seq, n)
        spr = to_problem(sub)
        out, smax, ssum_r = orc.forward(spr, q, k, v)
        dq, dk, dv = orc.backward(spr, q, k, v, dy)
        label = f"{name} seq {seq} head {n}"
        check_forward(got, out.reshape(got["out"].shape), smax.reshape(got["smax"].shape),
                      ssum_r.reshape(got["ssum"].shape), label)
        check_grads(got, dq.reshape(got["dq"].shape), dk.reshape(got["dk"].shape), dv.reshape(got["dv"].shape),
                    label)
