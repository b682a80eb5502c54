"""GPU parity on seeded random geometries: libswa against the fp64 CPU oracle.

The hand-picked cases in test_parity_gpu.py cover each feature on purpose;
these draw every parameter at once from a fixed seed per case, so that
combinations nobody listed get exercised too: layout, batch and sequence
lengths (zero-length TND sequences and skipped trailing batches included),
query and key/value heads (GQA / MQA), head dims that are multiples of 8 up
to 128, no mask or a BAND with either edge negative, the scale, dropout from
a packed mask or generated from a seed, and the element type.  The gates
are those of the hand-picked cases (tests/helpers.py).

The draw stays in the workloads' regime: scale within D^-0.5 x [0.5, 1]
(either sign), keep_prob within [0.8, 0.95], and a key/value length drawn
apart from the query length at least 64.  dS is rounded to the MMA operand
type before dQ = dS K and dK = dS^T Q, an error of up to 2^-8 of each
|dS_ij k_j| (or |dS_ij q_i|) term.  A larger scale, heavier dropout or a
few keys seen by many query rows make those terms large enough to pass the
flat 2e-2 element gate where the result itself is small (measured: 0.033 on
dQ with scale 1.9 D^-0.5, keep 0.7 and 39 keys; 0.035 on dK of fp32 outputs
with 6 keys seen by 1077 query rows).
"""
import numpy as np
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw
from oracle import swa_oracle as orc
from tests.helpers import (TOL_ABS, TOL_GRAD, TOL_OUT, check_stat, check_tensor, half_ulp, out_dtype, rel_l2,
                           to_problem)

N_CASES = 64


@pytest.fixture(scope="module")
def built():
    B.build()
    orc.build()
    swa.lib()


def random_geometry(seed: int) -> dict:
    """Geometry keyword arguments drawn from `seed` (valid by construction)."""
    rng = np.random.default_rng(1_000_003 * seed + 17)
    n_kv = int(rng.integers(1, 4))
    group = int(rng.choice([1, 1, 2, 3]))
    D = int(rng.choice([8, 16, 24, 32, 40, 56, 64, 72, 80, 96, 112, 128]))
    kw = dict(N=n_kv * group, D=D)
    if group > 1 or rng.random() < 0.3:
        kw["N_kv"] = n_kv
    if rng.random() < 0.55:
        kw.update(layout="BNSD", B=int(rng.integers(1, 3)))
        s_q = int(rng.integers(1, 480))
        s_kv = s_q if rng.random() < 0.6 else int(rng.integers(64, 480))
        kw.update(S_q=s_q, S_kv=s_kv)
    else:
        b = int(rng.integers(1, 6))
        lq = rng.integers(0, 300, b)
        lq[rng.random(b) < 0.2] = 0  # empty sequences
        if lq.sum() == 0:
            lq[0] = int(rng.integers(1, 300))
        lkv = lq.copy() if rng.random() < 0.6 else rng.integers(64, 300, b)
        lkv[lq == 0] = 0
        if lkv.sum() == 0:
            lkv[int(np.argmax(lq))] = int(rng.integers(1, 300))
        cq, ckv = np.cumsum(lq).tolist(), np.cumsum(lkv).tolist()
        # a skipped last batch is written as a trailing zero in both lists
        if b > 1 and lq[-1] == 0 and lkv[-1] == 0 and rng.random() < 0.5:
            cq[-1] = 0
            ckv[-1] = 0
        kw.update(layout="TND", B=b, cu_seqlens_q=cq, cu_seqlens_kv=ckv)
    if rng.random() < 0.7:
        pre = int(rng.integers(-64, 320))
        nxt = int(rng.integers(max(-64, -pre), 320))
        kw.update(sparse_mode=4, pre_tokens=pre, next_tokens=nxt)
    else:
        kw.update(sparse_mode=0)
    kw["scale"] = float(D ** -0.5 * rng.uniform(0.5, 1.0) * (-1.0 if rng.random() < 0.08 else 1.0))
    if rng.random() < 0.35:
        kw["keep_prob"] = float(rng.uniform(0.8, 0.95))
        if rng.random() < 0.4:
            kw.update(dropout_gen=1, dropout_seed=int(rng.integers(0, 2 ** 31)), dropout_offset=int(rng.integers(0, 64)))
    kw["dtype"] = str(rng.choice(["bf16", "bf16", "bf16", "fp16", "fp32"]))
    return kw


def test_random_geometries_are_distinct_and_valid():
    """The draw covers both layouts, both masks, GQA, dropout in both forms and every element type."""
    kws = [random_geometry(s) for s in range(N_CASES)]
    assert {k["layout"] for k in kws} == {"BNSD", "TND"}
    assert {k["sparse_mode"] for k in kws} == {0, 4}
    assert {k["dtype"] for k in kws} == {"bf16", "fp16", "fp32"}
    assert any(k.get("N_kv", k["N"]) < k["N"] for k in kws)
    assert any(k.get("keep_prob", 1.0) < 1.0 and not k.get("dropout_gen") for k in kws)
    assert any(k.get("dropout_gen") for k in kws)
    for k in kws:
        Geometry(**k)


def run_gpu(inp):
    g = inp.geom
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    out, smax, ssum = swa.forward(g, q, k, v, mask)
    ws = torch.empty(swa.swa_backward_workspace_size(swa.Params(g)), dtype=torch.uint8, device=dev)
    dq, dk, dv = swa.backward(g, q, k, v, dy, out, smax, ssum, mask, workspace=ws)
    swa.check_workspace(ws)
    torch.cuda.synchronize()
    return {n: t.cpu().double().numpy() for n, t in
            (("out", out), ("smax", smax), ("ssum", ssum), ("dq", dq), ("dk", dk), ("dv", dv))}


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_geometry_parity(seed, built):
    kw = random_geometry(seed)
    geom = Geometry(**kw)
    inp = draw(geom, 90_000 + seed)
    geom = inp.geom
    pr = to_problem(geom)
    res = run_gpu(inp)
    dt = out_dtype(geom)
    ops = (inp.q, inp.k, inp.v, inp.dy)
    if dt == "fp32":  # computed on the bf16 roundings of fp32 inputs (include/swa.h)
        ops = tuple(t.to(torch.bfloat16).to(torch.float32) for t in ops)
    mask = inp.drop_mask
    if geom.dropout_gen:  # the oracle's own Philox4x32-10 draws the bits the seed / offset stand for
        mask = orc.generate_keep_mask(pr, geom.dropout_seed, geom.dropout_offset)
    out, smax, ssum = orc.forward(pr, *ops[:3], mask)
    dq, dk, dv = orc.backward(pr, *ops, mask)
    label = f"seed {seed}: {kw}"
    check_tensor(label, "out", res["out"], out, dt, TOL_OUT)
    check_stat(label, "softmax_max", res["smax"], smax)
    check_stat(label, "softmax_sum", res["ssum"], ssum)
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tensor(label, name, res[name], ref, dt, TOL_GRAD)


# ------------------------------------------------- outside that regime --
# Scales up to 2.5 D^-0.5, keep_prob down to 0.5 and key ranges of any
# length.  There the products' 16-bit operands (P~ for out and dV, dS for
# dQ and dK) carry rounding errors up to u = 2^-8 of each term, D_i is
# formed from the stored, rounded O, and the sums of those terms' absolute
# values can far exceed the results.  The element gate adds the oracle's
# first-order bound of those roundings (orc_rounding_error, u = 2^-8) to
# the flat one.

EXTREME = {
    # the two draws outside the regime that missed the flat gate
    "gqa_39_keys_scale_1.9_keep_0.7": dict(layout="BNSD", B=2, N=6, N_kv=2, D=56, S_q=349, S_kv=39, scale=0.249,
                                           sparse_mode=4, pre_tokens=130, next_tokens=108, keep_prob=0.7),
    "mqa_6_keys_fp32": dict(layout="BNSD", B=1, N=3, N_kv=1, D=112, S_q=359, S_kv=6, scale=0.0765, sparse_mode=0,
                            dtype="fp32"),
}


def extreme_geometry(seed: int) -> dict:
    rng = np.random.default_rng(2_000_033 * seed + 5)
    kw = random_geometry(10_000 + seed)
    D = kw["D"]
    kw["scale"] = float(D ** -0.5 * rng.uniform(1.0, 2.5) * (-1.0 if rng.random() < 0.15 else 1.0))
    if kw["layout"] == "BNSD":
        kw["S_kv"] = int(rng.integers(1, 80))
    kw.pop("dropout_gen", None), kw.pop("dropout_seed", None), kw.pop("dropout_offset", None)
    kw.pop("keep_prob", None)
    if rng.random() < 0.5:
        kw["keep_prob"] = float(rng.uniform(0.5, 0.95))
        if rng.random() < 0.4:
            kw.update(dropout_gen=1, dropout_seed=int(rng.integers(0, 2 ** 31)), dropout_offset=int(rng.integers(0, 64)))
    return kw


_EXTREME_RUNS = sorted(EXTREME) + [f"draw{s}" for s in range(16)]


@pytest.mark.gpu
@pytest.mark.parametrize("name", _EXTREME_RUNS)
def test_outside_regime_within_rounding_budget(name, built):
    kw = EXTREME[name] if name in EXTREME else extreme_geometry(int(name[4:]))
    geom = Geometry(**kw)
    inp = draw(geom, 95_000 + sum(map(ord, name)))
    geom = inp.geom
    pr = to_problem(geom)
    res = run_gpu(inp)
    dt = out_dtype(geom)
    ops = (inp.q, inp.k, inp.v, inp.dy)
    if dt == "fp32":
        ops = tuple(t.to(torch.bfloat16).to(torch.float32) for t in ops)
    mask = inp.drop_mask
    if geom.dropout_gen:
        mask = orc.generate_keep_mask(pr, geom.dropout_seed, geom.dropout_offset)
    out, smax, ssum = orc.forward(pr, *ops[:3], mask)
    dq, dk, dv = orc.backward(pr, *ops, mask)
    bounds = orc.rounding_error(pr, *ops, mask, u=2.0 ** -8)
    label = f"{name}: {kw}"
    check_stat(label, "softmax_max", res["smax"], smax)
    check_stat(label, "softmax_sum", res["ssum"], ssum)
    for tname, ref, bound, tol in (("out", out, bounds[0], TOL_OUT), ("dq", dq, bounds[1], TOL_GRAD),
                                   ("dk", dk, bounds[2], TOL_GRAD), ("dv", dv, bounds[3], TOL_GRAD)):
        got = res[tname]
        assert np.all(np.isfinite(got)), (label, tname)
        excess = np.abs(got - ref) - (TOL_ABS + half_ulp(ref, dt) + bound)
        assert float(excess.max()) <= 0.0, (label, tname, "element gate with the rounding bound", float(excess.max()))
        assert rel_l2(got, ref) <= tol, (label, tname, "relative L2", rel_l2(got, ref))
