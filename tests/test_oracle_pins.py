"""Pins for the fp64 CPU oracle, against things other than itself.

- closed forms of the pages' own samples (tests/golden/*.json);
- central finite differences of L = sum(dY * O) for dQ, dK, dV;
- torch.nn.functional.scaled_dot_product_attention in float64 with an
  explicit boolean mask (a library routine), and autograd for its gradients;
- invariants: softmax rows sum to one, logsumexp of the visible scores,
  BAND wider than the sequence == sparse_mode 0, keep mask all ones ==
  no dropout, TND sequence == BNSD with B = 1, Skv = 1 -> out = v,
  pre = next = 0 -> out_i = v_i, empty rows, dropout bit order checked with
  numpy.unpackbits;
- the sampled-row / sampled-column entry points equal the full ones;
- key_ranges (the visible window of each row) equals the dense BAND mask on
  every row, empty rows included;
- the edge probe the GPU masked-set tests use moves dV and dQ far past the
  element gate on every row and key that a window error of one pair touches.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from attention_swa_forward_gb300.workloads import Geometry, draw
from oracle import swa_oracle as orc
from attention_swa_forward_gb300.workloads import edge_probe_inputs
from tests.helpers import TOL_ABS, half_ulp, to_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _tnd_problem(g, **over):
    d = dict(layout="TND", B=len(g["cu_seqlens_q"]), N=g["N"], D=g["D"], cu_seqlens_q=g["cu_seqlens_q"],
             cu_seqlens_kv=g["cu_seqlens_kv"], scale=g["scale"], pre_tokens=g["pre_tokens"],
             next_tokens=g["next_tokens"], sparse_mode=g["sparse_mode"], keep_prob=g["keep_prob"])
    d.update(over)
    return orc.Problem(**d)


# ------------------------------------------------------------ pages' samples --
@pytest.mark.parametrize("reading", ["value_one", "fp16_bit_pattern_one"])
def test_pages_forward_sample_closed_form(reading):
    g = _load("aclnn_varlen_forward_sample.json")
    c = g["fill_readings"][reading]
    pr = _tnd_problem(g)
    x = np.full((g["T"], g["N"], g["D"]), c)
    out, smax, ssum = orc.forward(pr, x, x, x)
    assert np.allclose(out, c, rtol=1e-12, atol=0)
    assert np.allclose(smax, g["scale"] * g["D"] * c * c, rtol=1e-12, atol=0)
    assert np.allclose(ssum, g["T"], rtol=1e-12, atol=0)


def test_pages_backward_sample_given_stats_closed_form():
    g = _load("aclnn_unpadding_grad_v2_sample.json")
    f = g["fill"]
    pr = _tnd_problem(g)
    shape = (g["T"], g["N"], g["D"])
    q, k, v, dy = (np.full(shape, f[n]) for n in ("q", "k", "v", "dy"))
    given_out = np.full(shape, f["attention_in"])
    gm = np.full((g["T"], g["N"]), f["softmax_max"])
    gs = np.full((g["T"], g["N"]), f["softmax_sum"])
    dq, dk, dv = orc.backward(pr, q, k, v, dy, None, given_out, gm, gs)
    p = math.exp(g["scale"] * g["D"] * f["q"] * f["k"] - f["softmax_max"]) / f["softmax_sum"]
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    assert np.allclose(dv, g["T"] * p * f["dy"], rtol=1e-12, atol=0)


def test_pages_backward_sample_exact_mode():
    g = _load("aclnn_unpadding_grad_v2_sample.json")
    pr = _tnd_problem(g)
    x = np.ones((g["T"], g["N"], g["D"]))
    dq, dk, dv = orc.backward(pr, x, x, x, x)
    assert np.allclose(dq, 0.0, atol=1e-12) and np.allclose(dk, 0.0, atol=1e-12)
    assert np.allclose(dv, 1.0, rtol=1e-12)


# ------------------------------------------------------- finite differences --
FD_CASES = {
    "bnsd_nomask": dict(layout="BNSD", B=1, N=2, D=4, S_q=6, S_kv=6, scale=0.7, sparse_mode=0),
    "bnsd_band": dict(layout="BNSD", B=1, N=1, D=4, S_q=7, S_kv=7, scale=0.9, sparse_mode=4, pre_tokens=2,
                      next_tokens=1),
    "bnsd_band_negative_pre": dict(layout="BNSD", B=1, N=1, D=3, S_q=6, S_kv=6, scale=1.1, sparse_mode=4,
                                   pre_tokens=-1, next_tokens=2),
    "bnsd_rect_band": dict(layout="BNSD", B=2, N=1, D=3, S_q=5, S_kv=8, scale=0.8, sparse_mode=4, pre_tokens=1,
                           next_tokens=3),
    "bnsd_dropout": dict(layout="BNSD", B=1, N=2, D=4, S_q=5, S_kv=5, scale=0.6, sparse_mode=4, pre_tokens=2,
                         next_tokens=2, keep_prob=0.7),
    "tnd_varlen": dict(layout="TND", B=4, N=2, D=3, cu_seqlens_q=[3, 3, 8, 0], cu_seqlens_kv=[4, 6, 9, 0],
                       scale=0.75, sparse_mode=0),
    "tnd_band_dropout": dict(layout="TND", B=2, N=1, D=4, cu_seqlens_q=[4, 9], cu_seqlens_kv=[4, 9], scale=0.9,
                             sparse_mode=4, pre_tokens=1, next_tokens=1, keep_prob=0.6),
    # the pages put no sign on scale: a negative one reverses the score order
    "bnsd_band_negative_scale": dict(layout="BNSD", B=1, N=2, D=4, S_q=7, S_kv=7, scale=-0.8, sparse_mode=4,
                                     pre_tokens=3, next_tokens=1),
}


def _fd_inputs(case, seed):
    geom = Geometry(**case)
    inp = draw(geom, seed)
    return geom, inp


@pytest.mark.parametrize("name", sorted(FD_CASES))
def test_finite_differences(name):
    case = FD_CASES[name]
    geom, inp = _fd_inputs(case, 1000 + len(name))
    pr = to_problem(geom)
    q, k, v, dy = (t.double().numpy() for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask
    dq, dk, dv = orc.backward(pr, q, k, v, dy, mask)

    def loss(qq, kk, vv):
        out, _, _ = orc.forward(pr, qq, kk, vv, mask)
        return float(np.sum(out * dy))

    h = 1e-6
    for which, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(base)
        flat = base.reshape(-1)
        for idx in range(flat.size):
            save = flat[idx]
            flat[idx] = save + h
            lp = loss(q, k, v)
            flat[idx] = save - h
            lm = loss(q, k, v)
            flat[idx] = save
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm((num - grad).ravel()) / max(np.linalg.norm(num.ravel()), 1e-30)
        assert err <= 1e-6, (name, which, err)


# ------------------------------------------------------- library routine ----
def _dense_mask(pr, lq, lk):
    i = np.arange(lq)[:, None]
    j = np.arange(lk)[None, :]
    if pr.sparse_mode == 4:
        return (j >= i - pr.pre_tokens) & (j <= i + pr.next_tokens)
    return np.ones((lq, lk), dtype=bool)


SDPA_CASES = {
    "nomask": dict(layout="BNSD", B=2, N=2, D=8, S_q=33, S_kv=33, scale=0.35, sparse_mode=0),
    "band": dict(layout="BNSD", B=1, N=3, D=16, S_q=70, S_kv=70, scale=0.25, sparse_mode=4, pre_tokens=9,
                 next_tokens=3),
    "band_sym": dict(layout="BNSD", B=2, N=1, D=8, S_q=40, S_kv=40, scale=0.4, sparse_mode=4, pre_tokens=5,
                     next_tokens=5),
    "rect": dict(layout="BNSD", B=1, N=2, D=8, S_q=20, S_kv=37, scale=0.3, sparse_mode=4, pre_tokens=4,
                 next_tokens=12),
    "band_negative_scale": dict(layout="BNSD", B=1, N=2, D=8, S_q=40, S_kv=40, scale=-0.3, sparse_mode=4,
                                pre_tokens=11, next_tokens=0),
    "nomask_zero_scale": dict(layout="BNSD", B=1, N=2, D=8, S_q=21, S_kv=21, scale=0.0, sparse_mode=0),
}


@pytest.mark.parametrize("name", sorted(SDPA_CASES))
def test_against_sdpa_float64(name):
    case = SDPA_CASES[name]
    geom = Geometry(**case)
    inp = draw(geom, 2000 + len(name))
    pr = to_problem(geom)
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy)
    q = inp.q.double().requires_grad_(True)
    k = inp.k.double().requires_grad_(True)
    v = inp.v.double().requires_grad_(True)
    m = torch.from_numpy(_dense_mask(pr, geom.S_q, geom.S_kv))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=geom.scale)
    ref.backward(inp.dy.double())
    assert np.allclose(out, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dq, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    assert np.allclose(dk, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    assert np.allclose(dv, v.grad.numpy(), rtol=1e-9, atol=1e-11)
    # statistics: softmax_max is the max visible scaled score, and
    # softmax_max + log(softmax_sum) is the logsumexp of the visible scores
    s = geom.scale * torch.einsum("bnid,bnjd->bnij", inp.q.double(), inp.k.double())
    s = s.masked_fill(~m, float("-inf"))
    assert np.allclose(smax, torch.amax(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(smax + np.log(ssum), torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- invariants ---
def test_probability_rows_sum_to_one():
    # V = identity (one-hot per key) makes out_i = P_i
    S = 48
    geom = Geometry("BNSD", 1, 2, S, S_q=S, S_kv=S, scale=0.2, sparse_mode=4, pre_tokens=7, next_tokens=2)
    inp = draw(geom, 7)
    eye = torch.eye(S, dtype=torch.bfloat16).expand(1, 2, S, S).contiguous()
    out, _, _ = orc.forward(to_problem(geom), inp.q, inp.k, eye)
    assert np.allclose(out.sum(-1), 1.0, rtol=0, atol=1e-13)
    # and P vanishes outside the band
    band = _dense_mask(to_problem(geom), S, S)
    assert np.all(out[..., ~band] == 0.0)


def test_wide_band_equals_no_mask():
    base = dict(layout="BNSD", B=1, N=2, D=16, S_q=50, S_kv=50, scale=0.3)
    g0 = Geometry(**base, sparse_mode=0)
    g4 = Geometry(**base, sparse_mode=4, pre_tokens=50, next_tokens=50)
    inp = draw(g0, 11)
    a = orc.forward(to_problem(g0), inp.q, inp.k, inp.v)
    b = orc.forward(to_problem(g4), inp.q, inp.k, inp.v)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    ga = orc.backward(to_problem(g0), inp.q, inp.k, inp.v, inp.dy)
    gb = orc.backward(to_problem(g4), inp.q, inp.k, inp.v, inp.dy)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)


def test_keep_all_is_identity():
    g = Geometry("BNSD", 1, 2, 8, S_q=30, S_kv=30, scale=0.5, sparse_mode=4, pre_tokens=6, next_tokens=6)
    inp = draw(g, 12)
    ones = np.full((g.mask_bits() + 7) // 8, 0xFF, dtype=np.uint8)
    a = orc.forward(to_problem(g), inp.q, inp.k, inp.v, None)
    b = orc.forward(to_problem(g), inp.q, inp.k, inp.v, ones)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    ga = orc.backward(to_problem(g), inp.q, inp.k, inp.v, inp.dy, None)
    gb = orc.backward(to_problem(g), inp.q, inp.k, inp.v, inp.dy, ones)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)


def test_dropout_mask_bit_order_and_element_order():
    # V = identity: out = P * z / keep, with z decoded by numpy.unpackbits
    B, N, S, keep = 2, 2, 24, 0.75
    g = Geometry("BNSD", B, N, S, S_q=S, S_kv=S, scale=0.3, sparse_mode=4, pre_tokens=5, next_tokens=3,
                 keep_prob=keep)
    inp = draw(g, 13)
    eye = torch.eye(S, dtype=torch.bfloat16).expand(B, N, S, S).contiguous()
    p_nodrop, _, _ = orc.forward(to_problem(Geometry(**{**g.as_dict(), "keep_prob": 1.0})), inp.q, inp.k, eye)
    p_drop, _, _ = orc.forward(to_problem(g), inp.q, inp.k, eye, inp.drop_mask)
    z = np.unpackbits(inp.drop_mask.numpy(), bitorder="little")[: B * N * S * S].reshape(B, N, S, S)
    assert 0 < z.mean() < 1
    assert np.allclose(p_drop, p_nodrop * z / keep, rtol=1e-14, atol=1e-15)


def test_tnd_sequence_equals_bnsd():
    lens_q, lens_kv = [5, 0, 17, 9], [7, 3, 17, 4]
    cu_q, cu_kv = list(np.cumsum(lens_q)), list(np.cumsum(lens_kv))
    g = Geometry("TND", 4, 2, 8, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, scale=0.4, sparse_mode=4, pre_tokens=3,
                 next_tokens=2, keep_prob=0.8)
    inp = draw(g, 14)
    pr = to_problem(g)
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    z = np.unpackbits(inp.drop_mask.numpy(), bitorder="little")
    qs = ks = zoff = 0
    for lq, lk in zip(lens_q, lens_kv):
        if lq and lk:
            sub = Geometry("BNSD", 1, 2, 8, S_q=lq, S_kv=lk, scale=0.4, sparse_mode=4, pre_tokens=3, next_tokens=2,
                           keep_prob=0.8)
            nb = 2 * lq * lk
            sub_mask = np.packbits(z[zoff:zoff + nb], bitorder="little")
            t = lambda x, s, l: x[s:s + l].permute(1, 0, 2).unsqueeze(0).contiguous()  # [L,N,D] -> [1,N,L,D]
            o2, m2, l2 = orc.forward(to_problem(sub), t(inp.q, qs, lq), t(inp.k, ks, lk), t(inp.v, ks, lk), sub_mask)
            g2 = orc.backward(to_problem(sub), t(inp.q, qs, lq), t(inp.k, ks, lk), t(inp.v, ks, lk),
                              t(inp.dy, qs, lq), sub_mask)
            assert np.array_equal(out[qs:qs + lq], o2[0].transpose(1, 0, 2))
            assert np.array_equal(smax[qs:qs + lq], m2[0].T)
            assert np.array_equal(ssum[qs:qs + lq], l2[0].T)
            assert np.allclose(dq[qs:qs + lq], g2[0][0].transpose(1, 0, 2), rtol=1e-13, atol=1e-15)
            assert np.allclose(dk[ks:ks + lk], g2[1][0].transpose(1, 0, 2), rtol=1e-13, atol=1e-15)
            assert np.allclose(dv[ks:ks + lk], g2[2][0].transpose(1, 0, 2), rtol=1e-13, atol=1e-15)
            zoff += nb
        elif lq:  # no keys: every row is empty
            assert np.all(out[qs:qs + lq] == 0) and np.all(ssum[qs:qs + lq] == 0)
            assert np.all(np.isneginf(smax[qs:qs + lq]))
        qs += lq
        ks += lk
    assert zoff == g.mask_bits()


def test_single_key_returns_value():
    g = Geometry("BNSD", 2, 2, 8, S_q=9, S_kv=1, scale=0.5, sparse_mode=0)
    inp = draw(g, 15)
    out, _, ssum = orc.forward(to_problem(g), inp.q, inp.k, inp.v)
    assert np.array_equal(out, np.broadcast_to(inp.v.double().numpy(), out.shape))
    assert np.all(ssum == 1.0)


def test_zero_width_band_returns_own_value():
    g = Geometry("BNSD", 1, 2, 8, S_q=12, S_kv=12, scale=0.5, sparse_mode=4, pre_tokens=0, next_tokens=0)
    inp = draw(g, 16)
    out, smax, ssum = orc.forward(to_problem(g), inp.q, inp.k, inp.v)
    assert np.array_equal(out, inp.v.double().numpy())
    assert np.all(ssum == 1.0)
    qk = g.scale * (inp.q.double() * inp.k.double()).sum(-1).numpy()
    assert np.allclose(smax, qk, rtol=1e-14, atol=1e-15)


def test_empty_rows_convention():
    # window [i+1, i+2]: the last row sees nothing
    g = Geometry("BNSD", 1, 1, 4, S_q=6, S_kv=6, scale=0.5, sparse_mode=4, pre_tokens=-1, next_tokens=2)
    inp = draw(g, 17)
    out, smax, ssum = orc.forward(to_problem(g), inp.q, inp.k, inp.v)
    dq, dk, dv = orc.backward(to_problem(g), inp.q, inp.k, inp.v, inp.dy)
    assert np.all(out[0, 0, 5] == 0) and np.isneginf(smax[0, 0, 5]) and ssum[0, 0, 5] == 0
    assert np.all(dq[0, 0, 5] == 0)
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    # key 0 is seen by nobody (j >= i + 1 >= 1)
    assert np.all(dk[0, 0, 0] == 0) and np.all(dv[0, 0, 0] == 0)
    # an entirely empty band
    g2 = Geometry(**{**g.as_dict(), "pre_tokens": -3, "next_tokens": 1})
    out2, smax2, ssum2 = orc.forward(to_problem(g2), inp.q, inp.k, inp.v)
    assert np.all(out2 == 0) and np.all(np.isneginf(smax2)) and np.all(ssum2 == 0)


def test_given_stats_mode_matches_exact_mode():
    g = Geometry("BNSD", 1, 2, 8, S_q=20, S_kv=20, scale=0.4, sparse_mode=4, pre_tokens=4, next_tokens=1,
                 keep_prob=0.85)
    inp = draw(g, 18)
    pr = to_problem(g)
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    a = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    b = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask, out, smax, ssum)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-15)


# ---------------------------------------------- sampled entry points -------
@pytest.mark.parametrize("layout", ["BNSD", "TND"])
def test_sampled_entry_points_match_full(layout):
    if layout == "BNSD":
        g = Geometry("BNSD", 2, 2, 8, S_q=40, S_kv=40, scale=0.4, sparse_mode=4, pre_tokens=6, next_tokens=2,
                     keep_prob=0.9)
        nq, nk = 2 * 40 * 2, 2 * 40 * 2
    else:
        g = Geometry("TND", 3, 2, 8, cu_seqlens_q=[10, 30, 37], cu_seqlens_kv=[10, 30, 37], scale=0.4,
                     sparse_mode=4, pre_tokens=5, next_tokens=5, keep_prob=0.9)
        nq, nk = 37 * 2, 37 * 2
    inp = draw(g, 19)
    pr = to_problem(g)
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    rows = np.array([0, 3, 17, nq - 1, nq // 2])
    cols = np.array([0, 5, 21, nk - 1, nk // 3])
    o_s, m_s, l_s = orc.forward_rows(pr, inp.q, inp.k, inp.v, inp.drop_mask, rows)
    dq_s = orc.backward_dq_rows(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask, rows)
    dk_s, dv_s = orc.backward_dkv_cols(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask, cols)
    D = g.D
    if layout == "BNSD":
        flat_q = lambda a: a.reshape(-1, D)
        flat_s = lambda a: a.reshape(-1)
    else:  # TND rows are (t, n) -> flat id t*N + n, same as reshape
        flat_q = lambda a: a.reshape(-1, D)
        flat_s = lambda a: a.reshape(-1)
    assert np.array_equal(o_s, flat_q(out)[rows])
    assert np.array_equal(m_s, flat_s(smax)[rows])
    assert np.array_equal(l_s, flat_s(ssum)[rows])
    assert np.allclose(dq_s, flat_q(dq)[rows], rtol=1e-13, atol=1e-15)
    assert np.allclose(dk_s, flat_q(dk)[cols], rtol=1e-13, atol=1e-15)
    assert np.allclose(dv_s, flat_q(dv)[cols], rtol=1e-13, atol=1e-15)


def test_visible_pair_count_matches_dense_mask():
    for case in SDPA_CASES.values():
        pr = to_problem(Geometry(**case))
        dense = _dense_mask(pr, pr.S_q, pr.S_kv).sum() * pr.B * pr.N
        assert orc.visible_pairs(pr) == dense


# ------------------------------------------- grouped key/value heads (GQA) --
# The rule (aclnnFlashAttentionUnpaddingScoreGradV2 article §6.2): N is a
# non-zero integer multiple of N_kv; query head n reads key/value head
# n // (N / N_kv).  Pinned three ways: against the oracle's own per-head path
# on explicitly repeated K / V (dK, dV summed over each group), against torch
# SDPA with repeated K / V and autograd, and by finite differences.
GQA_CASES = {
    "bnsd_g2_band": dict(layout="BNSD", B=2, N=4, N_kv=2, D=8, S_q=19, S_kv=19, scale=0.4, sparse_mode=4,
                         pre_tokens=5, next_tokens=2),
    "bnsd_mqa_nomask": dict(layout="BNSD", B=1, N=3, N_kv=1, D=8, S_q=17, S_kv=23, scale=0.3, sparse_mode=0),
    "bnsd_g3_dropout": dict(layout="BNSD", B=1, N=6, N_kv=2, D=4, S_q=12, S_kv=12, scale=0.5, sparse_mode=4,
                            pre_tokens=3, next_tokens=3, keep_prob=0.75),
    "tnd_g2_band": dict(layout="TND", B=3, N=4, N_kv=2, D=8, cu_seqlens_q=[7, 7, 20], cu_seqlens_kv=[7, 7, 20],
                        scale=0.45, sparse_mode=4, pre_tokens=4, next_tokens=0),
}


def _repeat_heads(x, geom, G):
    """Repeat each key/value head G times along the head axis (BNSD axis 1, TND axis 1)."""
    return np.repeat(np.asarray(x), G, axis=1)


def _sum_groups(x, geom, G):
    """Sum each run of G consecutive heads (the inverse bookkeeping of _repeat_heads)."""
    x = np.asarray(x)
    shp = list(x.shape)
    shp[1:2] = [shp[1] // G, G]
    return x.reshape(shp).sum(axis=2)


@pytest.mark.parametrize("name", sorted(GQA_CASES))
def test_gqa_equals_per_head_on_repeated_kv(name):
    case = GQA_CASES[name]
    geom = Geometry(**case)
    G = geom.N // geom.N_kv
    inp = draw(geom, 3000 + len(name))
    pr = to_problem(geom)
    mha = to_problem(Geometry(**{**case, "N_kv": 0}))
    q, k, v, dy = (t.double().numpy() for t in (inp.q, inp.k, inp.v, inp.dy))
    kr, vr = _repeat_heads(k, geom, G), _repeat_heads(v, geom, G)
    out, smax, ssum = orc.forward(pr, q, k, v, inp.drop_mask)
    out_r, smax_r, ssum_r = orc.forward(mha, q, kr, vr, inp.drop_mask)
    assert np.array_equal(out, out_r) and np.array_equal(smax, smax_r) and np.array_equal(ssum, ssum_r)
    dq, dk, dv = orc.backward(pr, q, k, v, dy, inp.drop_mask)
    dq_r, dk_r, dv_r = orc.backward(mha, q, kr, vr, dy, inp.drop_mask)
    assert dk.shape == k.shape and dv.shape == v.shape
    assert np.array_equal(dq, dq_r)
    assert np.allclose(dk, _sum_groups(dk_r, geom, G), rtol=1e-12, atol=1e-14)
    assert np.allclose(dv, _sum_groups(dv_r, geom, G), rtol=1e-12, atol=1e-14)
    # the key-column entry point agrees with the full backward
    cols = np.arange(geom.B * geom.n_kv * geom.S_kv if geom.layout == "BNSD" else geom.T_kv * geom.n_kv)
    ck, cv = orc.backward_dkv_cols(pr, q, k, v, dy, inp.drop_mask, cols)
    assert np.allclose(ck, dk.reshape(-1, geom.D), rtol=1e-12, atol=1e-14)
    assert np.allclose(cv, dv.reshape(-1, geom.D), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("name", ["bnsd_g2_band", "bnsd_mqa_nomask"])
def test_gqa_against_sdpa_float64(name):
    case = GQA_CASES[name]
    geom = Geometry(**case)
    G = geom.N // geom.N_kv
    inp = draw(geom, 4000 + len(name))
    pr = to_problem(geom)
    out, _, _ = orc.forward(pr, inp.q, inp.k, inp.v)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy)
    q = inp.q.double().requires_grad_(True)
    k = inp.k.double().requires_grad_(True)
    v = inp.v.double().requires_grad_(True)
    m = torch.from_numpy(_dense_mask(pr, geom.S_q, geom.S_kv))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k.repeat_interleave(G, dim=1),
                                                           v.repeat_interleave(G, dim=1), attn_mask=m,
                                                           scale=geom.scale)
    ref.backward(inp.dy.double())
    assert np.allclose(out, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dq, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    assert np.allclose(dk, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    assert np.allclose(dv, v.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_gqa_finite_differences():
    case = dict(layout="BNSD", B=1, N=4, N_kv=2, D=3, S_q=6, S_kv=6, scale=0.8, sparse_mode=4, pre_tokens=2,
                next_tokens=1, keep_prob=0.7)
    geom, inp = _fd_inputs(case, 5001)
    pr = to_problem(geom)
    q, k, v, dy = (t.double().numpy() for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask
    dq, dk, dv = orc.backward(pr, q, k, v, dy, mask)

    def loss(qq, kk, vv):
        out, _, _ = orc.forward(pr, qq, kk, vv, mask)
        return float(np.sum(out * dy))

    h = 1e-6
    for which, base, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(base)
        flat = base.reshape(-1)
        for idx in range(flat.size):
            save = flat[idx]
            flat[idx] = save + h
            lp = loss(q, k, v)
            flat[idx] = save - h
            lm = loss(q, k, v)
            flat[idx] = save
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm((num - grad).ravel()) / max(np.linalg.norm(num.ravel()), 1e-30)
        assert err <= 1e-6, (which, err)


def test_gqa_rejects_non_multiple():
    geom = Geometry("BNSD", 1, 4, 8, S_q=8, S_kv=8, N_kv=3)
    with pytest.raises(ValueError):
        orc.forward(to_problem(geom), np.zeros((1, 4, 8, 8)), np.zeros((1, 3, 8, 8)), np.zeros((1, 3, 8, 8)))


# ------------------------------------------------------ generated dropout --
# Philox4x32-10 (Salmon et al., SC'11) is pinned by the known-answer vectors
# published with its reference implementation (Random123): counter / key
# all zeros, all ones, and the hex digits of pi.
PHILOX_KAT = [
    ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    assert list(orc.philox4x32_10(ctr, key)) == want


def _mask_bits(mask, nbits):
    return np.unpackbits(mask, bitorder="little")[:nbits].astype(bool)


@pytest.mark.parametrize("keep", [0.5, 0.9, 0.25])
def test_generated_mask_keep_fraction(keep):
    geom = Geometry("BNSD", 2, 3, 8, S_q=160, S_kv=200, keep_prob=keep)
    pr = to_problem(geom)
    bits = _mask_bits(orc.generate_keep_mask(pr, seed=1234, offset=7), geom.mask_bits())
    p = round(keep * 256) / 256  # the generator's probability (an 8-bit threshold)
    n = bits.size
    # within 5 standard deviations of the binomial mean
    assert abs(bits.sum() - p * n) <= 5 * math.sqrt(n * p * (1 - p))
    # and no structure along keys: the 16 key positions of a block keep alike
    by_pos = bits.reshape(-1, 200)[:, :192].reshape(-1, 16).mean(axis=0)
    assert np.all(np.abs(by_pos - p) < 0.05)


def test_generated_mask_seed_offset_and_bounds():
    geom = Geometry("TND", 3, 2, 8, cu_seqlens_q=[40, 40, 97], cu_seqlens_kv=[35, 50, 120], keep_prob=0.8)
    pr = to_problem(geom)
    m0 = orc.generate_keep_mask(pr, 5, 0)
    assert np.array_equal(m0, orc.generate_keep_mask(pr, 5, 0))
    assert not np.array_equal(m0, orc.generate_keep_mask(pr, 6, 0))
    assert not np.array_equal(m0, orc.generate_keep_mask(pr, 5, 1))
    # keep_prob 1 keeps everything, a threshold of 0 nothing
    one = to_problem(Geometry(**{**geom.as_dict(), "keep_prob": 1.0}))
    assert _mask_bits(orc.generate_keep_mask(one, 5, 0), geom.mask_bits()).all()
    zero = to_problem(Geometry(**{**geom.as_dict(), "keep_prob": 1e-4}))
    assert not _mask_bits(orc.generate_keep_mask(zero, 5, 0), geom.mask_bits()).any()


# ------------------------------------------- visible windows (key_ranges) --
KEY_RANGE_CASES = {
    **SDPA_CASES,
    "band_negative_pre": dict(layout="BNSD", B=1, N=2, D=8, S_q=60, S_kv=60, scale=0.3, sparse_mode=4,
                              pre_tokens=-5, next_tokens=9),
    "band_negative_next": dict(layout="BNSD", B=2, N=1, D=8, S_q=50, S_kv=50, scale=0.3, sparse_mode=4,
                               pre_tokens=12, next_tokens=-4),
    "rect_wide_kv": dict(layout="BNSD", B=1, N=1, D=8, S_q=17, S_kv=90, scale=0.3, sparse_mode=4, pre_tokens=3,
                         next_tokens=40),
    "tnd_band_skipped": dict(layout="TND", B=5, N=3, D=8, cu_seqlens_q=[20, 20, 61, 0, 0],
                             cu_seqlens_kv=[31, 40, 70, 0, 0], scale=0.3, sparse_mode=4, pre_tokens=6,
                             next_tokens=2),
    "tnd_nomask": dict(layout="TND", B=3, N=2, D=8, cu_seqlens_q=[9, 30, 44], cu_seqlens_kv=[12, 12, 40],
                       scale=0.3, sparse_mode=0),
}


def _windows_dense(geom):
    """(lo, hi) of every statistics row from the dense BAND mask, -1 / -2 for
    a row that sees no key; rows in statistics order ([B,N,S] / [T,N])."""
    pr = to_problem(geom)
    out = []
    for b, (lq, lk) in enumerate(geom.seq_lens()):
        if lq == 0:
            continue
        if lk == 0:  # a sequence without keys: every row is empty
            out.append((np.full(lq, -1), np.full(lq, -2)))
            continue
        m = _dense_mask(pr, lq, lk)
        lo = np.where(m.any(1), m.argmax(1), -1)
        hi = np.where(m.any(1), lk - 1 - m[:, ::-1].argmax(1), -2)
        out.append((lo, hi))
    rows_lo, rows_hi = [], []
    if geom.layout == "BNSD":
        for lo, hi in out:
            for _ in range(geom.N):
                rows_lo.append(lo)
                rows_hi.append(hi)
        return np.concatenate(rows_lo), np.concatenate(rows_hi)
    for lo, hi in out:  # [T, N]: every head of a token in turn
        rows_lo.append(np.repeat(lo, geom.N))
        rows_hi.append(np.repeat(hi, geom.N))
    return np.concatenate(rows_lo), np.concatenate(rows_hi)


@pytest.mark.parametrize("name", sorted(KEY_RANGE_CASES))
def test_key_ranges_equal_dense_mask(name):
    geom = Geometry(**KEY_RANGE_CASES[name])
    pr = to_problem(geom)
    rows = np.arange(int(np.prod(geom.stat_shape())))
    lo, hi = orc.key_ranges(pr, rows)
    dlo, dhi = _windows_dense(geom)
    empty = dlo < 0
    assert np.array_equal(lo > hi, empty)
    # an empty row is reported as lo = 0, hi = -1
    assert np.all(lo[empty] == 0) and np.all(hi[empty] == -1)
    assert np.array_equal(lo[~empty], dlo[~empty]) and np.array_equal(hi[~empty], dhi[~empty])
    # rows past the table (beyond the last statistics row) see nothing
    lo2, hi2 = orc.key_ranges(pr, np.array([rows.size, rows.size + 7]))
    assert np.all(lo2 > hi2)


# -------------------------------- edge probe: one-pair window errors show --
EDGE_CASES = {
    "band": dict(layout="BNSD", B=1, N=2, D=64, S_q=400, S_kv=400, sparse_mode=4, pre_tokens=120, next_tokens=5),
    "band_negative_pre": dict(layout="BNSD", B=1, N=1, D=64, S_q=300, S_kv=300, sparse_mode=4, pre_tokens=-40,
                              next_tokens=90),
    "rect_band": dict(layout="BNSD", B=2, N=1, D=64, S_q=150, S_kv=400, sparse_mode=4, pre_tokens=10,
                      next_tokens=200),
    "tnd_band": dict(layout="TND", B=3, N=2, D=64, cu_seqlens_q=[150, 150, 420], cu_seqlens_kv=[130, 140, 500],
                     sparse_mode=4, pre_tokens=60, next_tokens=90),
    "gqa_band": dict(layout="BNSD", B=1, N=4, N_kv=2, D=64, S_q=300, S_kv=300, sparse_mode=4, pre_tokens=100,
                     next_tokens=30),
}


def _key_flat_ids(geom, b, j):
    """Flat key-row ids (rows of dk / dv reshaped to [-1, D]) of local key j of
    sequence b, one per key/value head."""
    nkv = geom.n_kv
    if geom.layout == "BNSD":
        return [(b * nkv + h) * geom.S_kv + j for h in range(nkv)]
    start = sum(lk for _, lk in geom.seq_lens()[:b])
    return [(start + j) * nkv + h for h in range(nkv)]


def _changed(geom, pr_a, pr_b):
    """Rows (statistics ids) whose window under pr_b differs from the true
    one under pr_a, and the flat key ids whose set of seeing rows differs.

    Only rows that see a key under pr_a count: a row the forward found empty
    has P = 0 in both backward passes whatever window they use, so an error
    there changes nothing.  A row left with no key by pr_b after one key
    under pr_a counts for its key (dV loses P * dY) but not for dQ: the
    dS of a lone pair is P * (dP - P dP) = 0."""
    rows = np.arange(int(np.prod(geom.stat_shape())))
    la, ha = orc.key_ranges(pr_a, rows)
    lb, hb = orc.key_ranges(pr_b, rows)
    ea, eb = la > ha, lb > hb
    diff = ~ea & ~((la == lb) & (ha == hb) & ~eb)
    lone_lost = diff & eb & (ha == la)
    keys = set()
    seq_of_row, local = [], []
    for b, (lq, _) in enumerate(geom.seq_lens()):
        seq_of_row += [b] * lq
        local += list(range(lq))
    for r in np.nonzero(diff)[0]:
        if geom.layout == "BNSD":
            b = r // (geom.N * geom.S_q)
        else:
            b = seq_of_row[r // geom.N]
        sa = set() if ea[r] else set(range(la[r], ha[r] + 1))
        sb = set() if eb[r] else set(range(lb[r], hb[r] + 1))
        for j in sa ^ sb:
            keys.update(_key_flat_ids(geom, b, j))
    return np.nonzero(diff & ~lone_lost)[0], np.array(sorted(keys), dtype=np.int64)


@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_edge_probe_exposes_one_pair_window_errors(name):
    """A backward pass whose window has one pair too many or too few at an
    edge (it recomputes P from the forward's statistics over the wrong set)
    moves dQ (query-major pass) on every row it touches and dV (key-major
    pass) on every key it touches by more than three times the element gate
    (2e-2 + half a bf16 ulp) of the GPU parity tests: the edge probe makes
    the GPU masked-set tests exact up to one pair."""
    geom = Geometry(**{**EDGE_CASES[name], "scale": math.log(2.0)})
    inp = draw(geom, 13)
    for alpha, edge in ((-1.0, "pre_tokens"), (1.0, "next_tokens")):
        q, k, v, dy = edge_probe_inputs(geom, inp.k, inp.dy, alpha)
        pr = to_problem(geom)
        out, m, l = orc.forward(pr, q, k, v)
        dq_t, _, dv_t = orc.backward(pr, q, k, v, dy, None, out, m, l)
        D = geom.D
        for delta in (+1, -1):
            bad = to_problem(Geometry(**{**geom.as_dict(), edge: getattr(geom, edge) + delta}))
            dq_b, _, dv_b = orc.backward(bad, q, k, v, dy, None, out, m, l)
            rows, keys = _changed(geom, pr, bad)
            assert rows.size > 0 and keys.size > 0, (name, edge, delta)
            rq_t, rq_b = dq_t.reshape(-1, D)[rows, 4:], dq_b.reshape(-1, D)[rows, 4:]
            gate = TOL_ABS + half_ulp(rq_t, "bf16")
            assert np.all(np.max(np.abs(rq_b - rq_t) - 3 * gate, axis=1) > 0), (name, edge, delta, "dq")
            kv_t, kv_b = dv_t.reshape(-1, D)[keys, 4:], dv_b.reshape(-1, D)[keys, 4:]
            gate = TOL_ABS + half_ulp(kv_t, "bf16")
            assert np.all(np.max(np.abs(kv_b - kv_t) - 3 * gate, axis=1) > 0), (name, edge, delta, "dv")


# ------------------------------------------------------- rounding budgets --
# orc_rounding_budget is test support: the per-element sums of absolute
# values that bound the drift of out / dQ / dK / dV when the products'
# operands are rounded to 16 bits (the tolerance of the GPU cases outside
# the workloads' regime).  Its pins: equality where every term has one sign
# (closed forms), the triangle inequality, and invariance / linearity in dY.

def test_budget_equals_result_when_every_term_is_positive():
    """v > 0 makes every term of out_i = sum_j P~_ij v_j positive, dY > 0
    every term of dV_j = sum_i P~_ij dY_i: there the budgets are the results
    (with dropout, so the z / keep weights are in both)."""
    g = Geometry(layout="BNSD", B=1, N=2, D=16, S_q=70, S_kv=70, scale=0.25, sparse_mode=4, pre_tokens=20,
                 next_tokens=5, keep_prob=0.8)
    inp = draw(g, 501)
    pr = to_problem(g)
    v = inp.v.double().abs().numpy() + 0.01
    dy = inp.dy.double().abs().numpy() + 0.01
    out, _, _ = orc.forward(pr, inp.q, inp.k, v, inp.drop_mask)
    _, _, dv = orc.backward(pr, inp.q, inp.k, v, dy, inp.drop_mask)
    out_b, _, _, dv_b = orc.rounding_budget(pr, inp.q, inp.k, v, dy, inp.drop_mask)
    np.testing.assert_allclose(out_b, out, rtol=1e-12, atol=0.0)
    np.testing.assert_allclose(dv_b, dv, rtol=1e-12, atol=0.0)


def test_dq_budget_is_exact_for_two_keys_of_opposite_sign():
    """D = 1 and every query sees keys i - 1 and i (BAND(1, 0)).  The two
    dS of a row sum to zero (sum_j P_ij (dP_ij - D_i) = 0), so
    dQ_i = scale dS_{i,i-1} (k_{i-1} - k_i); with k alternating in sign,
    |dQ_i| = |scale| |dS_{i,i-1}| (|k_{i-1}| + |k_i|), which is its budget."""
    S = 40
    g = Geometry(layout="BNSD", B=1, N=1, D=1, S_q=S, S_kv=S, scale=0.7, sparse_mode=4, pre_tokens=1, next_tokens=0)
    pr = to_problem(g)
    rng = np.random.default_rng(7)
    sign = np.where(np.arange(S) % 2 == 0, 1.0, -1.0).reshape(1, 1, S, 1)
    q = rng.normal(size=(1, 1, S, 1))
    k = (np.abs(rng.normal(size=(1, 1, S, 1))) + 0.1) * sign
    v = rng.normal(size=(1, 1, S, 1))
    dy = rng.normal(size=(1, 1, S, 1))
    dq, _, _ = orc.backward(pr, q, k, v, dy)
    _, dq_b, _, _ = orc.rounding_budget(pr, q, k, v, dy)
    assert np.max(np.abs(dq)) > 1e-3  # not a trivial zero
    np.testing.assert_allclose(dq_b, np.abs(dq), rtol=1e-10, atol=1e-15)


def test_budget_bounds_the_result_and_ignores_signs():
    """Every budget is at least the absolute result (triangle inequality),
    on a grouped-head BAND case with dropout; dY -> -dY flips dS and
    P~ dY but not their absolute values, and 2 dY doubles the three
    backward budgets while the forward's, which has no dY, stays."""
    g = Geometry(layout="BNSD", B=1, N=4, N_kv=2, D=32, S_q=150, S_kv=150, scale=0.2, sparse_mode=4, pre_tokens=60,
                 next_tokens=10, keep_prob=0.8)
    inp = draw(g, 502)
    pr = to_problem(g)
    out, _, _ = orc.forward(pr, inp.q, inp.k, inp.v, inp.drop_mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    b = orc.rounding_budget(pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    for got, bud in zip((out, dq, dk, dv), b):
        assert np.all(bud >= np.abs(got) * (1.0 - 1e-12) - 1e-15)
        assert np.max(bud - np.abs(got)) > 0.0  # strict somewhere: the terms do cancel
    bn = orc.rounding_budget(pr, inp.q, inp.k, inp.v, -inp.dy, inp.drop_mask)
    b2 = orc.rounding_budget(pr, inp.q, inp.k, inp.v, 2 * inp.dy, inp.drop_mask)
    for x, y in zip(b, bn):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=0.0)
    for x, y in zip(b[1:], b2[1:]):
        np.testing.assert_allclose(2.0 * x, y, rtol=1e-12, atol=0.0)
    np.testing.assert_allclose(b[0], b2[0], rtol=1e-12, atol=0.0)


def test_rounding_error_bound_composition():
    """The composed bounds are linear in the unit roundoff, and the forward's
    and dV's are u times their budgets (no D term there)."""
    g = Geometry(layout="BNSD", B=1, N=4, N_kv=2, D=32, S_q=150, S_kv=150, scale=0.2, sparse_mode=4, pre_tokens=60,
                 next_tokens=10, keep_prob=0.8)
    inp = draw(g, 503)
    pr = to_problem(g)
    args = (pr, inp.q, inp.k, inp.v, inp.dy, inp.drop_mask)
    u = 2.0 ** -8
    e1, e2 = orc.rounding_error(*args, u=u), orc.rounding_error(*args, u=2 * u)
    for x, y in zip(e1, e2):
        np.testing.assert_allclose(2.0 * x, y, rtol=1e-12, atol=0.0)
    b = orc.rounding_budget(*args)
    np.testing.assert_allclose(e1[0], u * b[0], rtol=1e-12, atol=0.0)
    np.testing.assert_allclose(e1[3], u * b[3], rtol=1e-12, atol=0.0)
    for j in (1, 2):  # dQ and dK carry the D term on top of u times their budgets
        assert np.all(e1[j] >= u * b[j] * (1.0 - 1e-12))
        assert np.max(e1[j] - u * b[j]) > 0.0


def test_rounding_error_d_term_matches_a_perturbed_output():
    """The D term through the oracle's own backward: with q, k > 0, shifting
    the given O by sign(dY) u (out_b + |O|) moves D_i by exactly dD_i, and
    the given-stats backward then moves dQ and dK by exactly the D terms of
    their bounds (dS_ij moves by -P_ij dD_i, and every P_ij k_j and P_ij q_i
    is positive)."""
    S, D = 90, 16
    g = Geometry(layout="BNSD", B=1, N=2, D=D, S_q=S, S_kv=S, scale=0.3, sparse_mode=4, pre_tokens=25, next_tokens=4)
    pr = to_problem(g)
    rng = np.random.default_rng(11)
    q = rng.uniform(0.1, 1.0, size=(1, 2, S, D))
    k = rng.uniform(0.1, 1.0, size=(1, 2, S, D))
    v = rng.normal(size=(1, 2, S, D))
    dy = rng.normal(size=(1, 2, S, D))
    u = 2.0 ** -8
    out, smax, ssum = orc.forward(pr, q, k, v)
    out_b, dq_b, dk_b, _ = orc.rounding_budget(pr, q, k, v, dy)
    _, dq_e, dk_e, _ = orc.rounding_error(pr, q, k, v, dy, u=u)
    shifted = out + np.sign(dy) * u * (out_b + np.abs(out))
    dq0, dk0, _ = orc.backward(pr, q, k, v, dy, None, given_out=out, given_max=smax, given_sum=ssum)
    dq1, dk1, _ = orc.backward(pr, q, k, v, dy, None, given_out=shifted, given_max=smax, given_sum=ssum)
    np.testing.assert_allclose(np.abs(dq1 - dq0), dq_e - u * dq_b, rtol=1e-7, atol=1e-15)
    np.testing.assert_allclose(np.abs(dk1 - dk0), dk_e - u * dk_b, rtol=1e-7, atol=1e-15)
