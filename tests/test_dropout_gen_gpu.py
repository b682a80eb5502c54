"""Dropout from a seed and an offset (dropout_gen = 1) on the GPU.

The keep mask a seed / offset pair stands for is defined in include/swa.h
(Philox4x32-10 over (key block, query row, offset), 8-bit threshold).  These
tests check, through the C ABI:
- swa_dropout_mask writes exactly the oracle's mask for that definition
  (bit for bit: integer work);
- forward and backward with the mask generated inside the kernels agree
  with the oracle run on the oracle's mask (the parity tolerances of the
  other GPU tests);
- the in-kernel generation and the materialised mask give the same results
  bit for bit.
"""
import numpy as np
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw
from oracle import swa_oracle as orc
from tests.helpers import TOL_GRAD, TOL_OUT, check_stat, check_tensor, out_dtype, to_problem

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    orc.build()
    swa.lib()


MASKS = {
    "bnsd_rect": dict(layout="BNSD", B=2, N=3, D=64, S_q=200, S_kv=130, keep_prob=0.8, dropout_gen=1,
                      dropout_seed=1, dropout_offset=0),
    "bnsd_big_seed": dict(layout="BNSD", B=1, N=2, D=128, S_q=77, S_kv=301, keep_prob=0.5, dropout_gen=1,
                          dropout_seed=2 ** 40 + 5, dropout_offset=12345),
    "tnd_varlen": dict(layout="TND", B=4, N=2, D=64, cu_seqlens_q=[50, 50, 197, 0], cu_seqlens_kv=[70, 100, 260, 0],
                       keep_prob=0.6, dropout_gen=1, dropout_seed=99, dropout_offset=7),
}


@pytest.mark.parametrize("name", sorted(MASKS))
def test_materialised_mask_matches_oracle(name):
    geom = Geometry(**MASKS[name])
    got = swa.dropout_mask(geom).cpu().numpy()
    ref = orc.generate_keep_mask(to_problem(geom), geom.dropout_seed, geom.dropout_offset)
    nbits = geom.mask_bits()
    gbits = np.unpackbits(got, bitorder="little")
    rbits = np.unpackbits(ref, bitorder="little")[:nbits]
    assert np.array_equal(gbits[:nbits], rbits)
    assert not gbits[nbits:].any()  # padding stays zero


CASES = {
    "bnsd_symband_d64": dict(layout="BNSD", B=2, N=2, D=64, S_q=400, S_kv=400, scale=0.125, sparse_mode=4,
                             pre_tokens=70, next_tokens=90, keep_prob=0.8, dropout_gen=1, dropout_seed=7,
                             dropout_offset=3),
    "bnsd_band_d128_ragged": dict(layout="BNSD", B=1, N=2, D=128, S_q=333, S_kv=333, scale=0.09, sparse_mode=4,
                                  pre_tokens=150, next_tokens=40, keep_prob=0.7, dropout_gen=1,
                                  dropout_seed=2 ** 33 + 1, dropout_offset=99),
    "tnd_band_d64": dict(layout="TND", B=4, N=3, D=64, cu_seqlens_q=[200, 201, 460, 0],
                         cu_seqlens_kv=[200, 201, 460, 0], scale=0.125, sparse_mode=4, pre_tokens=100,
                         next_tokens=17, keep_prob=0.85, dropout_gen=1, dropout_seed=11, dropout_offset=0),
    "bnsd_gqa_d128": dict(layout="BNSD", B=1, N=4, N_kv=2, D=128, S_q=290, S_kv=290, scale=0.09, sparse_mode=4,
                          pre_tokens=100, next_tokens=30, keep_prob=0.75, dropout_gen=1, dropout_seed=5,
                          dropout_offset=1),
    "bnsd_band_d64_fp16": dict(layout="BNSD", B=1, N=3, D=64, S_q=270, S_kv=270, scale=0.125, sparse_mode=4,
                               pre_tokens=90, next_tokens=10, keep_prob=0.9, dropout_gen=1, dropout_seed=3,
                               dropout_offset=2, dtype="fp16"),
    "bnsd_band_d72": dict(layout="BNSD", B=1, N=2, D=72, S_q=300, S_kv=300, scale=72 ** -0.5, sparse_mode=4,
                          pre_tokens=110, next_tokens=20, keep_prob=0.8, dropout_gen=1, dropout_seed=17,
                          dropout_offset=4),
}


def _gpu(geom, inp, mask=None):
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    out, smax, ssum = swa.forward(geom, q, k, v, mask)
    ws = torch.empty(swa.swa_backward_workspace_size(swa.Params(geom)), dtype=torch.uint8, device=dev)
    dq, dk, dv = swa.backward(geom, q, k, v, dy, out, smax, ssum, mask, workspace=ws)
    swa.check_workspace(ws)
    torch.cuda.synchronize()
    return {n: t.cpu().double().numpy() for n, t in
            (("out", out), ("smax", smax), ("ssum", ssum), ("dq", dq), ("dk", dk), ("dv", dv))}


# every case with the forward's default kernel choice; the D <= 64 cases also
# with the forward forced onto one CTA per pair of query tiles
_RUNS = [(n, 0) for n in sorted(CASES)] + [(n, 1) for n in sorted(CASES) if CASES[n]["D"] <= 64]


@pytest.mark.parametrize("name,pairs", _RUNS, ids=[n + ("-pairs" if p else "") for n, p in _RUNS])
def test_generated_dropout_parity(name, pairs):
    geom = Geometry(**CASES[name])
    inp = draw(geom, 6000 + sum(map(ord, name)))
    assert inp.drop_mask is None  # the seed / offset stand for the mask
    pr = to_problem(geom)
    mask = orc.generate_keep_mask(pr, geom.dropout_seed, geom.dropout_offset)
    out, smax, ssum = orc.forward(pr, inp.q, inp.k, inp.v, mask)
    dq, dk, dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy, mask)
    swa.swa_debug_forward_pairs(pairs)
    try:
        res = _gpu(geom, inp)
    finally:
        swa.swa_debug_forward_pairs(0)
    dt = out_dtype(geom)
    label = f"generated dropout {name}" + (" (query tile pairs)" if pairs else "")
    check_tensor(label, "out", res["out"], out, dt, TOL_OUT)
    check_stat(label, "softmax_max", res["smax"], smax)
    check_stat(label, "softmax_sum", res["ssum"], ssum)
    for n, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tensor(label, n, res[n], ref, dt, TOL_GRAD)
    # the materialised mask through the drop_mask path gives the same bits out
    gm = swa.dropout_mask(geom)
    geom_mask = Geometry(**{**CASES[name], "dropout_gen": 0})
    res_m = _gpu(geom_mask, inp, gm)
    for n in res:
        assert np.array_equal(res[n], res_m[n]), n
