"""swa_backward_noalloc: the backward for callers that cannot hand the library
device memory (a plugin whose host framework owns all device memory, a loop
that must not allocate after start-up).  It uses a fixed scratch array
compiled into the library instead of a workspace.

The GPU test calls it through the C ABI, twice in a row and then on a
different problem, and checks each result against swa_backward (the entry
point with a caller workspace) with the parity gates of the other GPU
tests (tests/helpers.py).  The file sorts last so that a run stopping at the first failure has
already run everything else; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw
from tests.helpers import TOL_GRAD, check_tensor

PROBLEMS = [
    Geometry("BNSD", 2, 3, 64, S_q=700, S_kv=700, scale=0.125, sparse_mode=4, pre_tokens=200, next_tokens=33,
             keep_prob=0.9),
    Geometry("TND", 3, 2, 128, cu_seqlens_q=[300, 300, 801], cu_seqlens_kv=[300, 300, 801], scale=128 ** -0.5,
             sparse_mode=0),
]


@pytest.fixture(scope="module")
def lib():
    B.build()
    return swa.lib()


def _case(geom, seed):
    inp = draw(geom, seed)
    dev = torch.device("cuda:0")
    t = {n: getattr(inp, n).to(dev) for n in ("q", "k", "v", "dy")}
    t["mask"] = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    t["out"], t["smax"], t["ssum"] = swa.forward(geom, t["q"], t["k"], t["v"], t["mask"])
    ref = swa.backward(geom, t["q"], t["k"], t["v"], t["dy"], t["out"], t["smax"], t["ssum"], t["mask"])
    torch.cuda.synchronize()
    return t, [r.double().cpu().numpy() for r in ref]


def _noalloc(geom, t):
    p = swa.Params(geom)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    ptr = lambda x: None if x is None else x.data_ptr()
    st = swa.swa_backward_noalloc(p, ptr(t["q"]), ptr(t["k"]), ptr(t["v"]), ptr(t["dy"]), ptr(t["out"]),
                                  ptr(t["smax"]), ptr(t["ssum"]), ptr(t["mask"]), ptr(dq), ptr(dk), ptr(dv),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == swa.SWA_OK, swa.swa_last_error()
    torch.cuda.synchronize()
    return [x.double().cpu().numpy() for x in (dq, dk, dv)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward(lib):
    t0, ref0 = _case(PROBLEMS[0], 31)
    t1, ref1 = _case(PROBLEMS[1], 32)
    # two calls in a row on the same problem, then a different problem:
    # the shared scratch must be cleared by every call
    for call, (geom, t, ref) in enumerate(((PROBLEMS[0], t0, ref0), (PROBLEMS[0], t0, ref0),
                                           (PROBLEMS[1], t1, ref1))):
        got = _noalloc(geom, t)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            check_tensor(f"no-alloc call {call}", name, g, r, "bf16", TOL_GRAD)


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    # 4 x 256 x 16384 query rows need 8 bytes each (134 MB) of scratch:
    # rejected on the host before any device work (no GPU needed)
    g = Geometry("BNSD", 4, 256, 128, S_q=16384, S_kv=16384, scale=0.088, sparse_mode=4, pre_tokens=4096,
                 next_tokens=0)
    p = swa.Params(g)
    fake = 1 << 20
    st = swa.swa_backward_noalloc(p, fake, fake, fake, fake, fake, fake, fake, None, fake, fake, fake, None)
    assert st == swa.SWA_ERR_WORKSPACE
    assert "64 MiB" in swa.swa_last_error()
