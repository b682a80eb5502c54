"""Bounded waits: a wait that runs out is reported, and the GPU stays usable.

Every mbarrier wait in the kernels gives up after 2 s, stores a code in the
workspace status word, lets the copies and tensor-core work already in
flight land, frees its tensor memory and returns; swa_workspace_status then
reports SWA_ERR_TIMEOUT (the operator-level "timeout" failure the
aclnnFlashAttentionUnpaddingScoreGradV2 article, §6.7, names for the
device).  The test hook swa_debug_stall makes the compute warps of one
kernel first wait on a barrier that nothing completes, so that wait runs out
for real: no fault, trap or endless loop is involved.  Afterwards a normal
call on fresh workspaces must still match the oracle.
"""
import numpy as np
import pytest
import torch

from attention_swa_forward_gb300 import build as B
from attention_swa_forward_gb300 import swa
from attention_swa_forward_gb300.workloads import Geometry, draw
from oracle import swa_oracle as orc
from tests.helpers import TOL_GRAD, TOL_OUT, check_stat, check_tensor, to_problem

pytestmark = pytest.mark.gpu

CASE = Geometry("BNSD", 1, 2, 128, S_q=600, S_kv=600, scale=128 ** -0.5, sparse_mode=4, pre_tokens=200,
                next_tokens=10)
KERNELS = {"forward": 1, "key_major": 2, "query_major": 4}


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    orc.build()
    swa.lib()


def _ws(geom, backward):
    p = swa.Params(geom)
    n = swa.swa_backward_workspace_size(p) if backward else swa.swa_forward_workspace_size(p)
    return torch.empty(n, dtype=torch.uint8, device="cuda:0")


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_wait_that_runs_out_is_reported(kernel):
    inp = draw(CASE, 31)
    dev = torch.device("cuda:0")
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    stream = torch.cuda.current_stream()
    ws_f, ws_b = _ws(CASE, False), _ws(CASE, True)
    try:
        if kernel == "forward":
            swa.swa_debug_stall(KERNELS[kernel])
        out, smax, ssum = swa.forward(CASE, q, k, v, workspace=ws_f)
        st_f = swa.swa_workspace_status(ws_f.data_ptr(), stream.cuda_stream)
        swa.swa_debug_stall(KERNELS[kernel])
        swa.backward(CASE, q, k, v, dy, out, smax, ssum, workspace=ws_b)
        st_b = swa.swa_workspace_status(ws_b.data_ptr(), stream.cuda_stream)
    finally:
        swa.swa_debug_stall(0)
    torch.cuda.synchronize()
    if kernel == "forward":
        assert st_f == swa.SWA_ERR_TIMEOUT, swa.swa_last_error()
    else:
        assert st_f == swa.SWA_OK
        assert st_b == swa.SWA_ERR_TIMEOUT, swa.swa_last_error()
    assert "bounded wait" in swa.swa_last_error()

    # the context is still usable: a normal call on fresh workspaces matches the oracle
    ws_f, ws_b = _ws(CASE, False), _ws(CASE, True)
    out, smax, ssum = swa.forward(CASE, q, k, v, workspace=ws_f)
    dq, dk, dv = swa.backward(CASE, q, k, v, dy, out, smax, ssum, workspace=ws_b)
    swa.check_workspace(ws_f)
    swa.check_workspace(ws_b)
    pr = to_problem(CASE)
    r_out, r_max, r_sum = orc.forward(pr, inp.q, inp.k, inp.v)
    r_dq, r_dk, r_dv = orc.backward(pr, inp.q, inp.k, inp.v, inp.dy)
    label = f"after a {kernel} timeout"
    got = lambda t: t.double().cpu().numpy()
    check_tensor(label, "out", got(out), r_out, "bf16", TOL_OUT)
    check_stat(label, "softmax_max", got(smax), r_max)
    check_stat(label, "softmax_sum", got(ssum), r_sum)
    for name, g, r in (("dq", dq, r_dq), ("dk", dk, r_dk), ("dv", dv, r_dv)):
        check_tensor(label, name, got(g), r, "bf16", TOL_GRAD)
    assert np.isfinite(got(out)).all()
