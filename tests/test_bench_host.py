"""Host logic of bench.py without a GPU: the multi-rank timing reduction over
gloo (world size 2), the whole-job throughput formula, the visible-pair count
against a brute-force mask, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from attention_swa_forward_gb300.workloads import WORKLOADS, Geometry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_time = 0.010 * (rank + 1)  # rank 1 is the slowest
    t = bench.max_over_ranks(my_time, world, torch.device("cpu"))
    bench.barrier(world)
    v = bench.whole_job_value(7.0e12, world, t)
    out_q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_rank_max_and_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == pytest.approx(0.020)
        assert v == pytest.approx(2 * 7.0e12 / 0.020 / 1e12)


def test_visible_pairs_brute_force():
    cases = [Geometry("BNSD", 2, 3, 64, S_q=37, S_kv=53, sparse_mode=4, pre_tokens=5, next_tokens=11),
             Geometry("BNSD", 1, 1, 64, S_q=40, S_kv=40, sparse_mode=0),
             Geometry("TND", 3, 2, 64, cu_seqlens_q=[10, 10, 30], cu_seqlens_kv=[5, 9, 30], sparse_mode=4,
                      pre_tokens=3, next_tokens=0)]
    for g in cases:
        brute = 0
        for lq, lk in g.seq_lens():
            i = np.arange(lq)[:, None]
            j = np.arange(lk)[None, :]
            m = np.ones((lq, lk), bool) if g.sparse_mode == 0 else (j >= i - g.pre_tokens) & (j <= i + g.next_tokens)
            brute += int(m.sum())
        assert bench.visible_pairs(g) == brute * g.N


def test_headline_flops():
    f = bench.flops(WORKLOADS["bnsd_1x32x32768x128_band4096"].geom)
    assert f["pairs"] == 32 * (4096 * 4097 // 2 + (32768 - 4096) * 4097)
    assert f["total"] == pytest.approx(14 * 128 * f["pairs"])


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "bnsd_1x2x256x64_nomask", "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "bnsd_1x2x256x64_nomask"
