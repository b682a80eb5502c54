"""Throughput benchmark of sliding-window attention forward + backward.

One step = one pass of the whole hot path over one batch of synthetic input:
swa_forward (band/varlen schedule, forward kernel) then swa_backward
(preprocess, key-major backward kernel, dQ conversion), through the C ABI.

Default workload: BNSD B=1, N=32, S=32768, D=128, BAND pre=4096 next=0, bf16
inputs ~N(0,1) from a fixed seed (the long sliding-window case).  Each of
q, k, v, dy is 268 MB, larger than the 129 MB L2, so no flush is needed
between steps.  The metric counts FLOPs over visible (i, j) pairs only:
4*D per pair forward, 10*D per pair backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl swa|reference]

For N > 1 (torchrun, one process per GPU) every rank runs its own replica of
the workload (weak scaling, no data-path collective); rank 0 prints one JSON
line with the whole-job throughput over the slowest rank's time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_swa_forward_gb300.workloads import HEADLINE, WORKLOADS, Geometry, draw  # noqa: E402

METRIC = "SWA fwd+bwd TFLOPS (unmasked FLOPs, bf16) and % of GB300 bf16 dense peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
KERNEL_SOURCES = ["attention_swa_forward_gb300/csrc/swa_fwd.cu", "attention_swa_forward_gb300/csrc/swa_bwd_dkv.cu",
                  "attention_swa_forward_gb300/csrc/swa_bwd_dq.cu",
                  "attention_swa_forward_gb300/csrc/swa_device.cuh", "attention_swa_forward_gb300/csrc/sm103.cuh"]


# ------------------------------------------------------------- counting --
def visible_pairs(g: Geometry) -> int:
    """Visible (i, j) pairs over all heads, by the BAND inequality i-pre <= j <= i+next."""
    total = 0
    for lq, lk in g.seq_lens():
        if lq == 0 or lk == 0:
            continue
        i = np.arange(lq, dtype=np.int64)
        if g.sparse_mode == 4:
            lo = np.maximum(0, i - g.pre_tokens)
            hi = np.minimum(lk - 1, i + g.next_tokens)
        else:
            lo, hi = np.zeros_like(i), np.full_like(i, lk - 1)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return total * g.N


def flops(g: Geometry) -> dict:
    p = visible_pairs(g)
    return {"pairs": p, "fwd": 4.0 * g.D * p, "bwd": 10.0 * g.D * p, "total": 14.0 * g.D * p}


def forward_kernel_name(g: Geometry, dev) -> str:
    """The forward kernel the library launches: at D <= 64 one CTA per pair
    of query tiles when the pairs fill every SM at least once, otherwise one
    CTA per query tile (the rule swa_forward applies)."""
    if g.D > 64:
        return "swa_fwd_kernel"
    tiles = g.N * sum(-(-lq // 128) for lq, _ in g.seq_lens())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return "swa_fwd_pair_kernel" if tiles >= 2 * sms else "swa_fwd_kernel"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.4)

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw_slowdown": parts[5], "hw_thermal_slowdown": parts[6],
                             "sw_thermal_slowdown": parts[7], "sw_power_cap": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = sorted({k for r in load for k in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                                   "sw_power_cap") if r[k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(load), "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------- oracle leg --
def oracle_sample(g: Geometry, inp, max_rows: int = 8192):
    """Bounded sample of the workload for the CPU oracle: head 0 of batch 0,
    the first `max_rows` query / key positions (the same per-pair work)."""
    if g.layout == "BNSD":
        S = min(g.S_q, max_rows)
        sub = Geometry(**{**g.as_dict(), "B": 1, "N": 1, "S_q": S, "S_kv": min(g.S_kv, max_rows),
                          "keep_prob": 1.0})
        sl = lambda t, L: t[:1, :1, :L].contiguous()
        q, k, v, dy = sl(inp.q, S), sl(inp.k, sub.S_kv), sl(inp.v, sub.S_kv), sl(inp.dy, S)
        desc = f"head 0 of batch 0, first {S} positions ({sub.S_q}x{sub.S_kv} pairs under the same mask)"
    else:
        lq, lk = g.seq_lens()[0]
        L = min(lq, max_rows)
        sub = Geometry("TND", 1, 1, g.D, cu_seqlens_q=[L], cu_seqlens_kv=[min(lk, max_rows)], scale=g.scale,
                       pre_tokens=g.pre_tokens, next_tokens=g.next_tokens, sparse_mode=g.sparse_mode)
        q, k, v, dy = (t[:L, :1].contiguous() for t in (inp.q, inp.k, inp.v, inp.dy))
        desc = f"sequence 0, head 0, first {L} positions"
    return sub, (q, k, v, dy), desc


def time_oracle_step(sub: Geometry, tensors) -> tuple[float, float]:
    from oracle import swa_oracle as orc

    orc.build()
    pr = orc.Problem(**sub.as_dict())
    q, k, v, dy = tensors
    t0 = time.perf_counter()
    orc.forward(pr, q, k, v)
    orc.backward(pr, q, k, v, dy)
    dt = time.perf_counter() - t0
    return dt, flops(sub)["total"]


def cpu_baseline(g: Geometry, inp) -> dict:
    sub, tensors, desc = oracle_sample(g, inp, max_rows=32768)
    dt, fl = time_oracle_step(sub, tensors)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": desc + f"; fwd+bwd in {dt:.1f} s"}


# ------------------------------------------------------------- helpers --
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def whole_job_value(total_flops_per_rank: float, ws: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return ws * total_flops_per_rank / max_seconds / 1e12


# ----------------------------------------------------------------- arms --
def run_reference(args, g: Geometry, name: str):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOADS[name]
    inp = draw(w.geom, w.seed, w.lengths)
    sub, tensors, desc = oracle_sample(inp.geom, inp, max_rows=args.ref_rows)
    for _ in range(args.warmup):
        time_oracle_step(sub, tensors)
    times = []
    fl = flops(sub)["total"]
    for _ in range(args.steps):
        dt, _ = time_oracle_step(sub, tensors)
        times.append(dt)
    t = sum(times) / len(times)
    value = fl / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(inp.geom, name),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(g: Geometry, name: str) -> dict:
    q_bytes = 2 * int(np.prod(g.q_shape()))
    l2 = ("inputs larger than L2 (q/k/v/dy each > 129 MB), no flush" if q_bytes > 129e6 else
          "inputs smaller than L2, not flushed between steps")
    cfg = {"workload": name, "layout": g.layout, "B": g.B, "N": g.N, "D": g.D, "sparse_mode": g.sparse_mode,
           "pre_tokens": g.pre_tokens, "next_tokens": g.next_tokens, "keep_prob": g.keep_prob,
           "scale": g.scale, "l2": l2}
    if g.N_kv:
        cfg["N_kv"] = g.N_kv
    if g.keep_prob < 1.0:
        cfg["dropout"] = "keep bits generated from seed / offset" if g.dropout_gen else "packed keep mask input"
    if g.layout == "BNSD":
        cfg.update(S_q=g.S_q, S_kv=g.S_kv)
    else:
        cfg.update(cu_seqlens_q=g.cu_seqlens_q)
    return cfg


def run_swa(args, name: str):
    from attention_swa_forward_gb300 import build as B
    from attention_swa_forward_gb300 import swa

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or ws == 1:
        B.build()
    barrier(ws)
    swa.lib()

    w = WORKLOADS[name]
    geom = w.geom if args.heads is None else Geometry(**{**w.geom.as_dict(), "N": args.heads})
    if args.keep_prob is not None:
        geom = Geometry(**{**geom.as_dict(), "keep_prob": args.keep_prob})
    if args.dropout_gen and geom.keep_prob < 1.0:  # keep bits from (seed, offset) instead of a mask
        geom = Geometry(**{**geom.as_dict(), "dropout_gen": 1, "dropout_seed": w.seed, "dropout_offset": 0})
    inp = draw(geom, w.seed, w.lengths)
    g = inp.geom
    fl = flops(g)
    p = swa.Params(g)
    stream = torch.cuda.current_stream(dev)
    q, k, v, dy = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dy))
    mask = inp.drop_mask.to(dev) if inp.drop_mask is not None else None
    out = torch.empty_like(q)
    smax = torch.empty(g.stat_shape(), dtype=torch.float32, device=dev)
    ssum = torch.empty_like(smax)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_f = torch.empty(swa.swa_forward_workspace_size(p), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(swa.swa_backward_workspace_size(p), dtype=torch.uint8, device=dev)
    n_tables_f = n_tables_b = 1  # one launch per family while the work table fits one kernel parameter

    def step():
        swa.forward(g, q, k, v, mask, out, smax, ssum, ws_f, stream)
        swa.backward(g, q, k, v, dy, out, smax, ssum, mask, dq, dk, dv, ws_b, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    swa.check_workspace(ws_b)

    # ---- timed region: K steps, kernel events around the main kernels
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    for quad in evs:  # materialise the event handles on this stream
        for e in quad:
            e.record(stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier(ws)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    t_start.record(stream)
    for i in range(args.steps):
        swa.swa_set_timing_events([e.cuda_event for e in evs[i]])
        step()
    t_end.record(stream)
    swa.swa_set_timing_events()
    torch.cuda.synchronize(dev)
    sampler.mark(False)
    barrier(ws)
    clocks = sampler.stop() if rank == 0 else None
    swa.check_workspace(ws_b)
    sec = t_start.elapsed_time(t_end) / 1e3 / args.steps
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    dkv_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
    dq_ms = sum(e[4].elapsed_time(e[5]) for e in evs) / args.steps
    prep_ms = sum(e[6].elapsed_time(e[7]) for e in evs) / args.steps
    sec_max = max_over_ranks(sec, ws, dev)
    value = whole_job_value(fl["total"], ws, sec_max)

    # ---- end to end through the public API: pinned host in, host out
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdy = (t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.dy))
        hmask = inp.drop_mask.pin_memory() if inp.drop_mask is not None else None
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (out, smax, ssum, dq, dk, dv)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdy)) + (
            hmask.numel() if hmask is not None else 0)
        d2h = sum(t.numel() * t.element_size() for t in h_out)

        # swa_step_host (host buffers through the C ABI, copies overlapped with
        # the computation in head groups) wherever it applies; a packed keep
        # mask has no host-step form, so that case copies and calls the device API
        chunks = 0
        if hmask is None:
            n_kv = g.N_kv or g.N
            chunks = next(c for c in ((args.chunks,) if args.chunks else (16, 8, 4, 2, 1))
                          if g.N % c == 0 and n_kv % c == 0 and (c == 1 or g.keep_prob == 1.0))
            step_buf = torch.empty(swa.swa_step_host_buffer_size(p, chunks), dtype=torch.uint8, device=dev)

        def e2e_step():
            if chunks:
                swa.step_host(g, hq, hk, hv, hdy, *h_out, chunks=chunks, device_buffer=step_buf, stream=stream)
                return
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            dy.copy_(hdy, non_blocking=True)
            if hmask is not None:
                mask.copy_(hmask, non_blocking=True)
            step()
            for h, d in zip(h_out, (out, smax, ssum, dq, dk, dv)):
                h.copy_(d, non_blocking=True)

        # as many untimed steps as the device leg: the first copies from
        # freshly pinned buffers are slower than the rest
        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(3, args.steps)
        # events around each step on the caller's stream give its duration
        # (steps run one after the other: each starts behind the last one's
        # results); the figure is the wall-clock mean, the median and the
        # slowest step show whether a rare stalled step is in it
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_e2e)]
        barrier(ws)
        t0 = time.perf_counter()
        for e_begin, e_end in step_ev:
            e_begin.record(stream)
            e2e_step()
            e_end.record(stream)
        torch.cuda.synchronize(dev)
        t_e2e = (time.perf_counter() - t0) / n_e2e
        t_e2e = max_over_ranks(t_e2e, ws, dev)
        per_step = sorted(a.elapsed_time(b) for a, b in step_ev)
        e2e = {"value": whole_job_value(fl["total"], ws, t_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3, "steps": n_e2e,
               "step_ms_median": per_step[len(per_step) // 2], "step_ms_max": per_step[-1],
               "api": f"swa_step_host, {chunks} head groups" if chunks else "copies + swa_forward / swa_backward"}
        if chunks:
            swa.check_step_host(g, chunks, step_buf, stream)

    if rank != 0:
        barrier(ws)
        return 0

    peaks, source = load_peaks()
    # The measured burst peak (best of a few cuBLAS GEMMs) fits a timed region
    # shorter than about a second, where the clocks stay at their maximum;
    # the sustained one (seconds of back-to-back GEMMs under the power cap)
    # fits longer regions.
    region_s = sec_max * args.steps
    peak_key = "bf16_tflops" if region_s < 1.0 else "bf16_tflops_sustained"
    peak = peaks.get(peak_key, FALLBACK_PEAKS[peak_key])
    # algorithmic FLOPs per launch: forward 4*D per visible pair (QK^T, PV);
    # dK/dV pass 8*D (QK^T, dY V^T, P^T dY, dS^T Q); dQ pass 6*D (QK^T,
    # dY V^T, dS K).  Only 14*D per pair counts toward the metric.
    pairs_d = fl["pairs"] * g.D
    kernels = {
        forward_kernel_name(g, dev): {"ms": fwd_ms, "tflops": 4.0 * pairs_d / (fwd_ms / 1e3) / 1e12},
        "swa_bwd_dkv_kernel": {"ms": dkv_ms, "tflops": 8.0 * pairs_d / (dkv_ms / 1e3) / 1e12},
        "swa_bwd_dq_kernel": {"ms": dq_ms, "tflops": 6.0 * pairs_d / (dq_ms / 1e3) / 1e12},
    }
    dom = max(kernels, key=lambda kname: kernels[kname]["ms"])
    traffic = None
    try:
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("source_hash") == kernel_source_hash() and tr.get("workload") == name:
            traffic = tr.get("kernels", {}).get(dom)
    except Exception:
        traffic = None
    achieved = kernels[dom]["tflops"]
    for kd in kernels.values():
        kd["frac"] = kd["tflops"] / peak
    # the memory-bound preprocess: reads dY and O and the two statistics,
    # writes lse2 and D (algorithmic bytes per launch)
    # (16-bit dY and O: fp32 inputs reach it as bf16 copies)
    rows = g.B * g.N * g.S_q if g.layout == "BNSD" else g.T_q * g.N
    prep_bytes = rows * (2 * g.D * 2 + 4 * 4)
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    prep_gbs = prep_bytes / (prep_ms / 1e3) / 1e9
    memory_bound = {"kernel": "swa_prep_bulk_kernel", "bound": "hbm",
                    "ms": prep_ms, "bytes": prep_bytes, "achieved": prep_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": prep_gbs / hbm_peak, "peak_source": f"{source} hbm_gbs"}
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{source} {peak_key} (timed region {region_s:.2f} s of back-to-back steps)",
                "kernels": kernels, "memory_bound": memory_bound}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_max * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, shapes of the workload)",
        "config": workload_config(g, name if args.heads is None else f"{name} with N={g.N}"),
        "pct_of_bf16_peak": 100.0 * value / ws / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
        "flops_per_step": fl["total"], "visible_pairs": fl["pairs"],
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": args.steps * (n_tables_f + 1 + 2 * n_tables_b),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(g, inp)
    print(json.dumps(line), flush=True)
    barrier(ws)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["swa", "reference"], default="swa")
    ap.add_argument("--workload", default=HEADLINE, choices=list(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=8192, help="positions per oracle sample (reference arm)")
    ap.add_argument("--keep-prob", type=float, default=None, help="override the workload's keep_prob")
    ap.add_argument("--dropout-gen", action="store_true",
                    help="dropout workloads: generate the keep mask in the kernels from a seed / offset")
    ap.add_argument("--chunks", type=int, default=None,
                    help="head groups of the end-to-end host step (default: the largest of 16, 8, 4, 2, 1 that divides)")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count N (smaller profiling captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args, WORKLOADS[args.workload].geom, args.workload)
    return run_swa(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
