"""Benchmark of the verify step on GB300.

One step = one sv_verify_sample call (lossless rejection sampling at T = 1:
streaming pass over every target and drafter row, residual draw, fp64 path)
over the lossless workload: B = 64 sequences, K = 16 draft tokens, V = 128256,
bf16 logits (541.75 MB of logits per step, larger than the 126 MB L2, so every
step streams from HBM).  Inputs are seeded synthetic tensors resident on the
GPU before the timed region.

Prints ONE JSON line (rank 0): verified draft rows/s for the whole job, the
roofline of the streaming kernel against the measured HBM copy bandwidth, the
end-to-end rate through the C ABI with host buffers, the CPU oracle baseline
and the SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): every rank verifies its own full batch (weak scaling, no
collective on the data path); value = all ranks' rows / max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import datagen  # noqa: E402

WORKLOAD = "lossless_t1"
METRIC = "verified draft rows/sec and logits HBM GB/s (fraction of GB300 peak), 1 GPU"
PROFILE = os.path.join(ROOT, "profiles", "pass_kernel_lossless_t1.md")
KERNEL_SOURCES = ["sv_pass.cu", "sv_common.cuh", "sv_dev.cuh", "sv_gumbel.cuh", "sv_job.cuh"]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "draft_block_verification_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic():
    """DRAM bytes per launch of the streaming kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != _kernel_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons every 50 ms; the
    timed region starts only after the first sample arrived."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        self.first = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = self.p.stdout.readline()  # sampler is running
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.p is None:
            return
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def _max_over_ranks(dist, x, dev):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist, dev):
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)


def _oracle_inputs(cfg, nseq):
    si = datagen.sample_inputs(nseq, cfg["K"], cfg["V"], dtype=cfg["dtype"], seed=cfg["seed"],
                               sigma=cfg["sigma"], T=cfg["T"], device="cpu")
    return (datagen.to_numpy_logits(si.target), datagen.to_numpy_logits(si.draft),
            si.draft_ids.numpy())


def _oracle_call(cfg, inputs):
    import oracle
    tgt, drf, ids = inputs
    t0 = time.perf_counter()
    oracle.verify_sample(tgt, drf, ids, seed=cfg["seed"], want_tv=False)
    return time.perf_counter() - t0


def cpu_baseline(cfg, nseq=None, inputs=None):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload:
    the first nseq sequences of the batch (all of them by default), generated
    on the CPU with the same recipe."""
    import oracle
    oracle.build()
    nseq = nseq or cfg["B"]
    inputs = inputs or _oracle_inputs(cfg, nseq)
    dt = _oracle_call(cfg, inputs)
    rows = nseq * cfg["K"]
    return {"value": rows / dt, "unit": "rows/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of %d sequences x %d drafts x V=%d (%s), one oracle verify call, "
                      "%.3f s wall" % (nseq, cfg["B"], cfg["K"], cfg["V"], cfg["dtype"], dt)}


def run_reference(args):
    """The reference arm is the CPU oracle (the pages ship no code): every step
    verifies a sample of the workload, sized so that the whole run stays
    within about two minutes."""
    dist, rank, ws = _dist()
    cfg = datagen.CONFIGS[WORKLOAD]
    if rank != 0:
        return
    import oracle
    oracle.build()
    full = _oracle_inputs(cfg, cfg["B"])
    t_full = _oracle_call(cfg, full)
    n_calls = max(1, args.warmup + args.steps)
    nseq = int(max(1, min(cfg["B"], cfg["B"] * 120.0 / (n_calls * max(t_full, 1e-6)))))
    inputs = full if nseq == cfg["B"] else tuple(a[:nseq] for a in full)
    vals = []
    cb = None
    for _ in range(n_calls):
        cb = cpu_baseline(cfg, nseq, inputs)
        vals.append(cb["value"])
    value = statistics.median(vals[args.warmup:]) if args.steps else cb["value"]
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * nseq * cfg["K"] / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": cfg["B"], "K": cfg["K"], "V": cfg["V"],
                       "logits": cfg["dtype"], "T": cfg["T"], "l2": "inputs larger than L2",
                       "sample_sequences_per_step": nseq},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ours(args):
    import draft_block_verification_gb300 as dbv
    dist, rank, ws = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dbv.build()
    cfg = dict(datagen.CONFIGS[WORKLOAD])
    if args.batch:
        cfg["B"] = args.batch
    B, K, V = cfg["B"], cfg["K"], cfg["V"]
    si = datagen.sample_inputs(B, K, V, dtype=cfg["dtype"], seed=cfg["seed"], sigma=cfg["sigma"],
                               T=cfg["T"], device=dev)
    h = dbv.default_handle(dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: dbv.sv_verify_sample(si.target, si.draft, si.draft_ids, T_p=cfg["T"],
                                        T_q=cfg["T"], seed=cfg["seed"], handle=h)
    for _ in range(max(args.warmup, 3)):
        call()
    h.sync_status()
    # per-launch events around the streaming kernel (recorded by the library
    # on the call's stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:  # torch creates the CUDA events at their first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    ptrs = [np.array([e[0].cuda_event, e[1].cuda_event], dtype=np.uint64) for e in evs]
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        _barrier(dist, dev)
        t_start.record(stream)
        for i in range(args.steps):
            h.set_option(dbv.SV_OPT_TIMING_EVENTS, int(ptrs[i].ctypes.data))
            call()
        t_stop.record(stream)
        _barrier(dist, dev)
    h.set_option(dbv.SV_OPT_TIMING_EVENTS, 0)
    h.sync_status()
    ms = t_start.elapsed_time(t_stop) / args.steps
    ms = _max_over_ranks(dist, ms, dev)
    kern_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    rows = B * K
    value = ws * rows / (ms / 1000.0)
    alg_bytes = B * (2 * K + 1) * V * 2
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (kern_ms / 1000.0) / 1e9

    # end to end: pinned host inputs -> device, the call, results -> host
    host = [t.detach().cpu().pin_memory() for t in (si.target, si.draft, si.draft_ids)]
    dst = [torch.empty_like(t, device=dev) for t in host]
    h2d = sum(t.numel() * t.element_size() for t in host)
    out_bytes = 0
    _barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(2, min(args.steps, 5))
    e0.record(stream)
    for _ in range(e_steps):
        for d, s in zip(dst, host):
            d.copy_(s, non_blocking=True)
        out = dbv.sv_verify_sample(dst[0], dst[1], dst[2], T_p=cfg["T"], T_q=cfg["T"],
                                   seed=cfg["seed"], handle=h)
        res = [out[k].to("cpu", non_blocking=True) for k in ("accept_len", "next_token",
                                                             "p_at_draft", "q_at_draft")]
        out_bytes = sum(r.numel() * r.element_size() for r in res)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = _max_over_ranks(dist, e0.elapsed_time(e1) / e_steps, dev)
    h.sync_status()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD if B == datagen.CONFIGS[WORKLOAD]["B"] else
                   "%s with B=%d" % (WORKLOAD, B), "B": B, "K": K, "V": V, "logits": "bf16",
                   "T": cfg["T"], "mode": "lossless", "outputs": "accept_len, next_token, "
                   "p/q at draft ids, lse",
                   "l2": "inputs larger than L2 (%.2f MB/step)" % (B * (2 * K + 1) * V * 2 / 1e6)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _profiled_traffic(),
                     "peak_source": peak_kind, "kernel": "pass_kernel", "kernel_ms": kern_ms,
                     "alg_bytes_per_launch": alg_bytes},
        "e2e": {"value": ws * rows / (e_ms / 1000.0), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_bytes},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the number of sequences (small cases for ncu captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
