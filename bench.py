"""Benchmark of the verify step on GB300.

One step = one verify call over one batch of a named workload (default: the
Packed-SS step at T = 1 -- sv_packed_step over B = 256 sequences, K = 32
verify rows and W = 32 proposal rows per sequence, V = 151936, bf16 logits;
the call reads the required rows, about 3.7 GB per step, far larger than the
126 MB L2, so every step streams from HBM).  A call runs the whole verify
path: the streaming pass over every required row, the decisions, the
residual draw from the stored proposal rows and the fp64 check.  Inputs are
seeded synthetic tensors resident on the GPU before the timed region.

Prints ONE JSON line (rank 0): verified draft rows/s for the whole job, the
roofline of the streaming kernel against the measured HBM copy bandwidth, the
end-to-end rate through the C ABI with host buffers, the CPU oracle baseline
and the SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload packed|lossless_t1|lenient_sweep|tree|greedy_tiny]
                  [--T t] [--sigma s] [--lam l] [--mode lossless|ratio|linear]
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

WORKLOAD = "packed"
METRIC = "verified draft rows/sec and logits HBM GB/s (fraction of GB300 peak), 1 GPU"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["sv_pass.cu", "sv_common.cuh", "sv_dev.cuh", "sv_gumbel.cuh", "sv_job.cuh"]
TOPK_SOURCES = ["sv_topk.cu", "sv_topk.cuh", "sv_common.cuh", "sv_dev.cuh", "sv_gumbel.cuh"]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_hash(w=None):
    h = hashlib.sha256()
    for f in (TOPK_SOURCES if w is not None and w.kind == "packed_topk" else KERNEL_SOURCES):
        with open(os.path.join(ROOT, "draft_block_verification_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_path(w):
    """The committed ncu summary of the streaming kernel on this workload."""
    t = "" if w.kind == "greedy" or w.name.endswith("_t%g" % w.T) else "_t%g" % w.T
    return os.path.join(ROOT, "profiles", "%s_%s%s.md" % (w.kernel(), w.name, t))


def _profiled_traffic(w):
    """DRAM bytes per launch of the streaming kernel from the committed ncu
    summary of this workload, if it was taken on the current kernel source;
    else None."""
    try:
        text = open(_profile_path(w)).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != _kernel_hash(w):
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons every 20 ms.  The
    timed region starts only after the first sample arrived; that sample is
    kept (taken just before the region), so that a region shorter than the
    sampling interval still has a clock record; `in_region` counts the
    samples taken while it ran."""

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
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = self.p.stdout.readline()  # sampler is running
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        self.rows = []
        self.in_region = 0
        if self.p is None:
            return
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        lines = ([self.first] if self.first else []) + out.splitlines()
        for i, line in enumerate(lines):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)
                self.in_region += 1 if i > 0 else 0

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
                "samples": len(rows), "in_region": getattr(self, "in_region", 0)}


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
    if dev.type == "cuda":
        torch.cuda.synchronize(dev)


def job_rate(world_size, units_per_rank, ms_max):
    """Whole-job throughput: every rank processed units_per_rank units; the
    job took the slowest rank's time (ms)."""
    return world_size * units_per_rank / (ms_max / 1000.0)


def _percentiles(xs):
    """Median, 10th and 90th percentiles (ms) of per-step times."""
    a = np.asarray(xs, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# Workloads.  Each is one verify call on seeded synthetic inputs of the shapes
# and distributions the method is measured on.
# ---------------------------------------------------------------------------
class Workload:
    """One verify call of a named workload: inputs, the call through the
    library, the same call through the oracle, and the algorithmic bytes of
    the streaming kernel (required logit rows x V x element size)."""

    def __init__(self, name, args):
        self.name = name
        self.cfg = dict(datagen.CONFIGS[name])
        self.kind = self.cfg["kind"]
        c = self.cfg
        if args.batch:
            c["B"] = args.batch
        pick = lambda v, d: d if v is None else v
        if self.kind == "sample":
            # one point of the sweep (the lossless workload has a single point)
            self.T = pick(args.T, c["T"] if not isinstance(c["T"], tuple) else 1.0)
            self.sigma = pick(args.sigma, c["sigma"] if not isinstance(c["sigma"], tuple) else 1.0)
            self.mode = {"lossless": 0, "ratio": 1, "linear": 2, "cactus": 3}[
                args.mode or ("lossless" if name == "lossless_t1" else "ratio")]
            self.lam = pick(args.lam, 1.0 if self.mode == 0 else 2.0)
            if self.mode == 2 and args.lam is None:
                self.lam = 0.5  # mu = 1 - 1/lambda at lambda = 2
            # the lenient sweep reports the per-row TV(p, q) as well (a second
            # pass over every row pair); --no-tv leaves it out
            self.tv = name == "lenient_sweep" and not args.no_tv
        elif self.kind in ("tree", "packed", "spot"):
            self.T = pick(args.T, 1.0)
        elif self.kind == "anyorder":
            self.T = 0.0  # Alg. 3 is greedy
        elif self.kind == "packed_topk":
            self.T = pick(args.T, c["T"])
        else:
            self.T = 0.0
        self.esz = 2 if c["dtype"] == "bf16" else 4

    def point(self):
        c = self.cfg
        d = {"workload": self.name}
        if self.kind == "sample":
            d.update(B=c["B"], K=c["K"], V=c["V"], T=self.T, sigma=self.sigma,
                     mode=["lossless", "ratio", "linear", "cactus"][self.mode], lam=self.lam,
                     tv=self.tv)
        elif self.kind == "greedy":
            d.update(B=c["B"], K=c["K"], V=c["V"])
        elif self.kind == "tree":
            d.update(B=c["B"], N=c["N"], V=c["V"], T=self.T, max_depth=c["max_depth"],
                     max_children=c["max_children"])
        elif self.kind == "spot":
            d.update(B=c["B"], N=c["N"], L=c["L"], V=c["V"], T=self.T, max_depth=c["max_depth"],
                     max_children=c["max_children"])
        elif self.kind == "anyorder":
            d.update(B=c["B"], Kv=c["K"], W=c["W"], V=c["V"], T=0.0)
        elif self.kind == "packed_topk":
            d.update(B=c["B"], K=c["K"], W=c["W"], V=c["V"], T=self.T, top_k_p=c["kp"],
                     top_k_q=c["kq"])
        else:
            d.update(B=c["B"], K=c["K"], W=c["W"], V=c["V"], T=self.T)
        d["logits"] = c["dtype"]
        return d

    def inputs(self, device, nseq=None):
        c = self.cfg
        B = nseq or c["B"]
        if self.kind == "sample":
            si = datagen.sample_inputs(B, c["K"], c["V"], dtype=c["dtype"], seed=c["seed"],
                                       sigma=self.sigma, T=self.T, device=device)
            return {"target": si.target, "draft": si.draft, "draft_ids": si.draft_ids}
        if self.kind == "greedy":
            gi = datagen.greedy_inputs(B, c["K"], c["V"], dtype=c["dtype"], seed=c["seed"],
                                       device=device)
            return {"target": gi.target, "draft_ids": gi.draft_ids, "draft_len": gi.draft_len}
        if self.kind == "tree":
            ti = datagen.tree_inputs(B, c["N"], c["V"], dtype=c["dtype"], seed=c["seed"],
                                     L=c["L"], max_depth=c["max_depth"],
                                     max_children=c["max_children"], device=device)
            return {"node_logits": ti.node_logits, "parent": ti.parent, "node_pos": ti.node_pos,
                    "node_tok": ti.node_tok}
        if self.kind == "anyorder":
            ai = datagen.anyorder_inputs(B, c["K"], c["W"], c["V"], dtype=c["dtype"],
                                         seed=c["seed"], device=device)
            return {"logits": ai.logits, "u": ai.u, "win_pos": ai.win_pos, "order": ai.order,
                    "draft": ai.draft, "end_pos": ai.end_pos}
        if self.kind == "spot":
            si = datagen.spot_inputs(B, c["N"], c["L"], c["V"], dtype=c["dtype"], seed=c["seed"],
                                     max_depth=c["max_depth"], max_children=c["max_children"],
                                     device=device)
            return {"state_logits": si.state_logits, "parent": si.parent,
                    "node_pos": si.node_pos, "node_tok": si.node_tok, "root_mask": si.root_mask}
        if self.kind == "packed_topk":
            return self.topk_inputs(B, device)
        pi = datagen.packed_inputs(B, c["K"], c["W"], c["V"], dtype=c["dtype"], seed=c["seed"],
                                   T=self.T, device=device)
        d = {"logits": pi.logits, "prev_draft": pi.prev_draft, "prev_len": pi.prev_len}
        if self.T > 0:
            d.update(prev_q_at_draft=pi.prev_q_at_draft, prev_draft_logits=pi.prev_draft_logits,
                     prev_q_offset=pi.prev_q_offset)
        return d

    def topk_inputs(self, B, device):
        """This call's rows and the state a previous call leaves: that call
        (no previous draft) runs on the previous rows -- through the library
        on a GPU, through the oracle on the CPU -- and is taken to have
        stopped at a_prev."""
        c = self.cfg
        K, W, kp, kq = c["K"], c["W"], c["kp"], c["kq"]
        ti = datagen.packed_topk_inputs(B, K, W, c["V"], dtype=c["dtype"], seed=c["seed"],
                                        device=device)
        if torch.device(device).type == "cuda":
            import draft_block_verification_gb300 as dbv
            z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device=device)
            prev = dbv.sv_packed_topk_step(ti.prev_logits, K, W, kp, kq, z(B, K - 1), z(B),
                                           z(B, W, kq), z(B, W, kq, dt=torch.float32), z(B),
                                           T=self.T, seed=c["seed"], it=1)
            a_prev = torch.maximum(ti.a_prev, prev["commit_len"])
        else:
            import oracle
            lg = datagen.to_numpy_logits
            prev = oracle.packed_topk_step(
                lg(ti.prev_logits), K, W, kp, kq, np.zeros((B, K - 1), np.int32),
                np.zeros(B, np.int32), np.zeros((B, W, kq), np.int32),
                np.zeros((B, W, kq), np.float32), np.zeros(B, np.int32), self.T, seed=c["seed"],
                it=1)
            prev = {k: torch.from_numpy(np.asarray(v)) for k, v in prev.items()}
            prev["q_probs"] = prev["q_probs"].float()
            a_prev = torch.maximum(ti.a_prev, prev["commit_len"])
        st = datagen.packed_state_from(prev["next_draft"], prev["commit_len"], prev["q_ids"],
                                       prev["q_probs"], a_prev, K, W)
        st["logits"] = ti.logits
        return st

    def call(self, dbv, inp, h):
        c = self.cfg
        if self.kind == "packed_topk":
            return dbv.sv_packed_topk_step(inp["logits"], c["K"], c["W"], c["kp"], c["kq"],
                                           inp["prev_draft"], inp["prev_len"],
                                           inp["prev_q_ids"], inp["prev_q_probs"],
                                           inp["prev_q_offset"], T=self.T, seed=c["seed"], it=2,
                                           handle=h)
        if self.kind == "sample":
            return dbv.sv_verify_sample(inp["target"], inp["draft"], inp["draft_ids"], T_p=self.T,
                                        T_q=self.T, mode=self.mode, lam=self.lam, seed=c["seed"],
                                        want_tv=self.tv, handle=h)
        if self.kind == "greedy":
            acc, nxt = dbv.sv_verify_greedy(inp["target"], inp["draft_ids"], inp["draft_len"],
                                            handle=h)
            return {"accept_len": acc, "next_token": nxt}
        if self.kind == "tree":
            return dbv.sv_verify_tree(inp["node_logits"], inp["parent"], inp["node_pos"],
                                      inp["node_tok"], T=self.T, seed=c["seed"], handle=h)
        if self.kind == "anyorder":
            return dbv.sv_packed_anyorder_step(inp["logits"], c["K"], c["W"], inp["u"],
                                               inp["win_pos"], inp["order"], inp["draft"],
                                               inp["end_pos"], handle=h)
        if self.kind == "spot":
            return dbv.sv_verify_spot(inp["state_logits"], inp["parent"], inp["node_pos"],
                                      inp["node_tok"], inp["root_mask"], T=self.T,
                                      seed=c["seed"], handle=h)
        return dbv.sv_packed_step(inp["logits"], c["K"], c["W"], inp["prev_draft"],
                                  inp["prev_len"], prev_q_at_draft=inp.get("prev_q_at_draft"),
                                  prev_draft_logits=inp.get("prev_draft_logits"),
                                  prev_q_offset=inp.get("prev_q_offset"), T=self.T,
                                  seed=c["seed"], it=1, handle=h)

    def oracle_call(self, inp):
        """The same call through the oracle; inputs as returned by inputs() on
        the CPU.  Returns the wall time in seconds."""
        import oracle
        c = self.cfg
        n = lambda t: t.numpy()
        lg = datagen.to_numpy_logits
        t0 = time.perf_counter()
        if self.kind == "sample":
            oracle.verify_sample(lg(inp["target"]), lg(inp["draft"]), n(inp["draft_ids"]),
                                 T_p=self.T, T_q=self.T, mode=self.mode, lam=self.lam,
                                 seed=c["seed"], want_tv=self.tv)
        elif self.kind == "greedy":
            oracle.verify_greedy(lg(inp["target"]), n(inp["draft_ids"]), n(inp["draft_len"]))
        elif self.kind == "tree":
            oracle.verify_tree(lg(inp["node_logits"]), n(inp["parent"]), n(inp["node_pos"]),
                               n(inp["node_tok"]), T=self.T, seed=c["seed"])
        elif self.kind == "anyorder":
            oracle.packed_anyorder_step(lg(inp["logits"]), c["K"], c["W"], n(inp["u"]),
                                        n(inp["win_pos"]), n(inp["order"]), n(inp["draft"]),
                                        n(inp["end_pos"]))
        elif self.kind == "spot":
            oracle.verify_spot(lg(inp["state_logits"]), n(inp["parent"]), n(inp["node_pos"]),
                               n(inp["node_tok"]), n(inp["root_mask"]).astype(np.uint64),
                               T=self.T, seed=c["seed"])
        elif self.kind == "packed_topk":
            oracle.packed_topk_step(lg(inp["logits"]), c["K"], c["W"], c["kp"], c["kq"],
                                    n(inp["prev_draft"]), n(inp["prev_len"]),
                                    n(inp["prev_q_ids"]), n(inp["prev_q_probs"]),
                                    n(inp["prev_q_offset"]), self.T, seed=c["seed"], it=2)
        else:
            pdl = inp.get("prev_draft_logits")
            oracle.packed_step(lg(inp["logits"]), c["K"], c["W"], n(inp["prev_draft"]),
                               n(inp["prev_len"]),
                               prev_q_at_draft=None if pdl is None else n(inp["prev_q_at_draft"]),
                               prev_draft_logits=None if pdl is None else lg(pdl),
                               prev_q_offset=None if pdl is None else n(inp["prev_q_offset"]),
                               T=self.T, seed=c["seed"], it=1)
        return time.perf_counter() - t0

    def units(self, inp):
        """Verified draft rows of one call (the metric's unit)."""
        c = self.cfg
        if self.kind in ("sample", "greedy"):
            if "draft_len" in inp:
                return int(inp["draft_len"].sum().item())
            return int(inp["draft_ids"].shape[0]) * c["K"]
        if self.kind in ("tree", "spot"):
            return int(inp["parent"].numel())
        if self.kind == "anyorder":
            return int(sum(k for k, _ in self.anyorder_rows(inp)))
        return int(inp["prev_len"].sum().item())

    def alg_bytes(self, inp):
        """Bytes of logits the streaming kernel must read: every row the
        verify rule needs, once."""
        c = self.cfg
        row = c["V"] * self.esz
        if self.kind == "sample":
            B = inp["target"].shape[0]
            return B * (2 * c["K"] + 1) * row
        if self.kind == "greedy":
            return int((inp["draft_len"].long() + 1).sum().item()) * row
        if self.kind == "tree":
            return int(inp["parent"].numel()) * row
        if self.kind == "spot":
            return self.spot_rows(inp) * row
        if self.kind == "anyorder":
            return int(sum(min(k + 1, u) + u for k, u in self.anyorder_rows(inp))) * row
        B = inp["logits"].shape[0]
        return int((inp["prev_len"].long() + 1).sum().item() + B * c["W"]) * row

    def anyorder_rows(self, inp):
        """(kappa, u) of every sequence of an any-order call: kappa verified
        draft tokens; min(kappa + 1, u) verify rows and u proposal rows read."""
        u = inp["u"].cpu().numpy()
        od, dr = inp["order"].cpu().numpy(), inp["draft"].cpu().numpy()
        out = []
        for b in range(len(u)):
            k = 0
            while k < u[b] and dr[b, od[b, k]] >= 0:
                k += 1
            out.append((k, int(u[b])))
        return out

    def spot_rows(self, inp):
        """Rows a SPOT call streams: every masked position of every state."""
        m = inp["root_mask"].cpu().numpy().astype(np.uint64)
        par, pos = inp["parent"].cpu().numpy(), inp["node_pos"].cpu().numpy()
        total = 0
        for b in range(par.shape[0]):
            masks = [int(m[b])]
            for n in range(par.shape[1]):
                masks.append(masks[par[b, n] + 1] & ~(1 << int(pos[b, n])))
            total += sum(bin(x).count("1") for x in masks)
        return total

    def decisions(self, out):
        """Per-call decision summary of a call's outputs: near-threshold flags,
        mean accepted draft tokens per sequence (tree: mean accepted path
        depth), and for Packed-SS the mean stopping index a."""
        t = lambda k: out[k].detach().float().cpu() if isinstance(out, dict) and k in out else None
        d = {}
        if self.kind in ("tree", "spot"):
            d["mean_path_len"] = float(t("path_len").mean())
        else:
            d["mean_accept_len"] = float(t("accept_len").mean())
        if self.kind in ("packed", "packed_topk"):
            d["mean_commit_len"] = float(t("commit_len").mean())
        f = t("flags")
        d["flags"] = None if f is None else int(f.sum())
        return d

    def kernel(self):
        """The streaming kernel the roofline is taken on."""
        return "topk_select_kernel" if self.kind == "packed_topk" else "pass_kernel"

    def launches(self):
        """Library kernels per call: the streaming pass; the seed kernel
        before it when rows carry a Gumbel-max (trees, SPOT and Packed-SS
        steps at T > 0); the residual pass (the correction or the bonus
        token) and the fp64 check after a sampling call or a Packed-SS step
        at T > 0 (and the TV pass when TV is asked for); the per-sequence
        preparation of a SPOT or any-order call.  The truncated Packed-SS step
        is a selection and a decision kernel."""
        if self.kind == "packed_topk":
            return 2
        if self.kind == "sample":
            return 4 if self.tv else 3
        if self.kind == "anyorder":
            return 2
        if self.kind == "spot":
            return 3 if self.T > 0 else 2
        if self.kind == "tree":
            return 2 if self.T > 0 else 1
        return 4 if (self.kind == "packed" and self.T > 0) else 1


def _cpu_sample(w, seconds, nmax=None):
    """Inputs for the oracle on the CPU: as many sequences of the workload as
    fit in about `seconds` of oracle time, in whole rounds of one sequence per
    oracle thread (the oracle runs its sequences in parallel), measured on one
    sequence."""
    import oracle
    oracle.build()
    B = nmax or w.cfg["B"]
    one = w.inputs("cpu", 1)
    t1 = max(w.oracle_call(one), 1e-4)
    P = max(1, oracle.num_threads())
    nseq = int(max(1, min(B, P * max(1, int(seconds / t1)))))
    return nseq, (one if nseq == 1 else w.inputs("cpu", nseq))


def _threads_used(nseq):
    import oracle
    return int(min(nseq, max(1, oracle.num_threads())))


def cpu_baseline(w, seconds=15.0):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload
    (the first sequences of a batch drawn on the CPU with the same recipe),
    repeating the call until about `seconds` have passed."""
    nseq, inp = _cpu_sample(w, seconds / 3)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        times.append(w.oracle_call(inp))
        if time.perf_counter() >= t_end or len(times) >= 50:
            break
    dt = statistics.median(times)
    units = w.units(inp)
    return {"value": units / dt, "unit": "rows/s", "cores": _threads_used(nseq), "kind": "oracle",
            "cpu_model": _cpu_model(),
            "sample": "%d of %d sequences of %s, %d oracle calls, median %.3f s wall"
                      % (nseq, w.cfg["B"], w.name, len(times), dt)}


REF_BUDGET_S = 100.0  # oracle time of a whole reference run


def run_reference(args):
    """The reference arm is the CPU oracle (the pages ship no code): every step
    verifies a sample of the workload (whole rounds of one sequence per oracle
    thread).  The run stays within about two minutes: when the requested
    warm-up and steps would not fit, it times as many steps as fit (at least
    three, after one warm-up call) and reports that count as `steps`, next to
    `steps_requested`."""
    dist, rank, ws = _dist()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    w = Workload(args.workload, args)
    n_calls = max(1, args.warmup + args.steps)
    nseq, inp = _cpu_sample(w, REF_BUDGET_S / n_calls)
    t0 = time.perf_counter()
    vals = [w.units(inp) / w.oracle_call(inp)]  # first call: warm-up, and sizes the run
    t_call = time.perf_counter() - t0
    fit = max(4, int(REF_BUDGET_S / max(t_call, 1e-3)))
    n_run = min(n_calls, fit)
    warm = min(max(args.warmup, 1), max(1, n_run - 3)) if args.steps else n_run
    for _ in range(n_run - 1):
        vals.append(w.units(inp) / w.oracle_call(inp))
    timed = vals[warm:]
    value = statistics.median(timed) if timed else vals[-1]
    cb = {"value": value, "unit": "rows/s", "cores": _threads_used(nseq), "kind": "oracle",
          "cpu_model": _cpu_model(),
          "sample": "%d of %d sequences of %s per step" % (nseq, w.cfg["B"], w.name)}
    cfg = w.point()
    cfg.update(sample_sequences_per_step=nseq)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": ws, "steps": len(timed), "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": 1000.0 * w.units(inp) / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg, "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def _tensors(out):
    return [t for t in (out.values() if isinstance(out, dict) else out) if torch.is_tensor(t)]


def run_ours(args):
    import draft_block_verification_gb300 as dbv
    dist, rank, ws = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dbv.build()
    w = Workload(args.workload, args)
    inp = w.inputs(dev)
    h = dbv.default_handle(dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: w.call(dbv, inp, h)
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
    # Inputs smaller than a few L2s: flush L2 between steps (a write of twice
    # its size, outside the per-step events) and time each step on its own.
    flush = None
    if w.alg_bytes(inp) < 3 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    # one event pair per step (start, end) on the launching stream
    steps_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    with Clocks(local) as clk:
        _barrier(dist, dev)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(float(i))
            steps_ev[i][0].record(stream)
            out = call()
            steps_ev[i][1].record(stream)
        _barrier(dist, dev)
    h.sync_status()
    dec = w.decisions(out)
    # The streaming kernel's own duration: the same steps again, with the
    # library recording an event pair around that kernel on the call's stream
    # (kept out of the timed steps above, where events between the kernels
    # would serialise their launches).
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(float(i))
        h.set_option(dbv.SV_OPT_TIMING_EVENTS, int(ptrs[i].ctypes.data))
        call()
    h.set_option(dbv.SV_OPT_TIMING_EVENTS, 0)
    h.sync_status()
    step_ms = [a.elapsed_time(b) for a, b in steps_ev]
    ms = sum(step_ms) / args.steps
    ms = _max_over_ranks(dist, ms, dev)
    kern_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    units = w.units(inp)
    value = job_rate(ws, units, ms)
    alg_bytes = w.alg_bytes(inp)
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (kern_ms / 1000.0) / 1e9

    # end to end: pinned host inputs -> device, the call, results -> host
    host = {k: t.detach().cpu().pin_memory() for k, t in inp.items()}
    dst = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    out_bytes = 0
    _barrier(dist, dev)
    # one event pair per step; the median step (host-link traffic from other
    # work on the machine can slow single steps)
    e_steps = max(3, min(args.steps, 10))
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(e_steps)]
    for i in range(e_steps):
        e_ev[i][0].record(stream)
        for k, t in host.items():
            dst[k].copy_(t, non_blocking=True)
        res = [t.to("cpu", non_blocking=True) for t in _tensors(w.call(dbv, dst, h))]
        out_bytes = sum(r.numel() * r.element_size() for r in res)
        e_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    e_ms = _max_over_ranks(dist, statistics.median(a.elapsed_time(b) for a, b in e_ev), dev)
    h.sync_status()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    cfg = w.point()
    cfg["l2"] = ("inputs larger than L2 (%.2f MB of logits/step)" % (alg_bytes / 1e6)
                 if flush is None else "L2 flushed between steps (%.2f MB of logits/step)"
                 % (alg_bytes / 1e6))
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.cfg["dtype"], "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": _profiled_traffic(w),
                     "peak_source": peak_kind, "kernel": w.kernel(), "kernel_ms": kern_ms,
                     "alg_bytes_per_launch": alg_bytes},
        "e2e": {"value": job_rate(ws, units, e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out_bytes,
                "ms_per_step": e_ms, "steps": e_steps},
        "step_ms": _percentiles(step_ms),
        "decisions": dec,
        "gpu_launches": w.launches() * args.steps,
        "clocks": clk.summary(),
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
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
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(datagen.CONFIGS),
                    help="which verify workload one step runs (default: %s)" % WORKLOAD)
    ap.add_argument("--T", type=float, default=None, help="temperature (sample, tree, packed)")
    ap.add_argument("--sigma", type=float, default=None, help="drafter noise (sample)")
    ap.add_argument("--lam", type=float, default=None,
                    help="lambda (ratio), mu (linear) or the KL budget delta (cactus)")
    ap.add_argument("--mode", default=None, choices=["lossless", "ratio", "linear", "cactus"])
    ap.add_argument("--no-tv", action="store_true",
                    help="lenient sweep: leave out the per-row TV pass")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
