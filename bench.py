#!/usr/bin/env python
"""Benchmark of the DLRM sparse hot path on one or more GPUs (one JSON line).

A step is one pass of the whole path over one batch of the workload:
embedding-bag forward -> interaction forward -> interaction backward ->
embedding-bag backward with row-wise SGD (for a workload without interaction,
forward -> backward with a resident pooled gradient).  The default workload is
"multi-hot": 26 fp16 tables x 4M rows x d = 128, batch 65536, Poisson(20) bag
lengths, Zipf(1.2) indices, strict pairs -- the one configuration that runs
all of the path's steps at a size that is not launch-bound.

Timing: W warm-up steps, then K steps between two CUDA events on the launch
stream, with a barrier and a device synchronize on both sides; the max over
ranks is reported.  Inputs are larger than L2 (tables of tens of GB, indices
of hundreds of MB per step), so no L2 flush is inserted.  Every kernel of the
timed steps is also bracketed by CUDA events (recorded on the launch stream
through the library's profiling hook) to time the dominant kernel for the
roofline.  SM clocks and throttle reasons are sampled with nvidia-smi during
the timed region.

``--impl reference`` times the CPU oracle (plain fp64 loops, one core) on a
bounded sample of the same workload instead.

Multi-GPU: replicas only.  The path's one exchange step (the all-to-all of
pooled vectors between model-parallel table shards) is not part of this
build, so N ranks run N independent replicas (weak scaling), one per GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_dense_interaction_gb300 import workloads as W  # noqa: E402

METRIC = "emb-bag+interaction fwd/bwd/SGD samples/s; gathered GB/s as % of HBM peak"


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=250)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="multi-hot", choices=sorted(W.CONFIG_IDS))
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement (kernel experiments)")
    p.add_argument("--schedule", choices=["overlap", "serial"], default="overlap",
                   help="overlap: the backward's coalescing runs on a side stream next to the forward")
    p.add_argument("--optimizer", choices=["sgd", "adagrad"], default="sgd",
                   help="row-wise update of the touched rows (adagrad: one fp32 accumulator per row)")
    p.add_argument("--fwd", choices=["separate", "fused"], default="separate",
                   help="fused: one kernel for the lookup and the interaction forward")
    p.add_argument("--update", choices=["sorted", "atomic"], default="sorted",
                   help="atomic: the SGD update by atomic reductions without coalescing (fp32 tables)")
    p.add_argument("--targets", choices=["auto", "on", "off"], default="auto",
                   help="also measure the capacity and uniform multi-hot workloads stage by stage "
                        "(auto: with the default workload on one GPU)")
    p.add_argument("--no-graph", action="store_true",
                   help="skip the second measurement: the same steps replayed from one CUDA graph")
    p.add_argument("--target-steps", type=int, default=40)
    p.add_argument("--batch", type=int, default=None, help="override the batch size (profiling runs)")
    p.add_argument("--tables", type=int, default=None, help="override the table count (profiling runs)")
    p.add_argument("--rows", type=int, default=None, help="override the rows per table (profiling runs)")
    return p.parse_args()


def workload_config(args):
    over = {}
    if args.tables is not None:
        over["T"] = args.tables
    if args.rows is not None:
        over["rows"] = [args.rows] * (args.tables or W.make_config(args.workload)["T"])
    if args.batch is not None:
        over["B"] = args.batch
    return W.make_config(args.workload, **over)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ the oracle ---

def oracle_sample(cfg, offsets, indices, Bs, seed):
    """A bounded sample of the workload for the CPU oracle: the first Bs
    samples of the batch, each table restricted to the rows those samples
    look up (renumbered in increasing order, so every result is unchanged)."""
    T, B, d = cfg["T"], cfg["B"], cfg["d"]
    sub_off = [np.zeros(1, dtype=np.int64)]
    sub_idx, tables, rows = [], [], []
    run = 0
    for t in range(T):
        lo, hi = int(offsets[t * B]), int(offsets[t * B + Bs])
        idx = indices[lo:hi]
        uniq, inv = np.unique(idx, return_inverse=True)
        if uniq.size == 0:
            uniq = np.zeros(1, dtype=np.int64)
        tables.append(W.table_rows_host(cfg, t, uniq, seed))
        rows.append(int(uniq.size))
        sub_idx.append(inv.astype(np.int64))
        sub_off.append(offsets[t * B + 1:t * B + Bs + 1] - lo + run)
        run += hi - lo
    sub = W.make_config(cfg["name"], B=Bs, rows=rows)
    sub["T"] = T
    return dict(cfg=sub, tables=tables, offsets=np.concatenate(sub_off),
                indices=np.concatenate(sub_idx) if sub_idx else np.zeros(0, np.int64),
                e0=W.make_e0(cfg, seed)[:Bs], dy=W.make_dy(cfg, seed)[:Bs],
                dpooled=W.make_dpooled(cfg, seed)[:Bs])


def oracle_step(s, optimizer="sgd"):
    import oracle
    cfg = s["cfg"]
    B, dt = cfg["B"], cfg["dtype"]
    pooled, pmag = oracle.emb_bag_fwd(s["tables"], dt, s["offsets"], s["indices"], B)
    if cfg["interaction"]:
        oracle.interact_fwd(s["e0"], pooled, cfg["include_self"], emb_mag=pmag)
        _, _, dp, dpm = oracle.interact_bwd(s["e0"], pooled, s["dy"], cfg["include_self"], emb_mag=pmag)
    else:
        dp, dpm = s["dpooled"], None
    co = oracle.coalesce(cfg["rows"], s["offsets"], s["indices"], B)
    if optimizer == "adagrad":
        oracle.adagrad(s["tables"], dt, s["offsets"], B, s["indices"].size, dp, cfg["lr"], ADAGRAD_EPS,
                       np.zeros(co["U"]), co, dpooled_mag=dpm)
    else:
        oracle.sgd(s["tables"], dt, s["offsets"], B, s["indices"].size, dp, cfg["lr"], co, dpooled_mag=dpm)


def calibrate_oracle(cfg, offsets, indices, seed, seconds, optimizer="sgd"):
    """Picks a sample size whose oracle step takes about `seconds`."""
    probe = min(128, cfg["B"])
    s = oracle_sample(cfg, offsets, indices, probe, seed)
    oracle_step(s, optimizer)  # first call loads the library and warms the caches
    t0 = time.perf_counter()
    oracle_step(s, optimizer)
    per_sample = (time.perf_counter() - t0) / probe
    return int(max(probe, min(cfg["B"], seconds / max(per_sample, 1e-9))))


def cpu_model():
    """The host CPU's model name (lscpu), or the platform's description."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(cfg, offsets, indices, seed, seconds, optimizer="sgd"):
    """The oracle timed on the host: the serial build (the parity oracle) on
    one core, then its OpenMP build (the same loops, identical results) on all
    cores, each on a sample sized for about `seconds`."""
    import oracle
    oracle.build()
    oracle.use_openmp(False)
    Bs = calibrate_oracle(cfg, offsets, indices, seed, seconds, optimizer)
    s = oracle_sample(cfg, offsets, indices, Bs, seed)
    t0 = time.perf_counter()
    oracle_step(s, optimizer)
    el = time.perf_counter() - t0
    out = {"value": Bs / el, "unit": "samples/s", "cores": 1, "kind": "oracle",
           "sample": f"first {Bs} of {cfg['B']} samples of the same batch (all {cfg['T']} tables, "
                     f"{s['indices'].size} lookups), full step in fp64 on one host core, {el:.1f} s",
           "cpu_model": cpu_model(), "host_cores": os.cpu_count()}
    if oracle.use_openmp(True):
        try:
            Ba = calibrate_oracle(cfg, offsets, indices, seed, seconds, optimizer)
            sa = oracle_sample(cfg, offsets, indices, Ba, seed)
            t0 = time.perf_counter()
            oracle_step(sa, optimizer)
            ela = time.perf_counter() - t0
            out["all_cores"] = {"value": Ba / ela, "unit": "samples/s", "cores": os.cpu_count(),
                                "kind": "oracle, OpenMP build",
                                "sample": f"first {Ba} of {cfg['B']} samples ({sa['indices'].size} lookups), "
                                          f"{ela:.1f} s on all {os.cpu_count()} host cores"}
        finally:
            oracle.use_openmp(False)
    else:
        out["all_cores"] = None
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = workload_config(args)
    offsets, indices = W.make_indices(cfg, args.seed)
    budget = 90.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    Bs = calibrate_oracle(cfg, offsets, indices, args.seed, min(3.0, budget), args.optimizer)
    s = oracle_sample(cfg, offsets, indices, Bs, args.seed)
    for _ in range(args.warmup):
        oracle_step(s, args.optimizer)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(s, args.optimizer)
    el = time.perf_counter() - t0
    value = Bs * args.steps / el
    sample = (f"first {Bs} of {cfg['B']} samples of the batch per step (all {cfg['T']} tables, "
              f"{s['indices'].size} lookups), fp64 oracle on one host core")
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": "samples/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_of(cfg), schedule=args.schedule, forward=args.fwd, optimizer=args.optimizer),
        "cpu_baseline": {"value": value, "unit": "samples/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def config_of(cfg):
    return {"workload": cfg["name"], "tables": cfg["T"], "rows_per_table": cfg["rows"][0]
            if len(set(cfg["rows"])) == 1 else f"{min(cfg['rows'])}..{max(cfg['rows'])}",
            "d": cfg["d"], "table_dtype": cfg["dtype"], "global_batch": cfg["B"],
            "bag": "x".join(str(v) for v in cfg["bag"]), "index": "x".join(str(v) for v in cfg["index"]),
            "pairs": ("self-inclusive" if cfg["include_self"] else "strict") if cfg["interaction"] else "none",
            "update": cfg["update"], "lr": cfg["lr"], "parallelism": "replicas",
            "l2": "inputs larger than L2 (no flush)"}


def aggregate_over_ranks(ms, units, device=None):
    """(max elapsed ms, total units) over the ranks of the default process
    group; the local values when there is no group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(units)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                smax.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.file.name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ the GPU run ---

ADAGRAD_EPS = 1e-8


class Step:
    """Device buffers and the launches of one step of the path."""

    def __init__(self, cfg, seed, dev, schedule="overlap", fwd="separate", optimizer="sgd", update="sorted"):
        import torch

        import sparse_dense_interaction_gb300 as sdi
        self.sdi, self.torch, self.cfg, self.dev = sdi, torch, cfg, dev
        B, T, d = cfg["B"], cfg["T"], cfg["d"]
        self.offsets_h, self.indices_h = W.make_indices(cfg, seed)
        self.nnz = int(self.indices_h.size)
        self.tables = W.make_tables_device(cfg, seed, dev)
        self.offsets = torch.from_numpy(self.offsets_h).to(dev)
        self.indices = torch.from_numpy(self.indices_h).to(dev)
        self.inter = cfg["interaction"]
        self.P = sdi.dlrm_num_pairs(T, cfg["include_self"]) if self.inter else 0
        self.pooled = torch.empty((B, T, d), device=dev)
        self.dpooled = torch.empty((B, T, d), device=dev)
        if self.inter:
            self.e0 = torch.from_numpy(W.make_e0(cfg, seed)).to(dev)
            self.dy = torch.from_numpy(W.make_dy(cfg, seed)).to(dev)
            self.y = torch.empty((B, d + self.P), device=dev)
            self.de0 = torch.empty((B, d), device=dev)
        else:
            self.dpooled.copy_(torch.from_numpy(W.make_dpooled(cfg, seed)))
        self.update = update
        if update == "atomic":
            if cfg["dtype"] != "f32" or cfg["update"] != "sgd" or optimizer != "sgd":
                raise ValueError("the atomic update serves fp32 tables with plain SGD")
            schedule = "serial"  # nothing to coalesce ahead of the forward
        self.ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, self.nnz, d) if update == "sorted" else 0,
                              dtype=torch.uint8, device=dev)
        self.grad = torch.empty((self.nnz, d), device=dev) if cfg["update"] == "grad" else None
        self.flag = torch.zeros(1, dtype=torch.int32, device=dev)
        self.schedule, self.fwd, self.optimizer = schedule, fwd, optimizer
        self.state = ([torch.zeros(r, dtype=torch.float32, device=dev) for r in cfg["rows"]]
                      if optimizer == "adagrad" else None)
        self.side = torch.cuda.Stream(dev, priority=-1)  # its small sort kernels go first when SMs free up
        self.coalesced = torch.cuda.Event()

    def run(self, prof=None):
        """One step: lookup, interaction forward and backward, lookup backward with the
        update.  With the overlapped schedule the backward's coalescing (which needs
        only the indices) runs on a side stream next to the forward kernels, and the
        reduce waits for it.  With `prof`, every library kernel is bracketed by events."""
        sdi, c, torch = self.sdi, self.cfg, self.torch
        main = torch.cuda.current_stream(self.dev)

        def call(name, fn, stream):
            if prof is None:
                fn()
            else:
                prof.begin(name, stream)
                fn()
                prof.end()

        if self.schedule == "overlap":
            self.side.wait_stream(main)  # this step's inputs, the previous step's reduce
            with torch.cuda.stream(self.side):
                call("coalesce", lambda: sdi.dlrm_emb_bag_coalesce(
                    c["rows"], c["d"], self.offsets, self.indices, c["B"], self.ws, err_flag=self.flag,
                    stream=self.side), self.side)
                self.coalesced.record(self.side)
        if self.inter and self.fwd == "fused":
            call("emb_bag_interact_fwd", lambda: sdi.dlrm_emb_bag_interact_fwd(
                self.tables, self.offsets, self.indices, c["B"], self.e0, c["include_self"], self.y,
                pooled=self.pooled, err_flag=self.flag), main)
        else:
            call("emb_bag_fwd", lambda: sdi.dlrm_emb_bag_fwd(self.tables, self.offsets, self.indices, c["B"],
                                                             self.pooled, err_flag=self.flag), main)
            if self.inter:
                call("interact_fwd", lambda: sdi.dlrm_interact_fwd(self.e0, self.pooled, c["include_self"],
                                                                   self.y), main)
        if self.inter:
            call("interact_bwd", lambda: sdi.dlrm_interact_bwd(
                self.e0, self.pooled, c["include_self"], self.dy, self.de0, self.dpooled), main)
        if self.update == "atomic":
            call("emb_bag_bwd_atomic", lambda: sdi.dlrm_emb_bag_bwd_sgd_atomic(
                self.tables, self.offsets, self.indices, c["B"], self.dpooled, c["lr"], err_flag=self.flag), main)
        elif self.schedule == "overlap":
            main.wait_event(self.coalesced)
            if self.state is None:
                call("reduce_sgd", lambda: sdi.dlrm_emb_bag_reduce_sgd(
                    self.tables, self.nnz, c["B"], self.dpooled, c["lr"], self.ws, grad_rows=self.grad,
                    err_flag=self.flag), main)
            else:
                call("reduce_sgd", lambda: sdi.dlrm_emb_bag_reduce_adagrad(
                    self.tables, self.state, self.nnz, c["B"], self.dpooled, c["lr"], ADAGRAD_EPS, self.ws,
                    grad_rows=self.grad, err_flag=self.flag), main)
        elif self.state is None:
            call("emb_bag_bwd", lambda: sdi.dlrm_emb_bag_bwd_sgd(
                self.tables, self.offsets, self.indices, c["B"], self.dpooled, c["lr"], self.ws,
                grad_rows=self.grad, err_flag=self.flag), main)
        else:
            call("emb_bag_bwd", lambda: sdi.dlrm_emb_bag_bwd_adagrad(
                self.tables, self.state, self.offsets, self.indices, c["B"], self.dpooled, c["lr"], ADAGRAD_EPS,
                self.ws, grad_rows=self.grad, err_flag=self.flag), main)


class KernelProfiler:
    """Brackets every library kernel of the timed steps with CUDA events."""

    BWD_NAMES = None

    def __init__(self, torch, sdi, stream, n_steps, max_per_call=24):
        self.torch, self.sdi, self.stream = torch, sdi, stream
        self.pool = []
        self.calls = []  # (call name, start event, [events after each kernel])
        n = n_steps * 5
        for _ in range(n):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(max_per_call + 1)]
            for e in evs:
                e.record(stream)  # creates the CUDA handle
            self.pool.append(evs)
        torch.cuda.synchronize()
        self.next = 0
        self.cur = None

    def begin(self, name, stream=None):
        evs = self.pool[self.next]
        self.next += 1
        evs[0].record(stream if stream is not None else self.stream)
        self.sdi.dlrm_profile_events(evs[1:])
        self.cur = (name, evs, self.sdi.dlrm_kernel_launch_count())

    def end(self):
        name, evs, before = self.cur
        self.sdi.dlrm_profile_events([])
        n = self.sdi.dlrm_kernel_launch_count() - before
        self.calls.append((name, evs, n))

    def per_kernel_ms(self):
        """{(call, kernel index): [ms per launch]} over all recorded steps."""
        out = {}
        for name, evs, n in self.calls:
            for k in range(n):
                out.setdefault((name, k), []).append(evs[k].elapsed_time(evs[k + 1]))
        return out


class CallTimer:
    """Brackets every library call (not each of its kernels) with CUDA events:
    a call's time without the events the per-kernel profile inserts between
    its kernels."""

    def __init__(self, torch, stream, n_steps):
        self.torch, self.stream = torch, stream
        self.pool = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(n_steps * 5)]
        self.next, self.calls, self.cur = 0, [], None

    def begin(self, name, stream=None):
        a, b = self.pool[self.next]
        self.next += 1
        a.record(stream if stream is not None else self.stream)
        self.cur = (name, a, b, stream if stream is not None else self.stream)

    def end(self):
        name, a, b, stream = self.cur
        b.record(stream)
        self.calls.append((name, a, b))

    def per_call_ms(self):
        out = {}
        for name, a, b in self.calls:
            out.setdefault(name, []).append(a.elapsed_time(b))
        return {k: float(np.mean(v)) for k, v in out.items()}


BWD_KERNELS_PREFIX = ["bwd_prep", "bag_ids"]


NUMBER_KERNELS = ["seg_count", "seg_scan"]  # number the unique keys: for a view or gradient rows


def coalesce_kernel_names(plan, numbered=False):
    """Kernels of one coalescing; ``plan`` = (LSD passes, MSD bucket sort used), as the
    library reports it (with the bucket sort the first pass sorts by the top digit and the
    later passes return at once)."""
    passes, msd = plan
    names = list(BWD_KERNELS_PREFIX) + ["sort_hist", "sort_digit_scan", "sort_pass[0]"]
    names += ["bucket_sort"] if msd else []
    names += [f"sort_pass[{p}]" for p in range(1, passes)]
    return names + (NUMBER_KERNELS if numbered else [])


REDUCE_KERNELS = ["seg_reduce", "seg_block_sum", "seg_finalize"]


def reduce_kernel_names(grad_rows):
    # the reduce numbers the unique keys first when it is given gradient rows (no view is asked
    # for here, so the coalescing leaves them unnumbered)
    return (NUMBER_KERNELS if grad_rows else []) + REDUCE_KERNELS


def bwd_kernel_names(plan, grad_rows=False):
    return coalesce_kernel_names(plan) + reduce_kernel_names(grad_rows)


def kernel_name(call, k, plan, grad_rows=False):
    """Name of the k-th kernel that a library call launched."""
    if call == "emb_bag_bwd":
        return bwd_kernel_names(plan, grad_rows)[k]
    if call == "coalesce":
        return coalesce_kernel_names(plan)[k]
    if call == "reduce_sgd":
        return reduce_kernel_names(grad_rows)[k]
    if call == "emb_bag_interact_fwd" and k > 0:  # the two-kernel path of the fused call
        return "interact_fwd"
    return call


def algorithmic_bytes(cfg, st):
    """Compulsory HBM bytes of each single-kernel call per launch (each
    distinct table row counted once; streams read or written once)."""
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    es = W.ELEM_BYTES[cfg["dtype"]]
    nb = T * B
    uniq = 0
    for t in range(T):
        lo, hi = st.offsets_h[t * B], st.offsets_h[(t + 1) * B]
        uniq += np.unique(st.indices_h[lo:hi]).size
    out = {
        "emb_bag_fwd": st.nnz * 8 + (nb + 1) * 8 + uniq * d * es + nb * d * 4,
    }
    if st.inter:
        width = d + st.P
        # fused call: the lookup's reads, e0 in, y and the pooled block out
        out["emb_bag_interact_fwd"] = out["emb_bag_fwd"] + B * d * 4 + B * width * 4
        out["interact_fwd"] = B * (T + 1) * d * 4 + B * width * 4
        out["interact_bwd"] = B * (T + 1) * d * 4 + B * width * 4 + B * (T + 1) * d * 4
    # the reduce + update kernel: the sorted keys and the bags the sort carried
    # (no view is asked for), the pooled gradient, and one read-modify-write of
    # every unique row
    out["seg_reduce"] = st.nnz * 8 + nb * d * 4 + 2 * uniq * d * es
    # the whole backward (coalescing + reduce, or the atomic update): the
    # indices and offsets, the pooled gradient, one read-modify-write of every
    # unique row (the sort's own passes are not compulsory traffic)
    out["backward"] = st.nnz * 8 + (nb + 1) * 8 + nb * d * 4 + 2 * uniq * d * es
    out["emb_bag_bwd_atomic"] = out["backward"]
    if st.state is not None:  # AdaGrad: read-modify-write of each touched row's accumulator
        out["seg_reduce"] += 2 * uniq * 4
        out["backward"] += 2 * uniq * 4
    return out, uniq


def stage_times(kernel_ms, plan):
    """Per-stage milliseconds of one step from the per-kernel times."""
    coal = sum(kernel_ms.get(k, 0.0) for k in coalesce_kernel_names(plan, numbered=True))
    red = sum(kernel_ms.get(k, 0.0) for k in REDUCE_KERNELS)
    out = {"lookup": kernel_ms.get("emb_bag_fwd"), "coalesce": coal or None, "reduce": red or None}
    if "emb_bag_bwd_atomic" in kernel_ms:
        out["backward"] = kernel_ms["emb_bag_bwd_atomic"]
    elif coal and red:
        out["backward"] = coal + red
    return out


def measure_overlapped_step(name, args, dev):
    """The step of a workload with the coalescing on a second stream beside the
    lookup (the schedule a training loop would use): CUDA events around the
    steps only."""
    import torch

    import sparse_dense_interaction_gb300 as sdi
    cfg = W.make_config(name)
    st = Step(cfg, args.seed, dev, "overlap", "separate", "sgd", "sorted")
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    if sdi.dlrm_read_error(st.flag) != 0:
        raise RuntimeError(f"device error flag in the overlapped {name} step")
    K = args.target_steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        st.run()
    b.record(stream)
    torch.cuda.synchronize()
    ms_step = a.elapsed_time(b) / K
    out = {"config": config_of(cfg), "update": "sorted", "schedule": "overlap", "ms_per_step": ms_step,
           "samples_per_s": cfg["B"] / (ms_step / 1e3), "steps": K}
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_target(name, args, dev, update="sorted"):
    """One workload measured stage by stage (serial schedule): the lookup and
    the whole backward timed per call (CUDA events around each library call),
    the coalescing and the reduce from a second run with every kernel
    bracketed by events; each with its algorithmic bytes and its fraction of
    the measured HBM peak."""
    import torch

    import sparse_dense_interaction_gb300 as sdi
    cfg = W.make_config(name)
    st = Step(cfg, args.seed, dev, "serial", "separate", "sgd", update)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    if sdi.dlrm_read_error(st.flag) != 0:
        raise RuntimeError(f"device error flag in the {name} target")
    K = args.target_steps
    calls = CallTimer(torch, stream, K)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        st.run(calls)
    b.record(stream)
    torch.cuda.synchronize()
    ms_step = a.elapsed_time(b) / K
    call_ms = calls.per_call_ms()
    prof = KernelProfiler(torch, sdi, stream, K)
    for _ in range(K):
        st.run(prof)
    torch.cuda.synchronize()
    plan = sdi.dlrm_emb_bag_sort_plan(cfg["rows"], st.nnz)
    kernel_ms = {kernel_name(c, k, plan, st.grad is not None): float(np.mean(v))
                 for (c, k), v in prof.per_kernel_ms().items()}
    alg, uniq = algorithmic_bytes(cfg, st)
    peak, _ = measured_peaks()
    stages = {}
    times = stage_times(kernel_ms, plan)
    kernel_sum_bwd = times.get("backward")
    times["lookup"] = call_ms.get("emb_bag_fwd")  # one kernel: call and kernel times agree
    times["backward"] = call_ms.get("emb_bag_bwd_atomic" if update == "atomic" else "emb_bag_bwd")
    for stage, ms in times.items():
        if ms is None:
            continue
        nbytes = {"lookup": alg["emb_bag_fwd"], "reduce": alg["seg_reduce"], "backward": alg["backward"]}.get(stage)
        e = {"ms": ms}
        if nbytes is not None:
            gbs = nbytes / (ms / 1e3) / 1e9
            e.update(bytes=nbytes, gbs=gbs, frac=gbs / peak)
        stages[stage] = e
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):  # DRAM bytes of a full launch from ncu (scaled from small cases)
        with open(tpath) as f:
            tr = json.load(f).get(name, {})
        for stage, kern in (("reduce", "seg_reduce"), ("backward", "emb_bag_bwd_atomic")):
            if stage in stages and kern in tr and (stage == "reduce" or update == "atomic"):
                stages[stage]["traffic"] = tr[kern]
    if "backward" in stages and kernel_sum_bwd is not None:
        stages["backward"]["kernel_sum_ms"] = kernel_sum_bwd  # with events between its kernels
    out = {"config": config_of(cfg), "update": update, "ms_per_step": ms_step,
           "samples_per_s": cfg["B"] / (ms_step / 1e3), "steps": K, "unique_rows": uniq, "lookups": st.nnz,
           "stages": stages, "stage_timing": "lookup and backward: events around each library call; coalescing "
                                             "and reduce: sums of per-kernel events (a second run)"}
    del st, prof, calls
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_targets(args, dev):
    """The workloads the >= 70 % of HBM goal is set on: capacity (uniform
    indices over 131 GB of fp32 tables) with both update paths, and the
    multi-hot shapes with uniform indices."""
    out = {}
    for key, name, update in (("capacity", "capacity", "sorted"), ("capacity_atomic", "capacity", "atomic"),
                              ("multi_hot_uniform", "multi-hot-uniform", "sorted")):
        out[key] = measure_target(name, args, dev, update)
    out["capacity_overlapped"] = measure_overlapped_step("capacity", args, dev)
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_dense_interaction_gb300 as sdi
    from sparse_dense_interaction_gb300 import build as cuda_build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    sdi.load()

    cfg = workload_config(args)
    st = Step(cfg, args.seed + rank, dev, args.schedule, args.fwd, args.optimizer, args.update)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    status = sdi.dlrm_read_error(st.flag)
    if status != 0:
        raise RuntimeError(f"device error flag after warm-up: {sdi.status_string(status)}")

    # timed region: K steps between two events, kernels bracketed by events
    prof = KernelProfiler(torch, sdi, stream, args.steps)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = sdi.dlrm_kernel_launch_count()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        st.run(prof)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = sdi.dlrm_kernel_launch_count() - launches0
    ms, samples = aggregate_over_ranks(t0.elapsed_time(t1), cfg["B"] * args.steps, dev)
    ms_step = ms / args.steps
    value = samples / (ms / 1e3)

    # the same steps replayed from one captured CUDA graph (the library launches on the
    # capturing stream, never synchronises and never allocates)
    graph_line = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        before = sdi.dlrm_kernel_launch_count()
        with torch.cuda.graph(graph):
            st.run()
        per_step = sdi.dlrm_kernel_launch_count() - before
        for _ in range(3):
            graph.replay()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        gms, _ = aggregate_over_ranks(t0.elapsed_time(t1), cfg["B"] * args.steps, dev)
        graph_line = {"value": samples / (gms / 1e3), "unit": "samples/s", "ms_per_step": gms / args.steps,
                      "steps": args.steps, "gpu_launches": per_step * args.steps}
        del graph

    # per-kernel times (events on the launch stream) and the roofline
    per = prof.per_kernel_ms()
    plan = sdi.dlrm_emb_bag_sort_plan(cfg["rows"], st.nnz)
    names = {}
    for (call, k) in per:
        names[(call, k)] = kernel_name(call, k, plan, st.grad is not None)
    kernel_ms = {names[key]: float(np.mean(v)) for key, v in per.items()}
    alg, uniq = algorithmic_bytes(cfg, st)
    peak, peak_kind = measured_peaks()
    dominant = max(kernel_ms, key=kernel_ms.get)
    rl_kernel = dominant if dominant in alg else max((k for k in kernel_ms if k in alg), key=kernel_ms.get)
    achieved = alg[rl_kernel] / (kernel_ms[rl_kernel] / 1e3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            # the captures are of the SGD kernels; other optimizers have their own entry, or none
            key = cfg["name"] if st.optimizer == "sgd" else f'{cfg["name"]}+{st.optimizer}'
            traffic = json.load(f).get(key, {}).get(rl_kernel)
    roofline = {"kernel": rl_kernel, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "algorithmic_bytes": alg[rl_kernel], "peak_source": peak_kind,
                "kernel_ms": kernel_ms[rl_kernel]}
    es = W.ELEM_BYTES[cfg["dtype"]]
    fwd_key = "emb_bag_fwd" if "emb_bag_fwd" in kernel_ms else "emb_bag_interact_fwd"
    gathered = st.nnz * cfg["d"] * es / (kernel_ms[fwd_key] / 1e3) / 1e9

    # end to end through the public API with host buffers
    e2e = None if args.no_e2e else e2e_measure(args, st, torch, sdi, stream, dev)

    status = sdi.dlrm_read_error(st.flag)
    if status != 0:
        raise RuntimeError(f"device error flag after timing: {sdi.status_string(status)}")

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(cfg, st.offsets_h, st.indices_h, args.seed, args.cpu_seconds, args.optimizer)
    gathered_bytes, unique_rows, lookups = st.nnz * cfg["d"] * es, uniq, st.nnz
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    targets = None
    if world == 1 and (args.targets == "on" or (args.targets == "auto" and args.workload == "multi-hot"
                                                  and args.batch is None and args.tables is None
                                                  and args.rows is None)):
        targets = run_targets(args, dev)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 accumulate, " + cfg["dtype"] + " tables",
            "data": "synthetic (seeded; Zipf/uniform indices, counter-hash tables)",
            "config": dict(config_of(cfg), schedule=args.schedule, forward=args.fwd, optimizer=args.optimizer,
                           update=args.update),
            "gathered": {"gbs": gathered, "frac_of_hbm_peak": gathered / peak,
                         "bytes": gathered_bytes, "unique_rows": unique_rows, "lookups": lookups},
            "roofline": roofline,
            "kernels_ms": kernel_ms,
            "e2e": e2e,
            "graph": graph_line,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": base,
            "targets": targets,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def e2e_measure(args, st, torch, sdi, stream, dev):
    """Same metric through the public API, every step's inputs copied from
    pinned host memory and its results read back, pipelined as a training
    loop would be: two device buffer sets; the inputs of step i+1 are copied
    on one copy stream while step i computes, and the results of step i are
    read back on another while step i+1 computes (the two directions overlap).
    Events order every copy against the steps that use the buffer.  The timed
    region covers K steps from the first input copy to the last result read
    back."""
    c = st.cfg
    K = args.e2e_steps or max(3, args.steps // 2)
    names_in = ["offsets", "indices"] + (["e0", "dy"] if st.inter else ["dpooled"])
    names_out = ["y", "de0"] if st.inter else ["pooled"]
    host_in = {"offsets": torch.from_numpy(st.offsets_h).pin_memory(),
               "indices": torch.from_numpy(st.indices_h).pin_memory()}
    for n in names_in[2:]:
        host_in[n] = getattr(st, n).cpu().pin_memory()
    sets = [{n: getattr(st, n) for n in names_in + names_out},
            {n: torch.empty_like(getattr(st, n)) for n in names_in + names_out}]
    host_out = [{n: torch.empty(getattr(st, n).shape, dtype=getattr(st, n).dtype, pin_memory=True)
                 for n in names_out} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def load(i):  # inputs of step i into set i % 2, once step i - 2 no longer reads it
        k = i % 2
        with torch.cuda.stream(copy_in):
            if i >= 2:
                copy_in.wait_event(step_done[k])
            for n in names_in:
                sets[k][n].copy_(host_in[n], non_blocking=True)
            in_ready[k].record(copy_in)

    def step(i):  # step i on set i % 2, then its results read back
        k = i % 2
        stream.wait_event(in_ready[k])
        if i >= 2:
            stream.wait_event(out_done[k])  # step i - 2's results have left the buffers
        for n, t in sets[k].items():
            setattr(st, n, t)
        st.run()
        step_done[k].record(stream)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(step_done[k])
            for n in names_out:
                host_out[k][n].copy_(sets[k][n], non_blocking=True)
            out_done[k].record(copy_out)

    def loop(n):
        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            step(i)
        stream.wait_event(out_done[(n - 1) % 2])

    loop(2)  # warm-up of the pipeline and both buffer sets
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy_in.wait_event(a)
    copy_out.wait_event(a)
    loop(K)
    b.record(stream)
    torch.cuda.synchronize()
    for n, t in sets[0].items():  # the step's own buffers again
        setattr(st, n, t)
    ms = a.elapsed_time(b) / K
    return {"value": c["B"] / (ms / 1e3), "unit": "samples/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "pipelined": "inputs of step i+1 copied while step i computes; results of step i read back "
                         "while step i+1 computes (two buffer sets, one copy stream per direction)"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
