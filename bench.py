#!/usr/bin/env python
"""Benchmark one DSpark draft round (sample + schedule + verify) on GB300.

Workload (default, --workload 3): R=128 requests, gamma=16, V=151936, r=256,
d=4096, bf16 inputs, synthetic structured logits (top-1 boosted +6 on 70% of
positions), T in {0.6, 1.0}, staircase SPS, synchronous scheduler. A step is
one whole round over one batch; inputs stay resident in HBM, `round` advances
so every step draws fresh noise, and L2 is flushed (256 MiB write) between
steps outside the timed events.

Prints one JSON line. Metric: draft tokens per second (sum of gamma_r over the
batch / round time). Multi-GPU (torchrun): every rank runs an independent
replica on its own batch (weak scaling, no collective on the data path); the
value is all ranks' draft tokens over the slowest rank's time.

--impl reference times the CPU oracle (test infrastructure, the only
reference this method has) on a bounded sample of the same workload.
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
sys.path.insert(0, ROOT)

METRIC = "DSpark round: draft tokens/s (sample+schedule+verify) & % of HBM roofline"
UNIT = "draft tokens/s"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s replica: every rank runs the whole workload with its own noise."""
    return int(seed) + 1000 * int(rank)


def job_times(times_s, device):
    """Max over ranks of each per-rank duration (seconds); identity on one rank."""
    t = torch.tensor([float(x) for x in times_s], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized() \
            and torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", "dspark_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------ accounting

def round_bytes(rnd, keep_sum: int, n_rejected: int) -> dict:
    """Compulsory HBM bytes of one round, each tensor read once (algorithmic)."""
    es = 2 if rnd.dtype == "bf16" else 4
    g = rnd.gamma.cpu().numpy() if rnd.gamma is not None else np.full(rnd.R, rnd.gamma_max)
    drafted = int(g.sum())
    b = {
        "U": drafted * rnd.V * es,
        "W": rnd.r * rnd.V * es,
        "h": drafted * rnd.d * es,
        "E_rows": 2 * drafted * rnd.r * es,                       # bias rows + confidence rows
        "target_rows": (keep_sum + rnd.R) * rnd.V * es,
        "residual_recompute": n_rejected * rnd.V * es + (rnd.r * rnd.V * es if n_rejected else 0),
    }
    b["total"] = sum(b.values())
    return b


def draft_stats_launch_bytes(rnd, w_every_step: bool = False) -> float:
    """Algorithmic bytes of one draft_stats launch: that step's U slice, the
    conditioning E rows and the partial statistics written (one (max, sum) pair per
    request for each of the kernel's CTAs, one per SM: 152 on GB300), plus W counted
    once per round (its share per step), as the round's compulsory traffic counts it.
    With w_every_step, W is counted whole in every step instead: the L2 cannot keep a
    78 MB operand between steps on this GPU (measured retention 32-48 MB)."""
    es = 2 if rnd.dtype == "bf16" else 4
    g = rnd.gamma.cpu().numpy() if rnd.gamma is not None else np.full(rnd.R, rnd.gamma_max)
    drafted = int(g.sum())
    ctas = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    w = rnd.r * rnd.V * es
    per_round = drafted * rnd.V * es + drafted * rnd.r * es + rnd.R * rnd.gamma_max * ctas * 8
    return (per_round + (w * rnd.gamma_max if w_every_step else w)) / rnd.gamma_max


def host_to_device_copier():
    """cudaMemcpyAsync(dst, src, bytes, host-to-device, stream) through the CUDA runtime the
    process already loaded: one call per copy, without torch's per-call tensor overhead."""
    import ctypes
    rt = None
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        raise RuntimeError("the CUDA runtime library is not loadable")
    fn = rt.cudaMemcpyAsync
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int

    def copy(dst, src, nbytes, stream):
        rc = fn(dst, src, nbytes, 1, stream)
        if rc:
            raise RuntimeError("cudaMemcpyAsync failed (%d)" % rc)
    return copy


def host_to_device_copier_2d():
    """cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, host-to-device, stream)."""
    import ctypes
    rt = None
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        raise RuntimeError("the CUDA runtime library is not loadable")
    fn = rt.cudaMemcpy2DAsync
    fn.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t,
                   ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int

    def copy(dst, dpitch, src, spitch, width, height, stream):
        rc = fn(dst, dpitch, src, spitch, width, height, 1, stream)
        if rc:
            raise RuntimeError("cudaMemcpy2DAsync failed (%d)" % rc)
    return copy


def kernel_hash(files) -> str:
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[2] == src_hash:
                return float(parts[3])
    return None


# ------------------------------------------------------------------ CPU oracle

def run_oracle_round(rnd, ids, threads, rnd_index):
    import oracle

    def to_np(t):
        t = t.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    idx = torch.as_tensor(ids, dtype=torch.long, device=rnd.U.device)
    U = to_np(rnd.U.index_select(0, idx))
    h = to_np(rnd.h.index_select(0, idx))
    target = to_np(rnd.target.index_select(0, idx))
    E, W = to_np(rnd.E), to_np(rnd.W)
    T = to_np(rnd.temperature)[ids]
    anchor = to_np(rnd.anchor)[ids]
    gamma = None if rnd.gamma is None else to_np(rnd.gamma)[ids]
    sps = to_np(rnd.sps).astype(np.float64)
    t0 = time.perf_counter()
    s = oracle.sample_block(U, E, W, h, to_np(rnd.w_h), to_np(rnd.w_e), rnd.b, T, anchor, rnd.seed, rnd_index,
                            gamma=gamma, req_ids=np.asarray(ids), conf_token=rnd.conf_token,
                            bias_first=rnd.bias_first, threads=threads)
    mode = rnd.mode
    cap = s["surv"] if mode == 1 else None   # the sample has no older round; reuse current survivals
    c = oracle.schedule(s["surv"], sps, mode, gamma=gamma, surv_capacity=cap)
    oracle.verify(target, U, E, W, anchor, np.where(s["tokens"] < 0, 0, s["tokens"]), s["lse"], s["logit"],
                  c["keep"], T, rnd.seed, rnd_index, gamma=gamma, req_ids=np.asarray(ids),
                  bias_first=rnd.bias_first, threads=threads)
    dt = time.perf_counter() - t0
    drafted = int(gamma.sum()) if gamma is not None else len(ids) * rnd.gamma_max
    return drafted, dt


def cpu_threads():
    return max(1, min(16, os.cpu_count() or 1))


def library_draft_logp(ds, rnd, rnd_index):
    """Input preparation for the controlled-distance workload: its target rows are scored on the
    drafted prefix, so they are built from the realised draft distribution. The library drafts
    round `rnd_index` once (outside any timing); log p_d of every drafted position is then
    formed with plain torch ops from those tokens (softmax((U_k + W_1[x_{k-1}] W_2) / T))."""
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd_index, gamma=rnd.gamma)
    tokens = out["tokens"].clamp(min=0).long()
    W = rnd.W.float()

    def fn(ids):
        q = torch.as_tensor(ids, device=rnd.U.device)
        prev = torch.cat([rnd.anchor[q].long().unsqueeze(1), tokens[q, :-1]], dim=1)
        bias = rnd.E[prev].float() @ W
        if not rnd.bias_first:
            bias[:, 0] = 0.0
        logits = (rnd.U[q].float() + bias) / rnd.temperature[q].view(-1, 1, 1)
        return torch.log_softmax(logits, dim=2)
    return fn


def oracle_draft_logp(rnd, rnd_index, threads):
    """The same input preparation from the oracle's own draft (the reference arm runs no library
    code)."""
    import oracle

    def to_np(t):
        t = t.detach().contiguous().cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    def fn(ids):
        idx = torch.as_tensor(ids, dtype=torch.long, device=rnd.U.device)
        g = None if rnd.gamma is None else to_np(rnd.gamma)[ids]
        o = oracle.sample_block(to_np(rnd.U.index_select(0, idx)), to_np(rnd.E), to_np(rnd.W),
                                to_np(rnd.h.index_select(0, idx)), to_np(rnd.w_h), to_np(rnd.w_e), rnd.b,
                                to_np(rnd.temperature)[ids], to_np(rnd.anchor)[ids], rnd.seed, rnd_index, gamma=g,
                                req_ids=np.asarray(ids), logp=True, threads=threads)
        return torch.from_numpy(o["logp"])
    return fn


def make_workload(wl, n, dev, ds=None, threads=None):
    """Workload n on device dev; the controlled-distance one gets its target from the round-0
    draft (the library's, or the oracle's when ds is None)."""
    rnd = wl.WORKLOADS[n](device=dev)
    if "tv_delta" in rnd.extra:
        fn = library_draft_logp(ds, rnd, 0) if ds is not None else oracle_draft_logp(rnd, 0, threads or 1)
        wl.fill_controlled_tv_target(rnd, fn)
    return rnd


def sfu_floor(rnd, keep_sum, n_rej, sm_mhz, sms):
    """Special-function-unit operations of one round and the time they take at the documented
    rate of 16 per SM per clock (exp2 / log2 on the MUFU pipe), at the SM clock measured under
    load. Counted: one exp2 per draft vocabulary element (block statistics), one per target
    element read (verify rows), two per element of each rejected row (the residual), and the
    block- and element-level Gumbel logs (two each)."""
    g = rnd.gamma.cpu().numpy() if rnd.gamma is not None else np.full(rnd.R, rnd.gamma_max)
    drafted = int(g.sum())
    nblk = (rnd.V + 127) // 128
    ops = {"draft_exp2": drafted * rnd.V,
           "draft_gumbel_logs": 2 * drafted * (nblk + 128),
           "verify_exp2": (keep_sum + rnd.R) * rnd.V,
           "residual_exp2": 2 * n_rej * rnd.V}
    ops["total"] = sum(ops.values())
    rate = 16.0 * sms * sm_mhz * 1e6
    return {"ops_per_round": ops, "rate_ops_per_s": rate, "floor_us": ops["total"] / rate * 1e6,
            "basis": "16 MUFU results per SM per clock x %d SMs x %.0f MHz (median under load)" % (sms, sm_mhz)}


def time_rounds(ds, rnd, runner, flush, n, stream, first_round):
    """n whole rounds between CUDA events on the launch stream, L2 flushed before each outside the
    events; returns the per-round milliseconds."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    for s in range(n):
        flush.zero_()
        runner.set_round(first_round + s)
        starts[s].record(stream)
        runner.run()
        stops[s].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, stops)]


def percentiles(ms):
    a = np.asarray(ms)
    return {"median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "mean_ms": float(a.mean())}


def other_workloads(ds, wl, dev, flush, stream, n=10, sm_mhz=None):
    """The other full-size workloads, timed like the headline in the same run: resident inputs,
    n rounds between events on the launch stream, L2 flushed between rounds."""
    peaks = measured_peaks()
    rows = {}
    for w in (2, 4, 5):
        rnd = make_workload(wl, w, dev, ds=ds)
        cap = None
        if rnd.mode == wl.SCHED_ASYNC_CAPACITY:
            cap = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                                  rnd.seed, 0, gamma=rnd.gamma)["surv"].clone()
        runner = ds.RoundRunner(rnd, surv_capacity=cap)
        for i in range(3):
            runner.set_round(2 + i)
            runner.run()
        ms = time_rounds(ds, rnd, runner, flush, n, stream, 3000)
        status = runner.check()
        if status:
            raise RuntimeError("device status %d in workload %d" % (status, w))
        res = runner.results()
        keep_sum = int(res["keep"].sum())
        n_rej = int(res["resampled"].to(torch.int32).sum())
        rb = round_bytes(rnd, keep_sum, n_rej)
        mean_s = float(np.mean(ms)) / 1e3
        rows[rnd.name] = {"draft_tokens_per_s": rnd.draft_tokens() / mean_s, "rounds_per_s": 1.0 / mean_s,
                          **percentiles(ms), "admitted_per_round": keep_sum,
                          "committed_per_round": int(res["accepted"].sum()) + rnd.R,
                          "round_roofline_frac": rb["total"] / mean_s / 1e9 / peaks["hbm_gbs"],
                          "round_floor_us": rb["total"] / (peaks["hbm_gbs"] * 1e9) * 1e6,
                          "sched_mode": {0: "sync", 1: "async_capacity", 2: "full_scan"}[rnd.mode]}
        del runner, rnd, res
        torch.cuda.empty_cache()
    rows["note"] = ("same event protocol as the headline, %d rounds each; the controlled-distance workload's "
                    "target rows are built from the library's round-0 draft (its timed rounds draw other "
                    "tokens, so their distance is near, not at, the set value)" % n)
    return rows


# ------------------------------------------------------------------ arms

def bench_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    from speculative_decoding_draft_round_gb300 import workloads as wl
    dev = "cuda:%d" % local if torch.cuda.is_available() else "cpu"
    threads = cpu_threads()
    rnd = make_workload(wl, args.workload, dev, ds=None, threads=threads)
    n_req = threads
    ids = list(range(0, rnd.R, max(1, rnd.R // n_req)))[:n_req]
    for i in range(args.warmup):
        run_oracle_round(rnd, ids, threads, i)
    tok = 0
    tot = 0.0
    for i in range(args.steps):
        d, dt = run_oracle_round(rnd, ids, threads, args.warmup + i)
        tok += d
        tot += dt
    value = tok / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": rnd.name, "R": rnd.R, "gamma": rnd.gamma_max, "V": rnd.V,
                                           "r": rnd.r, "d": rnd.d, "sample_requests": len(ids)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d of %d requests per step, whole round (sample+schedule+verify)"
                                       % (len(ids), rnd.R)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_next_rows(ds, rnd, res, flush, n=20):
    """Times of the calls beyond the headline round, on this round's inputs and outputs: the
    flat verify batch and the static-threshold admission (median of isolated launches), and the
    sampler call in its variants -- the Markov head as in the headline, the RNN sequential head,
    greedy decoding at temperature 0 and per-position confidence temperatures -- each a whole
    dspark_sample_block call between CUDA events with L2 flushed before it, plus the median
    launch of the per-step kernels the variant changes."""
    from speculative_decoding_draft_round_gb300 import workloads as wl

    def per_launch(family, fn, reps=n):
        timer = ds.KernelTimer(family, reps * max(1, rnd.gamma_max))
        with timer:
            for _ in range(reps):
                fn()
        d = timer.durations_ms()
        return round(1e3 * float(np.median(d)), 2) if d else None

    def call_us(fn, reps=5):
        fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return round(1e3 * float(np.median([a.elapsed_time(b) for a, b in ev])), 1)

    tokens = torch.where(res["tokens"] < 0, torch.zeros_like(res["tokens"]), res["tokens"])
    a_out = ds.assemble(res["keep"], rnd.anchor, tokens)
    s_out = ds.schedule(res["surv"], rnd.sps, ds.SCHED_THRESHOLD, gamma=rnd.gamma, threshold=0.5)
    flat = per_launch("assemble", lambda: ds.assemble(res["keep"], rnd.anchor, tokens, out=a_out,
                                                     workspace=a_out["workspace"]))
    thr = per_launch("schedule", lambda: ds.schedule(res["surv"], rnd.sps, ds.SCHED_THRESHOLD, gamma=rnd.gamma,
                                                    threshold=0.5, out=s_out, workspace=s_out["workspace"]))
    rows = {"assemble_us": flat, "threshold_schedule_us": thr,
            "flat_tokens": int(res["keep"].sum().item()) + rnd.R}

    base = (rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b)
    variants = {
        "markov": dict(temperature=rnd.temperature),
        "rnn": dict(temperature=rnd.temperature, head=ds.HEAD_RNN, W_rnn=wl.rnn_weights(rnd)),
        "greedy": dict(temperature=torch.zeros_like(rnd.temperature)),
        "sts": dict(temperature=rnd.temperature,
                    sts_temp=torch.linspace(0.8, 1.6, rnd.gamma_max, device=rnd.U.device)),
    }
    for name, kw in variants.items():
        temp = kw.pop("temperature")
        out = ds.sample_block(*base, temp, rnd.anchor, rnd.seed, 7, gamma=rnd.gamma, **kw)
        ws = out.pop("workspace")
        fn = lambda: ds.sample_block(*base, temp, rnd.anchor, rnd.seed, 7, gamma=rnd.gamma, out=out, workspace=ws,
                                     **kw)
        row = {"sampler_us": call_us(fn), "draft_stats_us": per_launch("draft_stats", fn, reps=2),
               "draft_commit_us": per_launch("draft_commit", fn, reps=2)}
        if name == "rnn":
            row["rnn_step_us"] = per_launch("rnn_step", fn, reps=2)
            row["W_rnn"] = [3 * rnd.r, 2 * rnd.r + rnd.d]
        status = ds.check(ws)
        if status:
            raise RuntimeError("device status %d in the %s sampler" % (status, name))
        rows["sampler_" + name] = row
    torch.cuda.synchronize()
    rows["note"] = ("kernel times: medians of isolated launches under per-kernel events; sampler_us: median of "
                    "5 whole calls, L2 flushed before each")
    return rows


def bench_ours(args):
    import speculative_decoding_draft_round_gb300 as ds
    from speculative_decoding_draft_round_gb300 import build as dsbuild
    from speculative_decoding_draft_round_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    dsbuild.build()
    path = {"auto": ds.PATH_AUTO, "cuda_core": ds.PATH_CUDA_CORE, "tensor_core": ds.PATH_TENSOR_CORE,
            "resident": ds.PATH_RESIDENT}[args.path]
    rnd = wl.WORKLOADS[args.workload](device=dev)
    if world > 1:   # independent replica per rank
        rnd.seed = replica_seed(rnd.seed, rank)
    if "tv_delta" in rnd.extra:
        wl.fill_controlled_tv_target(rnd, library_draft_logp(ds, rnd, 0))
    cap = None
    if rnd.mode == wl.SCHED_ASYNC_CAPACITY:
        old = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, 0, gamma=rnd.gamma, path=path)
        cap = old["surv"].clone()
    runner = ds.RoundRunner(rnd, surv_capacity=cap, path=path)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    spath = ds.sample_path(runner.sa)
    uses_tc = spath in (ds.PATH_TENSOR_CORE, ds.PATH_RESIDENT)

    clocks = ClockSampler(gpu_id_for(local))
    clocks.start()
    # warm-up: at least W rounds and at least one second of work, so the clock sampler sees load
    t_start = time.time()
    i = 0
    while i < args.warmup or time.time() - t_start < 1.0:
        runner.set_round(2 + i)
        runner.run()
        torch.cuda.synchronize()
        i += 1
    status = runner.check()
    if status:
        raise RuntimeError("device status %d after warm-up" % status)

    n_timed = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    launches0 = ds.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # headline: K whole rounds, each bracketed by events on the launch stream, L2 flushed between
    # rounds outside the events; no per-kernel events here (they would break the overlap of
    # consecutive kernels that programmatic dependent launch provides)
    for s in range(n_timed):
        flush.zero_()
        runner.set_round(1000 + s)
        starts[s].record(stream)
        runner.run()
        stops[s].record(stream)
    torch.cuda.synchronize()
    launches = ds.launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, stops)]
    total_ms = sum(step_ms)
    # the same K rounds again with events around every launch of the dominant kernel, for its
    # average launch duration
    dom = "draft_loop" if spath == ds.PATH_RESIDENT else "draft_stats"
    timer = ds.KernelTimer(dom, n_timed * rnd.gamma_max)
    keep_tot = torch.zeros((), dtype=torch.int64, device=dev)
    commit_tot = torch.zeros((), dtype=torch.int64, device=dev)
    with timer:
        for s in range(n_timed):
            flush.zero_()
            runner.set_round(1000 + s)
            runner.run()
            # the same rounds as the timed ones: admitted and committed tokens (device sums, untimed)
            keep_tot += runner.cout["keep"].sum()
            commit_tot += runner.vout["accepted"].sum() + rnd.R
    stats_ms = timer.durations_ms()
    if spath == ds.PATH_RESIDENT:   # one launch per round covers every step: per-step average
        stats_ms = [m / rnd.gamma_max for m in stats_ms]
    admitted_total, committed_total = int(keep_tot.item()), int(commit_tot.item())
    status = runner.check()
    if status:
        raise RuntimeError("device status %d after timing" % status)
    res = runner.results()
    keep_sum = int(res["keep"].sum())
    n_rej = int(res["resampled"].to(torch.int32).sum())

    # end to end through the public API: per-round inputs copied from pinned host memory,
    # results read back, every step. U is copied one position at a time on a second stream and
    # the sampler's step k waits for its slice (step_ready events), so the draft steps run under
    # the copy. The target logits are copied after the scheduler, and only the rows verification
    # reads (rows 0..keep[r] of each request: what the target model would have scored): row 0 of
    # every request in one strided copy, then one copy per request that admitted tokens; the host
    # reads keep back to know them.
    host_in = {k: getattr(rnd, k).cpu().pin_memory() for k in ("h", "temperature", "anchor", "sps")}
    U_h = rnd.U.cpu().pin_memory()
    copy_stream = torch.cuda.Stream()
    slice_ready = [torch.cuda.Event() for _ in range(rnd.gamma_max)]
    es_u = rnd.U.element_size()
    memcpy_2d = host_to_device_copier_2d()
    if rnd.gamma is not None:
        host_in["gamma"] = rnd.gamma.cpu().pin_memory()
    dev_in = {k: getattr(rnd, k) for k in host_in}
    target_h = rnd.target.cpu().pin_memory()
    keep_h = torch.empty(rnd.R, dtype=torch.int32).pin_memory()
    outs = [res["tokens"], res["keep"], res["accepted"], res["next_token"], res["stats"]]
    host_out = [o.cpu().pin_memory() for o in outs]
    h2d_fixed = sum(t.numel() * t.element_size() for t in host_in.values()) + U_h.numel() * es_u
    d2h = sum(t.numel() * t.element_size() for t in host_out) + keep_h.numel() * 4
    row_bytes = rnd.V * rnd.target.element_size()
    req_bytes = (rnd.gamma_max + 1) * row_bytes
    memcpy_async = host_to_device_copier()
    n_e2e = max(3, min(args.steps, 10))
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e_stops = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    target_rows = 0
    torch.cuda.synchronize()
    for s in range(n_e2e):
        e_starts[s].record(stream)
        for k, t in host_in.items():
            dev_in[k].copy_(t, non_blocking=True)
        # U[:, k, :] for every request: R rows of V elements, G*V apart, on the copy stream
        copy_stream.wait_stream(stream)
        for k in range(rnd.gamma_max):
            memcpy_2d(rnd.U.data_ptr() + k * rnd.V * es_u, rnd.gamma_max * rnd.V * es_u,
                      U_h.data_ptr() + k * rnd.V * es_u, rnd.gamma_max * rnd.V * es_u, rnd.V * es_u, rnd.R,
                      copy_stream.cuda_stream)
            slice_ready[k].record(copy_stream)
        runner.set_round(5000 + s)
        runner.run_draft(step_ready=slice_ready)
        keep_h.copy_(res["keep"], non_blocking=True)
        stream.synchronize()
        # row 0 of every request (always verified) in one strided copy, then rows 1..keep[r] of the
        # requests that admitted tokens, one copy each
        memcpy_2d(rnd.target.data_ptr(), req_bytes, target_h.data_ptr(), req_bytes, row_bytes, rnd.R,
                  stream.cuda_stream)
        target_rows += rnd.R
        for q, kq in enumerate(keep_h.tolist()):
            n = min(max(kq, 0), rnd.gamma_max)
            if n:
                memcpy_async(rnd.target.data_ptr() + q * req_bytes + row_bytes,
                             target_h.data_ptr() + q * req_bytes + row_bytes, n * row_bytes, stream.cuda_stream)
                target_rows += n
        runner.run_verify()
        for o, h in zip(outs, host_out):
            h.copy_(o, non_blocking=True)
        e_stops[s].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(e_starts, e_stops))
    h2d = h2d_fixed + target_rows * row_bytes // n_e2e
    next_rows = time_next_rows(ds, rnd, res, flush)
    others = other_workloads(ds, wl, dev, flush, stream) if (world == 1 and not args.no_other_workloads) else None
    clock = clocks.stop()

    drafted = rnd.draft_tokens()
    total_s = total_ms / 1e3
    total_s, e2e_s = job_times([total_s, e2e_ms / 1e3], dev)
    value = job_rate(drafted * n_timed, world, total_s)
    e2e_value = job_rate(drafted * n_e2e, world, e2e_s)

    peaks = measured_peaks()
    launch_bytes = draft_stats_launch_bytes(rnd)
    reread_bytes = draft_stats_launch_bytes(rnd, w_every_step=True)
    stats_mean_s = (sum(stats_ms) / len(stats_ms)) / 1e3 if stats_ms else float("nan")
    achieved = launch_bytes / stats_mean_s / 1e9
    resident = spath == ds.PATH_RESIDENT
    src = ["speculative_decoding_draft_round_gb300/csrc/%s" % f for f in
           (("draft_loop.cu",) if resident else ("sample_tc.cu",) if uses_tc else ("sample.cu",)) + ("common.cuh",)]
    kname = "draft_loop" if resident else "draft_stats_tc" if uses_tc else "draft_stats_simt"
    traffic = profiled_traffic(kname, rnd.name, kernel_hash(src))
    rb = round_bytes(rnd, keep_sum, n_rej)
    round_s = total_s / n_timed
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_timed, "warmup": args.warmup,
        "ms_per_step": 1e3 * round_s, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if uses_tc else "f32", "data": "synthetic",
        "config": {"workload": rnd.name, "R": rnd.R, "gamma": rnd.gamma_max, "V": rnd.V, "r": rnd.r, "d": rnd.d,
                   "sched_mode": {0: "sync", 1: "async_capacity", 2: "full_scan"}[rnd.mode],
                   "path": "resident" if resident else "tensor_core" if uses_tc else "cuda_core",
                   "parallelism": "replica x%d" % world,
                   "l2": "flushed between steps (256 MiB write, outside the timed events)",
                   "inputs": "resident in HBM"},
        "rounds_per_s": world * n_timed / total_s,
        "admitted_per_round": keep_sum,
        "admitted_tokens_per_s": world * admitted_total / total_s,
        "committed_tokens_per_s": world * committed_total / total_s,
        "round_ms": percentiles(step_ms),
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "bytes_per_launch": launch_bytes, "launch_us": stats_mean_s * 1e6,
                     "launches_timed": len(stats_ms), "peak_source": peaks["source"],
                     "bytes_per_launch_w_reread": reread_bytes,
                     "frac_w_reread": reread_bytes / stats_mean_s / 1e9 / peaks["hbm_gbs"]},
        "round_roofline": {"bytes_per_round": rb["total"], "achieved_gbs": rb["total"] / round_s / 1e9,
                           "frac": rb["total"] / round_s / 1e9 / peaks["hbm_gbs"],
                           "floor_us": rb["total"] / (peaks["hbm_gbs"] * 1e9) * 1e6,
                           "bias_gemm_tflops": 2.0 * rnd.r * rnd.V * drafted / round_s / 1e12,
                           "breakdown": rb},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": n_e2e, "note": "per-round inputs copied in: h, T, anchor, SPS before the round, U one position at a "
                                        "time on a second stream with the sampler's step k waiting for its slice, the "
                                        "target rows verification reads (rows 0..keep[r], after keep is read back) "
                                        "copied in after the scheduler, results copied out; E, W, w_h, w_e stay "
                                        "resident"},
        "gpu_launches": launches,
        "next_rows": next_rows,
        "clocks": clock,
    }
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = (clock or {}).get("sm_mhz") or 2070.0
    line["sfu_floor"] = sfu_floor(rnd, keep_sum, n_rej, sm_mhz, sms)
    if others is not None:
        line["other_workloads"] = others
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle on this host's cores over a bounded sample of the same round: chunks of
        # `threads` requests (one per thread), each a whole round for those requests, until about
        # ten seconds of work have been timed
        threads = cpu_threads()
        d_tot, t_tot, n_req, n_chunks = 0, 0.0, 0, 0
        while t_tot < 10.0 and n_chunks < 64:
            lo = (n_chunks * threads) % rnd.R
            ids = [(lo + j) % rnd.R for j in range(min(threads, rnd.R))]
            d, dt = run_oracle_round(rnd, ids, threads, 7 + n_chunks)
            d_tot += d
            t_tot += dt
            n_req += len(ids)
            n_chunks += 1
        line["cpu_baseline"] = {"value": d_tot / t_tot, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": "%d request-rounds of the %d-request workload in %d chunks of %d, "
                                          "each a whole round (sample+schedule+verify), %.1f s"
                                          % (n_req, rnd.R, n_chunks, min(threads, rnd.R), t_tot)}
        # and on one core: two requests, one whole round each
        d1, t1 = run_oracle_round(rnd, [0, 1], 1, 3)
        line["cpu_baseline"]["single_thread"] = {"value": d1 / t1, "unit": UNIT, "cores": 1,
                                                 "sample": "2 request-rounds, %.1f s" % t1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_profile(args):
    """Plain rounds for an external profiler: warm-up W rounds, then K rounds, no clocks,
    no end-to-end leg and no CPU baseline."""
    import speculative_decoding_draft_round_gb300 as ds
    from speculative_decoding_draft_round_gb300 import build as dsbuild
    from speculative_decoding_draft_round_gb300 import workloads as wl
    dsbuild.build()
    path = {"auto": ds.PATH_AUTO, "cuda_core": ds.PATH_CUDA_CORE, "tensor_core": ds.PATH_TENSOR_CORE,
            "resident": ds.PATH_RESIDENT}[args.path]
    rnd = make_workload(wl, args.workload, "cuda", ds=ds)
    cap = None
    if rnd.mode == wl.SCHED_ASYNC_CAPACITY:
        cap = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, 0, gamma=rnd.gamma, path=path)["surv"].clone()
    if args.head == "rnn":
        W_rnn = wl.rnn_weights(rnd)
        status = 0
        for i in range(args.warmup + args.steps):
            out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                                  rnd.seed, 2 + i, gamma=rnd.gamma, path=path, head=ds.HEAD_RNN, W_rnn=W_rnn)
            status = status or ds.check(out["workspace"])
        print(json.dumps({"profile_rounds": args.warmup + args.steps, "workload": rnd.name, "head": "rnn",
                          "status": status, "launches": ds.launch_count()}))
        if status:
            raise SystemExit(1)
        return
    runner = ds.RoundRunner(rnd, surv_capacity=cap, path=path)
    for i in range(args.warmup + args.steps):
        runner.set_round(2 + i)
        runner.run()
    torch.cuda.synchronize()
    status = runner.check()
    print(json.dumps({"profile_rounds": args.warmup + args.steps, "workload": rnd.name, "status": status,
                      "launches": ds.launch_count()}))
    if status:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--path", choices=["auto", "cuda_core", "tensor_core", "resident"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true", help="skip timing workloads 2, 4 and 5")
    ap.add_argument("--profile", action="store_true", help="plain rounds for ncu (no timing, no baselines)")
    ap.add_argument("--head", choices=["markov", "rnn"], default="markov",
                    help="with --profile: rnn runs only the sampler, with the RNN sequential head")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        bench_profile(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
