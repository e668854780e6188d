#!/usr/bin/env python
"""Throughput of block-causal varlen chunked attention (forward + backward).

One step = the whole hot path over one batch of synthetic input: the forward
of every query chunk of every sequence, then the backward (statistics, main
kernel) and, for needed-only K/V windows, the owner summation of the dK/dV
partials. Inputs are resident in HBM when the timed region starts; L2 is
flushed (256 MiB write) between steps, outside the step's CUDA events.

Headline metric: useful TFLOP/s of forward + backward, where useful FLOPs are
14 * d * N (N = unmasked (query, key, head) triples; forward 4 d N, backward
10 d N including the recomputation of Q K^T). Masked pairs are never counted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 3] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs its own replica of the
workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "useful TFLOP/s (fwd, fwd+bwd) and % of GB300 dense BF16 peak, 1 GPU"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                out[k] = float(v) if v is not None else FALLBACK[k]
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def host_info():
    """CPU model and torch's BLAS, reported with the CPU baseline."""
    import platform
    import re

    import torch
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, flags=re.M)
        model = m.group(1).strip() if m else None
    except Exception:
        pass
    if not model:
        try:
            m = re.search(r"^model name\s*:\s*(.+)$", open("/proc/cpuinfo").read(), flags=re.M)
            model = m.group(1).strip() if m else None
        except OSError:
            pass
    m = re.search(r"BLAS_INFO=([^,\s]+)", torch.__config__.show())
    return {"cpu_model": model or platform.processor() or platform.machine(), "arch": platform.machine(),
            "blas": m.group(1) if m else "unknown"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.window = None

    def mark(self, t0, t1):
        """Wall-clock bounds of the timed region; only samples inside it count."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if self.window and ts is not None and not (self.window[0] <= ts <= self.window[1]):
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
                power.append(float(f[4]))
            except ValueError:
                continue
            for n, val in zip(names, f[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w": statistics.median(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# the sources each timed kernel is compiled from (its own file and the headers it includes)
KERNEL_SOURCES = {
    "bd_fwd_kernel": ("attn_fwd.cu", "ptx.cuh", "plan_layout.h", "host_util.h", "common.h"),
    "bd_bwd_kernel": ("attn_bwd.cu", "ptx.cuh", "plan_layout.h", "host_util.h", "common.h", "bwd_aux.h",
                      "bwd_kernel.cuh"),
    "bd_bwd256_kernel": ("attn_bwd256.cu", "ptx.cuh", "plan_layout.h", "host_util.h", "common.h", "bwd_kernel.cuh"),
}


def kernel_source_digest(kernel):
    """sha256 over the kernel's source files (in the listed order) with comments
    and blank lines removed, so that only code changes make recorded counters stale."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_causal_varlen_gb300", "csrc", f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


def kernel_traffic(kernel, workload):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from the ncu
    capture recorded in profiles/traffic.json, or None when there is none or the
    kernel's sources changed since the counters were taken."""
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(prof) or kernel not in KERNEL_SOURCES:
        return None
    try:
        rec = json.load(open(prof)).get(f"{kernel}:{workload}")
        if rec and rec.get("source_sha256") == kernel_source_digest(kernel):
            return rec.get("bytes")
    except Exception:
        pass
    return None


def tile_stats(plan, wl):
    """128 x 128 (query, key) tiles per head: those the kernels visit (tiles that
    are fully masked are never loaded) against the dense causal tiles of every chunk."""
    import math
    per_head = plan.fwd_tiles() * plan.slots() / wl.H  # a forward work unit serves slots() heads
    qt = math.ceil(wl.L / 128)
    dense = 0
    for c in range(wl.cp):         # causal: chunk c's query tiles against keys [0, (c+1) L)
        for t in range(qt):
            dense += math.ceil(min(wl.S, c * wl.L + (t + 1) * 128) / 128)
    dense *= wl.B
    return {"visited_per_head": per_head, "dense_causal_per_head": dense,
            "skipped_fraction": 1.0 - per_head / dense if dense else 0.0,
            # useful (query, key) pairs over the pairs of the visited tiles
            "visited_density": plan.useful_pairs() / (per_head * 128 * 128) if per_head else 0.0}


def useful_flops(plan, wl):
    n = plan.useful_pairs() * wl.H
    return n, 4.0 * wl.d * n, 10.0 * wl.d * n


# ------------------------------------------------------------------ oracle timing

DROPOUT_SEED = 0x5EED0F0D0F0A77E0  # fixed seed of the --dropout runs


def oracle_sample(wl, q, k, v, do, chunks, heads=None, budget_s=None, dropout=0.0, dtype=None):
    """Time the oracle (fwd + bwd) on the host cores over the given chunks, one
    K/V head's query heads at a time (heads: how many query heads; with budget_s,
    stop once that many seconds have been spent, after at least one group), in
    ``dtype`` (default fp32, the precision the oracle is specified in; the tests
    run it in fp64). Returns (seconds, useful (pair, head) items)."""
    import torch
    dtype = torch.float32 if dtype is None else dtype

    import oracle
    G = wl.H // wl.Hkv
    nh = wl.H if heads is None else heads
    pairs = 0
    t0 = time.perf_counter()
    done = False
    for b, c in chunks:
        hdr = oracle.segment_chunk(wl.cu[b], wl.S, wl.cp, c)
        h = hdr["hdr"]
        a, e = h["kv_start"], h["kv_end"]
        rows = slice(c * wl.L, (c + 1) * wl.L)
        n_chunk = sum(ql * (kl - ql) + ql * (ql + 1) // 2 for _, _, ql, _, kl, _ in hdr["segs"])
        for g in range((nh + G - 1) // G):
            hq = slice(g * G, min(nh, (g + 1) * G))
            kw, vw = k[b, a:e, g:g + 1], v[b, a:e, g:g + 1]
            if dropout > 0:
                # the head index only selects the keep mask; timing is what matters here
                oracle.chunk_fwd_dropout(q[b, rows, hq], kw, vw, wl.cu[b], wl.S, c * wl.L, dropout, DROPOUT_SEED,
                                         b=b, kv_base=a, dtype=dtype)
                oracle.chunk_bwd_dropout(q[b, rows, hq], kw, vw, do[b, rows, hq], wl.cu[b], wl.S, c * wl.L,
                                         dropout, DROPOUT_SEED, b=b, kv_base=a, dtype=dtype)
            else:
                oracle.chunk_fwd(q[b, rows, hq], kw, vw, wl.cu[b], wl.S, c * wl.L, kv_base=a, dtype=dtype)
                oracle.chunk_bwd(q[b, rows, hq], kw, vw, do[b, rows, hq], wl.cu[b], wl.S, c * wl.L, kv_base=a,
                                 dtype=dtype)
            pairs += n_chunk * (hq.stop - hq.start)
            if budget_s is not None and time.perf_counter() - t0 > budget_s:
                done = True
                break
        if done:
            break
    del torch
    return time.perf_counter() - t0, pairs


def oracle_cost(wl, b, c):
    """Dense size of the oracle's score block for chunk c of sequence b (its window length x L)."""
    import oracle
    h = oracle.segment_chunk(wl.cu[b], wl.S, wl.cp, c)["hdr"]
    return (h["kv_end"] - h["kv_start"]) * wl.L


def run_reference(args):
    """The oracle as the reference arm, on the host cores, same metric and workload."""
    import torch

    import workloads
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    torch.set_num_threads(len(os.sched_getaffinity(0)))
    wl = bench_workload(args)
    q, k, v, do = workloads.tensors(wl)
    chunks_all = [(b, c) for b in range(wl.B) for c in range(wl.cp) if wl.cu[b][-1] > c * wl.L]
    times, pairs = [], []
    for s in range(args.warmup + args.steps):
        t, p = oracle_sample(wl, q, k, v, do, [chunks_all[s % len(chunks_all)]], heads=1, budget_s=0.0,
                             dtype=torch.float32)
        if s >= args.warmup:
            times.append(t)
            pairs.append(p)
    flops = 14.0 * wl.d * sum(pairs)
    value = flops / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "S": wl.S, "cp": wl.cp, "H": wl.H, "Hkv": wl.Hkv,
                       "d": wl.d, "kv_mode": wl.kv_mode},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": torch.get_num_threads(), "kind": "oracle",
                             "dtype": "f32",
                             "sample": "each step: one query chunk x one query head (fwd+bwd, fp32), chunks in turn",
                             **host_info()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_workload(args):
    """The workload `--workload` names, with `--head-dim` replacing its head dim and,
    for the single-document workload 4, `--seq-len` / `--cp` shrinking it (a reduced
    case for profiler captures)."""
    import dataclasses

    import workloads
    wl = workloads.config(args.workload)
    if args.head_dim and args.head_dim != wl.d:
        wl = dataclasses.replace(wl, d=args.head_dim, name=wl.name.replace(f"_d{wl.d}", f"_d{args.head_dim}"))
    seq_len, cp_arg = getattr(args, "seq_len", 0), getattr(args, "cp", 0)
    if seq_len or cp_arg:
        if args.workload != 4:
            raise SystemExit("--seq-len / --cp reshape only the single-document workload 4")
        S = seq_len or wl.S
        cp = cp_arg or wl.cp
        if S % cp or (S // cp) % 128:
            raise SystemExit("--seq-len must be a multiple of 128 * cp")
        wl = dataclasses.replace(wl, S=S, cp=cp, cu=[[0, S]], name=f"single_doc_s{S}_h{wl.H}kv{wl.Hkv}_d{wl.d}_cp{cp}")
    return wl


def plan_timing(bd, plan, wl, mode, dev, reps=5):
    """Host build time of the plan (median of `reps` builds) and the time of its
    one copy to the device (median of `reps` uploads, CUDA events on the current
    stream): both stay outside the timed step, once per step in training and
    shared by every layer. None where a measurement could not be taken."""
    import torch
    out = {"bytes": int(plan.host.nbytes), "build_ms": None, "upload_ms": None}
    try:
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
            ts.append(1e3 * (time.perf_counter() - t0))
        out["build_ms"] = statistics.median(ts)
        if torch.cuda.is_available():
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                plan.upload(dev)
                e1.record()
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            out["upload_ms"] = statistics.median(ts)
    except Exception as e:  # a report field; it never stops the benchmark
        out["error"] = repr(e)[:200]
    return out


# ------------------------------------------------------------------ our path

def workloads_block(bd, dev, flush, steps=20, warmup=3):
    """Every other workload (and head dim 256 on the 16k layout) timed the same
    way as the headline: inputs resident, L2 flushed between steps outside the
    events, median of `steps` steps; forward alone and forward + backward."""
    import dataclasses

    import torch

    import workloads
    cases = [(1, 0), (2, 0), (4, 0), (5, 0), (3, 256)]
    out = {}
    stream = torch.cuda.current_stream(dev)
    for i, hd in cases:
        wl = workloads.config(i)
        if hd:
            wl = dataclasses.replace(wl, d=hd, name=wl.name.replace(f"_d{wl.d}", f"_d{hd}"))
        mode = bd.BD_KV_WINDOW if wl.kv_mode == "window" else bd.BD_KV_GATHER
        plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode).upload(dev)
        fused = mode == bd.BD_KV_WINDOW and plan.owner_units() > 0
        q, k, v, do = workloads.tensors(wl)
        qd = q.to(dev).view(wl.B, wl.cp, wl.L, wl.H, wl.d)
        dod = do.to(dev).view_as(qd)
        del q, do
        if mode == bd.BD_KV_WINDOW:
            W = plan.kv_rows()
            kd = torch.zeros(wl.B, wl.cp, W, wl.Hkv, wl.d, dtype=torch.bfloat16, device=dev)
            vd = torch.zeros_like(kd)
            for b in range(wl.B):
                for c in range(wl.cp):
                    hdr, _ = plan.chunk(b * wl.cp + c)
                    a, e = hdr["kv_start"], hdr["kv_end"]
                    kd[b, c, :e - a] = k[b, a:e].to(dev)
                    vd[b, c, :e - a] = v[b, a:e].to(dev)
        else:
            kd, vd = k.to(dev).unsqueeze(1), v.to(dev).unsqueeze(1)
        del k, v
        out_t = torch.empty_like(qd)
        lse = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device=dev)
        dq = torch.empty(qd.shape, dtype=torch.float32, device=dev)
        gshape = (wl.B, 1, wl.S, wl.Hkv, wl.d) if fused else kd.shape
        dk = torch.empty(gshape, dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        wsp = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device=dev)
        flags = bd.BD_BWD_OWNER_ROWS if fused else 0
        n_pairs, f_fwd, f_bwd = useful_flops(plan, wl)

        def one(with_bwd):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            flush.zero_()
            ev[0].record(stream)
            if with_bwd:  # the forward's idle warp zeroes the backward's dQ accumulator
                bd.bd_attn_fwd_ex(plan, qd, kd, vd, out_t, lse, dq_zero=dq, stream=stream)
            else:
                bd.bd_attn_fwd(plan, qd, kd, vd, out_t, lse, stream=stream)
            ev[1].record(stream)
            if with_bwd:
                bd.bd_attn_bwd_ex(plan, qd, kd, vd, out_t, dod, lse, dq, dk, dv, wsp,
                                  flags | bd.BD_BWD_DQ_ZEROED, stream=stream)
            ev[2].record(stream)
            return ev

        evs = [one(True) for _ in range(warmup + steps)][warmup:]
        torch.cuda.synchronize(dev)
        bd.bd_check_status(plan)
        t_f = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
        t_s = statistics.median(e[0].elapsed_time(e[2]) for e in evs)
        out[wl.name] = {"fwd_ms": t_f, "fwd_bwd_ms": t_s, "fwd_tflops": f_fwd / (t_f * 1e-3) / 1e12,
                        "fwd_bwd_tflops": (f_fwd + f_bwd) / (t_s * 1e-3) / 1e12, "useful_pairs": n_pairs,
                        "kv_mode": wl.kv_mode,
                        "path": ("owner-row backward" if fused else "backward") + "; dQ zeroed by the forward",
                        "tiles": tile_stats(plan, wl), "steps": steps}
        del qd, dod, kd, vd, out_t, lse, dq, dk, dv, wsp, plan
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    import block_causal_varlen_gb300 as bd
    import workloads
    from block_causal_varlen_gb300 import build as bdbuild

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bdbuild.build()
    bd.load()

    wl = bench_workload(args)
    mode = bd.BD_KV_WINDOW if wl.kv_mode == "window" else bd.BD_KV_GATHER
    q, k, v, do = workloads.tensors(wl)
    plan = bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode)
    if args.dropout > 0:
        plan.set_dropout(args.dropout, DROPOUT_SEED)
    plan.upload(dev)
    plan_cost = plan_timing(bd, plan, wl, mode, dev)
    n_pairs, f_fwd, f_bwd = useful_flops(plan, wl)
    f_step = f_fwd + f_bwd

    qd = q.to(dev).view(wl.B, wl.cp, wl.L, wl.H, wl.d)
    dod = do.to(dev).view_as(qd)
    if mode == bd.BD_KV_WINDOW:
        W = plan.kv_rows()
        kd = torch.zeros(wl.B, wl.cp, W, wl.Hkv, wl.d, dtype=torch.bfloat16, device=dev)
        vd = torch.zeros_like(kd)
        for b in range(wl.B):
            for c in range(wl.cp):
                hdr, _ = plan.chunk(b * wl.cp + c)
                a, e = hdr["kv_start"], hdr["kv_end"]
                kd[b, c, :e - a] = k[b, a:e].to(dev)
                vd[b, c, :e - a] = v[b, a:e].to(dev)
    else:
        kd, vd = k.to(dev).unsqueeze(1), v.to(dev).unsqueeze(1)
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.cp, wl.H, wl.L, dtype=torch.float32, device=dev)
    dq = torch.empty(qd.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(kd.shape, dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    dk_own = torch.zeros(wl.B, 1, wl.S, wl.Hkv, wl.d, dtype=torch.float32, device=dev)
    dv_own = torch.zeros_like(dk_own)
    wsp = torch.empty(bd.bd_attn_bwd_workspace(plan), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # needed-only windows over every chunk: dK / dV summed at their owners inside the
    # backward kernel (no owner-sum kernel). The forward's otherwise idle warp 3 zeroes
    # the fp32 dQ accumulator (bd_attn_fwd_ex); --dq-in-pre moves that back to the
    # statistics kernel
    fused = (not args.split) and mode == bd.BD_KV_WINDOW and plan.owner_units() > 0
    zero_in_fwd = not args.dq_in_pre
    launches_per_step = 3 if fused else 3 + (1 if mode == bd.BD_KV_WINDOW else 0)

    def step(ev):
        ev[0].record(stream)
        if zero_in_fwd:
            bd.bd_attn_fwd_ex(plan, qd, kd, vd, out, lse, dq_zero=dq, stream=stream)
        else:
            bd.bd_attn_fwd(plan, qd, kd, vd, out, lse, stream=stream)
        ev[1].record(stream)
        bd.bd_attn_bwd_pre(plan, out, dod, lse, dq, wsp, stream=stream, clear_dq=not zero_in_fwd)
        ev[2].record(stream)
        if fused:
            bd.bd_attn_bwd_main_ex(plan, qd, kd, vd, dod, dq, dk_own, dv_own, wsp, bd.BD_BWD_OWNER_ROWS,
                                   stream=stream)
        else:
            bd.bd_attn_bwd_main(plan, qd, kd, vd, dod, dq, dk, dv, wsp, stream=stream)
        ev[3].record(stream)
        if mode == bd.BD_KV_WINDOW and not fused:  # stores every owner row: nothing to clear between steps
            bd.bd_owner_sum(plan, dk, dv, dk_own, dv_own, stream=stream, accumulate=False)
        ev[4].record(stream)

    def prep():
        flush.zero_()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    warm = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    props = torch.cuda.get_device_properties(dev)
    clocks = Clocks(f"GPU-{props.uuid}" if getattr(props, "uuid", None) is not None else str(local))
    clocks.start()  # nvidia-smi needs a moment to start: launch it before the warm-up
    for _ in range(args.warmup):
        prep()
        step(warm)
    torch.cuda.synchronize(dev)
    bd.bd_check_status(plan)

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for s in range(args.steps):
        prep()
        step(evs[s])
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    time.sleep(0.1)
    clocks.mark(t_wall0, t_wall1)
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    bd.bd_check_status(plan)
    seg = [[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in evs]  # ms
    # medians over the timed steps (the mean is reported beside the step time)
    t_fwd = statistics.median(x[0] for x in seg)
    t_pre = statistics.median(x[1] for x in seg)
    t_main = statistics.median(x[2] for x in seg)
    t_own = statistics.median(x[3] for x in seg)
    t_step = statistics.median(sum(x) for x in seg)
    t_step_mean = sum(sum(x) for x in seg) / args.steps
    if ws > 1:
        tt = torch.tensor([t_step], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        t_step = float(tt.item())
    value = ws * f_step / (t_step * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region.
    # Two buffer sets: while step t computes, step t+1's inputs copy in and step
    # t-1's results copy out on their own streams (every step moves all its bytes).
    e2e = None
    if not args.no_e2e:
        n_e2e = max(4, args.steps // 4)
        host_in = [dict(q=qd.cpu().pin_memory(), k=kd.cpu().pin_memory(), v=vd.cpu().pin_memory(),
                        do=dod.cpu().pin_memory()) for _ in range(2)]
        gk_shape = dk_own.shape if mode == bd.BD_KV_WINDOW else dk.shape
        host_out = [dict(o=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                         l=torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
                         dq=torch.empty(dq.shape, dtype=dq.dtype).pin_memory(),
                         dk=torch.empty(gk_shape, dtype=torch.float32).pin_memory(),
                         dv=torch.empty(gk_shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
        sets = []
        for i in range(2):
            dset = dict(q=torch.empty_like(qd), k=torch.empty_like(kd), v=torch.empty_like(vd),
                        do=torch.empty_like(dod), o=torch.empty_like(out), l=torch.empty_like(lse),
                        dq=torch.empty_like(dq), dkw=torch.empty_like(dk), dvw=torch.empty_like(dv),
                        dk=torch.zeros_like(dk_own), dv=torch.zeros_like(dv_own),
                        ws=torch.empty_like(wsp))
            sets.append(dset)
        # the plan blob goes up once per step too (host build stays outside: it is the same blob every step),
        # with the step's inputs, into the buffer set's own device copy of the plan
        plan_pinned = torch.from_numpy(plan.host).pin_memory()
        plans = [bd.Plan(wl.cu, wl.S, wl.cp, wl.H, wl.Hkv, wl.d, kv_mode=mode).upload(dev) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in[0].values()) + plan_pinned.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        for i in range(2):
            comp_done[i].record(stream)
            out_done[i].record(stream)

        def e2e_step(t):
            i = t % 2
            D_, Hi, Ho = sets[i], host_in[i], host_out[i]
            P_ = plans[i]
            with torch.cuda.stream(s_in):
                s_in.wait_event(comp_done[i])            # step t-2 finished reading this set
                P_.dev.copy_(plan_pinned, non_blocking=True)
                for key in ("q", "k", "v", "do"):
                    D_[key].copy_(Hi[key], non_blocking=True)
                in_ready[i].record(s_in)
            stream.wait_event(in_ready[i])
            stream.wait_event(out_done[i])               # step t-2's results have left this set
            if zero_in_fwd:
                bd.bd_attn_fwd_ex(P_, D_["q"], D_["k"], D_["v"], D_["o"], D_["l"], dq_zero=D_["dq"], stream=stream)
            else:
                bd.bd_attn_fwd(P_, D_["q"], D_["k"], D_["v"], D_["o"], D_["l"], stream=stream)
            zflag = bd.BD_BWD_DQ_ZEROED if zero_in_fwd else 0
            if fused:
                bd.bd_attn_bwd_ex(P_, D_["q"], D_["k"], D_["v"], D_["o"], D_["do"], D_["l"], D_["dq"], D_["dk"],
                                  D_["dv"], D_["ws"], bd.BD_BWD_OWNER_ROWS | zflag, stream=stream)
            else:
                bd.bd_attn_bwd_ex(P_, D_["q"], D_["k"], D_["v"], D_["o"], D_["do"], D_["l"], D_["dq"], D_["dkw"],
                                  D_["dvw"], D_["ws"], zflag, stream=stream)
                if mode == bd.BD_KV_WINDOW:
                    bd.bd_owner_sum(P_, D_["dkw"], D_["dvw"], D_["dk"], D_["dv"], stream=stream,
                                    accumulate=False)
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                gk_, gv_ = (D_["dk"], D_["dv"]) if mode == bd.BD_KV_WINDOW else (D_["dkw"], D_["dvw"])
                for key, src_t in (("o", D_["o"]), ("l", D_["l"]), ("dq", D_["dq"]), ("dk", gk_), ("dv", gv_)):
                    Ho[key].copy_(src_t, non_blocking=True)
                out_done[i].record(s_out)

        for t in range(args.warmup):
            e2e_step(t)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for t in range(n_e2e):
            e2e_step(t)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        for P_ in plans:
            bd.bd_check_status(P_)
        te = e0.elapsed_time(e1) / n_e2e
        e2e = {"value": ws * f_step / (te * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": te, "steps": n_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipeline": "double-buffered: next step's H2D and previous step's D2H overlap this step's kernels"}

    others = None
    if not args.no_workloads and ws == 1:
        others = workloads_block(bd, dev, flush)
    pk, src = peaks()
    if others:
        for rec in others.values():
            rec["frac_of_peak"] = rec["fwd_bwd_tflops"] / pk["bf16_tflops"]
    bwd_name = "bd_bwd256_kernel" if wl.d == 256 else "bd_bwd_kernel"  # head dim 256 has its own kernel
    dominant = bwd_name if t_main >= t_fwd else "bd_fwd_kernel"
    dom_ms = t_main if dominant == bwd_name else t_fwd
    dom_flops = f_bwd if dominant == bwd_name else f_fwd
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    # the recorded counters are for the dropout-free instantiation
    traffic = kernel_traffic(dominant, wl.name) if args.dropout == 0 else None

    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu and ws == 1:
            import torch as _t
            _t.set_num_threads(len(os.sched_getaffinity(0)))
            b0 = 0
            chunks = [(b0, c) for c in range(wl.cp) if wl.cu[b0][-1] > c * wl.L]
            # cheapest chunks first, one K/V head's query heads at a time, until ~12 s of oracle work
            chunks.sort(key=lambda bc: oracle_cost(wl, *bc))
            secs, pairs = oracle_sample(wl, q, k, v, do, chunks, budget_s=10.0, dropout=args.dropout)
            secs64, pairs64 = oracle_sample(wl, q, k, v, do, chunks, budget_s=5.0, dropout=args.dropout,
                                            dtype=_t.float64)
            v32 = 14.0 * wl.d * pairs / secs / 1e12
            v64 = 14.0 * wl.d * pairs64 / secs64 / 1e12
            cpu = {"value": v32, "unit": "TFLOP/s", "cores": _t.get_num_threads(),
                   "kind": "oracle", "seconds": secs, "dtype": "f32", **host_info(),
                   "fp64": {"value": v64, "seconds": secs64, "pairs": pairs64, "fp32_over_fp64": v32 / v64},
                   "sample": f"oracle fwd+bwd in fp32 (the precision the oracle is specified in) on chunks of "
                             f"sequence 0, cheapest first, one K/V head's query heads at a time until ~10 s "
                             f"({pairs} useful (pair, head) items); the same in fp64 (the tests' precision) for "
                             f"~5 s; TFLOP/s counts the same useful FLOPs"}
        result = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step, "ms_per_step_mean": t_step_mean,
            "step_statistic": "median of the timed steps' CUDA-event intervals",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "S": wl.S, "cp": wl.cp, "L": wl.L, "H": wl.H,
                       "Hkv": wl.Hkv, "d": wl.d, "kv_mode": wl.kv_mode, "layout_seed": wl.seed,
                       "useful_pairs": n_pairs, "useful_flops_fwd": f_fwd, "useful_flops_bwd": f_bwd,
                       "dropout": args.dropout,
                       "path": ("owner-row backward" if fused else
                                "window partials + owner-sum kernel" if mode == bd.BD_KV_WINDOW else
                                "all-gathered K/V, dK/dV summed in the kernel")
                               + ("; dQ zeroed by the forward" if zero_in_fwd else "; dQ zeroed by the statistics kernel"),
                       "tiles": tile_stats(plan, wl),
                       "plan": plan_cost,
                       "l2": "flushed between steps by a 256 MiB write outside the step events"},
            "fwd_tflops": f_fwd / (t_fwd * 1e-3) / 1e12,
            "bwd_tflops": f_bwd / ((t_pre + t_main + t_own) * 1e-3) / 1e12,
            "fwd_bwd_tflops_12dn": ws * 12.0 * wl.d * n_pairs / (t_step * 1e-3) / 1e12,
            "frac_of_peak": value / ws / pk["bf16_tflops"],
            "frac_of_sustained_peak": value / ws / pk["bf16_tflops_sustained"],
            "peak_source": src,
            "kernels_ms": {"bd_fwd_kernel": t_fwd, "bd_bwd_pre_kernel": t_pre, bwd_name: t_main,
                           **({} if fused or mode != bd.BD_KV_WINDOW else {"bd_owner_sum_kernel": t_own})},
            "roofline": {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                         "peak_source": f"bf16_tflops ({src})"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "workloads": others,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=3, help="1..5 (default 3: lognormal 16k, GQA, window)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="attention dropout probability (default 0, as in every benchmarked configuration)")
    ap.add_argument("--head-dim", type=int, default=0, choices=[0, 64, 128, 256],
                    help="replace the workload's head dim (default: keep it)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="workload 4 only: the single document's length (a reduced case for profiler captures)")
    ap.add_argument("--cp", type=int, default=0, help="workload 4 only: the number of chunks")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload block (the other workloads and head dim 256, timed after the headline)")
    ap.add_argument("--dq-in-pre", action="store_true",
                    help="zero the fp32 dQ accumulator in the backward's statistics kernel instead of with the "
                         "forward's idle warp (bd_attn_fwd_ex, the default)")
    ap.add_argument("--split", action="store_true",
                    help="needed-only windows: time window partials + the owner-sum kernel instead of the "
                         "owner-row backward")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
