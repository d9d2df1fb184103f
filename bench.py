#!/usr/bin/env python
"""Benchmark of the top-k sparse flash-attention backward (sfa_grad) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sfa|reference]
                    [--workload mla] [--deterministic]

One step is one sfa_grad call (phase 2: workspace zeroing, token metadata,
Dsum, score/softmax-gradient, key-side and query-side contractions, output
cast) over the whole workload, inputs already resident in HBM.  The metric is
TFLOP/s with 2 * (3 * (D + Dr) + 2 * D) = 5504 flops per valid
(query, head, key).  Each timed step is bracketed by CUDA events on the
launching stream; L2 is flushed (a 256 MB write) between steps, outside the
events.  Prints one JSON line (rank 0).

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling, no collective); the time is the max
over ranks and the value counts the work of all ranks.

--impl reference times the fp64 CPU oracle instead, on a bounded token
sample of the same workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "sparse-attn bwd TFLOP/s (1×GB300) and % of dense bf16 tensor peak"
FLOPS_PER_QHK = 2 * (3 * (512 + 64) + 2 * 512)
# Peaks used when MEASURED_PEAKS.json is absent (one earlier GB300 measurement).
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = dict(FALLBACK_PEAKS)
        for k in FALLBACK_PEAKS:
            for cand in (k, k.replace("_gbs", "_GBs")):
                if cand in d and isinstance(d[cand], (int, float)):
                    out[k] = float(d[cand])
        return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def valid_pairs(w, inp) -> int:
    """Valid (query, key) slot count; every workload here draws in-range keys,
    and mode-3 workloads draw them below each query's limit."""
    idx = inp["indices"].reshape(-1, w.K)
    return int((idx >= 0).sum().item()) * w.block_size


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled during the timed region."""

    def __init__(self, dev_index: int):
        self.proc = None
        self.lines = []
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={dev_index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks of the default process group (x itself
    when running alone).  Every rank must call it."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs flops_per_rank of work (independent
    replicas, weak scaling) and the job takes the slowest rank's ms."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def cpu_oracle_sample(w, inp, n_tokens: int):
    """Runs the fp64 oracle backward on a few query tokens of the workload with
    their full K/V segment; returns (seconds, flops, sample description).
    BSND: the first n tokens of batch 0.  TND: the last n tokens of the first
    non-empty batch, which keeps each token's causal limit kvlen - qlen + i."""
    import oracle
    sub = {}
    if w.layout == "TND":
        aq = inp["act_seq_q"].tolist()
        akv = inp["act_seq_kv"].tolist()
        b = next(i for i, x in enumerate(aq) if x > 0)
        q0, kv0, qlen, kvlen = sum(aq[:b]), sum(akv[:b]), aq[b], akv[b]
        n = min(n_tokens, qlen)
        sl = slice(q0 + qlen - n, q0 + qlen)
        kvs = slice(kv0, kv0 + kvlen)
        for name in ("q", "q_rope", "d_out", "indices"):
            sub[name] = inp[name][sl]
        kw = dict(k=inp["k"][kvs], v=inp["v"][kvs], k_rope=inp["k_rope"][kvs], scale=w.scale_value,
                  sparse_block_size=w.block_size, layout="TND", sparse_mode=w.mode,
                  act_seq_q=torch.tensor([n], dtype=torch.int32), act_seq_kv=torch.tensor([kvlen], dtype=torch.int32))
        what = f"last {n} query tokens of batch {b} of {w.name} (its full K/V segment), fp64 numpy"
    else:
        n = min(n_tokens, w.S1)
        sl = slice(0, n)
        for name in ("q", "q_rope", "d_out", "indices"):
            sub[name] = inp[name][:1, sl]
        kw = dict(k=inp["k"][:1], v=inp["v"][:1], k_rope=inp["k_rope"][:1], scale=w.scale_value,
                  sparse_block_size=w.block_size, layout="BSND", sparse_mode=w.mode)
        what = f"first {n} query tokens of {w.name} (full K/V), fp64 numpy"
    out, smax, ssum = oracle.sfa_fwd(q=sub["q"], indices=sub["indices"], q_rope=sub["q_rope"], **kw)
    t0 = time.perf_counter()
    oracle.sfa_bwd(q=sub["q"], indices=sub["indices"], q_rope=sub["q_rope"], d_out=sub["d_out"], out=out,
                   softmax_max=smax, softmax_sum=ssum, **kw)
    dt = time.perf_counter() - t0
    pairs = int((sub["indices"] >= 0).sum().item()) * w.block_size
    return dt, pairs * w.N1 * FLOPS_PER_QHK, what


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    per_step = 2
    times, flops = [], 0
    for i in range(args.warmup + args.steps):
        dt, fl, sample = cpu_oracle_sample(w, inp, per_step)
        if i >= args.warmup:
            times.append(dt)
            flops = fl
    ms = 1e3 * statistics.mean(times)
    value = flops / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w, False), "sample_tokens_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_desc(w, det, shared_kv=False):
    return (f"{w.name}: {w.layout} B={w.B} S1={w.S1} S2={w.S2} N1={w.N1} N2=1 D=512 Dr=64 K={w.K} "
            f"sparseBlockSize={w.block_size} sparseMode={w.mode} {w.dtype} deterministic={int(det)}"
            + (" value=key" if shared_kv else ""))


# DRAM bytes (read + write) per query token of one launch, from ncu captures
# of 512-token profiling workloads, scaled by tokens for other token counts of
# the same shape (heads, indices per token, block size, mode): the per-token
# traffic of another shape differs.  Reported only while the kernel source
# still hashes to the value it had when the counters were taken.
TRAFFIC = {
    "kvq": {"sources": ["kvq.cu", "common.cuh"],
            "sha256": "f54b31958027f5a265f0752651eca38ce939c0eec7c8ad81aa04bf232718526b",
            "shapes": [
                # mla_q512: 915.9 MB read + 83.0 MB written per launch
                {"N1": 128, "K": 2048, "bs": 1, "det": False, "bytes_per_token": 998.9e6 / 512},
                # mla_q512 --deterministic: 935.0 MB read + 2313.0 MB written (bf16 partial rows)
                {"N1": 128, "K": 2048, "bs": 1, "det": True, "bytes_per_token": 3248.0e6 / 512},
            ]},
}


def _source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sfa_grad_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def kernel_traffic(name, tokens, shape):
    """Recorded DRAM bytes of `name` for `tokens` query tokens of `shape`
    (dict with N1, K, bs, det), or None when no capture of that shape on the
    current source exists."""
    ent = TRAFFIC.get(name)
    if not ent or ent["sha256"] is None:
        return None
    if _source_hash(ent["sources"]) != ent["sha256"]:
        return None
    for sh in ent["shapes"]:
        if all(sh[k] == shape.get(k) for k in ("N1", "K", "bs", "det")):
            return sh["bytes_per_token"] * tokens
    return None


# Contraction work per valid (query, head, key) of each tensor-core kernel,
# in flops: sdp and sdpb recompute S (576-deep) and dP (512-deep); kvq forms
# dV (512 features), [dK | dKRope] (576) and [dQ | dQRope] (576); kvb forms dV
# and [dK | dKRope] per block; dqb forms [dQ | dQRope].
TENSOR_FLOPS = {"sdp": 2 * (576 + 512), "sdpb": 2 * (576 + 512), "kvq": 2 * (512 + 576 + 576),
                "kvb": 2 * (512 + 576), "dqb": 2 * 576}
# Bytes a streaming kernel must move per valid (query, key) pair: det_reduce
# reads each pair's 1088-element bf16 partial row once.
STREAM_BYTES = {"det_reduce": 1088 * 2}
# L2-resident fp32 vector reductions (red.global.add.v4.f32, four key rows x
# 128 B per warp instruction) measured on this GPU by bench_l2_red.cu
# (`bench.py --l2-red-ceiling`): the ceiling of the key-side scatter, which
# never reaches DRAM.
L2_RED_CEILING_GBS = 7040.0


def roofline(dname, names, qhk, pairs, k_ms, peaks, det):
    """Roofline of the dominant kernel over all its launches of one step
    (work of the launches over their summed time = per-launch work over the
    mean launch time).  Tensor-core kernels: algorithmic flops against the
    measured dense bf16 peak (burst: the step is milliseconds long and timed
    alone).  Streaming kernels: algorithmic bytes against the HBM copy peak."""
    t = k_ms * 1e-3
    if dname in TENSOR_FLOPS:
        per = TENSOR_FLOPS[dname]
        achieved = qhk * per / t / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "flops_per_query_head_key": per}
        if dname == "kvq" and not det:
            # the key side's scatter: 1088 fp32 reductions (4352 B) per pair
            gbs = pairs * 4352 / t / 1e9
            roof["l2_red"] = {"achieved_gbs": gbs, "ceiling_gbs": L2_RED_CEILING_GBS,
                              "frac": gbs / L2_RED_CEILING_GBS,
                              "ceiling_source": "bench_l2_red.cu: red.global.add.v4.f32, 4 rows x 128 B per warp instruction, 152 SMs"}
        return roof
    per_b = STREAM_BYTES.get(dname)
    if per_b is None:
        return {"bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": None,
                "note": f"no algorithmic byte count for {dname}"}
    achieved = pairs * per_b / t / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "bytes_per_pair": per_b}


def kernel_names(p, det):
    import sfa_grad_gb300 as sfa
    return sfa.plan_names(p)


def run_sfa(args):
    import sfa_grad_gb300 as sfa
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    det = args.deterministic
    inp = make_inputs(w)
    if args.shared_kv:
        inp["v"] = inp["k"]
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items() if not (args.shared_kv and k == "v")}
    if args.shared_kv:
        d["v"] = d["k"]
    kw = dict(q_rope=d["q_rope"], k_rope=d["k_rope"], sparse_block_size=w.block_size, layout=w.layout,
              sparse_mode=w.mode, act_seq_q=d.get("act_seq_q"), act_seq_kv=d.get("act_seq_kv"))
    out, smax, ssum = sfa.fwd(d["q"], d["k"], d["v"], d["indices"], w.scale_value, **kw)
    p = sfa.make_params(d["q"], d["k"], d["indices"], w.scale_value, layout=w.layout,
                        sparse_block_size=w.block_size, sparse_mode=w.mode, deterministic=det,
                        batch=w.B if w.layout == "TND" else None)
    _, launches = sfa.plan_info(p)
    names = kernel_names(p, det)
    ws = torch.empty(sfa.grad_workspace_size(p), dtype=torch.uint8, device=dev)
    outs = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
            torch.empty_like(d["q_rope"]), torch.empty_like(d["k_rope"]))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    pairs = valid_pairs(w, inp)
    flops = pairs * w.N1 * FLOPS_PER_QHK

    def step(events=None):
        sfa.grad(d["q"], d["k"], d["v"], d["indices"], d["d_out"], out, smax, ssum, w.scale_value,
                 deterministic=det, outputs=outs, workspace=ws, events=events, **kw)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    nev = launches + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    for row in ev:
        for e in row:
            e.record(stream)   # materialise the event handles
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        step(ev[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps)]
    per_launch = [statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                  for j in range(launches)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms = total_ms / args.steps
    value = job_tflops(world, flops, ms)
    err = sfa.read_device_error(ws)
    if err != 0:
        raise RuntimeError(f"device error word {err}")

    # ---- end to end through the C ABI from pinned host buffers: sfa_grad_host
    # copies every input to the device and every result back inside the
    # timed region, overlapping the copies of one token chunk with the
    # kernels of its neighbours
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inp.items()}
    if args.shared_kv:
        host["v"] = host["k"]
    h_out, h_m, h_l = out.cpu().pin_memory(), smax.cpu().pin_memory(), ssum.cpu().pin_memory()
    res_host = tuple(torch.empty(o.shape, dtype=o.dtype).pin_memory() if o is not None else None for o in outs)
    in_list = [host["q"], host["k"], None if args.shared_kv else host["v"], host["indices"], host["d_out"], h_out,
               h_m, h_l, host["q_rope"], host["k_rope"], host.get("act_seq_q"), host.get("act_seq_kv")]
    h2d = sum(x.numel() * x.element_size() for x in in_list if x is not None)
    d2h = sum(x.numel() * x.element_size() for x in res_host if x is not None)
    # copy bandwidth of these pinned buffers on this machine (outside the
    # timed region): the bound on the copies the call overlaps with its kernels
    def copy_gbs(dst, src):
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            t = a.elapsed_time(b)
            best = t if best is None else min(best, t)
        return src.numel() * src.element_size() / best / 1e6
    h2d_gbs = copy_gbs(d["q"], host["q"])
    d2h_gbs = copy_gbs(res_host[0], outs[0])
    del ws
    torch.cuda.empty_cache()
    ws_h = torch.empty(sfa.grad_host_workspace_size(p), dtype=torch.uint8, device=dev)
    hkw = dict(q_rope=host["q_rope"], k_rope=host["k_rope"], sparse_block_size=w.block_size, layout=w.layout,
               sparse_mode=w.mode, act_seq_q=host.get("act_seq_q"), act_seq_kv=host.get("act_seq_kv"))
    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms, call_ms = [], []
    for i in range(e2e_steps + 2):
        flush.fill_(2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        c0 = time.perf_counter()
        sfa.grad_host(host["q"], host["k"], host["v"], host["indices"], host["d_out"], h_out, h_m, h_l,
                      w.scale_value, deterministic=det, outputs=res_host, workspace=ws_h, **hkw)
        c1 = time.perf_counter()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
            call_ms.append((c1 - c0) * 1e3)
    err = sfa.read_device_error(ws_h)
    if err != 0:
        raise RuntimeError(f"device error word {err} (host-buffer path)")
    e2e_mean = max_over_ranks(statistics.mean(e2e_ms), world, dev)
    e2e_value = job_tflops(world, flops, e2e_mean)

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    # Dominant kernel (largest summed time per step; a workload in several
    # token chunks launches each kernel once per chunk) and its roofline:
    # algorithmic work of all its launches over their summed time, which is the
    # per-launch work over the mean launch duration.
    by_name, n_by_name = {}, {}
    for j in range(launches):
        nm = names[j] if j < len(names) else f"launch{j}"
        by_name[nm] = by_name.get(nm, 0.0) + per_launch[j]
        n_by_name[nm] = n_by_name.get(nm, 0) + 1
    dname = max(by_name, key=by_name.get)
    k_ms, k_n = by_name[dname], n_by_name[dname]
    roof = roofline(dname, names, pairs * w.N1, pairs, k_ms, peaks, det)
    if args.traffic is not None:
        roof["traffic"] = args.traffic                        # given per launch
    else:
        shape = {"N1": w.N1, "K": w.K, "bs": w.block_size, "det": bool(det)}
        tr = kernel_traffic(dname, p.T1, shape)               # all tokens of the step
        roof["traffic"] = None if tr is None else tr / k_n    # per launch
    if roof["traffic"] is not None:
        # the kernel's measured DRAM traffic over its mean launch time, against
        # the HBM copy peak (a secondary bound: the contractions read mostly L2)
        gbs = roof["traffic"] / (k_ms / k_n * 1e-3) / 1e9
        roof["dram"] = {"achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"]}
    roof["kernel"] = dname
    roof["launches_per_step"] = k_n
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        # bounded sample: size the token count from a short probe run so the
        # timed oracle run takes about 12 s
        n0 = 8
        dt0, _, _ = cpu_oracle_sample(w, inp, n0)
        n = int(min(w.S1, max(n0, n0 * 12.0 / max(dt0, 1e-3))))
        dt, fl, sample = cpu_oracle_sample(w, inp, n)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample, "seconds": dt}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(w, det, args.shared_kv), "l2": "flushed between steps (256 MB write, outside the events)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "valid_query_head_key": pairs * w.N1},
        "frac_of_dense_bf16_peak": value / world / peaks["bf16_tflops"],
        "peak_source": peak_src,
        "per_kernel_ms": {f"{j}:{names[j] if j < len(names) else j}": round(per_launch[j], 4) for j in range(launches)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_mean, "h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
                "host_call_ms": round(statistics.mean(call_ms), 3),
                "call": "sfa_grad_host: pinned host inputs and outputs, copies overlapped with the kernels per token chunk"},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_forward(args):
    """Times the companion forward sfa_fwd (out, softmaxMax, softmaxSum) on the
    workload, same timing rules as the backward; one JSON line.  Work counted
    as 2 * (576 + 512) flops per valid (query, head, key): S and P.V."""
    import sfa_grad_gb300 as sfa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    kw = dict(q_rope=d["q_rope"], k_rope=d["k_rope"], sparse_block_size=w.block_size, layout=w.layout,
              sparse_mode=w.mode, act_seq_q=d.get("act_seq_q"), act_seq_kv=d.get("act_seq_kv"))
    p = sfa.make_params(d["q"], d["k"], d["indices"], w.scale_value, layout=w.layout,
                        sparse_block_size=w.block_size, sparse_mode=w.mode, has_rope=True,
                        batch=w.B if w.layout == "TND" else None)
    ws = torch.empty(max(sfa.fwd_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flops = valid_pairs(w, inp) * w.N1 * 2 * (576 + 512)
    for _ in range(args.warmup):
        flush.fill_(1)
        sfa.fwd(d["q"], d["k"], d["v"], d["indices"], w.scale_value, workspace=ws, **kw)
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sfa.fwd(d["q"], d["k"], d["v"], d["indices"], w.scale_value, workspace=ws, **kw)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.mean(times)
    peaks, peak_src = load_peaks()
    value = flops / (ms * 1e-3) / 1e12
    print(json.dumps({"metric": "sparse-attn fwd TFLOP/s (1×GB300)", "value": value, "unit": "TFLOP/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
                      "frac_of_dense_bf16_peak": value / peaks["bf16_tflops"], "peak_source": peak_src,
                      "config": {"workload": workload_desc(w, False),
                                 "l2": "flushed between steps (256 MB write, outside the events)"}}), flush=True)
    return 0


def run_l2_red_ceiling():
    """Builds and runs bench_l2_red.cu (L2-resident fp32 reduction rates by
    instruction shape) and prints its JSON line."""
    import tempfile
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bench_l2_red.cu")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "bench_l2_red")
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        print(r.stdout.strip(), flush=True)
        return r.returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["sfa", "reference"], default="sfa")
    ap.add_argument("--workload", default="mla", choices=list(WORKLOADS))
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--shared-kv", action="store_true",
                    help="pass the key tensor as the value tensor too (value identical to key)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward", action="store_true", help="time the companion forward sfa_fwd instead")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    ap.add_argument("--l2-red-ceiling", action="store_true",
                    help="measure the L2 fp32 reduction ceiling (bench_l2_red.cu) and exit")
    args = ap.parse_args()
    if args.l2_red_ceiling:
        return run_l2_red_ceiling()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.forward:
        return run_forward(args)
    return run_sfa(args)


if __name__ == "__main__":
    sys.exit(main())
