#!/usr/bin/env python3
"""Benchmark of UniPrefill block scoring + top-p selection + compaction on GB300.

One step = one pass of the whole hot path (up_score_blocks, up_select_topp,
up_compact) over one batch of synthetic Llama-3.1-8B-layer-shaped input
(default: one 131072-token sequence, 32 query / 8 KV heads, head_dim 128,
hidden 4096, n = 128, G = 64, p = 0.99).  Inputs are resident in HBM when the
timed region starts; k (268 MB) and x (1.07 GB) are larger than the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank processes its own copy of the batch (the
path shards by sequence; there is no data-path collective): weak scaling.
--impl reference times the fp64 CPU oracle on the host cores instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scored+compacted prefill tokens/s at N=128K Llama-8B shape; % of roofline"
UNIT = "tokens/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama31_8b_128k")
    ap.add_argument("--gain", default="5", help="logit gain of the planted shifts, or 'literal'")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def gain_of(s):
    return None if s == "literal" else float(s)


# ---------------------------------------------------------------- work model

def valid_pairs(inp):
    """Visible (query, key) pairs per query head: sum_s n_s*L_s - n_s(n_s-1)/2."""
    tot = 0
    for s in range(inp.num_seqs):
        L = int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s])
        ns = min(inp.n, L)
        tot += ns * L - ns * (ns - 1) // 2
    return tot


def work_model(inp, G):
    pairs = valid_pairs(inp)
    flops = 2.0 * inp.d * inp.Hq * pairs
    exps = float(inp.Hq * pairs)
    nb = sum((int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s]) + G - 1) // G
             for s in range(inp.num_seqs))
    score_bytes = inp.k.nbytes + inp.q_last.nbytes + 4 * nb + 4 * (inp.num_seqs + 1)
    return dict(flops=flops, exps=exps, score_bytes=score_bytes, blocks=nb)


def step_roofline(wm, cbytes, tflops, hbm_gbs, ex2_rate, tokens, ms_step):
    """Tokens/s of one step if every phase ran at its roof: scoring at the larger
    of its tensor time and its K/Q/score HBM time, plus compaction at HBM speed
    (the form the workload names), and the same with the exponential roof as a
    third scoring term."""
    t_mma = wm["flops"] / (tflops * 1e12)
    t_bytes = wm["score_bytes"] / (hbm_gbs * 1e9)
    t_exp = wm["exps"] / ex2_rate
    t_cmp = cbytes / (hbm_gbs * 1e9)
    roof = tokens / (max(t_mma, t_bytes) + t_cmp)
    roof_exp = tokens / (max(t_mma, t_bytes, t_exp) + t_cmp)
    value = tokens / (ms_step * 1e-3)
    return dict(tokens_per_s=roof, frac=value / roof, tokens_per_s_with_exp=roof_exp,
                frac_with_exp=value / roof_exp,
                terms_us=dict(score_tensor=t_mma * 1e6, score_hbm=t_bytes * 1e6,
                              score_exp=t_exp * 1e6, compact_hbm=t_cmp * 1e6))


def compact_bytes(kept_tokens, hidden):
    # x rows read + written, positions read + written
    return kept_tokens * (2 * 2 * hidden + 8)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profiled_traffic(workload, d, G):
    """DRAM bytes per launch of the scoring kernel from the committed ncu summary,
    or None when the summary is for another workload or the kernel source has
    changed since the counters were taken."""
    import hashlib
    if workload != "llama31_8b_128k" or d != 128 or G != 64:
        return None
    summary = os.path.join(ROOT, "profiles", "score_tc_llama31_8b_128k.md")
    src = os.path.join(ROOT, "block_sparse_long_up_gb300", "csrc", "score_tc.cu")
    try:
        text = open(summary).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines()
                  if line.startswith(("source_sha256_16:", "dram_bytes_per_launch:")))
    if fields.get("source_sha256_16", "").strip() != sha:
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(inp, heads, queries, threads, G, p, cache=None):
    """Time the fp64 oracle on a sample: the first `heads` query heads (with
    their KV heads) and the last `queries` queries of every sequence, over all
    keys, then top-p and compaction of the result.  Returns (seconds, fraction
    of the full workload's scoring work, heads used, queries used).  `cache`
    (a dict) keeps the sliced inputs of a sample size between calls."""
    import oracle
    g = inp.Hq // inp.Hk
    hs = max(1, min(heads, inp.Hq))
    kv = (hs + g - 1) // g
    hs = min(inp.Hq, kv * g) if hs > g else hs
    nq = max(1, min(queries, inp.n))
    key = (hs, nq)
    if cache is not None and key in cache:
        q, k, rows = cache[key]
    else:
        rows, qsel = [], []
        off = 0
        for s in range(inp.num_seqs):
            L = int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s])
            ns = min(inp.n, L)
            keep_q = min(nq, ns)
            qsel.append(inp.q_last[off + ns - keep_q: off + ns, :hs])
            rows.append(keep_q)
            off += ns
        q = np.ascontiguousarray(np.concatenate(qsel, axis=0))
        k = np.ascontiguousarray(inp.k[:, :kv])
        if cache is not None:
            cache[key] = (q, k, rows)
    t0 = time.perf_counter()
    sc, cb = oracle.score_blocks(q, k, inp.cu_seqlens, hs, kv, inp.d, nq, G, nthreads=threads)
    keep, _, _, _ = oracle.select_topp(sc, cb, inp.cu_seqlens, G, p)
    oracle.compact(inp.x, inp.pos, inp.cu_seqlens, G, keep, cb, with_x=inp.x is not None)
    dt = time.perf_counter() - t0
    full_rows = sum(min(inp.n, int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s]))
                    for s in range(inp.num_seqs)) * inp.Hq
    frac = (sum(rows) * hs) / max(1, full_rows)
    return dt, frac, hs, nq


def cpu_model():
    parts = {"0xd4f": "Arm Neoverse V2"}  # Arm's CPU part numbers
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":", 1)[0].strip().lower()
            if key == "model name":
                return line.split(":", 1)[1].strip()
            if key == "cpu part":
                part = line.split(":", 1)[1].strip()
                return f"{parts.get(part, 'Arm')} (CPU part {part})"
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, inp, w):
    """--impl reference: the oracle, as it stands, on the host cores."""
    cores = cpu_cores()
    threads = cores
    budget = 150.0 / max(1, args.steps + args.warmup)  # seconds per step
    cache = {}
    # calibrate on one query of one head (one thread), select and compact included
    dt1, frac1, _, _ = oracle_sample(inp, 1, 1, 1, w["G"], w["p"], cache)
    per_row = max(dt1, 1e-4)
    # the oracle's threads split the query heads, so `threads` heads cost the time
    # of one: sample that many heads (or all), then as many queries as fit the
    # budget, then further heads in whole batches of `threads`
    heads = min(inp.Hq, threads)
    queries = max(1, min(inp.n, int(budget / per_row)))
    if queries == inp.n:
        batches = max(1, int(budget / (per_row * inp.n)))
        heads = min(inp.Hq, threads * batches)
    times = []
    for i in range(args.warmup + args.steps):
        dt, frac, hs, nq = oracle_sample(inp, heads, queries, threads, w["G"], w["p"], cache)
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    value = inp.total_tokens * frac / t
    used = min(threads, hs)
    sample = (f"{hs} of {inp.Hq} query heads x last {nq} of {inp.n} queries over all "
              f"{inp.total_tokens} keys per step (fraction {frac:.4g} of the scoring work), "
              f"value scaled to the full workload")
    return dict(metric=METRIC, value=value, unit=UNIT, impl="reference", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=t * 1e3 / frac,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=workload_config(args, inp, w, 1),
                cpu_baseline=dict(value=value, unit=UNIT, cores=used, kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


# ---------------------------------------------------------------- GPU arm

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(args, inp, w, world):
    return dict(workload=args.workload, tokens=inp.total_tokens, num_seqs=inp.num_seqs,
                Hq=inp.Hq, Hk=inp.Hk, head_dim=inp.d, hidden=inp.hidden, n=inp.n, G=w["G"],
                p=w["p"], gain=args.gain,
                parallelism=f"replica x{world}" if world > 1 else "single",
                l2="inputs larger than L2 (k %.0f MB, x %.0f MB > 129 MB); no flush"
                   % (inp.k.nbytes / 1e6, (inp.x.nbytes if inp.x is not None else 0) / 1e6))


def run_ours(args, inp, w, rank, world):
    import torch
    import block_sparse_long_up_gb300 as up

    up.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    G, p, n = w["G"], w["p"], inp.n

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    h_q = bf16(inp.q_last).pin_memory()
    h_k = bf16(inp.k).pin_memory()
    h_x = bf16(inp.x).pin_memory()
    h_cu = torch.from_numpy(inp.cu_seqlens).pin_memory()
    h_pos = torch.from_numpy(inp.pos).pin_memory()
    q, k, x = h_q.to(dev), h_k.to(dev), h_x.to(dev)
    cu, pos = h_cu.to(dev), h_pos.to(dev)
    sp = up.Sparsifier(inp.num_seqs, inp.total_tokens, inp.Hq, inp.Hk, inp.d, inp.hidden, n, G, p,
                       device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        sp.run(q, k, cu, x, pos)
    torch.cuda.synchronize()
    if up.get_device_error():
        raise RuntimeError("device error during warm-up")
    kept = int(sp.total_kept.item())
    kept_blocks = int(sp.keep[: int(sp.cu_blocks[-1].item())].sum().item())
    ex2_rate = up.measure_ex2_rate()  # the exponential roof, measured on this GPU

    # timed region: K steps.  The scoring kernel is timed live by the pair of
    # events the library records around it, on every KS-th step only: an event
    # between two kernels cuts their programmatic overlap, so recording it every
    # step would slow the step it measures.  Per-call events are left out for the
    # same reason; the per-call breakdown is taken in a separate loop below,
    # outside the headline number.
    K = args.steps
    KS = 16
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range((K + KS - 1) // KS)]
    KB = min(K, 200)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KB)]
    for group in ev + evb:
        for event in group:
            event.record(stream)  # creates the CUDA events before the timed region
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_uuid)
    start.record(stream)
    for i in range(K):
        sampled = i % KS == 0
        if sampled:
            up.set_kernel_timing_events(ev[i // KS][0], ev[i // KS][1])
        sp.run(q, k, cu, x, pos)
        if sampled:
            up.set_kernel_timing_events(None, None)
    end.record(stream)
    up.set_kernel_timing_events(None, None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms_total = start.elapsed_time(end)
    ms_step = max_over_ranks(ms_total / K, world)
    t_kernel = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    if up.get_device_error():
        raise RuntimeError("device error during the timed region")

    # per-call breakdown (not part of the headline): events between the calls
    keep_k = torch.empty_like(sp.keep)
    kt_k = torch.empty_like(sp.kept_tokens)
    for i in range(KB):
        e = evb[i]
        e[0].record(stream)
        up.score_blocks(q, k, cu, n, G, sp.scores, sp.cu_blocks, sp.ws_score)
        e[1].record(stream)
        up.select_topp(sp.scores, sp.cu_blocks, cu, G, p, sp.keep, sp.kept_tokens)
        e[2].record(stream)
        up.compact(x, pos, cu, G, sp.keep, sp.cu_blocks, sp.x_out, sp.pos_out, sp.cu_out,
                   sp.src_idx, sp.total_kept, sp.ws_compact)
        e[3].record(stream)
        # the top-k rule (same ranking) at the block count top-p kept, into scratch flags
        up.select_blocks(sp.scores, sp.cu_blocks, cu, G, mode="top_k", k=max(1, kept_blocks),
                         keep=keep_k, kept_tokens=kt_k)
        e[4].record(stream)
    torch.cuda.synchronize()
    t_score = statistics.mean(e[0].elapsed_time(e[1]) for e in evb)
    t_select = statistics.mean(e[1].elapsed_time(e[2]) for e in evb)
    t_compact = statistics.mean(e[2].elapsed_time(e[3]) for e in evb)
    t_select_k = statistics.mean(e[3].elapsed_time(e[4]) for e in evb)

    # end to end: host (pinned) inputs -> device, the three calls, result -> host
    E = args.e2e_steps
    h_total = torch.empty(1, dtype=torch.int32).pin_memory()
    h_cuo = torch.empty(inp.num_seqs + 1, dtype=torch.int32).pin_memory()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(max(E, 1) if E > 0 else 0):
        q.copy_(h_q, non_blocking=True)
        k.copy_(h_k, non_blocking=True)
        x.copy_(h_x, non_blocking=True)
        cu.copy_(h_cu, non_blocking=True)
        pos.copy_(h_pos, non_blocking=True)
        sp.run(q, k, cu, x, pos)
        h_total.copy_(sp.total_kept, non_blocking=True)
        h_cuo.copy_(sp.cu_out, non_blocking=True)
        torch.cuda.synchronize()
        assert int(h_total[0]) == kept
    e2e_s = max_over_ranks((time.perf_counter() - t0) / max(E, 1), world) if E > 0 else None
    h2d = h_q.nbytes + h_k.nbytes + h_x.nbytes + h_cu.nbytes + h_pos.nbytes
    d2h = h_total.nbytes + h_cuo.nbytes

    wm = work_model(inp, G)
    peaks, peak_src = measured_peaks()
    tc_peak = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    achieved = wm["flops"] / (t_kernel * 1e-3) / 1e12
    traffic = profiled_traffic(args.workload, inp.d, w["G"])
    cbytes = compact_bytes(kept, inp.hidden)
    value = world * inp.total_tokens / (ms_step * 1e-3)
    out = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
        ms_per_step=ms_step, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16", data="synthetic",
        config=workload_config(args, inp, w, world),
        clocks=clk,
        e2e=(dict(value=world * inp.total_tokens / e2e_s, unit=UNIT, h2d_bytes_per_step=h2d,
                  d2h_bytes_per_step=d2h, ms_per_step=e2e_s * 1e3) if e2e_s else None),
        gpu_launches=K * sp.launches_per_step(),
        roofline=dict(kernel="score_tc_kernel (tcgen05 scoring)", bound="tensor",
                      achieved=achieved, peak=tc_peak, unit="TFLOP/s", frac=achieved / tc_peak,
                      traffic=traffic, kernel_ms=t_kernel,
                      algorithmic_bytes=wm["score_bytes"],
                      peak_source=f"{peak_src} bf16 sustained (kernel timed inside a long loop)",
                      kernel_timing=f"CUDA events around the kernel on every {KS}th timed step "
                                    f"({len(ev)} samples)",
                      exp_rate_per_s=wm["exps"] / (t_kernel * 1e-3)),
        exp_roof=dict(kernel="score_tc_kernel", achieved=wm["exps"] / (t_kernel * 1e-3),
                      peak=ex2_rate, unit="exp/s", frac=wm["exps"] / (t_kernel * 1e-3) / ex2_rate,
                      peak_source="measured in this run (up_measure_ex2_rate microbenchmark)"),
        step_roofline=step_roofline(wm, cbytes, tc_peak, float(peaks["hbm_gbs"]), ex2_rate,
                                    inp.total_tokens * world, ms_step),
        calls_ms=dict(score=t_score, score_kernel=t_kernel, select=t_select, compact=t_compact,
                      select_topk=t_select_k),
        compact_roofline=dict(bound="hbm", achieved=cbytes / (t_compact * 1e-3) / 1e9,
                              peak=float(peaks["hbm_gbs"]), unit="GB/s",
                              frac=cbytes / (t_compact * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                              bytes=cbytes),
        kept=dict(tokens=kept, blocks=kept_blocks, blocks_total=wm["blocks"],
                  rho=kept / inp.total_tokens),
    )
    return out


def main():
    args = parse_args()
    from block_sparse_long_up_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        inp = synth.make_workload(args.workload, gain=gain_of(args.gain))
        out = run_reference(args, inp, w)
        out["n_gpus"] = world
        out["config"] = workload_config(args, inp, w, world)
        print(json.dumps(out), flush=True)
        return 0
    rank, world = dist_setup()
    inp = synth.make_workload(args.workload, gain=gain_of(args.gain))
    out = run_ours(args, inp, w, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            # one query head per host core (the oracle's threads split the heads)
            threads = max(1, min(cpu_cores(), inp.Hq))
            dt, frac, hs, nq = oracle_sample(inp, threads, inp.n, threads, w["G"], w["p"])
            out["cpu_baseline"] = dict(
                value=inp.total_tokens * frac / dt, unit=UNIT, cores=min(threads, hs),
                kind="oracle", cpu=cpu_model(),
                sample=f"{hs} of {inp.Hq} query heads x {nq} queries over all {inp.total_tokens} "
                       f"keys (fraction {frac:.4g} of the scoring work) plus top-p and "
                       f"compaction; tokens/s scaled to the full workload")
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
