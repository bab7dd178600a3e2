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

Besides the headline the JSON line carries: the scoring kernel's roofline
(burst bf16 peak, >= 100 CUDA-event samples), clocks sampled while the same
step runs for over a second, a per-call breakdown (also the paged-key,
tensor-parallel-shard and block-CSR calls), select + compact against HBM on
the headline keep set and on the dense keep set of the literal input reading,
every other workload's step and scoring-kernel time, and the parity of the
headline run against the fp64 oracle.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
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
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama31_8b_128k")
    ap.add_argument("--gain", default="5", help="logit gain of the planted shifts, or 'literal'")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--kernel-samples", type=int, default=200)
    ap.add_argument("--clock-window-s", type=float, default=1.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads, the literal keep set and the extra calls")
    return ap.parse_args()


def gain_of(s):
    return None if s == "literal" else float(s)


# ---------------------------------------------------------------- work model

def valid_pairs(cu_seqlens, n):
    """Visible (query, key) pairs per query head: sum_s n_s*L_s - n_s(n_s-1)/2."""
    tot = 0
    for s in range(len(cu_seqlens) - 1):
        L = int(cu_seqlens[s + 1] - cu_seqlens[s])
        ns = min(n, L)
        tot += ns * L - ns * (ns - 1) // 2
    return tot


def work_model(inp, G, n=None):
    n = inp.n if n is None else n
    pairs = valid_pairs(inp.cu_seqlens, n)
    flops = 2.0 * inp.d * inp.Hq * pairs
    exps = float(inp.Hq * pairs)
    nb = sum((int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s]) + G - 1) // G
             for s in range(inp.num_seqs))
    nq = sum(min(n, int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s])) for s in range(inp.num_seqs))
    score_bytes = inp.k.nbytes + nq * inp.Hq * inp.d * 2 + 4 * nb + 4 * (inp.num_seqs + 1)
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
    """nvidia-smi polled every 50 ms in the background; samples carry their
    wall-clock time, so those inside a given interval can be picked out."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.rows = []

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None  # an unreadable time stamp: the sample counts for every window
                try:
                    self.rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]),
                                      {nm for nm, v in zip(self.REASONS, parts[6:10])
                                       if v.lower() == "active"}))
                except ValueError:
                    continue
        os.unlink(self.path)

    def summary(self, t0, t1, label):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sel = [r for r in self.rows if r[0] is None or t0 - 0.06 <= r[0] <= t1 + 0.06]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "window": label}
        reasons = set()
        for r in sel:
            reasons |= r[4]
        return {"sm_mhz": statistics.median(r[1] for r in sel),
                "sm_max_mhz": max(r[2] for r in sel), "power_w_max": max(r[3] for r in sel),
                "samples": len(sel), "reasons": sorted(reasons), "window": label}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash():
    """Hash of the sources the tensor-core scoring kernel is compiled from."""
    h = hashlib.sha256()
    for fn in ("score_tc.cu", "sm100.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "block_sparse_long_up_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, d, G):
    """DRAM bytes per launch of the scoring kernel from the committed ncu
    counters (profiles/score_tc_counters.json), or None when there are none for
    this workload or the kernel's sources have changed since they were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "score_tc_counters.json")) as f:
            entry = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, "no counters file"
    if not entry or entry.get("head_dim") != d or entry.get("G") != G:
        return None, "no counters for this workload"
    if entry.get("source_sha256_16") != kernel_source_hash():
        return None, "kernel source changed since the counters were taken"
    return int(entry["dram_bytes_per_launch"]), "ncu, " + entry.get("file", "profiles/")


# ---------------------------------------------------------------- CPU oracle timing

def _slice_inputs(inp, heads, queries):
    """The first `heads` query heads (whole GQA groups past the first) and the
    last `queries` queries of every sequence, over all keys."""
    g = inp.Hq // inp.Hk
    hs = max(1, min(heads, inp.Hq))
    kv = (hs + g - 1) // g
    hs = min(inp.Hq, kv * g) if hs > g else hs
    nq = max(1, min(queries, inp.n))
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
    full_rows = sum(min(inp.n, int(inp.cu_seqlens[s + 1] - inp.cu_seqlens[s]))
                    for s in range(inp.num_seqs)) * inp.Hq
    return q, k, hs, kv, nq, (sum(rows) * hs) / max(1, full_rows)


def oracle_score(inp, sliced, threads, G):
    """Time the oracle's scoring on a slice (see _slice_inputs)."""
    import oracle
    q, k, hs, kv, nq, frac = sliced
    t0 = time.perf_counter()
    sc, cb = oracle.score_blocks(q, k, inp.cu_seqlens, hs, kv, inp.d, nq, G, nthreads=threads)
    return time.perf_counter() - t0, sc, cb


def oracle_select_compact(inp, sc, cb, G, p):
    """Time the oracle's top-p selection and compaction at full size (their cost
    does not depend on how many heads or queries the scores came from)."""
    import oracle
    t0 = time.perf_counter()
    keep, _, ci, ce = oracle.select_topp(sc, cb, inp.cu_seqlens, G, p)
    oracle.compact(inp.x, inp.pos, inp.cu_seqlens, G, keep, cb, with_x=inp.x is not None)
    return time.perf_counter() - t0, keep, ci, ce


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
    """--impl reference: the oracle, as it stands, on the host cores.  Each step
    scores a sample of the workload (as many query heads as host threads, the
    oracle's threads split the heads, and as many of the last queries as fit the
    per-step budget) and scales that time to the full workload; selection and
    compaction are timed at full size and added unscaled."""
    threads = cpu_cores()
    G, p = w["G"], w["p"]
    budget = 150.0 / max(1, args.steps + args.warmup)  # seconds per step
    one = _slice_inputs(inp, 1, 1)
    dt1, sc1, cb1 = oracle_score(inp, one, 1, G)
    t_sc, _, _, _ = oracle_select_compact(inp, sc1, cb1, G, p)
    per_row = max(dt1, 1e-4)
    heads = min(inp.Hq, threads)
    queries = max(1, min(inp.n, int(max(budget - t_sc, 0.0) / per_row)))
    if queries == inp.n:
        batches = max(1, int(max(budget - t_sc, 0.0) / (per_row * inp.n)))
        heads = min(inp.Hq, threads * batches)
    sliced = _slice_inputs(inp, heads, queries)
    frac = sliced[5]
    times = []
    for i in range(args.warmup + args.steps):
        dt, sc, cb = oracle_score(inp, sliced, threads, G)
        ds, _, _, _ = oracle_select_compact(inp, sc, cb, G, p)
        if i >= args.warmup:
            times.append(dt / frac + ds)
    t = sum(times) / len(times)
    value = inp.total_tokens / t
    hs, nq = sliced[2], sliced[4]
    sample = (f"scoring: {hs} of {inp.Hq} query heads x last {nq} of {inp.n} queries over all "
              f"{inp.total_tokens} keys per step (fraction {frac:.4g} of the scoring work), its "
              f"time scaled to the full workload; top-p and compaction at full size, unscaled")
    return dict(metric=METRIC, value=value, unit=UNIT, impl="reference", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=t * 1e3,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=workload_config(args, inp, w, 1),
                cpu_baseline=dict(value=value, unit=UNIT, cores=min(threads, hs), kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def cpu_baseline_and_parity(inp, w, g_scores, g_keep, g_kept):
    """The oracle at full size on the host cores (scoring, then top-p and
    compaction) -- the CPU baseline -- and the headline run's parity against it:
    block scores, kept set (mismatches inside the band around p counted, not
    failed), kept tokens, and the mass split between the sink block, the planted
    salient blocks and the rest."""
    threads = max(1, min(cpu_cores(), inp.Hq))
    G, p = w["G"], w["p"]
    full = _slice_inputs(inp, inp.Hq, inp.n)
    dt, sc, cb = oracle_score(inp, full, threads, G)
    ds, keep, ci, ce = oracle_select_compact(inp, sc, cb, G, p)
    base = dict(value=inp.total_tokens / (dt + ds), unit=UNIT, cores=threads, kind="oracle",
                cpu=cpu_model(), score_s=dt, select_compact_s=ds,
                sample=f"the full workload: all {inp.Hq} query heads x {inp.n} queries over all "
                       f"{inp.total_tokens} keys ({threads} threads), then top-p and compaction")
    nb = len(sc)
    g = g_scores[:nb].astype(np.float64)
    rel = np.abs(g - sc) / np.maximum(np.abs(sc), 1e-30)
    tol_ok = np.abs(g - sc) <= np.maximum(1e-3 * np.abs(sc), 1e-6)
    diff = g_keep[:nb].astype(bool) != keep.astype(bool)
    band = (np.abs(ci - p) <= 1e-4) | (np.abs(ce - p) <= 1e-4)
    split = {}
    if inp.num_seqs == 1 and G == 64 and inp.planted:
        sal = np.asarray(inp.planted[0], dtype=np.int64)
        split = dict(sink=float(g[0]), salient=float(g[sal].sum()),
                     rest=float(1.0 - g[0] - g[sal].sum()), salient_blocks=int(len(sal)))
    parity = dict(scores_within_tolerance=bool(tol_ok.all()),
                  max_rel_score_err=float(rel.max()), max_abs_score_err=float(np.abs(g - sc).max()),
                  kept_set_equal=bool(not diff.any()), kept_mismatch_hard=int((diff & ~band).sum()),
                  kept_mismatch_excused=int((diff & band).sum()),
                  kept_blocks=int(g_keep[:nb].sum()), kept_blocks_oracle=int(keep.sum()),
                  kept_tokens=int(g_kept), rho=g_kept / inp.total_tokens, mass_split=split,
                  tolerance="|gpu-oracle| <= max(1e-3*|oracle|, 1e-6) per block; kept sets "
                            "bit-exact outside |cumulative mass - p| <= 1e-4")
    return base, parity


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


def _bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _dev_x(tokens, hidden, seed, dev):
    """Hidden states drawn on the device (seeded N(0,1) rounded to bf16) for the
    timing-only workloads: a bit copy's time does not depend on the values, and
    drawing gigabytes on the host would take minutes."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return torch.randn(tokens, hidden, generator=gen, device=dev, dtype=torch.float32).to(
        torch.bfloat16)


def _kernel_times(up, sp, q, k, cu, x, pos, reps, flush=None):
    """Scoring-kernel durations (ms) over `reps` full steps: the library records
    a pair of events around its tensor-core kernel on each step."""
    import torch
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for a, b in ev:
        if flush is not None:
            flush()
        up.set_kernel_timing_events(a, b)
        sp.run(q, k, cu, x, pos)
    up.set_kernel_timing_events(None, None)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def _time_steps(up, sp, q, k, cu, x, pos, steps, flush=None):
    """Mean step time (ms): back to back between two events, or, with an L2
    flush between steps, each step between its own pair of events."""
    import torch
    stream = torch.cuda.current_stream()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            sp.run(q, k, cu, x, pos)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        sp.run(q, k, cu, x, pos)
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def other_workloads(up, dev, peaks, tc_peak_burst):
    """GPU-only step and scoring-kernel timings of the other workloads at
    n = 128, G = 64 (q and k from the seeded host recipe, x drawn on the device).
    The 4K and 32K workloads fit in L2 and are timed one step at a time with a
    flush (a 2 x L2 write) before each step; the others exceed L2."""
    import torch
    from block_sparse_long_up_gb300 import synth
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    out = {}
    for name in ("gqa8x2_d64_4k", "llama31_8b_32k", "llama31_8b_varlen8_392k",
                 "gqa16x2_d256_128k_sweep"):
        w = synth.WORKLOADS[name]
        G, p = 64, w["p"]
        inp = synth.make_workload(name, with_x=False, n=128)
        q, k = _bf16(inp.q_last).to(dev), _bf16(inp.k).to(dev)
        cu = torch.from_numpy(inp.cu_seqlens).to(dev)
        pos = torch.from_numpy(np.concatenate(
            [np.arange(int(L), dtype=np.int32) for L in np.diff(inp.cu_seqlens)])).to(dev)
        x = _dev_x(inp.total_tokens, w["hidden"], w["seed"], dev)
        sp = up.Sparsifier(inp.num_seqs, inp.total_tokens, inp.Hq, inp.Hk, inp.d, w["hidden"],
                           128, G, p, device=dev)
        # keys within twice the L2 size could stay partly cached between steps
        fits_l2 = inp.k.nbytes < 2 * L2_BYTES
        fl = flush if fits_l2 else None
        for _ in range(5):
            sp.run(q, k, cu, x, pos)
        torch.cuda.synchronize()
        steps = 100 if fits_l2 else max(20, min(200, int(0.05 / (inp.total_tokens / 1.0e9))))
        ms = _time_steps(up, sp, q, k, cu, x, pos, steps, fl)
        kt = _kernel_times(up, sp, q, k, cu, x, pos, 100, fl)
        if up.get_device_error():
            raise RuntimeError(f"device error in workload {name}")
        kept = int(sp.total_kept.item())
        wm = work_model(inp, G, 128)
        k_ms = statistics.mean(kt)
        ach = wm["flops"] / (k_ms * 1e-3) / 1e12
        out[name] = dict(
            tokens=inp.total_tokens, n=128, G=G, p=p, ms_per_step=ms,
            tokens_per_s=inp.total_tokens / (ms * 1e-3), score_kernel_us=k_ms * 1e3,
            score_kernel_samples=len(kt), score_tflops=ach, score_frac_burst=ach / tc_peak_burst,
            kept_tokens=kept, rho=kept / inp.total_tokens,
            l2="flushed before each step (k within 2x L2)" if fl else "inputs larger than L2",
            x="drawn on the device (seeded); q, k from the host recipe",
            note="launch-bound (4096 tokens): the roofline fraction is not meaningful"
                 if inp.total_tokens <= 4096 else None)
        del q, k, cu, pos, x, sp
        torch.cuda.empty_cache()
    del flush_buf
    torch.cuda.empty_cache()
    return out


def run_ours(args, inp, w, rank, world):
    import torch
    import block_sparse_long_up_gb300 as up
    from block_sparse_long_up_gb300 import synth

    up.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    G, p, n = w["G"], w["p"], inp.n

    h_q = _bf16(inp.q_last).pin_memory()
    h_k = _bf16(inp.k).pin_memory()
    h_x = _bf16(inp.x).pin_memory()
    h_cu = torch.from_numpy(inp.cu_seqlens).pin_memory()
    h_pos = torch.from_numpy(inp.pos).pin_memory()
    q, k, x = h_q.to(dev), h_k.to(dev), h_x.to(dev)
    cu, pos = h_cu.to(dev), h_pos.to(dev)
    sp = up.Sparsifier(inp.num_seqs, inp.total_tokens, inp.Hq, inp.Hk, inp.d, inp.hidden, n, G, p,
                       device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):  # first calls: per-device set-up, kernel attributes
        sp.run(q, k, cu, x, pos)
    torch.cuda.synchronize()
    if up.get_device_error():
        raise RuntimeError("device error during warm-up")
    kept = int(sp.total_kept.item())
    nb = int(sp.cu_blocks[-1].item())
    kept_blocks = int(sp.keep[:nb].sum().item())
    g_scores = sp.scores[:nb].cpu().numpy()
    g_keep = sp.keep[:nb].cpu().numpy()
    ex2_rate = up.measure_ex2_rate()  # the exponential roof, measured on this GPU

    # timed region: K steps back to back on one stream.  The scoring kernel is
    # also timed live by the pair of events the library records around it, on
    # every KS-th step only: an event between two kernels cuts their
    # programmatic overlap, so recording it every step would slow the step it
    # measures.  A dedicated loop below takes >= 100 samples.
    K = args.steps
    KS = 16
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range((K + KS - 1) // KS)]
    for group in ev:
        for event in group:
            event.record(stream)  # creates the CUDA events before the timed region
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid)
    time.sleep(0.2)  # the sampler's first reading comes before the timed region
    # the W warm-up steps run right before the timed region, so the GPU is not
    # left idle (clocks down) between them
    for _ in range(max(args.warmup, 3)):
        sp.run(q, k, cu, x, pos)
    barrier(world)
    torch.cuda.synchronize()
    t_region0 = time.time()
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
    t_region1 = time.time()
    barrier(world)
    ms_total = start.elapsed_time(end)
    ms_step = max_over_ranks(ms_total / K, world)
    t_kernel_region = [e[0].elapsed_time(e[1]) for e in ev]
    if up.get_device_error():
        raise RuntimeError("device error during the timed region")

    # clock window: the same step, back to back, for a second or more, so the
    # sampler sees the clocks under this load (the timed region at small K is
    # shorter than its period)
    t_win0 = time.time()
    while time.time() - t_win0 < args.clock_window_s:
        for _ in range(200):
            sp.run(q, k, cu, x, pos)
        torch.cuda.synchronize()
    t_win1 = time.time()
    clocks.stop()
    clk = clocks.summary(t_region0, t_win1, "the timed region and a %.1f s run of the same step "
                         "right after it" % (t_win1 - t_win0))
    clk["samples_in_timed_region"] = len([r for r in clocks.rows if r[0] is not None and
                                          t_region0 - 0.06 <= r[0] <= t_region1 + 0.06])

    # the scoring kernel alone: >= 100 samples
    kt = _kernel_times(up, sp, q, k, cu, x, pos, max(100, args.kernel_samples))
    t_kernel = statistics.mean(kt)

    # per-call breakdown (not part of the headline): events between the calls
    KB = 100
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KB)]
    keep_k = torch.empty_like(sp.keep)
    kt_k = torch.empty_like(sp.kept_tokens)
    torch.cuda.synchronize()
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
        # select and compact with no event between them (their kernels overlap)
        up.select_topp(sp.scores, sp.cu_blocks, cu, G, p, sp.keep, sp.kept_tokens)
        up.compact(x, pos, cu, G, sp.keep, sp.cu_blocks, sp.x_out, sp.pos_out, sp.cu_out,
                   sp.src_idx, sp.total_kept, sp.ws_compact)
        e[5].record(stream)
    torch.cuda.synchronize()
    calls = dict(score=statistics.mean(e[0].elapsed_time(e[1]) for e in evb),
                 score_kernel=t_kernel,
                 select=statistics.mean(e[1].elapsed_time(e[2]) for e in evb),
                 compact=statistics.mean(e[2].elapsed_time(e[3]) for e in evb),
                 select_topk=statistics.mean(e[3].elapsed_time(e[4]) for e in evb),
                 select_compact=statistics.mean(e[4].elapsed_time(e[5]) for e in evb))
    if not args.no_extras:
        calls.update(extra_calls(up, sp, q, k, cu, inp, n, G, KB))

    # end to end: host (pinned) inputs -> device, the three calls, result -> host
    # Every step's inputs come from pinned host memory: q, k and cu_seqlens are
    # copied to the device; x and pos are read in place by the compaction,
    # which takes only the kept rows across the host link (up_compact accepts
    # pinned host rows); the kept count and cu_seqlens_out are read back.
    E = args.e2e_steps
    h_total = torch.empty(1, dtype=torch.int32).pin_memory()
    h_cuo = torch.empty(inp.num_seqs + 1, dtype=torch.int32).pin_memory()

    def e2e_loop(steps, copy_rows):
        # one untimed step first: the first pass over the pinned buffers pays
        # one-off costs (35-120 ms in one run of this bench, 3 ms in isolation)
        if steps <= 0:
            return None
        barrier(world)
        torch.cuda.synchronize()
        t0 = None
        for i in range(steps + 1):
            if i == 1:
                t0 = time.perf_counter()
            q.copy_(h_q, non_blocking=True)
            k.copy_(h_k, non_blocking=True)
            cu.copy_(h_cu, non_blocking=True)
            if copy_rows:
                x.copy_(h_x, non_blocking=True)
                pos.copy_(h_pos, non_blocking=True)
                sp.run(q, k, cu, x, pos)
            else:
                sp.run(q, k, cu, h_x, h_pos)
            h_total.copy_(sp.total_kept, non_blocking=True)
            h_cuo.copy_(sp.cu_out, non_blocking=True)
            torch.cuda.synchronize()
            assert int(h_total[0]) == kept
        return max_over_ranks((time.perf_counter() - t0) / steps, world)

    e2e_s = e2e_loop(E, copy_rows=False)
    # diagnostic: the same steps with x and pos copied to the device whole first
    e2e_copy_s = e2e_loop(min(E, 3), copy_rows=True)
    # the copies' own bandwidth (events around each, one pass after the loop, on
    # the pinned buffers the timed steps have already used)
    cev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize()
    cev[0].record(stream)
    k.copy_(h_k, non_blocking=True)
    cev[1].record(stream)
    x.copy_(h_x, non_blocking=True)
    cev[2].record(stream)
    torch.cuda.synchronize()
    h2d_gbs = dict(k=h_k.nbytes / (cev[0].elapsed_time(cev[1]) * 1e-3) / 1e9,
                   x=h_x.nbytes / (cev[1].elapsed_time(cev[2]) * 1e-3) / 1e9)
    h2d_copied = h_q.nbytes + h_k.nbytes + h_cu.nbytes
    h2d_in_place = kept * (h_x.shape[1] * h_x.element_size() + h_pos.element_size())
    h2d = h2d_copied + h2d_in_place
    d2h = h_total.nbytes + h_cuo.nbytes

    wm = work_model(inp, G)
    peaks, peak_src = measured_peaks()
    tc_burst = float(peaks["bf16_tflops"])
    tc_sust = float(peaks.get("bf16_tflops_sustained") or tc_burst)
    hbm = float(peaks["hbm_gbs"])
    achieved = wm["flops"] / (t_kernel * 1e-3) / 1e12
    traffic, traffic_src = profiled_traffic(args.workload, inp.d, w["G"])
    cbytes = compact_bytes(kept, inp.hidden)
    value = world * inp.total_tokens / (ms_step * 1e-3)
    out = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
        ms_per_step=ms_step, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16", data="synthetic",
        config=workload_config(args, inp, w, world),
        clocks=clk,
        e2e=(dict(value=world * inp.total_tokens / e2e_s, unit=UNIT, h2d_bytes_per_step=h2d,
                  d2h_bytes_per_step=d2h, ms_per_step=e2e_s * 1e3,
                  h2d_copied_bytes=h2d_copied, h2d_read_in_place_bytes=h2d_in_place,
                  inputs="q, k, cu_seqlens copied from pinned host memory; x and pos read in "
                         "place from pinned host memory by the compaction (kept rows only); "
                         "one untimed step before the timed ones",
                  copy_all_rows=dict(value=world * inp.total_tokens / e2e_copy_s,
                                     ms_per_step=e2e_copy_s * 1e3,
                                     h2d_bytes_per_step=h2d_copied + h_x.nbytes + h_pos.nbytes),
                  h2d_copy_gbs={n: round(v, 1) for n, v in h2d_gbs.items()})
             if e2e_s else None),
        gpu_launches=K * sp.launches_per_step(),
        roofline=dict(kernel="score_tc_kernel (tcgen05 scoring)", bound="tensor",
                      achieved=achieved, peak=tc_burst, unit="TFLOP/s", frac=achieved / tc_burst,
                      traffic=traffic, traffic_source=traffic_src, kernel_ms=t_kernel,
                      kernel_ms_median=statistics.median(kt),
                      kernel_ms_timed_region=(statistics.mean(t_kernel_region)
                                              if t_kernel_region else None),
                      algorithmic_flops=wm["flops"], algorithmic_bytes=wm["score_bytes"],
                      peak_source=f"{peak_src} bf16 burst (the kernel runs ~0.1 ms at a time)",
                      frac_of_sustained=achieved / tc_sust,
                      kernel_timing=f"CUDA events around the kernel on each of {len(kt)} steps "
                                    f"after the timed region ({len(t_kernel_region)} more inside "
                                    f"it, every {KS}th step)"),
        exp_roof=dict(kernel="score_tc_kernel", achieved=wm["exps"] / (t_kernel * 1e-3),
                      peak=ex2_rate, unit="exp/s", frac=wm["exps"] / (t_kernel * 1e-3) / ex2_rate,
                      peak_source="measured in this run (up_measure_ex2_rate microbenchmark)"),
        step_roofline=step_roofline(wm, cbytes, tc_burst, hbm, ex2_rate,
                                    inp.total_tokens * world, ms_step),
        calls_ms=calls,
        compact_roofline=dict(bound="hbm", achieved=cbytes / (calls["compact"] * 1e-3) / 1e9,
                              peak=hbm, unit="GB/s",
                              frac=cbytes / (calls["compact"] * 1e-3) / 1e9 / hbm, bytes=cbytes,
                              select_compact_frac=cbytes / (calls["select_compact"] * 1e-3) / 1e9
                              / hbm,
                              # select + compact inside the pipelined step: the step's time
                              # less the scoring call's (plan + scoring kernel), both timed here
                              in_step_us=(ms_step - calls["score"]) * 1e3,
                              in_step_frac=(cbytes / ((ms_step - calls["score"]) * 1e-3) / 1e9 / hbm
                                            if ms_step > calls["score"] else None)),
        kept=dict(tokens=kept, blocks=kept_blocks, blocks_total=wm["blocks"],
                  rho=kept / inp.total_tokens),
    )
    if not args.no_extras and inp.num_seqs == 1 and args.gain != "literal":
        out["compact_roofline_literal"] = literal_compact(up, dev, args, w, x, pos, cu, hbm)
        out["workloads"] = other_workloads(up, dev, peaks, tc_burst)
    return out, g_scores, g_keep, kept


def extra_calls(up, sp, q, k, cu, inp, n, G, reps):
    """Times of the calls outside the three-call step: scoring from a paged
    KV-head-major cache (pages of 256 keys in shuffled order), scoring one
    tensor-parallel shard (half the KV heads with their query heads, the mean
    over all query heads), and the block-CSR of the kept blocks."""
    import torch
    stream = torch.cuda.current_stream()
    page = 256
    T, Hk, d = k.shape
    npg = (T + page - 1) // page
    kp = torch.zeros(npg * page, Hk, d, dtype=k.dtype, device=k.device)
    kp[:T] = k
    pages = kp.view(npg, page, Hk, d).transpose(1, 2).contiguous()  # [pages, Hk, page, d]
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(5)).to(k.device)
    pool = torch.empty_like(pages)
    pool[perm] = pages
    table = perm.to(torch.int32).view(1, npg)
    del kp, pages
    qs, ks = up.shard_heads(q, k, 0, 2)
    ws_shard = torch.empty(up.score_blocks_workspace(inp.num_seqs, T, qs.shape[1], ks.shape[1], d,
                                                     n, G), dtype=torch.uint8, device=k.device)
    indptr = torch.empty(inp.num_seqs + 1, dtype=torch.int32, device=k.device)
    indices = torch.empty_like(sp.scores, dtype=torch.int32)
    sc2 = torch.empty_like(sp.scores)
    cb2 = torch.empty_like(sp.cu_blocks)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    torch.cuda.synchronize()
    for e in ev:
        e[0].record(stream)
        up.score_blocks_paged(q, pool, table, cu, T, n, G, sc2, cb2, sp.ws_score)
        e[1].record(stream)
        up.score_blocks(qs, ks, cu, n, G, sc2, cb2, ws_shard, Hq_total=inp.Hq)
        e[2].record(stream)
        up.block_csr(sp.keep, sp.cu_blocks, indptr, indices)
        e[3].record(stream)
    torch.cuda.synchronize()
    if up.get_device_error():
        raise RuntimeError("device error in the extra calls")
    res = dict(score_paged=statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
               score_shard_half_heads=statistics.mean(e[1].elapsed_time(e[2]) for e in ev),
               block_csr=statistics.mean(e[2].elapsed_time(e[3]) for e in ev),
               extra_calls_note=f"paged: {npg} pages of {page} keys, shuffled; shard: "
                                f"{qs.shape[1]}/{inp.Hq} query and {ks.shape[1]}/{Hk} KV heads")
    del pool, table, qs, ks, ws_shard
    torch.cuda.empty_cache()
    return res


def literal_compact(up, dev, args, w, x, pos, cu, hbm):
    """Selection + compaction on the dense keep set: the same 128K layer drawn
    with the literal unit-vector shifts (rho ~ 0.99, ~2.1 GB gathered), where
    compaction is HBM-bound.  Scored once on the GPU; select + compact timed
    together (one event pair, so their kernels overlap as in the step)."""
    import torch
    from block_sparse_long_up_gb300 import synth
    lit = synth.make_workload(args.workload, gain=None, with_x=False)
    q, k = _bf16(lit.q_last).to(dev), _bf16(lit.k).to(dev)
    sp = up.Sparsifier(lit.num_seqs, lit.total_tokens, lit.Hq, lit.Hk, lit.d, x.shape[1], lit.n,
                       w["G"], w["p"], device=dev)
    up.score_blocks(q, k, cu, lit.n, w["G"], sp.scores, sp.cu_blocks, sp.ws_score)
    del q, k
    stream = torch.cuda.current_stream()

    def sel_cmp():
        up.select_topp(sp.scores, sp.cu_blocks, cu, w["G"], w["p"], sp.keep, sp.kept_tokens)
        up.compact(x, pos, cu, w["G"], sp.keep, sp.cu_blocks, sp.x_out, sp.pos_out, sp.cu_out,
                   sp.src_idx, sp.total_kept, sp.ws_compact)

    for _ in range(3):
        sel_cmp()
    torch.cuda.synchronize()
    reps = 20
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        sel_cmp()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    kept = int(sp.total_kept.item())
    if up.get_device_error():
        raise RuntimeError("device error in the literal keep set")
    by = compact_bytes(kept, x.shape[1])
    del sp
    torch.cuda.empty_cache()
    return dict(bound="hbm", achieved=by / (ms * 1e-3) / 1e9, peak=hbm, unit="GB/s",
                frac=by / (ms * 1e-3) / 1e9 / hbm, bytes=by, ms=ms, kept_tokens=kept,
                rho=kept / lit.total_tokens,
                what="select + compact, back to back (inputs > L2, no flush)")


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
    out, g_scores, g_keep, kept = run_ours(args, inp, w, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            base, parity = cpu_baseline_and_parity(inp, w, g_scores, g_keep, kept)
            out["cpu_baseline"] = base
            out["parity"] = parity
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
