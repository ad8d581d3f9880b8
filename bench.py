#!/usr/bin/env python3
"""Benchmark of one decode-attention step (all of: split plan, phi-frame split partials, window
test, fallback recompute, combine) through libfdpp's C ABI on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl fdpp|reference]

Prints ONE JSON line (rank 0). The default workload is the paged continuous batch, the largest
single-GPU one: batch 64, 64 query / 8 kv heads, head_dim 128, seq_lens uniform in [512, 16384],
paged bf16 cache (block 16, permuted block table), split 512, phi 0, window [-30, 10]. `--config`
names one of workloads.ALL (e.g. long_context, gqa_decode, fallback_stress).

  value      KV-read GB/s: algorithmic K+V bytes of all ranks' steps (tokens t < L_b only) over the
             max-over-ranks device time of the K timed steps (CUDA events, inputs resident in HBM).
             The steps rotate over R copies of K/V totalling >= 4x the L2 size, so no step reuses
             the previous step's bytes from L2.
  e2e        the same metric through the C ABI with HOST buffers: each step copies q, seq_lens
             (and the block table) host->device from pinned memory, runs the step, copies the
             output back and synchronises. The K/V cache is resident device state.
  roofline   the split kernel: algorithmic KV bytes per launch over its launch time, against the
             measured HBM copy bandwidth of MEASURED_PEAKS.json. The launch time is the median of
             a separate pass after the timed region, CUDA events recorded right around each
             split kernel by fdpp_decode_attn_timed (>= 50 launches). Such events keep the launch
             from overlapping the previous kernel, so where that median exceeds the whole step's
             time (small steps) the step time is used instead, and `kernel_time_from` says so.
  cpu_baseline  the fp64 oracle on the host cores over a bounded sample of the same workload.

With --gpus N > 1 (torchrun) every rank runs its own seeded batch (weak scaling, no collective on
the data path); value sums all ranks' bytes over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-read GB/s (% of ~8 TB/s HBM peak) and µs/step at 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES_FALLBACK = 129 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="paged_batch")
    ap.add_argument("--impl", default="fdpp", choices=["fdpp", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--split-samples", type=int, default=100,
                    help="launches of the split-kernel timing pass (at least 50)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--kernel", type=int, default=0, help="fdpp_kernel (0 auto, 1 tensor, 2 simt)")
    ap.add_argument("--mode", type=int, default=0, help="fdpp_mode (0 normal, 1 fast, 2 online)")
    ap.add_argument("--tc-stages", type=int, default=0)
    ap.add_argument("--tc-ctas", type=int, default=0)
    ap.add_argument("--tc-prefetch", type=int, default=0)
    ap.add_argument("--tc-mma", type=int, default=0,
                    help="tensor kernel build for > 8 rows per kv head (0 auto, 1 mma.sync, 2 tcgen05)")
    ap.add_argument("--split-len", type=int, default=-1, help="override split_len (0 = auto)")
    ap.add_argument("--q-tokens", type=int, default=0,
                    help="override the workload's query tokens per sequence (rows per kv head = q_tokens G)")
    ap.add_argument("--stress-frac", type=float, default=-1.0,
                    help="override the workload's fraction of units given a hot key (fallback rate)")
    ap.add_argument("--split-k", type=int, default=0, help="flat GEMM configs: split_k (0 = auto)")
    ap.add_argument("--noalloc", action="store_true",
                    help="time fdpp_decode_attn_noalloc (the library's static scratch) in the "
                         "timed region instead of fdpp_decode_attn with a workspace")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--calibrate", action="store_true",
                    help="per-head phi chosen from the score ranges of a seeded sample of the "
                         "workload (another seed), then used for the timed steps")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.split_samples = max(50, args.split_samples)
    return args


# ------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier + max-over-ranks timing only)
# ------------------------------------------------------------------------------------------

class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend)
            self.pg = dist
        if n_gpus != self.world and not (n_gpus >= 1 and self.world == 1 and n_gpus == 1):
            if self.world == 1 and n_gpus > 1:
                raise SystemExit("--gpus N > 1 must be launched with torchrun (one rank per GPU)")

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(per_rank_bytes: float, per_rank_seconds: float, dist: Dist):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    total = dist.sum(per_rank_bytes)
    t = dist.max(per_rank_seconds)
    return total, t, (total / t / 1e9 if t > 0 else 0.0)


# ------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, enabled: bool):
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            # raw samples (the JSON line carries their summary): FDPP_BENCH_LOG_DIR, else the
            # system temporary directory
            out_dir = os.environ.get("FDPP_BENCH_LOG_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return None
        sm = [r[0] for r in rows]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), r[2:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def split_kernel_source_hash():
    h = hashlib.sha256()
    for name in ("split_tc.cu", "split_um.cu", "split_tc_common.cuh", "split_simt.cu", "combine.cu",
                 "device_common.cuh", "tcgen05.cuh", "fdpp_internal.h"):
        with open(os.path.join(ROOT, "split_kv_async_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gemm_kernel_source_hash():
    h = hashlib.sha256()
    for name in ("flat_gemm.cu", "device_common.cuh", "tcgen05.cuh", "fdpp_internal.h"):
        with open(os.path.join(ROOT, "split_kv_async_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config_name: str, kernel_name: str):
    """DRAM bytes per split-kernel launch from the committed ncu summary, when it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{config_name}/{kernel_name}")
    want = gemm_kernel_source_hash() if kernel_name == "flat_gemm" else split_kernel_source_hash()
    if not e or e.get("source_hash") != want:
        return None
    return e.get("dram_bytes_per_launch")


def _dev_tensor(a, dev):
    import numpy as np
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


# ------------------------------------------------------------------------------------------
# reference arm: the fp64 oracle, timed as it stands, on the host cores
# ------------------------------------------------------------------------------------------

def oracle_sample_rate(inp, budget_s=None, max_groups=None):
    """Times the oracle over whole (b, g) groups (all G query heads) until `budget_s` seconds
    are spent or `max_groups` groups are done. Returns (GB/s of algorithmic KV bytes, threads
    used, sample description, seconds, bytes)."""
    import numpy as np

    import oracle
    wl = inp.wl
    prob = oracle.make_problem(
        batch=wl.batch, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
        head_dim=wl.head_dim, dtype=oracle.F32 if wl.dtype == "f32" else oracle.BF16,
        scale=wl.scale, phi=wl.phi, lo=wl.lo, hi=wl.hi, max_seq_len=inp.max_seq_len,
        paged=wl.paged, block_size=wl.block_size, max_blocks_per_seq=inp.max_blocks_per_seq,
        q_tokens=wl.q_tokens)
    es = 4 if wl.dtype == "f32" else 2
    Tq = max(1, wl.q_tokens)
    groups = [(b, g) for b in range(wl.batch) for g in range(wl.num_kv_heads)]
    rng = np.random.default_rng(wl.seed ^ 0xC0FFEE)
    order = rng.permutation(len(groups))
    threads = oracle.default_threads()
    done_bytes, done_s, n_groups, i = 0, 0.0, 0, 0
    chunk = max(1, threads // max(1, wl.group))
    while (budget_s is None or done_s < budget_s) and (max_groups is None or n_groups < max_groups):
        c_n = chunk if max_groups is None else min(chunk, max_groups - n_groups)
        sel = [groups[order[(i + c) % len(groups)]] for c in range(c_n)]
        i += c_n
        # every query token of the group: query row b Tq + i, head g G + h
        rows = np.array([(b * Tq + i, g * wl.group + h) for (b, g) in sel for i in range(Tq)
                         for h in range(wl.group)], np.int32)
        t0 = time.perf_counter()
        _, used = oracle.attention(prob, inp.q, inp.k, inp.v, inp.seq_lens,
                                   block_table=inp.block_table, rows=rows, n_threads=threads)
        done_s += time.perf_counter() - t0
        threads = used if n_groups == 0 else threads
        done_bytes += sum(int(inp.seq_lens[b]) * wl.head_dim * 2 * es for (b, g) in sel)
        n_groups += len(sel)
    gbs = done_bytes / done_s / 1e9 if done_s > 0 else 0.0
    desc = (f"{n_groups} (sequence, kv-head) groups x {wl.group * Tq} query rows of {wl.name}, "
            f"{done_s:.1f} s of fp64 oracle work on {threads} threads")
    return gbs, threads, desc, done_s, done_bytes


def run_reference(args, dist: Dist):
    import workloads as W
    if dist.rank != 0:
        return None
    wl = W.ALL[args.config]
    inp = W.generate(wl)
    # each step is a bounded sample: a fixed number of (b, g) groups sized so that
    # warmup + steps fit in about args.cpu_budget_s * 10 seconds
    gbs, threads, _, _, _ = oracle_sample_rate(inp, budget_s=1.0)
    total_budget = 10.0 * args.cpu_budget_s
    avg_group_bytes = inp.kv_bytes / (wl.batch * wl.num_kv_heads)
    group_s = avg_group_bytes / (gbs * 1e9) if gbs > 0 else 1.0
    groups_per_step = max(1, int(total_budget / (args.steps + args.warmup) / group_s))
    groups_per_step = min(groups_per_step, wl.batch * wl.num_kv_heads)
    for _ in range(args.warmup):
        oracle_sample_rate(inp, max_groups=groups_per_step)
    t_sum, b_sum = 0.0, 0
    for _ in range(args.steps):
        _, _, _, t, b = oracle_sample_rate(inp, max_groups=groups_per_step)
        t_sum += t
        b_sum += b
    value = b_sum / t_sum / 1e9
    sample = (f"each step: the fp64 oracle on {groups_per_step} (sequence, kv-head) groups x "
              f"{wl.group} query heads of {wl.name} (of {wl.batch * wl.num_kv_heads}), "
              f"{threads} host threads")
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_sum / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
                   "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "split_len": wl.split_len},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------------------------------
# fdpp arm
# ------------------------------------------------------------------------------------------

def run_fdpp(args, dist: Dist):
    import numpy as np
    import torch

    import split_kv_async_gb300 as F
    import workloads as W

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    wl = W.ALL[args.config]
    if args.stress_frac >= 0:
        wl = wl.replace(stress_frac=args.stress_frac)
    if args.q_tokens > 0:
        wl = wl.replace(q_tokens=args.q_tokens)
    if dist.world > 1:
        wl = wl.replace(seed=wl.seed + 1000 * dist.rank)      # each rank its own batch
    # the heuristic dataflow's table, measured offline on this GPU model (attn_lut.py): kernel
    # choice for kernel 0, split scheduler targets for split_len 0
    from split_kv_async_gb300 import attn_lut
    lut_rows = attn_lut.apply()
    inp = W.generate(wl)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    kv_pool_bytes = inp.k.nbytes + inp.v.nbytes
    R = max(1, min(8, math.ceil(4 * l2 / kv_pool_bytes)))

    q = _dev_tensor(inp.q, dev)
    ks = [_dev_tensor(inp.k, dev)]
    vs = [_dev_tensor(inp.v, dev)]
    for _ in range(R - 1):
        ks.append(ks[0].clone())
        vs.append(vs[0].clone())
    sl = torch.from_numpy(inp.seq_lens).to(dev)
    bt = None if inp.block_table is None else torch.from_numpy(inp.block_table).to(dev)
    out = torch.empty_like(q)
    split_len = wl.split_len if args.split_len < 0 else args.split_len
    kw = dict(batch=wl.batch, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
              head_dim=wl.head_dim, dtype=F.FDPP_F32 if wl.dtype == "f32" else F.FDPP_BF16,
              max_seq_len=inp.max_seq_len, scale=wl.scale, phi=wl.phi, lo=wl.lo, hi=wl.hi,
              split_len=split_len, q_tokens=wl.q_tokens, mode=args.mode, kernel=args.kernel,
              tc_stages=args.tc_stages,
              tc_ctas_per_sm=args.tc_ctas, tc_prefetch=args.tc_prefetch, tc_mma=args.tc_mma)
    if wl.paged:
        kw.update(block_size=wl.block_size, max_blocks_per_seq=inp.max_blocks_per_seq,
                  num_kv_blocks=inp.num_kv_blocks,
                  max_seq_len=inp.max_blocks_per_seq * wl.block_size)
    p = F.make_params(**kw)
    ws = F.alloc_workspace(p, dev)
    calib = None
    if args.calibrate:
        # phi observed in advance: score ranges of a sample drawn with another seed, one phi per
        # head picked from them on the host; the timed steps then run with those values
        sample = W.generate(wl.replace(seed=wl.seed + 1))
        sq = _dev_tensor(sample.q, dev)
        sk = _dev_tensor(sample.k, dev)
        ssl = torch.from_numpy(sample.seq_lens).to(dev)
        sbt = None if sample.block_table is None else torch.from_numpy(sample.block_table).to(dev)
        pk = dict(kw)
        if wl.paged:
            pk.update(max_blocks_per_seq=sample.max_blocks_per_seq,
                      num_kv_blocks=sample.num_kv_blocks,
                      max_seq_len=sample.max_blocks_per_seq * wl.block_size)
        else:
            pk.update(max_seq_len=sample.max_seq_len)
        ps = F.make_params(**pk)
        wss = F.alloc_workspace(ps, dev)
        smin, smax, ns = F.fdpp_score_ranges(sq, sk, sbt, ssl, ps, wss)
        phi_np, kept = F.fdpp_pick_phi(smin, smax, ns, wl.lo, wl.hi, fallback=wl.phi)
        phi_dev = torch.from_numpy(phi_np).to(dev)
        kw["phi_heads"] = phi_dev
        p = F.make_params(**kw)
        calib = {"sample_seed": wl.seed + 1, "sample_row_splits": int(ns.sum()) * wl.num_q_heads,
                 "kept": int(kept.sum()), "phi_min": float(phi_np.min()),
                 "phi_max": float(phi_np.max())}
        del sq, sk, wss
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # raw C calls with pre-built arguments (the binding's per-call marshalling is not timed)
    call = F.lib.fdpp_decode_attn_timed
    pp = ctypes.byref(p)
    ws_bytes = ws.numel()
    argsets = [(q.data_ptr(), ks[i].data_ptr(), vs[i].data_ptr(),
                None if bt is None else bt.data_ptr(), sl.data_ptr(), pp, ws.data_ptr(), ws_bytes,
                out.data_ptr(), sh) for i in range(R)]

    noalloc = F.lib.fdpp_decode_attn_noalloc

    def step(i, eb=None, ee=None):
        if args.noalloc and eb is None:
            a_ = argsets[i % R]
            st = noalloc(a_[0], a_[1], a_[2], a_[3], a_[4], pp, a_[8], sh)
            if st != 0:
                raise F.FdppError(st, "fdpp_decode_attn_noalloc", F.fdpp_last_error())
            return
        st = call(*argsets[i % R], eb, ee)
        if st != 0:
            raise F.FdppError(st, "fdpp_decode_attn_timed", F.fdpp_last_error())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    diag, _, _ = F.fdpp_read_diag_noalloc(p) if args.noalloc else F.fdpp_read_diag(ws, p)
    kernel_name = {1: "tensor", 2: "simt"}.get(diag["kernel"], "?")

    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0,
                           enabled=not args.no_clocks and dist.local_rank == 0)
    time.sleep(0.25 if sampler.proc else 0.0)
    dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(K):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    diag, _, _ = F.fdpp_read_diag_noalloc(p) if args.noalloc else F.fdpp_read_diag(ws, p)

    # The split kernel alone, in a pass of its own after the timed region: events right around
    # it (fdpp_decode_attn_timed) and around the whole call, on every launch. torch creates an
    # event's CUDA handle on its first record: record each once first so that the raw handles
    # handed to the C call exist.
    n_samp = args.split_samples
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_samp)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_samp)]
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_samp)]
    for ev in ev_b + ev_e + ev_s:
        ev.record(stream)
    torch.cuda.synchronize()
    for k in range(n_samp):
        step(K + k, ev_b[k].cuda_event, ev_e[k].cuda_event)
        ev_s[k].record(stream)
    torch.cuda.synchronize()
    split_ms = sorted(ev_b[k].elapsed_time(ev_e[k]) for k in range(n_samp))
    alone_ms = sorted(ev_b[k].elapsed_time(ev_s[k]) for k in range(n_samp))

    def pct(xs, f):
        return xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]

    kv_bytes = inp.kv_bytes
    tot_bytes, t_max, value = aggregate(kv_bytes * K, total_ms / 1e3, dist)
    ms_per_step = t_max * 1e3 / K
    split_med_ms = statistics.median(split_ms)
    peak, peak_kind = measured_peaks()
    # the kernel cannot take longer than the step it is part of: events around a launch cost it
    # the overlap with the kernel before it, which matters only for short steps
    kernel_ms, kernel_from = split_med_ms, "split-kernel events, median of the separate pass"
    if split_med_ms > total_ms / K:
        kernel_ms, kernel_from = total_ms / K, "whole step (split-kernel median exceeded it)"
    achieved = kv_bytes / (kernel_ms / 1e3) / 1e9

    # End to end through the C ABI with host buffers: every step sends that step's inputs (q,
    # seq_lens and, paged, the block table), packed in one pinned host buffer, with one
    # host-to-device copy, runs fdpp_decode_attn, copies the output back to pinned host memory
    # and waits for it on the host. The step is captured once per K/V copy as a CUDA graph (the
    # two copies and the two kernels), so a step costs one graph launch and one wait.
    e2e = None
    if not args.no_e2e:
        def al(x):
            return (x + 255) // 256 * 256
        q_np = inp.q.view(np.uint8).reshape(-1)
        sl_np = inp.seq_lens.view(np.uint8).reshape(-1)
        bt_np = None if inp.block_table is None else inp.block_table.view(np.uint8).reshape(-1)
        off_sl = al(q_np.size)
        off_bt = al(off_sl + sl_np.size)
        h2d = off_bt + (0 if bt_np is None else bt_np.size)
        hin = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        hin_np = hin.numpy()
        hin_np[:q_np.size] = q_np
        hin_np[off_sl:off_sl + sl_np.size] = sl_np
        if bt_np is not None:
            hin_np[off_bt:off_bt + bt_np.size] = bt_np
        din = torch.empty(h2d, dtype=torch.uint8, device=dev)
        base = din.data_ptr()
        hout = torch.empty(out.numel() * out.element_size(), dtype=torch.uint8).pin_memory()
        out_bytes = out.view(-1).view(torch.uint8)
        d2h = out.numel() * out.element_size()

        def e2e_call(i, sh_):
            st = call(base, ks[i % R].data_ptr(), vs[i % R].data_ptr(),
                      None if bt_np is None else base + off_bt, base + off_sl, pp, ws.data_ptr(),
                      ws_bytes, out.data_ptr(), sh_, None, None)
            if st != 0:
                raise F.FdppError(st, "fdpp_decode_attn_timed", F.fdpp_last_error())

        def eager_step(i):
            din.copy_(hin, non_blocking=True)
            e2e_call(i, sh)
            hout.copy_(out_bytes, non_blocking=True)
            stream.synchronize()

        graphs, mode = [], "graph"
        try:
            side = torch.cuda.Stream(dev)
            for r in range(R):
                eager_step(r)                        # warm every path before capture
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
                    din.copy_(hin, non_blocking=True)
                    e2e_call(r, side.cuda_stream)
                    hout.copy_(out_bytes, non_blocking=True)
                graphs.append(g)
        except Exception as exc:                     # no graph capture here: eager steps
            graphs, mode = [], f"eager ({type(exc).__name__})"
        torch.cuda.synchronize()

        def e2e_step(i):
            if graphs:
                graphs[i % R].replay()
                stream.synchronize()
            else:
                eager_step(i)

        for i in range(3):
            e2e_step(i)
        dist.barrier()
        n = max(1, args.e2e_steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        _, t_e2e, v_e2e = aggregate(kv_bytes * n, e0.elapsed_time(e1) / 1e3, dist)
        e2e = {"value": v_e2e, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "us_per_step": t_e2e * 1e6 / n, "mode": mode}

    cpu = None
    if not args.no_cpu and dist.rank == 0:
        gbs, threads, desc, _, _ = oracle_sample_rate(inp, budget_s=args.cpu_budget_s)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc}

    if dist.rank != 0:
        return None
    traffic = recorded_traffic(wl.name, kernel_name)
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "pct_of_8TBps": 100.0 * value / dist.world / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * value / dist.world / peak,
        "config": {"workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
                   "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "seq_len": wl.seq_len if wl.seq_len else list(wl.seq_len_range),
                   "paged": wl.paged, "block_size": wl.block_size if wl.paged else None,
                   "q_tokens": max(1, wl.q_tokens),
                   "stress_frac": wl.stress_frac,
                   "split_len": diag["split_len"],
                   "split_len_from": ("lookup table" if lut_rows and split_len == 0 else
                                      "scheduler defaults" if split_len == 0 else "workload"),
                   "phi": wl.phi, "window": [wl.lo, wl.hi],
                   "kv_bytes_per_step": kv_bytes, "kernel": kernel_name,
                   "tensor_build": {0: None, 1: "mma.sync", 2: "tcgen05"}.get(diag.get("tc_build", 0)),
                   "tensor_parts": diag.get("tc_parts", 0) or None,
                   "tensor_phantom_tiles": diag.get("tc_seg_tiles", 0) if diag.get("tc_parts", 0) else None,
                   "l2_policy": f"rotate {R} K/V copies ({R * kv_pool_bytes / 2**20:.0f} MiB >= "
                                f"4x L2 {l2 / 2**20:.0f} MiB); no flush",
                   "parallelism": f"replicas{dist.world}" if dist.world > 1 else "single",
                   "entry_point": "fdpp_decode_attn_noalloc" if args.noalloc else "fdpp_decode_attn"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": traffic, "kernel": f"split_{kernel_name}",
                     "kernel_us": kernel_ms * 1e3, "kernel_time_from": kernel_from,
                     "split_kernel_us": {"median": split_med_ms * 1e3, "p10": pct(split_ms, 0.1) * 1e3,
                                         "p90": pct(split_ms, 0.9) * 1e3},
                     "timed_launches": n_samp},
        "step_alone_us": {"median": statistics.median(alone_ms) * 1e3,
                          "p10": pct(alone_ms, 0.1) * 1e3, "p90": pct(alone_ms, 0.9) * 1e3,
                          "about": "one call with events around it (no overlap with the step "
                                   "before), same pass as split_kernel_us"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "traffic_note": None if traffic is not None else
        "no ncu capture at the current kernel sources for this workload",
        "fallback": {"flagged_row_splits": diag["n_flagged_row_splits"],
                     "flagged_units": diag["n_flagged_units"], "units": diag["n_units"],
                     "unit_rate": diag["n_flagged_units"] / max(1, diag["n_units"])},
        "clocks": clocks,
        "error_bits": diag["error_bits"],
    }
    if calib is not None:
        res["config"]["phi"] = "per head, calibrated"
        res["calibration"] = calib
    return res


GEMM_METRIC = "flat-GEMM (decode linear layer y = x W^T) bytes GB/s and µs/call at 1 GB300"


def gemm_oracle_rate(x, w, budget_s):
    """The oracle's rate on sampled entries of the product, as bytes of the whole call per
    second (time per entry x M x N for the whole product)."""
    import numpy as np
    import oracle
    M, K = x.shape
    N = w.shape[0]
    rng = np.random.default_rng(1)
    threads = oracle.default_threads()
    done, t_sum, n = 0, 0.0, 4 * threads
    while t_sum < budget_s:
        ent = np.stack([rng.integers(0, M, n), rng.integers(0, N, n)], axis=1)
        t0 = time.perf_counter()
        oracle.flat_gemm(x, w, entries=ent, n_threads=threads)
        t_sum += time.perf_counter() - t0
        done += n
        n = min(n * 2, 1 << 20)
    per_entry = t_sum / done
    call_bytes = (N * K + M * K + M * N) * 2
    return call_bytes / (per_entry * M * N) / 1e9, threads, (
        f"{done} sampled entries of the {M}x{N}x{K} product, {t_sum:.1f} s of fp64 oracle work on "
        f"{threads} threads, scaled to the whole product")


def run_gemm(args, dist: Dist):
    import numpy as np
    import torch

    import split_kv_async_gb300 as F
    import workloads as W

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    wl = W.GEMM[args.config]
    if dist.world > 1:
        wl = wl.replace(seed=wl.seed + 1000 * dist.rank)
    x_np, w_np = W.gemm_inputs(wl)
    M, N, K = wl.M, wl.N, wl.K
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    w_bytes = w_np.nbytes
    R = max(1, min(64, math.ceil(4 * l2 / w_bytes)))
    x = _dev_tensor(x_np, dev)
    ws_ = [_dev_tensor(w_np, dev)]
    for _ in range(R - 1):
        ws_.append(ws_[0].clone())
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    # the heuristic dataflow's table, measured offline on this GPU model (gemm_lut.py)
    from split_kv_async_gb300 import gemm_lut
    lut_rows = gemm_lut.apply() if args.split_k == 0 else 0
    split = F.fdpp_flat_gemm_split_k(M, N, K, args.split_k)
    work = F.alloc_flat_gemm_workspace(M, N, K, split, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    call = F.lib.fdpp_flat_gemm
    wsb = work.numel()

    def step(i):
        st = call(x.data_ptr(), ws_[i % R].data_ptr(), y.data_ptr(), M, N, K, split, work.data_ptr(),
                  wsb, sh)
        if st != 0:
            raise F.FdppError(st, "fdpp_flat_gemm", F.fdpp_last_error())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    Ksteps = args.steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0,
                           enabled=not args.no_clocks and dist.local_rank == 0)
    time.sleep(0.25 if sampler.proc else 0.0)
    dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(Ksteps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    call_bytes = (N * K + M * K + M * N) * 2
    _, t_max, value = aggregate(call_bytes * Ksteps, total_ms / 1e3, dist)
    us = t_max * 1e6 / Ksteps
    peak, peak_kind = measured_peaks()
    achieved = call_bytes / (total_ms / 1e3 / Ksteps) / 1e9
    err = F.fdpp_flat_gemm_read_error(work)

    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

        def e2e_step(i):
            x.copy_(hx, non_blocking=True)
            step(i)
            hy.copy_(y, non_blocking=True)
            stream.synchronize()

        for i in range(3):
            e2e_step(i)
        n = max(1, args.e2e_steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        _, t_e2e, v_e2e = aggregate(call_bytes * n, e0.elapsed_time(e1) / 1e3, dist)
        e2e = {"value": v_e2e, "unit": "GB/s", "h2d_bytes_per_step": int(x_np.nbytes),
               "d2h_bytes_per_step": int(M * N * 2), "us_per_step": t_e2e * 1e6 / n, "mode": "eager"}

    cpu = None
    if not args.no_cpu and dist.rank == 0:
        gbs, threads, desc = gemm_oracle_rate(x_np, w_np, args.cpu_budget_s)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc}
    if dist.rank != 0:
        return None
    return {
        "metric": GEMM_METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": Ksteps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "us_per_step": us, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tflops": 2.0 * M * N * K / (us * 1e-6) / 1e12 * dist.world,
        "config": {"workload": wl.name, "M": M, "N": N, "K": K, "split_k": split,
                   "split_k_from": ("request" if args.split_k else
                                    "lookup table" if lut_rows else "heuristic"),
                   "bytes_per_call": call_bytes,
                   "l2_policy": f"rotate {R} weight copies ({R * w_bytes / 2**20:.0f} MiB >= 4x L2 "
                                f"{l2 / 2**20:.0f} MiB); no flush",
                   "parallelism": f"replicas{dist.world}" if dist.world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": recorded_traffic(wl.name, "flat_gemm"), "kernel": "flat_gemm_kernel",
                     "kernel_us": us},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": Ksteps, "clocks": clocks, "error_bits": err,
    }


def main(argv=None):
    args = parse_args(argv)
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            res = run_reference(args, dist)
        else:
            import __graft_entry__
            if dist.rank == 0:
                __graft_entry__.build()
            dist.barrier()
            __graft_entry__.build()
            res = run_gemm(args, dist) if args.config.startswith("gemm_") else run_fdpp(args, dist)
        if res is not None and dist.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
