"""The heuristic dataflow's lookup table for the flat GEMM, made offline by measurement.

opt.ai.kr "FlashDecoding++ async softmax -- theory", s4: a model's linear layers come down to a
few weight shapes N x K (Q/K/V generation, O projection, the two FFN matrices) that never change,
while M (the batch's query tokens) does; so the kernel configuration is chosen per M range from a
table measured in advance, instead of one static choice for every shape.

Here the configuration is split_k, the number of K ranges per 128-row weight tile. ``sweep``
times every candidate split for each (N, K) at the top of each M range on the current GPU and
keeps the fastest; ``entries`` turns the result into rows (m_max, N, K, split_k) for
``fdpp_flat_gemm_set_lut``. ``apply`` loads a table file written by this module, when it was
measured on a GPU with the current device's SM count.

    python -m split_kv_async_gb300.gemm_lut --out split_kv_async_gb300/gemm_lut_gb300.json
"""
from __future__ import annotations

import argparse
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_TABLE = os.path.join(HERE, "gemm_lut_gb300.json")

# The decoder-block linear layers of the bench (hidden 4096, 8 kv heads of 128, FFN 14336).
LAYERS = ((6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336))
M_BUCKETS = (1, 8, 16, 32, 64, 128)
SPLITS = (1, 2, 3, 4, 5, 6, 7, 8)


def _weights(torch, N, K):
    """Seeded weight copies totalling >= 4x L2, so that every timed call reads W from HBM."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(N * 131 + K)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20)
    copies = max(1, min(32, math.ceil(4 * l2 / (N * K * 2))))
    return [torch.randn((N, K), generator=g, device=dev).to(torch.bfloat16) for _ in range(copies)]


def _time_us(F, torch, ws_, M, split, iters=60, reps=3):
    """Median per-call time of fdpp_flat_gemm with the weights rotated over `ws_`."""
    dev = torch.device("cuda")
    N, K = ws_[0].shape
    copies = len(ws_)
    g = torch.Generator(device=dev)
    g.manual_seed(M)
    x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    work = F.alloc_flat_gemm_workspace(M, N, K, split)
    for i in range(5):
        F.fdpp_flat_gemm(x, ws_[i % copies], y, work, split_k=split)
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(iters):
            F.fdpp_flat_gemm(x, ws_[i % copies], y, work, split_k=split)
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / iters)
    if F.fdpp_flat_gemm_read_error(work):
        raise RuntimeError(f"device error bits after M={M} N={N} K={K} split={split}")
    out.sort()
    return out[len(out) // 2]


def sweep(layers=LAYERS, m_buckets=M_BUCKETS, splits=SPLITS):
    """{(N, K, M): {split: us}} on the current GPU."""
    import torch
    import split_kv_async_gb300 as F
    res = {}
    for N, K in layers:
        kb = (K + 63) // 64
        ws_ = _weights(torch, N, K)
        for M in m_buckets:
            t = {}
            for s in splits:
                if s <= min(kb, 8):
                    t[s] = _time_us(F, torch, ws_, M, s)
            res[(N, K, M)] = t
        del ws_
        torch.cuda.empty_cache()
    return res


def entries(res):
    """Rows (m_max, N, K, split_k): the fastest split at the top of each M range."""
    rows = []
    for (N, K, M), t in sorted(res.items()):
        best = min(t, key=t.get)
        rows.append((M, N, K, best))
    return rows


def apply(path=DEFAULT_TABLE) -> int:
    """Loads the table at `path` into the library when it was measured on a GPU with this
    device's SM count; returns the number of entries set (0: no table or another GPU)."""
    import torch
    import split_kv_async_gb300 as F
    if not os.path.exists(path):
        return 0
    with open(path) as f:
        t = json.load(f)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if t.get("sms") != sms:
        return 0
    F.fdpp_flat_gemm_set_lut(t["entries"])
    return len(t["entries"])


def main(argv=None):
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=DEFAULT_TABLE)
    args = ap.parse_args(argv)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    res = sweep()
    table = {
        "about": "flat GEMM split_k per (M range, N, K), fastest measured by gemm_lut.sweep",
        "device": props.name, "sms": props.multi_processor_count,
        "entries": [list(r) for r in entries(res)],
        "timings_us": {f"{N}x{K}@M{M}": {str(s): round(v, 2) for s, v in t.items()}
                       for (N, K, M), t in sorted(res.items())},
    }
    with open(args.out, "w") as f:
        json.dump(table, f, indent=1)
    print(json.dumps({"entries": table["entries"]}))


if __name__ == "__main__":
    main()
