"""The heuristic dataflow's lookup table for decode attention, made offline by measurement.

opt.ai.kr "FlashDecoding++ async softmax -- theory", sections 2(3) and 4: one static dataflow
loses on some shapes, so the configuration is chosen per shape range from a table measured in
advance. For decode attention the shape is (batch, cache length, query rows per kv head) and
the configuration is the split kernel (tensor cores or CUDA cores) and the split scheduler's
target of units per SM, which sets the split length when a call asks for split_len = 0.

``sweep`` times every candidate on the current GPU for each shape at the top of each range,
``rows`` keeps the fastest per range as rows for ``fdpp_attn_set_lut`` (ranges ascending, so
the first row that holds a shape is its range), and ``apply`` loads a table file written by this
module when it was measured on a GPU with the current device's SM count.

    python -m split_kv_async_gb300.attn_lut --out split_kv_async_gb300/attn_lut_gb300.json
"""
from __future__ import annotations

import argparse
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_TABLE = os.path.join(HERE, "attn_lut_gb300.json")

HKV, HEAD_DIM = 8, 128
BATCHES = (1, 8, 64)                  # range tops; the last range is open
SEQ_LENS = (2048, 16384, 131072)
ROWS = (4, 8, 16, 64)                 # query rows per kv head (one query token: G; 64: a prefill chunk)
UNITS = (1, 2, 4, 8, 16)
MIN_SPLIT = 256
MAX_TOKENS = 1 << 21                  # batch x length measured (larger shapes take their range)
OPEN = 1 << 30


def _time_us(F, torch, p, q, ks, vs, sl, ws, out, iters=30, reps=3):
    """Median per-call time of chained fdpp_decode_attn calls over rotated K/V copies."""
    copies = len(ks)
    for i in range(5):
        F.fdpp_decode_attn(q, ks[i % copies], vs[i % copies], None, sl, p, ws, out)
    torch.cuda.synchronize()
    res = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(iters):
            F.fdpp_decode_attn(q, ks[i % copies], vs[i % copies], None, sl, p, ws, out)
        e1.record()
        torch.cuda.synchronize()
        res.append(e0.elapsed_time(e1) * 1e3 / iters)
    diag, _, _ = F.fdpp_read_diag(ws, p)
    if diag["error_bits"]:
        raise RuntimeError(f"device error bits {diag['error_bits']}")
    res.sort()
    return res[len(res) // 2]


def sweep(batches=BATCHES, seq_lens=SEQ_LENS, rows=ROWS, units=UNITS):
    """{(B, L, R): {(kernel, units): us}} on the current GPU (bf16, head_dim 128, 8 kv heads,
    one query token, N(0, 1) inputs)."""
    import torch
    import split_kv_async_gb300 as F
    dev = torch.device("cuda")
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20)
    F.fdpp_attn_set_lut([])
    res = {}
    for B in batches:
        for L in seq_lens:
            if B * L > MAX_TOKENS:
                continue
            kv_bytes = B * L * HKV * HEAD_DIM * 2
            copies = max(1, min(8, math.ceil(4 * l2 / (2 * kv_bytes))))
            g = torch.Generator(device=dev)
            g.manual_seed(B * 7919 + L)
            ks = [torch.randn((B, L, HKV, HEAD_DIM), generator=g, device=dev).to(torch.bfloat16)
                  for _ in range(copies)]
            vs = [torch.randn((B, L, HKV, HEAD_DIM), generator=g, device=dev).to(torch.bfloat16)
                  for _ in range(copies)]
            sl = torch.full((B,), L, dtype=torch.int32, device=dev)
            for R in rows:
                Hq = R * HKV
                q = torch.randn((B, Hq, HEAD_DIM), generator=g, device=dev).to(torch.bfloat16)
                out = torch.empty_like(q)
                t = {}
                kernels = [F.FDPP_KERNEL_TENSOR] + ([F.FDPP_KERNEL_SIMT] if R <= 16 else [])
                for kern in kernels:
                    for u in units:
                        F.fdpp_attn_set_lut([(OPEN, OPEN, OPEN, kern, u, MIN_SPLIT)])
                        p = F.make_params(batch=B, num_q_heads=Hq, num_kv_heads=HKV,
                                          head_dim=HEAD_DIM, dtype=F.FDPP_BF16, max_seq_len=L,
                                          scale=float(HEAD_DIM ** -0.5), split_len=0)
                        ws = F.alloc_workspace(p, dev)
                        t[(kern, u)] = _time_us(F, torch, p, q, ks, vs, sl, ws, out)
                        del ws
                res[(B, L, R)] = t
            del ks, vs
            torch.cuda.empty_cache()
    F.fdpp_attn_set_lut([])
    return res


def rows_from(res, batches=BATCHES, seq_lens=SEQ_LENS, rows=ROWS):
    """Rows (max_batch, max_seq_len, max_rows, kernel, units_per_sm, min_split), ranges
    ascending; each range takes the fastest configuration measured at its top (or, for a shape
    too large to measure, at the largest measured shape below it in the same column)."""
    out = []
    b_tops = list(batches[:-1]) + [OPEN]
    l_tops = list(seq_lens[:-1]) + [OPEN]
    r_tops = list(rows[:-1]) + [64]
    for bi, B in enumerate(batches):
        for li, L in enumerate(seq_lens):
            for ri, R in enumerate(rows):
                key = (B, L, R)
                b2 = bi
                while key not in res and b2 > 0:      # too large: the largest measured batch
                    b2 -= 1
                    key = (batches[b2], L, R)
                if key not in res:
                    continue
                t = res[key]
                (kern, u), _ = min(t.items(), key=lambda kv: kv[1])
                out.append((b_tops[bi], l_tops[li], r_tops[ri], kern, u, MIN_SPLIT))
    return out


def apply(path=DEFAULT_TABLE) -> int:
    """Loads the table file into libfdpp when it was measured on a GPU with this SM count;
    returns the rows installed (0: none)."""
    import torch
    import split_kv_async_gb300 as F
    if not os.path.exists(path):
        return 0
    with open(path) as f:
        d = json.load(f)
    sms = torch.cuda.get_device_properties(torch.device("cuda")).multi_processor_count
    if int(d.get("num_sms", -1)) != sms:
        return 0
    rows = [tuple(r) for r in d["rows"]]
    F.fdpp_attn_set_lut(rows)
    return len(rows)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=DEFAULT_TABLE)
    args = ap.parse_args(argv)
    import torch
    props = torch.cuda.get_device_properties(torch.device("cuda"))
    res = sweep()
    rows = rows_from(res)
    doc = {
        "about": "heuristic dataflow table of decode attention: the fastest (kernel, units per SM) "
                 "per (batch, max_seq_len, rows per kv head) range, measured by attn_lut.sweep "
                 "(bf16, head_dim 128, 8 kv heads, one query token); rows for fdpp_attn_set_lut",
        "gpu": props.name, "num_sms": props.multi_processor_count,
        "columns": ["max_batch", "max_seq_len", "max_rows", "kernel", "units_per_sm", "min_split"],
        "rows": rows,
        "measured_us": {f"B{B}_L{L}_R{R}": {f"k{k}_u{u}": round(v, 2) for (k, u), v in t.items()}
                        for (B, L, R), t in res.items()},
    }
    with open(args.out, "w") as f:
        json.dump(doc, f, indent=1)
    print(f"{len(rows)} rows -> {args.out}")


if __name__ == "__main__":
    main()
