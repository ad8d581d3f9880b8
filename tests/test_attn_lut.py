"""The heuristic dataflow table of decode attention on the host (no GPU): the library's lookup
(fdpp_attn_set_lut / fdpp_attn_auto_choice) against the oracle's restatement of the table rule,
on the table measured on GB300 and on random tables; the argument checks; and the offline
builder's pick of the fastest configuration per range.

opt.ai.kr "FlashDecoding++ async softmax -- theory", s2(3) and s4: a static dataflow loses on
some shapes, so the configuration is taken per shape range from a table measured in advance."""
import json
import os

import numpy as np
import pytest

import oracle
import split_kv_async_gb300 as F
from split_kv_async_gb300 import attn_lut


@pytest.fixture(autouse=True)
def _clear_table():
    F.fdpp_attn_set_lut([])
    yield
    F.fdpp_attn_set_lut([])


def _params(B, L, Hq, Hkv, dtype, q_tokens=1):
    return F.make_params(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, dtype=dtype,
                         max_seq_len=L, scale=0.088388, split_len=0, q_tokens=q_tokens)


def _shapes(rng, n):
    for _ in range(n):
        Hkv = int(rng.choice([1, 2, 8]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        Tq = int(rng.choice([1, 1, 2, 4]))
        if G * Tq > 64:
            Tq = 1
        yield (int(rng.integers(1, 2000)), int(rng.integers(1, 300000)), G * Hkv, Hkv,
               int(rng.choice([F.FDPP_BF16, F.FDPP_F32])), Tq)


def _check_against_oracle(rows, shapes):
    for (B, L, Hq, Hkv, dt, Tq) in shapes:
        got = F.fdpp_attn_auto_choice(_params(B, L, Hq, Hkv, dt, Tq))
        want = oracle.dataflow_choice(rows, B, L, Tq * Hq // Hkv, dt == F.FDPP_BF16,
                                      F.FDPP_AUTO_UNITS_PER_SM, F.FDPP_AUTO_MIN_SPLIT)
        assert got == want, ((B, L, Hq, Hkv, dt, Tq), got, want)


def test_without_a_table_the_defaults_apply():
    rng = np.random.default_rng(1)
    _check_against_oracle([], _shapes(rng, 200))


def test_the_measured_table_matches_the_oracle_rule():
    with open(attn_lut.DEFAULT_TABLE) as f:
        rows = [tuple(r) for r in json.load(f)["rows"]]
    assert rows
    F.fdpp_attn_set_lut(rows)
    rng = np.random.default_rng(2)
    _check_against_oracle(rows, _shapes(rng, 500))


def test_random_tables_match_the_oracle_rule():
    rng = np.random.default_rng(3)
    for _ in range(20):
        rows = [(int(rng.integers(1, 3000)), int(rng.integers(1, 400000)), int(rng.integers(1, 65)),
                 int(rng.integers(0, 3)), int(rng.integers(1, 65)), 256 + 64 * int(rng.integers(0, 40)))
                for _ in range(int(rng.integers(1, 12)))]
        F.fdpp_attn_set_lut(rows)
        _check_against_oracle(rows, _shapes(rng, 50))


@pytest.mark.parametrize("row", [
    (0, 10, 10, 0, 4, 256), (10, 0, 10, 0, 4, 256), (10, 10, 0, 0, 4, 256),
    (10, 10, 10, 3, 4, 256), (10, 10, 10, -1, 4, 256), (10, 10, 10, 0, 0, 256),
    (10, 10, 10, 0, 65, 256), (10, 10, 10, 0, 4, 128), (10, 10, 10, 0, 4, 300),
    (10, 10, 10, 0, 4, (1 << 20) + 64)])
def test_bad_rows_are_rejected_and_leave_the_table(row):
    good = [(1 << 30, 1 << 30, 64, 1, 8, 512)]
    F.fdpp_attn_set_lut(good)
    with pytest.raises(F.FdppError):
        F.fdpp_attn_set_lut([row])
    assert F.fdpp_attn_auto_choice(_params(8, 4096, 32, 8, F.FDPP_BF16))[1:] == (8, 512)


def test_the_builder_keeps_the_fastest_per_range():
    res = {}
    rng = np.random.default_rng(4)
    best = {}
    for B in attn_lut.BATCHES:
        for L in attn_lut.SEQ_LENS:
            if B * L > attn_lut.MAX_TOKENS:
                continue
            for R in attn_lut.ROWS:
                t = {(k, u): float(rng.uniform(10, 20)) for k in (1, 2) for u in attn_lut.UNITS}
                res[(B, L, R)] = t
                best[(B, L, R)] = min(t, key=t.get)
    rows = attn_lut.rows_from(res)
    b_tops = list(attn_lut.BATCHES[:-1]) + [attn_lut.OPEN]
    l_tops = list(attn_lut.SEQ_LENS[:-1]) + [attn_lut.OPEN]
    for (mb, ml, mr, k, u, m) in rows:
        B = attn_lut.BATCHES[b_tops.index(mb)]
        L = attn_lut.SEQ_LENS[l_tops.index(ml)]
        R = attn_lut.ROWS[list(attn_lut.ROWS[:-1]).index(mr)] if mr in attn_lut.ROWS[:-1] else attn_lut.ROWS[-1]
        key = (B, L, R)
        while key not in res:                      # too large: the measured batch below
            B = attn_lut.BATCHES[attn_lut.BATCHES.index(B) - 1]
            key = (B, L, R)
        assert (k, u) == best[key]
        assert m == attn_lut.MIN_SPLIT
    # every shape falls in some row: the last ranges are open
    assert rows[-1][0] == attn_lut.OPEN and rows[-1][1] == attn_lut.OPEN
