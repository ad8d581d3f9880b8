"""A CPU model of the tensor kernel's partition of its own work and of the combine's lookup of run
slots, checked for the properties the two must share.

The tensor kernel cuts the 64-token tiles of all (sequence, kv head) units into P parts, one per CTA,
in a stream that counts K phantom tiles after each unit (split_tc_common.cuh, `Producer::run` and
`run_parts`); each CTA walks its part as runs, one per unit it touches, and leaves one partial per run
in run slot c + u. The combine (combine.cu) finds a head's runs from the cut alone: the parts whose
range meets the head's tiles, and for a part that starts inside a split, that split's edge flags.
This model restates both in plain Python with C integer semantics, so that the properties hold for the
algorithm whatever the batch:
  * every real tile is in exactly one run, and every run starts at a tile of its unit (k >= 0);
  * the combine's parts for a head are exactly the parts that wrote a run for it, with the same start
    offsets (the edge-flag decisions follow from those offsets).
The GPU parity tests check the kernels themselves against the oracle.
"""
import numpy as np
import pytest

TILE = 64


def cdiv(a, b):
    """C's truncating integer division."""
    q = abs(a) // abs(b)
    return q if (a >= 0) == (b >= 0) else -q


def cut(seq_lens, hkv, split, k_req, p_cap):
    """The cut: tiles per sequence and kv head, P parts, K phantoms (none where units of equal length
    fall evenly on the parts), the stream's length TV."""
    ts = -(-split // TILE)
    tplan = [0]
    for L in (int(x) for x in seq_lens):
        nb = -(-L // split)
        nt = 0 if nb == 0 else (nb - 1) * ts + -(-min(L - (nb - 1) * split, split) // TILE)
        tplan.append(tplan[-1] + nt)
    T = tplan[-1] * hkv
    U = len(seq_lens) * hkv
    P = min(p_cap, T)
    even = all(tplan[b + 1] - tplan[b] == tplan[1] - tplan[0] for b in range(len(seq_lens)))
    K = 0 if (even and P > 0 and P % U == 0) else k_req
    return tplan, P, K, T + K * U


def walk(seq_lens, hkv, split, k_req, p_cap):
    """Each part's runs as the producer walks them: {(b, kvh): [(part, first tile, end tile)]}."""
    tplan, P, K, TV = cut(seq_lens, hkv, split, k_req, p_cap)
    runs = {}
    for c in range(P):
        q, r = divmod(TV, P)
        tb, te = c * q + (c * r) // P, (c + 1) * q + ((c + 1) * r) // P
        cursor = [0]                         # the sequence the walk is in (moves forward only)

        def seg_at(v):
            while True:
                if v >= te:
                    return None, v
                cb = cursor[0]
                while hkv * (tplan[cb + 1] + K * (cb + 1)) <= v:
                    cb += 1
                cursor[0] = cb
                ntb = tplan[cb + 1] - tplan[cb]
                rr = v - hkv * (tplan[cb] + K * cb)
                kvh = cdiv(rr, ntb + K)
                k = rr - kvh * (ntb + K)
                if k >= ntb:                 # a phantom: the next unit's first tile
                    v += ntb + K - k
                    continue
                return (cb, kvh, k, min(ntb, k + (te - v))), v

        cur, t = seg_at(tb)
        while cur is not None:
            b, kvh, k, kend = cur
            runs.setdefault((b, kvh), []).append((c, k, kend))
            tn = t + (kend - k)
            last = tn >= te
            if not last and K > 0:
                if te <= tn + K:
                    last = True
                elif kvh + 1 >= hkv:         # the look ahead keeps the cursor where it was
                    keep = cursor[0]
                    last = seg_at(tn)[0] is None
                    cursor[0] = keep
            if last:
                break
            cur, t = seg_at(tn)
    return runs, tplan, P, K, TV


def combine_lookup(tplan, hkv, P, K, TV):
    """The combine's parts per head: {(b, kvh): [(part, offset of its first tile in the head)]}."""
    q, r = divmod(TV, P)
    out = {}
    for b in range(len(tplan) - 1):
        nt = tplan[b + 1] - tplan[b]
        if nt == 0:
            continue
        for kvh in range(hkv):
            u = b * hkv + kvh
            V = hkv * tplan[b] + kvh * nt + K * u
            c_first = ((V + 1) * P - 1) // TV
            n_r = ((V + nt) * P - 1) // TV - c_first + 1
            out[(b, kvh)] = [(c, max(c * q + (c * r) // P - V, 0)) for c in range(c_first, c_first + n_r)]
    return out


def _random_batch(rng):
    b = int(rng.integers(1, 70))
    sl = rng.integers(0, 5000, b)
    sl[rng.random(b) < 0.2] = 0
    return (sl, int(rng.choice([1, 2, 4, 8])), int(rng.choice([64, 128, 192, 256, 512, 1024])),
            int(rng.choice([0, 1, 6, 9])), int(rng.choice([17, 152, 256, 512])))


@pytest.mark.parametrize("seed", range(4))
def test_every_tile_in_exactly_one_run(seed):
    rng = np.random.default_rng([0x5EED1800, seed])
    for _ in range(50):
        sl, hkv, split, k, p_cap = _random_batch(rng)
        runs, tplan, P, K, TV = walk(sl, hkv, split, k, p_cap)
        cover = {}
        for (b, kvh), lst in runs.items():
            assert 0 <= kvh < hkv
            for c, k0, k1 in lst:
                assert 0 <= k0 < k1 <= tplan[b + 1] - tplan[b]
                for x in range(k0, k1):
                    cover[(b, kvh, x)] = cover.get((b, kvh, x), 0) + 1
        want = {(b, kvh, x) for b in range(len(sl)) for kvh in range(hkv)
                for x in range(tplan[b + 1] - tplan[b])}
        assert set(cover) == want and all(n == 1 for n in cover.values())


@pytest.mark.parametrize("seed", range(4))
def test_combine_finds_the_runs_the_parts_wrote(seed):
    rng = np.random.default_rng([0x5EED1900, seed])
    for _ in range(50):
        sl, hkv, split, k, p_cap = _random_batch(rng)
        runs, tplan, P, K, TV = walk(sl, hkv, split, k, p_cap)
        if P == 0:
            continue
        look = combine_lookup(tplan, hkv, P, K, TV)
        assert set(look) == set(runs)
        for head, lst in runs.items():
            assert sorted((c, k0) for c, k0, _ in lst) == sorted(look[head])


def test_phantoms_only_where_the_cut_misses_unit_boundaries():
    """Units of equal length whose count divides P need no phantoms (long_context: 8 units on 152
    parts); otherwise K is counted (prefill_chunk_tq16: 64 units on 152 parts)."""
    assert cut([131072], 8, 1024, 9, 152)[2] == 0
    assert cut([4096] * 8, 8, 512, 9, 152)[2] == 9
    assert cut([4096, 4000] * 4, 2, 512, 6, 16)[2] == 6       # 64 and 63 tiles: unequal units
    assert cut([4096, 4095] * 4, 2, 512, 6, 16)[2] == 0       # 64 tiles each, 16 units on 16 parts
