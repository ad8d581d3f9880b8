"""GPU parity: libfdpp (through its C ABI) against the fp64 oracle on the same seeded inputs.

Small cases the oracle finishes in seconds span several 64-token tiles, splits with ragged tails,
GQA groups of 1, 4 and 8, head_dim 64 and 128, contiguous and paged caches (block sizes 16..128),
and the degenerate cases of the method: empty and one-token sequences, NaN past seq_len, hot keys
that must take the fallback, the forced-online and forced-fast modes, the automatic split length.
Window decisions and the split plan are compared with the oracle's bit-exactly.
"""
import numpy as np
import pytest

import fdpp_harness as H
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

try:
    import split_kv_async_gb300 as F
except ImportError:        # the library must exist where these tests run; fail loudly there
    F = None


def _wl(base, **kw):
    return base.replace(**kw)


SMALL = {
    # (workload, explicit seq_lens)
    "gqa_ragged": (_wl(W.GQA, name="gqa_ragged", batch=3, split_len=512), [1000, 513, 71]),
    "gqa_d64": (_wl(W.GQA, name="gqa_d64", batch=2, head_dim=64, split_len=256), [777, 64]),
    "mha_g1": (_wl(W.GQA, name="mha_g1", batch=2, num_q_heads=8, num_kv_heads=8, split_len=128),
               [300, 129]),
    "g8": (_wl(W.PAGED, name="g8_contig", batch=3, paged=False, seq_len_range=None, seq_len=700,
               split_len=256), [700, 1, 333]),
    "paged_bs16": (_wl(W.PAGED, name="paged_bs16", batch=5, seq_len_range=(17, 1500),
                       split_len=512), None),
    "paged_bs32": (_wl(W.PAGED, name="paged_bs32", batch=4, block_size=32, seq_len_range=(33, 900),
                       split_len=256), None),
    "paged_bs128": (_wl(W.PAGED, name="paged_bs128", batch=3, block_size=128,
                        seq_len_range=(100, 1100), split_len=256), None),
    "tiny": (W.TINY, None),
    # several query tokens per sequence (the last Tq positions, causal): 8 query rows per kv head
    # on the tensor kernel, 16 on the SIMT kernel only; sequences shorter than Tq included
    "tq2_gqa": (_wl(W.GQA, name="tq2_gqa", batch=3, num_q_heads=8, num_kv_heads=2, q_tokens=2,
                    split_len=256), [700, 65, 1]),
    "tq8_mha": (_wl(W.GQA, name="tq8_mha", batch=3, num_q_heads=4, num_kv_heads=4, head_dim=64,
                    q_tokens=8, split_len=64), [300, 9, 5]),
    "tq2_g8_simt": (_wl(W.GQA, name="tq2_g8", batch=2, num_q_heads=16, num_kv_heads=2, q_tokens=2,
                        split_len=128), [400, 130]),
    # more than 8 query rows per kv head: the tensor kernel takes them in groups of 8
    "tq16_g4": (_wl(W.GQA, name="tq16_g4", batch=3, num_q_heads=8, num_kv_heads=2, q_tokens=16,
                    split_len=256), [900, 300, 40]),
    "tq3_g4": (_wl(W.GQA, name="tq3_g4", batch=2, num_q_heads=8, num_kv_heads=2, q_tokens=3,
                   split_len=128), [700, 129]),
    "g16": (_wl(W.GQA, name="g16", batch=2, num_q_heads=32, num_kv_heads=2, split_len=256),
            [1000, 333]),
    "tq8_paged_g2": (_wl(W.PAGED, name="tq8_paged_g2", batch=3, num_q_heads=4, num_kv_heads=2,
                         q_tokens=8, seq_len_range=(40, 1200), split_len=256), None),
    "tq4_paged": (_wl(W.PAGED, name="tq4_paged", batch=4, num_q_heads=4, num_kv_heads=2,
                      q_tokens=4, seq_len_range=(3, 700), split_len=128), None),
    # the tcgen05 build's shapes (bf16, d = 128, 9..64 rows per kv head, padded to 16, 32 or 64):
    # sequences shorter than the chunk (rows that see no key), splits that are no multiple of
    # the 64-token tile (ragged tiles inside a sequence), 20 rows on a paged cache
    "tq16_short": (_wl(W.GQA, name="tq16_short", batch=6, num_q_heads=8, num_kv_heads=2,
                       q_tokens=16, split_len=64), [5, 16, 17, 64, 65, 200]),
    "tq4_g4_s100": (_wl(W.GQA, name="tq4_g4_s100", batch=3, num_q_heads=8, num_kv_heads=2,
                        q_tokens=4, split_len=100), [777, 100, 3]),
    "tq8_g4": (_wl(W.GQA, name="tq8_g4", batch=2, num_q_heads=8, num_kv_heads=2, q_tokens=8,
                   split_len=256), [1000, 257]),
    "tq5_paged_g4": (_wl(W.PAGED, name="tq5_paged_g4", batch=4, num_q_heads=8, num_kv_heads=2,
                         q_tokens=5, seq_len_range=(2, 1300), split_len=256), None),
}

# More than 8 query rows per kv head with bf16 K/V and d = 128: the tcgen05 build by default,
# the mma.sync build (rows in groups of 8) when asked for.
MANY_ROWS = ["tq16_g4", "tq3_g4", "g16", "tq8_paged_g2", "tq16_short", "tq4_g4_s100", "tq8_g4",
             "tq5_paged_g4"]


_cache = {}


def _inputs(name, poison=False):
    key = (name, poison)
    if key not in _cache:
        wl, sl = SMALL[name]
        inp = W.generate(wl, seq_lens=None if sl is None else np.array(sl, np.int32),
                         poison_tail=poison)
        _cache[key] = (inp, H.DeviceInputs(inp))
    return _cache[key]


def _kernels(inp):
    R = inp.wl.group * max(1, inp.wl.q_tokens)
    ks = [F.FDPP_KERNEL_SIMT] if R <= 16 else []
    if inp.wl.dtype == W.BF16 and R <= 64:
        ks.insert(0, F.FDPP_KERNEL_TENSOR)
    return ks


@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity(name):
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    for kernel in _kernels(inp):
        got, diag, flags, ns, _ = H.run(dinp, kernel=kernel)
        H.assert_parity(got, ref, f"{name} kernel {kernel}")
        assert diag["error_bits"] == 0
        assert diag["kernel"] == kernel
        # split plan = the oracle's scheduler, bit for bit
        S = inp.wl.split_len
        o_ns, _, o_units = oracle.plan(inp.seq_lens, inp.wl.num_kv_heads, 1 << 30, S)
        assert diag["split_len"] == S
        np.testing.assert_array_equal(ns, o_ns)
        assert diag["n_units"] == o_units
        # N(0,1) inputs never leave the window
        assert diag["n_flagged_row_splits"] == 0 and (flags & F.FDPP_FLAG_OUT).sum() == 0


@pytest.mark.parametrize("name", MANY_ROWS)
@pytest.mark.parametrize("build", ["tcgen05", "mma_sync"])
def test_many_rows_on_both_tensor_builds(name, build):
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    tc = F.FDPP_TC_MMA_TCGEN05 if build == "tcgen05" else F.FDPP_TC_MMA_SYNC
    got, diag, flags, ns, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=tc)
    H.assert_parity(got, ref, f"{name} {build}")
    assert diag["error_bits"] == 0
    assert diag["kernel"] == F.FDPP_KERNEL_TENSOR and diag["tc_build"] == tc
    o_ns, _, o_units = oracle.plan(inp.seq_lens, inp.wl.num_kv_heads, 1 << 30, inp.wl.split_len)
    np.testing.assert_array_equal(ns, o_ns)
    assert diag["n_units"] == o_units
    assert diag["n_flagged_row_splits"] == 0 and (flags & F.FDPP_FLAG_OUT).sum() == 0


def test_many_rows_default_to_the_tcgen05_build():
    inp, dinp = _inputs("tq16_g4")
    _, diag, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR)
    assert diag["tc_build"] == F.FDPP_TC_MMA_TCGEN05
    # two CTAs per SM asked for: only the mma.sync build runs that geometry
    _, diag, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_ctas_per_sm=2)
    assert diag["tc_build"] == F.FDPP_TC_MMA_SYNC
    # head_dim 64 has no tcgen05 build
    inp64, dinp64 = _inputs("tq8_mha")
    _, diag, _, _, _ = H.run(dinp64, kernel=F.FDPP_KERNEL_TENSOR)
    assert diag["tc_build"] == F.FDPP_TC_MMA_SYNC


@pytest.mark.parametrize("name", ["gqa_ragged", "paged_bs16", "tiny", "tq4_paged", "tq16_short",
                                  "tq5_paged_g4"])
def test_nan_past_seq_len_is_never_read_into_results(name):
    inp, dinp = _inputs(name, poison=True)
    ref = H.oracle_out(inp)
    assert np.isfinite(ref).all()
    for kernel in _kernels(inp):
        got, diag, _, _, _ = H.run(dinp, kernel=kernel)
        H.assert_parity(got, ref, f"{name} poisoned kernel {kernel}")
        assert diag["n_flagged_row_splits"] == 0


def test_empty_and_single_token_sequences():
    wl = _wl(W.GQA, name="edge", batch=4, split_len=64)
    inp = W.generate(wl, seq_lens=np.array([0, 1, 64, 65], np.int32))
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    for kernel in _kernels(inp):
        got, diag, _, ns, _ = H.run(dinp, kernel=kernel)
        g = got.reshape(4, 32, 128)
        assert np.all(g[0] == 0.0)                          # L = 0: zero row
        v0 = W.bf16_bits_to_f32(inp.v[1, 0]).astype(np.float64)      # [Hkv][d]
        np.testing.assert_array_equal(g[1], np.repeat(v0, 4, axis=0))  # L = 1: exactly v0
        H.assert_parity(got, ref, f"edge kernel {kernel}")
        assert list(ns) == [0, 1, 1, 2]


def test_constant_values_give_v0():
    """Rows of A sum to one, so V rows all equal to v0 give v0 (hwan-h-heo.github.io,
    'Optimizing sparse 3D generation inference', s2.2)."""
    inp, _ = _inputs("gqa_ragged")
    v = inp.v.copy()
    v[:] = inp.v[:, :1]                       # every token of sequence b carries v[b, 0]
    inp2 = W.Inputs(**{**inp.__dict__, "v": v})
    dinp = H.DeviceInputs(inp2)
    for kernel in _kernels(inp2):
        got, _, _, _, _ = H.run(dinp, kernel=kernel)
        g = got.reshape(inp.wl.batch, inp.wl.num_q_heads, -1)
        for b in range(inp.wl.batch):
            v0 = W.bf16_bits_to_f32(v[b, 0]).astype(np.float64)
            np.testing.assert_array_equal(g[b], np.repeat(v0, inp.wl.group, axis=0))


def test_paged_equals_contiguous_bit_for_bit():
    inp, dinp = _inputs("paged_bs16")
    wl = inp.wl
    B, bs = wl.batch, wl.block_size
    Lmax = int(inp.seq_lens.max())
    kc = np.zeros((B, Lmax, wl.num_kv_heads, wl.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for t in range(int(inp.seq_lens[b])):
            kc[b, t] = inp.k[inp.block_table[b, t // bs], t % bs]
            vc[b, t] = inp.v[inp.block_table[b, t // bs], t % bs]
    cont = W.Inputs(wl.replace(paged=False), inp.seq_lens, inp.q, kc, vc, None, Lmax, 0, 0, [])
    dcont = H.DeviceInputs(cont)
    for kernel in _kernels(inp):
        gp, _, _, _, _ = H.run(dinp, kernel=kernel)
        gc, _, _, _, _ = H.run(dcont, kernel=kernel)
        np.testing.assert_array_equal(gp, gc)


def test_runs_are_bit_identical():
    inp, dinp = _inputs("paged_bs16")
    for kernel in _kernels(inp):
        a, _, _, _, ws = H.run(dinp, kernel=kernel)
        b, _, _, _, _ = H.run(dinp, ws=ws, kernel=kernel)
        np.testing.assert_array_equal(a, b)


def _stress_inputs(batch=8, seq_len=1024, split_len=256, frac=0.05, seed_offset=0, **kw):
    """Hot-key workload whose scores all sit at least 1e-3 from a window edge (the decision
    replay compares booleans; a score closer than that could round either way in fp32).
    Seeds advance deterministically until the margin holds."""
    for k in range(16):
        wl = W.STRESS.replace(batch=batch, seq_len=seq_len, split_len=split_len,
                              stress_frac=frac, seed=W.STRESS.seed + 101 * (seed_offset + k), **kw)
        inp = W.generate(wl)
        ms = -(-seq_len // split_len)
        flags, margin = H.oracle_flags(inp, split_len, ms)
        if margin.min() > 1e-3:
            return inp, flags
    raise AssertionError("no seed with a 1e-3 decision margin")


@pytest.mark.parametrize("kernel", ["tensor", "simt"])
def test_fallback_decisions_and_results(kernel):
    inp, oflags = _stress_inputs()
    dinp = H.DeviceInputs(inp)
    kid = F.FDPP_KERNEL_TENSOR if kernel == "tensor" else F.FDPP_KERNEL_SIMT
    ref = H.oracle_out(inp)
    got, diag, flags, _, _ = H.run(dinp, kernel=kid)
    # decisions: the OUT/ABOVE/BELOW/NAN bits equal the oracle's exactly
    np.testing.assert_array_equal(flags & 0x0F, oflags)
    hot_rows = (oflags & oracle.FLAG_OUT) != 0
    assert hot_rows.sum() >= len(inp.hot)
    # only flagged row-splits were recomputed, and all of them
    np.testing.assert_array_equal((flags & F.FDPP_FLAG_RECOMPUTED) != 0, hot_rows)
    assert diag["n_flagged_row_splits"] == hot_rows.sum()
    H.assert_parity(got, ref, f"stress {kernel}")


@pytest.mark.parametrize("build", ["tcgen05", "mma_sync"])
def test_fallback_with_many_rows(build):
    """Four query tokens of four heads per kv head: 16 rows, one unit of the tcgen05 build or two
    row groups of the mma.sync build. Hot keys send segments to the fallback lists; the tcgen05
    build streams a recomputed piece twice (the rows' maxima, then the sums in that frame).
    Decisions and results as for one query token."""
    inp, oflags = _stress_inputs(batch=4, seq_len=1024, split_len=256, frac=0.1, num_q_heads=16,
                                 num_kv_heads=4, q_tokens=4)
    dinp = H.DeviceInputs(inp)
    tc = F.FDPP_TC_MMA_TCGEN05 if build == "tcgen05" else F.FDPP_TC_MMA_SYNC
    got, diag, flags, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=tc)
    assert diag["tc_build"] == tc
    np.testing.assert_array_equal(flags & 0x0F, oflags)
    hot_rows = (oflags & oracle.FLAG_OUT) != 0
    assert hot_rows.sum() >= len(inp.hot)
    np.testing.assert_array_equal((flags & F.FDPP_FLAG_RECOMPUTED) != 0, hot_rows)
    assert diag["error_bits"] == 0
    H.assert_parity(got, H.oracle_out(inp), f"stress, many rows, {build}")


@pytest.mark.parametrize("q_tokens,build", [(1, "mma_sync"), (4, "mma_sync"), (4, "tcgen05")])
def test_every_unit_falls_back(q_tokens, build):
    """A hot key in every unit: the mma.sync build finishes every such row-split in place with the
    running max (most warps switch mid-segment, and the merge weighs their frames); the tcgen05
    build streams every tainted piece twice. Decisions, recompute marks and results as for the
    oracle."""
    inp, oflags = _stress_inputs(batch=4, seq_len=1024, split_len=256, frac=1.0, num_q_heads=16,
                                 num_kv_heads=4, q_tokens=q_tokens)
    tc = F.FDPP_TC_MMA_TCGEN05 if build == "tcgen05" else F.FDPP_TC_MMA_SYNC
    diag = _check_fallback(inp, oflags, f"every unit falls back, {q_tokens} tokens, {build}", tc_mma=tc)
    # (a hot key in a sequence's last positions is hidden from the chunk's first query tokens)
    assert diag["n_flagged_units"] >= 0.8 * diag["n_units"]
    if q_tokens > 1:
        assert diag["tc_build"] == tc


def _check_fallback(inp, oflags, what, **kw):
    dinp = H.DeviceInputs(inp)
    got, diag, flags, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, **kw)
    np.testing.assert_array_equal(flags & 0x0F, oflags)
    hot_rows = (oflags & oracle.FLAG_OUT) != 0
    assert hot_rows.sum() >= len(inp.hot)
    np.testing.assert_array_equal((flags & F.FDPP_FLAG_RECOMPUTED) != 0, hot_rows)
    assert diag["error_bits"] == 0
    H.assert_parity(got, H.oracle_out(inp), what)
    return diag


def _random_fallback_case(i):
    """A seeded random hot-key shape for the tensor kernel: 1-12 sequences of 200..3000 keys, 1-4
    kv heads, groups of 1-8, query tokens so that 9..64 rows share a kv head, a split length of
    64..1000, 5-100 % of units with a hot key."""
    rng = np.random.default_rng([0x5EED1500, i])
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    tq = int(rng.integers(-(-9 // g), 64 // g + 1))
    kw = dict(batch=int(rng.integers(1, 13)), seq_len=int(rng.integers(200, 3001)),
              split_len=int(rng.choice([64, 128, 192, 256, 500, 1000])),
              frac=float(rng.choice([0.05, 0.2, 0.5, 1.0])), num_q_heads=hkv * g, num_kv_heads=hkv,
              q_tokens=tq, seed_offset=50 + 17 * i)
    return kw


@pytest.mark.parametrize("i", range(6))
@pytest.mark.parametrize("build", ["tcgen05", "mma_sync"])
def test_fallback_random_shapes_with_many_rows(i, build):
    """Decisions, recompute marks and results of seeded random hot-key shapes on both tensor
    builds: the tcgen05 build's pushed runs and redo pieces over its phantom-tile partition, the
    mma.sync row groups' in-place finish."""
    kw = _random_fallback_case(i)
    inp, oflags = _stress_inputs(**kw)
    tc = F.FDPP_TC_MMA_TCGEN05 if build == "tcgen05" else F.FDPP_TC_MMA_SYNC
    diag = _check_fallback(inp, oflags, f"random fallback case {i} ({build}): {kw}", tc_mma=tc)
    assert diag["tc_build"] == tc


def test_one_split_spread_over_many_parts():
    """The tensor kernel cuts the tiles of all units into equal parts, one per CTA. One split of
    64 tiles becomes 64 one-tile parts: 63 of them leave their share in an extra slot that the
    combine adds in, and the hot key's share is recomputed from its own extra slot. The flag
    byte of the split is the OR over all its parts."""
    inp, oflags = _stress_inputs(batch=1, seq_len=4096, split_len=4096, frac=1.0,
                                 num_q_heads=4, num_kv_heads=1)
    assert inp.hot and inp.hot[0][3] >= 64           # the hot key is not in the first part
    diag = _check_fallback(inp, oflags, "one split over 64 parts")
    assert diag["n_units"] == 1


def test_one_split_over_many_parts_with_many_rows():
    """The same on the tcgen05 build: four query tokens of four heads (16 rows) per kv head, one
    split of 64 tiles cut into one-tile parts, whose run slots hold all 16 rows."""
    inp, oflags = _stress_inputs(batch=1, seq_len=4096, split_len=4096, frac=1.0,
                                 num_q_heads=4, num_kv_heads=1, q_tokens=4)
    diag = _check_fallback(inp, oflags, "one split over 64 parts, 16 rows",
                           tc_mma=F.FDPP_TC_MMA_TCGEN05)
    assert diag["n_units"] == 1 and diag["tc_build"] == F.FDPP_TC_MMA_TCGEN05


# The tcgen05 build cuts its tiles in a stream that counts phantom tiles after every (sequence,
# kv head) unit, so that a part holding a run boundary takes fewer tiles: empty sequences (units
# of phantoms only) at the start, inside and at the end; many more tiles than CTAs (boundaries
# inside parts); and units of equal length whose count divides the parts (no phantoms).
PHANTOM_CASES = {
    "empty_units": (_wl(W.GQA, name="ph_empty", batch=6, num_q_heads=8, num_kv_heads=2, q_tokens=16,
                        split_len=128), [0, 300, 0, 0, 130, 0]),
    "many_units": (_wl(W.GQA, name="ph_many", batch=12, num_q_heads=8, num_kv_heads=2, q_tokens=16,
                       split_len=256),
                   [2900, 150, 1777, 64, 3000, 999, 2048, 65, 1200, 2500, 333, 1800]),
    "many_units_16_rows": (_wl(W.GQA, name="ph_many16", batch=12, num_q_heads=8, num_kv_heads=2,
                               q_tokens=4, split_len=192),
                           [2900, 150, 1777, 64, 3000, 999, 2048, 65, 1200, 2500, 333, 1800]),
    "even_units": (_wl(W.GQA, name="ph_even", batch=1, num_q_heads=32, num_kv_heads=8, q_tokens=16,
                       split_len=512), [2048]),
}


@pytest.mark.parametrize("name", list(PHANTOM_CASES))
def test_tcgen05_partition_with_phantom_tiles(name):
    wl, sl = PHANTOM_CASES[name]
    inp = W.generate(wl, seq_lens=np.array(sl, np.int32))
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    got, diag, flags, ns, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=F.FDPP_TC_MMA_TCGEN05)
    H.assert_parity(got, ref, f"{name} tcgen05")
    assert diag["error_bits"] == 0 and diag["tc_build"] == F.FDPP_TC_MMA_TCGEN05
    o_ns, _, o_units = oracle.plan(inp.seq_lens, wl.num_kv_heads, 1 << 30, wl.split_len)
    np.testing.assert_array_equal(ns, o_ns)
    assert diag["n_units"] == o_units
    # the cut: P parts, and phantoms unless units of equal length fall evenly on the parts
    units = wl.batch * wl.num_kv_heads
    tiles = wl.num_kv_heads * sum(-(-L // 64) for L in sl)     # splits are whole tiles here
    rows = wl.q_tokens * wl.group
    assert diag["tc_parts"] > 0
    even = len(set(sl)) == 1 and diag["tc_parts"] % units == 0
    assert diag["tc_seg_tiles"] == (0 if even else (9 if rows > 32 else 6))
    assert diag["tc_parts"] <= tiles
    g = got.reshape(wl.batch, wl.q_tokens, wl.num_q_heads, wl.head_dim)
    for b, L in enumerate(sl):
        if L == 0:
            assert np.all(g[b] == 0.0)                        # no key: zero rows
    # the mma.sync build cuts the same tiles without phantoms
    got2, diag2, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=F.FDPP_TC_MMA_SYNC)
    H.assert_parity(got2, ref, f"{name} mma.sync")
    assert diag2["tc_build"] == F.FDPP_TC_MMA_SYNC and diag2["tc_seg_tiles"] == 0


# Parts that run on past a sequence's last kv head into the next sequence, many times over: 48
# sequences of 0..3499 keys, 2 kv heads, parts of ~10 tiles. (The look ahead that decides whether a
# part holds another run must leave the walk's sequence cursor where it was.)
SEQ_CROSS_LENS = np.random.default_rng([0x5EED1700, 44]).integers(0, 3500, 48).astype(np.int32)


@pytest.mark.parametrize("tq,split,paged", [(4, 256, False), (16, 512, False), (4, 256, True)])
def test_tcgen05_parts_across_sequences(tq, split, paged):
    kw = dict(name=f"seqx{tq}", batch=48, num_q_heads=8, num_kv_heads=2, head_dim=128, dtype=W.BF16,
              q_tokens=tq, split_len=split, seed=0x5EED1701)
    if paged:
        kw.update(block_size=32, seq_len_range=None)
    wl = _wl(W.PAGED if paged else W.GQA, **kw)
    inp = W.generate(wl, seq_lens=SEQ_CROSS_LENS)
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    got, diag, flags, ns, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=F.FDPP_TC_MMA_TCGEN05)
    assert diag["error_bits"] == 0 and diag["tc_build"] == F.FDPP_TC_MMA_TCGEN05
    assert diag["tc_seg_tiles"] == (9 if tq * wl.group > 32 else 6)
    H.assert_parity(got, ref, f"parts across sequences, Tq {tq}, S {split}, paged {paged}")
    o_ns, _, o_units = oracle.plan(inp.seq_lens, wl.num_kv_heads, 1 << 30, wl.split_len)
    np.testing.assert_array_equal(ns, o_ns)
    assert (flags & F.FDPP_FLAG_OUT).sum() == 0


def _random_tc_case(i):
    """A seeded random shape for the tcgen05 build: 1-4 kv heads, groups of 1-8, query tokens
    so that 9..64 rows share a kv head, 1-6 sequences of 0..1199 keys (one no longer than the
    chunk, often an empty one), split lengths that are and are not tile multiples, contiguous or
    paged caches (blocks of 16, 32 or 64; the split a whole number of blocks), NaN past every
    sequence's end."""
    rng = np.random.default_rng([0x5EED1100, i])
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    tq = int(rng.integers(-(-9 // g), 64 // g + 1))
    b = int(rng.integers(1, 7))
    sl = rng.integers(0, 1200, b)
    sl[int(rng.integers(0, b))] = int(rng.integers(0, tq + 1))
    if b > 2:
        sl[int(rng.integers(0, b))] = 0
    split = int(rng.choice([64, 100, 128, 192, 256, 500, 512]))
    paged = bool(rng.random() < 0.4)
    kw = dict(name=f"rnd{i}", batch=b, num_q_heads=hkv * g, num_kv_heads=hkv, head_dim=128,
              dtype=W.BF16, q_tokens=tq, split_len=split, seed=0x5EED1200 + i)
    if paged:
        bs = int(rng.choice([16, 32, 64]))
        # a paged split is a whole number of blocks (the API's contract), still often no whole tile
        kw.update(block_size=bs, seq_len_range=None, split_len=max(bs, split // bs * bs))
    return _wl(W.PAGED if paged else W.GQA, **kw), sl.astype(np.int32)


@pytest.mark.parametrize("i", range(16))
@pytest.mark.parametrize("build", ["tcgen05", "mma_sync"])
def test_many_rows_random_shapes(i, build):
    wl, sl = _random_tc_case(i)
    inp = W.generate(wl, seq_lens=sl, poison_tail=True)
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    tc = F.FDPP_TC_MMA_TCGEN05 if build == "tcgen05" else F.FDPP_TC_MMA_SYNC
    got, diag, flags, ns, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_mma=tc)
    what = (f"random case {i} ({build}): B {wl.batch}, Hkv {wl.num_kv_heads}, G {wl.group}, "
            f"Tq {wl.q_tokens}, S {wl.split_len}, paged {wl.paged}, L {[int(x) for x in sl]}")
    H.assert_parity(got, ref, what)
    assert diag["error_bits"] == 0 and diag["tc_build"] == tc, what
    o_ns, _, o_units = oracle.plan(inp.seq_lens, wl.num_kv_heads, 1 << 30, wl.split_len)
    np.testing.assert_array_equal(ns, o_ns)
    assert diag["n_units"] == o_units


def _random_decode_case(i):
    """A seeded random decode shape: 1-8 kv heads, groups of 1-16, one or two query tokens (at most
    16 rows per kv head), d = 64 or 128, bf16 or fp32, 1-8 sequences of 0..2999 keys (often an
    empty and a one-key one), splits of whole or partial tiles, contiguous or paged caches, NaN
    past every sequence's end; every kernel that takes the shape runs it."""
    rng = np.random.default_rng([0x5EED1300, i])
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    tq = int(rng.choice([1, 2])) if g <= 8 else 1
    b = int(rng.integers(1, 9))
    sl = rng.integers(0, 3000, b)
    if b > 1:
        sl[int(rng.integers(0, b))] = int(rng.integers(0, 2))
    d = int(rng.choice([64, 128]))
    dt = W.F32 if rng.random() < 0.25 else W.BF16
    split = int(rng.choice([64, 96, 128, 200, 256, 512, 1000]))
    paged = bool(rng.random() < 0.4)
    kw = dict(name=f"drnd{i}", batch=b, num_q_heads=hkv * g, num_kv_heads=hkv, head_dim=d, dtype=dt,
              q_tokens=tq, split_len=split, seed=0x5EED1400 + i)
    if paged:
        bs = int(rng.choice([16, 32, 64, 128]))
        kw.update(block_size=bs, seq_len_range=None, split_len=max(bs, split // bs * bs))
    return _wl(W.PAGED if paged else W.GQA, **kw), sl.astype(np.int32)


@pytest.mark.parametrize("i", range(16))
def test_decode_random_shapes(i):
    wl, sl = _random_decode_case(i)
    inp = W.generate(wl, seq_lens=sl, poison_tail=True)
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    ks = _kernels(inp)
    assert ks
    for kernel in ks:
        got, diag, flags, ns, _ = H.run(dinp, kernel=kernel)
        what = (f"random decode case {i} (kernel {kernel}): B {wl.batch}, Hkv {wl.num_kv_heads}, "
                f"G {wl.group}, Tq {wl.q_tokens}, d {wl.head_dim}, {wl.dtype}, S {wl.split_len}, "
                f"paged {wl.paged}, L {[int(x) for x in sl]}")
        H.assert_parity(got, ref, what)
        assert diag["error_bits"] == 0 and diag["kernel"] == kernel, what
        o_ns, _, o_units = oracle.plan(inp.seq_lens, wl.num_kv_heads, 1 << 30, wl.split_len)
        np.testing.assert_array_equal(ns, o_ns)
        assert diag["n_units"] == o_units


def test_batch_beyond_the_shared_memory_plan():
    """Batches above 1024 sequences are dealt out to the CTAs as whole units (no extra slots);
    results, decisions and the fallback must be the same as for the part-balanced path."""
    inp, oflags = _stress_inputs(batch=1100, seq_len=256, split_len=128, frac=0.01,
                                 num_q_heads=8, num_kv_heads=2, head_dim=64)
    diag = _check_fallback(inp, oflags, "batch 1100")
    assert diag["n_units"] == 1100 * 2 * 2


def test_batch_beyond_the_shared_memory_plan_with_row_groups():
    """The whole-unit path with row groups: five query tokens of four heads per kv head are 20
    rows, three groups of 8, 8 and 4. Units are dealt out per (sequence, row group, split); the
    reported unit count stays per kv head."""
    inp, oflags = _stress_inputs(batch=1100, seq_len=256, split_len=128, frac=0.01,
                                 num_q_heads=8, num_kv_heads=2, head_dim=64, q_tokens=5)
    diag = _check_fallback(inp, oflags, "batch 1100, row groups")
    assert diag["n_units"] == 1100 * 2 * 2


def test_batch_beyond_the_shared_memory_plan_with_many_rows():
    """The whole-unit path of the tcgen05 build: 20 rows per kv head (padded to 32), d = 128,
    units dealt out per (sequence, kv head, split), fallback pieces in their split slots."""
    inp, oflags = _stress_inputs(batch=1100, seq_len=256, split_len=128, frac=0.01,
                                 num_q_heads=8, num_kv_heads=2, q_tokens=5)
    diag = _check_fallback(inp, oflags, "batch 1100, 20 rows", tc_mma=F.FDPP_TC_MMA_TCGEN05)
    assert diag["n_units"] == 1100 * 2 * 2 and diag["tc_build"] == F.FDPP_TC_MMA_TCGEN05


def test_many_rows_share_combine_blocks():
    """735 softmax rows: the combine gives a row fewer than 8 warps when the rows would not fit
    on the GPU at once, and packs several rows into one block (the last block has a row to
    spare). Every row must still be right."""
    wl = _wl(W.GQA, name="many_rows", batch=245, num_q_heads=3, num_kv_heads=3, head_dim=64,
             seq_len=300, split_len=64)
    rng = np.random.default_rng(7)
    inp = W.generate(wl, seq_lens=rng.integers(1, 301, size=245).astype(np.int32))
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    for kernel in _kernels(inp):
        got, diag, _, _, _ = H.run(dinp, kernel=kernel)
        assert diag["error_bits"] == 0
        H.assert_parity(got, ref, f"many rows kernel {kernel}")


@pytest.mark.parametrize("kernel", ["tensor", "simt"])
def test_fallback_state_resets_between_calls(kernel):
    """The device-wide fallback list and its counters live in the workspace and must be back at
    zero after every call, so repeated calls on one workspace agree."""
    inp, oflags = _stress_inputs(seed_offset=3)
    dinp = H.DeviceInputs(inp)
    kid = F.FDPP_KERNEL_TENSOR if kernel == "tensor" else F.FDPP_KERNEL_SIMT
    ref = H.oracle_out(inp)
    first, _, f1, _, ws = H.run(dinp, kernel=kid)
    H.assert_parity(first, ref, "call 1")
    for call in range(2, 6):
        got, diag, fl, _, _ = H.run(dinp, ws=ws, kernel=kid)
        np.testing.assert_array_equal(got, first)
        np.testing.assert_array_equal(fl, f1)
        assert diag["error_bits"] == 0


@pytest.mark.parametrize("kernel", ["tensor", "simt"])
def test_force_fast_is_wrong_exactly_where_flagged(kernel):
    """Negative control: without the fallback, the rows with a hot key overflow (inf/NaN or far
    off) and every other row still matches. This shows the recompute is what keeps them right."""
    inp, oflags = _stress_inputs()
    dinp = H.DeviceInputs(inp)
    kid = F.FDPP_KERNEL_TENSOR if kernel == "tensor" else F.FDPP_KERNEL_SIMT
    ref = H.oracle_out(inp)
    got, diag, flags, _, _ = H.run(dinp, kernel=kid, mode=F.FDPP_MODE_FORCE_FAST)
    above = ((oflags & oracle.FLAG_ABOVE) != 0).any(axis=2).reshape(-1)
    bound = np.maximum(H.ABS_TOL, H.BF16_RESOLUTION * np.abs(ref))
    bad = ~np.isfinite(got).all(axis=1) | (np.abs(got - ref) > bound).any(axis=1)
    # every row whose split crossed the overflow side goes wrong, and no other row does
    hot = np.zeros_like(above)
    for (b, g, j, t) in inp.hot:
        hot[b * inp.wl.num_q_heads + g * inp.wl.group] = True
    assert bad[hot].all()
    assert not bad[~above].any()
    assert (flags & F.FDPP_FLAG_RECOMPUTED).sum() == 0


@pytest.mark.parametrize("name", ["gqa_ragged", "paged_bs16", "tiny", "tq16_short", "tq5_paged_g4"])
def test_force_online_matches(name):
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    rows = inp.wl.group * max(1, inp.wl.q_tokens)
    for kernel in _kernels(inp):
        got, diag, flags, _, _ = H.run(dinp, kernel=kernel, mode=F.FDPP_MODE_FORCE_ONLINE)
        H.assert_parity(got, ref, f"{name} online kernel {kernel}")
        assert diag["n_recomputed_row_splits"] == diag["n_units"] * rows


@pytest.mark.parametrize("name", ["gqa_ragged", "paged_bs16"])
def test_auto_split_len_matches_replay(name):
    import torch
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for kernel in _kernels(inp):
        got, diag, _, ns, _ = H.run(dinp, kernel=kernel, split_len=0)
        p = H.params_for(inp, split_len=0)
        gran = max(F.FDPP_AUTO_GRANULE, inp.wl.block_size if inp.wl.paged else 0)
        S = oracle.split_len(inp.seq_lens, inp.wl.num_kv_heads, p.max_seq_len, 0, sms,
                             F.FDPP_AUTO_UNITS_PER_SM, gran, F.FDPP_AUTO_MIN_SPLIT)
        assert diag["split_len"] == S
        o_ns, _, o_units = oracle.plan(inp.seq_lens, inp.wl.num_kv_heads, p.max_seq_len, S)
        np.testing.assert_array_equal(ns, o_ns)
        assert diag["n_units"] == o_units
        H.assert_parity(got, ref, f"{name} auto split kernel {kernel}")


@pytest.mark.parametrize("name", ["gqa_ragged", "paged_bs16", "tiny"])
def test_dataflow_table_sets_kernel_and_split_as_replayed(name):
    """split_len = 0 and kernel AUTO with the heuristic dataflow table installed: the kernel,
    units per SM and least split the table gives for the shape (replayed by the oracle's table
    rule) set the split length, which the device's plan must equal bit for bit, and the result
    still matches the oracle. Three tables: the one measured on GB300, and two that force each
    kernel with other split targets."""
    import json
    import torch
    from split_kv_async_gb300 import attn_lut
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with open(attn_lut.DEFAULT_TABLE) as f:
        measured = [tuple(r) for r in json.load(f)["rows"]]
    open_ = 1 << 30
    tables = [measured, [(open_, open_, 64, F.FDPP_KERNEL_SIMT, 16, 320)],
              [(open_, open_, 64, F.FDPP_KERNEL_TENSOR, 1, 512)]]
    try:
        for rows in tables:
            F.fdpp_attn_set_lut(rows)
            p = H.params_for(inp, split_len=0)
            R = inp.wl.group * max(1, inp.wl.q_tokens)
            kern, units, min_split = oracle.dataflow_choice(
                rows, p.batch, p.max_seq_len, R, inp.wl.dtype == W.BF16,
                F.FDPP_AUTO_UNITS_PER_SM, F.FDPP_AUTO_MIN_SPLIT)
            got, diag, _, ns, _ = H.run(dinp, split_len=0)
            assert diag["kernel"] == kern
            gran = max(F.FDPP_AUTO_GRANULE, inp.wl.block_size if inp.wl.paged else 0)
            S = oracle.split_len(inp.seq_lens, inp.wl.num_kv_heads, p.max_seq_len, 0, sms,
                                 units, gran, min_split)
            assert diag["split_len"] == S
            o_ns, _, o_units = oracle.plan(inp.seq_lens, inp.wl.num_kv_heads, p.max_seq_len, S)
            np.testing.assert_array_equal(ns, o_ns)
            assert diag["n_units"] == o_units
            H.assert_parity(got, ref, f"{name} table {rows[:1]}")
    finally:
        F.fdpp_attn_set_lut([])


@pytest.mark.parametrize("name,stages,ctas", [("paged_bs16", 2, 1), ("paged_bs16", 3, 2),
                                               ("paged_bs16", 6, 1), ("gqa_ragged", 2, 2),
                                               ("gqa_ragged", 6, 1), ("gqa_d64", 12, 1),
                                               ("gqa_d64", 6, 2), ("mha_g1", 3, 2),
                                               ("paged_bs128", 4, 1), ("paged_bs32", 3, 2)])
def test_pipeline_geometries(name, stages, ctas):
    inp, dinp = _inputs(name)
    ref = H.oracle_out(inp)
    got, diag, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_stages=stages,
                               tc_ctas_per_sm=ctas)
    H.assert_parity(got, ref, f"{name} stages {stages} ctas {ctas}")
    assert diag["error_bits"] == 0


@pytest.mark.parametrize("name", ["paged_bs16", "gqa_ragged", "paged_bs128"])
@pytest.mark.parametrize("prefetch", [-1, 1, 12])
def test_l2_prefetch_distances(name, prefetch):
    """The L2 prefetch ahead of the TMA ring moves no data the kernel reads: any distance (or
    none) gives bit-identical results."""
    inp, dinp = _inputs(name)
    base, _, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR)
    got, diag, _, _, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_prefetch=prefetch)
    np.testing.assert_array_equal(got, base)
    assert diag["error_bits"] == 0


def test_geometry_that_does_not_fit_is_rejected():
    inp, dinp = _inputs("paged_bs16")              # 4 stages of 32 KB do not fit twice per SM
    with pytest.raises(F.FdppError) as e:
        H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR, tc_stages=4, tc_ctas_per_sm=2)
    assert e.value.status == F.FDPP_ERR_UNSUPPORTED


def test_out_of_range_seq_len_sets_error_bit():
    inp, dinp = _inputs("gqa_ragged")
    import torch
    bad = dinp.seq_lens.clone()
    bad[0] = inp.max_seq_len + 5
    saved = dinp.seq_lens
    dinp.seq_lens = bad
    try:
        _, diag, _, ns, _ = H.run(dinp, kernel=F.FDPP_KERNEL_TENSOR)
    finally:
        dinp.seq_lens = saved
    assert diag["error_bits"] & F.FDPP_ERRBIT_SEQ_LEN
    assert ns[0] == -(-inp.max_seq_len // inp.wl.split_len)      # clamped to the capacity
    torch.cuda.synchronize()


def test_bad_block_table_entry_sets_error_bit():
    inp, dinp = _inputs("paged_bs16")
    saved = dinp.block_table
    bt = saved.clone()
    bt[0, 0] = inp.num_kv_blocks + 7          # outside the pool: never read, reported
    dinp.block_table = bt
    try:
        for kernel in _kernels(inp):
            _, diag, _, _, _ = H.run(dinp, kernel=kernel)
            assert diag["error_bits"] & F.FDPP_ERRBIT_BLOCK_TABLE
    finally:
        dinp.block_table = saved
