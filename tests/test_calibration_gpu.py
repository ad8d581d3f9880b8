"""GPU parity of per-head phi and of choosing phi in advance.

opt.ai.kr "FlashDecoding++ async softmax -- theory", section 3: phi is set by observing the score
distribution beforehand, and a split whose scores leave the window falls back. Workloads here
give every query head its own score level (workloads.score_shift), so one scalar phi sends most
splits to the fallback while per-head values chosen from sample scores send none.

Checked against the fp64 oracle: score ranges (fp32 sums vs fp64), the per-head pick (counts
exact, values close), window decisions with per-head phi (bit-exact wherever the decision does
not change when the window moves by 1e-3, which must be nearly everywhere), and outputs (parity
tolerance), on both split kernels.
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


def _shifted(paged=False, seed_offset=0):
    """Per-head score levels in [0, 30] (a few hundred tokens per row)."""
    if paged:
        wl = W.PAGED.replace(name="shift_paged", batch=3, seq_len_range=(200, 900), split_len=256,
                             score_shift=30.0, seed=W.PAGED.seed + 17 * seed_offset)
    else:
        wl = W.GQA.replace(name="shift_gqa", batch=4, seq_len=1024, split_len=256,
                           score_shift=30.0, seed=W.GQA.seed + 17 * seed_offset)
    return W.generate(wl)


def _assert_decisions(flags, oflags, robust, what):
    """OUT/ABOVE/BELOW/NAN bits equal the oracle's wherever the decision is robust (almost
    everywhere), and the OUT bit equals it everywhere robust."""
    assert robust.mean() > 0.97, f"{what}: only {robust.mean():.3f} of decisions are robust"
    np.testing.assert_array_equal((flags & 0x0F)[robust], (oflags & 0x0F)[robust], err_msg=what)


def _kernels(inp):
    return [F.FDPP_KERNEL_TENSOR, F.FDPP_KERNEL_SIMT]


@pytest.mark.parametrize("paged", [False, True])
def test_score_ranges_match_oracle(paged):
    inp = _shifted(paged)
    dinp = H.DeviceInputs(inp)
    p = H.params_for(inp)
    ws = F.alloc_workspace(p, dinp.dev)
    smin, smax, ns = F.fdpp_score_ranges(dinp.q, dinp.k, dinp.block_table, dinp.seq_lens, p, ws)
    ms = smin.shape[2]
    omin, omax = oracle.score_ranges(H.oracle_problem(inp), inp.q, inp.k, inp.seq_lens,
                                     inp.wl.split_len, ms, block_table=inp.block_table)
    np.testing.assert_array_equal(ns, -(-inp.seq_lens // inp.wl.split_len))
    np.testing.assert_array_equal(np.isnan(smin), np.isnan(omin))
    ok = ~np.isnan(omin)
    np.testing.assert_allclose(smin[ok], omin[ok], rtol=0, atol=1e-3)
    np.testing.assert_allclose(smax[ok], omax[ok], rtol=0, atol=1e-3)


@pytest.mark.parametrize("paged", [False, True])
def test_calibrated_phi_removes_the_fallbacks(paged):
    """Scalar phi = 0: most row-splits fall back (decisions equal the oracle's bit for bit).
    phi picked per head from the GPU's score ranges: the same count of kept splits as the
    oracle's pick, no fallback, decisions equal the oracle's replay with those values, outputs
    equal the exact softmax on both kernels."""
    import torch
    inp = _shifted(paged)
    dinp = H.DeviceInputs(inp)
    ref = H.oracle_out(inp)
    wl = inp.wl
    ms = -(-inp.max_seq_len // wl.split_len)
    oflags0, robust0 = H.oracle_flags_robust(inp, wl.split_len, ms)
    for kernel in _kernels(inp):
        got, diag, flags, _, _ = H.run(dinp, kernel=kernel)
        _assert_decisions(flags, oflags0, robust0, f"scalar phi kernel {kernel}")
        assert diag["n_flagged_row_splits"] > flags[..., 0].size // 2
        H.assert_parity(got, ref, f"scalar phi kernel {kernel}")

    p = H.params_for(inp)
    ws = F.alloc_workspace(p, dinp.dev)
    smin, smax, ns = F.fdpp_score_ranges(dinp.q, dinp.k, dinp.block_table, dinp.seq_lens, p, ws)
    phi, kept = F.fdpp_pick_phi(smin, smax, ns, wl.lo, wl.hi, fallback=wl.phi)
    omin, omax = oracle.score_ranges(H.oracle_problem(inp), inp.q, inp.k, inp.seq_lens,
                                     wl.split_len, smin.shape[2], block_table=inp.block_table)
    ophi, okept = oracle.pick_phi(omin, omax, ns, wl.lo, wl.hi, fallback=wl.phi)
    np.testing.assert_array_equal(kept, okept)
    np.testing.assert_allclose(phi, ophi, rtol=0, atol=1e-3)

    oflags, margin = H.oracle_flags(inp, wl.split_len, smin.shape[2], phi_heads=phi)
    assert margin.min() > 1e-3
    assert not (oflags & oracle.FLAG_OUT).any()
    dphi = torch.from_numpy(phi).to(dinp.dev)
    for kernel in _kernels(inp):
        got, diag, flags, _, _ = H.run(dinp, kernel=kernel, phi_heads=dphi)
        np.testing.assert_array_equal(flags & 0x0F, oflags)
        assert diag["n_flagged_row_splits"] == 0 and diag["error_bits"] == 0
        H.assert_parity(got, ref, f"calibrated phi kernel {kernel}")


def test_mixed_per_head_phi_matches_oracle():
    """Arbitrary per-head values, some of which leave splits outside the window and some not:
    per-head decisions, recomputed rows and outputs all follow the oracle."""
    import torch
    inp = _shifted(False, seed_offset=5)
    dinp = H.DeviceInputs(inp)
    wl = inp.wl
    ms = -(-inp.max_seq_len // wl.split_len)
    phi = np.random.default_rng(3).uniform(-5.0, 35.0, size=wl.num_q_heads).astype(np.float32)
    oflags, robust = H.oracle_flags_robust(inp, wl.split_len, ms, phi_heads=phi)
    out_rows = (oflags & oracle.FLAG_OUT) != 0
    assert out_rows.any() and not out_rows.all()
    ref = H.oracle_out(inp)
    dphi = torch.from_numpy(phi).to(dinp.dev)
    for kernel in _kernels(inp):
        got, diag, flags, _, _ = H.run(dinp, kernel=kernel, phi_heads=dphi)
        _assert_decisions(flags, oflags, robust, f"mixed phi kernel {kernel}")
        # the flagged row-splits, and only they, were recomputed
        np.testing.assert_array_equal((flags & F.FDPP_FLAG_RECOMPUTED) != 0,
                                      (flags & F.FDPP_FLAG_OUT) != 0)
        H.assert_parity(got, ref, f"mixed phi kernel {kernel}")
