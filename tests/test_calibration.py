"""Choosing phi in advance, on the host: the library's fdpp_pick_phi against the oracle's pick on
the same score ranges, and the argument checks of the calibration entry points. No GPU.

opt.ai.kr "FlashDecoding++ async softmax -- theory", section 3: phi is set by observing the score
distribution beforehand. The reading both sides follow: phi_h keeps the most sample row-splits
of head h inside the window; among all values that do, the middle of the widest run."""
import ctypes

import numpy as np
import pytest

import oracle
import split_kv_async_gb300 as F
from fdpp_harness import no_fake_pointer_calls_on_a_gpu


def _random_ranges(seed, B=5, Hq=6, ms=7):
    rng = np.random.default_rng(seed)
    mid = rng.normal(0.0, 15.0, size=(B, Hq, ms))
    half = rng.uniform(0.0, 25.0, size=(B, Hq, ms))
    smin = (mid - half).astype(np.float32)
    smax = (mid + half).astype(np.float32)
    ns = rng.integers(0, ms + 1, size=B).astype(np.int32)
    for b in range(B):
        smin[b, :, ns[b]:] = np.nan
        smax[b, :, ns[b]:] = np.nan
    return smin, smax, ns


@pytest.mark.parametrize("seed", range(8))
def test_library_pick_matches_oracle(seed):
    smin, smax, ns = _random_ranges(seed)
    lo, hi = -30.0, 10.0
    phi_l, kept_l = F.fdpp_pick_phi(smin, smax, ns, lo, hi, fallback=1.25)
    phi_o, kept_o = oracle.pick_phi(smin.astype(np.float64), smax.astype(np.float64), ns, lo, hi,
                                    fallback=1.25)
    np.testing.assert_array_equal(kept_l, kept_o)
    np.testing.assert_allclose(phi_l, phi_o, rtol=1e-6, atol=1e-6)


def test_pick_with_every_split_unkeepable_gives_fallback():
    smin = np.zeros((2, 3, 4), np.float32)
    smax = np.full((2, 3, 4), 100.0, np.float32)      # range 100 > hi - lo = 40
    phi, kept = F.fdpp_pick_phi(smin, smax, np.array([4, 2], np.int32), -30.0, 10.0, fallback=-2.0)
    np.testing.assert_array_equal(phi, -2.0)
    np.testing.assert_array_equal(kept, 0)


def test_pick_ignores_splits_past_nsplit():
    smin = np.full((1, 1, 3), 0.0, np.float32)
    smax = np.full((1, 1, 3), 1.0, np.float32)
    smin[0, 0, 2], smax[0, 0, 2] = 500.0, 501.0      # only j < nsplit counts
    phi, kept = F.fdpp_pick_phi(smin, smax, np.array([2], np.int32), -30.0, 10.0)
    assert kept[0] == 2
    assert -9.0 <= phi[0] <= 30.0


def test_calibration_argument_errors():
    vp = ctypes.c_void_p
    buf = np.zeros(8, np.float32)
    ns = np.zeros(1, np.int32)
    st = F.lib.fdpp_pick_phi(None, buf.ctypes.data, ns.ctypes.data, 1, 1, 1, -30.0, 10.0, 0.0,
                             buf.ctypes.data, None)
    assert st == F.FDPP_ERR_INVALID_ARG
    st = F.lib.fdpp_pick_phi(buf.ctypes.data, buf.ctypes.data, ns.ctypes.data, 1, 1, 1, 10.0,
                             -30.0, 0.0, buf.ctypes.data, None)
    assert st == F.FDPP_ERR_INVALID_ARG                 # lo > hi
    p = F.make_params(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, dtype=F.FDPP_F32,
                      max_seq_len=256, scale=0.125, split_len=64)
    no_fake_pointer_calls_on_a_gpu()
    fake = vp(1 << 20)                                  # never dereferenced: rejected first
    st = F.lib.fdpp_score_ranges(None, fake, None, fake, ctypes.byref(p), fake, 1 << 30,
                                 buf.ctypes.data, buf.ctypes.data, None, None)
    assert st == F.FDPP_ERR_INVALID_ARG
    p_bad = F.make_params(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, dtype=F.FDPP_F32,
                          max_seq_len=256, scale=0.125, split_len=64, phi_heads=(1 << 20) + 2)
    size = ctypes.c_size_t(0)
    assert F.lib.fdpp_workspace_size(ctypes.byref(p_bad), ctypes.byref(size)) == F.FDPP_ERR_INVALID_ARG
