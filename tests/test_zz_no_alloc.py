"""fdpp_decode_attn_noalloc: the decode step for callers that cannot allocate device memory (for
example a plugin inside a runtime that owns every device allocation, or a serving loop whose
memory is fixed at start-up). Its scratch is the library's own static device array, so it takes
no workspace. It runs the same kernels as fdpp_decode_attn on the same inputs, so its output must
equal that entry point's bit for bit, call after call, and agree with the oracle; what it found
on the device is read with fdpp_read_diag_noalloc.

The static array keeps the last call's contents, whatever its shape; the alternation test runs
calls of different layouts (hot-key fallback lists, a ragged batch, the fp32 SIMT kernel, a paged
cache) one after another through it.

This file is named to be collected last: if it fails, a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import fdpp_harness as H
import oracle
import workloads as W

try:
    import split_kv_async_gb300 as F
except ImportError:
    F = None


def _run_noalloc(dinp, p):
    import torch
    out = torch.full_like(dinp.q, float("nan"))      # rows the library fails to write show up
    F.fdpp_decode_attn_noalloc(dinp.q, dinp.k, dinp.v, dinp.block_table, dinp.seq_lens, p, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(-1, dinp.inp.wl.head_dim).astype(np.float64)
    diag, flags, ns = F.fdpp_read_diag_noalloc(p, want_flags=True, want_nsplit=True)
    return got, diag, flags, ns


def _case(name):
    if name == "gqa_ragged":
        wl = W.GQA.replace(name="noalloc_gqa", batch=4, split_len=256)
        return W.generate(wl, seq_lens=np.array([1000, 513, 71, 300], np.int32)), {}
    if name == "hot_keys":
        # hot keys: the fallback lists inside the static array are used and must be left clean
        # for the next call
        wl = W.STRESS.replace(name="noalloc_hot", batch=4, seq_len=768, split_len=256,
                              stress_frac=0.1)
        return W.generate(wl), {}
    if name == "tiny_simt":
        wl = W.TINY.replace(name="noalloc_tiny", batch=2, split_len=64)
        return W.generate(wl, seq_lens=np.array([256, 97], np.int32)), {"kernel": F.FDPP_KERNEL_SIMT}
    if name == "paged":
        wl = W.PAGED.replace(name="noalloc_paged", batch=5, seq_len_range=(17, 1500), split_len=512)
        return W.generate(wl), {}
    raise KeyError(name)


def _check_against_workspace_path(name, inp, dinp, kw, calls):
    p = H.params_for(inp, **kw)
    assert F.fdpp_workspace_size(p) <= F.FDPP_NOALLOC_WORKSPACE_BYTES
    ref, diag, flags, ns, _ = H.run(dinp, **kw)          # the workspace entry point
    assert diag["error_bits"] == 0
    want = H.oracle_out(inp)
    for call in range(calls):
        got, d2, f2, n2 = _run_noalloc(dinp, p)
        what = f"{name} no-alloc call {call + 1}"
        # the same kernels on the same inputs: identical bits
        np.testing.assert_array_equal(got, ref, err_msg=what)
        H.assert_parity(got, want, what)
        assert d2["error_bits"] == 0, what
        assert d2["split_len"] == diag["split_len"] and d2["n_units"] == diag["n_units"], what
        np.testing.assert_array_equal(n2, ns, err_msg=what)
        # flag bytes of the splits each sequence has (slots past them keep older calls' bytes)
        Tq = max(1, inp.wl.q_tokens)
        ms = flags.shape[-1]
        valid = (np.arange(ms)[None, :] < np.repeat(ns, Tq)[:, None])[:, None, :]
        valid = np.broadcast_to(valid, flags.shape)
        np.testing.assert_array_equal(f2[valid], flags[valid], err_msg=what)
        f2 = np.where(valid, f2, 0)
        # every flagged row-split was recomputed, and only those
        assert d2["n_recomputed_row_splits"] == d2["n_flagged_row_splits"], what
        if inp.wl.stress_frac > 0:
            assert d2["n_flagged_row_splits"] >= len(inp.hot) > 0, what
            np.testing.assert_array_equal((f2 & F.FDPP_FLAG_RECOMPUTED) != 0,
                                          (f2 & oracle.FLAG_OUT) != 0, err_msg=what)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["gqa_ragged", "hot_keys"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    inp, kw = _case(name)
    _check_against_workspace_path(name, inp, H.DeviceInputs(inp), kw, calls=2)


@pytest.mark.gpu
def test_noalloc_state_left_by_other_shapes_is_harmless():
    """Calls of different layouts in a row through the one static array: the fallback lists of a
    hot-key call, then a ragged batch, the fp32 SIMT kernel, a paged cache, and the hot keys
    again; each agrees with the workspace entry point bit for bit and with the oracle."""
    cases = {}
    for name in ["hot_keys", "gqa_ragged", "tiny_simt", "paged", "hot_keys", "gqa_ragged"]:
        if name not in cases:
            inp, kw = _case(name)
            cases[name] = (inp, H.DeviceInputs(inp), kw)
        inp, dinp, kw = cases[name]
        _check_against_workspace_path(name, inp, dinp, kw, calls=1)


def test_noalloc_rejects_a_problem_beyond_its_static_size():
    p = F.make_params(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype=F.FDPP_BF16,
                      max_seq_len=16384, scale=0.088388, split_len=512)
    assert F.fdpp_workspace_size(p) > F.FDPP_NOALLOC_WORKSPACE_BYTES
    d = F.fdpp_diag()
    assert F.lib.fdpp_read_diag_noalloc(ctypes.byref(p), ctypes.byref(d), None, None) == \
        F.FDPP_ERR_WORKSPACE                               # host check, no CUDA call
    assert "static workspace" in F.fdpp_last_error()
    H.no_fake_pointer_calls_on_a_gpu()
    fake = 1 << 20                                       # never dereferenced: rejected first
    st = F.lib.fdpp_decode_attn_noalloc(fake, fake, fake, None, fake, ctypes.byref(p), fake, None)
    assert st == F.FDPP_ERR_WORKSPACE
    assert "static workspace" in F.fdpp_last_error()
