"""fdpp_decode_attn_noalloc: the decode step for callers that cannot allocate device memory (for
example a plugin inside a runtime that owns every device allocation, or a serving loop whose
memory is fixed at start-up). Its scratch is the library's own static device array, so it takes
no workspace. Its output must agree with fdpp_decode_attn's on the same inputs, call after call.

This file is named to be collected last: if it fails, a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import fdpp_harness as H
import workloads as W

try:
    import split_kv_async_gb300 as F
except ImportError:
    F = None


def _run_noalloc(dinp, p):
    import torch
    out = torch.full_like(dinp.q, float("nan"))
    F.fdpp_decode_attn_noalloc(dinp.q, dinp.k, dinp.v, dinp.block_table, dinp.seq_lens, p, out)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(-1, dinp.inp.wl.head_dim).astype(np.float64)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["gqa_ragged", "hot_keys"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    if case == "gqa_ragged":
        wl = W.GQA.replace(name="noalloc_gqa", batch=4, split_len=256)
        inp = W.generate(wl, seq_lens=np.array([1000, 513, 71, 300], np.int32))
    else:
        # hot keys: the fallback list inside the static array is used and must
        # be left clean for the next call
        wl = W.STRESS.replace(name="noalloc_hot", batch=4, seq_len=768, split_len=256,
                              stress_frac=0.1)
        inp = W.generate(wl)
    dinp = H.DeviceInputs(inp)
    p = H.params_for(inp)
    assert F.fdpp_workspace_size(p) <= F.FDPP_NOALLOC_WORKSPACE_BYTES
    ref, diag, _, _, _ = H.run(dinp)                  # the workspace entry point
    assert diag["error_bits"] == 0
    for call in range(2):
        got = _run_noalloc(dinp, p)
        H.assert_parity(got, ref, f"{case} no-alloc call {call + 1}")


def test_noalloc_rejects_a_problem_beyond_its_static_size():
    p = F.make_params(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype=F.FDPP_BF16,
                      max_seq_len=16384, scale=0.088388, split_len=512)
    assert F.fdpp_workspace_size(p) > F.FDPP_NOALLOC_WORKSPACE_BYTES
    fake = 1 << 20                                       # never dereferenced: rejected first
    st = F.lib.fdpp_decode_attn_noalloc(fake, fake, fake, None, fake, ctypes.byref(p), fake, None)
    assert st == F.FDPP_ERR_WORKSPACE
    assert "static workspace" in F.fdpp_last_error()
