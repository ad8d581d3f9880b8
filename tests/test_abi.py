"""The C ABI without a GPU: the library loads, exports every function fdpp.h declares, and every
argument error is reported synchronously with the documented status before any CUDA call."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import split_kv_async_gb300 as F
from fdpp_harness import no_fake_pointer_calls_on_a_gpu

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
HEADER = os.path.join(INCLUDE, "fdpp.h")
GEMM_HEADER = os.path.join(INCLUDE, "fdpp_gemm.h")


def _declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(fdpp_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_names():
    assert _declared_functions() == sorted(F.EXPORTED)


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(F.lib, name)


def test_params_struct_matches_header_field_order():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct fdpp_params \{(.*?)\} fdpp_params;", text, re.S).group(1)
    names = re.findall(r"\b(\w+)\s*[;,]", body)
    assert names == [n for n, _ in F.fdpp_params._fields_]
    body = re.search(r"typedef struct fdpp_diag \{(.*?)\} fdpp_diag;", text, re.S).group(1)
    names = re.findall(r"\b(\w+)\s*;", body)
    assert names == [n for n, _ in F.fdpp_diag._fields_]


def test_binding_constants_match_header_defines():
    text = open(HEADER).read()
    found = re.findall(r"#define (FDPP_\w+) \(?(\d+)u?(?: << (\d+))?", text)
    defines = {name: int(v) << int(sh or 0) for name, v, sh in found}
    for name in ("FDPP_AUTO_UNITS_PER_SM", "FDPP_AUTO_GRANULE", "FDPP_AUTO_MIN_SPLIT",
                 "FDPP_TC_MAX_PARTS", "FDPP_NOALLOC_WORKSPACE_BYTES"):
        assert getattr(F, name) == defines[name], name
    gemm = dict((n, int(v)) for n, v in re.findall(r"#define (FDPP_\w+) (\d+)", open(GEMM_HEADER).read()))
    assert F.FDPP_GEMM_MAX_M == gemm["FDPP_GEMM_MAX_M"]


def _gqa_params(**kw):
    base = dict(batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype=F.FDPP_BF16,
                max_seq_len=4096, scale=float(np.float32(128 ** -0.5)), split_len=512)
    base.update(kw)
    return F.make_params(**base)


def test_max_splits_and_workspace_size():
    p = _gqa_params()
    assert F.fdpp_max_splits(p) == 8
    ws = F.fdpp_workspace_size(p)
    # partials o (d floats), l, m and a flag byte per split slot and per run slot (G = 4 rows
    # for each of FDPP_TC_MAX_PARTS parts plus one per (sequence, kv head)), the fallback lists
    # (8 lists of 32-byte entries, one per split piece: units, parts and (sequence, kv head)
    # pairs), plus header and plan
    slots = 8 * 32 * 8 + (F.FDPP_TC_MAX_PARTS + 8 * 8) * 4
    lists = 8 * (8 * 8 * 8 + F.FDPP_TC_MAX_PARTS + 8 * 8) * 32
    fixed = slots * (128 * 4 + 4 + 4 + 1) + lists
    assert fixed <= ws <= fixed + 64 * 1024
    assert ws % 256 == 0
    p0 = _gqa_params(split_len=0)
    assert F.fdpp_max_splits(p0) == 4096 // F.FDPP_AUTO_MIN_SPLIT
    p1 = _gqa_params(split_len=1000, max_seq_len=4097)
    assert F.fdpp_max_splits(p1) == 5


def test_workspace_size_with_row_groups():
    # 16 query tokens of 4 heads per kv head: R = 64 rows. Partials per (query row, split). The
    # run slots serve either build: the mma.sync build's hold one run of one row group of 8 rows
    # (one per part plus one per (sequence, kv head, row group)), the tcgen05 build's one run of
    # all R rows (one per part, at most FDPP_TC_UM_MAX_CTAS, plus one per (sequence, kv head));
    # the larger count is reserved. The fallback lists hold an entry per (sequence, kv head, row
    # group, split) and per part.
    p = _gqa_params(q_tokens=16)
    ws = F.fdpp_workspace_size(p)
    runs = max((F.FDPP_TC_MAX_PARTS + 8 * 8 * 8) * 8, (F.FDPP_TC_UM_MAX_CTAS + 8 * 8) * 64)
    slots = 8 * 16 * 32 * 8 + runs
    lists = 8 * (8 * 8 * 8 * 8 + F.FDPP_TC_MAX_PARTS + 8 * 8 * 8) * 32
    fixed = slots * (128 * 4 + 4 + 4 + 1) + lists
    assert fixed <= ws <= fixed + 64 * 1024
    # 12 rows: two groups (8 + 4), lists twice the one-group count
    p12 = _gqa_params(q_tokens=3)
    ws12 = F.fdpp_workspace_size(p12)
    runs = max((F.FDPP_TC_MAX_PARTS + 8 * 8 * 2) * 8, (F.FDPP_TC_UM_MAX_CTAS + 8 * 8) * 12)
    slots = 8 * 3 * 32 * 8 + runs
    lists = 8 * (8 * 8 * 2 * 8 + F.FDPP_TC_MAX_PARTS + 8 * 8 * 2) * 32
    fixed = slots * (128 * 4 + 4 + 4 + 1) + lists
    assert fixed <= ws12 <= fixed + 64 * 1024
    # head_dim 64 has no tcgen05 build: row-group run slots only
    p64 = _gqa_params(q_tokens=16, head_dim=64)
    ws64 = F.fdpp_workspace_size(p64)
    slots = 8 * 16 * 32 * 8 + (F.FDPP_TC_MAX_PARTS + 8 * 8 * 8) * 8
    lists = 8 * (8 * 8 * 8 * 8 + F.FDPP_TC_MAX_PARTS + 8 * 8 * 8) * 32
    fixed = slots * (64 * 4 + 4 + 4 + 1) + lists
    assert fixed <= ws64 <= fixed + 64 * 1024


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, F.FDPP_ERR_INVALID_ARG),
    ("num_q_heads", 30, F.FDPP_ERR_INVALID_ARG),        # not a multiple of 8 kv heads
    ("num_kv_heads", 0, F.FDPP_ERR_INVALID_ARG),
    ("head_dim", 96, F.FDPP_ERR_UNSUPPORTED),
    ("dtype", 7, F.FDPP_ERR_INVALID_ARG),
    ("max_seq_len", 0, F.FDPP_ERR_INVALID_ARG),
    ("split_len", -1, F.FDPP_ERR_INVALID_ARG),
    ("scale", float("nan"), F.FDPP_ERR_INVALID_ARG),
    ("scale", 0.0, F.FDPP_ERR_INVALID_ARG),
    ("scale", -0.125, F.FDPP_ERR_INVALID_ARG),
    ("phi", float("inf"), F.FDPP_ERR_INVALID_ARG),
    ("lo", 20.0, F.FDPP_ERR_INVALID_ARG),               # lo > hi
    ("mode", 3, F.FDPP_ERR_INVALID_ARG),
    ("kernel", 9, F.FDPP_ERR_INVALID_ARG),
    ("tc_stages", 1, F.FDPP_ERR_INVALID_ARG),
    ("tc_ctas_per_sm", 3, F.FDPP_ERR_INVALID_ARG),
    ("tc_prefetch", 33, F.FDPP_ERR_INVALID_ARG),
    ("tc_prefetch", -2, F.FDPP_ERR_INVALID_ARG),
    ("tc_mma", 3, F.FDPP_ERR_INVALID_ARG),
    ("tc_mma", -1, F.FDPP_ERR_INVALID_ARG),
])
def test_bad_params_are_rejected_on_the_host(field, value, status):
    p = _gqa_params()
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    assert F.lib.fdpp_workspace_size(ctypes.byref(p), ctypes.byref(n)) == status
    assert F.fdpp_last_error()
    no_fake_pointer_calls_on_a_gpu()
    fake = 1 << 20                                          # never dereferenced
    st = F.lib.fdpp_decode_attn(fake, fake, fake, None, fake, ctypes.byref(p), fake * 256,
                                1 << 30, fake, None)
    assert st == status


@pytest.mark.parametrize("kw", [
    dict(q_tokens=16, head_dim=64),                   # tcgen05 build: d = 128 only
    dict(q_tokens=2),                                 # 8 rows per kv head: the mma.sync build's
    dict(q_tokens=16, dtype=F.FDPP_F32),              # bf16 only
    dict(q_tokens=16, tc_ctas_per_sm=2),              # one CTA per SM
])
def test_tcgen05_build_outside_its_shapes_is_unsupported(kw):
    p = _gqa_params(kernel=F.FDPP_KERNEL_TENSOR, tc_mma=F.FDPP_TC_MMA_TCGEN05, **kw)
    assert F.fdpp_workspace_size(p) > 0
    assert _call(p) == F.FDPP_ERR_UNSUPPORTED
    assert F.fdpp_last_error()


def test_group_too_large_is_unsupported():
    p = _gqa_params(num_q_heads=128 * 8, num_kv_heads=8)    # G = 128 > 64 query rows per kv head
    n = ctypes.c_size_t(0)
    assert F.lib.fdpp_workspace_size(ctypes.byref(p), ctypes.byref(n)) == F.FDPP_ERR_UNSUPPORTED


def _call(p, q=1 << 20, k=1 << 20, v=1 << 20, bt=None, sl=1 << 20, ws=1 << 28, ws_bytes=None,
          out=1 << 20):
    # made-up device addresses: only where no kernel can be launched on them
    no_fake_pointer_calls_on_a_gpu()
    if ws_bytes is None:
        ws_bytes = F.fdpp_workspace_size(p)
    return F.lib.fdpp_decode_attn(q, k, v, bt, sl, ctypes.byref(p), ws, ws_bytes, out, None)


def test_pointer_and_workspace_errors():
    p = _gqa_params()
    assert _call(p, q=None) == F.FDPP_ERR_INVALID_ARG
    assert _call(p, out=None) == F.FDPP_ERR_INVALID_ARG
    assert _call(p, sl=None) == F.FDPP_ERR_INVALID_ARG
    assert _call(p, k=(1 << 20) + 8) == F.FDPP_ERR_INVALID_ARG       # 16-byte alignment
    assert _call(p, sl=(1 << 20) + 2) == F.FDPP_ERR_INVALID_ARG      # 4-byte alignment
    assert _call(p, ws=None) == F.FDPP_ERR_WORKSPACE
    assert _call(p, ws=(1 << 28) + 128) == F.FDPP_ERR_WORKSPACE      # 256-byte alignment
    assert _call(p, ws_bytes=F.fdpp_workspace_size(p) - 1) == F.FDPP_ERR_WORKSPACE
    assert "needed" in F.fdpp_last_error()


def test_paged_contract_errors():
    base = dict(block_size=16, max_blocks_per_seq=256, num_kv_blocks=1000)
    bt = 1 << 20
    assert _call(_gqa_params(**dict(base, block_size=24)), bt=bt) == F.FDPP_ERR_INVALID_ARG
    assert _call(_gqa_params(**dict(base, block_size=512)), bt=bt) == F.FDPP_ERR_INVALID_ARG
    assert _call(_gqa_params(**dict(base, max_blocks_per_seq=100)), bt=bt) == F.FDPP_ERR_INVALID_ARG
    assert _call(_gqa_params(**dict(base, num_kv_blocks=0)), bt=bt) == F.FDPP_ERR_INVALID_ARG
    assert _call(_gqa_params(split_len=520, **base), bt=bt) == F.FDPP_ERR_INVALID_ARG
    # The same parameters without a block table are a contiguous cache: the host checks ignore
    # the block fields, and with no device the call stops at the device query.
    assert _call(_gqa_params(**dict(base, block_size=24))) == F.FDPP_ERR_CUDA


def test_tensor_kernel_limits():
    fp32 = _gqa_params(dtype=F.FDPP_F32, kernel=F.FDPP_KERNEL_TENSOR)
    assert _call(fp32) == F.FDPP_ERR_UNSUPPORTED
    too_many_rows = _gqa_params(num_q_heads=128, num_kv_heads=1, kernel=F.FDPP_KERNEL_TENSOR)
    assert _call(too_many_rows, ws_bytes=1 << 30) == F.FDPP_ERR_UNSUPPORTED   # 128 rows > 64
    simt_rows = _gqa_params(num_q_heads=64, num_kv_heads=2, kernel=F.FDPP_KERNEL_SIMT)
    assert _call(simt_rows) == F.FDPP_ERR_UNSUPPORTED              # 32 rows > the SIMT kernel's 16


def test_status_strings():
    for s, name in [(0, "FDPP_OK"), (1, "FDPP_ERR_INVALID_ARG"), (2, "FDPP_ERR_UNSUPPORTED"),
                    (3, "FDPP_ERR_WORKSPACE"), (4, "FDPP_ERR_CUDA")]:
        assert F.fdpp_status_str(s) == name


def test_no_gpu_gives_cuda_error_not_a_crash():
    assert _call(_gqa_params()) == F.FDPP_ERR_CUDA


# ---- flat GEMM: argument errors before any CUDA call ----------------------------------------

def _gemm_status(x=16, w=16, y=16, M=8, N=256, K=512, split_k=0, ws=256, ws_bytes=1 << 20):
    no_fake_pointer_calls_on_a_gpu()
    return F.lib.fdpp_flat_gemm(x, w, y, M, N, K, split_k, ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(M=0), dict(M=129), dict(N=0), dict(K=4), dict(K=100),
                                dict(x=None), dict(w=None), dict(y=None), dict(x=24),
                                dict(w=8), dict(split_k=-1), dict(split_k=9), dict(K=4096, split_k=9)])
def test_flat_gemm_rejects_bad_arguments(kw):
    assert _gemm_status(**kw) == F.FDPP_ERR_INVALID_ARG
    assert F.fdpp_last_error()


def test_flat_gemm_rejects_a_misaligned_workspace():
    assert _gemm_status(ws=256 + 64) == F.FDPP_ERR_WORKSPACE


def test_flat_gemm_split_k_and_size_reject_bad_shapes():
    assert F.fdpp_flat_gemm_split_k(0, 128, 64) == 0
    assert F.fdpp_flat_gemm_split_k(8, 128, 63) == 0
    assert F.fdpp_flat_gemm_workspace_size(8, 0, 64) == 0


@pytest.mark.parametrize("rows", [[(0, 128, 64, 1)], [(8, 128, 4, 1)], [(8, 128, 64, 0)]])
def test_flat_gemm_lut_rejects_bad_entries(rows):
    with pytest.raises(F.FdppError):
        F.fdpp_flat_gemm_set_lut(rows)


def test_flat_gemm_lut_accepts_and_clears():
    F.fdpp_flat_gemm_set_lut([(16, 4096, 4096, 10)])
    F.fdpp_flat_gemm_set_lut([])
