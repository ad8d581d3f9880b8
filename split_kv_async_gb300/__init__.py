"""Python binding of libfdpp: unified-max split-KV decode attention on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the library's CUDA kernels. The
functions keep the C names of ``include/fdpp.h`` (``fdpp_decode_attn``, ``fdpp_workspace_size``,
...) and take torch tensors (device memory and streams come from PyTorch; no torch op computes
anything here). Importing this module loads ``libfdpp.so``; if it was not built this raises, there
is no fallback.

The operation (opt.ai.kr "FlashDecoding++ async softmax -- theory", sections 1 and 3): one query
token per sequence attends to its K/V cache; the cache is cut into splits that each work against a
unified max phi, a split whose scores leave lo <= s - phi <= hi is recomputed with online softmax,
and the split partials are combined by a (max-rescaled, otherwise plain) sum.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfdpp.so")

FDPP_OK, FDPP_ERR_INVALID_ARG, FDPP_ERR_UNSUPPORTED, FDPP_ERR_WORKSPACE, FDPP_ERR_CUDA = range(5)
FDPP_F32, FDPP_BF16 = 0, 1
FDPP_MODE_NORMAL, FDPP_MODE_FORCE_FAST, FDPP_MODE_FORCE_ONLINE = 0, 1, 2
FDPP_KERNEL_AUTO, FDPP_KERNEL_TENSOR, FDPP_KERNEL_SIMT = 0, 1, 2
FDPP_TC_MMA_AUTO, FDPP_TC_MMA_SYNC, FDPP_TC_MMA_TCGEN05 = 0, 1, 2
FDPP_FLAG_OUT, FDPP_FLAG_ABOVE, FDPP_FLAG_BELOW, FDPP_FLAG_NAN, FDPP_FLAG_RECOMPUTED = 1, 2, 4, 8, 16
FDPP_FLAG_SLOT = 32
FDPP_ERRBIT_SEQ_LEN, FDPP_ERRBIT_BLOCK_TABLE, FDPP_ERRBIT_TIMEOUT = 1, 2, 4
FDPP_AUTO_UNITS_PER_SM, FDPP_AUTO_GRANULE, FDPP_AUTO_MIN_SPLIT = 4, 64, 256

# Names every build of the library exports (the C ABI of include/fdpp.h and include/fdpp_gemm.h).
EXPORTED = ("fdpp_max_splits", "fdpp_workspace_size", "fdpp_workspace_init", "fdpp_decode_attn",
            "fdpp_decode_attn_timed", "fdpp_decode_attn_noalloc", "fdpp_score_ranges",
            "fdpp_pick_phi", "fdpp_read_diag", "fdpp_read_diag_noalloc", "fdpp_status_str",
            "fdpp_last_error", "fdpp_attn_set_lut", "fdpp_attn_auto_choice",
            "fdpp_flat_gemm_split_k", "fdpp_flat_gemm_workspace_size", "fdpp_flat_gemm",
            "fdpp_flat_gemm_set_lut", "fdpp_flat_gemm_read_error")
FDPP_GEMM_MAX_M = 128
FDPP_NOALLOC_WORKSPACE_BYTES = 16 << 20
FDPP_TC_MAX_PARTS = 512
FDPP_TC_UM_MAX_CTAS = 256


class FdppError(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {reason}")
        self.status = status


_STATUS_NAMES = {0: "FDPP_OK", 1: "FDPP_ERR_INVALID_ARG", 2: "FDPP_ERR_UNSUPPORTED",
                 3: "FDPP_ERR_WORKSPACE", 4: "FDPP_ERR_CUDA"}


class fdpp_params(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("block_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
        ("num_kv_blocks", ctypes.c_int),
        ("scale", ctypes.c_float), ("phi", ctypes.c_float), ("lo", ctypes.c_float),
        ("hi", ctypes.c_float),
        ("split_len", ctypes.c_int), ("mode", ctypes.c_int), ("kernel", ctypes.c_int),
        ("tc_stages", ctypes.c_int), ("tc_ctas_per_sm", ctypes.c_int),
        ("tc_prefetch", ctypes.c_int), ("phi_heads", ctypes.c_void_p),
        ("q_tokens", ctypes.c_int), ("tc_mma", ctypes.c_int),
    ]


class fdpp_diag(ctypes.Structure):
    _fields_ = [
        ("split_len", ctypes.c_int32), ("max_splits", ctypes.c_int32),
        ("n_units", ctypes.c_int64), ("n_flagged_row_splits", ctypes.c_int64),
        ("n_flagged_units", ctypes.c_int64), ("n_recomputed_row_splits", ctypes.c_int64),
        ("error_bits", ctypes.c_uint32), ("kernel", ctypes.c_int32),
        ("tc_build", ctypes.c_int32), ("tc_parts", ctypes.c_int32), ("tc_seg_tiles", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class fdpp_attn_lut_row(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in ("max_batch", "max_seq_len", "max_rows", "kernel",
                                                  "units_per_sm", "min_split")]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(fdpp_params)
    vp = ctypes.c_void_p
    lib.fdpp_max_splits.argtypes = [P]
    lib.fdpp_max_splits.restype = ctypes.c_int
    lib.fdpp_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.fdpp_workspace_size.restype = ctypes.c_int
    lib.fdpp_workspace_init.argtypes = [vp, ctypes.c_size_t, vp]
    lib.fdpp_workspace_init.restype = ctypes.c_int
    lib.fdpp_decode_attn.argtypes = [vp, vp, vp, vp, vp, P, vp, ctypes.c_size_t, vp, vp]
    lib.fdpp_decode_attn.restype = ctypes.c_int
    lib.fdpp_decode_attn_timed.argtypes = [vp, vp, vp, vp, vp, P, vp, ctypes.c_size_t, vp, vp, vp,
                                           vp]
    lib.fdpp_decode_attn_timed.restype = ctypes.c_int
    lib.fdpp_decode_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, P, vp, vp]
    lib.fdpp_decode_attn_noalloc.restype = ctypes.c_int
    lib.fdpp_score_ranges.argtypes = [vp, vp, vp, vp, P, vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.fdpp_score_ranges.restype = ctypes.c_int
    lib.fdpp_pick_phi.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_float, ctypes.c_float, vp, vp]
    lib.fdpp_pick_phi.restype = ctypes.c_int
    lib.fdpp_read_diag.argtypes = [vp, ctypes.c_size_t, P, ctypes.POINTER(fdpp_diag), vp, vp]
    lib.fdpp_read_diag.restype = ctypes.c_int
    lib.fdpp_read_diag_noalloc.argtypes = [P, ctypes.POINTER(fdpp_diag), vp, vp]
    lib.fdpp_read_diag_noalloc.restype = ctypes.c_int
    lib.fdpp_attn_set_lut.argtypes = [ctypes.POINTER(fdpp_attn_lut_row), ctypes.c_int]
    lib.fdpp_attn_set_lut.restype = ctypes.c_int
    ip = ctypes.POINTER(ctypes.c_int)
    lib.fdpp_attn_auto_choice.argtypes = [P, ip, ip, ip]
    lib.fdpp_attn_auto_choice.restype = ctypes.c_int
    lib.fdpp_status_str.argtypes = [ctypes.c_int]
    lib.fdpp_status_str.restype = ctypes.c_char_p
    lib.fdpp_last_error.argtypes = []
    lib.fdpp_last_error.restype = ctypes.c_char_p
    ci = ctypes.c_int
    lib.fdpp_flat_gemm_split_k.argtypes = [ci, ci, ci, ci]
    lib.fdpp_flat_gemm_split_k.restype = ci
    lib.fdpp_flat_gemm_workspace_size.argtypes = [ci, ci, ci, ci]
    lib.fdpp_flat_gemm_workspace_size.restype = ctypes.c_size_t
    lib.fdpp_flat_gemm.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.c_size_t, vp]
    lib.fdpp_flat_gemm.restype = ci
    lib.fdpp_flat_gemm_set_lut.argtypes = [vp, ci]
    lib.fdpp_flat_gemm_set_lut.restype = ci
    lib.fdpp_flat_gemm_read_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.fdpp_flat_gemm_read_error.restype = ci
    return lib


lib = _load()


def _check(status: int, where: str) -> None:
    if status != FDPP_OK:
        raise FdppError(status, where, lib.fdpp_last_error().decode())


def make_params(*, batch, num_q_heads, num_kv_heads, head_dim, dtype, max_seq_len, scale,
                phi=0.0, lo=-30.0, hi=10.0, split_len=0, block_size=0, max_blocks_per_seq=0,
                num_kv_blocks=0, mode=FDPP_MODE_NORMAL, kernel=FDPP_KERNEL_AUTO, tc_stages=0,
                tc_ctas_per_sm=0, tc_prefetch=0, phi_heads=None, q_tokens=1,
                tc_mma=FDPP_TC_MMA_AUTO) -> fdpp_params:
    """phi_heads: a float32 device tensor [num_q_heads] (or its address), or None. q_tokens:
    query tokens per sequence (q and out are then [batch][q_tokens][num_q_heads][head_dim]).
    tc_mma: the tensor kernel's build for more than 8 query rows per kv head."""
    ph = phi_heads if phi_heads is None or isinstance(phi_heads, int) else phi_heads.data_ptr()
    return fdpp_params(batch, num_q_heads, num_kv_heads, head_dim, dtype, max_seq_len, block_size,
                       max_blocks_per_seq, num_kv_blocks, scale, phi, lo, hi, split_len, mode,
                       kernel, tc_stages, tc_ctas_per_sm, tc_prefetch, ph, q_tokens, tc_mma)


def fdpp_max_splits(p: fdpp_params) -> int:
    n = lib.fdpp_max_splits(ctypes.byref(p))
    if n < 0:
        raise FdppError(FDPP_ERR_INVALID_ARG, "fdpp_max_splits", lib.fdpp_last_error().decode())
    return n


def fdpp_workspace_size(p: fdpp_params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.fdpp_workspace_size(ctypes.byref(p), ctypes.byref(n)), "fdpp_workspace_size")
    return n.value


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def fdpp_workspace_init(workspace, stream=None) -> None:
    _check(lib.fdpp_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream)), "fdpp_workspace_init")


def alloc_workspace(p: fdpp_params, device="cuda", stream=None):
    """Allocates (torch) and zeroes a workspace for `p`. The library itself allocates nothing."""
    import torch
    ws = torch.empty(fdpp_workspace_size(p), dtype=torch.uint8, device=device)
    fdpp_workspace_init(ws, stream)
    return ws


def fdpp_decode_attn(q, k_cache, v_cache, block_table, seq_lens, p: fdpp_params, workspace, out,
                     stream=None) -> None:
    """Enqueues one decode-attention step (tensors must be contiguous device tensors)."""
    _check(lib.fdpp_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                _ptr(seq_lens), ctypes.byref(p), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(out),
                                _stream_handle(stream)), "fdpp_decode_attn")


def fdpp_decode_attn_timed(q, k_cache, v_cache, block_table, seq_lens, p: fdpp_params, workspace,
                           out, ev_split_begin=None, ev_split_end=None, stream=None) -> None:
    """fdpp_decode_attn that also records two torch.cuda.Event around the split kernel."""
    _check(lib.fdpp_decode_attn_timed(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), ctypes.byref(p),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _stream_handle(stream), None if ev_split_begin is None else ev_split_begin.cuda_event,
        None if ev_split_end is None else ev_split_end.cuda_event), "fdpp_decode_attn_timed")


def fdpp_decode_attn_noalloc(q, k_cache, v_cache, block_table, seq_lens, p: fdpp_params, out,
                             stream=None) -> None:
    """The decode step for callers that cannot allocate: no workspace argument, the library's
    own static device array is the scratch (see include/fdpp.h for its size and sharing rules)."""
    _check(lib.fdpp_decode_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                        _ptr(seq_lens), ctypes.byref(p), _ptr(out),
                                        _stream_handle(stream)), "fdpp_decode_attn_noalloc")


def fdpp_score_ranges(q, k_cache, block_table, seq_lens, p: fdpp_params, workspace, stream=None):
    """Least and greatest score of every row-split on sample inputs (synchronous). Returns
    (smin, smax float32 numpy [B*Tq][Hq][max_splits], NaN where a query row has no key of the
    split; nsplit int32 [B*Tq])."""
    import numpy as np
    ms = fdpp_max_splits(p)
    rows = p.batch * max(1, p.q_tokens)
    smin = np.empty((rows, p.num_q_heads, ms), np.float32)
    smax = np.empty_like(smin)
    ns = np.empty(rows, np.int32)
    _check(lib.fdpp_score_ranges(_ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(seq_lens),
                                 ctypes.byref(p), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), smin.ctypes.data,
                                 smax.ctypes.data, ns.ctypes.data, _stream_handle(stream)),
           "fdpp_score_ranges")
    return smin, smax, ns


def fdpp_pick_phi(smin, smax, nsplit, lo, hi, fallback=0.0):
    """Per-head phi from score ranges (host only). Returns (phi float32 [Hq], kept int32 [Hq])."""
    import numpy as np
    smin = np.ascontiguousarray(smin, dtype=np.float32)
    smax = np.ascontiguousarray(smax, dtype=np.float32)
    ns = np.ascontiguousarray(nsplit, dtype=np.int32)
    B, Hq, ms = smin.shape
    phi = np.empty(Hq, np.float32)
    kept = np.empty(Hq, np.int32)
    _check(lib.fdpp_pick_phi(smin.ctypes.data, smax.ctypes.data, ns.ctypes.data, B, Hq, ms,
                             lo, hi, fallback, phi.ctypes.data, kept.ctypes.data), "fdpp_pick_phi")
    return phi, kept


def fdpp_read_diag(workspace, p: fdpp_params, want_flags=False, want_nsplit=False):
    """Returns (diag dict, flags uint8 numpy [B][Hq][max_splits] or None, nsplit or None)."""
    import numpy as np
    d = fdpp_diag()
    ms = fdpp_max_splits(p)
    flags = np.zeros((p.batch * max(1, p.q_tokens), p.num_q_heads, ms), np.uint8) if want_flags else None
    ns = np.zeros(p.batch, np.int32) if want_nsplit else None
    _check(lib.fdpp_read_diag(_ptr(workspace), workspace.numel() * workspace.element_size(),
                              ctypes.byref(p), ctypes.byref(d),
                              None if flags is None else flags.ctypes.data,
                              None if ns is None else ns.ctypes.data), "fdpp_read_diag")
    return d.as_dict(), flags, ns


def fdpp_read_diag_noalloc(p: fdpp_params, want_flags=False, want_nsplit=False):
    """fdpp_read_diag for the no-alloc entry point's static array on the current device."""
    import numpy as np
    d = fdpp_diag()
    ms = fdpp_max_splits(p)
    flags = np.zeros((p.batch * max(1, p.q_tokens), p.num_q_heads, ms), np.uint8) if want_flags else None
    ns = np.zeros(p.batch, np.int32) if want_nsplit else None
    _check(lib.fdpp_read_diag_noalloc(ctypes.byref(p), ctypes.byref(d),
                                      None if flags is None else flags.ctypes.data,
                                      None if ns is None else ns.ctypes.data),
           "fdpp_read_diag_noalloc")
    return d.as_dict(), flags, ns


def fdpp_attn_set_lut(rows) -> None:
    """rows: (max_batch, max_seq_len, max_rows, kernel, units_per_sm, min_split) tuples, first
    match wins; an empty list removes the table."""
    arr = (fdpp_attn_lut_row * max(1, len(rows)))()
    for i, r in enumerate(rows):
        arr[i] = fdpp_attn_lut_row(*[int(x) for x in r])
    _check(lib.fdpp_attn_set_lut(arr if rows else None, len(rows)), "fdpp_attn_set_lut")


def fdpp_attn_auto_choice(p: fdpp_params):
    """(kernel, units_per_sm, min_split) a call with `p` uses (host only)."""
    k, u, m = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.fdpp_attn_auto_choice(ctypes.byref(p), ctypes.byref(k), ctypes.byref(u),
                                     ctypes.byref(m)), "fdpp_attn_auto_choice")
    return k.value, u.value, m.value


def fdpp_status_str(status: int) -> str:
    return lib.fdpp_status_str(status).decode()


def fdpp_last_error() -> str:
    return lib.fdpp_last_error().decode()


# ---- flat GEMM (include/fdpp_gemm.h) --------------------------------------------------------

def fdpp_flat_gemm_split_k(M: int, N: int, K: int, split_k: int = 0) -> int:
    """split_k fdpp_flat_gemm uses on the current device (0: the shape is invalid)."""
    return int(lib.fdpp_flat_gemm_split_k(M, N, K, split_k))


def fdpp_flat_gemm_workspace_size(M: int, N: int, K: int, split_k: int = 0) -> int:
    return int(lib.fdpp_flat_gemm_workspace_size(M, N, K, split_k))


def alloc_flat_gemm_workspace(M: int, N: int, K: int, split_k: int = 0, device="cuda"):
    """A zeroed uint8 device tensor large enough for fdpp_flat_gemm(M, N, K, split_k)."""
    import torch
    n = fdpp_flat_gemm_workspace_size(M, N, K, split_k)
    if n == 0:
        raise FdppError(FDPP_ERR_INVALID_ARG, "fdpp_flat_gemm_workspace_size",
                        f"invalid shape M={M} N={N} K={K}")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def fdpp_flat_gemm(x, w, y, workspace, split_k: int = 0, stream=None) -> None:
    """y = x W^T: x [M][K], w [N][K], y [M][N], bf16 device tensors (or addresses with shapes
    given by the tensors)."""
    M, K = int(x.shape[0]), int(x.shape[1])
    N = int(w.shape[0])
    _check(lib.fdpp_flat_gemm(_ptr(x), _ptr(w), _ptr(y), M, N, K, split_k, _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream_handle(stream)), "fdpp_flat_gemm")


def fdpp_flat_gemm_set_lut(entries) -> None:
    """entries: rows of (m_max, N, K, split_k); an empty list clears the table."""
    import numpy as np
    e = np.ascontiguousarray(np.asarray(entries, np.int32).reshape(-1, 4))
    _check(lib.fdpp_flat_gemm_set_lut(e.ctypes.data if len(e) else None, len(e)),
           "fdpp_flat_gemm_set_lut")


def fdpp_flat_gemm_read_error(workspace) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib.fdpp_flat_gemm_read_error(_ptr(workspace), ctypes.byref(bits)),
           "fdpp_flat_gemm_read_error")
    return int(bits.value)
