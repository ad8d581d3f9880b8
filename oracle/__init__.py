"""fp64 CPU oracle for unified-max split-KV decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package. The CUDA library shares
no code with it.

All arithmetic lives in ``oracle.c`` (plain C, double precision, pthreads over rows); this module
only compiles it with gcc, loads it with ctypes and marshals numpy arrays. Each C function cites
the passage of the pages it follows:

* ``attention``        -- the plain definition softmax(scale * q K^T) V, max-shifted
  (opt.ai.kr "FlashDecoding++ async softmax -- theory", section 3, first formula).
* ``attention_shifted`` -- the same softmax shifted by a fixed value phi (same page, section 3,
  second formula).
* ``window_flags``     -- the per-(sequence, head, split) out-of-window decision (same page,
  section 3: a score past the phi criterion sends its block back to online softmax).
* ``split_method``     -- the method's steps in fp64: phi-frame partials per split, detect,
  online recompute, max-rescaled (plain when nothing fell back) sum.
* ``inplace_partial``  -- one row's partial when a block continues in place with the running max
  from its first tile holding an out-of-window score (oracle.c, R11).
* ``split_len`` / ``plan`` -- the split scheduler restated: n_b = ceil(L_b / S).
* several query tokens per sequence (``make_problem(q_tokens=Tq)``): the last Tq positions,
  causal (oracle.c, R9); every function above then works on the B*Tq query rows.
* ``score_ranges`` / ``pick_phi`` -- phi observed in advance (same page, section 3): the score
  range of every row-split on sample inputs, and per head the phi that keeps the most row-splits
  inside the window (the reading is stated in oracle.c, R8).

``window_flags`` and ``split_method`` take an optional per-head phi (oracle.c, R7).

Parity status: every function above is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
MODE_NORMAL, MODE_FORCE_FAST, MODE_FORCE_ONLINE = 0, 1, 2
FLAG_OUT, FLAG_ABOVE, FLAG_BELOW, FLAG_NAN = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (IEEE double, no contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("paged", ctypes.c_int),
        ("max_seq_len", ctypes.c_int), ("block_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("scale", ctypes.c_float), ("phi", ctypes.c_float), ("lo", ctypes.c_float),
        ("hi", ctypes.c_float), ("q_tokens", ctypes.c_int),
    ]

    @property
    def query_rows(self) -> int:
        """B * Tq: q, out, flags and ranges are [B*Tq][Hq][...] (oracle.c, R9)."""
        return self.batch * max(1, self.q_tokens)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER(Problem)
            vp, ip = ctypes.c_void_p, ctypes.c_void_p
            lib.or_attention.argtypes = [P, vp, vp, vp, ip, ip, ip, ctypes.c_int, vp, ctypes.c_int]
            lib.or_attention.restype = ctypes.c_int
            lib.or_attention_shifted.argtypes = [P, vp, vp, vp, ip, ip, ip, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, vp, ctypes.c_int]
            lib.or_attention_shifted.restype = ctypes.c_int
            lib.or_window_flags.argtypes = [P, vp, vp, ip, ip, ctypes.c_int, ctypes.c_int, vp, vp,
                                            vp, ctypes.c_int]
            lib.or_window_flags.restype = ctypes.c_int
            lib.or_split_method.argtypes = [P, vp, vp, vp, ip, ip, ip, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_int]
            lib.or_split_method.restype = ctypes.c_int
            lib.or_score_ranges.argtypes = [P, vp, vp, ip, ip, ctypes.c_int, ctypes.c_int, vp, vp,
                                            ctypes.c_int]
            lib.or_score_ranges.restype = ctypes.c_int
            lib.or_pick_phi.argtypes = [vp, vp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_double, vp, vp]
            lib.or_pick_phi.restype = ctypes.c_int
            lib.or_split_len.argtypes = [ip] + [ctypes.c_int] * 8
            lib.or_split_len.restype = ctypes.c_int
            lib.or_plan.argtypes = [ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ip, ip]
            lib.or_plan.restype = ctypes.c_longlong
            lib.or_flat_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         vp, vp, ip, ctypes.c_int, vp, ctypes.c_int]
            lib.or_flat_gemm.restype = ctypes.c_int
            lib.or_inplace_partial.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                               vp, vp, vp]
            lib.or_inplace_partial.restype = ctypes.c_int
            lib.or_default_threads.argtypes = []
            lib.or_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _kv_array(a, dtype):
    """Inputs are uint16 bf16 bit patterns (dtype BF16) or float32 (dtype F32), C-contiguous."""
    want = np.uint16 if dtype == BF16 else np.float32
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"expected {want} array, got {a.dtype}")
    return a


def make_problem(*, batch, num_q_heads, num_kv_heads, head_dim, dtype, scale, phi, lo, hi,
                 max_seq_len=0, block_size=0, max_blocks_per_seq=0, paged=False,
                 q_tokens=1) -> Problem:
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    return Problem(batch, num_q_heads, num_kv_heads, head_dim, dtype, 1 if paged else 0,
                   max_seq_len, block_size, max_blocks_per_seq,
                   np.float32(scale), np.float32(phi), np.float32(lo), np.float32(hi),
                   max(1, int(q_tokens)))


def _rows_arg(prob, rows):
    if rows is None:
        return None, prob.query_rows * prob.num_q_heads
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    return r, r.shape[0]


def default_threads() -> int:
    return _load().or_default_threads()


def attention(prob, q, k, v, seq_lens, block_table=None, rows=None, n_threads=0):
    """Exact attention rows in fp64. Returns (out [n_rows][d] float64, threads used)."""
    lib = _load()
    q, k, v = (_kv_array(x, prob.dtype) for x in (q, k, v))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    r, n = _rows_arg(prob, rows)
    out = np.zeros((n, prob.head_dim), dtype=np.float64)
    used = lib.or_attention(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                            _ptr(r), n, _ptr(out), n_threads)
    return out, used


def attention_shifted(prob, q, k, v, seq_lens, shift=None, block_table=None, rows=None,
                      n_threads=0):
    """exp(s - shift)-weighted attention (shift = prob.phi when None)."""
    lib = _load()
    q, k, v = (_kv_array(x, prob.dtype) for x in (q, k, v))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    r, n = _rows_arg(prob, rows)
    out = np.zeros((n, prob.head_dim), dtype=np.float64)
    lib.or_attention_shifted(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                             _ptr(r), n, 0 if shift is None else 1,
                             0.0 if shift is None else float(shift), _ptr(out), n_threads)
    return out


def _phi_arg(prob, phi_heads):
    if phi_heads is None:
        return None
    a = np.ascontiguousarray(phi_heads, dtype=np.float32).reshape(-1)
    if a.size != prob.num_q_heads:
        raise ValueError("phi_heads needs one value per query head")
    return a


def window_flags(prob, q, k, seq_lens, split_len, max_splits, block_table=None, phi_heads=None,
                 n_threads=0):
    """Returns (flags uint8 [B][Hq][max_splits], row_margin float64 [B][Hq])."""
    lib = _load()
    q, k = (_kv_array(x, prob.dtype) for x in (q, k))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    ph = _phi_arg(prob, phi_heads)
    flags = np.zeros((prob.query_rows, prob.num_q_heads, max_splits), dtype=np.uint8)
    margin = np.zeros((prob.query_rows, prob.num_q_heads), dtype=np.float64)
    lib.or_window_flags(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(bt), _ptr(sl), split_len,
                        max_splits, _ptr(flags), _ptr(margin), _ptr(ph), n_threads)
    return flags, margin


def score_ranges(prob, q, k, seq_lens, split_len, max_splits, block_table=None, n_threads=0):
    """Least and greatest score of every row-split: (smin, smax) float64 [B][Hq][max_splits],
    NaN past a sequence's splits."""
    lib = _load()
    q, k = (_kv_array(x, prob.dtype) for x in (q, k))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    smin = np.zeros((prob.query_rows, prob.num_q_heads, max_splits), dtype=np.float64)
    smax = np.zeros_like(smin)
    lib.or_score_ranges(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(bt), _ptr(sl), split_len,
                        max_splits, _ptr(smin), _ptr(smax), n_threads)
    return smin, smax


def pick_phi(smin, smax, nsplit, lo, hi, fallback):
    """Per-head phi from score ranges [B][Hq][max_splits] (oracle.c, R8). Returns (phi float64
    [Hq], kept int32 [Hq]: the row-splits each head's phi keeps inside the window)."""
    lib = _load()
    smin = np.ascontiguousarray(smin, dtype=np.float64)
    smax = np.ascontiguousarray(smax, dtype=np.float64)
    B, Hq, ms = smin.shape
    ns = np.ascontiguousarray(nsplit, dtype=np.int32)
    phi = np.zeros(Hq, dtype=np.float64)
    kept = np.zeros(Hq, dtype=np.int32)
    lib.or_pick_phi(_ptr(smin), _ptr(smax), _ptr(ns), B, Hq, ms, float(lo), float(hi),
                    float(fallback), _ptr(phi), _ptr(kept))
    return phi, kept


def split_method(prob, q, k, v, seq_lens, split_len, max_splits, mode=MODE_NORMAL,
                 block_table=None, rows=None, want_partials=False, phi_heads=None, n_threads=0):
    """The method's steps in fp64. Returns dict(out, flags[, part_o, part_l, part_m])."""
    lib = _load()
    q, k, v = (_kv_array(x, prob.dtype) for x in (q, k, v))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    r, n = _rows_arg(prob, rows)
    d = prob.head_dim
    res = {"out": np.zeros((n, d), dtype=np.float64),
           "flags": np.zeros((n, max_splits), dtype=np.uint8)}
    if want_partials:
        res["part_o"] = np.zeros((n, max_splits, d), dtype=np.float64)
        res["part_l"] = np.zeros((n, max_splits), dtype=np.float64)
        res["part_m"] = np.zeros((n, max_splits), dtype=np.float64)
    ph = _phi_arg(prob, phi_heads)
    lib.or_split_method(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                        _ptr(r), n, split_len, max_splits, mode, _ptr(res["out"]),
                        _ptr(res.get("part_o")), _ptr(res.get("part_l")),
                        _ptr(res.get("part_m")), _ptr(res["flags"]), _ptr(ph), n_threads)
    return res


def inplace_partial(s, v, tile, phi, lo, hi):
    """One softmax row's partial by oracle.c R11 (the in-place finish of a block whose scores
    leave the window). s: scaled scores [n], v: values [n][d]. Returns (o [d], l, m, switched)."""
    lib = _load()
    s = np.ascontiguousarray(s, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64).reshape(len(s), -1)
    o = np.zeros(v.shape[1], dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    sw = lib.or_inplace_partial(_ptr(s), _ptr(v), len(s), v.shape[1], int(tile), float(phi),
                                float(lo), float(hi), _ptr(o), _ptr(l), _ptr(m))
    if sw < 0:
        raise ValueError("or_inplace_partial: bad arguments")
    return o, float(l[0]), float(m[0]), bool(sw)


def split_len(seq_lens, num_kv_heads, max_seq_len, split_len_req, num_sms, units_per_sm,
              granule, min_split):
    lib = _load()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    return lib.or_split_len(_ptr(sl), sl.shape[0], num_kv_heads, max_seq_len, split_len_req,
                            num_sms, units_per_sm, granule, min_split)


def dataflow_choice(rows, batch, max_seq_len, rows_per_kv_head, bf16,
                    default_units=4, default_min_split=256):
    """The heuristic dataflow table's choice for one call shape (opt.ai.kr "FlashDecoding++
    async softmax -- theory", s4: the configuration comes from a table measured in advance, per
    shape range). rows: (max_batch, max_seq_len, max_rows, kernel, units_per_sm, min_split); the
    first row whose ranges hold (batch, max_seq_len, rows_per_kv_head) applies. Kernel ids: 0 no
    preference, 1 tensor cores (bf16, at most 64 rows per kv head), 2 CUDA cores (at most 16);
    without a usable preference the tensor kernel is taken where it applies, else CUDA cores.
    Returns (kernel, units_per_sm, min_split)."""
    kernel, units, min_split = 0, default_units, default_min_split
    for (mb, ml, mr, k, u, m) in rows:
        if batch <= mb and max_seq_len <= ml and rows_per_kv_head <= mr:
            kernel, units, min_split = k, u, m
            break
    tensor_ok = bf16 and rows_per_kv_head <= 64
    simt_ok = rows_per_kv_head <= 16
    if not ((kernel == 1 and tensor_ok) or (kernel == 2 and simt_ok)):
        kernel = 1 if tensor_ok else 2
    return kernel, units, min_split


def plan(seq_lens, num_kv_heads, max_seq_len, S):
    """Returns (nsplit int32 [B], split_off int32 [B+1], n_units)."""
    lib = _load()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.shape[0]
    nsplit = np.zeros(B, dtype=np.int32)
    off = np.zeros(B + 1, dtype=np.int32)
    n_units = lib.or_plan(_ptr(sl), B, num_kv_heads, max_seq_len, S, _ptr(nsplit), _ptr(off))
    return nsplit, off, int(n_units)


def flat_gemm(x, w, entries=None, dtype=BF16, n_threads=0):
    """C = x W^T in float64 on the widened inputs (oracle.c, R10).

    x: [M][K], w: [N][K], uint16 bf16 bit patterns (dtype BF16) or float32 (dtype F32).
    entries: None for the whole [M][N] product, or an int array of (m, n) pairs, giving
    float64 [len(entries)]."""
    lib = _load()
    x = _kv_array(x, dtype)
    w = _kv_array(w, dtype)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"shapes {x.shape} and {w.shape} do not make x W^T")
    M, K = x.shape
    N = w.shape[0]
    if entries is None:
        out = np.empty((M, N), np.float64)
        e, ne = None, 0
    else:
        e = np.ascontiguousarray(np.asarray(entries, np.int32).reshape(-1, 2))
        ne = e.shape[0]
        out = np.empty(ne, np.float64)
    used = lib.or_flat_gemm(M, N, K, dtype, _ptr(x), _ptr(w), _ptr(e), ne, _ptr(out), n_threads)
    if used < 0:
        raise ValueError("or_flat_gemm rejected its arguments")
    return out
