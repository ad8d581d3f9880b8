"""Seeded synthetic decode-attention workloads (and the decode-time linear layers' GEMMs).

This module only builds inputs: shapes, seeded random draws, bf16 rounding and cache layout. It
holds none of the attention arithmetic, and both the CUDA path (through its tests and the bench)
and the CPU oracle read the inputs it produces.

Workloads follow the problem statement of opt.ai.kr "FlashDecoding++ async softmax -- theory",
section 1: one query token per sequence against a long K/V cache. The shapes below are the five
decode workloads this library is measured on (tiny MHA, GQA decode, long context, paged
continuous batch, fallback stress).

Recipe:
  * every array has its own numpy ``Generator(PCG64)`` seeded with ``[seed, stream_id]``, so
    changing one array's size does not shift another array's draws;
  * values are float32 standard normals; bf16 inputs are the float32 draws rounded to nearest
    even (ties to even) into bf16;
  * ``seq_lens`` are fixed, or uniform integers in [lo, hi] (inclusive);
  * contiguous caches are [B][Lmax][Hkv][d] with Lmax = max seq_len;
  * paged caches are one pool [num_blocks][block_size][Hkv][d] holding exactly
    sum_b ceil(L_b / block_size) blocks; the block table maps each sequence's logical blocks to
    a seeded random permutation of the pool; unused table entries are -1;
  * ``poison_tail`` writes NaN into every cache slot at or past L_b (masking tests);
  * the fallback-stress workload replaces, in round(frac * units) seeded splits, one key at a
    seeded position by k = 12 * q_h0 / ||q_h0|| * sqrt(d) (h0 = first query head of the kv
    group, computed in float32 from the rounded query, then rounded to bf16), so that head's
    score is about 12 ||q|| and far above phi + 10.
  * ``score_shift`` > 0 moves each query head's scores to its own level: per kv head g a seeded
    unit direction u_g, per query head h a seeded level mu_h uniform in [0, score_shift]; the keys
    of kv head g gain a * u_g and query h gains (mu_h sqrt(d) / a) * u_g, a = sqrt(score_shift
    sqrt(d)) (float32, then rounded to bf16), so that head h's scaled scores centre near mu_h.
    Heads then need a unified max of their own (tests of per-head phi and of its calibration).
    The levels and directions come from ``shift_seed`` alone, like a property of the model's
    weights, so samples drawn with other seeds share them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32, BF16 = "f32", "bf16"
_CHUNK = 1 << 24

# stream ids of the per-array generators
_S_SEQ, _S_Q, _S_K, _S_V, _S_PERM, _S_STRESS, _S_SHIFT = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str
    split_len: int
    seq_len: Optional[int] = None              # fixed length for every sequence
    seq_len_range: Optional[tuple] = None      # (lo, hi) inclusive, uniform
    paged: bool = False
    block_size: int = 16
    phi: float = 0.0
    lo: float = -30.0
    hi: float = 10.0
    stress_frac: float = 0.0
    score_shift: float = 0.0                   # > 0: per-head score levels in [0, score_shift]
    q_tokens: int = 1                          # query tokens per sequence (the last positions)
    shift_seed: int = 0x5EED00FF               # the levels and directions (fixed across samples)
    seed: int = 0x5EED0000

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five decode workloads, in order (seed = 0x5EED0000 + index).
TINY = Workload("tiny", 1, 4, 4, 64, F32, split_len=64, seq_len=256, seed=0x5EED0000)
GQA = Workload("gqa_decode", 8, 32, 8, 128, BF16, split_len=512, seq_len=4096, seed=0x5EED0001)
LONG = Workload("long_context", 1, 32, 8, 128, BF16, split_len=1024, seq_len=131072,
                seed=0x5EED0002)
PAGED = Workload("paged_batch", 64, 64, 8, 128, BF16, split_len=512, seq_len_range=(512, 16384),
                 paged=True, block_size=16, seed=0x5EED0003)
STRESS = Workload("fallback_stress", 8, 32, 8, 128, BF16, split_len=512, seq_len=4096,
                  stress_frac=0.02, seed=0x5EED0004)
# GQA decode shapes whose query heads score at their own levels in [0, 30]: one scalar phi sends
# most splits to the fallback; phi chosen per head from a sample keeps them on the fast path.
SHIFTED = Workload("gqa_head_levels", 8, 32, 8, 128, BF16, split_len=512, seq_len=4096,
                   score_shift=30.0, seed=0x5EED0005)
# A speculative-decoding step on gqa_decode shapes: two query tokens per sequence (the last two
# positions, causal), 8 query rows per kv head.
SPEC = Workload("spec_decode_tq2", 8, 32, 8, 128, BF16, split_len=512, seq_len=4096, q_tokens=2,
                seed=0x5EED0006)
# A 16-token prefill chunk against gqa_decode's caches: 64 query rows per kv head, one unit of
# the tensor kernel's tcgen05 build.
CHUNK = Workload("prefill_chunk_tq16", 8, 32, 8, 128, BF16, split_len=512, seq_len=4096, q_tokens=16,
                 seed=0x5EED0007)
ALL = {w.name: w for w in (TINY, GQA, LONG, PAGED, STRESS, SHIFTED, SPEC, CHUNK)}


@dataclasses.dataclass(frozen=True)
class GemmWorkload:
    """A decode-time linear layer y = x W^T: x [M][K] activations, W [N][K] weight, both bf16
    standard normals (W scaled by 1/sqrt(K), as an initialised layer's weight)."""
    name: str
    M: int
    N: int
    K: int
    seed: int

    def replace(self, **kw) -> "GemmWorkload":
        return dataclasses.replace(self, **kw)


# The four linear layers of a decoder block with the attention workloads' geometry (hidden
# 4096 = 32 query heads x 128, 8 kv heads, FFN width 14336 with gate and up fused), at the batch of
# gqa_decode (M = 8) and of paged_batch (M = 64).
_LAYERS = (("qkv", 6144, 4096), ("o_proj", 4096, 4096), ("gate_up", 28672, 4096),
           ("down", 4096, 14336))
GEMM = {f"gemm_{n}_m{m}": GemmWorkload(f"gemm_{n}_m{m}", m, N, K, seed=0x5EEDA000 + 16 * i + m)
        for i, (n, N, K) in enumerate(_LAYERS) for m in (8, 64)}

_S_GX, _S_GW = 11, 12


def gemm_inputs(wl: GemmWorkload):
    """(x, w) as uint16 bf16 bit patterns, [M][K] and [N][K]."""
    x = _normals(_rng(wl.seed, _S_GX), wl.M * wl.K, BF16).reshape(wl.M, wl.K)
    rng = _rng(wl.seed, _S_GW)
    scale = np.float32(1.0 / math.sqrt(wl.K))
    w = np.empty(wl.N * wl.K, np.uint16)
    for i in range(0, w.size, _CHUNK):
        n = min(_CHUNK, w.size - i)
        w[i:i + n] = f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32) * scale)
    return x, w.reshape(wl.N, wl.K)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed & 0xFFFFFFFFFFFFFFFF, stream]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _normals(rng: np.random.Generator, n: int, dtype: str) -> np.ndarray:
    """n standard normals, as float32 (F32) or bf16 bit patterns (BF16), drawn in chunks."""
    out = np.empty(n, dtype=np.float32 if dtype == F32 else np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32)
        out[s:e] = x if dtype == F32 else f32_to_bf16_bits(x)
    return out


@dataclasses.dataclass
class Inputs:
    """Host arrays of one workload instance (bf16 as uint16 bit patterns)."""
    wl: Workload
    seq_lens: np.ndarray            # int32 [B]
    q: np.ndarray                   # [B][Hq][d], or [B][Tq][Hq][d] for several query tokens
    k: np.ndarray                   # contiguous [B][Lmax][Hkv][d] or paged [N][bs][Hkv][d]
    v: np.ndarray
    block_table: Optional[np.ndarray]   # int32 [B][max_blocks_per_seq] or None
    max_seq_len: int
    max_blocks_per_seq: int
    num_kv_blocks: int
    hot: list                       # stress injections: (b, g, j, t)

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes of one step: only tokens t < L_b, every kv head, K and V."""
        es = 4 if self.wl.dtype == F32 else 2
        return int(self.seq_lens.astype(np.int64).sum()) * self.wl.num_kv_heads * \
            self.wl.head_dim * 2 * es


def make_seq_lens(wl: Workload) -> np.ndarray:
    if wl.seq_len is not None:
        return np.full(wl.batch, wl.seq_len, dtype=np.int32)
    lo, hi = wl.seq_len_range
    return _rng(wl.seed, _S_SEQ).integers(lo, hi + 1, size=wl.batch).astype(np.int32)


def generate(wl: Workload, *, seq_lens: Optional[np.ndarray] = None, poison_tail: bool = False,
             max_blocks_per_seq: Optional[int] = None) -> Inputs:
    """Build one seeded instance of `wl` on the host."""
    B, Hq, Hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    sl = make_seq_lens(wl) if seq_lens is None else np.asarray(seq_lens, dtype=np.int32)
    assert sl.shape == (B,)
    Lmax = max(1, int(sl.max()))
    Tq = max(1, wl.q_tokens)
    q = _normals(_rng(wl.seed, _S_Q), B * Tq * Hq * d, wl.dtype)
    q = q.reshape(B, Hq, d) if Tq == 1 else q.reshape(B, Tq, Hq, d)
    nan_val = np.float32(np.nan) if wl.dtype == F32 else np.uint16(0x7FC0)

    table = None
    nblk_total = 0
    mbps = 0
    if not wl.paged:
        shape = (B, Lmax, Hkv, d)
        k = _normals(_rng(wl.seed, _S_K), int(np.prod(shape)), wl.dtype).reshape(shape)
        v = _normals(_rng(wl.seed, _S_V), int(np.prod(shape)), wl.dtype).reshape(shape)
        if poison_tail:
            for b in range(B):
                k[b, sl[b]:] = nan_val
                v[b, sl[b]:] = nan_val
    else:
        bs = wl.block_size
        nblk = [(int(L) + bs - 1) // bs for L in sl]
        nblk_total = max(1, sum(nblk))
        mbps = max(nblk) if max_blocks_per_seq is None else max_blocks_per_seq
        mbps = max(mbps, 1)
        perm = _rng(wl.seed, _S_PERM).permutation(nblk_total).astype(np.int32)
        table = np.full((B, mbps), -1, dtype=np.int32)
        pos = 0
        for b in range(B):
            table[b, :nblk[b]] = perm[pos:pos + nblk[b]]
            pos += nblk[b]
        shape = (nblk_total, bs, Hkv, d)
        k = _normals(_rng(wl.seed, _S_K), int(np.prod(shape)), wl.dtype).reshape(shape)
        v = _normals(_rng(wl.seed, _S_V), int(np.prod(shape)), wl.dtype).reshape(shape)
        if poison_tail:
            for b in range(B):
                L = int(sl[b])
                if L % bs and nblk[b]:
                    last = table[b, nblk[b] - 1]
                    k[last, L % bs:] = nan_val
                    v[last, L % bs:] = nan_val

    if wl.score_shift > 0:
        _shift_scores(wl, q, k)
    hot = []
    if wl.stress_frac > 0:
        hot = _inject_hot_keys(wl, sl, q, k, table)
    return Inputs(wl, sl, q, k, v, table, Lmax, mbps, nblk_total, hot)


def _shift_scores(wl, q, k):
    """Per-head score levels (see the module docstring), in place."""
    rng = _rng(wl.shift_seed, _S_SHIFT)
    Hkv, G, d = wl.num_kv_heads, wl.group, wl.head_dim
    u = rng.standard_normal((Hkv, d)).astype(np.float32)
    u /= np.linalg.norm(u, axis=1, keepdims=True).astype(np.float32)
    mu = rng.uniform(0.0, wl.score_shift, size=wl.num_q_heads).astype(np.float32)
    a = np.float32(math.sqrt(wl.score_shift * math.sqrt(d)))

    def widen(x):
        return x if wl.dtype == F32 else bf16_bits_to_f32(x)

    def narrow(x):
        return x.astype(np.float32) if wl.dtype == F32 else f32_to_bf16_bits(x)

    for g in range(Hkv):
        kg = widen(k[..., g, :]) + a * u[g]
        k[..., g, :] = narrow(kg)
        for h in range(g * G, (g + 1) * G):
            qh = widen(q[..., h, :]) + (mu[h] * np.float32(math.sqrt(d)) / a) * u[g]
            q[..., h, :] = narrow(qh)


def _inject_hot_keys(wl, sl, q, k, table):
    """Replace one key in round(frac * units) seeded splits (see the module docstring)."""
    rng = _rng(wl.seed, _S_STRESS)
    S, G, d = wl.split_len, wl.group, wl.head_dim
    units = [(b, g, j) for b in range(wl.batch) for g in range(wl.num_kv_heads)
             for j in range((int(sl[b]) + S - 1) // S)]
    n_hot = int(round(wl.stress_frac * len(units)))
    order = rng.permutation(len(units))
    hot = []
    for u in order[:n_hot]:
        b, g, j = units[int(u)]
        t0, t1 = j * S, min((j + 1) * S, int(sl[b]))
        t = int(rng.integers(t0, t1))
        h0 = g * G
        qrow = q[b, h0] if q.ndim == 3 else q[b, 0, h0]     # several query tokens: the first
        qv = qrow.astype(np.float32) if wl.dtype == F32 else bf16_bits_to_f32(qrow)
        kv = (np.float32(12.0) * qv / np.float32(np.linalg.norm(qv))
              * np.float32(math.sqrt(d))).astype(np.float32)
        row = kv if wl.dtype == F32 else f32_to_bf16_bits(kv)
        if table is None:
            k[b, t, g] = row
        else:
            bs = wl.block_size
            k[table[b, t // bs], t % bs, g] = row
        hot.append((b, g, j, t))
    return hot


def to_float(a: np.ndarray, dtype: str) -> np.ndarray:
    """View helper: bf16 bit patterns -> float32 values (F32 arrays returned as float32)."""
    return a.astype(np.float32) if dtype == F32 else bf16_bits_to_f32(a)
