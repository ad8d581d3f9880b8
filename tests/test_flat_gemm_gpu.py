"""Flat GEMM (y = x W^T, a decode-time linear layer) on the GPU against the fp64 oracle.

Source: opt.ai.kr "FlashDecoding++ async softmax -- theory", s2 (2) and s4. The kernel pads M only
to the next multiple of 16 and splits K across the CTAs of a cluster when the weight tiles are too
few; these cases
cover single and split K, ragged M, N and K (tails inside a 128-row tile, a 64-wide K slice and a
16-row MMA column block), and every layer shape of the bench at its full size (sampled entries).

Tolerance, from the arithmetic: products of bf16 are exact in fp32; the fp32 sum adds at most a
few units of 2^-24 per term of sum_k |x_k w_k| (bounded here by 2^-14 of it), and rounding the
result to bf16 adds at most 2^-9 of |y| (bounded by 2^-8).
"""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import split_kv_async_gb300 as F


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _host(t):
    return W.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _bound(x, w, ref, entries=None):
    xa = np.abs(W.bf16_bits_to_f32(x).astype(np.float64))
    wa = np.abs(W.bf16_bits_to_f32(w).astype(np.float64))
    if entries is None:
        s = xa @ wa.T
    else:
        s = np.array([xa[m] @ wa[n] for m, n in entries])
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * s


def _run(x, w, split_k=0):
    M, K = x.shape
    N = w.shape[0]
    ws = F.alloc_flat_gemm_workspace(M, N, K, split_k)
    xd, wd = _dev(x), _dev(w)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    F.fdpp_flat_gemm(xd, wd, y, ws, split_k=split_k)
    torch.cuda.synchronize()
    assert F.fdpp_flat_gemm_read_error(ws) == 0
    return y, ws, (xd, wd)


def _inputs(M, N, K, seed):
    return W.gemm_inputs(W.GemmWorkload("t", M, N, K, seed))


SMALL = [
    # M, N, K, split_k
    (1, 128, 64, 1),       # one tile, one slice
    (5, 200, 72, 1),       # ragged N (two tiles) and K (a slice of 8)
    (3, 130, 8, 1),        # K smaller than a slice
    (16, 384, 512, 3),     # split K, full 16-row column block
    (17, 256, 320, 2),     # M one past a 16-row block
    (33, 1000, 1000, 0),   # automatic split, ragged everything
    (64, 512, 2048, 0),
    (40, 130, 4096, 8),    # the largest split, N not a multiple of 4
    (128, 256, 256, 2),    # the largest M
    (8, 4096, 4096, 0),
]


@pytest.mark.parametrize("M,N,K,split_k", SMALL)
def test_matches_oracle(M, N, K, split_k):
    x, w = _inputs(M, N, K, seed=1000 + M + N + K)
    y, _, _ = _run(x, w, split_k)
    ref = oracle.flat_gemm(x, w)
    got = _host(y)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= _bound(x, w, ref)), f"max err {err.max():.3e}"


@pytest.mark.parametrize("split_k", [1, 2, 5, 8])
def test_split_k_gives_the_same_product(split_k):
    x, w = _inputs(8, 640, 1024, seed=77)
    y, _, _ = _run(x, w, split_k)
    ref = oracle.flat_gemm(x, w)
    assert np.all(np.abs(_host(y) - ref) <= _bound(x, w, ref))


def test_repeated_calls_are_bitwise_equal():
    x, w = _inputs(24, 1536, 2048, seed=5)
    M, K = x.shape
    N = w.shape[0]
    split = F.fdpp_flat_gemm_split_k(M, N, K, 0)
    assert split > 1
    ws = F.alloc_flat_gemm_workspace(M, N, K)
    xd, wd = _dev(x), _dev(w)
    ys = []
    for _ in range(3):
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        F.fdpp_flat_gemm(xd, wd, y, ws)
        ys.append(y)
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_lookup_table_sets_the_split():
    M, N, K = 8, 1024, 2048
    try:
        F.fdpp_flat_gemm_set_lut([(16, N, K, 4), (64, N, K, 2)])
        assert F.fdpp_flat_gemm_split_k(M, N, K) == 4
        assert F.fdpp_flat_gemm_split_k(40, N, K) == 2
        x, w = _inputs(M, N, K, seed=9)
        y, _, _ = _run(x, w, 0)
        ref = oracle.flat_gemm(x, w)
        assert np.all(np.abs(_host(y) - ref) <= _bound(x, w, ref))
    finally:
        F.fdpp_flat_gemm_set_lut([])


@pytest.mark.parametrize("name", sorted(W.GEMM))
def test_layer_shapes_at_full_size(name):
    wl = W.GEMM[name]
    x, w = W.gemm_inputs(wl)
    y, _, _ = _run(x, w, 0)
    got = _host(y)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(wl.seed)
    ent = [(int(m), int(n)) for m, n in zip(rng.integers(0, wl.M, 400), rng.integers(0, wl.N, 400))]
    # tile edges and the last row and column
    ent += [(0, 127), (wl.M - 1, 128), (wl.M - 1, wl.N - 1), (wl.M // 2, wl.N - 129)]
    ref = oracle.flat_gemm(x, w, entries=ent)
    g = np.array([got[m, n] for m, n in ent])
    assert np.all(np.abs(g - ref) <= _bound(x, w, ref, ent))


def test_chained_layers_read_the_previous_output():
    # y1 = x W1^T, y2 = y1 W2^T back to back on one stream: the second call starts streaming W2
    # while the first finishes, and must read y1 only after the first call has written it
    x, w1 = _inputs(8, 1024, 2048, seed=21)
    _, w2 = _inputs(8, 3072, 1024, seed=22)
    ws1 = F.alloc_flat_gemm_workspace(8, 1024, 2048)
    ws2 = F.alloc_flat_gemm_workspace(8, 3072, 1024)
    xd, w1d, w2d = _dev(x), _dev(w1), _dev(w2)
    y1 = torch.empty((8, 1024), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((8, 3072), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        y1.fill_(float("nan"))
        y2.fill_(float("nan"))
        F.fdpp_flat_gemm(xd, w1d, y1, ws1)
        F.fdpp_flat_gemm(y1, w2d, y2, ws2)
    torch.cuda.synchronize()
    y1_bits = y1.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.flat_gemm(y1_bits, w2)
    assert np.all(np.abs(_host(y2) - ref) <= _bound(y1_bits, w2, ref))
    ref1 = oracle.flat_gemm(x, w1)
    assert np.all(np.abs(_host(y1) - ref1) <= _bound(x, w1, ref1))
