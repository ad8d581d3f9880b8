"""Pins of the oracle's flat GEMM (a decode-time linear layer, y = x W^T) against plain facts.

Source: opt.ai.kr "FlashDecoding++ async softmax -- theory" s2 (2) and s4: in decoding, the linear
layers' matrices are flat (M, the number of query tokens, is very small) while the weight N x K is
fixed. The pages give no worked example, so every pin here is a closed form, a special case with a
known answer, or a relation between two differently-shaped products. Together they catch a
transposed operand, a swapped (m, n), a dropped or extra term of the k sum, and a wrong sign.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def _bf16(a):
    return W.f32_to_bf16_bits(np.asarray(a, np.float32))


def _widen(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def test_two_by_two_by_hand():
    # [[1, 2], [3, 4]] times the transpose of [[5, 6], [7, 8]]: rows of x against rows of W
    got = oracle.flat_gemm(_bf16([[1, 2], [3, 4]]), _bf16([[5, 6], [7, 8]]))
    assert got.tolist() == [[17.0, 23.0], [39.0, 53.0]]


def test_fp32_inputs_take_the_same_definition():
    got = oracle.flat_gemm(np.array([[1, 2], [3, 4]], np.float32),
                           np.array([[5, 6], [7, 8]], np.float32), dtype=oracle.F32)
    assert got.tolist() == [[17.0, 23.0], [39.0, 53.0]]


def test_identity_weight_returns_the_activations():
    rng = np.random.default_rng(7)
    K = 48
    x = _bf16(rng.standard_normal((5, K)))
    got = oracle.flat_gemm(x, _bf16(np.eye(K)))
    assert np.array_equal(got, _widen(x))


def test_one_hot_rows_select_weight_columns():
    rng = np.random.default_rng(8)
    M, N, K = 6, 9, 40
    w = _bf16(rng.standard_normal((N, K)))
    cols = [3, 0, 39, 17, 17, 5]
    x = np.zeros((M, K), np.float32)
    for m, k in enumerate(cols):
        x[m, k] = 1.0
    got = oracle.flat_gemm(_bf16(x), w)
    assert np.array_equal(got, _widen(w)[:, cols].T)


def test_integer_closed_form_with_an_odd_k():
    # x[m][k] = m + 1, W[n][k] = n - 3: C[m][n] = (m + 1)(n - 3) K, exact in bf16 and double
    M, N, K = 4, 7, 37
    x = np.repeat(np.arange(1, M + 1, dtype=np.float32)[:, None], K, axis=1)
    w = np.repeat(np.arange(-3, N - 3, dtype=np.float32)[:, None], K, axis=1)
    got = oracle.flat_gemm(_bf16(x), _bf16(w))
    want = np.outer(np.arange(1, M + 1), np.arange(-3, N - 3)).astype(np.float64) * K
    assert np.array_equal(got, want)


def test_swapping_the_operands_transposes_the_product():
    rng = np.random.default_rng(9)
    x = _bf16(rng.standard_normal((3, 64)))
    w = _bf16(rng.standard_normal((11, 64)))
    assert np.array_equal(oracle.flat_gemm(x, w), oracle.flat_gemm(w, x).T)


def test_stacked_weights_repeat_the_columns():
    rng = np.random.default_rng(10)
    x = _bf16(rng.standard_normal((4, 32)))
    w = _bf16(rng.standard_normal((6, 32)))
    one = oracle.flat_gemm(x, w)
    two = oracle.flat_gemm(x, np.concatenate([w, w]))
    assert np.array_equal(two, np.concatenate([one, one], axis=1))


def test_entries_are_the_product_at_those_places():
    rng = np.random.default_rng(11)
    x = _bf16(rng.standard_normal((5, 96)))
    w = _bf16(rng.standard_normal((13, 96)))
    full = oracle.flat_gemm(x, w)
    ent = [(0, 0), (4, 12), (2, 7), (4, 0)]
    got = oracle.flat_gemm(x, w, entries=ent)
    assert np.array_equal(got, np.array([full[m, n] for m, n in ent]))


def test_bad_shapes_and_entries_are_rejected():
    x = _bf16(np.ones((2, 8)))
    with pytest.raises(ValueError):
        oracle.flat_gemm(x, _bf16(np.ones((3, 9))))
    with pytest.raises(ValueError):
        oracle.flat_gemm(x, _bf16(np.ones((3, 8))), entries=[(2, 0)])
