"""Pins for the oracle's attention: brute force and special cases with known answers."""
import numpy as np
import pytest

from oracle.attention import attention_bruteforce, attention_fp64


def test_matches_bruteforce_triple_loop():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 2, 4))
    k = rng.standard_normal((5, 2, 4))
    v = rng.standard_normal((5, 2, 4))
    got = attention_fp64(q, k, v)
    want = np.array(attention_bruteforce(q.tolist(), k.tolist(), v.tolist()))
    assert np.max(np.abs(got - want)) < 1e-13


def test_one_key_returns_its_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 3, 8)) * 10
    k = rng.standard_normal((1, 3, 8))
    v = rng.standard_normal((1, 3, 8))
    assert np.allclose(attention_fp64(q, k, v), np.broadcast_to(v, (4, 3, 8)), rtol=0, atol=1e-14)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 2, 8))
    k = np.broadcast_to(rng.standard_normal((1, 2, 8)), (7, 2, 8))
    v = rng.standard_normal((7, 2, 8))
    assert np.allclose(attention_fp64(q, k, v), v.mean(axis=0, keepdims=True), atol=1e-14)


def test_dominant_logit_selects_value():
    d = 16
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 100.0
    k = np.zeros((5, 1, d)); k[3, 0, 0] = 100.0       # logit 10000/4 for key 3, 0 for the rest
    v = np.arange(5 * d, dtype=np.float64).reshape(5, 1, d)
    assert np.allclose(attention_fp64(q, k, v)[0, 0], v[3, 0], atol=1e-12)


def test_scale_is_one_over_sqrt_d():
    # two keys with logits a and 0 (before scaling): weight of key 0 = sigmoid(a / sqrt(d))
    d = 64
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, d)); k[0, 0, 0] = 3.0
    v = np.zeros((2, 1, d)); v[0, 0, 1] = 1.0
    w = 1.0 / (1.0 + np.exp(-3.0 / np.sqrt(d)))
    assert abs(attention_fp64(q, k, v)[0, 0, 1] - w) < 1e-15


def test_rows_are_convex_combinations_and_key_order_free():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((6, 2, 8)) * 3
    k = rng.standard_normal((11, 2, 8))
    v = np.ones((11, 2, 8))
    assert np.allclose(attention_fp64(q, k, v), 1.0, atol=1e-14)     # rows of P sum to 1
    v = rng.standard_normal((11, 2, 8))
    perm = rng.permutation(11)
    a = attention_fp64(q, k, v)
    b = attention_fp64(q, k[perm], v[perm])
    assert np.max(np.abs(a - b)) < 1e-13


@pytest.mark.parametrize("shape", [(3, 5), (5, 3)])
def test_operands_not_transposed(shape):
    # different T, N and heads with different data catch a swapped head or operand
    T, N = shape
    rng = np.random.default_rng(4)
    q = rng.standard_normal((T, 3, 4))
    k = rng.standard_normal((N, 3, 4))
    v = rng.standard_normal((N, 3, 4))
    got = attention_fp64(q, k, v)
    want = np.array(attention_bruteforce(q.tolist(), k.tolist(), v.tolist()))
    assert got.shape == (T, 3, 4)
    assert np.max(np.abs(got - want)) < 1e-13
