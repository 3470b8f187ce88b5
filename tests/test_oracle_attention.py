"""Pins for the oracle's decode attention, split/combine and sparse restriction (no GPU)."""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle.attention import page_token_indices


def brute_force(q, k, v, sm_scale):
    """Pure-Python softmax attention without max subtraction (tiny inputs only)."""
    n, d = len(k), len(q)
    e = [math.exp(sm_scale * sum(q[i] * k[t][i] for i in range(d))) for t in range(n)]
    z = sum(e)
    return [sum(e[t] * v[t][i] for t in range(n)) / z for i in range(d)]


@pytest.mark.parametrize("n,d", [(1, 4), (2, 3), (5, 8), (8, 2)])
def test_brute_force_tiny(n, d):
    rng = np.random.default_rng(100 + n * 10 + d)
    q = rng.standard_normal(d)
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    got = oracle.decode_attention_tokens(q, k, v, 0.37)
    want = brute_force(q.tolist(), k.tolist(), v.tolist(), 0.37)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_one_token_returns_its_value():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((1, 16))
    got = oracle.decode_attention_tokens(rng.standard_normal(16), rng.standard_normal((1, 16)), v, 0.25)
    assert np.array_equal(got, v[0])


def test_uniform_values_and_zero_query():
    rng = np.random.default_rng(2)
    k = rng.standard_normal((40, 8))
    v = np.tile(np.arange(8.0), (40, 1))
    assert np.allclose(oracle.decode_attention_tokens(rng.standard_normal(8), k, v, 1.0), np.arange(8.0))
    v2 = rng.standard_normal((40, 8))
    assert np.allclose(oracle.decode_attention_tokens(np.zeros(8), k, v2, 1.0), v2.mean(axis=0), atol=1e-14)


def test_two_token_closed_form():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal(6), rng.standard_normal((2, 6)), rng.standard_normal((2, 6))
    delta = 0.5 * (q @ k[0] - q @ k[1])
    w0 = 1.0 / (1.0 + math.exp(-delta))
    want = w0 * v[0] + (1 - w0) * v[1]
    assert np.allclose(oracle.decode_attention_tokens(q, k, v, 0.5), want, atol=1e-14)


def test_dominant_token():
    k = np.eye(4) * 50.0
    v = np.arange(16.0).reshape(4, 4)
    q = np.array([0.0, 0.0, 1.0, 0.0])
    assert np.allclose(oracle.decode_attention_tokens(q, k, v, 1.0), v[2], atol=1e-12)


def test_token_permutation_invariance():
    # the physical order of tokens (pages) does not change the result
    rng = np.random.default_rng(4)
    k, v, q = rng.standard_normal((33, 16)), rng.standard_normal((33, 16)), rng.standard_normal(16)
    p = rng.permutation(33)
    a = oracle.decode_attention_tokens(q, k, v, 0.25)
    b = oracle.decode_attention_tokens(q, k[p], v[p], 0.25)
    assert np.allclose(a, b, atol=1e-14)


def test_gqa_head_mapping():
    # kv head g holds constant values g; query head h must read kv head h // G
    Hq, Hkv, L, d = 8, 2, 5, 4
    rng = np.random.default_rng(6)
    k = rng.standard_normal((L, Hkv, d))
    v = np.zeros((L, Hkv, d))
    for g in range(Hkv):
        v[:, g, :] = g + 1
    out = oracle.decode_attention(rng.standard_normal((Hq, d)), k, v, 0.5)
    for h in range(Hq):
        assert np.allclose(out[h], h // (Hq // Hkv) + 1)


def test_empty_sequence_gives_zeros():
    out = oracle.decode_attention(np.ones((2, 4)), np.zeros((0, 2, 4)), np.zeros((0, 2, 4)), 1.0)
    assert (out == 0).all()


@pytest.mark.parametrize("bounds", [[0, 100], [0, 1, 100], [0, 0, 37, 37, 99, 100], [0, 10, 20, 30, 100]])
def test_split_combine_identity(bounds):
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal(32), rng.standard_normal((100, 32)) * 3, rng.standard_normal((100, 32))
    parts = oracle.split_partials(q, k, v, 0.2, bounds)
    got = oracle.combine_partials(parts)
    want = oracle.decode_attention_tokens(q, k, v, 0.2)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_sparse_with_all_pages_equals_dense():
    rng = np.random.default_rng(10)
    L, Hkv, Hq, d, ps = 75, 2, 4, 8, 16
    k, v = rng.standard_normal((L, Hkv, d)), rng.standard_normal((L, Hkv, d))
    q = rng.standard_normal((Hq, d))
    P = -(-L // ps)
    dense = oracle.decode_attention(q, k, v, 0.3)
    sparse = oracle.sparse_decode_attention(q, k, v, 0.3, [list(range(P))] * Hq, ps)
    assert np.array_equal(dense, sparse)


def test_sparse_restricts_tokens():
    rng = np.random.default_rng(12)
    L, d, ps = 64, 4, 16
    k, v = rng.standard_normal((L, 1, d)), rng.standard_normal((L, 1, d))
    q = rng.standard_normal((1, d))
    got = oracle.sparse_decode_attention(q, k, v, 0.5, [[1, 3]], ps)
    t = list(range(16, 32)) + list(range(48, 64))
    want = brute_force(q[0].tolist(), k[t, 0].tolist(), v[t, 0].tolist(), 0.5)
    assert np.allclose(got[0], want, atol=1e-12)
    assert page_token_indices([3], 16, 50).tolist() == [48, 49]
