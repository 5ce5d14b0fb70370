"""Pins of the oracle's variable-length (packed) batch: every sequence is its
own attention problem ("Flash Attention (4)" §5; "Lecture 25" §7.2 item 2)."""
import math

import numpy as np
import pytest

import oracle


def _brute_row(q, k, v, i, Nq, Nk, causal, scale):
    s = scale * (k @ q)
    if causal:
        s = np.where(np.arange(Nk) <= i + Nk - Nq, s, -np.inf)
    if not np.isfinite(s).any():
        return np.zeros(v.shape[1]), -np.inf
    m = s.max()
    p = np.exp(s - m)
    return p @ v / p.sum(), m + math.log(p.sum())


@pytest.mark.parametrize("causal", [False, True])
def test_against_brute_force_with_empty_and_keyless_sequences(causal):
    g = np.random.default_rng(7)
    cu_q = [0, 3, 3, 8, 9]      # lengths 3, 0, 5, 1
    cu_k = [0, 4, 6, 6, 11]     # lengths 4, 2, 0, 5
    H, H_kv, d = 4, 2, 6
    q = g.standard_normal((cu_q[-1], H, d))
    k = g.standard_normal((cu_k[-1], H_kv, d))
    v = g.standard_normal((cu_k[-1], H_kv, d))
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal, 0.4)
    for s in range(len(cu_q) - 1):
        Nq, Nk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        for i in range(Nq):
            for h in range(H):
                t = cu_q[s] + i
                ob, lb = _brute_row(q[t, h], k[cu_k[s]:cu_k[s + 1], h // 2], v[cu_k[s]:cu_k[s + 1], h // 2],
                                    i, Nq, Nk, causal, 0.4)
                np.testing.assert_allclose(o[t, h], ob, rtol=0, atol=1e-12)
                assert (lse[h, t] == lb) if np.isinf(lb) else abs(lse[h, t] - lb) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_are_a_dense_batch(causal):
    g = np.random.default_rng(8)
    B, H, N, d = 3, 2, 7, 4
    q, k, v = (g.standard_normal((B, H, N, d)) for _ in range(3))
    o_dense, l_dense = oracle.attention(q, k, v, causal, 0.3)
    pack = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(B * N, H, d))
    cu = [b * N for b in range(B + 1)]
    o, lse = oracle.attention_varlen(pack(q), pack(k), pack(v), cu, cu, causal, 0.3)
    np.testing.assert_allclose(o, pack(o_dense), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l_dense.transpose(1, 0, 2).reshape(H, B * N), rtol=0, atol=1e-12)


def test_a_sequence_never_sees_its_neighbours():
    g = np.random.default_rng(9)
    cu = [0, 5, 12, 20]
    q, k, v = (g.standard_normal((20, 2, 4)) for _ in range(3))
    o1, l1 = oracle.attention_varlen(q, k, v, cu, cu, False, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[:5] *= 2.0  # adding one constant vector to every key would cancel in the softmax
    v2[12:] *= -2.0
    o2, l2 = oracle.attention_varlen(q, k2, v2, cu, cu, False, 0.5)
    np.testing.assert_array_equal(o1[5:12], o2[5:12])   # the middle sequence is untouched
    np.testing.assert_array_equal(l1[:, 5:12], l2[:, 5:12])
    assert np.abs(o1[:5] - o2[:5]).max() > 1e-3 and np.abs(o1[12:] - o2[12:]).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_equal_lengths_are_a_dense_batch(causal):
    g = np.random.default_rng(21)
    B, H, N, d = 3, 2, 7, 4
    q, k, v, G = (g.standard_normal((B, H, N, d)) for _ in range(4))
    dense = oracle.attention_bwd(q.reshape(B * H, N, d), k.reshape(B * H, N, d), v.reshape(B * H, N, d),
                                 G.reshape(B * H, N, d), causal, 0.3)
    pack = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(B * N, H, d))
    cu = [b * N for b in range(B + 1)]
    got = oracle.attention_bwd_varlen(pack(q), pack(k), pack(v), pack(G), cu, cu, causal, 0.3)
    for x, y in zip(got, dense):
        np.testing.assert_allclose(x, pack(y.reshape(B, H, N, d)), rtol=0, atol=1e-12)


def test_bwd_varlen_finite_differences_with_an_empty_and_a_keyless_sequence():
    """Central differences of L = sum(O * G) through oracle.attention_varlen."""
    g = np.random.default_rng(22)
    cu_q = [0, 3, 3, 6]      # lengths 3, 0, 3
    cu_k = [0, 4, 6, 6]      # lengths 4, 2, 0 (the third sequence's rows see no key)
    H, H_kv, d = 2, 1, 3
    q = g.standard_normal((cu_q[-1], H, d))
    k = g.standard_normal((cu_k[-1], H_kv, d))
    v = g.standard_normal((cu_k[-1], H_kv, d))
    G = g.standard_normal((cu_q[-1], H, d))
    for causal in (False, True):
        got = oracle.attention_bwd_varlen(q, k, v, G, cu_q, cu_k, causal, 0.7)
        for x, gx in zip((q, k, v), got):
            fd = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                old = x[idx]
                x[idx] = old + 1e-6
                op, _ = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal, 0.7)
                x[idx] = old - 1e-6
                om, _ = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal, 0.7)
                x[idx] = old
                fd[idx] = ((op - om) * G).sum() / 2e-6
            np.testing.assert_allclose(gx, fd, rtol=0, atol=1e-8)
