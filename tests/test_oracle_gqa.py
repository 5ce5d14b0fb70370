"""Pins of the oracle's grouped-query attention (head mapping) against closed
forms and independent computations ("Flash Attention (4)" §5: the K/V index of
query head h is mapped to its group, h // (H // H_kv))."""
import math

import numpy as np
import pytest
import torch

import oracle


def _brute(q, k, v, causal, scale, group):
    """Plain numpy fp64 attention, one (b, h, i) row at a time, K/V head h // group."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, h // group], v[b, h // group]
            for i in range(Nq):
                s = scale * (kh @ q[b, h, i])
                if causal:
                    s = np.where(np.arange(Nk) <= i + Nk - Nq, s, -np.inf)
                m = s.max()
                p = np.exp(s - m)
                o[b, h, i] = p @ vh / p.sum()
                lse[b, h, i] = m + math.log(p.sum())
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_when_every_head_has_its_own_kv(causal):
    g = np.random.default_rng(1)
    q, k, v = (g.standard_normal((2, 3, 9, 8)) for _ in range(3))
    o1, l1 = oracle.attention_gqa(q, k, v, causal, 0.35)
    o2, l2 = oracle.attention(q, k, v, causal, 0.35)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_mqa_against_brute_force(causal):
    g = np.random.default_rng(2)
    q = g.standard_normal((2, 4, 5, 6))
    k = g.standard_normal((2, 1, 7, 6))
    v = g.standard_normal((2, 1, 7, 6))
    o, l = oracle.attention_gqa(q, k, v, causal, 0.5)
    ob, lb = _brute(q, k, v, causal, 0.5, group=4)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_is_mha_with_each_kv_head_repeated_for_its_group(causal):
    g = np.random.default_rng(3)
    B, H, H_kv, N, d = 2, 6, 2, 11, 8
    q = g.standard_normal((B, H, N, d))
    k = g.standard_normal((B, H_kv, N, d)) * np.arange(1, H_kv + 1)[None, :, None, None]  # heads differ in scale
    v = g.standard_normal((B, H_kv, N, d))
    o, l = oracle.attention_gqa(q, k, v, causal, 0.3)
    rep = H // H_kv
    o_ref, l_ref = oracle.attention(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), causal, 0.3)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)
    # The other plausible mapping, h % H_kv, gives a different result on these inputs.
    o_bad, _ = oracle.attention(q, np.tile(k, (1, rep, 1, 1)), np.tile(v, (1, rep, 1, 1)), causal, 0.3)
    assert np.abs(o - o_bad).max() > 1e-3


def test_kv_head_of_maps_consecutive_query_heads_to_one_kv_head():
    assert [oracle.kv_head_of(bh, 8, 2) for bh in range(16)] == [0, 0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2, 3, 3, 3, 3]
    assert [oracle.kv_head_of(bh, 4, 1) for bh in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(bh, 3, 3) for bh in range(6)] == list(range(6))


def test_sampled_rows_follow_the_group_mapping():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(2, 4, 6, 8, generator=g)
    k = torch.randn(2, 2, 9, 8, generator=g)
    v = torch.randn(2, 2, 9, 8, generator=g)
    o, l = oracle.attention_gqa(q, k, v, True, 0.4)
    pairs = [(0, 0), (3, 5), (5, 2), (7, 4)]
    so, sl = oracle.sampled_rows(q, k, v, pairs, True, 0.4)
    for n, (bh, r) in enumerate(pairs):
        np.testing.assert_allclose(so[n], o.reshape(8, 6, 8)[bh, r], rtol=0, atol=1e-12)
        np.testing.assert_allclose(sl[n], l.reshape(8, 6)[bh, r], rtol=0, atol=1e-12)


def test_rejects_a_head_count_that_does_not_divide():
    q = np.zeros((1, 3, 2, 4)); k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention_gqa(q, k, k, False, 1.0)


def test_bwd_gqa_finite_differences():
    """The grouped-query backward is the derivative of the grouped-query forward:
    central differences of L = sum(O * G) through oracle.attention_gqa."""
    g = np.random.default_rng(12)
    B, H, H_kv, Nq, Nk, d = 1, 4, 2, 5, 6, 3
    q = g.standard_normal((B, H, Nq, d))
    k = g.standard_normal((B, H_kv, Nk, d))
    v = g.standard_normal((B, H_kv, Nk, d))
    G = g.standard_normal((B, H, Nq, d))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd_gqa(q, k, v, G, causal, 0.6)
        for x, got in ((q, dq), (k, dk), (v, dv)):
            fd = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                old = x[idx]
                x[idx] = old + 1e-6
                op, _ = oracle.attention_gqa(q, k, v, causal, 0.6)
                x[idx] = old - 1e-6
                om, _ = oracle.attention_gqa(q, k, v, causal, 0.6)
                x[idx] = old
                fd[idx] = ((op - om) * G).sum() / 2e-6
            assert np.allclose(got, fd, atol=1e-8, rtol=0)


def test_bwd_gqa_with_one_query_head_per_kv_head_is_plain_bwd():
    g = np.random.default_rng(13)
    q, k, v, G = (g.standard_normal((2, 3, 7, 4)) for _ in range(4))
    a = oracle.attention_bwd_gqa(q, k, v, G, True, 0.5)
    b = oracle.attention_bwd(q.reshape(6, 7, 4), k.reshape(6, 7, 4), v.reshape(6, 7, 4), G.reshape(6, 7, 4), True, 0.5)
    for x, y in zip(a, b):
        assert np.array_equal(x.reshape(y.shape), y)
