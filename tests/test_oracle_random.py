"""Randomised shapes for the oracle (CPU): hypothesis draws the problem sizes, the
mask and the tiling, and the oracle must agree with an independent library
routine (torch fp64 scaled_dot_product_attention, logsumexp and autograd) and
with its own tiled loop.  The fixed-shape pins cover the worked cases; these
cover the shape space around them (Nq > Nk and Nq < Nk under the causal mask,
single rows and keys, tiles that do not divide the key count).
"""
import math

import numpy as np
import pytest
import torch

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


def _mask(Nq, Nk):
    return torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)


shapes = st.tuples(st.integers(1, 2), st.integers(1, 3), st.integers(1, 40), st.integers(1, 40),
                   st.sampled_from([1, 3, 8, 16]), st.booleans(), st.integers(0, 2 ** 31 - 1))


@settings(max_examples=60, deadline=None)
@given(shapes)
def test_forward_against_torch(shape):
    B, H, Nq, Nk, d, causal, seed = shape
    lib = oracle.load()
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, n, d, generator=g, dtype=torch.float64) for n in (Nq, Nk, Nk))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, causal, scale, lib=lib)
    s = scale * (q @ k.transpose(-1, -2))
    if causal:
        s = s.masked_fill(~_mask(Nq, Nk), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)   # rows with no key: weight 0
    ref_o = p @ v
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse.numpy()))
    fin = np.isfinite(lse)
    assert np.allclose(lse[fin], ref_lse.numpy()[fin], atol=1e-12, rtol=0)
    assert np.allclose(o, ref_o.numpy(), atol=1e-12, rtol=0)


@settings(max_examples=40, deadline=None)
@given(shapes, st.integers(1, 48))
def test_tiled_loop_equals_full(shape, Bc):
    B, H, Nq, Nk, d, causal, seed = shape
    lib = oracle.load()
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, n, d, generator=g, dtype=torch.float64) for n in (Nq, Nk, Nk))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, causal, scale, lib=lib)
    ot, lt = oracle.attention_tiled(q, k, v, causal, scale, 16, Bc, lib=lib)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lt))
    fin = np.isfinite(lse)
    assert np.allclose(lt[fin], lse[fin], atol=1e-12, rtol=0)
    assert np.allclose(ot, o, atol=1e-12, rtol=0)


@settings(max_examples=30, deadline=None)
@given(shapes)
def test_backward_against_torch_autograd(shape):
    B, H, Nq, Nk, d, causal, seed = shape
    if causal and Nq > Nk:
        Nq = Nk   # rows with no key have no gradient path through torch's softmax (NaN there)
    lib = oracle.load()
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, n, d, generator=g, dtype=torch.float64, requires_grad=True) for n in (Nq, Nk, Nk))
    dout = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float64)
    scale = 1.0 / math.sqrt(d)
    s = scale * (q @ k.transpose(-1, -2))
    if causal:
        s = s.masked_fill(~_mask(Nq, Nk), float("-inf"))
    (torch.softmax(s, dim=-1) @ v).backward(dout)
    dq, dk, dv = oracle.attention_bwd(q.detach(), k.detach(), v.detach(), dout, causal, scale, lib=lib)
    for got, want in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
        assert np.allclose(got, want.numpy(), atol=1e-11, rtol=0)
