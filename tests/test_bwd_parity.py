"""fa_bwd (tcgen05 attention backward) against the fp64 oracle's gradients.

The GPU side runs the product pipeline: fa_fwd gives (O, LSE), fa_bwd the
gradients from them.  The oracle side recomputes everything from q, k, v, dO
(oracle.attention_bwd).  The tolerance is derived in parity.py (compare_grads).
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs
import oracle
from parity import compare_grads, grad_magnitudes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    oracle.set_threads(16)
    return fa


def _np(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def _floors(dtype, Nq, Nk, q, k, dout, scale):
    if dtype != torch.float16:
        return 0.0, 0.0, 0.0
    e = 2.0 ** -25
    return (e * Nk * scale * np.abs(k).max(), e * Nq * scale * np.abs(q).max(), e * Nq * np.abs(dout).max())


def run_bwd(fa, B, H, Nq, Nk, d, dtype, causal, seed):
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, seed, "cuda")
    dout = attn_inputs.make_dout(B, H, Nq, d, dtype, seed, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(q, k, v, o, dout, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    qn, kn, vn, gn = (_np(x).reshape(B * H, -1, d) for x in (q, k, v, dout))
    ref = oracle.attention_bwd(qn, kn, vn, gn, causal, scale)
    o_ref, lse_ref = oracle.attention(qn, kn, vn, causal, scale)
    mags = grad_magnitudes(qn, kn, vn, o_ref, gn, lse_ref, causal, scale)
    floors = _floors(q.dtype, Nq, Nk, qn, kn, gn, scale)
    return compare_grads((dq, dk, dv), ref, mags, floors, q.dtype,
                         f"bwd B{B} H{H} Nq{Nq} Nk{Nk} d{d} {dtype} causal={causal}")


CASES = [
    # B, H, Nq, Nk, d, dtype, causal
    (1, 2, 128, 128, 128, "bf16", False),   # one tile
    (2, 2, 300, 300, 128, "bf16", True),    # ragged tails, diagonal tiles
    (1, 2, 257, 513, 64, "f16", False),     # d = 64, Nq != Nk
    (1, 2, 520, 200, 128, "bf16", True),    # Nq > Nk: the first rows see no key
    (1, 2, 200, 520, 128, "bf16", True),    # Nq < Nk: the first key blocks are seen by every row
    (1, 2, 1, 300, 128, "bf16", False),     # one query row
    (1, 4, 1024, 1024, 128, "bf16", True),  # several query blocks per key block
    (1, 2, 384, 384, 64, "bf16", True),
    (1, 2, 640, 640, 128, "f16", False),
    (1, 1, 129, 1, 128, "bf16", True),      # a single key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}Nq{}Nk{}d{}{}{}".format(*c[:6], "c" if c[6] else ""))
def test_bwd(fa, case):
    B, H, Nq, Nk, d, dtype, causal = case
    run_bwd(fa, B, H, Nq, Nk, d, dtype, causal, 300 + Nq + Nk)


def test_bwd_full_size_invariants_and_one_head():
    """B=2, H=32, N=8192, d=128, bf16, causal (the forward benchmark's shape): on
    every head the dK rows sum to zero and the dV rows sum to the dO rows
    (properties of the gradient at any size), and one head against the oracle."""
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    oracle.set_threads(16)
    B, H, N, d = 2, 32, 8192, 128
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 1000, "cuda")
    dout = attn_inputs.make_dout(B, H, N, d, "bf16", 1000, "cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    dq, dk, dv = fa.bwd(q, k, v, o, dout, lse, causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    u = 2.0 ** -8
    dk64, dv64 = dk.double(), dv.double()
    # sum_j dK_j = 0 (shift invariance of the keys): each term is off by at most
    # u |dK_j| (output rounding) plus its own rounding of dS, so allow 2u sum |dK_j|.
    s_dk = dk64.sum(dim=2).abs()
    assert (s_dk <= 2 * u * dk64.abs().sum(dim=2) + 1e-6).all()
    # sum_j dV_j = sum_i dO_i (rows of P sum to one; every row sees key 0)
    s_dv = dv64.sum(dim=2)
    s_do = dout.double().sum(dim=2)
    assert ((s_dv - s_do).abs() <= 2 * u * dv64.abs().sum(dim=2) + 2 * u * dout.double().abs().sum(dim=2)).all()
    # one head (b = 1, h = 17) element-wise against the oracle
    b, h = 1, 17
    qn, kn, vn, gn = (_np(x[b, h]).reshape(1, N, d) for x in (q, k, v, dout))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_bwd(qn, kn, vn, gn, True, scale)
    o_ref, lse_ref = oracle.attention(qn, kn, vn, True, scale)
    mags = grad_magnitudes(qn, kn, vn, o_ref, gn, lse_ref, True, scale)
    compare_grads((dq[b, h], dk[b, h], dv[b, h]), ref, mags, (0.0, 0.0, 0.0), torch.bfloat16, "bwd full-size head")


def test_bwd_full_size_noncausal_one_head(fa):
    """B=2, H=32, N=8192, d=128, bf16 without the mask: one head element-wise."""
    B, H, N, d = 2, 32, 8192, 128
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 1100, "cuda")
    dout = attn_inputs.make_dout(B, H, N, d, "bf16", 1100, "cuda")
    o, lse = fa.fwd(q, k, v, causal=False)
    dq, dk, dv = fa.bwd(q, k, v, o, dout, lse, causal=False)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    b, h = 0, 7
    qn, kn, vn, gn = (_np(x[b, h]).reshape(1, N, d) for x in (q, k, v, dout))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_bwd(qn, kn, vn, gn, False, scale)
    o_ref, lse_ref = oracle.attention(qn, kn, vn, False, scale)
    mags = grad_magnitudes(qn, kn, vn, o_ref, gn, lse_ref, False, scale)
    compare_grads((dq[b, h], dk[b, h], dv[b, h]), ref, mags, (0.0, 0.0, 0.0), torch.bfloat16,
                  "bwd full-size non-causal head")


def test_dk_dv_deterministic_dq_close(fa):
    q, k, v = attn_inputs.make_qkv(1, 4, 700, 700, 128, "bf16", 77, "cuda")
    dout = attn_inputs.make_dout(1, 4, 700, 128, "bf16", 77, "cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    a = fa.bwd(q, k, v, o, dout, lse, causal=True)
    b = fa.bwd(q, k, v, o, dout, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2.0 ** -6 * a[0].float().abs().max().item()


def test_autograd_wrapper_matches_bwd(fa):
    q, k, v = attn_inputs.make_qkv(2, 2, 333, 333, 64, "bf16", 88, "cuda")
    dout = attn_inputs.make_dout(2, 2, 333, 64, "bf16", 88, "cuda")
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    out = fa.attention(qq, kk, vv, causal=True)
    out.backward(dout)
    o, lse = fa.fwd(q, k, v, causal=True)
    dq, dk, dv = fa.bwd(q, k, v, o, dout, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out, o)
    assert torch.equal(kk.grad, dk) and torch.equal(vv.grad, dv)
    assert (qq.grad.float() - dq.float()).abs().max().item() <= 2.0 ** -6 * dq.float().abs().max().item()


def test_bwd_rejects_bad_arguments(fa):
    q, k, v = attn_inputs.make_qkv(1, 2, 100, 100, 128, "bf16", 5, "cuda")
    dout = torch.randn_like(q)
    o, lse = fa.fwd(q, k, v)
    lib = fa.load_library()
    need = fa.bwd_workspace_bytes(1, 2, 100, 128)
    assert need == 1 * 2 * 128 * 128 * 4 + 2 * 1024
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    args = lambda nbytes: (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, 2, 100, 100, 128, 0, 0.1, fa.FA_BF16,
                           ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    assert lib.fa_bwd(*args(need - 1)) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd(*args(need)) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK


GQA = [
    # B, H, H_kv, Nq, Nk, d, dtype, causal
    (2, 4, 2, 300, 300, 128, "bf16", True),
    (1, 8, 1, 257, 513, 64, "f16", False),     # multi-query
    (1, 6, 3, 520, 200, 128, "bf16", True),    # Nq > Nk
]


@pytest.mark.parametrize("case", GQA, ids=lambda c: "B{}H{}Hkv{}Nq{}Nk{}d{}{}{}".format(*c[:7], "c" if c[7] else ""))
def test_bwd_gqa(fa, case):
    """Grouped K/V heads: dK, dV of a K/V head sum its query heads' contributions."""
    B, H, H_kv, Nq, Nk, d, dtype, causal = case
    q, _, _ = attn_inputs.make_qkv(B, H, Nq, 1, d, dtype, 500 + Nq, "cuda")
    _, k, v = attn_inputs.make_qkv(B, H_kv, 1, Nk, d, dtype, 600 + Nk, "cuda")
    dout = attn_inputs.make_dout(B, H, Nq, d, dtype, 700, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(q, k, v, o, dout, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    ref = oracle.attention_bwd_gqa(q, k, v, dout, causal, scale)
    group = H // H_kv
    # magnitudes per query head against its K/V head, then summed like the gradients
    rep = lambda x: _np(x).repeat(group, axis=1).reshape(B * H, -1, d)
    qn, gn = _np(q).reshape(B * H, Nq, d), _np(dout).reshape(B * H, Nq, d)
    o_ref, lse_ref = oracle.attention(qn, rep(k), rep(v), causal, scale)
    mq, mk, mv = grad_magnitudes(qn, rep(k), rep(v), o_ref, gn, lse_ref, causal, scale)
    mk = mk.reshape(B, H_kv, group, Nk, d).sum(axis=2)
    mv = mv.reshape(B, H_kv, group, Nk, d).sum(axis=2)
    floors = _floors(q.dtype, Nq * group, Nk, qn, _np(k), gn, scale)  # dK, dV sum Nq * group terms
    compare_grads((dq, dk, dv), ref, (mq.reshape(ref[0].shape), mk, mv), floors, q.dtype,
                  f"bwd gqa {case}")


def test_bwd_gqa_autograd(fa):
    q, _, _ = attn_inputs.make_qkv(1, 4, 200, 1, 64, "bf16", 81, "cuda")
    _, k, v = attn_inputs.make_qkv(1, 1, 1, 200, 64, "bf16", 82, "cuda")
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    out = fa.attention(qq, kk, vv, causal=True)
    out.backward(torch.ones_like(out))
    torch.cuda.synchronize()
    assert kk.grad.shape == k.shape and torch.isfinite(kk.grad).all() and torch.isfinite(qq.grad).all()
