"""fa_bwd_varlen (backward of packed variable-length batches) against the fp64 oracle.

Layouts as fa_fwd_varlen: q, o, dout, dq packed [total_q, H, d]; k, v, dk, dv
[total_k, H_kv, d]; lse [H, total_q].  The GPU side runs fa_fwd_varlen then
fa_bwd_varlen; the oracle recomputes each sequence's gradients from q, k, v, dO
(oracle.attention_bwd_varlen).  Tolerance as in parity.compare_grads, with the
magnitudes taken sequence by sequence.
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


def _packed(lens_q, lens_k, H, H_kv, d, dtype, seed):
    total_q, total_k = sum(lens_q), sum(lens_k)
    q, _, _ = attn_inputs.make_qkv(1, total_q, H, 1, d, dtype, seed, "cuda")
    _, k, v = attn_inputs.make_qkv(1, total_k, 1, H_kv, d, dtype, seed + 5, "cuda")
    dout = attn_inputs.make_dout(1, total_q, H, d, dtype, seed, "cuda")
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    return q[0].contiguous(), k[0].contiguous(), v[0].contiguous(), dout[0].contiguous(), cu_q, cu_k


def _magnitudes(q, k, v, dout, o_ref, lse_ref, lens_q, lens_k, causal, scale):
    """grad_magnitudes sequence by sequence (K/V heads repeated per group, their
    magnitudes summed like the gradients), in the packed layouts."""
    H, H_kv, d = q.shape[1], k.shape[1], q.shape[2]
    group = H // H_kv
    mq, mk, mv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    cq, ck = np.concatenate([[0], np.cumsum(lens_q)]), np.concatenate([[0], np.cumsum(lens_k)])
    tr = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))           # [n, h, d] -> [h, n, d]
    rep = lambda x: tr(x).repeat(group, axis=0)
    for s in range(len(lens_q)):
        a, b, c, e = cq[s], cq[s + 1], ck[s], ck[s + 1]
        if b == a or e == c:
            continue
        m = grad_magnitudes(tr(q[a:b]), rep(k[c:e]), rep(v[c:e]), tr(o_ref[a:b]), tr(dout[a:b]),
                            lse_ref[:, a:b], causal, scale)
        mq[a:b] = m[0].transpose(1, 0, 2)
        mk[c:e] = m[1].reshape(H_kv, group, e - c, d).sum(axis=1).transpose(1, 0, 2)
        mv[c:e] = m[2].reshape(H_kv, group, e - c, d).sum(axis=1).transpose(1, 0, 2)
    return mq, mk, mv


def run_varlen_bwd(fa, lens_q, lens_k, H, H_kv, d, dtype, causal, seed):
    q, k, v, dout, cu_q, cu_k = _packed(lens_q, lens_k, H, H_kv, d, dtype, seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd_varlen(q, k, v, cu_q, cu_k, max(lens_q), causal=causal, scale=scale)
    dq, dk, dv = fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, max(lens_k), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    qn, kn, vn, gn = (_np(x) for x in (q, k, v, dout))
    ref = oracle.attention_bwd_varlen(qn, kn, vn, gn, cu_q.cpu(), cu_k.cpu(), causal, scale)
    o_ref, lse_ref = oracle.attention_varlen(qn, kn, vn, cu_q.cpu(), cu_k.cpu(), causal, scale)
    mags = _magnitudes(qn, kn, vn, gn, o_ref, lse_ref, lens_q, lens_k, causal, scale)
    floors = (0.0, 0.0, 0.0)
    if q.dtype == torch.float16:  # fp32 accumulation of up to max-length sums, as in the dense test
        e = 2.0 ** -25
        group = H // H_kv
        floors = (e * max(lens_k) * scale * np.abs(kn).max(), e * max(lens_q) * group * scale * np.abs(qn).max(),
                  e * max(lens_q) * group * np.abs(gn).max())
    compare_grads((dq, dk, dv), ref, mags, floors, q.dtype, f"bwd varlen q{lens_q} k{lens_k} H{H}/{H_kv} d{d}")
    return dq, dk, dv, ref


CASES = [
    # lens_q, lens_k, H, H_kv, d, dtype, causal
    ([1, 127, 128, 129, 300], None, 4, 4, 128, "bf16", True),
    ([1, 127, 128, 129, 300], None, 4, 2, 64, "f16", False),
    ([513, 7, 256], [600, 7, 100], 2, 1, 128, "bf16", True),     # Nq != Nk per sequence, some rows see no key
    ([64, 0, 200], [64, 50, 0], 4, 2, 128, "bf16", False),        # an empty sequence and a keyless one
    ([130, 0, 70], [0, 90, 70], 2, 2, 64, "bf16", True),          # keys without queries and queries without keys
    ([1000, 1, 333, 1100], None, 8, 2, 128, "bf16", True),
    # 100 short sequences (several 32-sequence chunks of the row plan), lengths 0..300, some empty
    ([int(x) for x in np.random.default_rng(5).integers(0, 301, 100)], None, 2, 1, 64, "bf16", True),
]


def _case_id(c):
    lens = "-".join(map(str, c[0])) if len(c[0]) <= 6 else f"{len(c[0])}seqs"
    return f"q{lens}_H{c[2]}kv{c[3]}_d{c[4]}{c[5]}{'c' if c[6] else ''}"


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_bwd_varlen(fa, case):
    lens_q, lens_k, H, H_kv, d, dtype, causal = case
    lens_k = lens_k or lens_q
    dq, dk, dv, ref = run_varlen_bwd(fa, lens_q, lens_k, H, H_kv, d, dtype, causal, 300 + sum(lens_q) % 97)
    # sequences without keys: dQ exactly 0; keys of sequences without queries: dK = dV = 0
    cq, ck = np.concatenate([[0], np.cumsum(lens_q)]), np.concatenate([[0], np.cumsum(lens_k)])
    for s in range(len(lens_q)):
        if lens_k[s] == 0 and lens_q[s] > 0:
            assert (dq[cq[s]:cq[s + 1]] == 0).all()
        if lens_q[s] == 0 and lens_k[s] > 0:
            assert (dk[ck[s]:ck[s + 1]] == 0).all() and (dv[ck[s]:ck[s + 1]] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_the_dense_backward(fa, causal):
    """Packed sequences of one length are a dense batch.  Rows and keys past a
    sequence end get weight exactly 0, so dK and dV (no atomics) agree with fa_bwd
    to the bit; dQ (fp32 atomic sums, order not fixed) within a few ulp."""
    B, H, N, d = 3, 4, 300, 128
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 211, "cuda")
    dout = attn_inputs.make_dout(B, H, N, d, "bf16", 211, "cuda")
    o, lse = fa.fwd(q, k, v, causal=causal)
    dq_d, dk_d, dv_d = fa.bwd(q, k, v, o, dout, lse, causal=causal)
    pack = lambda x: x.transpose(1, 2).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    lse_p = lse.transpose(0, 1).reshape(H, B * N).contiguous()
    dq, dk, dv = fa.bwd_varlen(pack(q), pack(k), pack(v), pack(o), pack(dout), lse_p, cu, cu, N, causal=causal)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(dk, pack(dk_d))
    assert torch.equal(dv, pack(dv_d))
    diff = (dq.float() - pack(dq_d).float()).abs()
    assert (diff <= 2.0 ** -6 * pack(dq_d).float().abs() + 1e-6).all()


def test_varlen_bwd_deterministic_dk_dv(fa):
    q, k, v, dout, cu_q, cu_k = _packed([300, 5, 700], [300, 5, 700], 4, 2, 128, "bf16", 77)
    o, lse = fa.fwd_varlen(q, k, v, cu_q, cu_k, 700, causal=True)
    a = fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 700, causal=True)
    b = fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 700, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_varlen_bwd_rejects_bad_arguments(fa):
    q, k, v, dout, cu_q, cu_k = _packed([10, 20], [10, 20], 2, 2, 64, "bf16", 5)
    o, lse = fa.fwd_varlen(q, k, v, cu_q, cu_k, 20)
    with pytest.raises(fa.FaError) as e:
        fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 0)    # max_seqlen_k must be >= 1
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FaError) as e:
        fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 31)   # more than total_k
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    short = torch.empty(fa.bwd_varlen_workspace_bytes(2, 30, 30, 2, 64) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 20, workspace=short)
    assert e.value.code == fa.FA_ERR_WORKSPACE
    assert fa.get_device_status() == fa.FA_OK


def test_varlen_autograd(fa):
    """attention_varlen under autograd gives the gradients of fa_bwd_varlen."""
    q, k, v, dout, cu_q, cu_k = _packed([90, 200, 31], [120, 200, 40], 4, 2, 64, "bf16", 91)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    out = fa.attention_varlen(qq, kk, vv, cu_q, cu_k, 200, 200, causal=True)
    out.backward(dout)
    o, lse = fa.fwd_varlen(q, k, v, cu_q, cu_k, 200, causal=True)
    dq, dk, dv = fa.bwd_varlen(q, k, v, o, dout, lse, cu_q, cu_k, 200, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o)
    assert torch.equal(kk.grad, dk) and torch.equal(vv.grad, dv)
    assert ((qq.grad.float() - dq.float()).abs() <= 2.0 ** -6 * dq.float().abs() + 1e-6).all()


def _segment_sums(x, cu):
    """Per-sequence sums over tokens of a [total, H, d] tensor (fp64): [num_seqs, H, d]."""
    c = torch.cat([torch.zeros_like(x[:1], dtype=torch.float64), x.double().cumsum(dim=0)])
    return c[cu[1:].long()] - c[cu[:-1].long()]


def test_bwd_varlen_benchmarked_batch(fa):
    """The benchmarked packed batch (16 causal sequences of 256..8192 tokens, H=32,
    d=128, bf16): on every sequence and head the dK rows sum to zero and the dV rows
    to the dO rows, and one head of the longest sequence against the oracle."""
    import itertools

    vw = attn_inputs.VARLEN_WORKLOAD
    lens = attn_inputs.varlen_lengths(vw["num_seqs"], vw["lo"], vw["hi"], vw["seed"])
    total, H, d = sum(lens), vw["H"], vw["d"]
    q = attn_inputs.make_qkv(1, total, H, 1, d, vw["dtype"], vw["seed"], "cuda")[0][0]
    _, k, v = attn_inputs.make_qkv(1, total, 1, H, d, vw["dtype"], vw["seed"] + 5, "cuda")
    k, v = k[0], v[0]
    dout = attn_inputs.make_dout(1, total, H, d, vw["dtype"], vw["seed"], "cuda")[0]
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device="cuda")
    o, lse = fa.fwd_varlen(q, k, v, cu, cu, max(lens), causal=True)
    dq, dk, dv = fa.bwd_varlen(q, k, v, o, dout, lse, cu, cu, max(lens), causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    u = 2.0 ** -8
    s_dk = _segment_sums(dk, cu).abs()
    assert (s_dk <= 2 * u * _segment_sums(dk.abs(), cu) + 1e-6).all()
    s_dv, s_do = _segment_sums(dv, cu), _segment_sums(dout, cu)
    assert ((s_dv - s_do).abs() <= 2 * u * (_segment_sums(dv.abs(), cu) + _segment_sums(dout.abs(), cu))).all()
    s = int(np.argmax(lens))
    a, b, h = int(cu[s]), int(cu[s + 1]), 11
    one = lambda x: _np(x[a:b, h]).reshape(1, b - a, d)
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_bwd(one(q), one(k), one(v), one(dout), True, scale)
    o_ref, lse_ref = oracle.attention(one(q), one(k), one(v), True, scale)
    mags = grad_magnitudes(one(q), one(k), one(v), o_ref, one(dout), lse_ref, True, scale)
    compare_grads((dq[a:b, h], dk[a:b, h], dv[a:b, h]), ref, mags, (0.0, 0.0, 0.0), torch.bfloat16,
                  f"bwd varlen benchmarked batch, sequence {s} ({lens[s]} tokens), head {h}")
