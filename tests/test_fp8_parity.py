"""FP8 (E4M3) path against the oracle: the block quantization bit for bit, and
fa_fwd_fp8 against attention on the dequantized inputs (oracle.fp8).

Tolerance of the FP8 forward, from the kernel's arithmetic: with the scores exact
up to fp32 (E4M3 products are exact, sums in fp32), the only coarse rounding is
P to E4M3 after scaling by kappa_j = 2^7 s_v(j) / max s_v.  A normal E4M3 value
is within 2^-4 (relative) of its input, a subnormal one (below 2^-6) within
2^-10 (absolute), so for every output element
    |O - O_ref| <= 2^-4 sum_j P_ij |v_j| / l_i
                 + 2^-10 sum_{j: P_ij kappa_j < 2^-6} |v_j| / (kappa_j l_i)
                 + half an output ulp,
with P_ij = exp(s_ij - max_j s_ij) and l_i = sum_j P_ij on the dequantized inputs
(the kernel's running max only moves P and l by one common factor per row).  The
test allows that bound plus 1e-4.  LSE does not involve the rounded P: 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs
import oracle
from oracle import fp8

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


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_bit_exact(fa, dtype, transpose):
    B, H, N, d = 1, 3, 300, 128
    x = attn_inputs.make_qkv(B, H, N, 1, d, dtype, 21, "cuda")[0]
    x[0, 1] *= 40.0                 # a head of large values
    x[0, 2, :256] = 0               # head 2: block 1 all zero (scale 1, codes 0) ...
    x[0, 2, 5, 7] = 1e-3            # ... and block 0 holding one tiny value
    codes, scales = fa.fp8_quantize(x, transpose=transpose)
    torch.cuda.synchronize()
    ref_codes, ref_scales = fp8.quantize_blocks(x.reshape(B * H, N, d).cpu())
    assert np.array_equal(scales.cpu().numpy(), ref_scales)
    got = codes.cpu().numpy().reshape(B * H, *codes.shape[2:])
    if transpose:
        assert got.shape == (B * H, d, 384)
        assert np.array_equal(got[:, :, :N].transpose(0, 2, 1), ref_codes)
        assert (got[:, :, N:] == 0).all()
    else:
        assert np.array_equal(got, ref_codes)


def _fp8_tolerance(q, k, v, qs, ks, vs, causal, scale, o_ref, out_dtype):
    """Element-wise bound of the docstring for [BH, N, d] dequantized q, k, v."""
    BH, Nq, d = q.shape
    Nk = k.shape[1]
    kappa = 128.0 * vs / vs.max(axis=1, keepdims=True)               # [BH, key blocks]
    kap_j = kappa[:, np.arange(Nk) // 128]                            # [BH, Nk]
    allowed = np.ones((Nq, Nk), bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    tol = np.empty_like(o_ref)
    for b in range(BH):
        s = scale * (q[b] @ k[b].T)
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        p = np.where(allowed, np.exp(s - m), 0.0)
        l = p.sum(axis=1, keepdims=True)
        l = np.where(l > 0, l, np.inf)
        small = (p * kap_j[b][None, :] < 2.0 ** -6) & allowed
        rel = 2.0 ** -4 * (p @ np.abs(v[b])) / l
        absol = 2.0 ** -10 * ((small / kap_j[b][None, :]) @ np.abs(v[b])) / l
        tol[b] = rel + absol
    ulp_half = (2.0 ** -9 if out_dtype == torch.bfloat16 else 2.0 ** -12) * np.abs(o_ref)
    return tol + ulp_half + 1e-4


CASES = [
    # B, H, Nq, Nk, causal, input dtype
    (1, 2, 128, 128, False, "bf16"),
    (2, 2, 300, 300, True, "bf16"),
    (1, 2, 257, 513, False, "f16"),
    (1, 2, 520, 200, True, "bf16"),     # Nq > Nk: the first rows see no key
    (1, 2, 200, 520, True, "bf16"),
    (1, 2, 1, 300, False, "bf16"),
    (1, 4, 1024, 1024, True, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}Nq{}Nk{}{}{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_fwd_fp8(fa, case):
    B, H, Nq, Nk, causal, dtype = case
    d = 128
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, 400 + Nq + Nk, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd_fp8_from(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    # the oracle quantizes the same inputs itself
    q8, qs = fp8.quantize_blocks(q.reshape(B * H, Nq, d).cpu())
    k8, ks = fp8.quantize_blocks(k.reshape(B * H, Nk, d).cpu())
    v8, vs = fp8.quantize_blocks(v.reshape(B * H, Nk, d).cpu())
    o_ref, lse_ref = fp8.attention_fp8(q8, qs, k8, ks, v8, vs, causal, scale)
    og = _np(o).reshape(o_ref.shape)
    assert np.isfinite(og).all()
    tol = _fp8_tolerance(fp8.dequantize_blocks(q8, qs), fp8.dequantize_blocks(k8, ks), fp8.dequantize_blocks(v8, vs),
                         qs, ks, vs.astype(np.float64), causal, scale, o_ref, q.dtype)
    err = np.abs(og - o_ref)
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} O elements out of tolerance; worst {np.unravel_index(np.argmax(err / tol), err.shape)}"
    lg = _np(lse).reshape(lse_ref.shape)
    assert (np.isneginf(lg) == np.isneginf(lse_ref)).all()
    fin = np.isfinite(lse_ref)
    assert np.abs(lg[fin] - lse_ref[fin]).max(initial=0) <= 1e-3


def test_fwd_fp8_close_to_the_16_bit_forward(fa):
    """On N(0, 1) inputs the FP8 path stays near the 16-bit forward.  The gap is the
    quantization of the inputs (up to 2^-4 relative per element), not the kernel:
    a score s = scale q.k moves by up to about 2^-3 scale sum|q||k|, typically a few
    hundredths, and LSE by a P-weighted mean of those moves."""
    q, k, v = attn_inputs.make_qkv(1, 4, 777, 777, 128, "bf16", 31, "cuda")
    o16, l16 = fa.fwd(q, k, v, causal=True)
    o8, l8 = fa.fwd_fp8_from(q, k, v, causal=True)
    torch.cuda.synchronize()
    rel = (o8.float() - o16.float()).norm() / o16.float().norm()
    assert rel.item() < 0.05
    assert (l8 - l16).abs().max().item() < 0.15


def test_fp8_rejects_bad_arguments(fa):
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fp8_quantize(q)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    assert fa.get_device_status() == fa.FA_OK


def test_fwd_fp8_full_size_one_head(fa):
    """B=2, H=32, N=8192, d=128, causal (the benchmarked FP8 launch): the codes of one
    head bit for bit and that head's output element-wise within the bound above."""
    B, H, N, d = 2, 32, 8192, 128
    w = attn_inputs.WORKLOADS["b2h32_n8192_d128_bf16_causal"]
    q, k, v = attn_inputs.make_workload(w, "cuda")
    q8, qs = fa.fp8_quantize(q)
    k8, ks = fa.fp8_quantize(k)
    v8t, vs = fa.fp8_quantize(v, transpose=True)
    o, lse = fa.fwd_fp8(q8, qs, k8, ks, v8t, vs, causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    b, h = 1, 30
    bh = b * H + h
    qr, kr, vr = (x[b, h].reshape(1, N, d).cpu() for x in (q, k, v))
    rq8, rqs = fp8.quantize_blocks(qr)
    rk8, rks = fp8.quantize_blocks(kr)
    rv8, rvs = fp8.quantize_blocks(vr)
    assert np.array_equal(q8[b, h].cpu().numpy(), rq8[0]) and np.array_equal(qs[bh].cpu().numpy(), rqs[0])
    assert np.array_equal(k8[b, h].cpu().numpy(), rk8[0]) and np.array_equal(ks[bh].cpu().numpy(), rks[0])
    assert np.array_equal(v8t[b, h].cpu().numpy().T, rv8[0]) and np.array_equal(vs[bh].cpu().numpy(), rvs[0])
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = fp8.attention_fp8(rq8, rqs, rk8, rks, rv8, rvs, True, scale)
    tol = _fp8_tolerance(fp8.dequantize_blocks(rq8, rqs), fp8.dequantize_blocks(rk8, rks),
                         fp8.dequantize_blocks(rv8, rvs), rqs, rks, rvs.astype(np.float64), True, scale, o_ref,
                         torch.bfloat16)
    err = np.abs(_np(o[b, h]).reshape(o_ref.shape) - o_ref)
    assert (err <= tol).all(), f"{int((err > tol).sum())} elements out of tolerance"
    assert np.abs(_np(lse[b, h]) - lse_ref[0]).max() <= 1e-3
