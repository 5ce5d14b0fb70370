"""Pins of the oracle's FP8 (E4M3) format, block quantization and FP8 attention
("Flash Attention (4)" §5.4: E4M3 operands with per-block scale factors)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_decode_closed_forms():
    v = fp8.e4m3_decode(np.array([0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x40, 0x7E, 0xFE, 0x7F, 0xFF], np.uint8))
    want = [0.0, -0.0, 2 ** -9, 7 * 2 ** -9, 2 ** -6, 1.0, 1.875, 2.0, 448.0, -448.0]
    assert np.array_equal(v[:10], np.array(want))
    assert np.isnan(v[10]) and np.isnan(v[11])
    assert np.signbit(v[1])


def test_decode_matches_torch_float8_e4m3fn():
    """Independent library routine: torch's float8_e4m3fn on all 256 codes."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_encode_ties_to_even_and_saturates():
    # midpoint of 1.0 (0x38, even) and 1.125 (0x39): to 1.0; of 1.125 and 1.25 (0x3A): to 1.25
    assert fp8.e4m3_encode([1.0625, 1.1875])[0] == 0x38
    assert fp8.e4m3_encode([1.1875])[0] == 0x3A
    # midpoint of the two smallest subnormals 2^-9 (0x01) and 2^-8 (0x02): to 0x02; 2^-10 to 0 (even)
    assert fp8.e4m3_encode([1.5 * 2 ** -9, 2 ** -10, -2 ** -10]).tolist() == [0x02, 0x00, 0x80]
    assert fp8.e4m3_encode([448.0, 460.0, 1e9, -1e9, np.inf]).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]
    assert fp8.e4m3_encode([np.nan])[0] == 0x7F


def test_encode_matches_torch_in_range():
    """torch's fp32 -> float8_e4m3fn cast (round to nearest even) on random in-range values."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(200000, generator=g) * torch.exp2(torch.randint(-14, 9, (200000,), generator=g).float())
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp8.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_quantize_blocks_error_bound_and_scales():
    g = np.random.default_rng(4)
    x = (g.standard_normal((2, 300, 64)) * np.exp2(g.integers(-6, 6, (2, 300, 1)))).astype(np.float32)
    codes, s = fp8.quantize_blocks(x)
    assert codes.shape == x.shape and s.shape == (2, 3)
    for h in range(2):
        for b in range(3):
            blk = x[h, 128 * b:128 * (b + 1)]
            assert s[h, b] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
    deq = fp8.dequantize_blocks(codes, s)
    rows = np.arange(300) // 128
    sb = s[:, rows][:, :, None].astype(np.float64)
    # normal range: half an ulp = 2^-4 relative; subnormal range: half of 2^-9, times the scale
    assert (np.abs(deq - x) <= 2 ** -4 * np.abs(x) + 2 ** -10 * sb * (1 + 1e-6)).all()
    # the block's largest element maps to the largest code (up to the fp32 division)
    for h in range(2):
        for b in range(3):
            blk = codes[h, 128 * b:128 * (b + 1)] & 0x7F
            assert blk.max() == 0x7E


def test_quantize_blocks_power_of_two_equivariance_and_zero_block():
    g = np.random.default_rng(5)
    x = g.standard_normal((1, 256, 32)).astype(np.float32)
    y = x.copy()
    y[0, 128:] *= 8.0
    y[0, :128] = 0.0
    cx, sx = fp8.quantize_blocks(x)
    cy, sy = fp8.quantize_blocks(y)
    assert np.array_equal(cy[0, 128:], cx[0, 128:]) and sy[0, 1] == 8 * sx[0, 1]
    assert (cy[0, :128] == 0).all() and sy[0, 0] == 1.0


def test_attention_fp8_is_attention_of_dequantized_inputs():
    """With inputs exactly on the E4M3 grid and unit scales, the FP8 oracle is the
    plain oracle; a power-of-two factor on a K block moves into its scale."""
    g = np.random.default_rng(6)
    BH, N, d = 2, 200, 16
    q8, k8, v8 = (fp8.e4m3_encode(g.standard_normal((BH, N, d)) * 4) for _ in range(3))
    ones = np.ones((BH, 2), np.float32)
    q, k, v = (fp8.e4m3_decode(c) for c in (q8, k8, v8))
    for causal in (False, True):
        o1, l1 = fp8.attention_fp8(q8, ones, k8, ones, v8, ones, causal, 0.25)
        o2, l2 = oracle.attention(q, k, v, causal, 0.25)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    k_scale = ones.copy()
    k_scale[:, 1] = 0.5
    o3, l3 = fp8.attention_fp8(q8, ones, k8, k_scale, v8, ones, False, 0.25)
    k_half = k.copy()
    k_half[:, 128:] *= 0.5
    o4, l4 = oracle.attention(q, k_half, v, False, 0.25)
    assert np.allclose(o3, o4, atol=1e-12, rtol=0) and np.allclose(l3, l4, atol=1e-12, rtol=0)
