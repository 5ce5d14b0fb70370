"""FP8 (E4M3) side of the oracle: the format, block quantization, and attention
on dequantized inputs.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only the tests, the
package smoke check and the benchmark's CPU legs call it, and it shares no code
with the CUDA library.

The pages use E4M3 for the operands of both products and per-block scale
factors against underflow ("Flash Attention (4)" §5.4, FP8 support and error
control; the exercise on FP8 underflow in §8.3).  The format is written out
here from its definition, plain numpy:

  E4M3 (no infinities): bit 7 sign, bits 6..3 exponent e (bias 7), bits 2..0
  mantissa m.  e = 0: value m * 2^-9 (subnormal); 0 < e: (1 + m/8) * 2^(e-7);
  e = 15 and m = 7 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.

Quantization of a [BH, N, d] tensor in blocks of 128 rows of one head: with
amax the largest |x| of the block (fp32), the block's scale is s = amax / 448
in fp32 (s = 1 when amax = 0), and each element's code is x / s (fp32
division) rounded to the nearest E4M3 value, ties to an even mantissa, with
magnitudes above 448 saturating to 448.  x is represented as codes * s.
"""
from __future__ import annotations

import numpy as np

from . import attention, to_f64

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_decode(codes) -> np.ndarray:
    """Values (fp64) of E4M3 codes (uint8); NaN for 0x7F and 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the non-negative finite values in code order (codes 0x00 .. 0x7E); increasing
_POS_VALUES = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """Round fp32/fp64 values to E4M3 codes: nearest, ties to even mantissa,
    finite magnitudes above 448 saturate to 448, NaN to 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a_sat, side="left")  # first value >= a
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = _POS_VALUES[hi] - a_sat
    d_lo = a_sat - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0))
    code = np.where(pick_lo, lo, hi).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_blocks(x, block: int = BLOCK):
    """(codes uint8 [BH, N, d], scales float32 [BH, ceil(N / block)]) of x [BH, N, d]."""
    x32 = np.asarray(to_f64(x), dtype=np.float64).astype(np.float32)
    if x32.ndim == 2:
        x32 = x32[None]
    BH, N, d = x32.shape
    nb = -(-N // block)
    codes = np.zeros((BH, N, d), dtype=np.uint8)
    scales = np.ones((BH, nb), dtype=np.float32)
    for h in range(BH):
        for b in range(nb):
            blk = x32[h, b * block:(b + 1) * block]
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            s = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
            scales[h, b] = s
            codes[h, b * block:(b + 1) * block] = e4m3_encode((blk / s).astype(np.float32))
    return codes, scales


def dequantize_blocks(codes, scales, block: int = BLOCK) -> np.ndarray:
    """codes * scale of their block, fp64 [BH, N, d]."""
    vals = e4m3_decode(codes)
    BH, N, _ = vals.shape
    rows = np.arange(N) // block
    return vals * np.asarray(scales, dtype=np.float64)[:, rows][:, :, None]


def attention_fp8(q8, q_scale, k8, k_scale, v8, v_scale, causal: bool, scale: float, lib=None):
    """The attention definition (fp64) on the dequantized inputs: Q = q8 * q_scale,
    K = k8 * k_scale, V = v8 * v_scale, each scale per 128-row block of a head;
    all arrays [BH, N, d] / [BH, blocks].  Returns (O, LSE)."""
    q = dequantize_blocks(q8, q_scale)
    k = dequantize_blocks(k8, k_scale)
    v = dequantize_blocks(v8, v_scale)
    return attention(q, k, v, causal, scale, lib=lib)


def p_quant_step() -> float:
    """Spacing of the E4M3 subnormals (2^-9) — the absolute rounding step below 2^-6."""
    return 2.0 ** -9


def e4m3_rel_half_ulp() -> float:
    """Largest relative rounding error of a normal E4M3 value (half of 2^-3)."""
    return 2.0 ** -4


__all__ = ["e4m3_decode", "e4m3_encode", "quantize_blocks", "dequantize_blocks", "attention_fp8", "E4M3_MAX",
           "BLOCK", "p_quant_step", "e4m3_rel_half_ulp"]
