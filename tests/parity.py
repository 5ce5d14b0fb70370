"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerance (written out once, used by every GPU parity test):
  O:   |O_gpu - rnd(O_ref)| <= max(2e-3, ulp(rnd(O_ref)))   element-wise,
       where rnd() rounds the fp64 oracle to the output dtype (nearest even)
       and ulp() is the spacing of that dtype at that magnitude.  Below
       |O| = 0.5 in bf16 (and everywhere in fp16 for |O| < 2) this is the
       plain 2e-3 bound; above it, one output ulp is already larger than 2e-3
       and two correct roundings of nearly equal values can differ by one ulp.
  LSE: |LSE_gpu - LSE_ref| <= 1e-3, and -inf exactly where the oracle has -inf.
"""
from __future__ import annotations

import math

import numpy as np
import torch

O_ABS_TOL = 2e-3
LSE_ABS_TOL = 1e-3

_MANT = {torch.float16: 10, torch.bfloat16: 7}
_EMIN = {torch.float16: -14, torch.bfloat16: -126}


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of `dtype` numbers at |x| (x already representable in dtype)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, _EMIN[dtype])
    return np.exp2(e - _MANT[dtype])


def round_to(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).to(torch.float64).numpy()


def compare(o_gpu, o_ref: np.ndarray, lse_gpu, lse_ref: np.ndarray, dtype: torch.dtype, what: str = ""):
    """Assert parity; returns a dict of error statistics for reporting."""
    og = o_gpu.detach().to("cpu").to(torch.float64).numpy() if isinstance(o_gpu, torch.Tensor) else o_gpu
    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(og.shape)
    assert np.isfinite(og).all(), f"{what}: non-finite O"
    rr = round_to(o_ref, dtype)
    tol = np.maximum(O_ABS_TOL, ulp(rr, dtype))
    err = np.abs(og - rr)
    bad = err > tol
    stats = {"o_max_err_vs_rounded": float(err.max(initial=0.0)),
             "o_max_err_vs_fp64": float(np.abs(og - o_ref).max(initial=0.0)),
             "o_over_2e-3": int((np.abs(og - o_ref) > O_ABS_TOL).sum())}
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} O elements out of tolerance; worst at {idx}: "
                             f"gpu={og[idx]!r} ref={o_ref[idx]!r} tol={tol[idx]!r}")
    if lse_gpu is not None:
        lg = lse_gpu.detach().to("cpu").to(torch.float64).numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        lr = np.asarray(lse_ref, dtype=np.float64).reshape(lg.shape)
        fin = np.isfinite(lr)
        assert (np.isneginf(lg) == np.isneginf(lr)).all(), f"{what}: -inf LSE pattern differs"
        assert np.isfinite(lg[fin]).all(), f"{what}: non-finite LSE"
        lerr = np.abs(lg[fin] - lr[fin])
        stats["lse_max_err"] = float(lerr.max(initial=0.0))
        assert stats["lse_max_err"] <= LSE_ABS_TOL, f"{what}: LSE error {stats['lse_max_err']}"
    return stats


def sdpa_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
