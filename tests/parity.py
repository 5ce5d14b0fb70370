"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerance (written out once, used by every GPU parity test):
  O:   |O_gpu - rnd(O_ref)| <= max(2e-3, ulp(rnd(O_ref)))   element-wise,
       where rnd() rounds the fp64 oracle to the output dtype (nearest even)
       and ulp() is the spacing of that dtype at that magnitude.  Below
       |O| = 0.5 in bf16 (and everywhere in fp16 for |O| < 2) this is the
       plain 2e-3 bound; above it, one output ulp is already larger than 2e-3
       and two correct roundings of nearly equal values can differ by one ulp.
  Where half an output ulp leaves room for it, the literal bound holds against
  the unrounded fp64 oracle as well: |O_gpu - O_ref| <= 2e-3 for every fp16
  element with |O_ref| < 2 (half an ulp there is at most 2^-11 = 4.9e-4) and
  every bf16 element with |O_ref| < 0.25 (at most 2^-11 as well).
  LSE: |LSE_gpu - LSE_ref| <= 1e-3, and -inf exactly where the oracle has -inf.

Every comparison's error statistics are appended to RECORDS; the test
session prints them at its end (tests/conftest.py).
"""
from __future__ import annotations

import math

import numpy as np
import torch

O_ABS_TOL = 2e-3
LSE_ABS_TOL = 1e-3

# |O_ref| below which the literal 2e-3 bound is asserted against unrounded fp64
LITERAL_BELOW = {torch.float16: 2.0, torch.bfloat16: 0.25}
RECORDS: list[tuple[str, dict]] = []

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
    err64 = np.abs(og - o_ref)
    lit = np.abs(o_ref) < LITERAL_BELOW[dtype]
    stats = {"o_max_err_vs_rounded": float(err.max(initial=0.0)),
             "o_max_err_vs_fp64": float(err64.max(initial=0.0)),
             "o_max_err_vs_fp64_literal_region": float(err64[lit].max(initial=0.0)),
             "o_over_2e-3": int((err64 > O_ABS_TOL).sum()), "o_elements": int(err64.size),
             "o_literal_elements": int(lit.sum())}
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} O elements out of tolerance; worst at {idx}: "
                             f"gpu={og[idx]!r} ref={o_ref[idx]!r} tol={tol[idx]!r}")
    bad_lit = lit & (err64 > O_ABS_TOL)
    if bad_lit.any():
        idx = np.unravel_index(np.argmax(np.where(lit, err64, 0.0)), err64.shape)
        raise AssertionError(f"{what}: {int(bad_lit.sum())} O elements with |O_ref| < {LITERAL_BELOW[dtype]} are "
                             f"more than 2e-3 from the fp64 oracle; worst at {idx}: gpu={og[idx]!r} ref={o_ref[idx]!r}")
    if lse_gpu is not None:
        lg = lse_gpu.detach().to("cpu").to(torch.float64).numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        lr = np.asarray(lse_ref, dtype=np.float64).reshape(lg.shape)
        fin = np.isfinite(lr)
        assert (np.isneginf(lg) == np.isneginf(lr)).all(), f"{what}: -inf LSE pattern differs"
        assert np.isfinite(lg[fin]).all(), f"{what}: non-finite LSE"
        lerr = np.abs(lg[fin] - lr[fin])
        stats["lse_max_err"] = float(lerr.max(initial=0.0))
        assert stats["lse_max_err"] <= LSE_ABS_TOL, f"{what}: LSE error {stats['lse_max_err']}"
    RECORDS.append((what, stats))
    return stats


def sdpa_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# ---------------------------------------------------------------- backward
#
# Tolerance of the gradients, from the arithmetic of the kernel.  With inputs
# exactly representable in the 16-bit type and fp32 accumulation, the rounding
# steps are: P to 16 bits (for dV), dS to 16 bits (for dK, dQ), D computed from
# the 16-bit forward output O, and the final rounding of each gradient.  Each is
# a relative error of at most u/2 (u = 2^-8 for bf16, 2^-11 for fp16) of the
# rounded value, so with the magnitudes
#     mag_dV = P^T |dO|,
#     mag_dS = P o (|dP| + rowsum(|dO| o |O|)),
#     mag_dK = scale mag_dS^T |Q|,   mag_dQ = scale mag_dS |K|,
# every element satisfies |g_gpu - g_ref| <= u/2 (mag_g + |g_ref|) plus fp32
# accumulation terms far below that.  The test allows twice that much,
#     |g_gpu - g_ref| <= u (mag_g + |g_ref|) + floor,
# where floor covers fp16 subnormals (P or dS below 2^-14 keep an absolute
# error up to 2^-25): floor = 2^-25 x (number of summed terms) x max|operand|.

GRAD_U = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def grad_magnitudes(q, k, v, o, dout, lse, causal: bool, scale: float):
    """(mag_dq, mag_dk, mag_dv) in fp64 for [BH, N, d] numpy arrays (lse [BH, Nq])."""
    Nq, Nk = q.shape[-2], k.shape[-2]
    allowed = np.ones((Nq, Nk), dtype=bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    mags = [np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)]
    for b in range(q.shape[0]):
        s = scale * (q[b] @ k[b].T)
        with np.errstate(invalid="ignore", over="ignore"):
            p = np.exp(s - lse[b][:, None])
        p = np.where(allowed & np.isfinite(lse[b])[:, None], p, 0.0)
        del s
        dp = np.abs(dout[b] @ v[b].T)
        mag_d = (np.abs(dout[b]) * np.abs(o[b])).sum(axis=1)
        mag_ds = p * (dp + mag_d[:, None])
        del dp
        mags[0][b] = scale * (mag_ds @ np.abs(k[b]))
        mags[1][b] = scale * (mag_ds.T @ np.abs(q[b]))
        mags[2][b] = p.T @ np.abs(dout[b])
    return tuple(mags)


def compare_grads(got, ref, mags, floors, dtype: torch.dtype, what: str = ""):
    """Assert |g_gpu - g_ref| <= u (mag + |g_ref|) + floor for g in (dq, dk, dv)."""
    u = GRAD_U[dtype]
    stats = {}
    for name, g, r, m, fl in zip(("dq", "dk", "dv"), got, ref, mags, floors):
        gg = g.detach().to("cpu").to(torch.float64).numpy().reshape(r.shape)
        assert np.isfinite(gg).all(), f"{what}: non-finite {name}"
        err = np.abs(gg - r)
        tol = u * (m + np.abs(r)) + fl
        stats[name + "_max_err"] = float(err.max(initial=0.0))
        ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
        stats[name + "_max_err_over_tol"] = float(ratio.max(initial=0.0))
        bad = err > tol
        if bad.any():
            idx = np.unravel_index(np.argmax(ratio), err.shape)
            raise AssertionError(f"{what}: {int(bad.sum())} {name} elements out of tolerance; worst at {idx}: "
                                 f"gpu={gg[idx]!r} ref={r[idx]!r} tol={tol[idx]!r}")
    return stats
