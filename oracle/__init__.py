"""Python binding of the fp64 CPU attention oracle (``attn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports this module and this module never imports the CUDA library.

``build()`` compiles ``attn_oracle.c`` with the system C compiler into
``oracle/_build/libattn_oracle.so`` (OpenMP when available, no fast-math).
All entry points take and return float64 numpy arrays; 16-bit inputs are
widened exactly by ``to_f64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libattn_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile the oracle shared library; returns its path.

    ``src``/``out`` let a test compile a modified copy of the source elsewhere.
    """
    src = src or _SRC
    out = out or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def _bind(lib):
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = ctypes.c_int
    lib.oracle_has_openmp.argtypes = []
    lib.oracle_has_openmp.restype = ctypes.c_int
    lib.oracle_attn_full.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, _dp, _dp]
    lib.oracle_attn_full.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double, _dp, _dp, _dp]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [_dp, _i64p, _i64p, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_tiled.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, _dp, _dp]
    lib.oracle_attn_tiled.restype = ctypes.c_int
    lib.oracle_attn_split_partials.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                               ctypes.c_long, _dp, _dp]
    lib.oracle_attn_split_partials.restype = ctypes.c_int
    lib.oracle_combine.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_long, ctypes.c_int, _dp, _dp]
    lib.oracle_combine.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library. A ``path`` loads a separate copy."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def set_threads(n: int) -> int:
    return load().oracle_set_threads(int(n))


def has_openmp() -> bool:
    return bool(load().oracle_has_openmp())


def to_f64(x) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype) or array to contiguous float64 numpy."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu").to(torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_dp)


def attention(q, k, v, causal: bool, scale: float, lib=None):
    """Exact attention.  q: [..., Nq, d], k, v: [..., Nk, d] -> (O [..., Nq, d], LSE [..., Nq])."""
    lib = lib or load()
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(lead + (Nq,), dtype=np.float64)
    rc = lib.oracle_attn_full(_p(q), _p(k), _p(v), BH, Nq, Nk, d, int(bool(causal)), float(scale), _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_full failed ({rc})")
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float, lib=None):
    """Gradients (dQ, dK, dV) of O = softmax(scale * Q K^T + mask) V for the given dO
    ("Lecture 25" §3.3).  q, dout: [..., Nq, d]; k, v: [..., Nk, d]."""
    lib = lib or load()
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    rc = lib.oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dout), BH, Nq, Nk, d, int(bool(causal)), float(scale),
                             _p(dq), _p(dk), _p(dv))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd failed ({rc})")
    return dq, dk, dv


def attention_tiled(q, k, v, causal: bool, scale: float, Br: int, Bc: int, lib=None):
    """The online-softmax loop of "6.2 FlashAttention V2 explained" §6 in fp64 (for the
    tiled == full invariant)."""
    lib = lib or load()
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(lead + (Nq,), dtype=np.float64)
    rc = lib.oracle_attn_tiled(_p(q), _p(k), _p(v), BH, Nq, Nk, d, int(bool(causal)), float(scale),
                               int(Br), int(Bc), _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_tiled failed ({rc})")
    return o, lse


def split_partials(q, k, v, causal: bool, scale: float, num_splits: int, split_len: int, lib=None):
    """Per-split normalised partials: (O_s [S, ..., Nq, d], LSE_s [S, ..., Nq])."""
    lib = lib or load()
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    o = np.zeros((num_splits,) + q.shape, dtype=np.float64)
    lse = np.zeros((num_splits,) + lead + (Nq,), dtype=np.float64)
    rc = lib.oracle_attn_split_partials(_p(q), _p(k), _p(v), BH, Nq, Nk, d, int(bool(causal)), float(scale),
                                        int(num_splits), int(split_len), _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_split_partials failed ({rc})")
    return o, lse


def combine(o_part, lse_part, lib=None):
    """LSE-weighted merge.  o_part: [S, ..., d], lse_part: [S, ...] -> (O [..., d], LSE [...])."""
    lib = lib or load()
    o_part, lse_part = to_f64(o_part), to_f64(lse_part)
    S = o_part.shape[0]
    d = o_part.shape[-1]
    rows = int(np.prod(o_part.shape[1:-1])) if o_part.ndim > 2 else 1
    o = np.zeros(o_part.shape[1:], dtype=np.float64)
    lse = np.zeros(lse_part.shape[1:], dtype=np.float64)
    rc = lib.oracle_combine(_p(o_part), _p(lse_part), S, rows, d, _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_combine failed ({rc})")
    return o, lse


def attention_rows(q_rows, row_index, kv_slot, k, v, Nq: int, causal: bool, scale: float, lib=None):
    """Selected rows.  q_rows: [n, d]; row_index, kv_slot: [n] ints; k, v: [slots, Nk, d]."""
    lib = lib or load()
    q_rows, k, v = to_f64(q_rows), to_f64(k), to_f64(v)
    ri = np.ascontiguousarray(np.asarray(row_index, dtype=np.int64))
    ks = np.ascontiguousarray(np.asarray(kv_slot, dtype=np.int64))
    n, d = q_rows.shape
    Nk = k.shape[-2]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_attn_rows(_p(q_rows), ri.ctypes.data_as(_i64p), ks.ctypes.data_as(_i64p), _p(k), _p(v),
                              n, int(Nq), Nk, d, int(bool(causal)), float(scale), _p(o), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed ({rc})")
    return o, lse


def kv_head_of(bh: int, H: int, H_kv: int) -> int:
    """K/V head read by query head bh = b*H + h under grouped-query attention:
    H // H_kv consecutive query heads share one K/V head, so it is b*H_kv + h // (H // H_kv)
    ("Flash Attention (4)" §5: the K/V index mapped per group of query heads)."""
    return (bh // H) * H_kv + (bh % H) // (H // H_kv)


def attention_gqa(q, k, v, causal: bool, scale: float, lib=None):
    """Exact grouped-query attention.  q: [B, H, Nq, d]; k, v: [B, H_kv, Nk, d] with H_kv
    dividing H -> (O [B, H, Nq, d], LSE [B, H, Nq]).  Every query row is the plain
    definition (attention_rows) against the K/V head of its group; H_kv = H is
    multi-head attention and H_kv = 1 multi-query attention."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, Nq, d = q64.shape
    H_kv, Nk = k64.shape[1], k64.shape[2]
    if H_kv <= 0 or H % H_kv != 0 or k64.shape != v64.shape or k64.shape[0] != B or k64.shape[3] != d:
        raise ValueError("attention_gqa: k, v must be [B, H_kv, Nk, d] with H_kv dividing H")
    bh = np.repeat(np.arange(B * H), Nq)
    rows = np.tile(np.arange(Nq), B * H)
    slots = np.array([kv_head_of(int(x), H, H_kv) for x in range(B * H)], dtype=np.int64)[bh]
    o, lse = attention_rows(q64.reshape(B * H * Nq, d), rows, slots, k64.reshape(B * H_kv, Nk, d),
                            v64.reshape(B * H_kv, Nk, d), Nq, causal, scale, lib=lib)
    return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)


def attention_bwd_gqa(q, k, v, dout, causal: bool, scale: float, lib=None):
    """Gradients of grouped-query attention ("Lecture 25" §3.3 per query head;
    "Flash Attention (4)" §5 for the head mapping).  q, dout: [B, H, Nq, d]; k, v:
    [B, H_kv, Nk, d].  Each query head's gradients are those of plain attention
    against its group's K/V head; a K/V head's dK, dV are the sums over the query
    heads that read it.  Returns (dQ [B, H, Nq, d], dK, dV [B, H_kv, Nk, d])."""
    q64, k64, v64, g64 = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, H, Nq, d = q64.shape
    H_kv, Nk = k64.shape[1], k64.shape[2]
    if H_kv <= 0 or H % H_kv != 0:
        raise ValueError("attention_bwd_gqa: H_kv must divide H")
    group = H // H_kv
    k_rep = np.repeat(k64, group, axis=1)  # query head h reads K/V head h // group
    v_rep = np.repeat(v64, group, axis=1)
    dq, dk_rep, dv_rep = attention_bwd(q64.reshape(B * H, Nq, d), k_rep.reshape(B * H, Nk, d),
                                       v_rep.reshape(B * H, Nk, d), g64.reshape(B * H, Nq, d), causal, scale, lib=lib)
    dk = dk_rep.reshape(B, H_kv, group, Nk, d).sum(axis=2)
    dv = dv_rep.reshape(B, H_kv, group, Nk, d).sum(axis=2)
    return dq.reshape(B, H, Nq, d), dk, dv


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float, lib=None):
    """Exact attention of a packed variable-length batch.  q: [total_q, H, d], k, v:
    [total_k, H_kv, d], cu_seqlens_q/k: num_seqs + 1 token offsets.  Sequence s is
    its own problem (attention_gqa on tokens [cu_q[s], cu_q[s+1]) of q and
    [cu_k[s], cu_k[s+1]) of k and v, causal diagonal at its bottom-right corner);
    a row with no key gets O = 0, LSE = -inf.  Returns (O [total_q, H, d], LSE [H, total_q])."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    cq = [int(x) for x in np.asarray(to_f64(cu_seqlens_q))]
    ck = [int(x) for x in np.asarray(to_f64(cu_seqlens_k))]
    total_q, H, d = q64.shape
    o = np.zeros_like(q64)
    lse = np.full((H, total_q), -np.inf)
    for s in range(len(cq) - 1):
        q_s = q64[cq[s]:cq[s + 1]]
        k_s, v_s = k64[ck[s]:ck[s + 1]], v64[ck[s]:ck[s + 1]]
        if q_s.shape[0] == 0 or k_s.shape[0] == 0:
            continue  # no rows, or rows that see no key (O = 0, LSE = -inf)
        o_s, l_s = attention_gqa(np.ascontiguousarray(q_s.transpose(1, 0, 2))[None],
                                 np.ascontiguousarray(k_s.transpose(1, 0, 2))[None],
                                 np.ascontiguousarray(v_s.transpose(1, 0, 2))[None], causal, scale, lib=lib)
        o[cq[s]:cq[s + 1]] = o_s[0].transpose(1, 0, 2)
        lse[:, cq[s]:cq[s + 1]] = l_s[0]
    return o, lse


def attention_bwd_varlen(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float, lib=None):
    """Gradients of a packed variable-length batch (layouts as attention_varlen; dout
    like q): every sequence is its own problem (attention_bwd_gqa on its tokens), and
    keys of a sequence with no query rows get zero gradients.
    Returns (dQ [total_q, H, d], dK, dV [total_k, H_kv, d])."""
    q64, k64, v64, g64 = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    cq = [int(x) for x in np.asarray(to_f64(cu_seqlens_q))]
    ck = [int(x) for x in np.asarray(to_f64(cu_seqlens_k))]
    dq, dk, dv = np.zeros_like(q64), np.zeros_like(k64), np.zeros_like(v64)
    tr = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))[None]
    for s in range(len(cq) - 1):
        q_s, g_s = q64[cq[s]:cq[s + 1]], g64[cq[s]:cq[s + 1]]
        k_s, v_s = k64[ck[s]:ck[s + 1]], v64[ck[s]:ck[s + 1]]
        if q_s.shape[0] == 0 or k_s.shape[0] == 0:
            continue
        a, b, c = attention_bwd_gqa(tr(q_s), tr(k_s), tr(v_s), tr(g_s), causal, scale, lib=lib)
        dq[cq[s]:cq[s + 1]] = a[0].transpose(1, 0, 2)
        dk[ck[s]:ck[s + 1]] = b[0].transpose(1, 0, 2)
        dv[ck[s]:ck[s + 1]] = c[0].transpose(1, 0, 2)
    return dq, dk, dv


def sampled_rows(q, k, v, pairs, causal: bool, scale: float, heads_per_batch: int = 16):
    """Oracle values for the (bh, row) pairs of ``[B, H, N, d]`` tensors (any device).

    Only the heads that appear in ``pairs`` are copied to the host, a few at a
    time, so that large workloads stay within host memory.
    Returns (O [n, d], LSE [n]) in the order of ``pairs``.
    """
    d = q.shape[-1]
    Nq = q.shape[-2]
    H, H_kv = q.shape[1], k.shape[1]  # H_kv < H: grouped-query attention (kv_head_of)
    qf = q.reshape(-1, Nq, d)
    kf = k.reshape(-1, k.shape[-2], d)
    vf = v.reshape(-1, v.shape[-2], d)
    by_bh: dict[int, list[int]] = {}
    for n, (bh, _r) in enumerate(pairs):
        by_bh.setdefault(int(bh), []).append(n)
    o = np.zeros((len(pairs), d))
    lse = np.zeros((len(pairs),))
    bhs = sorted(by_bh)
    for s in range(0, len(bhs), heads_per_batch):
        group = bhs[s:s + heads_per_batch]
        kk = np.stack([to_f64(kf[kv_head_of(bh, H, H_kv)]) for bh in group])
        vv = np.stack([to_f64(vf[kv_head_of(bh, H, H_kv)]) for bh in group])
        idx, rows, slots, qr = [], [], [], []
        for slot, bh in enumerate(group):
            for n in by_bh[bh]:
                idx.append(n)
                rows.append(pairs[n][1])
                slots.append(slot)
                qr.append(to_f64(qf[bh, pairs[n][1]]))
        oo, ll = attention_rows(np.stack(qr), rows, slots, kk, vv, Nq, causal, scale)
        o[idx] = oo
        lse[idx] = ll
    return o, lse


class WidenedWorkload:
    """A workload's Q, K and V widened to fp64 once, for repeated row queries.

    ``sampled_rows`` widens the heads it touches on every call; a caller that
    evaluates many row samples of one workload (a timing loop) widens once
    here, gathers each sample's query rows with ``gather`` and then calls
    ``rows``, whose only work is the oracle's own arithmetic (attention_rows:
    the plain definition per row over the row's full key range).
    q: [B, H, Nq, d]; k, v: [B, H_kv, Nk, d] (H_kv divides H).
    """

    def __init__(self, q, k, v):
        self.Nq, self.d = int(q.shape[-2]), int(q.shape[-1])
        self.H, self.H_kv = int(q.shape[1]), int(k.shape[1])
        self.q = to_f64(q).reshape(-1, self.Nq, self.d)
        self.k = to_f64(k).reshape(-1, int(k.shape[-2]), self.d)
        self.v = to_f64(v).reshape(-1, int(v.shape[-2]), self.d)

    def gather(self, pairs):
        """(query rows [n, d], row indices [n], K/V head slots [n]) of the (bh, row) pairs."""
        a = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
        bh, rows = a[:, 0], a[:, 1]
        slots = (bh // self.H) * self.H_kv + (bh % self.H) // (self.H // self.H_kv)  # kv_head_of, vectorised
        return np.ascontiguousarray(self.q[bh, rows]), np.ascontiguousarray(rows), np.ascontiguousarray(slots)

    def rows(self, gathered, causal: bool, scale: float):
        """Oracle (O [n, d], LSE [n]) of gathered rows."""
        q_rows, rows, slots = gathered
        return attention_rows(q_rows, rows, slots, self.k, self.v, self.Nq, causal, scale)
