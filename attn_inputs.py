"""Seeded synthetic inputs for attention workloads.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmark.  It holds no attention arithmetic: it only draws Q, K, V.

Recipe (the same everywhere): each of Q, K and V gets its own
``torch.Generator`` on the target device, seeded with ``seed + 1``,
``seed + 2`` and ``seed + 3``; values are drawn with ``torch.randn`` in fp32
(standard normal, the distribution the pages' benchmarks use) and then cast
to the 16-bit storage dtype.  Layout is contiguous ``[B, H, N, d]``.

Large tensors are drawn in chunks of whole ``[N, d]`` head slices so that the
fp32 staging buffer stays small; the chunking is deterministic, so the same
(seed, shape, device) always yields the same tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One attention workload: shapes, dtype, masking and seed."""

    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    seed: int
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 means H

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def flops(self) -> float:
        """Forward FLOPs, 4*B*H*Nq*Nk*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2.0 if self.causal else f

    def compulsory_bytes(self) -> int:
        """Bytes every implementation must move: Q, K, V read, O written (16-bit), LSE written (fp32)."""
        e = 2
        q = self.B * self.H * self.Nq * self.d * e
        kv = 2 * self.B * self.kv_heads * self.Nk * self.d * e
        o = q
        lse = self.B * self.H * self.Nq * 4
        return q + kv + o + lse


# The five workloads: sizes and dtypes as the attention-forward benchmark defines them.
WORKLOADS = {
    "tiny_d64_f16": Workload("tiny_d64_f16", 1, 1, 128, 128, 64, "f16", False, 1000),
    "tiny_d64_f16_causal": Workload("tiny_d64_f16_causal", 1, 1, 128, 128, 64, "f16", True, 1000),
    "b4h16_n1024_d64_f16": Workload("b4h16_n1024_d64_f16", 4, 16, 1024, 1024, 64, "f16", False, 2000),
    "b4h16_n1024_d64_f16_causal": Workload("b4h16_n1024_d64_f16_causal", 4, 16, 1024, 1024, 64, "f16", True, 2000),
    "b2h32_n8192_d128_bf16_causal": Workload("b2h32_n8192_d128_bf16_causal", 2, 32, 8192, 8192, 128, "bf16", True, 3000),
    "b2h32_n8192_d128_bf16": Workload("b2h32_n8192_d128_bf16", 2, 32, 8192, 8192, 128, "bf16", False, 3000),
    "b1h32_n32768_d128_bf16_causal": Workload("b1h32_n32768_d128_bf16_causal", 1, 32, 32768, 32768, 128, "bf16", True, 4000),
    "decode_b32h32_nk16384_d128_bf16": Workload("decode_b32h32_nk16384_d128_bf16", 32, 32, 1, 16384, 128, "bf16", False, 5000),
    # Grouped-query decode: 32 query heads over 8 K/V heads (4 per group).
    "decode_b32h32kv8_nk16384_d128_bf16": Workload("decode_b32h32kv8_nk16384_d128_bf16", 32, 32, 1, 16384, 128, "bf16",
                                                   False, 6000, H_kv=8),
}


def _randn(shape, dtype: torch.dtype, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1, shape[-2], shape[-1])  # [B*H, N, d]
    per = shape[-2] * shape[-1]
    chunk = max(1, (1 << 26) // max(per, 1))  # ~64M fp32 elements of staging at most
    for s in range(0, flat.shape[0], chunk):
        e = min(flat.shape[0], s + chunk)
        tmp = torch.randn((e - s, shape[-2], shape[-1]), generator=g, dtype=torch.float32, device=device)
        flat[s:e].copy_(tmp)
        del tmp
    return out


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, dtype="f16", seed: int = 0, device="cpu"):
    """Draw (q, k, v) with the module's recipe. dtype is 'f16', 'bf16' or a torch dtype."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    q = _randn((B, H, Nq, d), tdt, seed + 1, device)
    k = _randn((B, H, Nk, d), tdt, seed + 2, device)
    v = _randn((B, H, Nk, d), tdt, seed + 3, device)
    return q, k, v


def make_dout(B: int, H: int, Nq: int, d: int, dtype="f16", seed: int = 0, device="cpu"):
    """Draw the output gradient dO [B, H, Nq, d] with the same recipe (standard normal)."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return _randn((B, H, Nq, d), tdt, seed + 4, device)


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> list[int]:
    """Seeded sequence lengths, log-uniform in [lo, hi] (a packed batch of mixed
    short and long sequences)."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(num_seqs, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


# Packed variable-length batch: 16 sequences of 256..8192 tokens, 32 heads, d = 128,
# bf16, causal (q and k have the same lengths).
VARLEN_WORKLOAD = {"name": "varlen16_l256-8192_h32_d128_bf16_causal", "num_seqs": 16, "lo": 256, "hi": 8192,
                   "H": 32, "d": 128, "dtype": "bf16", "causal": True, "seed": 7000}


def make_workload(w: Workload, device="cpu"):
    if w.kv_heads == w.H:
        return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, w.seed, device)
    tdt = DTYPES[w.dtype]
    q = _randn((w.B, w.H, w.Nq, w.d), tdt, w.seed + 1, device)
    k = _randn((w.B, w.kv_heads, w.Nk, w.d), tdt, w.seed + 2, device)
    v = _randn((w.B, w.kv_heads, w.Nk, w.d), tdt, w.seed + 3, device)
    return q, k, v


def sample_rows(Nq: int, BH: int, count: int, seed: int, tile: int = 128):
    """A seeded sample of (bh, row) pairs that always includes the tile-boundary rows.

    Always present for bh = 0 and bh = BH - 1: rows 0, 1, tile-1, tile, tile+1,
    Nq-1, and the first and last row of a middle tile (clipped to [0, Nq)).
    The rest are drawn uniformly without replacement, in the order of one
    seeded permutation of all BH * Nq pairs.  Linear in `count`: membership is
    tested against a set.
    """
    g = torch.Generator().manual_seed(seed)
    mid = (Nq // tile // 2) * tile
    fixed_rows = [0, 1, tile - 1, tile, tile + 1, Nq - 1, mid, mid + tile - 1]
    out: list[tuple[int, int]] = []
    seen: set[tuple[int, int]] = set()
    n_fixed = 0
    for bh in sorted({0, BH - 1}):
        for r in fixed_rows:
            if 0 <= r < Nq:
                n_fixed += 1
                if (bh, r) not in seen:
                    seen.add((bh, r))
                    out.append((bh, r))
    total = BH * Nq
    target = min(count, total)
    if len(out) < target:
        # every fixed pair can collide with at most one drawn pair, so this prefix always suffices
        idx = torch.randperm(total, generator=g)[: target - len(out) + n_fixed].tolist()
        for flat in idx:
            p = (flat // Nq, flat % Nq)
            if p not in seen:
                seen.add(p)
                out.append(p)
                if len(out) >= target:
                    break
    return out
