"""Grouped-query attention (fa_fwd_gqa, fa_fwd_splitkv_gqa) against the fp64 oracle.

H query heads share H_kv K/V heads, H // H_kv consecutive query heads per K/V
head ("Flash Attention (4)" §5); H_kv = 1 is multi-query attention.  The oracle
side is oracle.attention_gqa (each query row against its group's K/V head).
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs
import oracle
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    oracle.set_threads(16)
    return fa


def _inputs(B, H, H_kv, Nq, Nk, d, dtype, seed):
    q, _, _ = attn_inputs.make_qkv(B, H, Nq, 1, d, dtype, seed, "cuda")
    _, k, v = attn_inputs.make_qkv(B, H_kv, 1, Nk, d, dtype, seed + 7, "cuda")
    return q, k, v


FWD = [
    # B, H, H_kv, Nq, Nk, d, dtype, causal
    (2, 8, 2, 300, 300, 128, "bf16", True),
    (1, 8, 1, 257, 513, 64, "f16", False),     # multi-query, ragged tails
    (2, 6, 3, 128, 128, 64, "bf16", True),
    (1, 16, 4, 520, 200, 128, "bf16", True),   # Nq > Nk: early rows see no key
    (1, 32, 8, 1024, 1024, 128, "bf16", True),
    # d = 64 grids of a few waves, run two CTAs per SM: causal (the group's heads
    # mapped to their K/V head in the kernel) and non-causal (the group's rows
    # merged into one head of 4 x 1000 rows)
    (4, 16, 4, 1000, 1000, 64, "f16", True),
    (4, 16, 4, 1000, 1000, 64, "bf16", False),
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: "B{}H{}Hkv{}Nq{}Nk{}d{}{}{}".format(*c[:7], "c" if c[7] else ""))
def test_fwd_gqa(fa, case):
    B, H, H_kv, Nq, Nk, d, dtype, causal = case
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, d, dtype, 50 + Nq + H_kv)
    o, lse = fa.fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention_gqa(q, k, v, causal, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, q.dtype, f"gqa fwd {case}")


def test_fwd_gqa_entry_point_with_one_kv_head_per_query_head_is_fa_fwd(fa):
    q, k, v = attn_inputs.make_qkv(2, 4, 200, 200, 128, "bf16", 61, "cuda")
    o1, l1 = fa.fwd(q, k, v, causal=True)
    lib = fa.load_library()
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    rc = lib.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), 2, 4, 4, 200, 200,
                        128, 1, 1 / math.sqrt(128), fa.FA_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_gqa_sampled_rows_of_a_large_head_group(fa):
    """B=1, H=32 query heads over H_kv=4 K/V heads, N=8192, d=128, causal: sampled rows."""
    B, H, H_kv, N, d = 1, 32, 4, 8192, 128
    q, k, v = _inputs(B, H, H_kv, N, N, d, "bf16", 71)
    o, lse = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    pairs = attn_inputs.sample_rows(N, B * H, 96, seed=5)
    o_ref, lse_ref = oracle.sampled_rows(q, k, v, pairs, True, 1 / math.sqrt(d))
    of = o.reshape(B * H, N, d)
    lf = lse.reshape(B * H, N)
    got_o = torch.stack([of[bh, r] for bh, r in pairs])
    got_l = torch.stack([lf[bh, r] for bh, r in pairs])
    compare(got_o, o_ref, got_l, lse_ref, q.dtype, "gqa sampled rows")


SPLIT = [
    # B, H, H_kv, Nq, Nk, d, dtype, causal, num_splits
    (4, 32, 8, 1, 4096, 128, "bf16", False, 8),
    (2, 8, 1, 3, 1000, 64, "f16", True, 5),
    (2, 16, 4, 1, 16384, 128, "bf16", False, 0),   # automatic split count
]


@pytest.mark.parametrize("case", SPLIT, ids=lambda c: "B{}H{}Hkv{}Nq{}Nk{}d{}{}{}S{}".format(*c[:7], "c" if c[7] else "", c[8]))
def test_splitkv_gqa(fa, case):
    B, H, H_kv, Nq, Nk, d, dtype, causal, S = case
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, d, dtype, 80 + Nk % 97 + H_kv)
    o, lse = fa.fwd_splitkv(q, k, v, causal=causal, num_splits=S)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention_gqa(q, k, v, causal, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, q.dtype, f"gqa split-KV {case}")


def test_splitkv_gqa_matches_fused_forward(fa):
    """The two GQA entry points agree on a prefill-shaped problem."""
    q, k, v = _inputs(1, 8, 2, 256, 700, 128, "bf16", 91)
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd_splitkv(q, k, v, causal=True, num_splits=3)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3
