"""fa_fwd_varlen and fa_fwd_varlen_ws (packed variable-length batches) against
the fp64 oracle.

Each sequence is its own attention problem: q, o packed as [total_q, H, d],
k, v as [total_k, H_kv, d], lse as [H, total_q], sequence boundaries in
cu_seqlens_q / cu_seqlens_k.  fa_fwd_varlen launches a grid sized by the
longest sequence; fa_fwd_varlen_ws launches over a device-built list of the row
blocks that hold rows (the binding's default, plan=True).
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


def _packed(lens_q, lens_k, H, H_kv, d, dtype, seed):
    total_q, total_k = sum(lens_q), sum(lens_k)
    q, _, _ = attn_inputs.make_qkv(1, total_q, H, 1, d, dtype, seed, "cuda")
    _, k, v = attn_inputs.make_qkv(1, total_k, 1, H_kv, d, dtype, seed + 5, "cuda")
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    return q[0].contiguous(), k[0].contiguous(), v[0].contiguous(), cu_q, cu_k


CASES = [
    # lens_q, lens_k, H, H_kv, d, dtype, causal
    ([1, 127, 128, 129, 300], None, 4, 4, 128, "bf16", True),
    ([1, 127, 128, 129, 300], None, 4, 2, 64, "f16", False),
    ([513, 7, 256], [600, 7, 100], 2, 1, 128, "bf16", True),     # Nq != Nk per sequence, some rows see no key
    ([64, 0, 200], [64, 50, 0], 4, 2, 128, "bf16", False),        # an empty sequence and a keyless one
    ([1000, 1, 333, 2048], None, 8, 2, 128, "bf16", True),
    # 100 short sequences, lengths 0..300 (two of them empty)
    ([int(x) for x in np.random.default_rng(5).integers(0, 301, 100)], None, 2, 1, 64, "bf16", True),
]


def _case_id(c):
    lens = "-".join(map(str, c[0])) if len(c[0]) <= 6 else f"{len(c[0])}seqs"
    return f"q{lens}_H{c[2]}kv{c[3]}_d{c[4]}{c[5]}{'c' if c[6] else ''}"


@pytest.mark.parametrize("plan", [True, False], ids=["planned", "grid"])
@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_varlen(fa, case, plan):
    lens_q, lens_k, H, H_kv, d, dtype, causal = case
    lens_k = lens_k or lens_q
    q, k, v, cu_q, cu_k = _packed(lens_q, lens_k, H, H_kv, d, dtype, 100 + sum(lens_q) % 89)
    o, lse = fa.fwd_varlen(q, k, v, cu_q, cu_k, max(lens_q), causal=causal, plan=plan)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention_varlen(q, k, v, cu_q.cpu(), cu_k.cpu(), causal, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, q.dtype, f"varlen {'planned' if plan else 'grid'} {case}")


BENCH_LENS = [424, 356, 1647, 312, 625, 6797, 744, 427, 5051, 6597, 2127, 326, 1395, 1870, 318, 7539]


@pytest.mark.parametrize("lens,H,H_kv,d,causal", [
    ([1, 127, 128, 129, 300], 4, 4, 128, True),
    ([64, 0, 200], 4, 2, 64, False),
    ([int(x) for x in np.random.default_rng(5).integers(0, 301, 100)], 2, 1, 64, True),
    (BENCH_LENS, 32, 32, 128, True),
], ids=["ragged", "empty_seq", "100seqs", "bench_batch"])
def test_planned_equals_grid_bit_for_bit(fa, lens, H, H_kv, d, causal):
    """The work list only changes which CTA computes a row block, not how: both
    launches give the same bits (the benchmarked batch of 16 sequences included)."""
    q, k, v, cu, _ = _packed(lens, lens, H, H_kv, d, "bf16", 7)
    o_ref, l_ref = fa.fwd_varlen(q, k, v, cu, cu, max(lens), causal=causal, plan=False)
    ws = torch.full((fa.fwd_varlen_workspace_bytes(len(lens), sum(lens)),), 0xAB, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call runs over the first call's list
        o, l = fa.fwd_varlen(q, k, v, cu, cu, causal=causal, workspace=ws)
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_the_dense_kernel_bit_for_bit(fa, causal):
    """Packed sequences of one length are a dense batch; keys past a sequence end
    get weight exactly 0, so the outputs agree to the bit."""
    B, H, N, d = 3, 4, 300, 128
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 111, "cuda")
    o_dense, l_dense = fa.fwd(q, k, v, causal=causal)
    pack = lambda x: x.transpose(1, 2).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    for plan in (True, False):
        o, lse = fa.fwd_varlen(pack(q), pack(k), pack(v), cu, cu, N, causal=causal, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(o, pack(o_dense))
        assert torch.equal(lse, l_dense.transpose(0, 1).reshape(H, B * N))


def test_rejects_bad_arguments(fa):
    q, k, v, cu_q, cu_k = _packed([10, 20], [10, 20], 2, 2, 64, "bf16", 5)
    with pytest.raises(fa.FaError) as e:
        fa.fwd_varlen(q, k, v, cu_q, cu_k, 0, plan=False)   # max_seqlen_q must be >= 1
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FaError) as e:
        fa.fwd_varlen(q, k, v, cu_q, cu_k, 31, plan=False)  # more than total_q
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    short = torch.empty(fa.fwd_varlen_workspace_bytes(2, 30) - 8, dtype=torch.uint8, device="cuda")
    lib = fa.load_library()
    rc = lib.fa_fwd_varlen_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), None, cu_q.data_ptr(),
                              cu_k.data_ptr(), 2, 30, 30, 2, 2, 64, 0, 0.125, 1, short.data_ptr(), short.numel(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_WORKSPACE                        # a workspace one pair short
    assert fa.get_device_status() == fa.FA_OK
