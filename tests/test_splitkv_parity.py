"""fa_fwd_splitkv (split partials + combine) and fa_splitkv_combine against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import attn_inputs
import oracle
from parity import compare, round_to, ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    oracle.set_threads(16)
    return fa


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, num_splits
    (2, 3, 1, 1000, 128, "bf16", False, 8),
    (1, 4, 1, 16384, 128, "bf16", False, 16),
    (2, 2, 1, 333, 64, "f16", False, 3),
    (1, 2, 1, 65, 128, "bf16", False, 32),   # more splits than tiles: empty splits
    (1, 1, 1, 1, 64, "bf16", False, 1),
    (2, 2, 5, 700, 128, "bf16", True, 4),    # several rows, causal bottom-right
    (1, 2, 40, 30, 64, "f16", True, 2),      # Nq > Nk: rows with no key
    (1, 1, 130, 130, 128, "f16", False, 0),  # auto split count
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}_q{}_k{}_d{}_{}_{}_S{}".format(*c[:6], "c" if c[6] else "nc", c[7]))
def test_splitkv_against_oracle(fa, case):
    B, H, Nq, Nk, d, dtype, causal, S = case
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, 11 * Nk + Nq, "cuda")
    o, lse = fa.fwd_splitkv(q, k, v, causal=causal, num_splits=S)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention(q, k, v, causal, 1 / math.sqrt(d))
    compare(o, o_ref, lse, lse_ref, q.dtype, str(case))


@pytest.mark.parametrize("S", [0, 8, 16, 32])
def test_decode_b32h32_nk16384_sampled(fa, S):
    """The decode workload at the benchmark's split counts (0: the automatic choice),
    checked on 256 sampled (b, h) rows, each over its full 16384 keys."""
    w = attn_inputs.WORKLOADS["decode_b32h32_nk16384_d128_bf16"]
    q, k, v = attn_inputs.make_workload(w, "cuda")
    o, lse = fa.fwd_splitkv(q, k, v, causal=False, num_splits=S)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    pairs = attn_inputs.sample_rows(1, w.B * w.H, 256, seed=w.seed + S)
    o_ref, lse_ref = oracle.sampled_rows(q, k, v, pairs, False, w.scale)
    idx = torch.tensor([p[0] for p in pairs], device=o.device)
    compare(o.view(-1, w.d)[idx], o_ref, lse.view(-1)[idx], lse_ref, q.dtype, f"decode S={S}")


def test_partials_match_oracle_partials(fa):
    """The workspace holds each split's normalised (O_s, LSE_s); compare them with the oracle's."""
    B, H, Nq, Nk, d, S = 1, 3, 2, 900, 128, 5
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, "bf16", 41, "cuda")
    ws = fa.splitkv_workspace(q, k, S)
    fa.fwd_splitkv(q, k, v, causal=True, num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    op, lp = fa.workspace_views(ws, B, H, Nq, d, S)
    L = fa.splitkv_split_len(Nk, S)
    assert L % 64 == 0 and L * S >= Nk
    o_ref, lse_ref = oracle.split_partials(q, k, v, True, 1 / math.sqrt(d), S, L)
    og = op.double().cpu().numpy()
    assert np.abs(og - o_ref).max() < 1e-4
    lg = lp.double().cpu().numpy()
    assert (np.isneginf(lg) == np.isneginf(lse_ref)).all()
    fin = np.isfinite(lse_ref)
    assert np.abs(lg[fin] - lse_ref[fin]).max() < 1e-4


def test_combine_of_oracle_partials(fa):
    """fa_splitkv_combine on partials made by the oracle (cast to fp32), including empty splits."""
    B, H, Nq, Nk, d, S = 2, 2, 3, 100, 64, 6
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, "f16", 42, "cpu")
    L = 32
    op, lp = oracle.split_partials(q, k, v, True, 0.3, S, L)  # splits 4, 5 are empty
    o_ref, lse_ref = oracle.combine(op, lp)
    o, lse = fa.splitkv_combine(torch.from_numpy(op).float().cuda().contiguous(),
                                torch.from_numpy(lp).float().cuda().contiguous(), dtype=torch.float16)
    compare(o, o_ref, lse, lse_ref, torch.float16, "combine")


def test_splitkv_equals_fused_forward(fa):
    """The split-KV path and the fused forward on the same causal problem (Nq = 64
    rows against 2048 keys, 7 splits): each within the parity bound of the fp64
    oracle, so the two differ element-wise by at most twice that bound (two output
    ulps above 2e-3)."""
    q, k, v = attn_inputs.make_qkv(2, 2, 64, 2048, 128, "bf16", 43, "cuda")
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd_splitkv(q, k, v, causal=True, num_splits=7)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(q, k, v, True, 1 / math.sqrt(128))
    compare(o1, o_ref, l1, lse_ref, q.dtype, "fused forward, split-KV problem")
    compare(o2, o_ref, l2, lse_ref, q.dtype, "split-KV, 7 splits")
    a, b = o1.double().cpu().numpy(), o2.double().cpu().numpy()
    bound = 2 * np.maximum(2e-3, ulp(round_to(np.asarray(o_ref).reshape(a.shape), q.dtype), q.dtype))
    assert (np.abs(a - b) <= bound).all()
    assert (l1 - l2).abs().max().item() <= 2e-3


def test_workspace_errors(fa):
    q, k, v = attn_inputs.make_qkv(1, 1, 1, 256, 128, "bf16", 44, "cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd_splitkv(q, k, v, num_splits=4, workspace=small)
    assert e.value.code == fa.FA_ERR_WORKSPACE
