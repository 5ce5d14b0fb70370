"""fa_fwd_splitkv_noalloc: the split-KV forward that allocates nothing.

Some callers cannot allocate device memory when they call the library (code
recorded into a CUDA graph, runtimes without a device allocator, services that
fix their memory footprint at start-up).  This entry point keeps the split
partials in the library's own 16 MiB scratch array instead of a workspace.
These tests call it through the C ABI and check it against fa_fwd_splitkv (the
entry point with a caller workspace), twice in a row with different shapes so
that the second call runs over the first call's leftovers in the scratch.  Both
entry points run the same split and combine kernels with the same split count,
so their outputs must be equal bit for bit; each case is also checked against
the fp64 oracle.

The file name makes pytest collect it last.
"""
import math

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
    return fa


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, num_splits
    (4, 8, 1, 4096, 128, "bf16", False, 8),
    (2, 4, 3, 1000, 64, "f16", True, 5),
]


def _against_workspace_version(fa, case):
    B, H, Nq, Nk, d, dtype, causal, S = case
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, 17 * Nk + S, "cuda")
    o_ref, lse_ref = fa.fwd_splitkv(q, k, v, causal=causal, num_splits=S)
    o, lse = fa.fwd_splitkv_noalloc(q, k, v, causal=causal, num_splits=S)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    assert torch.equal(o, o_ref), f"noalloc {case}: O differs from the workspace entry point"
    assert torch.equal(lse, lse_ref), f"noalloc {case}: LSE differs from the workspace entry point"
    o64, lse64 = oracle.attention(q, k, v, causal, 1.0 / math.sqrt(d))
    compare(o, o64, lse, lse64, q.dtype, f"noalloc {case} vs oracle")


def test_two_calls_in_a_row_match_workspace_entry_point(fa):
    assert fa.load_library().fa_splitkv_noalloc_capacity_bytes() == 16 << 20
    for case in CASES:
        _against_workspace_version(fa, case)


def test_oversize_problem_is_rejected_before_launch(fa):
    # 256 splits x 128 rows x (128 + 1) fp32 values is just over 16 MiB.
    q, k, v = attn_inputs.make_qkv(1, 128, 1, 64, 128, "bf16", 3, "cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd_splitkv_noalloc(q, k, v, num_splits=256)
    assert e.value.code == fa.FA_ERR_SCRATCH_LIMIT
    assert fa.get_device_status() == fa.FA_OK
