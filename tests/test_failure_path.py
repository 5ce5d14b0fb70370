"""Device-side failure reporting, exercised without a fault: a wait that nothing
completes runs out after a short limit, the host reads FA_ERR_DEVICE_TIMEOUT,
and the same context then runs attention normally."""
import math

import pytest
import torch

import attn_inputs
import oracle
from parity import compare

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_the_context_stays_usable():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    assert fa.get_device_status() == fa.FA_OK
    fa.selftest_timeout(50)
    assert fa.get_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.get_device_status() == fa.FA_OK        # read-and-clear
    q, k, v = attn_inputs.make_qkv(1, 2, 200, 200, 64, "f16", 9, "cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention(q, k, v, True, 1 / math.sqrt(64))
    compare(o, o_ref, lse, lse_ref, q.dtype, "after the timeout self-test")
    with pytest.raises(fa.FaError):
        fa.selftest_timeout(0)
