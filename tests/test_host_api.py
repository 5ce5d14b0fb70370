"""fa_fwd_host: the forward from and to host memory with chunked, overlapped copies.

Each chunk runs the fa_fwd_gqa kernels on its heads, so the outputs must equal
the device-resident forward bit for bit, whatever the chunking; one small case
is also checked against the fp64 oracle.
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
    oracle.set_threads(16)
    return fa


def _inputs(B, H, H_kv, Nq, Nk, d, dtype, seed):
    q, _, _ = attn_inputs.make_qkv(B, H, Nq, 1, d, dtype, seed, "cuda")
    _, k, v = attn_inputs.make_qkv(B, H_kv, 1, Nk, d, dtype, seed + 7, "cuda")
    return q, k, v


CASES = [
    # B, H, H_kv, Nq, Nk, d, dtype, causal, chunks
    (2, 4, 4, 300, 300, 128, "bf16", True, 0),
    (2, 4, 4, 300, 300, 128, "bf16", True, 3),       # chunks of unequal size
    (1, 8, 2, 257, 513, 64, "f16", False, 2),        # grouped heads (rows of a group merged)
    (3, 2, 1, 1, 700, 128, "bf16", False, 100),      # more chunks asked than K/V heads
    (1, 6, 3, 520, 200, 128, "bf16", True, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}Nq{}Nk{}d{}{}{}ch{}".format(*c[:7], "c" if c[7] else "", c[8]))
def test_host_forward_equals_device_forward(fa, case):
    B, H, H_kv, Nq, Nk, d, dtype, causal, chunks = case
    q, k, v = _inputs(B, H, H_kv, Nq, Nk, d, dtype, 40 + Nq)
    o_dev, lse_dev = fa.fwd(q, k, v, causal=causal)
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(qh, kh, vh, causal=causal, num_chunks=chunks)
    assert fa.get_device_status() == fa.FA_OK
    assert not o.is_cuda and not lse.is_cuda
    assert torch.equal(o, o_dev.cpu())
    assert torch.equal(lse, lse_dev.cpu())


def test_host_forward_against_the_oracle(fa):
    q, k, v = _inputs(1, 2, 2, 200, 333, 128, "bf16", 5)
    o, lse = fa.fwd_host(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(), causal=True)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 1 / math.sqrt(128))
    compare(o, o_ref, lse, lse_ref, q.dtype, "fa_fwd_host")


def test_host_forward_pageable_memory_and_side_stream(fa):
    """Pageable host buffers give the same result; the call is ordered on the stream
    it is given, after the work queued there before it."""
    q, k, v = _inputs(2, 4, 4, 256, 256, 64, "bf16", 9)
    o_dev, lse_dev = fa.fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    o, lse = fa.fwd_host(q.cpu(), k.cpu(), v.cpu(), causal=True, stream=s, num_chunks=4)
    assert torch.equal(o, o_dev.cpu()) and torch.equal(lse, lse_dev.cpu())
    # a kernel queued on the side stream first: the copies must wait for it
    qh = torch.zeros(q.shape, dtype=q.dtype, pin_memory=True)
    ws = torch.empty(fa.fwd_host_workspace_bytes(2, 4, 4, 256, 256, 64), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        ws.fill_(0)                                           # work before the call on s
    out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    fa.fwd_host(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(), causal=True, out=out,
                workspace=ws, stream=s, synchronize=False)
    s.synchronize()
    assert torch.equal(out, o_dev.cpu())
    del qh


def test_host_forward_rejects_bad_arguments(fa):
    q, k, v = _inputs(1, 2, 2, 64, 64, 64, "bf16", 3)
    qh, kh, vh = q.cpu(), k.cpu(), v.cpu()
    short = torch.empty(fa.fwd_host_workspace_bytes(1, 2, 2, 64, 64, 64) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd_host(qh, kh, vh, workspace=short)
    assert e.value.code == fa.FA_ERR_WORKSPACE
    assert fa.get_device_status() == fa.FA_OK
