"""Every output and workspace is written inside its own bounds.

Each buffer a call writes (outputs and workspaces) is a view into a larger
allocation whose bytes before and after the view hold a sentinel pattern; after
the call the sentinels must be intact.  Ragged sizes (rows and keys that are not
multiples of the 128-row tiles, packed sequences of odd lengths) put the edge
tiles of every kernel next to the guards.
"""
import itertools
import math

import pytest
import torch

import attn_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (keeps every view 16-byte aligned)
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    return fa


class Guarded:
    """A tensor of `shape` and `dtype` (or `nbytes` raw bytes) between two sentinel bands."""

    def __init__(self, shape=None, dtype=torch.uint8, nbytes=None):
        if nbytes is None:
            nbytes = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
        self.nbytes = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        body = self.raw[GUARD:GUARD + nbytes]
        self.t = body if shape is None else body.view(dtype).view(shape)

    def intact(self):
        return bool((self.raw[:GUARD] == SENTINEL).all()) and bool((self.raw[GUARD + self.nbytes:] == SENTINEL).all())


def _check(fa, *bufs):
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    for name, g in bufs:
        assert g.intact(), f"{name}: a sentinel byte next to the buffer changed"


@pytest.mark.parametrize("d,dtype,causal", [(128, "bf16", True), (64, "f16", False)])
def test_forward_and_backward(fa, d, dtype, causal):
    B, H, Nq, Nk = 2, 3, 300, 257
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, 61, "cuda")
    dout = attn_inputs.make_dout(B, H, Nq, d, dtype, 61, "cuda")
    o, lse = Guarded(q.shape, q.dtype), Guarded((B, H, Nq), torch.float32)
    fa.fwd(q, k, v, causal=causal, out=o.t, lse=lse.t)
    _check(fa, ("o", o), ("lse", lse))
    dq, dk, dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    ws = Guarded(nbytes=fa.bwd_workspace_bytes(B, H, Nq, d))
    fa.bwd(q, k, v, o.t, dout, lse.t, causal=causal, dq=dq.t, dk=dk.t, dv=dv.t, workspace=ws.t)
    _check(fa, ("dq", dq), ("dk", dk), ("dv", dv), ("workspace", ws))


def test_split_kv(fa):
    B, H, Nq, Nk, d = 3, 2, 1, 1001, 128
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, "bf16", 62, "cuda")
    o, lse = Guarded(q.shape, q.dtype), Guarded((B, H, Nq), torch.float32)
    ws = Guarded(nbytes=fa.splitkv_workspace_bytes(B, H, Nq, Nk, d, 7))
    fa.fwd_splitkv(q, k, v, num_splits=7, workspace=ws.t, out=o.t, lse=lse.t)
    _check(fa, ("o", o), ("lse", lse), ("workspace", ws))


def test_packed_variable_length(fa):
    lens = [1, 130, 0, 257, 77]
    H, H_kv, d = 4, 2, 128
    total = sum(lens)
    q = attn_inputs.make_qkv(1, total, H, 1, d, "bf16", 63, "cuda")[0][0]
    _, k, v = attn_inputs.make_qkv(1, total, 1, H_kv, d, "bf16", 64, "cuda")
    k, v = k[0], v[0]
    dout = attn_inputs.make_dout(1, total, H, d, "bf16", 63, "cuda")[0]
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device="cuda")
    o, lse = Guarded(q.shape, q.dtype), Guarded((H, total), torch.float32)
    fa.fwd_varlen(q, k, v, cu, cu, max(lens), causal=True, out=o.t, lse=lse.t)
    _check(fa, ("o", o), ("lse", lse))
    dq, dk, dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    ws = Guarded(nbytes=fa.bwd_varlen_workspace_bytes(len(lens), total, total, H, d))
    fa.bwd_varlen(q, k, v, o.t, dout, lse.t, cu, cu, max(lens), causal=True, dq=dq.t, dk=dk.t, dv=dv.t,
                  workspace=ws.t)
    _check(fa, ("dq", dq), ("dk", dk), ("dv", dv), ("workspace", ws))


def test_fp8(fa):
    B, H, N, d = 1, 2, 300, 128
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 65, "cuda")
    nb = (N + 127) // 128
    q8, qs = Guarded(q.shape, torch.uint8), Guarded((B * H, nb), torch.float32)
    k8, ks = Guarded(k.shape, torch.uint8), Guarded((B * H, nb), torch.float32)
    v8t, vs = Guarded((B, H, d, nb * 128), torch.uint8), Guarded((B * H, nb), torch.float32)
    fa.fp8_quantize(q, out=q8.t, scales=qs.t)
    fa.fp8_quantize(k, out=k8.t, scales=ks.t)
    fa.fp8_quantize(v, transpose=True, out=v8t.t, scales=vs.t)
    _check(fa, ("q8", q8), ("q scales", qs), ("k8", k8), ("k scales", ks), ("v8t", v8t), ("v scales", vs))
    o, lse = Guarded(q.shape, q.dtype), Guarded((B, H, N), torch.float32)
    fa.fwd_fp8(q8.t, qs.t, k8.t, ks.t, v8t.t, vs.t, causal=True, out=o.t, lse=lse.t)
    _check(fa, ("o", o), ("lse", lse))


def test_host_buffers_workspace(fa):
    B, H, N, d = 2, 2, 200, 64
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, "bf16", 66, "cuda")
    ws = Guarded(nbytes=fa.fwd_host_workspace_bytes(B, H, H, N, N, d))
    fa.fwd_host(q.cpu(), k.cpu(), v.cpu(), causal=True, workspace=ws.t, num_chunks=3)
    _check(fa, ("workspace", ws))
