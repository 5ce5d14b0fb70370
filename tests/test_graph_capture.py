"""The device entry points record into CUDA graphs.

A call is host-side argument checks and tensor-map encodes followed by kernel
launches on the caller's stream: no synchronisation, no allocation inside the
library (workspaces are the caller's), so a stream capture records it whole.
One graph here holds a causal forward, a packed-batch forward (its work-list
launch included), a split-KV decode (partials and combine) and a backward.
Replays must reproduce the eager results bit for bit (dQ to within its
summation order), and must read the inputs as they are at replay time (inputs
overwritten in place between replays)."""
import itertools

import pytest
import torch

import attn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    return fa


NAMES = "o lse vo vlse do dlse dq dk dv".split()


def same(name, a, b):
    """Bit for bit, except dQ: it is summed across key blocks with fp32 atomic adds
    in no fixed order, so two runs may round its 16-bit result one ulp apart."""
    if name != "dq":
        return torch.equal(a, b)
    a, b = a.float(), b.float()
    return bool(((a - b).abs() <= b.abs() * 2.0**-7 + 1e-6).all())


def _problems(seed):
    dense = attn_inputs.make_qkv(2, 4, 1000, 1000, 128, "bf16", seed, "cuda")
    dout = attn_inputs.make_dout(2, 4, 1000, 128, "bf16", seed, "cuda")
    lens = [300, 1000, 57]
    total = sum(lens)
    # packed [tokens, heads, d] tensors: 4 query heads over 2 K/V heads
    vq = attn_inputs.make_qkv(1, total, 4, 1, 64, "f16", seed + 1, "cuda")[0][0]
    _, vk, vv = attn_inputs.make_qkv(1, total, 1, 2, 64, "f16", seed + 2, "cuda")
    varlen = (vq, vk[0], vv[0])
    decode = attn_inputs.make_qkv(4, 8, 1, 4096, 128, "bf16", seed + 3, "cuda")
    return dense, dout, varlen, lens, decode


def test_graph_replay_matches_eager(fa):
    dense, dout, varlen, lens, decode = _problems(seed=610)
    q, k, v = dense
    vq, vk, vv = varlen
    dq_, dk_, dv_ = decode
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device="cuda")
    total = sum(lens)

    # Static outputs and workspaces, allocated before the capture.
    o = torch.empty_like(q)
    lse = torch.empty((2, 4, 1000), dtype=torch.float32, device="cuda")
    vo = torch.empty_like(vq)
    vlse = torch.empty((4, total), dtype=torch.float32, device="cuda")
    vws = torch.empty(fa.fwd_varlen_workspace_bytes(len(lens), total), dtype=torch.uint8, device="cuda")
    do_ = torch.empty_like(dq_)
    dlse = torch.empty((4, 8, 1), dtype=torch.float32, device="cuda")
    dws = fa.splitkv_workspace(dq_, dk_, 8)
    gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(fa.bwd_workspace_bytes(2, 4, 1000, 128), dtype=torch.uint8, device="cuda")

    def step():
        fa.fwd(q, k, v, causal=True, out=o, lse=lse)
        fa.fwd_varlen(vq, vk, vv, cu, cu, max(lens), causal=True, out=vo, lse=vlse, plan=True, workspace=vws)
        fa.fwd_splitkv(dq_, dk_, dv_, num_splits=8, workspace=dws, out=do_, lse=dlse)
        fa.bwd(q, k, v, o, dout, lse, causal=True, dq=gq, dk=gk, dv=gv, workspace=bws)

    def snapshot():
        return [t.clone() for t in (o, lse, vo, vlse, do_, dlse, gq, gk, gv)]

    # Eager reference (also the warm-up: first calls set up per-device state).
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    eager = snapshot()

    graph = torch.cuda.CUDAGraph()
    for t in (o, lse, vo, vlse, do_, dlse, gq, gk, gv):
        t.zero_()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    for name, a, b in zip(NAMES, snapshot(), eager):
        assert same(name, a, b), f"{name}: graph replay differs from the eager call"

    # New inputs written in place: the replay reads them, and matches eager again.
    (nq, nk, nv), ndout, (nvq, nvk, nvv), _, (ndq, ndk, ndv) = _problems(seed=611)
    for dst, src in ((q, nq), (k, nk), (v, nv), (dout, ndout), (vq, nvq), (vk, nvk), (vv, nvv),
                     (dq_, ndq), (dk_, ndk), (dv_, ndv)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    replayed = snapshot()
    step()
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    for name, a, b, old in zip(NAMES, replayed, snapshot(), eager):
        assert same(name, a, b), f"{name}: replay on new inputs differs from the eager call"
        assert not torch.equal(a, old), f"{name}: replay did not see the new inputs"
