"""Concurrent use of the library: calls on different streams, and from different
host threads, each with its own outputs and workspaces, give exactly the results
of the same calls made one at a time.  The library keeps no per-call state of its
own (the per-device status word aside), so nothing is shared between the calls."""
import itertools
import threading

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


def _problem(seed):
    q, k, v = attn_inputs.make_qkv(2, 4, 700, 700, 128, "bf16", seed, "cuda")
    lens = [300, 700, 57]
    total = sum(lens)
    vq = attn_inputs.make_qkv(1, total, 4, 1, 64, "f16", seed + 1, "cuda")[0][0]
    _, vk, vv = attn_inputs.make_qkv(1, total, 1, 2, 64, "f16", seed + 2, "cuda")
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device="cuda")
    dq, dk, dv = attn_inputs.make_qkv(4, 8, 1, 4096, 128, "bf16", seed + 3, "cuda")
    return (q, k, v), (vq, vk[0], vv[0], cu, max(lens)), (dq, dk, dv)


def _run(fa, prob, stream):
    (q, k, v), (vq, vk, vv, cu, mq), (dq, dk, dv) = prob
    with torch.cuda.stream(stream):
        o, lse = fa.fwd(q, k, v, causal=True)
        vo, vl = fa.fwd_varlen(vq, vk, vv, cu, cu, mq, causal=True)
        do, dl = fa.fwd_splitkv(dq, dk, dv, num_splits=8)
    return [o, lse, vo, vl, do, dl]


def test_two_streams_interleaved(fa):
    probs = [_problem(700), _problem(800)]
    ref = []
    for p in probs:  # one at a time on the default stream
        ref.append([t.clone() for t in _run(fa, p, torch.cuda.current_stream())])
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [_run(fa, p, s) for p, s in zip(probs, streams)]  # enqueued back to back, run concurrently
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    for got, want in zip(outs, ref):
        for a, b in zip(got, want):
            assert torch.equal(a, b)


def test_two_host_threads(fa):
    probs = [_problem(900), _problem(1000)]
    ref = []
    for p in probs:
        ref.append([t.clone() for t in _run(fa, p, torch.cuda.current_stream())])
        torch.cuda.synchronize()
    results, errors = [None, None], []

    def worker(idx):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.default_stream())
            out = None
            for _ in range(5):  # repeated calls, racing the other thread's
                out = _run(fa, probs[idx], s)
            s.synchronize()
            results[idx] = out
        except Exception as e:  # reported below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert fa.get_device_status() == fa.FA_OK
    for got, want in zip(results, ref):
        assert got is not None
        for a, b in zip(got, want):
            assert torch.equal(a, b)
