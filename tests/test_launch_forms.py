"""Which form of the fused forward a call launches: on a d = 64 grid of three to
eight waves whose CTAs visit few K/V tiles, the form with two CTAs per SM (one
score buffer each); elsewhere the one-CTA form with three score buffers.  The
kernel names come from the CUDA activity the profiler records; the tests skip if
the runtime records none."""
import re

import pytest
import torch

import attn_inputs

pytestmark = pytest.mark.gpu

PAIRED = re.compile(r"fa_fwd_kernel<64, (?:false|0), (?:false|0), (?:true|1)>")
ONE_CTA = re.compile(r"fa_fwd_kernel<(?:64|128), (?:false|true|0|1), (?:false|0), (?:false|0)>")


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    # The first profiling session of a process may record no kernel activity while
    # the activity API starts up: open one before the tests' own.
    x = torch.ones(1024, device="cuda")
    with torch.profiler.profile(activities=[torch.profiler.ProfilerActivity.CUDA]):
        (x * 2).sum().item()
    torch.cuda.synchronize()
    return fa


def _launched(fa, B, H, N, d, dtype, causal):
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, dtype, 61, "cuda")
    fa.fwd(q, k, v, causal=causal)  # device set-up outside the recorded region
    torch.cuda.synchronize()
    with torch.profiler.profile(activities=[torch.profiler.ProfilerActivity.CUDA]) as prof:
        fa.fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if "fa_fwd_kernel" in e.name]
    if not names:
        pytest.skip("the profiler recorded no CUDA kernel activity")
    assert fa.get_device_status() == fa.FA_OK
    return names


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("causal", [False, True])
def test_few_wave_d64_grid_runs_two_ctas_per_sm(fa, causal):
    # B4 H16 N1024: 512 CTAs of at most 8 K/V tiles, 3.4 waves on 152 SMs
    if not 3 * _sms() <= 512 <= 8 * _sms():
        pytest.skip("grid is not three to eight waves on this GPU")
    names = _launched(fa, 4, 16, 1024, 64, "f16", causal)
    assert all(PAIRED.search(n) for n in names), names


@pytest.mark.parametrize("shape", [
    (1, 1, 128, 64, "f16", True),        # one CTA
    (1, 8, 4096, 64, "bf16", True),      # 256 CTAs: under three waves
    (2, 16, 4096, 64, "bf16", False),    # 32 K/V tiles per CTA
    (4, 16, 1024, 128, "bf16", True),    # d = 128 never pairs
])
def test_other_grids_run_one_cta_per_sm(fa, shape):
    B, H, N, d, dtype, causal = shape
    names = _launched(fa, B, H, N, d, dtype, causal)
    assert all(ONE_CTA.search(n) and not PAIRED.search(n) for n in names), names
