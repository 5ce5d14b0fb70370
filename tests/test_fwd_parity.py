"""fa_fwd (tcgen05 fused forward) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import attn_inputs
import oracle
from parity import LSE_ABS_TOL, compare, round_to, ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_03_gb300 as fa
    from exact_attention_forward_03_gb300 import build

    build.build()
    fa.load_library()
    oracle.set_threads(16)
    return fa


def run_case(fa, B, H, Nq, Nk, d, dtype, causal, seed, scale=None):
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, seed, "cuda")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    return compare(o, o_ref, lse, lse_ref, q.dtype, f"B{B} H{H} Nq{Nq} Nk{Nk} d{d} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_d64_f16(fa, causal):
    w = attn_inputs.WORKLOADS["tiny_d64_f16_causal" if causal else "tiny_d64_f16"]
    run_case(fa, w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, causal, w.seed)


@pytest.mark.parametrize("causal", [False, True])
def test_b4h16_n1024_d64_f16_all_rows(fa, causal):
    w = attn_inputs.WORKLOADS["b4h16_n1024_d64_f16"]
    run_case(fa, w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, causal, w.seed)


RAGGED = [
    # B, H, Nq, Nk, d, dtype, causal
    (1, 2, 1, 1, 64, "f16", False),
    (1, 2, 17, 17, 128, "bf16", True),
    (2, 1, 127, 129, 64, "bf16", False),
    (1, 3, 129, 127, 128, "f16", False),
    (1, 2, 255, 255, 128, "bf16", True),
    (1, 1, 300, 300, 64, "f16", True),
    (2, 2, 384, 384, 128, "bf16", True),
    (1, 2, 200, 520, 128, "bf16", True),   # Nq < Nk: bottom-right diagonal
    (1, 2, 520, 200, 64, "f16", True),     # Nq > Nk: first 320 rows see no key
    (1, 1, 1, 700, 128, "bf16", False),    # one query row, many tiles
    (1, 1, 640, 1, 64, "bf16", False),     # one key
    (2, 3, 700, 333, 128, "f16", False),
]


@pytest.mark.parametrize("case", RAGGED, ids=lambda c: "B{}H{}_q{}_k{}_d{}_{}_{}".format(*c[:6], "c" if c[6] else "nc"))
def test_ragged_shapes(fa, case):
    B, H, Nq, Nk, d, dtype, causal = case
    run_case(fa, B, H, Nq, Nk, d, dtype, causal, seed=7 * Nq + Nk)


@pytest.mark.parametrize("B,H", [(1, 17), (3, 11)])
def test_launch_order_with_a_partial_head_group(fa, B, H):
    """Grids of a few waves interleave the row blocks of up to 16 heads; with 17 and 33
    heads the last group holds one head.  Every row is checked."""
    for causal in (False, True):
        run_case(fa, B, H, 300, 300, 64, "f16", causal, seed=53 + B * H)


# Grids of three to eight waves whose CTAs visit few K/V tiles run the d = 64 forward
# with two CTAs per SM (one score buffer each, so every tile's S waits for the last
# PV); on a 152-SM GPU each of these shapes takes that form.
PAIRED = [
    # B, H, Nq, Nk, d, dtype, causal
    (4, 16, 1000, 1000, 64, "f16", True),    # ragged last row and key blocks
    (4, 16, 1000, 1000, 64, "bf16", False),
    (2, 16, 2048, 2048, 64, "bf16", True),   # 16 K/V tiles for the last row block
    (4, 16, 900, 1024, 64, "f16", True),     # Nq < Nk: bottom-right diagonal
    (4, 16, 1024, 512, 64, "f16", True),     # Nq > Nk: the first four row blocks see no key
]


@pytest.mark.parametrize("case", PAIRED, ids=lambda c: "B{}H{}_q{}_k{}_d{}_{}_{}".format(*c[:6], "c" if c[6] else "nc"))
def test_two_ctas_per_sm_form(fa, case):
    B, H, Nq, Nk, d, dtype, causal = case
    run_case(fa, B, H, Nq, Nk, d, dtype, causal, seed=11 * Nq + Nk)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_two_ctas_per_sm_form_moves_its_max(fa, dtype):
    """The rescale paths in the two-CTAs-per-SM form (64 heads of N = 1024 at d = 64):
    on even rows of the first 48 heads the scores jump by ~20 (natural-log units) on
    K/V tile 5, and on the last 16 heads the keys' scores rise with the key index, so
    the running max moves on every tile (the magnitudes of the d = 128 edge-case tests
    above).  The output must equal, bit for bit, that of the one-CTA-per-SM form (the
    same heads four at a time, a grid too small for the paired form), also at scale
    1/8 (a jump of ~28).  Against the oracle: f16 within the 2e-3 bound; bf16 within
    the bound its 16-bit weights allow when a few keys dominate a row, 2^-9 max|v|
    (each weight rounded once, relative error 2^-9, and l summed from the unrounded
    weights) plus half an output ulp -- on these rows that can exceed 2e-3 by a little
    (2.2e-3 seen, in both forms alike)."""
    B, H, N, d = 1, 64, 1024, 64
    q, k, v = attn_inputs.make_qkv(B, H, N, N, d, dtype, 43, "cuda")
    q[:, :48, 0::2, 0] += 15.0
    k[:, :48, 640:768, 0] += 15.0
    ramp = torch.linspace(-2.0, 2.0, N, device="cuda")[:, None].expand(N, d)
    q[:, 48:] = math.sqrt(0.5)
    k[:, 48:] = ramp.to(q.dtype)
    for scale in (1 / math.sqrt(128), 0.125):
        for causal in (False, True):
            o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
            torch.cuda.synchronize()
            assert fa.get_device_status() == fa.FA_OK
            for h in range(0, H, 4):
                hs = slice(h, h + 4)
                o1, lse1 = fa.fwd(q[:, hs].contiguous(), k[:, hs].contiguous(), v[:, hs].contiguous(),
                                  causal=causal, scale=scale)
                assert torch.equal(o1, o[:, hs]) and torch.equal(lse1, lse[:, hs]), (scale, causal, h)
            if scale < 0.1:
                o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
                what = f"paired form, moving max {dtype} causal={causal}"
                if dtype == "f16":
                    compare(o, o_ref, lse, lse_ref, q.dtype, what)
                else:
                    og = o.double().cpu().numpy()
                    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(og.shape)
                    half_ulp = 0.5 * ulp(round_to(o_ref, q.dtype), q.dtype)
                    bound = 2.0 ** -9 * v.abs().max().item() + half_ulp + 1e-4
                    assert (np.abs(og - o_ref) <= bound).all(), what
                    lerr = np.abs(lse.double().cpu().numpy() - np.asarray(lse_ref).reshape(lse.shape))
                    assert lerr.max() <= LSE_ABS_TOL, what


def _sampled(fa, wname, count=1024):
    w = attn_inputs.WORKLOADS[wname]
    q, k, v = attn_inputs.make_workload(w, "cuda")
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    pairs = attn_inputs.sample_rows(w.Nq, w.B * w.H, count, seed=w.seed)
    o_ref, lse_ref = oracle.sampled_rows(q, k, v, pairs, w.causal, w.scale)
    of = o.view(-1, w.Nq, w.d)
    lf = lse.view(-1, w.Nq)
    idx_bh = torch.tensor([p[0] for p in pairs], device=o.device)
    idx_r = torch.tensor([p[1] for p in pairs], device=o.device)
    stats = compare(of[idx_bh, idx_r], o_ref, lf[idx_bh, idx_r], lse_ref, q.dtype, wname)
    assert torch.isfinite(o).all()
    return stats


def test_b2h32_n8192_d128_bf16_causal_sampled(fa):
    _sampled(fa, "b2h32_n8192_d128_bf16_causal")


def test_b2h32_n8192_d128_bf16_noncausal_sampled(fa):
    _sampled(fa, "b2h32_n8192_d128_bf16")


def test_b1h32_n32768_d128_bf16_causal_sampled(fa):
    _sampled(fa, "b1h32_n32768_d128_bf16_causal")


def test_one_long_sequence_sampled(fa):
    """N = 131072 (1024 K/V tiles per causal row block at the end), one head, 256 sampled
    rows each over its full key range."""
    N, d = 131072, 128
    q, k, v = attn_inputs.make_qkv(1, 1, N, N, d, "bf16", 39, "cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == fa.FA_OK
    pairs = attn_inputs.sample_rows(N, 1, 256, seed=39)
    o_ref, lse_ref = oracle.sampled_rows(q, k, v, pairs, True, 1 / math.sqrt(d))
    rows = torch.tensor([p[1] for p in pairs], device=o.device)
    compare(o[0, 0, rows], o_ref, lse[0, 0, rows], lse_ref, q.dtype, "N131072 causal sampled")


def test_constant_v_gives_constant_o(fa):
    q, k, _ = attn_inputs.make_qkv(1, 2, 300, 300, 128, "bf16", 31, "cuda")
    v = torch.full_like(k, 0.8125)
    for causal in (False, True):
        o, _ = fa.fwd(q, k, v, causal=causal)
        compare(o, np.full(o.shape, 0.8125), None, None, q.dtype, f"constant V causal={causal}")


def test_causal_row0_is_v0(fa):
    for d, dt in ((64, "f16"), (128, "bf16")):
        q, k, v = attn_inputs.make_qkv(2, 2, 256, 256, d, dt, 32, "cuda")
        o, lse = fa.fwd(q, k, v, causal=True)
        assert torch.equal(o[:, :, 0], v[:, :, 0])
        s00 = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) / math.sqrt(d)
        assert torch.allclose(lse[:, :, 0].double(), s00, atol=1e-4, rtol=0)


def test_most_heads_the_grid_allows(fa):
    """B * H = 65535 (the largest grid y the launch allows) of three-row problems, every
    head checked; one head more is refused before any launch."""
    q, k, v = attn_inputs.make_qkv(1, 65535, 3, 5, 64, "f16", 37, "cuda")
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 1 / math.sqrt(64))
        compare(o, o_ref, lse, lse_ref, q.dtype, f"65535 heads causal={causal}")
    q2, k2, v2 = attn_inputs.make_qkv(1, 65536, 1, 1, 64, "f16", 38, "cuda")
    with pytest.raises(fa.FaError):
        fa.fwd(q2, k2, v2)


def test_causal_never_reads_future_tiles(fa):
    """NaN in V rows 128..255 must not reach rows 0..127 (their K/V tile range ends at 128)."""
    q, k, v = attn_inputs.make_qkv(1, 2, 256, 256, 128, "bf16", 33, "cuda")
    v2 = v.clone()
    v2[:, :, 128:] = float("nan")
    k2 = k.clone()
    k2[:, :, 128:] = float("nan")
    o, lse = fa.fwd(q, k2, v2, causal=True)
    o_ref, lse_ref = oracle.attention(q[:, :, :128], k[:, :, :128], v[:, :, :128], True, 1 / math.sqrt(128))
    compare(o[:, :, :128], o_ref, lse[:, :, :128], lse_ref, q.dtype, "future tiles")


def test_growing_row_max_needs_l_rescale(fa):
    """Keys whose scores rise with j: the running max moves in every tile (l * alpha matters)."""
    Nk, d = 1024, 128
    q = torch.ones(1, 1, 256, d, device="cuda", dtype=torch.bfloat16) * 0.25
    ramp = torch.linspace(-2.0, 2.0, Nk, device="cuda")[:, None].expand(Nk, d)
    k = ramp[None, None].to(torch.bfloat16).contiguous()
    v = torch.randn(1, 1, Nk, d, device="cuda", generator=torch.Generator("cuda").manual_seed(5)).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal, scale=0.125)
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 0.125)
        compare(o, o_ref, lse, lse_ref, q.dtype, f"growing max causal={causal}")


def test_large_scores_stay_finite(fa):
    """Scores of size ~1e3 (scale 1, large q and k) must not overflow."""
    q, k, v = attn_inputs.make_qkv(1, 2, 200, 300, 64, "bf16", 34, "cuda")
    q = (q * 8).contiguous()
    k = (k * 8).contiguous()
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal, scale=1.0)
        assert torch.isfinite(o).all()
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 1.0)
        compare(o, o_ref, lse, lse_ref, q.dtype, f"large scores causal={causal}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_scores_jump_on_a_later_unmasked_tile(fa, dtype):
    """Even rows meet keys on tile 5 whose scores sit ~20 (natural-log units) above
    everything before: the exponentials taken against the running max overshoot
    there, and those rows (not their odd neighbours in the same warp) must move
    their max, rescale O and redo the tile."""
    B, H, Nq, Nk, d = 1, 2, 256, 1024, 128
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dtype, 41, "cuda")
    q[:, :, 0::2, 0] += 15.0
    k[:, :, 640:768, 0] += 15.0
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 1 / math.sqrt(d))
        compare(o, o_ref, lse, lse_ref, q.dtype, f"score jump {dtype} causal={causal}")


def test_joint_kv_permutation_leaves_output_unchanged(fa):
    """Without a mask, attention is invariant to permuting the K and V rows together:
    the kernel on the permuted keys (which reorders every tile's contents and moves
    keys across tiles and the ragged tail) matches the oracle of the unpermuted ones."""
    for d, dtype in ((128, "bf16"), (64, "f16")):
        q, k, v = attn_inputs.make_qkv(2, 3, 300, 700, d, dtype, 71 + d, "cuda")
        perm = torch.from_numpy(np.random.default_rng(72).permutation(700)).to("cuda")
        o, lse = fa.fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), causal=False)
        torch.cuda.synchronize()
        assert fa.get_device_status() == fa.FA_OK
        o_ref, lse_ref = oracle.attention(q, k, v, False, 1 / math.sqrt(d))
        compare(o, o_ref, lse, lse_ref, q.dtype, f"K/V rows permuted, d={d}")


def test_affine_v_moves_output_affinely(fa):
    """V -> a V + b gives O -> a O + b (the weights sum to 1).  On the GPU: the output
    for the shifted and scaled values (|O| near b = 1.25, where a bf16 ulp is 2^-7)
    matches the oracle, and differs from a O + b of the unshifted run by no more than
    the two runs' tolerances plus the rounding of a v + b to bf16 (half an ulp of
    a max|v| + b); the LSE does not change."""
    a, b = 0.5, 1.25
    q, k, v = attn_inputs.make_qkv(1, 4, 500, 500, 128, "bf16", 73, "cuda")
    v2 = (a * v.float() + b).to(v.dtype)
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal)
        o2, lse2 = fa.fwd(q, k, v2, causal=causal)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.attention(q, k, v2, causal, 1 / math.sqrt(128))
        compare(o2, o_ref, lse2, lse_ref, q.dtype, f"affine V causal={causal}")
        assert torch.equal(lse, lse2)  # the weights do not depend on V
        o1, o2d = o.double().cpu().numpy(), o2.double().cpu().numpy()
        vmax = float(v.abs().max())
        # each run within max(2e-3, ulp) + ulp/2 of fp64, with ulp <= 2^-6 for |O| < 4
        u = 2.0 ** -6
        tol = 1.5 * u * (1 + a) + 2.0 ** -9 * (a * vmax + b)
        assert np.abs(o2d - (a * o1 + b)).max() <= tol


def test_lse_optional(fa):
    q, k, v = attn_inputs.make_qkv(1, 1, 130, 130, 64, "f16", 35, "cuda")
    o1, _ = fa.fwd(q, k, v, causal=True, want_lse=False)
    o2, _ = fa.fwd(q, k, v, causal=True)
    assert torch.equal(o1, o2)


def test_deterministic(fa):
    q, k, v = attn_inputs.make_qkv(2, 4, 1000, 1000, 128, "bf16", 36, "cuda")
    a = fa.fwd(q, k, v, causal=True)
    b = fa.fwd(q, k, v, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_nonzero_stream(fa):
    q, k, v = attn_inputs.make_qkv(1, 4, 512, 512, 128, "bf16", 37, "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.fwd(q, k, v, causal=False)
    s.synchronize()
    o2, lse2 = fa.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
