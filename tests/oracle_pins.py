"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes a loaded oracle library and raises
``AssertionError`` when the oracle disagrees with a closed form, an invariant
of the method, brute force on a tiny input, or an independent library routine
(torch's CPU scaled_dot_product_attention / logsumexp / autograd in fp64).  The same
functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show that the pins catch plausible mistakes.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

TOL = 1e-12


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def pin_two_key_closed_form(lib):
    """d = 1, two keys: O = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1, LSE = log(e^s0 + e^s1).

    Softmax of two scores is the logistic function of their difference
    ("Lecture 25", §2.1 safe softmax; "6.2 FlashAttention V2 explained" §6: L = m + log l).
    """
    for (qv, k0, k1, v0, v1, sc) in [(1.0, 0.5, -1.5, 2.0, -3.0, 0.7), (-2.0, 1.0, 3.0, 0.25, 4.0, 1.0),
                                     (0.3, 0.0, 0.0, 1.0, 5.0, 2.0)]:
        q = np.array([[[qv]]])
        k = np.array([[[k0], [k1]]])
        v = np.array([[[v0], [v1]]])
        o, lse = oracle.attention(q, k, v, False, sc, lib=lib)
        s0, s1 = sc * qv * k0, sc * qv * k1
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        assert abs(o[0, 0, 0] - (w0 * v0 + w1 * v1)) < TOL
        mx = max(s0, s1)
        assert abs(lse[0, 0] - (mx + math.log1p(math.exp(-abs(s0 - s1))))) < TOL


def pin_zero_query_uniform(lib):
    """Q = 0 makes every score 0: softmax is uniform.

    Non-causal: O_i = mean_j V_j, LSE_i = ln Nk.  Causal (Nq = Nk): O_i is the
    prefix mean of V_0..V_i and LSE_i = ln(i + 1) ("6.2 FlashAttention V2 explained" §5.1: row i sees j <= i).
    """
    BH, N, d = 2, 9, 5
    q = np.zeros((BH, N, d))
    k = _rand((BH, N, d), 1)
    v = _rand((BH, N, d), 2)
    o, lse = oracle.attention(q, k, v, False, 0.5, lib=lib)
    assert np.allclose(o, v.mean(axis=1, keepdims=True).repeat(N, axis=1), atol=TOL, rtol=0)
    assert np.allclose(lse, math.log(N), atol=TOL, rtol=0)
    o, lse = oracle.attention(q, k, v, True, 0.5, lib=lib)
    prefix = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None]
    assert np.allclose(o, prefix, atol=TOL, rtol=0)
    assert np.allclose(lse, np.log(np.arange(1, N + 1))[None, :], atol=TOL, rtol=0)


def pin_constant_and_affine_v(lib):
    """Rows of P sum to 1, so V = c gives O = c and V -> aV + b gives O -> aO + b."""
    BH, Nq, Nk, d = 3, 7, 11, 4
    q = _rand((BH, Nq, d), 3)
    k = _rand((BH, Nk, d), 4)
    v = _rand((BH, Nk, d), 5)
    for causal in (False, True):
        c = np.full((BH, Nk, d), 0.375)
        o, _ = oracle.attention(q, k, c, causal, 0.4, lib=lib)
        assert np.allclose(o, 0.375, atol=TOL, rtol=0)
        o1, l1 = oracle.attention(q, k, v, causal, 0.4, lib=lib)
        o2, l2 = oracle.attention(q, k, -1.5 * v + 0.25, causal, 0.4, lib=lib)
        assert np.allclose(o2, -1.5 * o1 + 0.25, atol=1e-11, rtol=0)
        assert np.allclose(l1, l2, atol=TOL, rtol=0)


def pin_causal_row0(lib):
    """Causal with Nq = Nk: row 0 sees only key 0, so O_0 = V_0 and LSE_0 = s_00."""
    BH, N, d = 2, 6, 8
    q = _rand((BH, N, d), 6)
    k = _rand((BH, N, d), 7)
    v = _rand((BH, N, d), 8)
    o, lse = oracle.attention(q, k, v, True, 0.3, lib=lib)
    assert np.allclose(o[:, 0], v[:, 0], atol=TOL, rtol=0)
    s00 = 0.3 * np.einsum("bd,bd->b", q[:, 0], k[:, 0])
    assert np.allclose(lse[:, 0], s00, atol=TOL, rtol=0)


def pin_rows_of_p_sum_to_one(lib):
    """sum_j exp(s_ij - LSE_i) = 1 over the allowed keys ("Lecture 25" §2.1: p = e^{x-m}/l sums to 1)."""
    BH, Nq, Nk, d = 2, 5, 13, 6
    q = _rand((BH, Nq, d), 9)
    k = _rand((BH, Nk, d), 10)
    v = _rand((BH, Nk, d), 11)
    for causal in (False, True):
        _, lse = oracle.attention(q, k, v, causal, 0.6, lib=lib)
        s = 0.6 * np.einsum("bid,bjd->bij", q, k)
        if causal:
            allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
            s = np.where(allowed[None], s, -np.inf)
        tot = np.exp(s - lse[:, :, None]).sum(-1)
        assert np.allclose(tot, 1.0, atol=1e-12, rtol=0)


def pin_brute_force_tiny(lib):
    """Brute force on tiny inputs: every score enumerated with Python floats."""
    Nq, Nk, d = 3, 4, 2
    q = _rand((1, Nq, d), 12)
    k = _rand((1, Nk, d), 13)
    v = _rand((1, Nk, d), 14)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal, 1.25, lib=lib)
        for i in range(Nq):
            ws, num = [], [0.0] * d
            for j in range(Nk):
                if causal and j > i + (Nk - Nq):
                    continue
                sc = 1.25 * (q[0, i, 0] * k[0, j, 0] + q[0, i, 1] * k[0, j, 1])
                ws.append((sc, j))
            den = sum(math.exp(sc) for sc, _ in ws)
            for sc, j in ws:
                for t in range(d):
                    num[t] += math.exp(sc) * v[0, j, t]
            for t in range(d):
                assert abs(o[0, i, t] - num[t] / den) < 1e-12
            assert abs(lse[0, i] - math.log(den)) < 1e-12


def pin_sdpa_library(lib):
    """Independent library routine: torch CPU fp64 SDPA and logsumexp (square and bottom-right causal)."""
    cases = [(2, 3, 64, 64, 16, False), (1, 2, 96, 96, 32, True), (1, 1, 17, 40, 8, True),
             (2, 1, 33, 33, 64, False), (1, 2, 256, 256, 64, True)]
    for n, (B, H, Nq, Nk, d, causal) in enumerate(cases):
        g = torch.Generator().manual_seed(100 + n)
        q = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float64)
        k = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float64)
        v = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float64)
        scale = 1.0 / math.sqrt(d)
        o, lse = oracle.attention(q, k, v, causal, scale, lib=lib)
        mask = None
        if causal:
            mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        s = scale * (q @ k.transpose(-1, -2))
        if causal:
            s = s.masked_fill(~mask, float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1)
        assert np.allclose(o, ref.numpy(), atol=1e-12, rtol=0), f"case {n}"
        assert np.allclose(lse, ref_lse.numpy(), atol=1e-12, rtol=0), f"case {n}"


def pin_permutation_equivariance(lib):
    """Non-causal attention is invariant to a joint permutation of the K and V rows."""
    BH, Nq, Nk, d = 2, 6, 10, 5
    q = _rand((BH, Nq, d), 15)
    k = _rand((BH, Nk, d), 16)
    v = _rand((BH, Nk, d), 17)
    perm = np.random.default_rng(18).permutation(Nk)
    o1, l1 = oracle.attention(q, k, v, False, 0.5, lib=lib)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], False, 0.5, lib=lib)
    assert np.allclose(o1, o2, atol=TOL, rtol=0) and np.allclose(l1, l2, atol=TOL, rtol=0)


def pin_overflow_safety(lib):
    """Scores of magnitude ~1e4 stay finite ("Lecture 25" §2.2: the shifted exponent never overflows)."""
    q = np.full((1, 4, 2), 100.0)
    k = np.array([[[50.0, 50.0], [-50.0, 10.0], [49.0, 50.0], [0.0, 0.0]]])
    v = _rand((1, 4, 2), 19)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal, 1.0, lib=lib)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
    o, lse = oracle.attention(q, k, v, False, 1.0, lib=lib)
    # s = [10000, 4000, 9900, 0]: key 0 holds all but e^-100 of the weight
    assert np.allclose(o[0, 0], v[0, 0], atol=1e-30, rtol=1e-14)
    assert abs(lse[0, 0] - 10000.0) < 1e-9


def pin_fully_masked_rows(lib):
    """Causal with Nq > Nk: rows i < Nq - Nk see no key: O = 0, LSE = -inf."""
    q = _rand((1, 6, 3), 20)
    k = _rand((1, 2, 3), 21)
    v = _rand((1, 2, 3), 22)
    o, lse = oracle.attention(q, k, v, True, 1.0, lib=lib)
    assert (o[0, :4] == 0).all() and np.isneginf(lse[0, :4]).all()
    assert np.isfinite(lse[0, 4:]).all()
    assert np.allclose(o[0, 4], v[0, 0], atol=TOL)  # row 4 sees key 0 only


def pin_tiled_equals_full(lib):
    """The online-softmax loop of "6.2 FlashAttention V2 explained" §6 over KV tiles equals the full softmax (Bc in {1, 7, 64, 128, N})."""
    for causal, (Nq, Nk) in [(False, (70, 150)), (True, (150, 150)), (True, (40, 150)), (True, (20, 9))]:
        BH, d = 2, 8
        q = _rand((BH, Nq, d), 23, 1.5)
        k = _rand((BH, Nk, d), 24, 1.5)
        v = _rand((BH, Nk, d), 25)
        o, lse = oracle.attention(q, k, v, causal, 0.8, lib=lib)
        for Bc in (1, 7, 64, 128, Nk):
            ot, lt = oracle.attention_tiled(q, k, v, causal, 0.8, 32, Bc, lib=lib)
            assert np.allclose(ot, o, atol=1e-12, rtol=0), (causal, Bc)
            fin = np.isfinite(lse)
            assert (np.isfinite(lt) == fin).all()
            assert np.allclose(lt[fin], lse[fin], atol=1e-12, rtol=0), (causal, Bc)


def pin_tiled_growing_max(lib):
    """Row max that rises in a later tile (k_j grows with j): the l * alpha rescale matters.

    "Flash Attention (4)" §2.5 reports a first version that skipped the rescale of l and was
    caught only by a mismatch; here the tiled loop must still equal the full softmax.
    """
    Nk, d = 96, 4
    q = np.ones((1, 8, d))
    k = np.linspace(0.0, 3.0, Nk)[None, :, None].repeat(d, axis=2)[:, :, :] * np.ones((1, 1, d))
    v = _rand((1, Nk, d), 26)
    o, lse = oracle.attention(q, k, v, False, 1.0, lib=lib)
    ot, lt = oracle.attention_tiled(q, k, v, False, 1.0, 8, 16, lib=lib)
    assert np.allclose(ot, o, atol=1e-12, rtol=0) and np.allclose(lt, lse, atol=1e-12, rtol=0)


def pin_split_combine_equals_full(lib):
    """Split-KV partials merged by LSE weights equal the full result ("02 · FA2" §2, decode / split-KV).

    Includes more splits than keys, so some partials are empty (LSE_s = -inf).
    """
    for causal, (Nq, Nk) in [(False, (1, 200)), (False, (5, 130)), (True, (12, 40)), (True, (30, 7))]:
        BH, d = 3, 6
        q = _rand((BH, Nq, d), 27)
        k = _rand((BH, Nk, d), 28)
        v = _rand((BH, Nk, d), 29)
        o, lse = oracle.attention(q, k, v, causal, 0.7, lib=lib)
        for S in (1, 2, 8, 32, Nk + 3):
            split_len = max(1, -(-Nk // S))
            op, lp = oracle.split_partials(q, k, v, causal, 0.7, S, split_len, lib=lib)
            oc, lc = oracle.combine(op, lp, lib=lib)
            assert np.allclose(oc, o, atol=1e-12, rtol=0), (causal, S)
            fin = np.isfinite(lse)
            assert (np.isfinite(lc) == fin).all()
            assert np.allclose(lc[fin], lse[fin], atol=1e-12, rtol=0), (causal, S)


def pin_combine_two_halves_closed_form(lib):
    """Combining two single-key partials reproduces the two-key closed form."""
    s0, s1, v0, v1 = 0.4, -1.1, 3.0, -2.0
    op = np.array([[[v0]], [[v1]]])  # [S=2, rows=1, d=1]
    lp = np.array([[s0], [s1]])
    o, lse = oracle.combine(op, lp, lib=lib)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert abs(o[0, 0] - (w0 * v0 + (1 - w0) * v1)) < TOL
    assert abs(lse[0] - (s0 + math.log1p(math.exp(s1 - s0)))) < TOL


def pin_rows_matches_full(lib):
    """The selected-rows entry point equals the full computation on the same rows."""
    BH, Nq, Nk, d = 3, 9, 14, 5
    q = _rand((BH, Nq, d), 30)
    k = _rand((BH, Nk, d), 31)
    v = _rand((BH, Nk, d), 32)
    o, lse = oracle.attention(q, k, v, True, 0.9, lib=lib)
    pairs = [(0, 0), (2, 8), (1, 4), (2, 0)]
    kk = np.stack([k[bh] for bh in range(BH)])
    vv = np.stack([v[bh] for bh in range(BH)])
    qr = np.stack([q[bh, r] for bh, r in pairs])
    orow, lrow = oracle.attention_rows(qr, [r for _, r in pairs], [bh for bh, _ in pairs], kk, vv, Nq, True, 0.9,
                                       lib=lib)
    for n, (bh, r) in enumerate(pairs):
        assert np.allclose(orow[n], o[bh, r], atol=0, rtol=0)
        assert lrow[n] == lse[bh, r]


def _loss_grad_fd(q, k, v, g, causal, scale, lib, h=1e-6):
    """Central differences of L = sum(O * g) with respect to every entry of q, k and v."""
    out = []
    for x in (q, k, v):
        dx = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            op, _ = oracle.attention(q, k, v, causal, scale, lib=lib)
            x[idx] = old - h
            om, _ = oracle.attention(q, k, v, causal, scale, lib=lib)
            x[idx] = old
            dx[idx] = ((op - om) * g).sum() / (2 * h)
        out.append(dx)
    return out


def pin_bwd_finite_differences(lib):
    """The backward is the derivative of the forward: central differences of
    L = sum(O * dO) through the forward definition ("Lecture 25" §3.3).

    The cases include Nq != Nk and, causal with Nq > Nk, rows that see no key."""
    for n, (Nq, Nk, d, causal) in enumerate([(4, 6, 3, False), (5, 5, 2, True), (6, 3, 2, True)]):
        q = _rand((1, Nq, d), 40 + n)
        k = _rand((1, Nk, d), 50 + n)
        v = _rand((1, Nk, d), 60 + n)
        g = _rand((1, Nq, d), 70 + n)
        dq, dk, dv = oracle.attention_bwd(q, k, v, g, causal, 0.7, lib=lib)
        fq, fk, fv = _loss_grad_fd(q, k, v, g, causal, 0.7, lib)
        for got, want in ((dq, fq), (dk, fk), (dv, fv)):
            assert np.allclose(got, want, atol=1e-8, rtol=0), n


def pin_bwd_two_key_closed_form(lib):
    """d = 1, one query, two keys: O = w v0 + (1 - w) v1 with w = sigmoid(a),
    a = scale q (k0 - k1).  With dO = g: dv0 = w g, dv1 = (1 - w) g,
    dq = w(1-w) scale (k0 - k1)(v0 - v1) g, dk0 = -dk1 = w(1-w) scale q (v0 - v1) g."""
    for (qv, k0, k1, v0, v1, g, sc) in [(0.8, 0.5, -1.0, 2.0, -1.0, 1.5, 0.9), (-1.2, 2.0, 0.3, 0.5, 3.0, -0.7, 1.3)]:
        q = np.array([[[qv]]])
        k = np.array([[[k0], [k1]]])
        v = np.array([[[v0], [v1]]])
        dq, dk, dv = oracle.attention_bwd(q, k, v, np.array([[[g]]]), False, sc, lib=lib)
        w = 1.0 / (1.0 + math.exp(-sc * qv * (k0 - k1)))
        ww = w * (1.0 - w)
        assert abs(dv[0, 0, 0] - w * g) < TOL and abs(dv[0, 1, 0] - (1 - w) * g) < TOL
        assert abs(dq[0, 0, 0] - ww * sc * (k0 - k1) * (v0 - v1) * g) < TOL
        assert abs(dk[0, 0, 0] - ww * sc * qv * (v0 - v1) * g) < TOL
        assert abs(dk[0, 1, 0] + ww * sc * qv * (v0 - v1) * g) < TOL


def pin_bwd_autograd_library(lib):
    """Independent library routine: torch autograd in fp64 through CPU
    scaled_dot_product_attention (square and bottom-right causal)."""
    cases = [(1, 2, 40, 40, 16, True), (2, 1, 33, 70, 8, False), (1, 1, 20, 50, 32, True), (1, 2, 64, 64, 64, False)]
    for n, (B, H, Nq, Nk, d, causal) in enumerate(cases):
        gen = torch.Generator().manual_seed(200 + n)
        q = torch.randn(B, H, Nq, d, generator=gen, dtype=torch.float64, requires_grad=True)
        k = torch.randn(B, H, Nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        v = torch.randn(B, H, Nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        g = torch.randn(B, H, Nq, d, generator=gen, dtype=torch.float64)
        scale = 1.0 / math.sqrt(d)
        mask = None
        if causal:
            mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        o.backward(g)
        dq, dk, dv = oracle.attention_bwd(q.detach(), k.detach(), v.detach(), g, causal, scale, lib=lib)
        for got, want in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
            assert np.allclose(got, want.numpy(), atol=1e-11, rtol=0), f"case {n}"


def pin_bwd_invariants(lib):
    """Facts of the gradient that hold at any size.

    Adding one vector to every key leaves every softmax row unchanged, so the
    dK rows of a head sum to zero; rows of P sum to one, so the dV rows sum to
    the dO rows of the rows that see a key; a row that sees no key has dQ = 0;
    the gradient is linear in dO."""
    BH, Nq, Nk, d = 2, 9, 5, 4
    q = _rand((BH, Nq, d), 80)
    k = _rand((BH, Nk, d), 81)
    v = _rand((BH, Nk, d), 82)
    g1 = _rand((BH, Nq, d), 83)
    g2 = _rand((BH, Nq, d), 84)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g1, True, 0.6, lib=lib)
    assert np.allclose(dk.sum(axis=1), 0.0, atol=1e-12, rtol=0)
    seen = Nq - Nk  # causal, Nq > Nk: rows below this index see no key
    assert np.allclose(dv.sum(axis=1), g1[:, seen:].sum(axis=1), atol=1e-12, rtol=0)
    assert (dq[:, :seen] == 0).all() and np.abs(dq[:, seen:]).max() > 0
    a = oracle.attention_bwd(q, k, v, g1, True, 0.6, lib=lib)
    b = oracle.attention_bwd(q, k, v, g2, True, 0.6, lib=lib)
    c = oracle.attention_bwd(q, k, v, 2.0 * g1 - 3.0 * g2, True, 0.6, lib=lib)
    for x, y, z in zip(a, b, c):
        assert np.allclose(z, 2.0 * x - 3.0 * y, atol=1e-12, rtol=0)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def failing_pins(lib):
    """Names of the pins that fail (or crash) for ``lib``."""
    bad = []
    for fn in ALL_PINS:
        try:
            fn(lib)
        except Exception:  # noqa: BLE001 - any failure counts
            bad.append(fn.__name__)
    return bad
