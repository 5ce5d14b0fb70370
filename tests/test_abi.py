"""libfa.so builds, loads and exports every symbol include/fa.h declares; host-side checks (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_forward_03_gb300 import build
    import exact_attention_forward_03_gb300 as fa

    build.build()
    return fa.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    assert {"fa_fwd", "fa_fwd_splitkv", "fa_splitkv_combine", "fa_get_device_status"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    import exact_attention_forward_03_gb300 as fa

    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in fa.EXPORTS


def test_version_and_status_strings(lib):
    assert lib.fa_version() >= 100
    for code in range(-6, 1):
        assert lib.fa_status_string(code)
    assert lib.fa_status_string(12345) == b"unknown status"


def test_validation_without_gpu(lib):
    """Argument checks run before any CUDA call, so they work on a host without a GPU."""
    p = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the call is rejected first
    f = lib.fa_fwd
    assert f(None, p, p, p, None, 1, 1, 8, 8, 64, 0, 0.125, 0, None) == -1       # null q
    assert f(p, p, p, p, None, 0, 1, 8, 8, 64, 0, 0.125, 0, None) == -1          # B = 0
    assert f(p, p, p, p, None, 1, 1, 8, 8, 96, 0, 0.125, 0, None) == -2          # d = 96
    assert f(p, p, p, p, None, 1, 1, 8, 8, 64, 0, -1.0, 0, None) == -1           # scale <= 0
    assert f(p, p, p, p, None, 1, 1, 8, 8, 64, 0, float("nan"), 0, None) == -1  # scale NaN
    assert f(p, p, p, p, None, 1, 1, 8, 8, 64, 2, 0.125, 0, None) == -1          # causal = 2
    assert f(p, p, p, p, None, 1, 1, 8, 8, 64, 0, 0.125, 7, None) == -1          # dtype
    assert f(p, p, p, p, None, 256, 256, 8, 8, 64, 0, 0.125, 0, None) == -1      # B * H past the grid's y limit
    assert f(p, p, p, p, None, 1 << 16, 1 << 16, 8, 8, 64, 0, 0.125, 0, None) == -1  # B * H past int range
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert f(odd, p, p, p, None, 1, 1, 8, 8, 64, 0, 0.125, 0, None) == -3        # q not 16-byte aligned
    assert f(p, p, p, p, ctypes.c_void_p((1 << 20) + 2), 1, 1, 8, 8, 64, 0, 0.125, 0, None) == -3
    c = lib.fa_splitkv_combine
    assert c(None, p, p, None, 4, 1, 1, 1, 64, 0, None) == -1
    assert c(p, p, p, None, 0, 1, 1, 1, 64, 0, None) == -1
    assert c(p, p, p, None, 300, 1, 1, 1, 64, 0, None) == -1
    assert c(p, p, p, None, 4, 1, 1, 1, 32, 0, None) == -2


def test_planned_varlen_validation_without_gpu(lib):
    """fa_fwd_varlen_ws: workspace size formula and argument checks, before any CUDA call."""
    import exact_attention_forward_03_gb300 as fa

    fa.load_library()
    assert lib.fa_fwd_varlen_workspace_bytes(16, 10000) == 16 + 8 * (79 + 16)
    assert lib.fa_fwd_varlen_workspace_bytes(1, 1) == 16 + 8 * 2
    assert lib.fa_fwd_varlen_workspace_bytes(0, 10) == 0 and lib.fa_fwd_varlen_workspace_bytes(3, 0) == 0
    p = ctypes.c_void_p(1 << 20)
    need = lib.fa_fwd_varlen_workspace_bytes(2, 30)
    f = lib.fa_fwd_varlen_ws
    args = lambda ws, nbytes, nseq=2, H=2, H_kv=2: (p, p, p, p, None, p, p, nseq, 30, 30, H, H_kv, 64, 0, 0.125, 1,
                                                      ws, nbytes, None)
    assert f(*args(None, need)) == fa.FA_ERR_WORKSPACE                              # no workspace
    assert f(*args(p, need - 8)) == fa.FA_ERR_WORKSPACE                             # one pair short
    assert f(*args(ctypes.c_void_p((1 << 20) + 8), need)) == fa.FA_ERR_WORKSPACE   # not 16-byte aligned
    assert f(*args(p, need, nseq=0)) == fa.FA_ERR_INVALID_ARG                       # no sequence
    assert f(*args(p, need, H=3, H_kv=2)) == fa.FA_ERR_INVALID_ARG                 # H_kv does not divide H
    assert f(p, p, p, p, None, None, p, 2, 30, 30, 2, 2, 64, 0, 0.125, 1, p, need, None) == fa.FA_ERR_INVALID_ARG


def test_gqa_head_counts_are_checked_without_gpu(lib):
    """H must be a positive multiple of H_kv; checked before any CUDA call."""
    p = ctypes.c_void_p(1 << 20)
    g = lib.fa_fwd_gqa
    assert g(p, p, p, p, None, 1, 8, 3, 8, 8, 64, 0, 0.125, 0, None) == -1   # 8 % 3 != 0
    assert g(p, p, p, p, None, 1, 8, 0, 8, 8, 64, 0, 0.125, 0, None) == -1   # H_kv = 0
    assert g(p, p, p, p, None, 1, 8, -2, 8, 8, 64, 0, 0.125, 0, None) == -1  # H_kv < 0
    assert g(p, p, p, p, None, 1, 8, 2, 8, 8, 96, 0, 0.125, 0, None) == -2   # the common checks still apply
    s = lib.fa_fwd_splitkv_gqa
    assert s(p, p, p, p, None, 1, 6, 4, 1, 64, 64, 0, 0.125, 0, 4, p, 1 << 20, None) == -1
    assert s(p, p, p, p, None, 1, 6, 0, 1, 64, 64, 0, 0.125, 0, 4, p, 1 << 20, None) == -1


def test_split_planning(lib):
    assert lib.fa_splitkv_split_len(16384, 16) == 1024
    assert lib.fa_splitkv_split_len(1000, 8) == 128
    assert lib.fa_splitkv_split_len(65, 32) == 64
    for Nk, S in [(1, 1), (65, 32), (16384, 8), (999, 7)]:
        L = lib.fa_splitkv_split_len(Nk, S)
        assert L % 64 == 0 and L * S >= Nk and L * (S - 1) < Nk + 64 * S
    rows, d, S = 1024, 128, 16
    ws = lib.fa_splitkv_workspace_bytes(32, 32, 1, 16384, d, S)
    assert ws >= S * rows * (d + 1) * 4 and ws % 256 == 0
    assert lib.fa_splitkv_workspace_bytes(32, 32, 1, 16384, 96, S) == 0
    assert lib.fa_splitkv_workspace_bytes(32, 32, 1, 16384, d, 300) == 0


def test_python_binding_refuses_cpu_tensors():
    import torch
    import exact_attention_forward_03_gb300 as fa

    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)


def test_backward_and_fp8_validation_without_gpu(lib):
    """Argument checks of fa_bwd, fa_bwd_gqa, fa_fp8_quantize, fa_fwd_fp8 and the
    self-test run before any CUDA call."""
    p = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    ws = 1 << 30
    b = lib.fa_bwd
    assert b(p, p, p, p, None, p, p, p, p, 1, 2, 8, 8, 128, 0, 0.1, 1, p, ws, None) == -1    # null dout
    assert b(p, p, p, p, p, None, p, p, p, 1, 2, 8, 8, 128, 0, 0.1, 1, p, ws, None) == -1    # null lse
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 8, 8, 96, 0, 0.1, 1, p, ws, None) == -2       # d = 96
    assert b(p, p, p, p, odd, p, p, p, p, 1, 2, 8, 8, 128, 0, 0.1, 1, p, ws, None) == -3     # dout misaligned
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 8, 8, 128, 0, 0.1, 1, None, ws, None) == -4   # no workspace
    need = lib.fa_bwd_workspace_bytes(1, 2, 8, 128)
    assert need == 2 * 128 * 128 * 4 + 2 * 1024
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 8, 8, 128, 0, 0.1, 1, p, need - 1, None) == -4  # short workspace
    g = lib.fa_bwd_gqa
    assert g(p, p, p, p, p, p, p, p, p, 1, 6, 4, 8, 8, 128, 0, 0.1, 1, p, ws, None) == -1   # 6 % 4 != 0
    q = lib.fa_fp8_quantize
    assert q(None, p, p, 4, 128, 128, 0, 1, None) == -1
    assert q(p, p, p, 4, 128, 64, 0, 1, None) == -2      # d = 64
    assert q(p, p, p, 4, 128, 128, 2, 1, None) == -1     # transpose flag
    assert q(odd, p, p, 4, 128, 128, 0, 1, None) == -3
    f = lib.fa_fwd_fp8
    assert f(p, p, p, p, p, p, p, None, 1, 2, 8, 8, 64, 0, 0.1, 1, None) == -2       # d = 64
    assert f(p, None, p, p, p, p, p, None, 1, 2, 8, 8, 128, 0, 0.1, 1, None) == -1   # null q_scale
    assert f(p, p, p, p, odd, p, p, None, 1, 2, 8, 8, 128, 0, 0.1, 1, None) == -3    # v8t misaligned
    assert lib.fa_selftest_timeout(0, None) == -1
    vb = lib.fa_bwd_varlen
    two = ctypes.c_void_p((1 << 20) + 2)
    args = lambda **o: [o.get(n, x) for n, x in (
        ("q", p), ("k", p), ("v", p), ("o", p), ("dout", p), ("lse", p), ("dq", p), ("dk", p), ("dv", p),
        ("cu_q", p), ("cu_k", p), ("num_seqs", 2), ("max_k", 20), ("total_q", 30), ("total_k", 30), ("H", 2),
        ("H_kv", 2), ("d", 64), ("causal", 1), ("scale", 0.1), ("dtype", 1), ("ws", p), ("bytes", ws),
        ("stream", None))]
    assert vb(*args(dout=None)) == -1
    assert vb(*args(lse=None)) == -1
    assert vb(*args(cu_k=None)) == -1
    assert vb(*args(max_k=0)) == -1
    assert vb(*args(max_k=31)) == -1
    assert vb(*args(num_seqs=0)) == -1
    assert vb(*args(H=6, H_kv=4)) == -1
    assert vb(*args(d=96)) == -2
    assert vb(*args(dq=odd)) == -3
    assert vb(*args(cu_q=two)) == -3
    assert vb(*args(ws=None)) == -4
    need = lib.fa_bwd_varlen_workspace_bytes(2, 30, 30, 2, 64)
    # offsets, then per head 128 (ceil(30 / 128) + 2) rows of 64 floats and two vectors, then the
    # key-block work list: 16 + 8 (ceil(30 / 128) + 2) bytes, rounded up to 256
    assert need == 256 + 2 * 384 * 64 * 4 + 2 * (2 * 384 * 4) + 256
    assert lib.fa_bwd_varlen_workspace_bytes(2, 30, 0, 2, 64) == 0
    assert vb(*args(bytes=need - 1)) == -4
    h = lib.fa_fwd_host
    assert h(None, p, p, p, p, 1, 2, 2, 8, 8, 64, 0, 0.1, 1, 0, p, ws, None) == -1       # null q_host
    assert h(p, p, p, p, p, 1, 6, 4, 8, 8, 64, 0, 0.1, 1, 0, p, ws, None) == -1          # 6 % 4 != 0
    assert h(p, p, p, p, p, 1, 2, 2, 8, 8, 96, 0, 0.1, 1, 0, p, ws, None) == -2          # d = 96
    assert h(p, p, p, p, p, 1, 2, 2, 8, 8, 64, 0, 0.1, 1, 0, None, ws, None) == -4       # no workspace
    hneed = lib.fa_fwd_host_workspace_bytes(1, 2, 2, 8, 8, 64)
    assert hneed == 4 * 2048 + 256                        # q, o, k, v (2 heads x 8 x 64 x 2 B), lse
    assert h(p, p, p, p, p, 1, 2, 2, 8, 8, 64, 0, 0.1, 1, 0, p, hneed - 1, None) == -4  # short workspace
