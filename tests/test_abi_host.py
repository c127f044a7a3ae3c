"""Host-side checks of the C ABI (no GPU): every declared symbol is exported,
the host index builder is bit-exact against the oracle, the work lists cover
exactly the pairs the oracle's masks allow, and bad arguments give the
documented status codes."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from vlm_zigzag_head_gb300 import _binding as B
from vlm_zigzag_head_gb300 import cp_plan_pairs, cp_zigzag_index, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(cp_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(cplib):
    names = _declared_symbols()
    assert {"cp_attn_fwd", "cp_attn_bwd", "cp_lse_merge", "cp_zigzag_index"} <= names
    for n in names:
        assert hasattr(cplib, n), n
    assert cplib.cp_version() == 1
    assert set(B.SIGNATURES) >= names


def test_bounds_checked_library_builds_and_exports_every_symbol():
    """The debug build (-DCPATTN_BOUNDS_CHECK) compiles from the same sources
    and exports the same C ABI; its kernels run in the -m gpu tests."""
    from vlm_zigzag_head_gb300 import build
    path = build.build(checked=True)
    lib = ctypes.CDLL(path)
    for n in _declared_symbols():
        assert hasattr(lib, n), n
    lib.cp_status_string.restype = ctypes.c_char_p
    assert lib.cp_status_string(9) == b"CP_ERR_BOUNDS"


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


CASES = [(2, 0, [256]), (1, 0, [16]), (3, 5, [12, 0, 24]), (4, 576, [1024, 2048, 512]),
         (8, 3, [32, 16]), (8, 0, [131072]), (4, 2304, [16384, 16384])]


@pytest.mark.parametrize("P,N,texts", CASES)
def test_host_index_bit_exact_vs_oracle(cplib, P, N, texts):
    cu = _cu(N, texts)
    fwd, inv = cp_zigzag_index(cu, N, P)
    ofwd, oinv = oracle.zigzag_index(cu, N, P)
    assert np.array_equal(fwd.numpy().astype(np.int64), ofwd)
    assert np.array_equal(inv.numpy().astype(np.int64), oinv)


def test_host_index_on_named_workloads(cplib):
    for name in workloads.WORKLOADS:
        w = workloads.get(name)
        cu = workloads.cu_seqlens(w)
        fwd, inv = cp_zigzag_index(cu, w.prefix_len, w.P)
        ofwd, oinv = oracle.zigzag_index(cu, w.prefix_len, w.P)
        assert np.array_equal(fwd.numpy().astype(np.int64), ofwd), name
        assert np.array_equal(inv.numpy().astype(np.int64), oinv), name


@pytest.mark.parametrize("P,N,texts", [(2, 0, [256]), (1, 3, [8]), (3, 5, [12, 0, 24]),
                                       (4, 130, [1024, 512]), (8, 3, [32, 16]),
                                       (2, 200, [0, 384])])
def test_work_lists_cover_exactly_the_visible_pairs(cplib, P, N, texts):
    """Forward (query tiles x key runs) and backward (key tiles x query runs)
    work lists cover, per ring step, exactly the pairs the oracle's masks
    allow (prefix-query pairs in step 0)."""
    cu = _cu(N, texts)
    fwd_pairs, bwd_pairs, fwd_items, bwd_items = cp_plan_pairs(cu, N, P)
    counts, self_pairs = oracle.cp_pair_counts(cu, N, P)
    want = counts.sum(axis=0)
    want[0] += self_pairs
    assert fwd_pairs == want.tolist()
    assert bwd_pairs == want.tolist()


@pytest.mark.parametrize("name", ["text_llm", "vlm_prefix", "packed_vlm", "long"])
def test_work_lists_match_closed_form_on_workloads(cplib, name):
    w = workloads.get(name)
    cu = workloads.cu_seqlens(w)
    fwd_pairs, bwd_pairs, _, _ = cp_plan_pairs(cu, w.prefix_len, w.P)
    P, N = w.P, w.prefix_len
    want = [0] * P
    for L in workloads.text_lengths(w):
        c = L // (2 * P)
        want[0] += P * (c * c + c * (c + 1) + 2 * c * N) + N * (N + 1) // 2
        for s in range(1, P):
            want[s] += P * 2 * c * c
    assert fwd_pairs == want and bwd_pairs == want
    total = sum((N + L) * (N + L + 1) // 2 for L in workloads.text_lengths(w))
    assert sum(want) == total


def test_bad_arguments_return_status(cplib):
    L = cplib
    cu = B.cu_array([0, 10])
    assert L.cp_zigzag_index(cu, 1, 0, 2, None, None, 0, None) == 2        # 10 % 4 != 0
    assert L.cp_zigzag_index(None, 1, 0, 2, None, None, 0, None) == 1
    assert L.cp_zigzag_index(cu, 1, 0, 0, None, None, 0, None) == 1       # P < 1
    assert L.cp_zigzag_index(B.cu_array([0, 3]), 1, 4, 1, None, None, 0, None) == 2  # prefix > len
    assert L.cp_attn_fwd_workspace_size(1, 10, 1, 64, cu, 1, 2, 0, 0.1) == 0
    assert L.cp_attn_fwd_workspace_size(1, 8, 1, 64, B.cu_array([0, 8]), 1, 2, 0, 0.1) > 0
    # d not in {64,128}, wrong dtype, null tensors, misaligned pointers
    cu8 = B.cu_array([0, 8])
    fake = ctypes.c_void_p(1 << 20)
    def fwd(q, dt, T, d, lo=None):
        return L.cp_attn_fwd(q, fake, fake, dt, T, 1, d, cu8, 1, 2, 0, 1.0, fake, fake, lo, fake,
                             1 << 20, None)
    assert fwd(fake, 1, 8, 96) == 2                                        # d not in {64, 128}
    assert fwd(fake, 7, 8, 64) == 3                                        # dtype
    assert fwd(None, 1, 8, 64) == 1                                        # null tensor
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert fwd(odd, 1, 8, 64) == 4                                         # misaligned
    assert fwd(fake, 1, 9, 64) == 2                                        # T != cu[-1]
    assert fwd(fake, 0, 8, 64, lo=fake) == 3                               # out_lo with fp32
    L.cp_zigzag_index(cu, 1, 0, 2, None, None, 0, None)
    assert b"not divisible" in L.cp_last_error()
    assert L.cp_status_string(7) == b"CP_ERR_TIMEOUT"


def test_copy_rows_arguments(cplib):
    """cp_copy_rows checks its arguments before any CUDA call: nothing to copy
    is CP_OK, a null pointer or a row wider than a pitch is CP_ERR_INVALID_ARG."""
    L = cplib
    p = ctypes.c_void_p(1 << 20)
    assert L.cp_copy_rows(p, 64, p, 64, 64, 0, None) == 0
    assert L.cp_copy_rows(None, 64, p, 64, 64, 4, None) == 1
    assert L.cp_copy_rows(p, 32, p, 64, 64, 4, None) == 1
    assert b"pitch" in L.cp_last_error()


def test_grouped_kv_arguments(cplib):
    """The grouped-KV entry points: H must be a positive multiple of H_kv, the
    KV-side workspace shrinks with H_kv, and H_kv == H sizes like the plain
    calls."""
    L = cplib
    cu = B.cu_array([0, 16])
    assert L.cp_attn_fwd_workspace_size_gqa(1, 16, 6, 4, 128, cu, 1, 2, 0, 0.1) == 0
    assert L.cp_attn_bwd_workspace_size_gqa(1, 16, 4, 0, 128, cu, 1, 2, 0, 0.1) == 0
    assert L.cp_attn_fwd_workspace_size_gqa(1, 16, 8, 8, 128, cu, 1, 2, 0, 0.1) == \
        L.cp_attn_fwd_workspace_size(1, 16, 8, 128, cu, 1, 2, 0, 0.1)
    assert L.cp_attn_bwd_workspace_size_gqa(0, 16, 8, 8, 64, cu, 1, 2, 0, 0.1) == \
        L.cp_attn_bwd_workspace_size(0, 16, 8, 64, cu, 1, 2, 0, 0.1)
    assert 0 < L.cp_attn_fwd_workspace_size_gqa(1, 16, 8, 2, 128, cu, 1, 2, 0, 0.1) < \
        L.cp_attn_fwd_workspace_size_gqa(1, 16, 8, 8, 128, cu, 1, 2, 0, 0.1)
    fake = ctypes.c_void_p(1 << 20)
    st = L.cp_attn_fwd_gqa(fake, fake, fake, 1, 16, 6, 4, 128, cu, 1, 2, 0, 1.0, fake, fake,
                           None, fake, 1 << 20, None)
    assert st == 2 and b"multiple of H_kv" in L.cp_last_error()
    st = L.cp_attn_bwd_gqa(fake, fake, fake, fake, None, fake, fake, 1, 16, 4, 3, 128, cu, 1, 2,
                           0, 1.0, fake, fake, fake, None, fake, 1 << 20, None)
    assert st == 2


@pytest.mark.skipif(os.environ.get("CPATTN_FWD_PER_STEP") == "1",
                    reason="the per-step schedule merges through the running result")
def test_forward_workspace_is_sized_by_schedule(cplib):
    """The default bf16 forward merges its ring steps on chip, so its
    workspace holds the rank-local q/k/v but no fp32 running result; the fp32
    path merges through one ([rows][H][d] fp32 plus lse) and reserves it."""
    L = cplib
    rows, H, d = 4096, 8, 128
    cu = B.cu_array([0, rows])
    ws_bf16 = L.cp_attn_fwd_workspace_size(1, rows, H, d, cu, 1, 2, 0, 0.1)
    ws_f32 = L.cp_attn_fwd_workspace_size(0, rows, H, d, cu, 1, 2, 0, 0.1)
    qkv_bf16, qkv_f32 = 3 * rows * H * d * 2, 3 * rows * H * d * 4
    running = rows * H * (d + 1) * 4
    assert qkv_bf16 <= ws_bf16 < qkv_bf16 + running // 4
    assert ws_f32 >= qkv_f32 + running


def test_f16_operand_copies_are_sized_by_softmax_scale(cplib):
    """Above softmax scale 0.25 the bf16 forward keeps an f16 copy of V and the
    backward f16 copies of Q and K (plus one 256-byte block of factors); at or
    below it, and for fp32, nothing is added."""
    L = cplib
    rows, H, Hkv, d = 4096, 8, 2, 128
    cu = B.cu_array([0, rows])
    f = lambda dt, sc: L.cp_attn_fwd_workspace_size_gqa(dt, rows, H, Hkv, d, cu, 1, 2, 0, sc)  # noqa: E731
    b = lambda dt, sc: L.cp_attn_bwd_workspace_size_gqa(dt, rows, H, Hkv, d, cu, 1, 2, 0, sc)  # noqa: E731
    assert f(1, 0.25) == f(1, 0.088) and b(1, 0.25) == b(1, 0.088)
    assert f(1, 1.0) - f(1, 0.25) == 256 + rows * Hkv * d * 2
    assert b(1, 1.0) - b(1, 0.25) == 256 + rows * (H + Hkv) * d * 2
    assert f(0, 1.0) == f(0, 0.1) and b(0, 1.0) == b(0, 0.1)
