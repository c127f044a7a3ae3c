"""The fixed-scratch forward (cp_attn_fwd_noalloc), for callers that cannot
allocate device memory: through the C ABI it must give the same results as
cp_attn_fwd, on two calls in a row (the shared scratch keeps the previous
call's contents), and refuse problems larger than its scratch.

Collected last on purpose: a failure here leaves every other test already run.
Passes alone in a fresh process and after the other tests."""
import ctypes

import pytest
import torch

from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(cu, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((cu[-1], H, d), generator=g).to(torch.bfloat16).to(DEV) for _ in range(3)]


def _noalloc(B, q, k, v, cu, P, N, scale, out, lse, out_lo):
    T, H, d = q.shape
    return B.lib().cp_attn_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), B.CP_BF16, T, H, d, B.cu_array(cu), len(cu) - 1, P, N,
        scale, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(out_lo.data_ptr()), None)


def test_noalloc_forward_matches_workspace_forward_twice():
    import vlm_zigzag_head_gb300 as cp
    from vlm_zigzag_head_gb300 import _binding as B
    cases = [  # (P, N, texts, H): a packed VLM-like case, then a different shape
        (4, 130, [512, 1024], 2),
        (2, 0, [2048], 4),
    ]
    for P, N, texts, H in cases:
        cu = [0]
        for L in texts:
            cu.append(cu[-1] + N + L)
        q, k, v = _inputs(cu, H, 128, 7 + P)
        scale = 128 ** -0.5
        ref_out, ref_lse, ref_lo = cp.cp_attn_fwd(q, k, v, cu, P, N, scale, residual=True)
        torch.cuda.synchronize()
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            lse = torch.full((H, cu[-1]), float("nan"), device=DEV)
            lo = torch.full_like(q, float("nan"))
            st = _noalloc(B, q, k, v, cu, P, N, scale, out, lse, lo)
            assert st == 0, B.lib().cp_last_error()
            torch.cuda.synchronize()
            assert_close("out", out.cpu(), ref_out.cpu(), "bf16")
            assert_close("lse", lse.cpu(), ref_lse.cpu(), "bf16")
            assert_close("out_lo", lo.cpu().float() + out.cpu().float(),
                         ref_lo.cpu().float() + ref_out.cpu().float(), "bf16")


def test_noalloc_forward_rejects_problems_beyond_its_scratch():
    from vlm_zigzag_head_gb300 import _binding as B
    cu = [0, 65536]
    H, d = 8, 128
    x = torch.empty((8, 16), dtype=torch.bfloat16, device=DEV)   # never read: size check first
    p = ctypes.c_void_p(x.data_ptr())
    st = B.lib().cp_attn_fwd_noalloc(p, p, p, B.CP_BF16, cu[-1], H, d, B.cu_array(cu), 1, 2, 0,
                                     0.1, p, p, None, None)
    assert st == 5
    assert b"fixed scratch" in B.lib().cp_last_error()
