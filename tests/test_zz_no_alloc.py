"""The fixed-scratch forward (cp_attn_fwd_noalloc), for callers that cannot
allocate device memory (their memory belongs to another allocator, or to a
budget fixed up front).  Through the C ABI, on two calls in a row (the shared
scratch keeps the previous call's contents), it must match the fp64 oracle
within the method's tolerances and give the same results as cp_attn_fwd; it
must refuse problems larger than its scratch, and a device wait that gives up
must show in cp_workspace_status with no workspace.

Collected last on purpose: a failure here leaves every other test already run.
Passes alone in a fresh process and after the other tests."""
import ctypes

import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CP_ERR_TIMEOUT = 7


def _cu(N, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + N + L)
    return cu


def _inputs(cu, H, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    xs = [torch.randn((cu[-1], H, d), generator=g) for _ in range(3)]
    return [x.to(dtype) if dtype != torch.float32 else x for x in xs]


def _noalloc(B, q, k, v, cu, P, N, scale, out, lse, out_lo):
    T, H, d = q.shape
    dt = B.CP_BF16 if q.dtype == torch.bfloat16 else B.CP_F32
    return B.lib().cp_attn_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), dt, T, H, d, B.cu_array(cu), len(cu) - 1, P, N,
        scale, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(out_lo.data_ptr()) if out_lo is not None else None, None)


CASES = [  # (P, N, texts, H, d, dtype)
    (4, 130, [512, 1024], 2, 128, torch.bfloat16),   # packed, ragged prefix tiles
    (2, 0, [2048], 4, 64, torch.bfloat16),           # head_dim 64
    (3, 37, [384, 0, 192], 2, 64, torch.float32),    # fp32 (CUDA cores), text-less sample
    (2, 300, [0], 2, 128, torch.float32),            # prefix only
]


@pytest.mark.parametrize("P,N,texts,H,d,dtype", CASES)
def test_noalloc_forward_matches_oracle_and_workspace_forward_twice(P, N, texts, H, d, dtype):
    import vlm_zigzag_head_gb300 as cp
    from vlm_zigzag_head_gb300 import _binding as B
    cu = _cu(N, texts)
    q, k, v = _inputs(cu, H, d, dtype, 7 + P + d)
    scale = d ** -0.5
    tag = "bf16" if dtype == torch.bfloat16 else "f32"
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    bf16 = dtype == torch.bfloat16
    r = cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, residual=bf16)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(qd, float("nan"))
        lse = torch.full((H, cu[-1]), float("nan"), device=DEV)
        lo = torch.full_like(qd, float("nan")) if bf16 else None
        st = _noalloc(B, qd, kd, vd, cu, P, N, scale, out, lse, lo)
        assert st == 0, B.lib().cp_last_error()
        assert cp.cp_workspace_status() == 0
        assert_close("out vs oracle", out.cpu(), o_ref, tag)
        assert_close("lse vs oracle", lse.cpu(), l_ref, tag)
        assert_close("out vs cp_attn_fwd", out.cpu(), r[0].cpu(), tag)
        assert_close("lse vs cp_attn_fwd", lse.cpu(), r[1].cpu(), tag)
        if bf16:   # out + out_lo: the fp32 result, also within the bf16 bounds
            assert_close("out + out_lo vs oracle", lo.cpu().double() + out.cpu().double(),
                         o_ref, "bf16")
            assert_close("out_lo vs cp_attn_fwd", lo.cpu().double() + out.cpu().double(),
                         r[2].cpu().double() + r[0].cpu().double(), "bf16")


def test_noalloc_forward_scale_one_uses_the_f16_copy_of_v():
    """Softmax scale 1 on pre-scaled queries: PV on f16 operands, with the f16
    copy of V and its factors held in the fixed scratch."""
    import vlm_zigzag_head_gb300 as cp
    P, N, texts, H, d = 3, 37, [384, 0, 192], 2, 128
    cu = _cu(N, texts)
    q, k, v = _inputs(cu, H, d, torch.bfloat16, 23)
    q = (q.float() * d ** -0.5).to(torch.bfloat16)
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, 1.0)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    r = cp.cp_attn_fwd(qd, kd, vd, cu, P, N, 1.0)
    out, lse = cp.cp_attn_fwd_noalloc(qd, kd, vd, cu, P, N, 1.0)
    torch.cuda.synchronize()
    assert cp.cp_workspace_status() == 0
    assert_close("out vs oracle", out.cpu(), o_ref, "bf16")
    assert_close("lse vs oracle", lse.cpu(), l_ref, "bf16")
    assert torch.equal(out.cpu().view(torch.int16), r[0].cpu().view(torch.int16))
    assert torch.equal(lse.cpu(), r[1].cpu())


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


def test_noalloc_timeout_is_reported_and_the_next_call_is_exact():
    """A bounded wait cut to one polling round gives up inside the fixed-scratch
    forward; cp_workspace_status() without a workspace reports it, and the next
    call with the normal bound is exact again."""
    import vlm_zigzag_head_gb300 as cp
    from vlm_zigzag_head_gb300 import _binding as B
    P, N, texts, H, d = 2, 64, [2048, 1024], 4, 128
    cu = _cu(N, texts)
    q, k, v = _inputs(cu, H, d, torch.bfloat16, 5)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    scale = d ** -0.5
    out = torch.empty_like(qd)
    lse = torch.empty((H, cu[-1]), device=DEV)
    seen = []
    cp.cp_set_wait_limit(1)
    try:
        for _ in range(3):
            assert _noalloc(B, qd, kd, vd, cu, P, N, scale, out, lse, None) == 0
            seen.append(cp.cp_workspace_status())
    finally:
        cp.cp_set_wait_limit(0)
    assert all(s in (0, CP_ERR_TIMEOUT) for s in seen), seen
    assert CP_ERR_TIMEOUT in seen, seen
    assert _noalloc(B, qd, kd, vd, cu, P, N, scale, out, lse, None) == 0
    assert cp.cp_workspace_status() == 0
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    assert_close("out", out.cpu(), o_ref, "bf16")
    assert_close("lse", lse.cpu(), l_ref, "bf16")
