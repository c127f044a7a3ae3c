"""Failure detection without a GPU fault: every mbarrier wait of the
tensor-core kernels is bounded.  With the bound cut to one polling round,
waits give up; the kernels then wait (with a fixed bound) for their own
copies and products in flight, free TMEM, and report CP_ERR_TIMEOUT through
the workspace status word.  The context stays usable: the next call with the
normal bound is exact again."""
import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CP_ERR_TIMEOUT = 7


def test_timeout_is_reported_and_the_context_recovers():
    import vlm_zigzag_head_gb300 as cp
    P, N, texts, H, d = 2, 64, [2048, 1024], 4, 128
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + N + L)
    g = torch.Generator().manual_seed(5)
    q, k, v, do = (torch.randn((cu[-1], H, d), generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    scale = d ** -0.5
    ws_f, ws_b = cp.Workspace(DEV), cp.Workspace(DEV)
    seen = []
    cp.cp_set_wait_limit(1)
    try:
        for _ in range(3):
            out, lse, lo = cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, workspace=ws_f,
                                          residual=True)
            seen.append(cp.cp_workspace_status(ws_f))
            cp.cp_attn_bwd(qd, kd, vd, out, lse, dod, cu, P, N, scale, workspace=ws_b,
                           out_lo=lo)
            seen.append(cp.cp_workspace_status(ws_b))
    finally:
        cp.cp_set_wait_limit(0)
    torch.cuda.synchronize()
    assert all(s in (0, CP_ERR_TIMEOUT) for s in seen), seen
    assert CP_ERR_TIMEOUT in seen, seen
    # normal bound again: the same workspaces, exact results
    out, lse, lo = cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, workspace=ws_f, residual=True)
    dq, dk, dv = cp.cp_attn_bwd(qd, kd, vd, out, lse, dod, cu, P, N, scale, workspace=ws_b,
                                out_lo=lo)
    assert cp.cp_workspace_status(ws_f) == 0 and cp.cp_workspace_status(ws_b) == 0
    o_ref, lse_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    g_ref = oracle.causal_attention_bwd(q, k, v, do, cu, scale)
    assert_close("out", out.cpu(), o_ref, "bf16")
    assert_close("lse", lse.cpu(), lse_ref, "bf16")
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        assert_close(name, got.cpu(), want, "bf16")
