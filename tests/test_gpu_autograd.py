"""The torch.autograd binding: gradients through ``cp_attention`` equal the
oracle's, and the prefix hook sees the per-rank terms whose sum is the
prefix gradient (the multimodal CP page, §4.2 and §5.2)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import F32_REL, assert_close, to64

DEV = "cuda:0"


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


def _leaves(cu, H, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    ts = [torch.randn((cu[-1], H, d), generator=g).to(dtype) for _ in range(4)]
    return ts[:3], ts[3]


@pytest.mark.gpu
@pytest.mark.parametrize("P,N,texts", [(2, 64, [256, 512]), (4, 0, [1024])])
def test_autograd_matches_oracle_bf16(P, N, texts):
    from vlm_zigzag_head_gb300.autograd import cp_attention
    H, d = 2, 128
    cu = _cu(N, texts)
    (q, k, v), w = _leaves(cu, H, d, torch.bfloat16, 40 + P)
    scale = d ** -0.5
    qd, kd, vd = (x.to(DEV).requires_grad_(True) for x in (q, k, v))
    out, lse = cp_attention(qd, kd, vd, cu, P, N, scale)
    loss = (out.float() * w.to(DEV).float()).sum()
    loss.backward()
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    g_ref = oracle.causal_attention_bwd(q, k, v, w, cu, scale)
    assert_close("out", out.cpu(), o_ref, "bf16")
    assert_close("lse", lse.cpu(), lse_ref, "bf16")
    for name, got, want in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), g_ref):
        assert got.dtype == torch.bfloat16
        assert_close(name, got.cpu(), want, "bf16")


@pytest.mark.gpu
def test_autograd_fp32_and_partial_requires_grad():
    from vlm_zigzag_head_gb300.autograd import cp_attention
    P, N, texts, H, d = 2, 16, [256], 1, 64
    cu = _cu(N, texts)
    (q, k, v), w = _leaves(cu, H, d, torch.float32, 7)
    qd, kd = q.to(DEV), k.to(DEV)
    vd = v.to(DEV).requires_grad_(True)
    out, _ = cp_attention(qd, kd, vd, cu, P, N)
    (out * w.to(DEV)).sum().backward()
    torch.cuda.synchronize()
    assert qd.grad is None and kd.grad is None
    g_ref = oracle.causal_attention_bwd(q, k, v, w, cu, d ** -0.5)
    r = assert_close("dv", vd.grad.cpu(), g_ref[2], "f32")
    assert r <= F32_REL


@pytest.mark.gpu
def test_prefix_hook_sees_per_rank_terms():
    from vlm_zigzag_head_gb300.autograd import cp_attention
    P, N, texts, H, d = 4, 128, [1024, 512], 2, 128
    cu = _cu(N, texts)
    (q, k, v), w = _leaves(cu, H, d, torch.bfloat16, 11)
    seen = []
    qd, kd, vd = (x.to(DEV).requires_grad_(True) for x in (q, k, v))
    out, _ = cp_attention(qd, kd, vd, cu, P, N, prefix_hook=lambda t: seen.append(t.clone()))
    (out.float() * w.to(DEV).float()).sum().backward()
    torch.cuda.synchronize()
    assert len(seen) == 1
    terms = seen[0].cpu()
    n = len(texts)
    assert tuple(terms.shape) == (2, P + 1, n * N, H, d)
    # the fixed-order sum of the terms is the prefix gradient autograd received
    rows = np.concatenate([np.arange(cu[i], cu[i] + N) for i in range(n)])
    g_ref = oracle.causal_attention_bwd(q, k, v, w, cu, d ** -0.5)
    for slot, want in ((0, g_ref[1]), (1, g_ref[2])):
        total = to64(terms[slot]).sum(axis=0)
        assert_close("prefix sum %d" % slot, total, to64(want)[rows], "bf16")
    assert_close("dk prefix", kd.grad.cpu()[rows], to64(g_ref[1])[rows], "bf16")


def test_autograd_refuses_cpu_tensors():
    from vlm_zigzag_head_gb300 import CpError
    from vlm_zigzag_head_gb300.autograd import cp_attention
    q = torch.zeros((256, 1, 64), requires_grad=True)
    with pytest.raises(CpError):
        cp_attention(q, q, q, [0, 256], 2)


@pytest.mark.gpu
def test_autograd_grouped_kv_heads():
    """k / v with fewer heads than q (grouped-query attention): autograd
    receives dk / dv shaped like k / v, equal to the oracle's group sums."""
    from vlm_zigzag_head_gb300.autograd import cp_attention
    P, N, texts, H, H_kv, d = 2, 32, [512, 256], 4, 2, 128
    cu = _cu(N, texts)
    g = torch.Generator().manual_seed(19)
    q = torch.randn((cu[-1], H, d), generator=g).to(torch.bfloat16)
    k = torch.randn((cu[-1], H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((cu[-1], H_kv, d), generator=g).to(torch.bfloat16)
    w = torch.randn((cu[-1], H, d), generator=g).to(torch.bfloat16)
    qd, kd, vd = (x.to(DEV).requires_grad_(True) for x in (q, k, v))
    out, _ = cp_attention(qd, kd, vd, cu, P, N)
    (out.float() * w.to(DEV).float()).sum().backward()
    torch.cuda.synchronize()
    g_ref = oracle.causal_attention_bwd(q, k, v, w, cu, d ** -0.5)
    assert kd.grad.shape == k.shape and vd.grad.shape == v.shape
    for name, got, want in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), g_ref):
        assert_close(name, got.cpu(), want, "bf16")
