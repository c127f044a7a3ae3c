"""The host entry point (attention_host): inputs in pinned host memory, results
copied back, heads streamed through the device in chunks whose copies
overlap the kernels of other chunks.  Chunking by heads must not change the
results: the forward equals the device call bit for bit (each head's
arithmetic is the same), the gradients match it up to the order of fp32
reduce-adds, and all of them match the fp64 oracle."""
import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _case(seed, T_texts, N, H, H_kv, d, q_mul=1.0):
    cu = [0]
    for L in T_texts:
        cu.append(cu[-1] + N + L)
    T = cu[-1]
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((T, H, d), generator=g) * q_mul).to(torch.bfloat16)
    k = torch.randn((T, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, H_kv, d), generator=g).to(torch.bfloat16)
    do = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    return cu, q, k, v, do


@pytest.mark.parametrize("chunks,scale", [(1, None), (2, None), (4, None), (4, 1.0)])
def test_host_pipeline_matches_device_call_and_oracle(chunks, scale):
    import vlm_zigzag_head_gb300 as cp
    P, N, texts, H, H_kv, d = 2, 64, [512, 1024], 8, 4, 128
    cu, q, k, v, do = _case(40 + chunks, texts, N, H, H_kv, d,
                            q_mul=d ** -0.5 if scale == 1.0 else 1.0)
    sc = scale if scale is not None else d ** -0.5
    hq, hk, hv, hdo = (x.pin_memory() for x in (q, k, v, do))
    out, lse, dq, dk, dv = cp.attention_host(hq, hk, hv, hdo, cu, P, N, sc, device=DEV,
                                             chunks=chunks)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o2, l2, lo2 = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, sc, residual=True)
    g2 = cp.cp_attn_bwd_gqa(qd, kd, vd, o2, l2, dod, cu, P, N, sc, out_lo=lo2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o2.cpu().view(torch.int16))
    assert torch.equal(lse, l2.cpu())
    for name, a, b in (("dq", dq, g2[0]), ("dk", dk, g2[1]), ("dv", dv, g2[2])):
        b = b.cpu().double()
        err = float((a.double() - b).norm() / b.norm())
        assert err < 1e-5, (name, err)
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, sc)
    dq_ref, dk_ref, dv_ref = oracle.causal_attention_bwd(q, k, v, do, cu, sc)
    for name, got, want in (("out", out, o_ref), ("lse", lse, l_ref), ("dq", dq, dq_ref),
                            ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        assert_close(name, got, want, "bf16")


def test_host_pipeline_forward_only_and_chunk_choice():
    import vlm_zigzag_head_gb300 as cp
    assert cp.host_chunks(131072, 32, 32, 128, 2) == 4
    assert cp.host_chunks(8192, 16, 16, 128, 2) == 1
    assert cp.host_chunks(131072, 32, 2, 128, 2) == 2
    P, N, texts, H, H_kv, d = 2, 0, [1024], 4, 2, 64
    cu, q, k, v, _ = _case(77, texts, N, H, H_kv, d)
    out, lse = cp.attention_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), None, cu, P,
                                 N, 0.125, device=DEV, chunks=2)
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, 0.125)
    assert_close("out", out, o_ref, "bf16")
    assert_close("lse", lse, l_ref, "bf16")
