"""GPU parity of the grouped-KV-head variant (GQA / MQA) against the fp64 CPU
oracle, through the C ABI (cp_attn_fwd_gqa / cp_attn_bwd_gqa).

Query head h reads KV head h // (H / H_kv); dK / dV of a KV head sum its query
heads' terms.  Covered: the tensor-core forward and backward (both dS paths),
multi-query attention (H_kv = 1), the image prefix with per-rank prefix
gradients, packed samples, and the CUDA-core paths (fp32, and bf16 with
head_dim 64).  The forward must also be bit-identical to the plain call on
K / V whose heads were repeated to H."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def cp():
    import vlm_zigzag_head_gb300 as cp_mod
    cp_mod._binding.lib()   # loud failure if the library is missing
    return cp_mod


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


def _inputs(cu, H, H_kv, d, dtype, seed, q_mul=1.0):
    T = cu[-1]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((T, H, d), generator=g) * q_mul
    k = torch.randn((T, H_kv, d), generator=g)
    v = torch.randn((T, H_kv, d), generator=g)
    do = torch.randn((T, H, d), generator=g)
    if dtype != torch.float32:
        q, k, v, do = (x.to(dtype) for x in (q, k, v, do))
    return q, k, v, do


def _run(cp, q, k, v, do, cu, P, N, scale, per_rank=False):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    bf16 = q.dtype == torch.bfloat16
    r = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, scale, residual=bf16)
    out, lse = r[0], r[1]
    g = cp.cp_attn_bwd_gqa(qd, kd, vd, out, lse, dod, cu, P, N, scale,
                           per_rank_prefix=per_rank, out_lo=r[2] if bf16 else None)
    torch.cuda.synchronize()
    res = {"out": out, "lse": lse, "dq": g[0], "dk": g[1], "dv": g[2]}
    if per_rank:
        res["pgrad"] = g[3]
    return {k_: v_.cpu() for k_, v_ in res.items()}


CASES = [
    # (P, prefix, texts, H, H_kv, d, dtype, scale, q_mul)
    (2, 0, [2048], 8, 2, 128, torch.bfloat16, 128 ** -0.5, 1.0),        # text, G = 4
    (4, 192, [1024, 512], 8, 1, 128, torch.bfloat16, 128 ** -0.5, 1.0),  # MQA, prefix, packed
    (3, 37, [384, 0, 1152], 6, 3, 128, torch.bfloat16, 1.0, 128 ** -0.5),  # scale 1: f16 operands
    (2, 5, [256, 128], 4, 2, 64, torch.bfloat16, 0.125, 1.0),            # d = 64
    (3, 37, [384, 0, 768], 4, 2, 64, torch.bfloat16, 1.0, 64 ** -0.5),   # d = 64, scale 1
    (2, 0, [1024], 2, 2, 64, torch.bfloat16, 1.0, 64 ** -0.5),           # d = 64, scale 1, MHA
    (2, 5, [64, 32], 4, 2, 64, torch.float32, 0.125, 1.0),               # fp32 CUDA-core path
]


@pytest.mark.parametrize("P,N,texts,H,H_kv,d,dtype,scale,q_mul", CASES)
def test_gqa_matches_oracle(cp, P, N, texts, H, H_kv, d, dtype, scale, q_mul):
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, H_kv, d, dtype, 300 + P + H_kv, q_mul)
    got = _run(cp, q, k, v, do, cu, P, N, scale)
    assert got["dk"].shape == (cu[-1], H_kv, d) and got["dv"].shape == (cu[-1], H_kv, d)
    tag = "f32" if dtype == torch.float32 else "bf16"
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, scale)
    for name, want in (("out", o_ref), ("lse", l_ref), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, got[name], want, tag)


def test_gqa_per_rank_prefix_gradients(cp):
    """Per-rank prefix dK / dV (one slot per rank and one for the prefix
    queries), summed over each KV head's query heads, against the
    partitioned oracle."""
    P, N, texts, H, H_kv = 2, 300, [512], 4, 2
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, H_kv, 128, torch.bfloat16, 41)
    got = _run(cp, q, k, v, do, cu, P, N, 128 ** -0.5, per_rank=True)
    _, _, _, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, N, P, 128 ** -0.5)
    pg = got["pgrad"]
    assert pg.shape == (2, P + 1, N, H_kv, 128)
    assert_close("prefix dk slots", pg[0], pdk, "bf16")
    assert_close("prefix dv slots", pg[1], pdv, "bf16")


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_gqa_forward_equals_plain_call_on_repeated_kv(cp, dtype, d):
    """Each query head runs the same arithmetic as the plain call does on K / V
    with heads repeated to H, so the forward outputs agree bit for bit."""
    P, N, texts, H, H_kv = 4, 64, [512, 1024], 8, 2
    cu = _cu(N, texts)
    q, k, v, _ = _inputs(cu, H, H_kv, d, dtype, 77)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    o1, l1 = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, 0.1)
    G = H // H_kv
    kr, vr = (x.repeat_interleave(G, dim=1).contiguous() for x in (kd, vd))
    o2, l2 = cp.cp_attn_fwd(qd, kr, vr, cu, P, N, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o1.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       o2.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(l1.cpu(), l2.cpu())


def test_gqa_backward_close_to_plain_call_on_repeated_kv(cp):
    """dQ agrees with the plain call on repeated K / V, and dK / dV equal the
    plain call's gradients summed over each group (up to fp32 summation
    order)."""
    P, N, texts, H, H_kv = 2, 0, [1024], 8, 2
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, H_kv, 128, torch.bfloat16, 78)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, l, lo = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, 0.09, residual=True)
    g1 = cp.cp_attn_bwd_gqa(qd, kd, vd, o, l, dod, cu, P, N, 0.09, out_lo=lo)
    G = H // H_kv
    kr, vr = (x.repeat_interleave(G, dim=1).contiguous() for x in (kd, vd))
    g2 = cp.cp_attn_bwd(qd, kr, vr, o, l, dod, cu, P, N, 0.09, out_lo=lo)
    torch.cuda.synchronize()
    fold = lambda x: x.view(x.shape[0], H_kv, G, x.shape[2]).sum(2)  # noqa: E731
    for a, b in ((g1[0], g2[0]), (g1[1], fold(g2[1])), (g1[2], fold(g2[2]))):
        a, b = a.double().cpu(), b.double().cpu()
        assert float((a - b).norm() / b.norm()) < 1e-5
        assert np.isfinite(a.numpy()).all()


def test_gqa_large_grid_without_group_split(cp):
    """Enough key tiles that each KV head's group stays in one CTA (no
    reduce-add of partial dK / dV): checked on query heads 0, 1 and their KV
    head 0, the oracle computing those heads only."""
    P, N, texts, H, H_kv = 2, 0, [8192], 32, 16
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, H_kv, 128, torch.bfloat16, 91)
    got = _run(cp, q, k, v, do, cu, P, N, 128 ** -0.5)
    qs, ks, vs, ds = q[:, 0:2], k[:, 0:1], v[:, 0:1], do[:, 0:2]
    o_ref, l_ref = oracle.causal_attention_fwd(qs, ks, vs, cu, 128 ** -0.5)
    dq, dk, dv = oracle.causal_attention_bwd(qs, ks, vs, ds, cu, 128 ** -0.5)
    assert_close("out", got["out"][:, 0:2], o_ref, "bf16")
    assert_close("lse", got["lse"][0:2], l_ref, "bf16")
    assert_close("dq", got["dq"][:, 0:2], dq, "bf16")
    assert_close("dk", got["dk"][:, 0:1], dk, "bf16")
    assert_close("dv", got["dv"][:, 0:1], dv, "bf16")


def test_gqa_long_workload_sampled(cp):
    """128K tokens, P = 8, 32 query heads over 8 KV heads, at full size.
    out / lse / dQ on 2048 seeded rows of query heads 0 and 5, and dK / dV of
    KV head 0 (the sum of its 4 query heads' terms) on the last 64 keys of
    zigzag chunk 14, which rank 0's chunk-15 queries meet at ring step 7, and
    on the last 256 keys, from
    the oracle's row- and key-sampled forms.  At every key, per KV head,
    sum_j dV_j equals the sum of dO over the group's query heads, and
    sum_j dK_j = 0."""
    from gpu_util import BF16_REL, rel_l2
    from vlm_zigzag_head_gb300 import workloads as W
    w = W.get("long", H_kv=8)
    x = W.make_inputs(w)
    got = _run(cp, x.q, x.k, x.v, x.dout, x.cu_seqlens, w.P, w.prefix_len, x.scale)
    G = w.H // w.kv_heads
    rows = W.sample_rows(x.T, 2048, w.seed).numpy()
    r_t = torch.as_tensor(rows)
    for h in (0, 5):
        o_ref, l_ref, dq_ref = oracle.causal_attention_fwd_rows(
            x.q[:, h:h + 1], x.k[:, h // G:h // G + 1], x.v[:, h // G:h // G + 1], x.cu_seqlens,
            x.scale, rows, dout=x.dout[:, h:h + 1])
        assert_close("out rows h%d" % h, got["out"][r_t][:, h:h + 1], o_ref, "bf16")
        assert_close("lse rows h%d" % h, got["lse"][h:h + 1][:, r_t], l_ref, "bf16")
        assert_close("dq rows h%d" % h, got["dq"][r_t][:, h:h + 1], dq_ref, "bf16")
    c = x.T // (2 * w.P)
    keys = np.concatenate([np.arange(15 * c - 64, 15 * c), np.arange(x.T - 256, x.T)])
    dk_ref = dv_ref = 0
    for h in range(G):                      # the query heads of KV head 0
        a, b = oracle.causal_attention_bwd_keys(x.q[:, h:h + 1], x.k[:, 0:1], x.v[:, 0:1],
                                                x.dout[:, h:h + 1], x.cu_seqlens, x.scale, keys)
        dk_ref, dv_ref = dk_ref + a, dv_ref + b
    k_t = torch.as_tensor(keys)
    assert_close("dk keys", got["dk"][k_t][:, 0:1], dk_ref, "bf16")
    assert_close("dv keys", got["dv"][k_t][:, 0:1], dv_ref, "bf16")
    sum_dv = got["dv"].double().sum(0)
    sum_do = x.dout.double().view(x.T, w.kv_heads, G, w.d).sum(dim=(0, 2))
    assert rel_l2(sum_dv, sum_do) < BF16_REL
    sum_dk = got["dk"].double().sum(0)
    assert float(sum_dk.norm() / got["dk"].double().norm()) < BF16_REL
