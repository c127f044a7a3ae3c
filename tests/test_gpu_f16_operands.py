"""Above softmax scale 0.25 the bf16 path runs P V, S = Q K^T, dQ = dS K and
dK = dS^T Q on f16 operands: per-call f16 copies of V (forward) and of Q and K
(backward) scaled by powers of two found on the device, and dS scaled by a
power of two bounded through max |V| max |dO|.

Scaling the inputs by powers of two must therefore change nothing but the
exponents: with q * 2^-a, k * 2^a, v * 2^b and dO * 2^c (all exact in bf16)
the logits are unchanged and

    out -> out * 2^b      lse -> lse          dV -> dV * 2^c
    dS  -> dS * 2^(b+c)   dQ -> dQ * 2^(a+b+c)   dK -> dK * 2^(b+c-a)

bit for bit where the kernels sum in a fixed order (out, lse, dK, dV), and
up to the order of the fp32 reduce-adds for dQ.  A plain bf16 -> f16
conversion would overflow at these magnitudes (|v| near 2^30).  The unscaled
run is checked against the fp64 oracle as well."""
import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


def _run(cp, q, k, v, do, cu, P, N, scale):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, lo = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, scale, residual=True)
    dq, dk, dv = cp.cp_attn_bwd_gqa(qd, kd, vd, o, lse, dod, cu, P, N, scale, out_lo=lo)
    torch.cuda.synchronize()
    assert cp.cp_workspace_status(cp.default_workspace("fwd", qd.device)) == 0
    assert cp.cp_workspace_status(cp.default_workspace("bwd", qd.device)) == 0
    return {n: x.cpu() for n, x in zip(("out", "lse", "lo", "dq", "dk", "dv"),
                                       (o, lse, lo, dq, dk, dv))}


@pytest.mark.parametrize("P,N,texts,H,H_kv,d,a,b,c", [
    (3, 37, [384, 0, 1152], 2, 2, 128, 20, 30, -25),
    (2, 0, [1024], 4, 2, 64, -12, -40, 18),
])
def test_power_of_two_input_scaling_is_exact(P, N, texts, H, H_kv, d, a, b, c):
    import vlm_zigzag_head_gb300 as cp
    cu = _cu(N, texts)
    T = cu[-1]
    g = torch.Generator().manual_seed(1000 + d)
    q = (torch.randn((T, H, d), generator=g) * d ** -0.5).to(torch.bfloat16)
    k = torch.randn((T, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, H_kv, d), generator=g).to(torch.bfloat16)
    do = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    base = _run(cp, q, k, v, do, cu, P, N, 1.0)

    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, 1.0)
    dq_ref, dk_ref, dv_ref = oracle.causal_attention_bwd(q, k, v, do, cu, 1.0)
    for name, want in (("out", o_ref), ("lse", l_ref), ("dq", dq_ref), ("dk", dk_ref),
                       ("dv", dv_ref)):
        assert_close(name, base[name], want, "bf16")

    p2 = lambda e: 2.0 ** e  # noqa: E731
    scaled = _run(cp, q * p2(-a), k * p2(a), v * p2(b), do * p2(c), cu, P, N, 1.0)
    assert torch.equal(scaled["lse"], base["lse"])
    for name, e in (("out", b), ("lo", b)):
        assert torch.equal(scaled[name].float(), base[name].float() * p2(e)), name
    for name, e in (("dk", b + c - a), ("dv", c)):
        assert torch.equal(scaled[name], base[name] * p2(e)), name
    dq_s = scaled["dq"].double() * p2(-(a + b + c))
    err = (dq_s - base["dq"].double()).norm() / base["dq"].double().norm()
    assert err < 1e-6, err
