"""The bounds-checked debug build (libcpattn_checked.so, -DCPATTN_BOUNDS_CHECK)
on the small parity cases.

Its tensor-core kernels test every row and head index against the tensor's
extent before each TMA load, TMA reduce and global store, and report a failed
test as CP_ERR_BOUNDS through the workspace status word instead of touching
the address.  On valid problems no test may fail: every call here must leave
status CP_OK, match the fp64 oracle within the method's tolerances, and give
a forward bit-identical to the normal library's (the checks add no
arithmetic).  Covered: the all-steps and per-step forwards, the 128-query
backward (head_dim 128 and 64, grouped KV heads, per-rank prefix gradients),
the f16-operand products above softmax scale 0.25, and the fixed-scratch
forward.

The library is built on first use (a minute or two)."""
import os
import subprocess
import sys

import pytest
import torch

import oracle
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cp():
    import vlm_zigzag_head_gb300 as cp_mod
    from vlm_zigzag_head_gb300 import build
    build.build(checked=True)
    cp_mod._binding.lib()
    return cp_mod


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


def _inputs(cu, H, H_kv, d, seed, q_mul=1.0):
    g = torch.Generator().manual_seed(seed)
    T = cu[-1]
    q = (torch.randn((T, H, d), generator=g) * q_mul).to(torch.bfloat16)
    k, v = (torch.randn((T, H_kv, d), generator=g).to(torch.bfloat16) for _ in range(2))
    do = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    return q, k, v, do


def _fwd_bwd(cp, q, k, v, do, cu, P, N, scale, per_rank=False):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, lo = cp.cp_attn_fwd_gqa(qd, kd, vd, cu, P, N, scale, residual=True)
    g = cp.cp_attn_bwd_gqa(qd, kd, vd, o, lse, dod, cu, P, N, scale, per_rank_prefix=per_rank,
                           out_lo=lo)
    torch.cuda.synchronize()
    st_f = cp.cp_workspace_status(cp.default_workspace("fwd", qd.device))
    st_b = cp.cp_workspace_status(cp.default_workspace("bwd", qd.device))
    return [x.cpu() for x in (o, lse, lo) + tuple(g)], (st_f, st_b)


CASES = [
    # (P, prefix, texts, H, H_kv, d, scale, q_mul, per_rank)
    (4, 130, [512, 1024], 2, 2, 128, 128 ** -0.5, 1.0, False),   # packed, ragged prefix tiles
    (3, 37, [384, 0, 1152], 2, 2, 128, 1.0, 128 ** -0.5, False),  # scale 1: f16 operands
    (2, 5, [256, 128], 4, 4, 64, 0.125, 1.0, False),              # head_dim 64
    (2, 0, [2048], 8, 2, 128, 128 ** -0.5, 1.0, False),           # grouped KV heads
    (2, 300, [512], 4, 2, 128, 128 ** -0.5, 1.0, True),           # per-rank prefix gradients
]


@pytest.mark.parametrize("P,N,texts,H,H_kv,d,scale,q_mul,per_rank", CASES)
def test_checked_build_matches_oracle_and_normal_build(cp, P, N, texts, H, H_kv, d, scale,
                                                        q_mul, per_rank):
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, H_kv, d, 500 + P + H, q_mul)
    ref, st_ref = _fwd_bwd(cp, q, k, v, do, cu, P, N, scale, per_rank)
    with cp._binding.bounds_checked():
        got, st = _fwd_bwd(cp, q, k, v, do, cu, P, N, scale, per_rank)
    assert st == (0, 0) and st_ref == (0, 0), (st, st_ref)
    # the forward is deterministic and the checks add no arithmetic
    for name, a, b in zip(("out", "lse", "out_lo"), got[:3], ref[:3]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, scale)
    for name, x, want in (("out", got[0], o_ref), ("lse", got[1], l_ref), ("dq", got[3], dq),
                          ("dk", got[4], dk), ("dv", got[5], dv)):
        assert_close(name, x, want, "bf16")
    if per_rank:
        _, _, _, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, N, P, scale)
        assert_close("prefix dk slots", got[6][0], pdk, "bf16")
        assert_close("prefix dv slots", got[6][1], pdv, "bf16")


def test_checked_build_fixed_scratch_forward(cp):
    P, N, texts, H, d = 4, 130, [512, 1024], 2, 128
    cu = _cu(N, texts)
    q, k, v, _ = _inputs(cu, H, H, d, 61)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    ref = cp.cp_attn_fwd_noalloc(qd, kd, vd, cu, P, N, d ** -0.5)
    with cp._binding.bounds_checked():
        got = cp.cp_attn_fwd_noalloc(qd, kd, vd, cu, P, N, d ** -0.5)
        torch.cuda.synchronize()
        assert cp.cp_workspace_status() == 0
    torch.cuda.synchronize()
    assert torch.equal(got[0].cpu().view(torch.int16), ref[0].cpu().view(torch.int16))
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, d ** -0.5)
    assert_close("out", got[0].cpu(), o_ref, "bf16")
    assert_close("lse", got[1].cpu(), l_ref, "bf16")


CHILD = r"""
import sys, torch
import vlm_zigzag_head_gb300 as cp
a = torch.load(sys.argv[1])
dev = "cuda:0"
with cp._binding.bounds_checked():
    o, l, lo = cp.cp_attn_fwd(a["q"].to(dev), a["k"].to(dev), a["v"].to(dev), a["cu"], a["P"],
                              a["N"], a["scale"], residual=True)
    torch.cuda.synchronize()
    st = cp.cp_workspace_status(cp.default_workspace("fwd", torch.device(dev)))
torch.save({"out": o.cpu(), "lse": l.cpu(), "status": st}, sys.argv[2])
"""


def test_checked_build_per_step_forward(cp, tmp_path):
    """One launch per ring step with the fp32 running result in between
    (CPATTN_FWD_PER_STEP=1, read once per process: run in a child)."""
    P, N, texts, H, d = 3, 37, [384, 0, 1152], 2, 128
    cu = _cu(N, texts)
    q, k, v, _ = _inputs(cu, H, H, d, 62)
    src, dst = tmp_path / "in.pt", tmp_path / "out.pt"
    torch.save({"q": q, "k": k, "v": v, "cu": cu, "P": P, "N": N, "scale": d ** -0.5}, src)
    env = dict(os.environ, CPATTN_FWD_PER_STEP="1")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD, str(src), str(dst)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = torch.load(dst)
    assert res["status"] == 0
    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, d ** -0.5)
    assert_close("out", res["out"], o_ref, "bf16")
    assert_close("lse", res["lse"], l_ref, "bf16")
