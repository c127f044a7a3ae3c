"""The two tensor-core forward schedules against the fp64 CPU oracle.

By default the bf16 forward is one persistent launch in which every query
tile walks the KV tiles of all ring steps in ring order, so the log-sum-exp
merge of the per-step partials is its online softmax.  With
CPATTN_FWD_PER_STEP=1 (read once per process) it is one launch per ring step
that merges into an fp32 running result.  Both compute the same attention
(CP-VLM page §1 ring order, §4.1 prefix) and must meet the bf16 tolerance;
the per-step schedule runs in a child process with that variable set.
"""
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

CHILD = r"""
import sys, torch
import vlm_zigzag_head_gb300 as cp
d = torch.load(sys.argv[1])
q, k, v = (d[n].to("cuda:0") for n in ("q", "k", "v"))
out, lse, lo = cp.cp_attn_fwd(q, k, v, d["cu"], d["P"], d["N"], d["scale"], residual=True)
torch.cuda.synchronize()
torch.save({"out": out.cpu(), "lse": lse.cpu(), "lo": lo.cpu()}, sys.argv[2])
"""


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


CASES = [
    # (P, prefix, texts, H, scale, q_mul)
    (1, 0, [512], 2, 128 ** -0.5, 1.0),                 # one ring step
    (2, 0, [2048], 4, 1.0, 128 ** -0.5),                # text, scale 1: PV on f16 operands
    (4, 576, [1536, 512, 0], 2, 128 ** -0.5, 1.0),      # prefix, packed, text-less sample
    (8, 0, [4096], 2, 128 ** -0.5, 1.0),                # P = 8: 15 key runs per tile
    (3, 37, [384, 1152], 3, 128 ** -0.5, 1.0),          # ragged chunks (c = 64, 192)
]


@pytest.mark.parametrize("P,N,texts,H,scale,q_mul", CASES)
def test_all_steps_and_per_step_forward(cp, tmp_path, P, N, texts, H, scale, q_mul):
    cu = _cu(N, texts)
    T, d = cu[-1], 128
    g = torch.Generator().manual_seed(900 + P + H)
    q = (torch.randn((T, H, d), generator=g) * q_mul).to(torch.bfloat16)
    k = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, H, d), generator=g).to(torch.bfloat16)

    out, lse, lo = cp.cp_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cu, P, N, scale,
                                  residual=True)
    torch.cuda.synchronize()
    fused = {"out": out.cpu(), "lse": lse.cpu(), "lo": lo.cpu()}

    src, dst = tmp_path / "in.pt", tmp_path / "out.pt"
    torch.save({"q": q, "k": k, "v": v, "cu": cu, "P": P, "N": N, "scale": scale}, src)
    env = dict(os.environ, CPATTN_FWD_PER_STEP="1")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD, str(src), str(dst)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    step = torch.load(dst)

    o_ref, l_ref = oracle.causal_attention_fwd(q, k, v, cu, scale)
    for name, res in (("all-steps", fused), ("per-step", step)):
        assert_close(name + " out", res["out"], o_ref, "bf16")
        assert_close(name + " lse", res["lse"], l_ref, "bf16")
        # out + out_lo carries the fp32 result: much closer than bf16 out alone
        assert_close(name + " out+lo", res["out"].double() + res["lo"].double(), o_ref, "bf16")
    # the two schedules differ only in the order of the fp32 merge
    diff = (fused["out"].double() + fused["lo"].double()
            - step["out"].double() - step["lo"].double()).abs().max().item()
    assert diff <= 5e-3, diff
    assert (fused["lse"] - step["lse"]).abs().max().item() <= 1e-3
