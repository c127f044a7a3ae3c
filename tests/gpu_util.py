"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (stated by the method's correctness targets):
  * indices and permutations: bit-exact;
  * fp32 inputs: relative L2 error <= 1e-5;
  * bf16 inputs, fp32 accumulation: relative L2 <= 5e-3 and max |err| <= 2e-2,
    on out, lse, dQ, dK and dV.
"""
import numpy as np
import torch

F32_REL = 1e-5
BF16_REL = 5e-3
BF16_ABS = 2e-2


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2(got, want):
    got, want = to64(got), to64(want)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def max_abs(got, want):
    got, want = to64(got), to64(want)
    return float(np.abs(got - want).max()) if got.size else 0.0


def assert_close(name, got, want, dtype):
    got, want = to64(got), to64(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), name + ": non-finite values"
    r = rel_l2(got, want)
    if dtype == "f32":
        assert r <= F32_REL, "%s: rel-L2 %.3e > %.0e" % (name, r, F32_REL)
    else:
        m = max_abs(got, want)
        assert r <= BF16_REL, "%s: rel-L2 %.3e > %.0e" % (name, r, BF16_REL)
        assert m <= BF16_ABS, "%s: max-abs %.3e > %.0e" % (name, m, BF16_ABS)
    return r
