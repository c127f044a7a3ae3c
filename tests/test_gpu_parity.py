"""GPU parity of the CUDA path against the fp64 CPU oracle, through the C ABI.

Small cases are compared element by element over the whole output; the large
workloads on seeded heads / rows / keys the oracle computes one by one, and
at full length through identities that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import BF16_ABS, BF16_REL, assert_close, rel_l2, to64
from vlm_zigzag_head_gb300 import workloads as W

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


def _inputs(cu, H, d, dtype, seed, dout=True, q_mul=1.0):
    T = cu[-1]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((T, H, d), generator=g) * q_mul
    k = torch.randn((T, H, d), generator=g)
    v = torch.randn((T, H, d), generator=g)
    do = torch.randn((T, H, d), generator=g) if dout else None
    cast = (lambda x: x.to(dtype)) if dtype != torch.float32 else (lambda x: x)
    return [cast(x) if x is not None else None for x in (q, k, v, do)]


def _run(cp, q, k, v, do, cu, P, N, scale, per_rank=False):
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    keep = do is not None and q.dtype == torch.bfloat16
    r = cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, residual=keep)
    out, lse = r[0], r[1]
    res = {"out": out, "lse": lse}
    if do is not None:
        g = cp.cp_attn_bwd(qd, kd, vd, out, lse, do.to(DEV), cu, P, N, scale,
                           per_rank_prefix=per_rank, out_lo=r[2] if keep else None)
        res.update(dq=g[0], dk=g[1], dv=g[2])
        if per_rank:
            res["pgrad"] = g[3]
    torch.cuda.synchronize()
    return {k_: v_.cpu() for k_, v_ in res.items()}


def _check_full(cp, cu, P, N, H, d, dtype, seed, scale, bwd=True, heads=None, q_mul=1.0):
    q, k, v, do = _inputs(cu, H, d, dtype, seed, dout=bwd, q_mul=q_mul)
    got = _run(cp, q, k, v, do, cu, P, N, scale)
    hs = list(range(H)) if heads is None else list(heads)
    sel = lambda x: x[:, hs]  # noqa: E731
    o_ref, l_ref = oracle.causal_attention_fwd(sel(q), sel(k), sel(v), cu, scale)
    tag = "f32" if dtype == torch.float32 else "bf16"
    assert_close("out", got["out"][:, hs], o_ref, tag)
    assert_close("lse", got["lse"][hs], l_ref, tag)
    if bwd:
        dq, dk, dv = oracle.causal_attention_bwd(sel(q), sel(k), sel(v), sel(do), cu, scale)
        assert_close("dq", got["dq"][:, hs], dq, tag)
        assert_close("dk", got["dk"][:, hs], dk, tag)
        assert_close("dv", got["dv"][:, hs], dv, tag)
    return got


# ---------------------------------------------------------------------------
# zigzag index / permutation kernels: bit-exact
# ---------------------------------------------------------------------------
def _many_texts(P, n, seed):
    g = torch.Generator().manual_seed(seed)
    return [int(x) * 2 * P for x in torch.randint(0, 9, (n,), generator=g)]


# The device tables come from the same kernel cp_attn_fwd launches for its
# gather (sample tables travel in its parameters, 192 samples per launch: the
# 401-sample case spans three launches).
INDEX_CASES = [(1, 0, [256]), (2, 0, [256]), (3, 37, [384, 0, 1152]),
               (4, 576, [1024, 0, 3072]), (8, 3, [32, 16]), (8, 64, [1024, 2048, 0, 512]),
               (2, 5, _many_texts(2, 401, 3)), (3, 0, [0, 0, 6] + _many_texts(3, 200, 4))]


@pytest.mark.parametrize("P,N,texts", INDEX_CASES)
def test_index_and_permutation_bit_exact(cp, P, N, texts):
    cu = _cu(N, texts)
    fwd, inv = cp.cp_zigzag_index(cu, N, P, device=DEV)
    ofwd, oinv = oracle.zigzag_index(cu, N, P)
    assert np.array_equal(fwd.cpu().numpy().astype(np.int64), ofwd)
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), oinv)
    x = torch.randn((cu[-1], 3, 64), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    xd = x.to(DEV)
    g = cp.cp_zigzag_gather(xd, fwd)
    assert torch.equal(g.cpu().view(torch.int16), x[torch.as_tensor(ofwd)].view(torch.int16))
    back = torch.zeros_like(xd)
    cp.cp_zigzag_scatter(g, fwd, back)
    text = torch.as_tensor(ofwd)
    assert torch.equal(back.cpu()[text].view(torch.int16), x[text].view(torch.int16))


# ---------------------------------------------------------------------------
# standalone LSE merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge_matches_oracle(cp, out_dtype):
    g = torch.Generator().manual_seed(7)
    n, rows, H, d = 3, 200, 4, 128
    po = torch.randn((n, rows, H, d), generator=g)
    pl = torch.randn((n, H, rows), generator=g) * 3
    pl[1, :, :50] = float("-inf")          # a part that saw nothing
    pl[:, 0, 7] = float("-inf")            # a row no part saw
    out, lse = cp.cp_lse_merge(po.to(DEV), pl.to(DEV), out_dtype)
    o_ref, l_ref = oracle.lse_merge(list(po), list(pl))
    assert torch.isneginf(lse.cpu()[0, 7])
    assert torch.all(out.cpu()[7, 0] == 0)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(to64(lse)), fin)
    assert rel_l2(lse.cpu()[torch.as_tensor(fin)], l_ref[fin]) < 1e-6
    tag = "f32" if out_dtype == torch.float32 else "bf16"
    assert_close("merge out", out, o_ref, tag)


# ---------------------------------------------------------------------------
# fp32 path (CUDA cores): rel-L2 <= 1e-5
# ---------------------------------------------------------------------------
def test_tiny_workload_fp32(cp):
    w = W.get("tiny")
    x = W.make_inputs(w)
    got = _run(cp, x.q, x.k, x.v, None, x.cu_seqlens, w.P, w.prefix_len, x.scale)
    o_ref, l_ref = oracle.causal_attention_fwd(x.q, x.k, x.v, x.cu_seqlens, x.scale)
    assert_close("out", got["out"], o_ref, "f32")
    assert_close("lse", got["lse"], l_ref, "f32")


@pytest.mark.parametrize("P,N,texts,d", [(2, 0, [256], 64), (3, 70, [384, 0, 192], 64),
                                         (1, 0, [200], 128), (4, 130, [8, 1024], 128)])
def test_fp32_fwd_bwd_packed_prefix(cp, P, N, texts, d):
    _check_full(cp, _cu(N, texts), P, N, 2, d, torch.float32, 11 + P, d ** -0.5)


# ---------------------------------------------------------------------------
# bf16 path (tensor cores)
# ---------------------------------------------------------------------------
EDGE = [
    # (P, N, texts, H, d)
    (1, 0, [256], 2, 128),             # no ring: one step
    (2, 0, [4], 1, 128),               # c = 1
    (2, 0, [512], 2, 64),              # d = 64
    (4, 576, [1536, 512], 2, 128),     # ragged prefix tiles (576 = 4.5 x 128)
    (3, 37, [384, 0, 1152], 2, 128),   # text-less sample, c = 64 / 192 (ragged)
    (8, 0, [2048], 2, 128),            # P = 8
    (2, 300, [0], 2, 128),             # prefix only
    (2, 4, [8] * 200, 1, 64),          # 200 packed samples (index kernel batches of 192)
]


@pytest.mark.parametrize("P,N,texts,H,d", EDGE)
def test_bf16_edge_cases(cp, P, N, texts, H, d):
    _check_full(cp, _cu(N, texts), P, N, H, d, torch.bfloat16, 21 + P, d ** -0.5)


def test_bf16_text_llm_workload(cp):
    w = W.get("text_llm")
    x = W.make_inputs(w)
    got = _run(cp, x.q, x.k, x.v, x.dout, x.cu_seqlens, w.P, w.prefix_len, x.scale)
    hs = [0, 7, 15]
    sel = lambda t: t[:, hs]  # noqa: E731
    o_ref, l_ref = oracle.causal_attention_fwd(sel(x.q), sel(x.k), sel(x.v), x.cu_seqlens, x.scale)
    assert_close("out", got["out"][:, hs], o_ref, "bf16")
    assert_close("lse", got["lse"][hs], l_ref, "bf16")
    dq, dk, dv = oracle.causal_attention_bwd(sel(x.q), sel(x.k), sel(x.v), sel(x.dout),
                                             x.cu_seqlens, x.scale)
    assert_close("dq", got["dq"][:, hs], dq, "bf16")
    assert_close("dk", got["dk"][:, hs], dk, "bf16")
    assert_close("dv", got["dv"][:, hs], dv, "bf16")


def test_bf16_text_llm_double_scaling_reading(cp):
    """The other reading of the Text LLM workload: q pre-scaled by 1/sqrt(128)
    and the softmax scale 1/sqrt(d) applied as well (reduced length)."""
    _check_full(cp, [0, 2048], 2, 0, 4, 128, torch.bfloat16, 5, 128 ** -0.5, q_mul=128 ** -0.5)


@pytest.mark.parametrize("name,heads", [("vlm_prefix", [0, 31]), ("packed_vlm", [0, 31])])
def test_bf16_vlm_workloads(cp, name, heads):
    w = W.get(name)
    x = W.make_inputs(w)
    got = _run(cp, x.q, x.k, x.v, x.dout, x.cu_seqlens, w.P, w.prefix_len, x.scale)
    sel = lambda t: t[:, heads]  # noqa: E731
    o_ref, l_ref = oracle.causal_attention_fwd(sel(x.q), sel(x.k), sel(x.v), x.cu_seqlens, x.scale)
    assert_close("out", got["out"][:, heads], o_ref, "bf16")
    assert_close("lse", got["lse"][heads], l_ref, "bf16")
    dq, dk, dv = oracle.causal_attention_bwd(sel(x.q), sel(x.k), sel(x.v), sel(x.dout),
                                             x.cu_seqlens, x.scale)
    assert_close("dq", got["dq"][:, heads], dq, "bf16")
    assert_close("dk", got["dk"][:, heads], dk, "bf16")
    assert_close("dv", got["dv"][:, heads], dv, "bf16")


def test_per_rank_prefix_gradients(cp):
    """Per-rank prefix dK/dV before the sum match the partitioned oracle's
    per-rank terms, and the summed prefix rows match the plain gradient."""
    P, N, texts, H, d = 4, 130, [512, 1024], 2, 128
    cu = _cu(N, texts)
    q, k, v, do = _inputs(cu, H, d, torch.bfloat16, 31)
    got = _run(cp, q, k, v, do, cu, P, N, d ** -0.5, per_rank=True)
    _, dk, dv, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, N, P, d ** -0.5)
    pg = got["pgrad"]
    for r in range(P + 1):
        assert_close("prefix dk slot %d" % r, pg[0, r], pdk[r], "bf16")
        assert_close("prefix dv slot %d" % r, pg[1, r], pdv[r], "bf16")
    pre = [t for a in cu[:-1] for t in range(a, a + N)]
    assert_close("prefix dk", got["dk"][pre], dk[pre], "bf16")
    assert_close("prefix dv", got["dv"][pre], dv[pre], "bf16")


def _long_check_keys(T, c):
    """Keys whose gradients come from several ring steps: the last 64 keys of
    zigzag chunks 12, 13 and 14 (ranks 3, 2, 1 at P = 8) are met by their own
    rank at step 0 and by the ranks holding later chunks at steps 5..7; the
    last 256 keys (chunk 15) only by rank 0 at step 0."""
    ends = [13 * c, 14 * c, 15 * c]
    return np.concatenate([np.arange(e - 64, e) for e in ends] + [np.arange(T - 256, T)])


def test_bf16_long_workload_sampled(cp):
    """128K tokens, P=8: out/lse/dQ on 4096 seeded query rows (2 heads), dK/dV
    at 448 keys (2 heads) that include keys met at ring steps 5..7, and at
    every key the identities sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 per
    head."""
    w = W.get("long")
    x = W.make_inputs(w)
    got = _run(cp, x.q, x.k, x.v, x.dout, x.cu_seqlens, w.P, w.prefix_len, x.scale)
    heads = [0, 31]
    rows = W.sample_rows(x.T, 4096, w.seed).numpy()
    o_ref, l_ref, dq_ref = oracle.causal_attention_fwd_rows(x.q, x.k, x.v, x.cu_seqlens, x.scale,
                                                           rows, heads=heads, dout=x.dout)
    r_t = torch.as_tensor(rows)
    assert_close("out rows", got["out"][r_t][:, heads], o_ref, "bf16")
    assert_close("lse rows", got["lse"][heads][:, r_t], l_ref, "bf16")
    assert_close("dq rows", got["dq"][r_t][:, heads], dq_ref, "bf16")
    keys = _long_check_keys(x.T, W.text_lengths(w)[0] // (2 * w.P))
    dk_ref, dv_ref = oracle.causal_attention_bwd_keys(x.q, x.k, x.v, x.dout, x.cu_seqlens,
                                                      x.scale, keys, heads=heads)
    k_t = torch.as_tensor(keys)
    assert_close("dk keys", got["dk"][k_t][:, heads], dk_ref, "bf16")
    assert_close("dv keys", got["dv"][k_t][:, heads], dv_ref, "bf16")
    # The identities hold exactly; in finite precision the residual over all
    # 131072 keys of a sum of independent per-key errors is ||e|| ~ sqrt(n)
    # sigma_e against ||dK|| ~ sqrt(n) sigma_dK, i.e. the per-key relative
    # error, which the bf16 bound caps at BF16_REL.
    sum_dv = got["dv"].double().sum(0)
    sum_do = x.dout.double().sum(0)
    assert rel_l2(sum_dv, sum_do) < BF16_REL
    sum_dk = got["dk"].double().sum(0)
    assert float(sum_dk.norm() / got["dk"].double().norm()) < BF16_REL


# ---------------------------------------------------------------------------
# error paths on the device
# ---------------------------------------------------------------------------
def test_device_error_paths(cp):
    cu = [0, 256]
    q, k, v, _ = _inputs(cu, 1, 64, torch.bfloat16, 1, dout=False)
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    flat = torch.empty(256 * 64 + 8, dtype=torch.bfloat16, device=DEV)
    bad = flat[1:1 + 256 * 64].view(256, 1, 64)        # 2-byte offset: not 16-aligned
    with pytest.raises(cp.CpError) as e:
        cp.cp_attn_fwd(bad, kd, vd, cu, 2, 0, 0.125)
    assert e.value.status == 4
    tiny_ws = cp.Workspace(DEV)
    tiny_ws.buf = torch.empty(512, dtype=torch.uint8, device=DEV)
    import ctypes
    from vlm_zigzag_head_gb300 import _binding as B
    out = torch.empty_like(qd)
    lse = torch.empty((1, 256), device=DEV)
    st = B.lib().cp_attn_fwd(ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()),
                             ctypes.c_void_p(vd.data_ptr()), 1, 256, 1, 64, B.cu_array(cu), 1, 2,
                             0, 0.125, ctypes.c_void_p(out.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr()), None, ctypes.c_void_p(tiny_ws.ptr()),
                             tiny_ws.nbytes(), None)
    assert st == 5
    with pytest.raises(cp.CpError) as e:
        cp.cp_attn_fwd(qd, kd, vd, [0, 250, 256], 2, 0, 0.125)
    assert e.value.status == 2
    # empty input is a no-op
    z = torch.empty((0, 1, 64), dtype=torch.bfloat16, device=DEV)
    o, l = cp.cp_attn_fwd(z, z, z, [0, 0], 2, 0, 0.125)
    assert o.numel() == 0
