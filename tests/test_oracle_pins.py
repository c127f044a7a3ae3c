"""Pins for the CPU oracle: each test ties it to something other than itself
(the page's worked example, brute force with scalar loops, a library routine,
closed forms, finite differences).  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64).to(dtype)


def _qkv(T, H, d, seed):
    return _rand((T, H, d), seed), _rand((T, H, d), seed + 1), _rand((T, H, d), seed + 2)


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


# ---------------------------------------------------------------------------
# zigzag index
# ---------------------------------------------------------------------------
def _read_golden_example():
    ranks = {}
    P = None
    with open(os.path.join(GOLDEN, "zigzag_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("P="):
                P = int(line[2:])
            else:
                head, tail = line.split(":")
                ranks[int(head.split()[1])] = tuple(int(x) for x in tail.split())
    return P, ranks


def test_worked_example_cp2_chunk_assignment():
    P, ranks = _read_golden_example()
    assert P == 2
    assert oracle.zigzag_chunk_ids(P) == [ranks[0], ranks[1]]
    # the same example at token level: 4 chunks of c=3 text tokens
    fwd, inv = oracle.zigzag_index([0, 12], 0, 2)
    c = 3
    for r, chunks in ranks.items():
        got = fwd[r * 2 * c:(r + 1) * 2 * c].tolist()
        want = [t for ch in chunks for t in range(ch * c, (ch + 1) * c)]
        assert got == want


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8])
def test_index_matches_brute_force_chunk_rule(P):
    # packed samples with a prefix; every text token is classified by brute force
    rng = np.random.default_rng(P)
    prefix = int(rng.integers(0, 5))
    texts = [int(2 * P * rng.integers(0, 4)) for _ in range(3)]
    cu = _cu(prefix, texts)
    fwd, inv = oracle.zigzag_index(cu, prefix, P)
    want = []
    for r in range(P):
        for i in range(len(texts)):
            a = cu[i] + prefix
            c = texts[i] // (2 * P)
            for ch in (r, 2 * P - r - 1):          # the page's [cp_rank, 2*cp_size-cp_rank-1]
                for t in range(a, cu[i + 1]):
                    if (t - a) // max(c, 1) == ch and c > 0:
                        want.append(t)
    assert fwd.tolist() == want


@pytest.mark.parametrize("P", [1, 2, 3, 8])
def test_index_is_a_bijection_and_inverse(P):
    cu = _cu(3, [4 * P, 0, 8 * P])
    fwd, inv = oracle.zigzag_index(cu, 3, P)
    text = [t for i in range(3) for t in range(cu[i] + 3, cu[i + 1])]
    assert sorted(fwd.tolist()) == text
    assert [fwd[k] for k in inv] == text
    assert sorted(inv.tolist()) == list(range(len(text)))


def test_index_rejects_indivisible_text():
    with pytest.raises(ValueError):
        oracle.zigzag_index([0, 10], 0, 2)


# ---------------------------------------------------------------------------
# forward: brute force, library special case, partition invariant
# ---------------------------------------------------------------------------
def _brute_force_fwd(q, k, v, cu, scale):
    """Scalar loops with math.exp: no vectorisation, no shared helpers."""
    T, H, d = q.shape
    out = np.zeros((T, H, d))
    lse = np.zeros((H, T))
    for a, b in zip(cu, cu[1:]):
        for h in range(H):
            for i in range(a, b):
                scores = []
                for j in range(a, i + 1):
                    s = 0.0
                    for e in range(d):
                        s += float(q[i, h, e]) * float(k[j, h, e])
                    scores.append(scale * s)
                z = sum(math.exp(x) for x in scores)
                lse[h, i] = math.log(z)
                for e in range(d):
                    out[i, h, e] = sum(math.exp(x) / z * float(v[a + jj, h, e])
                                       for jj, x in enumerate(scores))
    return out, lse


def test_fwd_matches_scalar_brute_force_packed_prefix():
    cu = _cu(2, [4, 8])
    q, k, v = _qkv(cu[-1], 2, 3, 10)
    out, lse = oracle.causal_attention_fwd(q, k, v, cu, 0.7)
    bo, bl = _brute_force_fwd(q.numpy(), k.numpy(), v.numpy(), cu, 0.7)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("texts,prefix", [([64], 0), ([40, 24, 8], 5)])
def test_fwd_matches_torch_sdpa_per_sample(texts, prefix):
    cu = _cu(prefix, texts)
    q, k, v = _qkv(cu[-1], 3, 16, 20)
    scale = 0.31
    out, lse = oracle.causal_attention_fwd(q, k, v, cu, scale, row_block=7)
    for a, b in zip(cu, cu[1:]):
        qs, ks, vs = (x[a:b].transpose(0, 1) for x in (q, k, v))      # [H, n, d]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, is_causal=True,
                                                               scale=scale)
        np.testing.assert_allclose(out[a:b], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        n = b - a
        scores = scale * qs @ ks.transpose(1, 2)
        scores = scores.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(lse[:, a:b], torch.logsumexp(scores, dim=-1).numpy(),
                                   rtol=0, atol=1e-12)


CASES = [
    # (P, prefix, texts)
    (1, 0, [16]),
    (2, 0, [32]),
    (2, 4, [8, 16]),
    (3, 0, [36]),
    (3, 5, [12, 0, 24]),
    (4, 6, [16, 32]),
    (8, 0, [64]),
    (8, 3, [32, 16]),
]


@pytest.mark.parametrize("P,prefix,texts", CASES)
def test_partition_invariant_fwd(P, prefix, texts):
    """zigzag split -> per-rank ring steps -> LSE merge -> inverse == plain."""
    cu = _cu(prefix, texts)
    q, k, v = _qkv(cu[-1], 2, 8, 30 + P)
    o1, l1 = oracle.causal_attention_fwd(q, k, v, cu, 0.5)
    o2, l2 = oracle.cp_ring_fwd(q, k, v, cu, prefix, P, 0.5)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


def test_split_prefix_changes_the_result():
    """The failure mode of CP-VLM page §3: if a rank's text queries do not see
    the whole image prefix (here: the replicated prefix is left out of ring
    step 0), the merged result is no longer plain causal attention."""
    cu = _cu(4, [16])
    q, k, v = _qkv(cu[-1], 1, 4, 40)
    o_ref, _ = oracle.causal_attention_fwd(q, k, v, cu, 1.0)
    local = oracle.rank_local_rows(cu, 4, 2)
    sid, pos = oa._positions(cu)
    # rank 0's queries with only text KV at every step (no replicated prefix)
    qr = local[0]
    parts = []
    for s in range(2):
        kv = local[(0 - s) % 2]
        parts.append(oa._masked_partial(oa._f64(q)[qr], oa._f64(k)[kv], oa._f64(v)[kv],
                                        oa._visible(sid, pos, qr, kv), 1.0))
    o_bad, _ = oracle.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    assert np.abs(o_bad - o_ref[qr]).max() > 1e-3


# ---------------------------------------------------------------------------
# balance: closed-form pair counts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,P,N", [(256, 2, 0), (64, 4, 0), (96, 3, 0), (128, 8, 0),
                                   (64, 2, 5), (48, 3, 7)])
def test_pair_counts_closed_form(L, P, N):
    cu = _cu(N, [L])
    counts, self_pairs = oracle.cp_pair_counts(cu, N, P)
    c = L // (2 * P)
    for r in range(P):
        assert counts[r, 0] == c * c + c * (c + 1) + 2 * c * N
        for s in range(1, P):
            assert counts[r, s] == 2 * c * c
        assert counts[r].sum() == (2 * P - 1) * c * c + c * (c + 1) + 2 * c * N
    if P == 2 and N == 0:
        assert counts[0].sum() == 3 * c * c + c * (c + 1)
    assert self_pairs == N * (N + 1) // 2
    assert counts.sum() + self_pairs == (N + L) * (N + L + 1) // 2


# ---------------------------------------------------------------------------
# LSE merge
# ---------------------------------------------------------------------------
def test_merge_special_cases():
    H, n, d = 2, 3, 4
    o = np.arange(n * H * d, dtype=np.float64).reshape(n, H, d)
    l = np.array([[0.5, -1.0, 2.0], [1.0, 0.0, -3.0]])
    ninf = np.full((H, n), -np.inf)
    z = np.zeros((n, H, d))
    mo, ml = oracle.lse_merge([z, o], [ninf, l])          # -inf (+) x = x
    np.testing.assert_allclose(mo, o)
    np.testing.assert_allclose(ml, l)
    mo, ml = oracle.lse_merge([o, z], [l, ninf])
    np.testing.assert_allclose(mo, o)
    mo, ml = oracle.lse_merge([z, z], [ninf, ninf])       # empty (+) empty
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    mo, ml = oracle.lse_merge([o, o], [l, l])             # x (+) x: same o, lse + log 2
    np.testing.assert_allclose(mo, o, atol=1e-12)
    np.testing.assert_allclose(ml, l + math.log(2.0), atol=1e-15)


def test_merge_of_single_key_partials_closed_form():
    # two partials that each saw one key: o = v_j, lse = s_j
    s1, s2 = 0.3, -1.7
    v1, v2 = np.array([1.0, -2.0]), np.array([0.5, 4.0])
    mo, ml = oracle.lse_merge([v1.reshape(1, 1, 2), v2.reshape(1, 1, 2)],
                              [np.array([[s1]]), np.array([[s2]])])
    w1, w2 = math.exp(s1), math.exp(s2)
    np.testing.assert_allclose(mo[0, 0], (w1 * v1 + w2 * v2) / (w1 + w2), atol=1e-15)
    assert abs(ml[0, 0] - math.log(w1 + w2)) < 1e-15


# ---------------------------------------------------------------------------
# backward: autograd, finite differences, partition and prefix invariants
# ---------------------------------------------------------------------------
def _autograd_grads(q, k, v, do, cu, scale):
    qs, ks, vs = (x.clone().requires_grad_(True) for x in (q, k, v))
    for a, b in zip(cu, cu[1:]):
        o = torch.nn.functional.scaled_dot_product_attention(
            qs[a:b].transpose(0, 1), ks[a:b].transpose(0, 1), vs[a:b].transpose(0, 1),
            is_causal=True, scale=scale)
        (o.transpose(0, 1) * do[a:b]).sum().backward()
    return qs.grad.numpy(), ks.grad.numpy(), vs.grad.numpy()


@pytest.mark.parametrize("texts,prefix", [([48], 0), ([16, 32, 8], 6)])
def test_bwd_matches_torch_autograd(texts, prefix):
    cu = _cu(prefix, texts)
    q, k, v = _qkv(cu[-1], 2, 8, 50)
    do = _rand((cu[-1], 2, 8), 53)
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, 0.4, row_block=5)
    rq, rk, rv = _autograd_grads(q, k, v, do, cu, 0.4)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_bwd_central_finite_differences():
    cu = _cu(2, [4, 6])
    q, k, v = _qkv(cu[-1], 1, 3, 60)
    do = _rand((cu[-1], 1, 3), 63)
    scale = 0.8
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.causal_attention_fwd(qq, kk, vv, cu, scale)
        return float((o * do.numpy()).sum())

    eps = 1e-6
    base = [q.numpy().copy(), k.numpy().copy(), v.numpy().copy()]
    for which, grad in enumerate((dq, dk, dv)):
        for idx in [(0, 0, 0), (3, 0, 2), (7, 0, 1), (11, 0, 0)]:
            plus = [b.copy() for b in base]
            minus = [b.copy() for b in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7, (which, idx, fd, grad[idx])


@pytest.mark.parametrize("P,prefix,texts", [(1, 3, [8]), (2, 4, [8, 16]), (3, 5, [12, 0, 24]),
                                            (4, 2, [32]), (8, 0, [32])])
def test_partition_invariant_bwd(P, prefix, texts):
    cu = _cu(prefix, texts)
    q, k, v = _qkv(cu[-1], 2, 4, 70 + P)
    do = _rand((cu[-1], 2, 4), 75 + P)
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, 0.6)
    cq, ck, cv, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, prefix, P, 0.6)
    for a, b in ((cq, dq), (ck, dk), (cv, dv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("P", [2, 3, 4])
def test_per_rank_prefix_gradients_sum_to_plain_and_match_masked_autograd(P):
    """CP-VLM page §4.2: each rank holds its own image-prefix gradient and the
    sum equals the full one.  Each per-rank term is pinned on its own: it is
    the prefix gradient of plain attention with dO zeroed outside that rank's
    text rows (autograd of torch SDPA)."""
    prefix, texts = 5, [4 * P, 8 * P]
    cu = _cu(prefix, texts)
    q, k, v = _qkv(cu[-1], 2, 4, 80 + P)
    do = _rand((cu[-1], 2, 4), 85 + P)
    _, dk, dv, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, prefix, P, 0.5)
    pre = oa._prefix_rows(cu, prefix)
    rk, rv = _autograd_grads(q, k, v, do, cu, 0.5)[1:]
    np.testing.assert_allclose(pdk.sum(0), rk[pre], rtol=0, atol=1e-12)
    np.testing.assert_allclose(pdv.sum(0), rv[pre], rtol=0, atol=1e-12)
    local = oracle.rank_local_rows(cu, prefix, P)
    for r in range(P + 1):
        rows = local[r] if r < P else pre
        dmask = torch.zeros_like(do)
        dmask[torch.as_tensor(rows)] = do[torch.as_tensor(rows)]
        mk, mv = _autograd_grads(q, k, v, dmask, cu, 0.5)[1:]
        np.testing.assert_allclose(pdk[r], mk[pre], rtol=0, atol=1e-12)
        np.testing.assert_allclose(pdv[r], mv[pre], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# sampled-row / sampled-key variants used for very long workloads
# ---------------------------------------------------------------------------
def test_sampled_rows_and_keys_match_autograd():
    cu = _cu(3, [40, 24])
    q, k, v = _qkv(cu[-1], 3, 8, 90)
    do = _rand((cu[-1], 3, 8), 93)
    out = torch.zeros_like(q)
    for a, b in zip(cu, cu[1:]):
        out[a:b] = torch.nn.functional.scaled_dot_product_attention(
            q[a:b].transpose(0, 1), k[a:b].transpose(0, 1), v[a:b].transpose(0, 1),
            is_causal=True, scale=0.45).transpose(0, 1)
    rq, rk, rv = _autograd_grads(q, k, v, do, cu, 0.45)
    rows = np.array([0, 2, 5, 30, 42, 43, 69])
    heads = [0, 2]
    o, l, dq = oracle.causal_attention_fwd_rows(q, k, v, cu, 0.45, rows, heads=heads, dout=do,
                                                row_block=3)
    np.testing.assert_allclose(o, out.numpy()[rows][:, heads], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, rq[rows][:, heads], rtol=0, atol=1e-12)
    keys = np.array([1, 4, 20, 40, 50, 60, 69])
    dk, dv = oracle.causal_attention_bwd_keys(q, k, v, do, cu, 0.45, keys, heads=heads,
                                              row_block=4)
    np.testing.assert_allclose(dk, rk[keys][:, heads], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, rv[keys][:, heads], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# grouped KV heads (GQA / MQA): query head h reads KV head h // (H / H_kv)
# ---------------------------------------------------------------------------
def _gqa_inputs(T, H, H_kv, d, seed):
    return _rand((T, H, d), seed), _rand((T, H_kv, d), seed + 1), _rand((T, H_kv, d), seed + 2)


def _sdpa_gqa(q, k, v, do, cu, scale):
    """torch SDPA with its own grouped-query option (fp64), per sample, and its
    autograd gradients: an implementation of GQA independent of the oracle."""
    qs, ks, vs = (x.clone().requires_grad_(True) for x in (q, k, v))
    outs = []
    for a, b in zip(cu, cu[1:]):
        o = torch.nn.functional.scaled_dot_product_attention(
            qs[a:b].transpose(0, 1), ks[a:b].transpose(0, 1), vs[a:b].transpose(0, 1),
            is_causal=True, scale=scale, enable_gqa=True)
        outs.append(o.transpose(0, 1))
        (o.transpose(0, 1) * do[a:b]).sum().backward()
    out = torch.cat(outs).detach().numpy()
    return out, qs.grad.numpy(), ks.grad.numpy(), vs.grad.numpy()


@pytest.mark.parametrize("H,H_kv", [(4, 2), (6, 3), (4, 1), (3, 3)])
def test_gqa_matches_torch_sdpa_enable_gqa(H, H_kv):
    cu = _cu(3, [10, 6])
    q, k, v = _gqa_inputs(cu[-1], H, H_kv, 8, 90 + H)
    do = _rand((cu[-1], H, 8), 95 + H)
    out, _ = oracle.causal_attention_fwd(q, k, v, cu, 0.45, row_block=4)
    dq, dk, dv = oracle.causal_attention_bwd(q, k, v, do, cu, 0.45, row_block=4)
    ro, rq, rk, rv = _sdpa_gqa(q, k, v, do, cu, 0.45)
    assert dk.shape == (cu[-1], H_kv, 8) and dv.shape == (cu[-1], H_kv, 8)
    for a, b in ((out, ro), (dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_gqa_fwd_matches_scalar_brute_force():
    """Scalar loops that pick the KV head of query head h as h // G by hand."""
    cu = _cu(1, [5])
    H, H_kv, d = 4, 2, 3
    q, k, v = _gqa_inputs(cu[-1], H, H_kv, d, 100)
    out, lse = oracle.causal_attention_fwd(q, k, v, cu, 0.9)
    for h in range(H):
        hk = h // (H // H_kv)
        bo, bl = _brute_force_fwd(q[:, h:h + 1].numpy(), k[:, hk:hk + 1].numpy(),
                                  v[:, hk:hk + 1].numpy(), cu, 0.9)
        np.testing.assert_allclose(out[:, h:h + 1], bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[h:h + 1], bl, rtol=0, atol=1e-12)


def test_gqa_rejects_indivisible_heads():
    cu = _cu(0, [8])
    q, k, v = _gqa_inputs(8, 3, 2, 4, 110)
    with pytest.raises(ValueError):
        oracle.causal_attention_fwd(q, k, v, cu, 0.5)


@pytest.mark.parametrize("P,prefix,texts,H,H_kv", [(2, 4, [8, 16], 4, 2), (3, 5, [12, 0, 24], 6, 2),
                                                   (4, 2, [32], 4, 1)])
def test_gqa_partition_invariant_and_prefix_sum(P, prefix, texts, H, H_kv):
    cu = _cu(prefix, texts)
    q, k, v = _gqa_inputs(cu[-1], H, H_kv, 4, 120 + P)
    do = _rand((cu[-1], H, 4), 125 + P)
    o1, l1 = oracle.causal_attention_fwd(q, k, v, cu, 0.6)
    o2, l2 = oracle.cp_ring_fwd(q, k, v, cu, prefix, P, 0.6)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    _, rq, rk, rv = _sdpa_gqa(q, k, v, do, cu, 0.6)
    cq, ck, cv, pdk, pdv = oracle.cp_ring_bwd(q, k, v, do, cu, prefix, P, 0.6)
    for a, b in ((cq, rq), (ck, rk), (cv, rv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)
    pre = oa._prefix_rows(cu, prefix)
    assert pdk.shape == (P + 1, len(pre), H_kv, 4)
    np.testing.assert_allclose(pdk.sum(0), rk[pre], rtol=0, atol=1e-11)
    np.testing.assert_allclose(pdv.sum(0), rv[pre], rtol=0, atol=1e-11)
