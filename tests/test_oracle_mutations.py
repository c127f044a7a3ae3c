"""The pins bite: plant a plausible mistake in the oracle (on the CPU, by
monkeypatching one of its functions) and check that a pin catches it."""
import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

from test_oracle_pins import _autograd_grads, _cu, _qkv, _rand, _read_golden_example


def _check_worked_example():
    P, ranks = _read_golden_example()
    assert oracle.zigzag_chunk_ids(P) == [ranks[0], ranks[1]]
    fwd, _ = oracle.zigzag_index([0, 12], 0, 2)
    for r, chunks in ranks.items():
        assert fwd[r * 6:(r + 1) * 6].tolist() == [t for ch in chunks
                                                   for t in range(ch * 3, ch * 3 + 3)]


def _check_sdpa():
    cu = _cu(2, [12])
    q, k, v = _qkv(cu[-1], 1, 4, 5)
    out, _ = oa.causal_attention_fwd(q, k, v, cu, 0.5)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), is_causal=True, scale=0.5)
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), atol=1e-12)


def _check_partition():
    cu = _cu(3, [16])
    q, k, v = _qkv(cu[-1], 1, 4, 6)
    o1, l1 = oa.causal_attention_fwd(q, k, v, cu, 0.5)
    o2, l2 = oa.cp_ring_fwd(q, k, v, cu, 3, 2, 0.5)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)


def _check_bwd():
    cu = _cu(0, [16])
    q, k, v = _qkv(16, 1, 4, 7)
    do = _rand((16, 1, 4), 8)
    got = oa.causal_attention_bwd(q, k, v, do, cu, 0.5)
    ref = _autograd_grads(q, k, v, do, cu, 0.5)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, atol=1e-11)


def test_unmutated_checks_pass():
    _check_worked_example()
    _check_sdpa()
    _check_partition()
    _check_bwd()


def test_swapped_head_tail_pair_is_caught(monkeypatch):
    monkeypatch.setattr(oa, "zigzag_chunk_ids", lambda P: [(2 * P - 1 - r, r) for r in range(P)])
    monkeypatch.setattr(oracle, "zigzag_chunk_ids", oa.zigzag_chunk_ids)
    with pytest.raises(AssertionError):
        _check_worked_example()


def test_off_by_one_mask_is_caught(monkeypatch):
    real = oa._causal_rows

    def leaky(qb, kb, vb, q_pos0, scale):      # a query also sees the next key
        return real(qb, kb, vb, q_pos0 + 1, scale) if kb.shape[0] > q_pos0 + len(qb) else \
            real(qb, np.vstack([kb, kb[-1:]]), np.vstack([vb, vb[-1:]]), q_pos0 + 1, scale)
    monkeypatch.setattr(oa, "_causal_rows", leaky)
    with pytest.raises(AssertionError):
        _check_sdpa()


def test_swapped_merge_weights_are_caught(monkeypatch):
    real = oa._merge2
    monkeypatch.setattr(oa, "_merge2", lambda oa_, la, ob, lb: real(oa_, lb, ob, la))
    with pytest.raises(AssertionError):
        _check_partition()


def test_dropped_scale_in_dk_is_caught(monkeypatch):
    real = oa.causal_attention_bwd

    def no_scale(q, k, v, do, cu, scale, row_block=1024):
        dq, dk, dv = real(q, k, v, do, cu, scale, row_block)
        return dq, dk / scale, dv
    monkeypatch.setattr(oa, "causal_attention_bwd", no_scale)
    with pytest.raises(AssertionError):
        _check_bwd()


def _check_gqa():
    from test_oracle_pins import _gqa_inputs, _sdpa_gqa
    cu = _cu(2, [10])
    q, k, v = _gqa_inputs(cu[-1], 4, 2, 4, 9)
    do = _rand((cu[-1], 4, 4), 10)
    out, _ = oa.causal_attention_fwd(q, k, v, cu, 0.5)
    dk = oa.causal_attention_bwd(q, k, v, do, cu, 0.5)[1]
    ro, _, rk, _ = _sdpa_gqa(q, k, v, do, cu, 0.5)
    np.testing.assert_allclose(out, ro, atol=1e-11)
    np.testing.assert_allclose(dk, rk, atol=1e-11)


def test_unmutated_gqa_check_passes():
    _check_gqa()


def test_interleaved_kv_grouping_is_caught(monkeypatch):
    # query head h reading KV head h % H_kv instead of h // G
    monkeypatch.setattr(oa, "_expand_kv", lambda x, H: np.tile(x, (1, oa.kv_group(H, x.shape[1]), 1)))
    with pytest.raises(AssertionError):
        _check_gqa()
