"""Ring load balance of the zigzag split against a naive contiguous split
(the multimodal CP page, §1 and §1.1): exact pair counts, pinned to the
oracle's brute-force counts, to brute force over positions and to closed
forms."""
import numpy as np
import pytest

import oracle
from vlm_zigzag_head_gb300 import balance


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


@pytest.mark.parametrize("P,N,texts", [(1, 0, [8]), (2, 0, [16]), (2, 3, [8, 16]),
                                       (3, 5, [12, 24, 6]), (4, 2, [16, 32])])
def test_zigzag_counts_equal_oracle_brute_force(P, N, texts):
    cu = _cu(N, texts)
    got, pre = balance.rank_step_pairs(cu, N, P, "zigzag")
    want, want_pre = oracle.cp_pair_counts(cu, N, P)
    assert np.array_equal(got, want)
    assert pre == want_pre


def _brute_contiguous(cu, N, P):
    counts = np.zeros((P, P), dtype=np.int64)
    for i in range(len(cu) - 1):
        L = cu[i + 1] - cu[i] - N
        c = L // P
        owner = np.arange(L) // c                 # rank holding text position t
        for r in range(P):
            for s in range(P):
                j = (r - s) % P
                for t in np.nonzero(owner == r)[0]:
                    keys = np.nonzero(owner == j)[0]
                    counts[r, s] += int((keys <= t).sum())
                    if s == 0:
                        counts[r, s] += N         # the whole prefix
    return counts


@pytest.mark.parametrize("P,N,texts", [(2, 0, [8]), (3, 4, [9, 6]), (4, 1, [8, 16])])
def test_contiguous_counts_equal_brute_force(P, N, texts):
    cu = _cu(N, texts)
    got, pre = balance.rank_step_pairs(cu, N, P, "contiguous")
    assert np.array_equal(got, _brute_contiguous(cu, N, P))
    assert pre == len(texts) * N * (N + 1) // 2


@pytest.mark.parametrize("split", balance.SPLITS)
@pytest.mark.parametrize("P,N,texts", [(2, 7, [40, 24]), (8, 0, [256]), (4, 16, [64, 128])])
def test_pairs_sum_to_causal_total(split, P, N, texts):
    cu = _cu(N, texts)
    counts, pre = balance.rank_step_pairs(cu, N, P, split)
    assert int(counts.sum()) + pre == sum((N + L) * (N + L + 1) // 2 for L in texts)


def test_closed_forms_and_imbalance():
    P, L = 8, 1 << 14
    c = L // (2 * P)
    z, _ = balance.rank_step_pairs([0, L], 0, P, "zigzag")
    assert np.all(z.sum(axis=1) == (2 * P - 1) * c * c + c * (c + 1))
    cc = L // P
    n, _ = balance.rank_step_pairs([0, L], 0, P, "contiguous")
    for r in range(P):
        assert n[r].sum() == r * cc * cc + cc * (cc + 1) // 2
    sz = balance.ring_summary([0, L], 0, P, "zigzag")
    sn = balance.ring_summary([0, L], 0, P, "contiguous")
    assert sz["imbalance"] == pytest.approx(1.0, abs=1e-3)
    assert sn["imbalance"] == pytest.approx(2.0 - 1.0 / P, rel=1e-3)
    assert sn["ring_pairs"] > 1.8 * sz["ring_pairs"]


def test_rejects_bad_lengths():
    with pytest.raises(ValueError):
        balance.rank_step_pairs([0, 30], 0, 4, "zigzag")
    with pytest.raises(ValueError):
        balance.rank_step_pairs([0, 30], 0, 4, "contiguous")
    with pytest.raises(ValueError):
        balance.rank_step_pairs([0, 32], 0, 4, "striped")
