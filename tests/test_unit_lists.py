"""Host planner of the all-steps forward (CPU, no GPU needed).

The default tensor-core forward runs every ring step in one persistent
launch.  An item is a 256-query tile with the key runs of all P ring steps
(CP-VLM page §1 ring order, §1.1 zigzag chunks, §4.1 replicated prefix).
Its cost in KV tiles must equal what the tile's queries see under the global
causal mask, counted here from the mask itself.  The units (item, head) are
dealt to the persistent CTAs head by head, each to the least-loaded CTA.
This is list scheduling, so every CTA ends within one unit of the mean, and
the lists must be a permutation of all units.
"""
import numpy as np
import pytest

import oracle
from vlm_zigzag_head_gb300 import cp_plan_unit_lists, workloads

UNIT_COST = 2   # fixed cost per unit, in KV tiles, used by the planner
TILE_Q, TILE_K = 256, 128


def _cu(prefix, texts):
    cu = [0]
    for L in texts:
        cu.append(cu[-1] + prefix + L)
    return cu


def _expected_tiles(cu, N, P):
    """KV tiles of every 256-query tile, from the causal mask and the zigzag
    split: a text tile of rank r's chunk cq meets, per key chunk, the tiles
    that hold at least one key visible to one of its rows; prefix tiles meet
    their prefix causally."""
    out = []
    for i in range(len(cu) - 1):
        L = cu[i + 1] - cu[i] - N
        c = L // (2 * P)
        # prefix queries: causal over the prefix
        for t0 in range(0, N, TILE_Q):
            q_len = min(TILE_Q, N - t0)
            out.append(-(-(t0 + q_len) // TILE_K))
        if c == 0:
            continue
        ids = oracle.zigzag_chunk_ids(P)
        for r in range(P):
            for cq in ids[r]:
                for t0 in range(0, c, TILE_Q):
                    q_len = min(TILE_Q, c - t0)
                    n = -(-N // TILE_K) if N else 0     # the whole prefix
                    for ck in range(cq):                 # earlier chunks: all keys
                        n += -(-c // TILE_K)
                    n += -(-min(c, t0 + q_len) // TILE_K)  # own chunk: causal
                    out.append(n)
    return sorted(out, reverse=True)


CASES = [
    # (prefix, texts, P, H, grid)
    (0, [8192], 2, 16, 152),
    (2304, [16384, 16384], 4, 32, 152),
    (0, [131072], 8, 32, 152),
    (37, [384, 0, 1152], 3, 6, 7),
    (576, [1536, 512], 4, 2, 5),
    (300, [0], 2, 3, 4),
]


@pytest.mark.parametrize("N,texts,P,H,grid", CASES)
def test_items_cover_the_causal_mask(N, texts, P, H, grid):
    cu = _cu(N, texts)
    tiles, _, _ = cp_plan_unit_lists(cu, N, P, H, grid)
    assert sorted(tiles.tolist(), reverse=True) == _expected_tiles(cu, N, P)


@pytest.mark.parametrize("N,texts,P,H,grid", CASES)
def test_unit_lists_are_a_balanced_permutation(N, texts, P, H, grid):
    cu = _cu(N, texts)
    tiles, units, off = cp_plan_unit_lists(cu, N, P, H, grid)
    n = len(tiles)
    assert off[0] == 0 and off[-1] == n * H and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.sort(units), np.arange(n * H))
    cost = tiles[units % n].astype(np.int64) + UNIT_COST
    load = np.array([cost[off[b]:off[b + 1]].sum() for b in range(grid)])
    # list scheduling: the CTA that ends last was the least loaded when it
    # took its last unit, so it ends at most one unit above the mean
    assert load.max() <= load.sum() / grid + cost.max() + 1e-9
    for b in range(grid):                      # each CTA goes head by head
        heads = units[off[b]:off[b + 1]] // n
        assert np.all(np.diff(heads) >= 0)


def test_round_robin_would_be_unbalanced_on_the_vlm_workload():
    """The stride effect the lists remove: 146 items over 152 CTAs."""
    w = workloads.get("vlm_prefix")
    cu = workloads.cu_seqlens(w)
    tiles, units, off = cp_plan_unit_lists(cu, w.prefix_len, w.P, w.H, 152)
    n = len(tiles)
    rr = np.zeros(152)
    for u in range(n * w.H):
        rr[u % 152] += tiles[u % n] + UNIT_COST
    cost = tiles[units % n] + UNIT_COST
    lists = np.array([cost[off[b]:off[b + 1]].sum() for b in range(152)])
    assert rr.max() / rr.mean() > 1.1
    assert lists.max() / lists.mean() < 1.03


def test_bad_arguments_rejected():
    from vlm_zigzag_head_gb300 import CpError
    with pytest.raises(CpError):
        cp_plan_unit_lists([0, 100], 0, 2, 0, 4)      # H < 1
    with pytest.raises(CpError):
        cp_plan_unit_lists([0, 100], 0, 2, 4, 0)      # grid < 1
    with pytest.raises(CpError):
        cp_plan_unit_lists([0, 102], 0, 4, 4, 4)      # text not divisible by 2P
