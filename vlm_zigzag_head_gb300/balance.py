"""Load balance of the ring under the zigzag split and under a naive
contiguous split.

The multimodal context-parallel page (§1, the motivation of the zigzag
split) notes that a causal mask makes later tokens costlier: with the text cut
into P contiguous pieces, the rank holding the tail does the most work and the
rank holding the head the least. Pairing chunk r with chunk 2P-1-r gives every
rank the same work (§1.1).

This module counts, exactly and without a GPU, the visible (query, key)
pairs each rank meets at each ring step under either split. In a real ring
every step waits for its slowest rank, so the time of step s is the maximum
over ranks. Scaled by a per-pair cost (taken from a measured throughput), this
gives a simulated ring time for each split.

Geometry (the same as the kernels'):

- rank r at step s meets the KV of rank (r - s) mod P;
- step 0 adds the replicated prefix, which every text query sees whole;
- the prefix queries' own pairs are counted once, at rank 0, step 0.
"""
from __future__ import annotations

import argparse
import json
from typing import List, Sequence, Tuple

import numpy as np

SPLITS = ("zigzag", "contiguous")


def _block_pairs(a0: int, a1: int, b0: int, b1: int) -> int:
    """Causal pairs between text queries [a0, a1) and text keys [b0, b1) of one
    sample: sum over q of the keys k in [b0, b1) with k <= q."""
    n = 0
    if a1 <= a0 or b1 <= b0:
        return 0
    # queries with q >= b1 - 1 see the whole key block
    full_from = max(a0, b1 - 1)
    if full_from < a1:
        n += (a1 - full_from) * (b1 - b0)
    # queries q in [max(a0, b0), min(a1, b1 - 1)) see keys b0..q
    lo, hi = max(a0, b0), min(a1, b1 - 1)
    if hi > lo:
        # sum_{q=lo}^{hi-1} (q - b0 + 1)
        first, last = lo - b0 + 1, hi - b0
        n += (first + last) * (hi - lo) // 2
    return n


def _rank_chunks(L: int, P: int, split: str) -> List[List[Tuple[int, int]]]:
    """Text intervals held by each rank for one sample of text length L."""
    if split == "zigzag":
        if L % (2 * P):
            raise ValueError("text length %d is not a multiple of 2P = %d" % (L, 2 * P))
        c = L // (2 * P)
        return [[(r * c, (r + 1) * c), ((2 * P - 1 - r) * c, (2 * P - r) * c)] for r in range(P)]
    if split == "contiguous":
        if L % P:
            raise ValueError("text length %d is not a multiple of P = %d" % (L, P))
        c = L // P
        return [[(r * c, (r + 1) * c)] for r in range(P)]
    raise ValueError("split must be one of %s" % (SPLITS,))


def rank_step_pairs(cu_seqlens: Sequence[int], prefix_len: int, P: int,
                    split: str = "zigzag") -> Tuple[np.ndarray, int]:
    """Visible pairs per head: ``(counts[P ranks][P steps], prefix_self)``.
    counts covers text queries; prefix_self is the prefix queries' own causal
    pairs (computed once, by rank 0 at step 0, not included in counts)."""
    N = int(prefix_len)
    counts = np.zeros((P, P), dtype=np.int64)
    prefix_self = 0
    for i in range(len(cu_seqlens) - 1):
        L = int(cu_seqlens[i + 1]) - int(cu_seqlens[i]) - N
        if L < 0:
            raise ValueError("sample %d is shorter than the prefix" % i)
        prefix_self += N * (N + 1) // 2
        if L == 0:
            continue
        chunks = _rank_chunks(L, P, split)
        for r in range(P):
            nq = sum(b - a for a, b in chunks[r])
            counts[r, 0] += nq * N          # the whole prefix, at step 0
            for s in range(P):
                j = (r - s) % P
                counts[r, s] += sum(_block_pairs(a0, a1, b0, b1)
                                    for a0, a1 in chunks[r] for b0, b1 in chunks[j])
    return counts, prefix_self


def ring_summary(cu_seqlens: Sequence[int], prefix_len: int, P: int, split: str,
                 seconds_per_pair: float = 0.0) -> dict:
    """Per-rank totals, per-step maxima and the simulated ring time: the sum
    over steps of the slowest rank's pairs (prefix self pairs go to rank 0,
    step 0), times ``seconds_per_pair`` per head."""
    counts, pre = rank_step_pairs(cu_seqlens, prefix_len, P, split)
    c = counts.copy()
    c[0, 0] += pre
    step_max = c.max(axis=0)
    total = int(c.sum())
    return {
        "split": split,
        "per_rank": [int(x) for x in c.sum(axis=1)],
        "step_max": [int(x) for x in step_max],
        "total_pairs": total,
        "ring_pairs": int(step_max.sum()),          # pairs-time of the ring (slowest rank per step)
        "ideal_pairs": total / P,                   # perfectly balanced ring
        "imbalance": float(step_max.sum() / (total / P)) if total else 1.0,
        "simulated_s": float(step_max.sum()) * seconds_per_pair,
    }


def main(argv=None) -> int:
    from . import workloads as W
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="long", choices=sorted(W.WORKLOADS))
    ap.add_argument("--tflops", type=float, default=0.0,
                    help="measured forward TFLOP/s to turn pairs into seconds (4*d*H flop per pair)")
    args = ap.parse_args(argv)
    w = W.get(args.workload)
    cu = W.cu_seqlens(w)
    spp = (4.0 * w.d * w.H / (args.tflops * 1e12)) if args.tflops > 0 else 0.0
    for split in SPLITS:
        print(json.dumps(dict(workload=w.name, P=w.P, **ring_summary(cu, w.prefix_len, w.P,
                                                                      split, spp))))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
