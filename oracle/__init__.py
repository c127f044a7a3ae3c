"""Plain fp64 CPU oracle for zigzag context-parallel causal attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code, table
or helper with the CUDA library.

Source pages (cited by short name in every docstring):

* "CP-VLM page" -- *context-parallel-multimodal* (xuesongtap.github.io,
  2026-03-22): §1 (CP shards the sequence, Ring Attention across ranks),
  §1.1 (2P chunks, head-tail pairing, ``index_select``), §2 (``[image tokens,
  text tokens]`` layout), §4.1 (replicated image prefix, forward), §4.2
  (per-rank prefix gradients summed by AllReduce), §5.3 (packed samples with
  ``cu_seqlens``).
* "Parallelism page" -- *Parallelism* (lizn-zn.github.io), §6 (CP: attention
  cost grows with the square of the length; KV is exchanged around a ring).

Grouped KV heads (GQA / MQA) are not on the pages: where ``k``/``v`` hold
``H_kv < H`` heads, query head ``h`` reads KV head ``h // (H / H_kv)``, the
layout models with fewer KV heads use, and KV-side gradients are summed over
each KV head's query heads.

Every function is either the plain definition of the result (unpartitioned
causal softmax attention per sample and its gradient) or a literal, step by
step restatement of the partitioned method in the pages' order.  Pins that
tie it to something other than itself live in ``tests/test_oracle_*.py``.
"""
from .attention import (  # noqa: F401
    zigzag_chunk_ids,
    zigzag_index,
    rank_local_rows,
    causal_attention_fwd,
    causal_attention_bwd,
    causal_attention_fwd_rows,
    causal_attention_bwd_keys,
    lse_merge,
    cp_ring_fwd,
    cp_ring_bwd,
    cp_pair_counts,
    kv_group,
)
