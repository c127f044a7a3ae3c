"""Seeded synthetic inputs for context-parallel causal attention.

This module only draws random tensors and lays out sample boundaries; it
contains none of the attention arithmetic.  Both the CUDA path (through the
tests and ``bench.py``) and the CPU oracle consume what it returns, so the two
always see the same bits.

Workloads follow the shapes the multimodal context-parallel page describes
(8K-128K contexts, a replicated image-token prefix, packed samples): there is
no public dataset behind them, the values are i.i.d. normal draws.

Recipe (every tensor is drawn in fp32 on the CPU with ``torch.Generator``):

* q, k, v ~ N(0, 1), shape ``[T, H, d]`` (THD, natural token order), drawn in
  that order from one generator seeded with ``seed``; then cast to the
  workload dtype (bf16 rounds to nearest even).
* the "Text LLM" workload multiplies q by 1/sqrt(128) before the cast and uses
  softmax scale 1.0 (the scaling *is* the softmax scale); every other
  workload uses unscaled q and scale 1/sqrt(d).
* dO ~ N(0, 1) from a generator seeded with ``seed + 100``.
* packed text lengths ~ U{1024..6144} from a generator seeded with ``seed``
  (drawn before q/k/v), each rounded up to a multiple of 2*P*64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_seqs: int
    prefix_len: int          # N: image tokens at the head of every sample
    text_lens: tuple         # L_i per sample (() = drawn, see packed_range)
    P: int                   # simulated context-parallel degree
    H: int
    d: int
    dtype: str               # "f32" or "bf16"
    seed: int
    backward: bool
    q_prescaled: bool = False
    packed_range: Optional[tuple] = None   # (lo, hi) inclusive for drawn text lengths
    round_to: int = 0                      # round drawn lengths up to this multiple
    H_kv: int = 0                          # KV heads (grouped-query attention); 0: H

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H


WORKLOADS = {
    "tiny": Workload("tiny", 1, 0, (256,), 2, 1, 64, "f32", 0, False),
    "text_llm": Workload("text_llm", 1, 0, (8192,), 2, 16, 128, "bf16", 1, True,
                         q_prescaled=True),
    "vlm_prefix": Workload("vlm_prefix", 2, 2304, (16384, 16384), 4, 32, 128, "bf16", 2, True),
    "packed_vlm": Workload("packed_vlm", 8, 576, (), 4, 32, 128, "bf16", 3, True,
                           packed_range=(1024, 6144), round_to=2 * 4 * 64),
    "long": Workload("long", 1, 0, (131072,), 8, 32, 128, "bf16", 4, True),
}


def get(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields overridden (smaller test cases)."""
    w = WORKLOADS[name]
    if overrides:
        w = replace(w, **overrides)
    return w


def text_lengths(w: Workload) -> List[int]:
    if w.packed_range is None:
        assert len(w.text_lens) == w.n_seqs
        return [int(x) for x in w.text_lens]
    g = torch.Generator().manual_seed(w.seed)
    lo, hi = w.packed_range
    raw = torch.randint(lo, hi + 1, (w.n_seqs,), generator=g).tolist()
    m = w.round_to
    return [int(-(-x // m) * m) for x in raw]


def cu_seqlens(w: Workload) -> List[int]:
    cu = [0]
    for L in text_lengths(w):
        cu.append(cu[-1] + w.prefix_len + L)
    return cu


def softmax_scale(w: Workload) -> float:
    return 1.0 if w.q_prescaled else 1.0 / math.sqrt(w.d)


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


@dataclass
class Inputs:
    workload: Workload
    cu_seqlens: List[int]
    scale: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.cu_seqlens[-1]


def make_inputs(w: Workload, with_dout: Optional[bool] = None) -> Inputs:
    """Draw the CPU tensors of one workload (fp32 draw, then dtype cast)."""
    cu = cu_seqlens(w)
    T = cu[-1]
    g = torch.Generator().manual_seed(w.seed)
    if w.packed_range is not None:
        # the length draw consumes the generator first (same seed, same order)
        lo, hi = w.packed_range
        torch.randint(lo, hi + 1, (w.n_seqs,), generator=g)
    shape = (T, w.H, w.d)
    kv_shape = (T, w.kv_heads, w.d)
    dt = torch_dtype(w)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    if w.q_prescaled:
        q = q * (1.0 / math.sqrt(128.0))
    q, k, v = q.to(dt), k.to(dt), v.to(dt)
    dout = None
    if w.backward if with_dout is None else with_dout:
        g2 = torch.Generator().manual_seed(w.seed + 100)
        dout = torch.randn(shape, generator=g2, dtype=torch.float32).to(dt)
    return Inputs(w, cu, softmax_scale(w), q, k, v, dout)


def sample_rows(T: int, count: int, seed: int) -> torch.Tensor:
    """Seeded subset of natural-order query rows (sorted), for sampled checks."""
    g = torch.Generator().manual_seed(seed)
    count = min(count, T)
    return torch.sort(torch.randperm(T, generator=g)[:count]).values

