"""Seeded synthetic workloads for masked attention.

This module only draws inputs: shapes, random tensors, document lengths and
prefix lengths. It holds none of the attention arithmetic, so both the CPU
oracle (``oracle/``) and the CUDA path can be fed from it without sharing any
of the computation.

Recipe (the same for every workload, seed = the workload number by default):

1. ``rng = numpy.random.default_rng(seed)`` draws the mask parameters first:
   document lengths (uniform integers in ``[doc_lo, doc_hi]``, drawn until
   their sum reaches ``S``; the last one is truncated so the lengths sum to
   exactly ``S`` and may be shorter than ``doc_lo``), one list per batch
   element in batch order; then one prefix length per batch element, uniform
   in ``[prefix_lo, prefix_hi]``.
2. ``g = torch.Generator().manual_seed(seed)`` then draws Q, K, V (and dO for
   the training step) in that order with ``torch.randn(..., dtype=float32)``
   on the CPU. bf16 workloads round them to bf16 (round to nearest even).

Layouts are contiguous ``[B, H, S, D]`` (D innermost). ``doc_id`` is int32
``[B, max(Sq, Skv)]`` indexed by absolute position; ``prefix_len`` is int32
``[B]``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# The five workloads. Each names the mask and score modifications it uses; the
# meaning of those names lives in the oracle and in the kernels, not here.
WORKLOADS = {
    1: dict(name="tiny fp32 causal", dtype="f32", B=1, Hq=2, Hkv=2, S=128, D=64,
            causal=True),
    2: dict(name="bf16 causal + ALiBi", dtype="bf16", B=4, Hq=16, Hkv=16, S=2048, D=64,
            causal=True, alibi=True),
    3: dict(name="bf16 document + sliding window 1024 + causal", dtype="bf16", B=1, Hq=16,
            Hkv=16, S=16384, D=128, causal=True, window=1024, document=True,
            doc_lo=256, doc_hi=4096),
    4: dict(name="bf16 GQA PrefixLM + softcap 50", dtype="bf16", B=2, Hq=32, Hkv=8,
            S=8192, D=128, causal=True, prefix=True, softcap=50.0,
            prefix_lo=512, prefix_hi=4096),
    5: dict(name="bf16 causal forward + backward", dtype="bf16", B=8, Hq=16, Hkv=16,
            S=4096, D=128, causal=True, backward=True),
}


@dataclasses.dataclass
class Workload:
    """One seeded problem instance (all tensors on the CPU)."""
    name: str
    dtype: str                      # "bf16" or "f32": the type of Q, K, V, O
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    causal: bool = False
    window: Optional[int] = None
    document: bool = False
    prefix: bool = False
    alibi: bool = False
    softcap: Optional[float] = None
    backward: bool = False
    relbias: bool = False                    # relative-position bias table on
    seed: int = 0
    doc_lengths: Optional[list] = None       # per batch element
    doc_id: Optional[np.ndarray] = None      # int32 [B, max(Sq, Skv)]
    prefix_len: Optional[np.ndarray] = None  # int32 [B]
    q: Optional[torch.Tensor] = None
    k: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None
    do: Optional[torch.Tensor] = None
    rel_bias: Optional[torch.Tensor] = None  # fp32 [Hq, Sq + Skv - 1], entry i - j + Skv - 1

    def describe(self) -> dict:
        out = dict(name=self.name, dtype=self.dtype, B=self.B, Hq=self.Hq, Hkv=self.Hkv,
                   Sq=self.Sq, Skv=self.Skv, D=self.D, seed=self.seed)
        for key in ("causal", "document", "prefix", "alibi", "backward", "relbias"):
            if getattr(self, key):
                out[key] = True
        if self.window is not None:
            out["window"] = self.window
        if self.softcap is not None:
            out["softcap"] = self.softcap
        if self.doc_lengths is not None:
            out["doc_lengths"] = [list(map(int, d)) for d in self.doc_lengths]
        if self.prefix_len is not None:
            out["prefix_len"] = [int(p) for p in self.prefix_len]
        return out


def draw_doc_lengths(rng: np.random.Generator, S: int, lo: int, hi: int) -> list:
    """Uniform lengths in [lo, hi] until they cover S; the last is cut to fit."""
    lengths = []
    total = 0
    while total < S:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, S - total)
        lengths.append(n)
        total += n
    return lengths


def doc_ids_from_lengths(lengths: list, L: int) -> np.ndarray:
    """Document index of every position 0..L-1 (positions past the last
    document keep the last index)."""
    ids = np.empty(L, dtype=np.int32)
    pos = 0
    for d, n in enumerate(lengths):
        ids[pos:pos + n] = d
        pos += n
    if pos < L:
        ids[pos:] = len(lengths) - 1
    return ids


def make_workload(number: int = 0, *, seed: Optional[int] = None, with_tensors: bool = True,
                  **overrides) -> Workload:
    """Build workload ``number`` (1..5) or a custom one from ``overrides``.

    Any recipe field can be overridden (for example ``S=512`` for a reduced
    size parity case). ``Sq``/``Skv`` override ``S`` separately.
    """
    spec = dict(WORKLOADS.get(number, {}))
    spec.update(overrides)
    if seed is None:
        seed = number
    S = spec.get("S", 128)
    Sq = spec.get("Sq", S)
    Skv = spec.get("Skv", S)
    B, Hq, Hkv, D = spec["B"], spec["Hq"], spec.get("Hkv", spec["Hq"]), spec["D"]
    w = Workload(name=spec.get("name", "custom"), dtype=spec.get("dtype", "bf16"), B=B, Hq=Hq,
                 Hkv=Hkv, Sq=Sq, Skv=Skv, D=D, causal=spec.get("causal", False),
                 window=spec.get("window"), document=spec.get("document", False),
                 prefix=spec.get("prefix", False), alibi=spec.get("alibi", False),
                 softcap=spec.get("softcap"), backward=spec.get("backward", False),
                 relbias=spec.get("relbias", False), seed=seed)
    rng = np.random.default_rng(seed)
    L = max(Sq, Skv)
    if w.document:
        if "doc_lengths" in spec:
            lengths = [list(x) for x in spec["doc_lengths"]]
        else:
            lengths = [draw_doc_lengths(rng, L, spec.get("doc_lo", 256), spec.get("doc_hi", 4096))
                       for _ in range(B)]
        w.doc_lengths = lengths
        w.doc_id = np.stack([doc_ids_from_lengths(x, L) for x in lengths]).astype(np.int32)
    if w.prefix:
        if "prefix_len" in spec:
            w.prefix_len = np.asarray(spec["prefix_len"], dtype=np.int32)
        else:
            lo, hi = spec.get("prefix_lo", 512), spec.get("prefix_hi", 4096)
            w.prefix_len = np.array([int(rng.integers(lo, hi + 1)) for _ in range(B)],
                                    dtype=np.int32)
    if with_tensors:
        g = torch.Generator().manual_seed(seed)
        tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        w.q = torch.randn(B, Hq, Sq, D, dtype=torch.float32, generator=g).to(tdtype)
        w.k = torch.randn(B, Hkv, Skv, D, dtype=torch.float32, generator=g).to(tdtype)
        w.v = torch.randn(B, Hkv, Skv, D, dtype=torch.float32, generator=g).to(tdtype)
        if w.backward:
            w.do = torch.randn(B, Hq, Sq, D, dtype=torch.float32, generator=g).to(tdtype)
        if w.relbias:  # drawn last: the other tensors do not depend on it
            w.rel_bias = torch.randn(Hq, Sq + Skv - 1, dtype=torch.float32, generator=g)
    return w

