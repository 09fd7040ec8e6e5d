"""Seeded synthetic inputs for the fused attention forward.

This module only draws random numbers and lays out document boundaries. It
holds none of the attention arithmetic, so both the fp64 oracle (``oracle/``)
and the CUDA path (``attention_attn_fwd_04_gb300``) can take their inputs from
it without sharing any of the method's code.

Input recipe (the same for every workload):

* Q, K, V: one CPU ``torch.Generator`` seeded with ``seed`` (0 by default);
  Q, then K, then V are drawn as float32 standard normals in that order and
  rounded to bfloat16 (round to nearest even).  Both sides read these exact
  bf16 values.
* Document ids (packed-sequence workloads): a CPU generator seeded with
  ``doc_seed`` draws document lengths uniformly from the inclusive range
  [doc_min, doc_max] until the total reaches S; the last document is cut to
  fit.  ``doc_ids[j]`` is the 0-based index of the document holding token j.
* Row sample (large workloads): a CPU generator seeded with 2 picks
  ``n_rows`` flattened (b, h, i) indices uniformly without replacement, plus
  fixed edge rows.

The named workloads are the sizes the FlashAttention-4 / FlexAttention pages
discuss in prose (dense, causal, GQA, sliding window + soft-capping, document
packing + ALiBi); the pages publish no datasets, so synthetic inputs with
those shapes stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "get",
    "generate",
    "doc_ids_for",
    "sample_rows",
    "row_count",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and mods of one attention-forward problem.

    Layout is Q [B,H,S_q,D], K/V [B,H_kv,S_k,D] (bf16, contiguous), outputs
    O [B,H,S_q,D] bf16 and LSE [B,H,S_q] fp32.
    """

    name: str
    B: int
    H: int
    H_kv: int
    S_q: int
    S_k: int
    D: int
    scale: float
    causal: bool = False
    window: int = 0            # >0: key j visible iff qpos - window < j <= qpos
    document: bool = False     # packed documents, ids from doc_seed
    prefix_lm: bool = False    # uses prefix_len (per batch)
    alibi: bool = False        # default slopes m_h = 2^(-8(h+1)/H)
    softcap: float = 0.0       # >0: s <- softcap * tanh(s / softcap)
    q_offset: int = 0
    seed: int = 0
    doc_seed: int = 1
    doc_min: int = 256
    doc_max: int = 4096
    prefix_lens: Optional[tuple] = None

    @property
    def tiny(self) -> bool:
        return self.B * self.H * self.S_q <= 4096


def _wl(**kw) -> Workload:
    return Workload(**kw)


# The five problems the hot path is measured and checked on.  Names state the
# problem and its sizes.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        _wl(name="causal_b1_h2_s128_d64", B=1, H=2, H_kv=2, S_q=128, S_k=128,
            D=64, scale=1.0 / math.sqrt(64), causal=True),
        _wl(name="dense_b4_h16_s4096_d128", B=4, H=16, H_kv=16, S_q=4096,
            S_k=4096, D=128, scale=1.0 / math.sqrt(128)),
        _wl(name="causal_gqa_b2_h32_hkv8_s8192_d128", B=2, H=32, H_kv=8,
            S_q=8192, S_k=8192, D=128, scale=1.0 / math.sqrt(128),
            causal=True),
        _wl(name="window1024_softcap30_b1_h16_s16384_d128", B=1, H=16, H_kv=16,
            S_q=16384, S_k=16384, D=128, scale=1.0 / math.sqrt(128),
            causal=True, window=1024, softcap=30.0),
        _wl(name="docs_alibi_b1_h16_s32768_d128", B=1, H=16, H_kv=16,
            S_q=32768, S_k=32768, D=128, scale=1.0 / math.sqrt(128),
            causal=True, document=True, alibi=True),
    ]
}

# The workload the headline throughput is quoted on (dense, D=128).
HEADLINE = "dense_b4_h16_s4096_d128"


def get(name: str) -> Workload:
    return WORKLOADS[name]


def doc_ids_for(S: int, seed: int = 1, lo: int = 256, hi: int = 4096) -> torch.Tensor:
    """Document ids for a packed sequence of S tokens (int32 [S]).

    Lengths are drawn uniformly from the inclusive range [lo, hi] with a CPU
    generator seeded with ``seed`` until they cover S; the last one is cut.
    """
    g = torch.Generator().manual_seed(seed)
    lengths: List[int] = []
    total = 0
    while total < S:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        L = min(L, S - total)
        lengths.append(L)
        total += L
    ids = torch.repeat_interleave(torch.arange(len(lengths), dtype=torch.int32),
                                  torch.tensor(lengths))
    return ids.to(torch.int32)


def generate(w: Workload) -> Dict[str, torch.Tensor]:
    """Seeded CPU inputs for ``w``: q, k, v (bf16), plus doc_ids / prefix_len."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.H, w.S_q, w.D), generator=g, dtype=torch.float32)
    q = q.to(torch.bfloat16)
    k = torch.randn((w.B, w.H_kv, w.S_k, w.D), generator=g, dtype=torch.float32)
    k = k.to(torch.bfloat16)
    v = torch.randn((w.B, w.H_kv, w.S_k, w.D), generator=g, dtype=torch.float32)
    v = v.to(torch.bfloat16)
    out: Dict[str, torch.Tensor] = {"q": q, "k": k, "v": v}
    if w.document:
        ids = doc_ids_for(w.S_k, w.doc_seed, w.doc_min, w.doc_max)
        out["doc_ids"] = ids.unsqueeze(0).repeat(w.B, 1).contiguous()
    if w.prefix_lm:
        pl = w.prefix_lens if w.prefix_lens is not None else tuple([w.S_k // 4] * w.B)
        out["prefix_len"] = torch.tensor(pl, dtype=torch.int32)
    return out


def row_count(w: Workload) -> int:
    return w.B * w.H * w.S_q


def sample_rows(w: Workload, n_rows: int = 4096, seed: int = 2,
                doc_ids: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Flattened row indices ((b*H + h)*S_q + i) to check, sorted, int64.

    All rows when the problem is small; otherwise a seeded uniform sample
    without replacement plus edge rows: i in {0, 1, 2, 127, 128, S_q-1} of
    heads 0 and H-1 in the first and last batch, and the first two rows of
    every document.
    """
    N = row_count(w)
    if N <= n_rows:
        return torch.arange(N, dtype=torch.int64)
    g = torch.Generator().manual_seed(seed)
    picked = torch.randperm(N, generator=g)[:n_rows].to(torch.int64)
    edge: List[int] = []
    for b in sorted({0, w.B - 1}):
        for h in sorted({0, w.H - 1}):
            for i in (0, 1, 2, 127, 128, w.S_q - 1):
                if 0 <= i < w.S_q:
                    edge.append((b * w.H + h) * w.S_q + i)
    if doc_ids is not None:
        ids = doc_ids.reshape(-1, w.S_k)[0]
        starts = torch.nonzero(torch.diff(ids, prepend=ids[:1] - 1)).flatten()
        for s in starts.tolist():
            for i in (s, s + 1):
                if i < w.S_q:
                    edge.append(i)  # b = 0, h = 0
                    edge.append(((w.B - 1) * w.H + (w.H - 1)) * w.S_q + i)
    rows = torch.cat([picked, torch.tensor(edge, dtype=torch.int64)])
    return torch.unique(rows)
