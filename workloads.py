"""Seeded synthetic inputs for top-k sparse flash-attention backward.

This module holds no attention arithmetic: it only draws random tensors and
index lists with the shapes, dtypes and index structure of the workloads, so
that the CUDA library and the CPU oracle consume identical bytes.  It imports
neither of them.

Draw order (one ``torch.Generator`` on the CPU, seeded per workload):
lengths (TND only) -> q -> qRope -> k -> kRope -> v -> dO -> indices.
Values are N(0, std^2) drawn in fp32 and rounded to the dtype (round to
nearest even).  Index lists are distinct positions, sorted ascending, except
for the kinds that draw duplicates or out-of-range entries on purpose
("pile", "random_any").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "small_workload"]


@dataclass(frozen=True)
class Workload:
    name: str
    layout: str            # "BSND" or "TND"
    B: int
    S1: int                # BSND query length (TND: unused)
    S2: int                # BSND kv length (TND: unused)
    N1: int                # query heads G (N2 = 1)
    K: int                 # indices per query token
    block_size: int = 1    # sparseBlockSize
    mode: int = 0          # sparseMode (0 or 3)
    dtype: str = "bf16"
    std: float = 1.0
    seed: int = 101
    D: int = 512
    Dr: int = 64
    index_kind: str = "uniform"   # uniform | causal | block | skewed | all | pile | random_any
    kv_extra: int = 0             # TND: kvlen = qlen + kv_extra
    T1: int = 0                   # TND total query tokens
    deterministic: bool = False
    scale: Optional[float] = None
    act_q: Optional[tuple] = None  # TND lengths given explicitly

    @property
    def scale_value(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D + self.Dr)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def keff(self) -> int:
        return self.K * self.block_size


# The five workloads of the headline table: tiny parity case, MLA-style,
# TND varlen causal, block-sparse fp16, long context.
WORKLOADS = {
    "tiny": Workload("tiny", "BSND", B=1, S1=16, S2=2048, N1=4, K=1024, seed=101,
                     deterministic=True),
    "mla": Workload("mla", "BSND", B=1, S1=4096, S2=4096, N1=128, K=2048, seed=102),
    "tnd": Workload("tnd", "TND", B=4, S1=0, S2=0, N1=64, K=2048, mode=3, seed=103,
                    index_kind="causal", kv_extra=4096, T1=16384),
    "block": Workload("block", "BSND", B=2, S1=8192, S2=32768, N1=16, K=64, block_size=64,
                      dtype="fp16", std=0.5, seed=104, index_kind="block"),
    "long": Workload("long", "BSND", B=1, S1=8192, S2=65536, N1=128, K=8192, seed=105,
                     index_kind="skewed"),
    # MLA shape with 512 query tokens: the case the per-kernel profiles capture
    # (staged P/dS of 512 MB, larger than L2, a few GB on the device).
    "mla_q512": Workload("mla_q512", "BSND", B=1, S1=512, S2=4096, N1=128, K=2048, seed=106),
    # Block-sparse shape with 2048 query tokens: the key-major block kernel's
    # profiling case (2 GB of staged P/dS, 142 MB accumulator).
    "block_q2048": Workload("block_q2048", "BSND", B=1, S1=2048, S2=32768, N1=16, K=64, block_size=64,
                            dtype="fp16", std=0.5, seed=107, index_kind="block"),
}


def small_workload(**kw) -> Workload:
    base = dict(name="small", layout="BSND", B=1, S1=8, S2=512, N1=16, K=128, seed=7)
    base.update(kw)
    return Workload(**base)


def _randn(g, shape, w: Workload):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if w.std != 1.0:
        x = x * w.std
    return x.to(w.torch_dtype)


def _tnd_lengths(g, w: Workload):
    if w.act_q is not None:
        return list(w.act_q)
    # B-1 distinct cut points in [1, T1-1], sorted; lengths are the gaps.
    cuts = torch.randperm(w.T1 - 1, generator=g)[: w.B - 1] + 1
    cuts = torch.sort(cuts).values.tolist()
    edges = [0] + cuts + [w.T1]
    return [edges[i + 1] - edges[i] for i in range(w.B)]


def _indices_for_token(g, w: Workload, kvlen: int, qlen: int, i: int):
    K = w.K
    kind = w.index_kind
    if kind == "uniform":
        r = torch.randperm(kvlen, generator=g)[:K]
    elif kind == "all":
        r = torch.arange(K)
    elif kind == "causal":
        p = kvlen - qlen + i                       # query position in its kv sequence
        r = torch.randperm(p + 1, generator=g)[: min(K, p + 1)]
        if r.numel() < K:                          # pad with out-of-range entries
            r = torch.cat([r, torch.full((K - r.numel(),), -1, dtype=r.dtype)])
    elif kind == "block":
        nblk = kvlen // w.block_size
        r = torch.randperm(nblk, generator=g)[:K] * w.block_size
    elif kind == "skewed":
        recent = 8192
        half = K // 2
        a = torch.randperm(recent, generator=g)[:half] + (kvlen - recent)
        b = torch.randperm(kvlen - recent, generator=g)[: K - half]
        r = torch.cat([a, b])
    elif kind == "pile":
        # half the slots piled onto keys 0 and 1 (thousands of occurrences of
        # one key in a token chunk), half distinct uniform positions
        half = K // 2
        a = torch.randint(0, 2, (half,), generator=g)
        b = torch.randperm(kvlen, generator=g)[: K - half]
        r = torch.cat([a, b])
    elif kind == "random_any":
        # arbitrary (possibly duplicated / out-of-range / negative) entries
        r = torch.randint(-4, kvlen + 4, (K,), generator=g)
        return r.to(torch.int32)
    else:
        raise ValueError(kind)
    return torch.sort(r).values.to(torch.int32)


def make_inputs(w: Workload):
    """Returns a dict of CPU tensors: q, q_rope, k, k_rope, v, d_out, indices and,
    for TND, act_seq_q / act_seq_kv (int32)."""
    g = torch.Generator().manual_seed(w.seed)
    G, D, Dr = w.N1, w.D, w.Dr
    res = {}
    if w.layout == "TND":
        aq = _tnd_lengths(g, w)
        akv = [a + w.kv_extra for a in aq]
        T1, T2 = sum(aq), sum(akv)
        res["act_seq_q"] = torch.tensor(aq, dtype=torch.int32)
        res["act_seq_kv"] = torch.tensor(akv, dtype=torch.int32)
        qs, ks = (T1, G), (T2, 1)
        batches = [(aq[b], akv[b]) for b in range(w.B)]
    else:
        qs, ks = (w.B, w.S1, G), (w.B, w.S2, 1)
        batches = [(w.S1, w.S2)] * w.B
    res["q"] = _randn(g, qs + (D,), w)
    res["q_rope"] = _randn(g, qs + (Dr,), w) if Dr > 0 else None
    res["k"] = _randn(g, ks + (D,), w)
    res["k_rope"] = _randn(g, ks + (Dr,), w) if Dr > 0 else None
    res["v"] = _randn(g, ks + (D,), w)
    res["d_out"] = _randn(g, qs + (D,), w)
    rows = []
    for qlen, kvlen in batches:
        for i in range(qlen):
            rows.append(_indices_for_token(g, w, kvlen, qlen, i))
    idx = torch.stack(rows) if rows else torch.zeros((0, w.K), dtype=torch.int32)
    if w.layout == "TND":
        res["indices"] = idx.reshape(-1, 1, w.K).contiguous()
    else:
        res["indices"] = idx.reshape(w.B, w.S1, 1, w.K).contiguous()
    return res


def with_(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
