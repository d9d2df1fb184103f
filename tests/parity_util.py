"""Helpers shared by the GPU parity tests: feed identical bytes to the oracle
and to the library, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import Workload, make_inputs

# Float outputs, compared in fp32 per tensor: relative Frobenius error
# (bf16 1e-2, fp16 5e-3) and max abs error 3e-2.
REL_TOL = {"bf16": 1e-2, "fp16": 5e-3}
MAX_ABS = 3e-2
OUT_NAMES = ("dq", "dk", "dv", "dq_rope", "dk_rope")


def oracle_kwargs(w: Workload, inp: dict) -> dict:
    kw = dict(q=inp["q"], k=inp["k"], v=inp["v"], indices=inp["indices"], scale=w.scale_value,
              sparse_block_size=w.block_size, layout=w.layout, sparse_mode=w.mode,
              q_rope=inp.get("q_rope"), k_rope=inp.get("k_rope"))
    if w.layout == "TND":
        kw["act_seq_q"] = inp["act_seq_q"]
        kw["act_seq_kv"] = inp["act_seq_kv"]
    return kw


def oracle_saved(w: Workload, inp: dict):
    """out (dtype), softmaxMax / softmaxSum (fp32) from the oracle forward."""
    out, smax, ssum = oracle.sfa_fwd(**oracle_kwargs(w, inp))
    return (torch.from_numpy(out).to(w.torch_dtype), torch.from_numpy(smax).float(),
            torch.from_numpy(ssum).float())


def to_cuda(x):
    return None if x is None else x.cuda()


def gpu_call_kwargs(w: Workload, dev: dict) -> dict:
    kw = dict(q_rope=dev.get("q_rope"), k_rope=dev.get("k_rope"), sparse_block_size=w.block_size,
              layout=w.layout, sparse_mode=w.mode)
    if w.layout == "TND":
        kw["act_seq_q"] = dev["act_seq_q"]
        kw["act_seq_kv"] = dev["act_seq_kv"]
    return kw


def compare(name: str, got, ref, dtype: str, rows=None):
    a = got.detach().float().cpu().double().numpy()
    b = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        a = a.reshape(-1, *a.shape[-1:])[rows] if a.ndim > 1 else a[rows]
        b = b.reshape(-1, *b.shape[-1:])[rows]
    assert np.all(np.isfinite(a)), f"{name}: non-finite output"
    d = a - b
    nb = np.linalg.norm(b)
    rel = np.linalg.norm(d) / nb if nb > 0 else np.linalg.norm(d)
    mx = float(np.abs(d).max()) if d.size else 0.0
    assert rel <= REL_TOL[dtype] and mx <= MAX_ABS, f"{name}: rel_fro {rel:.3e} max_abs {mx:.3e}"
    return rel, mx


def flat_rows(x: torch.Tensor, width: int) -> torch.Tensor:
    return x.reshape(-1, width)
