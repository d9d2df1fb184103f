"""Plain fp64 CPU oracle for top-k sparse flash attention: forward and backward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  The product library
(``sfa_grad_gb300``) never imports it, and it imports nothing from the product.

Sources (cited by page title and section):

* [SFAG] "aclnnSparseFlashAttentionGrad" (CANN ops-transformer documentation):
  - 功能说明 (function): key/value rows are gathered by ``topkIndices``; each index
    selects ``selectedBlockSize`` = ``sparseBlockSize`` consecutive rows.
  - 阶段1 (stage 1): dP = dO @ V^T and dV[u] = P^T @ dO.
  - 阶段2 (stage 2): dS = P * (dP - FlashSoftmaxGrad(dO, O)); the product is
    elementwise (the MindSpore page computes it with an elementwise multiply).
  - 阶段3 (stage 3): dQ = dS @ K[u] * scale and dK[u] = dS^T @ Q * scale; the
    page writes 1/sqrt(d), which the ``scaleValue`` parameter replaces.
  - 参数说明 (parameter table): shapes (B,S1,N1,D)/(T1,N1,D) for q, dOut, out;
    (B,S2,N2,D)/(T2,N2,D) for k, v; (B,S1,N2,K)/(T1,N2,K) indices;
    (B,N2,S1,G)/(N2,T1,G) softmaxMax/softmaxSum; per-batch actual lengths for
    TND; the MLA rope tensors queryRope/keyRope (Dr = 64).
  - 约束说明 / Mask table: sparseMode 0 = no mask, 3 = rightDownCausal (lower
    triangle anchored at the bottom-right corner).
* [FABWD] MindSpore 2.2.0 ``flash_attention_bwd.py`` (dense FlashAttention
  backward in TIK):
  - ``compute_Pij``: P = exp(S - m) * (1 / l) from the saved row max m and row
    sum l (so l is a plain sum of exponentials, not a log-sum-exp).
  - ``compute_Di``: D_i = rowsum(dO * O).
  - ``compute_dSij``: dS = P * (dP - D_i).
  - ``update_dVj`` / ``update_dQi`` / ``update_dKj``: the three contractions,
    accumulated into zero-initialised fp32 outputs with atomic adds.

Readings where the pages are silent or garbled (each is repeated in the design
notes):

1. softmaxMax holds the max of the *scaled* scores and softmaxSum the sum of
   exp(x - max) over the selected keys ([FABWD] compute_Pij).
2. The rope parts are concatenated to the 512-wide parts in S, dQ and dK; V
   and dV have no rope part ([SFAG] parameter table, queryRope/keyRope rows).
3. An index r with block size bs selects keys r, r+1, ..., r+bs-1 (r is a key
   position, not a block number).
4. A key j of a query at local position i is valid iff 0 <= j < kvlen and, in
   sparseMode 3, j <= kvlen - qlen + i.  Invalid keys contribute nothing
   (negative or out-of-range indices are treated as padding).
5. Duplicate indices keep gather semantics: every occurrence is its own
   column of S, and the scatter-add adds every occurrence.
6. A query row with no valid key has out = 0, max = -inf, sum = 0 in the
   forward; in the backward a row with sum == 0 has P == 0.
7. TND indices are local to the batch's KV segment, whose start is the prefix
   sum of actualSeqLengthsKv; BSND batch b starts at b * S2.

Everything is computed in float64 from the given (already dtype-rounded)
input values.  Rows of dK / dV / dKRope that no valid key selects are zero.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "Problem",
    "make_problem",
    "token_keys",
    "token_terms",
    "sfa_fwd",
    "sfa_bwd",
]


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu")
        if a.dtype.is_floating_point:
            a = a.double()
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


def _i64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.asarray(a, dtype=np.int64)


class Problem:
    """Token-major view of one call.

    q: (T1, G, D); qr: (T1, G, Dr) or None; k: (T2, D); kr: (T2, Dr) or None;
    v: (T2, Dv); idx: (T1, K) int64; batches: list of (q_start, qlen, kv_start, kvlen).
    """

    def __init__(self, q, k, v, indices, scale, block_size, layout, mode,
                 act_seq_q=None, act_seq_kv=None, q_rope=None, k_rope=None):
        layout = layout.upper()
        if layout not in ("BSND", "TND"):
            raise ValueError("layout must be BSND or TND")
        if mode not in (0, 3):
            raise ValueError("sparse_mode must be 0 or 3")
        self.layout, self.mode = layout, int(mode)
        self.scale, self.bs = float(scale), int(block_size)
        q, k, v = _f64(q), _f64(k), _f64(v)
        qr, kr = _f64(q_rope), _f64(k_rope)
        idx = _i64(indices)
        if layout == "BSND":
            B, S1, N1, D = q.shape
            S2 = k.shape[1]
            if k.shape[2] != 1:
                raise ValueError("N2 must be 1")
            self.shape_q = (B, S1, N1)
            self.shape_kv = (B, S2)
            self.q = q.reshape(B * S1, N1, D)
            self.k = k.reshape(B * S2, k.shape[-1])
            self.v = v.reshape(B * S2, v.shape[-1])
            self.qr = None if qr is None else qr.reshape(B * S1, N1, qr.shape[-1])
            self.kr = None if kr is None else kr.reshape(B * S2, kr.shape[-1])
            self.idx = idx.reshape(B * S1, idx.shape[-1])
            self.batches = [(b * S1, S1, b * S2, S2) for b in range(B)]
        else:
            T1, N1, D = q.shape
            T2 = k.shape[0]
            if k.shape[1] != 1:
                raise ValueError("N2 must be 1")
            aq, akv = _i64(act_seq_q), _i64(act_seq_kv)
            if aq is None or akv is None or len(aq) != len(akv):
                raise ValueError("TND needs per-batch actual lengths of equal count")
            if (aq < 0).any() or (akv < 0).any():
                raise ValueError("actual lengths must be non-negative")
            if aq.sum() != T1 or akv.sum() != T2:
                raise ValueError("actual lengths must sum to T1 / T2")
            self.shape_q = (T1, N1)
            self.shape_kv = (T2,)
            self.q = q
            self.k = k.reshape(T2, k.shape[-1])
            self.v = v.reshape(T2, v.shape[-1])
            self.qr = qr
            self.kr = None if kr is None else kr.reshape(T2, kr.shape[-1])
            self.idx = idx.reshape(T1, idx.shape[-1])
            qs = np.concatenate([[0], np.cumsum(aq)])
            ks = np.concatenate([[0], np.cumsum(akv)])
            self.batches = [(int(qs[b]), int(aq[b]), int(ks[b]), int(akv[b])) for b in range(len(aq))]
        if (self.qr is None) != (self.kr is None):
            raise ValueError("queryRope and keyRope come together")
        self.T1, self.G = self.q.shape[0], self.q.shape[1]
        self.T2 = self.k.shape[0]
        self.tok_batch = np.empty(self.T1, dtype=np.int64)
        for b, (q0, ql, _, _) in enumerate(self.batches):
            self.tok_batch[q0:q0 + ql] = b

    def stats_view(self, a):
        """(B,N2,S1,G) or (N2,T1,G) -> (T1, G)."""
        a = _f64(a)
        if self.layout == "BSND":
            B, S1, _ = self.shape_q
            return a.reshape(B, S1, self.G).reshape(B * S1, self.G)
        return a.reshape(self.T1, self.G)

    def tok_view(self, a):
        """(B,S1,N1,X) or (T1,N1,X) -> (T1, G, X)."""
        a = _f64(a)
        return a.reshape(self.T1, self.G, a.shape[-1])


def make_problem(**kw) -> Problem:
    return Problem(**kw)


def token_keys(prob: Problem, t: int):
    """Expanded key positions of token t and their validity ([SFAG] 功能说明,
    Mask table; readings 3 and 4).  Returns (j, valid, kv_start) with j the
    batch-local key position of every (slot, block offset) column."""
    b = int(prob.tok_batch[t])
    q0, qlen, kv0, kvlen = prob.batches[b]
    i = t - q0
    r = prob.idx[t].astype(np.int64)
    j = (r[:, None] + np.arange(prob.bs, dtype=np.int64)[None, :]).reshape(-1)
    valid = (j >= 0) & (j < kvlen)
    if prob.mode == 3:
        valid &= j <= (kvlen - qlen + i)
    return j, valid, kv0


def _scores(prob: Problem, t: int, rows):
    """x = scale * ([q || qRope] . [k || kRope]) over the given kv rows, (G, n)."""
    x = prob.q[t] @ prob.k[rows].T
    if prob.qr is not None:
        x = x + prob.qr[t] @ prob.kr[rows].T
    return prob.scale * x


def token_terms(prob: Problem, t: int, d_out, out, smax, ssum, keep=None):
    """All intermediate terms of token t over its valid key columns.

    d_out, out: (T1, G, Dv) float64; smax, ssum: (T1, G) float64.
    keep (optional, bool per global kv row) restricts the columns to those rows;
    every term of a column depends only on that column and the token's row
    statistics, so a subset is exact.
    Returns dict(rows, x, P, dP, D, dS) where rows are global kv rows.
    """
    j, valid, kv0 = token_keys(prob, t)
    rows = kv0 + j[valid]
    if keep is not None:
        rows = rows[keep[rows]]
    x = _scores(prob, t, rows)
    m = smax[t][:, None]
    l = ssum[t][:, None]
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        P = np.where(l > 0, np.exp(x - m) / l, 0.0)           # [FABWD] compute_Pij
    D = np.sum(d_out[t] * out[t], axis=-1)                      # [FABWD] compute_Di
    dP = d_out[t] @ prob.v[rows].T                              # [SFAG] 阶段1
    dS = P * (dP - D[:, None])                                  # [SFAG] 阶段2
    return dict(rows=rows, x=x, P=P, dP=dP, D=D, dS=dS)


def sfa_fwd(q, k, v, indices, scale, sparse_block_size=1, layout="BSND", sparse_mode=0,
            act_seq_q=None, act_seq_kv=None, q_rope=None, k_rope=None, token_rows=None):
    """Forward: out, softmaxMax, softmaxSum (float64), shaped like the pages'
    tensors: out like q (last dim = v's), stats (B,1,S1,G) or (1,T1,G).

    Rows with no valid key: out = 0, max = -inf, sum = 0 (reading 6).
    token_rows (optional) computes only those query tokens; other rows are NaN."""
    prob = Problem(q, k, v, indices, scale, sparse_block_size, layout, sparse_mode,
                   act_seq_q, act_seq_kv, q_rope, k_rope)
    Dv = prob.v.shape[1]
    out = np.zeros((prob.T1, prob.G, Dv))
    smax = np.full((prob.T1, prob.G), -np.inf)
    ssum = np.zeros((prob.T1, prob.G))
    visit = range(prob.T1)
    if token_rows is not None:
        visit = sorted(set(int(x) for x in token_rows))
        keep = np.zeros(prob.T1, bool)
        keep[visit] = True
        out[~keep], smax[~keep], ssum[~keep] = np.nan, np.nan, np.nan
    for t in visit:
        j, valid, kv0 = token_keys(prob, t)
        rows = kv0 + j[valid]
        if rows.size == 0:
            continue
        x = _scores(prob, t, rows)
        m = x.max(axis=1)
        e = np.exp(x - m[:, None])
        l = e.sum(axis=1)
        out[t] = (e / l[:, None]) @ prob.v[rows]
        smax[t], ssum[t] = m, l
    if prob.layout == "BSND":
        B, S1, N1 = prob.shape_q
        out = out.reshape(B, S1, N1, Dv)
        smax = smax.reshape(B, 1, S1, N1)
        ssum = ssum.reshape(B, 1, S1, N1)
    else:
        out = out.reshape(prob.T1, prob.G, Dv)
        smax = smax.reshape(1, prob.T1, prob.G)
        ssum = ssum.reshape(1, prob.T1, prob.G)
    return out, smax, ssum


def sfa_bwd(q, k, v, indices, d_out, out, softmax_max, softmax_sum, scale,
            sparse_block_size=1, layout="BSND", sparse_mode=0, act_seq_q=None,
            act_seq_kv=None, q_rope=None, k_rope=None, token_rows=None, key_rows=None):
    """Backward: dict(dq, dk, dv, dq_rope, dk_rope) in float64, shaped like
    q, k, v, q_rope, k_rope ([SFAG] 阶段1-3, [FABWD] update_dVj/dQi/dKj).

    token_rows / key_rows (optional) restrict the work to those query tokens
    (dq, dq_rope) and those global kv rows (dk, dv, dk_rope); other rows of the
    results are left NaN.  Either one alone leaves the other output family NaN.
    """
    prob = Problem(q, k, v, indices, scale, sparse_block_size, layout, sparse_mode,
                   act_seq_q, act_seq_kv, q_rope, k_rope)
    dO = prob.tok_view(d_out)
    O = prob.tok_view(out)
    smax = prob.stats_view(softmax_max)
    ssum = prob.stats_view(softmax_sum)
    T1, G = prob.T1, prob.G
    D, Dv = prob.q.shape[2], prob.v.shape[1]
    has_rope = prob.qr is not None
    Dr = prob.qr.shape[2] if has_rope else 0
    full = token_rows is None and key_rows is None
    want_tok = np.ones(T1, bool) if full else np.zeros(T1, bool)
    if token_rows is not None:
        want_tok[np.asarray(token_rows, dtype=np.int64)] = True
    want_key = np.ones(prob.T2, bool) if full else np.zeros(prob.T2, bool)
    if key_rows is not None:
        want_key[np.asarray(key_rows, dtype=np.int64)] = True
    do_keys = full or key_rows is not None

    dq = np.zeros((T1, G, D)) if full or token_rows is not None else np.full((T1, G, D), np.nan)
    dqr = (np.zeros((T1, G, Dr)) if full or token_rows is not None else np.full((T1, G, Dr), np.nan)) if has_rope else None
    if do_keys:
        dk, dv = np.zeros((prob.T2, D)), np.zeros((prob.T2, Dv))
        dkr = np.zeros((prob.T2, Dr)) if has_rope else None
    else:
        dk, dv = np.full((prob.T2, D), np.nan), np.full((prob.T2, Dv), np.nan)
        dkr = np.full((prob.T2, Dr), np.nan) if has_rope else None

    for t in range(T1):
        if not full and not want_tok[t]:
            if not do_keys:
                continue
            j, valid, kv0 = token_keys(prob, t)
            if not np.any(want_key[(kv0 + j[valid])]):
                continue
        terms = token_terms(prob, t, dO, O, smax, ssum, keep=None if (full or want_tok[t]) else want_key)
        rows, P, dS = terms["rows"], terms["P"], terms["dS"]
        if want_tok[t]:
            dq[t] = prob.scale * (dS @ prob.k[rows])                  # [SFAG] 阶段3 dQ
            if has_rope:
                dqr[t] = prob.scale * (dS @ prob.kr[rows])
        if do_keys:
            sel = want_key[rows]
            if not sel.any():
                continue
            r = rows[sel]
            np.add.at(dk, r, prob.scale * (dS[:, sel].T @ prob.q[t]))  # [SFAG] 阶段3 dK
            if has_rope:
                np.add.at(dkr, r, prob.scale * (dS[:, sel].T @ prob.qr[t]))
            np.add.at(dv, r, P[:, sel].T @ dO[t])                     # [SFAG] 阶段1 dV
    if do_keys and not full:
        dk[~want_key] = np.nan
        dv[~want_key] = np.nan
        if has_rope:
            dkr[~want_key] = np.nan

    if prob.layout == "BSND":
        B, S1, N1 = prob.shape_q
        _, S2 = prob.shape_kv
        res = dict(dq=dq.reshape(B, S1, N1, D), dk=dk.reshape(B, S2, 1, D),
                   dv=dv.reshape(B, S2, 1, Dv),
                   dq_rope=None if not has_rope else dqr.reshape(B, S1, N1, Dr),
                   dk_rope=None if not has_rope else dkr.reshape(B, S2, 1, Dr))
    else:
        res = dict(dq=dq, dk=dk.reshape(prob.T2, 1, D), dv=dv.reshape(prob.T2, 1, Dv),
                   dq_rope=dqr, dk_rope=None if not has_rope else dkr.reshape(prob.T2, 1, Dr))
    return res
