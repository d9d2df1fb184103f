"""Pins for the fp64 oracle, independent of the oracle itself.

* central finite differences of L = sum(O * dO) (both sparse modes, block
  sizes 1 and 2, BSND and TND, rope on and off);
* the dense special case (indices select every key) against torch.autograd of
  ordinary dense attention, causal mask built with torch.tril;
* invariants: rowsum(P) = 1, Dsum = rowsum(P * dP), rowsum(dS) = 0, slot
  permutation invariance, linearity in dO;
* equivalences: block expansion, TND(B=1) == BSND, causal with all keys
  allowed == no mask, padding indices == absent indices;
* a scalar brute-force implementation (pure Python loops, duplicates included);
* the closed form of the documentation page's worked example.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import sfa_bwd, sfa_fwd, make_problem, token_terms

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_case(rng, B=2, S1=3, S2=7, G=2, D=8, Dr=4, K=3, bs=1, rope=True, layout="BSND",
               aq=None, akv=None, distinct=True):
    if layout == "BSND":
        q = rng.standard_normal((B, S1, G, D))
        k = rng.standard_normal((B, S2, 1, D))
        v = rng.standard_normal((B, S2, 1, D + 1))
        qr = rng.standard_normal((B, S1, G, Dr)) if rope else None
        kr = rng.standard_normal((B, S2, 1, Dr)) if rope else None
        dO = rng.standard_normal((B, S1, G, D + 1))
        nblk = S2 // bs if bs > 1 else S2
        idx = np.zeros((B, S1, 1, K), np.int64)
        for b in range(B):
            for i in range(S1):
                pick = rng.permutation(nblk)[:K] if distinct else rng.integers(0, nblk, K)
                idx[b, i, 0] = pick * bs
        return dict(q=q, k=k, v=v, q_rope=qr, k_rope=kr, indices=idx, layout="BSND"), dO
    T1, T2 = sum(aq), sum(akv)
    q = rng.standard_normal((T1, G, D))
    k = rng.standard_normal((T2, 1, D))
    v = rng.standard_normal((T2, 1, D + 1))
    qr = rng.standard_normal((T1, G, Dr)) if rope else None
    kr = rng.standard_normal((T2, 1, Dr)) if rope else None
    dO = rng.standard_normal((T1, G, D + 1))
    idx = np.zeros((T1, 1, K), np.int64)
    t = 0
    for b in range(len(aq)):
        for i in range(aq[b]):
            nblk = akv[b] // bs if bs > 1 else akv[b]
            idx[t, 0] = rng.permutation(max(nblk, K))[:K] * bs
            t += 1
    return dict(q=q, k=k, v=v, q_rope=qr, k_rope=kr, indices=idx, layout="TND",
                act_seq_q=np.array(aq), act_seq_kv=np.array(akv)), dO


def _loss(case, dO, scale, bs, mode):
    out, _, _ = sfa_fwd(scale=scale, sparse_block_size=bs, sparse_mode=mode, **case)
    return float(np.sum(out * dO))


FD_CASES = [
    dict(layout="BSND", bs=1, mode=0, rope=True),
    dict(layout="BSND", bs=1, mode=3, rope=True),
    dict(layout="BSND", bs=2, mode=0, rope=True),
    dict(layout="BSND", bs=2, mode=3, rope=False),
    dict(layout="TND", bs=1, mode=3, rope=True),
    dict(layout="TND", bs=2, mode=0, rope=True),
]


@pytest.mark.parametrize("cfg", FD_CASES, ids=lambda c: f"{c['layout']}-bs{c['bs']}-m{c['mode']}-r{int(c['rope'])}")
def test_finite_differences(cfg):
    rng = np.random.default_rng(11 + cfg["bs"] + 7 * cfg["mode"])
    if cfg["layout"] == "BSND":
        case, dO = _rand_case(rng, S1=3, S2=8, K=3, bs=cfg["bs"], rope=cfg["rope"])
    else:
        case, dO = _rand_case(rng, layout="TND", aq=[2, 3], akv=[6, 8], K=3, bs=cfg["bs"], rope=cfg["rope"])
    scale, bs, mode = 0.37, cfg["bs"], cfg["mode"]
    out, smax, ssum = sfa_fwd(scale=scale, sparse_block_size=bs, sparse_mode=mode, **case)
    g = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale,
                sparse_block_size=bs, sparse_mode=mode, **case)
    h = 1e-6
    names = [("q", "dq"), ("k", "dk"), ("v", "dv")]
    if cfg["rope"]:
        names += [("q_rope", "dq_rope"), ("k_rope", "dk_rope")]
    for src, dst in names:
        x = case[src]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            old = x[mi]
            x[mi] = old + h
            lp = _loss(case, dO, scale, bs, mode)
            x[mi] = old - h
            lm = _loss(case, dO, scale, bs, mode)
            x[mi] = old
            fd[mi] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g[dst], fd, rtol=1e-6, atol=1e-7, err_msg=f"{src}")


def _dense_torch(q, k, v, qr, kr, dO, scale, causal):
    """Ordinary dense attention over all keys, per batch and head, with autograd."""
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    tqr = torch.tensor(qr, requires_grad=True)
    tkr = torch.tensor(kr, requires_grad=True)
    # q (B,S1,G,D) ; k (B,S2,1,D)
    s = torch.einsum("bigd,bjd->bgij", tq, tk[:, :, 0]) + torch.einsum("bigd,bjd->bgij", tqr, tkr[:, :, 0])
    s = s * scale
    S1, S2 = q.shape[1], k.shape[1]
    if causal:
        allowed = torch.ones(S1, S2, dtype=torch.bool).tril(diagonal=S2 - S1)
        s = s.masked_fill(~allowed, float("-inf"))
    m = s.max(dim=-1).values
    l = torch.exp(s - m[..., None]).sum(-1)
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bgij,bjd->bigd", p, tv[:, :, 0])
    loss = (o * torch.tensor(dO)).sum()
    loss.backward()
    return dict(out=o.detach().numpy(), m=m.detach().numpy(), l=l.detach().numpy(),
                dq=tq.grad.numpy(), dk=tk.grad.numpy(), dv=tv.grad.numpy(),
                dq_rope=tqr.grad.numpy(), dk_rope=tkr.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_dense_special_case_matches_autograd(causal):
    rng = np.random.default_rng(5 + causal)
    B, S1, S2, G, D, Dr = 2, 5, 9, 3, 6, 4
    q = rng.standard_normal((B, S1, G, D)); k = rng.standard_normal((B, S2, 1, D))
    v = rng.standard_normal((B, S2, 1, D)); qr = rng.standard_normal((B, S1, G, Dr))
    kr = rng.standard_normal((B, S2, 1, Dr)); dO = rng.standard_normal((B, S1, G, D))
    scale = 0.41
    ref = _dense_torch(q, k, v, qr, kr, dO, scale, causal)
    idx = np.broadcast_to(np.arange(S2), (B, S1, 1, S2)).copy()
    mode = 3 if causal else 0
    # oracle forward against torch
    out, smax, ssum = sfa_fwd(q, k, v, idx, scale, 1, "BSND", mode, q_rope=qr, k_rope=kr)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(smax[:, 0], ref["m"].transpose(0, 2, 1), rtol=1e-12)
    np.testing.assert_allclose(ssum[:, 0], ref["l"].transpose(0, 2, 1), rtol=1e-12)
    # oracle backward fed torch's forward results
    m_in = ref["m"].transpose(0, 2, 1)[:, None]
    l_in = ref["l"].transpose(0, 2, 1)[:, None]
    g = sfa_bwd(q, k, v, idx, dO, ref["out"], m_in, l_in, scale, 1, "BSND", mode,
                q_rope=qr, k_rope=kr)
    for name in ("dq", "dk", "dv", "dq_rope", "dk_rope"):
        np.testing.assert_allclose(g[name], ref[name], rtol=1e-10, atol=1e-12, err_msg=name)


def test_invariants():
    rng = np.random.default_rng(3)
    case, dO = _rand_case(rng, B=1, S1=4, S2=40, G=3, D=7, Dr=5, K=9)
    scale = 0.3
    out, smax, ssum = sfa_fwd(scale=scale, **case)
    prob = make_problem(scale=scale, block_size=1, mode=0, **{k: v for k, v in case.items()})
    O = prob.tok_view(out); dOt = prob.tok_view(dO)
    mx, sm = prob.stats_view(smax), prob.stats_view(ssum)
    for t in range(prob.T1):
        tt = token_terms(prob, t, dOt, O, mx, sm)
        np.testing.assert_allclose(tt["P"].sum(axis=1), 1.0, rtol=1e-13)
        np.testing.assert_allclose(tt["D"], (tt["P"] * tt["dP"]).sum(axis=1), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(tt["dS"].sum(axis=1), 0.0, atol=1e-12)
    # slot permutation invariance
    g0 = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale, **case)
    c2 = dict(case); c2["indices"] = case["indices"][..., rng.permutation(case["indices"].shape[-1])]
    g1 = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale, **c2)
    for n in ("dq", "dk", "dv", "dq_rope", "dk_rope"):
        np.testing.assert_allclose(g0[n], g1[n], rtol=1e-12, atol=1e-13)
    # linearity in dO (out and the statistics held fixed)
    dO2 = rng.standard_normal(dO.shape)
    ga = sfa_bwd(d_out=dO2, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale, **case)
    gb = sfa_bwd(d_out=dO + 2 * dO2, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale, **case)
    for n in ("dq", "dk", "dv", "dq_rope", "dk_rope"):
        np.testing.assert_allclose(gb[n], g0[n] + 2 * ga[n], rtol=1e-10, atol=1e-12)


def _grads(case, dO, scale, bs, mode):
    out, smax, ssum = sfa_fwd(scale=scale, sparse_block_size=bs, sparse_mode=mode, **case)
    g = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=scale,
                sparse_block_size=bs, sparse_mode=mode, **case)
    return out, g


def test_block_expansion_equals_expanded_indices():
    rng = np.random.default_rng(21)
    case, dO = _rand_case(rng, B=2, S1=3, S2=16, K=3, bs=4)
    o1, g1 = _grads(case, dO, 0.5, 4, 0)
    c2 = dict(case)
    idx = case["indices"]
    c2["indices"] = (idx[..., :, None] + np.arange(4)).reshape(idx.shape[:-1] + (-1,))
    o2, g2 = _grads(c2, dO, 0.5, 1, 0)
    np.testing.assert_allclose(o1, o2, rtol=1e-13)
    for n in g1:
        np.testing.assert_allclose(g1[n], g2[n], rtol=1e-12, atol=1e-13)


def test_tnd_single_batch_equals_bsnd():
    rng = np.random.default_rng(22)
    case, dO = _rand_case(rng, B=1, S1=4, S2=10, K=5)
    o1, g1 = _grads(case, dO, 0.5, 1, 3)
    c2 = dict(q=case["q"][0], k=case["k"][0], v=case["v"][0], q_rope=case["q_rope"][0],
              k_rope=case["k_rope"][0], indices=case["indices"][0], layout="TND",
              act_seq_q=np.array([4]), act_seq_kv=np.array([10]))
    o2, g2 = _grads(c2, dO[0], 0.5, 1, 3)
    np.testing.assert_allclose(o1[0], o2, rtol=1e-13)
    for n in g1:
        np.testing.assert_allclose(g1[n][0], g2[n], rtol=1e-12, atol=1e-13)


def test_causal_with_all_keys_allowed_equals_no_mask():
    rng = np.random.default_rng(23)
    case, dO = _rand_case(rng, B=1, S1=4, S2=12, K=5)
    # query i may see keys <= 12 - 4 + i >= 8; draw indices from [0, 8]
    case["indices"] = np.stack([rng.permutation(9)[:5] for _ in range(4)]).reshape(1, 4, 1, 5)
    o0, g0 = _grads(case, dO, 0.5, 1, 0)
    o3, g3 = _grads(case, dO, 0.5, 1, 3)
    np.testing.assert_allclose(o0, o3, rtol=1e-14)
    for n in g0:
        np.testing.assert_allclose(g0[n], g3[n], rtol=1e-13, atol=1e-14)


def test_causal_mask_drops_future_keys():
    """Mode 3: a key past kvlen - qlen + i contributes exactly as if absent."""
    rng = np.random.default_rng(24)
    case, dO = _rand_case(rng, B=1, S1=3, S2=10, K=4)
    lim = [10 - 3 + i for i in range(3)]
    idx = np.zeros((1, 3, 1, 4), np.int64)
    for i in range(3):
        idx[0, i, 0] = [0, 2, lim[i], lim[i] + 1 if lim[i] + 1 < 10 else 9]
    idx[0, 2, 0, 3] = 9   # limit of the last row is 9: key 9 allowed there
    case["indices"] = idx
    o3, g3 = _grads(case, dO, 0.5, 1, 3)
    c2 = dict(case)
    idx2 = idx.copy()
    idx2[0, 0, 0, 3] = -1   # future key of row 0 replaced by padding
    idx2[0, 1, 0, 3] = -1
    c2["indices"] = idx2
    o2, g2 = _grads(c2, dO, 0.5, 1, 0)
    np.testing.assert_allclose(o3, o2, rtol=1e-14)
    for n in g3:
        np.testing.assert_allclose(g3[n], g2[n], rtol=1e-13, atol=1e-14)


def test_padding_indices_equal_absent_indices():
    rng = np.random.default_rng(25)
    case, dO = _rand_case(rng, B=1, S1=3, S2=9, K=3)
    idx = case["indices"]
    pad_a = np.concatenate([idx, np.full(idx.shape[:-1] + (2,), -1)], axis=-1)
    pad_b = np.concatenate([idx, np.stack([np.full(idx.shape[:-1], 9), np.full(idx.shape[:-1], -700)], -1)], axis=-1)
    o0, g0 = _grads(case, dO, 0.5, 1, 0)
    for pad in (pad_a, pad_b):
        c = dict(case); c["indices"] = pad
        o1, g1 = _grads(c, dO, 0.5, 1, 0)
        np.testing.assert_allclose(o0, o1, rtol=1e-14)
        for n in g0:
            np.testing.assert_allclose(g0[n], g1[n], rtol=1e-13, atol=1e-14)


def test_rows_without_valid_keys():
    """Mode 3 with S1 > S2: the first rows see no key; their out is 0, the
    statistics are (-inf, 0) and they contribute no gradient."""
    rng = np.random.default_rng(26)
    case, dO = _rand_case(rng, B=1, S1=6, S2=3, K=2)
    out, smax, ssum = sfa_fwd(scale=0.5, sparse_mode=3, **case)
    # row i sees keys <= 3 - 6 + i -> rows 0, 1, 2 see nothing
    assert np.all(out[0, :3] == 0) and np.all(np.isneginf(smax[0, 0, :3])) and np.all(ssum[0, 0, :3] == 0)
    g = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=0.5, sparse_mode=3, **case)
    assert np.all(g["dq"][0, :3] == 0)
    assert all(np.all(np.isfinite(g[n])) for n in g)


def _brute(case, dO, out, smax, ssum, scale, bs, mode):
    """Scalar loops over (batch, token, head, slot, offset, feature)."""
    q, k, v, qr, kr, idx = (case[n] for n in ("q", "k", "v", "q_rope", "k_rope", "indices"))
    B, S1, G, D = q.shape
    S2, Dv, Dr = k.shape[1], v.shape[3], qr.shape[3]
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    dqr = np.zeros_like(qr); dkr = np.zeros_like(kr)
    for b in range(B):
        for i in range(S1):
            cols = []
            for s in range(idx.shape[3]):
                for u in range(bs):
                    j = int(idx[b, i, 0, s]) + u
                    ok = 0 <= j < S2 and (mode == 0 or j <= S2 - S1 + i)
                    if ok:
                        cols.append(j)
            for h in range(G):
                Dsum = sum(dO[b, i, h, c] * out[b, i, h, c] for c in range(Dv))
                lsum, mval = ssum[b, 0, i, h], smax[b, 0, i, h]
                for j in cols:
                    x = sum(q[b, i, h, c] * k[b, j, 0, c] for c in range(D))
                    x += sum(qr[b, i, h, c] * kr[b, j, 0, c] for c in range(Dr))
                    x *= scale
                    p = math.exp(x - mval) / lsum if lsum > 0 else 0.0
                    dp = sum(dO[b, i, h, c] * v[b, j, 0, c] for c in range(Dv))
                    ds = p * (dp - Dsum)
                    for c in range(D):
                        dq[b, i, h, c] += scale * ds * k[b, j, 0, c]
                        dk[b, j, 0, c] += scale * ds * q[b, i, h, c]
                    for c in range(Dr):
                        dqr[b, i, h, c] += scale * ds * kr[b, j, 0, c]
                        dkr[b, j, 0, c] += scale * ds * qr[b, i, h, c]
                    for c in range(Dv):
                        dv[b, j, 0, c] += p * dO[b, i, h, c]
    return dict(dq=dq, dk=dk, dv=dv, dq_rope=dqr, dk_rope=dkr)


@pytest.mark.parametrize("mode,bs", [(0, 1), (3, 2)])
def test_scalar_brute_force_with_duplicates(mode, bs):
    rng = np.random.default_rng(31 + mode)
    case, dO = _rand_case(rng, B=2, S1=3, S2=8, G=2, D=3, Dr=2, K=4, bs=bs, distinct=False)
    case["indices"][0, 1, 0, :2] = case["indices"][0, 1, 0, 2]   # force a duplicate
    out, smax, ssum = sfa_fwd(scale=0.45, sparse_block_size=bs, sparse_mode=mode, **case)
    g = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=0.45,
                sparse_block_size=bs, sparse_mode=mode, **case)
    r = _brute(case, dO, out, smax, ssum, 0.45, bs, mode)
    for n in r:
        np.testing.assert_allclose(g[n], r[n], rtol=1e-12, atol=1e-13, err_msg=n)


@pytest.mark.parametrize("mode", [0, 3])
def test_scalar_brute_force_blocks_across_edges(mode):
    """Block starts below 0 and blocks running past the sequence end: only the
    keys inside [0, kvlen) (and under the causal limit) count."""
    rng = np.random.default_rng(41 + mode)
    case, dO = _rand_case(rng, B=1, S1=3, S2=10, G=2, D=3, Dr=2, K=3, bs=4, distinct=False)
    case["indices"][0, :, 0, :] = np.array([[-1, 3, 8], [-3, 0, 7], [-4, 6, 9]])   # -4: no key >= 0
    out, smax, ssum = sfa_fwd(scale=0.5, sparse_block_size=4, sparse_mode=mode, **case)
    g = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=0.5,
                sparse_block_size=4, sparse_mode=mode, **case)
    r = _brute(case, dO, out, smax, ssum, 0.5, 4, mode)
    for n in r:
        np.testing.assert_allclose(g[n], r[n], rtol=1e-12, atol=1e-13, err_msg=n)


def test_sampled_rows_match_full():
    rng = np.random.default_rng(41)
    case, dO = _rand_case(rng, B=2, S1=5, S2=12, K=6)
    out, smax, ssum = sfa_fwd(scale=0.5, **case)
    full = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=0.5, **case)
    toks, keys = [0, 7, 9], [1, 5, 13, 23]
    part = sfa_bwd(d_out=dO, out=out, softmax_max=smax, softmax_sum=ssum, scale=0.5,
                   token_rows=toks, key_rows=keys, **case)
    fq = full["dq"].reshape(10, 2, -1); pq = part["dq"].reshape(10, 2, -1)
    np.testing.assert_allclose(pq[toks], fq[toks], rtol=1e-13)
    fk = full["dk"].reshape(24, -1); pk = part["dk"].reshape(24, -1)
    fv = full["dv"].reshape(24, -1); pv = part["dv"].reshape(24, -1)
    np.testing.assert_allclose(pk[keys], fk[keys], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(pv[keys], fv[keys], rtol=1e-13, atol=1e-15)


def test_sampled_forward_rows_match_full():
    """The forward restricted to some query tokens (token_rows, used by the
    full-size GPU checks) gives exactly the full forward's rows for those
    tokens, and NaN elsewhere so that a wrong row set cannot pass unnoticed."""
    rng = np.random.default_rng(43)
    for layout in ("BSND", "TND"):
        if layout == "BSND":
            case, _ = _rand_case(rng, B=2, S1=5, S2=12, K=6)
        else:
            case, _ = _rand_case(rng, layout="TND", aq=[4, 6], akv=[12, 9], K=6)
        out, smax, ssum = sfa_fwd(scale=0.5, **case)
        toks = [0, 4, 7, 9]
        po, pm, pl = sfa_fwd(scale=0.5, token_rows=toks, **case)
        T1 = 10
        fo, ffo = out.reshape(T1, -1), po.reshape(T1, -1)
        np.testing.assert_array_equal(ffo[toks], fo[toks])
        np.testing.assert_array_equal(pm.reshape(T1, -1)[toks], smax.reshape(T1, -1)[toks])
        np.testing.assert_array_equal(pl.reshape(T1, -1)[toks], ssum.reshape(T1, -1)[toks])
        rest = [t for t in range(T1) if t not in toks]
        assert np.all(np.isnan(ffo[rest])) and np.all(np.isnan(pl.reshape(T1, -1)[rest]))


def test_documentation_example_closed_form():
    with open(os.path.join(HERE, "golden", "sfag_doc_example.json")) as f:
        ex = json.load(f)
    c = np.frombuffer(np.uint16(ex["fp16_bits"]).tobytes(), dtype=np.float16)[0].astype(np.float64)
    assert c == 2.0 ** -24
    T1, N1, T2, D, Dr, K = (ex[n] for n in ("T1", "N1", "T2", "D", "Dr", "K"))
    q = np.full((T1, N1, D), c); k = np.full((T2, 1, D), c); v = np.full((T2, 1, D), c)
    qr = np.full((T1, N1, Dr), c); kr = np.full((T2, 1, Dr), c)
    dO = np.full((T1, N1, D), c); out = np.full((T1, N1, D), c)
    idx = np.arange(K).reshape(T1, 1, K)
    smax = np.full((1, T1, N1), ex["softmax_max"]); ssum = np.full((1, T1, N1), ex["softmax_sum"])
    g = sfa_bwd(q, k, v, idx, dO, out, smax, ssum, ex["scale"], ex["sparse_block_size"], ex["layout"],
                ex["sparse_mode"], np.array(ex["act_seq_q"]), np.array(ex["act_seq_kv"]), qr, kr)
    x = ex["scale"] * (D + Dr) * c * c
    dv_row = N1 * math.exp(x - ex["softmax_max"]) / ex["softmax_sum"] * c
    for n in ("dq", "dk", "dq_rope", "dk_rope"):
        assert np.all(g[n] == 0), n
    np.testing.assert_allclose(g["dv"], dv_row, rtol=1e-14)


def test_empty_query():
    q = np.zeros((0, 4, 8)); k = np.ones((5, 1, 8)); v = np.ones((5, 1, 8))
    idx = np.zeros((0, 1, 3), np.int64)
    g = sfa_bwd(q, k, v, idx, np.zeros((0, 4, 8)), np.zeros((0, 4, 8)), np.zeros((1, 0, 4)),
                np.zeros((1, 0, 4)), 0.5, 1, "TND", 0, np.array([0]), np.array([5]))
    assert g["dq"].shape == (0, 4, 8)
    assert np.all(g["dk"] == 0) and g["dk"].shape == (5, 1, 8)
