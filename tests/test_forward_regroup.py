"""The companion forward scores each selected key once: P is formed relative
to the max of each group of 32 of a token's slots, then rescaled to the final
statistics (the per-token forward; the per-block forward groups by selected
block).  CPU checks of that arithmetic, independent of the GPU:

- in exact (fp64) arithmetic the regrouped P equals the plain softmax
  P = exp((s - max) * scale) / sum of the aclnnSparseFlashAttentionGrad page's
  阶段1 (the statistics' definition), and the merged group statistics equal
  the plain max and sum;
- with the three roundings to bf16 that the kernels apply (P~, the factor, and
  their product), out = P . V stays within a third of the bf16 parity
  tolerance and within twice the error of a single rounding of P.
"""
import numpy as np
import pytest
import torch

from parity_util import MAX_ABS, REL_TOL

GROUP = 32


def _case(seed, G=8, K=200, D=64, masked=0.2):
    rng = np.random.default_rng(seed)
    s = rng.normal(0.0, 24.0, size=(G, K))            # raw scores: q . k over 576 features
    valid = rng.random(K) >= masked
    valid[rng.integers(K)] = True
    v = rng.normal(size=(K, D))
    return s, valid, v, 1.0 / np.sqrt(576.0)


def _plain(s, valid, scale):
    x = np.where(valid, s, -np.inf)
    m = x.max(axis=1, keepdims=True)
    e = np.where(valid, np.exp((x - m) * scale), 0.0)
    return e / e.sum(axis=1, keepdims=True), m[:, 0], e.sum(axis=1)


def _group_stats(s, valid, scale):
    """Per group of 32 slots and head: (max of the raw score over valid keys, sum of exp)."""
    G, K = s.shape
    ng = (K + GROUP - 1) // GROUP
    mg = np.full((G, ng), -np.inf)
    lg = np.zeros((G, ng))
    for g in range(ng):
        sl = slice(g * GROUP, min(K, (g + 1) * GROUP))
        if valid[sl].any():
            x = np.where(valid[sl], s[:, sl], -np.inf)
            mg[:, g] = x.max(axis=1)
            lg[:, g] = np.where(valid[sl], np.exp((x - mg[:, g:g + 1]) * scale), 0.0).sum(axis=1)
    return mg, lg


def _merge(mg, lg, scale):
    """Online merge of the group pairs, rescaling the running sum when the max grows."""
    G, ng = mg.shape
    m = np.full(G, -np.inf)
    l = np.zeros(G)
    for g in range(ng):
        for h in range(G):
            if mg[h, g] == -np.inf:
                continue
            if mg[h, g] > m[h]:
                l[h] = l[h] * np.exp((m[h] - mg[h, g]) * scale) + lg[h, g]
                m[h] = mg[h, g]
            else:
                l[h] += lg[h, g] * np.exp((mg[h, g] - m[h]) * scale)
    return m, l


def _regrouped_p(s, valid, scale, rnd=None):
    """P from the group maxima and the merged statistics; rnd rounds a value to
    the input type (None: exact)."""
    rnd = rnd or (lambda a: a)
    G, K = s.shape
    mg, lg = _group_stats(s, valid, scale)
    m, l = _merge(mg, lg, scale)
    p = np.zeros((G, K))
    for g in range(mg.shape[1]):
        sl = slice(g * GROUP, min(K, (g + 1) * GROUP))
        pt = np.where(valid[sl], np.exp((s[:, sl] - mg[:, g:g + 1]) * scale), 0.0)      # P~, staged
        fac = np.where(mg[:, g] == -np.inf, 0.0, np.exp((mg[:, g] - m) * scale) / l)     # the group's factor
        p[:, sl] = rnd(rnd(pt) * rnd(fac)[:, None])                                     # one rounded multiply
    return p, m, l


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_regrouped_p_is_the_softmax(seed):
    s, valid, _, scale = _case(seed)
    p_ref, m_ref, l_ref = _plain(s, valid, scale)
    p, m, l = _regrouped_p(s, valid, scale)
    np.testing.assert_allclose(m, m_ref, rtol=0, atol=0)
    np.testing.assert_allclose(l, l_ref, rtol=1e-12)
    np.testing.assert_allclose(p, p_ref, rtol=1e-12, atol=1e-300)
    assert np.all(p[:, ~valid] == 0.0)


def test_group_without_valid_key_contributes_nothing():
    s, valid, _, scale = _case(3, K=160)
    valid[32:64] = False                                # one whole group masked
    p_ref, _, _ = _plain(s, valid, scale)
    p, _, _ = _regrouped_p(s, valid, scale)
    assert np.all(p[:, 32:64] == 0.0)
    np.testing.assert_allclose(p, p_ref, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("seed", [4, 5])
def test_three_bf16_roundings_stay_inside_the_tolerance(seed):
    s, valid, v, scale = _case(seed, K=2048, D=512, masked=0.0)
    v = _bf16(v)                                        # the inputs are in the input type on both sides
    p_ref, _, _ = _plain(s, valid, scale)
    out_ref = p_ref @ v
    p3, _, _ = _regrouped_p(s, valid, scale, rnd=_bf16)
    out3 = p3 @ v
    # the plain reading's single rounding of P, for comparison
    out1 = _bf16(p_ref) @ v
    rel3 = np.linalg.norm(out3 - out_ref) / np.linalg.norm(out_ref)
    rel1 = np.linalg.norm(out1 - out_ref) / np.linalg.norm(out_ref)
    # measured: about 2.5e-3 against 1.7e-3 for a single rounding of P
    assert rel3 <= REL_TOL["bf16"] / 3, rel3
    assert np.abs(out3 - out_ref).max() <= MAX_ABS / 3
    assert rel3 <= 2 * rel1, (rel3, rel1)
