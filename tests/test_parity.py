"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded bytes.  Index decode is compared bit for bit; float outputs with
the relative-Frobenius / max-abs tolerances of parity_util."""
import numpy as np
import pytest
import torch

import oracle
import sfa_grad_gb300 as sfa
from parity_util import OUT_NAMES, compare, gpu_call_kwargs, oracle_kwargs, oracle_saved, to_cuda
from workloads import WORKLOADS, make_inputs, small_workload, with_

pytestmark = pytest.mark.gpu

# Small cases that span several key tiles and a ragged tail.
SMALL = {
    "tiny": WORKLOADS["tiny"],
    "g16_ragged": small_workload(N1=16, S1=8, S2=512, K=300, seed=11),
    "g128_causal": small_workload(N1=128, S1=4, S2=1024, K=640, mode=3, seed=12),
    "g64_tnd": small_workload(name="tnd_small", layout="TND", B=3, N1=64, K=200, mode=3, index_kind="causal",
                              kv_extra=150, T1=8, act_q=(3, 0, 5), seed=13),
    "g16_block_fp16": small_workload(N1=16, S1=6, S2=1024, K=40, block_size=8, index_kind="block",
                                     dtype="fp16", std=0.5, seed=14),
    "g32_padding_dups": small_workload(N1=32, S1=5, S2=300, K=160, index_kind="random_any", seed=15),
    "g64_norope": small_workload(N1=64, S1=4, S2=700, K=256, Dr=0, seed=16),
    "g128_fp16": small_workload(N1=128, S1=3, S2=600, K=384, dtype="fp16", seed=17),
    # 128 heads and an even number of 128-key tiles (a ragged last tile; no rope part)
    "g128_pair_ragged": small_workload(N1=128, S1=5, S2=1024, K=500, mode=3, seed=39),
    "g128_pair_norope_fp16": small_workload(N1=128, S1=3, S2=700, K=256, Dr=0, dtype="fp16", seed=40),
    "g4_bs64": small_workload(N1=4, S1=4, S2=4096, K=5, block_size=64, index_kind="block", seed=18),
    # KV extent past 64 MB of fp32 key rows: key-side items run tile-group major
    "g64_wide_kv": small_workload(N1=64, S1=4, S2=16384, K=640, seed=23),
    # Blocks of >= 16 keys that many tokens select: the non-deterministic path
    # groups the (token, index) pairs by block start (key-major dK / dV)
    "g16_kvb_bs16": small_workload(N1=16, S1=64, S2=512, K=16, block_size=16, index_kind="block", seed=24),
    "g16_kvb_bs32_unaligned": small_workload(N1=16, S1=48, S2=640, K=8, block_size=32, seed=25),
    "g32_kvb_bs64_norope_fp16": small_workload(N1=32, S1=32, S2=512, K=4, block_size=64, index_kind="block", Dr=0,
                                               dtype="fp16", std=0.5, seed=26),
    "g12_kvb_tnd_causal": small_workload(name="tnd_kvb", layout="TND", B=2, N1=12, K=6, block_size=16, mode=3,
                                         index_kind="causal", kv_extra=64, T1=40, act_q=(24, 16), seed=27),
    "g16_kvb_padding_dups": small_workload(N1=16, S1=32, S2=256, K=8, block_size=16, index_kind="random_any", seed=28),
    "g64_kvb_bs32": small_workload(N1=64, S1=32, S2=512, K=8, block_size=32, index_kind="block", seed=38),
    # edge cases: a single index per token; a KV sequence shorter than one key tile, every key selected
    "g8_single_index": small_workload(N1=8, S1=6, S2=300, K=1, seed=29),
    "g32_short_kv_all": small_workload(N1=32, S1=5, S2=64, K=64, index_kind="all", seed=30),
    # blocks of 8 starting below 0 or running past the end, through the per-pair key side
    "g16_bs8_edges": small_workload(N1=16, S1=6, S2=200, K=10, block_size=8, index_kind="random_any", seed=31),
    # head counts that are not powers of two (the page's N1 list includes 3, 6,
    # 12, 24 and 48): padded to 16-row boxes and 64 or 128 MMA columns
    "g3_odd_heads": small_workload(N1=3, S1=5, S2=600, K=300, seed=33),
    "g6_causal": small_workload(N1=6, S1=7, S2=400, K=200, mode=3, seed=34),
    "g24_fp16": small_workload(N1=24, S1=4, S2=700, K=256, dtype="fp16", seed=35),
    "g48_bs16": small_workload(N1=48, S1=24, S2=512, K=12, block_size=16, index_kind="block", seed=36),
    "g12_tnd": small_workload(name="tnd_g12", layout="TND", B=2, N1=12, K=150, mode=3, index_kind="causal",
                              kv_extra=100, T1=9, act_q=(4, 5), seed=37),
    # one and two heads (the smallest N1 of the page's list) over many batches;
    # the TND lengths are random cuts of T1
    "g1_many_batches": small_workload(B=40, N1=1, S1=2, S2=256, K=96, seed=41),
    "g2_tnd_many_batches": small_workload(name="tnd_many", layout="TND", B=24, N1=2, K=64, mode=3,
                                          index_kind="causal", kv_extra=40, T1=60, seed=42),
    # ~5100 occurrences of each of two keys in one token chunk: the deterministic
    # sort takes its path for row segments longer than one warp sorts in shared memory
    "g4_pile_dups": small_workload(N1=4, S1=160, S2=512, K=128, index_kind="pile", std=0.15, seed=32),
}


def _run(w, det, inp=None, saved=None):
    inp = inp or make_inputs(w)
    out, smax, ssum = saved or oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    g = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
                 w.scale_value, deterministic=det, **gpu_call_kwargs(w, dev))
    torch.cuda.synchronize()
    return inp, (out, smax, ssum), g


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("det", [False, True])
def test_grad_small(name, det):
    w = SMALL[name]
    inp, (out, smax, ssum), g = _run(w, det)
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, **oracle_kwargs(w, inp))
    for n, x in zip(OUT_NAMES, g):
        if ref[n] is None:
            assert x is None
            continue
        compare(f"{name}/{n}", x, ref[n], w.dtype)


# Key and value given as one tensor (the documentation's own constraint,
# 约束说明: value identical to key): the library gathers each key row once.
SHARED_KV = {
    "g128_shared": small_workload(N1=128, S1=4, S2=1024, K=640, seed=19),
    "g64_shared_norope": small_workload(N1=64, S1=4, S2=700, K=300, Dr=0, seed=20),
    "g16_shared_block_fp16": small_workload(N1=16, S1=6, S2=1024, K=40, block_size=8, index_kind="block",
                                            dtype="fp16", std=0.5, seed=21),
    "g64_shared_tnd": small_workload(name="tnd_shared", layout="TND", B=3, N1=64, K=200, mode=3, index_kind="causal",
                                     kv_extra=150, T1=8, act_q=(3, 0, 5), seed=22),
}


@pytest.mark.parametrize("name", list(SHARED_KV))
@pytest.mark.parametrize("det", [False, True])
def test_grad_shared_kv(name, det):
    w = SHARED_KV[name]
    inp = make_inputs(w)
    inp["v"] = inp["k"]
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items() if k != "v"}
    dev["v"] = dev["k"]
    g = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
                 w.scale_value, deterministic=det, **gpu_call_kwargs(w, dev))
    torch.cuda.synchronize()
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, **oracle_kwargs(w, inp))
    for n, x in zip(OUT_NAMES, g):
        if ref[n] is None:
            assert x is None
            continue
        compare(f"{name}/{n}", x, ref[n], w.dtype)


@pytest.mark.parametrize("name", ["tiny", "g16_ragged", "g64_tnd", "g16_block_fp16", "g32_padding_dups"])
def test_decode_bit_exact(name):
    w = SMALL[name]
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    rows, _ = sfa.decode_keys(dev["q"], dev["k"], dev["indices"], sparse_block_size=w.block_size, layout=w.layout,
                              sparse_mode=w.mode, act_seq_q=kw.get("act_seq_q"), act_seq_kv=kw.get("act_seq_kv"),
                              has_rope=dev.get("q_rope") is not None)
    got = rows.cpu().numpy()
    prob = oracle.make_problem(**{k: v for k, v in oracle_kwargs(w, inp).items() if k not in ("sparse_block_size", "layout", "sparse_mode")},
                               block_size=w.block_size, layout=w.layout, mode=w.mode)
    exp = np.full_like(got, -1)
    for t in range(prob.T1):
        j, valid, kv0 = oracle.token_keys(prob, t)
        exp[t, valid] = kv0 + j[valid]
    assert np.array_equal(got, exp)


# the last seven: block indices that many tokens select, which the forward
# scores per block start (statistics and P) and multiplies by V per token
@pytest.mark.parametrize("name", ["tiny", "g128_causal", "g128_pair_ragged", "g128_pair_norope_fp16", "g64_tnd",
                                  "g1_many_batches", "g2_tnd_many_batches", "g3_odd_heads", "g6_causal", "g24_fp16",
                                  "g32_padding_dups", "g16_block_fp16", "g4_bs64", "g16_bs8_edges", "g64_norope",
                                  "g16_kvb_bs16",
                                  "g16_kvb_bs32_unaligned", "g32_kvb_bs64_norope_fp16", "g12_kvb_tnd_causal",
                                  "g16_kvb_padding_dups", "g64_kvb_bs32", "g48_bs16"])
def test_fwd_small(name):
    w = SMALL[name]
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    out, smax, ssum = sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, **kw)
    torch.cuda.synchronize()
    ro, rm, rl = oracle.sfa_fwd(**oracle_kwargs(w, inp))
    compare(f"{name}/out", out, ro, w.dtype)
    m = smax.cpu().double().numpy()
    fin = np.isfinite(rm)
    assert np.array_equal(np.isfinite(m), fin)
    np.testing.assert_allclose(m[fin], rm[fin], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(ssum.cpu().double().numpy(), rl, rtol=2e-4, atol=1e-6)


def test_deterministic_bitwise():
    w = SMALL["g128_causal"]
    inp, saved, g1 = _run(w, True)
    _, _, g2 = _run(w, True, inp, saved)
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_doc_example_closed_form_on_gpu():
    """The documentation page's example (fp16 0x0001 everywhere, constant stats 3.0):
    dS is exactly zero, so dQ, dK and the rope gradients are zero; dV is 16 *
    exp(x - 3) / 3 * 2^-24 per element, below half the smallest fp16 subnormal,
    so it rounds to zero as well."""
    T1, N1, T2, K = 1, 16, 2048, 2048
    c = torch.tensor([1], dtype=torch.int16).view(torch.float16)
    q = c.repeat(T1 * N1 * 512).reshape(T1, N1, 512).cuda()
    k = c.repeat(T2 * 512).reshape(T2, 1, 512).cuda()
    qr = c.repeat(T1 * N1 * 64).reshape(T1, N1, 64).cuda()
    kr = c.repeat(T2 * 64).reshape(T2, 1, 64).cuda()
    idx = torch.arange(K, dtype=torch.int32).reshape(T1, 1, K).cuda()
    st = torch.full((1, T1, N1), 3.0, device="cuda")
    aq = torch.tensor([1], dtype=torch.int32, device="cuda")
    akv = torch.tensor([2048], dtype=torch.int32, device="cuda")
    g = sfa.grad(q, k, k.clone(), idx, q.clone(), q.clone(), st, st.clone(), 0.088388, q_rope=qr, k_rope=kr,
                 layout="TND", act_seq_q=aq, act_seq_kv=akv)
    torch.cuda.synchronize()
    for x in g:
        assert torch.all(x == 0)


def test_tnd_bad_lengths_reported():
    w = SMALL["g64_tnd"]
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    kw["act_seq_kv"] = kw["act_seq_kv"] + 1   # no longer sums to T2
    ws = torch.empty(sfa.grad_workspace_size(sfa.make_params(dev["q"], dev["k"], dev["indices"], 1.0, layout="TND",
                                                             batch=3)), dtype=torch.uint8, device="cuda")
    g = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
                 w.scale_value, workspace=ws, **kw)
    assert sfa.read_device_error(ws) == 2
    for x in g:
        assert torch.all(x == 0)


# ------------------------------------------------------------------ full-size workloads, sampled rows
FULL = ["mla", "tnd", "block", "long"]


def _full_case(name, det):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    out, smax, ssum = sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, **kw)
    g = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out, smax, ssum, w.scale_value,
                 deterministic=det, **kw)
    torch.cuda.synchronize()
    return w, inp, dev, (out, smax, ssum), g


def _segments(w, inp):
    """Per query token: start row of its KV segment (global) and the segment length."""
    if w.layout == "TND":
        aq = inp["act_seq_q"].tolist()
        akv = inp["act_seq_kv"].tolist()
        starts = np.concatenate([[0], np.cumsum(akv)])[:-1]
        kv0 = np.repeat(starts, aq)
        kvlen = np.repeat(akv, aq)
    else:
        t = np.arange(w.B * w.S1)
        kv0 = (t // w.S1) * w.S2
        kvlen = np.full(t.shape, w.S2)
    return kv0.astype(np.int64), kvlen.astype(np.int64)


def _sample(w, inp, chunk, seed):
    """Query tokens and global key rows to check at full size: the first and
    last token, both sides of every token-chunk boundary (up to three
    boundaries), and random tokens; key rows that sampled tokens select at
    slots on both sides of the 128-slot tile and 512-slot tile-group
    boundaries (global rows: the token's segment start plus the index), plus
    random rows."""
    rng = np.random.default_rng(seed)
    T1 = inp["q"].reshape(-1, w.N1, 512).shape[0]
    T2 = inp["k"].reshape(-1, 512).shape[0]
    toks = {0, T1 - 1}
    bounds = list(range(chunk, T1, chunk))
    for b in bounds[:2] + bounds[-1:]:
        toks |= {b - 1, b}
    toks |= set(int(x) for x in rng.choice(T1, size=3, replace=False))
    toks = np.array(sorted(toks))
    kv0, kvlen = _segments(w, inp)
    idx = inp["indices"].reshape(T1, -1).numpy().astype(np.int64)
    keff = w.K * w.block_size
    keys = set()
    for t in toks[:4]:
        for slot in (0, 127, 128, 511, 512, keff - 1):
            if slot >= keff:
                continue
            j = idx[t, slot // w.block_size] + slot % w.block_size
            if 0 <= j < kvlen[t]:
                keys.add(int(kv0[t] + j))
    keys |= set(int(x) for x in rng.choice(T2, size=4, replace=False))
    return toks, np.array(sorted(keys))


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name, det):
    """The launch configuration bench.py times, on the full workloads, against
    the oracle on sampled tokens and key rows; in deterministic mode also
    bitwise equal across two calls."""
    w, inp, dev, (out, smax, ssum), g = _full_case(name, det)
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, layout=w.layout,
                        sparse_block_size=w.block_size, sparse_mode=w.mode, deterministic=det,
                        batch=w.B if w.layout == "TND" else None)
    chunk, _ = sfa.plan_info(p)
    T1 = inp["q"].reshape(-1, w.N1, 512).shape[0]
    T2 = inp["k"].reshape(-1, 512).shape[0]
    toks, keys = _sample(w, inp, chunk, seed=int(det))
    if det:
        g2 = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out, smax, ssum, w.scale_value,
                      deterministic=True, **gpu_call_kwargs(w, dev))
        torch.cuda.synchronize()
        for n, a, b in zip(OUT_NAMES, g, g2):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name}/{n} differs between two calls"
        del g2
    o_c, m_c, l_c = out.cpu(), smax.cpu(), ssum.cpu()
    # the companion forward on the sampled tokens
    ro, rm, rl = oracle.sfa_fwd(**oracle_kwargs(w, inp), token_rows=toks)
    compare(f"{name}/fwd_out", o_c.reshape(T1, w.N1, 512)[toks], ro.reshape(T1, w.N1, 512)[toks], w.dtype)
    np.testing.assert_allclose(l_c.reshape(T1, w.N1)[toks].double().numpy(), rl.reshape(T1, w.N1)[toks], rtol=2e-4)
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=o_c, softmax_max=m_c, softmax_sum=l_c, token_rows=toks,
                         key_rows=keys, **oracle_kwargs(w, inp))
    dq, dk, dv, dqr, dkr = g
    compare(f"{name}/dq", dq.reshape(T1, -1)[toks], ref["dq"].reshape(T1, -1)[toks], w.dtype)
    compare(f"{name}/dq_rope", dqr.reshape(T1, -1)[toks], ref["dq_rope"].reshape(T1, -1)[toks], w.dtype)
    compare(f"{name}/dk", dk.reshape(T2, -1)[keys], ref["dk"].reshape(T2, -1)[keys], w.dtype)
    compare(f"{name}/dv", dv.reshape(T2, -1)[keys], ref["dv"].reshape(T2, -1)[keys], w.dtype)
    compare(f"{name}/dk_rope", dkr.reshape(T2, -1)[keys], ref["dk_rope"].reshape(T2, -1)[keys], w.dtype)
    for x in g:
        assert torch.isfinite(x.float()).all()
    del g, dev, out, smax, ssum
    torch.cuda.empty_cache()


def test_full_size_shared_kv_sampled():
    """MLA shape with value = key: the shared-row path against the oracle on
    sampled tokens and key rows, and against the path that gathers value rows
    separately (the same tensor passed as two buffers) within tolerance."""
    w = WORKLOADS["mla"]
    inp = make_inputs(w)
    inp["v"] = inp["k"]
    dev = {k: to_cuda(v) for k, v in inp.items() if k != "v"}
    dev["v"] = dev["k"]
    kw = gpu_call_kwargs(w, dev)
    out, smax, ssum = sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, **kw)
    g = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out, smax, ssum, w.scale_value, **kw)
    g_sep = sfa.grad(dev["q"], dev["k"], dev["k"].clone(), dev["indices"], dev["d_out"], out, smax, ssum,
                     w.scale_value, **kw)
    torch.cuda.synchronize()
    T1, T2 = w.S1, w.S2
    rng = np.random.default_rng(1)
    toks = np.sort(rng.choice(T1, size=4, replace=False))
    keys = np.sort(rng.choice(T2, size=6, replace=False))
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out.cpu(), softmax_max=smax.cpu(), softmax_sum=ssum.cpu(),
                         token_rows=toks, key_rows=keys, **oracle_kwargs(w, inp))
    dq, dk, dv, dqr, dkr = g
    compare("shared/dq", dq.reshape(T1, -1)[toks], ref["dq"].reshape(T1, -1)[toks], w.dtype)
    compare("shared/dq_rope", dqr.reshape(T1, -1)[toks], ref["dq_rope"].reshape(T1, -1)[toks], w.dtype)
    compare("shared/dk", dk.reshape(T2, -1)[keys], ref["dk"].reshape(T2, -1)[keys], w.dtype)
    compare("shared/dv", dv.reshape(T2, -1)[keys], ref["dv"].reshape(T2, -1)[keys], w.dtype)
    compare("shared/dk_rope", dkr.reshape(T2, -1)[keys], ref["dk_rope"].reshape(T2, -1)[keys], w.dtype)
    for n, a, b in zip(OUT_NAMES, g, g_sep):
        compare(f"shared_vs_separate/{n}", a, b.float().cpu().double().numpy(), w.dtype)


def test_full_size_deterministic_vs_atomic():
    """MLA: the deterministic result agrees with the atomic one within tolerance."""
    w, inp, dev, (out, smax, ssum), g1 = _full_case("mla", True)
    g3 = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out, smax, ssum, w.scale_value,
                  deterministic=False, **gpu_call_kwargs(w, dev))
    torch.cuda.synchronize()
    for n, a, b in zip(OUT_NAMES, g1, g3):
        compare(f"mla/det_vs_atomic/{n}", a, b.float().cpu().double().numpy(), w.dtype)
