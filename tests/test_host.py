"""GPU parity of sfa_grad_host, the backward from host buffers: the library
copies the inputs to the device chunk by chunk, overlapping the copies with
the kernels, and copies the results back.  Its outputs are compared with the
fp64 oracle (same tolerances as the device-buffer path), checked bitwise
reproducible with deterministic = 1, and the empty query zeroes the key-side
outputs."""
import pytest
import torch

import oracle
import sfa_grad_gb300 as sfa
from parity_util import OUT_NAMES, compare, oracle_kwargs, oracle_saved
from workloads import make_inputs, small_workload

pytestmark = pytest.mark.gpu

# Chunk schedules (first chunk 128 tokens, growing, ragged last chunk): 200
# tokens run as 128, 72; 600 as 128, 160, 200, 112; 150 as 128, 22; 16 tokens
# as one chunk.
CASES = {
    "g16_chunks_ragged": small_workload(N1=16, S1=200, S2=512, K=128, seed=41),
    "g8_tnd_causal": small_workload(name="tnd_host", layout="TND", B=3, N1=8, K=96, mode=3, index_kind="causal",
                                    kv_extra=100, T1=150, act_q=(70, 0, 80), seed=42),
    "g16_kvb_fp16": small_workload(N1=16, S1=150, S2=512, K=8, block_size=16, index_kind="block", dtype="fp16",
                                   std=0.5, seed=43),
    "g4_ramp_norope": small_workload(N1=4, S1=600, S2=256, K=64, Dr=0, seed=44),
    "tiny_one_chunk": small_workload(N1=4, S1=16, S2=2048, K=1024, seed=45),
}


def _host(inp, out, smax, ssum, w, det, shared_kv=False):
    def pin(x):
        return None if x is None else x.contiguous().pin_memory()
    h = {k: pin(v) for k, v in inp.items()}
    if shared_kv:
        h["v"] = h["k"]
    kw = dict(q_rope=h.get("q_rope"), k_rope=h.get("k_rope"), sparse_block_size=w.block_size, layout=w.layout,
              sparse_mode=w.mode)
    if w.layout == "TND":
        kw["act_seq_q"] = h["act_seq_q"]
        kw["act_seq_kv"] = h["act_seq_kv"]
    g = sfa.grad_host(h["q"], h["k"], h["v"], h["indices"], h["d_out"], pin(out), pin(smax), pin(ssum),
                      w.scale_value, deterministic=det, **kw)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("det", [False, True])
def test_grad_host(name, det):
    w = CASES[name]
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    g = _host(inp, out, smax, ssum, w, det)
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, **oracle_kwargs(w, inp))
    for n, x in zip(OUT_NAMES, g):
        if ref[n] is None:
            assert x is None
            continue
        assert not x.is_cuda
        compare(f"host/{name}/{n}", x, ref[n], w.dtype)


def test_grad_host_shared_kv():
    w = small_workload(N1=32, S1=130, S2=700, K=256, seed=46)
    inp = make_inputs(w)
    inp["v"] = inp["k"]
    out, smax, ssum = oracle_saved(w, inp)
    g = _host(inp, out, smax, ssum, w, False, shared_kv=True)
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, **oracle_kwargs(w, inp))
    for n, x in zip(OUT_NAMES, g):
        compare(f"host/shared/{n}", x, ref[n], w.dtype)


def test_grad_host_deterministic_bitwise():
    w = CASES["g16_chunks_ragged"]
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    g1 = _host(inp, out, smax, ssum, w, True)
    g2 = _host(inp, out, smax, ssum, w, True)
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_grad_host_empty_query():
    w = small_workload(N1=4, S1=0, S2=300, K=16, seed=47)
    q = torch.zeros(1, 0, 4, 512, dtype=torch.bfloat16).pin_memory()
    k = torch.randn(1, 300, 1, 512).to(torch.bfloat16).pin_memory()
    qr = torch.zeros(1, 0, 4, 64, dtype=torch.bfloat16).pin_memory()
    kr = torch.randn(1, 300, 1, 64).to(torch.bfloat16).pin_memory()
    idx = torch.zeros(1, 0, 1, 16, dtype=torch.int32).pin_memory()
    st = torch.zeros(1, 1, 0, 4).pin_memory()
    outs = (torch.empty(q.shape, dtype=q.dtype).pin_memory(), torch.full(k.shape, 7.0, dtype=k.dtype).pin_memory(),
            torch.full(k.shape, 7.0, dtype=k.dtype).pin_memory(), torch.empty(qr.shape, dtype=qr.dtype).pin_memory(),
            torch.full(kr.shape, 7.0, dtype=kr.dtype).pin_memory())
    sfa.grad_host(q, k, k.clone(), idx, q, q, st, st, w.scale_value, q_rope=qr, k_rope=kr, outputs=outs)
    torch.cuda.synchronize()
    for x in outs[1:3] + outs[4:]:
        assert torch.all(x == 0)


def test_full_size_host_sampled():
    """The MLA workload through sfa_grad_host, as bench.py times it end to end
    (pinned host buffers, ramped chunks): dQ on sampled tokens and dK / dV /
    dKRope on sampled key rows against the oracle, and every output against
    the device-buffer call within tolerance."""
    import numpy as np
    from parity_util import gpu_call_kwargs, to_cuda
    from workloads import WORKLOADS
    w = WORKLOADS["mla"]
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    out, smax, ssum = sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, **kw)
    g_dev = sfa.grad(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out, smax, ssum, w.scale_value, **kw)
    torch.cuda.synchronize()
    o_c, m_c, l_c = out.cpu(), smax.cpu(), ssum.cpu()
    g = _host(inp, o_c, m_c, l_c, w, False)
    T1, T2 = w.S1, w.S2
    rng = np.random.default_rng(2)
    toks = np.sort(rng.choice(T1, size=4, replace=False))
    keys = np.sort(rng.choice(T2, size=6, replace=False))
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=o_c, softmax_max=m_c, softmax_sum=l_c, token_rows=toks,
                         key_rows=keys, **oracle_kwargs(w, inp))
    dq, dk, dv, dqr, dkr = g
    compare("host_full/dq", dq.reshape(T1, -1)[toks], ref["dq"].reshape(T1, -1)[toks], w.dtype)
    compare("host_full/dq_rope", dqr.reshape(T1, -1)[toks], ref["dq_rope"].reshape(T1, -1)[toks], w.dtype)
    compare("host_full/dk", dk.reshape(T2, -1)[keys], ref["dk"].reshape(T2, -1)[keys], w.dtype)
    compare("host_full/dv", dv.reshape(T2, -1)[keys], ref["dv"].reshape(T2, -1)[keys], w.dtype)
    compare("host_full/dk_rope", dkr.reshape(T2, -1)[keys], ref["dk_rope"].reshape(T2, -1)[keys], w.dtype)
    for n, a, b in zip(OUT_NAMES, g, g_dev):
        compare(f"host_vs_device/{n}", a, b.float().cpu().double().numpy(), w.dtype)
