"""The allocation-free backward entry point, sfa_grad_noalloc.

Some callers cannot call cudaMalloc (a plugin whose framework's memory pool
owns the device, code running under stream capture, a path that must not risk
the device-wide synchronisation of cudaMalloc/cudaFree); for them the library
offers a backward whose workspace is a static device array inside the
library.  These tests call it through the C ABI and check it against the
ordinary workspace-taking entry point, sfa_grad, on two calls in a row for
each of the atomic, deterministic and key-major block plans (the scratch
keeps the previous call's contents, so every call after the first checks that
everything that must start at zero is cleared), check that the device error
word in the scratch is readable, and check that a problem too large for the
scratch is refused with a clear error.

This file is collected last so that a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import sfa_grad_gb300 as sfa
from parity_util import OUT_NAMES, compare, gpu_call_kwargs, oracle_saved, to_cuda
from workloads import WORKLOADS, make_inputs, small_workload, with_

pytestmark = pytest.mark.gpu


# Plans whose workspace fits the static scratch: the atomic path; the
# deterministic path (counting-sort bins, sorted entries and partial rows live
# in the scratch); the key-major block path (block bins, group lists).  Run in
# this order, each call finds the previous plan's data in the scratch.
PLANS = {
    "tiny_atomic": (with_(WORKLOADS["tiny"], deterministic=False), "kvq"),
    "g16_deterministic": (small_workload(N1=16, S1=8, S2=512, K=300, seed=11, deterministic=True), "det_sort"),
    "g16_kvb_bs16": (small_workload(N1=16, S1=64, S2=512, K=16, block_size=16, index_kind="block", seed=24), "kvb"),
}


@pytest.mark.parametrize("name", list(PLANS))
def test_noalloc_matches_workspace_entry_twice(name):
    w, launch = PLANS[name]
    det = w.deterministic
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, sparse_block_size=w.block_size,
                        deterministic=det)
    assert sfa.grad_workspace_size(p) <= sfa.NOALLOC_SCRATCH_BYTES
    assert launch in sfa.plan_names(p)
    args = (dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
            w.scale_value)
    ref = sfa.grad(*args, deterministic=det, **gpu_call_kwargs(w, dev))
    torch.cuda.synchronize()
    ref_np = [x.float().cpu().double().numpy() for x in ref]
    for call in range(2):
        got = sfa.grad_noalloc(*args, deterministic=det, **gpu_call_kwargs(w, dev))
        torch.cuda.synchronize()
        assert sfa.noalloc_read_device_error() == 0
        for n, a, b, r in zip(OUT_NAMES, got, ref_np, ref):
            compare(f"{name}/call{call}/{n}", a, b, w.dtype)
            if det:   # same plan, same fixed summation order
                assert torch.equal(a.view(torch.int16), r.view(torch.int16)), f"{name}/call{call}/{n}"


def test_noalloc_device_error_word():
    """TND lengths that do not sum to T2 mask every key and are reported in the
    static scratch's error word; reading it clears it."""
    w = small_workload(name="tnd_small", layout="TND", B=3, N1=64, K=200, mode=3, index_kind="causal",
                       kv_extra=150, T1=8, act_q=(3, 0, 5), seed=13)
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    args = (dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
            w.scale_value)
    bad = dict(kw, act_seq_kv=kw["act_seq_kv"] + 1)
    g = sfa.grad_noalloc(*args, **bad)
    assert sfa.noalloc_read_device_error() == 2
    for x in g:
        assert torch.all(x == 0)
    assert sfa.noalloc_read_device_error() == 0
    sfa.grad_noalloc(*args, **kw)
    assert sfa.noalloc_read_device_error() == 0


def test_noalloc_refuses_oversize_problem():
    # deterministic, 64 tokens x 2048 keys: the partial rows alone exceed the static scratch
    w = small_workload(N1=16, S1=64, S2=4096, K=2048, seed=38, deterministic=True)
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, deterministic=True)
    assert sfa.grad_workspace_size(p) > sfa.NOALLOC_SCRATCH_BYTES
    st = torch.zeros(1, 1, 64, 16, device="cuda")
    with pytest.raises(sfa.SfaError) as e:
        sfa.grad_noalloc(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], dev["d_out"], st, st + 1,
                         w.scale_value, deterministic=True, **gpu_call_kwargs(w, dev))
    assert e.value.code == sfa.SFA_ERR_SHAPE
    assert "static scratch" in str(e.value)
