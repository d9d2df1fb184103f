"""The kernels' timeout path, run on the GPU without faulting it.

Every pipeline wait inside the kernels gives up after a wall-clock limit; the
kernel then raises its abort flag, records SFA_DEVERR_TIMEOUT in the
workspace's error word, waits for the copies and MMAs it already issued and
returns.  The limit is per call (sfa_params.wait_limit_us), so a call with a
limit of one microsecond makes the first wait that is not satisfied at once
run out, in every tensor-core kernel of the call.  The tests check that such a
call returns and completes, reports the timeout, leaves the context usable,
and that the next ordinary call on the same workspace matches the oracle.
"""
import time

import pytest
import torch

import oracle
import sfa_grad_gb300 as sfa
from parity_util import OUT_NAMES, compare, gpu_call_kwargs, oracle_kwargs, oracle_saved, to_cuda
from workloads import small_workload

pytestmark = pytest.mark.gpu

TIMEOUT = 1

# one plan per family of tensor-core kernels: score + combined key/query side;
# deterministic (counting sort, partial rows, fixed-order sums); key-major
# blocks, atomic and deterministic
CASES = {
    "atomic": (small_workload(N1=128, S1=4, S2=1024, K=640, mode=3, seed=12), False),
    "deterministic": (small_workload(N1=64, S1=6, S2=700, K=300, seed=16), True),
    "kvb": (small_workload(N1=16, S1=64, S2=512, K=16, block_size=16, index_kind="block", seed=24), False),
    "kvb_deterministic": (small_workload(N1=16, S1=64, S2=512, K=16, block_size=16, index_kind="block", seed=24),
                          True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_wait_timeout_then_recovery(name):
    w, det = CASES[name]
    inp = make_inputs_cached(w)
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    args = (dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
            w.scale_value)
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, sparse_block_size=w.block_size,
                        deterministic=det)
    ws = torch.empty(sfa.grad_workspace_size(p), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sfa.grad(*args, deterministic=det, workspace=ws, wait_limit_us=1, **kw)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert sfa.read_device_error(ws) == TIMEOUT
    # the wind-down waits only for work already issued: far below its own 2 s limit
    assert took < 1.0, f"timed-out call took {took:.2f} s"
    # same workspace, ordinary limit: complete and correct
    g = sfa.grad(*args, deterministic=det, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert sfa.read_device_error(ws) == 0
    ref = oracle.sfa_bwd(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, **oracle_kwargs(w, inp))
    for n, x in zip(OUT_NAMES, g):
        compare(f"{name}/{n}", x, ref[n], w.dtype)


# the per-token forward (one score pass, P.V with the per-group rescale) and
# the per-block one (scores per block start, O with the features on the MMA's
# rows)
@pytest.mark.parametrize("name", ["atomic", "kvb"])
def test_forward_wait_timeout_then_recovery(name):
    w, _ = CASES[name]
    inp = make_inputs_cached(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    kw = gpu_call_kwargs(w, dev)
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, sparse_mode=w.mode,
                        sparse_block_size=w.block_size)
    ws = torch.empty(max(sfa.fwd_workspace_size(p), 256), dtype=torch.uint8, device="cuda")
    sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, workspace=ws, wait_limit_us=1, **kw)
    torch.cuda.synchronize()
    assert sfa.read_device_error(ws) == TIMEOUT
    o, m, l = sfa.fwd(dev["q"], dev["k"], dev["v"], dev["indices"], w.scale_value, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert sfa.read_device_error(ws) == 0
    ro, _, _ = oracle.sfa_fwd(**oracle_kwargs(w, inp))
    compare(f"fwd_{name}/out", o, ro, w.dtype)


_CACHE = {}


def make_inputs_cached(w):
    from workloads import make_inputs
    if w not in _CACHE:
        _CACHE[w] = make_inputs(w)
    return _CACHE[w]
