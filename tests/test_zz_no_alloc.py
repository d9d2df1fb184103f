"""The allocation-free backward entry point, sfa_grad_noalloc.

Some callers cannot call cudaMalloc (a plugin whose framework's memory pool
owns the device, code running under stream capture, a path that must not risk
the device-wide synchronisation of cudaMalloc/cudaFree); for them the library
offers a backward whose workspace is a static device array inside the
library.  These tests call it through the C ABI and check it against the
ordinary workspace-taking entry point, sfa_grad, on two calls in a row (the
scratch keeps the previous call's contents, so the second call checks that
everything that must start at zero is cleared), and check that a problem too
large for the scratch is refused with a clear error.

This file is collected last so that a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import sfa_grad_gb300 as sfa
from parity_util import OUT_NAMES, compare, gpu_call_kwargs, oracle_saved, to_cuda
from workloads import WORKLOADS, make_inputs, with_

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_twice():
    w = with_(WORKLOADS["tiny"], deterministic=False)
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    args = (dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], out.cuda(), smax.cuda(), ssum.cuda(),
            w.scale_value)
    ref = sfa.grad(*args, deterministic=False, **gpu_call_kwargs(w, dev))
    torch.cuda.synchronize()
    ref = [x.float().cpu().double().numpy() for x in ref]
    for call in range(2):
        got = sfa.grad_noalloc(*args, deterministic=False, **gpu_call_kwargs(w, dev))
        torch.cuda.synchronize()
        for n, a, b in zip(OUT_NAMES, got, ref):
            compare(f"call{call}/{n}", a, b, w.dtype)


def test_noalloc_refuses_oversize_problem():
    w = WORKLOADS["tiny"]          # deterministic: its workspace exceeds the static scratch
    inp = make_inputs(w)
    dev = {k: to_cuda(v) for k, v in inp.items()}
    p = sfa.make_params(dev["q"], dev["k"], dev["indices"], w.scale_value, deterministic=True)
    assert sfa.grad_workspace_size(p) > sfa.NOALLOC_SCRATCH_BYTES
    with pytest.raises(sfa.SfaError) as e:
        sfa.grad_noalloc(dev["q"], dev["k"], dev["v"], dev["indices"], dev["d_out"], dev["d_out"],
                         torch.zeros(1, 1, 16, 4, device="cuda"), torch.ones(1, 1, 16, 4, device="cuda"),
                         w.scale_value, deterministic=True, **gpu_call_kwargs(w, dev))
    assert e.value.code == sfa.SFA_ERR_SHAPE
    assert "static scratch" in str(e.value)
