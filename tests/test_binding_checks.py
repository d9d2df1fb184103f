"""The binding's argument checks (CPU): every input set the parity tests and
the bench build passes them, and tensors whose size, dtype or device do not
match the problem are refused with ValueError before the library is called
(a short buffer would otherwise be read or written past its end)."""
import pytest
import torch

import sfa_grad_gb300 as sfa
from parity_util import oracle_saved
from workloads import WORKLOADS, make_inputs, small_workload

CASES = {
    "tiny": WORKLOADS["tiny"],
    "g64_tnd": small_workload(name="tnd_small", layout="TND", B=3, N1=64, K=200, mode=3, index_kind="causal",
                              kv_extra=150, T1=8, act_q=(3, 0, 5), seed=13),
    "g16_block_fp16": small_workload(N1=16, S1=6, S2=1024, K=40, block_size=8, index_kind="block", dtype="fp16",
                                     std=0.5, seed=14),
    "g64_norope": small_workload(N1=64, S1=4, S2=700, K=256, Dr=0, seed=16),
    "g4_bs64_two_batches": small_workload(B=2, N1=4, S1=4, S2=512, K=5, block_size=64, index_kind="block", seed=18),
}


def _args(w, inp, saved):
    out, smax, ssum = saved
    p = sfa.make_params(inp["q"], inp["k"], inp["indices"], w.scale_value, layout=w.layout,
                        sparse_block_size=w.block_size, sparse_mode=w.mode, has_rope=inp["q_rope"] is not None,
                        batch=inp["act_seq_q"].numel() if w.layout == "TND" else None)
    kw = dict(d_out=inp["d_out"], out=out, softmax_max=smax, softmax_sum=ssum, q_rope=inp["q_rope"],
              k_rope=inp["k_rope"], act_seq_q=inp.get("act_seq_q"), act_seq_kv=inp.get("act_seq_kv"))
    return p, kw


@pytest.mark.parametrize("name", list(CASES))
def test_valid_inputs_pass(name):
    w = CASES[name]
    inp = make_inputs(w)
    saved = oracle_saved(w, inp)
    p, kw = _args(w, inp, saved)
    outs = (torch.empty_like(inp["q"]), torch.empty_like(inp["k"]), torch.empty_like(inp["v"]),
            torch.empty_like(inp["q_rope"]) if inp["q_rope"] is not None else None,
            torch.empty_like(inp["k_rope"]) if inp["k_rope"] is not None else None)
    sfa.check_tensors(p, inp["q"], inp["k"], inp["v"], inp["indices"], outputs=outs, **kw)
    # value = key, and the forward's inputs alone
    sfa.check_tensors(p, inp["q"], inp["k"], inp["k"], inp["indices"], **kw)
    sfa.check_tensors(p, inp["q"], inp["k"], inp["v"], inp["indices"], backward=False, q_rope=kw["q_rope"],
                      k_rope=kw["k_rope"], act_seq_q=kw["act_seq_q"], act_seq_kv=kw["act_seq_kv"])


def test_mismatches_are_refused():
    w = CASES["tiny"]
    inp = make_inputs(w)
    saved = oracle_saved(w, inp)
    p, kw = _args(w, inp, saved)
    q, k, v, idx = inp["q"], inp["k"], inp["v"], inp["indices"]

    def refused(match, **over):
        a = dict(kw)
        a.update(over)
        with pytest.raises(ValueError, match=match):
            sfa.check_tensors(p, q, k, v, a.pop("indices", idx), **a)

    refused("d_out: dtype", d_out=kw["d_out"].to(torch.float16))
    refused("out: .* elements", out=kw["out"][..., :256])
    refused("softmax_max: dtype", softmax_max=kw["softmax_max"].double())
    refused("softmax_sum: .* elements", softmax_sum=kw["softmax_sum"][:, :, :-1])
    refused("indices: .* elements", indices=idx[:, :-1])
    refused("indices: dtype", indices=idx.long())
    refused("k_rope is required", k_rope=None)
    refused("d_out is required", d_out=None)
    with pytest.raises(ValueError, match="v: .* elements"):
        sfa.check_tensors(p, q, k, v[:, :-1], idx, **kw)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)[:, :-1], torch.empty_like(inp["q_rope"]),
            torch.empty_like(inp["k_rope"]))
    with pytest.raises(ValueError, match="dv: .* elements"):
        sfa.check_tensors(p, q, k, v, idx, outputs=outs, backward=False, q_rope=kw["q_rope"], k_rope=kw["k_rope"])
    # rope tensors must come as a pair
    p0 = sfa.make_params(q, k, idx, w.scale_value, has_rope=False)
    with pytest.raises(ValueError, match="k_rope given without q_rope"):
        sfa.check_tensors(p0, q, k, v, idx, backward=False, k_rope=kw["k_rope"])


def test_tnd_lengths_required():
    w = CASES["g64_tnd"]
    inp = make_inputs(w)
    saved = oracle_saved(w, inp)
    p, kw = _args(w, inp, saved)
    kw["act_seq_kv"] = None
    with pytest.raises(ValueError, match="act_seq_kv is required"):
        sfa.check_tensors(p, inp["q"], inp["k"], inp["v"], inp["indices"], **kw)


def test_grad_host_refuses_before_any_device_work():
    """grad_host checks its inputs before it allocates pinned outputs or a
    device workspace, so the mistake surfaces as ValueError even without a GPU."""
    w = CASES["tiny"]
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    with pytest.raises(ValueError, match="d_out: dtype"):
        sfa.grad_host(inp["q"], inp["k"], inp["v"], inp["indices"], inp["d_out"].to(torch.float16), out, smax, ssum,
                      w.scale_value, q_rope=inp["q_rope"], k_rope=inp["k_rope"])


class _Recorder:
    """Stands in for the library and for torch's device switch: records the
    device each call made current and the library calls made inside it."""

    def __init__(self):
        self.log = []
        self.current = None

    def on(self, device):
        rec = self

        class Ctx:
            def __enter__(self):
                rec.log.append(("enter", str(device)))
                rec.current = str(device)

            def __exit__(self, *a):
                rec.log.append(("exit", str(device)))
                rec.current = None
        return Ctx()

    def __getattr__(self, name):
        if not name.startswith("sfa_"):
            raise AttributeError(name)

        def call(*a):
            self.log.append((name, self.current))
            return 0
        return call


def test_library_calls_run_with_the_tensors_device_current(monkeypatch):
    """The C ABI launches on the current device (and sfa_grad_noalloc uses
    that device's static scratch), so the binding makes the tensors' device
    current around every library call."""
    w = CASES["tiny"]
    inp = make_inputs(w)
    out, smax, ssum = oracle_saved(w, inp)
    rec = _Recorder()
    monkeypatch.setattr(sfa, "lib", lambda: rec)
    monkeypatch.setattr(sfa, "_on", rec.on)
    monkeypatch.setattr(sfa, "_ptr", lambda t: None if t is None else 16)
    monkeypatch.setattr(sfa, "_stream", lambda s: 0)
    monkeypatch.setattr(sfa, "grad_workspace_size", lambda p: 256)
    monkeypatch.setattr(sfa, "fwd_workspace_size", lambda p: 256)
    dev = str(inp["q"].device)
    args = (inp["q"], inp["k"], inp["v"], inp["indices"], inp["d_out"], out, smax, ssum, w.scale_value)
    kw = dict(q_rope=inp["q_rope"], k_rope=inp["k_rope"])
    sfa.grad_noalloc(*args, **kw)
    sfa.grad(*args, workspace=torch.empty(256, dtype=torch.uint8), **kw)
    sfa.fwd(inp["q"], inp["k"], inp["v"], inp["indices"], w.scale_value, workspace=torch.empty(256, dtype=torch.uint8),
            **kw)
    calls = [e for e in rec.log if e[0].startswith("sfa_")]
    assert [c[0] for c in calls] == ["sfa_grad_noalloc", "sfa_grad", "sfa_fwd"]
    assert all(c[1] == dev for c in calls), rec.log
    # a caller's workspace on another device than the tensors is refused
    with pytest.raises(ValueError, match="workspace is on"):
        sfa._workspace(256, torch.device("cuda", 0), torch.empty(256, dtype=torch.uint8))
