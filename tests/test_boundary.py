"""C-ABI boundary on the CPU: the library loads, exports every function the
public header declares, and its host-side validation returns the documented
status codes without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sfa():
    from sfa_grad_gb300.build import build
    build()
    import sfa_grad_gb300 as m
    m.lib()
    return m


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(sfa_[a-z_]+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(sfa):
    names = _declared()
    assert {"sfa_grad", "sfa_grad_workspace_size", "sfa_fwd", "sfa_fwd_workspace_size"} <= names
    L = sfa.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(sfa.EXPORTS) <= names


def _p(sfa, **kw):
    p = sfa.SfaParams()
    base = dict(layout=0, dtype=0, B=1, S1=16, S2=2048, T1=0, T2=0, N1=4, N2=1, D=512, Dr=64, K=1024,
                scale=1 / 24, sparse_block_size=1, sparse_mode=0, deterministic=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


def _ws(sfa, p):
    n = ctypes.c_size_t(0)
    return sfa.lib().sfa_grad_workspace_size(ctypes.byref(p), ctypes.byref(n)), n.value


def test_workspace_size_ok(sfa):
    rc, n = _ws(sfa, _p(sfa))
    assert rc == 0 and n > 16 * 2048 * 4


def test_null_pointers(sfa):
    n = ctypes.c_size_t(0)
    assert sfa.lib().sfa_grad_workspace_size(None, ctypes.byref(n)) == sfa.SFA_ERR_NULLPTR
    p = _p(sfa)
    assert sfa.lib().sfa_grad_workspace_size(ctypes.byref(p), None) == sfa.SFA_ERR_NULLPTR
    # dk missing: rejected before any device work
    args = [None] * 18
    assert sfa.lib().sfa_grad(ctypes.byref(p), *args, 0, None) == sfa.SFA_ERR_NULLPTR


@pytest.mark.parametrize("field,value", [("dtype", 2), ("layout", 5), ("deterministic", 3), ("wait_limit_us", -1)])
def test_param_invalid(sfa, field, value):
    rc, _ = _ws(sfa, _p(sfa, **{field: value}))
    assert rc == sfa.SFA_ERR_PARAM_INVALID


@pytest.mark.parametrize("field,value", [
    ("N2", 2), ("D", 256), ("Dr", 32), ("N1", 0), ("N1", 129), ("sparse_mode", 1), ("sparse_mode", 4),
    ("sparse_block_size", 3), ("sparse_block_size", 128), ("K", 0), ("S1", -1), ("B", 0),
    ("scale", float("nan")),
])
def test_shape_errors(sfa, field, value):
    rc, _ = _ws(sfa, _p(sfa, **{field: value}))
    assert rc == sfa.SFA_ERR_SHAPE


def test_deterministic_large_keff(sfa):
    # the deterministic reduction sorts per kv row, not per token: no key-count limit
    assert _ws(sfa, _p(sfa, deterministic=1, K=8192))[0] == 0
    assert _ws(sfa, _p(sfa, deterministic=1, K=8192, sparse_block_size=8))[0] == 0


def test_workspace_too_small_and_empty_query(sfa):
    p = _p(sfa)
    # empty query (S1 = 0) with null outputs is still a null-pointer error...
    p0 = _p(sfa, S1=0)
    assert sfa.lib().sfa_grad(ctypes.byref(p0), *([None] * 18), 0, None) == sfa.SFA_ERR_NULLPTR
    # ...and a short workspace is rejected before any launch
    fake = ctypes.c_void_p(16)
    args = [fake] * 12 + [fake] * 5 + [fake]
    rc = sfa.lib().sfa_grad(ctypes.byref(p), *args, 8, None)
    assert rc == sfa.SFA_ERR_PARAM_INVALID


def test_tnd_workspace_independent_of_lengths(sfa):
    a = _ws(sfa, _p(sfa, layout=1, B=4, T1=16384, T2=32768, N1=64, K=2048, sparse_mode=3))
    assert a[0] == 0 and a[1] > 32768 * 1088 * 4


def test_status_strings(sfa):
    for c in (0, 161001, 161002, 361001, 561002):
        assert sfa.status_string(c).startswith("SFA_")


def test_plan_names(sfa):
    """The launch sequence a call plans, as sfa_grad_plan_names lists it: one
    chunk of the combined kernel for an MLA shape; the grouped key-major block
    path for block indices that many tokens select; the fixed-order path when
    deterministic; a batch prefix first for TND."""
    mla = sfa.plan_names(_p(sfa, S1=4096, S2=4096, N1=128, K=2048))
    assert mla == ["meta", "dsum", "rowtab", "sdp", "kvq", "cast"]
    assert sfa.plan_info(_p(sfa, S1=4096, S2=4096, N1=128, K=2048))[1] == len(mla)
    blk = sfa.plan_names(_p(sfa, dtype=1, B=2, S1=8192, S2=32768, N1=16, K=64, sparse_block_size=64))
    chunk = ["blk_count", "blk_scan", "blk_scatter", "sdpb", "kvb", "dqb"]
    assert blk[:2] == ["meta", "dsum"] and blk[-1] == "cast"
    ctok, nl = sfa.plan_info(_p(sfa, dtype=1, B=2, S1=8192, S2=32768, N1=16, K=64, sparse_block_size=64))
    nchunks = (2 * 8192 + ctok - 1) // ctok
    assert len(blk) == nl == 3 + len(chunk) * nchunks
    assert blk[2:2 + len(chunk)] == chunk
    # few selections per key row, or bs < 16, or more than 64 heads: per-pair path
    assert "kvb" not in sfa.plan_names(_p(sfa, S1=4, S2=4096, N1=16, K=5, sparse_block_size=64))
    assert "kvb" not in sfa.plan_names(_p(sfa, S1=2048, S2=4096, N1=16, K=64, sparse_block_size=8))
    assert "kvb" not in sfa.plan_names(_p(sfa, S1=2048, S2=4096, N1=128, K=64, sparse_block_size=64))
    det = sfa.plan_names(_p(sfa, deterministic=1))
    assert det == ["meta", "dsum", "rowtab", "sdp", "det_count", "det_scan", "det_scatter", "det_sort",
                   "det_sort_long", "kvq", "det_reduce", "cast"]
    # deterministic block indices: the key-major path with sorted groups, one
    # kvb launch per block-start residue
    bdet = sfa.plan_names(_p(sfa, dtype=1, B=2, S1=8192, S2=32768, N1=16, K=64, sparse_block_size=64,
                             deterministic=1))
    cdet = (["blk_count", "blk_scan", "blk_scatter", "blk_sort", "blk_sort_long", "sdpb"] + ["kvb"] * 64
            + ["dqb"])
    assert bdet[2:2 + len(cdet)] == cdet and "det_reduce" not in bdet
    assert sfa.plan_info(_p(sfa, dtype=1, B=2, S1=8192, S2=32768, N1=16, K=64, sparse_block_size=64,
                            deterministic=1))[0] == ctok
    tnd = sfa.plan_names(_p(sfa, layout=1, B=4, T1=16384, T2=32768, N1=64, K=2048, sparse_mode=3))
    assert tnd[0] == "batch_prefix" and "kvq" in tnd
    assert sfa.plan_names(_p(sfa, S1=0)) == []


def test_host_entry_validation(sfa):
    """sfa_grad_host: its workspace holds the backward's plus device copies of
    every input and output; missing pointers and a short workspace are
    rejected before any CUDA call."""
    p = _p(sfa, S1=4096, S2=4096, N1=128, K=2048)
    n = ctypes.c_size_t(0)
    assert sfa.lib().sfa_grad_host_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    t1, t2, g = 4096, 4096, 128
    io = (3 * t1 * g * 512 + t1 * g * 64) * 2 + t1 * 2048 * 4 + 2 * t1 * g * 4 + (2 * t2 * 512 + t2 * 64) * 2 \
        + (t1 * g * 576 + t2 * 1088) * 2
    assert n.value >= io
    # sfa_grad's workspace (same staging chunk) plus the copies, each 256-byte aligned
    assert 0 <= n.value - io - _ws(sfa, p)[1] < 17 * 256
    assert sfa.lib().sfa_grad_host_workspace_size(None, ctypes.byref(n)) == sfa.SFA_ERR_NULLPTR
    assert sfa.lib().sfa_grad_host(ctypes.byref(p), *([None] * 18), 0, None) == sfa.SFA_ERR_NULLPTR
    fake = ctypes.c_void_p(16)
    rc = sfa.lib().sfa_grad_host(ctypes.byref(p), *([fake] * 18), 8, None)
    assert rc == sfa.SFA_ERR_PARAM_INVALID
    bad = _p(sfa, N2=2)
    assert sfa.lib().sfa_grad_host(ctypes.byref(bad), *([fake] * 18), 1 << 40, None) == sfa.SFA_ERR_SHAPE
