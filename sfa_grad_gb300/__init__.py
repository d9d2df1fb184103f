"""Python binding of libsfa.so (include/sfa_grad.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
builds the parameter block from tensor shapes, allocates outputs/workspace
with torch when the caller does not pass them, and calls the C ABI on the
current CUDA stream.  There is no fallback: if the library is missing or a
tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsfa.so")

SFA_OK = 0
SFA_ERR_NULLPTR = 161001
SFA_ERR_PARAM_INVALID = 161002
SFA_ERR_RUNTIME = 361001
SFA_ERR_SHAPE = 561002

LAYOUTS = {"BSND": 0, "TND": 1}
DTYPES = {torch.bfloat16: 0, torch.float16: 1}

EXPORTS = ("sfa_grad_workspace_size", "sfa_grad", "sfa_grad_profile", "sfa_grad_plan_info", "sfa_grad_plan_names",
           "sfa_fwd_workspace_size", "sfa_fwd", "sfa_decode_keys", "sfa_read_device_error", "sfa_status_string",
           "sfa_last_error_message", "sfa_grad_noalloc", "sfa_noalloc_read_device_error",
           "sfa_grad_host_workspace_size", "sfa_grad_host")


class SfaParams(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("B", ctypes.c_int64), ("S1", ctypes.c_int64), ("S2", ctypes.c_int64),
        ("T1", ctypes.c_int64), ("T2", ctypes.c_int64),
        ("N1", ctypes.c_int64), ("N2", ctypes.c_int64), ("D", ctypes.c_int64),
        ("Dr", ctypes.c_int64), ("K", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("sparse_block_size", ctypes.c_int64), ("sparse_mode", ctypes.c_int64),
        ("deterministic", ctypes.c_int32), ("wait_limit_us", ctypes.c_int32),
    ]


class SfaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code in (SFA_ERR_RUNTIME, SFA_ERR_SHAPE):
            detail = " - " + lib().sfa_last_error_message().decode()
        super().__init__(f"{where}: {status_string(code)} ({code}){detail}")


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libsfa.so (built in-tree by sfa_grad_gb300.build); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m sfa_grad_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(SfaParams)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    L.sfa_grad_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    L.sfa_fwd_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    L.sfa_grad.argtypes = [P] + [vp] * 18 + [sz, vp]
    L.sfa_grad_profile.argtypes = [P] + [vp] * 18 + [sz, vp, ctypes.POINTER(vp), ctypes.c_int32]
    L.sfa_grad_plan_info.argtypes = [P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    L.sfa_grad_plan_names.argtypes = [P, ctypes.POINTER(ctypes.c_char_p), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    L.sfa_grad_noalloc.argtypes = [P] + [vp] * 17 + [vp]
    L.sfa_grad_host_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    L.sfa_grad_host.argtypes = [P] + [vp] * 18 + [sz, vp]
    L.sfa_fwd.argtypes = [P] + [vp] * 12 + [sz, vp]
    L.sfa_decode_keys.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    L.sfa_read_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    L.sfa_noalloc_read_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    L.sfa_last_error_message.argtypes = []
    L.sfa_last_error_message.restype = ctypes.c_char_p
    L.sfa_status_string.argtypes = [ctypes.c_int32]
    L.sfa_status_string.restype = ctypes.c_char_p
    for name in ("sfa_grad_workspace_size", "sfa_fwd_workspace_size", "sfa_grad", "sfa_grad_profile",
                 "sfa_grad_plan_info", "sfa_grad_plan_names", "sfa_fwd", "sfa_decode_keys", "sfa_read_device_error",
                 "sfa_grad_noalloc", "sfa_noalloc_read_device_error", "sfa_grad_host_workspace_size",
                 "sfa_grad_host"):
        getattr(L, name).restype = ctypes.c_int32
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().sfa_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != SFA_OK:
        raise SfaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def make_params(q: torch.Tensor, k: torch.Tensor, indices: torch.Tensor, scale: float, *, layout: str = "BSND",
                sparse_block_size: int = 1, sparse_mode: int = 0, deterministic: bool = False,
                has_rope: bool = True, batch: Optional[int] = None, wait_limit_us: int = 0) -> SfaParams:
    p = SfaParams()
    p.layout = LAYOUTS[layout.upper()]
    if q.dtype not in DTYPES:
        raise ValueError("q must be bfloat16 or float16")
    p.dtype = DTYPES[q.dtype]
    if p.layout == 0:
        p.B, p.S1, p.N1, p.D = q.shape
        p.S2, p.N2 = k.shape[1], k.shape[2]
        p.T1, p.T2 = p.B * p.S1, p.B * p.S2
    else:
        p.T1, p.N1, p.D = q.shape
        p.T2, p.N2 = k.shape[0], k.shape[1]
        p.B = int(batch) if batch is not None else 1
    p.Dr = 64 if has_rope else 0
    p.K = indices.shape[-1]
    p.scale = float(scale)
    p.sparse_block_size = int(sparse_block_size)
    p.sparse_mode = int(sparse_mode)
    p.deterministic = 1 if deterministic else 0
    p.wait_limit_us = int(wait_limit_us)
    return p


def check_tensors(p: SfaParams, q, k, v, indices, *, d_out=None, out=None, softmax_max=None, softmax_sum=None,
                  q_rope=None, k_rope=None, act_seq_q=None, act_seq_kv=None, outputs=None, backward=True):
    """Checks every tensor's element count and dtype against the problem `p`
    describes (from the shapes of q, k and indices), so that no buffer the
    library reads or writes is shorter than it assumes, and that all tensors
    share q's device.  Raises ValueError; called by grad, grad_host,
    grad_noalloc and fwd before the library is."""
    dt = q.dtype
    T1, T2, G, K = int(p.T1), int(p.T2), int(p.N1), int(p.K)
    rope = p.Dr == 64

    def need(name, t, numel, dtype):
        if t is None:
            raise ValueError(f"{name} is required")
        if t.dtype != dtype:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if t.numel() != numel:
            raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")

    need("q", q, T1 * G * 512, dt)
    need("k", k, T2 * 512, dt)
    need("v", v, T2 * 512, dt)
    need("indices", indices, T1 * K, torch.int32)
    if rope:
        need("q_rope", q_rope, T1 * G * 64, dt)
        need("k_rope", k_rope, T2 * 64, dt)
    elif k_rope is not None:
        raise ValueError("k_rope given without q_rope")
    if p.layout == 1:
        need("act_seq_q", act_seq_q, int(p.B), torch.int32)
        need("act_seq_kv", act_seq_kv, int(p.B), torch.int32)
    if backward:
        need("d_out", d_out, T1 * G * 512, dt)
        need("out", out, T1 * G * 512, dt)
        need("softmax_max", softmax_max, T1 * G, torch.float32)
        need("softmax_sum", softmax_sum, T1 * G, torch.float32)
    if outputs is not None:
        dq, dk, dv, dqr, dkr = outputs
        need("dq", dq, T1 * G * 512, dt)
        need("dk", dk, T2 * 512, dt)
        need("dv", dv, T2 * 512, dt)
        if rope:
            need("dq_rope", dqr, T1 * G * 64, dt)
            need("dk_rope", dkr, T2 * 64, dt)


def grad_workspace_size(p: SfaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().sfa_grad_workspace_size(ctypes.byref(p), ctypes.byref(n)), "sfa_grad_workspace_size")
    return n.value


def fwd_workspace_size(p: SfaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().sfa_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)), "sfa_fwd_workspace_size")
    return n.value


def plan_info(p: SfaParams):
    """(tokens per staging chunk, kernel launches per call) of sfa_grad."""
    c, n = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().sfa_grad_plan_info(ctypes.byref(p), ctypes.byref(c), ctypes.byref(n)), "sfa_grad_plan_info")
    return c.value, n.value


def plan_names(p: SfaParams) -> list:
    """Names of the kernels one sfa_grad call launches, in launch order."""
    n = ctypes.c_int32(0)
    _check(lib().sfa_grad_plan_names(ctypes.byref(p), None, 0, ctypes.byref(n)), "sfa_grad_plan_names")
    buf = (ctypes.c_char_p * max(n.value, 1))()
    _check(lib().sfa_grad_plan_names(ctypes.byref(p), buf, n.value, ctypes.byref(n)), "sfa_grad_plan_names")
    return [buf[i].decode() for i in range(n.value)]


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _on(device):
    """Makes `device` current for the library call: the C ABI launches on the
    current device (and sfa_grad_noalloc uses that device's static scratch),
    so a call on tensors of another device must switch to it first."""
    return torch.cuda.device(device)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        if workspace.device != torch.device(device):
            raise ValueError(f"workspace is on {workspace.device}, the call runs on {device}")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def grad(q, k, v, indices, d_out, out, softmax_max, softmax_sum, scale, *, q_rope=None, k_rope=None,
         sparse_block_size=1, layout="BSND", sparse_mode=0, deterministic=False, act_seq_q=None, act_seq_kv=None,
         outputs=None, workspace=None, stream=None, events=None, wait_limit_us=0):
    """sfa_grad on torch CUDA tensors; returns (dq, dk, dv, dq_rope, dk_rope).

    events: optional list of torch.cuda.Event; when given, sfa_grad_profile
    records events[0] before the first launch and events[i] after launch i.
    wait_limit_us: the kernels' wait limit (0: the library's default); a test
    hook for the timeout path."""
    has_rope = q_rope is not None
    batch = act_seq_q.numel() if act_seq_q is not None else None
    p = make_params(q, k, indices, scale, layout=layout, sparse_block_size=sparse_block_size,
                    sparse_mode=sparse_mode, deterministic=deterministic, has_rope=has_rope, batch=batch,
                    wait_limit_us=wait_limit_us)
    check_tensors(p, q, k, v, indices, d_out=d_out, out=out, softmax_max=softmax_max, softmax_sum=softmax_sum,
                  q_rope=q_rope, k_rope=k_rope, act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    if outputs is None:
        outputs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                   torch.empty_like(q_rope) if has_rope else None, torch.empty_like(k_rope) if has_rope else None)
    check_tensors(p, q, k, v, indices, outputs=outputs, backward=False, q_rope=q_rope, k_rope=k_rope,
                  act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    dq, dk, dv, dqr, dkr = outputs
    with _on(q.device):
        ws = _workspace(grad_workspace_size(p), q.device, workspace)
        args = (ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(indices), _ptr(d_out), _ptr(out), _ptr(softmax_max),
                _ptr(softmax_sum), _ptr(act_seq_q), _ptr(act_seq_kv), _ptr(q_rope), _ptr(k_rope), _ptr(dq), _ptr(dk),
                _ptr(dv), _ptr(dqr), _ptr(dkr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
        if events:
            handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
            _check(lib().sfa_grad_profile(*args, handles, len(events)), "sfa_grad_profile")
        else:
            _check(lib().sfa_grad(*args), "sfa_grad")
    return dq, dk, dv, dqr, dkr


NOALLOC_SCRATCH_BYTES = 64 << 20


def grad_noalloc(q, k, v, indices, d_out, out, softmax_max, softmax_sum, scale, *, q_rope=None, k_rope=None,
                 sparse_block_size=1, layout="BSND", sparse_mode=0, deterministic=False, act_seq_q=None,
                 act_seq_kv=None, outputs=None, stream=None):
    """sfa_grad_noalloc: the backward with its workspace taken from the
    library's static device scratch (for callers that cannot allocate device
    memory); outputs are allocated here unless passed in."""
    has_rope = q_rope is not None
    batch = act_seq_q.numel() if act_seq_q is not None else None
    p = make_params(q, k, indices, scale, layout=layout, sparse_block_size=sparse_block_size,
                    sparse_mode=sparse_mode, deterministic=deterministic, has_rope=has_rope, batch=batch)
    check_tensors(p, q, k, v, indices, d_out=d_out, out=out, softmax_max=softmax_max, softmax_sum=softmax_sum,
                  q_rope=q_rope, k_rope=k_rope, act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    if outputs is None:
        outputs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                   torch.empty_like(q_rope) if has_rope else None, torch.empty_like(k_rope) if has_rope else None)
    check_tensors(p, q, k, v, indices, outputs=outputs, backward=False, q_rope=q_rope, k_rope=k_rope,
                  act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    dq, dk, dv, dqr, dkr = outputs
    with _on(q.device):
        rc = lib().sfa_grad_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(indices), _ptr(d_out), _ptr(out),
                                    _ptr(softmax_max), _ptr(softmax_sum), _ptr(act_seq_q), _ptr(act_seq_kv),
                                    _ptr(q_rope), _ptr(k_rope), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dqr), _ptr(dkr),
                                    _stream(stream))
    _check(rc, "sfa_grad_noalloc")
    return dq, dk, dv, dqr, dkr


def noalloc_read_device_error(device=None, stream=None) -> int:
    """sfa_noalloc_read_device_error: reads and clears the device error word
    (SFA_DEVERR_*) of sfa_grad_noalloc's static scratch on `device` (default:
    the current device), after synchronising `stream`."""
    code = ctypes.c_int32(0)
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    with _on(dev):
        _check(lib().sfa_noalloc_read_device_error(_stream(stream), ctypes.byref(code)),
               "sfa_noalloc_read_device_error")
    return code.value


def grad_host_workspace_size(p: SfaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().sfa_grad_host_workspace_size(ctypes.byref(p), ctypes.byref(n)), "sfa_grad_host_workspace_size")
    return n.value


def _hptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("sfa_grad_host takes host (CPU) tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def grad_host(q, k, v, indices, d_out, out, softmax_max, softmax_sum, scale, *, q_rope=None, k_rope=None,
              sparse_block_size=1, layout="BSND", sparse_mode=0, deterministic=False, act_seq_q=None,
              act_seq_kv=None, outputs=None, workspace=None, device=None, stream=None):
    """sfa_grad_host on host (CPU, preferably pinned) tensors: the library
    copies them to the device chunk by chunk, overlapping the copies with the
    kernels, and copies the results back into `outputs` (pinned CPU tensors
    allocated here unless passed in).  The results are complete once the
    stream has been synchronised.  `workspace` is a device tensor of at least
    grad_host_workspace_size bytes (allocated on `device`, default the
    current CUDA device, unless passed in).  Returns (dq, dk, dv, dq_rope,
    dk_rope)."""
    has_rope = q_rope is not None
    batch = act_seq_q.numel() if act_seq_q is not None else None
    p = make_params(q, k, indices, scale, layout=layout, sparse_block_size=sparse_block_size,
                    sparse_mode=sparse_mode, deterministic=deterministic, has_rope=has_rope, batch=batch)
    check_tensors(p, q, k, v, indices, d_out=d_out, out=out, softmax_max=softmax_max, softmax_sum=softmax_sum,
                  q_rope=q_rope, k_rope=k_rope, act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    if outputs is None:
        def pinned(t):
            return torch.empty(t.shape, dtype=t.dtype).pin_memory()
        outputs = (pinned(q), pinned(k), pinned(v), pinned(q_rope) if has_rope else None,
                   pinned(k_rope) if has_rope else None)
    check_tensors(p, q, k, v, indices, outputs=outputs, backward=False, q_rope=q_rope, k_rope=k_rope,
                  act_seq_q=act_seq_q, act_seq_kv=act_seq_kv)
    dq, dk, dv, dqr, dkr = outputs
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    with _on(dev):
        ws = _workspace(grad_host_workspace_size(p), dev, workspace)
        rc = lib().sfa_grad_host(ctypes.byref(p), _hptr(q), _hptr(k), _hptr(v), _hptr(indices), _hptr(d_out),
                                 _hptr(out), _hptr(softmax_max), _hptr(softmax_sum), _hptr(act_seq_q),
                                 _hptr(act_seq_kv), _hptr(q_rope), _hptr(k_rope), _hptr(dq), _hptr(dk), _hptr(dv),
                                 _hptr(dqr), _hptr(dkr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "sfa_grad_host")
    return dq, dk, dv, dqr, dkr


def fwd(q, k, v, indices, scale, *, q_rope=None, k_rope=None, sparse_block_size=1, layout="BSND", sparse_mode=0,
        act_seq_q=None, act_seq_kv=None, workspace=None, stream=None, wait_limit_us=0):
    """sfa_fwd on torch CUDA tensors; returns (out, softmax_max, softmax_sum)."""
    has_rope = q_rope is not None
    batch = act_seq_q.numel() if act_seq_q is not None else None
    p = make_params(q, k, indices, scale, layout=layout, sparse_block_size=sparse_block_size,
                    sparse_mode=sparse_mode, has_rope=has_rope, batch=batch, wait_limit_us=wait_limit_us)
    check_tensors(p, q, k, v, indices, q_rope=q_rope, k_rope=k_rope, act_seq_q=act_seq_q, act_seq_kv=act_seq_kv,
                  backward=False)
    out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if p.layout == 0:
        st_shape = (p.B, 1, p.S1, p.N1)
    else:
        st_shape = (1, p.T1, p.N1)
    smax = torch.empty(st_shape, dtype=torch.float32, device=q.device)
    ssum = torch.empty(st_shape, dtype=torch.float32, device=q.device)
    with _on(q.device):
        ws = _workspace(fwd_workspace_size(p), q.device, workspace)
        rc = lib().sfa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(indices), _ptr(act_seq_q),
                           _ptr(act_seq_kv), _ptr(q_rope), _ptr(k_rope), _ptr(out), _ptr(smax), _ptr(ssum), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "sfa_fwd")
    return out, smax, ssum


def decode_keys(q, k, indices, *, sparse_block_size=1, layout="BSND", sparse_mode=0, act_seq_q=None,
                act_seq_kv=None, has_rope=True, workspace=None, stream=None):
    """sfa_decode_keys: the global kv row (or -1) of every expanded slot, int32 (T1, K*bs)."""
    batch = act_seq_q.numel() if act_seq_q is not None else None
    p = make_params(q, k, indices, 1.0, layout=layout, sparse_block_size=sparse_block_size,
                    sparse_mode=sparse_mode, has_rope=has_rope, batch=batch)
    rows = torch.empty((p.T1, p.K * p.sparse_block_size), dtype=torch.int32, device=q.device)
    with _on(q.device):
        ws = _workspace(grad_workspace_size(p), q.device, workspace)
        rc = lib().sfa_decode_keys(ctypes.byref(p), _ptr(indices), _ptr(act_seq_q), _ptr(act_seq_kv), _ptr(rows),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "sfa_decode_keys")
    return rows, ws


def read_device_error(workspace: torch.Tensor, stream=None) -> int:
    code = ctypes.c_int32(0)
    with _on(workspace.device):
        _check(lib().sfa_read_device_error(_ptr(workspace), _stream(stream), ctypes.byref(code)),
               "sfa_read_device_error")
    return code.value
