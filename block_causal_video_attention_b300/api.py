"""Python binding of the C ABI in include/od_attn.h (argument marshalling only).

Tensors are torch CUDA tensors: Q, O, dO, dQ [B,T,S,Hq,D] bf16; K, V, dK, dV
[B,T,S,Hkv,D] bf16; LSE [B,T,S,Hq] fp32.  Every call enqueues on the current torch
stream (or the `stream` given) and returns without synchronising.  All computation
happens in the CUDA library; there is no other implementation to fall back to.

    space_attn_fwd / time_attn_fwd            O, LSE (and O's residual with o_lo=True)
    space_attn_bwd / time_attn_bwd            dQ, dK, dV (fp32 copies with fp32_grads=True)
    *_fwd_packed / *_bwd_packed               Q, K, V from one [B,T,S,Hq+2Hkv,D] tensor
    space_attn_fwd_varlen / _bwd_varlen       per-timestep-block lengths (padded layout)
    time_attn_decode                          one rollout step over a ring-buffer KV cache
    get_device_status[_detail]                device-side timeouts since the last read
    selftest_expired_wait                     exercises the timeout path (no fault)
    debug_build / debug_library               route calls to the range-checked build
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_LIB_PATH = os.path.join(_PKG, "libod_attn.so")
_DEBUG_LIB_PATH = os.path.join(_PKG, "libod_attn_debug.so")
_HEADER = os.path.join(_ROOT, "include", "od_attn.h")
_lock = threading.Lock()
_lib = None
_debug_lib = None
_override = None   # set inside debug_build(): the binding's calls go to that library

# kernels one backward call launches: the K/V range kernel (with O_lo) or the Delta pass, the
# dQ pass, the dK/dV kernel
BWD_LAUNCHES = 3

STATUS = {0: "OD_OK", 1: "OD_ERR_INVALID_ARG", 2: "OD_ERR_UNSUPPORTED", 3: "OD_ERR_CUDA",
          4: "OD_ERR_TIMEOUT", 5: "OD_ERR_WORKSPACE", 6: "OD_ERR_RANGE"}


class ODError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__("%s: %s%s" % (what, STATUS.get(code, code),
                                       "" if _lib is None else
                                       " (%s)" % _lib.od_status_string(code).decode()))


def _declared_symbols():
    src = open(_HEADER).read()
    return re.findall(r"^\s*(?:od_status|size_t|const char\*)\s+(od_\w+)\s*\(", src, re.M)


EXPORTED_SYMBOLS = tuple(_declared_symbols()) if os.path.exists(_HEADER) else ()


def library_path() -> str:
    return _LIB_PATH


def library():
    """Load libod_attn.so (raises if it has not been built); inside debug_build(), the
    range-checked build instead."""
    global _lib
    if _override is not None:
        return _override
    with _lock:
        if _lib is None:
            _lib = _load(_LIB_PATH)
    return _lib


def debug_library():
    """Load libod_attn_debug.so, the build with device-side range checks (raises if it has
    not been built).  Same calls as library(); the binding's functions use library()."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _load(_DEBUG_LIB_PATH)
    return _debug_lib


@contextlib.contextmanager
def debug_build():
    """Within the block every call of this binding goes to libod_attn_debug.so (same
    results; device-side range checks reported as OD_ERR_RANGE by get_device_status)."""
    global _override
    prev = _override
    _override = debug_library()
    try:
        yield _override
    finally:
        _override = prev


def _load(path):
    if not os.path.exists(path):
        raise ODError(3, "%s is not built (run __graft_entry__.build())" % os.path.basename(path))
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fwd = [P] * 5 + [I] * 7 + [F, P]
    bwd = [P] * 9 + [I] * 7 + [F, P, Z, P]
    fwd_ex = [P] * 6 + [I] * 7 + [F, P]
    bwd_ex = [P] * 13 + [I] * 7 + [F, P, Z, P]
    for name, args in (("od_space_attn_fwd", fwd), ("od_time_attn_fwd", fwd),
                       ("od_space_attn_bwd", bwd), ("od_time_attn_bwd", bwd),
                       ("od_space_attn_fwd_ex", fwd_ex), ("od_time_attn_fwd_ex", fwd_ex),
                       ("od_space_attn_bwd_ex", bwd_ex), ("od_time_attn_bwd_ex", bwd_ex)):
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    fwdp = [P] * 4 + [I] * 7 + [F, P]
    bwdp = [P] * 9 + [I] * 7 + [F, P, Z, P]
    for name, args in (("od_space_attn_fwd_packed", fwdp), ("od_time_attn_fwd_packed", fwdp),
                       ("od_space_attn_bwd_packed", bwdp), ("od_time_attn_bwd_packed", bwdp)):
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.od_space_attn_fwd_varlen.argtypes = [P] * 7 + [I] * 7 + [F, P]
    lib.od_space_attn_fwd_varlen.restype = I
    lib.od_space_attn_bwd_varlen.argtypes = [P] * 14 + [I] * 7 + [F, P, Z, P]
    lib.od_space_attn_bwd_varlen.restype = I
    lib.od_time_attn_decode.argtypes = [P] * 7 + [I] * 6 + [ctypes.c_longlong, F, P]
    lib.od_time_attn_decode.restype = I
    lib.od_space_attn_bwd_static_ws.argtypes = [P] * 13 + [I] * 7 + [F, P]
    lib.od_space_attn_bwd_static_ws.restype = I
    lib.od_attn_bwd_workspace_bytes.argtypes = [I] * 7
    lib.od_attn_bwd_workspace_bytes.restype = Z
    lib.od_selftest_expired_wait.argtypes = [P]
    lib.od_selftest_expired_wait.restype = I
    lib.od_get_device_status.argtypes = [P]
    lib.od_get_device_status.restype = I
    lib.od_get_device_status_detail.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.od_get_device_status_detail.restype = I
    lib.od_status_string.argtypes = [I]
    lib.od_status_string.restype = ctypes.c_char_p
    lib.od_version.argtypes = []
    lib.od_version.restype = ctypes.c_char_p
    return lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError("%s must be a CUDA tensor" % name)
        if t.dtype != torch.bfloat16:
            raise TypeError("%s must be bfloat16" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
        if t.dim() != 5:
            raise ValueError("%s must be [B,T,S,H,D]" % name)
    if k.shape != v.shape or q.shape[:3] != k.shape[:3] or q.shape[4] != k.shape[4]:
        raise ValueError("shape mismatch: q %s, k %s, v %s" % (tuple(q.shape), tuple(k.shape),
                                                               tuple(v.shape)))
    B, T, S, Hq, D = q.shape
    return B, T, S, Hq, k.shape[3], D


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _residual_out(o_lo, shape, device):
    """o_lo: None (not requested), True (allocate) or a tensor to fill."""
    if o_lo is None or o_lo is False:
        return None
    if o_lo is True:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    if o_lo.shape != shape or o_lo.dtype != torch.bfloat16 or not o_lo.is_contiguous():
        raise ValueError("o_lo must be a contiguous bf16 tensor shaped like O")
    return o_lo


def _fwd(name, q, k, v, extra, scale, out, lse, o_lo, stream):
    B, T, S, Hq, Hkv, D = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, T, S, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if l.shape != (B, T, S, Hq) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,T,S,Hq]")
    r = _residual_out(o_lo, tuple(q.shape), q.device)
    if r is None:   # the plain call; the extended one only when the residual is wanted
        st = getattr(library(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, T, S, Hq,
                                      Hkv, D, int(extra), float(scale), _stream(stream))
    else:
        name += "_ex"
        st = getattr(library(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(r), B, T,
                                      S, Hq, Hkv, D, int(extra), float(scale), _stream(stream))
    if st:
        raise ODError(st, name)
    return (o, l) if r is None else (o, l, r)


def space_attn_fwd(q, k, v, agent_idx=-1, scale=None, out=None, lse=None, stream=None, o_lo=None):
    """Masked space attention forward -> (O bf16, LSE fp32) [, O_lo].

    o_lo=True (or a bf16 tensor shaped like O) also returns O's rounding residual
    bf16(O - o), which the backward can take to read Delta from memory."""
    return _fwd("od_space_attn_fwd", q, k, v, agent_idx, scale, out, lse, o_lo, stream)


def time_attn_fwd(q, k, v, window, scale=None, out=None, lse=None, stream=None, o_lo=None):
    """Sliding-window causal time attention forward -> (O bf16, LSE fp32) [, O_lo]."""
    return _fwd("od_time_attn_fwd", q, k, v, window, scale, out, lse, o_lo, stream)


def bwd_workspace_bytes(which, B, T, S, Hq, Hkv, D=64):
    return int(library().od_attn_bwd_workspace_bytes(int(which), B, T, S, Hq, Hkv, D))


def _bwd(name, which, q, k, v, o, lse, dout, extra, scale, fp32_grads, workspace, out, stream,
         o_lo=None):
    B, T, S, Hq, Hkv, D = _check_qkv(q, k, v)
    for nm, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("%s must be a contiguous bf16 CUDA tensor shaped like q" % nm)
    if lse.shape != (B, T, S, Hq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,T,S,Hq]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    f32 = (None, None, None)
    if fp32_grads:
        f32 = (torch.empty(q.shape, dtype=torch.float32, device=q.device),
               torch.empty(k.shape, dtype=torch.float32, device=q.device),
               torch.empty(v.shape, dtype=torch.float32, device=q.device))
    need = bwd_workspace_bytes(which, B, T, S, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if o_lo is not None and (o_lo.shape != q.shape or o_lo.dtype != torch.bfloat16
                             or not o_lo.is_contiguous()):
        raise ValueError("o_lo must be a contiguous bf16 tensor shaped like q")
    if o_lo is None and not fp32_grads:   # the plain call
        st = getattr(library(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                      _ptr(dq), _ptr(dk), _ptr(dv), B, T, S, Hq, Hkv, D,
                                      int(extra), float(scale), _ptr(workspace),
                                      ctypes.c_size_t(workspace.numel()), _stream(stream))
    else:
        name += "_ex"
        st = getattr(library(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_lo), _ptr(lse),
                                      _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(f32[0]),
                                      _ptr(f32[1]), _ptr(f32[2]), B, T, S, Hq, Hkv, D, int(extra),
                                      float(scale), _ptr(workspace),
                                      ctypes.c_size_t(workspace.numel()), _stream(stream))
    if st:
        raise ODError(st, name)
    if fp32_grads:
        return dq, dk, dv, f32
    return dq, dk, dv


def space_attn_bwd(q, k, v, o, lse, dout, agent_idx=-1, scale=None, fp32_grads=False,
                   workspace=None, out=None, stream=None, o_lo=None):
    """Space attention backward -> (dQ, dK, dV) bf16 [, (dQ, dK, dV) fp32].

    o_lo: the residual the forward returned (optional; Delta is recomputed without it)."""
    return _bwd("od_space_attn_bwd", 0, q, k, v, o, lse, dout, agent_idx, scale, fp32_grads,
                workspace, out, stream, o_lo)


def time_attn_bwd(q, k, v, o, lse, dout, window, scale=None, fp32_grads=False,
                  workspace=None, out=None, stream=None, o_lo=None):
    """Time attention backward -> (dQ, dK, dV) bf16 [, (dQ, dK, dV) fp32]."""
    return _bwd("od_time_attn_bwd", 1, q, k, v, o, lse, dout, window, scale, fp32_grads,
                workspace, out, stream, o_lo)


def _check_packed(qkv, num_q_heads):
    if not isinstance(qkv, torch.Tensor) or not qkv.is_cuda or qkv.dtype != torch.bfloat16:
        raise TypeError("qkv must be a bf16 CUDA tensor")
    if not qkv.is_contiguous() or qkv.dim() != 5:
        raise ValueError("qkv must be a contiguous [B,T,S,Hq+2*Hkv,D] tensor")
    B, T, S, P, D = qkv.shape
    Hq = int(num_q_heads)
    if Hq <= 0 or P <= Hq or (P - Hq) % 2:
        raise ValueError("qkv head count %d does not split as Hq=%d + 2*Hkv" % (P, Hq))
    return B, T, S, Hq, (P - Hq) // 2, D


def _fwd_packed(name, qkv, num_q_heads, extra, scale, out, lse, stream, o_lo=None):
    B, T, S, Hq, Hkv, D = _check_packed(qkv, num_q_heads)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty((B, T, S, Hq, D), dtype=torch.bfloat16, device=qkv.device) if out is None else out
    l = torch.empty((B, T, S, Hq), dtype=torch.float32, device=qkv.device) if lse is None else lse
    if o.shape != (B, T, S, Hq, D) or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor [B,T,S,Hq,D]")
    if l.shape != (B, T, S, Hq) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,T,S,Hq]")
    r = _residual_out(o_lo, (B, T, S, Hq, D), qkv.device)
    st = getattr(library(), name)(_ptr(qkv), _ptr(o), _ptr(l), _ptr(r), B, T, S, Hq, Hkv, D,
                                  int(extra), float(scale), _stream(stream))
    if st:
        raise ODError(st, name)
    return (o, l) if r is None else (o, l, r)


def space_attn_fwd_packed(qkv, num_q_heads, agent_idx=-1, scale=None, out=None, lse=None,
                          stream=None, o_lo=None):
    """Space attention forward reading Q, K, V from one packed [B,T,S,Hq+2*Hkv,D] tensor."""
    return _fwd_packed("od_space_attn_fwd_packed", qkv, num_q_heads, agent_idx, scale, out, lse,
                       stream, o_lo)


def time_attn_fwd_packed(qkv, num_q_heads, window, scale=None, out=None, lse=None, stream=None,
                         o_lo=None):
    """Time attention forward reading Q, K, V from one packed [B,T,S,Hq+2*Hkv,D] tensor."""
    return _fwd_packed("od_time_attn_fwd_packed", qkv, num_q_heads, window, scale, out, lse,
                       stream, o_lo)


def _bwd_packed(name, which, qkv, num_q_heads, o, lse, dout, extra, scale, fp32_grads,
                workspace, out, stream, o_lo=None):
    B, T, S, Hq, Hkv, D = _check_packed(qkv, num_q_heads)
    for nm, t in (("o", o), ("dout", dout)):
        if t.shape != (B, T, S, Hq, D) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 tensor [B,T,S,Hq,D]" % nm)
    if lse.shape != (B, T, S, Hq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,T,S,Hq]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dqkv = torch.empty_like(qkv) if out is None else out
    if dqkv.shape != qkv.shape or dqkv.dtype != torch.bfloat16 or not dqkv.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like qkv")
    f32 = (None, None, None)
    if fp32_grads:
        f32 = (torch.empty((B, T, S, Hq, D), dtype=torch.float32, device=qkv.device),
               torch.empty((B, T, S, Hkv, D), dtype=torch.float32, device=qkv.device),
               torch.empty((B, T, S, Hkv, D), dtype=torch.float32, device=qkv.device))
    need = bwd_workspace_bytes(which, B, T, S, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qkv.device)
    if o_lo is not None and (o_lo.shape != o.shape or o_lo.dtype != torch.bfloat16
                             or not o_lo.is_contiguous()):
        raise ValueError("o_lo must be a contiguous bf16 tensor shaped like o")
    st = getattr(library(), name)(_ptr(qkv), _ptr(o), _ptr(o_lo), _ptr(lse), _ptr(dout), _ptr(dqkv),
                                  _ptr(f32[0]), _ptr(f32[1]), _ptr(f32[2]), B, T, S, Hq, Hkv, D,
                                  int(extra), float(scale), _ptr(workspace),
                                  ctypes.c_size_t(workspace.numel()), _stream(stream))
    if st:
        raise ODError(st, name)
    if fp32_grads:
        return dqkv, f32
    return dqkv


def space_attn_bwd_packed(qkv, num_q_heads, o, lse, dout, agent_idx=-1, scale=None,
                          fp32_grads=False, workspace=None, out=None, stream=None, o_lo=None):
    """Space attention backward on packed QKV -> dQKV (packed like qkv) [, fp32 dQ, dK, dV]."""
    return _bwd_packed("od_space_attn_bwd_packed", 0, qkv, num_q_heads, o, lse, dout, agent_idx,
                       scale, fp32_grads, workspace, out, stream, o_lo)


def time_attn_bwd_packed(qkv, num_q_heads, o, lse, dout, window, scale=None, fp32_grads=False,
                         workspace=None, out=None, stream=None, o_lo=None):
    """Time attention backward on packed QKV -> dQKV (packed like qkv) [, fp32 dQ, dK, dV]."""
    return _bwd_packed("od_time_attn_bwd_packed", 1, qkv, num_q_heads, o, lse, dout, window,
                       scale, fp32_grads, workspace, out, stream, o_lo)


def _check_seqlen(seqlen, B, T, device):
    if not isinstance(seqlen, torch.Tensor) or seqlen.dtype != torch.int32 or not seqlen.is_cuda:
        raise TypeError("seqlen must be an int32 CUDA tensor of B*T block lengths")
    if seqlen.numel() != B * T or not seqlen.is_contiguous() or seqlen.data_ptr() % 16:
        raise ValueError("seqlen must be a contiguous, 16-byte aligned tensor of B*T lengths")


def space_attn_fwd_varlen(q, k, v, seqlen, agent_idx=-1, scale=None, out=None, lse=None,
                          stream=None, o_lo=None):
    """Space attention over variable-length timestep blocks on the padded [B,T,S,H,D] layout:
    block (b, t) holds its first seqlen[b*T+t] tokens.  Padding rows of the outputs are left
    as they were (allocate `out`/`lse` yourself to control them)."""
    B, T, S, Hq, Hkv, D = _check_qkv(q, k, v)
    _check_seqlen(seqlen, B, T, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.zeros_like(q) if out is None else out
    l = torch.zeros((B, T, S, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if l.shape != (B, T, S, Hq) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,T,S,Hq]")
    r = _residual_out(o_lo, tuple(q.shape), q.device)
    st = library().od_space_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(r),
                                            _ptr(seqlen), B, T, S, Hq, Hkv, D, int(agent_idx),
                                            float(scale), _stream(stream))
    if st:
        raise ODError(st, "od_space_attn_fwd_varlen")
    return (o, l) if r is None else (o, l, r)


def space_attn_bwd_varlen(q, k, v, o, lse, dout, seqlen, agent_idx=-1, scale=None,
                          fp32_grads=False, workspace=None, out=None, stream=None, o_lo=None):
    """Backward of space_attn_fwd_varlen -> (dQ, dK, dV) [, fp32 copies]; padding rows of
    the gradients are left as they were (zeros when allocated here)."""
    B, T, S, Hq, Hkv, D = _check_qkv(q, k, v)
    _check_seqlen(seqlen, B, T, q.device)
    for nm, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 tensor shaped like q" % nm)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    else:
        dq, dk, dv = out
    f32 = (None, None, None)
    if fp32_grads:
        f32 = (torch.zeros(q.shape, dtype=torch.float32, device=q.device),
               torch.zeros(k.shape, dtype=torch.float32, device=q.device),
               torch.zeros(v.shape, dtype=torch.float32, device=q.device))
    need = bwd_workspace_bytes(0, B, T, S, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = library().od_space_attn_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_lo), _ptr(lse), _ptr(dout), _ptr(seqlen),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(f32[0]), _ptr(f32[1]), _ptr(f32[2]), B, T, S, Hq, Hkv,
        D, int(agent_idx), float(scale), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream(stream))
    if st:
        raise ODError(st, "od_space_attn_bwd_varlen")
    if fp32_grads:
        return dq, dk, dv, f32
    return dq, dk, dv


def time_attn_decode(q, k_new, v_new, k_cache, v_cache, t, scale=None, out=None, lse=None,
                     stream=None):
    """One rollout step of time attention over a ring-buffer KV cache -> (O bf16, LSE fp32).

    q [B,S,Hq,D]; k_new, v_new [B,S,Hkv,D]; k_cache, v_cache [B,W,S,Hkv,D] (bf16, updated in
    place: the new frame goes to slot t mod W); t is the new frame's absolute index.  O is
    [B,S,Hq,D] bf16, LSE [B,S,Hq] fp32 -- the rows of time_attn_fwd at step t."""
    ts = (("q", q, 4), ("k_new", k_new, 4), ("v_new", v_new, 4), ("k_cache", k_cache, 5),
          ("v_cache", v_cache, 5))
    for name, x, nd in ts:
        if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.bfloat16:
            raise TypeError("%s must be a bf16 CUDA tensor" % name)
        if not x.is_contiguous() or x.dim() != nd:
            raise ValueError("%s must be a contiguous %d-D tensor" % (name, nd))
    B, S, Hq, D = q.shape
    Hkv = k_new.shape[2]
    W = k_cache.shape[1]
    if k_new.shape != (B, S, Hkv, D) or v_new.shape != k_new.shape or \
            k_cache.shape != (B, W, S, Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [B,S,Hq,D], k_new/v_new [B,S,Hkv,D], caches [B,W,S,Hkv,D]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, S, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if l.shape != (B, S, Hq) or l.dtype != torch.float32 or not l.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,S,Hq]")
    st = library().od_time_attn_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(o), _ptr(l), B, S, Hq, Hkv, D, W,
                                       int(t), float(scale), _stream(stream))
    if st:
        raise ODError(st, "od_time_attn_decode")
    return o, l


def selftest_expired_wait(stream=None) -> None:
    """Enqueue the failure-path self-test (a bounded wait that runs out after ~2 s)."""
    st = library().od_selftest_expired_wait(_stream(stream))
    if st:
        raise ODError(st, "od_selftest_expired_wait")


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status (0 = OK)."""
    return int(library().od_get_device_status(_stream(stream)))


def get_device_status_detail(stream=None):
    """(status, site word) -- the site word names the first expired wait (0 if none)."""
    w = ctypes.c_uint(0)
    st = library().od_get_device_status_detail(_stream(stream), ctypes.byref(w))
    return int(st), int(w.value)
