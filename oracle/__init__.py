"""fp64 CPU oracle for masked space attention and windowed causal time attention
(training forward/backward, the rollout decode step, and space attention over
variable-length timestep blocks as per-block calls of the fixed-length operator).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this package; the CUDA library never calls it, and it shares
no code with the CUDA path.  The arithmetic lives in od_oracle.c (plain loops,
double precision); this module compiles it with gcc and marshals numpy arrays.

Every function takes float64 arrays in the library's layouts
(Q/O/dO/dQ [B,T,S,Hq,D], K/V/dK/dV [B,T,S,Hkv,D], LSE [B,T,S,Hq]; the decode step
takes one frame [B,S,H,D] and a ring-buffer cache [B,W,S,Hkv,D]) and returns
float64 results.  Use `from_bf16` to widen the bf16 inputs exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "od_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile od_oracle.c into liboracle.so (gcc -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            fwd = [dp, dp, dp, dp, dp, i, i, i, i, i, i, i, ctypes.c_double, i]
            bwd = [dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, ctypes.c_double, i]
            for name, args in (("oracle_space_fwd", fwd), ("oracle_time_fwd", fwd),
                               ("oracle_space_bwd", bwd), ("oracle_time_bwd", bwd)):
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            lib.oracle_time_decode.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                               ctypes.c_longlong, ctypes.c_double]
            lib.oracle_time_decode.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = [i]
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def num_threads(requested: int = 0) -> int:
    return _load().oracle_num_threads(int(requested))


def from_bf16(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prep(q, k, v):
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    if q.ndim != 5 or k.shape != v.shape or q.shape[:3] != k.shape[:3] or q.shape[4] != k.shape[4]:
        raise ValueError("expected Q [B,T,S,Hq,D] and K, V [B,T,S,Hkv,D]")
    return q, k, v


def _fwd(name, q, k, v, extra, scale, nthreads):
    q, k, v = _prep(q, k, v)
    B, T, S, Hq, D = q.shape
    Hkv = k.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros_like(q)
    lse = np.zeros((B, T, S, Hq), dtype=np.float64)
    rc = getattr(_load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                B, T, S, Hq, Hkv, D, int(extra), float(scale), int(nthreads))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def _bwd(name, q, k, v, dout, extra, scale, nthreads):
    q, k, v = _prep(q, k, v)
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    if dout.shape != q.shape:
        raise ValueError("dO must have Q's shape")
    B, T, S, Hq, D = q.shape
    Hkv = k.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros_like(q)
    lse = np.zeros((B, T, S, Hq), dtype=np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = getattr(_load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, T, S, Hq, Hkv, D, int(extra),
                                float(scale), int(nthreads))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return o, lse, dq, dk, dv


def space_fwd(q, k, v, agent=-1, scale=None, nthreads=0):
    """Masked space attention forward. Returns (O, LSE)."""
    return _fwd("oracle_space_fwd", q, k, v, agent, scale, nthreads)


def time_fwd(q, k, v, window, scale=None, nthreads=0):
    """Windowed causal time attention forward. Returns (O, LSE)."""
    return _fwd("oracle_time_fwd", q, k, v, window, scale, nthreads)


def space_bwd(q, k, v, dout, agent=-1, scale=None, nthreads=0):
    """Space attention backward. Returns (O, LSE, dQ, dK, dV)."""
    return _bwd("oracle_space_bwd", q, k, v, dout, agent, scale, nthreads)


def time_bwd(q, k, v, dout, window, scale=None, nthreads=0):
    """Time attention backward. Returns (O, LSE, dQ, dK, dV)."""
    return _bwd("oracle_time_bwd", q, k, v, dout, window, scale, nthreads)


def _varlen_blocks(shape_q, seqlen):
    B, T, S = shape_q[:3]
    L = np.clip(np.asarray(seqlen, dtype=np.int64).reshape(B, T), 0, S)
    return B, T, S, L


def space_fwd_varlen(q, k, v, seqlen, agent=-1, scale=None, nthreads=0):
    """Space attention over variable-length timestep blocks: block (b, t) holds its first
    seqlen[b, t] tokens (clamped to [0, S]) and is plain space attention over them (the agent
    rule applies when agent < seqlen).  Returns (O, LSE) with NaN in the padding rows."""
    B, T, S, L = _varlen_blocks(np.shape(q), seqlen)
    o = np.full(np.shape(q), np.nan)
    lse = np.full(np.shape(q)[:4], np.nan)
    for b in range(B):
        for t in range(T):
            n = int(L[b, t])
            if n == 0:
                continue
            a = agent if 0 <= agent < n else -1
            ob, lb = space_fwd(q[b:b + 1, t:t + 1, :n], k[b:b + 1, t:t + 1, :n],
                               v[b:b + 1, t:t + 1, :n], a, scale, nthreads)
            o[b, t, :n] = ob[0, 0]
            lse[b, t, :n] = lb[0, 0]
    return o, lse


def space_bwd_varlen(q, k, v, dout, seqlen, agent=-1, scale=None, nthreads=0):
    """Backward of space_fwd_varlen.  Returns (O, LSE, dQ, dK, dV), NaN in padding rows."""
    B, T, S, L = _varlen_blocks(np.shape(q), seqlen)
    out = [np.full(np.shape(q), np.nan), np.full(np.shape(q)[:4], np.nan),
           np.full(np.shape(q), np.nan), np.full(np.shape(k), np.nan), np.full(np.shape(v), np.nan)]
    for b in range(B):
        for t in range(T):
            n = int(L[b, t])
            if n == 0:
                continue
            a = agent if 0 <= agent < n else -1
            res = space_bwd(q[b:b + 1, t:t + 1, :n], k[b:b + 1, t:t + 1, :n],
                            v[b:b + 1, t:t + 1, :n], dout[b:b + 1, t:t + 1, :n], a, scale, nthreads)
            for dst, r in zip(out, res):
                dst[b, t, :n] = r[0, 0]
    return tuple(out)


def time_decode(q, k_new, v_new, k_cache, v_cache, t, scale=None):
    """Decode step of time attention with a ring-buffer KV cache of W = k_cache.shape[1]
    frames: stores the new frame (absolute index t) in slot t mod W, then attends over frames
    max(0, t-W+1) .. t.  q [B,S,Hq,D]; k_new, v_new [B,S,Hkv,D]; caches [B,W,S,Hkv,D].
    Returns (O [B,S,Hq,D], LSE [B,S,Hq], K cache after, V cache after); the inputs are not
    modified."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k_new = np.ascontiguousarray(k_new, dtype=np.float64)
    v_new = np.ascontiguousarray(v_new, dtype=np.float64)
    kc = np.array(k_cache, dtype=np.float64, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.float64, copy=True, order="C")
    B, S, Hq, D = q.shape
    Hkv = k_new.shape[2]
    W = kc.shape[1]
    if k_new.shape != (B, S, Hkv, D) or v_new.shape != k_new.shape or kc.shape != (B, W, S, Hkv, D) \
            or vc.shape != kc.shape:
        raise ValueError("expected q [B,S,Hq,D], k_new/v_new [B,S,Hkv,D], caches [B,W,S,Hkv,D]")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros_like(q)
    lse = np.zeros((B, S, Hq), dtype=np.float64)
    rc = _load().oracle_time_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(o),
                                    _ptr(lse), B, S, Hq, Hkv, D, W, int(t), float(scale))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return o, lse, kc, vc
