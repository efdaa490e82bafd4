"""Timelines of one CTA from a profiling build of the library (diagnosis only).

The kernels carry trace points that compile to nothing unless the library is built with
-DOD_TRACE.  This module builds that variant (libod_attn_trace.so), routes the binding's
calls to it, selects which kernel records (od_trace_select), runs a call and reads the
records back (od_trace_read): per warp of CTA 7, the SM clock at each trace point and the
point's event number.  `phases` summarises a recording as the median cycles between
consecutive events of each warp, which is how waits are told apart from work.

    python -m block_causal_video_attention_b300.trace minecraft_fwd_bwd space dq

Events (see OD_TP in the sources): forward softmax 1-9, MMA issuers 10-13 and 44-45, producer
20-23, V converter 30; dQ pass dS warps 80-88 and MMA issuers 90-91; dK/dV elementwise 40-47,
producer 50-51, MMA issuer 61-64, converters 70-73.  Clocks of different warps share a base,
within a CTA.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from . import api, build

TRACE_LIB = os.path.join(build.PKG, "libod_attn_trace.so")
KERNELS = {"fwd": 0, "dq": 1, "dkdv": 2, "delta": 3}
WARPS, PER_WARP = 32, 8192


def build_trace(force: bool = False) -> str:
    """libod_attn_trace.so: the library's sources compiled with -DOD_TRACE."""
    if not force and not build.needs_build_of(TRACE_LIB):
        return TRACE_LIB
    cmd = [build.NVCC] + build.NVCC_FLAGS + ["-DOD_TRACE", "-I", os.path.join(build.ROOT, "include"),
                                             "-o", TRACE_LIB, os.path.join(build.CSRC, "od_api.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building libod_attn_trace.so")
    return TRACE_LIB


def _lib():
    lib = api._load(build_trace())
    lib.od_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.od_trace_read.restype = ctypes.c_int
    lib.od_trace_select.argtypes = [ctypes.c_int]
    lib.od_trace_select.restype = ctypes.c_int
    return lib


def record(fn, kernel: str, warmup: int = 2) -> np.ndarray:
    """Runs fn() (calls of this package's binding) with the trace build; returns the records of
    `kernel`'s CTA 7 from the last run as uint64: (clock << 32) | (warp << 26) | event word."""
    import torch
    lib = _lib()
    prev = api._override
    api._override = lib
    try:
        if lib.od_trace_select(KERNELS[kernel]) != 0:
            raise RuntimeError("od_trace_select failed")
        buf = np.zeros(WARPS * PER_WARP, dtype=np.uint64)
        cnt = np.zeros(WARPS, dtype=np.uint32)
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        lib.od_trace_read(buf.ctypes.data, cnt.ctypes.data)   # clears the counts
        fn()
        torch.cuda.synchronize()
        if lib.od_trace_read(buf.ctypes.data, cnt.ctypes.data) != 0:
            raise RuntimeError("od_trace_read failed")
        lib.od_trace_select(-1)
    finally:
        api._override = prev
    recs = [buf[w * PER_WARP: w * PER_WARP + min(int(cnt[w]), PER_WARP)] | np.uint64(w << 26)
            for w in range(WARPS)]
    return np.concatenate(recs)


def phases(recs: np.ndarray, top: int = 6):
    """Per warp: (span in cycles, [(from event, to event, count, median cycles, share)])."""
    clk = (recs >> np.uint64(32)).astype(np.int64)
    word = (recs & np.uint64(0xFFFFFFFF)).astype(np.int64)
    warp, ev = word >> 26, (word >> 18) & 0xFF
    out = {}
    for w in np.unique(warp):
        m = np.nonzero(warp == w)[0]
        c = clk[m]
        t = np.concatenate([[0], np.cumsum(np.diff(c) % (1 << 32))])   # 32-bit clock unwrapped
        e = ev[m]
        span = int(t[-1]) if len(t) else 0
        pairs = {}
        for j in range(len(t) - 1):
            pairs.setdefault((int(e[j]), int(e[j + 1])), []).append(int(t[j + 1] - t[j]))
        rows = sorted(((a, b, len(v), int(np.median(v)), sum(v) / max(span, 1))
                       for (a, b), v in pairs.items()), key=lambda r: -r[4])
        out[int(w)] = (span, rows[:top])
    return out


def main(argv):
    import torch
    from . import synth
    name, kind, kernel = (argv + ["minecraft_fwd_bwd", "space", "dq"])[:3]
    w = synth.WORKLOADS[name]
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    Q, K, V, DO = to(q), to(k), to(v), to(do)
    extra = w.agent if kind == "space" else w.window
    fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
    bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
    o, lse, lo = fwd(Q, K, V, extra, w.scale, o_lo=True)
    if kernel == "fwd":
        fn = lambda: fwd(Q, K, V, extra, w.scale, o_lo=True)  # noqa: E731
    else:
        fn = lambda: bwd(Q, K, V, o, lse, DO, extra, w.scale, o_lo=None if kernel == "delta" else lo)  # noqa: E731
    for wp, (span, rows) in sorted(phases(record(fn, kernel)).items()):
        print("warp %2d  span %9d  " % (wp, span) +
              "  ".join("%d>%d n%d med %d (%.0f%%)" % (a, b, n, med, 100 * sh) for a, b, n, med, sh in rows))


if __name__ == "__main__":
    main(sys.argv[1:])
