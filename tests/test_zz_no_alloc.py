"""The allocation-free space backward (od_space_attn_bwd_static_ws).

Some callers cannot allocate device memory -- an allocator-free runtime, or code at a point
where cudaMalloc is not allowed or would synchronise.  For them the library offers a space
attention backward whose scratch lives in a fixed array inside the library.  These tests call
it through the C ABI and check that it gives the same gradients as the regular entry point
(with a caller-provided workspace) -- bit for bit, since both run the same deterministic
kernels -- on two calls in a row, since every call reuses the same array, on both Delta routes
(recomputed, and read from O + O_lo); and that sizes beyond the fixed array are refused before
anything runs.  The tests build all their inputs themselves and assume nothing about what ran
before them; the file name only makes pytest collect them last, so that a run that stops at
the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api
from helpers import assert_close, inputs, to_dev, to_f64

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _ptr(t):
    return P(t.data_ptr()) if t is not None else P(0)


def _static_ws_bwd(lib, Q, K, V, O, L, DO, agent, scale, stream, O_lo=None):
    dq, dk, dv = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    fq = torch.empty(Q.shape, dtype=torch.float32, device=Q.device)
    fk = torch.empty(K.shape, dtype=torch.float32, device=Q.device)
    fv = torch.empty(V.shape, dtype=torch.float32, device=Q.device)
    B, T, S, Hq, D = Q.shape
    st = lib.od_space_attn_bwd_static_ws(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(O_lo), _ptr(L), _ptr(DO), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(fq), _ptr(fk), _ptr(fv), B, T, S, Hq, K.shape[3], D, agent,
        ctypes.c_float(scale), P(stream.cuda_stream))
    assert st == 0, api.STATUS.get(st, st)
    return (dq, dk, dv), (fq, fk, fv)


@pytest.mark.parametrize("with_lo", [False, True])
def test_static_workspace_backward_matches_regular_entry_point(with_lo):
    lib = api.library()
    B, T, S, Hq, Hkv, agent, scale = 2, 6, 150, 12, 2, 149, 0.125
    Q, K, V, DO = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=2024, with_dout=True))
    stream = torch.cuda.current_stream()
    if with_lo:
        O, L, O_lo = api.space_attn_fwd(Q, K, V, agent, scale, o_lo=True)
    else:
        (O, L), O_lo = api.space_attn_fwd(Q, K, V, agent, scale), None
    dq, dk, dv, (fq, fk, fv) = api.space_attn_bwd(Q, K, V, O, L, DO, agent, scale, fp32_grads=True,
                                                  o_lo=O_lo)
    ref = (dq, dk, dv, fq, fk, fv)
    for call in range(2):   # the second call reuses the array the first one left behind
        got_bf, got_f32 = _static_ws_bwd(lib, Q, K, V, O, L, DO, agent, scale, stream, O_lo)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        for name, g, r in zip(("dQ", "dK", "dV", "dQ fp32", "dK fp32", "dV fp32"),
                              got_bf + got_f32, ref):
            assert_close(to_f64(g), to_f64(r), "call %d %s" % (call, name),
                         bf16_out=g.dtype == torch.bfloat16)
            assert torch.equal(g, r), "call %d %s differs from the regular entry point" % (call, name)


def test_static_workspace_refuses_sizes_beyond_the_fixed_array():
    lib = api.library()
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    B, T, S, Hq, Hkv = 1, 1024, 1024, 8, 8     # 8M query rows x 4 bytes > the fixed array
    assert B * T * S * Hq * 4 > 16 << 20
    ptrs = [_ptr(small)] * 4 + [P(0)] + [_ptr(small)] * 5 + [P(0)] * 3
    st = lib.od_space_attn_bwd_static_ws(*ptrs, B, T, S, Hq, Hkv, 64, -1, ctypes.c_float(0.125),
                                         P(torch.cuda.current_stream().cuda_stream))
    assert st == 5   # OD_ERR_WORKSPACE
