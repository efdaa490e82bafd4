"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
and rejects invalid arguments before touching the device."""
import ctypes
import re

import pytest

from block_causal_video_attention_b300 import api


@pytest.fixture(scope="module")
def lib():
    from block_causal_video_attention_b300 import build
    build.build()
    return api.library()


def test_every_declared_symbol_is_exported(lib):
    src = open(api._HEADER).read()
    declared = set(re.findall(r"\b(od_\w+)\s*\(", src))
    assert {"od_space_attn_fwd", "od_time_attn_fwd", "od_space_attn_bwd", "od_time_attn_bwd",
            "od_space_attn_fwd_ex", "od_time_attn_fwd_ex", "od_space_attn_bwd_ex", "od_time_attn_bwd_ex",
            "od_attn_bwd_workspace_bytes", "od_get_device_status", "od_get_device_status_detail",
            "od_status_string", "od_space_attn_bwd_static_ws", "od_time_attn_decode",
            "od_space_attn_fwd_packed", "od_time_attn_fwd_packed", "od_space_attn_bwd_packed",
            "od_time_attn_bwd_packed", "od_space_attn_fwd_varlen", "od_space_attn_bwd_varlen", "od_selftest_expired_wait",
            "od_version"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(api.EXPORTED_SYMBOLS) == declared


def test_status_strings(lib):
    for code in range(7):
        assert lib.od_status_string(code)
    assert b"sm_103a" in lib.od_version()


P = ctypes.c_void_p
GOOD = P(4096)  # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("fn", ["od_space_attn_fwd_ex", "od_time_attn_fwd_ex"])
def test_forward_rejects_invalid_arguments(lib, fn):
    f = getattr(lib, fn)
    extra_ok = 0 if fn == "od_space_attn_fwd_ex" else 4
    base = dict(B=1, T=4, S=8, Hq=4, Hkv=2, D=64, extra=extra_ok, scale=0.125)

    def call(ptrs=None, **kw):
        a = dict(base, **kw)
        q, k, v, o, l = ptrs or (GOOD, GOOD, GOOD, GOOD, GOOD)
        return f(q, k, v, o, l, a.get("o_lo", P(0)), a["B"], a["T"], a["S"], a["Hq"], a["Hkv"], a["D"], a["extra"],
                 a["scale"], P(0))
    assert call(ptrs=(P(0), GOOD, GOOD, GOOD, GOOD)) == 1
    assert call(ptrs=(GOOD, GOOD, GOOD, P(4097), GOOD)) == 1      # misaligned
    assert call(o_lo=P(4100)) == 1                                  # misaligned residual
    assert call(B=0) == 1
    assert call(S=-3) == 1
    assert call(Hq=5, Hkv=2) == 1                                  # Hq % Hkv
    assert call(scale=float("nan")) == 1
    assert call(scale=-0.1) == 1
    assert call(D=128) == 2                                         # unsupported head dim
    assert call(Hq=258, Hkv=1) == 2                                 # group too large
    # shapes whose byte count would wrap a 64-bit product: each dimension is checked first
    assert call(B=1024, T=1 << 24, S=1 << 24, Hq=4, Hkv=2) == 2
    assert call(B=65535, T=1 << 24, S=1 << 24, Hq=65535, Hkv=65535) == 2
    assert call(B=1, T=1 << 20, S=1 << 20, Hq=2, Hkv=2, extra=0 if fn == "od_space_attn_fwd_ex" else 4) == 2
    if fn == "od_space_attn_fwd_ex":
        assert call(extra=8) == 1 and call(extra=-2) == 1           # agent index out of range
    else:
        assert call(extra=0) == 1                                   # window < 1


@pytest.mark.parametrize("fn", ["od_space_attn_bwd_ex", "od_time_attn_bwd_ex"])
def test_backward_rejects_invalid_arguments(lib, fn):
    f = getattr(lib, fn)
    extra = 0 if fn == "od_space_attn_bwd_ex" else 4
    ptrs = [GOOD] * 4 + [P(0)] + [GOOD] * 5 + [P(0)] * 3   # q k v o (no o_lo) lse dO dq dk dv
    ws = lib.od_attn_bwd_workspace_bytes(0 if "space" in fn else 1, 1, 4, 8, 4, 2, 64)
    assert ws > 0
    assert f(*ptrs, 1, 4, 8, 4, 2, 64, extra, 0.125, GOOD, ws - 16, P(0)) == 5  # too small
    bad = list(ptrs)
    bad[6] = P(0)                                                   # null dO
    assert f(*bad, 1, 4, 8, 4, 2, 64, extra, 0.125, GOOD, ws, P(0)) == 1
    assert f(*ptrs, 1, 4, 8, 4, 3, 64, extra, 0.125, GOOD, ws, P(0)) == 1           # Hq % Hkv
    bad = list(ptrs)
    bad[4] = P(4104)                                                # misaligned o_lo
    assert f(*bad, 1, 4, 8, 4, 2, 64, extra, 0.125, GOOD, ws, P(0)) == 1
    assert lib.od_attn_bwd_workspace_bytes(2, 1, 4, 8, 4, 2, 64) == 0
    # Delta (fp32 per query row, 256-byte rounded) + 1024 slots x 8 fp32 operand ranges
    for dims in ((1, 4, 8, 4), (2, 7, 33, 12), (1, 256, 290, 30)):
        rows = dims[0] * dims[1] * dims[2] * dims[3]
        want = ((rows * 4 + 255) // 256) * 256 + 32768
        assert lib.od_attn_bwd_workspace_bytes(0, *dims, 2 if dims[3] % 2 == 0 else 3, 64) == want
    # the fixed array of the allocation-free entry point serves up to 4,186,112 rows
    assert ((4186112 * 4 + 255) // 256) * 256 + 32768 <= 16 << 20
    assert ((4186176 * 4 + 255) // 256) * 256 + 32768 > 16 << 20
    assert lib.od_attn_bwd_workspace_bytes(0, 1, 4, 8, 4, 3, 64) == 0


@pytest.mark.parametrize("kind", ["space", "time"])
def test_plain_calls_take_the_boundary_arguments(lib, kind):
    """The plain calls carry exactly (q, k, v, o, lse, B, T, S, Hq, Hkv, D, agent|window,
    scale, stream) and (q, k, v, o, lse, dO, dQ, dK, dV, sizes, agent|window, scale,
    workspace, bytes, stream): no residual and no fp32 outputs.  They validate like the
    extended calls with those pointers NULL -- which the extended calls accept."""
    fwd, bwd = getattr(lib, "od_%s_attn_fwd" % kind), getattr(lib, "od_%s_attn_bwd" % kind)
    fwd_ex, bwd_ex = getattr(lib, "od_%s_attn_fwd_ex" % kind), getattr(lib, "od_%s_attn_bwd_ex" % kind)
    assert fwd.argtypes is not None and len(fwd.argtypes) == 14 and len(fwd_ex.argtypes) == 15
    assert len(bwd.argtypes) == 20 and len(bwd_ex.argtypes) == 24
    extra = 0 if kind == "space" else 4
    which = 0 if kind == "space" else 1
    dims = (1, 4, 8, 4, 2, 64)
    ws = lib.od_attn_bwd_workspace_bytes(which, *dims)
    # invalid in the same way -> the same status from the plain and the extended call
    for bad_dims, bad_extra, bad_scale in (((0, 4, 8, 4, 2, 64), extra, 0.125),
                                           ((1, 4, 8, 5, 2, 64), extra, 0.125),
                                           ((1, 4, 8, 4, 2, 128), extra, 0.125),
                                           (dims, 8 if kind == "space" else 0, 0.125),
                                           (dims, extra, float("inf"))):
        a = fwd(GOOD, GOOD, GOOD, GOOD, GOOD, *bad_dims, bad_extra, bad_scale, P(0))
        b = fwd_ex(GOOD, GOOD, GOOD, GOOD, GOOD, P(0), *bad_dims, bad_extra, bad_scale, P(0))
        assert a == b and a in (1, 2)
        a = bwd(*[GOOD] * 9, *bad_dims, bad_extra, bad_scale, GOOD, ws, P(0))
        b = bwd_ex(*[GOOD] * 4, P(0), *[GOOD] * 5, P(0), P(0), P(0), *bad_dims, bad_extra,
                   bad_scale, GOOD, ws, P(0))
        assert a == b and a in (1, 2)
    assert fwd(P(0), GOOD, GOOD, GOOD, GOOD, *dims, extra, 0.125, P(0)) == 1          # null q
    assert fwd(GOOD, GOOD, GOOD, P(4097), GOOD, *dims, extra, 0.125, P(0)) == 1       # misaligned o
    assert bwd(*[GOOD] * 5, P(0), *[GOOD] * 3, *dims, extra, 0.125, GOOD, ws, P(0)) == 1   # null dO
    assert bwd(*[GOOD] * 9, *dims, extra, 0.125, GOOD, ws - 16, P(0)) == 5            # workspace
    assert bwd(*[GOOD] * 9, *dims, extra, 0.125, P(0), ws, P(0)) == 1                 # null workspace


def test_decode_rejects_invalid_arguments(lib):
    f = lib.od_time_attn_decode
    base = dict(B=2, S=5, Hq=4, Hkv=2, D=64, W=6, t=3, scale=0.125)

    def call(ptrs=None, **kw):
        a = dict(base, **kw)
        p = ptrs or (GOOD,) * 7
        return f(*p, a["B"], a["S"], a["Hq"], a["Hkv"], a["D"], a["W"], a["t"], a["scale"], P(0))
    assert call(ptrs=(GOOD,) * 3 + (P(0),) + (GOOD,) * 3) == 1     # null cache
    assert call(ptrs=(GOOD,) * 6 + (P(4100),)) == 1                 # misaligned LSE
    assert call(t=-1) == 1
    assert call(W=0) == 1
    assert call(B=0) == 1
    assert call(Hq=5) == 1                                          # Hq % Hkv
    assert call(scale=float("inf")) == 1
    assert call(D=32) == 2
    assert call(Hq=34, Hkv=2) == 2                                  # G = 17 > 16
    assert call(W=(1 << 24) + 1) == 2


def test_packed_calls_reject_invalid_arguments(lib):
    f = lib.od_space_attn_fwd_packed
    assert f(P(0), GOOD, GOOD, P(0), 1, 4, 8, 4, 2, 64, 0, 0.125, P(0)) == 1    # null qkv
    assert f(GOOD, GOOD, GOOD, P(0), 1, 4, 8, 4, 2, 32, 0, 0.125, P(0)) == 2    # D != 64
    assert f(GOOD, GOOD, GOOD, P(0), 1, 4, 8, 5, 2, 64, 0, 0.125, P(0)) == 1    # Hq % Hkv
    assert lib.od_time_attn_fwd_packed(GOOD, GOOD, GOOD, P(0), 1, 4, 8, 4, 2, 64, 0, 0.125,
                                       P(0)) == 1
    b = lib.od_space_attn_bwd_packed
    ws = lib.od_attn_bwd_workspace_bytes(0, 1, 4, 8, 4, 2, 64)
    n = 1 * 4 * 8 * (4 + 2 * 2) * 64 * 2          # bytes of one packed tensor
    args = lambda qkv, dqkv: (qkv, GOOD, P(0), GOOD, GOOD, dqkv, P(0), P(0), P(0), 1, 4, 8, 4, 2,
                              64, 0, 0.125, GOOD, ws, P(0))
    assert b(*args(P(1 << 20), P(0))) == 1                                      # null dqkv
    assert b(*args(P(1 << 20), P((1 << 20) + n - 16))) == 1                     # overlapping
    assert b(*args(P((1 << 20) + n - 16), P(1 << 20))) == 1
    assert lib.od_time_attn_bwd_packed(*args(P(1 << 20), P(1 << 20))) == 1      # aliased


def test_varlen_calls_reject_invalid_arguments(lib):
    f = lib.od_space_attn_fwd_varlen
    good = (GOOD,) * 5 + (P(0),)
    assert f(*good, P(0), 1, 4, 8, 4, 2, 64, 0, 0.125, P(0)) == 1               # no lengths
    assert f(*good, P(4100), 1, 4, 8, 4, 2, 64, 0, 0.125, P(0)) == 1            # misaligned
    assert f(*good, GOOD, 1, 4, 8, 4, 2, 64, 9, 0.125, P(0)) == 1               # agent >= S
    b = lib.od_space_attn_bwd_varlen
    ws = lib.od_attn_bwd_workspace_bytes(0, 1, 4, 8, 4, 2, 64)
    ptrs = [GOOD] * 4 + [P(0), GOOD, GOOD]        # q k v o (no o_lo) lse dO
    assert b(*ptrs, P(0), *([GOOD] * 3), *([P(0)] * 3), 1, 4, 8, 4, 2, 64, 0, 0.125, GOOD, ws,
             P(0)) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 2, 3, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 3, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        api.space_attn_fwd(q, k, k, agent_idx=-1)


def test_every_operator_has_a_binding():
    """Each operator entry point of the C ABI has a same-named Python function (without the
    od_ prefix) exported by the package."""
    import inspect

    import block_causal_video_attention_b300 as pkg
    ops = [s for s in api.EXPORTED_SYMBOLS
           if re.match(r"od_(space|time)_attn_(fwd|bwd|decode)", s)
           and not s.endswith(("static_ws", "_ex"))]
    assert len(ops) == 11
    for sym in ops + ["od_selftest_expired_wait", "od_get_device_status",
                      "od_get_device_status_detail"]:
        name = sym[3:]
        assert callable(getattr(api, name)), name
        assert name in pkg.__all__, name
    # an extended call is reached through the plain call's binding and its optional arguments
    ext = [s for s in api.EXPORTED_SYMBOLS if s.endswith("_ex")]
    assert len(ext) == 4
    for sym in ext:
        params = inspect.signature(getattr(api, sym[3:-3])).parameters
        assert "o_lo" in params and ("fwd" in sym or "fp32_grads" in params), sym
