"""Backward parity: CUDA library vs the fp64 oracle.

Gates (the fp32 gradient outputs carry the stated tolerance; bf16 outputs add one rounding):
  fp32 dQ/dK/dV : max |err| <= 1e-2 and mean |err| / mean |ref| <= 2e-3
  bf16 dQ/dK/dV : per element |err| <= max(1e-2, one bf16 ulp of |ref|), and
                  mean |err| / mean |ref| <= 2e-3
"""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import assert_close, inputs, to_dev, to_f64

pytestmark = pytest.mark.gpu


def run_bwd(oracle_mod, kind, bits, extra, scale=0.125, with_lo=False):
    """with_lo: the forward also writes O's residual and the backward takes Delta from
    O + O_lo (instead of recomputing it from P and dP)."""
    q, k, v, do = bits
    Q, K, V, DO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    X = oracle_mod.from_bf16
    fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
    bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
    lo = None
    if with_lo:
        o, l, lo = fwd(Q, K, V, extra, scale, o_lo=True)
    else:
        o, l = fwd(Q, K, V, extra, scale)
    dq, dk, dv, (fq, fk, fv) = bwd(Q, K, V, o, l, DO, extra, scale, fp32_grads=True, o_lo=lo)
    if kind == "space":
        ref = oracle_mod.space_bwd(X(q), X(k), X(v), X(do), extra, scale)
    else:
        ref = oracle_mod.time_bwd(X(q), X(k), X(v), X(do), extra, scale)
    torch.cuda.synchronize()
    st, site = api.get_device_status_detail()
    assert st == 0, "device timeout at site word %#x" % site
    return (to_f64(dq), to_f64(dk), to_f64(dv)), (to_f64(fq), to_f64(fk), to_f64(fv)), ref[2:]


def check_bwd(oracle_mod, kind, bits, extra, scale=0.125, what="", with_lo=False):
    bf, f32, ref = run_bwd(oracle_mod, kind, bits, extra, scale, with_lo)
    what = "%s%s" % (what, " (Delta from O + O_lo)" if with_lo else "")
    for name, g, gb, r in zip(("dQ", "dK", "dV"), f32, bf, ref):
        assert_close(g, r, "%s %s %s fp32" % (what, kind, name), bf16_out=False)
        assert_close(gb, r, "%s %s %s bf16" % (what, kind, name))


def test_tiny_config_backward(oracle_mod):
    w = synth.WORKLOADS["tiny"]
    bits = synth.make_inputs(w, with_dout=True)
    check_bwd(oracle_mod, "space", bits, w.agent, w.scale, "tiny")
    check_bwd(oracle_mod, "time", bits, w.window, w.scale, "tiny")


SHAPES = [
    # B, T, S, Hq, Hkv, agent, window
    (2, 9, 37, 6, 2, 36, 5),
    (1, 5, 290, 30, 3, 289, 3),
    (1, 300, 3, 10, 1, 0, 192),
    (2, 70, 11, 8, 2, 5, 64),
    (1, 33, 130, 2, 2, -1, 200),
    (1, 3, 800, 4, 4, 799, 2),
    (3, 7, 1, 4, 2, 0, 1),
    (1, 1, 17, 16, 2, 0, 9),
    (1, 140, 2, 128, 1, 1, 130),
]


@pytest.mark.parametrize("with_lo", [False, True])
@pytest.mark.parametrize("B,T,S,Hq,Hkv,agent,window", SHAPES)
def test_backward_shapes(oracle_mod, B, T, S, Hq, Hkv, agent, window, with_lo):
    bits = inputs(B, T, S, Hq, Hkv, seed=7 * B + T + 3 * S, with_dout=True)
    check_bwd(oracle_mod, "space", bits, agent, what=str((B, T, S, Hq, Hkv)), with_lo=with_lo)
    check_bwd(oracle_mod, "time", bits, window, what=str((B, T, S, Hq, Hkv)), with_lo=with_lo)


def test_backward_gradient_invariants_on_gpu():
    """Keys no query reads get exactly zero gradient: the agent's K/V receive nothing from
    world rows, and frames after t receive nothing from rows <= t."""
    B, T, S, Hq, Hkv, a = 1, 6, 40, 4, 2, 39
    q, k, v, do = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=99, with_dout=True))
    do2 = do.clone()
    do2[:, :, a] = 0
    o, l = api.space_attn_fwd(q, k, v, a)
    dq, dk, dv = api.space_attn_bwd(q, k, v, o, l, do2, a)
    assert torch.count_nonzero(dk[:, :, a]) == 0 and torch.count_nonzero(dv[:, :, a]) == 0
    do3 = do.clone()
    do3[:, 3:] = 0
    o, l = api.time_attn_fwd(q, k, v, 4)
    dq, dk, dv = api.time_attn_bwd(q, k, v, o, l, do3, 4)
    assert torch.count_nonzero(dk[:, 3:]) == 0 and torch.count_nonzero(dv[:, 3:]) == 0
    assert torch.count_nonzero(dq[:, 3:]) == 0


@pytest.mark.parametrize("name", ["minecraft_fwd_bwd", "tokenizer_enc", "tokenizer_dec"])
def test_backward_full_size_sampled_units(oracle_mod, name):
    """Full-size backward (the bench's configuration): every gradient element is written and
    finite; whole sampled units are checked against the oracle."""
    w = synth.WORKLOADS[name]
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    Q, K, V, DO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    G = w.G
    X = oracle_mod.from_bf16
    rng = np.random.default_rng(w.seed + 11)
    for kind in ("space", "time"):
        extra = w.agent if kind == "space" else w.window
        fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
        bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
        o, l = fwd(Q, K, V, extra, w.scale)
        grads = [torch.full_like(x, float("nan")) for x in (Q, K, V)]
        dq, dk, dv, (fq, fk, fv) = bwd(Q, K, V, o, l, DO, extra, w.scale, fp32_grads=True, out=grads)
        torch.cuda.synchronize()
        st, site = api.get_device_status_detail()
        assert st == 0, "device timeout at site word %#x" % site
        for t_ in (dq, dk, dv, fq, fk, fv):
            assert bool(torch.isfinite(t_).all())
        F = w.T if kind == "space" else w.S
        for _ in range(4):
            b, f, h = int(rng.integers(w.B)), int(rng.integers(F)), int(rng.integers(w.Hkv))
            hs = slice(h * G, (h + 1) * G)
            if kind == "space":
                sel_q = (slice(b, b + 1), slice(f, f + 1), slice(None), hs)
                sel_k = (slice(b, b + 1), slice(f, f + 1), slice(None), slice(h, h + 1))
                ref = oracle_mod.space_bwd(X(q[sel_q]), X(k[sel_k]), X(v[sel_k]), X(do[sel_q]), extra, w.scale)
            else:
                sel_q = (slice(b, b + 1), slice(None), slice(f, f + 1), hs)
                sel_k = (slice(b, b + 1), slice(None), slice(f, f + 1), slice(h, h + 1))
                ref = oracle_mod.time_bwd(X(q[sel_q]), X(k[sel_k]), X(v[sel_k]), X(do[sel_q]), extra, w.scale)
            for nm, g, r in (("dQ", fq[sel_q], ref[2]), ("dK", fk[sel_k], ref[3]), ("dV", fv[sel_k], ref[4])):
                assert_close(to_f64(g), r, "%s %s %s unit %s" % (name, kind, nm, (b, f, h)), bf16_out=False)


def _scaled_bits(bits, e):
    """bf16 bit patterns times 2^e (exact: only the exponent field moves)."""
    x = synth.bf16_bits_to_f64(bits) * (2.0 ** e)
    return synth.f64_to_bf16_bits(x)


@pytest.mark.parametrize("kind", ["space", "time"])
def test_backward_operands_far_from_unit_range(oracle_mod, kind):
    """The dK/dV products run on fp16 operands scaled by powers of two taken from each
    tensor's largest magnitude.  Inputs far outside fp16's own range (tiny dO, huge V, small
    Q, large K) must give the same gradients, up to the exact power-of-two factors by which
    each gradient scales: dQ ~ dO V K, dK ~ dO V Q, dV ~ dO."""
    B, T, S, Hq, Hkv, agent, window = 1, 12, 150, 8, 2, 149, 7
    q, k, v, do = inputs(B, T, S, Hq, Hkv, seed=4242, with_dout=True)
    eq, ek, ev, edo = -9, 7, 20, -30
    bits = (_scaled_bits(q, eq), _scaled_bits(k, ek), _scaled_bits(v, ev), _scaled_bits(do, edo))
    extra = agent if kind == "space" else window
    bf, f32, ref = run_bwd(oracle_mod, kind, bits, extra)
    factors = (2.0 ** (edo + ev + ek), 2.0 ** (edo + ev + eq), 2.0 ** edo)
    for name, g, gb, r, f in zip(("dQ", "dK", "dV"), f32, bf, ref, factors):
        assert np.isfinite(g).all() and np.isfinite(gb).all()
        assert_close(g / f, r / f, "scaled %s %s fp32" % (kind, name), bf16_out=False)
        assert_close(gb / f, r / f, "scaled %s %s bf16" % (kind, name))


@pytest.mark.parametrize("with_lo", [False, True])
def test_backward_is_deterministic(with_lo):
    """No atomics anywhere in the backward: reruns give bit-identical bf16 and fp32 gradients
    (both Delta routes)."""
    B, T, S, Hq, Hkv, agent, window = 1, 12, 290, 30, 3, 289, 8
    q, k, v, do = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=2025, with_dout=True))
    for kind, extra in (("space", agent), ("time", window)):
        fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
        bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
        res = fwd(q, k, v, extra, 0.125, o_lo=(True if with_lo else None))
        o, l = res[0], res[1]
        lo = res[2] if with_lo else None
        runs = [bwd(q, k, v, o, l, do, extra, 0.125, fp32_grads=True, o_lo=lo) for _ in range(3)]
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        for r in runs[1:]:
            for a, b in zip(runs[0][:3] + tuple(runs[0][3]), r[:3] + tuple(r[3])):
                assert torch.equal(a, b), kind


@pytest.mark.parametrize("kind", ["space", "time"])
def test_backward_single_large_elements_in_v_and_dout(oracle_mod, kind):
    """N(0,1) V and dO that each carry one element near 1e3-1e4: the power-of-two scales of
    the fp16 products come from each tensor's largest magnitude, so one large element must not
    push the typical dS values into fp16's subnormal range."""
    B, T, S, Hq, Hkv, agent, window = 1, 10, 150, 8, 2, 149, 6
    q, k, v, do = inputs(B, T, S, Hq, Hkv, seed=5150, with_dout=True)
    vf, dof = synth.bf16_bits_to_f64(v), synth.bf16_bits_to_f64(do)
    vf[0, 3, 17, 1, 5] = 3000.0
    dof[0, 4, 40, 6, 9] = -7000.0
    bits = (q, k, synth.f64_to_bf16_bits(vf), synth.f64_to_bf16_bits(dof))
    extra = agent if kind == "space" else window
    for with_lo in (False, True):
        bf, f32, ref = run_bwd(oracle_mod, kind, bits, extra, with_lo=with_lo)
        for name, g, gb, r in zip(("dQ", "dK", "dV"), f32, bf, ref):
            # the reference gradients are large where the outliers act: judge relative to the
            # tensor's scale (max err <= 1e-2 * max|ref| is the absolute gate at unit scale)
            sc = max(1.0, float(np.abs(r).max()) / 10.0)
            assert_close(g / sc, r / sc, "outliers %s %s fp32 (lo=%s)" % (kind, name, with_lo), bf16_out=False)
            assert_close(gb / sc, r / sc, "outliers %s %s bf16 (lo=%s)" % (kind, name, with_lo))


@pytest.mark.parametrize("kind", ["space", "time"])
def test_plain_and_extended_calls_agree(kind):
    """The plain forward/backward calls and the extended ones with every optional pointer
    NULL run the same kernels: bit-identical O, LSE, dQ, dK, dV (called through the C ABI)."""
    import ctypes
    P = ctypes.c_void_p
    lib = api.library()
    B, T, S, Hq, Hkv, agent, window = 1, 9, 150, 8, 2, 149, 5
    q, k, v, do = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=8181, with_dout=True))
    extra = agent if kind == "space" else window
    stream = P(torch.cuda.current_stream().cuda_stream)
    dims = (B, T, S, Hq, Hkv, 64)
    ptr = lambda t: P(t.data_ptr())  # noqa: E731
    res = []
    for ex in (False, True):
        o, lse = torch.empty_like(q), torch.empty((B, T, S, Hq), dtype=torch.float32, device="cuda")
        if ex:
            st = getattr(lib, "od_%s_attn_fwd_ex" % kind)(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), P(0),
                                                          *dims, extra, 0.125, stream)
        else:
            st = getattr(lib, "od_%s_attn_fwd" % kind)(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), *dims,
                                                       extra, 0.125, stream)
        assert st == 0
        ws = torch.empty(api.bwd_workspace_bytes(0 if kind == "space" else 1, B, T, S, Hq, Hkv),
                         dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if ex:
            st = getattr(lib, "od_%s_attn_bwd_ex" % kind)(
                ptr(q), ptr(k), ptr(v), ptr(o), P(0), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv),
                P(0), P(0), P(0), *dims, extra, 0.125, ptr(ws), ws.numel(), stream)
        else:
            st = getattr(lib, "od_%s_attn_bwd" % kind)(
                ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv), *dims,
                extra, 0.125, ptr(ws), ws.numel(), stream)
        assert st == 0
        res.append((o, lse, dq, dk, dv))
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), *res):
        assert torch.equal(a, b), name


# Short time sequences are packed in the backward (G T <= 64: several token positions per
# tile, block-diagonal mask): T in {1, 3, 32, 33} x G in {1, 2}, S with a partial last group
# of token positions, windows shorter than, equal to and longer than T.
PACKED_SHAPES = [
    # B, T, S, Hq, Hkv, window
    (2, 1, 37, 2, 2, 1),
    (1, 1, 130, 4, 2, 3),
    (2, 3, 41, 2, 2, 2),
    (1, 3, 50, 4, 2, 3),
    (1, 32, 13, 2, 2, 7),
    (2, 32, 9, 4, 2, 32),
    (1, 33, 11, 2, 2, 40),
    (1, 33, 7, 4, 2, 5),
]


@pytest.mark.parametrize("shape", PACKED_SHAPES)
@pytest.mark.parametrize("with_lo", [False, True])
def test_time_backward_short_sequences_packed(oracle_mod, shape, with_lo):
    B, T, S, Hq, Hkv, window = shape
    bits = inputs(B, T, S, Hq, Hkv, seed=700 + 7 * T + S, with_dout=True)
    check_bwd(oracle_mod, "time", bits, window, 0.125, "packed %s" % (shape,), with_lo=with_lo)
