"""Forward parity: CUDA library vs the fp64 oracle, element by element.

Tolerances (stated for bf16 I/O with N(0,1) inputs): max |err| <= 1e-2, mean relative
error (mean |err| / mean |ref|) <= 2e-3 for O, and |err| <= 1e-3 for the logsumexp.
"""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import LSE_ERR, assert_close, inputs, to_dev, to_f64

pytestmark = pytest.mark.gpu


def run_both(oracle_mod, kind, bits, extra, scale=0.125):
    q, k, v = bits[:3]
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full_like(dq, float("nan"))
    lse = torch.full(dq.shape[:4], float("nan"), dtype=torch.float32, device="cuda")
    if kind == "space":
        api.space_attn_fwd(dq, dk, dv, agent_idx=extra, scale=scale, out=o, lse=lse)
        ro, rl = oracle_mod.space_fwd(oracle_mod.from_bf16(q), oracle_mod.from_bf16(k),
                                      oracle_mod.from_bf16(v), extra, scale)
    else:
        api.time_attn_fwd(dq, dk, dv, window=extra, scale=scale, out=o, lse=lse)
        ro, rl = oracle_mod.time_fwd(oracle_mod.from_bf16(q), oracle_mod.from_bf16(k),
                                     oracle_mod.from_bf16(v), extra, scale)
    torch.cuda.synchronize()
    st, site = api.get_device_status_detail()
    assert st == 0, "device timeout at site word %#x" % site
    return to_f64(o), to_f64(lse), ro, rl


def check(oracle_mod, kind, bits, extra, scale=0.125, what=""):
    go, gl, ro, rl = run_both(oracle_mod, kind, bits, extra, scale)
    assert_close(go, ro, "%s %s O" % (what, kind))
    assert np.isfinite(gl).all()
    assert np.abs(gl - rl).max() <= LSE_ERR, "%s %s LSE err %g" % (what, kind, np.abs(gl - rl).max())


def test_tiny_config_all_elements(oracle_mod):
    w = synth.WORKLOADS["tiny"]
    bits = synth.make_inputs(w)
    check(oracle_mod, "space", bits, w.agent, w.scale, "tiny")
    check(oracle_mod, "time", bits, w.window, w.scale, "tiny")


# shapes spanning several Q tiles, several key blocks and ragged tails
SHAPES = [
    # B, T, S, Hq, Hkv, agent, window
    (2, 9, 37, 6, 2, 36, 5),       # G=3 (nTok=42, rows=126)
    (1, 5, 290, 30, 3, 289, 3),    # the 1.6B dynamics head layout, 3 key blocks in space
    (1, 300, 3, 10, 1, 0, 192),    # G=10 time with 3 key blocks and a window edge
    (2, 70, 11, 8, 2, 5, 64),      # G=4
    (1, 33, 130, 2, 2, -1, 200),   # G=1, window >= T, no agent
    (1, 4, 800, 4, 4, 799, 2),     # S > 7 key blocks: K/V streamed through the ring
    (3, 7, 1, 4, 2, 0, 1),         # S = 1 (agent reads itself only), W = 1
    (1, 1, 17, 16, 2, 0, 9),       # T = 1, agent at 0, G = 8
    (1, 260, 2, 128, 1, 1, 130),   # G = 128: one token per tile
]


@pytest.mark.parametrize("B,T,S,Hq,Hkv,agent,window", SHAPES)
def test_shapes_all_elements(oracle_mod, B, T, S, Hq, Hkv, agent, window):
    bits = inputs(B, T, S, Hq, Hkv, seed=B * 1000 + T * 10 + S)
    check(oracle_mod, "space", bits, agent, what=str((B, T, S, Hq, Hkv)))
    check(oracle_mod, "time", bits, window, what=str((B, T, S, Hq, Hkv)))


def test_lazy_rescale_path(oracle_mod):
    """Logits that grow from key block to key block force the running-max rescale."""
    B, T, S, Hq, Hkv = 1, 2, 400, 4, 2
    q = np.full((B, T, S, Hq, 64), 1.0)
    k = np.zeros((B, T, S, Hkv, 64))
    k[:] = (np.arange(S) * 0.01)[None, None, :, None, None]
    rng = np.random.default_rng(5)
    v = rng.standard_normal((B, T, S, Hkv, 64))
    q = q + 0.1 * rng.standard_normal(q.shape)
    bits = tuple(synth.f64_to_bf16_bits(a) for a in (q, k, v))
    check(oracle_mod, "space", bits, 399, what="rescale")
    # time: logits growing along t
    q2 = np.full((B, 300, 2, Hq, 64), 1.0) + 0.1 * rng.standard_normal((B, 300, 2, Hq, 64))
    k2 = np.zeros((B, 300, 2, Hkv, 64))
    k2[:] = (np.arange(300) * 0.01)[None, :, None, None, None]
    v2 = rng.standard_normal((B, 300, 2, Hkv, 64))
    bits2 = tuple(synth.f64_to_bf16_bits(a) for a in (q2, k2, v2))
    check(oracle_mod, "time", bits2, 250, what="rescale")


def test_scale_argument(oracle_mod):
    bits = inputs(1, 6, 20, 4, 1, seed=77)
    check(oracle_mod, "space", bits, 3, scale=0.3, what="scale")
    check(oracle_mod, "time", bits, 4, scale=0.05, what="scale")


def test_agent_invariance_on_gpu():
    """World rows of space attention do not change when the agent's K/V change."""
    B, T, S, Hq, Hkv, a = 1, 3, 50, 4, 2, 17
    q, k, v = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=9))
    o1, l1 = api.space_attn_fwd(q, k, v, agent_idx=a)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, a] += 3.0
    v2[:, :, a] *= -2.0
    o2, l2 = api.space_attn_fwd(q, k2, v2, agent_idx=a)
    world = [s for s in range(S) if s != a]
    assert torch.equal(o1[:, :, world], o2[:, :, world])
    assert torch.equal(l1[:, :, world], l2[:, :, world])
    assert not torch.equal(o1[:, :, a], o2[:, :, a])


def test_causality_on_gpu():
    B, T, S, Hq, Hkv, W = 1, 40, 3, 4, 2, 7
    q, k, v = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=10))
    o1, l1 = api.time_attn_fwd(q, k, v, window=W)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, 21:] += 1.0
    k2[:, 21:] -= 2.0
    v2[:, 21:] *= 3.0
    o2, l2 = api.time_attn_fwd(q2, k2, v2, window=W)
    assert torch.equal(o1[:, :21], o2[:, :21]) and torch.equal(l1[:, :21], l2[:, :21])
    k3 = k.clone()
    k3[:, :10] += 5.0
    o3, _ = api.time_attn_fwd(q, k3, v, window=W)
    assert torch.equal(o1[:, 16:], o3[:, 16:])   # rows t >= 16 never see frames < 10


@pytest.mark.parametrize("name", ["coinrun", "minecraft_fwd", "tokenizer_enc", "tokenizer_dec"])
def test_full_size_sampled_units(oracle_mod, name):
    """Full-size launch (the bench's configuration); every element is checked for being
    written and finite, and whole sampled units are checked against the oracle."""
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_inputs(w, with_dout=False)
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    G = w.G
    rng = np.random.default_rng(w.seed)
    for kind in ("space", "time"):
        o = torch.full_like(dq, float("nan"))
        lse = torch.full(dq.shape[:4], float("nan"), dtype=torch.float32, device="cuda")
        if kind == "space":
            api.space_attn_fwd(dq, dk, dv, agent_idx=w.agent, scale=w.scale, out=o, lse=lse)
        else:
            api.time_attn_fwd(dq, dk, dv, window=w.window, scale=w.scale, out=o, lse=lse)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
        F = w.T if kind == "space" else w.S
        for _ in range(8):
            b, f, h = int(rng.integers(w.B)), int(rng.integers(F)), int(rng.integers(w.Hkv))
            hs = slice(h * G, (h + 1) * G)
            if kind == "space":
                sq, sk, sv = q[b:b+1, f:f+1, :, hs], k[b:b+1, f:f+1, :, h:h+1], v[b:b+1, f:f+1, :, h:h+1]
                ro, rl = oracle_mod.space_fwd(*(oracle_mod.from_bf16(x) for x in (sq, sk, sv)),
                                              w.agent, w.scale)
                go = to_f64(o[b:b+1, f:f+1, :, hs])
                gl = to_f64(lse[b:b+1, f:f+1, :, hs])
            else:
                sq, sk, sv = q[b:b+1, :, f:f+1, hs], k[b:b+1, :, f:f+1, h:h+1], v[b:b+1, :, f:f+1, h:h+1]
                ro, rl = oracle_mod.time_fwd(*(oracle_mod.from_bf16(x) for x in (sq, sk, sv)),
                                             w.window, w.scale)
                go = to_f64(o[b:b+1, :, f:f+1, hs])
                gl = to_f64(lse[b:b+1, :, f:f+1, hs])
            assert_close(go, ro, "%s %s unit %s" % (name, kind, (b, f, h)))
            assert np.abs(gl - rl).max() <= LSE_ERR


@pytest.mark.parametrize("vscale", [2.0 ** 17, 2.0 ** -14, 2.0 ** -30])
def test_v_outside_fp16_range_is_rescaled(oracle_mod, vscale):
    """P V runs on fp16 V; a V block whose magnitude is outside fp16's safe range is scaled by
    a power of two into it (and O rescaled between blocks of different scales).  Keys 32..63
    and 200.. of every frame are scaled; the rest stay N(0,1).  Both sides are divided by the
    power of two nearest mean |O|, which leaves bf16 ulps exact, and compared at the usual
    gates (per element max(1e-2, one bf16 ulp of the reference), mean relative 2e-3)."""
    B, T, S, Hq, Hkv = 1, 4, 300, 4, 2
    q, k, v = inputs(B, T, S, Hq, Hkv, seed=31)
    vf = oracle_mod.from_bf16(v)
    vf[:, :, 32:64] *= vscale
    vf[:, :, 200:] *= vscale
    v2 = synth.f64_to_bf16_bits(vf)
    go, gl, ro, rl = run_both(oracle_mod, "space", (q, k, v2), 5)
    sc = 2.0 ** round(np.log2(np.abs(ro).mean()))
    assert_close(go / sc, ro / sc, "V scaled by %g (output scale %g)" % (vscale, sc))
    assert np.abs(gl - rl).max() <= LSE_ERR


@pytest.mark.parametrize("kind", ["space", "time"])
def test_output_residual(oracle_mod, kind):
    """o_lo = bf16(O - o): requesting it leaves O and LSE bit-identical, and o + o_lo holds the
    kernel's fp32 O, much closer to the exact O than bf16 O alone."""
    B, T, S, Hq, Hkv, agent, window = 1, 40, 290, 30, 3, 289, 24
    bits = inputs(B, T, S, Hq, Hkv, seed=4242)
    Q, K, V = (to_dev(x) for x in bits[:3])
    fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
    extra = agent if kind == "space" else window
    o1, l1 = fwd(Q, K, V, extra, 0.125)
    o2, l2, lo = fwd(Q, K, V, extra, 0.125, o_lo=True)
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    X = oracle_mod.from_bf16
    ro, _ = (oracle_mod.space_fwd if kind == "space" else oracle_mod.time_fwd)(
        X(bits[0]), X(bits[1]), X(bits[2]), extra, 0.125)
    hi, both = to_f64(o2), to_f64(o2) + to_f64(lo)
    # the residual is below half a bf16 ulp of o
    from helpers import bf16_ulp
    assert (np.abs(to_f64(lo)) <= 0.5 * bf16_ulp(hi) + 1e-30).all()
    e_hi = np.abs(hi - ro).mean() / np.abs(ro).mean()
    e_both = np.abs(both - ro).mean() / np.abs(ro).mean()
    assert e_both < 0.25 * e_hi and np.abs(both - ro).max() <= 2e-3, (e_hi, e_both)


# Short time sequences are packed in the forward too (G T <= 64); every output element is
# written (O and LSE start as NaN), including partial last groups of token positions.
PACKED_TIME_SHAPES = [
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


@pytest.mark.parametrize("shape", PACKED_TIME_SHAPES)
def test_time_forward_short_sequences_packed(oracle_mod, shape):
    B, T, S, Hq, Hkv, window = shape
    bits = inputs(B, T, S, Hq, Hkv, seed=500 + 7 * T + S)
    check(oracle_mod, "time", bits, window, 0.125, "packed %s" % (shape,))
