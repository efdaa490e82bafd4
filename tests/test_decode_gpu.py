"""Decode-step parity: one rollout step of time attention over the ring-buffer KV cache,
CUDA library vs the fp64 oracle.

Tolerances as for the forward: max |err| <= 1e-2 and mean relative error <= 2e-3 for O,
|err| <= 1e-3 for the logsumexp; the cache update is compared bit for bit.
"""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import LSE_ERR, assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def normal(shape, seed, start=0):
    n = int(np.prod(shape))
    return synth.normal_bf16(seed, start, n).reshape(shape)


def bits_of(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def step(oracle_mod, q, kn, vn, kc, vc, t, scale, what):
    """One decode step on both sides; checks O, LSE and the caches, returns the GPU caches'
    bits after the step."""
    W = kc.shape[1]
    dkc, dvc = kc.clone(), vc.clone()
    kc_before, vc_before = bits_of(kc), bits_of(vc)
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    api.time_attn_decode(q, kn, vn, dkc, dvc, t, scale=scale, out=o, lse=lse)
    torch.cuda.synchronize()
    st, site = api.get_device_status_detail()
    assert st == 0, "device timeout at site word %#x" % site
    f = oracle_mod.from_bf16
    # the oracle reads only the window's slots; the others may hold anything (NaN here)
    ro, rl, rkc, rvc = oracle_mod.time_decode(f(bits_of(q)), f(bits_of(kn)), f(bits_of(vn)),
                                              f(kc_before), f(vc_before), t, scale)
    assert_close(to_f64(o), ro, "%s O" % what)
    gl = to_f64(lse)
    assert np.isfinite(gl).all()
    assert np.abs(gl - rl).max() <= LSE_ERR, "%s LSE err %g" % (what, np.abs(gl - rl).max())
    # cache: slot t mod W now holds the new frame; every other slot is untouched, bit for bit
    gk, gv = bits_of(dkc), bits_of(dvc)
    others = [i for i in range(W) if i != t % W]
    np.testing.assert_array_equal(gk[:, others], kc_before[:, others])
    np.testing.assert_array_equal(gv[:, others], vc_before[:, others])
    np.testing.assert_array_equal(gk[:, t % W], bits_of(kn))
    np.testing.assert_array_equal(gv[:, t % W], bits_of(vn))
    return dkc, dvc


@pytest.mark.parametrize("B,S,Hq,Hkv,W,T", [
    (2, 7, 4, 2, 5, 13),      # wraps the ring twice
    (1, 3, 10, 1, 70, 75),    # 2 key blocks, ragged tail, then the wrap
    (1, 2, 16, 1, 1, 4),      # W = 1: every step reads only its own frame; G = 16
    (2, 5, 3, 3, 64, 66),     # G = 1, a window of exactly one block
])
def test_rollout_from_an_uninitialised_cache(oracle_mod, B, S, Hq, Hkv, W, T):
    """Steps t = 0 .. T-1 from a cache whose unwritten slots hold NaN: no step may read a
    slot outside its window, and each step matches the oracle."""
    D, scale = 64, 0.125
    kc = torch.full((B, W, S, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    for t in range(T):
        q = to_dev(normal((B, S, Hq, D), 10 + t))
        kn = to_dev(normal((B, S, Hkv, D), 1000 + t))
        vn = to_dev(normal((B, S, Hkv, D), 2000 + t))
        kc, vc = step(oracle_mod, q, kn, vn, kc, vc, t, scale, "t=%d" % t)


@pytest.mark.parametrize("t,W", [(0, 192), (63, 192), (64, 192), (127, 192), (150, 192),
                                 (191, 192), (192, 192), (1000, 192), (700, 129), (5, 1)])
def test_window_edges_on_the_dynamics_head_layout(oracle_mod, t, W):
    """30 query / 3 KV heads; full caches of random frames; t spans 1 .. W keys, the exact
    block boundaries, the first wrap and a long rollout."""
    B, S, Hq, Hkv, D = 1, 9, 30, 3, 64
    kc = to_dev(normal((B, W, S, Hkv, D), 31))
    vc = to_dev(normal((B, W, S, Hkv, D), 32))
    q = to_dev(normal((B, S, Hq, D), 33))
    kn = to_dev(normal((B, S, Hkv, D), 34))
    vn = to_dev(normal((B, S, Hkv, D), 35))
    step(oracle_mod, q, kn, vn, kc, vc, t, 0.125, "t=%d W=%d" % (t, W))


def test_full_size_rollout_step_sampled(oracle_mod):
    """The measured decode workload (16 rollouts, S = 290, 30/3 heads, W = 192, steady state
    t = 500): the GPU step over all rollouts, checked against the oracle on rollouts 0, 7
    and 15 (units are independent across rollouts)."""
    B, S, Hq, Hkv, D, W, t = 16, 290, 30, 3, 64, 192, 500
    kc_bits = normal((B, W, S, Hkv, D), 41)
    vc_bits = normal((B, W, S, Hkv, D), 42)
    q_bits = normal((B, S, Hq, D), 43)
    kn_bits = normal((B, S, Hkv, D), 44)
    vn_bits = normal((B, S, Hkv, D), 45)
    kc, vc = to_dev(kc_bits), to_dev(vc_bits)
    o = torch.full((B, S, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    api.time_attn_decode(to_dev(q_bits), to_dev(kn_bits), to_dev(vn_bits), kc, vc, t,
                         scale=0.125, out=o, lse=lse)
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    go, gl = to_f64(o), to_f64(lse)
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    f = oracle_mod.from_bf16
    for b in (0, 7, 15):
        ro, rl, rkc, _ = oracle_mod.time_decode(f(q_bits[b:b + 1]), f(kn_bits[b:b + 1]),
                                                f(vn_bits[b:b + 1]), f(kc_bits[b:b + 1]),
                                                f(vc_bits[b:b + 1]), t, 0.125)
        assert_close(go[b:b + 1], ro, "rollout %d O" % b)
        assert np.abs(gl[b:b + 1] - rl).max() <= LSE_ERR
    gk = bits_of(kc)
    np.testing.assert_array_equal(gk[:, t % W], kn_bits)
    others = [i for i in range(W) if i != t % W]
    np.testing.assert_array_equal(gk[:, others[:5]], kc_bits[:, others[:5]])


def test_rollout_equals_the_training_time_forward():
    """Feeding frames 0..T-1 through the decode step gives the rows of the windowed time
    forward on the whole sequence (both CUDA paths, each held to the oracle elsewhere)."""
    B, T, S, Hq, Hkv, D, W = 1, 200, 4, 30, 3, 64, 192
    q = to_dev(normal((B, T, S, Hq, D), 51))
    k = to_dev(normal((B, T, S, Hkv, D), 52))
    v = to_dev(normal((B, T, S, Hkv, D), 53))
    o_full, l_full = api.time_attn_fwd(q, k, v, window=W, scale=0.125)
    kc = torch.zeros((B, W, S, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    o_dec = torch.empty_like(q)
    l_dec = torch.empty_like(l_full)
    for t in range(T):
        o, l = api.time_attn_decode(q[:, t].contiguous(), k[:, t].contiguous(),
                                    v[:, t].contiguous(), kc, vc, t, scale=0.125)
        o_dec[:, t] = o
        l_dec[:, t] = l
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    d = (o_dec.float() - o_full.float()).abs()
    assert d.max().item() <= 1.6e-2 and (d.mean() / o_full.float().abs().mean()).item() <= 2e-3
    assert (l_dec - l_full).abs().max().item() <= 1e-3


def test_decode_rejects_bad_tensors():
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros(1, 2, 2, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 3, 2, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        api.time_attn_decode(q, kn, kn, kc[:, :, :1].contiguous(), kc, 0)
    with pytest.raises(api.ODError):
        api.time_attn_decode(q, kn, kn, kc, kc.clone(), -1)
