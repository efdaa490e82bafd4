"""Pins for the fp64 oracle: it is checked here against things other than itself.

* an independent dense-mask formulation over the flattened B*T*S*H rows,
* torch's scaled_dot_product_attention / autograd in float64 on the CPU,
* closed forms (q = 0 gives a uniform softmax), special cases (W = 1, T = 1,
  S = 1, W >= T, no agent, G = 1, replicated KV heads),
* invariants named by the pages' rules: causality, the agent-token read
  restriction, the window, row-stochastic weights, permutation equivariance,
* fp64 central finite differences for the backward and two exact gradient
  identities.
"""
import json
import os

import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ----------------------------------------------------------------------------
# independent dense-mask formulation (written from the rules, not the oracle)
# ----------------------------------------------------------------------------
def dense_mask(B, T, S, Hq, Hkv, kind, agent=-1, window=1):
    G = Hq // Hkv
    qb, qt, qs, qh = [a.ravel() for a in np.meshgrid(np.arange(B), np.arange(T), np.arange(S),
                                                     np.arange(Hq), indexing="ij")]
    kb, kt, ks, kh = [a.ravel() for a in np.meshgrid(np.arange(B), np.arange(T), np.arange(S),
                                                     np.arange(Hkv), indexing="ij")]
    same = (qb[:, None] == kb[None, :]) & ((qh // G)[:, None] == kh[None, :])
    if kind == "space":
        agent_col = (ks[None, :] == agent) & (qs[:, None] != agent)
        return same & (qt[:, None] == kt[None, :]) & ~agent_col
    d = qt[:, None] - kt[None, :]
    return same & (qs[:, None] == ks[None, :]) & (d >= 0) & (d < window)


def dense_attention(q, k, v, mask, scale):
    B, T, S, Hq, D = q.shape
    Q = q.reshape(-1, D)
    K = k.reshape(-1, D)
    V = v.reshape(-1, D)
    logits = np.where(mask, scale * (Q @ K.T), -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    z = e.sum(axis=1, keepdims=True)
    P = e / z
    O = P @ V
    lse = (m + np.log(z)).ravel()
    return O.reshape(q.shape), lse.reshape(B, T, S, Hq), P


SHAPES = [
    # B, T, S, Hq, Hkv, agent, window
    (1, 8, 22, 4, 2, 21, 4),
    (2, 5, 7, 6, 3, 0, 2),
    (1, 6, 9, 4, 1, 4, 6),
    (2, 4, 5, 2, 2, -1, 9),
    (1, 3, 1, 3, 1, 0, 1),
]


@pytest.mark.parametrize("B,T,S,Hq,Hkv,agent,window", SHAPES)
def test_forward_matches_dense_formulation(oracle_mod, B, T, S, Hq, Hkv, agent, window):
    D = 16
    q, k, v = rnd((B, T, S, Hq, D), 1), rnd((B, T, S, Hkv, D), 2), rnd((B, T, S, Hkv, D), 3)
    sc = 0.3
    o, lse = oracle_mod.space_fwd(q, k, v, agent, sc, nthreads=2)
    O, L, _ = dense_attention(q, k, v, dense_mask(B, T, S, Hq, Hkv, "space", agent=agent), sc)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-12)
    o, lse = oracle_mod.time_fwd(q, k, v, window, sc, nthreads=2)
    O, L, _ = dense_attention(q, k, v, dense_mask(B, T, S, Hq, Hkv, "time", window=window), sc)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-12)


def _torch_reference(q, k, v, kind, agent, window, scale):
    """torch fp64: SDPA on per-frame / per-position sequences, KV repeated per group."""
    B, T, S, Hq, D = q.shape
    G = Hq // k.shape[3]
    tq, tk, tv = (torch.tensor(a) for a in (q, k, v))
    tk = tk.repeat_interleave(G, dim=3)
    tv = tv.repeat_interleave(G, dim=3)
    if kind == "space":   # sequences over s: [B,T,H,S,D]
        perm = (0, 1, 3, 2, 4)
        L = S
        i = torch.arange(L)
        allowed = ~((i[None, :] == agent) & (i[:, None] != agent))
    else:                 # sequences over t: [B,S,H,T,D]
        perm = (0, 2, 3, 1, 4)
        L = T
        i = torch.arange(L)
        d = i[:, None] - i[None, :]
        allowed = (d >= 0) & (d < window)
    qq, kk, vv = (x.permute(*perm) for x in (tq, tk, tv))
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=allowed,
                                                           scale=scale)
    logits = (qq @ kk.transpose(-1, -2)) * scale
    lse = torch.logsumexp(logits.masked_fill(~allowed, float("-inf")), dim=-1)
    inv = np.argsort(perm)
    return out.permute(*inv).numpy(), lse.permute(*inv[:4]).numpy()


@pytest.mark.parametrize("B,T,S,Hq,Hkv,agent,window", SHAPES)
def test_forward_matches_torch_sdpa(oracle_mod, B, T, S, Hq, Hkv, agent, window):
    D = 8
    q, k, v = rnd((B, T, S, Hq, D), 4), rnd((B, T, S, Hkv, D), 5), rnd((B, T, S, Hkv, D), 6)
    sc = 1.0 / np.sqrt(D)
    o, lse = oracle_mod.space_fwd(q, k, v, agent, sc)
    O, L = _torch_reference(q, k, v, "space", agent, window, sc)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-12)
    o, lse = oracle_mod.time_fwd(q, k, v, window, sc)
    O, L = _torch_reference(q, k, v, "time", agent, window, sc)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-12)


def test_zero_query_closed_form(oracle_mod):
    """q = 0 makes every allowed logit 0: LSE = ln |allowed set|, O = mean of allowed V."""
    B, T, S, Hq, Hkv, D, a, W = 2, 7, 6, 4, 2, 8, 2, 3
    q = np.zeros((B, T, S, Hq, D))
    k, v = rnd((B, T, S, Hkv, D), 7), rnd((B, T, S, Hkv, D), 8)
    G = Hq // Hkv
    o, lse = oracle_mod.space_fwd(q, k, v, a)
    for s in range(S):
        n = S if s == a else S - 1
        np.testing.assert_allclose(lse[:, :, s, :], np.log(n), rtol=0, atol=1e-14)
        keys = [j for j in range(S) if j == s or j != a] if s == a else [j for j in range(S) if j != a]
        for h in range(Hq):
            np.testing.assert_allclose(o[:, :, s, h], v[:, :, keys, h // G].mean(axis=2),
                                       rtol=0, atol=1e-14)
    o, lse = oracle_mod.time_fwd(q, k, v, W)
    for t in range(T):
        lo = max(0, t - W + 1)
        np.testing.assert_allclose(lse[:, t], np.log(t - lo + 1), rtol=0, atol=1e-14)
        for h in range(Hq):
            np.testing.assert_allclose(o[:, t, :, h], v[:, lo:t + 1, :, h // G].mean(axis=1),
                                       rtol=0, atol=1e-14)


def test_single_key_special_cases(oracle_mod):
    """W = 1, T = 1 (time) and S = 1 (space): each row reads only itself."""
    B, T, S, Hq, Hkv, D = 2, 5, 4, 6, 3, 8
    G = Hq // Hkv
    q, k, v = rnd((B, T, S, Hq, D), 9), rnd((B, T, S, Hkv, D), 10), rnd((B, T, S, Hkv, D), 11)
    kr = np.repeat(k, G, axis=3)
    vr = np.repeat(v, G, axis=3)
    self_logit = 0.125 * (q * kr).sum(-1)
    o, lse = oracle_mod.time_fwd(q, k, v, 1, 0.125)
    np.testing.assert_allclose(o, vr, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, self_logit, rtol=0, atol=1e-14)
    o, lse = oracle_mod.time_fwd(q[:, :1], k[:, :1], v[:, :1], 7, 0.125)
    np.testing.assert_allclose(o, vr[:, :1], rtol=0, atol=1e-15)
    o, lse = oracle_mod.space_fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], 0, 0.125)
    np.testing.assert_allclose(o, vr[:, :, :1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, self_logit[:, :, :1], rtol=0, atol=1e-14)


def test_window_at_least_T_is_plain_causal_and_gqa_equals_replicated_mha(oracle_mod):
    B, T, S, Hq, Hkv, D = 1, 9, 3, 4, 2, 8
    G = Hq // Hkv
    q, k, v = rnd((B, T, S, Hq, D), 12), rnd((B, T, S, Hkv, D), 13), rnd((B, T, S, Hkv, D), 14)
    o1, l1 = oracle_mod.time_fwd(q, k, v, T)
    o2, l2 = oracle_mod.time_fwd(q, k, v, T + 50)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    kr, vr = np.repeat(k, G, axis=3), np.repeat(v, G, axis=3)
    o3, l3 = oracle_mod.time_fwd(q, kr, vr, 4)
    o4, l4 = oracle_mod.time_fwd(q, k, v, 4)
    np.testing.assert_array_equal(o3, o4)
    o5, _ = oracle_mod.space_fwd(q, kr, vr, 1)
    o6, _ = oracle_mod.space_fwd(q, k, v, 1)
    np.testing.assert_array_equal(o5, o6)


def test_causality_and_window_invariants(oracle_mod):
    """Perturbing frames after t leaves rows <= t bit-identical; frames before
    t-W+1 do not affect row t."""
    B, T, S, Hq, Hkv, D, W = 1, 10, 3, 4, 2, 8, 3
    q, k, v = rnd((B, T, S, Hq, D), 15), rnd((B, T, S, Hkv, D), 16), rnd((B, T, S, Hkv, D), 17)
    o, lse = oracle_mod.time_fwd(q, k, v, W)
    for t0 in (0, 4, 9):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[:, t0 + 1:] += 5.0
        k2[:, t0 + 1:] -= 3.0
        v2[:, t0 + 1:] *= -7.0
        o2, l2 = oracle_mod.time_fwd(q2, k2, v2, W)
        np.testing.assert_array_equal(o2[:, :t0 + 1], o[:, :t0 + 1])
        np.testing.assert_array_equal(l2[:, :t0 + 1], lse[:, :t0 + 1])
    t = 7
    k3, v3 = k.copy(), v.copy()
    k3[:, :t - W + 1] += 9.0
    v3[:, :t - W + 1] += 9.0
    o3, l3 = oracle_mod.time_fwd(q, k3, v3, W)
    np.testing.assert_array_equal(o3[:, t], o[:, t])
    np.testing.assert_array_equal(l3[:, t], lse[:, t])
    assert not np.array_equal(o3[:, t - 1], o[:, t - 1])


@pytest.mark.parametrize("agent", [0, 5, 8])
def test_agent_token_is_unreadable_by_world_tokens(oracle_mod, agent):
    B, T, S, Hq, Hkv, D = 2, 3, 9, 4, 2, 8
    q, k, v = rnd((B, T, S, Hq, D), 18), rnd((B, T, S, Hkv, D), 19), rnd((B, T, S, Hkv, D), 20)
    o, lse = oracle_mod.space_fwd(q, k, v, agent)
    k2, v2, q2 = k.copy(), v.copy(), q.copy()
    k2[:, :, agent] += 4.0
    v2[:, :, agent] *= -3.0
    q2[:, :, agent] += 1.0
    o2, l2 = oracle_mod.space_fwd(q2, k2, v2, agent)
    world = [s for s in range(S) if s != agent]
    np.testing.assert_array_equal(o2[:, :, world], o[:, :, world])
    np.testing.assert_array_equal(l2[:, :, world], lse[:, :, world])
    assert not np.array_equal(o2[:, :, agent], o[:, :, agent])


def test_rows_are_stochastic(oracle_mod):
    """With one-hot values (D >= keys) O reveals the softmax weights: >= 0, sum 1."""
    T, S = 5, 6
    D = max(T, S)
    q = rnd((1, T, S, 2, D), 21)
    k = rnd((1, T, S, 1, D), 22)
    v = np.zeros((1, T, S, 1, D))
    for s in range(S):
        v[0, :, s, 0, s] = 1.0
    o, _ = oracle_mod.space_fwd(q, k, v, 2)
    assert (o >= 0).all()
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-15)
    assert np.all(o[0, :, [s for s in range(S) if s != 2], :, 2] == 0.0)
    v = np.zeros((1, T, S, 1, D))
    for t in range(T):
        v[0, t, :, 0, t] = 1.0
    o, _ = oracle_mod.time_fwd(q, k, v, 3)
    assert (o >= 0).all()
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-15)
    for t in range(T):
        for tp in range(T):
            if not (t - 3 < tp <= t):
                assert np.all(o[0, t, :, :, tp] == 0.0)


def test_permutation_equivariance_of_world_tokens(oracle_mod):
    B, T, S, Hq, Hkv, D, a = 1, 2, 7, 2, 1, 8, 6
    q, k, v = rnd((B, T, S, Hq, D), 23), rnd((B, T, S, Hkv, D), 24), rnd((B, T, S, Hkv, D), 25)
    perm = np.array([3, 0, 5, 1, 4, 2, 6])  # agent stays at 6
    o, lse = oracle_mod.space_fwd(q, k, v, a)
    o2, l2 = oracle_mod.space_fwd(q[:, :, perm], k[:, :, perm], v[:, :, perm], a)
    np.testing.assert_allclose(o2, o[:, :, perm], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l2, lse[:, :, perm], rtol=0, atol=1e-14)


# ----------------------------------------------------------------------------
# backward
# ----------------------------------------------------------------------------
def _loss(oracle_mod, kind, q, k, v, dout, extra):
    f = oracle_mod.space_fwd if kind == "space" else oracle_mod.time_fwd
    o, _ = f(q, k, v, extra, 0.5, nthreads=1)
    return float((o * dout).sum())


@pytest.mark.parametrize("kind,extra", [("space", 2), ("space", -1), ("time", 2), ("time", 5)])
def test_backward_matches_finite_differences(oracle_mod, kind, extra):
    B, T, S, Hq, Hkv, D = 1, 4, 4, 4, 2, 4
    q, k, v = rnd((B, T, S, Hq, D), 26), rnd((B, T, S, Hkv, D), 27), rnd((B, T, S, Hkv, D), 28)
    dout = rnd((B, T, S, Hq, D), 29)
    f = oracle_mod.space_bwd if kind == "space" else oracle_mod.time_bwd
    _, _, dq, dk, dv = f(q, k, v, dout, extra, 0.5, nthreads=1)
    h = 1e-5
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = x[i]
            x[i] = old + h
            lp = _loss(oracle_mod, kind, q, k, v, dout, extra)
            x[i] = old - h
            lm = _loss(oracle_mod, kind, q, k, v, dout, extra)
            x[i] = old
            num[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("kind,extra", [("space", 3), ("time", 3)])
def test_backward_matches_torch_autograd(oracle_mod, kind, extra):
    B, T, S, Hq, Hkv, D = 2, 6, 5, 6, 2, 8
    q, k, v = rnd((B, T, S, Hq, D), 30), rnd((B, T, S, Hkv, D), 31), rnd((B, T, S, Hkv, D), 32)
    dout = rnd((B, T, S, Hq, D), 33)
    sc = 1.0 / np.sqrt(D)
    f = oracle_mod.space_bwd if kind == "space" else oracle_mod.time_bwd
    o, lse, dq, dk, dv = f(q, k, v, dout, extra, sc)
    mask = dense_mask(B, T, S, Hq, Hkv, kind, agent=extra, window=extra)
    tq, tk, tv = (torch.tensor(a.reshape(-1, D), requires_grad=True) for a in (q, k, v))
    logits = (tq @ tk.T * sc).masked_fill(~torch.tensor(mask), float("-inf"))
    O = torch.softmax(logits, dim=1) @ tv
    (O * torch.tensor(dout.reshape(-1, D))).sum().backward()
    np.testing.assert_allclose(o.reshape(-1, D), O.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq.reshape(-1, D), tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk.reshape(-1, D), tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv.reshape(-1, D), tv.grad.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("kind,extra", [("space", 4), ("space", -1), ("time", 3)])
def test_backward_identities(oracle_mod, kind, extra):
    """sum over keys of dV equals the group's summed dO rows (rows of P sum to 1);
    sum over keys of dK is 0 (each row's dS sums to 0: softmax is shift-invariant)."""
    B, T, S, Hq, Hkv, D = 2, 5, 6, 6, 3, 8
    G = Hq // Hkv
    q, k, v = rnd((B, T, S, Hq, D), 34), rnd((B, T, S, Hkv, D), 35), rnd((B, T, S, Hkv, D), 36)
    dout = rnd((B, T, S, Hq, D), 37)
    f = oracle_mod.space_bwd if kind == "space" else oracle_mod.time_bwd
    _, _, dq, dk, dv = f(q, k, v, dout, extra, 0.125)
    grp = dout.reshape(B, T, S, Hkv, G, D).sum(axis=4)
    if kind == "space":
        np.testing.assert_allclose(dv.sum(axis=2), grp.sum(axis=2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    else:
        np.testing.assert_allclose(dv.sum(axis=1), grp.sum(axis=1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-12)


def test_backward_causal_and_agent_zero_gradients(oracle_mod):
    B, T, S, Hq, Hkv, D, a = 1, 6, 5, 4, 2, 8, 4
    q, k, v = rnd((B, T, S, Hq, D), 38), rnd((B, T, S, Hkv, D), 39), rnd((B, T, S, Hkv, D), 40)
    dout = rnd((B, T, S, Hq, D), 41)
    d2 = dout.copy()
    d2[:, 3:] = 0.0  # no upstream gradient from rows t >= 3
    _, _, dq, dk, dv = oracle_mod.time_bwd(q, k, v, d2, 4)
    assert np.all(dk[:, 3:] == 0.0) and np.all(dv[:, 3:] == 0.0) and np.all(dq[:, 3:] == 0.0)
    d3 = dout.copy()
    d3[:, :, a] = 0.0  # only world rows carry gradient: the agent's K/V get none
    _, _, dq, dk, dv = oracle_mod.space_bwd(q, k, v, d3, a)
    assert np.all(dk[:, :, a] == 0.0) and np.all(dv[:, :, a] == 0.0)
    assert not np.all(dk[:, :, 0] == 0.0)


# ----------------------------------------------------------------------------
# variable-length space attention
# ----------------------------------------------------------------------------
def test_varlen_space_attention_is_the_dense_rule_per_block(oracle_mod):
    """Each block equals the independent dense-mask formulation over its first L tokens;
    full lengths reproduce the fixed-length oracle bit for bit; padding tokens affect nothing."""
    B, T, S, Hq, Hkv, D, a, sc = 2, 3, 11, 4, 2, 8, 3, 0.3
    q, k, v = rnd((B, T, S, Hq, D), 80), rnd((B, T, S, Hkv, D), 81), rnd((B, T, S, Hkv, D), 82)
    L = np.array([[11, 1, 4], [0, 7, 3]])
    o, lse = oracle_mod.space_fwd_varlen(q, k, v, L, a, sc)
    for b in range(B):
        for t in range(T):
            n = L[b, t]
            assert np.isnan(o[b, t, n:]).all() and np.isnan(lse[b, t, n:]).all()
            if n == 0:
                continue
            sl = (slice(b, b + 1), slice(t, t + 1), slice(0, n))
            m = dense_mask(1, 1, n, Hq, Hkv, "space", a if a < n else -1)
            O, LSE, _ = dense_attention(q[sl], k[sl], v[sl], m, sc)
            np.testing.assert_allclose(o[b, t, :n], O[0, 0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, t, :n], LSE[0, 0], rtol=0, atol=1e-12)
    full = np.full((B, T), S)
    o1, l1 = oracle_mod.space_fwd_varlen(q, k, v, full, a, sc)
    o2, l2 = oracle_mod.space_fwd(q, k, v, a, sc)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # padding tokens (past each block's length) change no valid output
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for b in range(B):
        for t in range(T):
            n = L[b, t]
            q2[b, t, n:] += 5.0
            k2[b, t, n:] -= 3.0
            v2[b, t, n:] *= 7.0
    o3, l3 = oracle_mod.space_fwd_varlen(q2, k2, v2, L, a, sc)
    np.testing.assert_array_equal(np.nan_to_num(o3, nan=9.0), np.nan_to_num(o, nan=9.0))
    np.testing.assert_array_equal(np.nan_to_num(l3, nan=9.0), np.nan_to_num(lse, nan=9.0))
    # a one-token block reads only itself
    G = Hq // Hkv
    np.testing.assert_array_equal(o[0, 1, 0], np.repeat(v[0, 1, 0], G, axis=0))


def test_varlen_space_backward_matches_autograd_per_block(oracle_mod):
    B, T, S, Hq, Hkv, D, a, sc = 1, 2, 9, 4, 2, 8, 8, 0.25
    q, k, v = rnd((B, T, S, Hq, D), 83), rnd((B, T, S, Hkv, D), 84), rnd((B, T, S, Hkv, D), 85)
    do = rnd((B, T, S, Hq, D), 86)
    L = np.array([[9, 5]])
    _, _, dq, dk, dv = oracle_mod.space_bwd_varlen(q, k, v, do, L, a, sc)
    G = Hq // Hkv
    for t in range(T):
        n = L[0, t]
        qt = torch.tensor(q[0, t, :n], requires_grad=True)
        kt = torch.tensor(k[0, t, :n], requires_grad=True)
        vt = torch.tensor(v[0, t, :n], requires_grad=True)
        m = torch.ones(n, n, dtype=torch.bool)
        if a < n:
            m[:, a] = False
            m[a, a] = True
        kr, vr = kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt.transpose(0, 1), kr.transpose(0, 1), vr.transpose(0, 1), attn_mask=m, scale=sc)
        o.backward(torch.tensor(do[0, t, :n]).transpose(0, 1))
        np.testing.assert_allclose(dq[0, t, :n], qt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk[0, t, :n], kt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[0, t, :n], vt.grad.numpy(), rtol=0, atol=1e-12)
        assert np.isnan(dq[0, t, n:]).all() and np.isnan(dk[0, t, n:]).all()


# ----------------------------------------------------------------------------
# decode step over a ring-buffer KV cache
# ----------------------------------------------------------------------------
def _rollout(oracle_mod, q, k, v, W, scale, fill=0.0):
    """Feeds frames 0..T-1 one at a time through the decode step, starting from a
    cache filled with `fill`; returns the per-frame outputs and the final caches."""
    B, T, S, Hq, D = q.shape
    Hkv = k.shape[3]
    kc = np.full((B, W, S, Hkv, D), fill)
    vc = np.full((B, W, S, Hkv, D), fill)
    os_, ls_ = [], []
    for t in range(T):
        o, lse, kc, vc = oracle_mod.time_decode(q[:, t], k[:, t], v[:, t], kc, vc, t, scale)
        os_.append(o)
        ls_.append(lse)
    return np.stack(os_, 1), np.stack(ls_, 1), kc, vc


@pytest.mark.parametrize("B,T,S,Hq,Hkv,W", [(1, 9, 3, 4, 2, 4), (2, 6, 5, 6, 3, 6),
                                             (1, 7, 2, 3, 1, 1), (2, 5, 3, 2, 2, 9)])
def test_decode_rollout_matches_sdpa_over_the_window(oracle_mod, B, T, S, Hq, Hkv, W):
    """A rollout of T decode steps reproduces, frame by frame, torch's float64 SDPA over
    the frames max(0, t-W+1)..t (ring wrap-around included when T > W); the cache's
    unwritten slots hold values (1e300) that would poison any read of them."""
    D, sc = 8, 0.3
    G = Hq // Hkv
    q, k, v = rnd((B, T, S, Hq, D), 60), rnd((B, T, S, Hkv, D), 61), rnd((B, T, S, Hkv, D), 62)
    o, lse, kc, vc = _rollout(oracle_mod, q, k, v, W, sc, fill=1e300)
    for t in range(T):
        lo = max(0, t - W + 1)
        qt = torch.from_numpy(q[:, t]).permute(0, 1, 2, 3).reshape(B * S, Hq, 1, D)
        kt = torch.from_numpy(np.repeat(k[:, lo:t + 1], G, axis=3)).permute(0, 2, 3, 1, 4)
        vt = torch.from_numpy(np.repeat(v[:, lo:t + 1], G, axis=3)).permute(0, 2, 3, 1, 4)
        kt = kt.reshape(B * S, Hq, t + 1 - lo, D)
        vt = vt.reshape(B * S, Hq, t + 1 - lo, D)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=sc)
        np.testing.assert_allclose(o[:, t], ref.reshape(B, S, Hq, D).numpy(), rtol=0, atol=1e-12)
        logits = torch.einsum("nhd,nhkd->nhk", qt[:, :, 0], kt) * sc
        np.testing.assert_allclose(lse[:, t], torch.logsumexp(logits, -1).reshape(B, S, Hq).numpy(),
                                   rtol=0, atol=1e-12)
    # the final cache holds frame f in slot f mod W for the last min(T, W) frames
    for f in range(max(0, T - W), T):
        np.testing.assert_array_equal(kc[:, f % W], k[:, f])
        np.testing.assert_array_equal(vc[:, f % W], v[:, f])


def test_decode_rollout_equals_the_windowed_time_forward(oracle_mod):
    """The decode step and the full-sequence time forward are two routes to the same rows."""
    B, T, S, Hq, Hkv, D, W = 1, 11, 4, 6, 2, 8, 4
    q, k, v = rnd((B, T, S, Hq, D), 63), rnd((B, T, S, Hkv, D), 64), rnd((B, T, S, Hkv, D), 65)
    o, lse, _, _ = _rollout(oracle_mod, q, k, v, W, 0.125)
    O, L = oracle_mod.time_fwd(q, k, v, W, 0.125)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-13)


def test_decode_first_frame_and_zero_query_closed_forms(oracle_mod):
    """t = 0 reads only the new frame: O = v_new, LSE = scale <q, k_new>.  q = 0 gives
    LSE = ln min(t+1, W) and O = the mean of V over the window's frames."""
    B, S, Hq, Hkv, D, W = 2, 3, 4, 2, 8, 5
    G = Hq // Hkv
    q, kn, vn = rnd((B, S, Hq, D), 66), rnd((B, S, Hkv, D), 67), rnd((B, S, Hkv, D), 68)
    kc, vc = rnd((B, W, S, Hkv, D), 69), rnd((B, W, S, Hkv, D), 70)
    o, lse, _, _ = oracle_mod.time_decode(q, kn, vn, kc, vc, 0, 0.25)
    np.testing.assert_array_equal(o, np.repeat(vn, G, axis=2))
    np.testing.assert_allclose(lse, 0.25 * (q * np.repeat(kn, G, axis=2)).sum(-1), rtol=0, atol=1e-15)
    for t in (2, 4, 5, 13):
        o, lse, kc2, vc2 = oracle_mod.time_decode(np.zeros_like(q), kn, vn, kc, vc, t, 0.25)
        n = min(t + 1, W)
        np.testing.assert_allclose(lse, np.log(n), rtol=0, atol=1e-15)
        frames = [(f % W) for f in range(max(0, t - W + 1), t + 1)]
        mean_v = vc2[:, frames].mean(axis=1)
        np.testing.assert_allclose(o, np.repeat(mean_v, G, axis=2), rtol=0, atol=1e-14)


def test_decode_writes_only_the_new_frames_slot(oracle_mod):
    B, S, Hq, Hkv, D, W, t = 2, 3, 4, 2, 8, 6, 15
    q, kn, vn = rnd((B, S, Hq, D), 71), rnd((B, S, Hkv, D), 72), rnd((B, S, Hkv, D), 73)
    kc, vc = rnd((B, W, S, Hkv, D), 74), rnd((B, W, S, Hkv, D), 75)
    _, _, kc2, vc2 = oracle_mod.time_decode(q, kn, vn, kc, vc, t)
    others = [i for i in range(W) if i != t % W]
    np.testing.assert_array_equal(kc2[:, others], kc[:, others])
    np.testing.assert_array_equal(vc2[:, others], vc[:, others])
    np.testing.assert_array_equal(kc2[:, t % W], kn)
    np.testing.assert_array_equal(vc2[:, t % W], vn)


# ----------------------------------------------------------------------------
# workload shapes and the input generator
# ----------------------------------------------------------------------------
def test_workload_shapes_follow_the_pages():
    facts = {k: v["value"] for k, v in json.load(open(os.path.join(HERE, "golden",
                                                                   "page_facts.json"))).items()
             if not k.startswith("_")}
    mc = synth.WORKLOADS["minecraft_fwd"]
    spatial = facts["tokenizer_latents_per_frame"] // facts["packing_factor"]
    assert mc.S == spatial + facts["registers_per_timestep"] + 1 + 1  # + action + agent
    assert mc.Hq == facts["dynamics_q_heads"] and mc.Hkv == facts["dynamics_kv_heads"]
    assert mc.D == facts["dynamics_d_model"] // facts["dynamics_q_heads"]
    assert mc.window == facts["time_window_steps"] and mc.T == facts["frames_per_gpu"]
    assert mc.agent == mc.S - 1
    tk = synth.WORKLOADS["tokenizer_enc"]
    h, w = facts["padded_frame_hw"]
    p = facts["patch_size"]
    assert tk.S == (h // p) * (w // p) + facts["tokenizer_latents_per_frame"]
    assert tk.Hq * tk.D == facts["tokenizer_encoder_d_model"]
    td = synth.WORKLOADS["tokenizer_dec"]
    assert td.S == tk.S and td.Hq * td.D == facts["tokenizer_decoder_d_model"]
    assert (h // p) * (w // p) == facts["tokenizer_patches_per_frame"]
    # blocks of an encoder that drops its masked patches: 512 latents + the kept patches,
    # a mask ratio of at most 0.9 keeping at least 92 of the 920
    lat, pat = facts["tokenizer_latents_per_frame"], facts["tokenizer_patches_per_frame"]
    L = synth.mae_block_lengths(64, 32, 7)
    kept_min = round(pat * (1 - facts["mae_max_mask_probability"]))
    assert L.dtype == np.int32 and L.min() >= lat + kept_min and L.max() <= lat + pat
    assert L.max() - L.min() > 0.7 * pat   # the ratios cover most of [0, 0.9]
    assert synth.WORKLOADS["minecraft_fwd_bwd"].q_shape() == mc.q_shape()


def test_generator_is_the_stated_splitmix_box_muller():
    # splitmix64 from state 0: first output is the published test value.
    u = synth._uniform(0, 0, 1)
    first = 0xE220A8397B1DCDAF
    assert u[0] == ((first >> 11) + 1) * 2.0 ** -53
    a = synth.normal_bf16(7, 0, 1000)
    b = synth.normal_bf16(7, 0, 600)
    c = synth.normal_bf16(7, 600, 400)
    np.testing.assert_array_equal(a, np.concatenate([b, c]))
    z = synth.bf16_bits_to_f64(synth.normal_bf16(3, 0, 200000))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    q, k, v = synth.make_inputs(synth.WORKLOADS["tiny"])
    assert q.dtype == np.uint16 and q.shape == (1, 8, 22, 4, 64) and k.shape == (1, 8, 22, 2, 64)
