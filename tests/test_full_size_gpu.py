"""Full-size parity: the route the bench times, compared with the fp64 oracle element by element.

Minecraft dynamics layer (B=1, T=256, S=290, 30 Q / 3 KV heads, window 192, agent 289): the
forward writes O, LSE and O's residual; the backward takes Delta from O + O_lo and writes bf16
and fp32 gradients -- every element of O, LSE, dQ, dK and dV of both operators is checked.
CoinRun shapes (B=8, T=64, S=74, 8/2 heads): every element of the forward.  Tokenizer encoder
(B=2, T=32, S=1432, 24 MHA heads): 64 whole units per operator, forward and backward.

Gates (bf16 I/O, N(0,1) inputs): O per element within max(1e-2, one bf16 ulp of |ref|) and
mean |err| / mean |ref| <= 2e-3; LSE within 1e-3; fp32 gradients within 1e-2 and 2e-3;
bf16 gradients per element within max(1e-2, one bf16 ulp) and 2e-3.
"""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import LSE_ERR, MAX_ERR, MEAN_REL, bf16_ulp, to_dev

pytestmark = pytest.mark.gpu


class Acc:
    """Chunked comparison of a large tensor: worst err / bound and sum |err|, sum |ref|."""

    def __init__(self, what, max_err=MAX_ERR, mean_rel=MEAN_REL, bf16_out=True):
        self.what, self.max_err, self.mean_rel, self.bf16_out = what, max_err, mean_rel, bf16_out
        self.worst = 0.0
        self.err_sum = 0.0
        self.ref_sum = 0.0
        self.n = 0
        self.max_abs = 0.0

    def add(self, gpu, ref):
        assert np.isfinite(gpu).all(), "%s: non-finite values" % self.what
        d = np.abs(gpu - ref)
        bound = np.maximum(self.max_err, bf16_ulp(ref)) if self.bf16_out else self.max_err
        self.worst = max(self.worst, float((d / bound).max()))
        self.max_abs = max(self.max_abs, float(d.max()))
        self.err_sum += float(d.sum())
        self.ref_sum += float(np.abs(ref).sum())
        self.n += d.size

    def check(self):
        rel = (self.err_sum / self.n) / max(self.ref_sum / self.n, 1e-3)
        assert self.worst <= 1.0 and rel <= self.mean_rel, (
            "%s: max|err| %.3g (worst err/bound %.3g), mean rel %.3g (<= %.3g)" % (
                self.what, self.max_abs, self.worst, rel, self.mean_rel))
        return self.max_abs, rel


def _host(t):
    return t.detach().float().cpu().numpy()


def _compare_all(pairs, chunks=8):
    """pairs: (name, gpu tensor, oracle array, bf16_out); compares along axis 1 in chunks."""
    out = {}
    for name, g, r, bf16_out in pairs:
        acc = Acc(name, bf16_out=bf16_out)
        n1 = r.shape[1]
        step = max(1, (n1 + chunks - 1) // chunks)
        for a in range(0, n1, step):
            sl = (slice(None), slice(a, a + step))
            acc.add(_host(g[sl]).astype(np.float64), r[sl])
        out[name] = acc.check()
    return out


@pytest.mark.parametrize("kind", ["space", "time"])
def test_minecraft_fwd_bwd_every_element_bench_route(oracle_mod, kind):
    w = synth.WORKLOADS["minecraft_fwd_bwd"]
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    Q, K, V, DO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    extra = w.agent if kind == "space" else w.window
    fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
    bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
    # exactly the bench's calls: residual written by the forward, Delta from O + O_lo
    o, lse, lo = fwd(Q, K, V, extra, w.scale, o_lo=True)
    dq, dk, dv, (fq, fk, fv) = bwd(Q, K, V, o, lse, DO, extra, w.scale, fp32_grads=True, o_lo=lo)
    torch.cuda.synchronize()
    st, site = api.get_device_status_detail()
    assert st == 0, "device timeout at site word %#x" % site
    del Q, K, V, DO, lo
    X = oracle_mod.from_bf16
    orc = oracle_mod.space_bwd if kind == "space" else oracle_mod.time_bwd
    ro, rl, rdq, rdk, rdv = orc(X(q), X(k), X(v), X(do), extra, w.scale)
    del q, k, v, do
    lerr = float(np.abs(_host(lse).astype(np.float64) - rl).max())
    assert lerr <= LSE_ERR, "%s LSE max err %g" % (kind, lerr)
    res = _compare_all([
        ("%s O" % kind, o, ro, True),
        ("%s dQ fp32" % kind, fq, rdq, False), ("%s dQ bf16" % kind, dq, rdq, True),
        ("%s dK fp32" % kind, fk, rdk, False), ("%s dK bf16" % kind, dk, rdk, True),
        ("%s dV fp32" % kind, fv, rdv, False), ("%s dV bf16" % kind, dv, rdv, True),
    ])
    print("minecraft_fwd_bwd %s, every element: LSE max err %.2e; %s" % (
        kind, lerr, "; ".join("%s max %.2e mean rel %.2e" % (n, m, r) for n, (m, r) in res.items())))


def test_coinrun_forward_every_element(oracle_mod):
    w = synth.WORKLOADS["coinrun"]
    q, k, v = synth.make_inputs(w, with_dout=False)
    Q, K, V = to_dev(q), to_dev(k), to_dev(v)
    X = oracle_mod.from_bf16
    for kind in ("space", "time"):
        extra = w.agent if kind == "space" else w.window
        fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
        o, lse = fwd(Q, K, V, extra, w.scale)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        orc = oracle_mod.space_fwd if kind == "space" else oracle_mod.time_fwd
        ro, rl = orc(X(q), X(k), X(v), extra, w.scale)
        lerr = float(np.abs(_host(lse).astype(np.float64) - rl).max())
        assert lerr <= LSE_ERR, "coinrun %s LSE max err %g" % (kind, lerr)
        _compare_all([("coinrun %s O" % kind, o, ro, True)])


def test_tokenizer_encoder_64_whole_units(oracle_mod):
    """64 seeded whole units per operator: (b, t, head) blocks for space attention and
    (b, s, head) sequences for time attention, forward and backward on the bench route."""
    w = synth.WORKLOADS["tokenizer_enc"]
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    Q, K, V, DO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    X = oracle_mod.from_bf16
    rng = np.random.default_rng(w.seed + 64)
    n_units = 64
    for kind in ("space", "time"):
        extra = w.agent if kind == "space" else w.window
        fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
        bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
        o, lse, lo = fwd(Q, K, V, extra, w.scale, o_lo=True)
        dq, dk, dv, (fq, fk, fv) = bwd(Q, K, V, o, lse, DO, extra, w.scale, fp32_grads=True, o_lo=lo)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        F = w.T if kind == "space" else w.S
        picks = set()
        while len(picks) < n_units:
            picks.add((int(rng.integers(w.B)), int(rng.integers(F)), int(rng.integers(w.Hkv))))
        accs = {n: Acc("tokenizer_enc %s %s (%d units)" % (kind, n, n_units), bf16_out=bf)
                for n, bf in (("O", True), ("dQ fp32", False), ("dQ bf16", True), ("dK fp32", False),
                              ("dK bf16", True), ("dV fp32", False), ("dV bf16", True))}
        lerr = 0.0
        for b, f, h in sorted(picks):
            if kind == "space":
                sq = (slice(b, b + 1), slice(f, f + 1), slice(None), slice(h, h + 1))
            else:
                sq = (slice(b, b + 1), slice(None), slice(f, f + 1), slice(h, h + 1))
            orc = oracle_mod.space_bwd if kind == "space" else oracle_mod.time_bwd
            ro, rl, rdq, rdk, rdv = orc(X(q[sq]), X(k[sq]), X(v[sq]), X(do[sq]), extra, w.scale)
            lerr = max(lerr, float(np.abs(_host(lse[sq]).astype(np.float64) - rl).max()))
            for n, g, r in (("O", o, ro), ("dQ fp32", fq, rdq), ("dQ bf16", dq, rdq),
                            ("dK fp32", fk, rdk), ("dK bf16", dk, rdk), ("dV fp32", fv, rdv),
                            ("dV bf16", dv, rdv)):
                accs[n].add(_host(g[sq]).astype(np.float64), r)
        assert lerr <= LSE_ERR, "tokenizer_enc %s LSE max err %g" % (kind, lerr)
        for a in accs.values():
            a.check()
