"""Shared test helpers: seeded inputs on both sides, comparison against the oracle."""
import numpy as np
import torch

from block_causal_video_attention_b300 import synth

MAX_ERR = 1e-2      # max |gpu - oracle| for O (and fp32 gradients)
MEAN_REL = 2e-3     # mean |gpu - oracle| / mean |oracle|
LSE_ERR = 1e-3      # max |gpu - oracle| for the logsumexp


def to_dev(bits):
    """uint16 bf16 bit patterns (numpy) -> CUDA bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_f64(t):
    """CUDA tensor (bf16 or fp32) -> float64 numpy."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def inputs(B, T, S, Hq, Hkv, seed, with_dout=False):
    w = synth.custom(B, T, S, Hq, Hkv, seed=seed)
    return synth.make_inputs(w, with_dout=with_dout)


def errors(gpu, ref):
    """(max |err|, mean |err| / mean |ref|); the denominator is floored at 1e-3 so a
    reference that is exactly zero (e.g. dQ when every row reads only itself) is judged
    on absolute error."""
    d = np.abs(gpu - ref)
    return float(d.max()), float(d.mean() / max(np.abs(ref).mean(), 1e-3))


def bf16_ulp(x):
    """One unit in the last place of bf16 (8 significant bits) at |x|."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 0.0)


def assert_close(gpu, ref, what, max_err=MAX_ERR, mean_rel=MEAN_REL, bf16_out=True):
    """max |err| <= max_err per element -- for a bf16 output, max(max_err, 1 bf16 ulp of
    |ref|), since rounding the exact value to bf16 alone can exceed max_err once |ref| >= 4
    -- and mean |err| / mean |ref| <= mean_rel over the tensor."""
    assert np.isfinite(gpu).all(), "%s: non-finite values" % what
    m, r = errors(gpu, ref)
    bound = np.maximum(max_err, bf16_ulp(ref)) if bf16_out else max_err
    worst = float((np.abs(gpu - ref) / bound).max())
    assert worst <= 1.0 and r <= mean_rel, (
        "%s: max|err| %.3g (worst err/bound %.3g), mean rel %.3g (<= %.3g)" % (
            what, m, worst, r, mean_rel))
    return m, r
