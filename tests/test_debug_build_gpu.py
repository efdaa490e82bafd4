"""The range-checked debug build (libod_attn_debug.so, compiled with -DOD_DEBUG).

Its kernels check every TMA box start coordinate and every output row index against the
tensor's extent and report a failed check through the device status word (OD_ERR_RANGE),
without trapping.  On the edge shapes below -- ragged tiles, a single frame, MHA and a
10-head group, the packed short time sequences, variable-length blocks including empty
and one-token ones, the packed-QKV forms and rollout decode steps -- the debug build must
report a clean status and give results bit-identical to the regular build.
"""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api
from helpers import inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_causal_video_attention_b300 import build
    build.build_debug()
    assert b"debug" in api.debug_library().od_version()


def _both(fn):
    """fn() with the regular build, then with the debug build: (regular, debug) results."""
    torch.cuda.synchronize()
    ref = fn()
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    with api.debug_build():
        got = fn()
        torch.cuda.synchronize()
        st, site = api.get_device_status_detail()
        assert st == 0, "debug build: status %s, site word %#x" % (api.STATUS.get(st, st), site)
    return ref, got


def _flat(x):
    if isinstance(x, torch.Tensor):
        return [x]
    out = []
    for y in x:
        out += _flat(y)
    return out


def _same(ref, got, what):
    a, b = _flat(ref), _flat(got)
    assert len(a) == len(b)
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x, y), "%s: output %d differs between the builds" % (what, i)


SHAPES = [
    # B, T, S, Hq, Hkv, agent, window
    (2, 3, 150, 8, 2, 149, 2),     # ragged space tiles (32 tokens x 4 heads), short time
    (1, 33, 5, 10, 1, 0, 7),       # 10-head group, ragged 12-frame time tiles
    (1, 1, 37, 4, 4, 36, 1),       # one frame; MHA
    (1, 32, 9, 2, 1, -1, 32),      # packed time tiles (G T = 64)
    (1, 3, 21, 4, 2, 3, 3),        # packed time tiles (G T = 6), agent inside the block
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind", ["space", "time"])
def test_debug_build_matches_and_stays_in_range(shape, kind):
    B, T, S, Hq, Hkv, agent, window = shape
    q, k, v, do = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=77 + T + S, with_dout=True))
    fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
    bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
    extra = agent if kind == "space" else window

    def run():
        o, lse, lo = fwd(q, k, v, extra, 0.125, o_lo=True)
        g1 = bwd(q, k, v, o, lse, do, extra, 0.125, fp32_grads=True, o_lo=lo)
        g2 = bwd(q, k, v, o, lse, do, extra, 0.125, fp32_grads=True)
        return o, lse, lo, g1, g2
    ref, got = _both(run)
    _same(ref, got, "%s %s" % (kind, shape))


def test_debug_build_packed_qkv_and_varlen():
    B, T, S, Hq, Hkv = 2, 4, 130, 8, 2
    P = Hq + 2 * Hkv
    q, k, v, do = (to_dev(x) for x in inputs(B, T, S, Hq, Hkv, seed=99, with_dout=True))
    qkv = torch.cat([q, k, v], dim=3).contiguous()
    assert qkv.shape[3] == P
    seqlen = torch.tensor([0, 1, 130, 64, 129, 2, 96, 97], dtype=torch.int32, device="cuda")

    def run():
        res = []
        for kind, extra in (("space", 129), ("time", 3)):
            fwdp = api.space_attn_fwd_packed if kind == "space" else api.time_attn_fwd_packed
            bwdp = api.space_attn_bwd_packed if kind == "space" else api.time_attn_bwd_packed
            o, lse, lo = fwdp(qkv, Hq, extra, 0.125, o_lo=True)
            res += [o, lse, lo, bwdp(qkv, Hq, o, lse, do, extra, 0.125, fp32_grads=True, o_lo=lo)]
        o = torch.zeros_like(q)
        lse = torch.zeros((B, T, S, Hq), dtype=torch.float32, device="cuda")
        lo = torch.zeros_like(q)
        api.space_attn_fwd_varlen(q, k, v, seqlen, 5, 0.125, out=o, lse=lse, o_lo=lo)
        res += [o, lse, lo, api.space_attn_bwd_varlen(q, k, v, o, lse, do, seqlen, 5, 0.125,
                                                       fp32_grads=True, o_lo=lo)]
        return res
    ref, got = _both(run)
    _same(ref, got, "packed qkv / varlen")


def test_debug_build_decode_steps():
    B, S, Hq, Hkv, W = 2, 7, 10, 1, 5
    rng = np.random.default_rng(5)

    def bf(*shape):
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16).cuda()
    steps = [(bf(B, S, Hq, 64), bf(B, S, Hkv, 64), bf(B, S, Hkv, 64)) for _ in range(8)]

    def run():
        kc = torch.zeros((B, W, S, Hkv, 64), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        res = []
        for t, (qs, kn, vn) in enumerate(steps):
            res += list(api.time_attn_decode(qs, kn, vn, kc, vc, t, 0.125))
        return res + [kc, vc]
    ref, got = _both(run)
    _same(ref, got, "decode")
