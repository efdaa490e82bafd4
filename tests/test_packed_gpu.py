"""Packed-QKV calls: Q, K, V read from one [B,T,S,Hq+2*Hkv,D] tensor, dQ/dK/dV written into
one tensor of that shape.  They must give bit for bit what the unpacked calls give on the
same values, and match the fp64 oracle within the forward/backward tolerances."""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import LSE_ERR, assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, T, S, Hq, Hkv, agent, window
    (1, 8, 22, 4, 2, 21, 4),       # the tiny configuration
    (2, 9, 37, 6, 2, 36, 5),       # G = 3, ragged tiles
    (1, 6, 290, 30, 3, 289, 3),    # the dynamics head layout
    (1, 200, 3, 10, 1, 0, 192),    # G = 10 time attention with a window edge
    (1, 5, 40, 4, 4, -1, 5),       # MHA (tokenizer-like), no agent
]


def pack(q, k, v):
    return torch.cat([q, k, v], dim=3).contiguous()


@pytest.mark.parametrize("B,T,S,Hq,Hkv,agent,window", SHAPES)
def test_packed_equals_unpacked_and_matches_the_oracle(oracle_mod, B, T, S, Hq, Hkv, agent,
                                                       window):
    w = synth.custom(B, T, S, Hq, Hkv, window=window, agent=agent, seed=77)
    q_b, k_b, v_b, do_b = synth.make_inputs(w, with_dout=True)
    q, k, v, do = to_dev(q_b), to_dev(k_b), to_dev(v_b), to_dev(do_b)
    qkv = pack(q, k, v)
    X = oracle_mod.from_bf16
    for kind, extra in (("space", agent), ("time", window)):
        if kind == "space":
            o1, l1 = api.space_attn_fwd(q, k, v, extra, 0.125)
            o2, l2 = api.space_attn_fwd_packed(qkv, Hq, extra, 0.125)
            g1 = api.space_attn_bwd(q, k, v, o1, l1, do, extra, 0.125, fp32_grads=True)
            g2 = api.space_attn_bwd_packed(qkv, Hq, o2, l2, do, extra, 0.125, fp32_grads=True)
            ro, rl, rdq, rdk, rdv = oracle_mod.space_bwd(X(q_b), X(k_b), X(v_b), X(do_b), extra, 0.125)
        else:
            o1, l1 = api.time_attn_fwd(q, k, v, extra, 0.125)
            o2, l2 = api.time_attn_fwd_packed(qkv, Hq, extra, 0.125)
            g1 = api.time_attn_bwd(q, k, v, o1, l1, do, extra, 0.125, fp32_grads=True)
            g2 = api.time_attn_bwd_packed(qkv, Hq, o2, l2, do, extra, 0.125, fp32_grads=True)
            ro, rl, rdq, rdk, rdv = oracle_mod.time_bwd(X(q_b), X(k_b), X(v_b), X(do_b), extra, 0.125)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2), kind
        dq1, dk1, dv1, f1 = g1
        dqkv, f2 = g2
        assert torch.equal(pack(dq1, dk1, dv1), dqkv), kind
        for a, b in zip(f1, f2):
            assert torch.equal(a, b), kind
        # and against the oracle
        assert_close(to_f64(o2), ro, "%s packed O" % kind)
        assert np.abs(to_f64(l2) - rl).max() <= LSE_ERR
        for name, g, r in (("dQ", f2[0], rdq), ("dK", f2[1], rdk), ("dV", f2[2], rdv)):
            assert_close(to_f64(g), r, "%s packed %s" % (kind, name), bf16_out=False)


def test_packed_gradients_leave_the_inputs_untouched():
    w = synth.custom(1, 4, 30, 6, 2, window=3, agent=29, seed=78)
    q_b, k_b, v_b, do_b = synth.make_inputs(w, with_dout=True)
    qkv = pack(to_dev(q_b), to_dev(k_b), to_dev(v_b))
    before = qkv.clone()
    do = to_dev(do_b)
    o, l = api.space_attn_fwd_packed(qkv, 6, 29)
    dqkv = torch.full_like(qkv, float("nan"))
    api.space_attn_bwd_packed(qkv, 6, o, l, do, 29, out=dqkv)
    torch.cuda.synchronize()
    assert torch.equal(qkv, before)
    assert torch.isfinite(dqkv.float()).all()   # every head range of every token was written
    with pytest.raises(api.ODError):
        api.space_attn_bwd_packed(qkv, 6, o, l, do, 29, out=qkv)


def test_packed_with_output_residual_equals_unpacked():
    """Delta from O + O_lo, with Q/K/V (and the operand-range scan) read through the packed
    views: bit-identical to the separate tensors."""
    B, T, S, Hq, Hkv, agent, window = 1, 12, 290, 30, 3, 289, 8
    w = synth.custom(B, T, S, Hq, Hkv, window=window, agent=agent, seed=79)
    q_b, k_b, v_b, do_b = synth.make_inputs(w, with_dout=True)
    q, k, v, do = to_dev(q_b), to_dev(k_b), to_dev(v_b), to_dev(do_b)
    qkv = pack(q, k, v)
    for kind, extra in (("space", agent), ("time", window)):
        fwd = api.space_attn_fwd if kind == "space" else api.time_attn_fwd
        fwdp = api.space_attn_fwd_packed if kind == "space" else api.time_attn_fwd_packed
        bwd = api.space_attn_bwd if kind == "space" else api.time_attn_bwd
        bwdp = api.space_attn_bwd_packed if kind == "space" else api.time_attn_bwd_packed
        o1, l1, r1 = fwd(q, k, v, extra, 0.125, o_lo=True)
        o2, l2, r2 = fwdp(qkv, Hq, extra, 0.125, o_lo=True)
        assert torch.equal(r1, r2)
        g1 = bwd(q, k, v, o1, l1, do, extra, 0.125, o_lo=r1)
        g2 = bwdp(qkv, Hq, o2, l2, do, extra, 0.125, o_lo=r2)
        torch.cuda.synchronize()
        assert api.get_device_status() == 0
        assert torch.equal(pack(*g1), g2), kind
