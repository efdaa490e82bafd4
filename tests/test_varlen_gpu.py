"""Variable-length space attention parity: per-block lengths on the padded layout, CUDA
library vs the fp64 oracle (valid rows element by element; padding rows must be left as they
were)."""
import numpy as np
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import LSE_ERR, assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

SENT = 7.0  # sentinel the padding rows of every output must keep


def run(oracle_mod, B, T, S, Hq, Hkv, agent, lengths, seed, with_lo):
    w = synth.custom(B, T, S, Hq, Hkv, agent=agent, seed=seed)
    q_b, k_b, v_b, do_b = synth.make_inputs(w, with_dout=True)
    q, k, v, do = to_dev(q_b), to_dev(k_b), to_dev(v_b), to_dev(do_b)
    L = torch.tensor(np.asarray(lengths, dtype=np.int32).reshape(-1), device="cuda")
    o = torch.full_like(q, SENT)
    lse = torch.full((B, T, S, Hq), SENT, dtype=torch.float32, device="cuda")
    res = api.space_attn_fwd_varlen(q, k, v, L, agent, 0.125, out=o, lse=lse,
                                    o_lo=(True if with_lo else None))
    lo = res[2] if with_lo else None
    grads = [torch.full_like(q, SENT), torch.full_like(k, SENT), torch.full_like(v, SENT)]
    f32 = api.space_attn_bwd_varlen(q, k, v, o, lse, do, L, agent, 0.125, fp32_grads=True,
                                    out=grads, o_lo=lo)[3]
    torch.cuda.synchronize()
    st, site = api.get_device_status_detail()
    assert st == 0, "device timeout at site word %#x" % site
    X = oracle_mod.from_bf16
    ref = oracle_mod.space_bwd_varlen(X(q_b), X(k_b), X(v_b), X(do_b),
                                      np.asarray(lengths).reshape(B, T), agent, 0.125)
    Lh = np.clip(np.asarray(lengths).reshape(B, T), 0, S)
    valid = np.zeros((B, T, S), dtype=bool)
    for b in range(B):
        for t in range(T):
            valid[b, t, :Lh[b, t]] = True
    what = "varlen %s%s" % (str((B, T, S, Hq, Hkv)), " +O_lo" if with_lo else "")
    go, gl = to_f64(o), to_f64(lse)
    assert (go[~valid] == SENT).all() and (gl[~valid] == SENT).all(), what + ": padding O/LSE written"
    for name, g in zip(("dQ", "dK", "dV"), grads):
        assert (to_f64(g)[~valid] == SENT).all(), "%s: padding %s written" % (what, name)
    if valid.any():
        assert_close(go[valid], ref[0][valid], what + " O")
        assert np.abs(gl[valid] - ref[1][valid]).max() <= LSE_ERR
        for name, g, gb, r in zip(("dQ", "dK", "dV"), f32, grads, ref[2:]):
            assert_close(to_f64(g)[valid], r[valid], "%s %s fp32" % (what, name), bf16_out=False)
            assert_close(to_f64(gb)[valid], r[valid], "%s %s bf16" % (what, name))


@pytest.mark.parametrize("with_lo", [False, True])
def test_small_blocks_with_empty_single_and_full_lengths(oracle_mod, with_lo):
    run(oracle_mod, 2, 3, 37, 6, 2, 36, [[37, 1, 13], [0, 24, 25]], 90, with_lo)


def test_dynamics_head_layout(oracle_mod):
    """30/3 heads (12 tokens per Q tile), K/V resident: lengths across tile and block edges;
    the agent (index 289) exists only in the full block."""
    run(oracle_mod, 1, 4, 290, 30, 3, 289, [290, 150, 33, 128], 91, True)


def test_tokenizer_layout_streams_key_blocks(oracle_mod):
    """24 MHA heads on the padded 1432-token tokenizer frame (23 key blocks: K/V streamed),
    with frames that kept 10 % and 29 % of their 920 patches beside the 512 latents."""
    run(oracle_mod, 1, 2, 1432, 24, 24, -1, [604, 779], 92, True)


def test_full_lengths_equal_the_fixed_length_call():
    B, T, S, Hq, Hkv, agent = 1, 3, 130, 8, 2, 129
    w = synth.custom(B, T, S, Hq, Hkv, agent=agent, seed=93)
    q, k, v, do = (to_dev(x) for x in synth.make_inputs(w, with_dout=True))
    L = torch.full((B * T,), S, dtype=torch.int32, device="cuda")
    o1, l1, r1 = api.space_attn_fwd(q, k, v, agent, 0.125, o_lo=True)
    o2, l2, r2 = api.space_attn_fwd_varlen(q, k, v, L, agent, 0.125, o_lo=True)
    g1 = api.space_attn_bwd(q, k, v, o1, l1, do, agent, 0.125, o_lo=r1)
    g2 = api.space_attn_bwd_varlen(q, k, v, o2, l2, do, L, agent, 0.125, o_lo=r2)
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(r1, r2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
