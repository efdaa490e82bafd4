"""The launch path is capturable: a whole forward + backward step (space and time, with the O
residual) recorded into a CUDA graph replays to bit-identical results, and replays again
after its inputs are overwritten in place (the graph reads them, nothing was baked in)."""
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def test_fwd_bwd_step_replays_from_a_cuda_graph():
    B, T, S, Hq, Hkv, agent, window = 1, 24, 290, 30, 3, 289, 16
    w = synth.custom(B, T, S, Hq, Hkv, window=window, agent=agent, seed=95)
    q, k, v, do = (to_dev(x) for x in synth.make_inputs(w, with_dout=True))
    outs = {
        "o_s": torch.empty_like(q), "o_t": torch.empty_like(q),
        "lo_s": torch.empty_like(q), "lo_t": torch.empty_like(q),
        "l_s": torch.empty(q.shape[:4], dtype=torch.float32, device="cuda"),
        "l_t": torch.empty(q.shape[:4], dtype=torch.float32, device="cuda"),
    }
    g_s = [torch.empty_like(x) for x in (q, k, v)]
    g_t = [torch.empty_like(x) for x in (q, k, v)]
    ws_s = torch.empty(api.bwd_workspace_bytes(0, B, T, S, Hq, Hkv), dtype=torch.uint8, device="cuda")
    ws_t = torch.empty(api.bwd_workspace_bytes(1, B, T, S, Hq, Hkv), dtype=torch.uint8, device="cuda")

    def step(stream):
        api.space_attn_fwd(q, k, v, agent, 0.125, outs["o_s"], outs["l_s"], stream, o_lo=outs["lo_s"])
        api.time_attn_fwd(q, k, v, window, 0.125, outs["o_t"], outs["l_t"], stream, o_lo=outs["lo_t"])
        api.space_attn_bwd(q, k, v, outs["o_s"], outs["l_s"], do, agent, 0.125, workspace=ws_s,
                           out=g_s, stream=stream, o_lo=outs["lo_s"])
        api.time_attn_bwd(q, k, v, outs["o_t"], outs["l_t"], do, window, 0.125, workspace=ws_t,
                          out=g_t, stream=stream, o_lo=outs["lo_t"])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)                      # eager (also initialises the library on this device)
    torch.cuda.synchronize()
    eager = [t.clone() for t in list(outs.values()) + g_s + g_t]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for t in list(outs.values()) + g_s + g_t:
        t.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert api.get_device_status() == 0
    for a, b in zip(eager, list(outs.values()) + g_s + g_t):
        assert torch.equal(a, b)
    # new inputs written in place: the replay follows them
    q.mul_(0.5)
    graph.replay()
    torch.cuda.synchronize()
    o_new, l_new = api.space_attn_fwd(q, k, v, agent, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(o_new, outs["o_s"]) and torch.equal(l_new, outs["l_s"])
