"""The bench's algorithmic counts, checked by brute force on small shapes: allowed
(query, key) pairs enumerated from the masking rules, bytes summed from tensor sizes."""
import numpy as np

import bench
from block_causal_video_attention_b300 import synth


def count_space(S, agent):
    n = 0
    for s in range(S):
        for j in range(S):
            if j == agent and s != agent:
                continue
            n += 1
    return n


def count_time(T, W):
    return sum(1 for t in range(T) for j in range(T) if 0 <= t - j < W)


def test_pair_counts_match_enumeration():
    for (B, T, S, Hq, Hkv, agent, W) in [(1, 8, 22, 4, 2, 21, 4), (2, 5, 7, 6, 3, -1, 9),
                                         (1, 13, 3, 10, 1, 0, 1)]:
        w = synth.custom(B, T, S, Hq, Hkv, window=W, agent=agent)
        assert bench.pairs_space(w) == count_space(S, agent) * B * T * Hq
        assert bench.pairs_time(w) == count_time(T, W) * B * S * Hq
        f = bench.flops(w)
        assert f["space_fwd"] == 4 * w.D * bench.pairs_space(w)
        assert f["time_bwd"] == 2.5 * f["time_fwd"]


def test_minecraft_step_flops():
    w = synth.WORKLOADS["minecraft_fwd_bwd"]
    f = bench.flops(w)
    # 290 x 290 pairs minus the 289 world rows that may not read the agent, per (t, head)
    assert bench.pairs_space(w) == (290 * 290 - 289) * 256 * 30
    # steps t = 0..191 see t + 1 keys, the remaining 64 steps see 192
    assert bench.pairs_time(w) == (sum(range(1, 193)) + 64 * 192) * 290 * 30
    assert abs(sum(f.values()) - 816.94384128e9) < 1.0   # GFLOP per bench step


def test_varlen_flops_match_enumeration():
    w = synth.custom(1, 2, 9, 4, 2, agent=5)
    L = np.array([[9, 4]])
    fwd, bwd = bench.varlen_space_flops(w, L)
    pairs = count_space(9, 5) + count_space(4, -1)   # agent 5 is past the second block
    assert fwd == 4 * w.D * w.Hq * pairs and bwd == 2.5 * fwd


def test_decode_bytes_are_the_tensors_touched():
    w = synth.WORKLOADS["minecraft_decode"]
    n_valid = min(w.T, w.window)
    row = w.D * 2
    cache_reads = 2 * w.B * n_valid * w.S * w.Hkv * row
    new_rows = 2 * w.B * w.S * w.Hkv * row            # k_new, v_new read
    cache_writes = 2 * w.B * w.S * w.Hkv * row
    q_o = 2 * w.B * w.S * w.Hq * row
    lse = w.B * w.S * w.Hq * 4
    assert bench.decode_bytes(w) == cache_reads + new_rows + cache_writes + q_o + lse
    assert bench.decode_flops(w) == 4 * w.D * w.B * w.S * w.Hq * n_valid
