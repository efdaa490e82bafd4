"""The trace module's host side: decoding per-warp records into phase medians.

Records are (clock << 32) | (warp << 26) | (event << 18) | detail, as the trace build writes
them.  `phases` must give, per warp, the span and the median cycles between consecutive
events, and unwrap a 32-bit clock that overflows between two records.
"""
import numpy as np

from block_causal_video_attention_b300 import trace


def _rec(clock, warp, event, detail=0):
    return np.uint64(((clock & 0xFFFFFFFF) << 32) | (warp << 26) | (event << 18) | detail)


def test_phases_medians_and_span():
    # warp 3: events 1 -> 2 takes 10, 20, 30 cycles; 2 -> 1 takes 100 each time
    recs, t = [], 1000
    for d in (10, 20, 30):
        recs.append(_rec(t, 3, 1))
        t += d
        recs.append(_rec(t, 3, 2))
        t += 100
    recs.append(_rec(t, 3, 1))
    out = trace.phases(np.array(recs, dtype=np.uint64))
    span, rows = out[3]
    assert span == t - 1000
    got = {(a, b): (n, med) for a, b, n, med, _ in rows}
    assert got[(1, 2)] == (3, 20)
    assert got[(2, 1)] == (3, 100)
    shares = {(a, b): sh for a, b, _, _, sh in rows}
    assert abs(sum(shares.values()) - 1.0) < 1e-9


def test_phases_unwraps_the_32_bit_clock():
    recs = [_rec(0xFFFFFFF0, 0, 5), _rec(0x00000010, 0, 6)]   # 0x20 cycles across the wrap
    span, rows = trace.phases(np.array(recs, dtype=np.uint64))[0]
    assert span == 0x20
    assert rows[0][:4] == (5, 6, 1, 0x20)


def test_phases_keeps_warps_apart():
    recs = [_rec(100, 1, 1), _rec(150, 1, 2), _rec(100, 2, 1), _rec(400, 2, 2)]
    out = trace.phases(np.array(recs, dtype=np.uint64))
    assert out[1][1][0][3] == 50 and out[2][1][0][3] == 300
