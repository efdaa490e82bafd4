"""Seeded synthetic inputs and workload shapes.

Test and benchmark infrastructure: the tests, the bench and the smoke check
call it to make the inputs that they then hand both to the CUDA kernels (through
the C ABI) and to the oracle.  Neither the kernels nor the oracle import it, and
it holds no attention arithmetic: only shapes and a counter-based normal
generator, so both sides of every parity check consume identical bf16 bytes.

Generator (stated so that it can be re-implemented anywhere):
  * splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014).  Output i of the stream seeded with `seed` is
    mix(seed + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64), which is exactly the
    i-th value of the sequential generator started at state `seed`.
  * uniforms u = ((x >> 11) + 1) * 2**-53, in (0, 1].
  * Box-Muller (Box and Muller, 1958): values 2j and 2j+1 of the stream use
    u1 = U[2j], u2 = U[2j+1]; r = sqrt(-2 ln u1);
    z[2j] = r cos(2 pi u2), z[2j+1] = r sin(2 pi u2).
  * bf16: fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest even).
  * Fill order: Q, then K, then V, then dO, each in C order of its
    [B, T, S, H, D] tensor; one stream, the counter continues across tensors.

Workload shapes come from the Open Dreamer pages: the Minecraft dynamics model
(30 heads, 3 KV heads, d_model 1920, 32 registers, packing factor 2, a 192-step
time window; section "Configuracion de entrenamiento" of the edgex es-LA page),
the CoinRun stage, and the tokenizer geometry (368x640 frames, 16x16 patches,
512 latents, encoder d_model 1536).
"""
from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # normals generated per vectorised chunk (even)


def _mix(x: np.ndarray) -> np.ndarray:
    x = (x ^ (x >> np.uint64(30))) * _M1
    x = (x ^ (x >> np.uint64(27))) * _M2
    return x ^ (x >> np.uint64(31))


def _uniform(seed: int, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        x = _mix(x)
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def _f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even); returns uint16 bit patterns."""
    u = f.astype(np.float32).view(np.uint32)
    nan = np.isnan(f)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return _f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


def _normal_chunk(seed: int, start: int, m: int) -> np.ndarray:
    m2 = m + (m & 1)
    u = _uniform(seed, start, m2)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(m2, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return f64_to_bf16_bits(z[:m])


def normal_bf16(seed: int, start: int, n: int) -> np.ndarray:
    """Values [start, start+n) of the seeded N(0,1) stream, as bf16 bits.

    `start` must be even (Box-Muller works on pairs).  Chunks of the stream are independent
    (the generator is counter-based), so large requests are filled by several threads; the
    values do not depend on how the work is split."""
    if start % 2:
        raise ValueError("start must be even")
    out = np.empty(n, dtype=np.uint16)
    chunks = [(pos, min(_CHUNK, n - pos)) for pos in range(0, n, _CHUNK)]

    def fill(c):
        pos, m = c
        out[pos:pos + m] = _normal_chunk(seed, start + pos, m)
    if len(chunks) > 2:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, chunks))
    else:
        for c in chunks:
            fill(c)
    return out


@dataclass(frozen=True)
class Workload:
    """One synthetic attention workload (shapes only)."""
    name: str
    B: int
    T: int
    S: int
    Hq: int
    Hkv: int
    D: int
    window: int
    agent: int          # agent token index within a timestep block, -1 = none
    seed: int
    backward: bool
    note: str = field(default="", compare=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def q_shape(self):
        return (self.B, self.T, self.S, self.Hq, self.D)

    def kv_shape(self):
        return (self.B, self.T, self.S, self.Hkv, self.D)

    def lse_shape(self):
        return (self.B, self.T, self.S, self.Hq)


WORKLOADS = {
    # 16 spatial + 4 registers + action + agent (index 21); 4 Q / 2 KV heads.
    "tiny": Workload("tiny", 1, 8, 22, 4, 2, 64, 4, 21, 0, False,
                     "tiny correctness case"),
    # CoinRun scale: 64 spatial + 8 registers + action + agent.
    "coinrun": Workload("coinrun", 8, 64, 74, 8, 2, 64, 64, 73, 1, False,
                        "CoinRun-scale layer"),
    # Minecraft dynamics layer: 256 spatial (512 latents, packing 2)
    # + 32 registers + action + agent; 30 Q / 3 KV heads, window 192.
    "minecraft_fwd": Workload("minecraft_fwd", 1, 256, 290, 30, 3, 64, 192, 289, 2, False,
                              "Minecraft 1.6B dynamics layer, forward"),
    "minecraft_fwd_bwd": Workload("minecraft_fwd_bwd", 1, 256, 290, 30, 3, 64, 192, 289, 3, True,
                                  "Minecraft 1.6B dynamics layer, forward + backward"),
    # Tokenizer encoder: 23x40 = 920 patch tokens + 512 latents = 1432 per
    # frame; d_model 1536 as 24 heads x 64; no agent; window = T = 32.
    "tokenizer_enc": Workload("tokenizer_enc", 2, 32, 1432, 24, 24, 64, 32, -1, 4, True,
                              "tokenizer encoder layer, forward + backward"),
    # Tokenizer decoder: the same 1432 tokens per frame at d_model 1024, read as 16 heads x 64
    # (the pages give the width, not the head split).
    "tokenizer_dec": Workload("tokenizer_dec", 2, 32, 1432, 16, 16, 64, 32, -1, 6, True,
                              "tokenizer decoder layer, forward + backward"),
    # Rollout decode of the Minecraft dynamics layer: 16 concurrent rollouts, one new frame
    # per step attending to a full 192-frame window (T = absolute index of the new frame + 1).
    "minecraft_decode": Workload("minecraft_decode", 16, 501, 290, 30, 3, 64, 192, 289, 5, False,
                                 "Minecraft 1.6B dynamics layer, rollout decode step"),
}


def mae_block_lengths(B: int, T: int, seed: int, patches: int = 920, latents: int = 512,
                      max_mask: float = 0.9) -> np.ndarray:
    """Tokens per timestep block of a tokenizer encoder that drops its masked patches: the
    512 latents plus the kept patches, with a mask ratio drawn uniformly from [0, max_mask]
    per block (splitmix64 uniforms of stream `seed`).  int32 [B, T]."""
    u = _uniform(seed, 0, B * T)
    kept = np.rint(patches * (1.0 - max_mask * u)).astype(np.int64)
    return (latents + kept).astype(np.int32).reshape(B, T)


def make_decode_inputs(w: Workload):
    """Seeded bf16 inputs of one decode step (uint16 numpy): q [B,S,Hq,D], k_new and v_new
    [B,S,Hkv,D], and full K/V caches [B,W,S,Hkv,D]."""
    shapes = [(w.B, w.S, w.Hq, w.D), (w.B, w.S, w.Hkv, w.D), (w.B, w.S, w.Hkv, w.D),
              (w.B, w.window, w.S, w.Hkv, w.D), (w.B, w.window, w.S, w.Hkv, w.D)]
    out, start = [], 0
    for shp in shapes:
        n = int(np.prod(shp))
        out.append(normal_bf16(w.seed, start, n).reshape(shp))
        start += n + (n & 1)
    return tuple(out)


def make_inputs(w: Workload, with_dout: bool | None = None):
    """Seeded bf16 Q, K, V (and dO) as uint16 numpy arrays in [B,T,S,H,D]."""
    if with_dout is None:
        with_dout = w.backward
    nq = int(np.prod(w.q_shape()))
    nkv = int(np.prod(w.kv_shape()))
    sizes = [nq, nkv, nkv] + ([nq] if with_dout else [])
    shapes = [w.q_shape(), w.kv_shape(), w.kv_shape()] + ([w.q_shape()] if with_dout else [])
    out, start = [], 0
    for n, shp in zip(sizes, shapes):
        out.append(normal_bf16(w.seed, start, n).reshape(shp))
        start += n + (n & 1)
    return tuple(out)


def custom(B, T, S, Hq, Hkv, window=1, agent=-1, seed=123, D=64, backward=True, name="custom"):
    return Workload(name, B, T, S, Hq, Hkv, D, window, agent, seed, backward)
