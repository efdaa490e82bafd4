// od_decode.cuh -- one rollout step of time attention over a ring-buffer KV cache (sm_103a).
//
// During a rollout the dynamics model produces one frame at a time (the local rollout
// harness and the frame-by-frame browser demo of the Open Dreamer pages: 7minutos.es page,
// section "Lo que realmente se envió"), so each time layer attends, for every token
// position s of the new frame t, from that frame's queries to the frames
// max(0, t - W + 1) .. t of the same position (the time window W of the training layer).
// The cache keeps the last W frames of K and V, frame f in slot f mod W:
//   K cache, V cache : [B, W, S, Hkv, 64] bf16,
// so the frames in the window are always the slots 0 .. n_valid - 1, n_valid = min(t+1, W).
//
// Work unit = (b, s, kv head): G <= 16 query heads x n_valid keys, a 16 x 64 x n_valid
// contraction twice (Q K^T, then P V).  The step is HBM-bound (every cached K/V byte is read
// once; about 5 multiply-adds per byte at G = 10), so the kernel is built as a stream:
//  * persistent CTAs, kDecWarps independent warps each; a warp owns whole units (no
//    cross-warp combine) and walks them block by block (kDecBN keys per block), with an
//    online softmax across blocks;
//  * every warp keeps a private ring of kDecStages stages; its lane 0 refills a stage by TMA
//    (K and V blocks: one 5-D box of kDecBN frames each, 128-byte swizzle; the unit's query
//    rows and the new frame's K/V rows by untiled bulk copies) as soon as the warp has
//    consumed it, so several blocks per warp are always in flight;
//  * the contractions run on the warp-level tensor-core MMA (m16n8k16, bf16 in, fp32
//    accumulate): the unit's 10 query heads fill one 16-row fragment, the 64-key block eight
//    8-column ones.  tcgen05's smallest tile (M = 64) would have to transpose the problem
//    and go through TMEM and a cross-warp hand-off for a few hundred multiply-adds per
//    block; with the kernel bound by HBM the tensor pipe is idle most of the time either way;
//  * P is split into a bf16 high part and a bf16 residual (two MMAs), so the P V product
//    keeps about 16 bits of P.
// The new frame's K/V rows are written into cache slot t mod W by the warp that owns the unit
// and substituted for that slot's (stale) row in shared memory before use, so one launch both
// updates the cache and attends over it.
#pragma once
#include "od_common.cuh"

namespace od {

constexpr int kDecWarps = 4;                       // warps per CTA (each one independent)
constexpr int kDecStages = 3;                      // ring stages per warp
constexpr int kDecBN = 64;                         // frames (keys) per block
constexpr int kDecRowBytes = 128;                  // one 64-element bf16 row
constexpr int kDecKVBytes = kDecBN * kDecRowBytes; // 8 KiB per K or V block
constexpr int kDecQBytes = 16 * kDecRowBytes;      // 16 query-head rows (rows >= G stay zero)
constexpr int kDecStageBytes = 2 * kDecKVBytes + kDecQBytes;  // 18 KiB (multiple of 1024)
constexpr int kDecThreads = kDecWarps * 32;
constexpr size_t kDecSmemBytes = (size_t)kDecWarps * kDecStages * kDecStageBytes + 1024;
static_assert(kDecStageBytes % 1024 == 0, "128-byte swizzled boxes need 1024-byte stages");

struct DecParams {
  const __nv_bfloat16* q;      // [B, S, Hq, 64]
  const __nv_bfloat16* k_new;  // [B, S, Hkv, 64]
  const __nv_bfloat16* v_new;  // [B, S, Hkv, 64]
  __nv_bfloat16* k_cache;      // [B, W, S, Hkv, 64]
  __nv_bfloat16* v_cache;      // [B, W, S, Hkv, 64]
  __nv_bfloat16* o;            // [B, S, Hq, 64]
  float* lse;                  // [B, S, Hq]
  int B, S, Hq, Hkv, G, W;
  int n_valid;                 // frames in the window: min(t + 1, W)
  int slot;                    // the new frame's slot, t mod W
  int nb;                      // key blocks per unit: ceil(n_valid / kDecBN)
  int units;                   // B * S * Hkv
  float sl;                    // scale * log2(e)
  unsigned int* status;
};

struct DecUnit {
  int b, s, h;  // batch, token position, KV head
};
__device__ __forceinline__ DecUnit dec_unit(const DecParams& p, int u) {
  DecUnit d;
  d.h = u % p.Hkv;
  const int bs = u / p.Hkv;
  d.s = bs % p.S;
  d.b = bs / p.S;
  return d;
}

// Byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * kDecRowBytes + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kDecThreads, 1)
    od_decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const DecParams p) {
  extern __shared__ uint8_t dec_smem_raw[];
  __shared__ __align__(8) uint64_t full[kDecWarps][kDecStages];
  __shared__ __align__(16) uint8_t aux[kDecWarps][kDecStages][2 * kDecRowBytes];
  __shared__ Ctl ctl;

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = base + warp * (kDecStages * kDecStageBytes);

  // The query rows G..15 of every stage are read by the MMAs but never written by a copy:
  // they are zeroed once here.
  for (int st = 0; st < kDecStages; ++st) {
    uint4* qz = reinterpret_cast<uint4*>(ring + st * kDecStageBytes + 2 * kDecKVBytes);
    for (int i = lane; i < kDecQBytes / 16; i += 32) qz[i] = make_uint4(0, 0, 0, 0);
  }
  if (lane == 0) {
    for (int st = 0; st < kDecStages; ++st) mbar_init(&full[warp][st], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) ctl.abort = 0;
  fence_proxy_async_smem();  // the zeroing (generic proxy) before any copy (async proxy)
  __syncthreads();
  if (lane == 0) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }

  const int gw = blockIdx.x * kDecWarps + warp;
  const int nwt = gridDim.x * kDecWarps;
  if (gw >= p.units) return;
  const int my_units = (p.units - 1 - gw) / nwt + 1;
  const int n_items = my_units * p.nb;
  const int slot_blk = p.slot / kDecBN, slot_row = p.slot % kDecBN;
  const int G = p.G;

  // lane 0: refill stage `i % kDecStages` with item i = (my unit i / nb, key block i % nb)
  auto issue = [&](int i) {
    const int ui = i / p.nb, blk = i - ui * p.nb;
    const DecUnit d = dec_unit(p, gw + ui * nwt);
    const int st = i % kDecStages;
    uint8_t* sK = ring + st * kDecStageBytes;
    uint8_t* sV = sK + kDecKVBytes;
    uint8_t* sQ = sV + kDecKVBytes;
    uint64_t* bar = &full[warp][st];
    const size_t kv_row = (static_cast<size_t>(d.b) * p.S + d.s) * p.Hkv + d.h;
    uint32_t bytes = 2 * kDecKVBytes;
    if (blk == 0) bytes += G * kDecRowBytes;
    if (blk == slot_blk) bytes += 2 * kDecRowBytes;
    mbar_arrive_expect_tx(bar, bytes);
    (void)OD_TMA_OK(d.h, d.s, blk * kDecBN, d.b, p.Hkv, p.S, p.W, p.B, p.status, 240);
    tma_load_5d(sK, &tk, bar, 0, d.h, d.s, blk * kDecBN, d.b);
    tma_load_5d(sV, &tv, bar, 0, d.h, d.s, blk * kDecBN, d.b);
    if (blk == 0) {
      const __nv_bfloat16* qsrc = p.q + ((static_cast<size_t>(d.b) * p.S + d.s) * p.Hq +
                                         static_cast<size_t>(d.h) * G) * 64;
      bulk_load(sQ, qsrc, G * kDecRowBytes, bar);
    }
    if (blk == slot_blk) {
      bulk_load(aux[warp][st], p.k_new + kv_row * 64, kDecRowBytes, bar);
      bulk_load(aux[warp][st] + kDecRowBytes, p.v_new + kv_row * 64, kDecRowBytes, bar);
    }
  };

  if (lane == 0)
    for (int i = 0; i < kDecStages && i < n_items; ++i) issue(i);

  const int g = lane >> 2, qd = lane & 3;  // fragment row group and column pair
  uint32_t qa[4][4];                       // query fragments (16 heads x 64), per k-step
  float oacc[8][4];                        // O fragments (16 heads x 64), per 8-column tile
  float m0 = -INFINITY, m1 = -INFINITY;    // running max (log2 units) of rows g and g + 8
  float l0 = 0.f, l1 = 0.f;                // running partial sums of this lane's columns
  int ui = 0, blk = 0;
  int consumed = 0;
  bool ok = true;

  for (int i = 0; i < n_items; ++i) {
    const int st = i % kDecStages;
    if (!wait_bar(&full[warp][st], (i / kDecStages) & 1, &ctl, p.status, 90)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    uint8_t* sK = ring + st * kDecStageBytes;
    uint8_t* sV = sK + kDecKVBytes;
    const uint8_t* sQ = sV + kDecKVBytes;
    const DecUnit d = dec_unit(p, gw + ui * nwt);

    if (blk == 0) {
      // A fragments of the 16 query rows: matrices (rows 0-7 | 8-15) x (chunk 2kk | 2kk+1)
      const int r = (lane & 7) + (lane & 8);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ldsm_x4(smem_u32(sQ + r * kDecRowBytes + ((2 * kk + (lane >> 4)) << 4)), qa[kk]);
#pragma unroll
      for (int n = 0; n < 8; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }
    if (blk == slot_blk) {
      // the new frame replaces slot t mod W: in this block's copy and in the cache
      const uint32_t kn = reinterpret_cast<const uint32_t*>(aux[warp][st])[lane];
      const uint32_t vn = reinterpret_cast<const uint32_t*>(aux[warp][st] + kDecRowBytes)[lane];
      const uint32_t off = sw128(slot_row, lane >> 2) + (lane & 3) * 4;
      *reinterpret_cast<uint32_t*>(sK + off) = kn;
      *reinterpret_cast<uint32_t*>(sV + off) = vn;
      const size_t crow = ((static_cast<size_t>(d.b) * p.W + p.slot) * p.S + d.s) * p.Hkv + d.h;
      if (OD_IN_RANGE(static_cast<long long>(crow), static_cast<long long>(p.B) * p.W * p.S * p.Hkv,
                      p.status, 241)) {
        reinterpret_cast<uint32_t*>(p.k_cache + crow * 64)[lane] = kn;
        reinterpret_cast<uint32_t*>(p.v_cache + crow * 64)[lane] = vn;
      }
      __syncwarp();
    }

    // ---- S = Q K^T for the block's 64 keys (8 tiles of 8 keys)
    float sacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t bk[4];
        ldsm_x4(smem_u32(sK) + sw128(8 * j + (lane & 7), 4 * kp + (lane >> 3)), bk);
        mma16816_bf16(sacc[j], qa[2 * kp], bk[0], bk[1]);
        mma16816_bf16(sacc[j], qa[2 * kp + 1], bk[2], bk[3]);
      }
    }
    // keys past the window's last frame (zero-filled rows of the last block)
    const int key0 = blk * kDecBN;
    if (key0 + kDecBN > p.n_valid) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (key0 + 8 * j + 2 * qd + (c & 1) >= p.n_valid) sacc[j][c] = -INFINITY;
    }

    // ---- online softmax (rows g and g + 8; a row's 64 columns live in the 4 lanes of a quad)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mx0 = max3(mx0, sacc[j][0], sacc[j][1]);
      mx1 = max3(mx1, sacc[j][2], sacc[j][3]);
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // every block holds at least one key of the window, so the new maxima are finite
    const float mn0 = fmaxf(m0, mx0 * p.sl), mn1 = fmaxf(m1, mx1 * p.sl);
    const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      oacc[n][0] *= a0;
      oacc[n][1] *= a0;
      oacc[n][2] *= a1;
      oacc[n][3] *= a1;
    }
    const float nm0 = -mn0, nm1 = -mn1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sacc[j][0] = ex2(fmaf(sacc[j][0], p.sl, nm0));
      sacc[j][1] = ex2(fmaf(sacc[j][1], p.sl, nm0));
      sacc[j][2] = ex2(fmaf(sacc[j][2], p.sl, nm1));
      sacc[j][3] = ex2(fmaf(sacc[j][3], p.sl, nm1));
      l0 += sacc[j][0] + sacc[j][1];
      l1 += sacc[j][2] + sacc[j][3];
    }

    // ---- O += P V: P's accumulator layout is the A fragment layout of the next MMA
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
      ph[0] = split_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1], &pl[0]);
      ph[1] = split_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3], &pl[1]);
      ph[2] = split_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], &pl[2]);
      ph[3] = split_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], &pl[3]);
      const int key = 16 * kk + (lane & 7) + (lane & 8);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bv[4];
        ldsm_x4_trans(smem_u32(sV) + sw128(key, 2 * np + (lane >> 4)), bv);
        mma16816_bf16(oacc[2 * np], ph, bv[0], bv[1]);
        mma16816_bf16(oacc[2 * np], pl, bv[0], bv[1]);
        mma16816_bf16(oacc[2 * np + 1], ph, bv[2], bv[3]);
        mma16816_bf16(oacc[2 * np + 1], pl, bv[2], bv[3]);
      }
    }

    // the stage is consumed: refill it (reads done by this warp; order them, and the generic
    // writes of the slot substitution, before the asynchronous copy into the same stage)
    __syncwarp();
    if (lane == 0 && i + kDecStages < n_items) {
      fence_proxy_async_smem();
      issue(i + kDecStages);
    }

    if (blk == p.nb - 1) {
      // ---- epilogue of the unit: normalise, write O rows < G and their LSE
      float s0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      float s1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      const float inv0 = 1.f / s0, inv1 = 1.f / s1;
      const size_t qrow = (static_cast<size_t>(d.b) * p.S + d.s) * p.Hq + static_cast<size_t>(d.h) * G;
      const long long nq = static_cast<long long>(p.B) * p.S * p.Hq;  // query rows (range checks)
      (void)nq;
      if (g < G && OD_IN_RANGE(static_cast<long long>(qrow + g), nq, p.status, 242)) {
        uint32_t* orow = reinterpret_cast<uint32_t*>(p.o + (qrow + g) * 64);
#pragma unroll
        for (int n = 0; n < 8; ++n) orow[4 * n + qd] = pack_bf16x2(oacc[n][0] * inv0, oacc[n][1] * inv0);
        if (qd == 0) p.lse[qrow + g] = (m0 + __log2f(s0)) * 0.6931471805599453f;
      }
      if (g + 8 < G && OD_IN_RANGE(static_cast<long long>(qrow + g + 8), nq, p.status, 242)) {
        uint32_t* orow = reinterpret_cast<uint32_t*>(p.o + (qrow + g + 8) * 64);
#pragma unroll
        for (int n = 0; n < 8; ++n) orow[4 * n + qd] = pack_bf16x2(oacc[n][2] * inv1, oacc[n][3] * inv1);
        if (qd == 0) p.lse[qrow + g + 8] = (m1 + __log2f(s1)) * 0.6931471805599453f;
      }
      blk = 0;
      ++ui;
    } else {
      ++blk;
    }
  }

  if (!ok && lane == 0) {
    // drain the copies this warp still has in flight before the CTA's shared memory goes
    for (int i = consumed; i < n_items && i < consumed + kDecStages; ++i)
      drain_wait(&full[warp][i % kDecStages], (i / kDecStages) & 1);
  }
  __syncwarp();
}

}  // namespace od
