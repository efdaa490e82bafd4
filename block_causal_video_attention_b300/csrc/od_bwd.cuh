// od_bwd.cuh -- backward of space and time attention (sm_103a).
//
// With P recomputed from the forward's logsumexp (activation checkpointing; edgex es-LA
// page, "Rendimiento de computo y estrategia de memoria"), per query row with allowed
// keys j:  P_j = exp(scale <q, k_j> - LSE),  Delta = <dO, O>,  dP_j = <dO, v_j>,
// dS_j = P_j (dP_j - Delta),  dQ = scale sum_j dS_j k_j,  dK_j += scale dS_j q,
// dV_j += P_j dO  (dK, dV summed over the G query heads of a KV head).
//
// Three launches, no atomics, no zeroed workspace (results are deterministic):
//   1. Operand ranges, and Delta unless the dQ pass can form it.  Given O's rounding residual
//        O_lo from the forward: od_bwd_kv_range_kernel, max|K| and max|V| only (the dQ pass
//        forms Delta = <dO, O + O_lo> from its dO tile).  Otherwise od_bwd_dq_kernel<true, ...>,
//        Delta = sum_j P_j dP_j per row in fp32 into the caller's workspace (equal to <dO, O>
//        for the exact O; the bf16 O alone would give Delta only to ~1e-2 absolute, which the
//        gradients inherit).
//   2. od_bwd_dq_kernel<false, ...>: Q-tile stationary (the forward's work items and warp roles):
//        S = Q K^T and dP = dO V^T per 96-key block in TMEM; dS written in place over S as
//        fp16 times 2^eds; dQ += dS K into one fp32 accumulator, written once per tile.  Q
//        tiles and K blocks are rewritten as scaled fp16 in shared memory first (see "fp16
//        operand scaling"), so S runs on exact fp16 operands and dQ on fp16.  With O_lo it
//        also writes Delta to the workspace for the next launch.
//   3. od_bwd_dkdv_kernel:  key-block stationary: a CTA item is (unit, 128-key block);
//        for every Q tile that can see the block, S^T = K Q^T and dP^T = V dO^T in TMEM
//        (keys on TMEM lanes), P^T and dS^T written in place (scaled fp16), then
//        dV += P^T dO and dK += dS^T Q accumulate in TMEM.  All G heads of the group are
//        rows of the same Q tile, so the GQA reduction of dK/dV happens on chip.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include "od_ptx.cuh"
#include "od_common.cuh"

namespace od {

// Key blocks of the query-stationary backward kernels (Delta pass and dQ): 96 keys.
constexpr int kBN = 96;
constexpr int kKVTile = kBN * 128;  // bytes of one K or V stage

// ---------------------------------------------------------------- fp16 operand scaling
// The dQ and dK/dV products run on fp16 operands scaled by powers of two: every bf16 input
// value is exactly representable in fp16 once the tensor's (or Q tile's) largest magnitude is
// brought just below 2^15 (only values 2^25 times smaller than that largest one lose bits as
// fp16 subnormals), and power-of-two scales cancel exactly after accumulation.
// dS = P (dP - Delta) is a product whose range is not bounded by any one input's, so its
// scale is chosen per query row in the dQ pass and per key in the dK/dV kernel, from
//   |dS_ij| <= P_ij (|<dO_i, v_j>| + |Delta_i|) <= ||dO_i|| ||v_j|| + |Delta_i|
// with the row's own ||dO_i|| and Delta_i (dQ: ||v_j|| <= 8 max|V|) or the key's own ||v_j||
// (dK: ||dO_i|| <= 8 max|dO|, |Delta_i| <= max|Delta|).  A single large element of V or dO
// then lowers the scale only of the rows or keys it can reach.
// Operand ranges live in kAmaxSlots slots of kAmaxStride floats after the Delta array in the
// workspace, one slot per CTA of the launch that wrote it: the first launch writes max|K| and
// max|V|, and max|dO| and max|Delta| where it forms Delta (the Delta pass); the dQ pass writes
// max|Q| (it scales each Q tile by the tile's own range and records the maximum for the
// dK/dV kernel), and max|dO| and max|Delta| where it forms Delta from O.
constexpr int kAmaxSlots = 1024;
constexpr int kAmaxStride = 8;
constexpr int kAmK = 0, kAmV = 1, kAmDo = 2, kAmDelta = 3, kAmQ = 4;

// Running max of |x| over packed bf16 pairs, kept per 16-bit half as bf16 bit patterns
// (non-negative bf16 patterns order like their values; NaN sorts above infinity).
__device__ __forceinline__ uint32_t scan_amax(const uint8_t* buf, int bytes, int lane, uint32_t m) {
  const uint4* src = reinterpret_cast<const uint4*>(buf);
#pragma unroll 4
  for (int x = lane; x < (bytes >> 4); x += 32) {
    const uint4 d = src[x];
    m = __vmaxu2(m, d.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, d.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, d.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, d.w & 0x7FFF7FFFu);
  }
  return m;
}
// Warp-wide max of scan_amax results, as a float.
__device__ __forceinline__ float amax_reduce(uint32_t m) {
  uint32_t h = max(m >> 16, m & 0xFFFFu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
  return __uint_as_float(h << 16);
}
// E with a < 2^E for a finite a > 0; 0 marks "no scaling" (a zero, infinite or NaN).
__device__ __forceinline__ int amax_exp(float a, bool* usable) {
  const uint32_t bits = __float_as_uint(a);
  const int be = static_cast<int>((bits >> 23) & 0xFFu);
  *usable = (a > 0.f) && (be != 0xFF);
  return be == 0 ? -126 : be - 126;
}
// Power-of-two exponent e with a * 2^e < 2^15, clamped to [-60, 60].
__device__ __forceinline__ int fp16_shift(float a) {
  bool ok;
  const int E = amax_exp(a, &ok);
  return ok ? min(max(15 - E, -60), 60) : 0;
}

// Max over `nslots` operand-range slots of field `f` (whole warp; every lane gets the
// result).  NaN propagates (fmaxf alone would drop it), so that no scaling is applied.
__device__ __forceinline__ float slots_max(const float* amax, int nslots, int f, int lane) {
  float a = 0.f;
  bool bad = false;
  for (int sl = lane; sl < nslots; sl += 32) {
    const float v = amax[kAmaxStride * sl + f];
    a = fmaxf(a, v);
    bad |= !(v == v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  return bad ? __int_as_float(0x7fc00000) : a;
}
// Squared Euclidean norm of 64-element bf16 row `row` of a 128-byte-swizzled tile.  Chunk c
// is read at position c ^ (row & 7), so that lanes on 8 consecutive rows hit 8 different
// bank groups (the sum does not depend on the order).
__device__ __forceinline__ float row_norm2(const uint8_t* tile, int row) {
  const uint4* src = reinterpret_cast<const uint4*>(tile + row * 128);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 d = src[c ^ (row & 7)];
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 f = make_float2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
      acc = __ffma2_rn(f, f, acc);
    }
  }
  return acc.x + acc.y;
}

// Eight bf16 elements of dO (d) against the same elements of O (o) and its residual (l):
// returns sum dO (o + o_lo) in fp32 and adds sum dO^2 to *n2.
__device__ __forceinline__ float chunk_delta(const uint4& d, const uint4& o, const uint4& l, float* n2) {
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
  const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
  const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
  float2 acc = make_float2(0.f, 0.f), nn = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float2 f = make_float2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
    const float2 ov = make_float2(__uint_as_float(ow[h] << 16) + __uint_as_float(lw[h] << 16),
                                  __uint_as_float(ow[h] & 0xFFFF0000u) +
                                      __uint_as_float(lw[h] & 0xFFFF0000u));
    acc = __ffma2_rn(f, ov, acc);
    nn = __ffma2_rn(f, f, nn);
  }
  *n2 += nn.x + nn.y;
  return acc.x + acc.y;
}

// Rewrite `bytes` of packed bf16 pairs as fp16 pairs times 2^e, in place (one warp).
__device__ __forceinline__ void to_fp16_scaled(uint8_t* buf, int bytes, float s, int lane) {
  uint4* p = reinterpret_cast<uint4*>(buf);
  const float2 s2 = make_float2(s, s);
#pragma unroll 4
  for (int x = lane; x < (bytes >> 4); x += 32) {
    uint4 d = p[x];
    uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 f = __fmul2_rn(make_float2(__uint_as_float(w[h] << 16),
                                              __uint_as_float(w[h] & 0xFFFF0000u)), s2);
      w[h] = pack_f16x2(f.x, f.y);
    }
    p[x] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ============================================================================ dQ kernel
// Work items, Q tiles, key blocks and K/V staging as in the forward (FwdParams, fwd_decode).
// TMEM per tile x (256 columns at 256 x): S [0,96), dP [96,192), dQ [192,256).
constexpr int kDqThreads = 384;
constexpr int kDqStages = 5;
static_assert(2 * 128 * kQsSoftmaxRegs + 128 * kQsCtrlRegs == kDqThreads * kQsLaunchRegs,
              "register split must add up to the launch allocation");

struct DqParams {
  FwdParams f;            // shapes and item schedule (f.o unused)
  const float* lse;       // forward logsumexp (natural log)
  float* delta;           // Delta per query row (written by the Delta pass, read otherwise)
  float* amax;            // operand-range slots: the Delta pass writes its CTA's max|K|, max|V|,
                          // max|dO|, max|Delta|; the dQ pass its CTA's max|Q|
  int amax_slots;         // dQ pass: slots the first launch wrote (scales for the fp16 products)
  float scale;
  __nv_bfloat16* dq;
  int dq_rows;            // 64-element rows per token of dq (Hq, or Hq + 2 Hkv when packed)
  float* dq_f32;          // optional, contiguous [B,T,S,Hq,64]
  // dQ pass, optional: O and its residual O_lo (contiguous [B,T,S,Hq,64]).  Given, the pass
  // forms Delta = <dO_i, O_i> itself, writes it for the dK/dV kernel and records max|dO| and
  // max|Delta| in its slots; otherwise it reads Delta from the workspace.
  const __nv_bfloat16* o;
  const __nv_bfloat16* o_lo;
};

struct DqSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kDqStages], v_full[kDqStages], kv_empty[kDqStages];
  uint64_t q16[2], k16[kDqStages];  // dQ pass: Q tile / K stage rewritten as scaled fp16
  uint64_t s_full[2], ds_full[2], dq_done[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  Ctl ctl;
  int ek;                     // dQ pass: K's fp16 scale exponent
  float vn8;                  // dQ pass: 8 max|V| >= every ||v_j||
  unsigned int dmax_bits;     // max |Delta| of the CTA's rows (float bits): Delta pass, or
                              // the dQ pass when it forms Delta from O
  unsigned int domax_bits;    // max |dO| of the CTA's tiles (float bits), idem
  int eqt[2];                 // dQ pass: scale exponent of Q tile x
};
// smem: [Q0 Q1 dO0 dO1][K stages][V stages][dQ staging 8 x 4 KB][DqSmem]
constexpr size_t kDqTileBytes = size_t(4) * kTile + size_t(2 * kDqStages) * kKVTile + 8 * 4096;
constexpr size_t kDqSmemBytes = kDqTileBytes + 1024 + sizeof(DqSmem) + 64;
static_assert(kDqSmemBytes <= 227 * 1024, "shared memory budget");

// kDelta = true: the Delta pass -- S and dP per key block, Delta = sum_j P_j dP_j accumulated
// in fp32 per row and written to the workspace (no dS, no dQ).  This is <dO, O> for the exact
// forward output, which the bf16 O given to the backward only approximates.
// kPacked: packed short time sequences (PK; see FwdParams), a separate instantiation so
// that the other calls compile without its branches
template <bool kDelta, bool kVarlen, bool kPacked>
__global__ void __launch_bounds__(kDqThreads, 1)
    od_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DqParams dp) {
  const FwdParams& p = dp.f;
  const int PK = kPacked ? p.pk : 0;   // packed: token positions per tile
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start of the dynamic shared memory, formed by pointer arithmetic on the
  // __shared__ array (not through an integer) so that every tile is addressed as shared memory
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ[2] = {base, base + kTile};
  uint8_t* sdO[2] = {base + 2 * kTile, base + 3 * kTile};
  uint8_t* sK = base + 4 * kTile;
  uint8_t* sV = sK + kDqStages * kKVTile;
  uint8_t* sOst = sV + kDqStages * kKVTile;
  DqSmem& sm = *reinterpret_cast<DqSmem*>(base + kDqTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool resident = p.nkb <= kDqStages;
  OD_TRACE_INIT(kDelta ? 3 : 1);
  // items of this CTA: a contiguous range (consecutive items of a unit share its K/V); for
  // variable-length blocks every gridDim.x-th item, so that items of unequal cost spread
  // over all CTAs
  const bool strided = kVarlen;
  const long long istep = strided ? gridDim.x : 1;
  const long long i0 = strided ? blockIdx.x : (p.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = strided ? p.nitems : (p.nitems * (blockIdx.x + 1)) / gridDim.x;

  {  // zero the tile rows TMA never writes (and, packed, the K/V stage rows past pk T keys)
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kDqThreads * 16)
      for (int t = 0; t < 2; ++t) {
        *reinterpret_cast<uint4*>(sQ[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sdO[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
      }
    const int kvpad = (kBN - p.kvb) * 128;
    for (int x = tid * 16; x < kvpad; x += kDqThreads * 16)
      for (int st = 0; st < 2 * kDqStages; ++st)
        *reinterpret_cast<uint4*>(sK + st * kKVTile + p.kvb * 128 + x) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.q_full[x], 1);
      // Delta pass: MMA commit + the range scanner; dQ pass: MMA commit + the 4 dS warps of
      // the tile, which read the fill's eq and dO rows (so the slot is not refilled first)
      mbar_init(&sm.q_empty[x], kDelta ? 2 : 5);
      mbar_init(&sm.q16[x], 1);
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.ds_full[x], 4);
      mbar_init(&sm.dq_done[x], 1);
      mbar_init(&sm.drain[x], 1);
    }
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], kDelta ? 3 : 2);
      mbar_init(&sm.k16[s], 1);
    }
    sm.ctl.abort = 0;
    sm.dmax_bits = 0u;
    sm.domax_bits = 0u;
    fence_mbar_init();
  }
  if (!kDelta && warp == kQsProducerWarp) {
    // operand ranges recorded by the first launch -> K's scale and the bound on ||v_j||
    const float ak = slots_max(dp.amax, dp.amax_slots, kAmK, lane);
    const float av = slots_max(dp.amax, dp.amax_slots, kAmV, lane);
    if (lane == 0) {
      sm.ek = fp16_shift(ak);
      sm.vn8 = 8.f * av;
    }
  }
  if (warp == kQsMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  Ctl* ctl = &sm.ctl;
  unsigned int* status = p.status;
  const int ek = kDelta ? 0 : sm.ek;
  const float vn8 = kDelta ? 0.f : sm.vn8;

  if (warp >= 8) {
    regs_dec<kQsCtrlRegs>();
    if (!kDelta && warp == 11) {
      // ---------------------------------------------------------- operand conversion
      // dQ pass: every Q tile is rewritten in place as fp16 times 2^eq (eq from the tile's own
      // largest magnitude) and every K block as fp16 times 2^ek (S then runs on fp16 operands
      // -- exact, the scales fold into the exponent -- and dQ += dS K on fp16 dS); the tile's
      // eq goes to the dS warpgroups.  Released to the MMA issuers and the dS warpgroups
      // through q16 / k16.  Walks the producer's fills in its order.
      const float sk = ldexpf(1.f, ek);
      uint32_t mq = 0;  // running max|Q| over the CTA's tiles (bf16 bit pairs)
      long long prev_unit = -1;
      uint32_t unit_loads = 0, sbase = 0, qn[2] = {0, 0};
      bool ok = true;
      auto conv_k = [&](int stage, uint32_t parity) -> bool {
        if (!__all_sync(0xffffffffu, wait_bar(&sm.k_full[stage], parity, ctl, status, 19))) return false;
        to_fp16_scaled(sK + stage * kKVTile, kKVTile, sk, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.k16[stage]);
        return true;
      };
      for (long long i = i0; i < i1 && ok; i += istep) {
        const FwdItem it = fwd_decode<kVarlen, kPacked>(p, i);
        if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
        const int nb = it.kb_hi - it.kb_lo + 1;
        for (int x = 0; x < 2 && ok; ++x) {
          if (x == 1 && !it.validB) break;
          ok = __all_sync(0xffffffffu, wait_bar(&sm.q_full[x], qn[x] & 1u, ctl, status, 17));
          if (!ok) break;
          ++qn[x];
          const uint32_t mt = scan_amax(sQ[x], p.rows * 128, lane, 0u);
          mq = __vmaxu2(mq, mt);
          const int eqt = fp16_shift(amax_reduce(mt));
          to_fp16_scaled(sQ[x], p.rows * 128, ldexpf(1.f, eqt), lane);
          if (lane == 0) sm.eqt[x] = eqt;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.q16[x]);
        }
        if (!ok) break;
        if (resident) {
          if (it.unit != prev_unit) {
            ++unit_loads;
            prev_unit = it.unit;
            for (int st = 0; st < p.nkb && ok; ++st) ok = conv_k(st, (unit_loads - 1) & 1u);
          }
        } else {
          for (int bi = 0; bi < nb && ok; ++bi) {
            const uint32_t c = sbase + static_cast<uint32_t>(bi);
            ok = conv_k(static_cast<int>(c % kDqStages), (c / kDqStages) & 1u);
          }
        }
        sbase += nb;
      }
      const float aq = amax_reduce(mq);
      if (lane == 0) dp.amax[kAmaxStride * blockIdx.x + kAmQ] = aq;
    } else if (kDelta && warp == 11) {
      // ---------------------------------------------------------- operand range scan
      // Walks the producer's fills in its order; every fill is scanned and then released
      // (one more arrival on q_empty / kv_empty), so no buffer is refilled unscanned.  (Q's
      // range is taken per tile by the dQ pass.)
      uint32_t mk = 0, mv = 0, mdo = 0;
      long long prev_unit = -1;
      uint32_t unit_loads = 0, sbase = 0, qn[2] = {0, 0};
      bool ok = true;
      for (long long i = i0; i < i1 && ok; i += istep) {
        const FwdItem it = fwd_decode<kVarlen, kPacked>(p, i);
        if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
        const int nb = it.kb_hi - it.kb_lo + 1;
        for (int x = 0; x < 2 && ok; ++x) {
          if (x == 1 && !it.validB) break;
          ok = __all_sync(0xffffffffu, wait_bar(&sm.q_full[x], qn[x] & 1u, ctl, status, 17));
          if (!ok) break;
          ++qn[x];
          mdo = scan_amax(sdO[x], p.rows * 128, lane, mdo);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.q_empty[x]);
        }
        if (!ok) break;
        auto scan_kv = [&](int stage, uint32_t parity) -> bool {
          bool w = wait_bar(&sm.k_full[stage], parity, ctl, status, 18) &&
                   wait_bar(&sm.v_full[stage], parity, ctl, status, 18);
          if (!__all_sync(0xffffffffu, w)) return false;
          mk = scan_amax(sK + stage * kKVTile, kKVTile, lane, mk);
          mv = scan_amax(sV + stage * kKVTile, kKVTile, lane, mv);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.kv_empty[stage]);
          return true;
        };
        if (resident) {
          if (it.unit != prev_unit) {
            ++unit_loads;
            prev_unit = it.unit;
            for (int st = 0; st < p.nkb && ok; ++st) ok = scan_kv(st, (unit_loads - 1) & 1u);
          }
        } else {
          for (int bi = 0; bi < nb && ok; ++bi) {
            const uint32_t c = sbase + static_cast<uint32_t>(bi);
            ok = scan_kv(static_cast<int>(c % kDqStages), (c / kDqStages) & 1u);
          }
        }
        sbase += nb;
      }
      const float ak = amax_reduce(mk), av = amax_reduce(mv), ad = amax_reduce(mdo);
      if (lane == 0) {
        float* slot = dp.amax + kAmaxStride * blockIdx.x;
        slot[kAmK] = ak;
        slot[kAmV] = av;
        slot[kAmDo] = ad;
      }
    } else if (warp == kQsProducerWarp) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        long long prev_unit = -1;
        uint32_t unit_loads = 0, sbase = 0, qn[2] = {0, 0};
        bool ok = true;
        for (long long i = i0; i < i1 && ok; i += istep) {
          const FwdItem it = fwd_decode<kVarlen, kPacked>(p, i);
          if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
          const int nb = it.kb_hi - it.kb_lo + 1;
          auto load_kv = [&](int stage, int kb) {
            // box start (s, t): packed time, time, space
            const int kp = kb * kBN;
            const int cs = PK ? it.tok0[0] + kb * PK : (p.is_time ? it.fixed : kp);
            const int ct = PK ? 0 : (p.is_time ? kp : it.fixed);
            // (a packed unit without a tile B loads its second block from past the end on
            // purpose: TMA fills it with zeros, and every stage's phase count stays equal)
            if (!PK || kb == 0 || it.validB)
              (void)OD_TMA_OK(it.kvh, cs, ct, it.b, p.Hkv, p.S, p.T, p.B, status, 210);
            mbar_arrive_expect_tx(&sm.k_full[stage], p.kvb * 128);
            mbar_arrive_expect_tx(&sm.v_full[stage], p.kvb * 128);
            tma_load_5d(sK + stage * kKVTile, &tm_k, &sm.k_full[stage], 0, it.kvh, cs, ct, it.b);
            tma_load_5d(sV + stage * kKVTile, &tm_v, &sm.v_full[stage], 0, it.kvh, cs, ct, it.b);
          };
          for (int x = 0; x < 2 && ok; ++x) {
            if (x == 1 && !it.validB) break;
            if (qn[x] > 0) ok = wait_bar(&sm.q_empty[x], (qn[x] - 1) & 1u, ctl, status, 1);
            if (!ok) break;
            const int t0 = x ? it.tok0[1] : it.tok0[0];
            const int cs = PK ? t0 : (p.is_time ? it.fixed : t0);
            const int ct = PK ? 0 : (p.is_time ? t0 : it.fixed);
            (void)OD_TMA_OK(it.kvh * p.G, cs, ct, it.b, p.Hq, p.S, p.T, p.B, status, 211);
            mbar_arrive_expect_tx(&sm.q_full[x], 2 * p.rows * 128);
            tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, cs, ct, it.b);
            tma_load_5d(sdO[x], &tm_do, &sm.q_full[x], 0, it.kvh * p.G, cs, ct, it.b);
            ++qn[x];
          }
          if (!ok) break;
          if (resident) {
            if (it.unit != prev_unit) {
              if (unit_loads > 0)
                for (int s = 0; s < p.nkb && ok; ++s)
                  ok = wait_bar(&sm.kv_empty[s], (unit_loads - 1) & 1u, ctl, status, 2);
              if (!ok) break;
              for (int kb = 0; kb < p.nkb; ++kb) load_kv(kb, kb);
              ++unit_loads;
              prev_unit = it.unit;
            }
          } else {
            for (int bi = 0; bi < nb && ok; ++bi) {
              const uint32_t c = sbase + bi;
              const int stage = static_cast<int>(c % kDqStages);
              const uint32_t n = c / kDqStages;
              if (n > 0) ok = wait_bar(&sm.kv_empty[stage], (n - 1) & 1u, ctl, status, 3);
              if (ok) load_kv(stage, it.kb_lo + bi);
            }
          }
          sbase += nb;
        }
        for (int x = 0; x < 2; ++x)
          if (qn[x] > 0) drain_wait(&sm.q_full[x], (qn[x] - 1) & 1u);
        if (resident) {
          if (unit_loads > 0)
            for (int s = 0; s < p.nkb; ++s) {
              drain_wait(&sm.k_full[s], (unit_loads - 1) & 1u);
              drain_wait(&sm.v_full[s], (unit_loads - 1) & 1u);
            }
        } else {
          for (int s = 0; s < kDqStages; ++s) {
            const uint32_t uses = sbase / kDqStages + (static_cast<uint32_t>(s) < sbase % kDqStages ? 1u : 0u);
            if (uses > 0) {
              drain_wait(&sm.k_full[s], (uses - 1) & 1u);
              drain_wait(&sm.v_full[s], (uses - 1) & 1u);
            }
          }
        }
      }
    } else if (warp == kQsMmaWarp || warp == kQsMmaWarp + 1) {
      // ---------------------------------------------------------- MMA issuers (per tile)
      // In order per tile: S(0), dP(0); then for each block j: wait dS(j), dQ += dS(j) K;
      // S(j+1), dP(j+1) (they overwrite buffers whose last reader was issued before them).
      {  // whole warp in lockstep; one elected lane issues
        const int x = warp - kQsMmaWarp;
        const uint32_t tS = tmem + 256u * x, tP = tS + 96u, tQ = tS + 192u;
        const uint32_t idesc_dq = idesc_fp16(128, 64, 0, 1);
        // operand descriptors: this tile's Q and dO, stage 0's K and V (a stage's are these
        // plus its offset in 16-byte units; every address stays below 2^18, the field's range)
        const uint64_t d_q = sdesc_sw128(smem_u32(sQ[x]), 16, 1024);
        const uint64_t d_do = sdesc_sw128(smem_u32(sdO[x]), 16, 1024);
        const uint64_t d_k = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t d_v = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t d_kq = sdesc_sw128(smem_u32(sK), 1024, 1024);   // K as dQ's B (MN-major)
        // the dQ pass reads Q and K after their fp16 rewrite, the Delta pass as loaded
        uint64_t* const qb = kDelta ? sm.q_full : sm.q16;
        uint64_t* const kb16 = kDelta ? sm.k_full : sm.k16;
        uint32_t js = 0, jd = 0, qn = 0, unit_loads = 0, sbase = 0;
        long long prev_unit = -1;
        bool ok = true;
        for (long long i = i0; i < i1 && ok; i += istep) {
          const FwdItem it = fwd_decode<kVarlen, kPacked>(p, i);
          if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
          const int nb = it.kb_hi - it.kb_lo + 1;
          if (resident && it.unit != prev_unit) {
            if (prev_unit >= 0)
              for (int s = 0; s < p.nkb; ++s) mma_commit_w(&sm.kv_empty[s]);
            ++unit_loads;
            prev_unit = it.unit;
            for (int s = 0; s < p.nkb && ok; ++s)
              ok = __all_sync(0xffffffffu, wait_bar(&kb16[s], (unit_loads - 1) & 1u, ctl, status, 11));
            for (int s = 0; s < p.nkb && ok; ++s)
              ok = __all_sync(0xffffffffu, wait_bar(&sm.v_full[s], (unit_loads - 1) & 1u, ctl, status, 11));
          }
          if (!ok) break;
          auto slot = [&](int bi) -> KvSlot {
            KvSlot k;
            if (resident) {
              k.stage = it.kb_lo + bi;
              k.parity = (unit_loads - 1) & 1u;
            } else {
              const uint32_t c = sbase + static_cast<uint32_t>(bi);
              k.stage = static_cast<int>(c % kDqStages);
              k.parity = (c / kDqStages) & 1u;
            }
            return k;
          };
          if (x == 1 && !it.validB) {
            if (!resident)
              for (int bi = 0; bi < nb && ok; ++bi) {
                const KvSlot ks = slot(bi);
                ok = __all_sync(0xffffffffu, wait_bar(&kb16[ks.stage], ks.parity, ctl, status, 12)) &&
                     __all_sync(0xffffffffu, wait_bar(&sm.v_full[ks.stage], ks.parity, ctl, status, 12));
                if (ok) mma_commit_w(&sm.kv_empty[ks.stage]);
              }
            sbase += nb;
            continue;
          }
          if (!__all_sync(0xffffffffu, wait_bar(&qb[x], qn & 1u, ctl, status, 14))) break;
          ++qn;
          OD_TP(90, (int)i, 0);
          // this tile's blocks (packed: its own block only; packed units are always resident)
          const int b0 = (x ? it.blo[1] : it.blo[0]) - it.kb_lo, b1 = (x ? it.bhi[1] : it.bhi[0]) - it.kb_lo;
          auto issue_s = [&](int bi) -> bool {
            const KvSlot ks = slot(bi);
            if (!resident) {   // (a resident unit's stages were all waited for at its start)
              if (!__all_sync(0xffffffffu, wait_bar(&kb16[ks.stage], ks.parity, ctl, status, 15))) return false;
              if (!__all_sync(0xffffffffu, wait_bar(&sm.v_full[ks.stage], ks.parity, ctl, status, 15))) return false;
              tc_fence_after();
            }
            const int n = round16(block_keys<kPacked>(p, it, it.kb_lo + bi, kBN));
            const uint32_t idesc = idesc_bf16(128, n, 0, 0);
            const uint32_t idesc_s = kDelta ? idesc : idesc_fp16(128, n, 0, 0);
            const uint64_t so = static_cast<uint64_t>((ks.stage * kKVTile) >> 4);
            mma_ss_k64_w(tS, d_q, d_k + so, idesc_s);
            mma_ss_k64_w(tP, d_do, d_v + so, idesc);
            mma_commit_w(&sm.s_full[x]);
            ++js;
            if (bi == b1) mma_commit_w(&sm.q_empty[x]);
            return true;
          };
          ok = issue_s(b0);
          for (int bi = b0; bi <= b1 && ok; ++bi) {
            if (!__all_sync(0xffffffffu, wait_bar(&sm.ds_full[x], jd & 1u, ctl, status, 16))) { ok = false; break; }
            ++jd;
            OD_TP(91, (int)i, bi);
            tc_fence_after();
            const KvSlot ks = slot(bi);
            if (!kDelta) {
              const int ksteps = round16(block_keys<kPacked>(p, it, it.kb_lo + bi, kBN)) >> 4;
              const uint64_t so = static_cast<uint64_t>((ks.stage * kKVTile) >> 4);
              mma_ts_kn6_w(tQ, tS, d_kq + so, idesc_dq, bi > b0 ? 1u : 0u, static_cast<uint32_t>(ksteps));
            }
            if (!resident) mma_commit_w(&sm.kv_empty[ks.stage]);
            if (bi == b1) {
              if (!kDelta) mma_commit_w(&sm.dq_done[x]);
            } else {
              ok = issue_s(bi + 1);
            }
          }
          sbase += nb;
        }
        mma_commit_w(&sm.drain[x]);
        drain_wait(&sm.drain[x], 0);
      }
    }
  } else {
    regs_inc<kQsSoftmaxRegs>();
    // ------------------------------------------------------------ dS warpgroups
    const int x = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 256u * x + lane_off, tP = tS + 96u, tQ = tS + 192u;
    const int G = p.G;
    const int tok = r / G;
    const int g = r - tok * G;
    const float lg2e = 1.4426950408889634f;
    uint32_t jS = 0, jD = 0, jq = 0;
    uint32_t dmax = 0u;  // max |Delta| of this thread's rows (float bits; NaN on top)
    uint32_t mdo = 0u;   // dQ pass from O: max |dO| of this thread's tile rows (bf16 pairs)
    const bool from_o = !kDelta && dp.o != nullptr;
    // the row's sequence position (packed: pt its frame, sp its token within the tile)
    const int pt = PK ? tok / PK : 0;
    const int sp = PK ? tok - pt * PK : 0;
    // this thread's token of item `it` ([B,T,S] order), if the tile row exists; its query
    // row is token * Hq + kvh G + g
    auto token_of = [&](const FwdItem& it, long long* ti) -> bool {
      const int t0 = x ? it.tok0[1] : it.tok0[0];
      const int ps = PK ? pt : t0 + tok;
      if (!(r < p.rows && (PK ? t0 + sp < p.S : ps < (kVarlen ? it.L : p.L)))) return false;
      const long long t_idx = p.is_time ? ps : it.fixed;
      const long long s_idx = PK ? t0 + sp : (p.is_time ? it.fixed : ps);
      *ti = (static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx;
      return true;
    };
    bool first = true;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; i += istep) {
      const FwdItem it = fwd_decode<kVarlen, kPacked>(p, i);
      if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
      if (x == 1 && !it.validB) continue;
      const int mytok0 = x ? it.tok0[1] : it.tok0[0];
      const int pos = PK ? pt : mytok0 + tok;
      long long tix = 0, row = 0;
      float lse2 = INFINITY, dl = 0.f;
      float dacc[4] = {0.f, 0.f, 0.f, 0.f};
      bool row_ok = token_of(it, &tix);
      row = tix * p.Hq + it.kvh * G + g;
      if (row_ok) row_ok = OD_IN_RANGE(row, static_cast<long long>(p.B) * p.T * p.S * p.Hq, status, 212);
      if (row_ok) {
        lse2 = dp.lse[row] * lg2e;
        if (!kDelta && !from_o) dl = dp.delta[row];
      }
      // from O: the row's O and O_lo lines are sent towards L2 one item ahead (the first
      // item's now), so that the loads below, on the way to this item's first dS, hit L2
      if (from_o) {
        if (first && row_ok) {
          prefetch_l2(dp.o + row * 64);
          prefetch_l2(dp.o_lo + row * 64);
        }
        long long tn;
        if (i + istep < i1) {
          const FwdItem nx = fwd_decode<kVarlen, kPacked>(p, i + istep);
          if (!(kVarlen && !nx.validA) && !(x == 1 && !nx.validB) && token_of(nx, &tn)) {
            const long long rn = tn * p.Hq + nx.kvh * G + g;
            if (rn < static_cast<long long>(p.B) * p.T * p.S * p.Hq) {
              prefetch_l2(dp.o + rn * 64);
              prefetch_l2(dp.o_lo + rn * 64);
            }
          }
        }
      }
      first = false;
      // dQ pass: S carries 2^(eq + ek) (eq: this Q tile's); dS is written times 2^eds with eds
      // from the row's bound ||dO_i|| 8 max|V| + |Delta_i| on |dS|, and dQ undoes 2^(eds + ek)
      float slx = p.sl, c1 = 1.f, fq = dp.scale;
      OD_TP(80, (int)i, 0);
      if (!kDelta) {
        // the row's ||dO_i|| (and, from O, Delta_i) from the dO tile as loaded; every row of
        // the tile counts towards max|dO|, which scales whole tiles in the dK/dV kernel
        ok = __all_sync(0xffffffffu, wait_bar(&sm.q_full[x], jq & 1u, ctl, status, 7));
        if (!ok) break;
        OD_TP(86, (int)i, 0);
        float dn2 = 0.f;
        if (from_o) {
          // the warp's 32 rows 4 at a time, 8 lanes x 16 bytes per 128-byte row (coalesced
          // loads of O and O_lo); each row's sums go back to the row's own lane
          const int sub = lane >> 3, ch = lane & 7;
          uint4 ov[8], lv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const long long rw = __shfl_sync(0xffffffffu, row, 4 * k + sub);
            const bool rok = __shfl_sync(0xffffffffu, static_cast<int>(row_ok), 4 * k + sub) != 0;
            ov[k] = rok ? __ldg(reinterpret_cast<const uint4*>(dp.o) + rw * 8 + ch) : make_uint4(0, 0, 0, 0);
            lv[k] = rok ? __ldg(reinterpret_cast<const uint4*>(dp.o_lo) + rw * 8 + ch) : make_uint4(0, 0, 0, 0);
          }
          float dsel = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 32 * (warp & 3) + 4 * k + sub;   // tile row (zeros past p.rows)
            const uint4 d = *reinterpret_cast<const uint4*>(sdO[x] + rr * 128 + ((ch ^ (rr & 7)) << 4));
            mdo = __vmaxu2(mdo, d.x & 0x7FFF7FFFu);
            mdo = __vmaxu2(mdo, d.y & 0x7FFF7FFFu);
            mdo = __vmaxu2(mdo, d.z & 0x7FFF7FFFu);
            mdo = __vmaxu2(mdo, d.w & 0x7FFF7FFFu);
            float n = 0.f;
            float a = chunk_delta(d, ov[k], lv[k], &n);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
              a += __shfl_xor_sync(0xffffffffu, a, o);
              n += __shfl_xor_sync(0xffffffffu, n, o);
            }
            const float at = __shfl_sync(0xffffffffu, a, (lane & 3) * 8);   // row 4k + (lane & 3)
            const float nt = __shfl_sync(0xffffffffu, n, (lane & 3) * 8);
            if ((lane >> 2) == k) {
              dsel = at;
              dn2 = nt;
            }
          }
          if (row_ok) {
            dl = dsel;
            dp.delta[row] = dsel;
            dmax = max(dmax, __float_as_uint(fabsf(dsel)));
          }
        } else if (row_ok) {
          dn2 = row_norm2(sdO[x], r);
        }
        OD_TP(87, (int)i, 0);
        ok = __all_sync(0xffffffffu, wait_bar(&sm.q16[x], jq & 1u, ctl, status, 9));
        if (!ok) break;
        OD_TP(88, (int)i, 0);
        ++jq;
        const int eqt = sm.eqt[x];
        const float dn = row_ok ? sqrtf(dn2) : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.q_empty[x]);  // this warp is done with the fill's values
        const int eds = fp16_shift(fmaf(dn, vn8, fabsf(dl)));
        slx = p.sl * ldexpf(1.f, -(eqt + ek));
        c1 = ldexpf(1.f, eds);
        fq = dp.scale * ldexpf(1.f, -(eds + ek));
      }
      const float ndl = -dl * c1;
      const float2 sl2 = make_float2(slx, slx), c12 = make_float2(c1, c1), nd2 = make_float2(ndl, ndl);
      const float2 nl2 = make_float2(-lse2, -lse2);
      const int kb_first = x ? it.blo[1] : it.blo[0], kb_last = x ? it.bhi[1] : it.bhi[0];
      for (int kb = kb_first; kb <= kb_last; ++kb) {
        const int bi = kb - it.kb_lo;
        const int kbase = kb * kBN;
        const int ncols = block_keys<kPacked>(p, it, kb, kBN);
        const int n32 = (ncols + 31) >> 5;
        int lo, hi, ex;
        if (PK) {   // frames [lo, hi] of the row's own token (see keep_bits_packed)
          lo = max(0, pos - p.window + 1);
          hi = pos;
          ex = -1;
        } else if (p.is_time) {
          lo = pos - p.window + 1 - kbase;
          hi = min(ncols, pos + 1 - kbase);
          ex = -1;
        } else {
          lo = 0;
          hi = ncols;
          ex = (p.agent >= kbase && p.agent < kbase + kBN && pos != p.agent) ? p.agent - kbase : -1;
        }
        ok = wait_bar(&sm.s_full[x], jS & 1u, ctl, status, 5);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++jS;
        OD_TP(82, (int)i, bi);
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < n32; ++c) {
          float sv[32], pv[32];
          tmem_ld32(tS + 32 * c, sv);
          tmem_ld32(tP + 32 * c, pv);
          tmem_wait_ld_dep32(sv);
          tmem_wait_ld_dep32(pv);
          const uint32_t keep = PK ? keep_bits_packed(32 * c, PK, sp, lo, hi) : keep_bits32(32 * c, lo, hi, ex);
          if (kDelta) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 xx = __ffma2_rn(make_float2(sv[2 * j], sv[2 * j + 1]), sl2, nl2);
              const float e0 = ((keep >> (2 * j)) & 1u) ? ex2(xx.x) * pv[2 * j] : 0.f;
              const float e1 = ((keep >> (2 * j + 1)) & 1u) ? ex2(xx.y) * pv[2 * j + 1] : 0.f;
              dacc[j & 3] += e0 + e1;
            }
            continue;
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 xx = __ffma2_rn(make_float2(sv[2 * j], sv[2 * j + 1]), sl2, nl2);
            const float2 t = __ffma2_rn(make_float2(pv[2 * j], pv[2 * j + 1]), c12, nd2);
            const float2 d = __fmul2_rn(make_float2(ex2(xx.x), ex2(xx.y)), t);
            // masked (and stale, beyond the block's N) columns give exactly zero: select,
            // never multiply, since stale TMEM may hold NaN
            pk[j] = pack_f16x2(((keep >> (2 * j)) & 1u) ? d.x : 0.f, ((keep >> (2 * j + 1)) & 1u) ? d.y : 0.f);
          }
          tmem_st16(tS + 16 * c, pk);   // dS (fp16 pairs, times 2^eds) over the scores already read
        }
        OD_TP(83, (int)i, bi);
        if (!kDelta) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ds_full[x]);
        OD_TP(84, (int)i, bi);
      }
      if (!ok) break;
      if (kDelta) {
        if (row_ok) {
          const float d = (dacc[0] + dacc[1]) + (dacc[2] + dacc[3]);
          dp.delta[row] = d;
          dmax = max(dmax, __float_as_uint(fabsf(d)));
        }
        continue;
      }
      // ---------------------------------------------------------------- epilogue
      ok = wait_bar(&sm.dq_done[x], jD & 1u, ctl, status, 8);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++jD;
      OD_TP(85, (int)i, 0);
      tc_fence_after();
      float o[64];
      tmem_ld32(tQ, o);
      tmem_ld32(tQ + 32, o + 32);
      tmem_wait_ld_dep32(o);
      tmem_wait_ld_dep32(o + 32);
      if (row_ok && dp.dq_f32) {
        float4* dst = reinterpret_cast<float4*>(dp.dq_f32 + row * 64);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dst[c] = make_float4(o[4 * c] * fq, o[4 * c + 1] * fq, o[4 * c + 2] * fq, o[4 * c + 3] * fq);
      }
      {
        uint8_t* stg = sOst + (warp & 7) * 4096;
        const int wr = lane;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 wv;
          wv.x = pack_bf16x2(o[8 * c + 0] * fq, o[8 * c + 1] * fq);
          wv.y = pack_bf16x2(o[8 * c + 2] * fq, o[8 * c + 3] * fq);
          wv.z = pack_bf16x2(o[8 * c + 4] * fq, o[8 * c + 5] * fq);
          wv.w = pack_bf16x2(o[8 * c + 6] * fq, o[8 * c + 7] * fq);
          *reinterpret_cast<uint4*>(stg + wr * 128 + ((c ^ (wr & 7)) << 4)) = wv;
        }
        __syncwarp();
        // rows 4k + sub of the warp, 8 lanes x 16 bytes per row; each row's dQ row comes
        // from the row's own lane (-1: no row)
        const int sub = lane >> 3, ch = lane & 7;
        const long long rq = row_ok ? tix * dp.dq_rows + it.kvh * G + g : -1LL;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + sub;
          const long long rw = __shfl_sync(0xffffffffu, rq, rr);
          if (rw >= 0) {
            const uint4 wv = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
            if (OD_IN_RANGE(rw, static_cast<long long>(p.B) * p.T * p.S * dp.dq_rows, status, 213))
              reinterpret_cast<uint4*>(dp.dq + rw * 64)[ch] = wv;
          }
        }
        __syncwarp();
      }
    }
    if (kDelta || from_o) {
      __syncwarp();
      const uint32_t m = __reduce_max_sync(0xffffffffu, dmax);
      const float md = amax_reduce(mdo);
      if (lane == 0) {
        atomicMax(&sm.dmax_bits, m);
        atomicMax(&sm.domax_bits, __float_as_uint(md));
      }
    }
  }

  OD_TRACE_END();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if ((kDelta || dp.o != nullptr) && tid == 0) {
    dp.amax[kAmaxStride * blockIdx.x + kAmDelta] = __uint_as_float(sm.dmax_bits);
    if (!kDelta) dp.amax[kAmaxStride * blockIdx.x + kAmDo] = __uint_as_float(sm.domax_bits);
  }
  if (warp == kQsMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dK/dV kernel
// A CTA item is (unit, block of 128 keys); keys are TMEM lanes.  Every Q tile that can see
// the block (nTok positions x G heads, as in the forward) is processed as two 64-row halves
// h = 0, 1, each owned by its own warpgroup, so that the tensor core computes one half
// while the other half's elementwise work runs:
//   S^T_h = K Q_h^T and dP^T_h = V dO_h^T         (TMEM columns [128h, 128h+64), +64)
//   P^T = exp2(S^T sl - LSE2),  dS^T = P^T (dP^T - Delta)   written as fp16 in place
//   dV += P^T dO_h,  dK += dS^T Q_h                (TMEM [256,320) and [320,384))
// All four operands are fp16 scaled by powers of two (see "fp16 operand scaling").  K and V
// of the item are the A operands of the first two products and live in TMEM ([384,416) and
// [416,448)): the elementwise warpgroups write them there at the start of each item, so
// every MMA reads only its B operand (a 64-row half tile) from shared memory.  The
// converter warps rewrite each Q/dO tile in place as scaled fp16 after its TMA load.
// Warps: 0-3 half 0, 4-7 half 1 (elementwise, then the epilogue: dK by warps 0-3, dV by
// warps 4-7), 8 TMA producer + per-row LSE/Delta copies, 9 TMEM allocator + MMA issuer
// (whole warp, one elected lane issues), 10-15 converters (a third of Q or of dO each: with
// two converter warps the conversion paced the kernel).  K/V blocks are double-buffered in
// shared memory across items; Q/dO tiles stream through kKvQSlots slots.  CTA c takes items
// c, then 2*grid-1-c, then 2*grid+c, ... so the items in flight at any time are consecutive
// (the key blocks of one unit share its Q/dO tiles through L2) and alternate between cheaper
// and dearer blocks.
constexpr int kKvBN = 128;
constexpr int kKvThreads = 512;
constexpr int kKvLaunchRegs = 128;   // 65536 registers / 512 threads
constexpr int kKvQSlots = 4;
constexpr int kKvProducerWarp = 8;
constexpr int kKvMmaWarp = 9;
constexpr int kKvConvWarp = 10;   // warps 10-12 convert Q, 13-15 dO (a third of each tile)
constexpr int kKvConvParts = 3;

struct KvParams {
  FwdParams f;            // shapes (item fields unused)
  const float* lse;
  const float* delta;
  const float* amax;      // operand-range slots (see "fp16 operand scaling")
  int amax_slots;         // slots the first launch wrote (max|K|, max|V|)
  int dq_slots;           // slots the dQ pass wrote (max|Q|)
  int dd_slots;           // slots holding max|dO| and max|Delta| (the Delta pass's, or the
                          // dQ pass's when it formed Delta from O)
  float scale;
  long long nitems;       // units x key blocks
  int nkb;                // 128-key blocks per unit
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int kv_rows;            // 64-element rows per token of dk / dv (Hkv, or Hq + 2 Hkv when packed)
  float* dk_f32;          // optional, contiguous [B,T,S,Hkv,64]
  float* dv_f32;
};

struct KvSmem {
  uint64_t kv_full[2], kv_tmem[2];   // K/V block landed; copied into TMEM (slot reusable)
  uint64_t q_full[kKvQSlots], q16[kKvQSlots], q_empty[kKvQSlots];
  uint64_t sp_full[2], p_full[2], acc_done, acc_free;
  uint64_t drain;
  uint32_t tmem_base;
  Ctl ctl;
  int eq, ek, ev, edo;               // fp16 scale exponents
  float don8, dmax;                  // 8 max|dO| >= every ||dO_i||; max|Delta|
  alignas(16) float nlse2[kKvQSlots][128];  // -log2(e) LSE per tile row (-inf: no row)
  alignas(16) float ndel[kKvQSlots][128];   // -Delta per tile row
};
static_assert(offsetof(KvSmem, nlse2) % 16 == 0 && offsetof(KvSmem, ndel) % 16 == 0,
              "row arrays are read with 16-byte loads");
// smem: [K0 V0 K1 V1][Q dO per slot][KvSmem]
constexpr size_t kKvTileBytes = size_t(4) * kTile + size_t(2 * kKvQSlots) * kTile;
constexpr size_t kKvSmemBytes = kKvTileBytes + 1024 + sizeof(KvSmem) + 64;
static_assert(kKvSmemBytes <= 227 * 1024, "shared memory budget");
constexpr int kKvElemRegs = 176;   // elementwise warpgroups
constexpr int kKvCtrlRegs = 80;    // producer, issuer, converters
static_assert(2 * 128 * kKvElemRegs + 256 * kKvCtrlRegs == kKvThreads * kKvLaunchRegs,
              "register split must add up to the launch allocation");

struct KvItem {
  int b, fixed, kvh, kb;
  int L;           // the unit's sequence length
  int valid;       // 0: the key block starts past the unit's length (skipped by every role)
  int t_lo, t_hi;  // Q tiles [t_lo, t_hi] that can see the key block
};
template <bool kVarlen, bool kPacked>
__device__ __forceinline__ KvItem kv_decode(const KvParams& kp, long long i) {
  const FwdParams& p = kp.f;
  KvItem it;
  const uint32_t ii = static_cast<uint32_t>(i);
  const uint32_t unit = ii / static_cast<uint32_t>(kp.nkb);
  it.kb = static_cast<int>(ii - unit * static_cast<uint32_t>(kp.nkb));
  const uint32_t r = unit / static_cast<uint32_t>(p.Hkv);
  it.kvh = static_cast<int>(unit - r * static_cast<uint32_t>(p.Hkv));
  const uint32_t bq = r / static_cast<uint32_t>(p.F);
  it.fixed = static_cast<int>(r - bq * static_cast<uint32_t>(p.F));
  it.b = static_cast<int>(bq);
  if (kPacked && p.pk) {  // packed time attention: `fixed` counts groups of pk positions
    it.L = p.L;
    it.valid = 1;
    it.t_lo = it.t_hi = 0;
    return it;
  }
  int L = p.L;
  if (kVarlen) L = min(max(__ldg(p.seqlen + static_cast<long long>(it.b) * p.T + it.fixed), 0), p.L);
  it.L = L;
  const int k0 = it.kb * kKvBN;
  it.valid = kVarlen ? k0 < L : 1;
  const int k1 = min(L, k0 + kKvBN) - 1;
  if (p.is_time) {
    it.t_lo = k0 / p.nTok;
    it.t_hi = min(L - 1, k1 + p.window - 1) / p.nTok;
  } else {
    it.t_lo = 0;
    it.t_hi = kVarlen ? (L - 1) / p.nTok : p.ntiles - 1;
  }
  return it;
}

// The CTA's item sequence: round r takes item r*grid + c (r even) or r*grid + grid-1-c.
template <bool kVarlen, bool kPacked>
struct KvSeq {
  long long round = 0;
  __device__ __forceinline__ bool next(const KvParams& kp, KvItem* it) {
    for (;;) {
      const long long base = round * static_cast<long long>(gridDim.x);
      if (base >= kp.nitems) return false;
      const long long c = (round & 1) ? static_cast<long long>(gridDim.x - 1 - blockIdx.x)
                                      : static_cast<long long>(blockIdx.x);
      ++round;
      if (base + c < kp.nitems) {
        *it = kv_decode<kVarlen, kPacked>(kp, base + c);
        if (!kVarlen || it->valid) return true;  // blocks past the length: no role sees them
      }
    }
  }
};

// One 32-column chunk of a key lane's elementwise step: P = exp2(S sl + nlse2) (zero
// outside the lane's rows when kMasked), dS = (P sj) (dP c1 + ndel); both packed as fp16
// pairs.
template <bool kMasked>
__device__ __forceinline__ void dkdv_chunk(const float* sv, const float* dv, const float* NL,
                                           const float* ND, float2 sl2, float2 c12, float2 sj2,
                                           uint32_t keep, uint32_t* pk, uint32_t* dk) {
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 l4 = *reinterpret_cast<const float4*>(NL + 4 * j4);
    const float4 d4 = *reinterpret_cast<const float4*>(ND + 4 * j4);
    const float2 x0 = __ffma2_rn(make_float2(sv[4 * j4], sv[4 * j4 + 1]), sl2, make_float2(l4.x, l4.y));
    const float2 x1 = __ffma2_rn(make_float2(sv[4 * j4 + 2], sv[4 * j4 + 3]), sl2, make_float2(l4.z, l4.w));
    float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
    float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
    if (kMasked) {
      const uint32_t kb = keep >> (4 * j4);
      p0.x = (kb & 1u) ? p0.x : 0.f;
      p0.y = (kb & 2u) ? p0.y : 0.f;
      p1.x = (kb & 4u) ? p1.x : 0.f;
      p1.y = (kb & 8u) ? p1.y : 0.f;
    }
    const float2 t0 = __ffma2_rn(make_float2(dv[4 * j4], dv[4 * j4 + 1]), c12, make_float2(d4.x, d4.y));
    const float2 t1 = __ffma2_rn(make_float2(dv[4 * j4 + 2], dv[4 * j4 + 3]), c12, make_float2(d4.z, d4.w));
    const float2 s0 = __fmul2_rn(__fmul2_rn(p0, sj2), t0);
    const float2 s1 = __fmul2_rn(__fmul2_rn(p1, sj2), t1);
    pk[2 * j4] = pack_f16x2(p0.x, p0.y);
    pk[2 * j4 + 1] = pack_f16x2(p1.x, p1.y);
    dk[2 * j4] = pack_f16x2(s0.x, s0.y);
    dk[2 * j4 + 1] = pack_f16x2(s1.x, s1.y);
  }
}


template <bool kVarlen, bool kPacked>
__global__ void __launch_bounds__(kKvThreads, 1)
    od_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const KvParams kp) {
  const FwdParams& p = kp.f;
  const int PK = kPacked ? p.pk : 0;   // packed: token positions per key block
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start of the dynamic shared memory, formed by pointer arithmetic on the
  // __shared__ array (not through an integer) so that every tile is addressed as shared memory
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sKV = base;                     // slot s: K at 2s*kTile, V at (2s+1)*kTile
  uint8_t* sQD = base + 4 * kTile;         // slot q: Q at 2q*kTile, dO at (2q+1)*kTile
  KvSmem& sm = *reinterpret_cast<KvSmem*>(base + kKvTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  OD_TRACE_INIT(2);

  {  // tile rows that TMA never writes stay zero (after conversion too)
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kKvThreads * 16)
      for (int t = 0; t < 2 * kKvQSlots; ++t)
        *reinterpret_cast<uint4*>(sQD + t * kTile + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
    const int kvpad = (kKvBN - p.kvb) * 128;   // packed: K/V rows past the block's pk T keys
    for (int x = tid * 16; x < kvpad; x += kKvThreads * 16)
      for (int t = 0; t < 4; ++t)
        *reinterpret_cast<uint4*>(sKV + t * kTile + p.kvb * 128 + x) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    for (int x = tid; x < kKvQSlots * 128; x += kKvThreads) {
      (&sm.nlse2[0][0])[x] = 0.f;
      (&sm.ndel[0][0])[x] = 0.f;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_tmem[s], 8);
      mbar_init(&sm.sp_full[s], 1);
      mbar_init(&sm.p_full[s], 4);
    }
    for (int q = 0; q < kKvQSlots; ++q) {
      mbar_init(&sm.q_full[q], 1 + 32);  // TMA issuer + the producer lanes' row copies
      mbar_init(&sm.q16[q], 2 * kKvConvParts);
      mbar_init(&sm.q_empty[q], 1);
    }
    mbar_init(&sm.acc_done, 1);
    mbar_init(&sm.acc_free, 8);
    mbar_init(&sm.drain, 1);
    sm.ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kKvProducerWarp) {
    // operand ranges recorded by the first launch and the dQ pass -> scale exponents
    const float aq = slots_max(kp.amax, kp.dq_slots, kAmQ, lane);
    const float ak = slots_max(kp.amax, kp.amax_slots, kAmK, lane);
    const float av = slots_max(kp.amax, kp.amax_slots, kAmV, lane);
    const float ado = slots_max(kp.amax, kp.dd_slots, kAmDo, lane);
    const float adl = slots_max(kp.amax, kp.dd_slots, kAmDelta, lane);
    if (lane == 0) {
      sm.eq = fp16_shift(aq);
      sm.ek = fp16_shift(ak);
      sm.ev = fp16_shift(av);
      sm.edo = fp16_shift(ado);
      sm.don8 = 8.f * ado;
      sm.dmax = adl;
    }
  }
  if (warp == kKvMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  Ctl* ctl = &sm.ctl;
  unsigned int* status = p.status;
  const int eq = sm.eq, ek = sm.ek, ev = sm.ev, edo = sm.edo;

  if (warp >= 8) {
    regs_dec<kKvCtrlRegs>();
    if (warp == kKvProducerWarp) {
      // ---------------------------------------------------------- producer (whole warp)
      KvSeq<kVarlen, kPacked> seq;
      KvItem it;
      uint32_t n = 0, tau = 0;
      bool ok = true;
      while (ok && seq.next(kp, &it)) {
        const int slot = n & 1;
        if (n >= 2) {
          ok = __all_sync(0xffffffffu, wait_bar(&sm.kv_tmem[slot], ((n >> 1) - 1) & 1u, ctl, status, 20));
          if (!ok) break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.kv_full[slot], 2 * p.kvb * 128);
          const int k0 = it.kb * kKvBN;
          // box start (s, t): packed time, time, space
          const int cs = PK ? it.fixed * PK : (p.is_time ? it.fixed : k0);
          const int ct = PK ? 0 : (p.is_time ? k0 : it.fixed);
          (void)OD_TMA_OK(it.kvh, cs, ct, it.b, p.Hkv, p.S, p.T, p.B, status, 220);
          uint8_t* dK = sKV + (2 * slot) * kTile;
          uint8_t* dV = sKV + (2 * slot + 1) * kTile;
          tma_load_5d(dK, &tm_k, &sm.kv_full[slot], 0, it.kvh, cs, ct, it.b);
          tma_load_5d(dV, &tm_v, &sm.kv_full[slot], 0, it.kvh, cs, ct, it.b);
        }
        ++n;
        for (int tq = it.t_lo; tq <= it.t_hi && ok; ++tq, ++tau) {
          const int q = static_cast<int>(tau % kKvQSlots);
          OD_TP(50, (int)tau, 0);
          if (tau >= kKvQSlots) {
            ok = __all_sync(0xffffffffu,
                            wait_bar(&sm.q_empty[q], ((tau / kKvQSlots) - 1) & 1u, ctl, status, 21));
            if (!ok) break;
          }
          const int t0 = tq * p.nTok;
          const int s0 = it.fixed * PK;   // packed: the block's first token position
          if (lane == 0) {
            const int cs = PK ? s0 : (p.is_time ? it.fixed : t0);
            const int ct = PK ? 0 : (p.is_time ? t0 : it.fixed);
            (void)OD_TMA_OK(it.kvh * p.G, cs, ct, it.b, p.Hq, p.S, p.T, p.B, status, 221);
            uint8_t* dQ = sQD + (2 * q) * kTile;
            uint8_t* dO = sQD + (2 * q + 1) * kTile;
            mbar_arrive_expect_tx(&sm.q_full[q], 2 * p.rows * 128);
            tma_load_5d(dQ, &tm_q, &sm.q_full[q], 0, it.kvh * p.G, cs, ct, it.b);
            tma_load_5d(dO, &tm_do, &sm.q_full[q], 0, it.kvh * p.G, cs, ct, it.b);
          }
          // raw LSE and Delta of the tile's rows, copied asynchronously (the converters
          // rescale them); rows outside the sequence keep finite stale values, which only
          // ever meet the zero Q/dO rows of the tile
          for (int rr = lane; rr < p.rows; rr += 32) {
            const int tk = rr / p.G;
            const int tpk = PK ? tk / PK : 0;
            const int sp = PK ? tk - tpk * PK : 0;
            const int ps = PK ? tpk : t0 + tk;
            if (PK ? s0 + sp < p.S : ps < (kVarlen ? it.L : p.L)) {
              const long long t_idx = p.is_time ? ps : it.fixed;
              const long long s_idx = PK ? s0 + sp : (p.is_time ? it.fixed : ps);
              const long long row = ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq +
                                    it.kvh * p.G + (rr - tk * p.G);
              cp_async4(&sm.nlse2[q][rr], kp.lse + row);
              cp_async4(&sm.ndel[q][rr], kp.delta + row);
            }
          }
          cp_async_arrive_noinc(&sm.q_full[q]);
          OD_TP(51, (int)tau, 0);
        }
      }
      if (lane == 0) {  // no TMA load may still be writing when the CTA exits
        for (int s = 0; s < 2; ++s) {
          const uint32_t uses = n / 2 + (static_cast<uint32_t>(s) < (n & 1u) ? 1u : 0u);
          if (uses > 0) drain_wait(&sm.kv_full[s], (uses - 1) & 1u);
        }
        for (int q = 0; q < kKvQSlots; ++q) {
          const uint32_t uses = tau / kKvQSlots + (static_cast<uint32_t>(q) < tau % kKvQSlots ? 1u : 0u);
          if (uses > 0) drain_wait(&sm.q_full[q], (uses - 1) & 1u);
        }
      }
    } else if (warp == kKvMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      // Order: SP_0(0) SP_1(0); per tile t: [P_0(t)] DKV_0(t) SP_0(t+1) [P_1(t)] DKV_1(t)
      // SP_1(t+1).  SP_h(t+1) overwrites half h's buffer after DKV_h(t) has been issued
      // (tcgen05 MMAs of one thread run in issue order).  The whole warp runs this loop in
      // lockstep; one elected lane issues every MMA and commit.
      {
        const uint32_t idesc_sp = idesc_fp16(128, 64, 0, 0);   // M keys, N 64 tile rows
        const uint32_t idesc_acc = idesc_fp16(128, 64, 0, 1);  // M keys, N head dim, B MN-major
        const uint32_t tDK = tmem + 256, tDV = tmem + 320;
        KvSeq<kVarlen, kPacked> seq;
        KvItem cur, nxt;
        bool ok = seq.next(kp, &cur);
        uint32_t n = 0, tau = 0;      // item and tile ordinals of the current tile
        int k = 0;                    // tile within the current item
        // descriptors of slot 0's Q tile (K-major, and MN-major for the dK/dV products); a
        // half tile of a slot is these plus its offset in 16-byte units (addresses < 2^18)
        const uint64_t d_qk = sdesc_sw128(smem_u32(sQD), 16, 1024);
        const uint64_t d_qm = sdesc_sw128(smem_u32(sQD), 1024, 1024);
        auto half_off = [&](uint32_t t, int which, int h) -> uint64_t {
          const uint32_t q = t % kKvQSlots;
          return static_cast<uint64_t>(((2 * q + which) * kTile + h * 8192) >> 4);
        };
        auto issue_sp = [&](int h, uint32_t t) {
          const uint64_t bq = d_qk + half_off(t, 0, h);
          const uint64_t bo = d_qk + half_off(t, 1, h);
          const uint32_t dS = tmem + 128u * h, dP = dS + 64u;
          const uint32_t aK = tmem + 384u, aV = tmem + 416u;
          mma_ts_k64_kb_w(dS, aK, bq, idesc_sp);
          mma_ts_k64_kb_w(dP, aV, bo, idesc_sp);
          mma_commit_w(&sm.sp_full[h]);
        };
        auto issue_dkv = [&](int h, uint32_t t, bool first) {
          const uint64_t bq = d_qm + half_off(t, 0, h);
          const uint64_t bo = d_qm + half_off(t, 1, h);
          const uint32_t aP = tmem + 128u * h, aD = aP + 64u;
          mma_ts_k64_w(tDV, aP, bo, idesc_acc, first ? 0u : 1u);
          mma_ts_k64_w(tDK, aD, bq, idesc_acc, first ? 0u : 1u);
        };
        // waits for the operands of tile t (item ordinal item_n, new item or not)
        auto wait_operands = [&](uint32_t t, uint32_t item_n, bool new_item) -> bool {
          if (new_item && !__all_sync(0xffffffffu, wait_bar(&sm.kv_tmem[item_n & 1], (item_n >> 1) & 1u, ctl, status, 30))) return false;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.q16[t % kKvQSlots], (t / kKvQSlots) & 1u, ctl, status, 31))) return false;
          tc_fence_after();
          return true;
        };
        if (ok) {
          ok = wait_operands(0, 0, true);
          if (ok) {
            issue_sp(0, 0);
            issue_sp(1, 0);
          }
        }
        while (ok) {
          const int ntl = cur.t_hi - cur.t_lo + 1;
          // successor tile
          bool has_next = true, next_new = false;
          nxt = cur;
          if (k + 1 >= ntl) {
            has_next = seq.next(kp, &nxt);
            next_new = true;
          }
          const uint32_t n1 = next_new ? n + 1 : n;
          const int k1 = next_new ? 0 : k + 1;
          // ---- half 0
          if (!__all_sync(0xffffffffu, wait_bar(&sm.p_full[0], tau & 1u, ctl, status, 32))) break;
          if (k == 0 && n > 0 && !__all_sync(0xffffffffu, wait_bar(&sm.acc_free, (n - 1) & 1u, ctl, status, 33))) break;
          tc_fence_after();
          issue_dkv(0, tau, k == 0);
          OD_TP(61, (int)tau, 0);
          if (has_next && !next_new) {
            if (!wait_operands(tau + 1, n1, false)) break;
            issue_sp(0, tau + 1);
            OD_TP(62, (int)tau, 0);
          }
          // ---- half 1
          OD_TP(63, (int)tau, 0);
          if (!__all_sync(0xffffffffu, wait_bar(&sm.p_full[1], tau & 1u, ctl, status, 34))) break;
          tc_fence_after();
          issue_dkv(1, tau, false);
          OD_TP(64, (int)tau, 0);
          mma_commit_w(&sm.q_empty[tau % kKvQSlots]);
          if (k == ntl - 1) mma_commit_w(&sm.acc_done);
          if (!has_next) break;
          // A new item's K/V reach TMEM only after its warpgroups have read this item's
          // accumulators, which needs DKV_1 above: its first S/dP products go out here.
          if (next_new) {
            if (!wait_operands(tau + 1, n1, true)) break;
            issue_sp(0, tau + 1);
          }
          issue_sp(1, tau + 1);
          cur = nxt;
          n = n1;
          k = k1;
          ++tau;
        }
        mma_commit_w(&sm.drain);
        drain_wait(&sm.drain, 0);
      }
    } else {
      // ---------------------------------------------------------- converters (10-15)
      // Warps 10-12 rewrite a third each of every Q tile's rows as fp16 times 2^eq, warps
      // 13-15 the same of dO times 2^edo; warp 10 also turns the rows' raw LSE into
      // -log2(e) LSE and warp 13 the raw Delta into -Delta (0 for rows outside the sequence).
      const int which = (warp - kKvConvWarp) / kKvConvParts;  // 0: Q, 1: dO
      const int part = (warp - kKvConvWarp) % kKvConvParts;
      const float sqd = ldexpf(1.f, which ? edo : eq);
      const float rowf = which ? -1.f : -1.4426950408889634f;
      const int nch = p.rows * 8;                               // 16-byte chunks of a tile
      const int c0 = (nch * part) / kKvConvParts, c1 = (nch * (part + 1)) / kKvConvParts;
      int tok_of[4];                                            // (lane + 32 k) / G
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tok_of[k] = (lane + 32 * k) / p.G;
        if (PK) tok_of[k] %= PK;                            // packed: the row's token
      }
      KvSeq<kVarlen, kPacked> seq;
      KvItem it;
      uint32_t n = 0, tau = 0;
      bool ok = true;
      while (ok && seq.next(kp, &it)) {
        ++n;
        for (int tq = it.t_lo; tq <= it.t_hi && ok; ++tq, ++tau) {
          const int q = static_cast<int>(tau % kKvQSlots);
          OD_TP(70, (int)tau, 0);
          ok = __all_sync(0xffffffffu, wait_bar(&sm.q_full[q], (tau / kKvQSlots) & 1u, ctl, status, 36));
          if (!ok) break;
          OD_TP(71, (int)tau, 0);
          to_fp16_scaled(sQD + (2 * q + which) * kTile + c0 * 16, (c1 - c0) * 16, sqd, lane);
          OD_TP(72, (int)tau, 0);
          if (part == 0) {  // rows of the tile: -log2(e) LSE (Q warp) or -Delta (dO warp); 0 elsewhere
            float* rowv = which ? sm.ndel[q] : sm.nlse2[q];
            const int t0 = tq * p.nTok;
            const int L = kVarlen ? it.L : p.L;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rr = lane + 32 * k;
              const bool valid = rr < p.rows && (PK ? it.fixed * PK + tok_of[k] < p.S : t0 + tok_of[k] < L);
              rowv[rr] = valid ? rowv[rr] * rowf : 0.f;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.q16[q]);
          OD_TP(73, (int)tau, 0);
        }
      }
    }
  } else {
    regs_inc<kKvElemRegs>();
    // ------------------------------------------------------------ elementwise (key lanes)
    const int h = warp >> 2;               // tile half: rows [64h, 64h+64)
    const int j = tid & 127;               // key lane within the block
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128u * h + lane_off, tD = tS + 64u;
    // logits: S^T carries 2^(eq+ek), dP^T carries 2^(edo+ev); dS^T is written times 2^eds,
    // eds from this key's bound ||v_j|| 8 max|dO| + max|Delta| on |dS|
    const float slx = p.sl * ldexpf(1.f, -(eq + ek));
    const float c1 = ldexpf(1.f, -(edo + ev));
    const float2 sl2 = make_float2(slx, slx), c12 = make_float2(c1, c1);
    const float don8 = sm.don8, dmax = sm.dmax;
    int eds = 0;
    float2 sj2 = make_float2(1.f, 1.f);
    const int Weff = min(p.window, p.L);
    const float skv = ldexpf(1.f, h ? ev : ek);
    KvSeq<kVarlen, kPacked> seq;
    KvItem it;
    uint32_t n = 0, tau = 0;
    bool ok = true;
    while (ok && seq.next(kp, &it)) {
      // the key's sequence position kpos (packed: its frame; spk its token within the block)
      const int tkj = PK ? j / PK : 0;
      const int spk = PK ? j - tkj * PK : 0;
      const int kpos = PK ? tkj : it.kb * kKvBN + j;
      const bool key_ok = PK ? (j < p.kvb && it.fixed * PK + spk < p.S) : kpos < (kVarlen ? it.L : p.L);
      {  // this key's K (half 0) or V (half 1) row -> scaled fp16 -> TMEM A operand columns.
         // The previous item's MMAs have all completed (its epilogue waited for them).
        const int slot = n & 1;
        ok = __all_sync(0xffffffffu, wait_bar(&sm.kv_full[slot], (n >> 1) & 1u, ctl, status, 35));
        if (!ok) break;
        const uint8_t* row = sKV + (2 * slot + h) * kTile + j * 128;
        const float2 s2 = make_float2(skv, skv);
        eds = fp16_shift(fmaf(sqrtf(row_norm2(sKV + (2 * slot + 1) * kTile, j)), don8, dmax));
        sj2 = make_float2(ldexpf(1.f, eds), ldexpf(1.f, eds));
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row sits at chunk c ^ (j & 7)
          const uint4 d = *reinterpret_cast<const uint4*>(row + ((c ^ (j & 7)) << 4));
          const uint32_t x[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __fmul2_rn(make_float2(__uint_as_float(x[e] << 16),
                                                    __uint_as_float(x[e] & 0xFFFF0000u)), s2);
            w[4 * c + e] = pack_f16x2(f.x, f.y);
          }
        }
        tmem_st32(tmem + lane_off + 384u + 32u * h, w);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.kv_tmem[slot]);
      }
      for (int tq = it.t_lo; tq <= it.t_hi && ok; ++tq, ++tau) {
        const int q = static_cast<int>(tau % kKvQSlots);
        OD_TP(40, (int)tau, 0);
        ok = wait_bar(&sm.q16[q], (tau / kKvQSlots) & 1u, ctl, status, 37) &&
             wait_bar(&sm.sp_full[h], tau & 1u, ctl, status, 38);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        OD_TP(41, (int)tau, 0);
        tc_fence_after();
        float sv[64], dv[64];
        tmem_ld32(tS, sv);
        tmem_ld32(tS + 32, sv + 32);
        tmem_ld32(tD, dv);
        tmem_ld32(tD + 32, dv + 32);
        // rows [r_lo, r_hi) of the tile may read this key (rows past the sequence end of a
        // fixed-length unit hold zero Q and dO and contribute nothing)
        const int t0 = tq * p.nTok;
        int r_lo = 0, r_hi = 128;
        if (p.is_time) {
          const long long d = static_cast<long long>(kpos) - t0;
          r_lo = static_cast<int>(min(max(d * p.G, 0LL), 128LL));
          r_hi = static_cast<int>(min(max((d + Weff) * p.G, 0LL), 128LL));
        } else if (kpos == p.agent) {
          const long long d = static_cast<long long>(p.agent) - t0;
          r_lo = static_cast<int>(min(max(d * p.G, 0LL), 128LL));
          r_hi = static_cast<int>(min(max((d + 1) * p.G, 0LL), 128LL));
        }
        // rows past the unit's length (padding of a variable-length block) read nothing
        if (kVarlen && it.L < p.L) r_hi = min(r_hi, static_cast<int>(min(max(static_cast<long long>(it.L - t0) * p.G, 0LL), 128LL)));
        tmem_wait_ld_dep32(sv);
        tmem_wait_ld_dep32(sv + 32);
        tmem_wait_ld_dep32(dv);
        tmem_wait_ld_dep32(dv + 32);
        OD_TP(45, (int)tau, 0);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float* NL = &sm.nlse2[q][64 * h + 32 * c];
          const float* ND = &sm.ndel[q][64 * h + 32 * c];
          const uint32_t keep =
              PK ? (key_ok ? keep_rows_packed(64 * h + 32 * c, p.G, PK, spk, kpos, min(p.L - 1, kpos + Weff - 1)) : 0u)
                   : keep_bits32(64 * h + 32 * c, r_lo, r_hi, -1);
          uint32_t pk[16], dk[16];
          if (__any_sync(0xffffffffu, keep != 0xFFFFFFFFu))
            dkdv_chunk<true>(sv + 32 * c, dv + 32 * c, NL, ND, sl2, c12, sj2, keep, pk, dk);
          else
            dkdv_chunk<false>(sv + 32 * c, dv + 32 * c, NL, ND, sl2, c12, sj2, keep, pk, dk);
          tmem_st16(tS + 16 * c, pk);   // P^T (fp16 pairs) over the scores already read
          tmem_st16(tD + 16 * c, dk);   // dS^T (fp16 pairs, times 2^eds) over dP^T
        }
        OD_TP(46, (int)tau, 0);
        tmem_wait_st();
        OD_TP(47, (int)tau, 0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[h]);
        OD_TP(42, (int)tau, 0);
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue: dK (h 0), dV (h 1)
      OD_TP(43, (int)n, 0);
      ok = __all_sync(0xffffffffu, wait_bar(&sm.acc_done, n & 1u, ctl, status, 39));
      if (!ok) break;
      OD_TP(44, (int)n, 0);
      ++n;
      tc_fence_after();
      float g[64];
      const uint32_t tA = tmem + (h ? 320u : 256u) + lane_off;
      tmem_ld32(tA, g);
      tmem_ld32(tA + 32, g + 32);
      tmem_wait_ld_dep32(g);
      tmem_wait_ld_dep32(g + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_free);
      if (key_ok) {
        const float f = h ? ldexpf(1.f, -edo) : kp.scale * ldexpf(1.f, -(eds + eq));
        const long long t_idx = p.is_time ? kpos : it.fixed;
        const long long s_idx = PK ? it.fixed * PK + spk : (p.is_time ? it.fixed : kpos);
        const long long tok = (static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx;
        if (!OD_IN_RANGE(tok, static_cast<long long>(p.B) * p.T * p.S, status, 222)) continue;
        const long long row = tok * p.Hkv + it.kvh;
        uint4* out = reinterpret_cast<uint4*>((h ? kp.dv : kp.dk) + (tok * kp.kv_rows + it.kvh) * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 a;
          a.x = pack_bf16x2(g[8 * c + 0] * f, g[8 * c + 1] * f);
          a.y = pack_bf16x2(g[8 * c + 2] * f, g[8 * c + 3] * f);
          a.z = pack_bf16x2(g[8 * c + 4] * f, g[8 * c + 5] * f);
          a.w = pack_bf16x2(g[8 * c + 6] * f, g[8 * c + 7] * f);
          out[c] = a;
        }
        float* o32 = h ? kp.dv_f32 : kp.dk_f32;
        if (o32) {
          float4* a = reinterpret_cast<float4*>(o32 + row * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            a[c] = make_float4(g[4 * c] * f, g[4 * c + 1] * f, g[4 * c + 2] * f, g[4 * c + 3] * f);
        }
      }
    }
  }

  OD_TRACE_END();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kKvMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ host side
template <bool kVarlen, bool kPacked>
inline cudaError_t bwd_setup_one() {
  cudaError_t e = cudaFuncSetAttribute(od_bwd_dq_kernel<false, kVarlen, kPacked>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDqSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(od_bwd_dq_kernel<true, kVarlen, kPacked>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kDqSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(od_bwd_dkdv_kernel<kVarlen, kPacked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kKvSmemBytes));
  if (e != cudaSuccess) return e;
  // each kernel redistributes its launch registers between warpgroups (setmaxnreg); the split
  // is only valid for the register count it was designed for
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, od_bwd_dq_kernel<false, kVarlen, kPacked>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kQsLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncGetAttributes(&fa, od_bwd_dq_kernel<true, kVarlen, kPacked>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kQsLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncGetAttributes(&fa, od_bwd_dkdv_kernel<kVarlen, kPacked>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kKvLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}
inline cudaError_t bwd_setup() {
  cudaError_t e = bwd_setup_one<false, false>();
  if (e == cudaSuccess) e = bwd_setup_one<true, false>();
  return e != cudaSuccess ? e : bwd_setup_one<false, true>();
}

// ============================================================================ K/V ranges
// When the forward also wrote O's rounding residual O_lo (O ~ o + o_lo to about 16 significant
// bits), Delta = <dO, O> is a row-wise dot product that the dQ pass forms from its dO tile and
// two row loads (no recompute of P and dP, no extra pass over dO).  The dQ pass then needs
// only the ranges of K and V up front (for K's fp16 scale and the bound on ||v_j||); this
// streaming kernel records max|K| and max|V| per CTA, in the slots the Delta pass would fill.
constexpr int kKvRangeThreads = 256;

struct KvRangeParams {
  const __nv_bfloat16* k;       // views: token i starts at row i * kv_rows
  const __nv_bfloat16* v;
  long long ntok;               // B * T * S
  int Hkv, kv_rows;
  float* amax;                  // one slot of kAmaxStride floats per CTA
};

__global__ void __launch_bounds__(kKvRangeThreads)
    od_bwd_kv_range_kernel(const KvRangeParams p) {
  __shared__ float red[kKvRangeThreads / 32][2];  // per warp: K, V
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gw = static_cast<long long>(blockIdx.x) * (kKvRangeThreads / 32) + warp;
  const long long nw = static_cast<long long>(gridDim.x) * (kKvRangeThreads / 32);
  auto vmax4 = [](uint32_t m, const uint4& x) {
    m = __vmaxu2(m, x.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, x.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, x.z & 0x7FFF7FFFu);
    return __vmaxu2(m, x.w & 0x7FFF7FFFu);
  };
  // A contiguous tensor is one flat array (four 16-byte loads in flight per thread); a packed
  // view is walked token by token (the token's head rows are contiguous), again four loads in
  // flight per lane.
  auto scan = [&](const __nv_bfloat16* base) {
    uint32_t m = 0;
    const uint4* src = reinterpret_cast<const uint4*>(base);
    if (p.kv_rows == p.Hkv) {
      const long long n = p.ntok * p.Hkv * 8;
      const long long nt = static_cast<long long>(gridDim.x) * kKvRangeThreads;
      const long long t0 = static_cast<long long>(blockIdx.x) * kKvRangeThreads + threadIdx.x;
      for (long long c = t0; c < n; c += 4 * nt) {
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          x[u] = (c + u * nt < n) ? __ldg(src + c + u * nt) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) m = vmax4(m, x[u]);
      }
    } else {
      const int nchunk = p.Hkv * 8;
      for (long long t = gw; t < p.ntok; t += nw) {
        const uint4* row = src + t * p.kv_rows * 8;
        for (int c = lane; c < nchunk; c += 128) {
          uint4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            x[u] = (c + 32 * u < nchunk) ? __ldg(row + c + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 4; ++u) m = vmax4(m, x[u]);
        }
      }
    }
    return m;
  };
  const float a[2] = {amax_reduce(scan(p.k)), amax_reduce(scan(p.v))};
  if (lane == 0) {
    red[warp][0] = a[0];
    red[warp][1] = a[1];
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float m = 0.f;
    bool nan = false;
    for (int w = 0; w < kKvRangeThreads / 32; ++w) {
      const float x = red[w][threadIdx.x];
      nan |= !(x == x);
      m = fmaxf(m, x);
    }
    static_assert(kAmK == 0 && kAmV == 1, "slot fields in order");
    p.amax[kAmaxStride * blockIdx.x + threadIdx.x] = nan ? __int_as_float(0x7fc00000) : m;
  }
}

// workspace: Delta (fp32, one per query row), then kAmaxSlots x kAmaxStride fp32 operand ranges
inline size_t bwd_delta_bytes(int B, int T, int S, int Hq) {
  return (size_t(B) * T * S * Hq * sizeof(float) + 255) & ~size_t(255);
}
inline size_t bwd_workspace_bytes(int B, int T, int S, int Hq, int /*D*/) {
  return bwd_delta_bytes(B, T, S, Hq) + size_t(kAmaxSlots) * kAmaxStride * sizeof(float);
}

struct BwdArgs {
  int is_time;
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float *dq_f32, *dk_f32, *dv_f32;
  int B, T, S, Hq, Hkv, D, agent, window;
  float scale;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  unsigned int* status;
  int num_sms;
};

}  // namespace od
