// od_bwd.cuh -- backward of space and time attention (sm_103a).
//
// With P recomputed from the forward's logsumexp (activation checkpointing; edgex es-LA
// page, "Rendimiento de computo y estrategia de memoria"), per query row with allowed
// keys j:  P_j = exp(scale <q, k_j> - LSE),  Delta = <dO, O>,  dP_j = <dO, v_j>,
// dS_j = P_j (dP_j - Delta),  dQ = scale sum_j dS_j k_j,  dK_j += scale dS_j q,
// dV_j += P_j dO  (dK, dV summed over the G query heads of a KV head).
//
// Three launches, no atomics, no zeroed workspace (results are deterministic):
//   1. od_bwd_dq_kernel<true>: Delta = sum_j P_j dP_j per row in fp32 into the caller's
//        workspace.  It equals <dO, O> for the exact O; the bf16 O passed in would give
//        Delta only to ~1e-2 absolute, which the gradients inherit.
//   2. od_bwd_dq_kernel<false>: Q-tile stationary (the forward's work items and warp roles):
//        S = Q K^T and dP = dO V^T per 96-key block in TMEM; dS split into bf16 high parts
//        (in place over S) and bf16 residuals (in place over dP); dQ += dS K as two MMAs per
//        step into one fp32 accumulator, written once per tile.
//   3. od_bwd_dkdv_kernel:  key-block stationary: a CTA item is (unit, 128-key block);
//        for every Q tile that can see the block, S^T = K Q^T and dP^T = V dO^T in TMEM
//        (keys on TMEM lanes), P^T and dS^T written in place (bf16), then
//        dV += P^T dO and dK += dS^T Q accumulate in TMEM.  All G heads of the group are
//        rows of the same Q tile, so the GQA reduction of dK/dV happens on chip.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include "od_ptx.cuh"
#include "od_fwd.cuh"

namespace od {

// ============================================================================ dQ kernel
// Work items, Q tiles, key blocks and K/V staging as in the forward (FwdParams, fwd_decode).
// TMEM per tile x (256 columns at 256 x): S [0,96), dP [96,192), dQ [192,256).
constexpr int kDqThreads = 384;
constexpr int kDqStages = 5;
static_assert(2 * 128 * kFwdSoftmaxRegs + 128 * kFwdCtrlRegs == kDqThreads * kFwdLaunchRegs,
              "register split must add up to the launch allocation");

struct DqParams {
  FwdParams f;            // shapes and item schedule (f.o unused)
  const float* lse;       // forward logsumexp (natural log)
  float* delta;           // Delta per query row (written by the Delta pass, read otherwise)
  float scale;
  __nv_bfloat16* dq;
  float* dq_f32;          // optional
};

struct DqSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kDqStages], v_full[kDqStages], kv_empty[kDqStages];
  uint64_t s_full[2], ds_full[2], dq_done[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  Ctl ctl;
};
// smem: [Q0 Q1 dO0 dO1][K stages][V stages][dQ staging 8 x 4 KB][DqSmem]
constexpr size_t kDqTileBytes = size_t(4) * kTile + size_t(2 * kDqStages) * kKVTile + 8 * 4096;
constexpr size_t kDqSmemBytes = kDqTileBytes + 1024 + sizeof(DqSmem) + 64;
static_assert(kDqSmemBytes <= 227 * 1024, "shared memory budget");

// kDelta = true: the Delta pass -- S and dP per key block, Delta = sum_j P_j dP_j accumulated
// in fp32 per row and written to the workspace (no dS, no dQ).  This is <dO, O> for the exact
// forward output, which the bf16 O given to the backward only approximates.
template <bool kDelta>
__global__ void __launch_bounds__(kDqThreads, 1)
    od_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DqParams dp) {
  const FwdParams& p = dp.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ[2] = {base, base + kTile};
  uint8_t* sdO[2] = {base + 2 * kTile, base + 3 * kTile};
  uint8_t* sK = base + 4 * kTile;
  uint8_t* sV = sK + kDqStages * kKVTile;
  uint8_t* sOst = sV + kDqStages * kKVTile;
  DqSmem& sm = *reinterpret_cast<DqSmem*>(base + kDqTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long i0 = (p.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = (p.nitems * (blockIdx.x + 1)) / gridDim.x;
  const bool resident = p.nkb <= kDqStages;

  {  // zero the tile rows TMA never writes
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kDqThreads * 16)
      for (int t = 0; t < 2; ++t) {
        *reinterpret_cast<uint4*>(sQ[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sdO[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
      }
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.q_full[x], 1);
      mbar_init(&sm.q_empty[x], 1);
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.ds_full[x], 4);
      mbar_init(&sm.dq_done[x], 1);
      mbar_init(&sm.drain[x], 1);
    }
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 2);
    }
    sm.ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kFwdMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  Ctl* ctl = &sm.ctl;
  unsigned int* status = p.status;

  if (warp >= 8) {
    regs_dec<kFwdCtrlRegs>();
    if (warp == kFwdProducerWarp) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        long long prev_unit = -1;
        uint32_t unit_loads = 0, sbase = 0, qn[2] = {0, 0};
        bool ok = true;
        for (long long i = i0; i < i1 && ok; ++i) {
          const FwdItem it = fwd_decode(p, i);
          const int nb = it.kb_hi - it.kb_lo + 1;
          auto load_kv = [&](int stage, int kb) {
            const int kp = kb * kBN;
            mbar_arrive_expect_tx(&sm.k_full[stage], kKVTile);
            mbar_arrive_expect_tx(&sm.v_full[stage], kKVTile);
            if (p.is_time) {
              tma_load_5d(sK + stage * kKVTile, &tm_k, &sm.k_full[stage], 0, it.kvh, it.fixed, kp, it.b);
              tma_load_5d(sV + stage * kKVTile, &tm_v, &sm.v_full[stage], 0, it.kvh, it.fixed, kp, it.b);
            } else {
              tma_load_5d(sK + stage * kKVTile, &tm_k, &sm.k_full[stage], 0, it.kvh, kp, it.fixed, it.b);
              tma_load_5d(sV + stage * kKVTile, &tm_v, &sm.v_full[stage], 0, it.kvh, kp, it.fixed, it.b);
            }
          };
          for (int x = 0; x < 2 && ok; ++x) {
            if (x == 1 && !it.validB) break;
            if (qn[x] > 0) ok = wait_bar(&sm.q_empty[x], (qn[x] - 1) & 1u, ctl, status, 1);
            if (!ok) break;
            const int t0 = x ? it.tok0[1] : it.tok0[0];
            mbar_arrive_expect_tx(&sm.q_full[x], 2 * p.rows * 128);
            if (p.is_time) {
              tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, it.fixed, t0, it.b);
              tma_load_5d(sdO[x], &tm_do, &sm.q_full[x], 0, it.kvh * p.G, it.fixed, t0, it.b);
            } else {
              tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, t0, it.fixed, it.b);
              tma_load_5d(sdO[x], &tm_do, &sm.q_full[x], 0, it.kvh * p.G, t0, it.fixed, it.b);
            }
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
    } else if (warp == kFwdMmaWarp || warp == kFwdMmaWarp + 1) {
      // ---------------------------------------------------------- MMA issuers (per tile)
      // In order per tile: S(0), dP(0); then for each block j: wait dS(j), dQ += dS(j) K;
      // S(j+1), dP(j+1) (they overwrite buffers whose last reader was issued before them).
      if (lane == 0) {
        const int x = warp - kFwdMmaWarp;
        const uint32_t tS = tmem + 256u * x, tP = tS + 96u, tQ = tS + 192u;
        const uint32_t idesc_dq = idesc_bf16(128, 64, 0, 1);
        uint32_t js = 0, jd = 0, qn = 0, unit_loads = 0, sbase = 0;
        long long prev_unit = -1;
        bool ok = true;
        for (long long i = i0; i < i1 && ok; ++i) {
          const FwdItem it = fwd_decode(p, i);
          const int nb = it.kb_hi - it.kb_lo + 1;
          if (resident && it.unit != prev_unit) {
            if (prev_unit >= 0)
              for (int s = 0; s < p.nkb; ++s) mma_commit(&sm.kv_empty[s]);
            ++unit_loads;
            prev_unit = it.unit;
            for (int s = 0; s < p.nkb && ok; ++s)
              ok = wait_bar(&sm.k_full[s], (unit_loads - 1) & 1u, ctl, status, 11);
            for (int s = 0; s < p.nkb && ok; ++s)
              ok = wait_bar(&sm.v_full[s], (unit_loads - 1) & 1u, ctl, status, 11);
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
                ok = wait_bar(&sm.k_full[ks.stage], ks.parity, ctl, status, 12) &&
                     wait_bar(&sm.v_full[ks.stage], ks.parity, ctl, status, 12);
                if (ok) mma_commit(&sm.kv_empty[ks.stage]);
              }
            sbase += nb;
            continue;
          }
          if (!wait_bar(&sm.q_full[x], qn & 1u, ctl, status, 14)) break;
          ++qn;
          auto issue_s = [&](int bi) -> bool {
            const KvSlot ks = slot(bi);
            if (!wait_bar(&sm.k_full[ks.stage], ks.parity, ctl, status, 15)) return false;
            if (!wait_bar(&sm.v_full[ks.stage], ks.parity, ctl, status, 15)) return false;
            tc_fence_after();
            const int n = round16(block_ncols(it, it.kb_lo + bi));
            const uint32_t idesc = idesc_bf16(128, n, 0, 0);
            const uint64_t aq = sdesc_sw128(smem_u32(sQ[x]), 16, 1024);
            const uint64_t ado = sdesc_sw128(smem_u32(sdO[x]), 16, 1024);
            const uint64_t bk = sdesc_sw128(smem_u32(sK + ks.stage * kKVTile), 16, 1024);
            const uint64_t bv = sdesc_sw128(smem_u32(sV + ks.stage * kKVTile), 16, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss(tS, aq + 2 * k, bk + 2 * k, idesc, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss(tP, ado + 2 * k, bv + 2 * k, idesc, k > 0);
            mma_commit(&sm.s_full[x]);
            ++js;
            if (bi == nb - 1) mma_commit(&sm.q_empty[x]);
            return true;
          };
          ok = issue_s(0);
          for (int bi = 0; bi < nb && ok; ++bi) {
            if (!wait_bar(&sm.ds_full[x], jd & 1u, ctl, status, 16)) { ok = false; break; }
            ++jd;
            tc_fence_after();
            const KvSlot ks = slot(bi);
            if (!kDelta) {
              const int ksteps = round16(block_ncols(it, it.kb_lo + bi)) >> 4;
              const uint64_t bk = sdesc_sw128(smem_u32(sK + ks.stage * kKVTile), 1024, 1024);
              for (int k = 0; k < ksteps; ++k) {
                mma_ts(tQ, tS + 8 * k, bk + (2048 >> 4) * k, idesc_dq, (bi > 0 || k > 0));
                mma_ts(tQ, tP + 8 * k, bk + (2048 >> 4) * k, idesc_dq, 1);
              }
            }
            if (!resident) mma_commit(&sm.kv_empty[ks.stage]);
            if (bi == nb - 1) {
              if (!kDelta) mma_commit(&sm.dq_done[x]);
            } else {
              ok = issue_s(bi + 1);
            }
          }
          sbase += nb;
        }
        mma_commit(&sm.drain[x]);
        drain_wait(&sm.drain[x], 0);
      }
    }
  } else {
    regs_inc<kFwdSoftmaxRegs>();
    // ------------------------------------------------------------ dS warpgroups
    const int x = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 256u * x + lane_off, tP = tS + 96u, tQ = tS + 192u;
    const int G = p.G;
    const int tok = r / G;
    const int g = r - tok * G;
    const float lg2e = 1.4426950408889634f;
    uint32_t jS = 0, jD = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; ++i) {
      const FwdItem it = fwd_decode(p, i);
      if (x == 1 && !it.validB) continue;
      const int nb = it.kb_hi - it.kb_lo + 1;
      const int mytok0 = x ? it.tok0[1] : it.tok0[0];
      const int pos = mytok0 + tok;
      const bool row_ok = (r < p.rows) && (pos < p.L);
      long long row = 0;
      float lse2 = INFINITY, dlt = 0.f;
      float dacc[4] = {0.f, 0.f, 0.f, 0.f};
      if (row_ok) {
        const long long t_idx = p.is_time ? pos : it.fixed;
        const long long s_idx = p.is_time ? it.fixed : pos;
        row = ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + it.kvh * G + g;
        lse2 = dp.lse[row] * lg2e;
        if (!kDelta) dlt = dp.delta[row];
      }
      const float2 sl2 = make_float2(p.sl, p.sl);
      const float2 nl2 = make_float2(-lse2, -lse2);
      for (int bi = 0; bi < nb; ++bi) {
        const int kbase = (it.kb_lo + bi) * kBN;
        const int ncols = block_ncols(it, it.kb_lo + bi);
        const int n32 = (ncols + 31) >> 5;
        int lo, hi, ex;
        if (p.is_time) {
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
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < n32; ++c) {
          float sv[32], pv[32];
          tmem_ld32(tS + 32 * c, sv);
          tmem_ld32(tP + 32 * c, pv);
          tmem_wait_ld_dep32(sv);
          tmem_wait_ld_dep32(pv);
          const uint32_t keep = keep_bits32(32 * c, lo, hi, ex);
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
          uint32_t pk[16], lk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 xx = __ffma2_rn(make_float2(sv[2 * j], sv[2 * j + 1]), sl2, nl2);
            // masked (and stale, beyond the block's N) columns give exactly zero: select,
            // never multiply, since stale TMEM may hold NaN
            const float d0 = ((keep >> (2 * j)) & 1u) ? ex2(xx.x) * (pv[2 * j] - dlt) : 0.f;
            const float d1 = ((keep >> (2 * j + 1)) & 1u) ? ex2(xx.y) * (pv[2 * j + 1] - dlt) : 0.f;
            pk[j] = split_bf16x2(d0, d1, &lk[j]);
          }
          tmem_st16(tS + 16 * c, pk);   // dS high parts over the scores already read
          tmem_st16(tP + 16 * c, lk);   // dS residuals over dP already read
        }
        if (!kDelta) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ds_full[x]);
      }
      if (!ok) break;
      if (kDelta) {
        if (row_ok) dp.delta[row] = (dacc[0] + dacc[1]) + (dacc[2] + dacc[3]);
        continue;
      }
      // ---------------------------------------------------------------- epilogue
      ok = wait_bar(&sm.dq_done[x], jD & 1u, ctl, status, 8);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++jD;
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
          dst[c] = make_float4(o[4 * c] * dp.scale, o[4 * c + 1] * dp.scale, o[4 * c + 2] * dp.scale,
                               o[4 * c + 3] * dp.scale);
      }
      {
        uint8_t* stg = sOst + (warp & 7) * 4096;
        const int wr = lane;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 wv;
          wv.x = pack_bf16x2(o[8 * c + 0] * dp.scale, o[8 * c + 1] * dp.scale);
          wv.y = pack_bf16x2(o[8 * c + 2] * dp.scale, o[8 * c + 3] * dp.scale);
          wv.z = pack_bf16x2(o[8 * c + 4] * dp.scale, o[8 * c + 5] * dp.scale);
          wv.w = pack_bf16x2(o[8 * c + 6] * dp.scale, o[8 * c + 7] * dp.scale);
          *reinterpret_cast<uint4*>(stg + wr * 128 + ((c ^ (wr & 7)) << 4)) = wv;
        }
        __syncwarp();
        const int sub = lane >> 3, ch = lane & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + sub;
          const int rt = (warp & 3) * 32 + rr;
          const int tk = rt / G;
          const int gg = rt - tk * G;
          const int ps = mytok0 + tk;
          if (rt < p.rows && ps < p.L) {
            const long long t_idx = p.is_time ? ps : it.fixed;
            const long long s_idx = p.is_time ? it.fixed : ps;
            const long long rw =
                ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + it.kvh * G + gg;
            const uint4 wv = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
            reinterpret_cast<uint4*>(dp.dq + rw * 64)[ch] = wv;
          }
        }
        __syncwarp();
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dK/dV kernel
// A CTA item is (unit, key block of 128 keys).  TMEM: S^T [0,128) (P^T high parts in place),
// dP^T [128,256) (dS^T high parts in place), dK [256,320), dV [320,384), P^T residuals
// [384,448), dS^T residuals [448,512); each accumulating product runs as high + residual.  Keys are TMEM lanes; Q tiles (nTok positions x G heads, as in
// the forward) stream through two shared-memory slots together with dO and, per tile row,
// log2-scaled LSE, Delta and the row's sequence position.
constexpr int kKvBN = 128;
constexpr int kKvThreads = 256;  // warps 0-3 elementwise, 4 producer, 5 MMA, 6-7 idle

struct KvParams {
  FwdParams f;            // shapes (item fields unused)
  const float* lse;
  const float* delta;
  float scale;
  long long nitems;       // units x key blocks
  int nkb;                // 128-key blocks per unit
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dk_f32;
  float* dv_f32;
};

struct KvSmem {
  uint64_t kv_full, kv_free;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, p_full, acc_done;
  uint64_t drain;
  uint32_t tmem_base;
  Ctl ctl;
  alignas(16) float lse2[2][128];   // read as float4: 16-byte aligned
  alignas(16) float delta[2][128];
  alignas(16) int qpos[2][128];
};
static_assert(offsetof(KvSmem, lse2) % 16 == 0 && offsetof(KvSmem, delta) % 16 == 0 &&
                  offsetof(KvSmem, qpos) % 16 == 0,
              "row arrays are read with 16-byte loads");
// smem: [K V][Q0 Q1 dO0 dO1][KvSmem]
constexpr size_t kKvTileBytes = size_t(2) * kTile + size_t(4) * kTile;
constexpr size_t kKvSmemBytes = kKvTileBytes + 1024 + sizeof(KvSmem) + 64;

struct KvItem {
  int b, fixed, kvh, kb;
  int t_lo, t_hi;  // Q tiles [t_lo, t_hi] that can see the key block
};
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
  const int k0 = it.kb * kKvBN;
  const int k1 = min(p.L, k0 + kKvBN) - 1;
  if (p.is_time) {
    it.t_lo = k0 / p.nTok;
    it.t_hi = min(p.L - 1, k1 + p.window - 1) / p.nTok;
  } else {
    it.t_lo = 0;
    it.t_hi = p.ntiles - 1;
  }
  return it;
}

__global__ void __launch_bounds__(kKvThreads, 1)
    od_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const KvParams kp) {
  const FwdParams& p = kp.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = base + kTile;
  uint8_t* sQ[2] = {base + 2 * kTile, base + 3 * kTile};
  uint8_t* sdO[2] = {base + 4 * kTile, base + 5 * kTile};
  KvSmem& sm = *reinterpret_cast<KvSmem*>(base + kKvTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long i0 = (kp.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = (kp.nitems * (blockIdx.x + 1)) / gridDim.x;

  {
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kKvThreads * 16)
      for (int t = 0; t < 2; ++t) {
        *reinterpret_cast<uint4*>(sQ[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sdO[t] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
      }
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_free, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.q_full[x], 1);
      mbar_init(&sm.q_empty[x], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 4);
    mbar_init(&sm.acc_done, 1);
    mbar_init(&sm.drain, 1);
    sm.ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  Ctl* ctl = &sm.ctl;
  unsigned int* status = p.status;
  const float lg2e = 1.4426950408889634f;

  if (warp == 4) {
    // ---------------------------------------------------------- producer (whole warp)
    // lane 0 issues the TMA loads; all lanes stage the tile rows' LSE, Delta and position
    uint32_t nt = 0, ni = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; ++i) {
      const KvItem it = kv_decode(kp, i);
      if (ni > 0) {
        ok = wait_bar(&sm.kv_free, (ni - 1) & 1u, ctl, status, 20);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.kv_full, 2 * kKvBN * 128);
        const int k0 = it.kb * kKvBN;
        if (p.is_time) {
          tma_load_5d(sK, &tm_k, &sm.kv_full, 0, it.kvh, it.fixed, k0, it.b);
          tma_load_5d(sV, &tm_v, &sm.kv_full, 0, it.kvh, it.fixed, k0, it.b);
        } else {
          tma_load_5d(sK, &tm_k, &sm.kv_full, 0, it.kvh, k0, it.fixed, it.b);
          tma_load_5d(sV, &tm_v, &sm.kv_full, 0, it.kvh, k0, it.fixed, it.b);
        }
      }
      ++ni;
      for (int tq = it.t_lo; tq <= it.t_hi && ok; ++tq, ++nt) {
        const int sl = nt & 1;
        if (nt >= 2) {
          ok = wait_bar(&sm.q_empty[sl], ((nt >> 1) - 1) & 1u, ctl, status, 21);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        const int t0 = tq * p.nTok;
        // per tile row: log2-scaled LSE, Delta, sequence position (invalid rows: P = 0)
        for (int rr = lane; rr < 128; rr += 32) {
          const int tk = rr / p.G;
          const int gg = rr - tk * p.G;
          const int ps = t0 + tk;
          float l2 = INFINITY, dl = 0.f;
          int qp = 0x3FFFFFFF;
          if (rr < p.rows && ps < p.L) {
            const long long t_idx = p.is_time ? ps : it.fixed;
            const long long s_idx = p.is_time ? it.fixed : ps;
            const long long row =
                ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + it.kvh * p.G + gg;
            l2 = kp.lse[row] * lg2e;
            dl = kp.delta[row];
            qp = ps;
          }
          sm.lse2[sl][rr] = l2;
          sm.delta[sl][rr] = dl;
          sm.qpos[sl][rr] = qp;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.q_full[sl], 2 * p.rows * 128);
          if (p.is_time) {
            tma_load_5d(sQ[sl], &tm_q, &sm.q_full[sl], 0, it.kvh * p.G, it.fixed, t0, it.b);
            tma_load_5d(sdO[sl], &tm_do, &sm.q_full[sl], 0, it.kvh * p.G, it.fixed, t0, it.b);
          } else {
            tma_load_5d(sQ[sl], &tm_q, &sm.q_full[sl], 0, it.kvh * p.G, t0, it.fixed, it.b);
            tma_load_5d(sdO[sl], &tm_do, &sm.q_full[sl], 0, it.kvh * p.G, t0, it.fixed, it.b);
          }
        }
      }
    }
    if (lane == 0) {
      if (ni > 0) drain_wait(&sm.kv_full, (ni - 1) & 1u);
      for (int sl = 0; sl < 2; ++sl) {
        const uint32_t uses = nt / 2 + (static_cast<uint32_t>(sl) < (nt & 1u) ? 1u : 0u);
        if (uses > 0) drain_wait(&sm.q_full[sl], (uses - 1) & 1u);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t tST = tmem, tDP = tmem + 128, tDK = tmem + 256, tDV = tmem + 320;
      const uint32_t tPL = tmem + 384, tDL = tmem + 448;
      const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);   // M keys, N tile rows
      const uint32_t idesc_acc = idesc_bf16(128, 64, 0, 1);  // M keys, N head dim, B MN-major
      uint32_t nt = 0, ni = 0, jp = 0;
      bool ok = true;
      for (long long i = i0; i < i1 && ok; ++i) {
        const KvItem it = kv_decode(kp, i);
        if (!wait_bar(&sm.kv_full, ni & 1u, ctl, status, 22)) break;
        ++ni;
        const int ntl = it.t_hi - it.t_lo + 1;
        for (int k = 0; k < ntl && ok; ++k, ++nt) {
          const int sl = nt & 1;
          if (!wait_bar(&sm.q_full[sl], (nt >> 1) & 1u, ctl, status, 23)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ak = sdesc_sw128(smem_u32(sK), 16, 1024);
          const uint64_t av = sdesc_sw128(smem_u32(sV), 16, 1024);
          const uint64_t bq = sdesc_sw128(smem_u32(sQ[sl]), 16, 1024);
          const uint64_t bdo = sdesc_sw128(smem_u32(sdO[sl]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_ss(tST, ak + 2 * kk, bq + 2 * kk, idesc_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_ss(tDP, av + 2 * kk, bdo + 2 * kk, idesc_s, kk > 0);
          mma_commit(&sm.s_full);
          if (!wait_bar(&sm.p_full, jp & 1u, ctl, status, 24)) { ok = false; break; }
          ++jp;
          tc_fence_after();
          // dV += P^T dO and dK += dS^T Q (A from TMEM, B MN-major in shared memory)
          const uint64_t bdo_mn = sdesc_sw128(smem_u32(sdO[sl]), 1024, 1024);
          const uint64_t bq_mn = sdesc_sw128(smem_u32(sQ[sl]), 1024, 1024);
          for (int kk = 0; kk < 8; ++kk) {
            mma_ts(tDV, tST + 8 * kk, bdo_mn + (2048 >> 4) * kk, idesc_acc, (k > 0 || kk > 0));
            mma_ts(tDV, tPL + 8 * kk, bdo_mn + (2048 >> 4) * kk, idesc_acc, 1);
            mma_ts(tDK, tDP + 8 * kk, bq_mn + (2048 >> 4) * kk, idesc_acc, (k > 0 || kk > 0));
            mma_ts(tDK, tDL + 8 * kk, bq_mn + (2048 >> 4) * kk, idesc_acc, 1);
          }
          mma_commit(&sm.q_empty[sl]);
        }
        if (!ok) break;
        mma_commit(&sm.acc_done);
        mma_commit(&sm.kv_free);
      }
      mma_commit(&sm.drain);
      drain_wait(&sm.drain, 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- elementwise (key lanes)
    const int j = tid;  // key lane within the block
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tST = tmem + lane_off, tDP = tmem + 128 + lane_off;
    const uint32_t tDK = tmem + 256 + lane_off, tDV = tmem + 320 + lane_off;
    const uint32_t tPL = tmem + 384 + lane_off, tDL = tmem + 448 + lane_off;
    uint32_t nt = 0, js = 0, na = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; ++i) {
      const KvItem it = kv_decode(kp, i);
      const int kpos = it.kb * kKvBN + j;
      const bool key_ok = kpos < p.L;
      const bool is_agent = !p.is_time && kpos == p.agent;
      const int ntl = it.t_hi - it.t_lo + 1;
      for (int k = 0; k < ntl && ok; ++k, ++nt) {
        const int sl = nt & 1;
        // the tile rows' LSE/Delta/positions were staged by the producer before it armed
        // q_full for this slot: acquire them from that barrier directly
        ok = wait_bar(&sm.q_full[sl], (nt >> 1) & 1u, ctl, status, 27);
        ok = ok && wait_bar(&sm.s_full, js & 1u, ctl, status, 25);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++js;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float sv[32], pv[32];
          tmem_ld32(tST + 32 * c, sv);
          tmem_ld32(tDP + 32 * c, pv);
          tmem_wait_ld_dep32(sv);
          tmem_wait_ld_dep32(pv);
          uint32_t pk[16], dk[16], pl[16], dl[16];
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            const int col = 32 * c + q;
            const float4 l4 = *reinterpret_cast<const float4*>(&sm.lse2[sl][col & ~3]);
            const float4 d4 = *reinterpret_cast<const float4*>(&sm.delta[sl][col & ~3]);
            const int4 q4 = *reinterpret_cast<const int4*>(&sm.qpos[sl][col & ~3]);
            const int o = col & 3;  // 0 or 2
            const float la = o ? l4.z : l4.x, lb = o ? l4.w : l4.y;
            const float da = o ? d4.z : d4.x, db = o ? d4.w : d4.y;
            const int qa = o ? q4.z : q4.x, qb = o ? q4.w : q4.y;
            float p0 = ex2(fmaf(sv[q], p.sl, -la));
            float p1 = ex2(fmaf(sv[q + 1], p.sl, -lb));
            bool ka, kb2;
            if (p.is_time) {
              ka = qa >= kpos && qa - kpos < p.window;
              kb2 = qb >= kpos && qb - kpos < p.window;
            } else {
              ka = !is_agent || qa == p.agent;
              kb2 = !is_agent || qb == p.agent;
            }
            p0 = ka ? p0 : 0.f;
            p1 = kb2 ? p1 : 0.f;
            pk[q >> 1] = split_bf16x2(p0, p1, &pl[q >> 1]);
            dk[q >> 1] = split_bf16x2(p0 * (pv[q] - da), p1 * (pv[q + 1] - db), &dl[q >> 1]);
          }
          tmem_st16(tST + 16 * c, pk);
          tmem_st16(tDP + 16 * c, dk);
          tmem_st16(tPL + 16 * c, pl);
          tmem_st16(tDL + 16 * c, dl);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full);
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue: dK, dV rows
      ok = wait_bar(&sm.acc_done, na & 1u, ctl, status, 26);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++na;
      tc_fence_after();
      float gk[64], gv[64];
      tmem_ld32(tDK, gk);
      tmem_ld32(tDK + 32, gk + 32);
      tmem_ld32(tDV, gv);
      tmem_ld32(tDV + 32, gv + 32);
      tmem_wait_ld_dep32(gk);
      tmem_wait_ld_dep32(gk + 32);
      tmem_wait_ld_dep32(gv);
      tmem_wait_ld_dep32(gv + 32);
      if (key_ok) {
        const long long t_idx = p.is_time ? kpos : it.fixed;
        const long long s_idx = p.is_time ? it.fixed : kpos;
        const long long row = ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hkv + it.kvh;
        uint4* dk_out = reinterpret_cast<uint4*>(kp.dk + row * 64);
        uint4* dv_out = reinterpret_cast<uint4*>(kp.dv + row * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 a, b;
          a.x = pack_bf16x2(gk[8 * c + 0] * kp.scale, gk[8 * c + 1] * kp.scale);
          a.y = pack_bf16x2(gk[8 * c + 2] * kp.scale, gk[8 * c + 3] * kp.scale);
          a.z = pack_bf16x2(gk[8 * c + 4] * kp.scale, gk[8 * c + 5] * kp.scale);
          a.w = pack_bf16x2(gk[8 * c + 6] * kp.scale, gk[8 * c + 7] * kp.scale);
          b.x = pack_bf16x2(gv[8 * c + 0], gv[8 * c + 1]);
          b.y = pack_bf16x2(gv[8 * c + 2], gv[8 * c + 3]);
          b.z = pack_bf16x2(gv[8 * c + 4], gv[8 * c + 5]);
          b.w = pack_bf16x2(gv[8 * c + 6], gv[8 * c + 7]);
          dk_out[c] = a;
          dv_out[c] = b;
        }
        if (kp.dk_f32) {
          float4* a = reinterpret_cast<float4*>(kp.dk_f32 + row * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            a[c] = make_float4(gk[4 * c] * kp.scale, gk[4 * c + 1] * kp.scale, gk[4 * c + 2] * kp.scale,
                               gk[4 * c + 3] * kp.scale);
        }
        if (kp.dv_f32) {
          float4* b = reinterpret_cast<float4*>(kp.dv_f32 + row * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c) b[c] = make_float4(gv[4 * c], gv[4 * c + 1], gv[4 * c + 2], gv[4 * c + 3]);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ host side
inline cudaError_t bwd_setup() {
  cudaError_t e = cudaFuncSetAttribute(od_bwd_dq_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDqSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(od_bwd_dq_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kDqSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(od_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kKvSmemBytes));
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, od_bwd_dq_kernel<false>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kFwdLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncGetAttributes(&fa, od_bwd_dq_kernel<true>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kFwdLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

// workspace: Delta (fp32, one per query row)
inline size_t bwd_workspace_bytes(int B, int T, int S, int Hq, int /*D*/) {
  return (size_t(B) * T * S * Hq * sizeof(float) + 255) & ~size_t(255);
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
