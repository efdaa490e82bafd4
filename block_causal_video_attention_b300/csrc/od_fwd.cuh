// od_fwd.cuh -- forward kernel shared by space and time attention (sm_103a).
//
// Both operators are "masked attention over the sequence of one unit":
//   space: unit = (b, t, kv head), sequence = the S tokens of that timestep block,
//          mask = the agent-token read restriction (world-model tokens cannot read the
//          agent token; 7minutos.es page, "Arquitectura: una columna vertebral, dos modelos");
//   time:  unit = (b, s, kv head), sequence = the T timesteps at token position s,
//          mask = causal with a sliding window of W steps (edgex es-LA page,
//          "Configuracion de entrenamiento": a 192-step window).
// All G = Hq/Hkv query heads of a KV head are packed into one Q tile ("grouped-query
// attention"): a tile holds nTok = floor(128/G) consecutive sequence positions x G heads,
// which in the [B,T,S,H,D] layout is one 5-D TMA box (64, G, nTok) -- rows r = tok*G + g.
// K/V of a unit are loaded once per CTA visit and reused by all G heads and all Q tiles.
//
// One persistent CTA per SM walks a contiguous range of work items (every gridDim.x-th item
// for variable-length blocks); an item is (unit, pair of Q tiles A and B).  Keys come in blocks of 64.  Every score row is split
// between two threads: one takes columns 0-31 of each block ("half a"), the other columns
// 32-63 ("half b").  Each half keeps its own running maximum, its own row sum and its own
// output accumulator (O_a, O_b in TMEM), so the halves never synchronise per block; at the
// end of an item they exchange (max, sum) once through shared memory and combine
//   O = (O_a 2^(m_a - M) + O_b 2^(m_b - M)) / (l_a 2^(m_a - M) + l_b 2^(m_b - M)),
//   M = max(m_a, m_b).
// Warp roles (640 threads, five warpgroups):
//   warps 0-3 tile A half a, 4-7 tile A half b, 8-11 tile B half a, 12-15 tile B half b
//        (thread i of a warpgroup owns TMEM lane / row i)
//   warp 16  TMA producer (one thread)
//   warps 17, 18  TMEM allocator (17) and tcgen05.mma issuers for tiles A and B (whole warp,
//        one elected lane issues)
//   warp 19  converts each V tile to fp16 in shared memory (P V runs in fp16)
// The kernel launches with kFwdLaunchRegs registers per thread; the softmax warpgroups then
// drop to kFwdSoftmaxRegs and the control warpgroup rises to kFwdCtrlRegs.  The shares add
// up to the launch allocation, and the host refuses to launch if the compiled register count
// differs from kFwdLaunchRegs.
//
// TMEM (512 columns), per tile x at 256x: two 64-column score buffers [0,64) and [64,128)
// (block j of the tile goes to buffer j mod 2), O_a [128,192), O_b [192,256).  Each half
// writes its P (fp16 pairs, 16 columns) in place at the start of its own 32 columns; P V
// reads it from TMEM.  A tile's Q K^T number j is issued once both halves have taken scores
// j-1 and P V j-2 has been issued (tcgen05 MMAs of one thread run in issue order), so each
// tile has its next scores computed while its softmax works; the softmax never waits for a
// P V except to rescale O and at the end of an item.  Every mbarrier is waited on at
// most one phase ahead of or behind its completions (a parity wait cannot tell more apart).
// The key range of an item is the union of its rows' allowed ranges, so key blocks that are
// fully masked for the whole item are never loaded; partial blocks are masked per element.
// Online softmax with a lazy rescale: a half's running maximum only moves when a block's
// maximum exceeds it by more than 8 (log2 units); that half's O is then rescaled in TMEM.
// Statistics are fp32; LSE (natural log) is written from registers; O (and, on request, its
// rounding residual) leaves by TMA store of the tile halves staged in shared memory, or by
// per-thread stores for variable-length blocks, whose padding rows must stay untouched.
#pragma once
#include "od_common.cuh"

namespace od {

constexpr int kFwdBN = 64;                    // keys per key block
constexpr int kFwdStages = 5;                 // K/V shared-memory stages
constexpr int kFwdKVTile = kFwdBN * 128;      // bytes of one K or V stage
constexpr int kFwdThreads = 640;
constexpr int kFwdLaunchRegs = 96;
constexpr int kFwdSoftmaxRegs = 88;
constexpr int kFwdCtrlRegs = 128;
static_assert(512 * kFwdSoftmaxRegs + 128 * kFwdCtrlRegs == kFwdThreads * kFwdLaunchRegs,
              "register split must add up to the launch allocation");
constexpr int kFwdProducerWarp = 16;
constexpr int kFwdMmaWarp = 17;               // 17: tile A, 18: tile B
constexpr int kFwdConvWarp = 19;

struct FwdSmem {
  uint64_t q_full[2][2], q_empty[2][2];  // per tile, two Q slots (next item's tile prefetched)
  uint64_t k_full[kFwdStages], v_full[kFwdStages], v16_ready[kFwdStages], kv_empty[kFwdStages];
  // per tile: scores ready, scores taken by both halves, P ready, (m, l) posted; P V of
  // even / odd blocks complete (two barriers, so that a softmax that waits only when it
  // needs to -- to rescale O, and at the end of an item -- never has two phases of one
  // barrier outstanding: receiving scores j implies P V j-2 has completed)
  uint64_t s_full[2], s_taken[2], p_full[2], ml_ready[2];
  uint64_t o_done[2][2];
  // per tile and half (4 warps): output rows staged for the TMA stores; staging free again
  // (the previous stores have read it)
  uint64_t st_full[2][2], st_free[2][2];
  uint64_t drain[2];
  uint32_t tmem_base;
  Ctl ctl;
  uint8_t vfmt[kFwdStages][2];  // per 32-key half of a V stage: 0 = fp16, 1 = bf16
  uint16_t rowtg[128];          // tile row r -> (r / G) << 8 | (r % G)
  float2 ml[2][2][128];         // per tile, half, row: (running max, row sum)
};
// dynamic smem: [Q: tile A slots 0 1, tile B slots 0 1][K stages][V stages]
//               [O staging, 2 KB per softmax warp][O residual staging, likewise][FwdSmem]
constexpr size_t kFwdStageBytes = 2 * 16 * 2048;
constexpr size_t kFwdTileBytes =
    size_t(4) * kTile + size_t(2 * kFwdStages) * kFwdKVTile + kFwdStageBytes;
constexpr size_t kFwdSmemBytes = kFwdTileBytes + 1024 + sizeof(FwdSmem) + 64;
static_assert(kFwdSmemBytes <= 227 * 1024, "shared memory budget");

// One pending P V product of an MMA issuer.
struct PvJob {
  uint8_t stage, vpar, ksteps, acc_a, acc_b;
};

template <bool kVarlen>
__global__ void __launch_bounds__(kFwdThreads, 1)
    od_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_lo, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base;  // tile x, slot s at (2x + s) * kTile
  uint8_t* sK = base + 4 * kTile;
  uint8_t* sV = sK + kFwdStages * kFwdKVTile;
  uint8_t* sOst = sV + kFwdStages * kFwdKVTile;
  uint8_t* sLst = sOst + 16 * 2048;
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base + kFwdTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // items of this CTA: a contiguous range (consecutive items of a unit share its K/V); for
  // variable-length blocks every gridDim.x-th item, so that items of unequal cost spread
  // over all CTAs
  const bool strided = kVarlen;
  const long long istep = strided ? gridDim.x : 1;
  const long long i0 = strided ? blockIdx.x : (p.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = strided ? p.nitems : (p.nitems * (blockIdx.x + 1)) / gridDim.x;
  OD_TRACE_INIT();

  // zero the Q-tile rows that TMA never writes (rows >= p.rows)
  {
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kFwdThreads * 16)
      for (int t = 0; t < 4; ++t)
        *reinterpret_cast<uint4*>(sQ + t * kTile + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      for (int q = 0; q < 2; ++q) {
        mbar_init(&sm.q_full[x][q], 1);
        mbar_init(&sm.q_empty[x][q], 1);
      }
      mbar_init(&sm.o_done[x][0], 1);
      mbar_init(&sm.o_done[x][1], 1);
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.s_taken[x], 8);
      mbar_init(&sm.p_full[x], 8);
      mbar_init(&sm.ml_ready[x], 8);
      mbar_init(&sm.drain[x], 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(&sm.st_full[x][h], 4);
        mbar_init(&sm.st_free[x][h], 1);
      }
    }
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v16_ready[s], 1);
      mbar_init(&sm.kv_empty[s], 2);
    }
    sm.ctl.abort = 0;
    fence_mbar_init();
  }
  if (tid < 128) sm.rowtg[tid] = static_cast<uint16_t>(((tid / p.G) << 8) | (tid % p.G));
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

  if (warp >= 16) {
    regs_inc<kFwdCtrlRegs>();
    if (warp == kFwdProducerWarp) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        long long prev_unit = -1;
        uint32_t unit_loads = 0, stream_cnt = 0, qn0 = 0, qn1 = 0;
        bool ok = true;
        for (long long i = i0; i < i1 && ok; i += istep) {
          const FwdItem it = fwd_decode<kVarlen>(p, i);
          if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
          auto load_kv = [&](int stage, int kb) {
            const int kp = kb * kFwdBN;
            mbar_arrive_expect_tx(&sm.k_full[stage], kFwdKVTile);
            mbar_arrive_expect_tx(&sm.v_full[stage], kFwdKVTile);
            uint8_t* dk = sK + stage * kFwdKVTile;
            uint8_t* dv = sV + stage * kFwdKVTile;
            if (p.is_time) {
              tma_load_5d(dk, &tm_k, &sm.k_full[stage], 0, it.kvh, it.fixed, kp, it.b);
              tma_load_5d(dv, &tm_v, &sm.v_full[stage], 0, it.kvh, it.fixed, kp, it.b);
            } else {
              tma_load_5d(dk, &tm_k, &sm.k_full[stage], 0, it.kvh, kp, it.fixed, it.b);
              tma_load_5d(dv, &tm_v, &sm.v_full[stage], 0, it.kvh, kp, it.fixed, it.b);
            }
          };
          auto load_q = [&](int x, uint32_t& n) -> bool {
            const int q = n & 1;
            if (n >= 2 && !wait_bar(&sm.q_empty[x][q], ((n >> 1) - 1) & 1u, ctl, status, 1)) return false;
            uint8_t* dst = sQ + (2 * x + q) * kTile;
            mbar_arrive_expect_tx(&sm.q_full[x][q], p.rows * 128);
            if (p.is_time)
              tma_load_5d(dst, &tm_q, &sm.q_full[x][q], 0, it.kvh * p.G, it.fixed, it.tok0[x], it.b);
            else
              tma_load_5d(dst, &tm_q, &sm.q_full[x][q], 0, it.kvh * p.G, it.tok0[x], it.fixed, it.b);
            ++n;
            return true;
          };
          OD_TP(1, (int)i, 0);
          ok = load_q(0, qn0);
          if (ok && it.validB) ok = load_q(1, qn1);
          if (!ok) break;
          if (p.resident) {
            if (it.unit != prev_unit) {
              if (unit_loads > 0) {
                for (int s = 0; s < p.nkb && ok; ++s)
                  ok = wait_bar(&sm.kv_empty[s], (unit_loads - 1) & 1u, ctl, status, 2);
              }
              if (!ok) break;
              for (int kb = 0; kb < p.nkb; ++kb) load_kv(kb, kb);
              ++unit_loads;
              prev_unit = it.unit;
            }
          } else {
            const int nb = it.kb_hi - it.kb_lo + 1;
            for (int bi = 0; bi < nb && ok; ++bi) {
              const uint32_t c = stream_cnt + bi;
              const int stage = static_cast<int>(c % kFwdStages);
              const uint32_t n = c / kFwdStages;
              if (n > 0) ok = wait_bar(&sm.kv_empty[stage], (n - 1) & 1u, ctl, status, 3);
              if (ok) load_kv(stage, it.kb_lo + bi);
            }
            stream_cnt += nb;
          }
        }
        // make sure no TMA load is still writing into this CTA's smem when it exits
        for (int x = 0; x < 2; ++x)
          for (int q = 0; q < 2; ++q) {
            const uint32_t n = x ? qn1 : qn0;
            const uint32_t uses = n / 2 + (static_cast<uint32_t>(q) < (n & 1u) ? 1u : 0u);
            if (uses > 0) drain_wait(&sm.q_full[x][q], (uses - 1) & 1u);
          }
        if (p.resident) {
          if (unit_loads > 0)
            for (int s = 0; s < p.nkb; ++s) {
              drain_wait(&sm.k_full[s], (unit_loads - 1) & 1u);
              drain_wait(&sm.v_full[s], (unit_loads - 1) & 1u);
            }
        } else {
          for (int s = 0; s < kFwdStages; ++s) {
            const uint32_t uses =
                stream_cnt / kFwdStages + (static_cast<uint32_t>(s) < stream_cnt % kFwdStages ? 1u : 0u);
            if (uses > 0) {
              drain_wait(&sm.k_full[s], (uses - 1) & 1u);
              drain_wait(&sm.v_full[s], (uses - 1) & 1u);
            }
          }
        }
      }
    } else if (warp == kFwdMmaWarp || warp == kFwdMmaWarp + 1) {
      // ---------------------------------------------------------- MMA issuers
      // Warp 17 issues tile A's MMAs, warp 18 tile B's, each in order: Q K^T(0); then for
      // every block j: wait until both halves have taken scores j, issue Q K^T(j+1) into the
      // tile's other score buffer; wait for P(j), issue P V(j) as O_a += P_a V_a (keys 0-31)
      // and O_b += P_b V_b (keys 32-63).  At the end of an item the last P V goes out at
      // once.  Both issuers walk every item (tile B also the items it has no rows in) and
      // release every K/V fill they have seen arrive, so kv_empty counts two.
      {
        const int x = warp - kFwdMmaWarp;  // 0: tile A, 1: tile B
        const uint32_t idesc_pv_bf16 = idesc_bf16(128, 64, 0, 1);
        const uint32_t idesc_pv_fp16 = idesc_fp16(128, 64, 0, 1);
        const uint32_t tOa = tmem + 256u * x + 128u, tOb = tOa + 64u;
        uint32_t js = 0, jp = 0, qn = 0, unit_loads = 0, sbase = 0;
        int qs = 0;  // Q slot of the current item
        long long prev_unit = -1;
        PvJob f0{}, f1{};
        int npend = 0;  // pending P V products; the oldest is slot jp & 1
        bool ok = true;
        auto issue_pv = [&]() -> bool {
          const PvJob jb = (jp & 1u) ? f1 : f0;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.p_full[x], jp & 1u, ctl, status, 9))) return false;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.v16_ready[jb.stage], jb.vpar, ctl, status, 10))) return false;
          tc_fence_after();
          const uint64_t b = sdesc_sw128(smem_u32(sV + jb.stage * kFwdKVTile), 1024, 1024);
          const uint32_t a = tmem + 256u * x + 64u * (jp & 1u);
          const uint32_t ida = sm.vfmt[jb.stage][0] ? idesc_pv_bf16 : idesc_pv_fp16;
          const uint32_t idb = sm.vfmt[jb.stage][1] ? idesc_pv_bf16 : idesc_pv_fp16;
          // O_a takes keys 0-31 of the block; O_b keys 32-63 -- and on an item's first block
          // at least one k-step even when the block is shorter (its P_b is then all zero),
          // so that O_b always holds this item's (finite) sum
          const int ka = jb.ksteps < 2 ? jb.ksteps : 2;
          const int kb = jb.ksteps > 2 ? jb.ksteps - 2 : (jb.acc_b ? 0 : 1);
          for (int k = 0; k < ka; ++k)
            mma_ts_w(tOa, a + 8 * k, b + (2048 >> 4) * k, ida, (jb.acc_a || k > 0));
          for (int k = 0; k < kb; ++k)
            mma_ts_w(tOb, a + 32 + 8 * k, b + (2048 >> 4) * (2 + k), idb, (jb.acc_b || k > 0));
          mma_commit_w(&sm.o_done[x][jp & 1u]);
          OD_TP(12 + x, 0, (int)jp);
          ++jp;
          --npend;
          if (!p.resident) mma_commit_w(&sm.kv_empty[jb.stage]);
          return true;
        };
        for (long long i = i0; i < i1 && ok; i += istep) {
          const FwdItem it = fwd_decode<kVarlen>(p, i);
          if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
          const int nb = it.kb_hi - it.kb_lo + 1;
          if (p.resident && it.unit != prev_unit) {
            if (prev_unit >= 0) {
              while (ok && npend > 0) ok = issue_pv();
              for (int s2 = 0; s2 < p.nkb; ++s2) mma_commit_w(&sm.kv_empty[s2]);
            }
            ++unit_loads;
            prev_unit = it.unit;
            // observe the fill before this issuer can ever release it
            for (int s2 = 0; s2 < p.nkb && ok; ++s2)
              ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[s2], (unit_loads - 1) & 1u, ctl, status, 11));
          }
          if (!ok) break;
          if (x == 1 && !it.validB) {
            if (!p.resident) {
              for (int bi = 0; bi < nb && ok; ++bi) {
                const uint32_t c = sbase + static_cast<uint32_t>(bi);
                const int stage = static_cast<int>(c % kFwdStages);
                ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[stage], (c / kFwdStages) & 1u, ctl, status, 12));
                if (ok) mma_commit_w(&sm.kv_empty[stage]);
              }
            }
            sbase += static_cast<uint32_t>(nb);
            continue;
          }
          for (int bi = 0; bi < nb && ok; ++bi) {
            while (ok && npend >= 2) ok = issue_pv();
            if (!ok) break;
            if (js > 0 && !__all_sync(0xffffffffu, wait_bar(&sm.s_taken[x], (js - 1) & 1u, ctl, status, 13))) { ok = false; break; }
            if (bi == 0) {
              qs = qn & 1;
              if (!__all_sync(0xffffffffu, wait_bar(&sm.q_full[x][qs], (qn >> 1) & 1u, ctl, status, 14))) { ok = false; break; }
              ++qn;
            }
            const KvSlot ks = kv_slot(p, it, bi, unit_loads, sbase, kFwdStages);
            if (!__all_sync(0xffffffffu, wait_bar(&sm.k_full[ks.stage], ks.parity, ctl, status, 15))) { ok = false; break; }
            tc_fence_after();
            const int n = round16(block_ncols(it, it.kb_lo + bi, kFwdBN));
            const uint32_t idesc = idesc_bf16(128, n, 0, 0);
            const uint64_t a = sdesc_sw128(smem_u32(sQ + (2 * x + qs) * kTile), 16, 1024);
            const uint64_t b = sdesc_sw128(smem_u32(sK + ks.stage * kFwdKVTile), 16, 1024);
            const uint32_t d = tmem + 256u * x + 64u * (js & 1u);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss_w(d, a + 2 * k, b + 2 * k, idesc, k > 0);
            mma_commit_w(&sm.s_full[x]);
            OD_TP(10 + x, (int)i, bi);
            PvJob jb;
            jb.stage = static_cast<uint8_t>(ks.stage);
            jb.vpar = static_cast<uint8_t>(ks.parity);
            jb.ksteps = static_cast<uint8_t>(n >> 4);
            jb.acc_a = bi > 0;
            jb.acc_b = bi > 0;
            if (js & 1u) f1 = jb; else f0 = jb;
            ++js;
            ++npend;
            if (bi == nb - 1) mma_commit_w(&sm.q_empty[x][qs]);
            while (ok && npend >= 2) ok = issue_pv();
          }
          // the item's last P V goes out as soon as its P is ready
          while (ok && npend > 0) ok = issue_pv();
          sbase += static_cast<uint32_t>(nb);
        }
        // wait until every MMA issued by this warp has completed before TMEM is freed
        mma_commit_w(&sm.drain[x]);
        drain_wait(&sm.drain[x], 0);
      }
    } else {
      // ---------------------------------------------------------- V converter (warp 19)
      // P V runs in fp16: P in [0, 256] loses 8x less to rounding than in bf16.  Each fill
      // of a V stage is converted in place, per 32-key half, when the half's magnitude is
      // inside a safe fp16 range (2^-10 <= max|v| <= 2^15, or all zero); otherwise the half
      // stays bf16 and the softmax and MMA use bf16 for those keys.
      long long prev_unit = -1;
      uint32_t unit_loads = 0, stream_cnt = 0;
      bool ok = true;
      auto convert = [&](int stage, uint32_t parity) -> bool {
        bool w = wait_bar(&sm.v_full[stage], parity, ctl, status, 4);
        if (!__all_sync(0xffffffffu, w)) return false;
#pragma unroll 1
        for (int cc = 0; cc < kFwdBN / 32; ++cc) {
          uint4* chunk = reinterpret_cast<uint4*>(sV + stage * kFwdKVTile + cc * 32 * 128);
          float mx = 0.f;
#pragma unroll 2
          for (int jj = 0; jj < 8; ++jj) {
            const uint4 d = chunk[lane + 32 * jj];
            const uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              mx = fmaxf(mx, fabsf(__uint_as_float(wv[h] << 16)));
              mx = fmaxf(mx, fabsf(__uint_as_float(wv[h] & 0xFFFF0000u)));
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const bool fp16_ok = (mx == 0.f) || (mx >= 0.0009765625f && mx <= 32768.f);
          if (fp16_ok) {
#pragma unroll 2
            for (int jj = 0; jj < 8; ++jj) {
              const uint4 d = chunk[lane + 32 * jj];
              uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
              for (int h = 0; h < 4; ++h)
                wv[h] = pack_f16x2(__uint_as_float(wv[h] << 16), __uint_as_float(wv[h] & 0xFFFF0000u));
              chunk[lane + 32 * jj] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
          if (lane == 0) sm.vfmt[stage][cc] = fp16_ok ? 0 : 1;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.v16_ready[stage]);
        return true;
      };
      for (long long i = i0; i < i1 && ok; i += istep) {
        const FwdItem it = fwd_decode<kVarlen>(p, i);
        if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
        if (p.resident) {
          if (it.unit != prev_unit) {
            ++unit_loads;
            prev_unit = it.unit;
            for (int st = 0; st < p.nkb && ok; ++st) ok = convert(st, (unit_loads - 1) & 1u);
          }
        } else {
          const int nb = it.kb_hi - it.kb_lo + 1;
          for (int bi = 0; bi < nb && ok; ++bi) {
            const uint32_t c = stream_cnt + bi;
            ok = convert(static_cast<int>(c % kFwdStages), (c / kFwdStages) & 1u);
          }
          stream_cnt += nb;
        }
      }
    }
  } else {
    regs_dec<kFwdSoftmaxRegs>();
    // ------------------------------------------------------------ softmax warpgroups
    const int x = warp >> 3;         // 0: tile A, 1: tile B
    const int hf = (warp >> 2) & 1;  // 0: columns 0-31 of each block, 1: columns 32-63
    const int r = (warp & 3) * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tX = tmem + 256u * x + lane_off;
    const uint32_t tO = tX + 128u + 64u * hf;  // this half's accumulator
    const int G = p.G;
    const int tok = r / G;
    const int g = r - tok * G;
    uint32_t jS = 0, jP = 0, jM = 0, jE = 0;
    long long prev_unit = -1;
    uint32_t unit_loads = 0, stream_next = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; i += istep) {
      const FwdItem it = fwd_decode<kVarlen>(p, i);
      if (kVarlen && !it.validA) continue;  // past the unit's length: no role touches it
      if (p.resident && it.unit != prev_unit) {
        ++unit_loads;
        prev_unit = it.unit;
      }
      const int nb = it.kb_hi - it.kb_lo + 1;
      const uint32_t stream_cnt = stream_next;
      stream_next += nb;
      if (x == 1 && !it.validB) continue;
      const int mytok0 = x ? it.tok0[1] : it.tok0[0];
      const int pos = mytok0 + tok;
      const bool row_ok = (r < p.rows) && (pos < (kVarlen ? it.L : p.L));
      float m_used = -INFINITY, l = 0.f;
      for (int bi = 0; bi < nb; ++bi) {
        const int kb = it.kb_lo + bi;
        const int kbase = kb * kFwdBN;
        const int ncols = block_ncols(it, kb, kFwdBN);
        int lo, hi, ex;
        if (p.is_time) {
          lo = pos - p.window + 1 - kbase;
          hi = min(ncols, pos + 1 - kbase);
          ex = -1;
        } else {
          lo = 0;
          hi = ncols;
          ex = (p.agent >= kbase && p.agent < kbase + kFwdBN && pos != p.agent) ? p.agent - kbase : -1;
        }
        // masking is needed only when this half's 32 columns are not all allowed
        const int c0 = 32 * hf;
        const bool partial = (lo > c0) || (hi < c0 + 32) || (ex >= c0 && ex < c0 + 32);
        OD_TP(20, (int)i, bi);
        ok = __all_sync(0xffffffffu, wait_bar(&sm.s_full[x], jS & 1u, ctl, status, 5));
        if (!ok) break;
        const uint32_t tS = tX + 64u * (jS & 1u) + 32u * hf;
        ++jS;
        if (lane == 0) mbar_arrive(&sm.s_taken[x]);
        tc_fence_after();
        float v[32];
        tmem_ld32(tS, v);
        tmem_wait_ld_dep32(v);
        OD_TP(21, (int)i, bi);
        if (__any_sync(0xffffffffu, partial)) {
          const uint32_t keep = keep_bits32(c0, lo, hi, ex);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = ((keep >> j) & 1u) ? v[j] : -INFINITY;
        }
        // row maximum of the 32 columns: four chains of 3-input max over v[0..31]
        float mx0 = max3(v[0], v[1], v[2]), mx1 = max3(v[3], v[4], v[5]);
        float mx2 = max3(v[6], v[7], v[8]), mx3 = max3(v[9], v[10], v[11]);
#pragma unroll
        for (int jj = 12; jj < 28; jj += 8) {
          mx0 = max3(mx0, v[jj], v[jj + 1]);
          mx1 = max3(mx1, v[jj + 2], v[jj + 3]);
          mx2 = max3(mx2, v[jj + 4], v[jj + 5]);
          mx3 = max3(mx3, v[jj + 6], v[jj + 7]);
        }
        mx0 = max3(mx0, v[28], v[29]);
        mx1 = max3(mx1, v[30], v[31]);
        const float mb = fmaxf(max3(mx0, mx1, mx2), mx3);
        const float mnew = mb * p.sl;
        float alpha = 1.f;
        bool rescale = false;
        if (mb != -INFINITY && (m_used == -INFINITY || mnew > m_used + kRescaleThreshold)) {
          if (m_used != -INFINITY) {
            alpha = ex2(m_used - mnew);
            rescale = true;
          }
          m_used = mnew;
          l *= alpha;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // V of this block must be converted before P's format can be chosen
        const KvSlot ks = kv_slot(p, it, bi, unit_loads, stream_cnt, kFwdStages);
        ok = __all_sync(0xffffffffu, wait_bar(&sm.v16_ready[ks.stage], ks.parity, ctl, status, 6));
        if (!ok) break;
        const float2 sl2 = make_float2(p.sl, p.sl);
        const float2 nm2 = make_float2(-msub, -msub);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
        uint32_t pk[16];
        if (sm.vfmt[ks.stage][hf] == 0) {  // warp-uniform: the format of this half's V keys
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 xx = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]), sl2, nm2);
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            if (j & 1) acc1 = __fadd2_rn(acc1, pp); else acc0 = __fadd2_rn(acc0, pp);
            pk[j] = pack_f16x2(pp.x, pp.y);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 xx = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]), sl2, nm2);
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            if (j & 1) acc1 = __fadd2_rn(acc1, pp); else acc0 = __fadd2_rn(acc0, pp);
            pk[j] = pack_bf16x2(pp.x, pp.y);
          }
        }
        tmem_st16(tS, pk);  // P pairs over the first 16 of this half's 32 score columns
        {
          const float2 a = __fadd2_rn(acc0, acc1);
          l += a.x + a.y;
        }
        OD_TP(26, (int)i, bi);
        // A rescale of O needs the previous block's P V complete (this block's P V is issued
        // only after p_full below).  P(j) itself overwrites scores j, written after P V j-2.
        if (__any_sync(0xffffffffu, rescale && bi > 0)) {
          ok = __all_sync(0xffffffffu, wait_bar(&sm.o_done[x][(jP - 1) & 1u], ((jP - 1) >> 1) & 1u, ctl, status, 7));
          if (!ok) break;
          tc_fence_after();
          const float f = (rescale && bi > 0) ? alpha : 1.f;
#pragma unroll 1
          for (int h = 0; h < 8; ++h) {
            uint32_t u[8];
            tmem_ld8(tO + 8 * h, u);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * f);
            tmem_st8(tO + 8 * h, u);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[x]);
        OD_TP(27, (int)i, bi);
        ++jP;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      OD_TP(30, (int)i, 0);
      ok = __all_sync(0xffffffffu, wait_bar(&sm.o_done[x][(jP - 1) & 1u], ((jP - 1) >> 1) & 1u, ctl, status, 8));
      if (!ok) break;
      tc_fence_after();
      OD_TP(33, (int)i, 0);
      sm.ml[x][hf][r] = make_float2(m_used, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.ml_ready[x]);
      ok = __all_sync(0xffffffffu, wait_bar(&sm.ml_ready[x], jM & 1u, ctl, status, 16));
      if (!ok) break;
      ++jM;
      OD_TP(32, (int)i, 0);
      const float2 other = sm.ml[x][hf ^ 1][r];
      const float M = fmaxf(m_used, other.x);
      const float w_me = (m_used == -INFINITY) ? 0.f : ex2(m_used - M);
      const float w_ot = (other.x == -INFINITY) ? 0.f : ex2(other.x - M);
      const float lsum = l * w_me + other.y * w_ot;
      const float inv = 1.f / lsum;
      // (both accumulators hold this item's finite sums; a half that saw no allowed key
      // has weight 0)
      const float wa = (hf ? w_ot : w_me) * inv, wb = (hf ? w_me : w_ot) * inv;
      if (hf == 0 && row_ok) {
        const int hq = it.kvh * G + g;
        const long long t_idx = p.is_time ? pos : it.fixed;
        const long long s_idx = p.is_time ? it.fixed : pos;
        p.lse[((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + hq] =
            (M + log2f(lsum)) * 0.69314718055994531f;
      }
      const uint32_t tOa = tX + 128u + 32u * hf, tOb = tOa + 64u;
      if (!kVarlen && p.tma_out) {
        // This half's columns [32 hf, 32 hf + 32) of the tile's rows r = tok * G + g leave by
        // TMA store: the 4 warps of the half stage their rows (64 bytes each, 16-byte chunk c
        // of row r at c ^ ((r >> 1) & 3): the 64-byte TMA swizzle) in the half's 8 KB block,
        // bf16(O) and the residual O - bf16(O) side by side, and the half's first warp stores
        // each block as one box once all 4 warps have arrived.  Rows past the sequence fall
        // outside the tensor and are not written.  The staging is reused one item later,
        // after the issuing thread has seen the stores read it.
        if (jE > 0) {
          if ((warp & 3) == 0 && lane == 0) {
            bulk_wait_read0();
            mbar_arrive(&sm.st_free[x][hf]);
          }
          ok = __all_sync(0xffffffffu, wait_bar(&sm.st_free[x][hf], (jE - 1) & 1u, ctl, status, 21));
          if (!ok) break;
        }
        uint8_t* so = sOst + warp * 2048;
        uint8_t* sl = sLst + warp * 2048;
        const int swz = (lane >> 1) & 3;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float oa[16], ob[16];
          tmem_ld16(tOa + 16 * c2, oa);
          tmem_ld16(tOb + 16 * c2, ob);
          tmem_wait_ld_dep16(oa);
          tmem_wait_ld_dep16(ob);
          uint32_t w[8], wl[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 y = __ffma2_rn(make_float2(oa[2 * j], oa[2 * j + 1]), make_float2(wa, wa),
                                        __fmul2_rn(make_float2(ob[2 * j], ob[2 * j + 1]), make_float2(wb, wb)));
            w[j] = split_bf16x2(y.x, y.y, &wl[j]);
          }
          *reinterpret_cast<uint4*>(so + lane * 64 + (((2 * c2) ^ swz) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(so + lane * 64 + (((2 * c2 + 1) ^ swz) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          if (p.o_lo) {
            *reinterpret_cast<uint4*>(sl + lane * 64 + (((2 * c2) ^ swz) << 4)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            *reinterpret_cast<uint4*>(sl + lane * 64 + (((2 * c2 + 1) ^ swz) << 4)) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
          }
        }
        fence_proxy_async_smem();  // the staged rows, visible to the TMA stores
        __syncwarp();
        OD_TP(34, (int)i, 0);
        if (lane == 0) mbar_arrive(&sm.st_full[x][hf]);
        if ((warp & 3) == 0) {
          ok = __all_sync(0xffffffffu, wait_bar(&sm.st_full[x][hf], jE & 1u, ctl, status, 22));
          if (!ok) break;
          if (lane == 0) {
            const int c1 = it.kvh * G;
            const int c2s = p.is_time ? it.fixed : mytok0, c3t = p.is_time ? mytok0 : it.fixed;
            tma_store_5d(&tm_o, sOst + warp * 2048, 32 * hf, c1, c2s, c3t, it.b);
            if (p.o_lo) tma_store_5d(&tm_lo, sLst + warp * 2048, 32 * hf, c1, c2s, c3t, it.b);
            bulk_commit();
          }
          __syncwarp();
        }
        ++jE;
        OD_TP(31, (int)i, 0);
        continue;
      }
      // Generic stores (variable-length blocks, whose padding rows must stay untouched, or when
      // the host chose them): this half writes output columns [32 hf, 32 hf + 32); each warp
      // stages its 32 rows (64 bytes each, 16-byte chunks XOR-swizzled by row) and stores them
      // coalesced.  When requested, the residual O - bf16(O) (rounded to bf16) follows through
      // the same staging buffer; it is kept in registers meanwhile.
      uint8_t* stg = sOst + warp * 2048;
      uint32_t wl[2][8];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        float oa[16], ob[16];
        tmem_ld16(tOa + 16 * c2, oa);
        tmem_ld16(tOb + 16 * c2, ob);
        tmem_wait_ld_dep16(oa);
        tmem_wait_ld_dep16(ob);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 y = __ffma2_rn(make_float2(oa[2 * j], oa[2 * j + 1]), make_float2(wa, wa),
                                      __fmul2_rn(make_float2(ob[2 * j], ob[2 * j + 1]), make_float2(wb, wb)));
          w[j] = split_bf16x2(y.x, y.y, &wl[c2][j]);
        }
        *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * c2) ^ (lane & 3)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * c2 + 1) ^ (lane & 3)) << 4)) =
            make_uint4(w[4], w[5], w[6], w[7]);
      }
      __syncwarp();
      OD_TP(34, (int)i, 0);
      const int nparts = p.o_lo ? 2 : 1;
#pragma unroll 1
      for (int part = 0; part < nparts; ++part) {
        if (part) {
          // the residual into the staging buffer (the O rows have been stored)
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * c2) ^ (lane & 3)) << 4)) =
                make_uint4(wl[c2][0], wl[c2][1], wl[c2][2], wl[c2][3]);
            *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * c2 + 1) ^ (lane & 3)) << 4)) =
                make_uint4(wl[c2][4], wl[c2][5], wl[c2][6], wl[c2][7]);
          }
          __syncwarp();
        }
        __nv_bfloat16* dst = part ? p.o_lo : p.o;
        const int sub = lane >> 2, ch = lane & 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = 8 * k + sub;                // row within the warp
          const int rt = (warp & 3) * 32 + rr;       // row within the tile
          const int tg = sm.rowtg[rt];
          const int gg = tg & 0xFF;
          const int ps = mytok0 + (tg >> 8);
          if (rt < p.rows && ps < (kVarlen ? it.L : p.L)) {
            const long long t_idx = p.is_time ? ps : it.fixed;
            const long long s_idx = p.is_time ? it.fixed : ps;
            const long long row =
                ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + it.kvh * G + gg;
            const uint4 wv = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((ch ^ (rr & 3)) << 4));
            reinterpret_cast<uint4*>(dst + row * 64 + 32 * hf)[ch] = wv;
          }
        }
        __syncwarp();
      }
      OD_TP(31, (int)i, 0);
    }
  }

  // output stores issued by this thread: complete before the CTA's shared memory goes
  if (!kVarlen && p.tma_out && warp < 16 && (warp & 3) == 0 && lane == 0) bulk_wait0();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace od
