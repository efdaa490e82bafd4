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
// One persistent CTA per SM walks a contiguous range of work items; an item is
// (unit, pair of Q tiles A and B).  Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax warpgroup for Q tile A  (thread i owns TMEM lane / row i)
//   warps 4-7   softmax warpgroup for Q tile B
//   warp  8     TMA producer (one thread)
//   warp  9     TMEM allocator + tcgen05.mma issuer for tile A (one thread)
//   warp  10    tcgen05.mma issuer for tile B (one thread)
//   warp  11    converts each V tile to fp16 in shared memory (P V runs in fp16)
// The kernel launches with kFwdLaunchRegs registers per thread; the softmax warpgroups
// then raise their limit to kFwdSoftmaxRegs and the control warpgroup lowers its own to
// kFwdCtrlRegs.  2*128*kFwdSoftmaxRegs + 128*kFwdCtrlRegs equals the launch allocation, and
// the host refuses to launch if the compiled register count differs from kFwdLaunchRegs.
//
// TMEM (512 columns): per tile two 96-column score buffers -- tile A [0,192), tile B
// [192,384); a tile's j-th scores go to its buffer j mod 2 -- and O_A [384,448),
// O_B [448,512).  The softmax writes P (fp16 pairs) in place over the first 48 columns of the
// scores it came from; P V reads it from TMEM.  A tile's Q K^T number j is issued once its
// softmax has taken scores j-1 and P V j-2 has been issued (tcgen05 MMAs of one thread run
// in issue order), so each tile has its next scores computed while it works, independently
// of the other tile.  Every mbarrier is waited on at most one phase ahead of or behind its
// completions (a parity wait cannot tell more apart); the per-tile "taken" barrier bounds
// the lookahead.
// Key blocks are 96 keys; the key range of an item is the union of its rows' allowed
// ranges, so key blocks that are fully masked for the whole item are never loaded;
// partial blocks are masked per element.  Online softmax with a lazy rescale: the running
// maximum used for the exponentials only moves when a block's maximum exceeds it by more
// than 8 (log2 units); O is then rescaled in TMEM.  Statistics are fp32; LSE (natural log)
// and O are written straight from registers.
#pragma once
#include <cuda.h>
#include "od_ptx.cuh"

// Timeline trace points: compiled out unless OD_TRACE is defined (a profiling build that
// supplies od_trace(event, a, b)).
#ifdef OD_TRACE
#define OD_TP(ev, a, b) od_trace((ev), (a), (b))
#define OD_TRACE_INIT() od_trace_init()
#else
#define OD_TP(ev, a, b) ((void)0)
#define OD_TRACE_INIT() ((void)0)
#endif

namespace od {

constexpr int kBM = 128;           // query rows per tile (MMA M)
constexpr int kBN = 96;            // keys per key block (score buffer columns)
constexpr int kStages = 6;         // K/V shared-memory stages
constexpr int kTile = 128 * 128;   // bytes of one Q tile: 128 rows x 64 16-bit elements
constexpr int kKVTile = kBN * 128; // bytes of one K or V stage: 96 rows x 64 elements
constexpr int kFwdThreads = 384;
constexpr int kFwdLaunchRegs = 168;
constexpr int kFwdSoftmaxRegs = 200;
constexpr int kFwdCtrlRegs = 104;
static_assert(2 * 128 * kFwdSoftmaxRegs + 128 * kFwdCtrlRegs == kFwdThreads * kFwdLaunchRegs,
              "register split must add up to the launch allocation");
constexpr int kFwdProducerWarp = 8;
constexpr int kFwdMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
  int B, T, S, Hq, Hkv, G;
  int is_time;
  int L;          // sequence length of a unit (S for space, T for time)
  int F;          // second index of a unit (T for space, S for time)
  int agent;      // space: agent token index or -1
  int window;     // time: window length W >= 1
  float sl;       // scale * log2(e)
  int nTok;       // sequence positions per Q tile
  int rows;       // nTok * G <= 128
  int ntiles;     // Q tiles per unit
  int npairs;     // work items per unit
  long long nitems;
  int nkb;        // key blocks per unit
  int resident;   // nkb <= kStages: the unit's K/V stay in smem across its items
  __nv_bfloat16* o;
  float* lse;
  unsigned int* status;
};

struct FwdSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStages], v_full[kStages], v16_ready[kStages], kv_empty[kStages];
  // per tile: scores ready, scores taken by the softmax, P ready, P V complete
  uint64_t s_full[2], s_taken[2], p_full[2], o_done[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  Ctl ctl;
  uint8_t vfmt[kStages][4];  // per 32-key chunk of a V stage: 0 = fp16, 1 = bf16
};
// dynamic smem: [Q0 Q1][K0..][V0..][O staging, 4 KB per softmax warp][FwdSmem]
constexpr size_t kFwdStageBytes = 8 * 32 * 128;
constexpr size_t kFwdTileBytes =
    size_t(2) * kTile + size_t(2 * kStages) * kKVTile + kFwdStageBytes;
constexpr size_t kFwdSmemBytes = kFwdTileBytes + 1024 + sizeof(FwdSmem) + 64;
static_assert(kFwdSmemBytes <= 227 * 1024, "shared memory budget");

struct FwdItem {
  uint32_t unit;
  int b, fixed, kvh;
  int tok0[2];
  int validB;
  int key_lo, key_hi;  // allowed key positions of the item lie in [key_lo, key_hi)
  int kb_lo, kb_hi;    // inclusive key-block range
};

__device__ __forceinline__ FwdItem fwd_decode(const FwdParams& p, long long i) {
  // the host guarantees nitems < 2^31, so 32-bit unsigned division suffices
  FwdItem it;
  const uint32_t ii = static_cast<uint32_t>(i);
  const uint32_t unit = ii / static_cast<uint32_t>(p.npairs);
  const int pair = static_cast<int>(ii - unit * static_cast<uint32_t>(p.npairs));
  it.unit = unit;
  const uint32_t r = unit / static_cast<uint32_t>(p.Hkv);
  it.kvh = static_cast<int>(unit - r * static_cast<uint32_t>(p.Hkv));
  const uint32_t bq = r / static_cast<uint32_t>(p.F);
  it.fixed = static_cast<int>(r - bq * static_cast<uint32_t>(p.F));
  it.b = static_cast<int>(bq);
  const int tA = 2 * pair;
  it.tok0[0] = tA * p.nTok;
  it.tok0[1] = (tA + 1) * p.nTok;
  it.validB = (tA + 1) < p.ntiles;
  const int last = min(p.L, (it.validB ? tA + 2 : tA + 1) * p.nTok) - 1;
  if (p.is_time) {
    it.key_lo = max(0, it.tok0[0] - p.window + 1);
    it.key_hi = last + 1;
  } else {
    it.key_lo = 0;
    it.key_hi = p.L;
  }
  it.kb_lo = it.key_lo / kBN;
  it.kb_hi = (it.key_hi - 1) / kBN;
  return it;
}

__device__ __forceinline__ int block_ncols(const FwdItem& it, int kb) {
  return min(kBN, it.key_hi - kb * kBN);
}
__device__ __forceinline__ int round16(int x) { return (x + 15) & ~15; }

// K/V stage and phase parity of block index bi (0-based within the item).
struct KvSlot {
  int stage;
  uint32_t parity;
};
__device__ __forceinline__ KvSlot kv_slot(const FwdParams& p, const FwdItem& it, int bi,
                                          uint32_t unit_loads, uint32_t stream_cnt) {
  KvSlot s;
  if (p.resident) {
    s.stage = it.kb_lo + bi;
    s.parity = (unit_loads - 1) & 1u;
  } else {
    const uint32_t c = stream_cnt + bi;
    s.stage = static_cast<int>(c % kStages);
    s.parity = (c / kStages) & 1u;
  }
  return s;
}

// Bit j set <=> column c0 + j of a score row is allowed: lo <= col < hi and col != ex.
__device__ __forceinline__ uint32_t keep_bits32(int c0, int lo, int hi, int ex) {
  const int a = min(max(lo - c0, 0), 32);
  const int b = min(max(hi - c0, 0), 32);
  const uint32_t below_b = b >= 32 ? 0xFFFFFFFFu : ((1u << b) - 1u);
  const uint32_t below_a = a >= 32 ? 0xFFFFFFFFu : ((1u << a) - 1u);
  uint32_t m = below_b & ~below_a;
  if (ex >= c0 && ex < c0 + 32) m &= ~(1u << (ex - c0));
  return m;
}
__device__ __forceinline__ void apply_mask32(float* v, uint32_t keep) {
  if (__any_sync(0xffffffffu, keep != 0xFFFFFFFFu)) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = ((keep >> j) & 1u) ? v[j] : -INFINITY;
  }
}

// bounded wait that ignores the abort flag (used only to drain in-flight async work)
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > OD_WAIT_LIMIT_NS) break;
  }
}

// One pending P V product of the MMA issuer.
struct PvJob {
  uint8_t stage, acc, ksteps, vpar;
};


__global__ void __launch_bounds__(kFwdThreads, 1)
    od_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ[2] = {base, base + kTile};
  uint8_t* sK = base + 2 * kTile;
  uint8_t* sV = sK + kStages * kKVTile;
  uint8_t* sOst = sV + kStages * kKVTile;
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base + kFwdTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const long long i0 = (p.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = (p.nitems * (blockIdx.x + 1)) / gridDim.x;
  OD_TRACE_INIT();

  // zero the Q-tile rows that TMA never writes (rows >= p.rows)
  {
    const int pad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < pad; x += kFwdThreads * 16) {
      *reinterpret_cast<uint4*>(sQ[0] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sQ[1] + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.q_full[x], 1);
      mbar_init(&sm.q_empty[x], 1);
      mbar_init(&sm.o_done[x], 1);
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.s_taken[x], 4);
      mbar_init(&sm.p_full[x], 4);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v16_ready[s], 1);
      mbar_init(&sm.kv_empty[s], 2);
    }
    mbar_init(&sm.drain[0], 1);
    mbar_init(&sm.drain[1], 1);
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
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        long long prev_unit = -1;
        uint32_t unit_loads = 0, stream_cnt = 0, qn0 = 0, qn1 = 0;
        bool ok = true;
        for (long long i = i0; i < i1 && ok; ++i) {
          const FwdItem it = fwd_decode(p, i);
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
          auto load_q = [&](int x, uint32_t& n) -> bool {
            if (n > 0 && !wait_bar(&sm.q_empty[x], (n - 1) & 1u, ctl, status, 1)) return false;
            mbar_arrive_expect_tx(&sm.q_full[x], p.rows * 128);
            if (p.is_time)
              tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, it.fixed, it.tok0[x], it.b);
            else
              tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, it.tok0[x], it.fixed, it.b);
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
              const int stage = static_cast<int>(c % kStages);
              const uint32_t n = c / kStages;
              if (n > 0) ok = wait_bar(&sm.kv_empty[stage], (n - 1) & 1u, ctl, status, 3);
              if (ok) load_kv(stage, it.kb_lo + bi);
            }
            stream_cnt += nb;
          }
        }
        // make sure no TMA load is still writing into this CTA's smem when it exits
        if (qn0 > 0) drain_wait(&sm.q_full[0], (qn0 - 1) & 1u);
        if (qn1 > 0) drain_wait(&sm.q_full[1], (qn1 - 1) & 1u);
        if (p.resident) {
          if (unit_loads > 0)
            for (int s = 0; s < p.nkb; ++s) {
              drain_wait(&sm.k_full[s], (unit_loads - 1) & 1u);
              drain_wait(&sm.v_full[s], (unit_loads - 1) & 1u);
            }
        } else {
          for (int s = 0; s < kStages; ++s) {
            const uint32_t uses =
                stream_cnt / kStages + (static_cast<uint32_t>(s) < stream_cnt % kStages ? 1u : 0u);
            if (uses > 0) {
              drain_wait(&sm.k_full[s], (uses - 1) & 1u);
              drain_wait(&sm.v_full[s], (uses - 1) & 1u);
            }
          }
        }
      }
    } else if (warp == kFwdMmaWarp || warp == kFwdMmaWarp + 1) {
      // ---------------------------------------------------------- MMA issuers
      // Warp 9 issues tile A's MMAs, warp 10 tile B's, each in order: Q K^T(0); then for
      // every block j: wait until the softmax has taken scores j, issue Q K^T(j+1) into the
      // tile's other score buffer; wait for P(j), issue P V(j).  At the end of an item the last
      // P V goes out at once.  Both issuers walk every item (tile B also the items it has no
      // rows in) and release every K/V fill they have seen arrive, so kv_empty counts two.
      {  // whole warp in lockstep; one elected lane issues
        const int x = warp - kFwdMmaWarp;  // 0: tile A, 1: tile B
        const uint32_t idesc_pv_bf16 = idesc_bf16(128, 64, 0, 1);
        const uint32_t idesc_pv_fp16 = idesc_fp16(128, 64, 0, 1);
        const uint32_t tOx = tmem + 384u + 64u * x;
        uint32_t js = 0, jp = 0, qn = 0, unit_loads = 0, sbase = 0;
        long long prev_unit = -1;
        PvJob f0{}, f1{};
        int npend = 0;  // pending P V products; the oldest is slot jp & 1
        bool ok = true;
        auto issue_pv = [&]() -> bool {
          const PvJob jb = (jp & 1u) ? f1 : f0;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.p_full[x], jp & 1u, ctl, status, 9))) return false;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.v16_ready[jb.stage], jb.vpar, ctl, status, 10))) return false;
          tc_fence_after();
          const uint64_t b = sdesc_sw128(smem_u32(sV + jb.stage * kKVTile), 1024, 1024);
          const uint32_t a = tmem + 192u * x + 96u * (jp & 1u);
          const uint32_t fmt = *reinterpret_cast<const uint32_t*>(sm.vfmt[jb.stage]);
          for (int k = 0; k < jb.ksteps; ++k) {
            const uint32_t idesc = ((fmt >> (8 * (k >> 1))) & 0xFFu) ? idesc_pv_bf16 : idesc_pv_fp16;
            mma_ts_w(tOx, a + 8 * k, b + (2048 >> 4) * k, idesc, (jb.acc || k > 0));
          }
          mma_commit_w(&sm.o_done[x]);
          OD_TP(12 + x, 0, (int)jp);
          ++jp;
          --npend;
          if (!p.resident) mma_commit_w(&sm.kv_empty[jb.stage]);
          return true;
        };
        for (long long i = i0; i < i1 && ok; ++i) {
          const FwdItem it = fwd_decode(p, i);
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
                const int stage = static_cast<int>(c % kStages);
                ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[stage], (c / kStages) & 1u, ctl, status, 12));
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
              if (!__all_sync(0xffffffffu, wait_bar(&sm.q_full[x], qn & 1u, ctl, status, 14))) { ok = false; break; }
              ++qn;
            }
            KvSlot ks;
            if (p.resident) {
              ks.stage = it.kb_lo + bi;
              ks.parity = (unit_loads - 1) & 1u;
            } else {
              const uint32_t c = sbase + static_cast<uint32_t>(bi);
              ks.stage = static_cast<int>(c % kStages);
              ks.parity = (c / kStages) & 1u;
            }
            if (!__all_sync(0xffffffffu, wait_bar(&sm.k_full[ks.stage], ks.parity, ctl, status, 15))) { ok = false; break; }
            tc_fence_after();
            const int n = round16(block_ncols(it, it.kb_lo + bi));
            const uint32_t idesc = idesc_bf16(128, n, 0, 0);
            const uint64_t a = sdesc_sw128(smem_u32(sQ[x]), 16, 1024);
            const uint64_t b = sdesc_sw128(smem_u32(sK + ks.stage * kKVTile), 16, 1024);
            const uint32_t d = tmem + 192u * x + 96u * (js & 1u);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss_w(d, a + 2 * k, b + 2 * k, idesc, k > 0);
            mma_commit_w(&sm.s_full[x]);
            OD_TP(10 + x, (int)i, bi);
            PvJob jb;
            jb.stage = static_cast<uint8_t>(ks.stage);
            jb.vpar = static_cast<uint8_t>(ks.parity);
            jb.acc = bi > 0;
            jb.ksteps = static_cast<uint8_t>(n >> 4);
            if (js & 1u) f1 = jb; else f0 = jb;
            ++js;
            ++npend;
            if (bi == nb - 1) mma_commit_w(&sm.q_empty[x]);
            while (ok && npend >= 2) ok = issue_pv();
          }
          // the item's last P V goes out as soon as its P is ready
          while (ok && npend > 0) ok = issue_pv();
          sbase += static_cast<uint32_t>(nb);
        }
        // wait until every MMA issued by this thread has completed before TMEM is freed
        mma_commit_w(&sm.drain[x]);
        drain_wait(&sm.drain[x], 0);
      }
    } else {
      // ---------------------------------------------------------- V converter (warp 11)
      // P V runs in fp16: P in [0, 256] loses 8x less to rounding than in bf16.  Each fill
      // of a V stage is converted in place, per 32-key chunk, when the chunk's magnitude
      // is inside a safe fp16 range (2^-10 <= max|v| <= 2^15, or all zero); otherwise the
      // chunk stays bf16 and the softmax and MMA use bf16 for those keys.
      long long prev_unit = -1;
      uint32_t unit_loads = 0, stream_cnt = 0;
      bool ok = true;
      auto convert = [&](int stage, uint32_t parity) -> bool {
        bool w = wait_bar(&sm.v_full[stage], parity, ctl, status, 4);
        if (!__all_sync(0xffffffffu, w)) return false;
#pragma unroll 1
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint4* chunk = reinterpret_cast<uint4*>(sV + stage * kKVTile + cc * 32 * 128);
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
      for (long long i = i0; i < i1 && ok; ++i) {
        const FwdItem it = fwd_decode(p, i);
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
            ok = convert(static_cast<int>(c % kStages), (c / kStages) & 1u);
          }
          stream_cnt += nb;
        }
      }
    }
  } else {
    regs_inc<kFwdSoftmaxRegs>();
    // ------------------------------------------------------------ softmax warpgroups
    const int x = warp >> 2;         // 0: tile A, 1: tile B
    const int r = tid & 127;         // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + 384 + x * 64 + lane_off;
    const int G = p.G;
    const int tok = r / G;
    const int g = r - tok * G;
    uint32_t jS = 0, jP = 0;
    long long prev_unit = -1;
    uint32_t unit_loads = 0, stream_next = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; ++i) {
      const FwdItem it = fwd_decode(p, i);
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
      const bool row_ok = (r < p.rows) && (pos < p.L);
      float m_used = -INFINITY, l = 0.f;
      for (int bi = 0; bi < nb; ++bi) {
        const int kb = it.kb_lo + bi;
        const int kbase = kb * kBN;
        const int ncols = block_ncols(it, kb);
        const int n32 = (ncols + 31) >> 5;
        const uint32_t tS = tmem + 192u * x + 96u * (jS & 1u) + lane_off;
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
        OD_TP(20, (int)i, bi);
        ok = wait_bar(&sm.s_full[x], jS & 1u, ctl, status, 5);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++jS;
        if (lane == 0) mbar_arrive(&sm.s_taken[x]);
        OD_TP(21, (int)i, bi);
        tc_fence_after();
        // Pass 1 over the scores (32 columns per step, next step's TMEM load in flight):
        // masks and the row maximum.  The loops stay rolled to keep the code small.
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
        {
          // every chunk's TMEM load in flight at once: one round trip
          float v[96];
#pragma unroll
          for (int c = 0; c < 3; ++c)
            if (c < n32) tmem_ld32(tS + 32 * c, v + 32 * c);
          tmem_wait_ld_dep32(v);
          tmem_wait_ld_dep32(v + 32);
          tmem_wait_ld_dep32(v + 64);
#pragma unroll
          for (int c = 0; c < 3; ++c)
            if (c < n32) {
              apply_mask32(v + 32 * c, keep_bits32(32 * c, lo, hi, ex));
#pragma unroll
              for (int jj = 0; jj < 32; jj += 8) {
                mx0 = max3(mx0, v[32 * c + jj], v[32 * c + jj + 1]);
                mx1 = max3(mx1, v[32 * c + jj + 2], v[32 * c + jj + 3]);
                mx2 = max3(mx2, v[32 * c + jj + 4], v[32 * c + jj + 5]);
                mx3 = max3(mx3, v[32 * c + jj + 6], v[32 * c + jj + 7]);
              }
            }
        }
        const float mb = fmaxf(max3(mx0, mx1, mx2), mx3);
        OD_TP(23, (int)i, bi);
        const float mnew = mb * p.sl;
        float alpha = 1.f;
        bool rescale = false;
        if (mb != -INFINITY && (m_used == -INFINITY || mnew > m_used + kRescaleThreshold)) {
          if (m_used != -INFINITY) {
            alpha = ex2(m_used - mnew);
            rescale = bi > 0;
          }
          m_used = mnew;
          l *= alpha;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // V of this block must be converted before P's format can be chosen
        const KvSlot ks = kv_slot(p, it, bi, unit_loads, stream_cnt);
        ok = wait_bar(&sm.v16_ready[ks.stage], ks.parity, ctl, status, 6);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        OD_TP(25, (int)i, bi);
        const uint32_t fmt_bits = *reinterpret_cast<const uint32_t*>(sm.vfmt[ks.stage]);
        const float2 sl2 = make_float2(p.sl, p.sl);
        const float2 nm2 = make_float2(-msub, -msub);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
        // Pass 2: exponentials, row sum, and P written in place over the first half of the
        // score buffer (the P pairs of step c land in columns already read by steps <= c).
        {
          float va[32];
          tmem_ld32(tS, va);
#pragma unroll 1
          for (int c = 0; c < n32; ++c) {
            tmem_wait_ld_dep32(va);
            float2 pp[16];
            apply_mask32(va, keep_bits32(32 * c, lo, hi, ex));
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 xx = __ffma2_rn(make_float2(va[2 * j], va[2 * j + 1]), sl2, nm2);
              pp[j] = make_float2(ex2(xx.x), ex2(xx.y));
            }
            if (c + 1 < n32) tmem_ld32(tS + 32 * (c + 1), va);
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              acc0 = __fadd2_rn(acc0, pp[j]);
              acc1 = __fadd2_rn(acc1, pp[j + 1]);
              acc2 = __fadd2_rn(acc2, pp[j + 2]);
              acc3 = __fadd2_rn(acc3, pp[j + 3]);
            }
            uint32_t pk[16];
            if ((fmt_bits >> (8 * c)) & 0xFFu) {
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(pp[j].x, pp[j].y);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[j] = pack_f16x2(pp[j].x, pp[j].y);
            }
            tmem_st16(tS + 16 * c, pk);
          }
        }
        {
          const float2 a01 = __fadd2_rn(acc0, acc1);
          const float2 a23 = __fadd2_rn(acc2, acc3);
          const float2 a = __fadd2_rn(a01, a23);
          l += a.x + a.y;
        }
        OD_TP(26, (int)i, bi);
        // The previous block's P V must be complete before this block's P is released
        // (keeps o_done exactly one phase behind, and O stable for a rescale).
        if (jP > 0) {
          ok = wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status, 7);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? alpha : 1.f;
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
      ok = wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status, 8);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      OD_TP(30, (int)i, 0);
      tc_fence_after();
      float o[64];
      tmem_ld32(tO, o);
      tmem_ld32(tO + 32, o + 32);
      tmem_wait_ld_dep32(o);
      tmem_wait_ld_dep32(o + 32);
      // Each warp stages its 32 rows (bf16, 128 B each, XOR-swizzled by row to keep the
      // shared-memory accesses conflict free) and then stores them coalesced: one
      // instruction writes 4 whole rows, 8 lanes per row.
      {
        const float inv = 1.f / l;
        uint8_t* stg = sOst + (warp & 7) * 4096;
        const int wr = lane;  // row within the warp
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 wv;
          wv.x = pack_bf16x2(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
          wv.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
          wv.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
          wv.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
          *reinterpret_cast<uint4*>(stg + wr * 128 + ((c ^ (wr & 7)) << 4)) = wv;
        }
        if (row_ok) {
          const int hq = it.kvh * G + g;
          const long long t_idx = p.is_time ? pos : it.fixed;
          const long long s_idx = p.is_time ? it.fixed : pos;
          p.lse[((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + hq] =
              (m_used + log2f(l)) * 0.69314718055994531f;
        }
        __syncwarp();
        const int sub = lane >> 3, ch = lane & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 4 * k + sub;                // row within the warp
          const int rt = (warp & 3) * 32 + rr;       // row within the tile
          const int tk = rt / G;
          const int gg = rt - tk * G;
          const int ps = mytok0 + tk;
          if (rt < p.rows && ps < p.L) {
            const long long t_idx = p.is_time ? ps : it.fixed;
            const long long s_idx = p.is_time ? it.fixed : ps;
            const long long row =
                ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + it.kvh * G + gg;
            const uint4 wv = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
            reinterpret_cast<uint4*>(p.o + row * 64)[ch] = wv;
          }
        }
        __syncwarp();
      }
      OD_TP(31, (int)i, 0);
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

}  // namespace od
