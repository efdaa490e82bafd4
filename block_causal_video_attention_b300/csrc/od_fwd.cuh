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
// K/V for the unit are therefore read once per tile pair and reused by all G heads.
//
// One persistent CTA per SM walks a contiguous range of work items; an item is
// (unit, pair of Q tiles).  Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax warpgroup for Q tile A  (thread i owns TMEM lane / row i)
//   warps 4-7   softmax warpgroup for Q tile B
//   warp  8     TMA producer (one thread)
//   warp  9     TMEM allocator + tcgen05.mma issuer (one thread)
//   warps 10-11 convert each V tile to fp16 in shared memory (P V runs in fp16)
// The kernel launches with kFwdLaunchRegs registers per thread; the softmax warpgroups
// then raise their limit to kFwdSoftmaxRegs and the control warpgroup lowers its own to
// kFwdCtrlRegs.  2*128*kFwdSoftmaxRegs + 128*kFwdCtrlRegs equals the launch allocation, and
// the host refuses to launch if the compiled register count differs from kFwdLaunchRegs.
// TMEM (512 columns): S_A[0,128) S_B[128,256) P_A[256,320) P_B[320,384) O_A[384,448)
// O_B[448,512).  S = Q K^T is fp32 in TMEM; the softmax warps read it, write P as bf16 to
// TMEM, and O += P V runs with A = P taken from TMEM.  Key blocks are 128 keys; the key
// range of an item is the union of the rows' allowed ranges, so key blocks that are fully
// masked for the whole item are never loaded; partial blocks are masked per element.
// Online softmax with a lazy rescale: the running maximum used for the exponentials only
// moves when a block's maximum exceeds it by more than 8 (log2 units); O is then rescaled
// in TMEM.  Statistics are fp32; LSE (natural log) is written per row.
#pragma once
#include <cuda.h>
#include "od_ptx.cuh"

namespace od {

constexpr int kBM = 128;           // query rows per tile (MMA M)
constexpr int kBN = 128;           // keys per key block
constexpr int kStages = 4;         // K/V shared-memory stages
constexpr int kTile = 128 * 128;   // bytes of one 128-row x 64-bf16 tile
constexpr int kFwdThreads = 384;
constexpr int kFwdLaunchRegs = 168;
constexpr int kFwdSoftmaxRegs = 216;
constexpr int kFwdCtrlRegs = 72;
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
  float* lse;
  unsigned int* status;
};

struct FwdSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_empty[2], p_full[2], o_done[2];
  uint64_t st_full[2], st_free[2];
  uint64_t v16_ready[kStages];
  uint64_t drain;
  uint8_t vfmt[kStages][4];  // per 32-key chunk of a V stage: 0 = fp16, 1 = bf16
  uint32_t tmem_base;
  Ctl ctl;
};
// dynamic smem: [Q0 Q1][K0..K3][V0..V3][ST0 ST1][FwdSmem], 1024-byte aligned tiles
constexpr int kFwdTiles = 2 + 2 * kStages + 2;
constexpr size_t kFwdSmemBytes = size_t(kFwdTiles) * kTile + 1024 + sizeof(FwdSmem) + 64;

struct FwdItem {
  long long unit;
  int b, fixed, kvh;
  int tok0[2];
  int validB;
  int key_lo, key_hi;  // allowed key positions of the item lie in [key_lo, key_hi)
  int kb_lo, kb_hi;    // inclusive key-block range
};

__device__ __forceinline__ FwdItem fwd_decode(const FwdParams& p, long long i) {
  FwdItem it;
  const long long unit = i / p.npairs;
  const int pair = static_cast<int>(i - unit * p.npairs);
  it.unit = unit;
  it.kvh = static_cast<int>(unit % p.Hkv);
  const long long r = unit / p.Hkv;
  it.fixed = static_cast<int>(r % p.F);
  it.b = static_cast<int>(r / p.F);
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

// bounded wait that ignores the abort flag (used only to drain in-flight async work)
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > OD_WAIT_LIMIT_NS) break;
  }
}

__global__ void __launch_bounds__(kFwdThreads, 1)
    od_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ[2] = {base, base + kTile};
  uint8_t* sK = base + 2 * kTile;
  uint8_t* sV = base + (2 + kStages) * kTile;
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base + kFwdTiles * kTile);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const long long i0 = (p.nitems * blockIdx.x) / gridDim.x;
  const long long i1 = (p.nitems * (blockIdx.x + 1)) / gridDim.x;

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
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.s_empty[x], 4);
      mbar_init(&sm.p_full[x], 4);
      mbar_init(&sm.o_done[x], 1);
      mbar_init(&sm.st_full[x], 128);
      mbar_init(&sm.st_free[x], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v16_ready[s], 2);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.drain, 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      long long prev_unit = -1;
      uint32_t unit_loads = 0, stream_cnt = 0, qn0 = 0, qn1 = 0;
      bool ok = true;
      for (long long i = i0; i < i1 && ok; ++i) {
        const FwdItem it = fwd_decode(p, i);
        auto load_kv = [&](int stage, int kb) {
          const int kp = kb * kBN;
          mbar_arrive_expect_tx(&sm.k_full[stage], kTile);
          mbar_arrive_expect_tx(&sm.v_full[stage], kTile);
          if (p.is_time) {
            tma_load_5d(sK + stage * kTile, &tm_k, &sm.k_full[stage], 0, it.kvh, it.fixed, kp, it.b);
            tma_load_5d(sV + stage * kTile, &tm_v, &sm.v_full[stage], 0, it.kvh, it.fixed, kp, it.b);
          } else {
            tma_load_5d(sK + stage * kTile, &tm_k, &sm.k_full[stage], 0, it.kvh, kp, it.fixed, it.b);
            tma_load_5d(sV + stage * kTile, &tm_v, &sm.v_full[stage], 0, it.kvh, kp, it.fixed, it.b);
          }
        };
        if (p.resident && it.unit != prev_unit) {
          if (unit_loads > 0) {
            for (int s = 0; s < p.nkb && ok; ++s)
              ok = wait_bar(&sm.kv_empty[s], (unit_loads - 1) & 1u, ctl, status);
          }
          if (!ok) break;
          for (int kb = 0; kb < p.nkb; ++kb) load_kv(kb, kb);
          ++unit_loads;
          prev_unit = it.unit;
        }
        auto load_q = [&](int x, uint32_t& n) -> bool {
          if (n > 0 && !wait_bar(&sm.q_empty[x], (n - 1) & 1u, ctl, status)) return false;
          mbar_arrive_expect_tx(&sm.q_full[x], p.rows * 128);
          if (p.is_time)
            tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, it.fixed, it.tok0[x], it.b);
          else
            tma_load_5d(sQ[x], &tm_q, &sm.q_full[x], 0, it.kvh * p.G, it.tok0[x], it.fixed, it.b);
          ++n;
          return true;
        };
        ok = load_q(0, qn0);
        if (ok && it.validB) ok = load_q(1, qn1);
        if (!p.resident) {
          const int nb = it.kb_hi - it.kb_lo + 1;
          for (int bi = 0; bi < nb && ok; ++bi) {
            const uint32_t c = stream_cnt + bi;
            const int stage = static_cast<int>(c % kStages);
            const uint32_t n = c / kStages;
            if (n > 0) ok = wait_bar(&sm.kv_empty[stage], (n - 1) & 1u, ctl, status);
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
          const uint32_t uses = stream_cnt / kStages + (static_cast<uint32_t>(s) < stream_cnt % kStages ? 1u : 0u);
          if (uses > 0) {
            drain_wait(&sm.k_full[s], (uses - 1) & 1u);
            drain_wait(&sm.v_full[s], (uses - 1) & 1u);
          }
        }
      }
    }
   } else if (warp == kFwdMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tS[2] = {tmem + 0, tmem + 128};
      const uint32_t tP[2] = {tmem + 256, tmem + 320};
      const uint32_t tO[2] = {tmem + 384, tmem + 448};
      const uint32_t idesc_pv_bf16 = idesc_bf16(128, 64, 0, 1);
      const uint32_t idesc_pv_fp16 = idesc_fp16(128, 64, 0, 1);
      long long prev_unit = -1;
      uint32_t unit_loads = 0, stream_cnt = 0, qn[2] = {0, 0}, jS[2] = {0, 0}, jP[2] = {0, 0};
      bool ok = true;
      for (long long i = i0; i < i1 && ok; ++i) {
        const FwdItem it = fwd_decode(p, i);
        if (p.resident && it.unit != prev_unit) {
          if (unit_loads > 0)
            for (int s = 0; s < p.nkb; ++s) mma_commit(&sm.kv_empty[s]);
          ++unit_loads;
          prev_unit = it.unit;
        }
        const int nb = it.kb_hi - it.kb_lo + 1;
        ok = wait_bar(&sm.q_full[0], qn[0] & 1u, ctl, status);
        ++qn[0];
        if (ok && it.validB) {
          ok = wait_bar(&sm.q_full[1], qn[1] & 1u, ctl, status);
          ++qn[1];
        }
        if (!ok) break;
        auto issue_qk = [&](int x, int bi) -> bool {
          const KvSlot ks = kv_slot(p, it, bi, unit_loads, stream_cnt);
          if (!wait_bar(&sm.k_full[ks.stage], ks.parity, ctl, status)) return false;
          if (jS[x] > 0 && !wait_bar(&sm.s_empty[x], (jS[x] - 1) & 1u, ctl, status)) return false;
          tc_fence_after();
          const int n = round16(block_ncols(it, it.kb_lo + bi));
          const uint32_t idesc = idesc_bf16(128, n, 0, 0);
          const uint64_t a = sdesc_sw128(smem_u32(sQ[x]), 16, 1024);
          const uint64_t b = sdesc_sw128(smem_u32(sK + ks.stage * kTile), 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tS[x], a + 2 * k, b + 2 * k, idesc, k > 0);
          mma_commit(&sm.s_full[x]);
          ++jS[x];
          return true;
        };
        auto issue_pv = [&](int x, int bi) -> bool {
          const KvSlot ks = kv_slot(p, it, bi, unit_loads, stream_cnt);
          if (!wait_bar(&sm.v16_ready[ks.stage], ks.parity, ctl, status)) return false;
          if (!wait_bar(&sm.p_full[x], jP[x] & 1u, ctl, status)) return false;
          tc_fence_after();
          const int ksteps = round16(block_ncols(it, it.kb_lo + bi)) >> 4;
          const uint64_t b = sdesc_sw128(smem_u32(sV + ks.stage * kTile), 1024, 1024);
          for (int k = 0; k < ksteps; ++k) {
            const uint32_t idesc = sm.vfmt[ks.stage][k >> 1] ? idesc_pv_bf16 : idesc_pv_fp16;
            mma_ts(tO[x], tP[x] + 8 * k, b + (2048 >> 4) * k, idesc, (bi > 0 || k > 0));
          }
          mma_commit(&sm.o_done[x]);
          ++jP[x];
          return true;
        };
        ok = issue_qk(0, 0);
        if (ok && it.validB) ok = issue_qk(1, 0);
        for (int bi = 0; bi < nb && ok; ++bi) {
          if (bi + 1 < nb) ok = issue_qk(0, bi + 1);
          else mma_commit(&sm.q_empty[0]);
          if (ok) ok = issue_pv(0, bi);
          if (ok && it.validB) {
            if (bi + 1 < nb) ok = issue_qk(1, bi + 1);
            else mma_commit(&sm.q_empty[1]);
            if (ok) ok = issue_pv(1, bi);
          }
          if (ok && !p.resident) mma_commit(&sm.kv_empty[kv_slot(p, it, bi, 0, stream_cnt).stage]);
        }
        if (!p.resident) stream_cnt += nb;
      }
      // wait until every MMA issued by this thread has completed before TMEM is freed
      mma_commit(&sm.drain);
      drain_wait(&sm.drain, 0);
    }
   } else {
    // ------------------------------------------------------------ V converter (warps 10-11)
    // P V runs in fp16: P in [0, 256] loses 8x less to rounding than in bf16.  Each fill
    // of a V stage is converted in place, per 32-key chunk, when the chunk's magnitude
    // is inside a safe fp16 range (2^-10 <= max|v| <= 2^15, or all zero); otherwise the
    // chunk stays bf16 and the softmax and MMA use bf16 for those keys.
    const int cw = warp - 10;
    long long prev_unit = -1;
    uint32_t unit_loads = 0, stream_cnt = 0;
    bool ok = true;
    auto convert = [&](int stage, uint32_t parity) -> bool {
      bool w = wait_bar(&sm.v_full[stage], parity, ctl, status);
      if (!__all_sync(0xffffffffu, w)) return false;
#pragma unroll 1
      for (int cc = 2 * cw; cc < 2 * cw + 2; ++cc) {
        uint4* chunk = reinterpret_cast<uint4*>(sV + stage * kTile + cc * 32 * 128);
        float mx = 0.f;
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const uint4 d = chunk[lane + 32 * j];
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
          for (int j = 0; j < 8; ++j) {
            const uint4 d = chunk[lane + 32 * j];
            uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
              wv[h] = pack_f16x2(__uint_as_float(wv[h] << 16), __uint_as_float(wv[h] & 0xFFFF0000u));
            chunk[lane + 32 * j] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
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
    const uint32_t tS = tmem + x * 128 + lane_off;
    const uint32_t tP = tmem + 256 + x * 64 + lane_off;
    const uint32_t tO = tmem + 384 + x * 64 + lane_off;
    const int G = p.G;
    const int tok = r / G;
    const int g = r - tok * G;
    uint32_t jS = 0, jP = 0, e = 0;
    long long prev_unit = -1;
    uint32_t unit_loads = 0, stream_next = 0;
    bool ok = true;
    for (long long i = i0; i < i1 && ok; ++i) {
      const FwdItem it = fwd_decode(p, i);
      if (p.resident && it.unit != prev_unit) {
        ++unit_loads;
        prev_unit = it.unit;
      }
      const uint32_t stream_cnt = stream_next;
      stream_next += it.kb_hi - it.kb_lo + 1;
      if (x == 1 && !it.validB) continue;
      const int mytok0 = x ? it.tok0[1] : it.tok0[0];
      const int pos = mytok0 + tok;
      const bool row_ok = (r < p.rows) && (pos < p.L);
      float m_used = -INFINITY, l = 0.f;
      const int nb = it.kb_hi - it.kb_lo + 1;
      for (int bi = 0; bi < nb; ++bi) {
        const int kb = it.kb_lo + bi;
        const int kbase = kb * kBN;
        const int ncols = block_ncols(it, kb);
        const int nch = (ncols + 31) >> 5;
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
        ok = wait_bar(&sm.s_full[x], jS & 1u, ctl, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < nch) tmem_ld32(tS + 32 * c, s + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_empty[x]);
        ++jS;
        const bool need_mask = !(lo <= 0 && hi >= nch * 32 && ex < 0);
        if (__any_sync(0xffffffffu, need_mask)) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (c < nch) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int col = 32 * c + j;
                const bool keep = (col >= lo) && (col < hi) && (col != ex);
                s[32 * c + j] = keep ? s[32 * c + j] : -INFINITY;
              }
            }
        }
        float mb = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < nch) {
#pragma unroll
            for (int j = 0; j < 32; ++j) mb = fmaxf(mb, s[32 * c + j]);
          }
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
        // the previous P V of this tile must be done: P buffer free, O stable
        if (jP > 0) {
          ok = wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status);
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
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // V of this block must be converted before P's format can be chosen
        const KvSlot ks = kv_slot(p, it, bi, unit_loads, stream_cnt);
        ok = wait_bar(&sm.v16_ready[ks.stage], ks.parity, ctl, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < nch) {
            const bool as_bf16 = sm.vfmt[ks.stage][c] != 0;
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float p0 = ex2(fmaf(s[32 * c + j], p.sl, -msub));
              const float p1 = ex2(fmaf(s[32 * c + j + 1], p.sl, -msub));
              l += p0 + p1;
              pk[j >> 1] = as_bf16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            }
            tmem_st16(tP + 16 * c, pk);
          }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[x]);
        ++jP;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      ok = wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float o[64];
      tmem_ld32(tO, o);
      tmem_ld32(tO + 32, o + 32);
      tmem_wait_ld();
      if (e > 0) {
        ok = wait_bar(&sm.st_free[x], (e - 1) & 1u, ctl, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      const float inv = 1.f / l;
      uint8_t* const stile = base + (2 + 2 * kStages + x) * kTile;
      uint8_t* st = stile + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w;
        w.x = pack_bf16x2(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
        w.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
        w.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
        w.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
        *reinterpret_cast<uint4*>(st + ((c ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.st_full[x]);
      if (row_ok) {
        const int hq = it.kvh * G + g;
        const long long t_idx = p.is_time ? pos : it.fixed;
        const long long s_idx = p.is_time ? it.fixed : pos;
        const long long idx = ((static_cast<long long>(it.b) * p.T + t_idx) * p.S + s_idx) * p.Hq + hq;
        p.lse[idx] = (m_used + log2f(l)) * 0.69314718055994531f;
      }
      if (r == 0) {
        ok = wait_bar(&sm.st_full[x], e & 1u, ctl, status);
        if (ok) {
          if (p.is_time)
            tma_store_5d(&tm_o, stile, 0, it.kvh * G, it.fixed, mytok0, it.b);
          else
            tma_store_5d(&tm_o, stile, 0, it.kvh * G, mytok0, it.fixed, it.b);
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&sm.st_free[x]);
        }
      }
      ++e;
    }
    if (r == 0) bulk_wait0();
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
