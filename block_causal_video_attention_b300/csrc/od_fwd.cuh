// od_fwd.cuh -- forward kernel shared by space and time attention (sm_103a).
//
// Both operators are "masked attention over the sequence of one unit":
//   space: unit = (b, t, kv head), sequence = the S tokens of that timestep block,
//          mask = the agent-token read restriction (world-model tokens cannot read the
//          agent token; 7minutos.es page, "Arquitectura: una columna vertebral, dos modelos");
//   time:  unit = (b, s, kv head), sequence = the T timesteps at token position s,
//          mask = causal with a sliding window of W steps (edgex es-LA page,
//          "Configuracion de entrenamiento": a 192-step window).
// All G = Hq/Hkv query heads of a KV head are rows of one Q tile ("grouped-query
// attention"): a tile holds nTok = floor(128/G) consecutive sequence positions x G heads, which
// in the [B,T,S,H,D] layout is one 5-D TMA box (64, G, nTok) -- rows r = tok*G + g.  Short
// time sequences (G*T <= 64) are packed instead: a tile holds pk = floor(128/(G*T)) token
// positions x all T timesteps x G heads (box (64, G, pk, T), rows r = (t*pk + sp)*G + g), and
// its keys are the pk*T keys of the same positions (box (64, 1, pk, T), key c = t*pk + sp), so
// the mask is block-diagonal in sp and causal-windowed in t.
//
// Work item = (unit, pair of Q tiles A and B); one persistent CTA per SM walks a contiguous
// range of items (every gridDim.x-th item for variable-length blocks).  Keys come in blocks
// of 128 (one QK^T MMA of N = 128 reads 8 KB of shared memory per k-step, which the tensor
// core consumes at its full rate; N = 64 would be bound by shared-memory bandwidth).  K/V of a
// unit stay resident in shared memory across its items when they fit in the three stages, else
// stream through them.
//
// Roles (384 threads, three warpgroups):
//   warpgroup 0 (warps 0-3): softmax of tile A, one query row per thread (TMEM lane = row)
//   warpgroup 1 (warps 4-7): softmax of tile B
//   warp 8  TMA producer (one thread)
//   warps 9, 10  tcgen05.mma issuers of tiles A and B (whole warp, one elected lane issues);
//        warp 9 also allocates TMEM
//   warp 11  converts V stages to fp16 in place (P V runs in fp16)
// The kernel launches with kFwdLaunchRegs registers per thread; the softmax warpgroups rise to
// kFwdSoftmaxRegs and the control warpgroup drops to kFwdCtrlRegs.  The shares add up to the
// launch allocation, and the host refuses to launch if the compiled count differs.
//
// TMEM (512 columns), per tile x at 256x: scores S [0,128) fp32, P [128,192) (fp16 pairs),
// O [192,256) fp32.  Each tile's issuer keeps its QK^T one key block ahead of its P V:
// QK^T(j+1) goes out as soon as the softmax has loaded S(j) into registers, P V(j) as soon as
// P(j) is in TMEM.  The softmax computes P(j+1) in registers and only then waits for P V(j)
// (P is single-buffered), so that wait overlaps the exponentials.
//
// Online softmax with a lazy rescale: a row's running maximum only moves when a block's
// maximum exceeds it by more than 8 (log2 units); that row of O is then rescaled in TMEM.
// Statistics are fp32.  Output: the softmax threads stage bf16(O) (and, on request, the
// residual O - bf16(O)) in shared memory with the 128-byte swizzle and one thread per tile
// stores the tile with one TMA box (rows past the sequence fall outside the tensor and are not
// written); variable-length blocks store per thread (their padding rows must stay untouched).//
// Every wait is bounded (od_ptx.cuh), and every mbarrier is waited on at most one phase ahead
// of or behind its completions (a parity wait cannot tell more apart); the protocol comments
// below state why for each barrier.
#pragma once
#include "od_common.cuh"

namespace od {

constexpr int kFwdBN = 128;                   // keys per key block
constexpr int kFwdStages = 3;                 // K and V stages of 128 rows
constexpr int kFwdKVTile = kFwdBN * 128;      // bytes of one K or V stage
constexpr int kFwdThreads = 384;
constexpr int kFwdLaunchRegs = 168;
constexpr int kFwdSoftmaxRegs = 208;
constexpr int kFwdCtrlRegs = 88;
static_assert(256 * kFwdSoftmaxRegs + 128 * kFwdCtrlRegs == kFwdThreads * kFwdLaunchRegs,
              "register split must add up to the launch allocation");
constexpr int kFwdProducerWarp = 8;
constexpr int kFwdMmaWarp = 9;               // 9: tile A's MMAs (and the TMEM allocation), 10: tile B's
constexpr int kFwdConvWarp = 11;

// Layout modes of the forward.
constexpr int kModeSpace = 0;
constexpr int kModeTime = 1;
constexpr int kModeTimePacked = 2;

struct AttnFwdParams {
  int B, T, S, Hq, Hkv, G;
  int mode;       // kModeSpace, kModeTime or kModeTimePacked
  int L;          // sequence length of a unit (S for space, T for time)
  int F;          // units per (b, kv head): T (space), S (time), ceil(S / (2 pk)) (packed)
  int pk;         // packed time: token positions per tile (1 otherwise)
  int agent;      // space: agent token index or -1
  int window;     // time: window length W >= 1
  float sl;       // scale * log2(e)
  int nTok;       // sequence positions per Q tile (packed: T)
  int rows;       // Q rows per tile: nTok * G (packed: pk * T * G), <= 128
  int ntiles;     // Q tiles per unit
  int npairs;     // work items per unit
  long long nitems;
  int nkb;        // key blocks of a unit (packed: 2, one per tile)
  int kvb;        // keys per key block: 128, or pk * T when packed
  int resident;   // nkb <= kFwdStages: a unit's K/V stay in shared memory across its items
  // reciprocals for the item decode: floor(2^64 / d) + 1 for d = npairs, Hkv, F (0 when
  // d >= 2^16, where the plain division is used)
  unsigned long long rcp_npairs, rcp_hkv, rcp_f;
  // space attention with variable-length timestep blocks: block (b, t) holds its first
  // seqlen[b * T + t] tokens (clamped to [0, S]); the rest of the S slots are padding that
  // is neither read as a key nor written as a query row.  NULL: every block holds S tokens.
  const int* seqlen;
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;   // optional: O - bf16(O), rounded to bf16 (for the backward's Delta)
  int tma_out;           // O (and O_lo) leave by TMA store of staged tiles
  float* lse;
  unsigned int* status;
};

struct FwdItem2 {
  uint32_t unit;
  int b, fixed, kvh;
  int L;           // the unit's sequence length
  int valid[2];    // tile x has rows to compute
  int tok0[2];     // first sequence position of tile x (packed: first token position s)
  int lo[2], hi[2];  // inclusive key-block range of tile x
  int ulo, uhi;    // union of the ranges (the blocks the item loads)
  int key_hi;      // keys at or past key_hi are never read
};

template <bool kVarlen, int kMode>
__device__ __forceinline__ FwdItem2 fwd_item(const AttnFwdParams& p, int i) {
  // the host guarantees nitems < 2^31, so 32-bit unsigned division suffices
  FwdItem2 it;
  const uint32_t ii = static_cast<uint32_t>(i);
  const uint32_t unit = div_rcp(ii, static_cast<uint32_t>(p.npairs), p.rcp_npairs);
  const int pair = static_cast<int>(ii - unit * static_cast<uint32_t>(p.npairs));
  it.unit = unit;
  const uint32_t r = div_rcp(unit, static_cast<uint32_t>(p.Hkv), p.rcp_hkv);
  it.kvh = static_cast<int>(unit - r * static_cast<uint32_t>(p.Hkv));
  const uint32_t bq = div_rcp(r, static_cast<uint32_t>(p.F), p.rcp_f);
  it.fixed = static_cast<int>(r - bq * static_cast<uint32_t>(p.F));
  it.b = static_cast<int>(bq);
  if (kMode == kModeTimePacked) {
    const int s0 = it.fixed * 2 * p.pk;
    it.L = p.L;
    it.tok0[0] = s0;
    it.tok0[1] = s0 + p.pk;
    it.valid[0] = 1;
    it.valid[1] = s0 + p.pk < p.S;
    it.lo[0] = it.hi[0] = 0;
    it.lo[1] = it.hi[1] = 1;
    it.ulo = 0;
    it.uhi = it.valid[1] ? 1 : 0;
    it.key_hi = p.kvb;
    return it;
  }
  int L = p.L;
  if (kVarlen) L = min(max(__ldg(p.seqlen + static_cast<long long>(it.b) * p.T + it.fixed), 0), p.L);
  it.L = L;
  const int tA = 2 * pair;
  it.tok0[0] = tA * p.nTok;
  it.tok0[1] = (tA + 1) * p.nTok;
  it.valid[0] = kVarlen ? it.tok0[0] < L : 1;
  it.valid[1] = (tA + 1) < p.ntiles && (!kVarlen || it.tok0[1] < L);
  const int last = min(L, (it.valid[1] ? tA + 2 : tA + 1) * p.nTok) - 1;
  int key_lo;
  if (kMode == kModeTime) {
    key_lo = max(0, it.tok0[0] - p.window + 1);
    it.key_hi = last + 1;
  } else {
    key_lo = 0;
    it.key_hi = L;
  }
  it.ulo = key_lo / kFwdBN;
  it.uhi = it.valid[0] ? (it.key_hi - 1) / kFwdBN : it.ulo - 1;  // none if the item is skipped
  it.lo[0] = it.lo[1] = it.ulo;
  it.hi[0] = it.hi[1] = it.uhi;
  return it;
}

// Columns of key block kb that hold keys of the unit (the rest are masked).
template <int kMode>
__device__ __forceinline__ int fwd_ncols(const AttnFwdParams& p, const FwdItem2& it, int kb) {
  return kMode == kModeTimePacked ? p.kvb : min(kFwdBN, it.key_hi - kb * kFwdBN);
}

// Stage and phase parity of the key block of step s of tile x.
struct FwdSlot {
  int stage;
  uint32_t parity;
};
// blk: the key block; s: its fill ordinal within the item (blk - ulo)
template <bool kRes>
__device__ __forceinline__ FwdSlot fwd_slot(int blk, int s, uint32_t unit_loads,
                                            uint32_t stream_base) {
  FwdSlot f;
  if (kRes) {
    f.stage = blk;
    f.parity = (unit_loads - 1) & 1u;
  } else {
    const uint32_t c = stream_base + static_cast<uint32_t>(s);
    f.stage = static_cast<int>(c % kFwdStages);
    f.parity = (c / kFwdStages) & 1u;
  }
  return f;
}

struct FwdSmem {
  uint64_t q_full[2][2], q_empty[2][2];  // per tile, two Q slots (the next item's tile prefetched)
  uint64_t k_full[kFwdStages], v_full[kFwdStages], v16_ready[kFwdStages];
  uint64_t k_empty[kFwdStages], v_empty[kFwdStages];
  // per tile: scores ready (QK^T done), scores loaded by the 4 softmax warps, P ready (4
  // warps), P V done
  uint64_t s_full[2], s_taken[2], p_full[2], o_done[2];
  // per tile (4 warps): output rows staged for the TMA stores; staging free again (the
  // previous stores have read it)
  uint64_t st_full[2], st_free[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  Ctl ctl;
  int vexp[kFwdStages];  // per V stage fill: its keys hold fp16(v * 2^vexp)
};
// dynamic smem: [Q: tile A slots 0 1, tile B slots 0 1][K stages][V stages]
//               [O staging: tile A, tile B][O residual staging: tile A, tile B][FwdSmem]
constexpr size_t kFwdTileBytes =
    size_t(4) * kTile + size_t(2 * kFwdStages) * kFwdKVTile + size_t(4) * kTile;
constexpr size_t kFwdSmemBytes = kFwdTileBytes + 1024 + sizeof(FwdSmem) + 64;
static_assert(kFwdSmemBytes <= 227 * 1024, "shared memory budget");

// Ties 32 registers to a preceding wait (no instruction): their uses stay after it.
__device__ __forceinline__ void reg_dep32(float* v) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                 "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                 "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31]));
}

// Maximum of 32 values: four chains of 3-input max.
__device__ __forceinline__ float max32(const float* v) {
  float a = max3(v[0], v[1], v[2]), b = max3(v[3], v[4], v[5]);
  float c = max3(v[6], v[7], v[8]), d = max3(v[9], v[10], v[11]);
#pragma unroll
  for (int j = 12; j < 28; j += 8) {
    a = max3(a, v[j], v[j + 1]);
    b = max3(b, v[j + 2], v[j + 3]);
    c = max3(c, v[j + 4], v[j + 5]);
    d = max3(d, v[j + 6], v[j + 7]);
  }
  a = max3(a, v[28], v[29]);
  b = max3(b, v[30], v[31]);
  return fmaxf(max3(a, b, c), d);
}

// Bit j set <=> j == first, first + step, ... (< 32): the columns of one token position in a
// packed time tile (key column c belongs to position c mod step).
__device__ __forceinline__ uint32_t stride_bits32(int first, int step) {
  if (step == 1) return 0xFFFFFFFFu;
  uint32_t m = 0;
  for (int j = first; j < 32; j += step) m |= 1u << j;
  return m;
}

template <bool kVarlen, int kMode, bool kRes>
__global__ void __launch_bounds__(kFwdThreads, 1)
    od_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_lo, const AttnFwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start of the dynamic shared memory, formed by pointer arithmetic on the
  // __shared__ array (not through an integer) so that every tile is addressed as shared memory
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = base;  // tile x, slot s at (2x + s) * kTile
  uint8_t* sK = base + 4 * kTile;
  uint8_t* sV = sK + kFwdStages * kFwdKVTile;
  uint8_t* sOst = sV + kFwdStages * kFwdKVTile;  // tile x at x * kTile
  uint8_t* sLst = sOst + 2 * kTile;
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base + kFwdTileBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // (the host guarantees nitems < 2^31)
  const bool strided = kVarlen;
  const int istep = strided ? static_cast<int>(gridDim.x) : 1;
  const int i0 = strided ? static_cast<int>(blockIdx.x) : static_cast<int>((p.nitems * blockIdx.x) / gridDim.x);
  const int i1 = strided ? static_cast<int>(p.nitems) : static_cast<int>((p.nitems * (blockIdx.x + 1)) / gridDim.x);
  OD_TRACE_INIT(0);

  // Zero what TMA never writes: Q-tile rows >= p.rows, and K/V stage rows >= p.kvb (packed
  // tiles whose key blocks are shorter than 128 rows; the MMAs read up to 16-row multiples).
  {
    const int qpad = (kBM - p.rows) * 128;
    for (int x = tid * 16; x < qpad; x += kFwdThreads * 16)
      for (int t = 0; t < 4; ++t)
        *reinterpret_cast<uint4*>(sQ + t * kTile + p.rows * 128 + x) = make_uint4(0, 0, 0, 0);
    const int kvpad = (kFwdBN - p.kvb) * 128;
    for (int x = tid * 16; x < kvpad; x += kFwdThreads * 16)
      for (int t = 0; t < 2 * kFwdStages; ++t)
        *reinterpret_cast<uint4*>(sK + t * kFwdKVTile + p.kvb * 128 + x) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      for (int q = 0; q < 2; ++q) {
        mbar_init(&sm.q_full[x][q], 1);
        mbar_init(&sm.q_empty[x][q], 1);
      }
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.s_taken[x], 4);
      mbar_init(&sm.p_full[x], 4);
      mbar_init(&sm.o_done[x], 1);
      mbar_init(&sm.st_full[x], 4);
      mbar_init(&sm.st_free[x], 1);
      mbar_init(&sm.drain[x], 1);
    }
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v16_ready[s], 1);
      mbar_init(&sm.k_empty[s], 2);  // released by both MMA issuers
      mbar_init(&sm.v_empty[s], 2);
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
      // Q tiles go to alternating slots per tile (slot reuse waits for the MMA issuer's
      // release after the item's last QK^T).  K/V: resident -- a new unit's K blocks load as
      // soon as the old unit's last QK^T has read the stages (k_empty), its V blocks once the
      // last P V has (v_empty); streaming -- block by block through the ring, each stage
      // reloaded after both tiles' QK^T (K) / P V (V) of its previous fill.
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        long long prev_unit = -1;
        uint32_t unit_loads = 0, stream_cnt = 0, qn[2] = {0, 0};
        bool ok = true;
#pragma unroll 1
  #pragma unroll 1
    for (int i = i0; i < i1 && ok; i += istep) {
          const FwdItem2 it = fwd_item<kVarlen, kMode>(p, i);
          if (kVarlen && !it.valid[0]) continue;  // past the unit's length: no role touches it
          auto kv_coords = [&](int kb, int* c) {
            if (kMode == kModeSpace) {
              c[0] = kb * kFwdBN; c[1] = it.fixed;
            } else if (kMode == kModeTime) {
              c[0] = it.fixed; c[1] = kb * kFwdBN;
            } else {
              c[0] = it.tok0[0] + kb * p.pk; c[1] = 0;
            }
          };
          auto load_k = [&](int stage, int kb) {
            int c[2];
            kv_coords(kb, c);
            // (a packed unit without a tile B loads its second block from past the end on
            // purpose: TMA fills it with zeros)
            if (kMode != kModeTimePacked || kb == 0 || it.valid[1])
              (void)OD_TMA_OK(it.kvh, c[0], c[1], it.b, p.Hkv, p.S, p.T, p.B, status, 201);
            mbar_arrive_expect_tx(&sm.k_full[stage], p.kvb * 128);
            tma_load_5d(sK + stage * kFwdKVTile, &tm_k, &sm.k_full[stage], 0, it.kvh, c[0], c[1], it.b);
          };
          auto load_v = [&](int stage, int kb) {
            int c[2];
            kv_coords(kb, c);
            mbar_arrive_expect_tx(&sm.v_full[stage], p.kvb * 128);
            tma_load_5d(sV + stage * kFwdKVTile, &tm_v, &sm.v_full[stage], 0, it.kvh, c[0], c[1], it.b);
          };
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok || !it.valid[x]) continue;
            const uint32_t n = qn[x];
            const int q = n & 1;
            if (n >= 2) ok = wait_bar(&sm.q_empty[x][q], ((n >> 1) - 1) & 1u, ctl, status, 1);
            if (!ok) break;
            uint8_t* dst = sQ + (2 * x + q) * kTile;
            mbar_arrive_expect_tx(&sm.q_full[x][q], p.rows * 128);
            const int c1 = it.kvh * p.G;
            (void)OD_TMA_OK(c1, kMode == kModeTime ? it.fixed : it.tok0[x],
                            kMode == kModeSpace ? it.fixed : (kMode == kModeTime ? it.tok0[x] : 0),
                            it.b, p.Hq, p.S, p.T, p.B, status, 200);
            if (kMode == kModeSpace)
              tma_load_5d(dst, &tm_q, &sm.q_full[x][q], 0, c1, it.tok0[x], it.fixed, it.b);
            else if (kMode == kModeTime)
              tma_load_5d(dst, &tm_q, &sm.q_full[x][q], 0, c1, it.fixed, it.tok0[x], it.b);
            else
              tma_load_5d(dst, &tm_q, &sm.q_full[x][q], 0, c1, it.tok0[x], 0, it.b);
            qn[x] = n + 1;
            OD_TP(20 + x, (int)i, 0);
          }
          if (!ok) break;
          if (kRes) {
            if (it.unit != prev_unit) {
              // every block of the unit, whatever range this item needs (later items of the
              // unit may need more; a packed unit without a tile B loads its all-out-of-range
              // block too, which keeps every stage's phase count equal to the unit count)
              const int nload = p.nkb;
              for (int s = 0; s < nload && ok; ++s) {
                if (unit_loads > 0) ok = wait_bar(&sm.k_empty[s], (unit_loads - 1) & 1u, ctl, status, 2);
                if (ok) load_k(s, s);
              }
              OD_TP(22, (int)i, 0);
              for (int s = 0; s < nload && ok; ++s) {
                if (unit_loads > 0) ok = wait_bar(&sm.v_empty[s], (unit_loads - 1) & 1u, ctl, status, 3);
                if (ok) load_v(s, s);
              }
              OD_TP(23, (int)i, 0);
              ++unit_loads;
              prev_unit = it.unit;
            }
          } else {
            const int nb = it.uhi - it.ulo + 1;
            for (int s = 0; s < nb && ok; ++s) {
              const uint32_t c = stream_cnt + s;
              const int stage = static_cast<int>(c % kFwdStages);
              const uint32_t n = c / kFwdStages;
              if (n > 0) ok = wait_bar(&sm.k_empty[stage], (n - 1) & 1u, ctl, status, 4);
              if (ok) load_k(stage, it.ulo + s);
              if (ok && n > 0) ok = wait_bar(&sm.v_empty[stage], (n - 1) & 1u, ctl, status, 5);
              if (ok) load_v(stage, it.ulo + s);
            }
            stream_cnt += nb;
          }
        }
        // make sure no TMA load is still writing into this CTA's smem when it exits
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t uses = qn[x] / 2 + (static_cast<uint32_t>(q) < (qn[x] & 1u) ? 1u : 0u);
            if (uses > 0) drain_wait(&sm.q_full[x][q], (uses - 1) & 1u);
          }
        if (kRes) {
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
      // Warp 9 issues tile A's MMAs, warp 10 tile B's, each in order: per item, steps
      // s = 0 .. the tile's block count: QK^T(s) into S (after the softmax took the previous
      // S), then the P V still pending from the tile's previous step (after its P is in TMEM
      // and the V stage is fp16-ready).  The P V of an item's last step stays pending into the
      // next item, whose first QK^T thus overlaps the last softmax.  Both issuers release every
      // K/V fill they have seen (k_empty / v_empty count two), including fills of items in which
      // their tile has no rows, and observe each new fill before they can release it (a release
      // counts toward the phase of the fill it follows; an issuer whose tile has no rows would
      // otherwise run ahead and complete a phase alone).  Protocol:
      //  * s_taken[x] phase n is waited before QK^T n+1: the softmax takes S n+1 only after
      //    QK^T n+1 is issued, so the barrier is never two phases ahead;
      //  * p_full[x] phase n before P V n: the softmax writes P n+1 only after P V n has
      //    completed (o_done), which needs this issue first.
      {
        const int x = warp - kFwdMmaWarp;
        const uint32_t idesc_pv = idesc_fp16(128, 64, 0, 1);
        // Descriptor bases, computed once: the start-address field of a shared-memory
        // descriptor is the byte address / 16, so a tile at a byte offset adds offset / 16.
        const uint64_t dq0 = sdesc_sw128(smem_u32(sQ + 2 * x * kTile), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv0 = sdesc_sw128(smem_u32(sV), 1024, 1024);
        const uint32_t tS = tmem + 256u * x, tP = tS + 128u, tO = tS + 192u;
        uint32_t nqk = 0, npv = 0, qn = 0, unit_loads = 0, stream_cnt = 0;
        int prev_unit = -1;
        bool k_released = false;  // resident: this unit's K stages already released
        // the pending P V: on, stage, V phase parity, k-steps, accumulate
        int pon = 0, pst = 0, pks = 0;
        uint32_t pvp = 0, pacc = 0;
        bool ok = true;
        auto issue_pv = [&]() -> bool {
          if (!__all_sync(0xffffffffu, wait_bar(&sm.p_full[x], npv & 1u, ctl, status, 10) &&
                                       wait_bar(&sm.v16_ready[pst], pvp, ctl, status, 11)))
            return false;
          OD_TP(44 + x, 0, 0);
          tc_fence_after();
          const uint64_t bv = dv0 + static_cast<uint64_t>(pst * (kFwdKVTile >> 4));
          if (pks == 8) {
            mma_ts_k128_w(tO, tP, bv, idesc_pv, pacc);
          } else {
            for (int k = 0; k < pks; ++k)
              mma_ts_w(tO, tP + 8 * k, bv + (2048 >> 4) * k, idesc_pv, (pacc || k > 0) ? 1u : 0u);
          }
          mma_commit_w(&sm.o_done[x]);
          OD_TP(12 + x, 0, 0);
          ++npv;
          pon = 0;
          return true;
        };
#pragma unroll 1
        for (int i = i0; i < i1 && ok; i += istep) {
          const FwdItem2 it = fwd_item<kVarlen, kMode>(p, i);
          if (kVarlen && !it.valid[0]) continue;  // past the unit's length: no role touches it
          if (kRes && static_cast<int>(it.unit) != prev_unit) {
            if (prev_unit >= 0) {
              // every QK^T of the old unit is issued: its K stages go once those complete
              // (unless already released after the unit's last QK^T), its V stages once the
              // last P V (still pending) does
              if (!k_released)
                for (int s2 = 0; s2 < p.nkb; ++s2) mma_commit_w(&sm.k_empty[s2]);
              if (pon) ok = issue_pv();
              if (!ok) break;
              for (int s2 = 0; s2 < p.nkb; ++s2) mma_commit_w(&sm.v_empty[s2]);
            }
            ++unit_loads;
            prev_unit = static_cast<int>(it.unit);
            k_released = false;
            // observe the new fills before this issuer can ever release them
            for (int s2 = 0; s2 < p.nkb && ok; ++s2)
              ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[s2], (unit_loads - 1) & 1u, ctl, status, 15) &&
                                           wait_bar(&sm.v16_ready[s2], (unit_loads - 1) & 1u, ctl, status, 16));
            if (!ok) break;
          }
          const int lo = x ? it.lo[1] : it.lo[0];
          const int nb = (x ? it.valid[1] : it.valid[0]) ? (x ? it.hi[1] : it.hi[0]) - lo + 1 : 0;
          const int nload = it.uhi - it.ulo + 1;  // streaming: fills of this item
          if (nb == 0 && pon) {
            // no rows of this tile here: issue the pending P V now, so that its stage is not
            // held while the other tile works through this item's fills
            const int rel = pst;
            ok = issue_pv();
            if (!ok) break;
            if (!kRes) mma_commit_w(&sm.v_empty[rel]);
          }
          int qs = 0;
#pragma unroll 1
          for (int s = 0; s < nb && ok; ++s) {
            const int blk = lo + s;
            const FwdSlot f = fwd_slot<kRes>(blk, blk - it.ulo, unit_loads, stream_cnt);
            if (s == 0) {
              qs = qn & 1;
              ok = __all_sync(0xffffffffu, wait_bar(&sm.q_full[x][qs], (qn >> 1) & 1u, ctl, status, 12));
              if (!ok) break;
              ++qn;
            }
            ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[f.stage], f.parity, ctl, status, 13) &&
                                         (nqk == 0 || wait_bar(&sm.s_taken[x], (nqk - 1) & 1u, ctl, status, 14)));
            if (!ok) break;
            tc_fence_after();
            const int n = round16(fwd_ncols<kMode>(p, it, blk));
            const uint64_t a = dq0 + static_cast<uint64_t>(qs * (kTile >> 4));
            const uint64_t b = dk0 + static_cast<uint64_t>(f.stage * (kFwdKVTile >> 4));
            mma_ss_k64_w(tS, a, b, idesc_bf16(128, n, 0, 0));
            mma_commit_w(&sm.s_full[x]);
            OD_TP(10 + x, i, s);
            ++nqk;
            if (s == nb - 1) {
              mma_commit_w(&sm.q_empty[x][qs]);
              // resident: after the unit's last QK^T its K stages may take the next unit's
              // keys while the last blocks' softmax and P V still run
              // (fixed-length space calls only: there every item is processed, so the next
              // item of this CTA tells whether the unit ends here; for time attention releasing
              // at the unit change measured faster)
              if (kRes && !kVarlen && kMode == kModeSpace && (i + istep >= i1 || fwd_item<kVarlen, kMode>(p, i + istep).unit != it.unit)) {
                for (int s2 = 0; s2 < p.nkb; ++s2) mma_commit_w(&sm.k_empty[s2]);
                k_released = true;
              }
            }
            // streaming: this fill's K may be reloaded once both tiles' QK^T complete
            if (!kRes) mma_commit_w(&sm.k_empty[f.stage]);
            if (pon) {
              const int rel = pst;
              ok = issue_pv();
              if (!ok) break;
              if (!kRes) mma_commit_w(&sm.v_empty[rel]);
            }
            pon = 1;
            pst = f.stage;
            pvp = f.parity;
            pks = n >> 4;
            pacc = s > 0;
          }
          if (!ok) break;
          if (!kRes) {
            // fills of the item this tile did not use (no rows here, or, packed, the other
            // tile's block): observe and release them
            for (int s = 0; s < nload && ok; ++s) {
              if (s >= lo - it.ulo && s < lo - it.ulo + nb) continue;
              const FwdSlot f = fwd_slot<kRes>(it.ulo + s, s, unit_loads, stream_cnt);
              ok = __all_sync(0xffffffffu, wait_bar(&sm.k_full[f.stage], f.parity, ctl, status, 15) &&
                                           wait_bar(&sm.v16_ready[f.stage], f.parity, ctl, status, 16));
              if (!ok) break;
              mma_commit_w(&sm.k_empty[f.stage]);
              mma_commit_w(&sm.v_empty[f.stage]);
            }
            if (!ok) break;
            stream_cnt += nload;
          }
        }
        if (ok && pon) {
          const int rel = pst;
          ok = issue_pv();
          if (ok && !kRes) mma_commit_w(&sm.v_empty[rel]);
        }
        // wait until every MMA issued by this warp has completed before TMEM is freed
        mma_commit_w(&sm.drain[x]);
        drain_wait(&sm.drain[x], 0);
      }
    } else {
      // ---------------------------------------------------------- V converters (warps 10, 11)
      // P V runs in fp16: P in [0, 256] loses 8x less to rounding than in bf16.  Each V fill
      // is rewritten in place as fp16(v * 2^e): e = 0 when its magnitude is inside a safe fp16
      // range (2^-10 <= max|v| <= 2^15, or all zero), else the power of two that brings max|v|
      // into [2^14, 2^15) (the softmax rescales O when e changes between blocks and divides it
      // out at the end).
      long long prev_unit = -1;
      uint32_t unit_loads = 0, stream_cnt = 0;
      bool ok = true;
      auto convert = [&](int stage, uint32_t parity) -> bool {
        bool w = wait_bar(&sm.v_full[stage], parity, ctl, status, 6);
        if (!__all_sync(0xffffffffu, w)) return false;
        uint4* chunk = reinterpret_cast<uint4*>(sV + stage * kFwdKVTile);
        const int n16 = p.kvb * 8;  // 16-byte chunks holding keys
        float mx = 0.f;
#pragma unroll 4
        for (int jj = lane; jj < n16; jj += 32) {
          const uint4 d = chunk[jj];
          const uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            mx = fmaxf(mx, fabsf(__uint_as_float(wv[h] << 16)));
            mx = fmaxf(mx, fabsf(__uint_as_float(wv[h] & 0xFFFF0000u)));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const bool in_range = !(mx == mx) || mx == 0.f || (mx >= 0.0009765625f && mx <= 32768.f);
        int e = 0;
        if (!in_range) {
          // finite max|v| outside the range: 2^E <= mx < 2^(E+1), e = 14 - E (clamped)
          const int E = (mx < 1.17549435e-38f) ? -126 : static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
          e = (E == 128) ? 0 : min(max(14 - E, -60), 60);
        }
        const float2 sc = make_float2(__int_as_float((127 + (e >> 1)) << 23), __int_as_float((127 + e - (e >> 1)) << 23));
#pragma unroll 4
        for (int jj = lane; jj < n16; jj += 32) {
          const uint4 d = chunk[jj];
          uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float2 f2 = make_float2(__uint_as_float(wv[h] << 16), __uint_as_float(wv[h] & 0xFFFF0000u));
            if (e != 0) {  // two exact power-of-two steps (each within the normal range)
              f2 = __fmul2_rn(f2, make_float2(sc.x, sc.x));
              f2 = __fmul2_rn(f2, make_float2(sc.y, sc.y));
            }
            wv[h] = pack_f16x2(f2.x, f2.y);
          }
          chunk[jj] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        if (lane == 0) sm.vexp[stage] = e;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.v16_ready[stage]);
        OD_TP(30, stage, 0);
        return true;
      };
#pragma unroll 1
    for (int i = i0; i < i1 && ok; i += istep) {
        const FwdItem2 it = fwd_item<kVarlen, kMode>(p, i);
        if (kVarlen && !it.valid[0]) continue;  // past the unit's length: no role touches it
        if (kRes) {
          if (it.unit != prev_unit) {
            ++unit_loads;
            prev_unit = it.unit;
            for (int st = 0; st < p.nkb && ok; ++st) ok = convert(st, (unit_loads - 1) & 1u);
          }
        } else {
          const int nb = it.uhi - it.ulo + 1;
          for (int s = 0; s < nb && ok; ++s) {
            const uint32_t c = stream_cnt + s;
            ok = convert(static_cast<int>(c % kFwdStages), (c / kFwdStages) & 1u);
          }
          stream_cnt += nb;
        }
      }
    }
  } else {
    regs_inc<kFwdSoftmaxRegs>();
    // ------------------------------------------------------------ softmax warpgroups
    const int x = warp >> 2;                // 0: tile A, 1: tile B
    const int r = (warp & 3) * 32 + lane;   // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tX = tmem + 256u * x + lane_off;
    const uint32_t tS = tX, tP = tX + 128u, tO = tX + 192u;
    const int G = p.G;
    const int rr = r / G;
    const int g = r - rr * G;
    // sequence position within the tile; packed: timestep and token position within the tile
    const int tokr = kMode == kModeTimePacked ? rr / p.pk : rr;
    const int spr = kMode == kModeTimePacked ? rr - tokr * p.pk : 0;
    const bool packed = kMode == kModeTimePacked;
    uint32_t jS = 0, jP = 0, waited = 0, jE = 0;
    int prev_unit = -1;
    uint32_t unit_loads = 0, stream_next = 0;
    bool ok = true;
    const float2 sl2 = make_float2(p.sl, p.sl);
#pragma unroll 1
    for (int i = i0; i < i1 && ok; i += istep) {
      const FwdItem2 it = fwd_item<kVarlen, kMode>(p, i);
      if (kVarlen && !it.valid[0]) continue;  // past the unit's length: no role touches it
      if (kRes && static_cast<int>(it.unit) != prev_unit) {
        ++unit_loads;
        prev_unit = static_cast<int>(it.unit);
      }
      const uint32_t stream_cnt = stream_next;
      if (!kRes) stream_next += it.uhi - it.ulo + 1;
      if (!(x ? it.valid[1] : it.valid[0])) continue;
      // (the block loop keeps only what it needs; the epilogue decodes the item again)
      const int lo = x ? it.lo[1] : it.lo[0];
      const int nb = (x ? it.hi[1] : it.hi[0]) - lo + 1;
      const int key_hi = it.key_hi;
      const int pos = packed ? tokr : (x ? it.tok0[1] : it.tok0[0]) + tokr;  // query timestep / token
      float m_used = -INFINITY, l = 0.f;
      int e_cur = 0;  // O holds sum P fp16(V 2^e_cur)
#pragma unroll 1
      for (int s = 0; s < nb; ++s) {
        const int blk = lo + s;
        const int ncols = kMode == kModeTimePacked ? p.kvb : min(kFwdBN, key_hi - blk * kFwdBN);
        const int nch = (ncols + 31) >> 5;
        // allowed columns of this row: lo_c <= c < hi_c, c != ex, and (packed) c mod pk == spr
        int lo_c, hi_c, ex = -1;
        if (kMode == kModeSpace) {
          const int kbase = blk * kFwdBN;
          lo_c = 0;
          hi_c = ncols;
          if (p.agent >= kbase && p.agent < kbase + kFwdBN && pos != p.agent) ex = p.agent - kbase;
        } else if (kMode == kModeTime) {
          const int kbase = blk * kFwdBN;
          lo_c = pos - p.window + 1 - kbase;
          hi_c = min(ncols, pos + 1 - kbase);
        } else {
          lo_c = (pos - p.window + 1) * p.pk;
          hi_c = min(ncols, (pos + 1) * p.pk);
        }
        const bool need = packed || lo_c > 0 || hi_c < (nch << 5) || ex >= 0;
        ok = __all_sync(0xffffffffu, wait_bar(&sm.s_full[x], jS & 1u, ctl, status, 20));
        if (!ok) break;
        OD_TP(1, i, s);
        ++jS;
        tc_fence_after();
        float v[128];
        tmem_ld32(tS, v);
        if (nch > 1) tmem_ld32(tS + 32, v + 32);
        if (nch > 2) tmem_ld32(tS + 64, v + 64);
        if (nch > 3) tmem_ld32(tS + 96, v + 96);
        tmem_wait_ld_dep32(v);
        reg_dep32(v + 32);
        reg_dep32(v + 64);
        reg_dep32(v + 96);
        OD_TP(7, i, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_taken[x]);
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (ch < nch) {
              uint32_t keep = keep_bits32(32 * ch, lo_c, hi_c, ex);
              if (packed) {
                // first column c >= 32 ch with c mod pk == spr
                keep &= stride_bits32((spr - (32 * ch) % p.pk + p.pk) % p.pk, p.pk);
              }
              if (__any_sync(0xffffffffu, keep != 0xFFFFFFFFu)) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[32 * ch + j] = ((keep >> j) & 1u) ? v[32 * ch + j] : -INFINITY;
              }
            }
          }
        }
        float mb = max32(v);
        if (nch > 1) mb = fmaxf(mb, max32(v + 32));
        if (nch > 2) mb = fmaxf(mb, max32(v + 64));
        if (nch > 3) mb = fmaxf(mb, max32(v + 96));
        const float mnew = mb * p.sl;
        float alpha = 1.f;
        bool rescale = false;
        if (mb != -INFINITY && (m_used == -INFINITY || mnew > m_used + kRescaleThreshold)) {
          if (m_used != -INFINITY) {
            alpha = ex2(m_used - mnew);
            rescale = s > 0;
          }
          m_used = mnew;
          l *= alpha;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        OD_TP(8, i, s);
        // the V stage's scale exponent (its keys hold fp16(v * 2^e)); O is kept in the
        // scale of the item's latest block and rescaled when that changes
        const FwdSlot fs = fwd_slot<kRes>(blk, blk - it.ulo, unit_loads, stream_cnt);
        ok = __all_sync(0xffffffffu, wait_bar(&sm.v16_ready[fs.stage], fs.parity, ctl, status, 22));
        if (!ok) break;
        const int ev = sm.vexp[fs.stage];
        const int de = s > 0 ? ev - e_cur : 0;
        e_cur = ev;
        // P is single-buffered and O may need a rescale: both wait for the previous P V
        if (jP > waited) {
          ok = __all_sync(0xffffffffu, wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status, 21));
          if (!ok) break;
          waited = jP;
          tc_fence_after();
        }
        OD_TP(2, i, s);
        if (__any_sync(0xffffffffu, rescale || de != 0)) {
          const float f = (rescale ? alpha : 1.f) * __int_as_float((127 + de) << 23);
#pragma unroll 1
          for (int q = 0; q < 8; ++q) {
            uint32_t o[8];
            tmem_ld8(tO + 8 * q, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            tmem_st8(tO + 8 * q, o);
          }
        }
        const float2 nm2 = make_float2(-msub, -msub);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if (ch < nch) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t pk[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int c = 32 * ch + 16 * hh + 2 * j;
                const float2 xx = __ffma2_rn(make_float2(v[c], v[c + 1]), sl2, nm2);
                const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
                if (j & 1) acc1 = __fadd2_rn(acc1, pp); else acc0 = __fadd2_rn(acc0, pp);
                pk[j] = pack_f16x2(pp.x, pp.y);
              }
              tmem_st8(tP + 16 * ch + 8 * hh, pk);
            }
          }
        }
        {
          const float2 a = __fadd2_rn(acc0, acc1);
          l += a.x + a.y;
        }
        OD_TP(3, i, s);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[x]);
        OD_TP(4, i, s);
        ++jP;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // Space attention does what does not need O first (the item's last P V is still
      // running); for time attention waiting first measured faster.
      constexpr bool kLateWait = kMode == kModeSpace;
      if (!kLateWait && jP > waited) {
        ok = __all_sync(0xffffffffu, wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status, 23));
        if (!ok) break;
        waited = jP;
      }
      const FwdItem2 it2 = fwd_item<kVarlen, kMode>(p, i);
      const int tok0x = x ? it2.tok0[1] : it2.tok0[0];
      const int spos = packed ? tok0x + spr : 0;        // packed: token position
      const bool row_ok = (r < p.rows) && (packed ? spos < p.S : pos < it2.L);
      // 1 / l, and the V scale of the last block divided out (exact power of two)
      const float inv = l > 0.f ? (1.f / l) * __int_as_float((127 - e_cur) << 23) : 0.f;
      const int hq = it2.kvh * G + g;
      long long row;
      if (kMode == kModeSpace)
        row = ((static_cast<long long>(it2.b) * p.T + it2.fixed) * p.S + pos) * p.Hq + hq;
      else if (kMode == kModeTime)
        row = ((static_cast<long long>(it2.b) * p.T + pos) * p.S + it2.fixed) * p.Hq + hq;
      else
        row = ((static_cast<long long>(it2.b) * p.T + pos) * p.S + spos) * p.Hq + hq;
      // (row_w: row_ok, and in debug builds also the row inside the output)
      const bool row_w =
          row_ok && OD_IN_RANGE(row, static_cast<long long>(p.B) * p.T * p.S * p.Hq, status, 202);
      if (row_w) p.lse[row] = (m_used + log2f(l)) * 0.69314718055994531f;
      const bool want_lo = p.o_lo != nullptr;
      if (!kVarlen) {
        // stage the tile's rows (128 bytes each, 16-byte chunk c of row r at c ^ (r & 7): the
        // 128-byte TMA swizzle), then the tile's first thread stores the box once all 4 warps
        // have arrived.  The staging is reused an item later, after that thread has seen the
        // previous stores read it.
        const bool issuer = (warp & 3) == 0 && lane == 0;
        if (jE > 0) {
          if (issuer) {
            bulk_wait_read0();
            mbar_arrive(&sm.st_free[x]);
          }
          ok = __all_sync(0xffffffffu, wait_bar(&sm.st_free[x], (jE - 1) & 1u, ctl, status, 24));
          if (!ok) break;
        }
      }
      if (jP > waited) {
        ok = __all_sync(0xffffffffu, wait_bar(&sm.o_done[x], (jP - 1) & 1u, ctl, status, 23));
        if (!ok) break;
        waited = jP;
      }
      OD_TP(5, i, 0);
      tc_fence_after();
      uint8_t* so = sOst + x * kTile + r * 128;
      uint8_t* sl = sLst + x * kTile + r * 128;
      uint4* gdst = reinterpret_cast<uint4*>(p.o + (row_w ? row : 0) * 64);
      uint4* gdlo = want_lo ? reinterpret_cast<uint4*>(p.o_lo + (row_w ? row : 0) * 64) : nullptr;
      // (fixed-length space attention loads the whole row at once, the other modes in
      // quarters: each measured faster for its mode)
      if (kMode == kModeSpace && !kVarlen) {
        float o[64];
        tmem_ld32(tO, o);
        tmem_ld32(tO + 32, o + 32);
        tmem_wait_ld_dep32(o);
        reg_dep32(o + 32);
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk) {  // 16-byte chunk (8 columns) of the row
          uint32_t w[4], wl[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 y = __fmul2_rn(make_float2(o[8 * chunk + 2 * j], o[8 * chunk + 2 * j + 1]),
                                        make_float2(inv, inv));
            w[j] = split_bf16x2(y.x, y.y, &wl[j]);
          }
          const int sc = chunk ^ (r & 7);
          *reinterpret_cast<uint4*>(so + sc * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          if (want_lo) *reinterpret_cast<uint4*>(sl + sc * 16) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      } else
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t o16[16];
        tmem_ld16(tO + 16 * q4, reinterpret_cast<float*>(o16));
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int chunk = 2 * q4 + cc;  // 16-byte chunk (8 columns) of the row
          const uint32_t* o = o16 + 8 * cc;
          uint32_t w[4], wl[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 y = __fmul2_rn(make_float2(__uint_as_float(o[2 * j]), __uint_as_float(o[2 * j + 1])),
                                        make_float2(inv, inv));
            w[j] = split_bf16x2(y.x, y.y, &wl[j]);
          }
          if (!kVarlen) {
            const int sc = chunk ^ (r & 7);
            *reinterpret_cast<uint4*>(so + sc * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            if (want_lo) *reinterpret_cast<uint4*>(sl + sc * 16) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          } else if (row_w) {
            gdst[chunk] = make_uint4(w[0], w[1], w[2], w[3]);
            if (want_lo) gdlo[chunk] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          }
        }
      }
      if (!kVarlen) {
        fence_proxy_async_smem();  // the staged rows, visible to the TMA stores
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.st_full[x]);
        if ((warp & 3) == 0) {
          ok = __all_sync(0xffffffffu, wait_bar(&sm.st_full[x], jE & 1u, ctl, status, 25));
          if (!ok) break;
          if (lane == 0) {
            const int c1 = it2.kvh * G;
            int c2, c3;
            if (kMode == kModeSpace) { c2 = tok0x; c3 = it2.fixed; }
            else if (kMode == kModeTime) { c2 = it2.fixed; c3 = tok0x; }
            else { c2 = tok0x; c3 = 0; }
            if (OD_TMA_OK(c1, c2, c3, it2.b, p.Hq, p.S, p.T, p.B, status, 203)) {
              tma_store_5d(&tm_o, sOst + x * kTile, 0, c1, c2, c3, it2.b);
              if (want_lo) tma_store_5d(&tm_lo, sLst + x * kTile, 0, c1, c2, c3, it2.b);
            }
            bulk_commit();
          }
          __syncwarp();
        }
        ++jE;
      }
      OD_TP(6, i, 0);
    }
  }

  OD_TRACE_END();
  // output stores issued by this thread: complete before the CTA's shared memory goes
  if (!kVarlen && warp < 8 && (warp & 3) == 0 && lane == 0) bulk_wait0();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace od
