// od_common.cuh -- definitions shared by the query-stationary kernels (sm_103a).
//
// A unit is one (b, t, kv head) for space attention or one (b, s, kv head) for time
// attention; its sequence of L positions (S tokens of one timestep block, or T timesteps at
// one token position) is cut into Q tiles of nTok = floor(128 / G) positions x G query heads
// (rows r = tok * G + g, one 5-D TMA box), and its keys into blocks of `bn` keys.  A work item
// is (unit, pair of consecutive Q tiles A and B).
#pragma once
#include <cuda.h>
#include "od_ptx.cuh"

// Timeline trace points, compiled out unless OD_TRACE is defined.  A profiling build
// (nvcc -DOD_TRACE) records, for one kernel at a time (g_od_trace_sel, set by
// od_trace_select: 0 forward, 1 dQ pass, 2 dK/dV, 3 Delta pass), for the CTA with index
// OD_TRACE_CTA only and lane 0 of each warp, one 64-bit record per trace point into that
// warp's own region of OD_TRACE_PER_WARP records: the low 32 bits of the SM clock and a word
// (event << 18) | (a & 0x3FF) << 8 | (b & 0xFF).  The record count lives in a register
// (OD_TRACE_INIT declares it; OD_TRACE_END publishes it), so a trace point costs a clock read
// and one store.  od_trace_read (C ABI, same build) copies the regions out; the records show
// where each warp role waits.
#ifdef OD_TRACE
#ifndef OD_TRACE_CTA
#define OD_TRACE_CTA 7
#endif
#define OD_TRACE_WARPS 32
#define OD_TRACE_PER_WARP 8192
__device__ unsigned long long g_od_trace[OD_TRACE_WARPS * OD_TRACE_PER_WARP];
__device__ unsigned int g_od_trace_n[OD_TRACE_WARPS];
__device__ int g_od_trace_sel;
__device__ __forceinline__ void od_trace(unsigned int& n, bool on, int ev, int a, int b) {
  if (on && blockIdx.x == OD_TRACE_CTA && (threadIdx.x & 31) == 0 && n < OD_TRACE_PER_WARP) {
    const unsigned long long clk = static_cast<unsigned int>(clock64());
    const unsigned int w = (static_cast<unsigned int>(ev & 0xFF) << 18) |
                           (static_cast<unsigned int>(a & 0x3FF) << 8) | static_cast<unsigned int>(b & 0xFF);
    g_od_trace[(threadIdx.x >> 5) * OD_TRACE_PER_WARP + n] = (clk << 32) | w;
  }
  ++n;
}
#define OD_TP(ev, a, b) od_trace(od_tn, od_ton, (ev), (a), (b))
#define OD_TRACE_INIT(kid) \
  unsigned int od_tn = 0;  \
  const bool od_ton = g_od_trace_sel == (kid)
#define OD_TRACE_END()                                                                   \
  do {                                                                                   \
    if (od_ton && blockIdx.x == OD_TRACE_CTA && (threadIdx.x & 31) == 0)                 \
      g_od_trace_n[threadIdx.x >> 5] = od_tn < OD_TRACE_PER_WARP ? od_tn : OD_TRACE_PER_WARP; \
  } while (0)
#else
#define OD_TP(ev, a, b) ((void)0)
#define OD_TRACE_INIT(kid) ((void)0)
#define OD_TRACE_END() ((void)0)
#endif

namespace od {

constexpr int kBM = 128;           // query rows per tile (MMA M)
constexpr int kTile = 128 * 128;   // bytes of one Q tile: 128 rows x 64 16-bit elements
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// The 384-thread layout of the backward kernels: warps 0-7 elementwise (two warpgroups),
// 8-11 control; launched with kQsLaunchRegs registers, then rebalanced per warpgroup.
constexpr int kQsLaunchRegs = 168;
constexpr int kQsSoftmaxRegs = 200;
constexpr int kQsCtrlRegs = 104;
constexpr int kQsProducerWarp = 8;
constexpr int kQsMmaWarp = 9;

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
  int bn;         // keys per key block
  int nkb;        // key blocks per unit
  // packed time attention (short sequences, G T <= 64): a Q tile holds pk token positions x
  // all T frames x G heads, rows (t pk + sp) G + g, and its key block the same positions'
  // T frames, keys t pk + sp; query (t, sp) reads key (t', sp') iff sp' == sp and
  // t - window < t' <= t.  A unit is (b, 2 pk positions, kv head): tile x holds positions
  // [unit's first + x pk, + pk) and reads key block x only.  0: not packed.
  int pk;
  int kvb;        // keys a K/V block load brings in: bn, or pk T when packed
  int resident;   // nkb <= K/V stages: the unit's K/V stay in smem across its items
  // reciprocals for the item decode: floor(2^64 / d) + 1 for d = npairs, Hkv, F (0 when
  // d >= 2^16, where the plain division is used)
  unsigned long long rcp_npairs, rcp_hkv, rcp_f;
  // space attention with variable-length timestep blocks: block (b, t) holds its first
  // seqlen[b * T + t] tokens (clamped to [0, S]); the rest of the S slots are padding that
  // is neither read as a key nor written as a query row.  NULL: every block holds S tokens.
  const int* seqlen;
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;   // optional: O - bf16(O), rounded to bf16 (for the backward's Delta)
  int tma_out;           // forward: O (and O_lo) leave by TMA store of staged tile halves
  float* lse;
  unsigned int* status;
};

struct FwdItem {
  uint32_t unit;
  int b, fixed, kvh;
  int L;               // the unit's sequence length (p.L, or its block's length)
  int tok0[2];
  int validA;          // 0: tile A starts past the unit's length -- nothing to do
  int validB;
  int key_lo, key_hi;  // allowed key positions of the item lie in [key_lo, key_hi)
  int kb_lo, kb_hi;    // inclusive key-block range of the item
  int blo[2], bhi[2];  // inclusive key-block range of tile x
};

// n / d for n < 2^32 and 1 < d < 2^16 with rcp = floor(2^64 / d) + 1: the product's error
// term n (rcp d - 2^64) / (d 2^64) stays below n / 2^64 < 1 / d, so the high word is exact.
__device__ __forceinline__ uint32_t div_rcp(uint32_t n, uint32_t d, unsigned long long rcp) {
  if (rcp == 0ull) return n / d;
  return static_cast<uint32_t>(__umul64hi(static_cast<unsigned long long>(n), rcp));
}
// Host side: the reciprocal div_rcp expects (0 selects the plain division).
inline unsigned long long host_div_rcp(int d) {
  if (d <= 1 || d >= 65536) return 0ull;
  return (~0ull) / static_cast<unsigned long long>(d) + 1ull;
}

// kVarlen: space attention over variable-length blocks (p.seqlen); false compiles the
// fixed-length decode with no trace of the per-unit length.
template <bool kVarlen, bool kPacked = false>
__device__ __forceinline__ FwdItem fwd_decode(const FwdParams& p, long long i) {
  // the host guarantees nitems < 2^31, so 32-bit unsigned division suffices
  FwdItem it;
  const uint32_t ii = static_cast<uint32_t>(i);
  const uint32_t unit = div_rcp(ii, static_cast<uint32_t>(p.npairs), p.rcp_npairs);
  const int pair = static_cast<int>(ii - unit * static_cast<uint32_t>(p.npairs));
  it.unit = unit;
  const uint32_t r = div_rcp(unit, static_cast<uint32_t>(p.Hkv), p.rcp_hkv);
  it.kvh = static_cast<int>(unit - r * static_cast<uint32_t>(p.Hkv));
  const uint32_t bq = div_rcp(r, static_cast<uint32_t>(p.F), p.rcp_f);
  it.fixed = static_cast<int>(r - bq * static_cast<uint32_t>(p.F));
  it.b = static_cast<int>(bq);
  if (kPacked && p.pk) {  // packed time attention: `fixed` counts groups of 2 pk positions
    it.L = p.L;
    it.tok0[0] = it.fixed * 2 * p.pk;
    it.tok0[1] = it.tok0[0] + p.pk;
    it.validA = 1;
    it.validB = it.tok0[1] < p.S;
    it.key_lo = 0;
    it.key_hi = 2 * p.kvb;
    it.kb_lo = 0;
    it.kb_hi = it.validB ? 1 : 0;
    it.blo[0] = it.bhi[0] = 0;
    it.blo[1] = it.bhi[1] = 1;
    return it;
  }
  int L = p.L;
  if (kVarlen) L = min(max(__ldg(p.seqlen + static_cast<long long>(it.b) * p.T + it.fixed), 0), p.L);
  it.L = L;
  const int tA = 2 * pair;
  it.tok0[0] = tA * p.nTok;
  it.tok0[1] = (tA + 1) * p.nTok;
  it.validA = kVarlen ? it.tok0[0] < L : 1;
  it.validB = (tA + 1) < p.ntiles && (!kVarlen || it.tok0[1] < L);
  const int last = min(L, (it.validB ? tA + 2 : tA + 1) * p.nTok) - 1;
  if (p.is_time) {
    it.key_lo = max(0, it.tok0[0] - p.window + 1);
    it.key_hi = last + 1;
  } else {
    it.key_lo = 0;
    it.key_hi = L;
  }
  it.kb_lo = it.key_lo / p.bn;
  it.kb_hi = (!kVarlen || it.validA) ? (it.key_hi - 1) / p.bn : it.kb_lo - 1;  // none if skipped
  it.blo[0] = it.blo[1] = it.kb_lo;
  it.bhi[0] = it.bhi[1] = it.kb_hi;
  return it;
}

__device__ __forceinline__ int block_ncols(const FwdItem& it, int kb, int bn) {
  return min(bn, it.key_hi - kb * bn);
}
// Keys of block kb that the tile's rows may read (packed: the block's pk T keys).
template <bool kPacked>
__device__ __forceinline__ int block_keys(const FwdParams& p, const FwdItem& it, int kb, int bn) {
  return (kPacked && p.pk) ? p.kvb : block_ncols(it, kb, bn);
}

// Packed time attention, one query row (frame t, position sp within the tile): bit j set
// <=> key c0 + j = t' pk + sp with tlo <= t' <= thi.
__device__ __forceinline__ uint32_t keep_bits_packed(int c0, int pk, int sp, int tlo, int thi) {
  uint32_t m = 0u;
  for (int tt = max(tlo, (c0 - sp + pk - 1) / pk); tt <= thi; ++tt) {
    const int c = tt * pk + sp - c0;
    if (c >= 32) break;
    m |= 1u << c;
  }
  return m;
}
// Packed time attention, one key (frame t', position spk within the block): bit j set <=>
// row r0 + j = (t pk + spk) G + g with tlo <= t <= thi and 0 <= g < G.
__device__ __forceinline__ uint32_t keep_rows_packed(int r0, int G, int pk, int spk, int tlo, int thi) {
  uint32_t m = 0u;
  const int d = r0 / G - spk;   // frames before this one hold rows below r0
  for (int tt = max(tlo, d > 0 ? d / pk : 0); tt <= thi; ++tt) {
    const int c = (tt * pk + spk) * G - r0;   // the frame's G rows are [c, c + G)
    if (c >= 32) break;
    const int lo = max(c, 0), hi = min(c + G, 32);
    if (lo < hi) m |= (hi == 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
  }
  return m;
}
__device__ __forceinline__ int round16(int x) { return (x + 15) & ~15; }

// K/V stage and phase parity of block index bi (0-based within the item).
struct KvSlot {
  int stage;
  uint32_t parity;
};
__device__ __forceinline__ KvSlot kv_slot(const FwdParams& p, const FwdItem& it, int bi,
                                          uint32_t unit_loads, uint32_t stream_cnt, int stages) {
  KvSlot s;
  if (p.resident) {
    s.stage = it.kb_lo + bi;
    s.parity = (unit_loads - 1) & 1u;
  } else {
    const uint32_t c = stream_cnt + bi;
    s.stage = static_cast<int>(c % static_cast<uint32_t>(stages));
    s.parity = (c / static_cast<uint32_t>(stages)) & 1u;
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


}  // namespace od
