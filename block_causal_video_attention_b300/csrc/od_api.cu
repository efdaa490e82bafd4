// od_api.cu -- host side of the C ABI declared in include/od_attn.h.
//
// Validates arguments, encodes the TMA tensor maps for the [B,T,S,H,D] tensors, sizes the
// persistent grid to the SM count and launches on the caller's stream.  No allocation,
// no synchronisation on the launch path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "od_attn.h"
#include "od_fwd.cuh"
#include "od_bwd.cuh"
#include "od_decode.cuh"

// Device status words: [0] has bit OD_DEV_TIMEOUT set by any kernel whose bounded wait
// expired; [1] holds the first such wait's site word (site << 24 | parity << 23 | block).
__device__ unsigned int g_od_status[2];

namespace od {
// Exercises the failure path of the bounded waits: one warp waits on an mbarrier that nothing
// ever arrives on, gives up after the wait limit, records the timeout (site 120) and returns.
constexpr int kSelftestSite = 120;
__global__ void od_selftest_wait_kernel(unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ Ctl ctl;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    ctl.abort = 0;
  }
  __syncthreads();
  (void)wait_bar(&bar, 0u, &ctl, status, kSelftestSite);
}
}  // namespace od

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int range_ctas = 0;    // resident CTAs of the K/V range kernel (one wave), <= kAmaxSlots
  unsigned int* status = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

od_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OD_ERR_CUDA;
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_od_status) != cudaSuccess) return OD_ERR_CUDA;
    d.status = static_cast<unsigned int*>(sp);
    // The forward kernel redistributes its launch registers between warpgroups (setmaxnreg);
    // that split is only valid for the register count it was designed for.
    const void* fwd_fns[7] = {
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<false, od::kModeSpace, true>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<false, od::kModeSpace, false>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<true, od::kModeSpace, true>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<true, od::kModeSpace, false>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<false, od::kModeTime, true>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<false, od::kModeTime, false>),
        reinterpret_cast<const void*>(od::od_attn_fwd_kernel<false, od::kModeTimePacked, false>)};
    for (const void* fn : fwd_fns) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(od::kFwdSmemBytes)) != cudaSuccess)
        return OD_ERR_CUDA;
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || fa.numRegs != od::kFwdLaunchRegs)
        return OD_ERR_CUDA;
    }
    if (od::bwd_setup() != cudaSuccess) return OD_ERR_CUDA;
    {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, od::od_bwd_kv_range_kernel,
                                                        od::kKvRangeThreads, 0) != cudaSuccess ||
          per_sm < 1)
        return OD_ERR_CUDA;
      d.range_ctas = per_sm * d.num_sms < od::kAmaxSlots ? per_sm * d.num_sms : od::kAmaxSlots;
    }
    if (cudaFuncSetAttribute(od::od_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(od::kDecSmemBytes)) != cudaSuccess)
      return OD_ERR_CUDA;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return OD_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return OD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

od_status check_shape(int B, int T, int S, int Hq, int Hkv, int D, float scale) {
  if (B <= 0 || T <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return OD_ERR_INVALID_ARG;
  if (Hq % Hkv) return OD_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OD_ERR_INVALID_ARG;
  if (D != 64) return OD_ERR_UNSUPPORTED;
  if (Hq / Hkv > 128) return OD_ERR_UNSUPPORTED;
  // each dimension first (so that the product below cannot wrap), then the bytes of one Q-like
  // tensor: tensor-map coordinates are 32-bit and the tensor must stay below 2^40 bytes
  if (B > 65535 || T > (1 << 24) || S > (1 << 24) || Hq > 65535) return OD_ERR_UNSUPPORTED;
  const unsigned __int128 bytes = static_cast<unsigned __int128>(B) * static_cast<unsigned>(T) *
                                  static_cast<unsigned>(S) * static_cast<unsigned>(Hq) *
                                  static_cast<unsigned>(D) * 2u;
  if (bytes >= (static_cast<unsigned __int128>(1) << 40)) return OD_ERR_UNSUPPORTED;
  return OD_OK;
}

// 5-D tensor map over a [B,T,S,H,D] view of `elem` bytes per element whose consecutive tokens
// (b, t, s) are `tok_rows` D-element rows apart (tok_rows = H for a contiguous tensor, more for
// a view into a packed QKV tensor).
od_status make_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int elem, int B,
                   int T, int S, int H, int D, const uint32_t box[5],
                   CUtensorMapSwizzle swizzle, int tok_rows) {
  cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)T,
                        (cuuint64_t)B};
  cuuint64_t strides[4];
  strides[0] = (cuuint64_t)D * elem;
  strides[1] = strides[0] * tok_rows;
  strides[2] = strides[1] * S;
  strides[3] = strides[2] * T;
  cuuint32_t bx[5] = {box[0], box[1], box[2], box[3], box[4]};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 5, const_cast<void*>(ptr), dims, strides, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OD_OK : OD_ERR_CUDA;
}

// qkv_rows: 0 for separate contiguous Q, K, V; else the D-element rows per token of the packed
// [B,T,S,Hq+2Hkv,D] tensor that q, k and v point into.
od_status launch_fwd(int is_time, const void* q, const void* k, const void* v, void* o, float* lse,
                     void* o_lo, int B, int T, int S, int Hq, int Hkv, int D, int agent,
                     int window, float scale, void* stream, int qkv_rows = 0,
                     const int* seqlen = nullptr) {
  if (!q || !k || !v || !o || !lse) return OD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (o_lo && !aligned16(o_lo)))
    return OD_ERR_INVALID_ARG;
  od_status st = check_shape(B, T, S, Hq, Hkv, D, scale);
  if (st != OD_OK) return st;
  if (is_time) {
    if (window < 1) return OD_ERR_INVALID_ARG;
  } else {
    if (agent < -1 || agent >= S) return OD_ERR_INVALID_ARG;
  }
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != OD_OK) return st;

  od::AttnFwdParams p{};
  p.B = B; p.T = T; p.S = S; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  // short time sequences: several token positions share a tile (G * T <= 64)
  const bool packed = is_time && p.G * T <= 64;
  p.mode = packed ? od::kModeTimePacked : (is_time ? od::kModeTime : od::kModeSpace);
  p.L = is_time ? T : S;
  p.agent = is_time ? -1 : agent;
  p.window = is_time ? window : 1;
  p.sl = scale * 1.4426950408889634f;
  if (packed) {
    p.pk = od::kBM / (p.G * T);
    p.nTok = T;
    p.rows = p.pk * T * p.G;
    p.F = (S + 2 * p.pk - 1) / (2 * p.pk);
    p.ntiles = 2;
    p.npairs = 1;
    p.nkb = 2;
    p.kvb = p.pk * T;
  } else {
    p.pk = 1;
    p.nTok = od::kBM / p.G;
    p.rows = p.nTok * p.G;
    p.F = is_time ? S : T;
    p.ntiles = (p.L + p.nTok - 1) / p.nTok;
    p.npairs = (p.ntiles + 1) / 2;
    p.nkb = (p.L + od::kFwdBN - 1) / od::kFwdBN;
    p.kvb = od::kFwdBN;
  }
  p.nitems = 1LL * B * p.F * Hkv * p.npairs;
  if (p.nitems >= (1LL << 31)) return OD_ERR_UNSUPPORTED;
  p.rcp_npairs = od::host_div_rcp(p.npairs);
  p.rcp_hkv = od::host_div_rcp(p.Hkv);
  p.rcp_f = od::host_div_rcp(p.F);
  p.resident = !packed && p.nkb <= od::kFwdStages;
  p.lse = lse;
  p.status = dev->status;

  uint32_t qbox[5], kbox[5];
  if (p.mode == od::kModeSpace) {
    const uint32_t qb[5] = {64, (uint32_t)p.G, (uint32_t)p.nTok, 1, 1};
    const uint32_t kb[5] = {64, 1, (uint32_t)od::kFwdBN, 1, 1};
    for (int i = 0; i < 5; ++i) { qbox[i] = qb[i]; kbox[i] = kb[i]; }
  } else if (p.mode == od::kModeTime) {
    const uint32_t qb[5] = {64, (uint32_t)p.G, 1, (uint32_t)p.nTok, 1};
    const uint32_t kb[5] = {64, 1, 1, (uint32_t)od::kFwdBN, 1};
    for (int i = 0; i < 5; ++i) { qbox[i] = qb[i]; kbox[i] = kb[i]; }
  } else {
    const uint32_t qb[5] = {64, (uint32_t)p.G, (uint32_t)p.pk, (uint32_t)T, 1};
    const uint32_t kb[5] = {64, 1, (uint32_t)p.pk, (uint32_t)T, 1};
    for (int i = 0; i < 5; ++i) { qbox[i] = qb[i]; kbox[i] = kb[i]; }
  }
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_lo = static_cast<__nv_bfloat16*>(o_lo);
  p.seqlen = is_time ? nullptr : seqlen;
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int q_rows = qkv_rows ? qkv_rows : Hq, kv_rows = qkv_rows ? qkv_rows : Hkv;
  if ((st = make_map(&tq, q, bf, 2, B, T, S, Hq, D, qbox, sw, q_rows)) ||
      (st = make_map(&tk, k, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)) ||
      (st = make_map(&tv, v, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)))
    return st;

  const long long grid = p.nitems < dev->num_sms ? p.nitems : dev->num_sms;
  // fixed-length calls write O (and O_lo) by TMA store of whole staged tiles (the Q tile's
  // box over the output, 128-byte swizzle)
  CUtensorMap to = tq, tlo = tq;
  p.tma_out = p.seqlen ? 0 : 1;
  if (p.tma_out) {
    if ((st = make_map(&to, o, bf, 2, B, T, S, Hq, D, qbox, sw, Hq))) return st;
    if (o_lo && (st = make_map(&tlo, o_lo, bf, 2, B, T, S, Hq, D, qbox, sw, Hq))) return st;
  }

  const dim3 g((unsigned)grid), blk(od::kFwdThreads);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
#define OD_FWD_LAUNCH(V, M, R) \
  od::od_attn_fwd_kernel<V, M, R><<<g, blk, od::kFwdSmemBytes, strm>>>(tq, tk, tv, to, tlo, p)
  const bool res = p.resident != 0;
  if (p.seqlen) {
    if (res) OD_FWD_LAUNCH(true, od::kModeSpace, true); else OD_FWD_LAUNCH(true, od::kModeSpace, false);
  } else if (p.mode == od::kModeSpace) {
    if (res) OD_FWD_LAUNCH(false, od::kModeSpace, true); else OD_FWD_LAUNCH(false, od::kModeSpace, false);
  } else if (p.mode == od::kModeTime) {
    if (res) OD_FWD_LAUNCH(false, od::kModeTime, true); else OD_FWD_LAUNCH(false, od::kModeTime, false);
  } else {
    // packed: every item is a new unit of 2 blocks; streaming them through the stages lets
    // the next item's blocks load while this one computes
    OD_FWD_LAUNCH(false, od::kModeTimePacked, false);
  }
#undef OD_FWD_LAUNCH
  return cudaGetLastError() == cudaSuccess ? OD_OK : OD_ERR_CUDA;
}

od_status launch_bwd(int is_time, const void* q, const void* k, const void* v, const void* o,
                     const void* o_lo, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     float* dq_f32, float* dk_f32, float* dv_f32, int B, int T, int S, int Hq,
                     int Hkv, int D, int agent, int window, float scale, void* workspace,
                     size_t workspace_bytes, void* stream, int qkv_rows = 0,
                     const int* seqlen = nullptr) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return OD_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, o_lo, lse, dout, dq, dk, dv, dq_f32, dk_f32, dv_f32, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return OD_ERR_INVALID_ARG;
  od_status st = check_shape(B, T, S, Hq, Hkv, D, scale);
  if (st != OD_OK) return st;
  if (is_time) {
    if (window < 1) return OD_ERR_INVALID_ARG;
  } else {
    if (agent < -1 || agent >= S) return OD_ERR_INVALID_ARG;
  }
  if (workspace_bytes < od::bwd_workspace_bytes(B, T, S, Hq, D)) return OD_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != OD_OK) return st;
  od::BwdArgs a;
  a.is_time = is_time;
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dq_f32 = dq_f32; a.dk_f32 = dk_f32; a.dv_f32 = dv_f32;
  a.B = B; a.T = T; a.S = S; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
  a.agent = is_time ? -1 : agent;
  a.window = is_time ? window : 1;
  a.scale = scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = dev->status;
  a.num_sms = dev->num_sms;
  cudaStream_t strm = a.stream;

  // shapes shared by both gradient kernels (forward tiling)
  od::FwdParams f{};
  f.B = B; f.T = T; f.S = S; f.Hq = Hq; f.Hkv = Hkv; f.G = Hq / Hkv;
  f.is_time = is_time;
  f.L = is_time ? T : S;
  f.F = is_time ? S : T;
  f.agent = is_time ? -1 : agent;
  f.window = is_time ? window : 1;
  f.sl = scale * 1.4426950408889634f;
  f.nTok = od::kBM / f.G;
  f.rows = f.nTok * f.G;
  f.ntiles = (f.L + f.nTok - 1) / f.nTok;
  f.npairs = (f.ntiles + 1) / 2;
  f.nitems = 1LL * B * f.F * Hkv * f.npairs;
  f.rcp_npairs = od::host_div_rcp(f.npairs);
  f.rcp_hkv = od::host_div_rcp(f.Hkv);
  f.rcp_f = od::host_div_rcp(f.F);
  f.bn = od::kBN;
  f.nkb = (f.L + od::kBN - 1) / od::kBN;
  f.resident = 0;
  f.seqlen = is_time ? nullptr : seqlen;
  f.status = dev->status;
  f.pk = 0;
  if (f.nitems >= (1LL << 31)) return OD_ERR_UNSUPPORTED;
  if (1LL * B * f.F * Hkv * ((f.L + od::kKvBN - 1) / od::kKvBN) >= (1LL << 31)) return OD_ERR_UNSUPPORTED;
  // Short time sequences (G T <= 64) are packed: a Q tile holds pk token positions x all T
  // frames (rows (t pk + sp) G + g) and its key block the same positions' frames.  The dQ
  // passes take pk with pk T <= kBN keys per block, the dK/dV kernel pk with pk T G <= 128.
  od::FwdParams fk = f;   // the dK/dV kernel's tiling
  f.kvb = od::kBN;
  fk.kvb = od::kKvBN;
  const int Gq = Hq / Hkv;
  if (is_time && Gq * T <= 64) {
    const int pk_dq = od::kBM / (Gq * T) < od::kBN / T ? od::kBM / (Gq * T) : od::kBN / T;
    if (pk_dq >= 2) {
      f.pk = pk_dq;
      f.F = (S + 2 * pk_dq - 1) / (2 * pk_dq);
      f.nTok = T;
      f.rows = pk_dq * T * Gq;
      f.ntiles = 2;
      f.npairs = 1;
      f.nitems = 1LL * B * f.F * Hkv;
      f.rcp_npairs = od::host_div_rcp(f.npairs);
      f.rcp_f = od::host_div_rcp(f.F);
      f.kvb = pk_dq * T;
      f.nkb = 2;
    }
    const int pk_kv = od::kBM / (Gq * T);
    fk.pk = pk_kv;
    fk.F = (S + pk_kv - 1) / pk_kv;
    fk.nTok = T;
    fk.rows = pk_kv * T * Gq;
    fk.ntiles = 1;
    fk.kvb = pk_kv * T;
  }

  float* delta = static_cast<float*>(workspace);
  float* amax = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         od::bwd_delta_bytes(B, T, S, Hq));
  const int num_ctas = dev->num_sms < od::kAmaxSlots ? dev->num_sms : od::kAmaxSlots;
  int amax_slots = 0, dq_slots = 0;
  const uint32_t qbox_space[5] = {64, (uint32_t)f.G, (uint32_t)f.nTok, 1, 1};
  const uint32_t qbox_time[5] = {64, (uint32_t)f.G, 1, (uint32_t)f.nTok, 1};
  const uint32_t qbox_packed[5] = {64, (uint32_t)f.G, (uint32_t)f.pk, (uint32_t)T, 1};
  const uint32_t* qbox = f.pk ? qbox_packed : (is_time ? qbox_time : qbox_space);
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tdo, tk, tv;
  const int q_rows = qkv_rows ? qkv_rows : Hq, kv_rows = qkv_rows ? qkv_rows : Hkv;
  if ((st = make_map(&tq, q, bf, 2, B, T, S, Hq, D, qbox, sw, q_rows)) ||
      (st = make_map(&tdo, dout, bf, 2, B, T, S, Hq, D, qbox, sw, Hq)))
    return st;
  {
    const uint32_t kbox_space[5] = {64, 1, (uint32_t)od::kBN, 1, 1};
    const uint32_t kbox_time[5] = {64, 1, 1, (uint32_t)od::kBN, 1};
    const uint32_t kbox_packed[5] = {64, 1, (uint32_t)f.pk, (uint32_t)T, 1};
    const uint32_t* kbox = f.pk ? kbox_packed : (is_time ? kbox_time : kbox_space);
    if ((st = make_map(&tk, k, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)) ||
        (st = make_map(&tv, v, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)))
      return st;
    od::DqParams dp{};
    dp.f = f;
    dp.lse = lse;
    dp.delta = delta;
    dp.scale = scale;
    dp.dq = static_cast<__nv_bfloat16*>(dq);
    dp.dq_rows = q_rows;
    dp.dq_f32 = dq_f32;
    dp.amax = amax;
    const long long grid = f.nitems < num_ctas ? f.nitems : num_ctas;
    amax_slots = static_cast<int>(grid);
    dq_slots = static_cast<int>(grid);
    dp.amax_slots = amax_slots;
    // 1. the K/V ranges (the dQ pass forms Delta from O and its residual when the forward
    // wrote it), else the Delta pass; 2. dQ
    if (o_lo) {
      od::KvRangeParams d{};
      d.k = static_cast<const __nv_bfloat16*>(k);
      d.v = static_cast<const __nv_bfloat16*>(v);
      d.ntok = 1LL * B * T * S;
      d.Hkv = Hkv; d.kv_rows = kv_rows;
      d.amax = amax;
      // one wave of resident CTAs: every CTA streams an equal share
      const long long dgrid = dev->range_ctas;
      amax_slots = static_cast<int>(dgrid);
      dp.amax_slots = amax_slots;
      dp.o = static_cast<const __nv_bfloat16*>(o);
      dp.o_lo = static_cast<const __nv_bfloat16*>(o_lo);
      od::od_bwd_kv_range_kernel<<<(unsigned)dgrid, od::kKvRangeThreads, 0, strm>>>(d);
    } else {
      if (f.seqlen)
        od::od_bwd_dq_kernel<true, true, false><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
      else if (f.pk)
        od::od_bwd_dq_kernel<true, false, true><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
      else
        od::od_bwd_dq_kernel<true, false, false><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
    }
    if (cudaGetLastError() != cudaSuccess) return OD_ERR_CUDA;
    if (f.seqlen)
      od::od_bwd_dq_kernel<false, true, false><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
    else if (f.pk)
      od::od_bwd_dq_kernel<false, false, true><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
    else
      od::od_bwd_dq_kernel<false, false, false><<<(unsigned)grid, od::kDqThreads, od::kDqSmemBytes, strm>>>(tq, tdo, tk, tv, dp);
    if (cudaGetLastError() != cudaSuccess) return OD_ERR_CUDA;
  }
  // 3. dK, dV
  {
    const uint32_t kbox_space[5] = {64, 1, (uint32_t)od::kKvBN, 1, 1};
    const uint32_t kbox_time[5] = {64, 1, 1, (uint32_t)od::kKvBN, 1};
    const uint32_t kbox_packed[5] = {64, 1, (uint32_t)fk.pk, (uint32_t)T, 1};
    const uint32_t* kbox = fk.pk ? kbox_packed : (is_time ? kbox_time : kbox_space);
    if ((st = make_map(&tk, k, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)) ||
        (st = make_map(&tv, v, bf, 2, B, T, S, Hkv, D, kbox, sw, kv_rows)))
      return st;
    if (fk.pk) {   // Q/dO tiles of pk token positions x all T frames
      const uint32_t qbox_kv[5] = {64, (uint32_t)fk.G, (uint32_t)fk.pk, (uint32_t)T, 1};
      if ((st = make_map(&tq, q, bf, 2, B, T, S, Hq, D, qbox_kv, sw, q_rows)) ||
          (st = make_map(&tdo, dout, bf, 2, B, T, S, Hq, D, qbox_kv, sw, Hq)))
        return st;
    } else if (f.pk) {   // the dQ passes used packed boxes: back to the forward's tiles
      const uint32_t* qb = is_time ? qbox_time : qbox_space;
      if ((st = make_map(&tq, q, bf, 2, B, T, S, Hq, D, qb, sw, q_rows)) ||
          (st = make_map(&tdo, dout, bf, 2, B, T, S, Hq, D, qb, sw, Hq)))
        return st;
    }
    od::KvParams kp{};
    kp.f = fk;
    kp.lse = lse;
    kp.delta = delta;
    kp.scale = scale;
    kp.nkb = fk.pk ? 1 : (fk.L + od::kKvBN - 1) / od::kKvBN;
    kp.nitems = 1LL * B * fk.F * Hkv * kp.nkb;
    kp.dk = static_cast<__nv_bfloat16*>(dk);
    kp.dv = static_cast<__nv_bfloat16*>(dv);
    kp.kv_rows = kv_rows;
    kp.dk_f32 = dk_f32;
    kp.dv_f32 = dv_f32;
    kp.amax = amax;
    kp.amax_slots = amax_slots;
    kp.dq_slots = dq_slots;
    kp.dd_slots = o_lo ? dq_slots : amax_slots;
    const long long grid = kp.nitems < num_ctas ? kp.nitems : num_ctas;
    if (f.seqlen)
      od::od_bwd_dkdv_kernel<true, false><<<(unsigned)grid, od::kKvThreads, od::kKvSmemBytes, strm>>>(tq, tdo, tk, tv, kp);
    else if (fk.pk)
      od::od_bwd_dkdv_kernel<false, true><<<(unsigned)grid, od::kKvThreads, od::kKvSmemBytes, strm>>>(tq, tdo, tk, tv, kp);
    else
      od::od_bwd_dkdv_kernel<false, false><<<(unsigned)grid, od::kKvThreads, od::kKvSmemBytes, strm>>>(tq, tdo, tk, tv, kp);
    if (cudaGetLastError() != cudaSuccess) return OD_ERR_CUDA;
  }
  return OD_OK;
}

// One rollout step of time attention over the ring-buffer KV cache [B,W,S,Hkv,64].
od_status launch_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, void* o, float* lse, int B, int S, int Hq, int Hkv, int D,
                        int window, long long t, float scale, void* stream) {
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o, lse};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return OD_ERR_INVALID_ARG;
  if (t < 0 || window < 1) return OD_ERR_INVALID_ARG;
  od_status st = check_shape(B, 1, S, Hq, Hkv, D, scale);
  if (st != OD_OK) return st;
  if (Hq / Hkv > 16) return OD_ERR_UNSUPPORTED;
  // cache coordinates (frames x positions x heads) and the unit count stay 32-bit
  if (window > (1 << 24)) return OD_ERR_UNSUPPORTED;
  if (static_cast<unsigned __int128>(B) * static_cast<unsigned>(window) * static_cast<unsigned>(S) *
              static_cast<unsigned>(Hkv) * static_cast<unsigned>(D) * 2u >=
          (static_cast<unsigned __int128>(1) << 40) ||
      1LL * B * S * Hkv >= (1LL << 31))
    return OD_ERR_UNSUPPORTED;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != OD_OK) return st;

  od::DecParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B; p.S = S; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.W = window;
  p.n_valid = static_cast<int>(t + 1 < window ? t + 1 : window);
  p.slot = static_cast<int>(t % window);
  p.nb = (p.n_valid + od::kDecBN - 1) / od::kDecBN;
  p.units = B * S * Hkv;
  p.sl = scale * 1.4426950408889634f;
  p.status = dev->status;

  // The window's frames are the slots 0 .. n_valid - 1; the map's frame extent is n_valid, so
  // the rows of a last partial block come back zero-filled instead of reading unused slots.
  CUtensorMap tk, tv;
  const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)S,
                              (cuuint64_t)p.n_valid, (cuuint64_t)B};
  cuuint64_t strides[4];
  strides[0] = (cuuint64_t)D * 2;
  strides[1] = strides[0] * Hkv;
  strides[2] = strides[1] * S;
  strides[3] = strides[2] * window;
  const cuuint32_t box[5] = {64, 1, 1, (cuuint32_t)od::kDecBN, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  for (int which = 0; which < 2; ++which) {
    CUresult r = g_encode(which ? &tv : &tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                          which ? v_cache : k_cache, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return OD_ERR_CUDA;
  }
  const long long warps_needed = p.units;
  long long grid = (warps_needed + od::kDecWarps - 1) / od::kDecWarps;
  if (grid > dev->num_sms) grid = dev->num_sms;
  od::od_decode_kernel<<<(unsigned)grid, od::kDecThreads, od::kDecSmemBytes,
                         static_cast<cudaStream_t>(stream)>>>(tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? OD_OK : OD_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------
// Fixed scratch for od_space_attn_bwd_static_ws: callers that cannot allocate device memory
// (an allocator-free runtime, code running where cudaMalloc is forbidden or would
// synchronise) still need the backward's per-row Delta scratch.  It lives in this
// statically sized device array instead; each device that loads the library holds it until
// the process exits.  Host code must never pass the symbol itself to a kernel: on the host
// it is only a stand-in, so its device address is looked up once per device below.
static __device__ __align__(256) unsigned char g_od_static_ws[OD_STATIC_WORKSPACE_BYTES];
void* g_static_ws_ptr[kMaxDevices];

od_status static_ws_pointer(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_od_static_ws) != cudaSuccess || p == nullptr) return OD_ERR_CUDA;
    g_static_ws_ptr[dev] = p;
  }
  *out = g_static_ws_ptr[dev];
  return OD_OK;
}

}  // namespace

extern "C" {

od_status od_space_attn_bwd_static_ws(const void* q, const void* k, const void* v, const void* o,
                                      const void* o_lo, const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, float* dq_f32, float* dk_f32, float* dv_f32, int B,
                                      int T, int S, int Hq, int Hkv, int D, int agent_idx,
                                      float scale, void* stream) {
  if (B <= 0 || T <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return OD_ERR_INVALID_ARG;
  // the backward's scratch is one fp32 per query row; refuse what the fixed array cannot hold
  const size_t need = od::bwd_workspace_bytes(B, T, S, Hq, D);
  if (need > OD_STATIC_WORKSPACE_BYTES) return OD_ERR_WORKSPACE;
  void* ws = nullptr;
  od_status st = static_ws_pointer(&ws);
  if (st != OD_OK) return st;
  // the scratch is written completely before it is read, so nothing needs clearing
  return launch_bwd(0, q, k, v, o, o_lo, lse, dout, dq, dk, dv, dq_f32, dk_f32, dv_f32, B, T, S,
                    Hq, Hkv, D, agent_idx, 1, scale, ws, OD_STATIC_WORKSPACE_BYTES, stream);
}


od_status od_space_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* o_lo, int B, int T, int S, int Hq, int Hkv, int D,
                               int agent_idx, float scale, void* stream) {
  return launch_fwd(0, q, k, v, o, lse, o_lo, B, T, S, Hq, Hkv, D, agent_idx, 1, scale, stream);
}

od_status od_time_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* o_lo, int B, int T, int S, int Hq, int Hkv, int D, int window,
                              float scale, void* stream) {
  return launch_fwd(1, q, k, v, o, lse, o_lo, B, T, S, Hq, Hkv, D, -1, window, scale, stream);
}

od_status od_space_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                            float scale, void* stream) {
  return launch_fwd(0, q, k, v, o, lse, nullptr, B, T, S, Hq, Hkv, D, agent_idx, 1, scale, stream);
}

od_status od_time_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                           void* stream) {
  return launch_fwd(1, q, k, v, o, lse, nullptr, B, T, S, Hq, Hkv, D, -1, window, scale, stream);
}

size_t od_attn_bwd_workspace_bytes(int which, int B, int T, int S, int Hq, int Hkv, int D) {
  if ((which != 0 && which != 1) || check_shape(B, T, S, Hq, Hkv, D, 1.f) != OD_OK) return 0;
  return od::bwd_workspace_bytes(B, T, S, Hq, D);
}

od_status od_space_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                               const void* o_lo, const float* lse, const void* dout, void* dq,
                               void* dk, void* dv, float* dq_f32, float* dk_f32, float* dv_f32,
                               int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                               float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return launch_bwd(0, q, k, v, o, o_lo, lse, dout, dq, dk, dv, dq_f32, dk_f32, dv_f32, B, T, S, Hq,
                    Hkv, D, agent_idx, 1, scale, workspace, workspace_bytes, stream);
}

od_status od_time_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                              const void* o_lo, const float* lse, const void* dout, void* dq,
                              void* dk, void* dv, float* dq_f32, float* dk_f32, float* dv_f32,
                              int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return launch_bwd(1, q, k, v, o, o_lo, lse, dout, dq, dk, dv, dq_f32, dk_f32, dv_f32, B, T, S, Hq,
                    Hkv, D, -1, window, scale, workspace, workspace_bytes, stream);
}

od_status od_space_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                            float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return launch_bwd(0, q, k, v, o, nullptr, lse, dout, dq, dk, dv, nullptr, nullptr, nullptr, B, T,
                    S, Hq, Hkv, D, agent_idx, 1, scale, workspace, workspace_bytes, stream);
}

od_status od_time_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return launch_bwd(1, q, k, v, o, nullptr, lse, dout, dq, dk, dv, nullptr, nullptr, nullptr, B, T,
                    S, Hq, Hkv, D, -1, window, scale, workspace, workspace_bytes, stream);
}

od_status od_time_attn_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                              void* v_cache, void* o, float* lse, int B, int S, int Hq, int Hkv,
                              int D, int window, long long t, float scale, void* stream) {
  return launch_decode(q, k_new, v_new, k_cache, v_cache, o, lse, B, S, Hq, Hkv, D, window, t,
                       scale, stream);
}

// ---- packed QKV: q, k, v are the head ranges [0,Hq), [Hq,Hq+Hkv), [Hq+Hkv,Hq+2Hkv) of one
// [B,T,S,Hq+2Hkv,D] tensor (the output of a fused QKV projection, viewed as heads).
static od_status packed_views(const void* qkv, int B, int T, int S, int Hq, int Hkv, int D,
                              const void** q, const void** k, const void** v, int* rows) {
  if (!qkv || B <= 0 || T <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0)
    return OD_ERR_INVALID_ARG;
  if (D != 64) return OD_ERR_UNSUPPORTED;
  if (B > 65535 || T > (1 << 24) || S > (1 << 24) || Hq > 65535 || Hkv > 65535)
    return OD_ERR_UNSUPPORTED;
  *rows = Hq + 2 * Hkv;
  if (static_cast<unsigned __int128>(B) * static_cast<unsigned>(T) * static_cast<unsigned>(S) *
          static_cast<unsigned>(*rows) * static_cast<unsigned>(D) * 2u >=
      (static_cast<unsigned __int128>(1) << 40))
    return OD_ERR_UNSUPPORTED;
  const uint8_t* base = static_cast<const uint8_t*>(qkv);
  *q = base;
  *k = base + static_cast<size_t>(Hq) * D * 2;
  *v = base + static_cast<size_t>(Hq + Hkv) * D * 2;
  return OD_OK;
}

static od_status fwd_packed(int is_time, const void* qkv, void* o, float* lse, void* o_lo, int B,
                            int T, int S, int Hq, int Hkv, int D, int agent, int window,
                            float scale, void* stream) {
  const void *q, *k, *v;
  int rows = 0;
  od_status st = packed_views(qkv, B, T, S, Hq, Hkv, D, &q, &k, &v, &rows);
  if (st != OD_OK) return st;
  return launch_fwd(is_time, q, k, v, o, lse, o_lo, B, T, S, Hq, Hkv, D, agent, window, scale,
                    stream, rows);
}

static od_status bwd_packed(int is_time, const void* qkv, const void* o, const void* o_lo,
                            const float* lse,
                            const void* dout, void* dqkv, float* dq_f32, float* dk_f32,
                            float* dv_f32, int B, int T, int S, int Hq, int Hkv, int D, int agent,
                            int window, float scale, void* workspace, size_t workspace_bytes,
                            void* stream) {
  const void *q, *k, *v, *dq, *dk, *dv;
  int rows = 0;
  od_status st = packed_views(qkv, B, T, S, Hq, Hkv, D, &q, &k, &v, &rows);
  if (st != OD_OK) return st;
  if (!dqkv) return OD_ERR_INVALID_ARG;
  {  // the gradients must not overwrite the inputs they are computed from
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(qkv), b0 = reinterpret_cast<uintptr_t>(dqkv);
    const uintptr_t n = static_cast<uintptr_t>(1ULL * B * T * S * rows * D * 2);
    if (a0 < b0 + n && b0 < a0 + n) return OD_ERR_INVALID_ARG;
  }
  if ((st = packed_views(dqkv, B, T, S, Hq, Hkv, D, &dq, &dk, &dv, &rows)) != OD_OK) return st;
  return launch_bwd(is_time, q, k, v, o, o_lo, lse, dout, const_cast<void*>(dq), const_cast<void*>(dk),
                    const_cast<void*>(dv), dq_f32, dk_f32, dv_f32, B, T, S, Hq, Hkv, D, agent,
                    window, scale, workspace, workspace_bytes, stream, rows);
}

od_status od_space_attn_fwd_packed(const void* qkv, void* o, float* lse, void* o_lo, int B, int T,
                                   int S, int Hq, int Hkv, int D, int agent_idx, float scale,
                                   void* stream) {
  return fwd_packed(0, qkv, o, lse, o_lo, B, T, S, Hq, Hkv, D, agent_idx, 1, scale, stream);
}

od_status od_time_attn_fwd_packed(const void* qkv, void* o, float* lse, void* o_lo, int B, int T,
                                  int S, int Hq, int Hkv, int D, int window, float scale,
                                  void* stream) {
  return fwd_packed(1, qkv, o, lse, o_lo, B, T, S, Hq, Hkv, D, -1, window, scale, stream);
}

od_status od_space_attn_bwd_packed(const void* qkv, const void* o, const void* o_lo,
                                   const float* lse,
                                   const void* dout, void* dqkv, float* dq_f32, float* dk_f32,
                                   float* dv_f32, int B, int T, int S, int Hq, int Hkv, int D,
                                   int agent_idx, float scale, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return bwd_packed(0, qkv, o, o_lo, lse, dout, dqkv, dq_f32, dk_f32, dv_f32, B, T, S, Hq, Hkv, D,
                    agent_idx, 1, scale, workspace, workspace_bytes, stream);
}

od_status od_time_attn_bwd_packed(const void* qkv, const void* o, const void* o_lo,
                                  const float* lse,
                                  const void* dout, void* dqkv, float* dq_f32, float* dk_f32,
                                  float* dv_f32, int B, int T, int S, int Hq, int Hkv, int D,
                                  int window, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return bwd_packed(1, qkv, o, o_lo, lse, dout, dqkv, dq_f32, dk_f32, dv_f32, B, T, S, Hq, Hkv, D, -1,
                    window, scale, workspace, workspace_bytes, stream);
}

// ---- variable-length space attention: block (b, t) holds its first seqlen[b*T + t] tokens
od_status od_space_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o,
                                   float* lse, void* o_lo, const int* seqlen, int B, int T, int S,
                                   int Hq, int Hkv, int D, int agent_idx, float scale,
                                   void* stream) {
  if (!seqlen || !aligned16(seqlen)) return OD_ERR_INVALID_ARG;
  return launch_fwd(0, q, k, v, o, lse, o_lo, B, T, S, Hq, Hkv, D, agent_idx, 1, scale, stream, 0,
                    seqlen);
}

od_status od_space_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                   const void* o_lo, const float* lse, const void* dout,
                                   const int* seqlen, void* dq, void* dk, void* dv, float* dq_f32,
                                   float* dk_f32, float* dv_f32, int B, int T, int S, int Hq,
                                   int Hkv, int D, int agent_idx, float scale, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!seqlen || !aligned16(seqlen)) return OD_ERR_INVALID_ARG;
  return launch_bwd(0, q, k, v, o, o_lo, lse, dout, dq, dk, dv, dq_f32, dk_f32, dv_f32, B, T, S,
                    Hq, Hkv, D, agent_idx, 1, scale, workspace, workspace_bytes, stream, 0, seqlen);
}

od_status od_selftest_expired_wait(void* stream) {
  DeviceState* dev = nullptr;
  od_status st = device_state(&dev);
  if (st != OD_OK) return st;
  od::od_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status);
  return cudaGetLastError() == cudaSuccess ? OD_OK : OD_ERR_CUDA;
}

od_status od_get_device_status_detail(void* stream, unsigned int* site_word) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return OD_ERR_CUDA;
  unsigned int v[2] = {0, 0};
  if (cudaMemcpyFromSymbol(v, g_od_status, sizeof(v)) != cudaSuccess) return OD_ERR_CUDA;
  if (v[0] || v[1]) {
    const unsigned int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_od_status, zero, sizeof(zero)) != cudaSuccess) return OD_ERR_CUDA;
  }
  if (site_word) *site_word = v[1];
  if (v[0] & OD_DEV_RANGE) return OD_ERR_RANGE;
  return (v[0] & OD_DEV_TIMEOUT) ? OD_ERR_TIMEOUT : OD_OK;
}

od_status od_get_device_status(void* stream) { return od_get_device_status_detail(stream, nullptr); }

const char* od_status_string(od_status s) {
  switch (s) {
    case OD_OK: return "ok";
    case OD_ERR_INVALID_ARG: return "invalid argument";
    case OD_ERR_UNSUPPORTED: return "unsupported shape or head dimension";
    case OD_ERR_CUDA: return "CUDA error";
    case OD_ERR_TIMEOUT: return "device-side wait timed out";
    case OD_ERR_WORKSPACE: return "workspace too small";
    case OD_ERR_RANGE: return "device-side range check failed (debug build)";
  }
  return "unknown status";
}

#ifdef OD_DEBUG
const char* od_version(void) { return "od_attn 0.1 (sm_103a, debug: device-side range checks)"; }
#else
const char* od_version(void) { return "od_attn 0.1 (sm_103a)"; }
#endif

#ifdef OD_TRACE
// Profiling builds only: copies the per-warp trace regions (see od_common.cuh) into host
// memory -- dst holds OD_TRACE_WARPS * OD_TRACE_PER_WARP records, counts OD_TRACE_WARPS
// record counts -- and clears the counts.  Returns 0, or -1 on a CUDA error.
int od_trace_read(unsigned long long* dst, unsigned int* counts) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(counts, g_od_trace_n, OD_TRACE_WARPS * sizeof(unsigned int)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(dst, g_od_trace, sizeof(unsigned long long) * OD_TRACE_WARPS * OD_TRACE_PER_WARP) != cudaSuccess)
    return -1;
  unsigned int zero[OD_TRACE_WARPS] = {0};
  if (cudaMemcpyToSymbol(g_od_trace_n, zero, sizeof(zero)) != cudaSuccess) return -1;
  return 0;
}
// Profiling builds only: selects the kernel whose trace points record (0 forward, 1 dQ
// pass, 2 dK/dV, 3 Delta pass).  Returns 0, or -1 on a CUDA error.
int od_trace_select(int kernel) {
  return cudaMemcpyToSymbol(g_od_trace_sel, &kernel, sizeof(int)) == cudaSuccess ? 0 : -1;
}
#endif

}  // extern "C"
