/*
 * od_attn.h -- C ABI of the block-causal video attention library (B300, sm_103a).
 *
 * Two attention operators of the block-causal transformer backbone that the Open
 * Dreamer tokenizer and dynamics model share (7minutos.es page, section
 * "Arquitectura: una columna vertebral, dos modelos"; edgex es-LA page, section
 * "Arquitectura"): space attention inside one timestep block, where world-model tokens
 * cannot read the agent token, and causal time attention across timesteps at each token
 * position, limited to a sliding window (192 steps in the Minecraft configuration, edgex
 * es-LA page, section "Configuracion de entrenamiento"), with grouped-query heads
 * (30 query heads sharing 3 KV heads in that configuration).
 *
 * Notation: B batch, T timesteps, S tokens per timestep block, Hq query heads, Hkv KV
 * heads, G = Hq / Hkv, D head dimension (64), W time window, a agent token index
 * (-1 = none), scale = softmax scale (1/sqrt(D) in the pages' configs).
 * Query head h reads KV head floor(h / G).
 *
 * Space attention, for each (b, t, h) and query token s:
 *   keys s' of the same (b, t), except s' = a when s != a (the agent reads everything).
 * Time attention, for each (b, s, h) and query step t:
 *   keys t' of the same (b, s) with max(0, t - W + 1) <= t' <= t (W keys including t).
 * Per query row with logits l_j = scale * <q, k_j> over its allowed keys:
 *   LSE = ln sum_j exp(l_j),  O = sum_j exp(l_j - LSE) v_j.
 * Backward: dV_j += p_j dO, dP_j = <dO, v_j>, dS_j = p_j (dP_j - <dO, O>),
 *   dQ = scale sum_j dS_j k_j, dK_j += scale dS_j q, with dK and dV summed over the G
 *   query heads of a group.
 *
 * Layouts (row-major, contiguous, caller-owned device memory):
 *   Q, O, dO, dQ : [B, T, S, Hq, D]  bf16 (raw __nv_bfloat16 bits)
 *   K, V, dK, dV : [B, T, S, Hkv, D] bf16
 *   LSE          : [B, T, S, Hq]     fp32, natural log
 * Mixed precision follows the pages' stability notes (bf16 attention inputs, fp32
 * statistics; edgex es-LA page, section "Ingenieria de estabilidad", item 3): inputs and
 * outputs bf16, accumulation and softmax statistics fp32.
 *
 * Calls are asynchronous: they validate their arguments on the host, enqueue kernels on
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream) and return.
 * They never synchronise, allocate or free.  Outputs are fully overwritten (never
 * accumulated into).  Every device pointer must be 16-byte aligned.
 *
 * Errors: OD_ERR_INVALID_ARG for a null pointer, a non-positive size, Hq % Hkv != 0,
 * agent outside [-1, S), window < 1, a misaligned pointer, a scale that is not finite and
 * positive, or a workspace that is too small; OD_ERR_UNSUPPORTED for D != 64, G > 128 or
 * sizes beyond 32-bit tensor coordinates; OD_ERR_CUDA when a CUDA call or a launch
 * fails.  Nothing is enqueued when an error is returned.  Device-side timeouts (a bounded
 * wait that gave up) are reported later by od_get_device_status.
 */
#ifndef OD_ATTN_H
#define OD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OD_OK = 0,
  OD_ERR_INVALID_ARG = 1,
  OD_ERR_UNSUPPORTED = 2,
  OD_ERR_CUDA = 3,
  OD_ERR_TIMEOUT = 4,
  OD_ERR_WORKSPACE = 5,
  OD_ERR_RANGE = 6   /* debug builds (OD_DEBUG) only: a device-side range check failed */
} od_status;

/* Space attention forward.  Writes O [B,T,S,Hq,D] (bf16) and LSE [B,T,S,Hq] (fp32). */
od_status od_space_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                            float scale, void* stream);

/* Time attention forward (window >= 1; keys t-window+1 .. t).  Writes O and LSE. */
od_status od_time_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                           void* stream);

/* Space attention backward.  Inputs: Q, K, V, the forward's O and LSE, and dO.  Outputs
 * dQ [B,T,S,Hq,D], dK and dV [B,T,S,Hkv,D] in bf16 (overwritten).  Delta = <dO, O> per
 * query row is recomputed from P and dP (an extra pass over Q, K, V, dO with two matrix
 * products), because bf16 O alone does not give Delta to the accuracy the gradients need;
 * O is therefore not read (it must still be a valid, aligned pointer).  `workspace` is
 * caller-owned device scratch of at least od_attn_bwd_workspace_bytes(0, ...) bytes (Delta
 * per query row in fp32, rounded up to 256 bytes, then 32 KiB of per-CTA operand ranges);
 * its contents on entry do not matter. */
od_status od_space_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                            float scale, void* workspace, size_t workspace_bytes, void* stream);

/* Time attention backward; as od_space_attn_bwd with `window` in place of agent_idx
 * (workspace: od_attn_bwd_workspace_bytes(1, ...)). */
od_status od_time_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Extended forms: the calls above plus optional outputs.  With every added pointer NULL
 * each computes exactly what the corresponding call above computes (same kernels, same
 * results bit for bit).
 * Forward: o_lo (may be NULL), if given, also receives O's rounding residual [B,T,S,Hq,D]
 * bf16: o_lo = bf16(O - o) with O the fp32 result, so o + o_lo holds O to about 16
 * significant bits.  Passing it on to the backward lets the backward take Delta = <dO, O>
 * from memory instead of recomputing P and dP for it (a faster backward).
 * Backward: o_lo (may be NULL) is the residual the forward wrote; with it, Delta is the
 * row-wise dot product of dO with o + o_lo, read from memory (o is read then).  If
 * dq_f32/dk_f32/dv_f32 are non-NULL, the gradients are also written there in fp32 (same
 * layouts, contiguous), before rounding to bf16.  Errors as for the calls above, and
 * OD_ERR_INVALID_ARG for a misaligned optional pointer. */
od_status od_space_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* o_lo, int B, int T, int S, int Hq, int Hkv, int D,
                               int agent_idx, float scale, void* stream);
od_status od_time_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* o_lo, int B, int T, int S, int Hq, int Hkv, int D, int window,
                              float scale, void* stream);
od_status od_space_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                               const void* o_lo, const float* lse, const void* dout, void* dq,
                               void* dk, void* dv, float* dq_f32, float* dk_f32, float* dv_f32,
                               int B, int T, int S, int Hq, int Hkv, int D, int agent_idx,
                               float scale, void* workspace, size_t workspace_bytes, void* stream);
od_status od_time_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                              const void* o_lo, const float* lse, const void* dout, void* dq,
                              void* dk, void* dv, float* dq_f32, float* dk_f32, float* dv_f32,
                              int B, int T, int S, int Hq, int Hkv, int D, int window, float scale,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Packed-QKV forms.  Each layer of the block-causal backbone alternates space and time
 * attention (7minutos.es page, section "Arquitectura: una columna vertebral, dos modelos"),
 * and a fused QKV projection writes one [B, T, S, Hq + 2*Hkv, D] bf16 tensor per layer: per
 * token the Hq query heads, then the Hkv key heads, then the Hkv value heads.  These calls
 * read Q, K and V straight from that tensor (no split or copy) and compute exactly what the
 * unpacked calls compute, with the same kernels.  O, LSE and dO keep their contiguous
 * layouts; the backward writes dQ, dK and dV into `dqkv`, a second tensor of the packed shape
 * (heads in the same order), which must not be `qkv` (it may not overlap it at all).  The
 * optional fp32 gradient copies (dq_f32 ...) stay contiguous [B,T,S,H,D].  Errors as for the
 * unpacked calls. */
od_status od_space_attn_fwd_packed(const void* qkv, void* o, float* lse, void* o_lo, int B, int T,
                                   int S, int Hq, int Hkv, int D, int agent_idx, float scale,
                                   void* stream);
od_status od_time_attn_fwd_packed(const void* qkv, void* o, float* lse, void* o_lo, int B, int T,
                                  int S, int Hq, int Hkv, int D, int window, float scale,
                                  void* stream);
od_status od_space_attn_bwd_packed(const void* qkv, const void* o, const void* o_lo,
                                   const float* lse,
                                   const void* dout, void* dqkv, float* dq_f32, float* dk_f32,
                                   float* dv_f32, int B, int T, int S, int Hq, int Hkv, int D,
                                   int agent_idx, float scale, void* workspace,
                                   size_t workspace_bytes, void* stream);
od_status od_time_attn_bwd_packed(const void* qkv, const void* o, const void* o_lo,
                                  const float* lse,
                                  const void* dout, void* dqkv, float* dq_f32, float* dk_f32,
                                  float* dv_f32, int B, int T, int S, int Hq, int Hkv, int D,
                                  int window, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Variable-length space attention.  The tokenizer is a masked autoencoder (7minutos.es page,
 * section "Arquitectura: una columna vertebral, dos modelos"; up to 90 % of the patches
 * masked); an encoder that drops the masked patches instead of replacing them sees a
 * different number of tokens in each timestep block.  These calls take the padded layout
 * [B, T, S, H, D] (S = the longest block) and `seqlen`, a device array of B*T int32 (16-byte
 * aligned): block (b, t) holds its first seqlen[b*T + t] tokens (values are clamped to
 * [0, S]); the remaining slots are padding.  Per block the result is exactly space attention
 * over its first seqlen tokens (the agent rule applies when agent_idx < seqlen).  Work
 * scales with the lengths: tiles and key blocks past a block's length are never loaded or
 * computed.  Padding rows of Q, K, V and dO must hold finite values (zeros will do); the
 * outputs' padding rows (O, LSE, o_lo, dQ, dK, dV and the fp32 copies) are left unchanged.
 * The backward takes the forward's o_lo like od_space_attn_bwd_ex. */
od_status od_space_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o,
                                   float* lse, void* o_lo, const int* seqlen, int B, int T, int S,
                                   int Hq, int Hkv, int D, int agent_idx, float scale,
                                   void* stream);
od_status od_space_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                   const void* o_lo, const float* lse, const void* dout,
                                   const int* seqlen, void* dq, void* dk, void* dv, float* dq_f32,
                                   float* dk_f32, float* dv_f32, int B, int T, int S, int Hq,
                                   int Hkv, int D, int agent_idx, float scale, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* One rollout (decode) step of time attention over a ring-buffer KV cache.  A rollout
 * generates one frame at a time (the local rollout harness and the frame-by-frame demo,
 * 7minutos.es page, section "Lo que realmente se envió"); the time layer then needs, for
 * the new frame t only, the rows of od_time_attn_fwd at step t.  The cache holds the last
 * `window` (= W) frames of K and V, frame f in slot f mod W:
 *   q, o           : [B, S, Hq, D]     bf16, the new frame's queries / outputs
 *   k_new, v_new   : [B, S, Hkv, D]    bf16, the new frame's keys and values
 *   k_cache, v_cache: [B, W, S, Hkv, D] bf16, read and updated in place
 *   lse            : [B, S, Hq]        fp32, natural log
 * The call stores k_new / v_new in slot t mod W, then for every (b, s, h) attends from
 * q[b,s,h] to the frames max(0, t - W + 1) .. t of position s (KV head floor(h / G)), i.e.
 * the slots 0 .. min(t+1, W) - 1.  The slots a caller has not written yet (t < W - 1) are
 * never read.  t is the frame's absolute index (t >= 0); the caller feeds t = 0, 1, 2, ...
 * in order, or fills the slots of frames t-W+1 .. t-1 itself beforehand.
 * Errors as for od_time_attn_fwd (t < 0 or window < 1 is OD_ERR_INVALID_ARG), and
 * OD_ERR_UNSUPPORTED for G = Hq / Hkv > 16. */
od_status od_time_attn_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                              void* v_cache, void* o, float* lse, int B, int S, int Hq, int Hkv,
                              int D, int window, long long t, float scale, void* stream);

/* Size of the fixed device scratch used by od_space_attn_bwd_static_ws. */
#define OD_STATIC_WORKSPACE_BYTES (16u << 20)

/* Space attention backward for callers that cannot allocate device memory -- for example
 * code running under an allocator-free runtime, or at a point where cudaMalloc is not
 * allowed or would synchronise the device.  (The Open Dreamer pages have no counterpart;
 * this is a property of this library's interface.)  Same arguments and results as
 * od_space_attn_bwd_ex, minus the workspace: the scratch the backward needs (fp32 per query row
 * plus a fixed 32 KiB of operand ranges) lives in a fixed device array of
 * OD_STATIC_WORKSPACE_BYTES bytes inside the library, which every device that loads the
 * library keeps until the process exits.  Calls for which od_attn_bwd_workspace_bytes(0, ...)
 * exceeds OD_STATIC_WORKSPACE_BYTES (B*T*S*Hq above 4,186,112) are rejected with
 * OD_ERR_WORKSPACE before anything is enqueued.  This call never allocates or frees device
 * memory.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 * and caches it; make that first call before any stream capture on that device.
 * Every call shares the one array and leaves its contents behind: calls whose kernels can
 * overlap on the GPU (different streams, or different threads without ordering) race on it
 * and must be serialised by the caller.  The scratch is fully rewritten by each call before
 * it is read, so no clearing is needed. */
od_status od_space_attn_bwd_static_ws(const void* q, const void* k, const void* v, const void* o,
                                      const void* o_lo, const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, float* dq_f32, float* dk_f32, float* dv_f32, int B,
                                      int T, int S, int Hq, int Hkv, int D, int agent_idx,
                                      float scale, void* stream);

/* Bytes of device workspace the backward needs (which: 0 = space, 1 = time). Returns 0
 * for invalid sizes. */
size_t od_attn_bwd_workspace_bytes(int which, int B, int T, int S, int Hq, int Hkv, int D);

/* Synchronises `stream`, then reads and clears the device status word of the current
 * device.  Returns OD_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, OD_ERR_RANGE if a range check of the debug build failed (see below), OD_ERR_CUDA if
 * the synchronisation failed, OD_OK otherwise.
 * Debug build: libod_attn_debug.so, the same sources compiled with -DOD_DEBUG, exports the
 * same calls.  Its kernels check every TMA box start coordinate and every output row index
 * against the tensor's extent before the access; a failed check skips the access (a TMA
 * load is still issued -- the hardware clips it -- so that no wait is left without its
 * bytes), never traps, and is reported as OD_ERR_RANGE with the first check's site word
 * (bits 31-24: the check site, 200-249; bits 23-0: the CTA index).  Slower; for diagnosis. */
od_status od_get_device_status(void* stream);

/* As od_get_device_status; if site_word is non-NULL it receives the first expired wait's
 * site word since the last call (0 if none): bits 31-24 name the wait site inside the
 * kernel, bit 23 the phase parity waited for, bits 22-0 the CTA index.  For diagnosis. */
od_status od_get_device_status_detail(void* stream, unsigned int* site_word);

/* Self-test of the device-side failure path: enqueues one warp that waits on a barrier
 * nothing will complete.  The wait gives up after the library's wait limit (2 s), records a
 * timeout with site 120 and returns, so that the next od_get_device_status reports
 * OD_ERR_TIMEOUT while the context stays usable.  No fault, trap or unbounded wait is
 * involved.  For tests of error handling only. */
od_status od_selftest_expired_wait(void* stream);

/* Static description of a status code. */
const char* od_status_string(od_status s);

/* Library version string. */
const char* od_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OD_ATTN_H */
