/*
 * od_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the two attention operators of the
 * block-causal transformer backbone described on the Open Dreamer pages.  It
 * is the yardstick the CUDA library is checked against and is never called by
 * the library itself (only tests/, the smoke check and the bench's CPU
 * baseline use it).  It shares no code, header or constant with the CUDA path.
 *
 * What is computed (all arithmetic in double precision, straight from the
 * definitions, no tiling, no online softmax):
 *
 *   Space attention -- "spatial layers move information between the elements
 *   of one frame" and "world-model tokens cannot read the agent token"
 *   (7minutos.es page, section "Arquitectura: una columna vertebral, dos
 *   modelos"; edgex es-LA page, section "Arquitectura").  For every batch b,
 *   timestep t and query head h, query token s attends to the keys s' of the
 *   same (b, t) in the allowed set
 *       A(s) = {0..S-1} minus {a}   if s != a,
 *       A(s) = {0..S-1}             if s == a (the agent reads everything),
 *   with a = -1 meaning no agent token.
 *
 *   Time attention -- "causal time layers move information between frames",
 *   with "a sliding window of 192 steps" (same sections, and section
 *   "Configuracion de entrenamiento").  For every (b, s, h), query step t
 *   attends to key steps t' of the same token position s in
 *       C(t) = { t' : max(0, t - W + 1) <= t' <= t }   (W keys, self included).
 *
 *   Grouped-query heads ("30 attention heads and 3 KV heads", same section):
 *   query head h uses KV head floor(h / G), G = Hq / Hkv.
 *
 *   For a query row with logits l_j = scale * <q, k_j> over its allowed keys:
 *     m = max_j l_j,  LSE = m + ln sum_j exp(l_j - m),  p_j = exp(l_j - LSE),
 *     O = sum_j p_j v_j.
 *   Backward (activation checkpointing recomputes p from the saved LSE; the
 *   oracle simply recomputes everything):
 *     Delta = <dO, O>,  dP_j = <dO, v_j>,  dS_j = p_j (dP_j - Delta),
 *     dQ = scale sum_j dS_j k_j,  dK_j += scale dS_j q,  dV_j += p_j dO,
 *   where dK and dV sum over every query row and every query head of the group.
 *
 *   Decode step (oracle_time_decode, at the end of this file): one new frame of a
 *   rollout attends, per token position, to the last W frames held in a ring-buffer
 *   KV cache -- the time-attention rows above for the single step t, with the new
 *   frame stored into its cache slot first.
 *
 * Layouts (row-major, contiguous): Q, O, dQ, dO [B,T,S,Hq,D];
 * K, V, dK, dV [B,T,S,Hkv,D]; LSE [B,T,S,Hq] (natural log).
 *
 * Threads: independent units are spread over `nthreads` POSIX threads
 * (nthreads <= 0 means all online cores).  A space unit is (b, t, kv head), a
 * time unit is (b, s, kv head); a unit owns its slice of dK and dV, so there is
 * no sharing between threads.
 *
 * Return value: 0 on success, -1 on an invalid argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv;
    int B, T, S, Hq, Hkv, D;
    int agent;   /* space only */
    int window;  /* time only */
    double scale;
    int is_time;
    int backward;
    long nunits;
    long next;   /* shared work counter */
    pthread_mutex_t lock;
} job_t;

static long q_index(const job_t *J, int b, int t, int s, int h) {
    return ((((long)b * J->T + t) * J->S + s) * J->Hq + h) * (long)J->D;
}
static long kv_index(const job_t *J, int b, int t, int s, int h) {
    return ((((long)b * J->T + t) * J->S + s) * J->Hkv + h) * (long)J->D;
}
static long lse_index(const job_t *J, int b, int t, int s, int h) {
    return (((long)b * J->T + t) * J->S + s) * J->Hq + h;
}
static double dot(const double *x, const double *y, int n) {
    double acc = 0.0;
    for (int i = 0; i < n; ++i) acc += x[i] * y[i];
    return acc;
}

/* Allowed key positions of query position `pos` in a sequence of length L.
 * Space: pos/keys are token indices s within one frame.
 * Time:  pos/keys are timesteps t at one token position.
 * Returns the number of allowed keys written to `keys`. */
static int allowed_keys(const job_t *J, int pos, int L, int *keys) {
    int n = 0;
    if (J->is_time) {
        int lo = pos - J->window + 1;
        if (lo < 0) lo = 0;
        for (int j = lo; j <= pos; ++j) keys[n++] = j;
    } else {
        for (int j = 0; j < L; ++j) {
            if (j == J->agent && pos != J->agent) continue;  /* world tokens skip the agent */
            keys[n++] = j;
        }
    }
    return n;
}

/* One unit: (b, frame t, kv head g) for space; (b, token s, kv head g) for time. */
static void run_unit(job_t *J, long u, int *keys, double *logit, double *p, double *orow,
                     double *dp) {
    const int G = J->Hq / J->Hkv;
    const int D = J->D;
    int b, fixed, g;  /* fixed = t for space, s for time */
    g = (int)(u % J->Hkv);
    long rest = u / J->Hkv;
    if (J->is_time) { fixed = (int)(rest % J->S); b = (int)(rest / J->S); }
    else            { fixed = (int)(rest % J->T); b = (int)(rest / J->T); }
    const int L = J->is_time ? J->T : J->S;

    for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh;
        for (int pos = 0; pos < L; ++pos) {
            const int t = J->is_time ? pos : fixed;
            const int s = J->is_time ? fixed : pos;
            const double *qrow = J->q + q_index(J, b, t, s, h);
            const int n = allowed_keys(J, pos, L, keys);
            /* logits and the row maximum */
            double m = -INFINITY;
            for (int j = 0; j < n; ++j) {
                const int kt = J->is_time ? keys[j] : t;
                const int ks = J->is_time ? s : keys[j];
                logit[j] = J->scale * dot(qrow, J->k + kv_index(J, b, kt, ks, g), D);
                if (logit[j] > m) m = logit[j];
            }
            double z = 0.0;
            for (int j = 0; j < n; ++j) z += exp(logit[j] - m);
            const double lse = m + log(z);
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            for (int j = 0; j < n; ++j) {
                const int kt = J->is_time ? keys[j] : t;
                const int ks = J->is_time ? s : keys[j];
                p[j] = exp(logit[j] - lse);
                const double *vrow = J->v + kv_index(J, b, kt, ks, g);
                for (int d = 0; d < D; ++d) orow[d] += p[j] * vrow[d];
            }
            if (J->o) memcpy(J->o + q_index(J, b, t, s, h), orow, sizeof(double) * D);
            if (J->lse) J->lse[lse_index(J, b, t, s, h)] = lse;
            if (!J->backward) continue;

            const double *dorow = J->dout + q_index(J, b, t, s, h);
            double *dqrow = J->dq + q_index(J, b, t, s, h);
            const double delta = dot(dorow, orow, D);
            for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
            for (int j = 0; j < n; ++j) {
                const int kt = J->is_time ? keys[j] : t;
                const int ks = J->is_time ? s : keys[j];
                const long kvi = kv_index(J, b, kt, ks, g);
                dp[j] = dot(dorow, J->v + kvi, D);
                const double ds = p[j] * (dp[j] - delta);
                const double *krow = J->k + kvi;
                double *dkrow = J->dk + kvi;
                double *dvrow = J->dv + kvi;
                for (int d = 0; d < D; ++d) {
                    dqrow[d] += J->scale * ds * krow[d];
                    dkrow[d] += J->scale * ds * qrow[d];
                    dvrow[d] += p[j] * dorow[d];
                }
            }
        }
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int L = J->is_time ? J->T : J->S;
    int *keys = (int *)malloc(sizeof(int) * (size_t)L);
    double *logit = (double *)malloc(sizeof(double) * (size_t)L);
    double *p = (double *)malloc(sizeof(double) * (size_t)L);
    double *dp = (double *)malloc(sizeof(double) * (size_t)L);
    double *orow = (double *)malloc(sizeof(double) * (size_t)J->D);
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long u = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->nunits) break;
        run_unit(J, u, keys, logit, p, orow, dp);
    }
    free(keys); free(logit); free(p); free(dp); free(orow);
    return NULL;
}

static int run(job_t *J, int nthreads) {
    if (J->B <= 0 || J->T <= 0 || J->S <= 0 || J->Hq <= 0 || J->Hkv <= 0 || J->D <= 0) return -1;
    if (J->Hq % J->Hkv) return -1;
    if (J->is_time && J->window < 1) return -1;
    if (!J->is_time && (J->agent < -1 || J->agent >= J->S)) return -1;
    J->nunits = (long)J->B * (J->is_time ? J->S : J->T) * J->Hkv;
    J->next = 0;
    if (J->backward) {
        const size_t nkv = (size_t)J->B * J->T * J->S * J->Hkv * J->D;
        memset(J->dk, 0, nkv * sizeof(double));
        memset(J->dv, 0, nkv * sizeof(double));
    }
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > J->nunits) nthreads = (int)J->nunits;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->lock);
    return 0;
}

int oracle_space_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                     int B, int T, int S, int Hq, int Hkv, int D, int agent, double scale,
                     int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    J.B = B; J.T = T; J.S = S; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.agent = agent; J.scale = scale; J.is_time = 0; J.backward = 0;
    return run(&J, nthreads);
}

int oracle_time_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                    int B, int T, int S, int Hq, int Hkv, int D, int window, double scale,
                    int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    J.B = B; J.T = T; J.S = S; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.window = window; J.scale = scale; J.is_time = 1; J.backward = 0;
    return run(&J, nthreads);
}

int oracle_space_bwd(const double *q, const double *k, const double *v, const double *dout,
                     double *o, double *lse, double *dq, double *dk, double *dv,
                     int B, int T, int S, int Hq, int Hkv, int D, int agent, double scale,
                     int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.dout = dout; J.o = o; J.lse = lse;
    J.dq = dq; J.dk = dk; J.dv = dv;
    J.B = B; J.T = T; J.S = S; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.agent = agent; J.scale = scale; J.is_time = 0; J.backward = 1;
    return run(&J, nthreads);
}

int oracle_time_bwd(const double *q, const double *k, const double *v, const double *dout,
                    double *o, double *lse, double *dq, double *dk, double *dv,
                    int B, int T, int S, int Hq, int Hkv, int D, int window, double scale,
                    int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.dout = dout; J.o = o; J.lse = lse;
    J.dq = dq; J.dk = dk; J.dv = dv;
    J.B = B; J.T = T; J.S = S; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.window = window; J.scale = scale; J.is_time = 1; J.backward = 1;
    return run(&J, nthreads);
}

int oracle_num_threads(int requested) {
    if (requested > 0) return requested;
    return (int)sysconf(_SC_NPROCESSORS_ONLN);
}

/*
 * Decode step of time attention with a ring-buffer KV cache.  Rollout generates frames one
 * at a time (7minutos.es page, section "Lo que realmente se envió": the local rollout
 * harness; the time window of W frames as above).  The new frame has absolute index t; the
 * cache holds the last W frames, frame f in slot f mod W.  The step first stores the new
 * frame's K and V in slot t mod W; then every query head h of every token position s of the
 * new frame attends, at the same (b, s) and KV head floor(h / G), to the frames
 *     f = max(0, t - W + 1) .. t
 * with logits l_f = scale <q, k_f>:  LSE = ln sum_f exp(l_f),  O = sum_f exp(l_f - LSE) v_f.
 * Layouts: q, o [B,S,Hq,D]; k_new, v_new [B,S,Hkv,D]; k_cache, v_cache [B,W,S,Hkv,D] (updated
 * in place); lse [B,S,Hq].  Single-threaded: decode shapes are small.
 */
int oracle_time_decode(const double *q, const double *k_new, const double *v_new,
                       double *k_cache, double *v_cache, double *o, double *lse,
                       int B, int S, int Hq, int Hkv, int D, int W, long long t, double scale) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || t < 0 || Hq % Hkv) return 1;
    const int G = Hq / Hkv;
    const long slot_t = (long)(t % W);
    /* 1. the new frame's K/V into its slot */
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int h = 0; h < Hkv; ++h) {
                const long src = (((long)b * S + s) * Hkv + h) * D;
                const long dst = ((((long)b * W + slot_t) * S + s) * Hkv + h) * D;
                for (int d = 0; d < D; ++d) {
                    k_cache[dst + d] = k_new[src + d];
                    v_cache[dst + d] = v_new[src + d];
                }
            }
    /* 2. attention of the new frame's queries over the frames in the window */
    const long long f0 = t - W + 1 > 0 ? t - W + 1 : 0;
    const int nk = (int)(t - f0 + 1);
    double *logit = (double *)malloc(sizeof(double) * (size_t)nk);
    if (!logit) return 2;
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / G;
                const double *qr = q + (((long)b * S + s) * Hq + h) * D;
                double m = -INFINITY;
                for (int j = 0; j < nk; ++j) {
                    const long slot = (long)((f0 + j) % W);
                    const double *kr = k_cache + ((((long)b * W + slot) * S + s) * Hkv + kvh) * D;
                    logit[j] = scale * dot(qr, kr, D);
                    if (logit[j] > m) m = logit[j];
                }
                double sum = 0.0;
                for (int j = 0; j < nk; ++j) sum += exp(logit[j] - m);
                const double l = m + log(sum);
                lse[((long)b * S + s) * Hq + h] = l;
                double *orow = o + (((long)b * S + s) * Hq + h) * D;
                for (int d = 0; d < D; ++d) orow[d] = 0.0;
                for (int j = 0; j < nk; ++j) {
                    const long slot = (long)((f0 + j) % W);
                    const double *vr = v_cache + ((((long)b * W + slot) * S + s) * Hkv + kvh) * D;
                    const double pj = exp(logit[j] - l);
                    for (int d = 0; d < D; ++d) orow[d] += pj * vr[d];
                }
            }
    free(logit);
    return 0;
}
