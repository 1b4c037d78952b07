/*
 * kda_oracle.c -- fp64 CPU reference for the KDA forward (test infrastructure).
 *
 * This file is TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header or
 * table with the CUDA library; the CUDA library never loads it.
 *
 * What it computes: the KDA recurrence (the gated delta rule with a decay per
 * key dimension), token by token, in fp64.  For one sequence and one head,
 * with S a K x V state:
 *
 *     S <- Diag(exp(g_t)) S                       decay each key row d by exp(g_t[d])
 *     S <- S + beta_t k_t (v_t - S^T k_t)^T       delta-rule write of (k_t, v_t)
 *     o_t = scale * S^T q_t                        read-out after the write
 *
 * which is S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T.
 * Sources: kernel-fun "kda/_kernels/fwd_state.py" (module docstring: the
 * chunked form whose per-token limit this is -- the per-dimension gate sits on
 * the K rows of the state, h_{c+1}[d,:] = exp2(G_d) h_c[d,:] + ..., and the
 * output reads the state after the chunk's own writes, Aqk keeps i >= j), and
 * "KDA源码剖析之FlashKDA（下）" (the recurrence kernel walk-through: per-sequence
 * state taken from initial_state at bos and stored to final_state at eos, with
 * sequences delimited by cu_seqlens).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - the decay is applied before the delta write, and the delta uses the
 *    decayed state;
 *  - g is a natural-log decay (exp, not exp2); the log2 form is a GPU detail;
 *  - beta arrives already in (0,1); no sigmoid is applied here;
 *  - scale multiplies o only.
 *
 * Parity pins (tests/test_oracle.py): closed forms for beta=0, g=-inf,
 * orthonormal-key recall, overwrite, a constant-coefficient scalar recurrence,
 * a hand-worked 2x2 example, and agreement with the independently written
 * chunked form in chunked.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern (the top 16 bits of an IEEE fp32). */
static double bf16_bits_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Input element accessors: the same routine serves fp64 inputs (for pins with
 * values that bf16 cannot hold exactly) and the raw bf16/fp32 buffers that the
 * GPU path consumes (widened exactly). */
typedef struct {
    int kind; /* 0 = double, 1 = bf16 bits, 2 = float */
    const void* p;
} src_t;

static double src_at(const src_t* s, size_t i) {
    switch (s->kind) {
    case 0: return ((const double*)s->p)[i];
    case 1: return bf16_bits_to_f64(((const uint16_t*)s->p)[i]);
    default: return (double)((const float*)s->p)[i];
    }
}

typedef struct {
    src_t q, k, v, g, beta, h0; /* h0.p may be NULL: zero initial state */
    double scale;
    const int32_t* cu; /* [N+1] token offsets into the packed T axis */
    int N, H, K, V;
    const int32_t* units; /* [2*n_units] (seq, head) pairs, or NULL = all */
    int n_units;
    double* o;  /* [T_total, H, V], rows of the selected units are written */
    double* ht; /* [N, H, K, V] or NULL */
    int nthreads;
} job_t;

typedef struct {
    const job_t* job;
    int tid;
} worker_t;

/* One (sequence, head) unit: the token-by-token recurrence. */
static void run_unit(const job_t* J, int s, int h, double* S, double* kS) {
    const int H = J->H, K = J->K, V = J->V;
    const size_t KV = (size_t)K * V;
    if (J->h0.p) {
        const size_t base = ((size_t)s * H + h) * KV;
        for (size_t i = 0; i < KV; ++i) S[i] = src_at(&J->h0, base + i);
    } else {
        memset(S, 0, KV * sizeof(double));
    }
    const int bos = J->cu[s], eos = J->cu[s + 1];
    for (int t = bos; t < eos; ++t) {
        const size_t rk = ((size_t)t * H + h) * K; /* row of q, k, g */
        const size_t rv = ((size_t)t * H + h) * V; /* row of v, o */
        /* decay: row d of S scaled by exp(g_t[d]) */
        for (int d = 0; d < K; ++d) {
            const double a = exp(src_at(&J->g, rk + d));
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] *= a;
        }
        /* kS = S^T k_t (what the decayed state recalls for key k_t) */
        for (int j = 0; j < V; ++j) kS[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double kd = src_at(&J->k, rk + d);
            for (int j = 0; j < V; ++j) kS[j] += kd * S[(size_t)d * V + j];
        }
        /* delta write: S += beta k (v - kS)^T */
        const double b = src_at(&J->beta, (size_t)t * H + h);
        for (int j = 0; j < V; ++j) kS[j] = b * (src_at(&J->v, rv + j) - kS[j]);
        for (int d = 0; d < K; ++d) {
            const double kd = src_at(&J->k, rk + d);
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] += kd * kS[j];
        }
        /* read-out: o_t = scale S^T q_t */
        double* orow = J->o + rv;
        for (int j = 0; j < V; ++j) orow[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double qd = src_at(&J->q, rk + d);
            for (int j = 0; j < V; ++j) orow[j] += qd * S[(size_t)d * V + j];
        }
        for (int j = 0; j < V; ++j) orow[j] *= J->scale;
    }
    if (J->ht) memcpy(J->ht + ((size_t)s * H + h) * KV, S, KV * sizeof(double));
}

static void* worker_main(void* arg) {
    const worker_t* w = (const worker_t*)arg;
    const job_t* J = w->job;
    const int total = J->units ? J->n_units : J->N * J->H;
    double* S = (double*)malloc(sizeof(double) * ((size_t)J->K * J->V + J->V));
    if (!S) return (void*)1;
    double* kS = S + (size_t)J->K * J->V;
    for (int u = w->tid; u < total; u += J->nthreads) {
        int s, h;
        if (J->units) {
            s = J->units[2 * u];
            h = J->units[2 * u + 1];
        } else {
            s = u / J->H;
            h = u % J->H;
        }
        run_unit(J, s, h, S, kS);
    }
    free(S);
    return NULL;
}

static int run_job(job_t* J) {
    if (J->N < 0 || J->H <= 0 || J->K <= 0 || J->V <= 0 || !J->cu || !J->o) return 1;
    for (int s = 0; s < J->N; ++s)
        if (J->cu[s + 1] < J->cu[s]) return 2;
    if (J->units)
        for (int u = 0; u < J->n_units; ++u)
            if (J->units[2 * u] < 0 || J->units[2 * u] >= J->N || J->units[2 * u + 1] < 0 ||
                J->units[2 * u + 1] >= J->H)
                return 3;
    const int total = J->units ? J->n_units : J->N * J->H;
    if (J->nthreads < 1) J->nthreads = 1;
    if (J->nthreads > total) J->nthreads = total > 0 ? total : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * J->nthreads);
    worker_t* ws = (worker_t*)malloc(sizeof(worker_t) * J->nthreads);
    if (!th || !ws) {
        free(th);
        free(ws);
        return 4;
    }
    int rc = 0, started = 0;
    for (int i = 0; i < J->nthreads; ++i) {
        ws[i].job = J;
        ws[i].tid = i;
        if (pthread_create(&th[i], NULL, worker_main, &ws[i]) != 0) {
            rc = 5;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void* r = NULL;
        pthread_join(th[i], &r);
        if (r) rc = 6;
    }
    free(th);
    free(ws);
    return rc;
}

/*
 * fp64 inputs.  q, k, g: [T_total, H, K]; v: [T_total, H, V]; beta: [T_total, H];
 * h0: [N, H, K, V] or NULL; cu_seqlens: [N+1]; units: NULL or [2*n_units]
 * (sequence, head) pairs.  Writes o [T_total, H, V] rows of the selected units
 * and ht [N, H, K, V] (if non-NULL).  Returns 0 on success.
 */
int kda_oracle_fwd_f64(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, double scale, const double* h0,
                       const int32_t* cu_seqlens, int N, int H, int K, int V,
                       const int32_t* units, int n_units, double* o, double* ht,
                       int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = (src_t){0, q};
    J.k = (src_t){0, k};
    J.v = (src_t){0, v};
    J.g = (src_t){0, g};
    J.beta = (src_t){0, beta};
    J.h0 = (src_t){0, h0};
    J.scale = scale;
    J.cu = cu_seqlens;
    J.N = N;
    J.H = H;
    J.K = K;
    J.V = V;
    J.units = units;
    J.n_units = n_units;
    J.o = o;
    J.ht = ht;
    J.nthreads = nthreads;
    return run_job(&J);
}

/*
 * The storage formats of the GPU path: q, k, v, beta as bf16 bit patterns, g
 * and h0 as fp32; all widened exactly to fp64 before any arithmetic.
 */
int kda_oracle_fwd_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const float* g, const uint16_t* beta, double scale, const float* h0,
                        const int32_t* cu_seqlens, int N, int H, int K, int V,
                        const int32_t* units, int n_units, double* o, double* ht,
                        int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = (src_t){1, q};
    J.k = (src_t){1, k};
    J.v = (src_t){1, v};
    J.g = (src_t){2, g};
    J.beta = (src_t){1, beta};
    J.h0 = (src_t){2, h0};
    J.scale = scale;
    J.cu = cu_seqlens;
    J.N = N;
    J.H = H;
    J.K = K;
    J.V = V;
    J.units = units;
    J.n_units = n_units;
    J.o = o;
    J.ht = ht;
    J.nthreads = nthreads;
    return run_job(&J);
}
