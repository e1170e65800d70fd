/*
 * hypic_oracle.c -- plain, slow, fp64 CPU oracle for HYPIC's linear-layer state path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls this file:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg do. It shares
 * no code, header, table or helper with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - The per-segment pair (S(C|0), T_C). "Cut First-Token Latency by 3.25x: Introducing
 *    HYPIC ..." (besthub.dev), paragraph "For linear layers": HYPIC stores T_C and the
 *    zero-initial state S(C|0) of every cached segment C. "HYPIC: Cache Acceleration for
 *    Hybrid Attention Models" (agihunt.info), "Core Approach", Linear Layers: T_C is the
 *    segment-cumulative transition operator.
 *    S(C|0) is obtained by stepping the family's recurrence token by token from S = 0.
 *    T_C is obtained by left-multiplying the identity by every token's transition factor,
 *    in token order, so that the latest factor ends up leftmost.
 *
 *  - The sequential run over the concatenated segments, which is the ground truth the
 *    composition must reproduce ("Hypic: Position-Independent KV Caching for
 *    Hybrid-Attention LLM Serving", episode companion, introduction: composition provably
 *    matches sequential computation).
 *
 *  - The composition scan prefix_j = T_j . prefix_{j-1} + S_j (besthub.dev paragraph
 *    "For linear layers": reuse composes T_C2 . S(C1) + S(C2)), with explicit dense
 *    matrix products, and the transition of the composed entry, T_{n-1} ... T_0.
 *
 *  - The segment's outputs o_t = S_t^T q_t for every token t of a segment, with S_t the
 *    state after token t when the segment starts from S_init (zero: the zero-state outputs
 *    O(C|0) of the prefill that stores the pair; a prefix state: the outputs of the segment
 *    reused after that prefix). besthub.dev, paragraph "For linear layers" (the pair is
 *    stored during the first prefill) and paragraph "Segment parallelism" (cold segments
 *    are prefilled by the scatter workers).
 *
 * The pages name the families (plain linear attention, RetNet, Mamba2, GLA, DeltaNet,
 * GDN, KDA) but print no equation. The recurrences below are the standard published forms,
 * with the state S a d_k x d_v matrix (rows = key channels) and T acting on the left:
 *
 *   LINEAR  S_t = S_{t-1} + k_t v_t^T                             factor I
 *   SCALAR  S_t = g_t S_{t-1} + k_t v_t^T, g_t = exp(log_gate)     factor g_t I
 *   DIAG    S_t = Diag(g_t) S_{t-1} + k_t v_t^T                    factor Diag(g_t)
 *   DELTA   S_t = (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T      factor I - b_t k_t k_t^T
 *   GDN     S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T  factor a_t (I - b_t k_t k_t^T)
 *   KDA     S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T
 *                                                          factor (I - b_t k_t k_t^T) Diag(a_t)
 *
 * (GDN: "Gated Delta Networks: Improving Mamba2 with Delta Rule", reference 7 of the
 * episode companion page.) SCALAR covers RetNet (constant per-head gamma) and Mamba2
 * (per-token scalar gate). KDA is the channel-gated delta rule: the gated delta rule with a
 * per-key-channel decay a_t in (0, 1]^{d_k} applied before the delta update.
 *
 * Layouts (all row-major, fp64):
 *   k        [N_tok][H_k][d_k]      value head h reads key head h / (H_v / H_k)
 *   v        [N_tok][H_v][d_v]
 *   q        [N_tok][H_k][d_k]      (outputs only)
 *   log_gate SCALAR [N_tok][H_v], DIAG and KDA [N_tok][H_v][d_k], GDN [N_tok][H_v], else unused
 *   log_gamma SCALAR with a constant per-head gate: [H_v] (then log_gate is unused)
 *   beta     DELTA / GDN / KDA [N_tok][H_v]
 *   S        [n_seg][H_v][d_k][d_v], T [n_seg][H_v][d_k][d_k]
 *   O        [N_tok][H_v][d_v]
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FAM_LINEAR = 0, FAM_SCALAR = 1, FAM_DIAG = 2, FAM_DELTA = 3, FAM_GDN = 4, FAM_KDA = 5 };

typedef struct {
    int family, H_k, H_v, d_k, d_v;
    const double *k, *v, *log_gate, *log_gamma, *beta;
} recurrence;

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Left-multiply the d_k x ncols matrix X by token t's transition factor of head h.
 * w is scratch of ncols doubles. */
static void apply_factor(const recurrence *r, int64_t t, int h, double *X, int ncols, double *w) {
    const int dk = r->d_k;
    const int hk = h / (r->H_v / r->H_k);
    const double *kt = r->k + ((size_t)t * r->H_k + hk) * dk;
    switch (r->family) {
    case FAM_LINEAR:
        return;
    case FAM_SCALAR: {
        double lg = r->log_gamma ? r->log_gamma[h] : r->log_gate[(size_t)t * r->H_v + h];
        double g = exp(lg);
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < ncols; ++n) X[(size_t)i * ncols + n] *= g;
        return;
    }
    case FAM_DIAG: {
        const double *lg = r->log_gate + ((size_t)t * r->H_v + h) * dk;
        for (int i = 0; i < dk; ++i) {
            double g = exp(lg[i]);
            for (int n = 0; n < ncols; ++n) X[(size_t)i * ncols + n] *= g;
        }
        return;
    }
    case FAM_DELTA:
    case FAM_GDN: {
        double a = (r->family == FAM_GDN) ? exp(r->log_gate[(size_t)t * r->H_v + h]) : 1.0;
        double b = r->beta[(size_t)t * r->H_v + h];
        /* a (I - b k k^T) X = a (X - b k (k^T X)) */
        for (int n = 0; n < ncols; ++n) w[n] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < ncols; ++n) w[n] += kt[i] * X[(size_t)i * ncols + n];
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < ncols; ++n)
                X[(size_t)i * ncols + n] = a * (X[(size_t)i * ncols + n] - b * kt[i] * w[n]);
        return;
    }
    case FAM_KDA: {
        /* (I - b k k^T) Diag(a) X: the channel decay first, then the delta update */
        const double *lg = r->log_gate + ((size_t)t * r->H_v + h) * dk;
        double b = r->beta[(size_t)t * r->H_v + h];
        for (int i = 0; i < dk; ++i) {
            double g = exp(lg[i]);
            for (int n = 0; n < ncols; ++n) X[(size_t)i * ncols + n] *= g;
        }
        for (int n = 0; n < ncols; ++n) w[n] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < ncols; ++n) w[n] += kt[i] * X[(size_t)i * ncols + n];
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < ncols; ++n) X[(size_t)i * ncols + n] -= b * kt[i] * w[n];
        return;
    }
    }
}

/* Add token t's write term to the d_k x d_v state S of head h:
 * k_t v_t^T, scaled by b_t for DELTA / GDN. */
static void add_write(const recurrence *r, int64_t t, int h, double *S) {
    const int dk = r->d_k, dv = r->d_v;
    const int hk = h / (r->H_v / r->H_k);
    const double *kt = r->k + ((size_t)t * r->H_k + hk) * dk;
    const double *vt = r->v + ((size_t)t * r->H_v + h) * dv;
    double b = (r->family == FAM_DELTA || r->family == FAM_GDN || r->family == FAM_KDA)
                   ? r->beta[(size_t)t * r->H_v + h] : 1.0;
    for (int i = 0; i < dk; ++i)
        for (int n = 0; n < dv; ++n) S[(size_t)i * dv + n] += b * kt[i] * vt[n];
}

static int check_shape(int family, int H_k, int H_v, int d_k, int d_v) {
    if (family < FAM_LINEAR || family > FAM_KDA) return -1;
    if (H_k <= 0 || H_v <= 0 || d_k <= 0 || d_v <= 0) return -1;
    if (H_v % H_k != 0) return -1;
    return 0;
}

/* (S(C|0), T_C) for every segment and value head. */
int oracle_build(int family, int n_seg, const int64_t *seg_offsets, int H_k, int H_v, int d_k,
                 int d_v, const double *k, const double *v, const double *log_gate,
                 const double *log_gamma, const double *beta, double *S_out, double *T_out,
                 int nthreads) {
    if (check_shape(family, H_k, H_v, d_k, d_v)) return -1;
    recurrence r = {family, H_k, H_v, d_k, d_v, k, v, log_gate, log_gamma, beta};
    set_threads(nthreads);
    const int64_t units = (int64_t)n_seg * H_v;
    int err = 0;
#pragma omp parallel
    {
        int wn = d_k > d_v ? d_k : d_v;
        double *w = (double *)malloc(sizeof(double) * wn);
        if (!w) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            if (!w) continue;
            int seg = (int)(u / H_v), h = (int)(u % H_v);
            double *S = S_out + (size_t)u * d_k * d_v;
            double *T = T_out ? T_out + (size_t)u * d_k * d_k : NULL;
            memset(S, 0, sizeof(double) * d_k * d_v);
            if (T) {
                memset(T, 0, sizeof(double) * d_k * d_k);
                for (int i = 0; i < d_k; ++i) T[(size_t)i * d_k + i] = 1.0;
            }
            for (int64_t t = seg_offsets[seg]; t < seg_offsets[seg + 1]; ++t) {
                apply_factor(&r, t, h, S, d_v, w);
                add_write(&r, t, h, S);
                if (T) apply_factor(&r, t, h, T, d_k, w);
            }
        }
        free(w);
    }
    return err;
}

/* Sequential run over the concatenated segments from the initial state S0 (NULL = 0);
 * S_bound[j] receives the state after segment j. */
int oracle_run(int family, int n_seg, const int64_t *seg_offsets, int H_k, int H_v, int d_k,
               int d_v, const double *k, const double *v, const double *log_gate,
               const double *log_gamma, const double *beta, const double *S0, double *S_bound,
               int nthreads) {
    if (check_shape(family, H_k, H_v, d_k, d_v)) return -1;
    recurrence r = {family, H_k, H_v, d_k, d_v, k, v, log_gate, log_gamma, beta};
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * d_v);
        double *S = (double *)malloc(sizeof(double) * d_k * d_v);
        if (!w || !S) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int h = 0; h < H_v; ++h) {
            if (!w || !S) continue;
            if (S0) memcpy(S, S0 + (size_t)h * d_k * d_v, sizeof(double) * d_k * d_v);
            else memset(S, 0, sizeof(double) * d_k * d_v);
            for (int seg = 0; seg < n_seg; ++seg) {
                for (int64_t t = seg_offsets[seg]; t < seg_offsets[seg + 1]; ++t) {
                    apply_factor(&r, t, h, S, d_v, w);
                    add_write(&r, t, h, S);
                }
                memcpy(S_bound + ((size_t)seg * H_v + h) * d_k * d_v, S,
                       sizeof(double) * d_k * d_v);
            }
        }
        free(w);
        free(S);
    }
    return err;
}

/* prefix_j = T_j prefix_{j-1} + S_j, prefix_{-1} = S0 (NULL = 0), for every unit.
 * T [n_seg][n_units][d_k][d_k], S and prefix [n_seg][n_units][d_k][d_v]. */
int oracle_compose_scan(int n_seg, int64_t n_units, int d_k, int d_v, const double *T,
                        const double *S, const double *S0, double *prefix, int nthreads) {
    if (n_seg < 0 || n_units < 0 || d_k <= 0 || d_v <= 0) return -1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *cur = (double *)malloc(sizeof(double) * d_k * d_v);
        double *nxt = (double *)malloc(sizeof(double) * d_k * d_v);
        if (!cur || !nxt) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < n_units; ++u) {
            if (!cur || !nxt) continue;
            if (S0) memcpy(cur, S0 + (size_t)u * d_k * d_v, sizeof(double) * d_k * d_v);
            else memset(cur, 0, sizeof(double) * d_k * d_v);
            for (int j = 0; j < n_seg; ++j) {
                const double *Tj = T + ((size_t)j * n_units + u) * d_k * d_k;
                const double *Sj = S + ((size_t)j * n_units + u) * d_k * d_v;
                for (int i = 0; i < d_k; ++i)
                    for (int n = 0; n < d_v; ++n) {
                        double acc = 0.0;
                        for (int m = 0; m < d_k; ++m)
                            acc += Tj[(size_t)i * d_k + m] * cur[(size_t)m * d_v + n];
                        nxt[(size_t)i * d_v + n] = acc + Sj[(size_t)i * d_v + n];
                    }
                memcpy(cur, nxt, sizeof(double) * d_k * d_v);
                memcpy(prefix + ((size_t)j * n_units + u) * d_k * d_v, cur,
                       sizeof(double) * d_k * d_v);
            }
        }
        free(cur);
        free(nxt);
    }
    return err;
}

/* Dense T from the log-scaled storage T = exp(lam) P that the library exports:
 *   LINEAR           T = I                      (lam, P unused)
 *   SCALAR           T = exp(lam[u]) I           lam [n]
 *   DIAG             T = Diag(exp(lam[u][i]))    lam [n][d_k]
 *   DELTA / GDN / KDA T = exp(lam[u]) P[u]       lam [n], P [n][d_k][d_k]
 * n is the number of (segment, unit) matrices. */
int oracle_materialize_T(int family, int64_t n, int d_k, const double *lam, const double *P,
                         double *T_out) {
    if (family < FAM_LINEAR || family > FAM_KDA || n < 0 || d_k <= 0) return -1;
    for (int64_t u = 0; u < n; ++u) {
        double *T = T_out + (size_t)u * d_k * d_k;
        memset(T, 0, sizeof(double) * d_k * d_k);
        switch (family) {
        case FAM_LINEAR:
            for (int i = 0; i < d_k; ++i) T[(size_t)i * d_k + i] = 1.0;
            break;
        case FAM_SCALAR: {
            double s = exp(lam[u]);
            for (int i = 0; i < d_k; ++i) T[(size_t)i * d_k + i] = s;
            break;
        }
        case FAM_DIAG:
            for (int i = 0; i < d_k; ++i) T[(size_t)i * d_k + i] = exp(lam[(size_t)u * d_k + i]);
            break;
        default: {
            double s = exp(lam[u]);
            const double *Pu = P + (size_t)u * d_k * d_k;
            for (size_t e = 0; e < (size_t)d_k * d_k; ++e) T[e] = s * Pu[e];
        }
        }
    }
    return 0;
}

/* The transition of consecutive segments composed into one cache entry, in the log-scaled
 * storage of the library: T(C_0 ... C_{n-1}) = T_{n-1} ... T_0 (latest segment leftmost;
 * "Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For
 * linear layers": an entry is the pair (T_C, S(C|0)) and entries compose as
 * T_C2 . S(C1) + S(C2), whose transition is T_C2 T_C1). With T_j = exp(lam_j) P_j:
 *   lam_total = sum_j lam_j                      [n_units] (DIAG: [n_units][d_k])
 *   P_total   = P_{n-1} ... P_0                  DELTA / GDN / KDA: [n_units][d_k][d_k]
 * lam [n_seg][n_units] (DIAG [n_seg][n_units][d_k]; unused for LINEAR, whose lam_total is
 * 0), P [n_seg][n_units][d_k][d_k]. Explicit dense products, one segment at a time. */
int oracle_compose_transitions(int family, int n_seg, int64_t n_units, int d_k, const double *lam,
                               const double *P, double *lam_total, double *P_total, int nthreads) {
    if (family < FAM_LINEAR || family > FAM_KDA || n_seg < 1 || n_units < 0 || d_k <= 0) return -1;
    const int dense = family == FAM_DELTA || family == FAM_GDN || family == FAM_KDA;
    const int nl = family == FAM_DIAG ? d_k : 1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *nxt = dense ? (double *)malloc(sizeof(double) * d_k * d_k) : NULL;
        if (dense && !nxt) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < n_units; ++u) {
            for (int i = 0; i < nl; ++i) {
                double acc = 0.0;
                if (family != FAM_LINEAR)
                    for (int j = 0; j < n_seg; ++j) acc += lam[((size_t)j * n_units + u) * nl + i];
                lam_total[(size_t)u * nl + i] = acc;
            }
            if (!dense || !nxt) continue;
            double *cur = P_total + (size_t)u * d_k * d_k;
            memcpy(cur, P + (size_t)u * d_k * d_k, sizeof(double) * d_k * d_k);
            for (int j = 1; j < n_seg; ++j) {
                const double *Pj = P + ((size_t)j * n_units + u) * d_k * d_k;
                for (int i = 0; i < d_k; ++i)
                    for (int c = 0; c < d_k; ++c) {
                        double acc = 0.0;
                        for (int m = 0; m < d_k; ++m) acc += Pj[(size_t)i * d_k + m] * cur[(size_t)m * d_k + c];
                        nxt[(size_t)i * d_k + c] = acc;
                    }
                memcpy(cur, nxt, sizeof(double) * d_k * d_k);
            }
        }
        free(nxt);
    }
    return err;
}

/* o_t = S_t^T q_t for every token of every segment and value head: the recurrence stepped
 * token by token from S_init[seg][h] (NULL = zero), the output read after each token's
 * update. q [N_tok][H_k][d_k] (value head h reads key head h / (H_v / H_k)); O_out
 * [N_tok][H_v][d_v]. */
int oracle_outputs(int family, int n_seg, const int64_t *seg_offsets, int H_k, int H_v, int d_k,
                   int d_v, const double *k, const double *v, const double *q, const double *log_gate,
                   const double *log_gamma, const double *beta, const double *S_init, double *O_out,
                   int nthreads) {
    if (check_shape(family, H_k, H_v, d_k, d_v)) return -1;
    recurrence r = {family, H_k, H_v, d_k, d_v, k, v, log_gate, log_gamma, beta};
    set_threads(nthreads);
    const int64_t units = (int64_t)n_seg * H_v;
    int err = 0;
#pragma omp parallel
    {
        int wn = d_k > d_v ? d_k : d_v;
        double *w = (double *)malloc(sizeof(double) * wn);
        double *S = (double *)malloc(sizeof(double) * d_k * d_v);
        if (!w || !S) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            if (!w || !S) continue;
            int seg = (int)(u / H_v), h = (int)(u % H_v);
            const int hk = h / (H_v / H_k);
            if (S_init) memcpy(S, S_init + (size_t)u * d_k * d_v, sizeof(double) * d_k * d_v);
            else memset(S, 0, sizeof(double) * d_k * d_v);
            for (int64_t t = seg_offsets[seg]; t < seg_offsets[seg + 1]; ++t) {
                apply_factor(&r, t, h, S, d_v, w);
                add_write(&r, t, h, S);
                const double *qt = q + ((size_t)t * H_k + hk) * d_k;
                double *o = O_out + ((size_t)t * H_v + h) * d_v;
                for (int n = 0; n < d_v; ++n) {
                    double acc = 0.0;
                    for (int i = 0; i < d_k; ++i) acc += S[(size_t)i * d_v + n] * qt[i];
                    o[n] = acc;
                }
            }
        }
        free(w);
        free(S);
    }
    return err;
}

int oracle_version(void) { return 3; }
