/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for the exact attention
 * forward pass  O = softmax(scale * Q K^T [+ causal mask]) V,  LSE = m + log(l).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle for the CUDA
 * path.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library, and the CUDA library never calls it.
 *
 * What it follows (citations name the web page and the section on it):
 *   - "Chapter 26 Online Softmax & FlashAttention" (gowda.ai), Listing 26.2
 *     "Naive attention materializes the score matrix": scores = q k^T/sqrt(d),
 *     causal keeps key j for query i iff j <= i, row-wise stable softmax,
 *     output = weights @ v.  Equation (26.1): m = max_i s_i,
 *     l = sum_i exp(s_i - m).
 *   - "Understanding FlashAttention Pt 1" (wpnews.pro), section 2.2: the
 *     stable softmax p_j = exp(x_j - m) / l.
 *   - "FlashAttention-2 -- Deeper Math" (aicassindra.com), "Fix 2": the
 *     per-row statistic L = m + log(l), natural log, in scaled-score units.
 *
 * fa_oracle_fwd() is the plain definition, written out.  For each query row
 * it materialises the score row S[i][*] and the probability row P[i][*]
 * (fp64), in chunks of rows (rows of a softmax are independent, so this
 * changes no arithmetic).  Steps, in the pages' order:
 *   1. S[i][j] = scale * sum_k Q[i][k] * K[j][k]
 *   2. causal: S[i][j] = -inf for j > i
 *   3. m_i = max_j S[i][j];  P[i][j] = exp(S[i][j] - m_i);  l_i = sum_j P[i][j]
 *   4. O[i] = (sum_j P[i][j] * V[j]) / l_i;  LSE_i = m_i + log(l_i)
 * A row whose every score is masked has no softmax; it is defined here as
 * O = 0, LSE = -inf (the "has_scores" guard of Listing 26.3 treats such a
 * block as contributing nothing).
 *
 * fa_oracle_fwd_blockwise() is the online (blockwise) recurrence, used only
 * by the oracle's own self-tests ("blockwise == dense for any split").  It
 * follows "Understanding FlashAttention Pt 1", section 2.4 "The Blockwise
 * Merge Recurrence": m_b = max(s), m' = max(m, m_b), alpha = exp(m - m'),
 * p = exp(s - m'), l' = alpha*l + sum p, a' = alpha*a + p^T V_b, and o = a/l
 * at the end; plus the fully-masked-block guard of gowda.ai Listing 26.3.
 *
 * Layouts: Q, K are [BH, N, d]; V is [BH, N, dv]; all row-major fp64.
 * fa_oracle_fwd_q() takes Q as [BH, Nq, d] with Nq <= N query rows that
 * sit at the last Nq positions (decoding: Nq = 1 is the newest token).
 * rows == NULL computes every query row: O is [BH, N, dv], LSE is [BH, N].
 * rows != NULL is a [BH, R] table of query indices: O is [BH, R, dv],
 * LSE is [BH, R].  Work is spread over nthreads POSIX threads; each output
 * row is produced by exactly one thread in a fixed order, so results do not
 * depend on the thread count.
 *
 * Return value: 0 on success, -1 on a bad argument, -2 on allocation failure.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ROW_CHUNK 64

/* bf16 bit pattern -> fp64.  bf16 is the upper half of an IEEE binary32, so
 * widening the bits and reinterpreting is exact. */
int fa_oracle_bf16_to_f64(const uint16_t *src, double *dst, int64_t n) {
    if (!src || !dst || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t bits = ((uint32_t)src[i]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        dst[i] = (double)f;
    }
    return 0;
}

typedef struct {
    const double *Q, *K, *V;
    double *O, *LSE;
    int64_t BH, N, d, dv, R;
    int64_t Nq;   /* query rows per head (== N for self-attention) */
    const int64_t *rows; /* NULL -> all rows */
    int causal;
    double scale;
    /* blockwise only */
    const int64_t *bounds;
    int64_t nblocks;
    int reverse;
    double *M_out, *L_out, *A_out;
    /* work distribution */
    int64_t n_items, chunks_per_head;
    int64_t next; /* atomic counter */
    int failed;
} oracle_job;

static int64_t query_index(const oracle_job *jb, int64_t bh, int64_t r) {
    return jb->rows ? jb->rows[bh * jb->R + r] : r;
}

/* One chunk of query rows of one (b,h): the materialised definition. */
static int dense_chunk(oracle_job *jb, int64_t bh, int64_t r0, int64_t r1,
                       double *S, double *P) {
    const int64_t N = jb->N, d = jb->d, dv = jb->dv;
    const double *Qh = jb->Q + bh * jb->Nq * d;
    const double *Kh = jb->K + bh * N * d;
    const double *Vh = jb->V + bh * N * dv;
    const int64_t nr = r1 - r0;

    /* step 1: scores, and step 2: causal mask */
    for (int64_t r = 0; r < nr; ++r) {
        const int64_t i = query_index(jb, bh, r0 + r);
        const double *q = Qh + i * d;
        for (int64_t j = 0; j < N; ++j) {
            double dot = 0.0;
            const double *k = Kh + j * d;
            for (int64_t c = 0; c < d; ++c) dot += q[c] * k[c];
            S[r * N + j] = jb->scale * dot;
            /* query row i sits at key position i + (N - Nq) */
            if (jb->causal && j > i + (N - jb->Nq)) S[r * N + j] = -INFINITY;
        }
    }
    /* step 3: row max, probabilities, normaliser;  step 4: output, LSE */
    for (int64_t r = 0; r < nr; ++r) {
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (S[r * N + j] > m) m = S[r * N + j];
        double *o = jb->O + (bh * jb->R + r0 + r) * dv;
        double *lse = jb->LSE + bh * jb->R + r0 + r;
        if (m == -INFINITY) { /* every key masked: no softmax */
            for (int64_t c = 0; c < dv; ++c) o[c] = 0.0;
            *lse = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            P[r * N + j] = exp(S[r * N + j] - m);
            l += P[r * N + j];
        }
        for (int64_t c = 0; c < dv; ++c) o[c] = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double p = P[r * N + j];
            const double *v = Vh + j * dv;
            for (int64_t c = 0; c < dv; ++c) o[c] += p * v[c];
        }
        for (int64_t c = 0; c < dv; ++c) o[c] /= l;
        *lse = m + log(l);
    }
    return 0;
}

/* One query row through the blockwise merge recurrence. */
static void blockwise_row(oracle_job *jb, int64_t bh, int64_t r, double *s,
                          double *a) {
    const int64_t N = jb->N, d = jb->d, dv = jb->dv;
    const int64_t i = query_index(jb, bh, r);
    const double *q = jb->Q + (bh * jb->Nq + i) * d;
    const double *Kh = jb->K + bh * N * d;
    const double *Vh = jb->V + bh * N * dv;

    double m = -INFINITY, l = 0.0;
    for (int64_t c = 0; c < dv; ++c) a[c] = 0.0;

    for (int64_t t = 0; t < jb->nblocks; ++t) {
        const int64_t b = jb->reverse ? jb->nblocks - 1 - t : t;
        const int64_t j0 = jb->bounds[b], j1 = jb->bounds[b + 1];
        /* the block's scores, masked, and its max m_b */
        double m_b = -INFINITY;
        for (int64_t j = j0; j < j1; ++j) {
            double dot = 0.0;
            const double *k = Kh + j * d;
            for (int64_t c = 0; c < d; ++c) dot += q[c] * k[c];
            s[j - j0] = (jb->causal && j > i + (N - jb->Nq)) ? -INFINITY : jb->scale * dot;
            if (s[j - j0] > m_b) m_b = s[j - j0];
        }
        if (m_b == -INFINITY) continue; /* block has no scores: no change */
        const double m_new = m > m_b ? m : m_b;
        const double alpha = exp(m - m_new); /* m = -inf gives 0 */
        double sum_p = 0.0;
        for (int64_t c = 0; c < dv; ++c) a[c] *= alpha;
        for (int64_t j = j0; j < j1; ++j) {
            const double p = exp(s[j - j0] - m_new);
            sum_p += p;
            const double *v = Vh + j * dv;
            for (int64_t c = 0; c < dv; ++c) a[c] += p * v[c];
        }
        l = alpha * l + sum_p;
        m = m_new;
    }
    const int64_t out = bh * jb->R + r;
    double *o = jb->O + out * dv;
    if (l == 0.0) {
        for (int64_t c = 0; c < dv; ++c) o[c] = 0.0;
        jb->LSE[out] = -INFINITY;
    } else {
        for (int64_t c = 0; c < dv; ++c) o[c] = a[c] / l;
        jb->LSE[out] = m + log(l);
    }
    if (jb->M_out) jb->M_out[out] = m;
    if (jb->L_out) jb->L_out[out] = l;
    if (jb->A_out)
        for (int64_t c = 0; c < dv; ++c) jb->A_out[out * dv + c] = a[c];
}

static void *dense_worker(void *arg) {
    oracle_job *jb = (oracle_job *)arg;
    const int64_t N = jb->N;
    double *S = (double *)malloc(sizeof(double) * ORACLE_ROW_CHUNK * (size_t)N);
    double *P = (double *)malloc(sizeof(double) * ORACLE_ROW_CHUNK * (size_t)N);
    if (!S || !P) {
        __atomic_store_n(&jb->failed, 1, __ATOMIC_SEQ_CST);
        free(S);
        free(P);
        return NULL;
    }
    for (;;) {
        const int64_t item = __atomic_fetch_add(&jb->next, 1, __ATOMIC_SEQ_CST);
        if (item >= jb->n_items) break;
        const int64_t bh = item / jb->chunks_per_head;
        const int64_t r0 = (item % jb->chunks_per_head) * ORACLE_ROW_CHUNK;
        const int64_t r1 = r0 + ORACLE_ROW_CHUNK < jb->R ? r0 + ORACLE_ROW_CHUNK : jb->R;
        dense_chunk(jb, bh, r0, r1, S, P);
    }
    free(S);
    free(P);
    return NULL;
}

static void *blockwise_worker(void *arg) {
    oracle_job *jb = (oracle_job *)arg;
    int64_t widest = 1;
    for (int64_t b = 0; b < jb->nblocks; ++b)
        if (jb->bounds[b + 1] - jb->bounds[b] > widest)
            widest = jb->bounds[b + 1] - jb->bounds[b];
    double *s = (double *)malloc(sizeof(double) * (size_t)widest);
    double *a = (double *)malloc(sizeof(double) * (size_t)(jb->dv > 0 ? jb->dv : 1));
    if (!s || !a) {
        __atomic_store_n(&jb->failed, 1, __ATOMIC_SEQ_CST);
        free(s);
        free(a);
        return NULL;
    }
    for (;;) {
        const int64_t item = __atomic_fetch_add(&jb->next, 1, __ATOMIC_SEQ_CST);
        if (item >= jb->n_items) break;
        const int64_t bh = item / jb->chunks_per_head;
        const int64_t r0 = (item % jb->chunks_per_head) * ORACLE_ROW_CHUNK;
        const int64_t r1 = r0 + ORACLE_ROW_CHUNK < jb->R ? r0 + ORACLE_ROW_CHUNK : jb->R;
        for (int64_t r = r0; r < r1; ++r) blockwise_row(jb, bh, r, s, a);
    }
    free(s);
    free(a);
    return NULL;
}

static int run_threads(oracle_job *jb, void *(*fn)(void *), int nthreads) {
    jb->chunks_per_head = (jb->R + ORACLE_ROW_CHUNK - 1) / ORACLE_ROW_CHUNK;
    jb->n_items = jb->BH * jb->chunks_per_head;
    jb->next = 0;
    jb->failed = 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > jb->n_items) nthreads = (int)(jb->n_items > 0 ? jb->n_items : 1);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) return -2;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, jb) != 0) break;
        ++started;
    }
    if (started == 0) fn(jb); /* no thread could start: run inline */
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    return jb->failed ? -2 : 0;
}

static int check_common(const double *Q, const double *K, const double *V,
                        const double *O, const double *LSE, int64_t BH,
                        int64_t Nq, int64_t N, int64_t d, int64_t dv,
                        const int64_t *rows, int64_t R) {
    if (!Q || !K || !V || !O || !LSE) return -1;
    if (BH < 1 || N < 1 || Nq < 1 || Nq > N || d < 1 || dv < 1) return -1;
    if (rows) {
        if (R < 1) return -1;
        for (int64_t t = 0; t < BH * R; ++t)
            if (rows[t] < 0 || rows[t] >= Nq) return -1;
    }
    return 0;
}

/* Nq query rows (Q is [BH, Nq, d]) against N keys (K, V are [BH, N, *]),
 * Nq <= N.  Causal keeps key j for query row i iff j <= i + (N - Nq): the
 * query rows are the last Nq positions of the sequence (with Nq == N this
 * is j <= i).  rows index the Nq query rows. */
int fa_oracle_fwd_q(const double *Q, const double *K, const double *V, double *O,
                    double *LSE, int64_t BH, int64_t Nq, int64_t N, int64_t d, int64_t dv,
                    int causal, double scale, const int64_t *rows, int64_t R,
                    int nthreads) {
    if (check_common(Q, K, V, O, LSE, BH, Nq, N, d, dv, rows, R)) return -1;
    oracle_job jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = Q; jb.K = K; jb.V = V; jb.O = O; jb.LSE = LSE;
    jb.BH = BH; jb.N = N; jb.Nq = Nq; jb.d = d; jb.dv = dv;
    jb.rows = rows; jb.R = rows ? R : Nq;
    jb.causal = causal ? 1 : 0; jb.scale = scale;
    return run_threads(&jb, dense_worker, nthreads);
}

int fa_oracle_fwd(const double *Q, const double *K, const double *V, double *O,
                  double *LSE, int64_t BH, int64_t N, int64_t d, int64_t dv,
                  int causal, double scale, const int64_t *rows, int64_t R,
                  int nthreads) {
    return fa_oracle_fwd_q(Q, K, V, O, LSE, BH, N, N, d, dv, causal, scale, rows, R,
                           nthreads);
}

int fa_oracle_fwd_blockwise(const double *Q, const double *K, const double *V,
                            double *O, double *LSE, int64_t BH, int64_t N,
                            int64_t d, int64_t dv, int causal, double scale,
                            const int64_t *rows, int64_t R,
                            const int64_t *bounds, int64_t nblocks, int reverse,
                            double *M_out, double *L_out, double *A_out,
                            int nthreads) {
    if (check_common(Q, K, V, O, LSE, BH, N, N, d, dv, rows, R)) return -1;
    if (!bounds || nblocks < 1 || bounds[0] != 0 || bounds[nblocks] != N) return -1;
    for (int64_t b = 0; b < nblocks; ++b)
        if (bounds[b + 1] <= bounds[b]) return -1;
    oracle_job jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = Q; jb.K = K; jb.V = V; jb.O = O; jb.LSE = LSE;
    jb.BH = BH; jb.N = N; jb.d = d; jb.dv = dv;
    jb.rows = rows; jb.R = rows ? R : N; jb.Nq = N;
    jb.causal = causal ? 1 : 0; jb.scale = scale;
    jb.bounds = bounds; jb.nblocks = nblocks; jb.reverse = reverse ? 1 : 0;
    jb.M_out = M_out; jb.L_out = L_out; jb.A_out = A_out;
    return run_threads(&jb, blockwise_worker, nthreads);
}

/*
 * fa_oracle_bwd -- gradients of the attention forward pass, by the plain
 * definition ("Understanding FlashAttention Pt 1", section 3.6 "Backward
 * Pass: Recompute Instead of Save"), materialised in fp64 per (b, h):
 *   S = scale * Q K^T (causal: S_ij = -inf for j > i), P = softmax_rows(S),
 *   O = P V, dV = P^T dO, dP = dO V^T, D_i = sum_r dO_ir O_ir,
 *   dS = P * (dP - D_i), dQ = scale * dS K, dK = scale * dS^T Q.
 * O is recomputed here from Q, K, V (not taken from the caller).
 * D_in (optional, may be NULL) replaces the D_i computed from that exact O
 * by the caller's values: the same gradients with D taken from another O,
 * e.g. the forward's output rounded to bf16 (tests use it to size the
 * effect of that rounding on the gradients).
 * Layouts: Q, K, V, dO, dQ, dK, dV are [BH, N, d] fp64; D_out and D_in
 * (optional, may be NULL) are [BH, N].  Returns 0, -1 (bad argument) or -2
 * (memory).
 */
typedef struct {
    const double *Q, *K, *V, *dO;
    double *dQ, *dK, *dV, *D_out;
    const double *D_in;
    int64_t BH, N, d;
    int causal;
    double scale;
    int64_t next;
    int failed;
} bwd_job;

static void bwd_head(bwd_job *jb, int64_t bh, double *S, double *P, double *dP) {
    const int64_t N = jb->N, d = jb->d;
    const double *Q = jb->Q + bh * N * d, *K = jb->K + bh * N * d, *V = jb->V + bh * N * d;
    const double *dO = jb->dO + bh * N * d;
    double *dQ = jb->dQ + bh * N * d, *dK = jb->dK + bh * N * d, *dV = jb->dV + bh * N * d;
    /* forward: S, P (row softmax), O = P V is folded into D below */
    for (int64_t i = 0; i < N; ++i) {
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += Q[i * d + c] * K[j * d + c];
            S[i * N + j] = (jb->causal && j > i) ? -INFINITY : jb->scale * dot;
            if (S[i * N + j] > m) m = S[i * N + j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            P[i * N + j] = (m == -INFINITY) ? 0.0 : exp(S[i * N + j] - m);
            l += P[i * N + j];
        }
        for (int64_t j = 0; j < N; ++j) P[i * N + j] = (l > 0.0) ? P[i * N + j] / l : 0.0;
    }
    /* dP = dO V^T */
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += dO[i * d + c] * V[j * d + c];
            dP[i * N + j] = dot;
        }
    /* D_i = sum_r dO_ir O_ir with O = P V */
    for (int64_t i = 0; i < N; ++i) {
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            double o = 0.0;
            for (int64_t j = 0; j < N; ++j) o += P[i * N + j] * V[j * d + c];
            Di += dO[i * d + c] * o;
        }
        if (jb->D_in) Di = jb->D_in[bh * N + i];
        if (jb->D_out) jb->D_out[bh * N + i] = Di;
        /* dS overwrites dP */
        for (int64_t j = 0; j < N; ++j) dP[i * N + j] = P[i * N + j] * (dP[i * N + j] - Di);
    }
    /* dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K */
    for (int64_t j = 0; j < N; ++j)
        for (int64_t c = 0; c < d; ++c) {
            double v = 0.0, k = 0.0;
            for (int64_t i = 0; i < N; ++i) {
                v += P[i * N + j] * dO[i * d + c];
                k += dP[i * N + j] * Q[i * d + c];
            }
            dV[j * d + c] = v;
            dK[j * d + c] = jb->scale * k;
        }
    for (int64_t i = 0; i < N; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double q = 0.0;
            for (int64_t j = 0; j < N; ++j) q += dP[i * N + j] * K[j * d + c];
            dQ[i * d + c] = jb->scale * q;
        }
}

static void *bwd_worker(void *arg) {
    bwd_job *jb = (bwd_job *)arg;
    const size_t nn = (size_t)jb->N * (size_t)jb->N;
    double *S = (double *)malloc(sizeof(double) * nn);
    double *P = (double *)malloc(sizeof(double) * nn);
    double *dP = (double *)malloc(sizeof(double) * nn);
    if (!S || !P || !dP) {
        __atomic_store_n(&jb->failed, 1, __ATOMIC_SEQ_CST);
    } else {
        for (;;) {
            const int64_t bh = __atomic_fetch_add(&jb->next, 1, __ATOMIC_SEQ_CST);
            if (bh >= jb->BH) break;
            bwd_head(jb, bh, S, P, dP);
        }
    }
    free(S);
    free(P);
    free(dP);
    return NULL;
}

int fa_oracle_bwd(const double *Q, const double *K, const double *V, const double *dO,
                  double *dQ, double *dK, double *dV, double *D_out, const double *D_in,
                  int64_t BH, int64_t N, int64_t d, int causal, double scale, int nthreads) {
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return -1;
    if (BH < 1 || N < 1 || d < 1) return -1;
    bwd_job jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = Q; jb.K = K; jb.V = V; jb.dO = dO;
    jb.dQ = dQ; jb.dK = dK; jb.dV = dV; jb.D_out = D_out; jb.D_in = D_in;
    jb.BH = BH; jb.N = N; jb.d = d; jb.causal = causal ? 1 : 0; jb.scale = scale;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = (int)BH;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, bwd_worker, &jb) != 0) break;
        ++started;
    }
    if (started == 0) bwd_worker(&jb);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    return jb.failed ? -2 : 0;
}
