/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the attention forward pass that the
 * fused GPU kernel computes.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the product path never does.
 * It shares no code, header or helper with the CUDA library.
 *
 * What it computes (per batch b, head h, query row i), written out as the
 * plain definition of softmax attention with a per-row log-sum-exp:
 *
 *   J_i    = {0..Nkv-1}                  (non-causal)
 *          = {0..i + Nkv - Nq}           (causal: key j may be seen by query i iff
 *                                          j <= i + Nkv - Nq)
 *   s_ij   = scale * sum_d Q[i,d] * K[j,d]                 for j in J_i
 *   m_i    = max_j s_ij
 *   l_i    = sum_j exp(s_ij - m_i)
 *   LSE_i  = m_i + ln(l_i)                                 (natural log, scale included)
 *   O[i,d] = (sum_j exp(s_ij - m_i) * V[j,d]) / l_i
 *
 * Sources: "ThunderKittens" attention kernel as printed on the page
 * 10100.com/article/71410160, section "writing a kernel with TK"
 * (attn_fwd_template, consumer::compute forms Q K^T, takes the row max,
 * exponentiates, accumulates the row sum and P V; consumer::finish divides
 * by the row sum once); alanwu.xyz/posts/thunderkittens, the attention inner
 * loop excerpt (same steps, with the ragged key tail filled with -inf so that
 * keys past the sequence end take no weight).  The pages compute the
 * exponentials in base 2 with scale*log2(e) folded in; that is the same
 * number as exp() of the scaled score, so the definition is written with
 * exp/log here.  The pages store no LSE; the reading taken is
 * LSE = scale*max + ln(sum), in natural log.  The causal mask is not on the
 * pages; the reading taken is key j <= query i when queries and keys have
 * the same length N.  Nq queries against a longer sequence of Nkv keys
 * (attention inference over a cache, listed among the kernels on the
 * groovesquid.com summary of the ThunderKittens paper) place the queries at
 * the end of the key sequence: query i stands at position i + Nkv - Nq.
 * Causal problems need Nkv >= Nq, so that every query sees a key.
 *
 * Two passes, no streaming, no tiling, no blocking: pass 1 forms every score
 * of the row and its maximum, pass 2 forms the weights, their sum and the
 * weighted sum of V.  Inputs are bf16 bit patterns, converted exactly to
 * double.  Outputs are double.
 *
 * Parallelism: independent rows are handed to POSIX threads; each row is
 * computed by exactly one thread with the same loop order, so the result
 * does not depend on the thread count.
 *
 * The file also holds the backward's chain rule and the plain GEMM that the
 * same tile pipeline runs (at the end).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row of one head.  q: D values; K, V: Nkv x D (double, row-major);
 * offset = Nkv - Nq.  s: scratch of Nkv doubles. */
static void attention_row(const double *q, const double *K, const double *V,
                          int64_t Nkv, int64_t D, int causal, int64_t offset, double scale,
                          int64_t i, double *s, double *o_row, double *lse_out) {
    int64_t nkeys = causal ? (i + offset + 1) : Nkv;
    if (nkeys > Nkv) nkeys = Nkv;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double *k = K + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += q[d] * k[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }

    /* pass 2: weights, their sum, and the weighted sum of V rows */
    double l = 0.0;
    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        double p = exp(s[j] - m);
        l += p;
        const double *v = V + j * D;
        for (int64_t d = 0; d < D; ++d) o_row[d] += p * v[d];
    }
    for (int64_t d = 0; d < D; ++d) o_row[d] /= l;
    *lse_out = m + log(l);
}

/* ------------------------------------------------------------------------ */
/* work distribution                                                         */

typedef struct {
    /* one head, already widened to double */
    const double *Q, *K, *V;
    int64_t Nq, Nkv, D;
    int causal;
    double scale;
    const int64_t *rows; /* NULL: all rows 0..Nq-1 */
    int64_t nrows;
    double *O;   /* nrows x D */
    double *LSE; /* nrows */
    int64_t next;
    pthread_mutex_t lock;
} head_job;

static void *head_worker(void *arg) {
    head_job *job = (head_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(job->Nkv > 0 ? job->Nkv : 1));
    if (!s) return NULL;
    const int64_t chunk = 8;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t begin = job->next;
        job->next += chunk;
        pthread_mutex_unlock(&job->lock);
        if (begin >= job->nrows) break;
        int64_t end = begin + chunk < job->nrows ? begin + chunk : job->nrows;
        for (int64_t r = begin; r < end; ++r) {
            int64_t i = job->rows ? job->rows[r] : r;
            attention_row(job->Q + i * job->D, job->K, job->V, job->Nkv, job->D, job->causal,
                          job->Nkv - job->Nq, job->scale, i, s, job->O + r * job->D, job->LSE + r);
        }
    }
    free(s);
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int g_last_threads = 0;

/* Computes the listed rows of one head.  Returns 0, or -1 on bad arguments or
 * allocation failure. */
static int run_head(const uint16_t *Qb, const uint16_t *Kb, const uint16_t *Vb, int64_t Nq,
                    int64_t Nkv, int64_t D, int causal, double scale, const int64_t *rows,
                    int64_t nrows, double *O, double *LSE, int nthreads) {
    size_t nq = (size_t)Nq * (size_t)D, nkv = (size_t)Nkv * (size_t)D;
    double *Q = (double *)malloc(sizeof(double) * nq);
    double *K = (double *)malloc(sizeof(double) * nkv);
    double *V = (double *)malloc(sizeof(double) * nkv);
    if (!Q || !K || !V) {
        free(Q); free(K); free(V);
        return -1;
    }
    for (size_t t = 0; t < nq; ++t) Q[t] = bf16_bits_to_double(Qb[t]);
    for (size_t t = 0; t < nkv; ++t) {
        K[t] = bf16_bits_to_double(Kb[t]);
        V[t] = bf16_bits_to_double(Vb[t]);
    }
    head_job job;
    job.Q = Q; job.K = K; job.V = V;
    job.Nq = Nq; job.Nkv = Nkv; job.D = D; job.causal = causal; job.scale = scale;
    job.rows = rows; job.nrows = nrows; job.O = O; job.LSE = LSE;
    job.next = 0;
    pthread_mutex_init(&job.lock, NULL);

    int T = resolve_threads(nthreads);
    if ((int64_t)T > (nrows + 7) / 8) T = (int)((nrows + 7) / 8);
    if (T < 1) T = 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)T);
    int started = 0;
    for (int t = 1; tid && t < T; ++t) {
        if (pthread_create(&tid[started], NULL, head_worker, &job) != 0) break;
        ++started;
    }
    if (started + 1 > g_last_threads) g_last_threads = started + 1;
    head_worker(&job); /* the calling thread works too */
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    free(Q); free(K); free(V);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* exported entry points                                                     */

/* Whole problem.  Q: bf16 bits, contiguous [B,H,Nq,D]; K, V: [B,H,Nkv,D].
 * O: double [B,H,Nq,D].  LSE: double [B,H,Nq].  nthreads <= 0: all online CPUs.
 * Causal problems need Nkv >= Nq. */
int tkor_attn_fwd_kv(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O,
                     double *LSE, int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D,
                     int causal, double scale, int nthreads) {
    if (!Q || !K || !V || !O || !LSE || B < 1 || H < 1 || Nq < 1 || Nkv < 1 || D < 1) return -1;
    if (causal && Nkv < Nq) return -1;
    g_last_threads = 0;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        size_t qoff = (size_t)bh * (size_t)Nq * (size_t)D;
        size_t kvoff = (size_t)bh * (size_t)Nkv * (size_t)D;
        if (run_head(Q + qoff, K + kvoff, V + kvoff, Nq, Nkv, D, causal, scale, NULL, Nq,
                     O + qoff, LSE + (size_t)bh * (size_t)Nq, nthreads))
            return -1;
    }
    return 0;
}

/* The same-length problem: Nq = Nkv = N. */
int tkor_attn_fwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O,
                  double *LSE, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                  double scale, int nthreads) {
    return tkor_attn_fwd_kv(Q, K, V, O, LSE, B, H, N, N, D, causal, scale, nthreads);
}

/* Selected rows of one head.  Q: bf16 bits [Nq,D] of that head; K, V:
 * [Nkv,D].  rows: nrows query indices in [0,Nq).  O: double [nrows,D];
 * LSE: double [nrows]. */
int tkor_attn_fwd_kv_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t Nq,
                          int64_t Nkv, int64_t D, int causal, double scale, const int64_t *rows,
                          int64_t nrows, double *O, double *LSE, int nthreads) {
    if (!Q || !K || !V || !O || !LSE || !rows || Nq < 1 || Nkv < 1 || D < 1 || nrows < 0)
        return -1;
    if (causal && Nkv < Nq) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= Nq) return -1;
    g_last_threads = 0;
    return run_head(Q, K, V, Nq, Nkv, D, causal, scale, rows, nrows, O, LSE, nthreads);
}

int tkor_attn_fwd_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t N,
                       int64_t D, int causal, double scale, const int64_t *rows,
                       int64_t nrows, double *O, double *LSE, int nthreads) {
    return tkor_attn_fwd_kv_rows(Q, K, V, N, N, D, causal, scale, rows, nrows, O, LSE, nthreads);
}

/* The attention weights of one head, P[i,j] = exp(s_ij - m_i) / l_i, with
 * P[i,j] = 0 for masked keys.  Q, K: bf16 bits [N,D].  P: double [N,N].
 * Meant for tiny N (it materialises the N x N matrix). */
int tkor_attn_weights(const uint16_t *Qb, const uint16_t *Kb, int64_t N, int64_t D,
                      int causal, double scale, double *P) {
    if (!Qb || !Kb || !P || N < 1 || D < 1) return -1;
    for (int64_t i = 0; i < N; ++i) {
        int64_t nkeys = causal ? i + 1 : N;
        double m = -INFINITY;
        double *row = P + i * N;
        for (int64_t j = 0; j < N; ++j) row[j] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dot += bf16_bits_to_double(Qb[i * D + d]) * bf16_bits_to_double(Kb[j * D + d]);
            row[j] = scale * dot;
            if (row[j] > m) m = row[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            row[j] = exp(row[j] - m);
            l += row[j];
        }
        for (int64_t j = 0; j < nkeys; ++j) row[j] /= l;
    }
    return 0;
}

/* Largest number of threads used by the last call. */
int tkor_last_threads(void) { return g_last_threads; }

/* ======================================================================== */
/* Backward pass                                                             */
/*
 * The gradient of L = sum_{i,d} O[i,d] * dO[i,d] with respect to Q, K, V,
 * where O is the forward output above.  Written out from the definition of
 * softmax attention (the pages list attention backwards among the kernels
 * built with the same tiles: groovesquid.com summary of the ThunderKittens
 * paper; the quantities are the plain chain rule through the softmax):
 *
 *   p_ij   = exp(s_ij - m_i) / l_i            (the forward weights, j in J_i)
 *   dV_j   = sum_i p_ij dO_i
 *   dP_ij  = <dO_i, V_j>
 *   dS_ij  = p_ij (dP_ij - sum_k p_ik dP_ik)   (softmax Jacobian applied to dP)
 *   dQ_i   = scale * sum_j dS_ij K_j
 *   dK_j   = scale * sum_i dS_ij Q_i
 *
 * Computed per head, one query row at a time, in fp64 from the bf16 inputs
 * widened exactly.  Rows are split over threads; each thread accumulates
 * its own dK and dV partial sums, which are added at the end in thread
 * order (so the result does not depend on scheduling, only on the thread
 * count through the final summation order, to within rounding).
 */

typedef struct {
    const double *Q, *K, *V, *dO;
    int64_t N, D;
    int causal;
    double scale;
    double *dQ;            /* N x D, written by the thread owning the row */
    double *dK_part;       /* T x N x D */
    double *dV_part;       /* T x N x D */
    int T;
    int tid;
} bwd_job;

static void *bwd_worker(void *arg) {
    bwd_job *job = (bwd_job *)arg;
    const int64_t N = job->N, D = job->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *dp = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s || !dp) {
        free(s); free(dp);
        return NULL;
    }
    double *dK = job->dK_part + (size_t)job->tid * (size_t)N * (size_t)D;
    double *dV = job->dV_part + (size_t)job->tid * (size_t)N * (size_t)D;
    for (int64_t i = job->tid; i < N; i += job->T) {
        const double *q = job->Q + i * D;
        const double *g = job->dO + i * D;
        int64_t nkeys = job->causal ? i + 1 : N;
        /* forward weights of row i */
        double m = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += q[d] * job->K[j * D + d];
            s[j] = job->scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (int64_t j = 0; j < nkeys; ++j) s[j] /= l; /* s now holds p_ij */
        /* dP and the softmax Jacobian term */
        double pdp = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += g[d] * job->V[j * D + d];
            dp[j] = dot;
            pdp += s[j] * dot;
        }
        double *dq = job->dQ + i * D;
        for (int64_t d = 0; d < D; ++d) dq[d] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double ds = s[j] * (dp[j] - pdp);
            for (int64_t d = 0; d < D; ++d) {
                dq[d] += job->scale * ds * job->K[j * D + d];
                dK[j * D + d] += job->scale * ds * q[d];
                dV[j * D + d] += s[j] * g[d];
            }
        }
    }
    free(s); free(dp);
    return NULL;
}

/* Q, K, V, dO: bf16 bits [B,H,N,D].  dQ, dK, dV: double [B,H,N,D]. */
int tkor_attn_bwd(const uint16_t *Qb, const uint16_t *Kb, const uint16_t *Vb, const uint16_t *dOb,
                  double *dQ, double *dK, double *dV, int64_t B, int64_t H, int64_t N, int64_t D,
                  int causal, double scale, int nthreads) {
    if (!Qb || !Kb || !Vb || !dOb || !dQ || !dK || !dV || B < 1 || H < 1 || N < 1 || D < 1)
        return -1;
    int T = resolve_threads(nthreads);
    if ((int64_t)T > N) T = (int)N;
    const size_t n = (size_t)N * (size_t)D;
    double *buf = (double *)malloc(sizeof(double) * n * 4);
    double *dKp = (double *)malloc(sizeof(double) * n * (size_t)T);
    double *dVp = (double *)malloc(sizeof(double) * n * (size_t)T);
    bwd_job *jobs = (bwd_job *)malloc(sizeof(bwd_job) * (size_t)T);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)T);
    if (!buf || !dKp || !dVp || !jobs || !tid) {
        free(buf); free(dKp); free(dVp); free(jobs); free(tid);
        return -1;
    }
    g_last_threads = T;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const size_t off = (size_t)bh * n;
        double *Q = buf, *K = buf + n, *V = buf + 2 * n, *G = buf + 3 * n;
        for (size_t t = 0; t < n; ++t) {
            Q[t] = bf16_bits_to_double(Qb[off + t]);
            K[t] = bf16_bits_to_double(Kb[off + t]);
            V[t] = bf16_bits_to_double(Vb[off + t]);
            G[t] = bf16_bits_to_double(dOb[off + t]);
        }
        memset(dKp, 0, sizeof(double) * n * (size_t)T);
        memset(dVp, 0, sizeof(double) * n * (size_t)T);
        for (int t = 0; t < T; ++t) {
            jobs[t].Q = Q; jobs[t].K = K; jobs[t].V = V; jobs[t].dO = G;
            jobs[t].N = N; jobs[t].D = D; jobs[t].causal = causal; jobs[t].scale = scale;
            jobs[t].dQ = dQ + off; jobs[t].dK_part = dKp; jobs[t].dV_part = dVp;
            jobs[t].T = T; jobs[t].tid = t;
        }
        /* thread t >= 1 runs on its own pthread when one can be started,
           otherwise inline; each writes only its own partial buffers */
        unsigned char *spawned = (unsigned char *)calloc((size_t)T, 1);
        for (int t = 1; t < T; ++t) {
            if (spawned && pthread_create(&tid[t], NULL, bwd_worker, &jobs[t]) == 0)
                spawned[t] = 1;
            else
                bwd_worker(&jobs[t]);
        }
        bwd_worker(&jobs[0]);
        for (int t = 1; t < T; ++t)
            if (spawned && spawned[t]) pthread_join(tid[t], NULL);
        free(spawned);
        for (size_t e = 0; e < n; ++e) {
            double a = 0.0, b = 0.0;
            for (int t = 0; t < T; ++t) {
                a += dKp[(size_t)t * n + e];
                b += dVp[(size_t)t * n + e];
            }
            dK[off + e] = a;
            dV[off + e] = b;
        }
    }
    free(buf); free(dKp); free(dVp); free(jobs); free(tid);
    return 0;
}

/* ======================================================================== */
/* GEMM: C = A op(B), the second workload of the same tile pipeline          */
/*                                                                          */
/* The pages name GEMM as the workload the tile abstractions are built      */
/* around (10100.com/article/71410160, section on grid-level abstraction).  */
/* Definition, fp64 from the exact bf16 inputs, one plain dot product per   */
/* output element in k order:                                               */
/*   C[m,n] = sum_k A[m,k] * B'[k,n],  B' = B^T (B stored [N,K], b_kmajor)  */
/*                                     or B (B stored [K,N]).               */

typedef struct {
    const uint16_t *A, *B;
    int64_t M, N, K;
    int b_kmajor;
    const int64_t *rows; /* NULL: rows 0..M-1 */
    int64_t nrows;
    double *C;           /* nrows x N */
    int64_t next;
    pthread_mutex_t lock;
} gemm_job;

static void gemm_row(const gemm_job *job, int64_t m, double *c_row) {
    const int64_t N = job->N, K = job->K;
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = bf16_bits_to_double(job->A[m * K + k]);
            double b = job->b_kmajor ? bf16_bits_to_double(job->B[n * K + k])
                                     : bf16_bits_to_double(job->B[k * N + n]);
            acc += a * b;
        }
        c_row[n] = acc;
    }
}

static void *gemm_worker(void *arg) {
    gemm_job *job = (gemm_job *)arg;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t r = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->nrows) break;
        int64_t m = job->rows ? job->rows[r] : r;
        gemm_row(job, m, job->C + r * job->N);
    }
    return NULL;
}

/* Selected rows of C (rows == NULL: all M rows).  A: bf16 bits [M,K];
 * B: [N,K] if b_kmajor else [K,N].  C: double [nrows, N]. */
int tkor_gemm_rows(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K,
                   int b_kmajor, const int64_t *rows, int64_t nrows, double *C, int nthreads) {
    if (!A || !B || !C || M < 1 || N < 1 || K < 1 || nrows < 0) return -1;
    if (b_kmajor != 0 && b_kmajor != 1) return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    gemm_job job;
    job.A = A; job.B = B; job.M = M; job.N = N; job.K = K; job.b_kmajor = b_kmajor;
    job.rows = rows; job.nrows = nrows; job.C = C; job.next = 0;
    pthread_mutex_init(&job.lock, NULL);
    g_last_threads = 0;
    int T = resolve_threads(nthreads);
    if ((int64_t)T > nrows) T = (int)(nrows > 0 ? nrows : 1);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)T);
    int started = 0;
    for (int t = 1; tid && t < T; ++t) {
        if (pthread_create(&tid[started], NULL, gemm_worker, &job) != 0) break;
        ++started;
    }
    g_last_threads = started + 1;
    gemm_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    return 0;
}

int tkor_gemm(const uint16_t *A, const uint16_t *B, double *C, int64_t M, int64_t N, int64_t K,
              int b_kmajor, int nthreads) {
    return tkor_gemm_rows(A, B, M, N, K, b_kmajor, NULL, M, C, nthreads);
}

/* ======================================================================== */
/* Based linear attention (causal), the linear-attention variant the pages */
/* list ("Based Linear Attention", thebeat.tech "ThunderKittens 2.0", New    */
/* Kernels).  The pages name it without a formula; the reading taken is the */
/* Based feature map, the second-order Taylor expansion of exp, on query and */
/* key features of dimension Dqk:                                           */
/*   s_ij  = scale * <Q_i, K_j>                                             */
/*   w_ij  = 1 + s_ij + s_ij^2 / 2          (= phi(q_i) . phi(k_j))          */
/*   DEN_i = sum_{j <= i} w_ij                                              */
/*   O_i   = sum_{j <= i} w_ij V_j / DEN_i                                  */
/* written here in its plain quadratic form: one pass over the keys of each */
/* row, fp64 from the exact bf16 inputs.  w_ij >= 1/2, so DEN_i > 0.         */

typedef struct {
    const uint16_t *Q, *K, *V;
    int64_t N, Dqk, Dv;
    double scale;
    const int64_t *rows; /* NULL: rows 0..N-1 */
    int64_t nrows;
    double *O, *DEN;     /* nrows x Dv, nrows */
    int64_t next;
    pthread_mutex_t lock;
} based_job;

static void based_row(const based_job *job, int64_t i, double *o_row, double *den_out) {
    const int64_t Dqk = job->Dqk, Dv = job->Dv;
    double den = 0.0;
    for (int64_t d = 0; d < Dv; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < Dqk; ++d)
            dot += bf16_bits_to_double(job->Q[i * Dqk + d]) * bf16_bits_to_double(job->K[j * Dqk + d]);
        double s = job->scale * dot;
        double w = 1.0 + s + 0.5 * s * s;
        den += w;
        for (int64_t d = 0; d < Dv; ++d) o_row[d] += w * bf16_bits_to_double(job->V[j * Dv + d]);
    }
    for (int64_t d = 0; d < Dv; ++d) o_row[d] /= den;
    *den_out = den;
}

static void *based_worker(void *arg) {
    based_job *job = (based_job *)arg;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t r = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->nrows) break;
        int64_t i = job->rows ? job->rows[r] : r;
        based_row(job, i, job->O + r * job->Dv, job->DEN + r);
    }
    return NULL;
}

/* Selected rows of one head (rows == NULL: all N).  Q, K: bf16 bits [N,Dqk];
 * V: [N,Dv].  O: double [nrows,Dv]; DEN: double [nrows]. */
int tkor_based_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t N, int64_t Dqk,
                    int64_t Dv, double scale, const int64_t *rows, int64_t nrows, double *O, double *DEN,
                    int nthreads) {
    if (!Q || !K || !V || !O || !DEN || N < 1 || Dqk < 1 || Dv < 1 || nrows < 0) return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= N) return -1;
    based_job job;
    job.Q = Q; job.K = K; job.V = V; job.N = N; job.Dqk = Dqk; job.Dv = Dv; job.scale = scale;
    job.rows = rows; job.nrows = nrows; job.O = O; job.DEN = DEN; job.next = 0;
    pthread_mutex_init(&job.lock, NULL);
    g_last_threads = 0;
    int T = resolve_threads(nthreads);
    if ((int64_t)T > nrows) T = (int)(nrows > 0 ? nrows : 1);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)T);
    int started = 0;
    for (int t = 1; tid && t < T; ++t) {
        if (pthread_create(&tid[started], NULL, based_worker, &job) != 0) break;
        ++started;
    }
    g_last_threads = started + 1;
    based_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    return 0;
}

/* Whole problem: Q, K [B,H,N,Dqk]; V [B,H,N,Dv]; O [B,H,N,Dv]; DEN [B,H,N]. */
int tkor_based(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O, double *DEN, int64_t B,
               int64_t H, int64_t N, int64_t Dqk, int64_t Dv, double scale, int nthreads) {
    if (B < 1 || H < 1) return -1;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        if (tkor_based_rows(Q + (size_t)bh * N * Dqk, K + (size_t)bh * N * Dqk, V + (size_t)bh * N * Dv, N, Dqk,
                            Dv, scale, NULL, N, O + (size_t)bh * N * Dv, DEN + (size_t)bh * N, nthreads))
            return -1;
    }
    return 0;
}

/* ======================================================================== */
/* Hedgehog linear attention (causal), the other linear-attention variant   */
/* the pages list ("LoLCATS Hedgehog Linear Attention", thebeat.tech        */
/* "ThunderKittens 2.0", New Kernels), named without a formula.  Reading:   */
/* the Hedgehog feature map, a softmax over a learned projection and over   */
/* its negation, on queries and keys of dimension d with f features each:   */
/*   phi_q(x) = [softmax(x Wq), softmax(-x Wq)],  phi_k likewise with Wk    */
/*   w_ij  = phi_q(q_i) . phi_k(k_j)                      (> 0)             */
/*   DEN_i = sum_{j <= i} w_ij,   O_i = sum_{j <= i} w_ij V_j / DEN_i       */
/* in its plain quadratic form, fp64 from the exact bf16 inputs; every      */
/* softmax is taken with its maximum subtracted.                             */

static void hedgehog_phi(const uint16_t *x, const uint16_t *W, int64_t d, int64_t f, double *phi) {
    /* z = x W (f values), then the two softmaxes */
    double zmax = -INFINITY, zmin = INFINITY;
    for (int64_t c = 0; c < f; ++c) {
        double z = 0.0;
        for (int64_t a = 0; a < d; ++a) z += bf16_bits_to_double(x[a]) * bf16_bits_to_double(W[a * f + c]);
        phi[c] = z;
        if (z > zmax) zmax = z;
        if (z < zmin) zmin = z;
    }
    double sp = 0.0, sn = 0.0;
    for (int64_t c = 0; c < f; ++c) {
        double z = phi[c];
        phi[c] = exp(z - zmax);
        phi[f + c] = exp(zmin - z);
        sp += phi[c];
        sn += phi[f + c];
    }
    for (int64_t c = 0; c < f; ++c) {
        phi[c] /= sp;
        phi[f + c] /= sn;
    }
}

/* One head, selected rows (rows == NULL: all).  Q, K: bf16 bits [N,d];
 * Wq, Wk: [d,f]; V: [N,Dv].  O: double [nrows,Dv]; DEN: double [nrows]. */
int tkor_hedgehog_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *Wq,
                       const uint16_t *Wk, int64_t N, int64_t d, int64_t f, int64_t Dv, const int64_t *rows,
                       int64_t nrows, double *O, double *DEN) {
    if (!Q || !K || !V || !Wq || !Wk || !O || !DEN || N < 1 || d < 1 || f < 1 || Dv < 1 || nrows < 0) return -1;
    int64_t maxrow = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= N) return -1;
        if (i > maxrow) maxrow = i;
    }
    double *phik = (double *)malloc(sizeof(double) * (size_t)(maxrow + 1) * (size_t)(2 * f));
    double *phiq = (double *)malloc(sizeof(double) * (size_t)(2 * f));
    if (!phik || !phiq) {
        free(phik); free(phiq);
        return -1;
    }
    for (int64_t j = 0; j <= maxrow && nrows > 0; ++j) hedgehog_phi(K + j * d, Wk, d, f, phik + j * 2 * f);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        hedgehog_phi(Q + i * d, Wq, d, f, phiq);
        double den = 0.0;
        double *o = O + r * Dv;
        for (int64_t e = 0; e < Dv; ++e) o[e] = 0.0;
        for (int64_t j = 0; j <= i; ++j) {
            double w = 0.0;
            for (int64_t c = 0; c < 2 * f; ++c) w += phiq[c] * phik[j * 2 * f + c];
            den += w;
            for (int64_t e = 0; e < Dv; ++e) o[e] += w * bf16_bits_to_double(V[j * Dv + e]);
        }
        for (int64_t e = 0; e < Dv; ++e) o[e] /= den;
        DEN[r] = den;
    }
    free(phik); free(phiq);
    g_last_threads = 1;
    return 0;
}
