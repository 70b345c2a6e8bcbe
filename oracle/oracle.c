/*
 * CPU ORACLE for exact tiled attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  The product path (the CUDA library) never calls it and
 * shares no code, header, table or helper with it.
 *
 * Everything here is plain fp64 C with naive loops, written from the
 * definitions on the four source pages:
 *
 *   [FA2]  "解析 FlashAttention（4）：FlashAttention-v2"  (FA-v2 analysis page)
 *   [FA1]  "深入理解 FlashAttention：分块、算子融合与重计算的艺术" (FA-1 note)
 *   [WIKI] "分块 Attention：重建概率，累计梯度" (attention-kernels wiki page)
 *   [CH18] "第18章 FlashAttention" (book chapter 18)
 *
 * Conventions (all tensors contiguous row-major):
 *   q, k, v, o, dout, dq, dk, dv : [B, H, N, d]   (double)
 *   lse                          : [B, H, N]      (double, natural log)
 *   kv_lens                      : [B] int or NULL (NULL = every key valid)
 *   key j is visible to query i  iff  j < kv_len(b)  and  (!causal or j <= i)
 *     and, for the sliding window (wl, wr) of flash_attn_func's window_size
 *     ([CH18] §18.7.1; -1 = no bound on that side),
 *     (wl < 0 or j >= i - wl)  and  (wr < 0 or j <= i + wr)
 *     -- causal mask M_ij = -inf for j > i ([CH18] §18.2.2 eq. for M_ij);
 *        padding mask removes columns ([CH18] §18.2.2 Table 18-3).
 *     and, for a block-sparse mask ([CH18] §18.8.1: per query block the list
 *     of key blocks to compute; here a dense 0/1 matrix bm [nqb][nkb] of
 *     bs x bs blocks), bm[i / bs][j / bs] != 0.
 *   Entry points without "_win" / "_mask" have no window (wl = wr = -1) and
 *   no block mask.
 *   S = scale * Q K^T ([CH18] §18.2.2; [WIKI] §04 "S = QK^T/sqrt(d)").
 *   A row with no visible key has O = 0, LSE = -inf and zero gradients
 *   ([WIKI] §04, the explicit fully-masked-row convention).
 *
 * Parity status of each entry point is listed in the header of
 * oracle/__init__.py; every function here is pinned by tests/test_oracle_*.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_OK 0
#define OR_ERR 1

/* Which keys a query sees: key-padding length, causal flag, window edges,
 * optional block mask (bm NULL = none). */
typedef struct {
    int kv_len, causal, wl, wr;
    const unsigned char* bm;
    int bs, nkb;
} mask_t;

static int visible(int i, int j, const mask_t* m) {
    if (j >= m->kv_len) return 0;
    if (m->causal && j > i) return 0;
    if (m->wl >= 0 && j < i - m->wl) return 0;
    if (m->wr >= 0 && j > i + m->wr) return 0;
    if (m->bm && !m->bm[(size_t)(i / m->bs) * m->nkb + j / m->bs]) return 0;
    return 1;
}

static mask_t make_mask(int kv_len, int causal, int wl, int wr, const unsigned char* bm, int bs, int nkb) {
    mask_t m = {kv_len, causal, wl, wr, bm, bs, nkb};
    return m;
}

static int kvlen_of(const int* kv_lens, int b, int N) {
    if (!kv_lens) return N;
    int L = kv_lens[b];
    if (L < 0) L = 0;
    if (L > N) L = N;
    return L;
}

/* ------------------------------------------------------------------------ */
/* tiny thread pool: run fn(arg, item) for item in [0, n_items)             */
/* ------------------------------------------------------------------------ */
typedef void (*item_fn)(void* arg, long item);
typedef struct {
    item_fn fn;
    void* arg;
    long n_items;
    long next;
    pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* p) {
    pool_t* pl = (pool_t*)p;
    for (;;) {
        pthread_mutex_lock(&pl->mu);
        long it = pl->next++;
        pthread_mutex_unlock(&pl->mu);
        if (it >= pl->n_items) break;
        pl->fn(pl->arg, it);
    }
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_items(item_fn fn, void* arg, long n_items, int nthreads) {
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
    pool_t pl;
    pl.fn = fn;
    pl.arg = arg;
    pl.n_items = n_items;
    pl.next = 0;
    pthread_mutex_init(&pl.mu, NULL);
    if (nthreads <= 1) {
        pool_worker(&pl);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, pool_worker, &pl);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
        free(th);
    }
    pthread_mutex_destroy(&pl.mu);
}

/* ======================================================================== */
/* 1. Naive materialised attention, one (b,h) head at a time                */
/*    [CH18] §18.1.1 / §18.2.4 standard attention; [FA1] §1.1;              */
/*    safe softmax (subtract the row max) [FA1] §3.2.                       */
/* ======================================================================== */

/* Build S (N x N, -inf where masked) and P (N x N) for one head; write O and
 * LSE.  Returns nothing; S and P are caller scratch. */
static void naive_head_forward(const double* q, const double* k, const double* v,
                               double* o, double* lse, double* S, double* P,
                               int N, int d, double scale, const mask_t* mk) {
    for (int i = 0; i < N; ++i) {
        for (int j = 0; j < N; ++j) {
            double s = -INFINITY;
            if (visible(i, j, mk)) {
                double acc = 0.0;
                for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
                s = scale * acc;
            }
            S[(size_t)i * N + j] = s;
        }
    }
    for (int i = 0; i < N; ++i) {
        const double* Si = S + (size_t)i * N;
        double* Pi = P + (size_t)i * N;
        /* safe softmax: max, then sum of exp(s - max), then normalise */
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j)
            if (Si[j] > mx) mx = Si[j];
        if (mx == -INFINITY) { /* fully masked row */
            for (int j = 0; j < N; ++j) Pi[j] = 0.0;
            lse[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < N; ++j) sum += (Si[j] == -INFINITY) ? 0.0 : exp(Si[j] - mx);
        double L = mx + log(sum);
        lse[i] = L;
        for (int j = 0; j < N; ++j) Pi[j] = (Si[j] == -INFINITY) ? 0.0 : exp(Si[j] - L);
    }
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < d; ++t) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += P[(size_t)i * N + j] * v[(size_t)j * d + t];
            o[(size_t)i * d + t] = acc;
        }
}

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv, *Dout;
    int B, H, N, d;
    mask_t mk; /* kv_len filled per batch item */
    double scale;
    const int* kv_lens;
} naive_args;

static mask_t mask_of(const naive_args* a, int b) {
    mask_t m = a->mk;
    m.kv_len = kvlen_of(a->kv_lens, b, a->N);
    return m;
}

static void naive_fwd_item(void* a_, long bh) {
    naive_args* a = (naive_args*)a_;
    size_t N = (size_t)a->N, d = (size_t)a->d;
    size_t off = (size_t)bh * N * d;
    int b = (int)(bh / a->H);
    double* S = (double*)malloc(sizeof(double) * N * N);
    double* P = (double*)malloc(sizeof(double) * N * N);
    const mask_t mk = mask_of(a, b);
    naive_head_forward(a->q + off, a->k + off, a->v + off, a->o + off, a->lse + (size_t)bh * N, S, P,
                       a->N, a->d, a->scale, &mk);
    free(S);
    free(P);
}

/* Forward: O = softmax(scale Q K^T + M) V and LSE, materialising S and P.
 * bm: optional block mask [ceil(N/bs)][nkb], nkb = ceil(N/bs). */
int oracle_fwd_mask(const double* q, const double* k, const double* v, double* o, double* lse,
                    int B, int H, int N, int d, double scale, int causal, int wl, int wr,
                    const unsigned char* bm, int bs, const int* kv_lens, int nthreads) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || (bm && bs <= 0)) return OR_ERR;
    naive_args a = {q, k, v, NULL, o, lse, NULL, NULL, NULL, NULL, B, H, N, d,
                    make_mask(N, causal, wl, wr, bm, bs, bm ? (N + bs - 1) / bs : 0), scale, kv_lens};
    run_items(naive_fwd_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
               int B, int H, int N, int d, double scale, int causal, const int* kv_lens,
               int nthreads) {
    return oracle_fwd_mask(q, k, v, o, lse, B, H, N, d, scale, causal, -1, -1, NULL, 0, kv_lens, nthreads);
}

/* Backward of L = sum(O * dO) for one head, by the definitions of
 * [FA2] §5.1 (softmax Jacobian: dS = P (dP - D), D_i = sum_j P_ij dP_ij) and
 * [WIKI] §04 (dQ += dS K / sqrt(d), dK += dS^T Q / sqrt(d), dV += P^T G).
 * D is computed from its definition sum_j P_ij dP_ij, NOT from the dO.O
 * identity, so that identity stays a test. */
static void naive_bwd_item(void* a_, long bh) {
    naive_args* a = (naive_args*)a_;
    int N = a->N, d = a->d;
    size_t off = (size_t)bh * N * d;
    int b = (int)(bh / a->H);
    const double *q = a->q + off, *k = a->k + off, *v = a->v + off, *dO = a->dout + off;
    double *o = a->o + off, *dq = a->dq + off, *dk = a->dk + off, *dv = a->dv + off;
    double* lse = a->lse + (size_t)bh * N;
    double* S = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* P = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* dP = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* D = (double*)malloc(sizeof(double) * (size_t)N);
    const mask_t mk = mask_of(a, b);
    naive_head_forward(q, k, v, o, lse, S, P, N, d, a->scale, &mk);
    /* dP = dO V^T */
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int t = 0; t < d; ++t) acc += dO[(size_t)i * d + t] * v[(size_t)j * d + t];
            dP[(size_t)i * N + j] = acc;
        }
    /* D_i = sum_j P_ij dP_ij (definition) */
    for (int i = 0; i < N; ++i) {
        double acc = 0.0;
        for (int j = 0; j < N; ++j) acc += P[(size_t)i * N + j] * dP[(size_t)i * N + j];
        D[i] = acc;
    }
    if (a->Dout) memcpy(a->Dout + (size_t)bh * N, D, sizeof(double) * (size_t)N);
    /* dS = P (dP - D), stored in S */
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j)
            S[(size_t)i * N + j] = P[(size_t)i * N + j] * (dP[(size_t)i * N + j] - D[i]);
    /* dQ = scale dS K */
    for (int i = 0; i < N; ++i)
        for (int t = 0; t < d; ++t) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += S[(size_t)i * N + j] * k[(size_t)j * d + t];
            dq[(size_t)i * d + t] = a->scale * acc;
        }
    /* dK = scale dS^T Q ; dV = P^T dO */
    for (int j = 0; j < N; ++j)
        for (int t = 0; t < d; ++t) {
            double acck = 0.0, accv = 0.0;
            for (int i = 0; i < N; ++i) {
                acck += S[(size_t)i * N + j] * q[(size_t)i * d + t];
                accv += P[(size_t)i * N + j] * dO[(size_t)i * d + t];
            }
            dk[(size_t)j * d + t] = a->scale * acck;
            dv[(size_t)j * d + t] = accv;
        }
    free(S);
    free(P);
    free(dP);
    free(D);
}

/* Backward (also returns the forward O, LSE and, if D_out != NULL, D). */
int oracle_bwd_mask(const double* q, const double* k, const double* v, const double* dout,
                    double* o, double* lse, double* dq, double* dk, double* dv, double* D_out,
                    int B, int H, int N, int d, double scale, int causal, int wl, int wr,
                    const unsigned char* bm, int bs, const int* kv_lens, int nthreads) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || (bm && bs <= 0)) return OR_ERR;
    naive_args a = {q, k, v, dout, o, lse, dq, dk, dv, D_out, B, H, N, d,
                    make_mask(N, causal, wl, wr, bm, bs, bm ? (N + bs - 1) / bs : 0), scale, kv_lens};
    run_items(naive_bwd_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               double* o, double* lse, double* dq, double* dk, double* dv, double* D_out,
               int B, int H, int N, int d, double scale, int causal, const int* kv_lens,
               int nthreads) {
    return oracle_bwd_mask(q, k, v, dout, o, lse, dq, dk, dv, D_out, B, H, N, d, scale, causal, -1, -1, NULL, 0,
                           kv_lens, nthreads);
}

/* ======================================================================== */
/* 1b. Rectangular attention (N_q query rows, N_k keys): decoding against a  */
/*     key/value cache and cross-attention ([CH18] §18.8.2: the query of a   */
/*     decode step is [b, n_q, d] with n_q << n_kv; §18.7.1 varlen API with  */
/*     separate query and key lengths).  With the causal mask the queries    */
/*     are the last N_q positions of the N_k-long sequence: query i sees key */
/*     j iff j <= i + (N_k - N_q); key padding as above.                     */
/* ======================================================================== */

static void rect_head_forward(const double* q, const double* k, const double* v, double* o, double* lse,
                              double* s, int Nq, int Nk, int d, double scale, int causal, int kv_len) {
    const int off = Nk - Nq;
    for (int i = 0; i < Nq; ++i) {
        double mx = -INFINITY;
        for (int j = 0; j < Nk; ++j) {
            s[j] = -INFINITY;
            if (j < kv_len && (!causal || j <= i + off)) {
                double acc = 0.0;
                for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
                s[j] = scale * acc;
                if (s[j] > mx) mx = s[j];
            }
        }
        double* orow = o + (size_t)i * d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (mx == -INFINITY) { /* no visible key */
            lse[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < Nk; ++j) sum += (s[j] == -INFINITY) ? 0.0 : exp(s[j] - mx);
        const double L = mx + log(sum);
        lse[i] = L;
        for (int j = 0; j < Nk; ++j) {
            if (s[j] == -INFINITY) continue;
            const double pj = exp(s[j] - L);
            for (int t = 0; t < d; ++t) orow[t] += pj * v[(size_t)j * d + t];
        }
    }
}

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int H, Nq, Nk, d, causal;
    double scale;
    const int* kv_lens;
} rect_args;

static void rect_item(void* a_, long bh) {
    rect_args* a = (rect_args*)a_;
    const int b = (int)(bh / a->H);
    double* s = (double*)malloc(sizeof(double) * (size_t)a->Nk);
    rect_head_forward(a->q + (size_t)bh * a->Nq * a->d, a->k + (size_t)bh * a->Nk * a->d,
                      a->v + (size_t)bh * a->Nk * a->d, a->o + (size_t)bh * a->Nq * a->d,
                      a->lse + (size_t)bh * a->Nq, s, a->Nq, a->Nk, a->d, a->scale, a->causal,
                      kvlen_of(a->kv_lens, b, a->Nk));
    free(s);
}

/* Forward of rectangular attention: q [B,H,Nq,d], k, v [B,H,Nk,d] -> o
 * [B,H,Nq,d], lse [B,H,Nq]; kv_lens [B] or NULL (clamped to [0, Nk]). */
int oracle_fwd_rect(const double* q, const double* k, const double* v, double* o, double* lse, int B, int H,
                    int Nq, int Nk, int d, double scale, int causal, const int* kv_lens, int nthreads) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return OR_ERR;
    rect_args a = {q, k, v, o, lse, H, Nq, Nk, d, causal, scale, kv_lens};
    run_items(rect_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

/* Backward of rectangular attention for one head, by the same definitions as
 * naive_bwd_item: P materialised (Nq x Nk), dP = dO V^T, D_i = sum_j P_ij
 * dP_ij, dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO. */
static void rect_head_backward(const double* q, const double* k, const double* v, const double* dO,
                               double* dq, double* dk, double* dv, int Nq, int Nk, int d, double scale,
                               int causal, int kv_len) {
    const int off = Nk - Nq;
    double* P = (double*)malloc(sizeof(double) * (size_t)Nq * Nk);
    double* dS = (double*)malloc(sizeof(double) * (size_t)Nq * Nk);
    for (int i = 0; i < Nq; ++i) {
        double* Pi = P + (size_t)i * Nk;
        double mx = -INFINITY;
        for (int j = 0; j < Nk; ++j) {
            Pi[j] = -INFINITY;
            if (j < kv_len && (!causal || j <= i + off)) {
                double acc = 0.0;
                for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
                Pi[j] = scale * acc;
                if (Pi[j] > mx) mx = Pi[j];
            }
        }
        if (mx == -INFINITY) {
            for (int j = 0; j < Nk; ++j) Pi[j] = 0.0;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < Nk; ++j) sum += (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - mx);
        const double L = mx + log(sum);
        for (int j = 0; j < Nk; ++j) Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - L);
    }
    for (int i = 0; i < Nq; ++i) {
        double Di = 0.0;
        for (int j = 0; j < Nk; ++j) {
            double dp = 0.0;
            for (int t = 0; t < d; ++t) dp += dO[(size_t)i * d + t] * v[(size_t)j * d + t];
            dS[(size_t)i * Nk + j] = dp;
            Di += P[(size_t)i * Nk + j] * dp;
        }
        for (int j = 0; j < Nk; ++j) dS[(size_t)i * Nk + j] = P[(size_t)i * Nk + j] * (dS[(size_t)i * Nk + j] - Di);
    }
    for (int i = 0; i < Nq; ++i)
        for (int t = 0; t < d; ++t) {
            double acc = 0.0;
            for (int j = 0; j < Nk; ++j) acc += dS[(size_t)i * Nk + j] * k[(size_t)j * d + t];
            dq[(size_t)i * d + t] = scale * acc;
        }
    for (int j = 0; j < Nk; ++j)
        for (int t = 0; t < d; ++t) {
            double acck = 0.0, accv = 0.0;
            for (int i = 0; i < Nq; ++i) {
                acck += dS[(size_t)i * Nk + j] * q[(size_t)i * d + t];
                accv += P[(size_t)i * Nk + j] * dO[(size_t)i * d + t];
            }
            dk[(size_t)j * d + t] = scale * acck;
            dv[(size_t)j * d + t] = accv;
        }
    free(P);
    free(dS);
}

typedef struct {
    const double *q, *k, *v, *dO;
    double *dq, *dk, *dv;
    int H, Nq, Nk, d, causal;
    double scale;
    const int* kv_lens;
} rect_bwd_args;

static void rect_bwd_item(void* a_, long bh) {
    rect_bwd_args* a = (rect_bwd_args*)a_;
    const int b = (int)(bh / a->H);
    const size_t oq = (size_t)bh * a->Nq * a->d, ok = (size_t)bh * a->Nk * a->d;
    rect_head_backward(a->q + oq, a->k + ok, a->v + ok, a->dO + oq, a->dq + oq, a->dk + ok, a->dv + ok, a->Nq,
                       a->Nk, a->d, a->scale, a->causal, kvlen_of(a->kv_lens, b, a->Nk));
}

/* Backward of oracle_fwd_rect: dq [B,H,Nq,d], dk, dv [B,H,Nk,d]. */
int oracle_bwd_rect(const double* q, const double* k, const double* v, const double* dout, double* dq,
                    double* dk, double* dv, int B, int H, int Nq, int Nk, int d, double scale, int causal,
                    const int* kv_lens, int nthreads) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return OR_ERR;
    rect_bwd_args a = {q, k, v, dout, dq, dk, dv, H, Nq, Nk, d, causal, scale, kv_lens};
    run_items(rect_bwd_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

/* ======================================================================== */
/* 2. Row-sampled forms of the same definitions, for shapes whose N x N      */
/*    matrices are too large to materialise.  One head per call.            */
/* ======================================================================== */

/* O and LSE of selected query rows of one head (definition applied row by
 * row: the row's scores, its safe-softmax LSE, then P V). */
int oracle_fwd_rows_mask(const double* q, const double* k, const double* v, int N, int d, double scale,
                         int causal, int kv_len, int wl, int wr, const unsigned char* bm, int bs,
                         const int* rows, int nrows, double* o_rows, double* lse_rows) {
    if (N <= 0 || d <= 0 || (bm && bs <= 0)) return OR_ERR;
    if (kv_len < 0) kv_len = 0;
    if (kv_len > N) kv_len = N;
    const mask_t mk = make_mask(kv_len, causal, wl, wr, bm, bs, bm ? (N + bs - 1) / bs : 0);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    for (int r = 0; r < nrows; ++r) {
        int i = rows[r];
        if (i < 0 || i >= N) { free(s); return OR_ERR; }
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) {
            s[j] = -INFINITY;
            if (visible(i, j, &mk)) {
                double acc = 0.0;
                for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
                s[j] = scale * acc;
                if (s[j] > mx) mx = s[j];
            }
        }
        double* orow = o_rows + (size_t)r * d;
        if (mx == -INFINITY) {
            for (int t = 0; t < d; ++t) orow[t] = 0.0;
            lse_rows[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < N; ++j) sum += (s[j] == -INFINITY) ? 0.0 : exp(s[j] - mx);
        double L = mx + log(sum);
        lse_rows[r] = L;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        for (int j = 0; j < N; ++j) {
            if (s[j] == -INFINITY) continue;
            double p = exp(s[j] - L);
            for (int t = 0; t < d; ++t) orow[t] += p * v[(size_t)j * d + t];
        }
    }
    free(s);
    return OR_OK;
}

int oracle_fwd_rows(const double* q, const double* k, const double* v, int N, int d, double scale,
                    int causal, int kv_len, const int* rows, int nrows, double* o_rows,
                    double* lse_rows) {
    return oracle_fwd_rows_mask(q, k, v, N, d, scale, causal, kv_len, -1, -1, NULL, 0, rows, nrows, o_rows,
                                lse_rows);
}

typedef struct {
    const double *q, *k, *v, *dout;
    int N, d;
    mask_t mk;
    double scale;
    double *lse, *D; /* [N] each, filled per row */
} rowstat_args;

/* per query row i: LSE_i and D_i = sum_j P_ij dP_ij (definitions) */
static void rowstat_item(void* a_, long i_) {
    rowstat_args* a = (rowstat_args*)a_;
    int i = (int)i_, N = a->N, d = a->d;
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
        s[j] = -INFINITY;
        if (visible(i, j, &a->mk)) {
            double acc = 0.0;
            for (int t = 0; t < d; ++t) acc += a->q[(size_t)i * d + t] * a->k[(size_t)j * d + t];
            s[j] = a->scale * acc;
            if (s[j] > mx) mx = s[j];
        }
    }
    if (mx == -INFINITY) {
        a->lse[i] = -INFINITY;
        a->D[i] = 0.0;
        free(s);
        return;
    }
    double sum = 0.0;
    for (int j = 0; j < N; ++j) sum += (s[j] == -INFINITY) ? 0.0 : exp(s[j] - mx);
    double L = mx + log(sum);
    double Dacc = 0.0;
    for (int j = 0; j < N; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - L);
        double dp = 0.0;
        for (int t = 0; t < d; ++t) dp += a->dout[(size_t)i * d + t] * a->v[(size_t)j * d + t];
        Dacc += p * dp;
    }
    a->lse[i] = L;
    a->D[i] = Dacc;
    free(s);
}

typedef struct {
    rowstat_args* rs;
    const int* keys;
    int nkeys;
    double *dk_part, *dv_part; /* [N_chunks][nkeys][d] partial sums */
    int chunk;
} keygrad_args;

/* partial dK/dV of the selected keys over one chunk of query rows */
static void keygrad_item(void* a_, long c) {
    keygrad_args* ka = (keygrad_args*)a_;
    rowstat_args* a = ka->rs;
    int N = a->N, d = a->d;
    int i0 = (int)c * ka->chunk, i1 = i0 + ka->chunk;
    if (i1 > N) i1 = N;
    double* dkp = ka->dk_part + (size_t)c * ka->nkeys * d;
    double* dvp = ka->dv_part + (size_t)c * ka->nkeys * d;
    for (int r = 0; r < ka->nkeys; ++r) {
        int j = ka->keys[r];
        for (int i = i0; i < i1; ++i) {
            if (!visible(i, j, &a->mk) || a->lse[i] == -INFINITY) continue;
            double acc = 0.0;
            for (int t = 0; t < d; ++t) acc += a->q[(size_t)i * d + t] * a->k[(size_t)j * d + t];
            double p = exp(a->scale * acc - a->lse[i]);
            double dp = 0.0;
            for (int t = 0; t < d; ++t) dp += a->dout[(size_t)i * d + t] * a->v[(size_t)j * d + t];
            double ds = p * (dp - a->D[i]);
            for (int t = 0; t < d; ++t) {
                dkp[(size_t)r * d + t] += a->scale * ds * a->q[(size_t)i * d + t];
                dvp[(size_t)r * d + t] += p * a->dout[(size_t)i * d + t];
            }
        }
    }
}

/* Gradients of selected rows of one head: dQ of rows[], dK and dV of keys[].
 * LSE and D of every query row come from their definitions (rowstat_item),
 * then dQ_i = scale sum_j dS_ij k_j and dK_j = scale sum_i dS_ij q_i,
 * dV_j = sum_i P_ij dO_i.  Optionally returns the full-head LSE and D. */
int oracle_bwd_rows_mask(const double* q, const double* k, const double* v, const double* dout, int N,
                         int d, double scale, int causal, int kv_len, int wl, int wr,
                         const unsigned char* bm, int bs, const int* rows, int nrows, double* dq_rows,
                         const int* keys, int nkeys, double* dk_rows, double* dv_rows, double* lse_all,
                         double* D_all, int nthreads) {
    if (N <= 0 || d <= 0 || (bm && bs <= 0)) return OR_ERR;
    if (kv_len < 0) kv_len = 0;
    if (kv_len > N) kv_len = N;
    double* lse = lse_all ? lse_all : (double*)malloc(sizeof(double) * (size_t)N);
    double* D = D_all ? D_all : (double*)malloc(sizeof(double) * (size_t)N);
    rowstat_args rs = {q, k, v, dout, N, d, make_mask(kv_len, causal, wl, wr, bm, bs, bm ? (N + bs - 1) / bs : 0),
                       scale, lse, D};
    run_items(rowstat_item, &rs, N, nthreads);
    for (int r = 0; r < nrows; ++r) {
        int i = rows[r];
        double* g = dq_rows + (size_t)r * d;
        for (int t = 0; t < d; ++t) g[t] = 0.0;
        if (lse[i] == -INFINITY) continue;
        for (int j = 0; j < N; ++j) {
            if (!visible(i, j, &rs.mk)) continue;
            double acc = 0.0;
            for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
            double p = exp(scale * acc - lse[i]);
            double dp = 0.0;
            for (int t = 0; t < d; ++t) dp += dout[(size_t)i * d + t] * v[(size_t)j * d + t];
            double ds = p * (dp - D[i]);
            for (int t = 0; t < d; ++t) g[t] += scale * ds * k[(size_t)j * d + t];
        }
    }
    if (nkeys > 0) {
        int chunk = 64;
        int nch = (N + chunk - 1) / chunk;
        keygrad_args ka;
        ka.rs = &rs;
        ka.keys = keys;
        ka.nkeys = nkeys;
        ka.chunk = chunk;
        ka.dk_part = (double*)calloc((size_t)nch * nkeys * d, sizeof(double));
        ka.dv_part = (double*)calloc((size_t)nch * nkeys * d, sizeof(double));
        run_items(keygrad_item, &ka, nch, nthreads);
        for (size_t e = 0; e < (size_t)nkeys * d; ++e) {
            double sk = 0.0, sv = 0.0;
            for (int c = 0; c < nch; ++c) {
                sk += ka.dk_part[(size_t)c * nkeys * d + e];
                sv += ka.dv_part[(size_t)c * nkeys * d + e];
            }
            dk_rows[e] = sk;
            dv_rows[e] = sv;
        }
        free(ka.dk_part);
        free(ka.dv_part);
    }
    if (!lse_all) free(lse);
    if (!D_all) free(D);
    return OR_OK;
}

int oracle_bwd_rows(const double* q, const double* k, const double* v, const double* dout, int N,
                    int d, double scale, int causal, int kv_len, const int* rows, int nrows,
                    double* dq_rows, const int* keys, int nkeys, double* dk_rows, double* dv_rows,
                    double* lse_all, double* D_all, int nthreads) {
    return oracle_bwd_rows_mask(q, k, v, dout, N, d, scale, causal, kv_len, -1, -1, NULL, 0, rows, nrows, dq_rows,
                                keys, nkeys, dk_rows, dv_rows, lse_all, D_all, nthreads);
}

/* ======================================================================== */
/* 3. Tiled fp64 reference: Algorithm 1 (forward) and Algorithm 2            */
/*    (backward) of [FA2] §4 and §5.4, with arbitrary Br/Bc and a ragged     */
/*    last block.  Exists to pin the blocking claims (tiled == unblocked).   */
/*    Shares no code with section 1.                                         */
/* ======================================================================== */

static double mask_score(double raw, int gi, int gj, int kv_len, int causal, double scale) {
    if (gj >= kv_len) return -INFINITY;
    if (causal && gj > gi) return -INFINITY;
    return scale * raw;
}

/* exp(a - b) where b may be -inf (then the block so far has no visible key
 * and the term is 0); never evaluates -inf - (-inf) ([WIKI] §04). */
static double exp_diff(double a, double b) {
    if (a == -INFINITY) return 0.0;
    return exp(a - b);
}

typedef struct {
    const double *q, *k, *v, *o_in, *lse_in, *dout;
    double *o, *lse, *dq, *dk, *dv;
    int B, H, N, d, causal, Br, Bc;
    double scale;
    const int* kv_lens;
} tiled_args;

/* Algorithm 1 for one head. For query block i: m = -inf, l = 0, O = 0; for
 * each key block j: S = scale Q_i K_j^T (+mask), m_new = max(m, rowmax S),
 * P~ = exp(S - m_new), l = exp(m - m_new) l + rowsum P~,
 * O = diag(exp(m - m_new)) O + P~ V_j (the rescale MULTIPLIES by
 * exp(m_old - m_new): [FA2] §2.3-2.4 scalar derivation, [FA1] §4.2,
 * [WIKI] §01); finally O = O / l and L = m + log l ([FA2] §4 steps 6-7). */
static void tiled_fwd_item(void* a_, long bh) {
    tiled_args* a = (tiled_args*)a_;
    int N = a->N, d = a->d, Br = a->Br, Bc = a->Bc;
    size_t off = (size_t)bh * N * d;
    int b = (int)(bh / a->H);
    int kv_len = kvlen_of(a->kv_lens, b, N);
    const double *q = a->q + off, *k = a->k + off, *v = a->v + off;
    double *o = a->o + off, *lse = a->lse + (size_t)bh * N;
    int Tr = (N + Br - 1) / Br, Tc = (N + Bc - 1) / Bc;
    double* m = (double*)malloc(sizeof(double) * Br);
    double* l = (double*)malloc(sizeof(double) * Br);
    double* O = (double*)malloc(sizeof(double) * (size_t)Br * d);
    double* S = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
    for (int bi = 0; bi < Tr; ++bi) {
        int r0 = bi * Br, nr = (r0 + Br <= N) ? Br : N - r0;
        for (int r = 0; r < nr; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.0;
            for (int t = 0; t < d; ++t) O[(size_t)r * d + t] = 0.0;
        }
        for (int bj = 0; bj < Tc; ++bj) {
            int c0 = bj * Bc, nc = (c0 + Bc <= N) ? Bc : N - c0;
            for (int r = 0; r < nr; ++r) {
                /* step 1: S = Q_i K_j^T (scaled, masked) */
                double rowmax = -INFINITY;
                for (int c = 0; c < nc; ++c) {
                    double acc = 0.0;
                    for (int t = 0; t < d; ++t) acc += q[(size_t)(r0 + r) * d + t] * k[(size_t)(c0 + c) * d + t];
                    double s = mask_score(acc, r0 + r, c0 + c, kv_len, a->causal, a->scale);
                    S[(size_t)r * Bc + c] = s;
                    if (s > rowmax) rowmax = s;
                }
                /* step 2: m_new */
                double m_new = m[r] > rowmax ? m[r] : rowmax;
                /* step 4 factor exp(m_old - m_new) (0 when m_old = -inf) */
                double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                /* step 3: P~ = exp(S - m_new); step 4: l; step 5: O */
                double rowsum = 0.0;
                for (int t = 0; t < d; ++t) O[(size_t)r * d + t] *= alpha;
                for (int c = 0; c < nc; ++c) {
                    double p = (m_new == -INFINITY) ? 0.0 : exp_diff(S[(size_t)r * Bc + c], m_new);
                    rowsum += p;
                    for (int t = 0; t < d; ++t) O[(size_t)r * d + t] += p * v[(size_t)(c0 + c) * d + t];
                }
                l[r] = alpha * l[r] + rowsum;
                m[r] = m_new;
            }
        }
        /* steps 6-7 */
        for (int r = 0; r < nr; ++r) {
            if (l[r] == 0.0) {
                for (int t = 0; t < d; ++t) o[(size_t)(r0 + r) * d + t] = 0.0;
                lse[r0 + r] = -INFINITY;
            } else {
                for (int t = 0; t < d; ++t) o[(size_t)(r0 + r) * d + t] = O[(size_t)r * d + t] / l[r];
                lse[r0 + r] = m[r] + log(l[r]);
            }
        }
    }
    free(m);
    free(l);
    free(O);
    free(S);
}

int oracle_tiled_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                     int B, int H, int N, int d, double scale, int causal, const int* kv_lens,
                     int Br, int Bc, int nthreads) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || Br <= 0 || Bc <= 0) return OR_ERR;
    tiled_args a;
    memset(&a, 0, sizeof(a));
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.B = B; a.H = H; a.N = N; a.d = d; a.causal = causal; a.Br = Br; a.Bc = Bc;
    a.scale = scale; a.kv_lens = kv_lens;
    run_items(tiled_fwd_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

/* Algorithm 2 for one head ([FA2] §5.4, loop order: outer over key blocks j,
 * inner over query blocks i).  D_i = rowsum(dO_i * O_i) ([FA2] §5.2),
 * P = exp(S - L_i) (0 where masked or L_i = -inf), dV_j += P^T dO_i,
 * dP = dO_i V_j^T, dS = P (dP - D_i), dQ_i += scale dS K_j,
 * dK_j += scale dS^T Q_i ([WIKI] §04 puts 1/sqrt(d) on dQ and dK). */
static void tiled_bwd_item(void* a_, long bh) {
    tiled_args* a = (tiled_args*)a_;
    int N = a->N, d = a->d, Br = a->Br, Bc = a->Bc;
    size_t off = (size_t)bh * N * d;
    int b = (int)(bh / a->H);
    int kv_len = kvlen_of(a->kv_lens, b, N);
    const double *q = a->q + off, *k = a->k + off, *v = a->v + off, *dO = a->dout + off;
    const double *o = a->o_in + off, *L = a->lse_in + (size_t)bh * N;
    double *dq = a->dq + off, *dk = a->dk + off, *dv = a->dv + off;
    int Tr = (N + Br - 1) / Br, Tc = (N + Bc - 1) / Bc;
    double* D = (double*)malloc(sizeof(double) * (size_t)N);
    double* P = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
    double* dS = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
    for (int i = 0; i < N; ++i) {
        double acc = 0.0;
        for (int t = 0; t < d; ++t) acc += dO[(size_t)i * d + t] * o[(size_t)i * d + t];
        D[i] = acc;
    }
    for (size_t e = 0; e < (size_t)N * d; ++e) dq[e] = 0.0;
    for (int bj = 0; bj < Tc; ++bj) {
        int c0 = bj * Bc, nc = (c0 + Bc <= N) ? Bc : N - c0;
        for (int c = 0; c < nc; ++c)
            for (int t = 0; t < d; ++t) {
                dk[(size_t)(c0 + c) * d + t] = 0.0;
                dv[(size_t)(c0 + c) * d + t] = 0.0;
            }
        for (int bi = 0; bi < Tr; ++bi) {
            int r0 = bi * Br, nr = (r0 + Br <= N) ? Br : N - r0;
            for (int r = 0; r < nr; ++r)
                for (int c = 0; c < nc; ++c) {
                    double acc = 0.0;
                    for (int t = 0; t < d; ++t) acc += q[(size_t)(r0 + r) * d + t] * k[(size_t)(c0 + c) * d + t];
                    double s = mask_score(acc, r0 + r, c0 + c, kv_len, a->causal, a->scale);
                    double Li = L[r0 + r];
                    double p = (s == -INFINITY || Li == -INFINITY) ? 0.0 : exp(s - Li);
                    P[(size_t)r * Bc + c] = p;
                }
            /* dV_j += P^T dO_i */
            for (int c = 0; c < nc; ++c)
                for (int t = 0; t < d; ++t) {
                    double acc = 0.0;
                    for (int r = 0; r < nr; ++r) acc += P[(size_t)r * Bc + c] * dO[(size_t)(r0 + r) * d + t];
                    dv[(size_t)(c0 + c) * d + t] += acc;
                }
            /* dP = dO_i V_j^T ; dS = P (dP - D_i) */
            for (int r = 0; r < nr; ++r)
                for (int c = 0; c < nc; ++c) {
                    double acc = 0.0;
                    for (int t = 0; t < d; ++t) acc += dO[(size_t)(r0 + r) * d + t] * v[(size_t)(c0 + c) * d + t];
                    dS[(size_t)r * Bc + c] = P[(size_t)r * Bc + c] * (acc - D[r0 + r]);
                }
            /* dQ_i += scale dS K_j */
            for (int r = 0; r < nr; ++r)
                for (int t = 0; t < d; ++t) {
                    double acc = 0.0;
                    for (int c = 0; c < nc; ++c) acc += dS[(size_t)r * Bc + c] * k[(size_t)(c0 + c) * d + t];
                    dq[(size_t)(r0 + r) * d + t] += a->scale * acc;
                }
            /* dK_j += scale dS^T Q_i */
            for (int c = 0; c < nc; ++c)
                for (int t = 0; t < d; ++t) {
                    double acc = 0.0;
                    for (int r = 0; r < nr; ++r) acc += dS[(size_t)r * Bc + c] * q[(size_t)(r0 + r) * d + t];
                    dk[(size_t)(c0 + c) * d + t] += a->scale * acc;
                }
        }
    }
    free(D);
    free(P);
    free(dS);
}

int oracle_tiled_bwd(const double* q, const double* k, const double* v, const double* o,
                     const double* lse, const double* dout, double* dq, double* dk, double* dv,
                     int B, int H, int N, int d, double scale, int causal, const int* kv_lens,
                     int Br, int Bc, int nthreads) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || Br <= 0 || Bc <= 0) return OR_ERR;
    tiled_args a;
    memset(&a, 0, sizeof(a));
    a.q = q; a.k = k; a.v = v; a.o_in = o; a.lse_in = lse; a.dout = dout;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.B = B; a.H = H; a.N = N; a.d = d; a.causal = causal; a.Br = Br; a.Bc = Bc;
    a.scale = scale; a.kv_lens = kv_lens;
    run_items(tiled_bwd_item, &a, (long)B * H, nthreads);
    return OR_OK;
}

/* ======================================================================== */
/* 4. FP8 E4M3 per-block quantisation ([CH18] §18.6.2: s = max|X| / 448,     */
/*    X8 = quant_E4M3(X / s)).  The code decision is taken in fp32, like the */
/*    device path: amax and X are bf16 values (exact in fp32), s = amax/448  */
/*    and X/s are IEEE fp32 divisions, then X/s is rounded to E4M3 with      */
/*    round-to-nearest-even and saturation to +-448.                         */
/*    E4M3 (OCP FP8 "E4M3FN"): 1 sign, 4 exponent bits (bias 7), 3 mantissa  */
/*    bits; no infinities; S.1111.111 is NaN; largest finite 448; smallest   */
/*    subnormal 2^-9.                                                        */
/* ======================================================================== */

double oracle_e4m3_decode(uint8_t code) {
    int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/* Round a finite fp32 value to the nearest E4M3 value (ties to even code),
 * saturating at +-448.  Done by exhaustive comparison against the 127
 * non-negative finite codes: slow but obviously correct. */
uint8_t oracle_e4m3_encode(float xf) {
    double x = (double)xf;
    if (x != x) return 0x7F;
    int neg = signbit(xf) ? 1 : 0;
    double ax = fabs(x);
    uint8_t best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double val = oracle_e4m3_decode((uint8_t)c);
        double err = fabs(val - ax);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_err = err;
        }
    }
    /* anything beyond the largest finite value saturates to it */
    if (ax > 448.0) best = 0x7E;
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* x: [B,H,N,d] fp32 values (bf16-representable); x8: [B,H,N,d] codes;
 * scales: [B,H,ceil(N/blk)]; block = blk consecutive rows x all d columns. */
int oracle_quantize_fp8(const float* x, uint8_t* x8, float* scales, int B, int H, int N, int d,
                        int blk) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || blk <= 0) return OR_ERR;
    int nb = (N + blk - 1) / blk;
    for (long bh = 0; bh < (long)B * H; ++bh) {
        for (int ib = 0; ib < nb; ++ib) {
            int r0 = ib * blk, r1 = r0 + blk < N ? r0 + blk : N;
            float amax = 0.0f;
            for (int r = r0; r < r1; ++r)
                for (int t = 0; t < d; ++t) {
                    float a = fabsf(x[((size_t)bh * N + r) * d + t]);
                    if (a > amax) amax = a;
                }
            volatile float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
            scales[(size_t)bh * nb + ib] = s;
            for (int r = r0; r < r1; ++r)
                for (int t = 0; t < d; ++t) {
                    size_t e = ((size_t)bh * N + r) * d + t;
                    volatile float y = x[e] / s;
                    x8[e] = oracle_e4m3_encode(y);
                }
        }
    }
    return OR_OK;
}
