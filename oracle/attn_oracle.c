/*
 * Exact scaled-dot-product attention on the CPU, in double precision.
 *
 * TEST INFRASTRUCTURE.  This file is the oracle that the GPU kernels are
 * checked against.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the product path never does.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * What it computes is the plain definition of attention, with S and P
 * written out row by row (no online recurrence, no tiling):
 *
 *   S_ij  = scale * q_i . k_j           (or -inf where key j is masked for query i)
 *   m_i   = max_j S_ij                  pass 1 of the safe softmax
 *   l_i   = sum_j exp(S_ij - m_i)       pass 2
 *   P_ij  = exp(S_ij - m_i) / l_i       pass 3
 *   O_i   = sum_j P_ij v_j
 *   LSE_i = m_i + ln(l_i)
 *
 * Sources: "注意力为什么受限于显存带宽：用算术强度与分块把 FlashAttention 推导清楚"
 * (magicnetworld.com), section 五 (standard attention: S = QK^T, P = softmax(S),
 * O = PV) and section 六 (subtract the row maximum before exponentiating);
 * "4. FlashAttention 深度剖析" (llm-training-tutorial), section 4.2.1 (the
 * three-pass safe softmax) and section 4.3.2 (the saved statistic
 * L = m + log l).
 *
 * Backward.  The pages name dS, dQ, dK, dV and say P is recomputed from the
 * saved statistics (magicnetworld section 八; llm-training-tutorial 4.3.4) but
 * print no gradient formulas.  The reading used here is the chain rule
 * through O = P V and the row softmax, for a loss whose gradient w.r.t. O
 * is dO:
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *
 * Masks.  Key j is visible to query i iff j < kv_len[b], j <= i when causal,
 * j >= i - window_left when window_left >= 0, and j <= i + window_right when
 * window_right >= 0 (square attention, N queries and N keys, 0-based
 * indices).  The window is the (left, right) pair of flash-attn's
 * window_size argument, (-1, -1) meaning no window ("炉案与百步之外的仓库：
 * Flash Attention 与注意力计算的工艺极限" section 六; "4. FlashAttention 深度
 * 剖析" 4.8.1, sliding window).  A block mask (the coarse block-level mask
 * matrix of "炉案与百步之外的仓库…" 第八部分, Block-Sparse FlashAttention)
 * hides further keys: with blocks of bs rows and bs columns, key j is
 * visible to query i only if entry (i / bs, j / bs) of the row-major
 * [ceil(N/bs), ceil(N/bs)] byte matrix is nonzero.  A row with no visible key
 * gets O = 0 and LSE = -inf.
 *
 * Grouped K/V heads (GQA / MQA, the same section 六 and the FlashAttention-2
 * summary in "注意力为什么受限于显存带宽…" section 九): K and V have
 * H_kv heads, H_kv divides H, and query head h reads K/V head
 * h / (H / H_kv).  dK and dV of a K/V head are the sums over the query heads
 * that read it.
 *
 * Layout: Q, O, dO, dQ are contiguous [B, H, N, d] arrays of doubles, K, V,
 * dK, dV are [B, H_kv, N, d], LSE and D are [B, H, N].  kv_len is NULL (no
 * padding) or an int array of length B.
 * Rows are spread over OpenMP threads when the file is built with -fopenmp;
 * the per-row arithmetic does not depend on the thread count, only the order
 * of the final dK/dV sums across threads does (a rounding-level effect).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

typedef struct {
    int causal;
    long len;          /* kv_len of the batch entry */
    long wl, wr;       /* window: -1 = unbounded on that side */
    const unsigned char *bm;   /* block mask or NULL */
    long bs, tk;       /* its block size and row length (blocks of keys) */
} mask_t;

static int key_visible(long i, long j, const mask_t *m)
{
    if (j >= m->len) return 0;
    if (m->causal && j > i) return 0;
    if (m->wl >= 0 && j < i - m->wl) return 0;
    if (m->wr >= 0 && j > i + m->wr) return 0;
    if (m->bm && !m->bm[(i / m->bs) * m->tk + j / m->bs]) return 0;
    return 1;
}

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += a[t] * b[t];
    return s;
}

/* One row of P for query i of one head: fills p[0..N) (0 for masked keys)
 * and returns the LSE of the row.  The three passes of the safe softmax. */
static double softmax_row(const double *qi, const double *K, int N, int d,
                          double scale, const mask_t *mk, long i, double *p)
{
    double m = -INFINITY;
    int any = 0;
    for (long j = 0; j < N; ++j) {               /* S row and pass 1: max */
        if (key_visible(i, j, mk)) {
            p[j] = scale * dot(qi, K + j * (long)d, d);
            if (p[j] > m) m = p[j];
            any = 1;
        } else {
            p[j] = -INFINITY;
        }
    }
    if (!any) {
        for (long j = 0; j < N; ++j) p[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (long j = 0; j < N; ++j) {               /* pass 2: sum of exp(S - m) */
        p[j] = key_visible(i, j, mk) ? exp(p[j] - m) : 0.0;
        l += p[j];
    }
    for (long j = 0; j < N; ++j) p[j] /= l;      /* pass 3: normalise */
    return m + log(l);
}

static int check_args(const void *a, const void *b, const void *c, int B, int H, int N, int d)
{
    if (!a || !b || !c) return 0;
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return 1;
}

static int check_heads(int H, int H_kv)
{
    return H_kv >= 1 && H_kv <= H && H % H_kv == 0;
}

int fa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over every (b, h) and every row; K/V head of query head h is
 * h / (H / H_kv), window (wl, wr) and block mask (bm, bs) as in the header
 * (bm NULL: none). */
int fa_oracle_forward_m(const double *q, const double *k, const double *v,
                        double *o, double *lse,
                        int B, int H, int H_kv, int N, int d, double scale, int causal,
                        const int *kv_len, int wl, int wr, const unsigned char *bm, int bs,
                        int nthreads)
{
    if (!check_args(q, k, v, B, H, N, d) || !o || !lse || !check_heads(H, H_kv) ||
        (bm && bs < 1))
        return ORACLE_EINVAL;
    const long tk = bm ? ((long)N + bs - 1) / bs : 0;
    if (nthreads < 1) nthreads = 1;
    const long hd = (long)N * d;
    const int group = H / H_kv;
    int err = ORACLE_OK;
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const long b = bh / H;
        const long kvh = b * H_kv + (bh % H) / group;
        const mask_t mk = {causal, kv_len ? kv_len[b] : N, wl, wr, bm, bm ? bs : 1, tk};
        const double *Q = q + bh * hd, *K = k + kvh * hd, *V = v + kvh * hd;
        double *O = o + bh * hd, *L = lse + bh * (long)N;
#pragma omp parallel num_threads(nthreads)
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)N);
            if (!p) {
#pragma omp atomic write
                err = ORACLE_ENOMEM;
            }
            /* every thread meets the work-sharing loop; one without a buffer skips rows */
#pragma omp for schedule(dynamic, 8)
            for (long i = 0; i < N; ++i) {
                if (!p) continue;
                {
                    L[i] = softmax_row(Q + i * d, K, N, d, scale, &mk, i, p);
                    double *oi = O + i * d;
                    for (int t = 0; t < d; ++t) oi[t] = 0.0;
                    for (long j = 0; j < N; ++j) {
                        if (p[j] == 0.0) continue;
                        const double *vj = V + j * d;
                        for (int t = 0; t < d; ++t) oi[t] += p[j] * vj[t];
                    }
                }
            }
            free(p);
        }
        if (err) return err;
    }
    return ORACLE_OK;
}

int fa_oracle_forward_v(const double *q, const double *k, const double *v,
                        double *o, double *lse,
                        int B, int H, int H_kv, int N, int d, double scale, int causal,
                        const int *kv_len, int wl, int wr, int nthreads)
{
    return fa_oracle_forward_m(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, kv_len, wl, wr,
                               NULL, 1, nthreads);
}

int fa_oracle_forward(const double *q, const double *k, const double *v,
                      double *o, double *lse,
                      int B, int H, int N, int d, double scale, int causal,
                      const int *kv_len, int nthreads)
{
    return fa_oracle_forward_v(q, k, v, o, lse, B, H, H, N, d, scale, causal, kv_len, -1, -1,
                               nthreads);
}

/* Forward for a chosen set of query rows of ONE head (q, k, v are [N, d]).
 * o_rows is [nrows, d], lse_rows is [nrows]; len is that head's kv_len. */
int fa_oracle_forward_rows_v(const double *q, const double *k, const double *v,
                             int N, int d, double scale, int causal, int len, int wl, int wr,
                             const int *rows, int nrows,
                             double *o_rows, double *lse_rows, int nthreads)
{
    const mask_t mk = {causal, len, wl, wr, NULL, 1, 0};
    if (!check_args(q, k, v, 1, 1, N, d) || !rows || !o_rows || !lse_rows || nrows < 0)
        return ORACLE_EINVAL;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return ORACLE_EINVAL;
    if (nthreads < 1) nthreads = 1;
    int err = ORACLE_OK;
#pragma omp parallel num_threads(nthreads)
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            if (!p) continue;
            {
                const long i = rows[r];
                lse_rows[r] = softmax_row(q + i * d, k, N, d, scale, &mk, i, p);
                double *oi = o_rows + (long)r * d;
                for (int t = 0; t < d; ++t) oi[t] = 0.0;
                for (long j = 0; j < N; ++j) {
                    if (p[j] == 0.0) continue;
                    const double *vj = v + j * d;
                    for (int t = 0; t < d; ++t) oi[t] += p[j] * vj[t];
                }
            }
        }
        free(p);
    }
    return err;
}

int fa_oracle_forward_rows(const double *q, const double *k, const double *v,
                           int N, int d, double scale, int causal, int len,
                           const int *rows, int nrows,
                           double *o_rows, double *lse_rows, int nthreads)
{
    return fa_oracle_forward_rows_v(q, k, v, N, d, scale, causal, len, -1, -1, rows, nrows,
                                    o_rows, lse_rows, nthreads);
}

/* Backward over every (b, h): dq is [B,H,N,d], dk and dv are [B,H_kv,N,d]
 * (sums over the query heads of each group); D is [B,H,N]
 * (D_i = sum_j P_ij dP_ij).  P is rebuilt from its definition, not from a
 * stored LSE, so the oracle does not depend on the forward's outputs. */
int fa_oracle_backward_m(const double *q, const double *k, const double *v,
                         const double *dout,
                         double *dq, double *dk, double *dv, double *D,
                         int B, int H, int H_kv, int N, int d, double scale, int causal,
                         const int *kv_len, int wl, int wr, const unsigned char *bm, int bs,
                         int nthreads)
{
    if (!check_args(q, k, v, B, H, N, d) || !dout || !dq || !dk || !dv || !D ||
        !check_heads(H, H_kv) || (bm && bs < 1))
        return ORACLE_EINVAL;
    const long tk = bm ? ((long)N + bs - 1) / bs : 0;
    if (nthreads < 1) nthreads = 1;
    const long hd = (long)N * d;
    const int group = H / H_kv;
    int err = ORACLE_OK;
    memset(dk, 0, sizeof(double) * (size_t)((long)B * H_kv * hd));
    memset(dv, 0, sizeof(double) * (size_t)((long)B * H_kv * hd));
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const long b = bh / H;
        const long kvh = b * H_kv + (bh % H) / group;
        const mask_t mk = {causal, kv_len ? kv_len[b] : N, wl, wr, bm, bm ? bs : 1, tk};
        const double *Q = q + bh * hd, *K = k + kvh * hd, *V = v + kvh * hd;
        const double *dO = dout + bh * hd;
        double *dQ = dq + bh * hd, *dK = dk + kvh * hd, *dV = dv + kvh * hd;
        double *Dh = D + bh * (long)N;
#pragma omp parallel num_threads(nthreads)
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)N);
            double *dp = (double *)malloc(sizeof(double) * (size_t)N);
            double *dk_loc = (double *)calloc((size_t)hd, sizeof(double));
            double *dv_loc = (double *)calloc((size_t)hd, sizeof(double));
            const int ok = p && dp && dk_loc && dv_loc;
            if (!ok) {
#pragma omp atomic write
                err = ORACLE_ENOMEM;
            }
#pragma omp for schedule(dynamic, 8)
            for (long i = 0; i < N; ++i) {
                if (!ok) continue;
                {
                    const double *qi = Q + i * d, *doi = dO + i * d;
                    softmax_row(qi, K, N, d, scale, &mk, i, p);
                    double Di = 0.0;
                    for (long j = 0; j < N; ++j) {        /* dP = dO V^T, D = rowsum(P o dP) */
                        dp[j] = (p[j] != 0.0) ? dot(doi, V + j * d, d) : 0.0;
                        Di += p[j] * dp[j];
                    }
                    Dh[i] = Di;
                    double *dqi = dQ + i * d;
                    for (int t = 0; t < d; ++t) dqi[t] = 0.0;
                    for (long j = 0; j < N; ++j) {
                        if (p[j] == 0.0) continue;
                        const double ds = p[j] * (dp[j] - Di);   /* dS = P o (dP - D) */
                        const double *kj = K + j * d;
                        double *dkj = dk_loc + j * d, *dvj = dv_loc + j * d;
                        for (int t = 0; t < d; ++t) {
                            dqi[t] += scale * ds * kj[t];
                            dkj[t] += scale * ds * qi[t];
                            dvj[t] += p[j] * doi[t];
                        }
                    }
                }
            }
            if (ok) {
#pragma omp critical
                {
                    for (long t = 0; t < hd; ++t) {
                        dK[t] += dk_loc[t];
                        dV[t] += dv_loc[t];
                    }
                }
            }
            free(p);
            free(dp);
            free(dk_loc);
            free(dv_loc);
        }
        if (err) return err;
    }
    return ORACLE_OK;
}

int fa_oracle_backward_v(const double *q, const double *k, const double *v,
                         const double *dout,
                         double *dq, double *dk, double *dv, double *D,
                         int B, int H, int H_kv, int N, int d, double scale, int causal,
                         const int *kv_len, int wl, int wr, int nthreads)
{
    return fa_oracle_backward_m(q, k, v, dout, dq, dk, dv, D, B, H, H_kv, N, d, scale, causal,
                                kv_len, wl, wr, NULL, 1, nthreads);
}

int fa_oracle_backward(const double *q, const double *k, const double *v,
                       const double *dout,
                       double *dq, double *dk, double *dv, double *D,
                       int B, int H, int N, int d, double scale, int causal,
                       const int *kv_len, int nthreads)
{
    return fa_oracle_backward_v(q, k, v, dout, dq, dk, dv, D, B, H, H, N, d, scale, causal,
                                kv_len, -1, -1, nthreads);
}

/* Decode-shaped attention: Nq queries per head against Nk keys.  Query t of
 * batch entry b sits at position pos = len_b - Nq + t of its sequence (the
 * newest Nq tokens of a key/value cache of len_b entries), so under causal it
 * sees keys j <= pos, and the window is taken around pos; keys j >= len_b are
 * never visible.  This is the shape FlashDecoding splits across SMs
 * ("4. FlashAttention 深度剖析" 4.8.3); the result is the plain definition, as
 * for fa_oracle_forward_v.  q, o: [B, H, Nq, d]; k, v: [B, H_kv, Nk, d]; lse:
 * [B, H, Nq]; kv_len NULL means len_b = Nk. */
int fa_oracle_decode(const double *q, const double *k, const double *v,
                     double *o, double *lse,
                     int B, int H, int H_kv, int Nq, int Nk, int d, double scale, int causal,
                     const int *kv_len, int wl, int wr, int nthreads)
{
    if (!check_args(q, k, v, B, H, Nq, d) || Nk < 1 || !o || !lse || !check_heads(H, H_kv))
        return ORACLE_EINVAL;
    if (nthreads < 1) nthreads = 1;
    const long qd = (long)Nq * d, kd = (long)Nk * d;
    const int group = H / H_kv;
    int err = ORACLE_OK;
    for (long bh = 0; bh < (long)B * H; ++bh) {
        const long b = bh / H;
        const long kvh = b * H_kv + (bh % H) / group;
        long len = kv_len ? kv_len[b] : Nk;
        if (len > Nk) len = Nk;
        const mask_t mk = {causal, len, wl, wr, NULL, 1, 0};
        const double *Q = q + bh * qd, *K = k + kvh * kd, *V = v + kvh * kd;
        double *O = o + bh * qd, *L = lse + bh * (long)Nq;
#pragma omp parallel num_threads(nthreads)
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
            if (!p) {
#pragma omp atomic write
                err = ORACLE_ENOMEM;
            }
#pragma omp for schedule(dynamic, 1)
            for (long t = 0; t < Nq; ++t) {
                if (!p) continue;
                {
                    const long pos = len - Nq + t;
                    L[t] = softmax_row(Q + t * d, K, Nk, d, scale, &mk, pos, p);
                    double *ot = O + t * d;
                    for (int c = 0; c < d; ++c) ot[c] = 0.0;
                    for (long j = 0; j < Nk; ++j) {
                        if (p[j] == 0.0) continue;
                        const double *vj = V + j * d;
                        for (int c = 0; c < d; ++c) ot[c] += p[j] * vj[c];
                    }
                }
            }
            free(p);
        }
        if (err) return err;
    }
    return ORACLE_OK;
}
