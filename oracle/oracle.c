/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the row softmax, the
 * attention forward and the attention backward (gradients).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library and includes nothing from it.
 *
 * Sources (the pages the method is defined on):
 *   [L22] "第二十二课：Softmax 为什么难以高效，以及 FlashAttention 如何减少显存访问"
 *         (lincklin.cn, lesson 22)
 *   [FG]  "少搬一趟：FlashAttention 四代进化史" (chengshu-blog, booklet)
 *   [OF]  "从 FlashAttention 看懂算子融合：为什么融合、少读写了什么、又会错在哪里"
 *         (jokeuncle.github.io notes)
 *
 * Every floating-point step runs in IEEE double.  Inputs arrive as float
 * (fp32 values, or bf16 values widened to fp32, which is exact) and are widened
 * to double before any arithmetic.
 *
 * Layouts (row-major, contiguous):
 *   softmax:   x, y  [rows, N]
 *   attention: Q, K, V, O  [total, H, d]  (token-major, heads, head dim)
 *              lse         [H, total]
 *              cu_seqlens  [B + 1], int32 prefix sums of the sequence lengths;
 *              sequence b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1.
 *   A dense [B, N, H, d] batch is the packed layout with
 *   cu_seqlens = {0, N, 2N, ..., B*N}.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Row softmax                                                               */
/* ------------------------------------------------------------------------ */

/*
 * Numerically stable softmax of one row, in the three passes of [L22] §三
 * ("稳定 Softmax 至少需要哪些步骤"), using the shift by the row maximum of
 * [L22] §二 ("数值稳定 Softmax"):
 *   pass 1  m = max_j x_j
 *   pass 2  s = sum_j exp(x_j - m)
 *   pass 3  y_j = exp(x_j - m) / s
 */
static void softmax_row(const float *x, double *y, int64_t N)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        double xj = (double)x[j];
        if (xj > m)
            m = xj;
    }
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j)
        s += exp((double)x[j] - m);
    for (int64_t j = 0; j < N; ++j)
        y[j] = exp((double)x[j] - m) / s;
}

/* Row softmax over a [rows, N] matrix; rows are independent ([L22] §五). */
void oracle_softmax_rows(const float *x, double *y, int64_t rows, int64_t N)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        softmax_row(x + r * N, y + r * N, N);
}

/* ------------------------------------------------------------------------ */
/* Online softmax: the block merge, used only to cross-check the oracle     */
/* ------------------------------------------------------------------------ */

/*
 * Running (m, l) of a row whose entries arrive in blocks.  Block k covers
 * x[block_ends[k-1] .. block_ends[k]-1] (block_ends[-1] = 0, the last entry of
 * block_ends is n).  Each block yields its own (m_B, l_B) by the stable form;
 * the running state absorbs it with the merge rule of [L22] §十九
 * ("Online Softmax 的最大值更新"):
 *   m = max(m_A, m_B)
 *   l = exp(m_A - m) * l_A + exp(m_B - m) * l_B
 * starting from m = -inf, l = 0 ([L22] §三十二).  A block of one entry is the
 * per-element update of [L22] §二十.  The first merge would compute
 * exp(-inf - (-inf)); since l_A = 0 there, the empty running state is simply
 * replaced by the first block.
 */
void oracle_online_softmax_state(const double *x, int64_t n, const int64_t *block_ends,
                                 int64_t nblocks, double *m_out, double *l_out)
{
    double m = -INFINITY, l = 0.0;
    int64_t begin = 0;
    for (int64_t k = 0; k < nblocks; ++k) {
        int64_t end = block_ends[k];
        if (end > n)
            end = n;
        if (end <= begin)
            continue;
        double mb = -INFINITY;
        for (int64_t j = begin; j < end; ++j)
            if (x[j] > mb)
                mb = x[j];
        double lb = 0.0;
        for (int64_t j = begin; j < end; ++j)
            lb += exp(x[j] - mb);
        if (l == 0.0 && m == -INFINITY) {
            m = mb;
            l = lb;
        } else {
            double mn = m > mb ? m : mb;
            l = exp(m - mn) * l + exp(mb - mn) * lb;
            m = mn;
        }
        begin = end;
    }
    *m_out = m;
    *l_out = l;
}

/* ------------------------------------------------------------------------ */
/* Attention forward                                                         */
/* ------------------------------------------------------------------------ */

/* Index of the sequence that owns token t (cu_seqlens is non-decreasing). */
static int64_t owner_sequence(const int32_t *cu_seqlens, int64_t B, int64_t t)
{
    int64_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int64_t mid = (lo + hi + 1) / 2;
        if ((int64_t)cu_seqlens[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/*
 * One query row of exact attention, straight from the definition
 * ([L22] §十二–§十三, [FG] §1.2):
 *   s_j  = scale * (q . k_j)                 for every visible key j
 *   p_j  = exp(s_j - m) / l,  m = max_j s_j,  l = sum_j exp(s_j - m)
 *   o    = sum_j p_j v_j
 *   lse  = m + ln(l) = ln sum_j exp(s_j)     ([FG] §2.4)
 * Visible keys: the keys of the query's own sequence, and, when causal,
 * only those at positions j <= i ([L22] §三十四; masked scores are -inf and
 * contribute exp(-inf) = 0, so they are simply left out of the sums).
 *
 * start: first token of the sequence; L: its length; i: query position in it.
 * s: scratch of at least L doubles.
 */
static void attention_row(const float *Q, const float *K, const float *V, int64_t H,
                          int64_t d, double scale, int causal, int64_t start, int64_t L,
                          int64_t i, int64_t h, double *s, double *o, double *lse)
{
    const float *q = Q + ((start + i) * H + h) * d;
    int64_t nvis = causal ? (i + 1 < L ? i + 1 : L) : L;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const float *k = K + ((start + j) * H + h) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += (double)q[c] * (double)k[c];
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    /* pass 2: normaliser */
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        l += exp(s[j] - m);
    /* pass 3: probabilities times values */
    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s[j] - m) / l;
        const float *v = V + ((start + j) * H + h) * d;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * (double)v[c];
    }
    *lse = nvis > 0 ? m + log(l) : -INFINITY;
}

/*
 * Full attention forward over all sequences, heads and query rows.
 * O: [total, H, d] doubles; lse: [H, total] doubles.
 */
void oracle_attention_fwd(const float *Q, const float *K, const float *V, double *O,
                          double *lse, int64_t B, int64_t H, int64_t d, double scale,
                          int causal, const int32_t *cu_seqlens)
{
    int64_t total = cu_seqlens[B];
    /* scratch for one row of scores; no sequence is longer than the packed total */
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(total > 0 ? total : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 16)
        for (int64_t w = 0; w < total * H; ++w) {
            int64_t t = w / H, h = w % H;
            int64_t b = owner_sequence(cu_seqlens, B, t);
            int64_t start = cu_seqlens[b];
            int64_t L = (int64_t)cu_seqlens[b + 1] - start;
            attention_row(Q, K, V, H, d, scale, causal, start, L, t - start, h, s,
                          O + (t * H + h) * d, lse + h * total + t);
        }
        free(s);
    }
}

/*
 * The same definition evaluated only on n sampled (token, head) pairs.
 * O_rows: [n, d]; lse_rows: [n].  Used where the full problem is too large for
 * the CPU within a test's time.
 */
void oracle_attention_rows(const float *Q, const float *K, const float *V, int64_t B,
                           int64_t H, int64_t d, double scale, int causal,
                           const int32_t *cu_seqlens, const int64_t *tok, const int64_t *head,
                           int64_t n, double *O_rows, double *lse_rows)
{
    int64_t total = cu_seqlens[B];
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(total > 0 ? total : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            int64_t t = tok[r], h = head[r];
            int64_t b = owner_sequence(cu_seqlens, B, t);
            int64_t start = cu_seqlens[b];
            int64_t L = (int64_t)cu_seqlens[b + 1] - start;
            attention_row(Q, K, V, H, d, scale, causal, start, L, t - start, h, s,
                          O_rows + r * d, lse_rows + r);
        }
        free(s);
    }
}

/*
 * Cross-check only (not what the GPU path is compared with): the tiled
 * online recurrence of [L22] §三十二 ("FlashAttention 的伪代码") and
 * [FG] §2.2, evaluated in fp64 with key tiles of T entries.  Per query row:
 *   m = -inf, l = 0, acc = 0
 *   for each key tile:  new_m = max(m, max_j s_j)
 *                       p_j   = exp(s_j - new_m)
 *                       c     = exp(m - new_m)
 *                       l     = c * l + sum_j p_j
 *                       acc   = c * acc + sum_j p_j v_j
 *                       m     = new_m
 *   o = acc / l,  lse = m + ln l
 * The first tile has m = -inf; its correction factor is taken as 0 (l and acc
 * are still 0 there), which avoids the undefined exp(-inf - (-inf)).
 */
void oracle_attention_fwd_online(const float *Q, const float *K, const float *V, double *O,
                                 double *lse, int64_t B, int64_t H, int64_t d, double scale,
                                 int causal, const int32_t *cu_seqlens, int64_t T)
{
    int64_t total = cu_seqlens[B];
    if (T < 1)
        T = 1;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)T * sizeof(double));
        double *acc = (double *)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 16)
        for (int64_t w = 0; w < total * H; ++w) {
            int64_t t = w / H, h = w % H;
            int64_t b = owner_sequence(cu_seqlens, B, t);
            int64_t start = cu_seqlens[b];
            int64_t L = (int64_t)cu_seqlens[b + 1] - start;
            int64_t i = t - start;
            int64_t nvis = causal ? (i + 1 < L ? i + 1 : L) : L;
            const float *q = Q + (t * H + h) * d;
            double m = -INFINITY, l = 0.0;
            for (int64_t c = 0; c < d; ++c)
                acc[c] = 0.0;
            for (int64_t j0 = 0; j0 < nvis; j0 += T) {
                int64_t j1 = j0 + T < nvis ? j0 + T : nvis;
                double bmax = -INFINITY;
                for (int64_t j = j0; j < j1; ++j) {
                    const float *k = K + ((start + j) * H + h) * d;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += (double)q[c] * (double)k[c];
                    s[j - j0] = scale * dot;
                    if (s[j - j0] > bmax)
                        bmax = s[j - j0];
                }
                double new_m = m > bmax ? m : bmax;
                double corr = (m == -INFINITY) ? 0.0 : exp(m - new_m);
                l *= corr;
                for (int64_t c = 0; c < d; ++c)
                    acc[c] *= corr;
                for (int64_t j = j0; j < j1; ++j) {
                    double p = exp(s[j - j0] - new_m);
                    const float *v = V + ((start + j) * H + h) * d;
                    l += p;
                    for (int64_t c = 0; c < d; ++c)
                        acc[c] += p * (double)v[c];
                }
                m = new_m;
            }
            double *o = O + (t * H + h) * d;
            for (int64_t c = 0; c < d; ++c)
                o[c] = nvis > 0 ? acc[c] / l : 0.0;
            lse[h * total + t] = nvis > 0 ? m + log(l) : -INFINITY;
        }
        free(acc);
        free(s);
    }
}

/*
 * Attention with separate query and key lengths (dense batches), the form used
 * when the keys of a query block are processed in several splits:
 *   Q, O: [B, Nq, H, d];  K, V: [B, Nk, H, d];  lse: [B, H, Nq].
 * Same definition as attention_row; when causal, query i sees the keys
 * j <= i + (Nk - Nq): the queries are the last Nq positions of a sequence of
 * Nk keys (bottom-right alignment; with Nq == Nk this is [L22] §三十四's j <= i).
 * Rows are evaluated only for the n sampled (b, i, h) triples given (all rows
 * when samp_b == NULL, in which case n must be B * Nq * H).
 */
void oracle_attention_qk(const float *Q, const float *K, const float *V, int64_t B, int64_t H,
                         int64_t Nq, int64_t Nk, int64_t d, double scale, int causal,
                         const int64_t *samp_b, const int64_t *samp_i, const int64_t *samp_h,
                         int64_t n, double *O_rows, double *lse_rows)
{
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            int64_t b, i, h;
            if (samp_b != NULL) {
                b = samp_b[r];
                i = samp_i[r];
                h = samp_h[r];
            } else {
                b = r / (Nq * H);
                i = (r / H) % Nq;
                h = r % H;
            }
            const float *q = Q + ((b * Nq + i) * H + h) * d;
            int64_t nvis = causal ? i + (Nk - Nq) + 1 : Nk;
            if (nvis > Nk)
                nvis = Nk;
            if (nvis < 0)
                nvis = 0;
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                const float *k = K + ((b * Nk + j) * H + h) * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += (double)q[c] * (double)k[c];
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                l += exp(s[j] - m);
            double *o = O_rows + r * d;
            for (int64_t c = 0; c < d; ++c)
                o[c] = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                double p = exp(s[j] - m) / l;
                const float *v = V + ((b * Nk + j) * H + h) * d;
                for (int64_t c = 0; c < d; ++c)
                    o[c] += p * (double)v[c];
            }
            lse_rows[r] = nvis > 0 ? m + log(l) : -INFINITY;
        }
        free(s);
    }
}

/* ------------------------------------------------------------------------ */
/* Attention backward                                                        */
/* ------------------------------------------------------------------------ */
/*
 * Gradients of the loss sum(dO * O) with respect to Q, K and V, for the forward
 * definition above on dense batches [B, N, H, d] (causal: j <= i).  The pages
 * recompute the probabilities from the saved row statistic instead of storing
 * them ([FG] §2.4: P_ij = exp(S_ij - L_i) with L = m + log l; [L22] §三十) and
 * leave the derivation of the gradients out ([FG], list of omitted topics at
 * the end).  Reading: the plain chain rule through S = scale Q K^T,
 * P = softmax(S) (row-wise over the visible keys), O = P V:
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (softmax Jacobian)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_i dS_ij Q_i
 * Everything is recomputed here from Q, K, V, dO in double; the row statistic
 * L_i = m_i + log l_i and D_i = sum_k P_ik dP_ik are returned for checks.
 * One (b, h) at a time; S and P are materialised (N x N doubles): small N.
 * Outputs: dQ, dK, dV, O [B, N, H, d]; lse, D [B, H, N] (O, lse, D may be NULL).
 */
void oracle_attention_bwd(const float *Q, const float *K, const float *V, const float *dO,
                          int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                          double *dQ, double *dK, double *dV, double *O, double *lse, double *D)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        double *P = (double *)calloc((size_t)(N * N > 0 ? N * N : 1), sizeof(double));
        double *dP = (double *)calloc((size_t)(N * N > 0 ? N * N : 1), sizeof(double));
#define ROW(X, t) ((X) + ((b * N + (t)) * H + h) * d)
        for (int64_t i = 0; i < N; ++i) {
            const int64_t nvis = causal ? i + 1 : N;
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += (double)ROW(Q, i)[c] * (double)ROW(K, j)[c];
                P[i * N + j] = scale * dot;             /* S for now */
                if (P[i * N + j] > m)
                    m = P[i * N + j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                l += exp(P[i * N + j] - m);
            const double L = m + log(l);
            for (int64_t j = 0; j < nvis; ++j)
                P[i * N + j] = exp(P[i * N + j] - L);   /* [FG] §2.4 */
            double Di = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += (double)ROW(dO, i)[c] * (double)ROW(V, j)[c];
                dP[i * N + j] = dot;
                Di += P[i * N + j] * dot;
            }
            if (lse)
                lse[(b * H + h) * N + i] = L;
            if (D)
                D[(b * H + h) * N + i] = Di;
            if (O)
                for (int64_t c = 0; c < d; ++c) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < nvis; ++j)
                        acc += P[i * N + j] * (double)ROW(V, j)[c];
                    ROW(O, i)[c] = acc;
                }
            /* dS overwrites dP */
            for (int64_t j = 0; j < nvis; ++j)
                dP[i * N + j] = P[i * N + j] * (dP[i * N + j] - Di);
        }
        for (int64_t i = 0; i < N; ++i)
            for (int64_t c = 0; c < d; ++c) {
                const int64_t nvis = causal ? i + 1 : N;
                double acc = 0.0;
                for (int64_t j = 0; j < nvis; ++j)
                    acc += dP[i * N + j] * (double)ROW(K, j)[c];
                ROW(dQ, i)[c] = scale * acc;
            }
        for (int64_t j = 0; j < N; ++j)
            for (int64_t c = 0; c < d; ++c) {
                double acc_k = 0.0, acc_v = 0.0;
                for (int64_t i = causal ? j : 0; i < N; ++i) {
                    acc_k += dP[i * N + j] * (double)ROW(Q, i)[c];
                    acc_v += P[i * N + j] * (double)ROW(dO, i)[c];
                }
                ROW(dK, j)[c] = scale * acc_k;
                ROW(dV, j)[c] = acc_v;
            }
#undef ROW
        free(P);
        free(dP);
    }
}

/*
 * The same gradients for one (b, h) of a large batch, for the listed query
 * rows (dQ) and keys (dK, dV) only.  First L_i and D_i of every query row of
 * the head are computed (one pass over its keys per row), then each listed
 * row or key costs one pass over the other side.  Outputs: dQ_rows [nq, d],
 * dK_rows, dV_rows [nk, d].
 */
void oracle_attention_bwd_head(const float *Q, const float *K, const float *V, const float *dO,
                               int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                               int causal, int64_t b, int64_t h, const int64_t *q_idx, int64_t nq,
                               const int64_t *k_idx, int64_t nk, double *dQ_rows,
                               double *dK_rows, double *dV_rows)
{
    (void)B;
    double *L = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *Dv = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#define ROW(X, t) ((X) + ((b * N + (t)) * H + h) * d)
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 8)
        for (int64_t i = 0; i < N; ++i) {
            const int64_t nvis = causal ? i + 1 : N;
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += (double)ROW(Q, i)[c] * (double)ROW(K, j)[c];
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                l += exp(s[j] - m);
            L[i] = m + log(l);
            double Di = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += (double)ROW(dO, i)[c] * (double)ROW(V, j)[c];
                Di += exp(s[j] - L[i]) * dot;
            }
            Dv[i] = Di;
        }
        free(s);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nq; ++r) {
            const int64_t i = q_idx[r];
            const int64_t nvis = causal ? i + 1 : N;
            double *out = dQ_rows + r * d;
            for (int64_t c = 0; c < d; ++c)
                out[c] = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                double sdot = 0.0, pdot = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    sdot += (double)ROW(Q, i)[c] * (double)ROW(K, j)[c];
                    pdot += (double)ROW(dO, i)[c] * (double)ROW(V, j)[c];
                }
                const double P = exp(scale * sdot - L[i]);
                const double dS = P * (pdot - Dv[i]);
                for (int64_t c = 0; c < d; ++c)
                    out[c] += scale * dS * (double)ROW(K, j)[c];
            }
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nk; ++r) {
            const int64_t j = k_idx[r];
            double *ok = dK_rows + r * d, *ov = dV_rows + r * d;
            for (int64_t c = 0; c < d; ++c)
                ok[c] = ov[c] = 0.0;
            for (int64_t i = causal ? j : 0; i < N; ++i) {
                double sdot = 0.0, pdot = 0.0;
                for (int64_t c = 0; c < d; ++c) {
                    sdot += (double)ROW(Q, i)[c] * (double)ROW(K, j)[c];
                    pdot += (double)ROW(dO, i)[c] * (double)ROW(V, j)[c];
                }
                const double P = exp(scale * sdot - L[i]);
                const double dS = P * (pdot - Dv[i]);
                for (int64_t c = 0; c < d; ++c) {
                    ok[c] += scale * dS * (double)ROW(Q, i)[c];
                    ov[c] += P * (double)ROW(dO, i)[c];
                }
            }
        }
    }
#undef ROW
    free(L);
    free(Dv);
}

/* Threads the OpenMP runtime will use for the parallel loops above. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the thread count of the parallel loops that follow (n >= 1); for
 * timing the oracle on one core. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
