/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file; it exists so
 * that tests, the smoke check and the CPU-baseline leg of the bench can
 * compare the GPU kernels against the plain definition of the operation.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the definition, written out with no tiling, no
 * streaming and no reordering beyond "for every row, for every key":
 *
 *   M4.3 "IO-Aware Attention and FlashAttention-1", 0x02A (the semantic graph):
 *       S_raw[b,h,i,j] = tau * <Q[b,h,i,:], K[b,g(h),j,:]>
 *       S = mask(S_raw)                       (mask before row normalisation)
 *       P = softmax_row(S),  O = P V
 *   M4.3 0x06B (safe softmax): m = max_j s_j, l = sum_j exp(s_j - m)
 *   M4.3 0x09A / 0x09E: O = u / l with u = sum_j exp(s_j - m) v_j,
 *                       LSE = m + log(l)
 *   M4.4 "FlashAttention-2 Work Partitioning and the Decode Boundary",
 *       0x06A (GQA):
 *       g = H_q / H_kv, kv_head = q_head / g  (integer division)
 *   M4.4 0x05.1A / 0x05.1F (causal):
 *       visible(q, k) iff k <= q + delta, delta = S_k - S_q (bottom-right)
 *
 * The backward pass (oracle_attn_bwd, below) is the gradient of that
 * definition as M4.4 0x06.1A writes it: dP = dO V^T, dS = P o (dP - rowsum(P o dP)),
 * dQ = tau dS K, dK = tau dS^T Q, dV = P^T dO, summed over query-head groups
 * for GQA (0x06.1H).
 *
 * Policies where the pages leave a choice open (each is a stated reading):
 *   - causal alignment is bottom-right, delta = S_k - S_q (M4.4 0x05.1F);
 *   - a row with no visible key (only possible when causal and S_q > S_k)
 *     returns O = 0 and LSE = -inf (M4.4 0x02F: zero payload, no LSE);
 *   - inputs are the already-rounded fp16/bf16 values, widened exactly to
 *     binary32 by the caller; every operation here is binary64.
 *
 * Layout: every tensor is contiguous [B, heads, S, d] (row-major), LSE is
 * [B, H, S_q].  Decode uses S_q = 1 and a per-batch valid key length L_b:
 * keys j >= L_b are padding and never read.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EARG (-1)

/* One query row against a set of visible keys [0, n_vis) of one K/V head:
 * materialise the scaled scores, then m, l, u, O, LSE exactly as defined
 * (M4.3 0x06B and 0x09A).  n_vis == 0 is the all-masked policy.           */
static void exact_row(const float *qrow, const float *kbase, const float *vbase,
                      long long n_vis, int d, double scale,
                      double *scores /* scratch [n_vis] */,
                      double *o /* [d] */, double *lse)
{
    if (n_vis <= 0) {
        for (int t = 0; t < d; ++t) o[t] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (long long j = 0; j < n_vis; ++j) {
        const float *krow = kbase + j * (long long)d;
        double dot = 0.0;
        for (int t = 0; t < d; ++t) dot += (double)qrow[t] * (double)krow[t];
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    double l = 0.0;
    for (int t = 0; t < d; ++t) o[t] = 0.0;
    for (long long j = 0; j < n_vis; ++j) {
        double p = exp(scores[j] - m);
        l += p;
        const float *vrow = vbase + j * (long long)d;
        for (int t = 0; t < d; ++t) o[t] += p * (double)vrow[t];
    }
    for (int t = 0; t < d; ++t) o[t] /= l;
    *lse = m + log(l);
}

/* Number of keys visible to query row i: keys 0 .. n-1 where the visible set
 * is { j : 0 <= j < Sk and (!causal or j <= i + Sk - Sq) }.  Because the
 * causal predicate is monotone in j the visible set is always a prefix.    */
static long long visible_prefix(int i, int Sq, int Sk, int causal)
{
    if (!causal) return Sk;
    long long last = (long long)i + (long long)Sk - (long long)Sq; /* largest visible j */
    if (last < 0) return 0;
    if (last >= Sk) return Sk;
    return last + 1;
}

static int check_heads(int H, int Hkv)
{
    return (H >= 1 && Hkv >= 1 && H % Hkv == 0) ? 0 : -1;
}

/*
 * Exact attention forward on a chosen subset of query rows.
 *   row_ids[r] = (b * H + h) * Sq + i   identifies the query row
 *   o   : [n_rows, d] fp64 output,  lse : [n_rows] fp64 output
 */
int oracle_attn_fwd_rows(const float *q, const float *k, const float *v,
                         int B, int H, int Hkv, int Sq, int Sk, int d,
                         double scale, int causal,
                         const long long *row_ids, long long n_rows,
                         double *o, double *lse)
{
    if (B < 1 || Sq < 1 || Sk < 1 || d < 1 || check_heads(H, Hkv)) return ORACLE_EARG;
    const int g = H / Hkv;
    const long long total_rows = (long long)B * H * Sq;
    for (long long r = 0; r < n_rows; ++r)
        if (row_ids[r] < 0 || row_ids[r] >= total_rows) return ORACLE_EARG;

    int bad = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (!scores) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long long r = 0; r < n_rows; ++r) {
                long long id = row_ids[r];
                int i = (int)(id % Sq);
                long long bh = id / Sq;
                int h = (int)(bh % H);
                int b = (int)(bh / H);
                int kvh = h / g;
                const float *qrow = q + id * (long long)d;
                const float *kbase = k + ((long long)b * Hkv + kvh) * (long long)Sk * d;
                const float *vbase = v + ((long long)b * Hkv + kvh) * (long long)Sk * d;
                exact_row(qrow, kbase, vbase, visible_prefix(i, Sq, Sk, causal), d, scale,
                          scores, o + r * (long long)d, lse + r);
            }
            free(scores);
        }
    }
    return bad ? ORACLE_EARG : ORACLE_OK;
}

/* Exact attention forward on every row: o [B,H,Sq,d], lse [B,H,Sq]. */
int oracle_attn_fwd(const float *q, const float *k, const float *v,
                    int B, int H, int Hkv, int Sq, int Sk, int d,
                    double scale, int causal, double *o, double *lse)
{
    if (B < 1 || H < 1 || Sq < 1) return ORACLE_EARG;
    long long n = (long long)B * H * Sq;
    long long *ids = (long long *)malloc(sizeof(long long) * (size_t)n);
    if (!ids) return ORACLE_EARG;
    for (long long r = 0; r < n; ++r) ids[r] = r;
    int rc = oracle_attn_fwd_rows(q, k, v, B, H, Hkv, Sq, Sk, d, scale, causal, ids, n, o, lse);
    free(ids);
    return rc;
}

/*
 * One-query decode against a padded KV cache:
 *   q [B,Hq,1,d], k/v [B,Hkv,Sk_max,d], seqlens[b] = L_b valid keys.
 * Row (b, h) sees keys 0 .. L_b-1 (padding masked).  Rows are selected by
 * row_ids[r] = b * Hq + h.  o [n_rows, d], lse [n_rows].
 */
int oracle_attn_decode_rows(const float *q, const float *k, const float *v,
                            const int *seqlens, int B, int Hq, int Hkv, int Sk_max, int d,
                            double scale, const long long *row_ids, long long n_rows,
                            double *o, double *lse)
{
    if (B < 1 || Sk_max < 1 || d < 1 || check_heads(Hq, Hkv)) return ORACLE_EARG;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > Sk_max) return ORACLE_EARG;
    for (long long r = 0; r < n_rows; ++r)
        if (row_ids[r] < 0 || row_ids[r] >= (long long)B * Hq) return ORACLE_EARG;
    const int g = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)Sk_max);
        if (!scores) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long r = 0; r < n_rows; ++r) {
                long long id = row_ids[r];
                int h = (int)(id % Hq);
                int b = (int)(id / Hq);
                int kvh = h / g;
                const float *kbase = k + ((long long)b * Hkv + kvh) * (long long)Sk_max * d;
                const float *vbase = v + ((long long)b * Hkv + kvh) * (long long)Sk_max * d;
                exact_row(q + id * (long long)d, kbase, vbase, seqlens[b], d, scale, scores,
                          o + r * (long long)d, lse + r);
            }
            free(scores);
        }
    }
    return bad ? ORACLE_EARG : ORACLE_OK;
}

/*
 * Split-KV chunk states for decode (Flash-Decoding: M4.4 0x01 work-axis
 * ledger; the split-KV tower of "Learning FlashAttention the Hard Way,
 * Part 2", Move 6).  Chunk c of row (b, h) covers keys
 *     [floor(c * L_b / n_split), floor((c + 1) * L_b / n_split))
 * and its state is the canonical summary of M4.3 0x08A, in natural units:
 *     m = max s_j,  l = sum exp(s_j - m),  u = sum exp(s_j - m) v_j.
 * An empty chunk is the identity (m = -inf, l = 0, u = 0) of M4.3 0x08C.
 * Outputs: m, l [B, Hq, n_split]; u [B, Hq, n_split, d]; count the same
 * shape as m (number of keys represented, for the partition check).
 */
int oracle_decode_chunk_states(const float *q, const float *k, const float *v,
                               const int *seqlens, int B, int Hq, int Hkv, int Sk_max, int d,
                               double scale, int n_split,
                               double *m_out, double *l_out, double *u_out, long long *count_out)
{
    if (B < 1 || Sk_max < 1 || d < 1 || n_split < 1 || check_heads(Hq, Hkv)) return ORACLE_EARG;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > Sk_max) return ORACLE_EARG;
    const int g = Hq / Hkv;
    const long long n_states = (long long)B * Hq * n_split;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long s = 0; s < n_states; ++s) {
        int c = (int)(s % n_split);
        long long bh = s / n_split;
        int h = (int)(bh % Hq);
        int b = (int)(bh / Hq);
        int kvh = h / g;
        long long L = seqlens[b];
        long long lo = (long long)c * L / n_split;
        long long hi = (long long)(c + 1) * L / n_split;
        const float *qrow = q + bh * (long long)d;
        const float *kbase = k + ((long long)b * Hkv + kvh) * (long long)Sk_max * d;
        const float *vbase = v + ((long long)b * Hkv + kvh) * (long long)Sk_max * d;
        double *u = u_out + s * (long long)d;
        for (int t = 0; t < d; ++t) u[t] = 0.0;
        count_out[s] = hi - lo;
        if (hi <= lo) {
            m_out[s] = -INFINITY;
            l_out[s] = 0.0;
            continue;
        }
        double m = -INFINITY;
        for (long long j = lo; j < hi; ++j) {
            double dot = 0.0;
            for (int t = 0; t < d; ++t) dot += (double)qrow[t] * (double)kbase[j * d + t];
            double sj = scale * dot;
            if (sj > m) m = sj;
        }
        double l = 0.0;
        for (long long j = lo; j < hi; ++j) {
            double dot = 0.0;
            for (int t = 0; t < d; ++t) dot += (double)qrow[t] * (double)kbase[j * d + t];
            double p = exp(scale * dot - m);
            l += p;
            for (int t = 0; t < d; ++t) u[t] += p * (double)vbase[j * d + t];
        }
        m_out[s] = m;
        l_out[s] = l;
    }
    return ORACLE_OK;
}

/*
 * Exact attention backward, M4.4 "FlashAttention-2 Work Partitioning and the
 * Decode Boundary", 0x06.1A: with S = tau Q K^T (masked before the row
 * normalisation), P = softmax_row(S), O = P V and the incoming gradient dO,
 *
 *     dP    = dO V^T
 *     dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)     (row softmax Jacobian
 *                                                  contracted with dP)
 *     dQ    = tau dS K,   dK = tau dS^T Q,   dV = P^T dO
 *
 * and, for grouped-query heads (0x06.1H), the K/V gradient of a KV head is
 * the sum over the g query heads that read it.  Invisible (masked) entries
 * have P = 0 and contribute nothing; a row with no visible key has
 * dQ = 0 and contributes nothing.
 *
 * The row scalar is computed here from its definition, sum_k P_ik dP_ik,
 * not from the saved-output shortcut dO_i . O_i that the pages derive from
 * it (the tests check that identity against this oracle).
 *
 * Organisation for one (b, kv_head) pair (no tiling, no streaming):
 *   pass 1, one query row at a time (h in the group, i): materialise the
 *           visible scores, P_i, dP_i, the row scalar D_i and dQ_i; keep
 *           LSE_i = m + log l and D_i;
 *   pass 2, one key row at a time: dK_j and dV_j as sums over the query
 *           rows that see key j, with P_ij = exp(S_ij - LSE_i) (the same
 *           softmax written through the row's log-normaliser).
 * The split only gives every output element a single writer.
 */
static void bwd_group(const float *q, const float *k, const float *v, const float *dout,
                      int b, int kvh, int H, int Hkv, int Sq, int Sk, int d, double scale,
                      int causal, double *dq /* [g, Sq, d] */, double *dk /* [Sk, d] */,
                      double *dv /* [Sk, d] */, double *lse_row /* [g * Sq] */,
                      double *D_row /* [g * Sq] */, int *bad)
{
    const int g = H / Hkv;
    const long long n_rows = (long long)g * Sq;
    const float *kb = k + ((long long)b * Hkv + kvh) * (long long)Sk * d;
    const float *vb = v + ((long long)b * Hkv + kvh) * (long long)Sk * d;
    /* query head h = kvh * g + hh of batch b */
#define QROW(hh, i) (q + (((long long)b * H + (long long)kvh * g + (hh)) * Sq + (i)) * (long long)d)
#define DOROW(hh, i) (dout + (((long long)b * H + (long long)kvh * g + (hh)) * Sq + (i)) * (long long)d)

    /* pass 1: per query row */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (!s || !dp) {
#pragma omp atomic write
            *bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long long r = 0; r < n_rows; ++r) {
                const int hh = (int)(r / Sq), i = (int)(r % Sq);
                const float *qi = QROW(hh, i), *doi = DOROW(hh, i);
                double *dqi = dq + r * (long long)d;
                const long long n_vis = visible_prefix(i, Sq, Sk, causal);
                for (int t = 0; t < d; ++t) dqi[t] = 0.0;
                if (n_vis <= 0) {
                    lse_row[r] = -INFINITY;
                    D_row[r] = 0.0;
                    continue;
                }
                double m = -INFINITY;
                for (long long j = 0; j < n_vis; ++j) {
                    double dot = 0.0, dpj = 0.0;
                    for (int t = 0; t < d; ++t) {
                        dot += (double)qi[t] * (double)kb[j * d + t];
                        dpj += (double)doi[t] * (double)vb[j * d + t];
                    }
                    s[j] = scale * dot;
                    dp[j] = dpj;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (long long j = 0; j < n_vis; ++j) l += exp(s[j] - m);
                double Di = 0.0;
                for (long long j = 0; j < n_vis; ++j) {
                    s[j] = exp(s[j] - m) / l; /* s now holds P_ij */
                    Di += s[j] * dp[j];
                }
                for (long long j = 0; j < n_vis; ++j) {
                    const double dsij = s[j] * (dp[j] - Di);
                    for (int t = 0; t < d; ++t) dqi[t] += scale * dsij * (double)kb[j * d + t];
                }
                lse_row[r] = m + log(l);
                D_row[r] = Di;
            }
        }
        free(s);
        free(dp);
    }
    if (*bad) return;

    /* pass 2: per key row */
#pragma omp parallel for schedule(dynamic, 4)
    for (long long j = 0; j < Sk; ++j) {
        double *dkj = dk + j * (long long)d, *dvj = dv + j * (long long)d;
        for (int t = 0; t < d; ++t) dkj[t] = dvj[t] = 0.0;
        for (long long r = 0; r < n_rows; ++r) {
            const int hh = (int)(r / Sq), i = (int)(r % Sq);
            if (j >= visible_prefix(i, Sq, Sk, causal)) continue;
            const float *qi = QROW(hh, i), *doi = DOROW(hh, i);
            double dot = 0.0, dpj = 0.0;
            for (int t = 0; t < d; ++t) {
                dot += (double)qi[t] * (double)kb[j * d + t];
                dpj += (double)doi[t] * (double)vb[j * d + t];
            }
            const double pij = exp(scale * dot - lse_row[r]);
            const double dsij = pij * (dpj - D_row[r]);
            for (int t = 0; t < d; ++t) {
                dkj[t] += scale * dsij * (double)qi[t];
                dvj[t] += pij * (double)doi[t];
            }
        }
    }
#undef QROW
#undef DOROW
}

/*
 * Backward for every head: dq [B,H,Sq,d], dk/dv [B,Hkv,Sk,d], and (if not
 * NULL) the row scalars D [B,H,Sq] and LSE [B,H,Sq].
 */
int oracle_attn_bwd(const float *q, const float *k, const float *v, const float *dout,
                    int B, int H, int Hkv, int Sq, int Sk, int d, double scale, int causal,
                    double *dq, double *dk, double *dv, double *D_out, double *lse_out)
{
    if (B < 1 || Sq < 1 || Sk < 1 || d < 1 || check_heads(H, Hkv)) return ORACLE_EARG;
    const int g = H / Hkv;
    double *lse = (double *)malloc(sizeof(double) * (size_t)g * Sq);
    double *D = (double *)malloc(sizeof(double) * (size_t)g * Sq);
    int bad = (!lse || !D);
    for (int b = 0; b < B && !bad; ++b)
        for (int kvh = 0; kvh < Hkv && !bad; ++kvh) {
            const long long h0 = (long long)b * H + (long long)kvh * g; /* first query head */
            bwd_group(q, k, v, dout, b, kvh, H, Hkv, Sq, Sk, d, scale, causal,
                      dq + h0 * Sq * (long long)d,
                      dk + ((long long)b * Hkv + kvh) * (long long)Sk * d,
                      dv + ((long long)b * Hkv + kvh) * (long long)Sk * d, lse, D, &bad);
            for (long long r = 0; r < (long long)g * Sq; ++r) {
                if (D_out) D_out[h0 * Sq + r] = D[r];
                if (lse_out) lse_out[h0 * Sq + r] = lse[r];
            }
        }
    free(lse);
    free(D);
    return bad ? ORACLE_EARG : ORACLE_OK;
}

/*
 * Backward restricted to chosen KV heads (for sampled checks of large
 * problems): kv_ids[n] = b * Hkv + kv_head.  For each chosen pair it returns
 * dq of its g query heads [n, g, Sq, d] and its dk, dv [n, Sk, d].
 */
int oracle_attn_bwd_kvheads(const float *q, const float *k, const float *v, const float *dout,
                            int B, int H, int Hkv, int Sq, int Sk, int d, double scale,
                            int causal, const long long *kv_ids, long long n,
                            double *dq, double *dk, double *dv)
{
    if (B < 1 || Sq < 1 || Sk < 1 || d < 1 || check_heads(H, Hkv)) return ORACLE_EARG;
    for (long long r = 0; r < n; ++r)
        if (kv_ids[r] < 0 || kv_ids[r] >= (long long)B * Hkv) return ORACLE_EARG;
    const int g = H / Hkv;
    double *lse = (double *)malloc(sizeof(double) * (size_t)g * Sq);
    double *D = (double *)malloc(sizeof(double) * (size_t)g * Sq);
    int bad = (!lse || !D);
    for (long long r = 0; r < n && !bad; ++r) {
        const int b = (int)(kv_ids[r] / Hkv), kvh = (int)(kv_ids[r] % Hkv);
        bwd_group(q, k, v, dout, b, kvh, H, Hkv, Sq, Sk, d, scale, causal,
                  dq + r * (long long)g * Sq * d, dk + r * (long long)Sk * d,
                  dv + r * (long long)Sk * d, lse, D, &bad);
    }
    free(lse);
    free(D);
    return bad ? ORACLE_EARG : ORACLE_OK;
}

/* Number of threads the oracle's parallel regions use (for reporting). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
