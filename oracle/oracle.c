/*
 * Exact softmax attention, forward and backward: the plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the test suite, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only in the seeded inputs the
 * tests hand to both.
 *
 * What it computes is the plain definition, written out without blocking,
 * fusion or reordering:
 *
 *   s_ij = scale * <q_i, k_j>                       for every allowed key j
 *   P_ij = exp(s_ij - mu) / Z,  Z = sum_j exp(s_ij - mu) [+ exp(sink - mu)]
 *   O_i  = sum_j P_ij v_j,      LSE_i = mu + ln Z
 *
 * with a two-pass safe softmax (row max first, then exponentials and sum), as
 * the flash-attention-tutorial README derives it ("Flash Attention Tutorial",
 * GitHub search results page, section 2 "Safe Softmax" and section 1
 * "Standard Self-Attention").  The backward is the chain rule of that
 * definition ("Flash Attention Tutorial", section 6 "Key derivations"), with
 * the softmax scale kept in dQ and dK:
 *
 *   D_i   = <dO_i, O_i>
 *   dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i)
 *   dV_j  = sum_i P_ij dO_i
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 *   dsink = - sum_i exp(sink - LSE_i) D_i
 *
 * Masks (vllm-project/flash-attention README, GitHub search results page,
 * flash_attn_func and flash_attn_with_kvcache docstrings; fa4-jax PyPI page,
 * "Varlen semantics"): with off = s_kv - s_q of the sequence, key j is
 * allowed for query i iff
 *   0 <= j < s_kv,
 *   causal      => j <= i + off              (bottom-right aligned),
 *   left  >= 0  => j >= i + off - left,
 *   right >= 0  => j <= i + off + right      (the window is inclusive).
 * A causal call with a window takes the intersection of the two masks.
 *
 * Grouped-query heads: query head h reads key/value head h / (h_q / h_kv)
 * (vllm-project/flash-attention README, flash_attn_func docstring, the
 * 6-query-head / 2-key-head example).
 *
 * Sinks: one logit per query head that joins every row's softmax
 * denominator and carries no value (dew-flash-attn PyPI page, the sinks
 * paragraph).  The returned LSE includes the sink; lse_nosink is the
 * logsumexp over the keys alone.
 *
 * Packed batches: with cu_q / cu_k given, sequence b owns rows
 * cu_q[b] .. cu_q[b+1]-1 of q (and cu_k[b] .. of k, v), indices are local to
 * the sequence and no sequence sees another (dew-flash-attn PyPI page,
 * "Packed sequences"; fa4-jax PyPI page, "Varlen semantics").  The LSE of a
 * packed call is laid out [h_q, T_q]; a dense one is [B, h_q, s_q].
 *
 * An empty row (no allowed key) has O = 0 and LSE = -inf, or LSE = sink when
 * the head has a sink (vllm-project/flash-attention README: "If the row of
 * the mask is all zero, the output will be zero").
 *
 * Layouts: q, o, dq, dout are [B, s_q, h_q, d] (dense) or [T_q, h_q, d]
 * (packed); k, v, dk, dv are [B, s_kv, h_kv, d] or [T_k, h_kv, d].  All
 * floating-point buffers are fp64; the caller allocates every buffer.
 *
 * Parallelism: OpenMP over independent (sequence, head) units only; every
 * sum inside a unit is a plain sequential fp64 loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, s_q, s_kv, h_q, h_kv, d;
    double scale;
    int causal, left, right;
    const double *sinks;   /* [h_q] or NULL */
    const int32_t *cu_q;   /* [B+1] or NULL (dense) */
    const int32_t *cu_k;   /* [B+1] or NULL (dense) */
} problem;

/* Rows of sequence b: first global row and count, for q and for k. */
static void seq_rows(const problem *p, int b, long *q0, long *nq, long *k0, long *nk) {
    if (p->cu_q) {
        *q0 = p->cu_q[b];
        *nq = (long)p->cu_q[b + 1] - p->cu_q[b];
        *k0 = p->cu_k[b];
        *nk = (long)p->cu_k[b + 1] - p->cu_k[b];
    } else {
        *q0 = (long)b * p->s_q;
        *nq = p->s_q;
        *k0 = (long)b * p->s_kv;
        *nk = p->s_kv;
    }
}

/* The mask predicate, written exactly as the pages state it. */
static int allowed(const problem *p, long i, long j, long nq, long nk) {
    long off = nk - nq;
    if (j < 0 || j >= nk) return 0;
    if (p->causal && j > i + off) return 0;
    if (p->left >= 0 && j < i + off - p->left) return 0;
    if (p->right >= 0 && j > i + off + p->right) return 0;
    return 1;
}

static double dot(const double *a, const double *b, int d) {
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += a[t] * b[t];
    return s;
}

/* LSE index of (sequence b, local row i, head h). */
static long lse_index(const problem *p, int b, long q0, long i, int h) {
    if (p->cu_q) {
        long T = p->cu_q[p->B];
        return (long)h * T + q0 + i;
    }
    return ((long)b * p->h_q + h) * p->s_q + i;
}

/*
 * One query row: fills srow[j] = s_ij for allowed j, and returns mu, Z
 * (with the sink when present), and the sink-less logsumexp.
 */
static void row_stats(const problem *p, const double *qi, const double *kbase, long nq, long nk,
                      long i, int hk, int h, double *srow, char *ok, double *mu_out, double *z_out,
                      double *lse_nosink_out) {
    const int d = p->d;
    double mu = -INFINITY;
    for (long j = 0; j < nk; ++j) {
        ok[j] = (char)allowed(p, i, j, nq, nk);
        if (!ok[j]) continue;
        const double *kj = kbase + (j * p->h_kv + hk) * (long)d;
        srow[j] = p->scale * dot(qi, kj, d);
        if (srow[j] > mu) mu = srow[j];
    }
    /* sink-less logsumexp, two passes */
    double z0 = 0.0;
    if (mu > -INFINITY)
        for (long j = 0; j < nk; ++j)
            if (ok[j]) z0 += exp(srow[j] - mu);
    *lse_nosink_out = (z0 > 0.0) ? mu + log(z0) : -INFINITY;

    double mus = mu;
    if (p->sinks && p->sinks[h] > mus) mus = p->sinks[h];
    double z = 0.0;
    if (mus > -INFINITY) {
        for (long j = 0; j < nk; ++j)
            if (ok[j]) z += exp(srow[j] - mus);
        if (p->sinks) z += exp(p->sinks[h] - mus);
    }
    *mu_out = mus;
    *z_out = z;
}

/* O_i and LSE_i for one row; returns them through oi / lse. */
static void row_forward(const problem *p, const double *qi, const double *kbase, const double *vbase,
                        long nq, long nk, long i, int hk, int h, double *srow, char *ok, double *oi,
                        double *lse, double *lse_nosink) {
    const int d = p->d;
    double mu, z;
    row_stats(p, qi, kbase, nq, nk, i, hk, h, srow, ok, &mu, &z, lse_nosink);
    for (int t = 0; t < d; ++t) oi[t] = 0.0;
    if (z > 0.0) {
        for (long j = 0; j < nk; ++j) {
            if (!ok[j]) continue;
            double pij = exp(srow[j] - mu) / z;
            const double *vj = vbase + (j * p->h_kv + hk) * (long)d;
            for (int t = 0; t < d; ++t) oi[t] += pij * vj[t];
        }
        *lse = mu + log(z);
    } else {
        *lse = -INFINITY;
    }
}

static int check(const problem *p) {
    if (p->B < 0 || p->h_q <= 0 || p->h_kv <= 0 || p->d <= 0) return 1;
    if (p->h_q % p->h_kv != 0) return 2;
    if ((p->cu_q == NULL) != (p->cu_k == NULL)) return 3;
    if (!p->cu_q && (p->s_q < 0 || p->s_kv < 0)) return 4;
    return 0;
}

static long max_kv_len(const problem *p) {
    long m = 0;
    for (int b = 0; b < p->B; ++b) {
        long q0, nq, k0, nk;
        seq_rows(p, b, &q0, &nq, &k0, &nk);
        if (nk > m) m = nk;
    }
    return m;
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward.  o: same layout as q.  lse, lse_nosink: [B, h_q, s_q] or [h_q, T_q]
 * (lse_nosink may be NULL).  Returns 0 on success, a positive code on bad
 * arguments, -1 when scratch memory could not be had.
 */
int oracle_fwd(int B, int s_q, int s_kv, int h_q, int h_kv, int d, double scale, int causal, int left,
               int right, const double *sinks, const int32_t *cu_q, const int32_t *cu_k, const double *q,
               const double *k, const double *v, double *o, double *lse, double *lse_nosink) {
    problem p = {B, s_q, s_kv, h_q, h_kv, d, scale, causal, left, right, sinks, cu_q, cu_k};
    int rc = check(&p);
    if (rc) return rc;
    const int G = h_q / h_kv;
    const long maxk = max_kv_len(&p);
    const long units = (long)B * h_q;
    int failed = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(maxk + 1));
        char *ok = (char *)malloc((size_t)(maxk + 1));
        if (!srow || !ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < units; ++u) {
            if (!srow || !ok) continue;
            int b = (int)(u / h_q), h = (int)(u % h_q), hk = h / G;
            long q0, nq, k0, nk;
            seq_rows(&p, b, &q0, &nq, &k0, &nk);
            const double *kbase = k + k0 * (long)h_kv * d;
            const double *vbase = v + k0 * (long)h_kv * d;
            for (long i = 0; i < nq; ++i) {
                const double *qi = q + ((q0 + i) * h_q + h) * (long)d;
                double *oi = o + ((q0 + i) * h_q + h) * (long)d;
                double l, l0;
                row_forward(&p, qi, kbase, vbase, nq, nk, i, hk, h, srow, ok, oi, &l, &l0);
                long li = lse_index(&p, b, q0, i, h);
                lse[li] = l;
                if (lse_nosink) lse_nosink[li] = l0;
            }
        }
        free(srow);
        free(ok);
    }
    return failed ? -1 : 0;
}

/*
 * Backward of L = sum(O * dout).  Recomputes O and LSE in fp64 itself.
 * dq: layout of q; dk, dv: layout of k; dsinks: [h_q] or NULL (required when
 * sinks is given).  Every output is overwritten.
 */
int oracle_bwd(int B, int s_q, int s_kv, int h_q, int h_kv, int d, double scale, int causal, int left,
               int right, const double *sinks, const int32_t *cu_q, const int32_t *cu_k, const double *q,
               const double *k, const double *v, const double *dout, double *dq, double *dk, double *dv,
               double *dsinks) {
    problem p = {B, s_q, s_kv, h_q, h_kv, d, scale, causal, left, right, sinks, cu_q, cu_k};
    int rc = check(&p);
    if (rc) return rc;
    if (sinks && !dsinks) return 5;
    const int G = h_q / h_kv;
    const long maxk = max_kv_len(&p);
    const long units = (long)B * h_kv; /* a unit owns dK, dV of one kv head and dQ of its G heads */
    long totq = cu_q ? (long)cu_q[B] : (long)B * s_q;
    long totk = cu_k ? (long)cu_k[B] : (long)B * s_kv;
    memset(dq, 0, sizeof(double) * (size_t)(totq * h_q * d));
    memset(dk, 0, sizeof(double) * (size_t)(totk * h_kv * d));
    memset(dv, 0, sizeof(double) * (size_t)(totk * h_kv * d));
    /* per-unit partial sink gradients, summed serially at the end */
    double *dsink_part = (double *)calloc((size_t)(units * G + 1), sizeof(double));
    if (!dsink_part) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)(maxk + 1));
        char *ok = (char *)malloc((size_t)(maxk + 1));
        double *oi = (double *)malloc(sizeof(double) * (size_t)d);
        if (!srow || !ok || !oi) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < units; ++u) {
            if (!srow || !ok || !oi) continue;
            int b = (int)(u / h_kv), hk = (int)(u % h_kv);
            long q0, nq, k0, nk;
            seq_rows(&p, b, &q0, &nq, &k0, &nk);
            const double *kbase = k + k0 * (long)h_kv * d;
            const double *vbase = v + k0 * (long)h_kv * d;
            for (int g = 0; g < G; ++g) {
                int h = hk * G + g;
                for (long i = 0; i < nq; ++i) {
                    const double *qi = q + ((q0 + i) * h_q + h) * (long)d;
                    const double *doi = dout + ((q0 + i) * h_q + h) * (long)d;
                    double *dqi = dq + ((q0 + i) * h_q + h) * (long)d;
                    double lse, l0;
                    row_forward(&p, qi, kbase, vbase, nq, nk, i, hk, h, srow, ok, oi, &lse, &l0);
                    double Di = dot(doi, oi, d);
                    if (sinks && lse > -INFINITY) dsink_part[u * G + g] -= exp(sinks[h] - lse) * Di;
                    if (!(lse > -INFINITY)) continue; /* an empty row has no gradient */
                    for (long j = 0; j < nk; ++j) {
                        if (!ok[j]) continue;
                        const double *kj = kbase + (j * h_kv + hk) * (long)d;
                        const double *vj = vbase + (j * h_kv + hk) * (long)d;
                        double *dkj = dk + ((k0 + j) * h_kv + hk) * (long)d;
                        double *dvj = dv + ((k0 + j) * h_kv + hk) * (long)d;
                        double pij = exp(srow[j] - lse);
                        double dpij = dot(doi, vj, d);
                        double dsij = pij * (dpij - Di);
                        for (int t = 0; t < d; ++t) {
                            dvj[t] += pij * doi[t];
                            dqi[t] += scale * dsij * kj[t];
                            dkj[t] += scale * dsij * qi[t];
                        }
                    }
                }
            }
        }
        free(srow);
        free(ok);
        free(oi);
    }
    if (dsinks) {
        for (int h = 0; h < h_q; ++h) dsinks[h] = 0.0;
        for (long u = 0; u < units; ++u) {
            int hk = (int)(u % h_kv);
            for (int g = 0; g < G; ++g) dsinks[hk * G + g] += dsink_part[u * G + g];
        }
    }
    free(dsink_part);
    return failed ? -1 : 0;
}
