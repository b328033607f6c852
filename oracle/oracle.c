/*
 * oracle.c -- plain, slow fp64 CPU oracle for pi-Attention and ECP attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes is the plain definition of the method, written out once per
 * query row with an explicit neighbour list:
 *
 *   pi-Attention ("pi-Attention: Periodic Sparse Transformers for Efficient
 *   Long-Context Modeling", section 2 "Methodology"):
 *     - 2.1 ring-local attention: token i attends to a local band of width k.
 *       Causal reading: keys j with max(0, i-k) <= j <= i.
 *     - 2.2 pi-skip attention: periodic keys at stride pi, restricted to
 *       earlier positions for causality: j = i - m*pi, m = 1..S, j >= 0.
 *       A skip key that already lies in the band (m*pi <= k) is not added a
 *       second time: the union holds each key once.
 *     - 2.3 adaptive fusion: one softmax over the union of local and skip
 *       neighbours, with the per-token, per-head gate alpha entering as a
 *       log-prior: +ln(alpha) on local logits, +ln(1-alpha) on skip logits.
 *   Bidirectional pi-Attention (same page, 2.1 and 2.2 in their general,
 *   non-causal form): the band is i-k .. i+k and the skip keys are i - m*pi and
 *   i + m*pi, each clipped to [0, N); the priors are those of the causal form.
 *   ECP ("Efficient Context Propagating Perceiver Architectures for
 *   Auto-Regressive Language Modeling", section 2, paired-segment PAR block):
 *     queries of half-segment s = floor(i/c) attend causally to keys of
 *     half-segments s-1 and s: max(0, (s-1)*c) <= j <= i.  No prior.
 *   GQA ("Long-context modelling with a GSS-Transformer hybrid", attention
 *   branch): query head h reads key/value head floor(h / (H/Hkv)).
 *
 *   Logit z_ij = (q_i . k_j) / sqrt(d) + prior_ij;  lse_i = ln sum_j exp(z_ij);
 *   p_ij = exp(z_ij - lse_i);  out_i = sum_j p_ij v_j.
 *   A row whose logits are all -inf (alpha = 0 and no skip key) has out = 0
 *   and lse = -inf.
 *
 * Backward (the chain rule applied to the definition above), with loss
 * gradient dout:
 *   D_i = dout_i . out_i ;  dz_ij = p_ij (dout_i . v_j - D_i)
 *   dq_i = sum_j dz_ij k_j / sqrt(d);  dk_j = sum_{h in group, i} dz_ij q_i / sqrt(d)
 *   dv_j = sum_{h in group, i} p_ij dout_i
 *   dalpha_i = sum_{j local} dz_ij / alpha_i - sum_{j skip} dz_ij / (1 - alpha_i),
 *   taken as 0 where alpha_i is 0 or 1 (there one prior is -inf: a saturated gate)
 *
 * Gate (same page, 2.3: a light neural network (MLP) producing alpha per token and
 * per head from the input content).  Reading: one hidden layer of F units with a
 * ReLU on the head's query, the output through a logistic function:
 *   hid_f = max(0, sum_t W1[h][f][t] q_t + b1[h][f]),  f = 0 .. F-1,
 *   alpha_{b,h,i} = 1 / (1 + exp(-(sum_f w2[h][f] hid_f + b2[h]))).
 *
 * Inputs may be fp64, fp32 or raw bf16 bits; bf16 is widened exactly.  All
 * arithmetic is fp64.  Parallel over query rows with OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DT_F64 0
#define DT_F32 1
#define DT_BF16 2

#define MODE_PI 0
#define MODE_ECP 1
#define MODE_PI_BIDIR 2

static double ld(const void *p, int dt, size_t idx) {
    if (dt == DT_F64) return ((const double *)p)[idx];
    if (dt == DT_F32) return (double)((const float *)p)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Upper bound on the neighbour count of one query row. */
static long max_neighbours(long N, int mode, long k_local, int S) {
    long n = (mode == MODE_PI) ? (k_local + 1 + S)
             : (mode == MODE_PI_BIDIR) ? (2 * k_local + 1 + 2 * (long)S) : (2 * k_local + 1);
    return n < N + 2 * (long)S + 1 ? n : N + 2 * (long)S + 1;
}

/* Neighbour list of query i (sequence length N): keys in idx[], tag 0 = local, 1 = skip. */
static long neighbours(long i, long N, int mode, long k_local, long period, int S,
                       long *idx, int *tag) {
    long n = 0, lo, hi, j;
    if (mode == MODE_PI_BIDIR) {
        lo = i - k_local;
        if (lo < 0) lo = 0;
        hi = i + k_local;
        if (hi > N - 1) hi = N - 1;
        for (j = lo; j <= hi; ++j) { idx[n] = j; tag[n] = 0; ++n; }
        for (int m = 1; m <= S; ++m) {
            long off = (long)m * period;
            if (off <= k_local) continue;    /* inside the band already */
            if (i - off >= 0) { idx[n] = i - off; tag[n] = 1; ++n; }
            if (i + off < N) { idx[n] = i + off; tag[n] = 1; ++n; }
        }
    } else if (mode == MODE_PI) {
        lo = i - k_local;
        if (lo < 0) lo = 0;
        for (j = lo; j <= i; ++j) { idx[n] = j; tag[n] = 0; ++n; }
        for (int m = 1; m <= S; ++m) {
            long back = (long)m * period;
            if (back <= k_local) continue;   /* inside the band already */
            j = i - back;
            if (j < 0) break;
            idx[n] = j; tag[n] = 1; ++n;
        }
    } else {
        long s = i / k_local;
        lo = (s - 1) * k_local;
        if (lo < 0) lo = 0;
        for (j = lo; j <= i; ++j) { idx[n] = j; tag[n] = 0; ++n; }
    }
    return n;
}

/* Per-row neighbour count and sum of key indices (identical for every b, h). */
void oracle_counts(long N, int mode, long k_local, long period, int S,
                   long long *count, long long *idx_sum) {
    long cap = max_neighbours(N, mode, k_local, S);
#pragma omp parallel
    {
        long *idx = (long *)malloc(sizeof(long) * cap);
        int *tag = (int *)malloc(sizeof(int) * cap);
#pragma omp for schedule(static)
        for (long i = 0; i < N; ++i) {
            long n = neighbours(i, N, mode, k_local, period, S, idx, tag);
            long long s = 0;
            for (long t = 0; t < n; ++t) s += idx[t];
            count[i] = n;
            idx_sum[i] = s;
        }
        free(idx);
        free(tag);
    }
}

/* Logits, softmax and output of one row (inputs already widened to fp64).
   z and p have room for n entries.  Writes out_row[d] and returns lse. */
static double one_row(const double *q, const double *k, const double *v, const float *alpha,
                      long H, long Hkv, long N, long d, int mode, long b, long h, long i, long n,
                      const long *idx, const int *tag, double *z, double *p, double *out_row) {
    long g = h / (H / Hkv);
    const double *qrow = q + (((size_t)b * H + h) * N + i) * d;
    double a = alpha ? (double)alpha[((size_t)b * H + h) * N + i] : 1.0;
    double scale = 1.0 / sqrt((double)d);
    double M = -INFINITY;
    for (long t = 0; t < n; ++t) {
        const double *krow = k + (((size_t)b * Hkv + g) * N + idx[t]) * d;
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += qrow[c] * krow[c];
        double prior = 0.0;
        if (mode != MODE_ECP) prior = (tag[t] == 0) ? log(a) : log1p(-a);
        z[t] = dot * scale + prior;
        if (z[t] > M) M = z[t];
    }
    for (long c = 0; c < d; ++c) out_row[c] = 0.0;
    if (M == -INFINITY) {
        for (long t = 0; t < n; ++t) p[t] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (long t = 0; t < n; ++t) l += exp(z[t] - M);
    for (long t = 0; t < n; ++t) p[t] = exp(z[t] - M) / l;
    for (long t = 0; t < n; ++t) {
        const double *vrow = v + (((size_t)b * Hkv + g) * N + idx[t]) * d;
        for (long c = 0; c < d; ++c) out_row[c] += p[t] * vrow[c];
    }
    return M + log(l);
}

/* Widen an input tensor of n elements to fp64 (exact for fp32 and bf16). */
static double *widen(const void *x, int dt, size_t n) {
    double *w = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (!w) return NULL;
#pragma omp parallel for schedule(static)
    for (long e = 0; e < (long)n; ++e) w[e] = ld(x, dt, (size_t)e);
    return w;
}

/*
 * Forward over query positions [i_begin, i_end) of every (b, h).
 * out: [B, H, i_end - i_begin, d] fp64; lse: [B, H, i_end - i_begin] fp64.
 * P (optional, may be NULL, requires i_begin = 0 and i_end = N): dense
 * [B, H, N, N] probabilities, zero outside the neighbour set.
 * Returns 0 on success, -1 on bad arguments.
 */
int oracle_fwd(const void *q, const void *k, const void *v, int dt, const float *alpha,
               long B, long H, long Hkv, long N, long d, long k_local, long period, int S,
               int mode, long i_begin, long i_end, double *out, double *lse, double *P) {
    if (B <= 0 || H <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || H % Hkv != 0) return -1;
    if (mode == MODE_ECP && k_local <= 0) return -1;
    if (mode != MODE_ECP && S > 0 && period <= 0) return -1;
    if (i_begin < 0 || i_end > N || i_begin > i_end) return -1;
    if (P && (i_begin != 0 || i_end != N)) return -1;
    long rows = i_end - i_begin;
    long cap = max_neighbours(N, mode, k_local, S);
    long total = B * H * rows;
    double *qd = widen(q, dt, (size_t)B * H * N * d);
    double *kd = widen(k, dt, (size_t)B * Hkv * N * d);
    double *vd = widen(v, dt, (size_t)B * Hkv * N * d);
    if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -2; }
#pragma omp parallel
    {
        long *idx = (long *)malloc(sizeof(long) * cap);
        int *tag = (int *)malloc(sizeof(int) * cap);
        double *z = (double *)malloc(sizeof(double) * cap);
        double *p = (double *)malloc(sizeof(double) * cap);
#pragma omp for schedule(dynamic, 64)
        for (long r = 0; r < total; ++r) {
            long b = r / (H * rows);
            long h = (r / rows) % H;
            long i = i_begin + r % rows;
            long n = neighbours(i, N, mode, k_local, period, S, idx, tag);
            double *orow = out + (size_t)r * d;
            lse[r] = one_row(qd, kd, vd, alpha, H, Hkv, N, d, mode, b, h, i, n, idx, tag, z, p,
                             orow);
            if (P) {
                double *prow = P + (((size_t)b * H + h) * N + i) * N;
                for (long j = 0; j < N; ++j) prow[j] = 0.0;
                for (long t = 0; t < n; ++t) prow[idx[t]] = p[t];
            }
        }
        free(idx); free(tag); free(z); free(p);
    }
    free(qd); free(kd); free(vd);
    return 0;
}

/*
 * Backward.  dout has the input dtype.  Writes dq [B,H,N,d], dk and dv
 * [B,Hkv,N,d], dalpha [B,H,N] (all fp64; dalpha may be NULL).
 * Parallel over (b, kv head) so that dk/dv accumulation has one writer.
 */
int oracle_bwd(const void *q, const void *k, const void *v, int dt, const float *alpha,
               const void *dout, long B, long H, long Hkv, long N, long d, long k_local,
               long period, int S, int mode, double *dq, double *dk, double *dv,
               double *dalpha) {
    if (B <= 0 || H <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || H % Hkv != 0) return -1;
    if (mode == MODE_ECP && k_local <= 0) return -1;
    if (mode != MODE_ECP && S > 0 && period <= 0) return -1;
    long G = H / Hkv;
    long cap = max_neighbours(N, mode, k_local, S);
    double scale = 1.0 / sqrt((double)d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * N * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * N * d);
    double *qd = widen(q, dt, (size_t)B * H * N * d);
    double *kd = widen(k, dt, (size_t)B * Hkv * N * d);
    double *vd = widen(v, dt, (size_t)B * Hkv * N * d);
    double *gd = widen(dout, dt, (size_t)B * H * N * d);
    if (!qd || !kd || !vd || !gd) { free(qd); free(kd); free(vd); free(gd); return -2; }
#pragma omp parallel
    {
        long *idx = (long *)malloc(sizeof(long) * cap);
        int *tag = (int *)malloc(sizeof(int) * cap);
        double *z = (double *)malloc(sizeof(double) * cap);
        double *p = (double *)malloc(sizeof(double) * cap);
        double *orow = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 1)
        for (long bg = 0; bg < B * Hkv; ++bg) {
            long b = bg / Hkv, g = bg % Hkv;
            double *dkg = dk + (size_t)bg * N * d;
            double *dvg = dv + (size_t)bg * N * d;
            const double *kg = kd + (size_t)bg * N * d;
            const double *vg = vd + (size_t)bg * N * d;
            for (long h = g * G; h < (g + 1) * G; ++h) {
                for (long i = 0; i < N; ++i) {
                    long n = neighbours(i, N, mode, k_local, period, S, idx, tag);
                    one_row(qd, kd, vd, alpha, H, Hkv, N, d, mode, b, h, i, n, idx, tag, z, p, orow);
                    size_t qoff = (((size_t)b * H + h) * N + i) * d;
                    const double *qrow = qd + qoff;
                    const double *grow = gd + qoff;
                    double D = 0.0;
                    for (long c = 0; c < d; ++c) D += grow[c] * orow[c];
                    double *dqrow = dq + qoff;
                    for (long c = 0; c < d; ++c) dqrow[c] = 0.0;
                    double sum_local = 0.0, sum_skip = 0.0;
                    for (long t = 0; t < n; ++t) {
                        size_t koff = (size_t)idx[t] * d;
                        double dp = 0.0;
                        for (long c = 0; c < d; ++c) dp += grow[c] * vg[koff + c];
                        double dz = p[t] * (dp - D);
                        if (tag[t] == 0) sum_local += dz; else sum_skip += dz;
                        for (long c = 0; c < d; ++c) {
                            dqrow[c] += dz * kg[koff + c] * scale;
                            dkg[koff + c] += dz * qrow[c] * scale;
                            dvg[koff + c] += p[t] * grow[c];
                        }
                    }
                    if (dalpha) {
                        /* At alpha = 0 or 1 one prior is -inf and its weights are exactly 0; the
                           derivative there is taken as 0 (a saturated gate passes no gradient). */
                        double g_a = 0.0;
                        double a = alpha ? (double)alpha[((size_t)b * H + h) * N + i] : 1.0;
                        if (mode != MODE_ECP && a > 0.0 && a < 1.0) {
                            g_a = sum_local / a - sum_skip / (1.0 - a);
                            if (sum_skip == 0.0) g_a = sum_local / a;
                        }
                        dalpha[((size_t)b * H + h) * N + i] = g_a;
                    }
                }
            }
        }
        free(idx); free(tag); free(z); free(p); free(orow);
    }
    free(qd); free(kd); free(vd); free(gd);
    return 0;
}

/*
 * Gate: alpha [B, H, N] fp64 from q [B, H, N, d] (any input dtype) through the MLP above:
 * W1 [H, F, d], b1 [H, F], w2 [H, F], b2 [H] (fp64).
 */
void oracle_gate(const void *q, int dt, const double *w1, const double *b1, const double *w2,
                 const double *b2, long B, long H, long N, long d, long F, double *alpha) {
#pragma omp parallel for schedule(static)
    for (long row = 0; row < B * H * N; ++row) {
        const long h = (row / N) % H;
        double z = b2[h];
        for (long f = 0; f < F; ++f) {
            double pre = b1[h * F + f];
            for (long t = 0; t < d; ++t) pre += ld(q, dt, (size_t)row * d + t) * w1[(h * F + f) * d + t];
            if (pre > 0.0) z += w2[h * F + f] * pre;
        }
        alpha[row] = 1.0 / (1.0 + exp(-z));
    }
}
