/*
 * attn_ref.c -- fp64 CPU oracle for the FlashAttention-2 forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written reference
 * that the CUDA path is checked against.  Only the test suite, the smoke check
 * in __graft_entry__.py and the CPU-baseline / reference legs of bench.py may
 * load it.  It shares no code, header, table or helper with the CUDA library,
 * and nothing in the library calls it.
 *
 * What it computes (for every batch*head slice and every query row i):
 *
 *   J      = { j < N : not causal, or j <= i }              (causal mask j > i)
 *   x_j    = s * sum_d Q[i,d] * K[j,d]          for j in J  (scaled scores)
 *   m      = max_{j in J} x_j
 *   l      = sum_{j in J} exp(x_j - m)
 *   O[i,:] = sum_{j in J} exp(x_j - m) * V[j,:] / l         (softmax(S) V)
 *   L[i]   = m + log(l)                                     (natural-log LSE)
 *
 * Sources: "A09 - Advanced Triton & FlashAttention", section 2 (First
 * Principles: S = QK^T/sqrt(d), P = softmax(S), O = PV); "Building a
 * Verifiable FlashAttention Forward from PyTorch to Triton", Part 1 (explicit
 * attention, causal mask triu(1) = keys strictly after the query);
 * "FlashAttention 2 from PyTorch to Triton", What I am building (L = m + log l,
 * natural log, equal to the log-sum-exp of the scaled scores).
 *
 * The scale s is the caller's value.  The pages hard-code 1/sqrt(d); the
 * library takes it as an argument, and the Python wrapper passes the same
 * float32 value widened to double.
 *
 * Inputs may be bf16 or fp16 bit patterns (decoded exactly to double from the
 * IEEE/bfloat16 format definitions) or float64.  Outputs are float64 and are
 * NOT rounded to the input dtype: output rounding counts against tolerance.
 *
 * attn_ref_forward_qkv() is the same definition for Nq queries against Nkv
 * keys (cross attention, decode).  Its causal mask is aligned bottom-right:
 * query i sees keys j <= i + (Nkv - Nq), so the last query sees every key --
 * the alignment under which decoding the last Nq positions of a sequence
 * gives the last Nq rows of its square causal attention; it equals the
 * top-left mask when Nq = Nkv ("How to profile and optimise kernels", causal
 * alignment).  A query that sees no key (possible when Nq > Nkv) gets O = 0
 * and LSE = -inf, the empty sum's value.
 *
 * attn_ref_forward_band() generalises the mask to a band (sliding window):
 * with i' = i + (Nkv - Nq), query i sees keys j in [i' - left, i' + right]
 * (a negative bound means unbounded on that side), so causal is the band
 * (unbounded, 0) and no mask is (unbounded, unbounded); a row whose band holds
 * no key gets O = 0 and LSE = -inf.
 *
 * attn_ref_backward_band() gives the gradients of that attention for an
 * upstream gradient dO (the same band mask; see its comment).
 *
 * Besides the explicit definition, attn_ref_tiled() runs the tiled online-
 * softmax recurrence in fp64, step by step in the order the pages give it, so
 * the tests can show that the recurrence equals the definition on small
 * brute-force cases.  It is never used as the parity reference.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_F64 = 2 };

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double fp16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double load_elem(const void *p, int dtype, size_t idx)
{
    if (dtype == ORC_BF16)
        return bf16_bits_to_double(((const uint16_t *)p)[idx]);
    if (dtype == ORC_FP16)
        return fp16_bits_to_double(((const uint16_t *)p)[idx]);
    return ((const double *)p)[idx];
}

/* Widen one [N, D] slice to double. */
static void load_slice(const void *p, int dtype, size_t base, long N, long D, double *dst)
{
    size_t n = (size_t)N * (size_t)D;
    for (size_t t = 0; t < n; ++t)
        dst[t] = load_elem(p, dtype, base + t);
}

int attn_ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Decode n bf16 (dtype 0) or fp16 (dtype 1) bit patterns; lets the tests pin
 * the decoder against an independent library conversion. */
void attn_ref_decode(const uint16_t *bits, int dtype, long n, double *out)
{
    for (long t = 0; t < n; ++t)
        out[t] = (dtype == ORC_BF16) ? bf16_bits_to_double(bits[t]) : fp16_bits_to_double(bits[t]);
}

/*
 * One query row, straight from the definition above, over the visible keys
 * 0 .. nvis-1.  q is the query row, Kh and Vh the key and value slices of its
 * head, x a scratch of at least nvis.  With no visible key, O = 0 and
 * LSE = -inf.
 */
static void ref_row_vis(const double *q, const double *Kh, const double *Vh, long nvis, long D, double s,
                        double *x, double *o, double *lse)
{
    if (nvis <= 0) {
        for (long d = 0; d < D; ++d)
            o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (long j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (long d = 0; d < D; ++d)
            dot += q[d] * Kh[j * D + d];
        x[j] = s * dot;
        if (x[j] > m)
            m = x[j];
    }
    double l = 0.0;
    for (long d = 0; d < D; ++d)
        o[d] = 0.0;
    for (long j = 0; j < nvis; ++j) {
        double w = exp(x[j] - m);
        l += w;
        for (long d = 0; d < D; ++d)
            o[d] += w * Vh[j * D + d];
    }
    for (long d = 0; d < D; ++d)
        o[d] /= l;
    *lse = m + log(l);
}

/* Row i of square attention: keys 0..i when causal, all N keys otherwise. */
static void ref_row(const double *q, const double *Kh, const double *Vh, long N, long D, long i,
                    int causal, double s, double *x, double *o, double *lse)
{
    ref_row_vis(q, Kh, Vh, causal ? i + 1 : N, D, s, x, o, lse);
}

/*
 * Full forward over contiguous [BH, N, D] inputs.  O is [BH, N, D] float64,
 * LSE is [BH, N] float64.  Returns 0, or -1 if a scratch allocation failed.
 */
int attn_ref_forward(const void *Q, const void *K, const void *V, int dtype,
                     long BH, long N, long D, int causal, double s,
                     double *O, double *LSE)
{
    size_t slice = (size_t)N * (size_t)D;
    double *Kh = (double *)malloc(slice * sizeof(double));
    double *Vh = (double *)malloc(slice * sizeof(double));
    double *Qh = (double *)malloc(slice * sizeof(double));
    if (!Kh || !Vh || !Qh) {
        free(Kh); free(Vh); free(Qh);
        return -1;
    }
    int failed = 0;
    for (long bh = 0; bh < BH; ++bh) {
        size_t base = (size_t)bh * slice;
        load_slice(Q, dtype, base, N, D, Qh);
        load_slice(K, dtype, base, N, D, Kh);
        load_slice(V, dtype, base, N, D, Vh);
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)N * sizeof(double));
            if (!x) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long i = 0; i < N; ++i)
                    ref_row(Qh + i * D, Kh, Vh, N, D, i, causal, s, x,
                            O + base + (size_t)i * D, LSE + (size_t)bh * N + i);
            }
            free(x);
        }
    }
    free(Kh); free(Vh); free(Qh);
    return failed ? -1 : 0;
}

/*
 * Full forward of Nq queries against Nkv keys: Q and O are [BH, Nq, D], K and
 * V are [BH, Nkv, D], LSE is [BH, Nq]; the causal mask is bottom-right (query
 * i sees keys j <= i + Nkv - Nq).  Returns 0, or -1 if a scratch allocation
 * failed.
 */
int attn_ref_forward_qkv(const void *Q, const void *K, const void *V, int dtype,
                         long BH, long Nq, long Nkv, long D, int causal, double s,
                         double *O, double *LSE)
{
    size_t qslice = (size_t)Nq * (size_t)D, kslice = (size_t)Nkv * (size_t)D;
    double *Kh = (double *)malloc(kslice * sizeof(double));
    double *Vh = (double *)malloc(kslice * sizeof(double));
    double *Qh = (double *)malloc(qslice * sizeof(double));
    if (!Kh || !Vh || !Qh) {
        free(Kh); free(Vh); free(Qh);
        return -1;
    }
    int failed = 0;
    for (long bh = 0; bh < BH; ++bh) {
        load_slice(Q, dtype, (size_t)bh * qslice, Nq, D, Qh);
        load_slice(K, dtype, (size_t)bh * kslice, Nkv, D, Kh);
        load_slice(V, dtype, (size_t)bh * kslice, Nkv, D, Vh);
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)Nkv * sizeof(double));
            if (!x) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long i = 0; i < Nq; ++i) {
                    long nvis = Nkv;
                    if (causal) {
                        long last = i + Nkv - Nq;   /* the last key query i sees */
                        nvis = last + 1 < Nkv ? last + 1 : Nkv;
                    }
                    ref_row_vis(Qh + i * D, Kh, Vh, nvis, D, s, x, O + (size_t)bh * qslice + (size_t)i * D,
                                LSE + (size_t)bh * Nq + i);
                }
            }
            free(x);
        }
    }
    free(Kh); free(Vh); free(Qh);
    return failed ? -1 : 0;
}

/*
 * Band-masked forward: Q and O are [BH, Nq, D], K and V are [BH, Nkv, D],
 * LSE is [BH, Nq]; query i sees keys j with i' - left <= j <= i' + right,
 * i' = i + Nkv - Nq (left or right < 0: unbounded).  Returns 0, or -1 if a
 * scratch allocation failed.
 */
int attn_ref_forward_band(const void *Q, const void *K, const void *V, int dtype,
                          long BH, long Nq, long Nkv, long D, long left, long right, double s,
                          double *O, double *LSE)
{
    size_t qslice = (size_t)Nq * (size_t)D, kslice = (size_t)Nkv * (size_t)D;
    double *Kh = (double *)malloc(kslice * sizeof(double));
    double *Vh = (double *)malloc(kslice * sizeof(double));
    double *Qh = (double *)malloc(qslice * sizeof(double));
    if (!Kh || !Vh || !Qh) {
        free(Kh); free(Vh); free(Qh);
        return -1;
    }
    int failed = 0;
    for (long bh = 0; bh < BH; ++bh) {
        load_slice(Q, dtype, (size_t)bh * qslice, Nq, D, Qh);
        load_slice(K, dtype, (size_t)bh * kslice, Nkv, D, Kh);
        load_slice(V, dtype, (size_t)bh * kslice, Nkv, D, Vh);
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)Nkv * sizeof(double));
            if (!x) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long i = 0; i < Nq; ++i) {
                    const long ii = i + Nkv - Nq;                        /* the query's position among the keys */
                    long lo = left < 0 ? 0 : ii - left, hi = right < 0 ? Nkv - 1 : ii + right;
                    if (lo < 0)
                        lo = 0;
                    if (hi > Nkv - 1)
                        hi = Nkv - 1;
                    const long nvis = hi >= lo ? hi - lo + 1 : 0;        /* keys lo .. hi */
                    ref_row_vis(Qh + i * D, Kh + (nvis > 0 ? lo : 0) * D, Vh + (nvis > 0 ? lo : 0) * D, nvis, D, s,
                                x, O + (size_t)bh * qslice + (size_t)i * D, LSE + (size_t)bh * Nq + i);
                }
            }
            free(x);
        }
    }
    free(Kh); free(Vh); free(Qh);
    return failed ? -1 : 0;
}

/*
 * Gradients of O = softmax(S) V, S = s Q K^T under the band mask of
 * attn_ref_forward_band, for an upstream gradient dO (same shape as O).  With
 * J_i the keys query i sees and L_i its log-sum-exp:
 *
 *   P[i,j]  = exp(s q_i.k_j - L_i)             for j in J_i, else 0
 *   dV[j,:] = sum_i P[i,j] dO[i,:]
 *   dP[i,j] = dO[i,:] . V[j,:]
 *   delta_i = sum_j P[i,j] dP[i,j]
 *   dS[i,j] = P[i,j] (dP[i,j] - delta_i)       (the softmax's Jacobian applied to dP)
 *   dQ[i,:] = s sum_j dS[i,j] K[j,:]
 *   dK[j,:] = s sum_i dS[i,j] Q[i,:]
 *
 * These are the chain rule through the definition, written out; the pages
 * name the backward's ingredients rather than its formulas ("FlashAttention 2
 * from PyTorch to Triton", What I am building: P is recovered as exp(S - L)
 * from the saved L; and its list of limitations: a precomputed
 * D = rowsum(dO o O), which equals delta_i here, since
 * dO_i . O_i = sum_j P[i,j] dO_i . V_j).  A row that sees no key has P = 0:
 * its dQ row is 0 and it adds nothing to dK or dV.
 *
 * Q, dO are [BH, Nq, D]; K, V are [BH, Nkv, D]; outputs are float64:
 * dQ [BH, Nq, D], dK and dV [BH, Nkv, D], and DELTA [BH, Nq] if not NULL.
 * Two passes per head: over query rows (L_i, delta_i, dQ_i), then over key
 * rows (dK_j, dV_j), each recomputing the P and dP entries it needs, so no
 * Nq x Nkv matrix is stored.  Returns 0, or -1 if a scratch allocation failed.
 */
static void band_range(long i, long Nq, long Nkv, long left, long right, long *lo, long *hi)
{
    const long ii = i + Nkv - Nq;   /* the query's position among the keys */
    long a = left < 0 ? 0 : ii - left, b = right < 0 ? Nkv - 1 : ii + right;
    if (a < 0)
        a = 0;
    if (b > Nkv - 1)
        b = Nkv - 1;
    *lo = a;
    *hi = b;   /* keys a .. b; none if b < a */
}

static double dot_d(const double *a, const double *b, long D)
{
    double acc = 0.0;
    for (long d = 0; d < D; ++d)
        acc += a[d] * b[d];
    return acc;
}

int attn_ref_backward_band(const void *Q, const void *K, const void *V, const void *dO, int dtype,
                           long BH, long Nq, long Nkv, long D, long left, long right, double s,
                           double *dQ, double *dK, double *dV, double *DELTA)
{
    size_t qslice = (size_t)Nq * (size_t)D, kslice = (size_t)Nkv * (size_t)D;
    double *Kh = (double *)malloc(kslice * sizeof(double));
    double *Vh = (double *)malloc(kslice * sizeof(double));
    double *Qh = (double *)malloc(qslice * sizeof(double));
    double *dOh = (double *)malloc(qslice * sizeof(double));
    double *Lr = (double *)malloc((size_t)Nq * sizeof(double));
    double *Dr = (double *)malloc((size_t)Nq * sizeof(double));
    if (!Kh || !Vh || !Qh || !dOh || !Lr || !Dr) {
        free(Kh); free(Vh); free(Qh); free(dOh); free(Lr); free(Dr);
        return -1;
    }
    int failed = 0;
    for (long bh = 0; bh < BH; ++bh) {
        load_slice(Q, dtype, (size_t)bh * qslice, Nq, D, Qh);
        load_slice(dO, dtype, (size_t)bh * qslice, Nq, D, dOh);
        load_slice(K, dtype, (size_t)bh * kslice, Nkv, D, Kh);
        load_slice(V, dtype, (size_t)bh * kslice, Nkv, D, Vh);
        double *dQh = dQ + (size_t)bh * qslice, *dKh = dK + (size_t)bh * kslice, *dVh = dV + (size_t)bh * kslice;
        /* Pass 1, query rows: L_i, delta_i, dQ_i. */
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)Nkv * sizeof(double));
            if (!x) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long i = 0; i < Nq; ++i) {
                    long lo, hi;
                    band_range(i, Nq, Nkv, left, right, &lo, &hi);
                    double *dq = dQh + (size_t)i * D;
                    for (long d = 0; d < D; ++d)
                        dq[d] = 0.0;
                    if (hi < lo) {   /* no key: P = 0 */
                        Lr[i] = -INFINITY;
                        Dr[i] = 0.0;
                        continue;
                    }
                    double m = -INFINITY;
                    for (long j = lo; j <= hi; ++j) {
                        x[j] = s * dot_d(Qh + i * D, Kh + j * D, D);
                        if (x[j] > m)
                            m = x[j];
                    }
                    double l = 0.0;
                    for (long j = lo; j <= hi; ++j)
                        l += exp(x[j] - m);
                    const double L = m + log(l);
                    double delta = 0.0;
                    for (long j = lo; j <= hi; ++j)
                        delta += exp(x[j] - L) * dot_d(dOh + i * D, Vh + j * D, D);
                    for (long j = lo; j <= hi; ++j) {
                        const double p = exp(x[j] - L);
                        const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - delta);
                        for (long d = 0; d < D; ++d)
                            dq[d] += s * ds * Kh[j * D + d];
                    }
                    Lr[i] = L;
                    Dr[i] = delta;
                }
            }
            free(x);
        }
        /* Pass 2, key rows: dK_j, dV_j over the queries that see key j. */
#pragma omp parallel for schedule(dynamic, 8)
        for (long j = 0; j < Nkv; ++j) {
            double *dk = dKh + (size_t)j * D, *dv = dVh + (size_t)j * D;
            for (long d = 0; d < D; ++d)
                dk[d] = dv[d] = 0.0;
            for (long i = 0; i < Nq; ++i) {
                long lo, hi;
                band_range(i, Nq, Nkv, left, right, &lo, &hi);
                if (j < lo || j > hi)
                    continue;
                const double p = exp(s * dot_d(Qh + i * D, Kh + j * D, D) - Lr[i]);
                const double ds = p * (dot_d(dOh + i * D, Vh + j * D, D) - Dr[i]);
                for (long d = 0; d < D; ++d) {
                    dv[d] += p * dOh[i * D + d];
                    dk[d] += s * ds * Qh[i * D + d];
                }
            }
        }
        if (DELTA)
            memcpy(DELTA + (size_t)bh * Nq, Dr, (size_t)Nq * sizeof(double));
    }
    free(Kh); free(Vh); free(Qh); free(dOh); free(Lr); free(Dr);
    return failed ? -1 : 0;
}

/*
 * Selected rows only: row r is (bh_idx[r], row_idx[r]).  bh_idx must be
 * non-decreasing so each head's K/V slice is widened once.  O_rows is
 * [nrows, D], LSE_rows is [nrows].  Returns 0, -1 on allocation failure,
 * -2 on a bad index.  Every row is independent, so a sampled row is exactly
 * the row the full forward would give.
 */
int attn_ref_rows(const void *Q, const void *K, const void *V, int dtype,
                  long BH, long N, long D, int causal, double s,
                  const long *bh_idx, const long *row_idx, long nrows,
                  double *O_rows, double *LSE_rows)
{
    for (long r = 0; r < nrows; ++r) {
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= N)
            return -2;
        if (r > 0 && bh_idx[r] < bh_idx[r - 1])
            return -2;
    }
    size_t slice = (size_t)N * (size_t)D;
    double *Kh = (double *)malloc(slice * sizeof(double));
    double *Vh = (double *)malloc(slice * sizeof(double));
    if (!Kh || !Vh) {
        free(Kh); free(Vh);
        return -1;
    }
    int failed = 0;
    long r0 = 0;
    while (r0 < nrows) {
        long bh = bh_idx[r0];
        long r1 = r0;
        while (r1 < nrows && bh_idx[r1] == bh)
            ++r1;
        size_t base = (size_t)bh * slice;
        load_slice(K, dtype, base, N, D, Kh);
        load_slice(V, dtype, base, N, D, Vh);
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)N * sizeof(double));
            double *q = (double *)malloc((size_t)D * sizeof(double));
            if (!x || !q) {
#pragma omp atomic write
                failed = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (long r = r0; r < r1; ++r) {
                    for (long d = 0; d < D; ++d)
                        q[d] = load_elem(Q, dtype, base + (size_t)row_idx[r] * D + d);
                    ref_row(q, Kh, Vh, N, D, row_idx[r], causal, s, x,
                            O_rows + (size_t)r * D, LSE_rows + r);
                }
            }
            free(x);
            free(q);
        }
        r0 = r1;
    }
    free(Kh); free(Vh);
    return failed ? -1 : 0;
}

/*
 * The explicit probability matrix P = softmax(S) of one [N, D] head (float64
 * inputs), P is [N, N].  Masked entries are exactly 0.  For small N only.
 */
void attn_ref_probs(const double *Q, const double *K, long N, long D, int causal, double s, double *P)
{
    for (long i = 0; i < N; ++i) {
        long nvis = causal ? i + 1 : N;
        double m = -INFINITY;
        for (long j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d)
                dot += Q[i * D + d] * K[j * D + d];
            P[i * N + j] = s * dot;
            if (P[i * N + j] > m)
                m = P[i * N + j];
        }
        double l = 0.0;
        for (long j = 0; j < nvis; ++j) {
            P[i * N + j] = exp(P[i * N + j] - m);
            l += P[i * N + j];
        }
        for (long j = 0; j < nvis; ++j)
            P[i * N + j] /= l;
        for (long j = nvis; j < N; ++j)
            P[i * N + j] = 0.0;
    }
}

/*
 * The tiled online-softmax recurrence (FlashAttention-2 forward), in fp64,
 * over float64 [BH, N, D] inputs with query tiles of BM rows and key tiles of
 * BN rows (either may leave a ragged last tile).
 *
 * Per query tile, following "FlashAttention 2 from PyTorch to Triton" (Step 1:
 * the tiled forward in PyTorch), "A09 - Advanced Triton & FlashAttention"
 * (3. Deep Dive: the rescaling update, written out; causal masking: skipping
 * beats masking) and "Triton: FlashAttention-2 Forward Pass" (the online-
 * softmax state; the rescale direction; masks and sentinels):
 *
 *   m = -inf, l = 0, acc = 0
 *   hi = min(end of this query tile, N) if causal else N   (later keys skipped)
 *   for each key tile starting below hi:
 *     S     = s * Q_tile K_tile^T, with -inf where key >= N or (causal) key > query
 *     m_new = max(m, rowmax(S))
 *     alpha = exp(m - m_new)                    (0 on the first tile: m = -inf)
 *     P     = exp(S - m_new)
 *     l     = alpha * l + rowsum(P)
 *     acc   = alpha * acc + P V_tile
 *     m     = m_new
 *   O = acc / l, L = m + log(l)
 *
 * A row whose visible keys so far are all masked has m_new = -inf; the pages
 * note that -inf - (-inf) is NaN there, so the shift used is 0 for such a row
 * (its P and alpha are then exactly 0).  A row that never sees a key keeps
 * l = 0 and is given O = 0, L = -inf.
 */
int attn_ref_tiled(const double *Q, const double *K, const double *V,
                   long BH, long N, long D, int causal, double s, long BM, long BN,
                   double *O, double *LSE)
{
    if (BM < 1 || BN < 1)
        return -2;
    double *S = (double *)malloc((size_t)BN * sizeof(double));
    double *acc = (double *)malloc((size_t)BM * (size_t)D * sizeof(double));
    double *m = (double *)malloc((size_t)BM * sizeof(double));
    double *l = (double *)malloc((size_t)BM * sizeof(double));
    if (!S || !acc || !m || !l) {
        free(S); free(acc); free(m); free(l);
        return -1;
    }
    for (long bh = 0; bh < BH; ++bh) {
        const double *Qh = Q + (size_t)bh * N * D;
        const double *Kh = K + (size_t)bh * N * D;
        const double *Vh = V + (size_t)bh * N * D;
        for (long q0 = 0; q0 < N; q0 += BM) {
            long rows = (N - q0 < BM) ? N - q0 : BM;
            for (long r = 0; r < rows; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (long d = 0; d < D; ++d)
                    acc[r * D + d] = 0.0;
            }
            long hi = N;
            if (causal)
                hi = (q0 + BM < N) ? q0 + BM : N;
            for (long k0 = 0; k0 < hi; k0 += BN) {
                for (long r = 0; r < rows; ++r) {
                    long qi = q0 + r;
                    double tile_max = -INFINITY;
                    for (long c = 0; c < BN; ++c) {
                        long kj = k0 + c;
                        if (kj >= N || (causal && kj > qi)) {
                            S[c] = -INFINITY;
                        } else {
                            double dot = 0.0;
                            for (long d = 0; d < D; ++d)
                                dot += Qh[qi * D + d] * Kh[kj * D + d];
                            S[c] = s * dot;
                        }
                        if (S[c] > tile_max)
                            tile_max = S[c];
                    }
                    double m_new = (m[r] > tile_max) ? m[r] : tile_max;
                    double shift = (m_new == -INFINITY) ? 0.0 : m_new;
                    double alpha = exp(m[r] - shift);
                    double rowsum = 0.0;
                    for (long c = 0; c < BN; ++c) {
                        S[c] = exp(S[c] - shift);       /* S now holds P */
                        rowsum += S[c];
                    }
                    l[r] = alpha * l[r] + rowsum;
                    for (long d = 0; d < D; ++d) {
                        double pv = 0.0;
                        for (long c = 0; c < BN; ++c)
                            if (k0 + c < N)
                                pv += S[c] * Vh[(k0 + c) * D + d];
                        acc[r * D + d] = alpha * acc[r * D + d] + pv;
                    }
                    m[r] = m_new;
                }
            }
            for (long r = 0; r < rows; ++r) {
                long qi = q0 + r;
                for (long d = 0; d < D; ++d)
                    O[((size_t)bh * N + qi) * D + d] = (l[r] > 0.0) ? acc[r * D + d] / l[r] : 0.0;
                LSE[(size_t)bh * N + qi] = (l[r] > 0.0) ? m[r] + log(l[r]) : -INFINITY;
            }
        }
    }
    free(S); free(acc); free(m); free(l);
    return 0;
}
