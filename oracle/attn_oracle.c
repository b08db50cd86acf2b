/*
 * CPU fp64 oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes is the plain definition of masked softmax attention, not
 * the tiled algorithm that reaches it:
 *
 *   for every (b, h, i):
 *     A(i)  = the attended key set of row i
 *               dense           : all j in [0, L)
 *               causal          : j <= i              ("Fused Attention" page,
 *                                                      stage-2 mask offs_m >= offs_n)
 *               block-diagonal  : floor(j/bs) == floor(i/bs)
 *                                                     ("TLX Block Attention" page,
 *                                                      definition of the diagonal
 *                                                      blocks at its top)
 *     s_j   = sm_scale * sum_d q[i,d] * k[j,d]     for j in A(i), ascending d
 *     m     = max_{j in A(i)} s_j
 *     l     = sum_{j in A(i)} exp(s_j - m)          (denominator starts at 0)
 *     O[i,:]= sum_{j in A(i)} exp(s_j - m) * v[j,:] / l
 *     lse_i = m + ln(l)                              ("Fused Attention" page,
 *                                                      epilogue m_i += log(l_i))
 *
 * The scores of one row are all computed and held in an L-long buffer before
 * the row is normalised (two passes over the row, no online update, no tiling
 * over j).  Everything is fp64; the inputs are the fp16/bf16 values the GPU
 * sees, widened exactly.  Rows are independent, so rows are spread over
 * OpenMP threads; the arithmetic inside a row is strictly sequential.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; the
 * CPU tests build every mutant and check that the pins catch each of them.
 *
 * attn_oracle_fp8v is the page's FP8 variant, which is not the plain
 * definition above: see its comment.  attn_oracle_bwd (at the end) is the
 * gradient of the definition above by the chain rule: see its comment.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { OR_DENSE = 0, OR_CAUSAL = 1, OR_BLOCK_DIAG = 2 };
enum { OR_F16 = 0, OR_BF16 = 1 };

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 -> double: bfloat16 is the upper half of an IEEE binary32. */
static double widen_bf16(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

double attn_oracle_widen(uint16_t bits, int dtype)
{
    return dtype == OR_BF16 ? widen_bf16(bits) : widen_f16(bits);
}

/* 1 if key j is in the attended set of query row i. */
static int attended(long i, long j, int mask_kind, long bs)
{
#if ORACLE_MUTANT == 1
    if (mask_kind == OR_CAUSAL) return j < i;          /* planted: drops the diagonal */
#endif
#if ORACLE_MUTANT == 6
    if (mask_kind == OR_BLOCK_DIAG) return (j % bs) == (i % bs);  /* planted: strided blocks */
#endif
    if (mask_kind == OR_CAUSAL) return j <= i;
    if (mask_kind == OR_BLOCK_DIAG) return (j / bs) == (i / bs);
    return 1;
}

/* One query row (b,h,i): fills o[0..D) and *lse.  q, k, v point at the
 * (b,h) slice [L, D] already widened to fp64; s is scratch of length L. */
static void one_row(const double *q, const double *k, const double *v,
                    long L, long D, long i, int mask_kind, long bs,
                    double sm_scale, double *s, double *o, double *lse)
{
    const double *qi = q + i * D;
    double m = -INFINITY;
    for (long j = 0; j < L; ++j) {
        if (!attended(i, j, mask_kind, bs)) {
            s[j] = -INFINITY;
            continue;
        }
#if ORACLE_MUTANT == 7
        const double *kj = v + j * D;                   /* planted: V in place of K */
#else
        const double *kj = k + j * D;
#endif
        double dot = 0.0;
#if ORACLE_MUTANT == 10
        for (long d = 0; d < D - 1; ++d)                /* planted: drops the last term */
#else
        for (long d = 0; d < D; ++d)
#endif
            dot += qi[d] * kj[d];
#if ORACLE_MUTANT == 2
        s[j] = dot;                                     /* planted: scale dropped */
#else
        s[j] = sm_scale * dot;
#endif
        if (s[j] > m) m = s[j];
    }

#if ORACLE_MUTANT == 3
    double l = 1.0;                                     /* planted: denominator starts at 1 */
#else
    double l = 0.0;
#endif
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long j = 0; j < L; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
#if ORACLE_MUTANT == 5
        const double *vj = v + i * D;                   /* planted: wrong row of V */
#elif ORACLE_MUTANT == 7
        const double *vj = k + j * D;
#else
        const double *vj = v + j * D;
#endif
#if ORACLE_MUTANT == 9
        p = exp(s[j]);                                  /* planted: max not removed in O only */
#endif
        for (long d = 0; d < D; ++d) o[d] += p * vj[d];
    }
    for (long d = 0; d < D; ++d) o[d] /= l;
#if ORACLE_MUTANT == 4
    *lse = log(l);                                      /* planted: max dropped from lse */
#elif ORACLE_MUTANT == 8
    *lse = m + log2(l);                                 /* planted: wrong log base */
#else
    *lse = m + log(l);
#endif
}

/*
 * Masked attention forward on [B,H,L,D] inputs given as raw fp16/bf16 bits.
 *
 *   rows == NULL : every row; O is [B,H,L,D] and lse is [B,H,L] (fp64).
 *   rows != NULL : only the nrows flat row ids r = (b*H + h)*L + i; O is
 *                  [nrows, D] and lse is [nrows], in the order given.
 *
 * Returns 0, or -1 on an argument error (nothing written).
 */
int attn_oracle(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                int dtype, long B, long H, long L, long D,
                int mask_kind, long bs, double sm_scale,
                const long *rows, long nrows,
                double *O, double *lse, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || D <= 0) return -1;
    if (mask_kind < OR_DENSE || mask_kind > OR_BLOCK_DIAG) return -1;
    if (mask_kind == OR_BLOCK_DIAG && (bs <= 0 || (L > 0 && L % bs != 0))) return -1;
    if (dtype != OR_F16 && dtype != OR_BF16) return -1;
    const long BH = B * H;
    const long total = rows ? nrows : BH * L;
    if (total == 0) return 0;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= BH * L) return -1;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
    /* Rows are grouped by (b,h): each group widens its slice once. */
#pragma omp parallel
    {
        double *qs = malloc(sizeof(double) * L * D);
        double *ks = malloc(sizeof(double) * L * D);
        double *vs = malloc(sizeof(double) * L * D);
        double *s = malloc(sizeof(double) * (L > 0 ? L : 1));
        long cur_bh = -1;
        if (!qs || !ks || !vs || !s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < total; ++t) {
            if (err) continue;
            long r = rows ? rows[t] : t;
            long bh = r / L, i = r % L;
            if (bh != cur_bh) {
                const size_t base = (size_t)bh * L * D;
                for (long e = 0; e < L * D; ++e) {
                    qs[e] = attn_oracle_widen(q[base + e], dtype);
                    ks[e] = attn_oracle_widen(k[base + e], dtype);
                    vs[e] = attn_oracle_widen(v[base + e], dtype);
                }
                cur_bh = bh;
            }
            one_row(qs, ks, vs, L, D, i, mask_kind, bs, sm_scale, s,
                    O + (size_t)t * D, lse + t);
        }
        free(qs); free(ks); free(vs); free(s);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------ fp8 P.V
 *
 * The "Fused Attention" page's FP8 variant: V is given in float8 e5m2 and
 * stored transposed ([B, H, D, L], keys innermost: the page notes that an
 * e5m2 V is transposed), P is cast to e5m2 before P.V (`p.to(tl.float8e5)`),
 * and the softmax denominator sums the unrounded p (`l_ij = tl.sum(p, 1)`).
 * The result then depends on where P is rounded, so this function follows the
 * page's tiled algorithm rather than the definition: key tiles of 128 keys
 * from key 0, taken in order; per tile the running max m_new = max(m, tile
 * max), p = exp(s - m_new) rounded to e5m2 for the P.V product, acc and l
 * rescaled by exp(m - m_new).  Tiles without an attended key are skipped (they
 * would change nothing).
 */

/* float8 e5m2 -> double: 1 sign bit, 5 exponent bits (bias 15), 2 fraction
 * bits. */
static double widen_e5m2(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int f = b & 3;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -16);               /* subnormal: f/4 * 2^-14 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(4 + f), e - 17);      /* (1 + f/4) * 2^(e-15) */
    return sign ? -mag : mag;
}

double attn_oracle_widen_e5m2(uint8_t b)
{
    return widen_e5m2(b);
}

/* Round a finite x >= 0 to e5m2: nearest, ties to even, saturating at the
 * largest finite value 57344.  *quantum receives the spacing of e5m2 values
 * around x (the step a rounding decision spans). */
static double round_e5m2(double x, double *quantum)
{
    double qv;
    if (x < 0x1p-14) {
        qv = 0x1p-16;                              /* subnormal spacing */
    } else {
        int ex;
        frexp(x, &ex);                             /* x in [2^(ex-1), 2^ex) */
        qv = ldexp(1.0, ex - 1 - 2);               /* 2 fraction bits */
    }
    if (quantum) *quantum = qv;
#if ORACLE_MUTANT == 11
    double r = floor(x / qv) * qv;                 /* planted: truncation */
#else
    double r = nearbyint(x / qv) * qv;             /* default rounding: ties to even */
#endif
    return r > 57344.0 ? 57344.0 : r;
}

double attn_oracle_round_e5m2(double x)
{
    return round_e5m2(x, NULL);
}

/* One query row of the FP8 variant.  q, k: the (b,h) slice [L, D] widened to
 * fp64; vt: the (b,h) slice of V^T [D, L] as e5m2 bytes.  s: scratch of 2L.
 * *slack receives a bound on how far a single-precision computation of p can
 * move O by rounding a p that lies near an e5m2 rounding tie to the other
 * neighbour.  "Near" is the error bound of such a computation of the exponent
 * s_j - m (natural-log units): the rounding of a D-term dot product, at most
 * D * 2^-24 * sum_d |q_d k_d| scaled by |sm_scale| (the standard bound of a
 * recursive sum), the rounding of the scaled score and of the subtraction of
 * the max, 2^-23 * (|s_j| + |m|), and 5e-5 for an approximate exponential. */
static void one_row_fp8v(const double *q, const double *k, const uint8_t *vt, long L, long D, long i,
                         int mask_kind, long bs, double sm_scale, double *s, double *o, double *lse,
                         double *slack)
{
    const double *qi = q + i * D;
    double m = -INFINITY, l = 0.0, tie = 0.0;
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long t0 = 0; t0 < L; t0 += 128) {
        const long t1 = t0 + 128 < L ? t0 + 128 : L;
        double mt = -INFINITY;
        int any = 0;
        for (long j = t0; j < t1; ++j) {
            if (!attended(i, j, mask_kind, bs)) continue;
            double dot = 0.0, absdot = 0.0;
            for (long d = 0; d < D; ++d) {
                dot += qi[d] * k[j * D + d];
                absdot += fabs(qi[d] * k[j * D + d]);
            }
            s[j] = sm_scale * dot;
            s[L + j] = fabs(sm_scale) * absdot;
            if (s[j] > mt) mt = s[j];
            any = 1;
        }
        if (!any) continue;
        const double m_new = mt > m ? mt : m;
        const double alpha = exp(m - m_new);           /* 0 on the first tile */
        for (long d = 0; d < D; ++d) o[d] *= alpha;
        l *= alpha;
        tie *= alpha;
        for (long j = t0; j < t1; ++j) {
            if (!attended(i, j, mask_kind, bs)) continue;
            const double p = exp(s[j] - m_new);
            double qv;
            const double p8 = round_e5m2(p, &qv);
#if ORACLE_MUTANT == 12
            l += p8;                                   /* planted: sums the rounded p */
#else
            l += p;
#endif
            double vmax = 0.0;
#if ORACLE_MUTANT == 15
            double vsum = 0.0;
#endif
            for (long d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 13
                const double vj = widen_e5m2(vt[j * D + d]);   /* planted: V read untransposed */
#else
                const double vj = widen_e5m2(vt[d * L + j]);
#endif
                o[d] += p8 * vj;
                if (fabs(vj) > vmax) vmax = fabs(vj);
#if ORACLE_MUTANT == 15
                vsum += fabs(vj);
#endif
            }
            /* p within the single-precision error of a tie (relative band
             * delta, see above) may round to the other neighbour; one such
             * flip moves each element of O by qv |v_jd| / l, so the row's
             * largest change is qv max_d |v_jd| / l */
            double delta = (double)D * 0x1p-24 * s[L + j] +
                           0x1p-23 * (fabs(s[j]) + fabs(m_new)) + 5e-5;
#if ORACLE_MUTANT == 14
            delta *= 100.0;                            /* planted: band 100x too wide */
#endif
            const double frac = p / qv - floor(p / qv);
#if ORACLE_MUTANT == 15
            if (fabs(frac - 0.5) < delta * (p / qv)) tie += qv * vsum;   /* planted: per column */
#else
            if (fabs(frac - 0.5) < delta * (p / qv)) tie += qv * vmax;
#endif
        }
        m = m_new;
    }
    for (long d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
    *slack = tie / l;
}

/*
 * FP8 variant on Q, K as fp16/bf16 bits ([B,H,L,D]) and V^T as e5m2 bytes
 * ([B,H,D,L]).  Same row selection and outputs as attn_oracle, plus slack
 * ([B,H,L] or [nrows]): per row, the tie bound described above.
 * Returns 0, or -1 on an argument error.
 */
int attn_oracle_fp8v(const uint16_t *q, const uint16_t *k, const uint8_t *vt, int dtype, long B, long H,
                     long L, long D, int mask_kind, long bs, double sm_scale, const long *rows, long nrows,
                     double *O, double *lse, double *slack, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || D <= 0) return -1;
    if (mask_kind < OR_DENSE || mask_kind > OR_BLOCK_DIAG) return -1;
    if (mask_kind == OR_BLOCK_DIAG && (bs <= 0 || (L > 0 && L % bs != 0))) return -1;
    if (dtype != OR_F16 && dtype != OR_BF16) return -1;
    const long BH = B * H;
    const long total = rows ? nrows : BH * L;
    if (total == 0) return 0;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= BH * L) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *qs = malloc(sizeof(double) * L * D);
        double *ks = malloc(sizeof(double) * L * D);
        double *s = malloc(sizeof(double) * (L > 0 ? 2 * L : 1));
        long cur_bh = -1;
        if (!qs || !ks || !s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < total; ++t) {
            if (err) continue;
            long r = rows ? rows[t] : t;
            long bh = r / L, i = r % L;
            if (bh != cur_bh) {
                const size_t base = (size_t)bh * L * D;
                for (long e = 0; e < L * D; ++e) {
                    qs[e] = attn_oracle_widen(q[base + e], dtype);
                    ks[e] = attn_oracle_widen(k[base + e], dtype);
                }
                cur_bh = bh;
            }
            one_row_fp8v(qs, ks, vt + (size_t)bh * D * L, L, D, i, mask_kind, bs, sm_scale, s,
                         O + (size_t)t * D, lse + t, slack + t);
        }
        free(qs); free(ks); free(s);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------ backward
 *
 * Gradients of the masked softmax attention above with respect to q, k and v
 * for an output gradient dO (the pages save q, k, v, O and the row statistic
 * for a backward they do not define; this follows from the definition by the
 * chain rule through the softmax), per head, for every row i and key j:
 *
 *   P[i,j]  = exp(s_ij - lse_i)   for j in A(i), 0 otherwise
 *   dV[j,:] = sum_i P[i,j] dO[i,:]
 *   dP[i,j] = sum_d dO[i,d] v[j,d]
 *   Di      = sum_j P[i,j] dP[i,j]
 *   dS[i,j] = P[i,j] (dP[i,j] - Di)
 *   dQ[i,:] = sm_scale sum_j dS[i,j] k[j,:]
 *   dK[j,:] = sm_scale sum_i dS[i,j] q[i,:]
 *
 * with s and lse as in one_row.  Inputs are fp64 [B,H,L,D] arrays (16-bit
 * callers widen them first; the finite-difference pins perturb them).
 *
 * Also returned, per element, the magnitudes a computation that rounds P and
 * dS to a 16-bit type and takes Di from a rounded O is sensitive to:
 *   bV[j,d] = sum_i P[i,j] |dO[i,d]|
 *   bK[j,d] = |sm_scale| sum_i (|dS[i,j]| + P[i,j] a_i) |q[i,d]|
 *   bQ[i,d] = |sm_scale| sum_j (|dS[i,j]| + P[i,j] a_i) |k[j,d]|
 * with a_i = sum_d |dO[i,d] O[i,d]|.  (Each may be NULL.)
 */
static void one_head_bwd(const double *q, const double *k, const double *v, const double *dO,
                         long L, long D, int mask_kind, long bs, double sm_scale,
                         double *dQ, double *dK, double *dV, double *bQ, double *bK, double *bV,
                         double *s, double *P, double *dS, double *o)
{
    for (long e = 0; e < L * D; ++e) {
        dQ[e] = dK[e] = dV[e] = 0.0;
        if (bQ) bQ[e] = 0.0;
        if (bK) bK[e] = 0.0;
        if (bV) bV[e] = 0.0;
    }
    for (long i = 0; i < L; ++i) {
        double lse;
        one_row(q, k, v, L, D, i, mask_kind, bs, sm_scale, s, o, &lse);
        const double *dOi = dO + i * D;
        double Di = 0.0, ai = 0.0;
        for (long d = 0; d < D; ++d) ai += fabs(dOi[d] * o[d]);
        for (long j = 0; j < L; ++j) {
            if (!attended(i, j, mask_kind, bs)) {
                P[j] = 0.0;
                dS[j] = 0.0;
                continue;
            }
            P[j] = exp(s[j] - lse);
            double dp = 0.0;
            for (long d = 0; d < D; ++d) dp += dOi[d] * v[j * D + d];
            dS[j] = dp;                                   /* dP for now */
            Di += P[j] * dp;
        }
        for (long j = 0; j < L; ++j) {
            if (P[j] == 0.0 && dS[j] == 0.0) continue;
#if ORACLE_MUTANT == 21
            dS[j] = P[j] * dS[j];                         /* planted: Di dropped */
#else
            dS[j] = P[j] * (dS[j] - Di);
#endif
        }
        for (long j = 0; j < L; ++j) {
            if (!attended(i, j, mask_kind, bs)) continue;
            const double w = fabs(dS[j]) + P[j] * ai;
            for (long d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 23
                dV[i * D + d] += P[j] * dO[j * D + d];    /* planted: P transposed */
#else
                dV[j * D + d] += P[j] * dOi[d];
#endif
                dQ[i * D + d] += sm_scale * dS[j] * k[j * D + d];
#if ORACLE_MUTANT == 22
                dK[j * D + d] += dS[j] * q[i * D + d];    /* planted: scale dropped */
#else
                dK[j * D + d] += sm_scale * dS[j] * q[i * D + d];
#endif
#if ORACLE_MUTANT == 24
                if (bQ) bQ[i * D + d] += 4.0 * fabs(sm_scale) * w * fabs(k[j * D + d]);  /* planted: 4x */
#else
                if (bQ) bQ[i * D + d] += fabs(sm_scale) * w * fabs(k[j * D + d]);
#endif
#if ORACLE_MUTANT == 25
                if (bK) bK[j * D + d] += 4.0 * fabs(sm_scale) * w * fabs(q[i * D + d]);  /* planted: 4x */
#else
                if (bK) bK[j * D + d] += fabs(sm_scale) * w * fabs(q[i * D + d]);
#endif
#if ORACLE_MUTANT == 26
                if (bV) bV[j * D + d] += 4.0 * P[j] * fabs(dOi[d]);                      /* planted: 4x */
#else
                if (bV) bV[j * D + d] += P[j] * fabs(dOi[d]);
#endif
            }
        }
    }
}

/* Backward over [B,H,L,D] fp64 inputs; outputs [B,H,L,D] fp64 (bQ, bK, bV may
 * be NULL).  Heads are spread over OpenMP threads.  Returns 0, or -1 on an
 * argument error. */
int attn_oracle_bwd(const double *q, const double *k, const double *v, const double *dO, long B, long H,
                    long L, long D, int mask_kind, long bs, double sm_scale, double *dQ, double *dK,
                    double *dV, double *bQ, double *bK, double *bV, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || D <= 0) return -1;
    if (mask_kind < OR_DENSE || mask_kind > OR_BLOCK_DIAG) return -1;
    if (mask_kind == OR_BLOCK_DIAG && (bs <= 0 || (L > 0 && L % bs != 0))) return -1;
    const long BH = B * H;
    if (BH * L == 0) return 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * L);
        double *P = malloc(sizeof(double) * L);
        double *dS = malloc(sizeof(double) * L);
        double *o = malloc(sizeof(double) * D);
        if (!s || !P || !dS || !o) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            if (err) continue;
            const size_t base = (size_t)bh * L * D;
            one_head_bwd(q + base, k + base, v + base, dO + base, L, D, mask_kind, bs, sm_scale,
                         dQ + base, dK + base, dV + base, bQ ? bQ + base : NULL, bK ? bK + base : NULL,
                         bV ? bV + base : NULL, s, P, dS, o);
        }
        free(s); free(P); free(dS); free(o);
    }
    return err ? -1 : 0;
}

/* The forward of attn_oracle on fp64 inputs (for the backward's
 * finite-difference pins): O [B,H,L,D] and lse [B,H,L]. */
int attn_oracle_f64(const double *q, const double *k, const double *v, long B, long H, long L, long D,
                    int mask_kind, long bs, double sm_scale, double *O, double *lse)
{
    if (B < 0 || H < 0 || L < 0 || D <= 0) return -1;
    if (mask_kind < OR_DENSE || mask_kind > OR_BLOCK_DIAG) return -1;
    if (mask_kind == OR_BLOCK_DIAG && (bs <= 0 || (L > 0 && L % bs != 0))) return -1;
    double *s = malloc(sizeof(double) * (L > 0 ? L : 1));
    if (!s) return -1;
    for (long bh = 0; bh < B * H; ++bh) {
        const size_t base = (size_t)bh * L * D;
        for (long i = 0; i < L; ++i)
            one_row(q + base, k + base, v + base, L, D, i, mask_kind, bs, sm_scale, s,
                    O + base + i * D, lse + bh * L + i);
    }
    free(s);
    return 0;
}
