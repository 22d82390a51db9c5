/*
 * fp64 CPU oracle for frozen-prefix chunk attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (one window, one KV head and the g query heads that read
 * it), written out as the plain definition, with no tiling or online softmax:
 *
 *   The chunk's queries attend to the frozen prefix, which the walk reads as
 *   constants ("train: walk the window", "What it is"), plus the chunk's own
 *   causal keys.  Chunk row t sits at absolute position Lp + t, so it sees
 *   every prefix key and chunk keys j <= t (bottom-right causal mask).
 *
 *     S_tj   = scale * q_t . k_j                     j visible to t
 *     LSE_t  = ln sum_j exp(S_tj)
 *     P_tj   = exp(S_tj - LSE_t)
 *     O_t    = sum_j P_tj v_j
 *
 *   Backward for the loss L = sum <O, dO>, gradients stopped at the prefix
 *   ("Context-Frozen Training", "Phase 2"; "train: walk the window", "Why it's
 *   a draft": cached prefixes are stop-gradient constants), i.e. the
 *   query-split attention backward that the prime-rl POC lists under "Known
 *   gaps":
 *
 *     delta_t = dO_t . O_t
 *     dP_tj   = dO_t . v_j
 *     dS_tj   = P_tj (dP_tj - delta_t)
 *     dQ_t    = scale * sum_{j visible} dS_tj k_j          (prefix and chunk keys)
 *     dK_c,j  = scale * sum_{h in group} sum_{t >= j} dS_tj q_t   (chunk keys only)
 *     dV_c,j  =         sum_{h in group} sum_{t >= j} P_tj dO_t    (chunk keys only)
 *
 *   The prefix gets no gradient from cfa_oracle_group; the horizon
 *   extension below (cfa_oracle_group_prefix_grad) gives the exact one for the
 *   rows a caller keeps.
 *
 * q8_0 (the llama.cpp cache type named in "train: walk the window"): a block
 * is a little-endian IEEE binary16 scale d followed by 32 signed 8-bit codes;
 * value i is d * q_i.  The fp32 value fp32(d)*q_i is exact (11 x 8 significant
 * bits); the bf16 that a kernel multiplies with is that value rounded to
 * nearest, ties to even.  The attention itself uses the exact values.
 *
 * This file is the plain definition and nothing else.  The tests that check
 * that the pins catch mistakes compile copies of it with a mistake planted by
 * a textual edit (tests/oracle_mutants.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats, from their definitions ---------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                    /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);        /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a finite fp32 value to bf16 (keep the top 16 bits), nearest, ties to
 * even.  Operates on the bit pattern: add 0x7fff plus the lowest kept bit,
 * then truncate.  Used only on finite values. */
static uint16_t float_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/*
 * Dequantise n_blocks q8_0 blocks (34 bytes each, contiguous).
 * out_f64 / out_f32 / out_bf16 may each be NULL; each receives 32 values per
 * block in order.
 */
void cfa_oracle_dequant_q8_0(const uint8_t *blocks, long n_blocks, double *out_f64,
                             float *out_f32, uint16_t *out_bf16)
{
    for (long b = 0; b < n_blocks; ++b) {
        const uint8_t *blk = blocks + 34 * b;
        uint16_t hbits = (uint16_t)(blk[0] | (blk[1] << 8));
        double d = half_bits_to_double(hbits);
        for (int i = 0; i < 32; ++i) {
            int qi = (int)(int8_t)blk[2 + i];
            double v = d * (double)qi;                 /* exact in double */
            long k = 32 * b + i;
            if (out_f64) out_f64[k] = v;
            if (out_f32) out_f32[k] = (float)v;         /* exact: v fits fp32 */
            if (out_bf16) out_bf16[k] = float_to_bf16_rne((float)v);
        }
    }
}

/* fp32 -> IEEE 754 binary16 bits, round to nearest, ties to even, from the
 * format's definition: |x| = (1 + m/1024) * 2^(e-15) for biased exponent e in
 * [1, 30], m/1024 * 2^-14 for e = 0; magnitudes from 65520 up (halfway past
 * the largest finite value, 65504, whose fraction is odd) become infinity.
 * The scaled magnitudes below are exact in double; rint rounds them to the
 * nearest integer, ties to even (the default rounding mode). */
static uint16_t float_to_half_rne(float x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double v = fabs((double)x);
    if (v == 0.0) return sign;
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    int k;
    frexp(v, &k);                   /* v = f * 2^k, f in [0.5, 1): v in [2^(k-1), 2^k) */
    int E = k - 1;                  /* unbiased exponent of v */
    if (E < -14) {                  /* subnormal: a multiple of 2^-24 */
        const double m = rint(ldexp(v, 24));
        return (uint16_t)(sign | (uint16_t)m);       /* m = 1024 is the smallest normal */
    }
    double m = rint(ldexp(v, 10 - E));               /* in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        ++E;
    }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/*
 * Quantise n_blocks blocks of 32 bf16 values (given as bit patterns) to q8_0,
 * the cache write of the walk ("train: walk the window": the chunk's keys and
 * values go into the q8_0 cache for the next chunk).  Per block, in fp32:
 * d = absmax / 127 (an all-zero block gets d = 0 and zero codes), code
 * q_i = x_i / d rounded half away from zero, clamped to [-127, 127]; the
 * stored scale is fp16(d), nearest even, little-endian.
 */
void cfa_oracle_quantize_q8_0(const uint16_t *x_bf16, long n_blocks, uint8_t *out)
{
    for (long b = 0; b < n_blocks; ++b) {
        float v[32];
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            const uint32_t u = (uint32_t)x_bf16[32 * b + i] << 16;   /* bf16 -> fp32, exact */
            memcpy(&v[i], &u, 4);
            const float a = fabsf(v[i]);
            amax = a > amax ? a : amax;
        }
        const float d = amax / 127.0f;
        const uint16_t dh = float_to_half_rne(d);
        uint8_t *blk = out + 34 * b;
        blk[0] = (uint8_t)(dh & 0xff);
        blk[1] = (uint8_t)(dh >> 8);
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (d > 0.0f) {
                const float r = v[i] / d;
                q = (int)roundf(r);
                q = q > 127 ? 127 : (q < -127 ? -127 : q);
            }
            blk[2 + i] = (uint8_t)(int8_t)q;
        }
    }
}

/* ---- attention ---------------------------------------------------------- */

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/*
 * One window, one KV head, its g query heads.
 *   q, dout : [lc][g][d]      kp, vp : [lp][d]      kc, vc : [lc][d]
 *   o, dq   : [lc][g][d]      lse, delta : [g][lc]  dkc, dvc : [lc][d]
 * Any output pointer may be NULL except that the backward needs o/lse/delta
 * internally (allocated here when NULL).  Returns 0, or -1 on allocation
 * failure.
 */
int cfa_oracle_group(int lp, int lc, int g, int d, double scale,
                     const double *q, const double *kp, const double *vp,
                     const double *kc, const double *vc, const double *dout,
                     double *o, double *lse, double *delta,
                     double *dq, double *dkc, double *dvc)
{
    const int nrow = lc * g;
    double *o_own = NULL, *lse_own = NULL, *delta_own = NULL;
    if (!o) o = o_own = (double *)malloc(sizeof(double) * (size_t)nrow * d + 8);
    if (!lse) lse = lse_own = (double *)malloc(sizeof(double) * (size_t)nrow + 8);
    if (!delta) delta = delta_own = (double *)malloc(sizeof(double) * (size_t)nrow + 8);
    if (!o || !lse || !delta) {
        free(o_own); free(lse_own); free(delta_own);
        return -1;
    }
    int fail = 0;

    /* Pass 1, one query row at a time: S, LSE, P, O, delta and dQ. */
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * ((size_t)lp + lc + 1));
        double *P = (double *)malloc(sizeof(double) * ((size_t)lp + lc + 1));
        if (!S || !P) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < nrow; ++r) {
            if (!S || !P) continue;
            const int t = r / g, hh = r % g;
            const double *qt = q + (size_t)r * d;
            const double *dot_ = dout + (size_t)r * d;
            const int nc = t + 1;                 /* visible chunk keys: j <= t */
            const int n = lp + nc;
            for (int j = 0; j < lp; ++j) S[j] = scale * dot(qt, kp + (size_t)j * d, d);
            for (int j = 0; j < nc; ++j) S[lp + j] = scale * dot(qt, kc + (size_t)j * d, d);
            double m = -INFINITY;
            for (int j = 0; j < n; ++j) m = S[j] > m ? S[j] : m;
            double sum = 0.0;
            for (int j = 0; j < n; ++j) sum += exp(S[j] - m);
            const double L = m + log(sum);
            lse[(size_t)hh * lc + t] = L;
            for (int j = 0; j < n; ++j) P[j] = exp(S[j] - L);
            double *ot = o + (size_t)r * d;
            for (int c = 0; c < d; ++c) ot[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                const double *vj = j < lp ? vp + (size_t)j * d : vc + (size_t)(j - lp) * d;
                for (int c = 0; c < d; ++c) ot[c] += P[j] * vj[c];
            }
            const double dl = dot(dot_, ot, d);
            delta[(size_t)hh * lc + t] = dl;
            if (dq) {
                double *dqt = dq + (size_t)r * d;
                for (int c = 0; c < d; ++c) dqt[c] = 0.0;
                for (int j = 0; j < n; ++j) {
                    const double *vj = j < lp ? vp + (size_t)j * d : vc + (size_t)(j - lp) * d;
                    const double *kj = j < lp ? kp + (size_t)j * d : kc + (size_t)(j - lp) * d;
                    const double dpj = dot(dot_, vj, d);
                    const double dsj = P[j] * (dpj - dl);
                    const double f = scale * dsj;
                    for (int c = 0; c < d; ++c) dqt[c] += f * kj[c];
                }
            }
        }
        free(S);
        free(P);
    }

    /* Pass 2, one chunk key at a time: dK_c and dV_c, summed over the group. */
    if (!fail && (dkc || dvc)) {
#pragma omp parallel for schedule(dynamic, 4)
        for (int j = 0; j < lc; ++j) {
            const double *kj = kc + (size_t)j * d, *vj = vc + (size_t)j * d;
            double *dk = dkc ? dkc + (size_t)j * d : NULL;
            double *dv = dvc ? dvc + (size_t)j * d : NULL;
            if (dk) for (int c = 0; c < d; ++c) dk[c] = 0.0;
            if (dv) for (int c = 0; c < d; ++c) dv[c] = 0.0;
            for (int t = j; t < lc; ++t) {
                for (int hh = 0; hh < g; ++hh) {      /* the group's query heads */
                    const int r = t * g + hh;
                    const double *qt = q + (size_t)r * d;
                    const double *dot_ = dout + (size_t)r * d;
                    const double s = scale * dot(qt, kj, d);
                    const double p = exp(s - lse[(size_t)hh * lc + t]);
                    const double dp = dot(dot_, vj, d);
                    const double ds = p * (dp - delta[(size_t)hh * lc + t]);
                    const double fk = scale * ds;
                    if (dk) for (int c = 0; c < d; ++c) dk[c] += fk * qt[c];
                    if (dv) for (int c = 0; c < d; ++c) dv[c] += p * dot_[c];
                }
            }
        }
    }

    free(o_own);
    free(lse_own);
    free(delta_own);
    return fail ? -1 : 0;
}

/*
 * Gradients of the frozen prefix's keys and values under the same loss, for
 * the "exact reverse pass with horizon H" that "train: walk the window" ("Why
 * it's a draft") asks for, and for the full k/v backward on context rows of
 * the prime-rl POC ("Mechanism"): every chunk row sees every prefix key, so
 * for prefix key j
 *
 *     dK_p,j = scale * sum_{h in group} sum_{t < Lc} dS_tj q_t
 *     dV_p,j =         sum_{h in group} sum_{t < Lc} P_tj dO_t
 *
 * with P_tj = exp(S_tj - LSE_t) and dS_tj = P_tj (dO_t . v_j - delta_t), LSE
 * and delta as cfa_oracle_group returns them.  Which prefix rows receive a
 * gradient (the horizon) is the caller's choice; this returns all of them.
 *   q, dout : [lc][g][d]   kp, vp, dkp, dvp : [lp][d]   lse, delta : [g][lc]
 */
void cfa_oracle_group_prefix_grad(int lp, int lc, int g, int d, double scale,
                                  const double *q, const double *kp, const double *vp,
                                  const double *dout, const double *lse,
                                  const double *delta, double *dkp, double *dvp)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int j = 0; j < lp; ++j) {
        const double *kj = kp + (size_t)j * d, *vj = vp + (size_t)j * d;
        double *dkr = dkp + (size_t)j * d, *dvr = dvp + (size_t)j * d;
        for (int c = 0; c < d; ++c) dkr[c] = dvr[c] = 0.0;
        for (int t = 0; t < lc; ++t) {
            for (int hh = 0; hh < g; ++hh) {      /* every query head of the group */
                const int r = t * g + hh;
                const double *qt = q + (size_t)r * d;
                const double *dot_ = dout + (size_t)r * d;
                const double p = exp(scale * dot(qt, kj, d) - lse[(size_t)hh * lc + t]);
                const double ds = p * (dot(dot_, vj, d) - delta[(size_t)hh * lc + t]);
                const double fkp = scale * ds;
                for (int c = 0; c < d; ++c) dkr[c] += fkp * qt[c];
                for (int c = 0; c < d; ++c) dvr[c] += p * dot_[c];
            }
        }
    }
}

/* Number of threads the parallel regions above use. */
int cfa_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
