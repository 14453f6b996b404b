/*
 * oracle.c -- plain single-threaded CPU definition of the k-quant prefill
 * matmul.  TEST INFRASTRUCTURE ONLY (see oracle.h): tests, the smoke check
 * and the benchmark's CPU-baseline leg use it; the product path never does.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC
 * (no FMA contraction, IEEE division: the quantizer's rounding decisions
 * must be the ones the definition states).
 *
 * Nothing here is blocked, fused or reordered beyond the definition: the GEMM
 * evaluates, for each output (m, n) and each superblock b in ascending order,
 * the per-superblock contribution c_b in block-integer form.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>
#include <stdlib.h>

double oracle_half_to_double(uint16_t h)
{
    /* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
     * bits.  Exact in double. */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }

/* ---------------------------------------------------------------- Q4_K --
 * Byte layout (144 B; GGUF reading):
 *   [0,2)    d     fp16
 *   [2,4)    dmin  fp16
 *   [4,16)   scales[12]: 8 six-bit sub-scales sc_j and 8 six-bit sub-mins m_j
 *            j < 4 : sc_j = s[j] & 63,            m_j = s[j+4] & 63
 *            j >= 4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4
 *                    m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 *   [16,144) qs[128]: for chunk c = 0..3 and l = 0..31, byte qs[32c+l] holds
 *            weight 64c+l in its low nibble and weight 64c+32+l in its high
 *            nibble.  Weight i belongs to sub-block i/32.
 */
void oracle_q4k_fields(const uint8_t *blk, double *d, double *dmin,
                       int sc[8], int mn[8], int q[256])
{
    const uint8_t *s = blk + 4;
    const uint8_t *qs = blk + 16;
    *d = oracle_half_to_double(rd16(blk));
    *dmin = oracle_half_to_double(rd16(blk + 2));
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        mn[j] = s[j + 4] & 63;
    }
    for (int j = 4; j < 8; ++j) {
        sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l) {
            q[64 * c + l] = qs[32 * c + l] & 15;
            q[64 * c + 32 + l] = qs[32 * c + l] >> 4;
        }
}

void oracle_q4k_pack(uint16_t d_bits, uint16_t dmin_bits, const int sc[8],
                     const int mn[8], const int q[256], uint8_t *blk)
{
    uint8_t *s = blk + 4;
    uint8_t *qs = blk + 16;
    wr16(blk, d_bits);
    wr16(blk + 2, dmin_bits);
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
    }
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            qs[32 * c + l] = (uint8_t)((q[64 * c + l] & 15) | ((q[64 * c + 32 + l] & 15) << 4));
}

/* ---------------------------------------------------------------- Q6_K --
 * Byte layout (210 B; GGUF reading):
 *   [0,128)   ql[128]  low 4 bits of each quant
 *   [128,192) qh[64]   high 2 bits of each quant
 *   [192,208) scales[16] int8, one per sub-block of 16 weights
 *   [208,210) d fp16
 * For half h = 0,1 (weights 128h .. 128h+127), with L = ql + 64h,
 * H = qh + 32h and l = 0..31:
 *   q[128h+l]    = (L[l]    & 15) | ((H[l] >> 0) & 3) << 4
 *   q[128h+l+32] = (L[l+32] & 15) | ((H[l] >> 2) & 3) << 4
 *   q[128h+l+64] = (L[l]    >> 4) | ((H[l] >> 4) & 3) << 4
 *   q[128h+l+96] = (L[l+32] >> 4) | ((H[l] >> 6) & 3) << 4
 * Weight i belongs to sub-block i/16.
 */
void oracle_q6k_fields(const uint8_t *blk, double *d, int sc[16], int q[256])
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *s = (const int8_t *)(blk + 192);
    *d = oracle_half_to_double(rd16(blk + 208));
    for (int j = 0; j < 16; ++j)
        sc[j] = s[j];
    for (int h = 0; h < 2; ++h) {
        const uint8_t *L = ql + 64 * h;
        const uint8_t *H = qh + 32 * h;
        int *o = q + 128 * h;
        for (int l = 0; l < 32; ++l) {
            o[l] = (L[l] & 15) | (((H[l] >> 0) & 3) << 4);
            o[l + 32] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);
            o[l + 64] = (L[l] >> 4) | (((H[l] >> 4) & 3) << 4);
            o[l + 96] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
        }
    }
}

void oracle_q6k_pack(uint16_t d_bits, const int sc[16], const int q[256],
                     uint8_t *blk)
{
    uint8_t *ql = blk;
    uint8_t *qh = blk + 128;
    for (int j = 0; j < 16; ++j)
        blk[192 + j] = (uint8_t)(int8_t)sc[j];
    wr16(blk + 208, d_bits);
    for (int h = 0; h < 2; ++h) {
        uint8_t *L = ql + 64 * h;
        uint8_t *H = qh + 32 * h;
        const int *o = q + 128 * h;
        for (int l = 0; l < 32; ++l) {
            L[l] = (uint8_t)((o[l] & 15) | ((o[l + 64] & 15) << 4));
            L[l + 32] = (uint8_t)((o[l + 32] & 15) | ((o[l + 96] & 15) << 4));
            H[l] = (uint8_t)(((o[l] >> 4) & 3) | (((o[l + 32] >> 4) & 3) << 2) |
                             (((o[l + 64] >> 4) & 3) << 4) | (((o[l + 96] >> 4) & 3) << 6));
        }
    }
}

void oracle_dequant_q4k(const uint8_t *blk, double w[256])
{
    double d, dmin;
    int sc[8], mn[8], q[256];
    oracle_q4k_fields(blk, &d, &dmin, sc, mn, q);
    for (int i = 0; i < 256; ++i)
        w[i] = d * sc[i / 32] * q[i] - dmin * mn[i / 32];
}

void oracle_dequant_q6k(const uint8_t *blk, double w[256])
{
    double d;
    int sc[16], q[256];
    oracle_q6k_fields(blk, &d, sc, q);
    for (int i = 0; i < 256; ++i)
        w[i] = d * sc[i / 16] * (q[i] - 32);
}

/* ---------------------------------------------------------------- Q8_K --
 * Per 256-element chunk of a row:
 *   amax = max |x_i| (fp32, exact);
 *   d = amax / 127 (fp32, correctly rounded division);
 *   d == 0 (amax == 0, or amax/127 underflowing to zero) -> every q = 0,
 *              every bsum = 0 (the pages leave this case open; x/0 has no
 *              value, so the chunk is taken as all zeros);
 *   otherwise  q_i = clamp(roundf(x_i / d), -127, 127), x_i / d again a
 *              correctly rounded fp32 division and roundf rounding halves
 *              away from zero;
 *   bsums[g] = sum of q_{16g .. 16g+15}.
 */
/* ---- PTQ1_0: 24 qs bytes (5 trits each), 2 qh bytes (4 trits each), fp16 d */
static int ptq1_digit(int byte, int i)
{
    int v = byte;
    for (int k = 0; k < i; ++k)
        v /= 3;
    return v % 3;
}

void oracle_ptq1_fields(const uint8_t *blk, double *d, int t[128])
{
    for (int k = 0; k < 120; ++k)
        t[k] = ptq1_digit(blk[k % 24], k / 24);
    for (int r = 0; r < 8; ++r)
        t[120 + r] = ptq1_digit(blk[24 + r % 2], r / 2);
    *d = oracle_half_to_double(rd16(blk + 26));
}

void oracle_ptq1_pack(uint16_t d_bits, const int t[128], uint8_t *blk)
{
    for (int j = 0; j < 24; ++j) {
        int v = 0;
        for (int i = 4; i >= 0; --i)
            v = 3 * v + t[24 * i + j];
        blk[j] = (uint8_t)v;
    }
    for (int h = 0; h < 2; ++h) {
        int v = 0;
        for (int i = 3; i >= 0; --i)
            v = 3 * v + t[120 + 2 * i + h];
        blk[24 + h] = (uint8_t)v;
    }
    wr16(blk + 26, d_bits);
}

void oracle_dequant_ptq1(const uint8_t *blk, double w[128])
{
    double d;
    int t[128];
    oracle_ptq1_fields(blk, &d, t);
    for (int k = 0; k < 128; ++k)
        w[k] = d * (double)(t[k] - 1);
}

void oracle_gemm_ptq1(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                      const int8_t *qs, const float *dx, int64_t M, const int64_t *rows, int64_t nrows,
                      double *y, double *absc)
{
    int64_t nb = K / 256;
    int64_t *own = NULL;
    if (!rows) {
        own = (int64_t *)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
        for (int64_t i = 0; i < M; ++i)
            own[i] = i;
        rows = own;
        nrows = M;
    }
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t n = 0; n < N; ++n) {
            y[r * N + n] = 0.0;
            if (absc)
                absc[r * N + n] = 0.0;
        }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            double d[2];
            int t[2][128];
            for (int h = 0; h < 2; ++h)
                oracle_ptq1_fields(w + n * ldw + (2 * b + h) * ORACLE_PTQ1_BYTES, &d[h], t[h]);
            for (int64_t r = 0; r < nrows; ++r) {
                const int8_t *xq = qs + rows[r] * K + b * 256;
                int64_t I[2] = {0, 0};
                for (int h = 0; h < 2; ++h)
                    for (int k = 0; k < 128; ++k)
                        I[h] += (int64_t)(t[h][k] - 1) * xq[128 * h + k];
                double cb = (double)dx[rows[r] * nb + b] * (d[0] * (double)I[0] + d[1] * (double)I[1]);
                y[r * N + n] += cb;
                if (absc)
                    absc[r * N + n] += fabs(cb);
            }
        }
    free(own);
}

void oracle_quantize_q8k(const float *x, int64_t M, int64_t K, int64_t ldx,
                         int8_t *qs, float *d, int16_t *bsums)
{
    int64_t nb = K / 256;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + m * ldx + b * 256;
            int8_t *qb = qs + m * K + b * 256;
            int16_t *sb = bsums + m * (K / 16) + b * 16;
            float amax = 0.0f;
            for (int i = 0; i < 256; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax)
                    amax = a;
            }
            float db = amax / 127.0f;
            if (db == 0.0f) {
                /* amax == 0, or amax so small that amax/127 underflows to
                 * zero: x/d is undefined, the chunk quantizes to zero. */
                d[m * nb + b] = 0.0f;
                memset(qb, 0, 256);
                memset(sb, 0, 16 * sizeof(int16_t));
                continue;
            }
            d[m * nb + b] = db;
            for (int i = 0; i < 256; ++i) {
                float r = roundf(xb[i] / db);
                if (r > 127.0f)
                    r = 127.0f;
                if (r < -127.0f)
                    r = -127.0f;
                qb[i] = (int8_t)r;
            }
            for (int g = 0; g < 16; ++g) {
                int s = 0;
                for (int i = 0; i < 16; ++i)
                    s += qb[16 * g + i];
                sb[g] = (int16_t)s;
            }
        }
    }
}

void oracle_q8k_to_aos(const int8_t *qs, const float *d, const int16_t *bsums,
                       int64_t M, int64_t K, uint8_t *aos)
{
    int64_t nb = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            uint8_t *o = aos + (m * nb + b) * ORACLE_Q8K_BYTES;
            memcpy(o, &d[m * nb + b], 4);
            memcpy(o + 4, qs + m * K + b * 256, 256);
            memcpy(o + 260, bsums + m * (K / 16) + b * 16, 32);
        }
}

void oracle_q8k_from_aos(const uint8_t *aos, int64_t M, int64_t K, int8_t *qs,
                         float *d, int16_t *bsums)
{
    int64_t nb = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *o = aos + (m * nb + b) * ORACLE_Q8K_BYTES;
            memcpy(&d[m * nb + b], o, 4);
            memcpy(qs + m * K + b * 256, o + 4, 256);
            memcpy(bsums + m * (K / 16) + b * 16, o + 260, 32);
        }
}

/* ---------------------------------------------------------------- GEMM --
 * Y[m][n] = sum_b c_b with, for superblock b of weight row n and token m,
 *   Q4_K: c_b = dx[m,b] * ( d * sum_j sc_j * I_j  -  dmin * sum_j m_j * B_j )
 *         I_j = sum_{i in sub-block j} q_i * qx_i   (exact integer)
 *         B_j = bsums[2j] + bsums[2j+1]             (sum of qx over j)
 *   Q6_K: c_b = dx[m,b] * d * sum_j sc_j * ( I_j - 32 * bsums[j] )
 *         I_j over the unsigned 6-bit q (0..63); equal to using q-32.
 * The integer parts are exact; scale products and the sum over b are fp64.
 */
static int64_t *all_rows(int64_t M)
{
    int64_t *r = (int64_t *)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
    for (int64_t i = 0; i < M; ++i)
        r[i] = i;
    return r;
}

void oracle_gemm_q4k(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                     const int8_t *qs, const float *dx, const int16_t *bsums,
                     int64_t M, const int64_t *rows, int64_t nrows,
                     double *y, double *absc)
{
    int64_t nb = K / 256;
    int64_t *own = NULL;
    if (!rows) {
        own = all_rows(M);
        rows = own;
        nrows = M;
    }
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t n = 0; n < N; ++n) {
            y[r * N + n] = 0.0;
            if (absc)
                absc[r * N + n] = 0.0;
        }
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            double d, dmin;
            int sc[8], mn[8], q[256];
            oracle_q4k_fields(w + n * ldw + b * ORACLE_Q4K_BYTES, &d, &dmin, sc, mn, q);
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t m = rows[r];
                const int8_t *xq = qs + m * K + b * 256;
                const int16_t *bs = bsums + m * (K / 16) + b * 16;
                int64_t dot = 0, corr = 0;
                for (int j = 0; j < 8; ++j) {
                    int64_t I = 0;
                    for (int i = 32 * j; i < 32 * j + 32; ++i)
                        I += (int64_t)q[i] * xq[i];
                    dot += (int64_t)sc[j] * I;
                    corr += (int64_t)mn[j] * (bs[2 * j] + bs[2 * j + 1]);
                }
                double cb = (double)dx[m * nb + b] * (d * (double)dot - dmin * (double)corr);
                y[r * N + n] += cb;
                if (absc)
                    absc[r * N + n] += fabs(cb);
            }
        }
    }
    free(own);
}

void oracle_gemm_q6k(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                     const int8_t *qs, const float *dx, const int16_t *bsums,
                     int64_t M, const int64_t *rows, int64_t nrows,
                     double *y, double *absc)
{
    int64_t nb = K / 256;
    int64_t *own = NULL;
    if (!rows) {
        own = all_rows(M);
        rows = own;
        nrows = M;
    }
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t n = 0; n < N; ++n) {
            y[r * N + n] = 0.0;
            if (absc)
                absc[r * N + n] = 0.0;
        }
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            double d;
            int sc[16], q[256];
            oracle_q6k_fields(w + n * ldw + b * ORACLE_Q6K_BYTES, &d, sc, q);
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t m = rows[r];
                const int8_t *xq = qs + m * K + b * 256;
                const int16_t *bs = bsums + m * (K / 16) + b * 16;
                int64_t dot = 0;
                for (int j = 0; j < 16; ++j) {
                    int64_t I = 0;
                    for (int i = 16 * j; i < 16 * j + 16; ++i)
                        I += (int64_t)q[i] * xq[i];
                    dot += (int64_t)sc[j] * (I - 32 * (int64_t)bs[j]);
                }
                double cb = (double)dx[m * nb + b] * d * (double)dot;
                y[r * N + n] += cb;
                if (absc)
                    absc[r * N + n] += fabs(cb);
            }
        }
    }
    free(own);
}

void oracle_gemm_id(int type, const uint8_t *w, int64_t E, int64_t N, int64_t K, int64_t ldw,
                    const int8_t *qs, const float *dx, const int16_t *bsums, int64_t M,
                    const int32_t *ids, int64_t top_k, double *y, double *absc)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t s = 0; s < top_k; ++s) {
            const int64_t pair = m * top_k + s;
            const int64_t e = ids[pair];
            if (e < 0 || e >= E)
                continue;
            /* expert e's rows, token m only */
            const uint8_t *we = w + e * N * ldw;
            double *yr = y + pair * N;
            double *ar = absc ? absc + pair * N : NULL;
            if (type == 4)
                oracle_gemm_q4k(we, N, K, ldw, qs, dx, bsums, M, &m, 1, yr, ar);
            else
                oracle_gemm_q6k(we, N, K, ldw, qs, dx, bsums, M, &m, 1, yr, ar);
        }
}

void oracle_epilogue(double *y, int64_t R, int64_t N, const float *bias, int act)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t n = 0; n < N; ++n) {
            double v = y[r * N + n] + (bias ? (double)bias[n] : 0.0);
            if (act == 1)
                v = v > 0.0 ? v : 0.0;
            else if (act == 2)
                v = v / (1.0 + exp(-v));
            else if (act == 3)
                v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
            y[r * N + n] = v;
        }
}

void oracle_brute(int type, const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                  const int8_t *qs, const float *dx, int64_t M, double *y)
{
    int64_t nb = K / 256;
    double *wd = (double *)malloc((size_t)K * sizeof(double));
    double *xd = (double *)malloc((size_t)(M * K) * sizeof(double));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            xd[m * K + k] = (double)dx[m * nb + k / 256] * (double)qs[m * K + k];
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            if (type == 1) {   /* PTQ1_0: two 128-weight blocks per 256 */
                oracle_dequant_ptq1(w + n * ldw + (2 * b) * ORACLE_PTQ1_BYTES, wd + b * 256);
                oracle_dequant_ptq1(w + n * ldw + (2 * b + 1) * ORACLE_PTQ1_BYTES, wd + b * 256 + 128);
                continue;
            }
            const uint8_t *blk = w + n * ldw + b * (type == 4 ? ORACLE_Q4K_BYTES : ORACLE_Q6K_BYTES);
            if (type == 4)
                oracle_dequant_q4k(blk, wd + b * 256);
            else
                oracle_dequant_q6k(blk, wd + b * 256);
        }
        for (int64_t m = 0; m < M; ++m) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += wd[k] * xd[m * K + k];
            y[m * N + n] = s;
        }
    }
    free(wd);
    free(xd);
}
