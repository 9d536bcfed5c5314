/*
 * kq_oracle.c -- plain, slow, fp64 reference for k-quant decoding and products.
 *
 * TEST INFRASTRUCTURE ONLY (see kq_oracle.h): used by the tests, the smoke
 * check and the benchmark's CPU-baseline leg; never by the product library.
 * No blocking, fusion or reordering: each function is the definition written
 * out as loops, in the order the format is described.
 */
#include "kq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_block_bytes(int type)
{
    switch (type) {
    case ORACLE_Q4_K: return 2 + 2 + 12 + 128;       /* d, dmin, scales, qs     */
    case ORACLE_Q5_K: return 2 + 2 + 12 + 32 + 128;  /* d, dmin, scales, qh, qs */
    case ORACLE_Q6_K: return 128 + 64 + 16 + 2;      /* ql, qh, scales, d       */
    case ORACLE_IA4: return 8 + 8 + 128;             /* scales, biases, codes   */
    default: return 0;
    }
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0 -> subnormal (or zero): (-1)^s * 2^-14 * f/1024
 * exponent 31 -> infinity (f == 0) or NaN
 * otherwise   -> (-1)^s * 2^(e-15) * (1 + f/1024) */
double oracle_half_to_double(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(1024.0 + (double)f, e - 25);
    return s ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32 pattern. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }

/* 8 six-bit scales and 8 six-bit mins in 12 bytes s[0..11]:
 *   j < 4 : sc_j = low 6 bits of s[j],   m_j = low 6 bits of s[j+4]
 *   j >= 4: low 4 bits of sc_j / m_j are the low / high nibble of s[j+4];
 *           their top 2 bits are the top 2 bits of s[j-4] / s[j]. */
static void unpack_scale_min_6bit(const uint8_t *s, int sc[8], int m[8])
{
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        m[j] = s[j + 4] & 63;
    }
    for (int j = 4; j < 8; ++j) {
        sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        m[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

static void pack_scale_min_6bit(const int sc[8], const int m[8], uint8_t *s)
{
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | (((sc[j + 4] >> 4) & 3) << 6));
        s[j + 4] = (uint8_t)((m[j] & 63) | (((m[j + 4] >> 4) & 3) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
}

int oracle_unpack(int type, const uint8_t *blk, oracle_fields *f)
{
    memset(f, 0, sizeof(*f));
    if (type == ORACLE_Q4_K || type == ORACLE_Q5_K) {
        const uint8_t *scales = blk + 4;
        const uint8_t *qh = blk + 16;                       /* Q5_K only */
        const uint8_t *qs = blk + (type == ORACLE_Q4_K ? 16 : 48);
        f->d_bits = rd16(blk);
        f->dmin_bits = rd16(blk + 2);
        unpack_scale_min_6bit(scales, f->sc, f->m);
        /* chunk g of 32 bytes: low nibbles are weights 64g..64g+31 (sub-block
         * 2g), high nibbles are weights 64g+32..64g+63 (sub-block 2g+1).
         * Q5_K: the 5th bit of weight 64g+l is bit 2g of qh[l], of weight
         * 64g+32+l bit 2g+1 of qh[l]. */
        for (int g = 0; g < 4; ++g) {
            for (int l = 0; l < 32; ++l) {
                int lo = qs[32 * g + l] & 15;
                int hi = qs[32 * g + l] >> 4;
                if (type == ORACLE_Q5_K) {
                    lo |= ((qh[l] >> (2 * g)) & 1) << 4;
                    hi |= ((qh[l] >> (2 * g + 1)) & 1) << 4;
                }
                f->q[64 * g + l] = lo;
                f->q[64 * g + 32 + l] = hi;
            }
        }
        return 0;
    }
    if (type == ORACLE_Q6_K) {
        const uint8_t *ql = blk;
        const uint8_t *qh = blk + 128;
        const int8_t *sc = (const int8_t *)(blk + 192);
        f->d_bits = rd16(blk + 208);
        for (int i = 0; i < 16; ++i) f->sc[i] = sc[i];
        /* half h of 128 weights: ql[64h+l] holds the low 4 bits of weights
         * 128h+l (low nibble) and 128h+64+l (high nibble); ql[64h+32+l] those
         * of 128h+32+l and 128h+96+l; qh[32h+l] holds their top 2 bits in bit
         * pairs 0-1, 2-3, 4-5, 6-7 for weights 128h+l, +32, +64, +96. */
        for (int h = 0; h < 2; ++h) {
            for (int l = 0; l < 32; ++l) {
                int a = ql[64 * h + l], b = ql[64 * h + 32 + l], c = qh[32 * h + l];
                f->q[128 * h + l] = (a & 15) | (((c >> 0) & 3) << 4);
                f->q[128 * h + 32 + l] = (b & 15) | (((c >> 2) & 3) << 4);
                f->q[128 * h + 64 + l] = (a >> 4) | (((c >> 4) & 3) << 4);
                f->q[128 * h + 96 + l] = (b >> 4) | (((c >> 6) & 3) << 4);
            }
        }
        return 0;
    }
    return -1;
}

int oracle_pack(int type, const oracle_fields *f, uint8_t *blk)
{
    int nbytes = oracle_block_bytes(type);
    if (!nbytes) return -1;
    memset(blk, 0, (size_t)nbytes);
    if (type == ORACLE_Q4_K || type == ORACLE_Q5_K) {
        uint8_t *qh = blk + 16;
        uint8_t *qs = blk + (type == ORACLE_Q4_K ? 16 : 48);
        wr16(blk, f->d_bits);
        wr16(blk + 2, f->dmin_bits);
        pack_scale_min_6bit(f->sc, f->m, blk + 4);
        for (int g = 0; g < 4; ++g) {
            for (int l = 0; l < 32; ++l) {
                int lo = f->q[64 * g + l], hi = f->q[64 * g + 32 + l];
                qs[32 * g + l] = (uint8_t)((lo & 15) | ((hi & 15) << 4));
                if (type == ORACLE_Q5_K) {
                    qh[l] |= (uint8_t)(((lo >> 4) & 1) << (2 * g));
                    qh[l] |= (uint8_t)(((hi >> 4) & 1) << (2 * g + 1));
                }
            }
        }
        return 0;
    }
    /* Q6_K */
    for (int h = 0; h < 2; ++h) {
        for (int l = 0; l < 32; ++l) {
            int q1 = f->q[128 * h + l], q2 = f->q[128 * h + 32 + l];
            int q3 = f->q[128 * h + 64 + l], q4 = f->q[128 * h + 96 + l];
            blk[64 * h + l] = (uint8_t)((q1 & 15) | ((q3 & 15) << 4));
            blk[64 * h + 32 + l] = (uint8_t)((q2 & 15) | ((q4 & 15) << 4));
            blk[128 + 32 * h + l] = (uint8_t)(((q1 >> 4) & 3) | (((q2 >> 4) & 3) << 2) |
                                              (((q3 >> 4) & 3) << 4) | (((q4 >> 4) & 3) << 6));
        }
    }
    for (int i = 0; i < 16; ++i) blk[192 + i] = (uint8_t)(int8_t)f->sc[i];
    wr16(blk + 208, f->d_bits);
    return 0;
}

int oracle_dequant_block_f64(int type, const uint8_t *blk, double w[256])
{
    if (type == ORACLE_IA4) {
        /* group g = weights 64g..64g+63: scale at bytes 2g, bias at 8+2g (bf16);
         * code byte 16+32g+l holds weight 64g+l (low nibble) and 64g+32+l (high) */
        for (int g = 0; g < 4; ++g) {
            double scale = oracle_bf16_to_double(rd16(blk + 2 * g));
            double bias = oracle_bf16_to_double(rd16(blk + 8 + 2 * g));
            for (int l = 0; l < 32; ++l) {
                int byte = blk[16 + 32 * g + l];
                w[64 * g + l] = scale * (double)(byte & 15) + bias;
                w[64 * g + 32 + l] = scale * (double)(byte >> 4) + bias;
            }
        }
        return 0;
    }
    oracle_fields f;
    if (oracle_unpack(type, blk, &f)) return -1;
    double d = oracle_half_to_double(f.d_bits);
    if (type == ORACLE_Q6_K) {
        for (int i = 0; i < 256; ++i)
            w[i] = d * (double)f.sc[i / 16] * (double)(f.q[i] - 32);
        return 0;
    }
    double dmin = oracle_half_to_double(f.dmin_bits);
    for (int i = 0; i < 256; ++i) {
        int j = i / 32;
        w[i] = d * (double)f.sc[j] * (double)f.q[i] - dmin * (double)f.m[j];
    }
    return 0;
}

int oracle_dequant(int type, const uint8_t *blocks, int64_t n_blocks, float *out)
{
    int nbytes = oracle_block_bytes(type);
    if (!nbytes || n_blocks < 0) return -1;
    double w[256];
    for (int64_t b = 0; b < n_blocks; ++b) {
        oracle_dequant_block_f64(type, blocks + b * nbytes, w);
        for (int i = 0; i < 256; ++i) out[b * 256 + i] = (float)w[i];
    }
    return 0;
}

/* All blocks -> their exact weights in fp64 (the values every product uses). */
int oracle_dequant_f64(int type, const uint8_t *blocks, int64_t n_blocks, double *out)
{
    int nbytes = oracle_block_bytes(type);
    if (!nbytes || n_blocks < 0) return -1;
    for (int64_t b = 0; b < n_blocks; ++b)
        oracle_dequant_block_f64(type, blocks + b * nbytes, out + b * 256);
    return 0;
}

static double x_value(const void *x, int x_dtype, int64_t idx)
{
    if (x_dtype == ORACLE_X_BF16) return oracle_bf16_to_double(((const uint16_t *)x)[idx]);
    return (double)((const float *)x)[idx];
}

/* One output: sum over k < K of w[k] * x[k] for one row of blocks. */
static void row_dot(int type, const uint8_t *row, int64_t K, const void *x, int x_dtype,
                    int64_t x_off, double *y, double *s)
{
    int nbytes = oracle_block_bytes(type);
    int64_t nb = (K + 255) / 256;
    double acc = 0.0, acc_abs = 0.0, w[256];
    for (int64_t b = 0; b < nb; ++b) {
        oracle_dequant_block_f64(type, row + b * nbytes, w);
        for (int i = 0; i < 256; ++i) {
            int64_t k = b * 256 + i;
            if (k >= K) break;
            double t = w[i] * x_value(x, x_dtype, x_off + k);
            acc += t;
            acc_abs += fabs(t);
        }
    }
    *y = acc;
    if (s) *s = acc_abs;
}

int oracle_matvec(int type, const uint8_t *W, int64_t N, int64_t K,
                  const void *x, int x_dtype, int64_t M,
                  double *y, double *s, int n_threads)
{
    int nbytes = oracle_block_bytes(type);
    if (!nbytes || N < 0 || K < 0 || M < 0) return -1;
    if (x_dtype != ORACLE_X_F32 && x_dtype != ORACLE_X_BF16) return -1;
    int64_t row_bytes = ((K + 255) / 256) * nbytes;
    int64_t total = M * N;
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(n_threads)
#endif
    for (int64_t i = 0; i < total; ++i) {
        int64_t m = i / N, n = i % N;
        row_dot(type, W + n * row_bytes, K, x, x_dtype, m * K, &y[i], s ? &s[i] : NULL);
    }
    (void)n_threads;
    return 0;
}

int oracle_moe_matvec(int type, const uint8_t *W_experts, int n_experts,
                      const int32_t *ids, const float *gate,
                      const void *x, int x_dtype, int x_per_slot,
                      int64_t N, int64_t K, int64_t M, int top_k,
                      double *y, double *s, int n_threads)
{
    int nbytes = oracle_block_bytes(type);
    if (!nbytes || N < 0 || K < 0 || M < 0 || top_k < 1 || n_experts < 1) return -1;
    if (x_dtype != ORACLE_X_F32 && x_dtype != ORACLE_X_BF16) return -1;
    for (int64_t i = 0; i < M * top_k; ++i)
        if (ids[i] < 0 || ids[i] >= n_experts) return -2;
    int64_t row_bytes = ((K + 255) / 256) * nbytes;
    int64_t expert_bytes = N * row_bytes;
    /* per-slot products first: p[m][t][n] */
    int64_t total = M * top_k * N;
    double *p = (double *)malloc(sizeof(double) * (size_t)(total ? total : 1));
    double *pa = (double *)malloc(sizeof(double) * (size_t)(total ? total : 1));
    if (!p || !pa) { free(p); free(pa); return -1; }
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(n_threads)
#endif
    for (int64_t i = 0; i < total; ++i) {
        int64_t mt = i / N, n = i % N;          /* mt = m * top_k + t */
        int64_t m = mt / top_k;
        const uint8_t *Wm = W_experts + (int64_t)ids[mt] * expert_bytes;
        int64_t x_off = (x_per_slot ? mt : m) * K;
        row_dot(type, Wm + n * row_bytes, K, x, x_dtype, x_off, &p[i], &pa[i]);
    }
    (void)n_threads;
    if (!gate) {
        memcpy(y, p, sizeof(double) * (size_t)total);
        if (s) memcpy(s, pa, sizeof(double) * (size_t)total);
    } else {
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0, acc_abs = 0.0;
                for (int t = 0; t < top_k; ++t) {
                    double g = (double)gate[m * top_k + t];
                    acc += g * p[(m * top_k + t) * N + n];
                    acc_abs += fabs(g) * pa[(m * top_k + t) * N + n];
                }
                y[m * N + n] = acc;
                if (s) s[m * N + n] = acc_abs;
            }
        }
    }
    free(p);
    free(pa);
    return 0;
}
