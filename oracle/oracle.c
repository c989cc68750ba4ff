/*
 * oracle.c -- fp64 CPU reference (test infrastructure; see oracle.h).
 *
 * Deliberately plain: one code at a time, one bit at a time, sequential fp64
 * sums, no blocking and no reordering beyond the definitions in oracle.h.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

static int valid_bits(int b) {
    return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8;
}

static int valid_group(int g) { return g == 32 || g == 64 || g == 128; }

int64_t oracle_words_per_row(int64_t K, int bits) { return K * bits / 32; }

/* Bit p of row n's bitstream: byte p/8 of the row, bit p%8 of that byte. */
static unsigned row_bit(const uint32_t *W, int64_t K, int bits, int64_t n, int64_t p) {
    const uint8_t *row = (const uint8_t *)(W + n * oracle_words_per_row(K, bits));
    return (row[p / 8] >> (p % 8)) & 1u;
}

uint32_t oracle_code(const uint32_t *W, int64_t K, int bits, int64_t n, int64_t k) {
    uint32_t q = 0;
    for (int j = 0; j < bits; ++j)
        q |= (uint32_t)row_bit(W, K, bits, n, k * bits + j) << j;
    return q;
}

double oracle_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int check_shape(int64_t N, int64_t K, int bits, int group) {
    if (!valid_bits(bits) || !valid_group(group)) return ORACLE_EINVAL;
    if (N < 0 || K <= 0 || K % group != 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

static double weight(const uint32_t *W, const uint16_t *s, const uint16_t *b,
                     int64_t K, int bits, int group, int64_t n, int64_t k) {
    int64_t g = k / group;
    int64_t ng = K / group;
    double q = (double)oracle_code(W, K, bits, n, k);
    return oracle_bf16(s[n * ng + g]) * q + oracle_bf16(b[n * ng + g]);
}

int oracle_weights(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                   int64_t N, int64_t K, int bits, int group, int64_t n0, int64_t n1,
                   double *w_out) {
    int rc = check_shape(N, K, bits, group);
    if (rc) return rc;
    if (n0 < 0 || n1 > N || n0 > n1) return ORACLE_EINVAL;
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = 0; k < K; ++k)
            w_out[(n - n0) * K + k] = weight(W, scales, biases, K, bits, group, n, k);
    return ORACLE_OK;
}

struct qmm_job {
    const uint16_t *x;
    int rows;
    int64_t K;
    const uint32_t *W;
    const uint16_t *s, *b;
    int bits, group;
    const int64_t *cols;
    int64_t ncols, j0, j1;
    double *y64, *absum;
};

static void qmm_columns(const struct qmm_job *jb) {
    for (int64_t j = jb->j0; j < jb->j1; ++j) {
        int64_t n = jb->cols ? jb->cols[j] : j;
        for (int r = 0; r < jb->rows; ++r) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < jb->K; ++k) {
                double w = weight(jb->W, jb->s, jb->b, jb->K, jb->bits, jb->group, n, k);
                double t = oracle_bf16(jb->x[(int64_t)r * jb->K + k]) * w;
                acc += t;
                mag += fabs(t);
            }
            jb->y64[(int64_t)r * jb->ncols + j] = acc;
            jb->absum[(int64_t)r * jb->ncols + j] = mag;
        }
    }
}

static void *qmm_thread(void *arg) {
    qmm_columns((const struct qmm_job *)arg);
    return NULL;
}

int oracle_qmm(const uint16_t *x, int rows, int64_t K,
               const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
               int64_t N, int bits, int group,
               const int64_t *cols, int64_t ncols,
               double *y64, double *absum, int nthreads) {
    int rc = check_shape(N, K, bits, group);
    if (rc) return rc;
    if (rows < 1 || ncols < 0) return ORACLE_EINVAL;
    if (!cols && ncols != N) return ORACLE_EINVAL;
    if (cols)
        for (int64_t j = 0; j < ncols; ++j)
            if (cols[j] < 0 || cols[j] >= N) return ORACLE_EINVAL;

    struct qmm_job base = {x, rows, K, W, scales, biases, bits, group, cols, ncols, 0, ncols,
                           y64, absum};
    if (nthreads > ncols) nthreads = (int)ncols;
    if (nthreads <= 1) {
        qmm_columns(&base);
        return ORACLE_OK;
    }
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *running = (int *)calloc((size_t)nthreads, sizeof(int));
    struct qmm_job *jobs = (struct qmm_job *)calloc((size_t)nthreads, sizeof(struct qmm_job));
    if (!th || !running || !jobs) {
        free(th);
        free(running);
        free(jobs);
        qmm_columns(&base);
        return ORACLE_OK;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].j0 = ncols * t / nthreads;
        jobs[t].j1 = ncols * (t + 1) / nthreads;
        running[t] = pthread_create(&th[t], NULL, qmm_thread, &jobs[t]) == 0;
        if (!running[t]) qmm_columns(&jobs[t]); /* no thread: do this share here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t]) pthread_join(th[t], NULL);
    free(th);
    free(running);
    free(jobs);
    return ORACLE_OK;
}

/* Set bit p of a row's bitstream to v. */
static void put_bit(uint8_t *row, int64_t p, unsigned v) {
    if (v)
        row[p / 8] = (uint8_t)(row[p / 8] | (1u << (p % 8)));
    else
        row[p / 8] = (uint8_t)(row[p / 8] & ~(1u << (p % 8)));
}

int oracle_widen(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                 int64_t N, int64_t K, int bits, int group,
                 uint32_t *W_out, uint16_t *s_out, uint16_t *b_out,
                 int bits_out, int group_out) {
    int rc = check_shape(N, K, bits, group);
    if (rc) return rc;
    if (!valid_bits(bits_out) || !valid_group(group_out)) return ORACLE_EINVAL;
    if (bits_out < bits) return ORACLE_ENARROW;
    if (group_out > group || group % group_out != 0) return ORACLE_EGROUP;

    int64_t wpr_out = oracle_words_per_row(K, bits_out);
    for (int64_t n = 0; n < N; ++n) {
        uint8_t *row = (uint8_t *)(W_out + n * wpr_out);
        memset(row, 0, (size_t)(wpr_out * 4));
        for (int64_t k = 0; k < K; ++k) {
            uint32_t q = oracle_code(W, K, bits, n, k);
            for (int j = 0; j < bits_out; ++j) put_bit(row, k * bits_out + j, (q >> j) & 1u);
        }
    }
    int64_t ng_in = K / group, ng_out = K / group_out;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < ng_out; ++g) {
            int64_t parent = g * group_out / group;
            s_out[n * ng_out + g] = scales[n * ng_in + parent];
            b_out[n * ng_out + g] = biases[n * ng_in + parent];
        }
    return ORACLE_OK;
}

int oracle_common_width(const int *bits, const int *groups, int n,
                        int *bits_out, int *group_out) {
    if (n < 1) return ORACLE_EINVAL;
    int b = 0, g = 1 << 30;
    for (int i = 0; i < n; ++i) {
        if (!valid_bits(bits[i]) || !valid_group(groups[i])) return ORACLE_EINVAL;
        if (bits[i] > b) b = bits[i];
        if (groups[i] < g) g = groups[i];
    }
    *bits_out = b;
    *group_out = g;
    return ORACLE_OK;
}

void oracle_relu2(const double *y, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) {
        const double v = y[i] > 0.0 ? y[i] : 0.0;
        out[i] = v * v;
    }
}
