/*
 * oracle.h -- fp64 CPU reference for the MLX-affine quantized row product.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline / reference leg may load this library.  It shares no
 * code, header, table or helper with the CUDA library, and neither includes
 * nor links the other.
 *
 * What it computes (TensorFold PR #788 "faster kernels in Zig engine": the
 * row-kernel commit "every MLX affine width in the row kernel" and the
 * tf-affine-ref commit; TensorFold PR #774 "oQ support", Exactness, the
 * Precision bullet):
 *
 *   code(n,k)   = bits [k*b, k*b+b) of row n's little-endian bitstream, read
 *                 one bit at a time, low code first (3- and 5-bit rows hold
 *                 eight codes in three or five bytes, low code first, as MLX
 *                 packs them; the same contiguous rule covers 2/4/6/8 bits);
 *   w(n,k)      = bf16(scale[n][k/G]) * code + bf16(bias[n][k/G])  (exact in fp64);
 *   y64[r][n]   = sum_k bf16(x[r][k]) * w(n,k), summed sequentially in fp64;
 *   absum[r][n] = sum_k |x[r][k] * w(n,k)|, the magnitude the fp32 bound uses.
 *
 * Widen / regroup (PR #788, the widen commit "mixed-width members read as one
 * matrix"): a matrix is re-packed at more bits with every code's integer value
 * unchanged, and its scale/bias are copied to each finer group; narrowing
 * bits, growing groups, groups that do not divide the source group and
 * unsupported widths are refused.
 */
#ifndef TF_ORACLE_H
#define TF_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)   /* unsupported bits/group, K % group, rows, sizes */
#define ORACLE_ENARROW (-2)  /* widen to fewer bits */
#define ORACLE_EGROUP (-3)   /* widen to a group that does not divide the source group */

/* Packed words per row: K*bits/32 (K is a multiple of 32 whenever the group is). */
int64_t oracle_words_per_row(int64_t K, int bits);

/* One code, extracted bit by bit.  W is [N][K*bits/32] uint32 (little endian). */
uint32_t oracle_code(const uint32_t *W, int64_t K, int bits, int64_t n, int64_t k);

/* bf16 bit pattern -> exact double. */
double oracle_bf16(uint16_t h);

/* Dequantized fp64 weights of rows [n0, n1): w_out[(n-n0)*K + k]. */
int oracle_weights(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                   int64_t N, int64_t K, int bits, int group, int64_t n0, int64_t n1,
                   double *w_out);

/*
 * y64[r*ncols + j] and absum[r*ncols + j] for the columns cols[j]
 * (cols == NULL means all N columns; ncols must then equal N).
 * nthreads <= 1 runs on the calling thread; otherwise the columns are split
 * over nthreads POSIX threads.  Returns ORACLE_OK or a negative code.
 */
int oracle_qmm(const uint16_t *x, int rows, int64_t K,
               const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
               int64_t N, int bits, int group,
               const int64_t *cols, int64_t ncols,
               double *y64, double *absum, int nthreads);

/* Decode every code and rebuild it at (bits_out, group_out). */
int oracle_widen(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                 int64_t N, int64_t K, int bits, int group,
                 uint32_t *W_out, uint16_t *s_out, uint16_t *b_out,
                 int bits_out, int group_out);

/*
 * Squared-ReLU output epilogue (TensorFold PR #788, row-kernel commit: relu2
 * calls in the bit-exact window gate; the pages name it without a formula, so
 * it is read as its name says): out[i] = max(y[i], 0)^2, in fp64.
 */
void oracle_relu2(const double *y, int64_t n, double *out);

/* The common width of n members: the most bits and the smallest group. */
int oracle_common_width(const int *bits, const int *groups, int n,
                        int *bits_out, int *group_out);

#ifdef __cplusplus
}
#endif
#endif
