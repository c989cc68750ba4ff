/*
 * tfqmm.h -- C ABI of the MLX-affine quantized row product for GB300 (sm_103a).
 *
 * The operation (TensorFold PR #788 "faster kernels in Zig engine", commit
 * "every MLX affine width in the row kernel"; PR #774 "oQ support",
 * Exactness, the Precision bullet):
 *
 *     y[r][n] = sum_k x[r][k] * (scale[n][k/G] * q[n][k] + bias[n][k/G])
 *
 * for activation rows r (1..16 in one launch).  q[n][k] is an unsigned code of `bits` bits
 * (2, 3, 4, 5, 6 or 8), stored low code first in row n's little-endian
 * bitstream (3- and 5-bit rows hold eight codes in three or five bytes; every
 * row ends on a 32-bit word).  scale and bias are bf16, one per group of G = 32,
 * 64 or 128 consecutive k.  x is bf16; y is fp32, accumulated in fp32.
 *
 * Results: every output lies within (K * 2^-24 + 2^-20) * sum_k |x_k * w_k| of
 * the exact product; a row's bits depend on its own inputs only (the same in a
 * window of any size), and a strided or stacked output equals the contiguous
 * one bit for bit (the canonical order below fixes the arithmetic).
 *
 * Canonical order of one output y[r][n]: K is cut into segments of 256 k and
 * chunks of 2048 k (the last of each may be shorter).  Inside a segment, group
 * by group in k order,
 *     T = sum over the group of x*q     (tensor-core dot products, exact codes)
 *     p = fma(scale, T, p); p = fma(bias, sum_group(x), p)     (p starts at 0)
 * where sum_group(x) is the sequential fp32 sum of the group's x.  A chunk's
 * sum is C = p_0 + p_1 + ... over its segments in order, and y = C_0 + C_1 +
 * ... over the chunks in order.  Row count, N, output stride, split-K, launch
 * mode and stack membership never enter this order.
 *
 * Memory: every pointer of tf_qmm / tf_qmm_stack / tf_widen is DEVICE memory
 * owned by the caller; the library never frees or retains it.  Calls are
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * The library keeps, per device and stream, a small workspace for split-K
 * partials and a device status word (allocated on first use, held until exit).
 * Errors are returned as negative status codes; nothing throws across the ABI.
 */
#ifndef TFQMM_H
#define TFQMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define TF_OK 0
#define TF_EINVAL_BITS (-1)   /* bits not in {2,3,4,5,6,8} */
#define TF_EINVAL_GROUP (-2)  /* group not in {32,64,128}, or K % group != 0, or K < 1 */
#define TF_EINVAL_ROWS (-3)   /* rows not in [1, 16] (tf_qmm / tf_qmm_ex: [1, 65536]) */
#define TF_EINVAL_STRIDE (-4) /* y_stride < N (a strided call writes rows at least a matrix wide) */
#define TF_EINVAL_PTR (-5)    /* NULL pointer, or x / W not 16-byte aligned, y not 4-byte aligned */
#define TF_EINVAL_SIZE (-6)   /* N < 1, or sizes too large for 32-bit indexing of one row */
#define TF_ENARROW (-7)       /* tf_widen to fewer bits */
#define TF_EGROUP (-8)        /* tf_widen to a group that does not divide the source group */
#define TF_ESTACK (-9)        /* bad stack table: member range outside its run, overlapping
                                 destinations, a destination past y_stride, mixed K */
#define TF_ECUDA (-10)        /* a CUDA runtime call failed; see tf_last_error_string() */
#define TF_EDEVICE (-11)      /* a kernel reported a bounded wait that ran out (device status) */
#define TF_EINVAL_FLAGS (-12) /* output flags other than TF_OUT_BF16 | TF_EPI_RELU2 */
#define TF_EGATHER (-13)      /* empty slot table, or a slot naming a missing expert or x row */
#define TF_EBOUNDS (-14)      /* the bounds-checking debug build (libtfqmm_debug.so) found an index
                                 outside its buffer (device status; the access was skipped) */

/*
 * tf_qmm -- one quantized product.
 *   x        [rows][K] bf16 (uint16 bit patterns), contiguous, 16-byte aligned.
 *   W        [N][K*bits/32] uint32, 16-byte aligned.
 *   scales   [N][K/group] bf16; biases likewise.
 *   y        fp32; row r, column n is y[r*y_stride + n] for n < N.  Columns
 *            N..y_stride-1 of each row are not touched.
 *   rows     1..65536: more than 16 rows run as 16-row windows (independent
 *            launches that overlap under programmatic dependent launch; the
 *            weights are read once per window), each row's bits those of the
 *            row alone -- the row / window gate of PR #788 extended past 16 rows.
 * Returns TF_OK or a negative status (checked on the host before any launch).
 * Allocation: the first call on a device allocates the device status word, and
 * a call whose plan splits K allocates (or grows, with cudaFree + cudaMalloc)
 * the split-K workspace of its (device, stream).  A caller that must not let
 * the library allocate uses tf_qmm_noalloc instead.
 */
int tf_qmm(const uint16_t *x, int rows, int K,
           const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
           int N, int bits, int group,
           float *y, int64_t y_stride, void *stream);

/*
 * tf_qmm_noalloc -- tf_qmm for callers that cannot let a library allocate
 * device memory: code running while a stream is captured into a CUDA graph,
 * engines that give all device memory to their own pool at start-up, and
 * processes that must not grow their footprint later.  The paper has no
 * counterpart; it is a deployment variant of tf_qmm.
 *
 * Same arguments, layouts and results as tf_qmm, bit for bit, rows 1..65536
 * (more than 16 rows run as 16-row windows, one launch after another), with
 * plain launches whatever the launch mode.  Its split-K scratch and status
 * word come from one fixed 4 MiB device array built into the library instead
 * of a cudaMalloc: every GPU that loads the library holds that array until
 * exit, and the call allocates nothing.  A product whose split-K partials need
 * more than the array holds (window rows * N * ceil(K/2048) * 4 bytes, about
 * 4 MiB, when the planner splits K) is refused with TF_EINVAL_SIZE before any
 * launch.  The first call on a device looks up the array's device address and
 * clears its status word (set-up); make that first call before any stream
 * capture.  All calls share the array: each clears the counters it needs at
 * zero on its own stream, and calls that overlap on the GPU race.  A bounded
 * wait that runs out is recorded in the array's status word, which
 * tf_noalloc_status reads (not tf_device_status).
 */
int tf_qmm_noalloc(const uint16_t *x, int rows, int K,
                   const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                   int N, int bits, int group,
                   float *y, int64_t y_stride, void *stream);

/*
 * Reads and clears the status word of tf_qmm_noalloc's fixed array on the
 * current device (synchronizes the device; allocates nothing).  TF_OK, or
 * TF_EDEVICE if a no-allocation product gave up a bounded wait since the last
 * read.  The paper has no counterpart.
 */
int tf_noalloc_status(void);

/*
 * Fused stack of members written through one strided output (PR #788, "a
 * fused stack of 48-column members at mixed widths written through the
 * stride"; PR #774, runs and members of the _stacked split rule and the
 * column map that writes each member's columns in place).
 *
 * A run is one matrix at one width (usually widened by tf_widen).  A member
 * takes n_cols consecutive columns of its run starting at src_col and writes
 * them to y columns [dst_col, dst_col + n_cols).  Members of a run need not be
 * adjacent in y.  Every member's columns equal the run's own tf_qmm result
 * bit for bit.  The table is read on the host only.  Each run is one launch;
 * under TF_LAUNCH_PDL / TF_LAUNCH_EARLY_WEIGHTS the runs after the first
 * overlap it (they start once the first run's dependency on the previous
 * kernel of the stream has resolved, and a run with split K waits for the run
 * before it), and the last launch completes after every run, so the next
 * kernel of the stream sees the whole stack.
 */
typedef struct tf_run {
    const uint32_t *W;
    const uint16_t *scales;
    const uint16_t *biases;
    int N;
    int bits;
    int group;
} tf_run;

typedef struct tf_member {
    int run;
    int src_col;
    int n_cols;
    int dst_col;
} tf_member;

int tf_qmm_stack(const uint16_t *x, int rows, int K,
                 const tf_run *runs, int n_runs,
                 const tf_member *members, int n_members,
                 float *y, int64_t y_stride, void *stream);

/*
 * Output options (PR #788, row-kernel commit: the one-row / window gate covers
 * relu2 calls and strided outputs bit for bit; tf-affine-ref commit: bf16
 * outputs are bounded by one more bf16 ulp).
 *   TF_OUT_BF16:  y is bf16 (uint16 bit patterns), each output rounded to
 *                 nearest even from the fp32 result; y 2-byte aligned.
 *   TF_EPI_RELU2: y = max(v, 0)^2 of the fp32 result v, in fp32 (then
 *                 rounded when TF_OUT_BF16 is also set).
 * The fp32 result v itself is the one tf_qmm computes, bit for bit.
 */
#define TF_OUT_BF16 1
#define TF_EPI_RELU2 2

/* tf_qmm with output options; y is float* or bf16* as flags say. */
int tf_qmm_ex(const uint16_t *x, int rows, int K,
              const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
              int N, int bits, int group,
              void *y, int64_t y_stride, int flags, void *stream);

/*
 * tf_qmm_prompt -- the product for many activation rows (a prompt), with the
 * weights read once per 64-row window (PR #788, the 2-bit affine_mm commit: the
 * prompt-side tiled product, checked row by row against windows of 1 to 65 rows).
 *   Same arguments, layouts and output options (flags as tf_qmm_ex) as tf_qmm_ex,
 *   rows 1..65536; K must be a multiple of 2048 (TF_EINVAL_SIZE otherwise) and
 *   scales / biases 16-byte aligned (TF_EINVAL_PTR).
 *   The group dot products run on the tcgen05 tensor cores (M = 128 output
 *   columns, N = the window's rows rounded up to 16, accumulators in tensor
 *   memory), so this entry point has its own canonical order: per output,
 *   p = fma(scale, T, p); p = fma(bias', sum_group(x), p) over the groups of each
 *   2048-k chunk from 0 (T the tensor-core group dot product; bias' = bias - 128
 *   scale for 4-6-bit codes, which enter as 128 + c), y = C_0 + C_1 + ... over the
 *   chunks in order.  Every row's result is the same bit for bit in any window of
 *   any size and position of this entry point, and whether or not the chunks are
 *   split over work items; it is within the tolerance of tf_qmm but not
 *   bit-identical to it (whose segment order and MMA instruction differ).
 *   Allocates a per-(device, stream) workspace for the permuted activations,
 *   their group sums and, when the column tiles are fewer than the SMs and K
 *   holds more than one chunk, the chunk partials of one window (rows * K * 2 +
 *   (K / group) * ceil(rows / 64) * 256 + [(K / 2048) * 64 * N * 4] bytes, grown
 *   on demand; the first call on a stream must precede any graph capture on it).
 *   Plain launches: one prepass, then per 64 rows one launch and, with split
 *   chunks, one fold.  Measured on GB300 it overtakes 16-row windows of tf_qmm
 *   from about 24 rows (the 248320 x 2048 LM head; about 30 rows at 12288 x
 *   2048) and is 2.3-2.4x faster at 64; below that, tf_qmm is faster.
 */
int tf_qmm_prompt(const uint16_t *x, int rows, int K,
                  const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                  int N, int bits, int group,
                  void *y, int64_t y_stride, int flags, void *stream);

/*
 * tf_qmm_gather -- indexed slots over a set of expert matrices (PR #788,
 * row-kernel commit: indexed slots in the bit-exact window gate; tf-affine-ref
 * commit: a one-expert gather equals the dense product).
 *   Slot i (0 <= i < n_slots) computes y row i = experts[slot_expert[i]] times
 *   x row slot_row[i] (x is [x_rows][K] bf16; y rows are y_stride elements
 *   apart, at least every used expert's N; columns past an expert's N are
 *   untouched).  Each slot equals, bit for bit, tf_qmm_ex of its expert on its
 *   x row alone.  The slot table is read on the host; experts may differ in
 *   bits, group and N.  Slots of one expert run together, 16 to a launch, and
 *   the launches may overlap under programmatic dependent launch (as stack runs).
 */
int tf_qmm_gather(const uint16_t *x, int x_rows, int K,
                  const tf_run *experts, int n_experts,
                  const int *slot_expert, const int *slot_row, int n_slots,
                  void *y, int64_t y_stride, int flags, void *stream);

/*
 * tf_widen -- exact widen / regroup on the device (PR #788, the widen commit:
 * mixed-width members read as one matrix at their common width, the most bits
 * and the smallest group; narrowing and groups that do not divide the source
 * group are refused).  Every code keeps its integer value and is re-packed at
 * bits_out; every finer group copies its parent group's scale and bias, so the
 * dequantized fp64 weights are identical bit for bit.
 *   W_out [N][K*bits_out/32], s_out/b_out [N][K/group_out]: caller-allocated
 *   device memory (sizes from tf_qmm_bytes).  W and W_out 16-byte aligned.
 */
int tf_widen(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
             int N, int K, int bits, int group,
             uint32_t *W_out, uint16_t *s_out, uint16_t *b_out,
             int bits_out, int group_out, void *stream);

/*
 * tf_widen_host -- the same widen / regroup on HOST memory, for loaders that
 * re-pack at load time before uploading (PR #788, the widen commit: the
 * packer writes mixed-width members as one matrix).  Same arguments, checks,
 * status codes and output bytes as tf_widen (W 16-byte aligned), with every
 * pointer in host memory owned by the caller; no CUDA call is made.
 */
int tf_widen_host(const uint32_t *W, const uint16_t *scales, const uint16_t *biases,
                  int N, int K, int bits, int group,
                  uint32_t *W_out, uint16_t *s_out, uint16_t *b_out,
                  int bits_out, int group_out);

/* Common width of n members: (max bits, min group).  Host only. */
int tf_common_width(const int *bits, const int *groups, int n, int *bits_out, int *group_out);

/* Byte sizes of W and of one of scales/biases for an (N, K, bits, group) matrix. */
int tf_qmm_bytes(int N, int K, int bits, int group, int64_t *w_bytes, int64_t *sb_bytes);

/*
 * Reads and clears the device status word of the current device (synchronizes
 * the device).  TF_OK, TF_EDEVICE if a kernel gave up a bounded wait, or (debug
 * build only) TF_EBOUNDS if a kernel found an index outside its buffer.
 */
int tf_device_status(void);

/*
 * Launch mode of later tf_qmm / tf_qmm_stack calls (process wide); returns the
 * previous mode.  Not on the pages: a GB300 launch option.
 *   TF_LAUNCH_PDL: programmatic dependent launch -- a product may start its
 *     prologue while the previous kernel of the stream finishes; it waits for
 *     that kernel before reading x or writing y (always safe).
 *   TF_LAUNCH_EARLY_WEIGHTS: as TF_LAUNCH_PDL, and the product also streams its
 *     weights, scales and biases before that wait.  Only valid when the kernel
 *     just before it in the stream does not write them (e.g. a decode step whose
 *     weights are fixed).
 *   TF_LAUNCH_EARLY_X: as TF_LAUNCH_EARLY_WEIGHTS, and the product also reads
 *     x and computes before that wait; it waits only before its first write
 *     of y (or of split-K partials), so consecutive independent products
 *     overlap.  Only valid when the kernel just before it in the stream writes
 *     neither x nor the weights (products that share an activation, or a
 *     sequence of independent products).  The runs of a stack, the windows of
 *     a call with more than 16 rows and the launches of a gather then overlap
 *     the same way.
 * 0 (the default) launches plainly.  Negative status for unknown bits.
 */
#define TF_LAUNCH_PDL 1
#define TF_LAUNCH_EARLY_WEIGHTS 2
#define TF_LAUNCH_EARLY_X 4
int tf_set_launch_mode(int mode);

/*
 * Test hook for the bounded waits (no GPU fault is involved): the next product
 * launch withholds every CTA's first stage of codes, so the consumers' wait
 * for it runs out after about 2 s; the kernel records that in the device
 * status word, stops waiting and runs to completion (its output is then
 * meaningless) and tf_device_status returns TF_EDEVICE.  The context stays
 * usable.  One shot; TF_OK.
 */
int tf_inject_stall(void);

/* Message for the last failing call on this host thread ("" if none). */
const char *tf_last_error_string(void);

const char *tf_version(void);

#ifdef __cplusplus
}
#endif
#endif
