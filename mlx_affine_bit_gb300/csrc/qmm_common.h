// qmm_common.h -- launch parameters shared by the host planner (api.cu) and
// the kernel template (qmm_kernel.cuh).  Internal to libtfqmm.
#pragma once
#include <cuda.h>   // CUtensorMap (type only; the encoder is fetched at run time)
#include <stdint.h>

#if defined(__CUDACC__)
#define TFQ_HD __host__ __device__
#else
#define TFQ_HD
#endif

namespace tfq {

constexpr int CHUNK = 512;     // canonical K chunk: y = p_0 + p_1 + ... in chunk order
constexpr int TN = 128;        // output columns per CTA tile (8 warps x 16)
constexpr int NCW = 8;         // consumer warps per CTA
constexpr int NTHREADS = (NCW + 1) * 32;   // + one producer warp
constexpr int MAXSEG = 16;     // column segments (stack members) per run
constexpr int MAX_STAGES = 8;
constexpr int XS_MAX = 64 * 1024;          // bytes of permuted x a CTA keeps resident
constexpr int SMEM_MAX = 227 * 1024;       // dynamic shared memory per CTA on sm_103a
constexpr int SMEM_PER_SM = 228 * 1024;    // shared memory per SM (each CTA reserves 1 KB)
constexpr int HDR_BYTES = 256;             // mbarriers + flags at the start of smem

// K length of one pipeline stage: 512 k for <= 4 bits, 256 k above (bytes balance).
TFQ_HD constexpr int stage_k(int bits) { return bits <= 4 ? 512 : 256; }

struct QmmParams {
    // 2D TMA descriptors (bulk mode): W as u32 [N][K*bits/32] with a box of
    // 128 rows x (stage bytes + 16); scales and biases as u16 [N][K/G] with a
    // box of 128 rows x max(8, stage groups).
    CUtensorMap tmW, tmS, tmB;
    const uint16_t *x;
    const uint32_t *W;
    const uint16_t *s;
    const uint16_t *b;
    float *y;
    float *ws;          // split-K chunk partials [nchunks][rows][N] (nsl > 1)
    int *counters;      // [nct] arrival tickets (nsl > 1), zero between launches
    int *status;        // device status word (bounded waits that ran out)
    long long y_stride;
    int rows, K, N;
    int nct;            // column tiles of TN
    int nsl, sl;        // K slices and slice length (multiple of CHUNK)
    int nchunks;
    int n_items;        // nct * nsl, slice-major
    int stages;         // pipeline depth
    int bulk;           // 1: tensor-map TMA copies; 0: copies by the producer warp
    int wpitch;         // bytes per W row in a stage
    int sbpitch;        // bytes per scale (or bias) row in a stage
    int stage_bytes;
    int x_off, sx_off, st_off;   // smem offsets
    int rows_even;      // padded rows of the B-fragment and sum_group(x) layouts (8*NT)
    int nseg;
    int seg_src[MAXSEG], seg_len[MAXSEG], seg_dst[MAXSEG];
};

}  // namespace tfq
