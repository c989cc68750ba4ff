// qmm_common.h -- launch parameters shared by the host planner (api.cu) and
// the kernel template (qmm_kernel.cuh).  Internal to libtfqmm.
#pragma once
#include <cuda.h>   // CUtensorMap (type only; the encoder is fetched at run time)

// The bounds-checking debug build and the phase-trace build put their
// internals in namespaces of their own, so that their symbols (kernels,
// launchers) never meet the product's when a process loads several libraries.
#ifdef TF_DEBUG_BOUNDS
#define tfq tfq_debug
#elif defined(TF_TRACE)
#define tfq tfq_trace
#endif
#include <stdint.h>

#if defined(__CUDACC__)
#define TFQ_HD __host__ __device__
#else
#define TFQ_HD
#endif

namespace tfq {

// Canonical order of one output (the same for every launch shape):
//   segment  = 256 k   : P = fma chain over the segment's groups, from 0
//   chunk    = 2048 k  : C = P_0 + P_1 + ... (segments in k order)
//   y        = C_0 + C_1 + ... (chunks in k order)
constexpr int SEG = 256;
constexpr int CHUNK = 2048;
constexpr int SEGS = CHUNK / SEG;          // segments per chunk = consumer warps
constexpr int TN = 16;                     // output columns per work item (one mma m-tile)
constexpr int NCW = SEGS;                  // consumer warps: one segment of a stage each
// Threads of a CTA with `cg` consumer groups of NCW warps, plus one producer warp.
TFQ_HD constexpr int block_threads(int cg) { return (cg * NCW + 1) * 32; }
constexpr int MAXCOLSEG = 16;              // column-map segments (stack members) per run
constexpr int MAX_STAGES = 8;
constexpr int XS_MAX = 64 * 1024;          // bytes of permuted x a CTA keeps resident
constexpr int SMEM_MAX = 227 * 1024;       // dynamic shared memory per CTA on sm_103a
constexpr int SMEM_PER_SM = 228 * 1024;    // shared memory per SM (each CTA reserves 1 KB)
constexpr int HDR_BYTES = 256;             // mbarriers + flags at the start of smem
// Phase-trace build: words a CTA record, records a buffer, header byte of the record index.
constexpr int TRACE_SLOTS = 9, TRACE_MAX = 1 << 16, TRACE_HDR = 192;

// Row bucket of a launch (a kernel template parameter): 1 (a single row),
// 2, 4, 8 or 16; the B-fragment layout holds layout_rows(bucket) rows.
TFQ_HD constexpr int row_bucket(int rows) {
    return rows == 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : rows <= 8 ? 8 : 16;
}
TFQ_HD constexpr int layout_rows(int rb) { return rb < 2 ? 2 : rb; }

// Zero words after each row segment of a stage (the TMA box reads them past the
// segment's extent).  Four in general; 4-bit rows with groups of 64 or 128 and
// 8-bit rows with groups of 64 take the pad at which no two lanes of a warp's
// code loads share a shared-memory bank (with four words they would in pairs).
TFQ_HD constexpr int seg_pad_words(int bits, int group) {
    return (bits == 4 && group == 64) ? 8 : ((bits == 4 && group == 128) || (bits == 8 && group == 64)) ? 16 : 4;
}
constexpr int ZERO_BYTES = 2048;           // zero block that idle lanes of small buckets read

struct QmmParams {
    // TMA descriptors (bulk mode).  W: [K/SEG segments][N rows][SEG*bits/32
    // words], box {segment + seg_pad_words past its extent (zero filled), the
    // stage's rows, 8 segments}; scales/biases: one stage's groups of its rows.
    CUtensorMap tmW, tmS, tmB;
    const uint16_t *x;
    const uint32_t *W;
    const uint16_t *s;
    const uint16_t *b;
    float *y;
    float *ws;          // split-K chunk sums [nchunks][rows][N] (nsl > 1)
    int *counters;      // [nmt] arrival tickets (nsl > 1), zero between launches
    int *status;        // device status word (bounded waits that ran out)
    long long y_stride;
    int rows, K, N;
    int nmt;            // column tiles of TN * MT columns (items per K slice)
    int nsl, sl;        // K slices and slice length (multiple of CHUNK)
    int nchunks;
    int stages;         // pipeline depth
    int bulk;           // 1: tensor-map TMA copies; 0: copies by the producer warp
    int sb3d;           // 1: scale/bias rows padded through a 3D map (K % CHUNK == 0)
    int early_w;        // 1: the producer may read W/scales/biases before the grid dependency resolves
    int early_x;        // 1: x is read and the product computed before the grid dependency
                        //    resolves; only the first write (y or split-K partials) waits for it
    int dep;            // programmatic dependent launch: 0 wait before x/y, release the next
                        // launch at once; 1 release it only after that wait (first run of a
                        // stack); 2 no wait before x/y, wait before exit (later runs of a stack)
    int sbpitch;        // bytes per scale (or bias) row in a stage
    int stage_bytes;    // W blocks + scales + biases
    int x_off, sx_off, pb_off, z_off, st_off;   // smem offsets
    int ncs;            // column-map segments
    int cs_src[MAXCOLSEG], cs_len[MAXCOLSEG], cs_dst[MAXCOLSEG];
    int stall;          // test hook: the producer withholds every CTA's first stage
    int out;            // OUT_* bits: bf16 output (y holds bf16), squared-ReLU epilogue
    int xrow[16];       // window row r reads x row xrow[r] (K elements apart) ...
    int yrow[16];       // ... and writes y row yrow[r] (y_stride elements apart)
    // Extents the call's arguments give each buffer, for the bounds checks of
    // the debug build: x rows, y rows, split-K partial floats, arrival counters.
    int x_rows, y_rows;
    long long ws_elems;
    int n_counters;
    // Phase-trace build only (null otherwise): per-CTA records, their counter,
    // and the launch's number.
    unsigned long long *trace;
    unsigned *trace_n;
    unsigned trace_seq;
};

#ifdef TF_TRACE
// Host (phase-trace build): the launch's parameters with the trace buffer and
// the next launch number.
QmmParams trace_params(const QmmParams &P);
#endif

// Bits of the device status word.
constexpr int STATUS_WAIT = 1;      // a bounded wait ran out
constexpr int STATUS_BOUNDS = 2;    // the debug build found an index outside its buffer

constexpr int OUT_BF16 = 1;    // y is bf16, each output rounded to nearest even
constexpr int OUT_RELU2 = 2;   // y = max(v, 0)^2 of the fp32 result v (before any bf16 rounding)

}  // namespace tfq
