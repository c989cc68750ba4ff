// api.cu -- C ABI of libtfqmm (declared in include/tfqmm.h).
//
// Host-side argument checks, the launch planner (column tiles x K slices),
// the per-(device, stream) split-K workspace, the stack dispatcher and the
// device widen / regroup kernels.  All arithmetic of the product runs in the
// kernels of qmm_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/tfqmm.h"
#ifdef TF_TRACE
#include "../../include/tfqmm_trace.h"
#endif
#include "internal.h"

using namespace tfq;

namespace {

thread_local std::string g_err;

int fail(int code, const std::string &msg) {
    g_err = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char *where) {
    g_err = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return TF_ECUDA;
}

bool valid_bits(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }
bool valid_group(int g) { return g == 32 || g == 64 || g == 128; }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_matrix(int K, const uint32_t *W, const uint16_t *s, const uint16_t *b, int N, int bits,
                 int group) {
    if (!valid_bits(bits)) return fail(TF_EINVAL_BITS, "bits must be 2, 3, 4, 5, 6 or 8");
    if (!valid_group(group) || K < group || K % group != 0)
        return fail(TF_EINVAL_GROUP, "group must be 32, 64 or 128 and divide K");
    if (N < 1 || K > (1 << 26)) return fail(TF_EINVAL_SIZE, "N must be >= 1 and K <= 2^26");
    if (!W || !s || !b) return fail(TF_EINVAL_PTR, "NULL weight, scale or bias pointer");
    if (!aligned(W, 16)) return fail(TF_EINVAL_PTR, "W must be 16-byte aligned");
    if (!aligned(s, 2) || !aligned(b, 2)) return fail(TF_EINVAL_PTR, "scales/biases must be 2-byte aligned");
    return TF_OK;
}

// Rows of one tf_qmm / tf_qmm_ex call: more than 16 run as 16-row windows.
constexpr int MAX_ROWS = 65536;

int check_io(const uint16_t *x, int rows, const float *y, int max_rows = 16) {
    if (rows < 1 || rows > max_rows)
        return fail(TF_EINVAL_ROWS, max_rows == 16 ? "rows must be in [1, 16]" : "rows must be in [1, 65536]");
    if (!x || !y) return fail(TF_EINVAL_PTR, "NULL x or y");
    if (!aligned(x, 16)) return fail(TF_EINVAL_PTR, "x must be 16-byte aligned");
    if (!aligned(y, 4)) return fail(TF_EINVAL_PTR, "y must be 4-byte aligned");
    return TF_OK;
}

// ---------------------------------------------------------------- planner --

struct Plan {
    int nmt, nsl, sl, nchunks, stages, smem, grid, segpitch, sbpitch, stage_bytes, x_off, sx_off,
        pb_off, z_off, st_off, rb, ctas, mt, cg;
    bool sb3d;
    bool half;      // one CTA per SM within half of its shared memory and registers
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

Plan layout(int N, int K, int bits, int group, int rows, int nsm, int ctas, bool sb3d, int mt, int cg = 1,
            bool half = false) {
    Plan p{};
    p.rb = row_bucket(rows);
    p.ctas = ctas;
    p.sb3d = sb3d;
    p.mt = mt;
    p.cg = cg;
    p.half = half;
    const int rws = TN * mt;                                // output columns (W rows) per item
    const bool halved = ctas == 2 || half;                  // half of the SM's shared memory
    const int xs_max = halved ? XS_MAX / 2 : XS_MAX;
    const int budget = halved ? SMEM_PER_SM / 2 - 1024 : SMEM_MAX;
    p.nmt = ceil_div(N, rws);
    p.nchunks = ceil_div(K, CHUNK);
    const int lr = layout_rows(p.rb);
    const int max_cps = std::max(1, xs_max / (lr * 2 * CHUNK));   // chunks of x a CTA holds
    const long long slots = (long long)ctas * nsm;
    double best = 1e30;
    int best_cps = p.nchunks;
    for (int nsl = 1; nsl <= p.nchunks; ++nsl) {
        const int cps = ceil_div(p.nchunks, nsl);
        if (cps > max_cps || (nsl - 1) * cps >= p.nchunks) continue;
        const long long team = std::max(1LL, slots / nsl);    // CTAs per K slice
        const double cost = (double)ceil_div(p.nmt, team) * (cps + (nsl > 1 ? 0.5 : 0.25)) * ctas;
        if (cost < best) {
            best = cost;
            best_cps = cps;
        }
    }
    p.sl = best_cps * CHUNK;
    p.nsl = ceil_div(p.nchunks, best_cps);
    const int len = std::min(p.sl, K);
    const int sbg = CHUNK / group;                          // groups of one stage
    p.segpitch = SEG * bits / 8 + 4 * seg_pad_words(bits, group);
    p.sbpitch = sb3d ? (sbg + 8) * 2 : sbg * 2;
    p.stage_bytes = SEGS * rws * p.segpitch + 2 * rws * p.sbpitch;
    const int x_bytes = (lr * len * 2 + 127) & ~127;
    const int sx_bytes = ((len / group) * lr * 4 + 127) & ~127;
    const int pb_bytes = cg * 2 * SEGS * rws * lr * 4;
    p.x_off = HDR_BYTES;
    p.sx_off = p.x_off + x_bytes;
    p.pb_off = p.sx_off + sx_bytes;
    p.z_off = (p.pb_off + pb_bytes + 127) & ~127;
    p.st_off = p.z_off + (lr < 8 ? ZERO_BYTES : 0);
    p.stages = std::min(MAX_STAGES, (budget - p.st_off) / p.stage_bytes);
    p.smem = p.st_off + p.stages * p.stage_bytes;
    // Whole teams: one team of CTAs per K slice (see ItemWalk).
    p.grid = p.nsl * (int)std::max(1LL, std::min<long long>(p.nmt, slots / p.nsl));
    return p;
}

// The launch plan, in order of preference (every choice gives the same bits):
//  0. when consecutive products may overlap (early-x launches), 1-2 rows and at
//     most eight column tiles per SM: one m-tile per item, at most one CTA per SM
//     within half of the SM, so that the next product's CTA is resident beside it
//     and computes while this one finishes (4096 x 4096 width sweep: 82 -> 69 us
//     for the 18 products);
//  1. up to 8 rows: two m-tiles (32 columns) per item, one CTA per SM, when two
//     stages fit and the items fill the SMs (two per SM at 1-2 rows, one per two
//     SMs at 3-8) -- computed by two consumer groups when the whole K is one
//     slice, three stages fit and the items are plentiful (2+ per SM at one
//     row, 4+ per SM from two rows on);
//  2. one m-tile per item, two CTAs per SM, when three stages fit, or two that
//     hold a whole item of two chunks;
//  3. one m-tile per item, one CTA per SM with a deeper ring: two consumer
//     groups for 9-16 rows over many column tiles, else for 9-16 rows two
//     m-tiles per item when those fill half the SMs.
Plan make_plan(int N, int K, int bits, int group, int rows, int nsm, bool sb3d, bool overlap = false) {
    if (overlap && row_bucket(rows) <= 2) {
        // The one-m-tile kernel is capped at 96 registers: two CTAs of nine warps fit an SM.
        Plan h = layout(N, K, bits, group, rows, nsm, 1, sb3d, 1, 1, true);
        if (h.nsl == 1 && h.stages >= 2 && (long long)h.nmt <= 8LL * nsm) {
            h.grid = std::min(h.grid, nsm);
            // Up to two items a CTA: as few CTAs as give the busiest one its items
            // (4096 columns: 128 CTAs of two items, not 152 of one or two); the
            // critical CTA is the same and the SMs left over take a later product's
            // CTAs early (width sweep 0.440 -> 0.449).  With more items a CTA the
            // spread grid measured faster (12288 columns: 6.1 against 7.2 us).
            const int per = (h.nmt + h.grid - 1) / h.grid;
            if (per <= 2) h.grid = (h.nmt + per - 1) / per;
            return h;
        }
    }
    if (row_bucket(rows) <= 8) {
        const Plan wide = layout(N, K, bits, group, rows, nsm, 1, sb3d, 2);
        // Two stages suffice for one consumer group: 6- and 8-bit codes at 4-8
        // rows leave room for no more, and the plan still beat the one-m-tile
        // plans there (12288 x 2048, 8 rows: 8.3 against 9.8 us).
        // With 4-8 rows a stage's compute is heavy enough that the wider item pays
        // even with idle SMs (2048 x 12288, 4 rows: 128 items on 152 SMs, 10.6
        // against 12.5 us); one or two rows want two items per SM.
        const long long min_items = row_bucket(rows) >= 4 ? nsm / 2 : 2LL * nsm;
        if (wide.stages >= 2 && (long long)wide.nmt * wide.nsl >= min_items) {
            // Two consumer groups (two stages computed at once) when three stages
            // fit; from two rows on only with at least four items per SM (at
            // 2.5 per SM one group measured 1.5-5 % faster, 12288 x 2048).
            if (wide.nsl == 1 && (row_bucket(rows) == 1 || (long long)wide.nmt >= 4LL * nsm)) {
                const Plan pp = layout(N, K, bits, group, rows, nsm, 1, sb3d, 2, 2);
                if (pp.stages >= 3 && pp.nsl == 1) return pp;
            }
            return wide;
        }
    }
    const Plan two = layout(N, K, bits, group, rows, nsm, 2, sb3d, 1);
    if (two.stages >= 3) return two;
    // Two stages suffice when they hold a whole item of two chunks (the second
    // loads while the first computes): 8-bit 4096 x 4096 products measured
    // 3.5-7.5 % faster than with one CTA per SM.
    if (two.stages == 2 && two.nsl == 1 && two.nchunks == 2) return two;
    const Plan one = layout(N, K, bits, group, rows, nsm, 1, sb3d, 1);
    if (row_bucket(rows) == 16 && one.nsl == 1 && (long long)one.nmt >= 2LL * nsm) {
        // Nine to sixteen rows over many column tiles: two consumer groups
        // (their compute per stage is long enough that one stage in flight keeps up).
        const Plan pp = layout(N, K, bits, group, rows, nsm, 1, sb3d, 1, 2);
        if (pp.stages >= 3 && pp.nsl == 1) return pp;
    }
    if (row_bucket(rows) == 16) {
        // Else two m-tiles per item for one consumer group (it shares the
        // activation loads; 2048 x 12288: 20.3 against 22.3 us).
        const Plan wide = layout(N, K, bits, group, rows, nsm, 1, sb3d, 2);
        if (wide.stages >= 2 && (long long)wide.nmt * wide.nsl >= nsm / 2) return wide;
    }
    return one;
}

// ------------------------------------------------------------ TMA maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once from the driver; read by callers on any thread (the
// no-allocation entry point runs outside the planner's mutex).
std::atomic<EncodeTiledFn> g_encode{nullptr};

int get_encoder() {
    if (g_encode.load(std::memory_order_acquire)) return TF_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(TF_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode.store(reinterpret_cast<EncodeTiledFn>(fn), std::memory_order_release);
    return TF_OK;
}

// 2D row-major tensor [rows][cols] of `esize`-byte elements, box [box_rows][box_cols].
int encode_2d(CUtensorMap *m, const void *base, CUtensorMapDataType t, int esize, long long cols,
              long long rows, int box_cols, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode.load(std::memory_order_acquire)(m, t, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TF_ECUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return TF_OK;
}

// A 3D view {d0, d1, d2} (d0 innermost, stride 4 or 2 bytes) with byte
// strides s1, s2 and box {b0, b1, b2}.
int encode_3d(CUtensorMap *m, const void *base, CUtensorMapDataType t, long long d0, long long d1,
              long long d2, long long s1, long long s2, int b0, int b1, int b2) {
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)s1, (cuuint64_t)s2};
    cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, (cuuint32_t)b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode.load(std::memory_order_acquire)(m, t, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TF_ECUDA, "cuTensorMapEncodeTiled(3D) failed (" + std::to_string((int)r) + ")");
    return TF_OK;
}

// Encoded maps of recently used matrices (a map holds only address and shape).
struct MapKey {
    const void *W, *s, *b;
    int N, K, bits, group, mt;
    bool operator<(const MapKey &o) const {
        if (W != o.W) return W < o.W;
        if (s != o.s) return s < o.s;
        if (b != o.b) return b < o.b;
        if (N != o.N) return N < o.N;
        if (K != o.K) return K < o.K;
        if (bits != o.bits) return bits < o.bits;
        if (mt != o.mt) return mt < o.mt;
        return group < o.group;
    }
};
struct MapSet {
    CUtensorMap W, s, b;
};
std::map<MapKey, MapSet> g_maps;
constexpr size_t MAP_CACHE_MAX = 512;

int tensor_maps(const uint32_t *W, const uint16_t *s, const uint16_t *b, int N, int K, int bits,
                int group, const Plan &pl, QmmParams &P) {
    const MapKey key{W, s, b, N, K, bits, group, pl.mt};
    auto it = g_maps.find(key);
    if (it == g_maps.end()) {
        int rc = get_encoder();
        if (rc) return rc;
        MapSet ms;
        const long long segw = SEG * bits / 32, rowb = (long long)K * bits / 8;
        // W as {segment words, rows, segments}: a box of 16 rows x 8 segments of
        // one stage lands segment-major with a row pitch of segment + 16 bytes
        // (the 4 words past each segment's extent are zero-filled, not read).
        rc = encode_3d(&ms.W, W, CU_TENSOR_MAP_DATA_TYPE_UINT32, segw, N, K / SEG, rowb, segw * 4,
                       (int)segw + seg_pad_words(bits, group), TN * pl.mt, SEGS);
        const int sbg = CHUNK / group;
        for (int i = 0; i < 2 && !rc; ++i) {
            CUtensorMap *m = i ? &ms.b : &ms.s;
            const void *base = i ? (const void *)b : (const void *)s;
            if (pl.sb3d)   // {stage groups, stages, rows}, box padded by 8 zero-filled groups
                rc = encode_3d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT16, sbg, K / CHUNK, N, sbg * 2,
                               (long long)(K / group) * 2, sbg + 8, 1, TN * pl.mt);
            else
                rc = encode_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / group, N, sbg, TN * pl.mt);
        }
        if (rc) return rc;
        if (g_maps.size() >= MAP_CACHE_MAX) g_maps.clear();
        it = g_maps.emplace(key, ms).first;
    }
    P.tmW = it->second.W;
    P.tmS = it->second.s;
    P.tmB = it->second.b;
    return TF_OK;
}

// ----------------------------------------------------- per-stream storage --

struct StreamWs {
    float *ws = nullptr;
    size_t ws_floats = 0;
    int *cnt = nullptr;
    size_t n_cnt = 0;
};

struct DevState {
    int nsm = 0;
    int *status = nullptr;
};

std::mutex g_mu;
std::atomic<int> g_launch_mode{0};
std::atomic<int> g_stall{0};          // test hook armed by tf_inject_stall (one launch)
#ifdef TF_DEBUG_BOUNDS
std::atomic<int> g_shrink{0};         // debug hook: rows to drop from the next launch's y extent
#endif
std::map<int, DevState> g_dev;
std::map<std::pair<int, cudaStream_t>, StreamWs> g_ws;

int dev_state(DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DevState &d = g_dev[dev];
    if (!d.nsm) {
        e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaMalloc(&d.status, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
        e = cudaMemset(d.status, 0, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    }
    *out = &d;
    return TF_OK;
}

int stream_ws(cudaStream_t st, size_t floats, size_t counters, StreamWs **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    StreamWs &w = g_ws[{dev, st}];
    if (w.ws_floats < floats) {
        if (w.ws) cudaFree(w.ws);
        w.ws = nullptr;
        w.ws_floats = 0;
        e = cudaMalloc(&w.ws, floats * sizeof(float));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
        w.ws_floats = floats;
    }
    if (w.n_cnt < counters) {
        if (w.cnt) cudaFree(w.cnt);
        w.cnt = nullptr;
        w.n_cnt = 0;
        e = cudaMalloc(&w.cnt, counters * sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(counters)");
        e = cudaMemsetAsync(w.cnt, 0, counters * sizeof(int), st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counters)");
        w.n_cnt = counters;
    }
    *out = &w;
    return TF_OK;
}

cudaError_t launch(int bits, int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                   cudaStream_t st, bool pdl) {
    switch (bits) {
        case 2: return launch_b2(group, rb, mt, cg, P, grid, smem, st, pdl);
        case 3: return launch_b3(group, rb, mt, cg, P, grid, smem, st, pdl);
        case 4: return launch_b4(group, rb, mt, cg, P, grid, smem, st, pdl);
        case 5: return launch_b5(group, rb, mt, cg, P, grid, smem, st, pdl);
        case 6: return launch_b6(group, rb, mt, cg, P, grid, smem, st, pdl);
        case 8: return launch_b8(group, rb, mt, cg, P, grid, smem, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

// One run (matrix) written through `nseg` column segments.
// Output options and row maps of one launch: window row r reads x row xrow[r]
// and writes y row yrow[r] (identity without a map).
struct Io {
    int out = 0;            // OUT_BF16 | OUT_RELU2
    bool map = false;
    int xrow[16] = {}, yrow[16] = {};
    int x_rows = 0, y_rows = 0;   // rows of the call's x and y (0: the launch's rows)
};

int run_product(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *s,
                const uint16_t *b, int N, int bits, int group, float *y, int64_t y_stride,
                int nseg, const int *seg_src, const int *seg_len, const int *seg_dst,
                cudaStream_t st, int stack_pos = -1, const Io *io = nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    DevState *d = nullptr;
    int rc = dev_state(&d);
    if (rc) return rc;
    const bool bulk = aligned(s, 16) && aligned(b, 16) && K % SEG == 0 && K % (8 * group) == 0;
    const bool sb3d = bulk && K % CHUNK == 0;
    // Early x: the kernel before this launch writes neither x nor the weights.
    // That holds for every run of a stack, window of a long call or gather
    // launch too (they only share x), so each launch then computes before its
    // dependency wait and waits only before its first write and at its exit.
    const int mode = g_launch_mode.load(std::memory_order_relaxed);
    const bool overlap = (mode & TF_LAUNCH_EARLY_X) != 0;
    const Plan pl = make_plan(N, K, bits, group, rows, d->nsm, sb3d, overlap);
    if (pl.cg > 1 && pl.nsl != 1) return fail(TF_EINVAL_SIZE, "internal: two consumer groups need one K slice");
    QmmParams P{};
    P.x = x;
    P.W = W;
    P.s = s;
    P.b = b;
    P.y = y;
    P.status = d->status;
    P.y_stride = y_stride;
    P.rows = rows;
    P.K = K;
    P.N = N;
    P.nmt = pl.nmt;
    P.nsl = pl.nsl;
    P.sl = pl.sl;
    P.nchunks = pl.nchunks;
    P.stages = pl.stages;
    P.bulk = bulk;
    P.sb3d = sb3d;
    if (bulk) {
        rc = tensor_maps(W, s, b, N, K, bits, group, pl, P);
        if (rc) return rc;
    }
    P.sbpitch = pl.sbpitch;
    P.stage_bytes = pl.stage_bytes;
    P.x_off = pl.x_off;
    P.sx_off = pl.sx_off;
    P.pb_off = pl.pb_off;
    P.z_off = pl.z_off;
    P.st_off = pl.st_off;
    P.ncs = nseg;
    for (int i = 0; i < nseg; ++i) {
        P.cs_src[i] = seg_src[i];
        P.cs_len[i] = seg_len[i];
        P.cs_dst[i] = seg_dst[i];
    }
    P.out = io ? io->out : 0;
    for (int r = 0; r < 16; ++r) {
        P.xrow[r] = io && io->map ? io->xrow[r] : r;
        P.yrow[r] = io && io->map ? io->yrow[r] : r;
    }
    P.x_rows = io && io->x_rows ? io->x_rows : rows;
    P.y_rows = io && io->y_rows ? io->y_rows : rows;
#ifdef TF_DEBUG_BOUNDS
    P.y_rows -= g_shrink.exchange(0);
#endif
    if (pl.nsl > 1) {
        StreamWs *w = nullptr;
        rc = stream_ws(st, (size_t)pl.nchunks * rows * N, (size_t)pl.nmt, &w);
        if (rc) return rc;
        P.ws = w->ws;
        P.counters = w->cnt;
        P.ws_elems = (long long)pl.nchunks * rows * N;
        P.n_counters = pl.nmt;
    }
    P.early_x = overlap;
    P.early_w = (mode & TF_LAUNCH_EARLY_WEIGHTS) != 0 || P.early_x;
    P.stall = g_stall.exchange(0);
    // Runs of a stack read x and write disjoint columns: after the first, a run
    // without split-K overlaps the runs before it (see QmmParams::dep).
    P.dep = stack_pos < 0 || overlap ? 0 : stack_pos == 0 ? 1 : pl.nsl == 1 ? 2 : 0;
    const cudaError_t e = launch(bits, group, pl.rb, pl.mt, pl.cg, P, pl.grid, pl.smem, st,
                                 (mode & (TF_LAUNCH_PDL | TF_LAUNCH_EARLY_WEIGHTS | TF_LAUNCH_EARLY_X)) != 0);
    if (e != cudaSuccess) return cuda_fail(e, "qmm kernel launch");
    return TF_OK;
}

// ------------------------------------------------------------------ widen --

// One thread re-packs 32 consecutive codes of one row (bits_in words in,
// bits_out words out); every code keeps its integer value.
__global__ void widen_codes(const uint32_t *W, uint32_t *Wo, long long N, int K, int bi, int bo) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const long long runs = K / 32;
    if (t >= N * runs) return;
    const long long n = t / runs, j = t - n * runs;
    const uint32_t *src = W + n * ((long long)K * bi / 32) + j * bi;
    uint32_t *dst = Wo + n * ((long long)K * bo / 32) + j * bo;
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const uint32_t mask = (1u << bi) - 1u;
    for (int i = 0; i < 32; ++i) {
        const int ib = i * bi, w = ib >> 5, sh = ib & 31;
        const uint64_t v = ((uint64_t)(w + 1 < bi ? src[w + 1] : 0u) << 32) | src[w];
        const uint32_t c = (uint32_t)(v >> sh) & mask;
        const int ob = i * bo, ow = ob >> 5, osh = ob & 31;
        out[ow] |= c << osh;
        if (osh + bo > 32) out[ow + 1] |= c >> (32 - osh);
    }
    for (int w = 0; w < bo; ++w) dst[w] = out[w];
}

// Each finer group copies its parent group's scale and bias.
__global__ void widen_groups(const uint16_t *s, const uint16_t *b, uint16_t *so, uint16_t *bo,
                             long long N, int ngi, int ngo, int ratio) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= N * ngo) return;
    const long long n = t / ngo, g = t - n * ngo;
    so[t] = s[n * ngi + g / ratio];
    bo[t] = b[n * ngi + g / ratio];
}

// One launch of up to 16 rows with caller-provided scratch: window rows
// r0 .. r0 + w - 1 of x and y (w <= 16).  Allocates nothing: the tensor maps
// are encoded into the launch parameters, no cache is grown.
int window_with_scratch(const uint16_t *x, int w, int r0, int total_rows, int K, const uint32_t *W,
                        const uint16_t *s, const uint16_t *b, int N, int bits, int group, float *y,
                        int64_t y_stride, cudaStream_t st, int nsm, float *ws, int *counters, int *status) {
    const bool bulk = aligned(s, 16) && aligned(b, 16) && K % SEG == 0 && K % (8 * group) == 0;
    const bool sb3d = bulk && K % CHUNK == 0;
    const Plan pl = make_plan(N, K, bits, group, w, nsm, sb3d);
    QmmParams P{};
    P.x = x;
    P.W = W;
    P.s = s;
    P.b = b;
    P.y = y;
    P.status = status;
    P.y_stride = y_stride;
    P.rows = w;
    P.K = K;
    P.N = N;
    P.nmt = pl.nmt;
    P.nsl = pl.nsl;
    P.sl = pl.sl;
    P.nchunks = pl.nchunks;
    P.stages = pl.stages;
    P.bulk = bulk;
    P.sb3d = sb3d;
    int rc = TF_OK;
    if (bulk) {
        rc = get_encoder();
        if (rc) return rc;
        const long long segw = SEG * bits / 32, rowb = (long long)K * bits / 8;
        rc = encode_3d(&P.tmW, W, CU_TENSOR_MAP_DATA_TYPE_UINT32, segw, N, K / SEG, rowb, segw * 4,
                       (int)segw + seg_pad_words(bits, group), TN * pl.mt, SEGS);
        const int sbg = CHUNK / group;
        for (int i = 0; i < 2 && !rc; ++i) {
            CUtensorMap *m = i ? &P.tmB : &P.tmS;
            const void *base = i ? (const void *)b : (const void *)s;
            if (sb3d)
                rc = encode_3d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT16, sbg, K / CHUNK, N, sbg * 2,
                               (long long)(K / group) * 2, sbg + 8, 1, TN * pl.mt);
            else
                rc = encode_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / group, N, sbg, TN * pl.mt);
        }
        if (rc) return rc;
    }
    P.sbpitch = pl.sbpitch;
    P.stage_bytes = pl.stage_bytes;
    P.x_off = pl.x_off;
    P.sx_off = pl.sx_off;
    P.pb_off = pl.pb_off;
    P.z_off = pl.z_off;
    P.st_off = pl.st_off;
    P.ncs = 1;
    P.cs_src[0] = 0;
    P.cs_len[0] = N;
    P.cs_dst[0] = 0;
    for (int r = 0; r < 16; ++r) P.xrow[r] = P.yrow[r] = r0 + std::min(r, w - 1);
    P.x_rows = P.y_rows = total_rows;
    P.stall = g_stall.exchange(0);
    cudaError_t e;
    if (pl.nsl > 1) {
        // The scratch keeps the last call's contents: the arrival counters must start at zero.
        e = cudaMemsetAsync(counters, 0, (size_t)pl.nmt * sizeof(int), st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch counters)");
        P.ws = ws;
        P.counters = counters;
        P.ws_elems = (long long)pl.nchunks * w * N;
        P.n_counters = pl.nmt;
    }
    e = launch(bits, group, pl.rb, pl.mt, pl.cg, P, pl.grid, pl.smem, st, false);
    if (e != cudaSuccess) return cuda_fail(e, "qmm kernel launch");
    return TF_OK;
}

}  // namespace

// Product with caller-provided scratch: the split-K partials, arrival counters
// and status word live in memory the caller owns (used by tf_qmm_noalloc).
// More than 16 rows run as 16-row windows, one launch after another on the
// stream, each reusing the scratch.  Every window's need is checked before the
// first launch.
int tfq::product_with_scratch(const uint16_t *x, int rows, int K, const uint32_t *W,
                              const uint16_t *s, const uint16_t *b, int N, int bits, int group,
                              float *y, int64_t y_stride, cudaStream_t st, int nsm, float *ws,
                              size_t ws_floats, int *counters, size_t n_counters, int *status) {
    g_err.clear();
    int rc = check_matrix(K, W, s, b, N, bits, group);
    if (rc) return rc;
    rc = check_io(x, rows, y, MAX_ROWS);
    if (rc) return rc;
    if (y_stride < N) return fail(TF_EINVAL_STRIDE, "y_stride below N is refused");
    const bool bulk = aligned(s, 16) && aligned(b, 16) && K % SEG == 0 && K % (8 * group) == 0;
    const bool sb3d = bulk && K % CHUNK == 0;
    // Windows hold 16 rows, the last one rows % 16 if that is not zero.
    for (int w : {std::min(16, rows), rows % 16}) {
        if (w == 0) continue;
        const Plan pl = make_plan(N, K, bits, group, w, nsm, sb3d);
        if (pl.nsl > 1 && ((size_t)pl.nchunks * w * N > ws_floats || (size_t)pl.nmt > n_counters))
            return fail(TF_EINVAL_SIZE, "split-K partials (" + std::to_string((size_t)pl.nchunks * w * N * 4) +
                                            " bytes) exceed the fixed scratch of the no-allocation entry point");
    }
    for (int r0 = 0; r0 < rows; r0 += 16) {
        rc = window_with_scratch(x, std::min(16, rows - r0), r0, rows, K, W, s, b, N, bits, group, y, y_stride, st,
                                 nsm, ws, counters, status);
        if (rc) return rc;
    }
    return TF_OK;
}

int tfq::fail_message(int code, const char *msg) { return fail(code, msg); }

int tfq::cuda_error(cudaError_t e, const char *where) { return cuda_fail(e, where); }

#ifdef TF_TRACE
// Per-device trace buffers (records, counter), allocated at the first traced
// launch; a failed allocation leaves the launch untraced.
namespace {
std::mutex g_tmu;
std::map<int, std::pair<unsigned long long *, unsigned *>> g_tbuf;
std::atomic<unsigned> g_tseq{0};
}  // namespace

tfq::QmmParams tfq::trace_params(const QmmParams &P) {
    QmmParams Q = P;
    Q.trace = nullptr;
    Q.trace_n = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q;
    std::lock_guard<std::mutex> lk(g_tmu);
    auto &b = g_tbuf[dev];
    if (!b.first) {
        unsigned long long *rec = nullptr;
        unsigned *cnt = nullptr;
        if (cudaMalloc(&rec, (size_t)TRACE_MAX * TRACE_SLOTS * 8) != cudaSuccess) return Q;
        if (cudaMalloc(&cnt, 4) != cudaSuccess || cudaMemset(cnt, 0, 4) != cudaSuccess) {
            cudaFree(rec);
            if (cnt) cudaFree(cnt);
            return Q;
        }
        b = {rec, cnt};
    }
    Q.trace = b.first;
    Q.trace_n = b.second;
    Q.trace_seq = g_tseq.fetch_add(1);
    return Q;
}
#endif

int tfq::check_product(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *s,
                       const uint16_t *b, int N, int bits, int group, const float *y, int64_t y_stride) {
    g_err.clear();
    int rc = check_matrix(K, W, s, b, N, bits, group);
    if (rc) return rc;
    rc = check_io(x, rows, y, MAX_ROWS);
    if (rc) return rc;
    if (y_stride < N) return fail(TF_EINVAL_STRIDE, "y_stride below N is refused");
    return TF_OK;
}

int tfq::tensor_map_2d(CUtensorMap *m, const void *base, int elem_bytes, long long cols, long long rows,
                       int box_cols, int box_rows) {
    const int rc = get_encoder();
    if (rc) return rc;
    const CUtensorMapDataType t = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                  : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return encode_2d(m, base, t, elem_bytes, cols, rows, box_cols, box_rows);
}

int tfq::tensor_map_3d(CUtensorMap *m, const void *base, int elem_bytes, long long d0, long long d1, long long d2,
                       long long s1, long long s2, int b0, int b1, int b2) {
    const int rc = get_encoder();
    if (rc) return rc;
    const CUtensorMapDataType t = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                  : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return encode_3d(m, base, t, d0, d1, d2, s1, s2, b0, b1, b2);
}

int tfq::device_info(int *nsm, int **status) {
    std::lock_guard<std::mutex> lk(g_mu);
    DevState *d = nullptr;
    const int rc = dev_state(&d);
    if (rc) return rc;
    *nsm = d->nsm;
    *status = d->status;
    return TF_OK;
}

// ============================================================== C ABI ====

// A product of any row count: up to 16 rows in one launch; more as 16-row
// windows (rows r0..r0+15 read x rows and write y rows r0..), which run as
// independent launches and overlap like the runs of a stack.  Each row's bits
// are those of the row alone.
int product_rows(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *s,
                 const uint16_t *b, int N, int bits, int group, float *y, int64_t y_stride, int out,
                 cudaStream_t st) {
    const int src = 0, len = N, dst = 0;
    Io io;
    io.out = out;
    if (rows <= 16) return run_product(x, rows, K, W, s, b, N, bits, group, y, y_stride, 1, &src, &len, &dst, st, -1, &io);
    io.map = true;
    io.x_rows = io.y_rows = rows;
    int pos = 0;
    for (int r0 = 0; r0 < rows; r0 += 16) {
        const int w = std::min(16, rows - r0);
        for (int r = 0; r < 16; ++r) io.xrow[r] = io.yrow[r] = r0 + std::min(r, w - 1);
        const int rc = run_product(x, w, K, W, s, b, N, bits, group, y, y_stride, 1, &src, &len, &dst, st, pos++, &io);
        if (rc) return rc;
    }
    return TF_OK;
}

extern "C" {

int tf_qmm(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *scales,
           const uint16_t *biases, int N, int bits, int group, float *y, int64_t y_stride,
           void *stream) {
    g_err.clear();
    int rc = check_matrix(K, W, scales, biases, N, bits, group);
    if (rc) return rc;
    rc = check_io(x, rows, y, MAX_ROWS);
    if (rc) return rc;
    if (y_stride < N) return fail(TF_EINVAL_STRIDE, "y_stride below N is refused");
    return product_rows(x, rows, K, W, scales, biases, N, bits, group, y, y_stride, 0,
                        static_cast<cudaStream_t>(stream));
}

int tf_qmm_stack(const uint16_t *x, int rows, int K, const tf_run *runs, int n_runs,
                 const tf_member *members, int n_members, float *y, int64_t y_stride,
                 void *stream) {
    g_err.clear();
    int rc = check_io(x, rows, y);
    if (rc) return rc;
    if (!runs || !members || n_runs < 1 || n_members < 1)
        return fail(TF_ESTACK, "empty run or member table");
    for (int i = 0; i < n_runs; ++i) {
        rc = check_matrix(K, runs[i].W, runs[i].scales, runs[i].biases, runs[i].N, runs[i].bits,
                          runs[i].group);
        if (rc) return rc;
    }
    for (int i = 0; i < n_members; ++i) {
        const tf_member &m = members[i];
        if (m.run < 0 || m.run >= n_runs) return fail(TF_ESTACK, "member names a missing run");
        if (m.n_cols < 1 || m.src_col < 0 || m.src_col + m.n_cols > runs[m.run].N)
            return fail(TF_ESTACK, "member columns outside its run");
        if (m.dst_col < 0 || (int64_t)m.dst_col + m.n_cols > y_stride)
            return fail(TF_ESTACK, "member destination past y_stride");
        for (int j = 0; j < i; ++j) {
            const tf_member &o = members[j];
            if (m.dst_col < o.dst_col + o.n_cols && o.dst_col < m.dst_col + m.n_cols)
                return fail(TF_ESTACK, "member destinations overlap");
            if (m.run == o.run && m.src_col < o.src_col + o.n_cols && o.src_col < m.src_col + m.n_cols)
                return fail(TF_ESTACK, "members take overlapping columns of one run");
        }
    }
    int pos = 0;                                    // launched runs so far
    for (int r = 0; r < n_runs; ++r) {
        int src[MAXCOLSEG], len[MAXCOLSEG], dst[MAXCOLSEG], n = 0;
        for (int i = 0; i < n_members; ++i) {
            if (members[i].run != r) continue;
            if (n == MAXCOLSEG) return fail(TF_ESTACK, "more than 16 members in one run");
            src[n] = members[i].src_col;
            len[n] = members[i].n_cols;
            dst[n] = members[i].dst_col;
            ++n;
        }
        if (n == 0) continue;
        rc = run_product(x, rows, K, runs[r].W, runs[r].scales, runs[r].biases, runs[r].N,
                         runs[r].bits, runs[r].group, y, y_stride, n, src, len, dst,
                         static_cast<cudaStream_t>(stream), pos++);
        if (rc) return rc;
    }
    return TF_OK;
}

int tf_qmm_ex(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *scales,
              const uint16_t *biases, int N, int bits, int group, void *y, int64_t y_stride,
              int flags, void *stream) {
    g_err.clear();
    if (flags & ~(TF_OUT_BF16 | TF_EPI_RELU2)) return fail(TF_EINVAL_FLAGS, "unknown output flags");
    int rc = check_matrix(K, W, scales, biases, N, bits, group);
    if (rc) return rc;
    if (rows < 1 || rows > MAX_ROWS) return fail(TF_EINVAL_ROWS, "rows must be in [1, 65536]");
    if (!x || !y || !aligned(x, 16) || !aligned(y, (flags & TF_OUT_BF16) ? 2 : 4))
        return fail(TF_EINVAL_PTR, "NULL pointer, x not 16-byte aligned, or y not aligned to its type");
    if (y_stride < N) return fail(TF_EINVAL_STRIDE, "y_stride below N is refused");
    return product_rows(x, rows, K, W, scales, biases, N, bits, group, static_cast<float *>(y), y_stride,
                        flags, static_cast<cudaStream_t>(stream));
}

int tf_qmm_gather(const uint16_t *x, int x_rows, int K, const tf_run *experts, int n_experts,
                  const int *slot_expert, const int *slot_row, int n_slots, void *y,
                  int64_t y_stride, int flags, void *stream) {
    g_err.clear();
    if (flags & ~(TF_OUT_BF16 | TF_EPI_RELU2)) return fail(TF_EINVAL_FLAGS, "unknown output flags");
    if (!x || !y || !aligned(x, 16) || !aligned(y, (flags & TF_OUT_BF16) ? 2 : 4))
        return fail(TF_EINVAL_PTR, "NULL pointer, x not 16-byte aligned, or y not aligned to its type");
    if (x_rows < 1) return fail(TF_EINVAL_ROWS, "x_rows must be at least 1");
    if (!experts || n_experts < 1 || !slot_expert || !slot_row || n_slots < 1)
        return fail(TF_EGATHER, "empty expert or slot table");
    for (int i = 0; i < n_slots; ++i) {
        if (slot_expert[i] < 0 || slot_expert[i] >= n_experts)
            return fail(TF_EGATHER, "a slot names a missing expert");
        if (slot_row[i] < 0 || slot_row[i] >= x_rows) return fail(TF_EGATHER, "a slot names a missing x row");
    }
    for (int e = 0; e < n_experts; ++e) {
        int used = 0;
        for (int i = 0; i < n_slots && !used; ++i) used = slot_expert[i] == e;
        if (!used) continue;
        const int rc = check_matrix(K, experts[e].W, experts[e].scales, experts[e].biases, experts[e].N,
                                    experts[e].bits, experts[e].group);
        if (rc) return rc;
        if (y_stride < experts[e].N) return fail(TF_EINVAL_STRIDE, "y_stride below an expert's N is refused");
    }
    // Slots grouped by expert in slot order, at most 16 to a launch; every
    // launch reads x and writes its own y rows, so they may overlap (as stack runs).
    int pos = 0;
    for (int e = 0; e < n_experts; ++e) {
        Io io;
        io.out = flags;
        io.map = true;
        io.x_rows = x_rows;
        io.y_rows = n_slots;
        int n = 0;
        for (int i = 0; i <= n_slots; ++i) {
            const bool take = i < n_slots && slot_expert[i] == e;
            if (take) {
                io.xrow[n] = slot_row[i];
                io.yrow[n] = i;
                ++n;
            }
            if (n == 16 || (i == n_slots && n > 0)) {
                const int src = 0, len = experts[e].N, dst = 0;
                const int rc = run_product(x, n, K, experts[e].W, experts[e].scales, experts[e].biases,
                                           experts[e].N, experts[e].bits, experts[e].group,
                                           static_cast<float *>(y), y_stride, 1, &src, &len, &dst,
                                           static_cast<cudaStream_t>(stream), pos++, &io);
                if (rc) return rc;
                n = 0;
            }
        }
    }
    return TF_OK;
}

int tf_widen(const uint32_t *W, const uint16_t *scales, const uint16_t *biases, int N, int K,
             int bits, int group, uint32_t *W_out, uint16_t *s_out, uint16_t *b_out, int bits_out,
             int group_out, void *stream) {
    g_err.clear();
    int rc = check_matrix(K, W, scales, biases, N, bits, group);
    if (rc) return rc;
    if (!valid_bits(bits_out)) return fail(TF_EINVAL_BITS, "bits_out must be 2, 3, 4, 5, 6 or 8");
    if (!valid_group(group_out)) return fail(TF_EINVAL_GROUP, "group_out must be 32, 64 or 128");
    if (bits_out < bits) return fail(TF_ENARROW, "narrowing bits is refused");
    if (group_out > group || group % group_out != 0)
        return fail(TF_EGROUP, "a group that does not divide the source group is refused");
    if (!W_out || !s_out || !b_out) return fail(TF_EINVAL_PTR, "NULL output pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long nrun = (long long)N * (K / 32);
    widen_codes<<<(unsigned)((nrun + 255) / 256), 256, 0, st>>>(W, W_out, N, K, bits, bits_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "widen_codes launch");
    const long long ng = (long long)N * (K / group_out);
    widen_groups<<<(unsigned)((ng + 255) / 256), 256, 0, st>>>(scales, biases, s_out, b_out, N,
                                                               K / group, K / group_out,
                                                               group / group_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "widen_groups launch");
    return TF_OK;
}

int tf_widen_host(const uint32_t *W, const uint16_t *scales, const uint16_t *biases, int N, int K,
                  int bits, int group, uint32_t *W_out, uint16_t *s_out, uint16_t *b_out, int bits_out,
                  int group_out) {
    g_err.clear();
    int rc = check_matrix(K, W, scales, biases, N, bits, group);
    if (rc) return rc;
    if (!valid_bits(bits_out)) return fail(TF_EINVAL_BITS, "bits_out must be 2, 3, 4, 5, 6 or 8");
    if (!valid_group(group_out)) return fail(TF_EINVAL_GROUP, "group_out must be 32, 64 or 128");
    if (bits_out < bits) return fail(TF_ENARROW, "narrowing bits is refused");
    if (group_out > group || group % group_out != 0)
        return fail(TF_EGROUP, "a group that does not divide the source group is refused");
    if (!W_out || !s_out || !b_out) return fail(TF_EINVAL_PTR, "NULL output pointer");
    // Every 32 codes of a row fill exactly `bits` words in and `bits_out` words
    // out; each code keeps its integer value.
    const long long wi = (long long)K * bits / 32, wo = (long long)K * bits_out / 32;
    const uint32_t mask = (1u << bits) - 1u;
    for (long long n = 0; n < N; ++n) {
        const uint32_t *src = W + n * wi;
        uint32_t *dst = W_out + n * wo;
        for (long long w = 0; w < wo; ++w) dst[w] = 0u;
        for (long long k = 0; k < K; ++k) {
            const long long ib = k * bits, ob = k * bits_out;
            const long long iw = ib >> 5, ow = ob >> 5;
            const int ish = (int)(ib & 31), osh = (int)(ob & 31);
            uint64_t v = src[iw];
            if (iw + 1 < wi) v |= (uint64_t)src[iw + 1] << 32;
            const uint64_t c = (v >> ish) & mask;
            dst[ow] |= (uint32_t)(c << osh);
            if (osh + bits_out > 32) dst[ow + 1] |= (uint32_t)(c >> (32 - osh));
        }
    }
    const long long ngi = K / group, ngo = K / group_out, ratio = group / group_out;
    for (long long n = 0; n < N; ++n)
        for (long long g = 0; g < ngo; ++g) {
            s_out[n * ngo + g] = scales[n * ngi + g / ratio];
            b_out[n * ngo + g] = biases[n * ngi + g / ratio];
        }
    return TF_OK;
}

int tf_common_width(const int *bits, const int *groups, int n, int *bits_out, int *group_out) {
    g_err.clear();
    if (!bits || !groups || !bits_out || !group_out || n < 1)
        return fail(TF_EINVAL_PTR, "empty member list");
    int b = 0, g = 1 << 30;
    for (int i = 0; i < n; ++i) {
        if (!valid_bits(bits[i])) return fail(TF_EINVAL_BITS, "unsupported member bits");
        if (!valid_group(groups[i])) return fail(TF_EINVAL_GROUP, "unsupported member group");
        b = std::max(b, bits[i]);
        g = std::min(g, groups[i]);
    }
    *bits_out = b;
    *group_out = g;
    return TF_OK;
}

int tf_qmm_bytes(int N, int K, int bits, int group, int64_t *w_bytes, int64_t *sb_bytes) {
    g_err.clear();
    if (!valid_bits(bits)) return fail(TF_EINVAL_BITS, "bits must be 2, 3, 4, 5, 6 or 8");
    if (!valid_group(group) || K < group || K % group) return fail(TF_EINVAL_GROUP, "bad group");
    if (N < 1) return fail(TF_EINVAL_SIZE, "N must be >= 1");
    if (w_bytes) *w_bytes = (int64_t)N * K * bits / 8;
    if (sb_bytes) *sb_bytes = (int64_t)N * (K / group) * 2;
    return TF_OK;
}

int tf_device_status(void) {
    g_err.clear();
    std::lock_guard<std::mutex> lk(g_mu);
    DevState *d = nullptr;
    int rc = dev_state(&d);
    if (rc) return rc;
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    if (v) {
        e = cudaMemset(d->status, 0, sizeof v);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
        if (v & STATUS_BOUNDS) return fail(TF_EBOUNDS, "the debug build found an index outside its buffer");
        return fail(TF_EDEVICE, "a kernel gave up a bounded wait");
    }
    return TF_OK;
}

int tf_set_launch_mode(int mode) {
    g_err.clear();
    if (mode & ~(TF_LAUNCH_PDL | TF_LAUNCH_EARLY_WEIGHTS | TF_LAUNCH_EARLY_X))
        return fail(TF_EINVAL_SIZE, "unknown launch mode bits");
    return g_launch_mode.exchange(mode);
}

int tf_inject_stall(void) {
    g_err.clear();
    g_stall.store(1);
    return TF_OK;
}

#ifdef TF_TRACE
int tf_trace_reset(void) {
    g_err.clear();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_tmu);
    auto it = g_tbuf.find(dev);
    if (it != g_tbuf.end()) {
        e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaMemset(it->second.second, 0, 4);
        if (e == cudaSuccess) e = cudaMemset(it->second.first, 0, (size_t)TRACE_MAX * TRACE_SLOTS * 8);
        if (e != cudaSuccess) return cuda_fail(e, "trace reset");
    }
    g_tseq.store(0);
    return TF_OK;
}

int tf_trace_read(uint64_t *buf, int max_records) {
    g_err.clear();
    if (!buf || max_records < 0) return fail(TF_EINVAL_PTR, "buf must be a host array of max_records records");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_tmu);
    auto it = g_tbuf.find(dev);
    if (it == g_tbuf.end()) return 0;
    e = cudaDeviceSynchronize();
    unsigned n = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&n, it->second.second, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "trace read");
    const int k = (int)std::min<unsigned>(std::min<unsigned>(n, (unsigned)TRACE_MAX), (unsigned)max_records);
    if (k > 0) {
        e = cudaMemcpy(buf, it->second.first, (size_t)k * TRACE_SLOTS * 8, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "trace read");
    }
    return k;
}
#endif

#ifdef TF_DEBUG_BOUNDS
int tf_debug_shrink_y(int rows) {
    g_err.clear();
    if (rows < 0 || rows > 16) return fail(TF_EINVAL_ROWS, "rows must be in [0, 16]");
    g_shrink.store(rows);
    return TF_OK;
}
#endif

const char *tf_last_error_string(void) { return g_err.c_str(); }

const char *tf_version(void) { return "tfqmm 0.1.0 (sm_103a)"; }

}  // extern "C"
