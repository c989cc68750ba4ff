// qmm_kernel.cuh -- the MLX-affine quantized row product for sm_103a.
//
// y[r][n] = sum_k x[r][k] * (scale[n][k/G] * q[n][k] + bias[n][k/G]), 1..16 rows
// (TensorFold PR #788, commit "every MLX affine width in the row kernel"; the
// group-sum form with fp32 group sums, PR #774 Exactness, Precision bullet).
//
// One CTA = 8 consumer warps + 1 producer warp, persistent over work items
// (a tile of 128 output columns x one K slice).  The producer streams each
// item's packed codes and scales/biases into a ring of shared-memory stages
// with cp.async.bulk (TMA, completion on mbarriers).  Each consumer warp owns
// 16 columns: it unpacks 8-code runs straight into bf16 A fragments (codes
// exact), multiplies them by the activations with mma.sync m16n8k16 (rows are
// the N dimension, so 1..8 rows cost one MMA and 9..16 two), and applies each
// group's scale and bias to the fp32 group sum in registers.
//
// Every wait on an mbarrier is bounded in time; on expiry the kernel records
// it in the device status word, stops waiting and runs to completion.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm_common.h"
#include "unpack.cuh"

namespace tfq {

// ------------------------------------------------------------ primitives --

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(tx)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;   // 2 s per wait

// Bounded wait for the phase of `parity`.  `abort` (shared) short-cuts every
// later wait once one has run out; `honor_abort` = false keeps waiting (the
// producer's final drain of its own copies).
__device__ __forceinline__ void mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *status, bool honor_abort = true) {
    if (mbar_try(bar, parity)) return;
    unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return;
        if ((it & 255u) == 0) {
            if (honor_abort && *abort) return;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                *abort = 1;
                atomicOr(status, 1);
                return;
            }
        }
    }
}

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ void named_bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

// ---------------------------------------------------------- item walking --

struct Item {
    int ct, slice, k_lo, k_hi;
};

__device__ __forceinline__ Item item_of(const QmmParams &P, int it) {
    Item I;
    I.slice = it / P.nct;
    I.ct = it - I.slice * P.nct;
    I.k_lo = I.slice * P.sl;
    I.k_hi = min(P.K, I.k_lo + P.sl);
    return I;
}

// Scale/bias placement of a stage: first group g0, `ng` groups, and the
// offset of g0 inside the copied row (bulk copies start on a 16-byte boundary).
template <int G>
__device__ __forceinline__ int sb_offset(const QmmParams &P, int g0, int ng) {
    return (P.bulk && ng * 2 < 16) ? (g0 & 7) : 0;
}

// -------------------------------------------------------------- producer --

template <int BITS, int G>
__device__ void producer(const QmmParams &P, uint8_t *smem, uint64_t *full, uint64_t *empty,
                         volatile int *abort) {
    constexpr int SK = stage_k(BITS);
    const int lane = threadIdx.x & 31;
    const int S = P.stages;
    const long long row_bytes = (long long)P.K * BITS / 8;
    const int ngK = P.K / G;
    if (P.bulk && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmW) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmS) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmB) : "memory");
    }
    uint32_t it = 0;
    for (int item = blockIdx.x; item < P.n_items; item += gridDim.x) {
        const Item I = item_of(P, item);
        const int n0 = I.ct * TN;
        const int nrows = min(TN, P.N - n0);
        for (int k0 = I.k_lo; k0 < I.k_hi; k0 += SK, ++it) {
            const int k1 = min(I.k_hi, k0 + SK);
            const int slot = it % S;
            mbar_wait(&empty[slot], ((it / S) & 1u) ^ 1u, abort, P.status);
            uint8_t *st = smem + P.st_off + slot * P.stage_bytes;
            uint8_t *sst = st + TN * P.wpitch;
            uint8_t *bst = sst + TN * P.sbpitch;
            const int wbytes = (k1 - k0) * BITS / 8;
            const int g0 = k0 / G, ng = (k1 - k0) / G;
            const int sboff = sb_offset<G>(P, g0, ng);
            if (P.bulk) {
                // One 2D tensor copy each for codes, scales and biases; rows past N
                // arrive zero-filled, and the full boxes count toward the bytes.
                if (lane == 0) {
                    mbar_arrive_tx(&full[slot], (uint32_t)P.stage_bytes);
                    tma_2d(st, &P.tmW, k0 * BITS / 32, n0, &full[slot]);
                    tma_2d(sst, &P.tmS, g0 - sboff, n0, &full[slot]);
                    tma_2d(bst, &P.tmB, g0 - sboff, n0, &full[slot]);
                }
            } else {
                // Odd shapes or alignments: plain 4-byte / 2-byte copies by the warp.
                const int wwords = wbytes / 4;
                for (int e = lane; e < nrows * wwords; e += 32) {
                    const int r = e / wwords, w = e - r * wwords;
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(
                        reinterpret_cast<const uint8_t *>(P.W) + (long long)(n0 + r) * row_bytes +
                        (long long)k0 * BITS / 8);
                    reinterpret_cast<uint32_t *>(st + r * P.wpitch)[w] = __ldg(src + w);
                }
                for (int e = lane; e < nrows * ng; e += 32) {
                    const int r = e / ng, g = e - r * ng;
                    const long long src = (long long)(n0 + r) * ngK + g0 + g;
                    reinterpret_cast<uint16_t *>(sst + r * P.sbpitch)[g] = __ldg(P.s + src);
                    reinterpret_cast<uint16_t *>(bst + r * P.sbpitch)[g] = __ldg(P.b + src);
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[slot]);
            }
        }
    }
    // Drain: the last stages' copies must land before the CTA may exit.
    if (P.bulk && lane == 0) {
        const uint32_t first = it > (uint32_t)S ? it - (uint32_t)S : 0u;
        for (uint32_t j = first; j < it; ++j)
            mbar_wait(&full[j % S], (j / S) & 1u, abort, P.status, false);
    }
}

// ------------------------------------------------------------- consumers --

// Activations of one K slice, permuted into mma B-fragment order, and the
// per-(group,row) sums of x.  Layout [k-step][R rows][4 quad lanes] of uint2
// with R = 8*NT (rows >= `rows` are zero), so every B load of a warp is one
// 8-byte access at a compile-time offset.  Entry (k-step, row, quad lane q)
// holds the four x values that meet quad lane q's four codes in that step:
// code i of an 8-code run is paired with code i+4, so a run x0..x7 feeds
// step 2m as {(x0,x4),(x1,x5)} and step 2m+1 as {(x2,x6),(x3,x7)}.
// sum_group(x) is the sequential fp32 sum of the group's x in k order.
template <int G, int NT>
__device__ void load_x_slice(const QmmParams &P, const Item &I, uint2 *Bf, float *sx, int tid) {
    constexpr int R = 8 * NT;
    const int rows = P.rows;
    const int ngs = (I.k_hi - I.k_lo) / G;
    for (int u = tid; u < R * ngs; u += NCW * 32) {
        const int r = u / ngs, gs = u - r * ngs;
        float acc = 0.f;
        const uint16_t *src = P.x + (long long)r * P.K + I.k_lo + gs * G;
#pragma unroll 4
        for (int t = 0; t < G / 8; ++t) {
            const int qq = (8 * t) / (G / 4), m = ((8 * t) % (G / 4)) / 8;
            const int ks = gs * (G / 16) + 2 * m;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows) v = *reinterpret_cast<const uint4 *>(src + 8 * t);
            Bf[(ks * R + r) * 4 + qq] = make_uint2(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u));
            Bf[((ks + 1) * R + r) * 4 + qq] = make_uint2(prmt(v.y, v.w, 0x5410u), prmt(v.y, v.w, 0x7632u));
            acc += bf16f((uint16_t)(v.x & 0xFFFF));
            acc += bf16f((uint16_t)(v.x >> 16));
            acc += bf16f((uint16_t)(v.y & 0xFFFF));
            acc += bf16f((uint16_t)(v.y >> 16));
            acc += bf16f((uint16_t)(v.z & 0xFFFF));
            acc += bf16f((uint16_t)(v.z >> 16));
            acc += bf16f((uint16_t)(v.w & 0xFFFF));
            acc += bf16f((uint16_t)(v.w >> 16));
        }
        sx[gs * R + r] = acc;
    }
}

// One group of this thread's two columns: T = tensor-core dot products of the
// group's exact codes with x, then p = fma(s,T,p); p = fma(b,sum_group(x),p).
// pr0/pr1[m]: run m of the thread's quarter in column rows g and g+8 (words);
// woff: the group's word offset in the stage row; bq: this lane's B entry of
// the group's first k-step; sxq: the group's sum_group(x) at rows 2q, 2q+1.
template <int BITS, int G, int NT>
__device__ __forceinline__ void group_body(const uint32_t *const (&pr0)[G / 32],
                                           const uint32_t *const (&pr1)[G / 32],
                                           const uint32_t (&sh)[G / 32], int woff, const uint2 *bq,
                                           const uint16_t *s0, const uint16_t *s1,
                                           const uint16_t *b0, const uint16_t *b1,
                                           const float *sxq, float (&p)[NT][4]) {
    constexpr int RUNS = G / 32, R = 8 * NT;
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
    for (int m = 0; m < RUNS; ++m) {
        uint32_t pa[4], pb[4];
        Unpack<BITS>::run(pr0[m] + woff, sh[m], pa);
        Unpack<BITS>::run(pr1[m] + woff, sh[m], pb);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint2 bb = bq[((2 * m + h) * R + nt * 8) * 4];
                mma_bf16(c[nt], pa[2 * h], pb[2 * h], pa[2 * h + 1], pb[2 * h + 1], bb.x, bb.y);
            }
    }
    const float sg0 = bf16f(*s0), bg0 = bf16f(*b0), sg1 = bf16f(*s1), bg1 = bf16f(*b1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float2 v = *reinterpret_cast<const float2 *>(sxq + nt * 8);
        p[nt][0] = fmaf(bg0, v.x, fmaf(sg0, c[nt][0], p[nt][0]));
        p[nt][1] = fmaf(bg0, v.y, fmaf(sg0, c[nt][1], p[nt][1]));
        p[nt][2] = fmaf(bg1, v.x, fmaf(sg1, c[nt][2], p[nt][2]));
        p[nt][3] = fmaf(bg1, v.y, fmaf(sg1, c[nt][3], p[nt][3]));
    }
}

__device__ __forceinline__ int dst_col(const QmmParams &P, int n) {
    for (int i = 0; i < P.nseg; ++i) {
        const int d = n - P.seg_src[i];
        if (d >= 0 && d < P.seg_len[i]) return P.seg_dst[i] + d;
    }
    return -1;
}

__device__ __forceinline__ void store_y(const QmmParams &P, int r, int n, float v) {
    if (r < P.rows && n < P.N) {
        const int d = dst_col(P, n);
        if (d >= 0) P.y[(long long)r * P.y_stride + d] = v;
    }
}

template <int BITS, int G, int NT>
__device__ void consumer(const QmmParams &P, uint8_t *smem, uint64_t *full, uint64_t *empty,
                         volatile int *abort, volatile int *flag) {
    constexpr int SK = stage_k(BITS);
    constexpr int NG = SK / G;               // groups in a full stage
    constexpr int QG = G / 4;                // codes of a group per quad lane
    constexpr int RUNS = G / 32;             // 8-code runs per quad lane per group
    constexpr int STEPS = G / 16;            // mma k-steps per group
    constexpr int GW = G * BITS / 32;        // words per group of one row
    constexpr int R = 8 * NT;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int S = P.stages, rows = P.rows;
    uint2 *Bf = reinterpret_cast<uint2 *>(smem + P.x_off);
    float *sx = reinterpret_cast<float *>(smem + P.sx_off);
    // This lane's runs inside any group: word offset and bit shift of run m.
    uint32_t wo[RUNS], sh[RUNS];
#pragma unroll
    for (int m = 0; m < RUNS; ++m) {
        const uint32_t bit = (uint32_t)(q * QG + 8 * m) * BITS;
        wo[m] = bit >> 5;
        sh[m] = bit & 31u;
    }
    const int row0 = warp * 16 + g;          // stage row of A row g (A row g+8 is row0+8)
    int cur_slice = -1;
    uint32_t it = 0;
    for (int item = blockIdx.x; item < P.n_items; item += gridDim.x) {
        const Item I = item_of(P, item);
        if (I.slice != cur_slice) {
            named_bar_consumers();
            load_x_slice<G, NT>(P, I, Bf, sx, tid);
            named_bar_consumers();
            cur_slice = I.slice;
        }
        const int col0 = I.ct * TN + row0;
        float p[NT][4], yv[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) p[nt][e] = yv[nt][e] = 0.f;

        for (int k0 = I.k_lo; k0 < I.k_hi; k0 += SK, ++it) {
            const int k1 = min(I.k_hi, k0 + SK);
            const int slot = it % S;
            mbar_wait(&full[slot], (it / S) & 1u, abort, P.status);
            const uint8_t *st = smem + P.st_off + slot * P.stage_bytes;
            const uint32_t *wr0 = reinterpret_cast<const uint32_t *>(st + row0 * P.wpitch);
            const uint32_t *wr1 = reinterpret_cast<const uint32_t *>(st + (row0 + 8) * P.wpitch);
            const uint32_t *pr0[RUNS], *pr1[RUNS];
#pragma unroll
            for (int m = 0; m < RUNS; ++m) {
                pr0[m] = wr0 + wo[m];
                pr1[m] = wr1 + wo[m];
            }
            const int ng = (k1 - k0) / G;
            const int sboff = sb_offset<G>(P, k0 / G, ng);
            const uint8_t *sbase = st + TN * P.wpitch;
            const uint16_t *s0 = reinterpret_cast<const uint16_t *>(sbase + row0 * P.sbpitch) + sboff;
            const uint16_t *s1 = reinterpret_cast<const uint16_t *>(sbase + (row0 + 8) * P.sbpitch) + sboff;
            const uint16_t *b0 = reinterpret_cast<const uint16_t *>(sbase + (TN + row0) * P.sbpitch) + sboff;
            const uint16_t *b1 = reinterpret_cast<const uint16_t *>(sbase + (TN + row0 + 8) * P.sbpitch) + sboff;
            const int gs0 = (k0 - I.k_lo) / G;
            const uint2 *bq = Bf + (gs0 * STEPS * R + g) * 4 + q;
            const float *sxq = sx + gs0 * R + 2 * q;
            if (ng == NG) {
#pragma unroll
                for (int gl = 0; gl < NG; ++gl)
                    group_body<BITS, G, NT>(pr0, pr1, sh, gl * GW, bq + gl * STEPS * R * 4, s0 + gl,
                                            s1 + gl, b0 + gl, b1 + gl, sxq + gl * R, p);
            } else {
#pragma unroll 1
                for (int gl = 0; gl < ng; ++gl)
                    group_body<BITS, G, NT>(pr0, pr1, sh, gl * GW, bq + gl * STEPS * R * 4, s0 + gl,
                                            s1 + gl, b0 + gl, b1 + gl, sxq + gl * R, p);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);

            if (k1 % CHUNK == 0 || k1 == P.K) {   // end of a canonical chunk
                const int chunk = (k1 - 1) / CHUNK;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (P.nsl == 1) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) yv[nt][e] = chunk == 0 ? p[nt][e] : yv[nt][e] + p[nt][e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = nt * 8 + 2 * q + (e & 1);
                            const int n = col0 + 8 * (e >> 1);
                            if (r < rows && n < P.N)
                                P.ws[((long long)chunk * rows + r) * P.N + n] = p[nt][e];
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) p[nt][e] = 0.f;
                }
            }
        }

        if (P.nsl == 1) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    store_y(P, nt * 8 + 2 * q + (e & 1), col0 + 8 * (e >> 1), yv[nt][e]);
        } else {
            // Split K: the last CTA to finish a column tile folds its chunk
            // partials in chunk order (an arrival ticket; nothing waits).
            __threadfence();
            named_bar_consumers();
            if (tid == 0) *flag = atomicAdd(&P.counters[I.ct], 1) == P.nsl - 1;
            named_bar_consumers();
            if (*flag) {
                __threadfence();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = nt * 8 + 2 * q + (e & 1);
                        const int n = col0 + 8 * (e >> 1);
                        if (r < rows && n < P.N) {
                            float v = __ldcg(P.ws + (long long)r * P.N + n);
                            for (int ch = 1; ch < P.nchunks; ++ch)
                                v = v + __ldcg(P.ws + ((long long)ch * rows + r) * P.N + n);
                            store_y(P, r, n, v);
                        }
                    }
                named_bar_consumers();
                if (tid == 0) P.counters[I.ct] = 0;
            }
        }
    }
}

// ------------------------------------------------------------------ kernel --

template <int BITS, int G, int NT>
__global__ void __launch_bounds__(NTHREADS, 2) qmm_kernel(const __grid_constant__ QmmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + MAX_STAGES;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + 16 * MAX_STAGES);
    volatile int *flag = abort + 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < P.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        *abort = 0;
        *flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= NCW * 32)
        producer<BITS, G>(P, smem, full, empty, abort);
    else
        consumer<BITS, G, NT>(P, smem, full, empty, abort, flag);
}

// Host-side launcher for one width: every group and row-tile count.
template <int BITS>
cudaError_t launch_width(int group, int nt, const QmmParams &P, int grid, int smem, cudaStream_t st) {
#define TFQ_CASE(G_, NT_)                                                                     \
    if (group == G_ && nt == NT_) {                                                           \
        auto k = qmm_kernel<BITS, G_, NT_>;                                                   \
        static unsigned attr_set = 0; /* one bit per device: smem limit raised */             \
        int dev = 0;                                                                          \
        cudaError_t e = cudaGetDevice(&dev);                                                  \
        if (e != cudaSuccess) return e;                                                       \
        const unsigned bit = 1u << (dev & 31);                                                \
        if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {                          \
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX); \
            if (e != cudaSuccess) return e;                                                   \
            __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);                              \
        }                                                                                     \
        k<<<grid, NTHREADS, smem, st>>>(P);                                                   \
        return cudaGetLastError();                                                            \
    }
    TFQ_CASE(32, 1) TFQ_CASE(32, 2) TFQ_CASE(64, 1) TFQ_CASE(64, 2) TFQ_CASE(128, 1) TFQ_CASE(128, 2)
#undef TFQ_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tfq
