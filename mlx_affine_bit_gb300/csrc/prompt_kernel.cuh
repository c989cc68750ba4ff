// prompt_kernel.cuh -- the MLX-affine quantized product for many activation rows
// (a prompt) on the fifth-generation tensor cores.
//
// y[r][n] = sum_k x[r][k] * (scale[n][k/G] * q[n][k] + bias[n][k/G]) (TensorFold PR
// #788, commit "every MLX affine width in the row kernel"; the group-sum form of PR
// #774, Exactness, Precision bullet), for a window of up to 64 rows that reads the
// weights once (PR #788, the 2-bit affine_mm commit: the prompt-side tiled product).
//
// A tile is 128 output columns (the MMA's M, one tensor-memory lane each) by the
// window's rows (the MMA's N: the rows rounded up to 16, at most 64).  Per group of
// G codes:
//   T      = tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in tensor memory) of
//            the group's codes (exact, or 128 + c at 4-6 bits) and x, K = 16 a step
//   p      = fma(s, T, p); p = fma(b', sum_group(x), p)      (b' = b - 128 s for offset codes)
// p runs over the groups of a 2048-k chunk from 0, and y = C_0 + C_1 + ... over the
// chunks in order.  Roles: a producer warp streams with TMA, per 128-k stage, the
// tile's codes and the window's x (permuted to the codes' pair order by a prepass),
// and per unit of up to 32 groups the scales, the biases and the per-group sums of
// x; four unpack warps write each stage's codes as bf16 into shared memory
// (canonical K-major layout); one thread of an MMA warp issues the stage's eight
// MMAs into the groups' accumulator slots; sixteen epilogue warps apply the group
// epilogue out of tensor memory.  Every wait is bounded.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm_kernel.cuh"

namespace tfq {
namespace prompt {

constexpr int PM = 128;                 // output columns per tile (MMA M, TMEM lanes)
constexpr int PN = 64;                  // activation rows per window (largest MMA N)
constexpr int PSTAGE = 128;             // k per pipeline stage (eight K = 16 MMAs)
constexpr int KSTEP = 16;               // k per MMA
constexpr int STAGES = 3;               // stage ring depth (codes and x)
constexpr int ABUF = 2;                 // unpacked stages in flight
constexpr int DSLOTS = 8;               // group accumulators in tensor memory (PN columns each)
constexpr int UNPACK_WARPS = 4;         // one column per thread
constexpr int EPI_WARPS = 16;           // four per tensor-memory lane quarter: rows 0-15, 16-31, 32-47, 48-63
constexpr int EPI_ROWS = PN / (EPI_WARPS / 4);   // window rows per epilogue warp
constexpr int PRODUCER = UNPACK_WARPS + EPI_WARPS, MMA_WARP = PRODUCER + 1;
constexpr int THREADS = (MMA_WARP + 1) * 32;
// Registers a thread: an SM's four schedulers hold 16K registers each and the
// CTA's 22 warps put six on two of them, so 6 x 32 x 80 <= 16384.
constexpr int MAX_REGS = 80;
constexpr int A_BYTES = PM * PSTAGE * 2;         // one unpacked stage (bf16)
constexpr int X_BYTES = PN * PSTAGE * 2;         // one stage of x (bf16)
constexpr int SX_BYTES = 32 * PN * 4;            // per-group sums of x of one scale/bias unit (<= 32 groups x 64 rows)
constexpr int TMEM_COLS = DSLOTS * PN;           // accumulator slots

// Groups of one stage, and stage-sized accumulator sets in tensor memory.
__host__ __device__ constexpr int groups_per_stage(int group) { return PSTAGE / group; }
__host__ __device__ constexpr int dsets(int group) { return DSLOTS / groups_per_stage(group); }
// Scales and biases travel in units of up to 32 groups (within one chunk).
__host__ __device__ constexpr int sb_groups(int group) { return CHUNK / group < 32 ? CHUNK / group : 32; }
__host__ __device__ constexpr int sb_k(int group) { return sb_groups(group) * group; }
// Pad words after each stage row of codes: the TMA box row is a multiple of 16
// bytes and row pitches of an odd number of 16-byte units keep the unpack warps'
// 16-byte reads of their own rows apart in the banks.
__host__ __device__ constexpr int code_pad_words(int bits) { return (bits & 1) ? 8 : 4; }
__host__ __device__ constexpr int code_pitch(int bits) { return (PSTAGE * bits / 32 + code_pad_words(bits)) * 4; }
// Scale/bias rows of a unit: its groups plus 8 padding values.
__host__ __device__ constexpr int sb_pitch(int group) { return (sb_groups(group) + 8) * 2; }

struct Layout {
    int w_off, x_off, stage_bytes, sb_off, sb_bytes, sx_off, a_off, smem;
};
__host__ __device__ inline Layout layout(int bits, int group) {
    Layout L;
    const int wbytes = (PM * code_pitch(bits) + 1023) & ~1023;
    L.w_off = 0;
    L.x_off = wbytes;
    L.stage_bytes = wbytes + X_BYTES;
    L.sb_bytes = (PM * sb_pitch(group) + 1023) & ~1023;   // scales (or biases) of one unit
    const int base = 1024;                                // header: barriers, TMEM address, flags
    L.sb_off = base + STAGES * L.stage_bytes;
    L.sx_off = L.sb_off + 4 * L.sb_bytes;                 // two slots x (scales, biases)
    L.a_off = L.sx_off + 2 * SX_BYTES;                    // two slots of group sums
    L.smem = L.a_off + ABUF * A_BYTES;
    return L;
}

struct Params {
    CUtensorMap tmW, tmSX, tmS, tmB;
    const uint16_t *xt;    // x operand tiles: [window][stage][16 k blocks][64 rows][8] bf16
    float *y;
    long long y_stride;
    int *status;
    int K, N, ntiles, nchunks;
    int r0, rows;          // window: x rows r0 .. r0 + rows - 1 (rows <= 64) -> y rows r0 ..
    int out;               // OUT_* bits
    // Work items: item w is column tile w / nsplit over chunks c0 = (w % nsplit) * cpi
    // .. min(c0 + cpi, nchunks) - 1.  With nsplit > 1 every chunk's partial goes to
    // part[c][window row][N] (fp32) and a fold sums them in chunk order.
    int nitems, nsplit, cpi;
    float *part;
};

struct Item {
    int tile, c0, c1;
    __device__ __forceinline__ Item(const Params &P, int w) {
        tile = w / P.nsplit;
        c0 = (w - tile * P.nsplit) * P.cpi;
        c1 = c0 + P.cpi < P.nchunks ? c0 + P.cpi : P.nchunks;
    }
};

// Shared-memory matrix descriptor (tcgen05): canonical K-major layout without
// swizzle; lbo = byte distance of core matrices adjacent in K, sbo = in M (or N).
// Shared addresses stay below 2^18, so a byte offset o moves a descriptor by o >> 4.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// Instruction descriptor: kind::f16, bf16 A and B (both K-major), fp32 D, M = 128,
// N = n (a multiple of 16, 16 .. 256).
__device__ __forceinline__ uint32_t idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
}

__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t id, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(id), "r"((uint32_t)acc)
        : "memory");
}
// One contiguous global -> shared copy completing on an mbarrier (16-byte
// aligned addresses, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// The scales (or biases) of the N <= 4 groups of one stage in one row: one
// shared-memory load of 2N bytes (2N-byte aligned); get(j) with j known at
// compile time.
template <int N>
struct SbRun {
    uint32_t lo = 0, hi = 0;
    __device__ __forceinline__ void load(const uint16_t *p) {
        if constexpr (N == 4) {
            const uint2 t = *reinterpret_cast<const uint2 *>(p);
            lo = t.x;
            hi = t.y;
        } else if constexpr (N == 2) {
            lo = *reinterpret_cast<const uint32_t *>(p);
        } else {
            lo = p[0];
        }
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t w = (j & 2) ? hi : lo;
        return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};

// Tensor-memory load of 16 columns of this warp's lane quarter, completed by
// tmem_wait16, which names the registers so that nothing reads them earlier.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Barriers of the header, in order.
struct Bars {
    uint64_t st_full[STAGES], st_empty[STAGES];
    uint64_t sb_full[2], sb_empty[2];
    uint64_t a_full[ABUF], a_empty[ABUF];
    uint64_t d_full[DSLOTS], d_empty[DSLOTS];
    uint64_t mma_done;
    uint32_t tmem;
    int abort;
};

// Every handshake is per 128-k stage: the producer fills a stage of codes and x
// (and its group sums), the unpack warps write the stage's A operand and arrive
// once, the MMA lane issues its eight MMAs into the groups' accumulator slots and
// commits once, the epilogue warps take the stage's groups out of tensor memory
// and release the slots once.
template <int BITS, int G, bool MC>
__global__ void __maxnreg__(MAX_REGS) prompt_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int SBP = sb_pitch(G) / 2;                     // scale/bias row pitch (bf16 values)
    constexpr int CP = code_pitch(BITS) / 4;                 // code row pitch (words)
    constexpr bool OFF = offset_codes(BITS);
    constexpr int GPS = groups_per_stage(G);                 // groups per stage
    constexpr int DST = dsets(G);                            // stage-sized accumulator sets
    constexpr int SPU = sb_k(G) / PSTAGE;                    // stages per scale/bias unit
    constexpr int UPC = CHUNK / sb_k(G);                     // units per chunk
    const Layout L = layout(BITS, G);
    Bars &B = *reinterpret_cast<Bars *>(smem);
    volatile int *abort = &B.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto stage_ptr = [&](uint32_t slot) { return smem + 1024 + slot * L.stage_bytes; };

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&B.st_full[i], 1);
            mbar_init(&B.st_empty[i], UNPACK_WARPS + 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.sb_full[i], 1);
            mbar_init(&B.sb_empty[i], EPI_WARPS);
        }
        for (int i = 0; i < ABUF; ++i) {
            mbar_init(&B.a_full[i], UNPACK_WARPS);
            mbar_init(&B.a_empty[i], 1);
        }
        for (int i = 0; i < DST; ++i) {
            mbar_init(&B.d_full[i], 1);
            mbar_init(&B.d_empty[i], EPI_WARPS);
        }
        mbar_init(&B.mma_done, 1);
        B.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&B.tmem)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = B.tmem;

    if (warp == PRODUCER) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmW) : "memory");
            const uint16_t *xw = P.xt + (long long)(P.r0 / PN) * (P.K / PSTAGE) * (X_BYTES / 2);
            uint32_t sit = 0, uit = 0;
            for (int w = blockIdx.x; w < P.nitems && !*abort; w += gridDim.x) {
                const Item it(P, w);
                const int n0 = it.tile * PM;
                for (int u = it.c0 * UPC; u < it.c1 * UPC && !*abort; ++u, ++uit) {
                    const int us = uit & 1;
                    mbar_wait(&B.sb_empty[us], ((uit >> 1) & 1) ^ 1, abort, P.status);
                    mbar_arrive_tx(&B.sb_full[us], 2u * PM * sb_pitch(G) + (uint32_t)(sb_groups(G) * PN * 4));
                    tma_3d(smem + L.sb_off + (2 * us) * L.sb_bytes, &P.tmS, 0, u, n0, &B.sb_full[us]);
                    tma_3d(smem + L.sb_off + (2 * us + 1) * L.sb_bytes, &P.tmB, 0, u, n0, &B.sb_full[us]);
                    tma_2d(smem + L.sx_off + us * SX_BYTES, &P.tmSX, P.r0, u * sb_groups(G), &B.sb_full[us]);
                    for (int st = 0; st < SPU && !*abort; ++st, ++sit) {
                        const uint32_t slot = sit % STAGES;
                        const int k0 = u * sb_k(G) + st * PSTAGE;
                        mbar_wait(&B.st_empty[slot], ((sit / STAGES) & 1) ^ 1, abort, P.status);
                        uint8_t *sp = stage_ptr(slot);
                        mbar_arrive_tx(&B.st_full[slot], (uint32_t)(PM * code_pitch(BITS) + X_BYTES));
                        tma_3d(sp + L.w_off, &P.tmW, 0, n0, k0 / PSTAGE, &B.st_full[slot]);
                        bulk_copy(sp + L.x_off, xw + (long long)(k0 / PSTAGE) * (X_BYTES / 2), X_BYTES,
                                  &B.st_full[slot]);
                    }
                }
            }
            // Drain: every issued copy has landed before the CTA may exit.
            for (uint32_t j = 0; j < (sit < (uint32_t)STAGES ? sit : (uint32_t)STAGES); ++j) {
                const uint32_t q = sit - 1 - j;
                mbar_wait(&B.st_full[q % STAGES], (q / STAGES) & 1, abort, P.status, false);
            }
            for (uint32_t j = 0; j < (uit < 2u ? uit : 2u); ++j) {
                const uint32_t q = uit - 1 - j;
                mbar_wait(&B.sb_full[q & 1], (q >> 1) & 1, abort, P.status, false);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            // MMA N: the window's rows rounded up to 16.
            const int nr = P.rows <= 16 ? 16 : P.rows <= 32 ? 32 : P.rows <= 48 ? 48 : 64;
            const uint32_t id = idesc(nr);
            // A stage: [16 column blocks][16 k blocks][8][16 B]; x stage:
            // [16 k blocks][64 rows][16 B].  K step j starts 2 k blocks further.
            const uint64_t a0 = smem_desc(smem_u32(smem + L.a_off), 128, (PSTAGE / 8) * 128);
            const uint64_t x0 = smem_desc(smem_u32(stage_ptr(0) + L.x_off), PN * 16, 128);
            uint32_t sit = 0;
            for (int w = blockIdx.x; w < P.nitems && !*abort; w += gridDim.x) {
                const Item it(P, w);
                for (int st = it.c0 * (CHUNK / PSTAGE); st < it.c1 * (CHUNK / PSTAGE) && !*abort; ++st, ++sit) {
                    const uint32_t slot = sit % STAGES, a = sit % ABUF, ds = sit % DST;
                    mbar_wait(&B.st_full[slot], (sit / STAGES) & 1, abort, P.status);
                    mbar_wait(&B.a_full[a], (sit / ABUF) & 1, abort, P.status);
                    mbar_wait(&B.d_empty[ds], ((sit / DST) & 1) ^ 1, abort, P.status);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint64_t ad = a0 + ((a * A_BYTES) >> 4);
                    const uint64_t bd = x0 + ((slot * L.stage_bytes) >> 4);
                    const uint32_t dt = tmem + ds * GPS * PN;
#pragma unroll
                    for (int j = 0; j < PSTAGE / KSTEP; ++j)
                        mma_issue(dt + (j * KSTEP / G) * PN, ad + ((j * 256) >> 4), bd + ((j * 2 * PN * 16) >> 4), id,
                                  (j * KSTEP) % G != 0);
                    mma_commit(&B.a_empty[a]);
                    mma_commit(&B.st_empty[slot]);
                    mma_commit(&B.d_full[ds]);
                }
            }
            mma_commit(&B.mma_done);
            mbar_wait(&B.mma_done, 0, abort, P.status, false);
        }
    } else if (warp < UNPACK_WARPS) {
        // Unpack warps: thread m unpacks output column n0 + m into the A stages.  The
        // stage row of codes comes in with 16-byte loads (row pitches of an odd
        // number of 16-byte units: no bank conflicts within a quarter warp); every
        // run's word and bit offsets are then compile-time constants.
        const int m = tid;
        const uint32_t mg = MAGIC, mq = QP<BITS>::value;
        constexpr int RW = PSTAGE * BITS / 32;                   // words of a stage row
        uint32_t sit = 0;
        for (int w = blockIdx.x; w < P.nitems && !*abort; w += gridDim.x) {
            const Item it(P, w);
            for (int st = it.c0 * (CHUNK / PSTAGE); st < it.c1 * (CHUNK / PSTAGE) && !*abort; ++st, ++sit) {
                const uint32_t slot = sit % STAGES, a = sit % ABUF;
                mbar_wait(&B.st_full[slot], (sit / STAGES) & 1, abort, P.status);
                uint32_t wv[RW + 1];                             // + one zero word: a run's second word
                const uint4 *src = reinterpret_cast<const uint4 *>(stage_ptr(slot) + L.w_off + m * code_pitch(BITS));
#pragma unroll
                for (int i = 0; i < RW / 4; ++i) {
                    const uint4 t = src[i];
                    wv[4 * i] = t.x;
                    wv[4 * i + 1] = t.y;
                    wv[4 * i + 2] = t.z;
                    wv[4 * i + 3] = t.w;
                }
                wv[RW] = 0u;
                mbar_wait(&B.a_empty[a], ((sit / ABUF) & 1) ^ 1, abort, P.status);
                uint8_t *ap = smem + L.a_off + a * A_BYTES + (m >> 3) * ((PSTAGE / 8) * 128) + (m & 7) * 16;
#pragma unroll
                for (int r = 0; r < PSTAGE / 8; ++r) {
                    // Run r (codes 8r .. 8r+7 of the stage) as pairs (c_i, c_i+4).
                    const uint32_t bit = (uint32_t)(r * 8 * BITS);
                    uint32_t ua, ub, v[4];
                    lane_args<BITS>(bit & 31u, ua, ub);
                    if constexpr (BITS == 6)
                        Unpack<6>::template run_words<1, OFF>(wv[bit >> 5], wv[(bit >> 5) + 1], ua, ub, mg, mq, v);
                    else
                        Unpack<BITS>::template run<1, OFF>(&wv[bit >> 5], ua, ub, mg, mq, v);
                    *reinterpret_cast<uint4 *>(ap + r * 128) = make_uint4(v[0], v[1], v[2], v[3]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&B.a_full[a]);
                    mbar_arrive(&B.st_empty[slot]);   // the stage's codes are read
                }
            }
        }
    } else {
        // Epilogue warps: column n0 + m (tensor-memory lane m), rows h*16 .. h*16 + 15;
        // a warp whose rows lie past the window only keeps the handshakes.
        const int e = warp - UNPACK_WARPS;
        const int q = e & 3, h = e >> 2;
        const int m = q * 32 + lane;
        const bool active = h * EPI_ROWS < P.rows;
        uint32_t sit = 0, uit = 0;
        float p[EPI_ROWS], y[MC ? EPI_ROWS : 1];             // chunk partial; chunk sums (K > one chunk)
#pragma unroll
        for (int r = 0; r < EPI_ROWS; ++r) p[r] = 0.f;
        // One group's epilogue: p = fma(s, T, p); p = fma(b', sum_group(x), p) per row.
        auto group_fma = [&](const uint32_t (&T)[16], float sg, float bg, const float *sxp) {
#pragma unroll
            for (int r = 0; r < EPI_ROWS; r += 4) {
                const float4 sx4 = *reinterpret_cast<const float4 *>(sxp + r);
                fma2(p[r], p[r + 1], sg, sg, __uint_as_float(T[r]), __uint_as_float(T[r + 1]));
                fma2(p[r], p[r + 1], bg, bg, sx4.x, sx4.y);
                fma2(p[r + 2], p[r + 3], sg, sg, __uint_as_float(T[r + 2]), __uint_as_float(T[r + 3]));
                fma2(p[r + 2], p[r + 3], bg, bg, sx4.z, sx4.w);
            }
        };
        for (int w = blockIdx.x; w < P.nitems && !*abort; w += gridDim.x) {
            const Item it(P, w);
            const int n0 = it.tile * PM;
            const int n = n0 + m;
            for (int c = it.c0; c < it.c1 && !*abort; ++c) {
                for (int u = 0; u < UPC && !*abort; ++u, ++uit) {
                    const int us = (int)(uit & 1);
                    mbar_wait(&B.sb_full[us], (uit >> 1) & 1, abort, P.status);
                    const uint16_t *srow = reinterpret_cast<const uint16_t *>(smem + L.sb_off + (2 * us) * L.sb_bytes) + m * SBP;
                    const uint16_t *brow =
                        reinterpret_cast<const uint16_t *>(smem + L.sb_off + (2 * us + 1) * L.sb_bytes) + m * SBP;
                    for (int st = 0; st < SPU && !*abort; ++st, ++sit) {
                        const uint32_t ds = sit % DST;
                        mbar_wait(&B.d_full[ds], (sit / DST) & 1, abort, P.status);
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const float *sxs = reinterpret_cast<const float *>(smem + L.sx_off + us * SX_BYTES) +
                                           st * GPS * PN + h * EPI_ROWS;
                        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + ds * GPS * PN + h * EPI_ROWS;
                        // Groups in order, the next group's accumulators and scale/bias
                        // fetched while this group's products are issued.
                        uint32_t TA[16], TB[16];
                        SbRun<GPS> sr, br;
                        sr.load(srow + st * GPS);
                        br.load(brow + st * GPS);
                        float sA = sr.get(0), sB = 0.f;
                        float bA = bias_term<BITS>(sA, br.get(0)), bB = 0.f;
                        if (active) {
                            tmem_ld16(tq, TA);
                            tmem_wait16(TA);
                        }
#pragma unroll
                        for (int j = 0; j < GPS; ++j) {
                            uint32_t(&Tc)[16] = (j & 1) ? TB : TA;
                            uint32_t(&Tn)[16] = (j & 1) ? TA : TB;
                            const float sc = (j & 1) ? sB : sA, bc = (j & 1) ? bB : bA;
                            if (j + 1 < GPS) {
                                const float sn = sr.get(j + 1);
                                const float bn = bias_term<BITS>(sn, br.get(j + 1));
                                if (j & 1) {
                                    sA = sn;
                                    bA = bn;
                                } else {
                                    sB = sn;
                                    bB = bn;
                                }
                                if (active) tmem_ld16(tq + (j + 1) * PN, Tn);
                            } else {
                                // Every accumulator of the stage is in registers: release the slots.
                                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&B.d_empty[ds]);
                            }
                            if (active) group_fma(Tc, sc, bc, sxs + j * PN);
                            if (j + 1 < GPS && active) tmem_wait16(Tn);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.sb_empty[us]);
                }
                if (P.part) {
                    // This chunk's partial, summed with the others in chunk order by the fold.
                    if (active && n < P.N && !*abort) {
#pragma unroll
                        for (int r = 0; r < EPI_ROWS; ++r)
                            P.part[((long long)c * PN + h * EPI_ROWS + r) * P.N + n] = p[r];
                    }
#pragma unroll
                    for (int r = 0; r < EPI_ROWS; ++r) p[r] = 0.f;
                } else if constexpr (MC) {
                    // Chunk sums in chunk order.
#pragma unroll
                    for (int r = 0; r < EPI_ROWS; ++r) {
                        y[r] = c == 0 ? p[r] : y[r] + p[r];
                        p[r] = 0.f;
                    }
                }
            }
            if (P.part) continue;
            // Store the window's rows h*16 .. h*16 + 15 of this column.
            if (active && n < P.N && !*abort) {
#pragma unroll
                for (int r = 0; r < EPI_ROWS; ++r) {
                    if (h * EPI_ROWS + r < P.rows) {
                        float v;
                        if constexpr (MC)
                            v = y[r];
                        else
                            v = p[r];
                        if (P.out & OUT_RELU2) {
                            const float u = fmaxf(v, 0.f);
                            v = u * u;
                        }
                        const long long at = (long long)(P.r0 + h * EPI_ROWS + r) * P.y_stride + n;
                        if (P.out & OUT_BF16)
                            reinterpret_cast<__nv_bfloat16 *>(P.y)[at] = __float2bfloat16_rn(v);
                        else
                            P.y[at] = v;
                    }
                }
            }
            if constexpr (!MC) {
#pragma unroll
                for (int r = 0; r < EPI_ROWS; ++r) p[r] = 0.f;
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

}  // namespace prompt
}  // namespace tfq
