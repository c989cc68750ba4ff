// prompt_kernel.cuh -- the MLX-affine quantized product for many activation rows
// (a prompt) on the fifth-generation tensor cores.
//
// y[r][n] = sum_k x[r][k] * (scale[n][k/G] * q[n][k] + bias[n][k/G]) (TensorFold PR
// #788, commit "every MLX affine width in the row kernel"; the group-sum form of PR
// #774, Exactness, Precision bullet), for a window of up to 64 rows that reads the
// weights once (PR #788, the 2-bit affine_mm commit: the prompt-side tiled product).
//
// A tile is 128 output columns (the MMA's M, one tensor-memory lane each) by the
// window's 64 rows (the MMA's N).  Per group of G codes:
//   T      = tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in tensor memory) of
//            the group's codes (exact, or 128 + c at 4-6 bits) and x, K = 16 a step
//   p      = fma(s, T, p); p = fma(b', sum_group(x), p)      (b' = b - 128 s for offset codes)
// p runs over the groups of a 2048-k chunk from 0, and y = C_0 + C_1 + ... over the
// chunks in order.  Roles: a producer warp streams, per 128-k stage, the tile's
// codes, the window's x (permuted to the codes' pair order by a prepass) and the
// per-group sums of x with TMA, and per chunk the scales and biases; four math
// warps unpack each 32-k piece of codes to bf16 in shared memory (canonical K-major
// layout) and run the group epilogue out of tensor memory; one thread of an MMA warp
// issues the MMAs and commits them to mbarriers.  Every wait is bounded.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm_kernel.cuh"

namespace tfq {
namespace prompt {

constexpr int PM = 128;                 // output columns per tile (MMA M, TMEM lanes)
constexpr int PN = 64;                  // activation rows per window (MMA N)
constexpr int PSTAGE = 128;             // k per pipeline stage
constexpr int PIECE = 32;               // k per unpacked piece (two K = 16 MMAs)
constexpr int NPIECE = PSTAGE / PIECE;  // pieces per stage
constexpr int STAGES = 3;               // stage ring depth (codes and x)
constexpr int SXR = 8;                  // ring depth of the per-group sums of x (one slot a stage)
constexpr int ABUF = 4;                 // unpacked pieces in flight
constexpr int DBUF = 4;                 // group accumulators in flight (tensor memory)
constexpr int UNPACK_WARPS = 4;         // one column per thread
constexpr int EPI_WARPS = 8;            // two per tensor-memory lane quarter: rows 0-31 and 32-63
constexpr int PRODUCER = UNPACK_WARPS + EPI_WARPS, MMA_WARP = PRODUCER + 1;
constexpr int THREADS = (MMA_WARP + 1) * 32;
constexpr int A_BYTES = PM * PIECE * 2;          // one unpacked piece (bf16)
constexpr int X_BYTES = PN * PSTAGE * 2;         // one stage of x (bf16)
constexpr int SX_BYTES = 1024;                   // per-group sums of x of one stage (<= 4 groups x 64 rows)
constexpr int TMEM_COLS = DBUF * PN;             // accumulator buffers

// Pad words after each stage row of codes: the TMA box row is a multiple of 16
// bytes and row pitches of an odd number of 16-byte units keep the math warps'
// vector reads of their own rows apart in the banks.
__host__ __device__ constexpr int code_pad_words(int bits) { return (bits & 1) ? 8 : 4; }
__host__ __device__ constexpr int code_pitch(int bits) { return (PSTAGE * bits / 32 + code_pad_words(bits)) * 4; }
// Scale/bias rows of a chunk: 2048/G values plus 8 padding values.
__host__ __device__ constexpr int sb_pitch(int group) { return (CHUNK / group + 8) * 2; }

struct Layout {
    int w_off, x_off, stage_bytes, sx_off, sb_off, sb_bytes, a_off, smem;
};
__host__ __device__ inline Layout layout(int bits, int group) {
    Layout L;
    const int wbytes = (PM * code_pitch(bits) + 1023) & ~1023;
    L.w_off = 0;
    L.x_off = wbytes;
    L.stage_bytes = wbytes + X_BYTES;
    L.sb_bytes = (PM * sb_pitch(group) + 1023) & ~1023;   // scales (or biases) of one chunk
    const int base = 1024;                                // header: barriers, TMEM address, flags
    L.sx_off = base + STAGES * L.stage_bytes;             // SXR slots of SX_BYTES
    L.sb_off = L.sx_off + SXR * SX_BYTES;
    L.a_off = L.sb_off + 4 * L.sb_bytes;                  // two slots x (scales, biases)
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
};

// Shared-memory matrix descriptor (tcgen05): canonical K-major layout without
// swizzle; lbo = byte distance of core matrices adjacent in K, sbo = in M (or N).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// Instruction descriptor: kind::f16, bf16 A and B (both K-major), fp32 D, M = 128, N = 64.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(PN >> 3) << 17) |
                           ((uint32_t)(PM >> 4) << 24);

__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t ad, uint64_t bd, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(IDESC), "r"((uint32_t)acc)
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
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Barriers of the header, in order.
struct Bars {
    uint64_t st_full[STAGES], st_empty[STAGES];
    uint64_t sx_full[SXR], sx_empty[SXR];
    uint64_t sb_full[2], sb_empty[2];
    uint64_t a_full[ABUF], a_empty[ABUF];
    uint64_t d_full[DBUF], d_empty[DBUF];
    uint64_t mma_done;
    uint32_t tmem;
    int abort;
};

template <int BITS, int G>
__global__ void __maxnreg__(128) prompt_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int SBP = sb_pitch(G) / 2;                     // scale/bias row pitch (bf16 values)
    constexpr int CP = code_pitch(BITS) / 4;                 // code row pitch (words)
    constexpr bool OFF = offset_codes(BITS);
    const Layout L = layout(BITS, G);
    Bars &B = *reinterpret_cast<Bars *>(smem);
    volatile int *abort = &B.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int SPC = CHUNK / PSTAGE;                      // stages per chunk
    auto stage_ptr = [&](uint32_t slot) { return smem + 1024 + slot * L.stage_bytes; };

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&B.st_full[i], 1);
            mbar_init(&B.st_empty[i], UNPACK_WARPS + 1);
        }
        for (int i = 0; i < SXR; ++i) {
            mbar_init(&B.sx_full[i], 1);
            mbar_init(&B.sx_empty[i], EPI_WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.sb_full[i], 1);
            mbar_init(&B.sb_empty[i], EPI_WARPS);
        }
        for (int i = 0; i < ABUF; ++i) {
            mbar_init(&B.a_full[i], UNPACK_WARPS);
            mbar_init(&B.a_empty[i], 1);
        }
        for (int i = 0; i < DBUF; ++i) {
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
            uint32_t sit = 0, cit = 0;
            for (int tile = blockIdx.x; tile < P.ntiles && !*abort; tile += gridDim.x) {
                const int n0 = tile * PM;
                for (int c = 0; c < P.nchunks && !*abort; ++c, ++cit) {
                    const int cs = cit & 1;
                    mbar_wait(&B.sb_empty[cs], ((cit >> 1) & 1) ^ 1, abort, P.status);
                    mbar_arrive_tx(&B.sb_full[cs], 2u * PM * sb_pitch(G));
                    tma_3d(smem + L.sb_off + (2 * cs) * L.sb_bytes, &P.tmS, 0, c, n0, &B.sb_full[cs]);
                    tma_3d(smem + L.sb_off + (2 * cs + 1) * L.sb_bytes, &P.tmB, 0, c, n0, &B.sb_full[cs]);
                    for (int st = 0; st < SPC && !*abort; ++st, ++sit) {
                        const uint32_t slot = sit % STAGES;
                        const int k0 = c * CHUNK + st * PSTAGE;
                        const uint32_t xslot = sit % SXR;
                        constexpr int GPS = PSTAGE / G >= 1 ? PSTAGE / G : 1;
                        mbar_wait(&B.sx_empty[xslot], ((sit / SXR) & 1) ^ 1, abort, P.status);
                        mbar_arrive_tx(&B.sx_full[xslot], (uint32_t)(GPS * PN * 4));
                        tma_2d(smem + L.sx_off + xslot * SX_BYTES, &P.tmSX, P.r0, k0 / G, &B.sx_full[xslot]);
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
            for (uint32_t j = 0; j < (cit < 2u ? cit : 2u); ++j) {
                const uint32_t q = cit - 1 - j;
                mbar_wait(&B.sb_full[q & 1], (q >> 1) & 1, abort, P.status, false);
            }
            for (uint32_t j = 0; j < (sit < (uint32_t)SXR ? sit : (uint32_t)SXR); ++j) {
                const uint32_t q = sit - 1 - j;
                mbar_wait(&B.sx_full[q % SXR], (q / SXR) & 1, abort, P.status, false);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            uint32_t sit = 0, pit = 0, git = 0;
            for (int tile = blockIdx.x; tile < P.ntiles && !*abort; tile += gridDim.x) {
                for (int c = 0; c < P.nchunks && !*abort; ++c) {
                    for (int st = 0; st < SPC && !*abort; ++st, ++sit) {
                        const uint32_t slot = sit % STAGES;
                        mbar_wait(&B.st_full[slot], (sit / STAGES) & 1, abort, P.status);
                        const uint32_t xs = smem_u32(stage_ptr(slot) + L.x_off);
                        for (int pc = 0; pc < NPIECE; ++pc, ++pit) {
                            const int kp = st * PSTAGE + pc * PIECE;            // piece's k within the chunk
                            const bool first = kp % G == 0, last = (kp + PIECE) % G == 0;
                            const uint32_t a = pit % ABUF, d = git % DBUF;
                            mbar_wait(&B.a_full[a], (pit / ABUF) & 1, abort, P.status);
                            if (first) mbar_wait(&B.d_empty[d], ((git / DBUF) & 1) ^ 1, abort, P.status);
                            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                            const uint32_t as = smem_u32(smem + L.a_off + a * A_BYTES);
                            const uint32_t dt = tmem + d * PN;
                            // A piece: [16 column blocks][4 k blocks][8][16 B]; x stage:
                            // [16 k blocks][64 rows][16 B].
                            mma_issue(dt, smem_desc(as, 128, 512), smem_desc(xs + (pc * 4) * 1024, 1024, 128), !first);
                            mma_issue(dt, smem_desc(as + 256, 128, 512), smem_desc(xs + (pc * 4 + 2) * 1024, 1024, 128),
                                      true);
                            mma_commit(&B.a_empty[a]);
                            if (last) {
                                mma_commit(&B.d_full[d]);
                                ++git;
                            }
                        }
                        mma_commit(&B.st_empty[slot]);
                    }
                }
            }
            mma_commit(&B.mma_done);
            mbar_wait(&B.mma_done, 0, abort, P.status, false);
        }
    } else if (warp < UNPACK_WARPS) {
        // Unpack warps: thread m unpacks output column n0 + m into the A pieces.
        const int m = tid;
        const uint32_t mg = MAGIC, mq = QP<BITS>::value;
        uint32_t ua[4], ub[4], wo[4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            const uint32_t bit = (uint32_t)(kb * 8) * BITS;      // run kb of a piece, from the piece's start
            wo[kb] = bit >> 5;
            lane_args<BITS>(bit & 31u, ua[kb], ub[kb]);
        }
        uint32_t sit = 0, pit = 0;
        for (int tile = blockIdx.x; tile < P.ntiles && !*abort; tile += gridDim.x) {
            for (int c = 0; c < P.nchunks && !*abort; ++c) {
                for (int st = 0; st < SPC && !*abort; ++st, ++sit) {
                    const uint32_t slot = sit % STAGES;
                    mbar_wait(&B.st_full[slot], (sit / STAGES) & 1, abort, P.status);
                    const uint32_t *wrow = reinterpret_cast<const uint32_t *>(stage_ptr(slot) + L.w_off) + m * CP;
#pragma unroll 1
                    for (int pc = 0; pc < NPIECE; ++pc, ++pit) {
                        const uint32_t a = pit % ABUF;
                        // The piece's four runs of this column, as pairs (c_i, c_i+4).
                        uint32_t v[16];
                        const uint32_t *pw = wrow + pc * BITS;
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb) {
                            if constexpr (BITS == 6)
                                Unpack<6>::template run_words<1, OFF>(pw[wo[kb]], pw[wo[kb] + 1], ua[kb], ub[kb], mg, mq,
                                                                      v + 4 * kb);
                            else
                                Unpack<BITS>::template run<1, OFF>(pw + wo[kb], ua[kb], ub[kb], mg, mq, v + 4 * kb);
                        }
                        mbar_wait(&B.a_empty[a], ((pit / ABUF) & 1) ^ 1, abort, P.status);
                        uint8_t *ap = smem + L.a_off + a * A_BYTES + (m >> 3) * 512 + (m & 7) * 16;
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb)
                            *reinterpret_cast<uint4 *>(ap + kb * 128) =
                                make_uint4(v[4 * kb], v[4 * kb + 1], v[4 * kb + 2], v[4 * kb + 3]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&B.a_full[a]);
                            if (pc == NPIECE - 1) mbar_arrive(&B.st_empty[slot]);   // the stage's codes are read
                        }
                    }
                }
            }
        }
    } else {
        // Epilogue warps: column n0 + m (tensor-memory lane m), rows h*32 .. h*32 + 31.
        const int e = warp - UNPACK_WARPS;
        const int q = e & 3, h = e >> 2;
        const int m = q * 32 + lane;
        uint32_t sit = 0, git = 0, cit = 0;
        float y[32], p[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) y[r] = p[r] = 0.f;
        for (int tile = blockIdx.x; tile < P.ntiles && !*abort; tile += gridDim.x) {
            const int n0 = tile * PM;
            for (int c = 0; c < P.nchunks && !*abort; ++c, ++cit) {
                const int cs = (int)(cit & 1);
                mbar_wait(&B.sb_full[cs], (cit >> 1) & 1, abort, P.status);
                const uint16_t *srow = reinterpret_cast<const uint16_t *>(smem + L.sb_off + (2 * cs) * L.sb_bytes) + m * SBP;
                const uint16_t *brow =
                    reinterpret_cast<const uint16_t *>(smem + L.sb_off + (2 * cs + 1) * L.sb_bytes) + m * SBP;
                for (int st = 0; st < SPC && !*abort; ++st, ++sit) {
                    const uint32_t xslot = sit % SXR;
                    mbar_wait(&B.sx_full[xslot], (sit / SXR) & 1, abort, P.status);
                    const float *sxs = reinterpret_cast<const float *>(smem + L.sx_off + xslot * SX_BYTES) + h * 32;
#pragma unroll 1
                    for (int kp = st * PSTAGE; kp < (st + 1) * PSTAGE; kp += G, ++git) {
                        const uint32_t d = git % DBUF;
                        const int gl = kp / G;                       // group within the chunk
                        const float s = bf16f(srow[gl]);
                        const float bb = bias_term<BITS>(s, bf16f(brow[gl]));
                        const float *sxp = sxs + ((kp % PSTAGE) / G) * PN;
                        mbar_wait(&B.d_full[d], (git / DBUF) & 1, abort, P.status);
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        float T[32];
                        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + d * PN + h * 32, T);
                        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&B.d_empty[d]);
#pragma unroll
                        for (int r = 0; r < 32; r += 4) {
                            const float4 sx4 = *reinterpret_cast<const float4 *>(sxp + r);
                            const float sxv[4] = {sx4.x, sx4.y, sx4.z, sx4.w};
#pragma unroll
                            for (int i = 0; i < 4; i += 2) {
                                fma2(p[r + i], p[r + i + 1], s, s, T[r + i], T[r + i + 1]);
                                fma2(p[r + i], p[r + i + 1], bb, bb, sxv[i], sxv[i + 1]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.sx_empty[xslot]);  // the stage's group sums are read
                }
                // Chunk sums in chunk order.
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    y[r] = c == 0 ? p[r] : y[r] + p[r];
                    p[r] = 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.sb_empty[cs]);
            }
            // Store the window's rows h*32 .. h*32 + 31 of this column.
            const int n = n0 + m;
            if (n < P.N && !*abort) {
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    if (h * 32 + r < P.rows) {
                        float v = y[r];
                        if (P.out & OUT_RELU2) {
                            const float u = fmaxf(v, 0.f);
                            v = u * u;
                        }
                        const long long at = (long long)(P.r0 + h * 32 + r) * P.y_stride + n;
                        if (P.out & OUT_BF16)
                            reinterpret_cast<__nv_bfloat16 *>(P.y)[at] = __float2bfloat16_rn(v);
                        else
                            P.y[at] = v;
                    }
                }
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
