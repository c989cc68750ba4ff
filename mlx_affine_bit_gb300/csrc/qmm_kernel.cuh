// qmm_kernel.cuh -- the MLX-affine quantized row product for sm_103a.
//
// y[r][n] = sum_k x[r][k] * (scale[n][k/G] * q[n][k] + bias[n][k/G]), 1..16 rows
// (TensorFold PR #788, commit "every MLX affine width in the row kernel"; the
// group-sum form with fp32 group sums, PR #774 Exactness, Precision bullet).
//
// One CTA = one or two consumer groups of 8 warps + 1 producer warp,
// persistent over work items (16 or 32 output columns x one K slice).  A
// pipeline stage is those rows x 2048 k: one 3D tensor-map TMA copy for the
// codes (a contiguous 8-64 KB of HBM when the slice is the whole row) and one
// each for scales and biases, completed on mbarriers.  Warp w of a group takes
// segment w (256 k) of a stage: it unpacks 8-code runs straight into bf16 A
// fragments (each code exact: c, or 128 + c at 4-6 bits with the offset taken
// back through the bias term), multiplies them by the activations with mma.sync
// m16n8k16 (rows are the N dimension: 1..8 rows cost one MMA, 9..16 two),
// applies each group's scale and bias to the fp32 group sum in registers, and
// the segment partials are folded in k order through shared memory.
//
// Every wait on an mbarrier is bounded in time; on expiry the kernel records
// it in the device status word, stops waiting and runs to completion.
//
// Built with TF_DEBUG_BOUNDS, every shared- and global-memory index the kernel
// computes is checked against its buffer before the access; an index outside
// it sets a bit of the device status word and the access is skipped (reads
// give zero).  The release build compiles each check to `true`.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm_common.h"
#include "unpack.cuh"

namespace tfq {

// ------------------------------------------------------------ primitives --

#ifdef TF_DEBUG_BOUNDS
static __device__ __noinline__ bool bounds_fail(int *status) {
    atomicOr(status, STATUS_BOUNDS);
    return false;
}
#define TFQ_IN(P, cond) ((cond) ? true : ::tfq::bounds_fail((P).status))
#else
#define TFQ_IN(P, cond) true
#endif

// [p, p + bytes) lies inside [lo, hi) of this CTA's shared memory.
__device__ __forceinline__ bool in_smem(const uint8_t *smem, const void *p, int bytes, int lo, int hi) {
    const long long off = reinterpret_cast<const uint8_t *>(p) - smem;
    return off >= lo && off + bytes <= hi;
}
// The stage ring, and the activation (or zero-block) and partial-sum regions.
__device__ __forceinline__ bool in_stages(const QmmParams &P, const uint8_t *smem, const void *p, int bytes) {
    return in_smem(smem, p, bytes, P.st_off, P.st_off + P.stages * P.stage_bytes);
}
__device__ __forceinline__ bool in_b(const QmmParams &P, const uint8_t *smem, const void *p, int bytes) {
    return in_smem(smem, p, bytes, P.x_off, P.sx_off) || in_smem(smem, p, bytes, P.z_off, P.z_off + ZERO_BYTES);
}
__device__ __forceinline__ bool in_sx(const QmmParams &P, const uint8_t *smem, const void *p, int bytes) {
    return in_smem(smem, p, bytes, P.sx_off, P.pb_off) || in_smem(smem, p, bytes, P.z_off, P.z_off + ZERO_BYTES);
}
__device__ __forceinline__ bool in_pbuf(const QmmParams &P, const uint8_t *smem, const void *p, int bytes) {
    return in_smem(smem, p, bytes, P.pb_off, P.z_off);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Phase-trace build (TF_TRACE): each CTA takes a record of TRACE_SLOTS words
// (its launch number, its SM and block, then %globaltimer at the phases below)
// in a device buffer that tf_trace_read copies out; the record's index sits in
// the shared header (byte TRACE_HDR).  In the product build the macros are empty.
enum TracePhase {
    TR_ENTER = 2,     // kernel entry
    TR_TMA0 = 3,      // producer: the CTA's first stage issued
    TR_LAND0 = 4,     // producer: the first stage landed (when the producer waits for it)
    TR_RELEASE = 5,   // consumer thread 0 past the dependency wait
    TR_XLOADED = 6,   // consumer thread 0: the first x slice placed and summed
    TR_STAGE0 = 7,    // consumer thread 0: the first stage's group products done
    TR_EXIT = 8,      // consumer thread 0: its last store issued
};
#ifdef TF_TRACE
__device__ __forceinline__ void trace_begin(const QmmParams &P, uint8_t *smem) {
    const unsigned s = P.trace ? atomicAdd(P.trace_n, 1u) : (unsigned)TRACE_MAX;
    *reinterpret_cast<unsigned *>(smem + TRACE_HDR) = s;
    if (s < (unsigned)TRACE_MAX) {
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        unsigned long long *r = P.trace + (unsigned long long)s * TRACE_SLOTS;
        r[0] = P.trace_seq;
        r[1] = ((unsigned long long)sm << 32) | blockIdx.x;
        for (int i = 2; i < TRACE_SLOTS; ++i) r[i] = 0ull;
        r[TR_ENTER] = global_ns();
    }
}
__device__ __forceinline__ void trace_at(const QmmParams &P, const uint8_t *smem, int phase) {
    const unsigned s = *reinterpret_cast<const volatile unsigned *>(smem + TRACE_HDR);
    if (s < (unsigned)TRACE_MAX) P.trace[(unsigned long long)s * TRACE_SLOTS + phase] = global_ns();
}
#define TFQ_TRACE_BEGIN(P, smem) trace_begin(P, smem)
#define TFQ_TRACE(smem, phase) trace_at(P, smem, phase)
#define TFQ_LAUNCH_PARAMS(P) trace_params(P)
#else
#define TFQ_TRACE_BEGIN(P, smem) ((void)0)
#define TFQ_TRACE(smem, phase) ((void)0)
#define TFQ_LAUNCH_PARAMS(P) (P)
#endif

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Relaxed arrive: the caller passes a value computed from every shared-memory
// read of the stage, so those reads have completed before the slot is released.
__device__ __forceinline__ void mbar_arrive_after(uint64_t *bar, float dep) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)), "f"(dep)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(tx)
                 : "memory");
}

// One test of the phase of `parity`; an incomplete phase suspends the thread
// until it completes or about SUSPEND_NS pass, so a waiting warp issues few
// instructions and leaves its scheduler's slots to the warps that compute.
constexpr uint32_t SUSPEND_NS = 1000000u;
__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(SUSPEND_NS)
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
        if ((it & 15u) == 0) {
            if (honor_abort && *abort) return;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                *abort = 1;
                atomicOr(status, STATUS_WAIT);
                return;
            }
        }
    }
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same copies with an L2 cache hint (a policy from createpolicy).  The
// weights, scales and biases are read once a launch: streamed with an
// evict-first policy they leave x, y and the split-K partials in L2.
#define TFQ_L2_HINT 1
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_3d_hint(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                            uint64_t pol) {
#if TFQ_L2_HINT
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
#else
    tma_3d(dst, map, x, y, z, bar);
#endif
}
__device__ __forceinline__ void tma_2d_hint(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t pol) {
#if TFQ_L2_HINT
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
#else
    tma_2d(dst, map, x, y, bar);
#endif
}

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Wait until the grids this one depends on (programmatic dependent launch) have
// completed and their memory is visible; returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// d = A*B with a zero accumulator (no registers to clear first).
__device__ __forceinline__ void mma_bf16_first(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// {d0, d1} = {a0 * b0 + d0, a1 * b1 + d1}: one fp32x2 FMA, each lane rounded
// exactly as fmaf.
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    unsigned long long A, B, D;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(D) : "f"(d0), "f"(d1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(D) : "l"(A), "l"(B));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(D));
}

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Named barrier `id` over `n` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------- item walking --

struct Item {
    int mt, slice, k_lo, k_hi;
};

// This CTA's work items.  The grid is a whole number of teams of
// gridDim.x / nsl CTAs, one team per K slice: CTA b of team s takes column
// tiles b, b + team, ... of slice s, so its activations are loaded once.
struct ItemWalk {
    int team, mt, slice;
    __device__ __forceinline__ explicit ItemWalk(const QmmParams &P) {
        team = gridDim.x / P.nsl;
        slice = blockIdx.x / team;
        mt = blockIdx.x - slice * team;
    }
    __device__ __forceinline__ bool more(const QmmParams &P) const { return mt < P.nmt; }
    __device__ __forceinline__ Item get(const QmmParams &P) const {
        Item I;
        I.mt = mt;
        I.slice = slice;
        I.k_lo = slice * P.sl;
        I.k_hi = min(P.K, I.k_lo + P.sl);
        return I;
    }
    __device__ __forceinline__ void next(const QmmParams &) { mt += team; }
};

// Ring position of the stage sequence: slot and mbarrier phase, no divisions.
struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next(int S) {
        if (++slot == (uint32_t)S) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// -------------------------------------------------------------- producer --

// Stage layout: W [SEGS segments][ROWS rows][SEGP bytes], then scales and
// biases [ROWS rows][sbpitch bytes] each.  SEGP = segment bytes + the pad.
template <int BITS, int G>
struct Pitch {
    static constexpr int SEGP = SEG * BITS / 8 + 4 * seg_pad_words(BITS, G);
};

template <int BITS, int G, int MT>
__device__ void producer(const QmmParams &P, uint8_t *smem, uint64_t *full, uint64_t *empty,
                         volatile int *abort) {
    constexpr int ROWS = TN * MT;
    constexpr int SEGP = Pitch<BITS, G>::SEGP;
    constexpr int SEGW = SEG * BITS / 32;     // words of one row segment
    const int lane = threadIdx.x & 31;
    const int S = P.stages;
    const long long row_words = (long long)P.K * BITS / 32;
    const int ngK = P.K / G;
    if (P.bulk && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmW) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmS) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&P.tmB) : "memory");
    }
    // Under programmatic dependent launch the previous kernel of the stream may
    // still run: wait for it unless the caller declared the weights unwritten by it.
    if (!P.early_w && P.dep != 2) grid_dependency_wait();
    uint32_t it = 0;
    Ring ring;
    for (ItemWalk w(P); w.more(P); w.next(P)) {
        const Item I = w.get(P);
        const int n0 = I.mt * ROWS;
        for (int k0 = I.k_lo; k0 < I.k_hi; k0 += CHUNK, ++it, ring.next(S)) {
            const int slot = (int)ring.slot;
            mbar_wait(&empty[slot], ring.phase ^ 1u, abort, P.status);
            uint8_t *st = smem + P.st_off + slot * P.stage_bytes;
            uint8_t *sst = st + SEGS * ROWS * SEGP;
            uint8_t *bst = sst + ROWS * P.sbpitch;
            if (!TFQ_IN(P, in_stages(P, smem, st, P.stage_bytes))) continue;
            // Test hook: the first stage is never sent, so its consumers' bounded
            // wait runs out (recorded in the status word) and the kernel completes.
            const bool withhold = P.stall && it == 0;
            if (withhold) {
            } else if (P.bulk) {
                // Rows past N and segments past K arrive zero-filled; the full
                // boxes count toward the transaction bytes.
                if (lane == 0) {
                    mbar_arrive_tx(&full[slot], (uint32_t)P.stage_bytes);
                    const uint64_t pol = l2_evict_first();
                    tma_3d_hint(st, &P.tmW, 0, n0, k0 / SEG, &full[slot], pol);
                    if (P.sb3d) {
                        tma_3d_hint(sst, &P.tmS, 0, k0 / CHUNK, n0, &full[slot], pol);
                        tma_3d_hint(bst, &P.tmB, 0, k0 / CHUNK, n0, &full[slot], pol);
                    } else {
                        tma_2d_hint(sst, &P.tmS, k0 / G, n0, &full[slot], pol);
                        tma_2d_hint(bst, &P.tmB, k0 / G, n0, &full[slot], pol);
                    }
                }
                // The CTA's first stage travels alone: every CTA's first stage
                // lands before later stages compete with it for DRAM -- except in
                // early-x launches of one or two rows, where the next stages follow
                // at once (their CTAs overlap the products around them; width sweep
                // 0.450 -> 0.454, while 3-16 rows measured slower without the rule).
                if (it == 0 && lane == 0) TFQ_TRACE(smem, TR_TMA0);
                if (it == 0 && !withhold && !(P.early_x && P.rows <= 2)) {
                    mbar_wait(&full[slot], ring.phase, abort, P.status);
                    if (lane == 0) TFQ_TRACE(smem, TR_LAND0);
                }
            } else {
                // Odd shapes or alignments: plain copies by the warp into the same layout.
                const int k1 = min(I.k_hi, k0 + CHUNK);
                const int nrows = min(ROWS, P.N - n0);
                const int kw = (k1 - k0) * BITS / 32;               // words of this stage per row
                for (int e = lane; e < nrows * kw; e += 32) {
                    const int r = e / kw, wd = e - r * kw;
                    const int seg = wd / SEGW, sw = wd - seg * SEGW;
                    uint32_t *d = reinterpret_cast<uint32_t *>(st + (seg * ROWS + r) * SEGP) + sw;
                    const long long src = (long long)(n0 + r) * row_words + (long long)k0 * BITS / 32 + wd;
                    if (TFQ_IN(P, in_stages(P, smem, d, 4) && n0 + r < P.N && (long long)k0 * BITS / 32 + wd < row_words))
                        *d = __ldg(P.W + src);
                }
                const int ng = (k1 - k0) / G;
                for (int e = lane; e < nrows * ng; e += 32) {
                    const int r = e / ng, gg = e - r * ng;
                    const long long src = (long long)(n0 + r) * ngK + k0 / G + gg;
                    uint16_t *ds = reinterpret_cast<uint16_t *>(sst + r * P.sbpitch) + gg;
                    uint16_t *db = reinterpret_cast<uint16_t *>(bst + r * P.sbpitch) + gg;
                    if (TFQ_IN(P, in_stages(P, smem, ds, 2) && in_stages(P, smem, db, 2) && n0 + r < P.N &&
                                      k0 / G + gg < ngK)) {
                        *ds = __ldg(P.s + src);
                        *db = __ldg(P.b + src);
                    }
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[slot]);
            }
        }
    }
    // Drain: the last stages' copies must land before the CTA may exit
    // (walk the ring back over the last min(it, S) stages).
    if (P.bulk && lane == 0) {
        const uint32_t n = it < (uint32_t)S ? it : (uint32_t)S;
        uint32_t slot = ring.slot, phase = ring.phase;
        for (uint32_t j = 0; j < n; ++j) {
            if (slot == 0) {
                slot = (uint32_t)S;
                phase ^= 1u;
            }
            --slot;
            if (P.stall && it - 1 - j == 0) continue;    // the withheld first stage
            mbar_wait(&full[slot], phase, abort, P.status, false);
        }
    }
}

// ------------------------------------------------------------- consumers --

// Activations of one K slice, permuted into mma B-fragment order, and the
// per-(group,row) sums of x.  Layout [run][RB rows][4 quad lanes] of uint4
// (rows >= `rows` are zero): entry (run, row, quad lane q) holds the B
// registers of the run's two k-steps, so one 16-byte load feeds two MMAs.
// Code i of an 8-code run is paired with code i+4, so a run x0..x7 feeds its
// first step as {(x0,x4),(x1,x5)} and its second as {(x2,x6),(x3,x7)}.
// sum_group(x) is the sequential fp32 sum of the group's x in k order, from 0.
// Two forms with the same result: one thread per (group, row) loads, places
// and sums its group (load_x_groups), or every thread places 8-value pieces and
// one thread per (group, row) then sums its group from shared memory
// (load_x_pieces).  With groups of 64 or 128 the first form's long per-group
// loops leave most threads idle: the second measured 0.3-0.5 us faster per
// 4096 x 4096 product and 0.4 us per 16-row 6192 x 2048 stack, but 0.3 us
// slower on that stack at one row (two rows and a 2048 slice keep the first
// form); with 32-wide groups the second pass's bank conflicts make it slower
// (0.3-1.4 us at 8-16 rows).  Threads 0..nthr-1 run either.
template <int G, int RB>
__device__ void load_x_groups(const QmmParams &P, const Item &I, uint4 *Bf, float *sx, int tid, int nthr) {
    static_assert(RB >= 2, "layout rows");
    const int rows = P.rows;
    const int ngs = (I.k_hi - I.k_lo) / G;
    [[maybe_unused]] const uint8_t *smem = reinterpret_cast<const uint8_t *>(Bf) - P.x_off;
    for (int u = tid; u < RB * ngs; u += nthr) {
        const int r = u / ngs, gs = u - r * ngs;
        float acc = 0.f;
        const int xr = r < rows ? P.xrow[r] : 0;
        const uint16_t *src = P.x + (long long)xr * P.K + I.k_lo + gs * G;
#pragma unroll 4
        for (int t = 0; t < G / 8; ++t) {
            const int qq = (8 * t) / (G / 4), m = ((8 * t) % (G / 4)) / 8;
            const int run = gs * (G / 32) + m;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows && TFQ_IN(P, xr >= 0 && xr < P.x_rows && I.k_lo + gs * G + 8 * t + 8 <= P.K))
                v = *reinterpret_cast<const uint4 *>(src + 8 * t);
            uint4 *d = Bf + (run * RB + r) * 4 + qq;
            if (TFQ_IN(P, in_b(P, smem, d, 16)))
                *d = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                                prmt(v.y, v.w, 0x7632u));
            acc += bf16f((uint16_t)(v.x & 0xFFFF));
            acc += bf16f((uint16_t)(v.x >> 16));
            acc += bf16f((uint16_t)(v.y & 0xFFFF));
            acc += bf16f((uint16_t)(v.y >> 16));
            acc += bf16f((uint16_t)(v.z & 0xFFFF));
            acc += bf16f((uint16_t)(v.z >> 16));
            acc += bf16f((uint16_t)(v.w & 0xFFFF));
            acc += bf16f((uint16_t)(v.w >> 16));
        }
        if (TFQ_IN(P, in_sx(P, smem, sx + gs * RB + r, 4))) sx[gs * RB + r] = acc;
    }
}

// B-layout slot of piece pc (the 8 x values at slice offset 8*pc) of row r.
template <int G, int RB>
__device__ __forceinline__ int piece_slot(int pc, int r) {
    constexpr int PPG = G / 8;                       // pieces of a group
    const int gs = pc / PPG, t = pc - gs * PPG;
    const int qq = (8 * t) / (G / 4), m = ((8 * t) % (G / 4)) / 8;
    return ((gs * (G / 32) + m) * RB + r) * 4 + qq;
}

// Piece form; `bar` is the threads' named barrier between the two passes.
template <int G, int RB>
__device__ void load_x_pieces(const QmmParams &P, const Item &I, uint4 *Bf, float *sx, int tid, int nthr,
                              int bar) {
    static_assert(RB >= 2, "layout rows");
    constexpr int BATCH = 4;                         // loads a thread keeps in flight
    const int rows = P.rows;
    [[maybe_unused]] const uint8_t *smem = reinterpret_cast<const uint8_t *>(Bf) - P.x_off;
    const int npc = (I.k_hi - I.k_lo) / 8;           // pieces of one row
    const int total = RB * npc;
    for (int u0 = tid; u0 < total; u0 += BATCH * nthr) {
        uint4 v[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int u = u0 + j * nthr;
            const int r = u / npc, pc = u - r * npc;
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (u < total && r < rows &&
                TFQ_IN(P, P.xrow[r] >= 0 && P.xrow[r] < P.x_rows && I.k_lo + 8 * pc + 8 <= P.K))
                v[j] = *reinterpret_cast<const uint4 *>(P.x + (long long)P.xrow[r] * P.K + I.k_lo + 8 * pc);
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int u = u0 + j * nthr;
            const int r = u / npc, pc = u - r * npc;
            uint4 *d = Bf + piece_slot<G, RB>(pc, r);
            if (u < total && TFQ_IN(P, in_b(P, smem, d, 16)))
                *d = make_uint4(prmt(v[j].x, v[j].z, 0x5410u), prmt(v[j].x, v[j].z, 0x7632u),
                                prmt(v[j].y, v[j].w, 0x5410u), prmt(v[j].y, v[j].w, 0x7632u));
        }
    }
    named_bar(bar, nthr);
    const int ngs = npc / (G / 8);
    for (int u = tid; u < RB * ngs; u += nthr) {
        const int r = u / ngs, gs = u - r * ngs;
        float acc = 0.f;
        if (r < rows) {
#pragma unroll
            for (int t = 0; t < G / 8; ++t) {
                // Stored pairs (x0,x4) (x1,x5) (x2,x6) (x3,x7): add x0..x7 in order.
                const uint4 *pw = Bf + piece_slot<G, RB>(gs * (G / 8) + t, r);
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (TFQ_IN(P, in_b(P, smem, pw, 16))) w = *pw;
                acc += bf16f((uint16_t)(w.x & 0xFFFF));
                acc += bf16f((uint16_t)(w.y & 0xFFFF));
                acc += bf16f((uint16_t)(w.z & 0xFFFF));
                acc += bf16f((uint16_t)(w.w & 0xFFFF));
                acc += bf16f((uint16_t)(w.x >> 16));
                acc += bf16f((uint16_t)(w.y >> 16));
                acc += bf16f((uint16_t)(w.z >> 16));
                acc += bf16f((uint16_t)(w.w >> 16));
            }
        }
        if (TFQ_IN(P, in_sx(P, smem, sx + gs * RB + r, 4))) sx[gs * RB + r] = acc;
    }
}

// Scales (or biases) of one segment for one row: NGS bf16 values, one vector load.
template <int NGS>
struct SegVals;
template <>
struct SegVals<8> {
    uint4 v;
    __device__ __forceinline__ void load(const uint16_t *p) { v = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ float get(int i) const {
        const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};
template <>
struct SegVals<4> {
    uint2 v;
    __device__ __forceinline__ void load(const uint16_t *p) { v = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ float get(int i) const {
        const uint32_t w = i < 2 ? v.x : v.y;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};
template <>
struct SegVals<2> {
    uint32_t v;
    __device__ __forceinline__ void load(const uint16_t *p) { v = *reinterpret_cast<const uint32_t *>(p); }
    __device__ __forceinline__ float get(int i) const {
        return __uint_as_float((i & 1) ? (v & 0xFFFF0000u) : (v << 16));
    }
};

// 4-, 5- and 6-bit codes enter the MMA as 128 + c (every pair of their runs
// sits at mantissa position 0, so this saves one instruction per pair); 2-,
// 3- and 8-bit codes enter exactly (the pages enter 2-bit codes exactly, and at
// 8 bits 128 + c does not fit the bf16 significand).
__host__ __device__ constexpr bool offset_codes(int bits) { return bits >= 4 && bits <= 6; }

// The group's bias coefficient: b, or b - 128 s (one rounding) for offset codes.
template <int BITS>
__device__ __forceinline__ float bias_term(float s, float b) {
    return offset_codes(BITS) ? fmaf(-128.f, s, b) : b;
}

// One group of this lane's 2*MT columns (rows t*16+g and t*16+g+8 of each
// m-tile t): T = tensor-core dot products of the group's codes with x (offset
// codes 128 + c at 4-6 bits, exact codes c otherwise), then p = fma(s,T,p);
// p = fma(b',sum_group(x),p); bg holds b' = b, or b - 128 s for offset codes.  pr[m]: run m of the lane's
// quarter in row g of m-tile 0 (other rows at compile-time offsets); for 6-bit
// codes pr[m] / pr2[m] are the run's first / second word in this lane's load
// order; woff: the group's word offset in the segment row; bq: this lane's B
// entry of the group's first run (shared by the m-tiles); sxq: the group's
// sum_group(x).
template <int BITS, int G, int RB, int MT>
__device__ __forceinline__ void group_body(const QmmParams &P, const uint8_t *smem,
                                           const uint32_t *const (&pr)[G / 32], const uint32_t *const (&pr2)[G / 32],
                                           const uint32_t (&ua)[G / 32], const uint32_t (&ub)[G / 32],
                                           uint32_t mg, uint32_t mq, int woff, const uint4 *bq, const float (&sg)[MT][2],
                                           const float (&bg)[MT][2], const float *sxq,
                                           float (&p)[MT][(RB > 8 ? 2 : 1)][4]) {
    constexpr int NT = RB > 8 ? 2 : 1;
    constexpr int LR = layout_rows(RB);
    constexpr int RUNS = G / 32;
    constexpr int RW = Pitch<BITS, G>::SEGP / 4;     // words between rows of a segment block
    // With offset codes the MMA takes 128 + c (one instruction per pair less):
    // T' = T + 128 sum_group(x), and bg holds b - 128 s.
    constexpr bool OFF = offset_codes(BITS);
    // 4- and 8-bit runs of a lane lie in consecutive aligned words: with two or
    // four runs a group, one vector load per row feeds them all.
    constexpr int VW = (BITS == 4 || BITS == 8) && RUNS >= 2 ? RUNS * BITS / 4 : 0;   // words
    uint32_t vw[MT][2][VW > 0 ? VW : 1];
    if (VW == 2 || VW == 4 || VW == 8) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t *src = pr[0] + woff + (t * 16 + 8 * h) * RW;
                const bool ok = TFQ_IN(P, in_stages(P, smem, src, 4 * (VW > 0 ? VW : 1)));
#pragma unroll
                for (int v = 0; v < VW; v += (VW >= 4 ? 4 : 2)) {
                    if (VW >= 4) {
                        uint4 u = make_uint4(0u, 0u, 0u, 0u);
                        if (ok) u = *reinterpret_cast<const uint4 *>(src + v);
                        vw[t][h][v] = u.x, vw[t][h][v + 1] = u.y, vw[t][h][v + 2] = u.z, vw[t][h][v + 3] = u.w;
                    } else {
                        uint2 u = make_uint2(0u, 0u);
                        if (ok) u = *reinterpret_cast<const uint2 *>(src + v);
                        vw[t][h][v] = u.x, vw[t][h][v + 1] = u.y;
                    }
                }
            }
    }
    float c[MT][NT][4];
#pragma unroll
    for (int m = 0; m < RUNS; ++m) {
        uint4 bb[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4 *pb = bq + (m * LR + nt * 8) * 4;
            bb[nt] = make_uint4(0u, 0u, 0u, 0u);
            if (TFQ_IN(P, in_b(P, smem, pb, 16))) bb[nt] = *pb;
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            // A registers in MMA operand order: a[2i] = pair i of row g, a[2i+1] of row g+8.
            uint32_t a[8];
            if (VW > 0) {
                Unpack<BITS>::template run<2, OFF>(&vw[t][0][m * BITS / 4], ua[m], ub[m], mg, mq, a);
                Unpack<BITS>::template run<2, OFF>(&vw[t][1][m * BITS / 4], ua[m], ub[m], mg, mq, a + 1);
            } else if constexpr (BITS == 6) {
                const int o0 = woff + (t * 16) * RW, o1 = woff + (t * 16 + 8) * RW;
                uint32_t w00 = 0u, w01 = 0u, w10 = 0u, w11 = 0u;
                if (TFQ_IN(P, in_stages(P, smem, pr[m] + o0, 4) && in_stages(P, smem, pr2[m] + o0, 4) &&
                                  in_stages(P, smem, pr[m] + o1, 4) && in_stages(P, smem, pr2[m] + o1, 4))) {
                    w00 = pr[m][o0], w01 = pr2[m][o0], w10 = pr[m][o1], w11 = pr2[m][o1];
                }
                Unpack<6>::template run_words<2, OFF>(w00, w01, ua[m], ub[m], mg, mq, a);
                Unpack<6>::template run_words<2, OFF>(w10, w11, ua[m], ub[m], mg, mq, a + 1);
            } else {
                // A run reads at most two words from its first.
                const uint32_t *r0 = pr[m] + woff + (t * 16) * RW, *r1 = pr[m] + woff + (t * 16 + 8) * RW;
                if (!TFQ_IN(P, in_stages(P, smem, r0, 8) && in_stages(P, smem, r1, 8)))
                    r0 = r1 = reinterpret_cast<const uint32_t *>(smem + P.st_off);
                Unpack<BITS>::template run<2, OFF>(r0, ua[m], ub[m], mg, mq, a);
                Unpack<BITS>::template run<2, OFF>(r1, ua[m], ub[m], mg, mq, a + 1);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (m == 0)
                    mma_bf16_first(c[t][nt], a[0], a[1], a[2], a[3], bb[nt].x, bb[nt].y);
                else
                    mma_bf16(c[t][nt], a[0], a[1], a[2], a[3], bb[nt].x, bb[nt].y);
                mma_bf16(c[t][nt], a[4], a[5], a[6], a[7], bb[nt].z, bb[nt].w);
            }
        }
    }
    if (RB == 1) {   // a single activation row: only row 0 of the tile is live
        float x0 = 0.f;
        if (TFQ_IN(P, in_sx(P, smem, sxq, 4))) x0 = *sxq;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            p[t][0][0] = fmaf(bg[t][0], x0, fmaf(sg[t][0], c[t][0][0], p[t][0][0]));
            p[t][0][2] = fmaf(bg[t][1], x0, fmaf(sg[t][1], c[t][0][2], p[t][0][2]));
        }
    } else {   // the two activation rows of a lane in one packed fp32x2 FMA each
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float2 v = make_float2(0.f, 0.f);
            if (TFQ_IN(P, in_sx(P, smem, sxq + nt * 8, 8))) v = *reinterpret_cast<const float2 *>(sxq + nt * 8);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                fma2(p[t][nt][0], p[t][nt][1], sg[t][0], sg[t][0], c[t][nt][0], c[t][nt][1]);
                fma2(p[t][nt][0], p[t][nt][1], bg[t][0], bg[t][0], v.x, v.y);
                fma2(p[t][nt][2], p[t][nt][3], sg[t][1], sg[t][1], c[t][nt][2], c[t][nt][3]);
                fma2(p[t][nt][2], p[t][nt][3], bg[t][1], bg[t][1], v.x, v.y);
            }
        }
    }
}

__device__ __forceinline__ int dst_col(const QmmParams &P, int n) {
    for (int i = 0; i < P.ncs; ++i) {
        const int d = n - P.cs_src[i];
        if (d >= 0 && d < P.cs_len[i]) return P.cs_dst[i] + d;
    }
    return -1;
}

// Output (window row r, column n) = v: the optional squared-ReLU epilogue in
// fp32, then an fp32 or a round-to-nearest-even bf16 store.
__device__ __forceinline__ void store_y(const QmmParams &P, int r, int n, float v) {
    if (r < P.rows && n < P.N) {
        const int d = dst_col(P, n);
        if (d < 0) return;
        if (P.out & OUT_RELU2) {
            const float u = fmaxf(v, 0.f);
            v = u * u;
        }
        const long long at = (long long)P.yrow[r] * P.y_stride + d;
        if (!TFQ_IN(P, P.yrow[r] >= 0 && P.yrow[r] < P.y_rows && d < P.y_stride)) return;
        if (P.out & OUT_BF16)
            reinterpret_cast<__nv_bfloat16 *>(P.y)[at] = __float2bfloat16_rn(v);
        else
            P.y[at] = v;
    }
}

// Consumer group `cg` of CG (eight warps each; warp w of a group takes segment
// w of a stage) computes every CG-th item of this CTA's walk, starting at item
// cg, and steps the ring over the other groups' stages without waiting on
// them; each ring slot is consumed by exactly one group.  With CG = 2 two
// stages are computed at once (twice the warps to hide unpack latency) while
// the activations stay shared: the plan gives CG = 2 only a single K slice.
template <int BITS, int G, int RB, int MT, int CG>
__device__ void consumer(const QmmParams &P, uint8_t *smem, uint64_t *full, uint64_t *empty,
                         volatile int *abort, const volatile uint32_t *magic) {
    constexpr int NT = RB > 8 ? 2 : 1;
    constexpr int ROWS = TN * MT;
    constexpr int SEGP = Pitch<BITS, G>::SEGP;
    constexpr int QG = G / 4;                // codes of a group per quad lane
    constexpr int RUNS = G / 32;             // 8-code runs per quad lane per group
    constexpr int GW = G * BITS / 32;        // words per group of one row
    constexpr int NGS = SEG / G;             // groups per segment
    constexpr int LR = layout_rows(RB);      // rows of the B / sum_group(x) layouts
    constexpr int NOUT = ROWS * LR;          // outputs of an item (padded rows)
    constexpr int GT = NCW * 32;             // threads of one consumer group
    constexpr int OUTS = (NOUT + GT - 1) / GT;   // outputs folded per thread
    const int tid = threadIdx.x;
    const int cg = CG == 1 ? 0 : tid / GT;
    const int gtid = tid - cg * GT;          // thread within the group
    const int warp = gtid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int S = P.stages, rows = P.rows;
    const int gbar = 2 + cg;                 // the group's named barrier (1: all consumers)
    uint4 *Bf = reinterpret_cast<uint4 *>(smem + P.x_off);
    float *sx = reinterpret_cast<float *>(smem + P.sx_off);
    float *pbuf = reinterpret_cast<float *>(smem + P.pb_off) + cg * (2 * SEGS * ROWS * LR);   // [2][SEGS][ROWS][LR]
    const uint8_t *zero = smem + P.z_off;
    // Lanes past the bucket's rows read a zero block instead of B / sum_group(x).
    const bool b_lane = g < LR, sx_lane = 2 * q < LR;
    if (LR < 8) {
        for (int i = tid; i < ZERO_BYTES / 4; i += CG * GT) reinterpret_cast<uint32_t *>(smem + P.z_off)[i] = 0u;
    }
    // This lane's runs inside any group: word offset and unpack arguments of run m.
    // A 6-bit run spans two words; with groups of 32 or 128 lanes whose quarter
    // starts at words {0,1,3,4} (or {0,6,12,18}) + a multiple of 4 per row would
    // meet in pairs on one bank, so half the lanes load the second word first
    // (their selectors flipped to match): every load is then conflict-free.
    // The one- and two-row kernels with two consumer groups keep the plain
    // order: under their 96-register cap the second pointer set spills (the
    // 6-bit LM head measured 6 % slower), and they wait least on shared memory.
    constexpr bool SWAP6 = BITS == 6 && !(RB <= 2 && CG == 2);
    const uint32_t d6 = (SWAP6 && ((G == 32 && !(q & 1)) || (G == 128 && q < 2))) ? 1u : 0u;
    uint32_t wo[RUNS], ua[RUNS], ub[RUNS];
#pragma unroll
    for (int m = 0; m < RUNS; ++m) {
        const uint32_t bit = (uint32_t)(q * QG + 8 * m) * BITS;
        wo[m] = bit >> 5;
        lane_args<BITS>(bit & 31u, ua[m], ub[m]);
        if (d6) {
            ua[m] ^= 0x4444u;
            ub[m] ^= 0x4444u;
        }
    }
    float yacc[OUTS];
#pragma unroll
    for (int i = 0; i < OUTS; ++i) yacc[i] = 0.f;
    const uint32_t mg = magic[0], mq = magic[1];   // MAGIC, QP<BITS>: read at run time, held in registers

    // x, y and the split-K workspace may be touched by the previous kernel of
    // the stream (programmatic dependent launch): wait for it first -- unless
    // this is a later run of a stack, which shares nothing it writes with the
    // runs before it, or the caller declared that the previous kernel writes
    // neither x nor the weights (early x): then only the first write below
    // waits.  The first run of a stack lets the later runs start only now, so
    // that they too read x after its producer finished.
    const bool early_x = P.early_x && P.dep == 0;
    if (P.dep != 2 && !early_x) grid_dependency_wait();
    if (tid == 0 && !early_x) TFQ_TRACE(smem, TR_RELEASE);
    if (P.dep == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    bool waited = !early_x;                  // this thread has passed the dependency wait
    // Early x: the outputs of an item finished before the dependency release wait
    // in registers and are stored after it, with the group's next item, so that the
    // group computes that item before the release.  One item is parked, in the one-
    // and two-row single-group instances only (their CTAs hold few items; more
    // parked items, or parking elsewhere, measured slower).
    constexpr bool PARK = RB <= 2 && CG == 1;
    float dv[OUTS];
    int dn0 = 0;
    bool parked = false;
    auto flush = [&]() {
        if (parked) {
#pragma unroll
            for (int i = 0; i < OUTS; ++i) {
                const int o = gtid + i * GT;
                if (o < NOUT) store_y(P, o - (o / LR) * LR, dn0 + o / LR, dv[i]);
            }
        }
        parked = false;
    };
    int cur_slice = -1;
    uint32_t it = 0;                         // stages this group has computed
    Ring ring;
    int own = 0;                             // position of the item in this CTA's walk
    for (ItemWalk iw(P); iw.more(P); iw.next(P), ++own) {
        const Item I = iw.get(P);
        if (I.slice != cur_slice) {
            // Every group walks every item, so all consumers meet here before the
            // x slice is overwritten (the first slice overwrites nothing: its
            // warps start placing x at once; the barrier after the placement
            // still orders it before every read).
            if (cur_slice >= 0) named_bar(1, CG * GT);
            if (G >= 64 && (LR > 2 || I.k_hi - I.k_lo >= 4096))
                load_x_pieces<G, LR>(P, I, Bf, sx, tid, CG * GT, 1);
            else
                load_x_groups<G, LR>(P, I, Bf, sx, tid, CG * GT);
            named_bar(1, CG * GT);
            if (tid == 0 && cur_slice < 0) TFQ_TRACE(smem, TR_XLOADED);
            cur_slice = I.slice;
        }
        if (CG > 1 && (own % CG) != cg) {    // another group's item: skip its stages
            for (int k0 = I.k_lo; k0 < I.k_hi; k0 += CHUNK) ring.next(S);
            continue;
        }
        const int n0 = I.mt * ROWS;
        for (int k0 = I.k_lo; k0 < I.k_hi; k0 += CHUNK, ++it, ring.next(S)) {
            const int k1 = min(I.k_hi, k0 + CHUNK);
            const int slot = (int)ring.slot;
            const int buf = it & 1;
            const int ks0 = k0 + warp * SEG;      // this warp's segment
            const bool active = ks0 < k1;
            // With two consumer groups a group skips the other's stages, so the
            // slot's previous fill may belong to the other group and may not
            // have landed yet; a parity wait on `full` alone could then pass a
            // phase early.  First wait, as the producer did before this fill,
            // for the previous fill's consumers to release the slot: `full` is
            // then exactly one phase from this fill.  (A fresh barrier passes
            // the parity-1 wait at once.)
            if (CG > 1) mbar_wait(&empty[slot], ring.phase ^ 1u, abort, P.status);
            mbar_wait(&full[slot], ring.phase, abort, P.status);
            float p[MT][NT][4];
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) p[t][nt][0] = p[t][nt][1] = p[t][nt][2] = p[t][nt][3] = 0.f;
            if (active) {
                const uint8_t *st = smem + P.st_off + slot * P.stage_bytes;
                const uint32_t *wr = reinterpret_cast<const uint32_t *>(st + (warp * ROWS + g) * SEGP);
                const uint32_t *pr[RUNS], *pr2[RUNS];
#pragma unroll
                for (int m = 0; m < RUNS; ++m) {
                    pr[m] = wr + wo[m] + d6;
                    pr2[m] = wr + wo[m] + (1u - d6);
                }
                const uint8_t *sbase = st + SEGS * ROWS * SEGP;
                const int gseg = warp * NGS;                             // segment's first group in the stage
                const int gs0 = (ks0 - I.k_lo) / G;                      // slice group index
                const uint4 *bq = (LR >= 8 || b_lane) ? Bf + (gs0 * RUNS * LR + g) * 4 + q
                                                      : reinterpret_cast<const uint4 *>(zero) + q;
                const float *sxq = (LR >= 8 || sx_lane) ? sx + gs0 * LR + 2 * q
                                                        : reinterpret_cast<const float *>(zero);
                const int ng = (min(k1, ks0 + SEG) - ks0) / G;
                const uint16_t *sp = reinterpret_cast<const uint16_t *>(sbase + g * P.sbpitch) + gseg;
                const uint16_t *bp = reinterpret_cast<const uint16_t *>(sbase + (ROWS + g) * P.sbpitch) + gseg;
                const int rstep = 8 * P.sbpitch / 2;                     // 8 rows, in bf16 elements
                if (ng == NGS) {
                    // Scales and biases in vector loads of NV groups: two for the
                    // two-m-tile kernels with two consumer groups (wider loads spill
                    // under their 96-register cap; the 6-bit LM head measured 5 %
                    // faster), four for 16 rows with two groups.
                    constexpr int NV = CG == 2 ? (MT == 2 ? (NGS >= 4 ? 2 : NGS) : (NGS == 8 ? 4 : NGS)) : NGS;
#pragma unroll
                    for (int g0 = 0; g0 < NGS; g0 += NV) {
                        SegVals<NV> Sv[MT][2], Bv[MT][2];
#pragma unroll
                        for (int t = 0; t < MT; ++t)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint16_t *ps = sp + (2 * t + h) * rstep + g0, *pb = bp + (2 * t + h) * rstep + g0;
                                if (TFQ_IN(P, in_stages(P, smem, ps, 2 * NV) && in_stages(P, smem, pb, 2 * NV))) {
                                    Sv[t][h].load(ps);
                                    Bv[t][h].load(pb);
                                } else {
                                    Sv[t][h].load(reinterpret_cast<const uint16_t *>(smem + P.st_off));
                                    Bv[t][h].load(reinterpret_cast<const uint16_t *>(smem + P.st_off));
                                }
                            }
#pragma unroll
                        for (int gv = 0; gv < NV; ++gv) {
                            const int gl = g0 + gv;
                            float sg[MT][2], bg[MT][2];
#pragma unroll
                            for (int t = 0; t < MT; ++t)
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    sg[t][h] = Sv[t][h].get(gv);
                                    bg[t][h] = bias_term<BITS>(sg[t][h], Bv[t][h].get(gv));
                                }
                            group_body<BITS, G, RB, MT>(P, smem, pr, pr2, ua, ub, mg, mq, gl * GW,
                                                        bq + gl * RUNS * LR * 4, sg, bg, sxq + gl * LR, p);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int gl = 0; gl < ng; ++gl) {
                        float sg[MT][2], bg[MT][2];
#pragma unroll
                        for (int t = 0; t < MT; ++t)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint16_t *ps = sp + (2 * t + h) * rstep + gl, *pb = bp + (2 * t + h) * rstep + gl;
                                const bool ok = TFQ_IN(P, in_stages(P, smem, ps, 2) && in_stages(P, smem, pb, 2));
                                sg[t][h] = ok ? bf16f(*ps) : 0.f;
                                bg[t][h] = bias_term<BITS>(sg[t][h], ok ? bf16f(*pb) : 0.f);
                            }
                        group_body<BITS, G, RB, MT>(P, smem, pr, pr2, ua, ub, mg, mq, gl * GW,
                                                    bq + gl * RUNS * LR * 4, sg, bg, sxq + gl * LR, p);
                    }
                }
            }
            {   // release the slot once every shared read of it has been consumed
                float dep = 0.f;
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) dep += p[t][nt][0] + p[t][nt][2];
                __syncwarp();
                if (lane == 0) mbar_arrive_after(&empty[slot], dep);
            }
            // Segment partial -> pbuf[buf][warp][row][padded activation row];
            // a lane's two activation rows are adjacent: one 8-byte store.
            float *pw = pbuf + ((buf * SEGS + warp) * ROWS) * LR;
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = nt * 8 + 2 * q;
                        const int c = t * 16 + g + 8 * h;
                        if (r < LR && TFQ_IN(P, in_pbuf(P, smem, pw + c * LR + r, 8)))
                            *reinterpret_cast<float2 *>(pw + c * LR + r) = make_float2(p[t][nt][2 * h], p[t][nt][2 * h + 1]);
                    }
            named_bar(gbar, GT);
            if (tid == 0 && it == 0) TFQ_TRACE(smem, TR_STAGE0);
            // Early x: every thread passes the dependency wait before the first
            // write of y or of split-K partials (the fold below); an item's final
            // outputs are parked instead while the group has a later item and room.
            bool park = false;
            if (!waited && (P.nsl > 1 || k0 + CHUNK >= I.k_hi)) {
                const bool later = iw.mt + CG * iw.team < P.nmt;
                if (PARK && P.nsl == 1 && later && !parked) {
                    park = true;
                } else {
                    grid_dependency_wait();
                    waited = true;
                    if (tid == 0) TFQ_TRACE(smem, TR_RELEASE);
                    flush();
                }
            }
            // Chunk sum C = P_0 + P_1 + ... in segment order, then the chunk fold.
            const int nseg = (k1 - k0 + SEG - 1) / SEG;
            const int chunk = k0 / CHUNK;
#pragma unroll
            for (int i = 0; i < OUTS; ++i) {
                const int o = gtid + i * GT;
                if (o < NOUT) {
                    const int fc = o / LR, fr = o - (o / LR) * LR;
                    const float *pf = pbuf + (buf * SEGS * ROWS + fc) * LR + fr;
                    // All segment partials are loaded first (independent loads in
                    // flight together), then added in segment order.
                    float v[SEGS];
#pragma unroll
                    for (int j = 0; j < SEGS; ++j)
                        v[j] = j < nseg && TFQ_IN(P, in_pbuf(P, smem, pf + j * ROWS * LR, 4)) ? pf[j * ROWS * LR] : 0.f;
                    float C = v[0];
#pragma unroll
                    for (int j = 1; j < SEGS; ++j)
                        if (j < nseg) C = C + v[j];
                    if (P.nsl == 1) {
                        yacc[i] = chunk == 0 ? C : yacc[i] + C;
                        if (k0 + CHUNK >= I.k_hi) {
                            if (park) {
                                dv[i] = yacc[i];
                            } else {
                                store_y(P, fr, n0 + fc, yacc[i]);
                            }
                        }
                    } else if (fr < rows && n0 + fc < P.N) {
                        const long long at = ((long long)chunk * rows + fr) * P.N + n0 + fc;
                        if (TFQ_IN(P, at < P.ws_elems)) P.ws[at] = C;
                    }
                }
            }
            if (park) {
                dn0 = n0;
                parked = true;
            }
        }
    }
    // Every thread passes the dependency wait before it exits, so that this
    // grid never completes before the one it depends on (a later kernel's
    // wait on this grid then covers every kernel before it).
    if (!waited) {
        grid_dependency_wait();
        if (tid == 0) TFQ_TRACE(smem, TR_RELEASE);
    }
    flush();
    if (CG == 1 && P.nsl > 1) {
        // Split K: once all of this CTA's chunk sums are out, one arrival ticket
        // per item, issued together; the last CTA to arrive at an item folds its
        // chunk sums in chunk order and rearms the counter.  Nothing waits on
        // another CTA.  The flags reuse the partial-sum buffer.
        int *last = reinterpret_cast<int *>(pbuf);
        const int team = gridDim.x / P.nsl;
        const int mt0 = blockIdx.x % team;                  // this CTA's first column tile
        const int nmine = mt0 < P.nmt ? (P.nmt - mt0 + team - 1) / team : 0;
        __threadfence();
        named_bar(gbar, GT);
        for (int b0 = 0; b0 < nmine; b0 += GT) {
            const int nb = min(GT, nmine - b0);
            if (gtid < nb) {
                const int mt = mt0 + (b0 + gtid) * team;
                int lst = 0;
                if (TFQ_IN(P, mt < P.n_counters)) {
                    lst = atomicAdd(&P.counters[mt], 1) == P.nsl - 1;
                    if (lst) P.counters[mt] = 0;            // no other arrival in this launch
                }
                if (TFQ_IN(P, in_pbuf(P, smem, last + gtid, 4))) last[gtid] = lst;
            }
            named_bar(gbar, GT);
            __threadfence();
            for (int j = 0; j < nb; ++j) {
                if (!TFQ_IN(P, in_pbuf(P, smem, last + j, 4)) || !last[j]) continue;   // the same for the whole group
                const int n0 = (mt0 + (b0 + j) * team) * ROWS;
#pragma unroll
                for (int i = 0; i < OUTS; ++i) {
                    const int o = gtid + i * GT;
                    if (o < NOUT) {
                        const int fc = o / LR, fr = o - (o / LR) * LR;
                        if (fr < rows && n0 + fc < P.N) {
                            const long long n = n0 + fc;
                            float v = 0.f;
                            if (TFQ_IN(P, (long long)fr * P.N + n < P.ws_elems)) v = __ldcg(P.ws + (long long)fr * P.N + n);
                            for (int ch = 1; ch < P.nchunks; ++ch) {
                                const long long at = ((long long)ch * rows + fr) * P.N + n;
                                if (TFQ_IN(P, at < P.ws_elems)) v = v + __ldcg(P.ws + at);
                            }
                            store_y(P, fr, (int)n, v);
                        }
                    }
                }
            }
            named_bar(gbar, GT);                             // before the flags are rewritten
        }
    }
    if (tid == 0) TFQ_TRACE(smem, TR_EXIT);
}

// ------------------------------------------------------------------ kernel --

// Register ceiling per thread.  An SM's 65,536 registers are split evenly
// over its four schedulers and each warp draws on its scheduler's share, so
// the busiest scheduler decides: two CTAs of nine warps (MT = 1) or one of
// 17 warps (CG = 2) put five warps on one scheduler (16,384 / (5 * 32),
// rounded down to a multiple of 8: 96); one CTA of nine warps puts three (168).
template <int MT, int CG>
struct RegCap {
    static constexpr int value = (CG == 2 || MT == 1) ? 96 : 168;
};

template <int BITS, int G, int RB, int MT, int CG>
__global__ void __maxnreg__((RegCap<MT, CG>::value)) qmm_kernel(const __grid_constant__ QmmParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + MAX_STAGES;
    volatile int *abort = reinterpret_cast<volatile int *>(empty + MAX_STAGES);
    volatile uint32_t *magic = reinterpret_cast<volatile uint32_t *>(abort + 2);
    if (threadIdx.x == 0) {
        TFQ_TRACE_BEGIN(P, smem);
        for (int i = 0; i < P.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        *abort = 0;
        magic[0] = MAGIC;
        magic[1] = QP<BITS>::value;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // The next kernel of the stream may start its prologue once every CTA of
    // this grid is resident (no effect without programmatic dependent launch).
    if (P.dep != 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x >= CG * NCW * 32)
        producer<BITS, G, MT>(P, smem, full, empty, abort);
    else
        consumer<BITS, G, RB, MT, CG>(P, smem, full, empty, abort, magic);
    // A later run of a stack completes only after the run before it, so the
    // stack's last launch completes after all of them.
    if (P.dep == 2) grid_dependency_wait();
}

// Host-side launcher for one width: every group and row bucket.
template <int BITS>
cudaError_t launch_width(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                         cudaStream_t st, bool pdl) {
#define TFQ_CASE(G_, RB_, MT_, CG_)                                                           \
    if (group == G_ && rb == RB_ && mt == MT_ && cg == CG_) {                                 \
        auto k = qmm_kernel<BITS, G_, RB_, MT_, CG_>;                                         \
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
        cudaLaunchConfig_t cfg = {};                                                          \
        cfg.gridDim = dim3(grid);                                                             \
        cfg.blockDim = dim3(block_threads(CG_));                                              \
        cfg.dynamicSmemBytes = smem;                                                          \
        cfg.stream = st;                                                                      \
        cudaLaunchAttribute attr[1];                                                          \
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                      \
        attr[0].val.programmaticStreamSerializationAllowed = 1;                               \
        cfg.attrs = attr;                                                                     \
        cfg.numAttrs = pdl ? 1 : 0;                                                           \
        return cudaLaunchKernelEx(&cfg, k, TFQ_LAUNCH_PARAMS(P));                             \
    }
#define TFQ_ROWS(G_) TFQ_CASE(G_, 1, 1, 1) TFQ_CASE(G_, 2, 1, 1) TFQ_CASE(G_, 4, 1, 1) TFQ_CASE(G_, 8, 1, 1) \
    TFQ_CASE(G_, 16, 1, 1) TFQ_CASE(G_, 1, 2, 1) TFQ_CASE(G_, 2, 2, 1) TFQ_CASE(G_, 4, 2, 1)                \
    TFQ_CASE(G_, 8, 2, 1) TFQ_CASE(G_, 16, 2, 1) TFQ_CASE(G_, 1, 2, 2) TFQ_CASE(G_, 2, 2, 2) TFQ_CASE(G_, 4, 2, 2) \
    TFQ_CASE(G_, 8, 2, 2) TFQ_CASE(G_, 16, 1, 2)
    TFQ_ROWS(32) TFQ_ROWS(64) TFQ_ROWS(128)
#undef TFQ_ROWS
#undef TFQ_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tfq
