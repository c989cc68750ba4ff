// prompt.cu -- tf_qmm_prompt: the product for many activation rows, weights read
// once per 64-row window, group dot products on the tcgen05 tensor cores
// (kernel in prompt_kernel.cuh).  Host side: checks, a per-(device, stream)
// workspace for the permuted activations, their per-group sums and the chunk
// partials of a split, the x prepass kernel, the work split, tensor maps, and per
// 64-row window one launch (plus the fold of the partials when chunks are split).
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/tfqmm.h"
#include "internal.h"
#include "prompt_kernel.cuh"

using namespace tfq;

namespace {

// x [rows][K] bf16 -> xt, the operand tiles of the prompt kernel: for each
// 64-row window and 128-k stage, [16 k blocks][64 rows][8 values] (one
// contiguous 16 KB block, copied with one bulk copy), every 8 values in the
// codes' pair order (x0, x4, x1, x5, x2, x6, x3, x7) and rows past `rows` zero;
// and sx [K/G][R64] fp32, the sequential sum of each group's x in k order from 0
// (0 past `rows`).  One thread per (group, row).
__global__ void prompt_prep(const uint16_t *x, int rows, int K, int G, int R64, uint16_t *xt, float *sx) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const int ng = K / G;
    if (t >= (long long)ng * R64) return;
    const int g = (int)(t / R64), r = (int)(t - (long long)g * R64);
    const int nst = K / prompt::PSTAGE, win = r / prompt::PN, wr = r % prompt::PN;
    float acc = 0.f;
    const uint16_t *src = x + (long long)r * K + (long long)g * G;
    for (int j = 0; j < G / 8; ++j) {
        const int k = g * G + 8 * j;
        const long long blk = ((long long)win * nst + k / prompt::PSTAGE) * (prompt::PSTAGE / 8) + (k % prompt::PSTAGE) / 8;
        uint4 *dst = reinterpret_cast<uint4 *>(xt + (blk * prompt::PN + wr) * 8);
        if (r >= rows) {
            *dst = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const uint4 v = reinterpret_cast<const uint4 *>(src)[j];
        *dst = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                          prmt(v.y, v.w, 0x7632u));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc += __uint_as_float(w[i] << 16);
            acc += __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    sx[t] = acc;
}

// y rows r0 .. r0 + rows - 1 = the chunk partials part[c][row][N] summed in chunk
// order (C_0 + C_1 + ...), then the output options.  One thread per (row, column).
__global__ void prompt_fold(const float *part, int nchunks, int N, int rows, int r0, void *y, long long y_stride,
                            int out) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= (long long)rows * N) return;
    const int r = (int)(t / N), n = (int)(t - (long long)r * N);
    float v = part[(long long)r * N + n];
    for (int c = 1; c < nchunks; ++c) v += part[((long long)c * prompt::PN + r) * N + n];
    if (out & OUT_RELU2) {
        const float u = fmaxf(v, 0.f);
        v = u * u;
    }
    const long long at = (long long)(r0 + r) * y_stride + n;
    if (out & OUT_BF16)
        static_cast<__nv_bfloat16 *>(y)[at] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(y)[at] = v;
}

struct Ws {
    void *p = nullptr;
    size_t bytes = 0;
};
std::mutex g_pmu;
std::map<std::pair<int, cudaStream_t>, Ws> g_pws;

int workspace(cudaStream_t st, size_t bytes, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_pmu);
    Ws &w = g_pws[{dev, st}];
    if (w.bytes < bytes) {
        if (w.p) {
            // The previous launches on this stream may still read it.
            e = cudaStreamSynchronize(st);
            if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
            cudaFree(w.p);
        }
        w.p = nullptr;
        w.bytes = 0;
        e = cudaMalloc(&w.p, bytes);
        if (e != cudaSuccess) return cuda_error(e, "cudaMalloc(prompt workspace)");
        w.bytes = bytes;
    }
    *out = w.p;
    return TF_OK;
}

template <int BITS, int G, bool MC>
cudaError_t launch_mc(const prompt::Params &P, int grid, int smem, cudaStream_t st) {
    auto k = prompt::prompt_kernel<BITS, G, MC>;
    static unsigned attr_set = 0;   // one bit per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned bit = 1u << (dev & 31);
    if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);
    }
    k<<<grid, prompt::THREADS, smem, st>>>(P);
    return cudaGetLastError();
}

// Chunk sums in registers only for whole-K items of more than one chunk.
template <int BITS, int G>
cudaError_t launch_one(const prompt::Params &P, int grid, int smem, cudaStream_t st) {
    return P.nchunks > 1 && !P.part ? launch_mc<BITS, G, true>(P, grid, smem, st)
                                    : launch_mc<BITS, G, false>(P, grid, smem, st);
}

template <int BITS>
cudaError_t launch_bits(int group, const prompt::Params &P, int grid, int smem, cudaStream_t st) {
    switch (group) {
        case 32: return launch_one<BITS, 32>(P, grid, smem, st);
        case 64: return launch_one<BITS, 64>(P, grid, smem, st);
        case 128: return launch_one<BITS, 128>(P, grid, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prompt(int bits, int group, const prompt::Params &P, int grid, int smem, cudaStream_t st) {
    switch (bits) {
        case 2: return launch_bits<2>(group, P, grid, smem, st);
        case 3: return launch_bits<3>(group, P, grid, smem, st);
        case 4: return launch_bits<4>(group, P, grid, smem, st);
        case 5: return launch_bits<5>(group, P, grid, smem, st);
        case 6: return launch_bits<6>(group, P, grid, smem, st);
        case 8: return launch_bits<8>(group, P, grid, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

extern "C" int tf_qmm_prompt(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *scales,
                             const uint16_t *biases, int N, int bits, int group, void *y, int64_t y_stride,
                             int flags, void *stream) {
    if (flags & ~(TF_OUT_BF16 | TF_EPI_RELU2)) return fail_message(TF_EINVAL_FLAGS, "unknown output flags");
    int rc = check_product(x, rows, K, W, scales, biases, N, bits, group, static_cast<const float *>(y), y_stride);
    if (rc) return rc;
    if (K % CHUNK != 0) return fail_message(TF_EINVAL_SIZE, "the prompt product needs K a multiple of 2048");
    if ((reinterpret_cast<uintptr_t>(scales) | reinterpret_cast<uintptr_t>(biases)) & 15)
        return fail_message(TF_EINVAL_PTR, "the prompt product needs 16-byte aligned scales and biases");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int nsm = 0, *status = nullptr;
    rc = device_info(&nsm, &status);
    if (rc) return rc;
    // Work split: whole-K items over the column tiles, or, when the tiles leave SMs
    // idle, each tile's chunks spread over up to nsm / ntiles items.
    const int ntiles = (N + prompt::PM - 1) / prompt::PM, nchunks = K / CHUNK;
    int nsplit = 1;
    if (ntiles < nsm && nchunks > 1) {
        nsplit = nsm / ntiles < nchunks ? nsm / ntiles : nchunks;
        if (nsplit < 1) nsplit = 1;
    }
    const int cpi = (nchunks + nsplit - 1) / nsplit;
    nsplit = (nchunks + cpi - 1) / cpi;
    // Workspace: x operand tiles [R64 / 64 windows][K / 128 stages][16 KB], the
    // group sums [K/G][R64] fp32, and with a split the chunk partials
    // [nchunks][64][N] fp32 of one window.
    const int R64 = (rows + prompt::PN - 1) / prompt::PN * prompt::PN;
    const size_t xp_bytes = (size_t)R64 * K * 2;
    const size_t sx_bytes = (size_t)(K / group) * R64 * 4;
    const size_t part_bytes = nsplit > 1 ? (size_t)nchunks * prompt::PN * N * 4 : 0;
    void *ws = nullptr;
    rc = workspace(st, xp_bytes + sx_bytes + part_bytes, &ws);
    if (rc) return rc;
    uint16_t *xp = static_cast<uint16_t *>(ws);
    float *sx = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + xp_bytes);
    float *part = nsplit > 1 ? reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + xp_bytes + sx_bytes) : nullptr;
    const long long nthreads = (long long)(K / group) * R64;
    prompt_prep<<<(unsigned)((nthreads + 255) / 256), 256, 0, st>>>(x, rows, K, group, R64, xp, sx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "prompt prepass launch");

    prompt::Params P{};
    const long long rowb = (long long)K * bits / 8;
    const int sw = prompt::PSTAGE * bits / 32;                  // words of one stage row
    rc = tensor_map_3d(&P.tmW, W, 4, sw, N, K / prompt::PSTAGE, rowb, (long long)sw * 4,
                       sw + prompt::code_pad_words(bits), prompt::PM, 1);
    P.xt = xp;
    if (!rc) {
        // One box: a scale/bias unit's groups (<= 32) x the window's 64 rows.
        rc = tensor_map_2d(&P.tmSX, sx, 4, R64, K / group, prompt::PN, prompt::sb_groups(group));
    }
    // Scales and biases as [N][K / unit][groups of a unit]: one box is a unit of
    // 128 columns, each row padded by 8 zero values.
    const int sbg = prompt::sb_groups(group);
    if (!rc)
        rc = tensor_map_3d(&P.tmS, scales, 2, sbg, K / prompt::sb_k(group), N, (long long)sbg * 2,
                           (long long)(K / group) * 2, sbg + 8, 1, prompt::PM);
    if (!rc)
        rc = tensor_map_3d(&P.tmB, biases, 2, sbg, K / prompt::sb_k(group), N, (long long)sbg * 2,
                           (long long)(K / group) * 2, sbg + 8, 1, prompt::PM);
    if (rc) return rc;
    P.y = static_cast<float *>(y);
    P.y_stride = y_stride;
    P.status = status;
    P.K = K;
    P.N = N;
    P.ntiles = ntiles;
    P.nchunks = nchunks;
    P.out = flags;
    P.nsplit = nsplit;
    P.cpi = cpi;
    P.nitems = ntiles * nsplit;
    P.part = part;
    const prompt::Layout L = prompt::layout(bits, group);
    const int grid = P.nitems < nsm ? P.nitems : nsm;
    for (int r0 = 0; r0 < rows; r0 += prompt::PN) {
        P.r0 = r0;
        P.rows = rows - r0 < prompt::PN ? rows - r0 : prompt::PN;
        e = launch_prompt(bits, group, P, grid, L.smem, st);
        if (e != cudaSuccess) return cuda_error(e, "prompt kernel launch");
        if (part) {
            const long long nt = (long long)P.rows * N;
            prompt_fold<<<(unsigned)((nt + 255) / 256), 256, 0, st>>>(part, nchunks, N, P.rows, r0, y, y_stride, flags);
            e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_error(e, "prompt fold launch");
        }
    }
    return TF_OK;
}
