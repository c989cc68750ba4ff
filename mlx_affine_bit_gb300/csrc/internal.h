// internal.h -- declarations shared by api.cu and the per-width kernel units.
#pragma once
#include <cuda_runtime.h>

#include <stddef.h>
#include <stdint.h>

#include "qmm_common.h"

namespace tfq {

// Defined in qmm_b<BITS>.cu, one translation unit per width.
cudaError_t launch_b2(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);
cudaError_t launch_b3(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);
cudaError_t launch_b4(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);
cudaError_t launch_b5(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);
cudaError_t launch_b6(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);
cudaError_t launch_b8(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl);

// Product whose split-K scratch and status word the caller provides (api.cu).
int product_with_scratch(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *s,
                         const uint16_t *b, int N, int bits, int group, float *y, int64_t y_stride,
                         cudaStream_t st, int nsm, float *ws, size_t ws_floats, int *counters,
                         size_t n_counters, int *status);

// Records `msg` as the calling thread's last error and returns `code` (api.cu).
int fail_message(int code, const char *msg);

}  // namespace tfq
