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
// The same for a failed CUDA runtime call.
int cuda_error(cudaError_t e, const char *where);

// Host checks shared by the entry points: the matrix, x / y pointers and rows
// (1..65536), and y_stride >= N; TF_OK or a status with the message recorded.
int check_product(const uint16_t *x, int rows, int K, const uint32_t *W, const uint16_t *s,
                  const uint16_t *b, int N, int bits, int group, const float *y, int64_t y_stride);

// Tiled tensor maps (row-major 2D [rows][cols]; 3D {d0, d1, d2} with byte
// strides s1, s2) of 1-, 2- or 4-byte elements; TF_OK or TF_ECUDA.
int tensor_map_2d(CUtensorMap *m, const void *base, int elem_bytes, long long cols, long long rows,
                  int box_cols, int box_rows);
int tensor_map_3d(CUtensorMap *m, const void *base, int elem_bytes, long long d0, long long d1, long long d2,
                  long long s1, long long s2, int b0, int b1, int b2);

// SM count and device status word of the current device (allocated on first use).
int device_info(int *nsm, int **status);

}  // namespace tfq
