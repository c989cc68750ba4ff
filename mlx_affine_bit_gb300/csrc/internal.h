// internal.h -- declarations shared by api.cu and the per-width kernel units.
#pragma once
#include <cuda_runtime.h>

#include "qmm_common.h"

namespace tfq {

// Defined in qmm_b<BITS>.cu, one translation unit per width.
cudaError_t launch_b2(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);
cudaError_t launch_b3(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);
cudaError_t launch_b4(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);
cudaError_t launch_b5(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);
cudaError_t launch_b6(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);
cudaError_t launch_b8(int group, int rb, const QmmParams &P, int grid, int smem, cudaStream_t st,
                      bool pdl);

}  // namespace tfq
