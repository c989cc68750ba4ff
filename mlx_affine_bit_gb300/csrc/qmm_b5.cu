// qmm_b5.cu -- kernel instantiations for 5-bit codes (groups 32/64/128, 1-8 and 9-16 rows).
#include "internal.h"
#include "qmm_kernel.cuh"

namespace tfq {
cudaError_t launch_b5(int group, int nt, const QmmParams &P, int grid, int smem, cudaStream_t st) {
    return launch_width<5>(group, nt, P, grid, smem, st);
}
}  // namespace tfq
