// qmm_b2.cu -- kernel instantiations for 2-bit codes (groups 32/64/128, 1-8 and 9-16 rows).
#include "internal.h"
#include "qmm_kernel.cuh"

namespace tfq {
cudaError_t launch_b2(int group, int nt, const QmmParams &P, int grid, int smem, cudaStream_t st) {
    return launch_width<2>(group, nt, P, grid, smem, st);
}
}  // namespace tfq
