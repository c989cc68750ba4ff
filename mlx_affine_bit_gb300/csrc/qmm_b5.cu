// qmm_b5.cu -- kernel instantiations for 5-bit codes (groups 32/64/128, row buckets 1/2/4/8/16, 1 or 2 m-tiles per item, 1 or 2 consumer groups).
#include "internal.h"
#include "qmm_kernel.cuh"

namespace tfq {
cudaError_t launch_b5(int group, int rb, int mt, int cg, const QmmParams &P, int grid, int smem,
                      cudaStream_t st, bool pdl) {
    return launch_width<5>(group, rb, mt, cg, P, grid, smem, st, pdl);
}
}  // namespace tfq
