// Host check of the launch planner (mlx_affine_bit_gb300/csrc/api.cu, make_plan):
// over a grid of shapes, widths, groups and row counts every plan fits the
// hardware and respects the kernel's assumptions.  Host code only: the kernel
// launchers are stubs and nothing touches a GPU.
#include "../mlx_affine_bit_gb300/csrc/api.cu"

#include <cstdio>

namespace tfq {
#define TFQ_STUB(n)                                                                                  \
    cudaError_t launch_b##n(int, int, int, int, const QmmParams &, int, int, cudaStream_t, bool) { \
        return cudaErrorInvalidValue;                                                                \
    }
TFQ_STUB(2) TFQ_STUB(3) TFQ_STUB(4) TFQ_STUB(5) TFQ_STUB(6) TFQ_STUB(8)
#undef TFQ_STUB
}  // namespace tfq

static int bad = 0;
static void check(bool ok, const char *what, int N, int K, int bits, int group, int rows, const Plan &p) {
    if (ok) return;
    if (bad < 20)
        printf("%s: N=%d K=%d %d/%d rows=%d -> mt %d cg %d ctas %d nsl %d sl %d stages %d grid %d smem %d\n", what, N,
               K, bits, group, rows, p.mt, p.cg, p.ctas, p.nsl, p.sl, p.stages, p.grid, p.smem);
    ++bad;
}

int main() {
    const int Ns[] = {1, 16, 17, 48, 300, 1024, 2048, 4096, 6192, 12288, 12304, 65536, 248320};
    const int Ks[] = {32, 256, 1024, 1536, 2048, 4096, 8192, 12288, 32768, 65536};
    const int bitss[] = {2, 3, 4, 5, 6, 8};
    const int groups[] = {32, 64, 128};
    const int nsms[] = {152, 132, 8};
    long long n = 0;
    for (int nsm : nsms)
        for (int N : Ns)
            for (int K : Ks)
                for (int bits : bitss)
                    for (int group : groups) {
                        if (K % group) continue;
                        for (int rows = 1; rows <= 16; ++rows)
                        for (int overlap = 0; overlap < 2; ++overlap) {
                            const bool sb3d = K % CHUNK == 0;
                            const Plan p = make_plan(N, K, bits, group, rows, nsm, sb3d, overlap != 0);
                            ++n;
                            const int budget = (p.ctas == 2 || p.half) ? SMEM_PER_SM / 2 - 1024 : SMEM_MAX;
                            // A half-SM plan leaves room for the next product's CTA: the
                            // 96-register one-m-tile kernel, one CTA per SM, only when asked.
                            check(!p.half || (overlap && p.mt == 1 && p.cg == 1 && p.ctas == 1 && p.grid <= nsm &&
                                              p.rb <= 2),
                                  "half-SM plan", N, K, bits, group, rows, p);
                            check(p.rb == row_bucket(rows), "row bucket", N, K, bits, group, rows, p);
                            check(p.ctas == 1 || p.ctas == 2, "CTAs per SM", N, K, bits, group, rows, p);
                            check(p.mt == 1 || p.mt == 2, "m-tiles", N, K, bits, group, rows, p);
                            check(p.cg == 1 || p.cg == 2, "consumer groups", N, K, bits, group, rows, p);
                            // instantiated kernels: (rb <= 8: mt 1/2, cg 1; mt 2 cg 2), (rb 16: mt 1 cg 1/2, mt 2 cg 1)
                            const bool inst = p.rb <= 8 ? (p.cg == 1 || p.mt == 2) : !(p.mt == 2 && p.cg == 2);
                            check(inst, "no such kernel instance", N, K, bits, group, rows, p);
                            check(p.stages >= 2 && p.stages <= MAX_STAGES, "ring stages", N, K, bits, group, rows, p);
                            check(p.cg == 1 || (p.nsl == 1 && p.stages >= 3), "two groups need one slice and 3 stages",
                                  N, K, bits, group, rows, p);
                            check(p.smem <= budget && p.smem == p.st_off + p.stages * p.stage_bytes, "shared memory",
                                  N, K, bits, group, rows, p);
                            check(p.st_off % 128 == 0 && p.stage_bytes % 128 == 0, "stage alignment", N, K, bits,
                                  group, rows, p);
                            check(p.sl % CHUNK == 0 && p.nsl >= 1 && (long long)p.nsl * p.sl >= K &&
                                      (long long)(p.nsl - 1) * p.sl < K,
                                  "K slices", N, K, bits, group, rows, p);
                            check(p.nmt == (N + TN * p.mt - 1) / (TN * p.mt), "column tiles", N, K, bits, group, rows,
                                  p);
                            // Whole teams (one per K slice) within the CTA slots, or one CTA per
                            // slice when there are more slices than slots (the kernel never
                            // waits on another CTA, so later CTAs simply run later).
                            check(p.grid >= p.nsl && p.grid % p.nsl == 0 &&
                                      p.grid <= std::max<long long>((long long)p.ctas * nsm, p.nsl),
                                  "grid: whole teams within the CTA slots", N, K, bits, group, rows, p);
                            check(p.grid / p.nsl <= p.nmt, "no team larger than its column tiles", N, K, bits, group,
                                  rows, p);
                        }
                    }
    if (bad)
        printf("FAIL %d of %lld plans\n", bad, n);
    else
        printf("PASS %lld plans\n", n);
    return bad ? 1 : 0;
}
