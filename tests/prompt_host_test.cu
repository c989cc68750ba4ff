// Host check of the prompt kernel's static resource plan (prompt_kernel.cuh):
// for every width and group the shared-memory layout fits a CTA and holds one
// CTA per SM (so the 512 tensor-memory columns are never contended), offsets and
// pitches meet the TMA and descriptor alignment rules, the accumulator sets tile
// the tensor memory, and the register cap fits the schedulers.  Host code only.
#include "prompt_kernel.cuh"

#include <cstdio>

using namespace tfq;
using namespace tfq::prompt;

static int bad = 0;
static void check(bool ok, const char *what, int bits, int group) {
    if (ok) return;
    if (bad < 20) printf("%s: %d-bit g%d\n", what, bits, group);
    ++bad;
}

int main() {
    const int bitss[] = {2, 3, 4, 5, 6, 8};
    const int groups[] = {32, 64, 128};
    int n = 0;
    // Registers: warps spread round-robin over four schedulers of 16K registers.
    const int warps = THREADS / 32, per_sched = (warps + 3) / 4;
    check(per_sched * 32 * MAX_REGS <= 16384, "registers per scheduler", 0, 0);
    check(THREADS <= 1024, "threads per CTA", 0, 0);
    check(TMEM_COLS == 512, "tensor-memory allocation", 0, 0);
    check(sizeof(Bars) <= 1024, "barrier header", 0, 0);
    check(EPI_WARPS % 4 == 0 && EPI_ROWS * (EPI_WARPS / 4) == PN, "epilogue rows", 0, 0);
    for (int bits : bitss)
        for (int group : groups) {
            ++n;
            const Layout L = layout(bits, group);
            check(L.smem <= SMEM_MAX, "shared memory of a CTA", bits, group);
            check(L.smem > SMEM_PER_SM / 2, "one CTA per SM", bits, group);
            check(L.stage_bytes % 1024 == 0 && L.sb_off % 1024 == 0 && L.sx_off % 1024 == 0 && L.a_off % 1024 == 0,
                  "1024-byte aligned regions", bits, group);
            check(L.x_off % 16 == 0 && L.w_off % 16 == 0, "16-byte aligned copies", bits, group);
            check((code_pitch(bits) / 16) % 2 == 1, "odd 16-byte code pitch", bits, group);
            check(PM * code_pitch(bits) <= L.x_off, "codes fit their region", bits, group);
            check(sb_pitch(group) % 16 == 0 && PM * sb_pitch(group) <= L.sb_bytes, "scale/bias box", bits, group);
            check(sb_groups(group) * PN * 4 <= SX_BYTES, "group-sum box", bits, group);
            check(CHUNK % sb_k(group) == 0 && sb_k(group) % PSTAGE == 0, "scale/bias unit", bits, group);
            check(PSTAGE % group == 0 && dsets(group) * groups_per_stage(group) == DSLOTS && dsets(group) >= 2,
                  "accumulator sets", bits, group);
            check(L.a_off + ABUF * A_BYTES == L.smem, "layout end", bits, group);
        }
    printf("%d configurations: %s\n", n, bad ? "FAIL" : "PASS");
    return bad ? 1 : 0;
}
