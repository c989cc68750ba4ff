// Host check of the kernel's run unpack (mlx_affine_bit_gb300/csrc/unpack.cuh):
// for every width, every bit phase a run can start at, and random words,
// the four bf16 pairs must hold exactly codes (c_i, c_{i+4}) read bit by bit.
#include <cstdio>
#include <cstdint>
#include <random>
#include "../mlx_affine_bit_gb300/csrc/unpack.cuh"

static uint32_t bit_code(const uint32_t *w, int bits, int start_bit, int i) {
    uint32_t q = 0;
    for (int j = 0; j < bits; ++j) {
        int p = start_bit + i * bits + j;
        q |= ((w[p / 32] >> (p % 32)) & 1u) << j;
    }
    return q;
}

static int bf16_int(uint16_t h) {
    float f = tfq::bf16_to_float_host(h);
    int v = (int)f;
    return ((float)v == f) ? v : -1000000;
}

template <int BITS>
static int check(std::mt19937 &rng, int sh) {
    int bad = 0;
    for (int t = 0; t < 20000; ++t) {
        uint32_t w[4];
        for (auto &x : w) x = rng();
        if (t < 4) for (auto &x : w) x = (t & 1) ? 0xFFFFFFFFu : 0u;
        uint32_t p[4];
        uint32_t ua, ub;
        tfq::lane_args<BITS>((uint32_t)sh, ua, ub);
        tfq::Unpack<BITS>::template run<1>(w, ua, ub, tfq::MAGIC, tfq::QP<BITS>::value, p);
        uint32_t p2[8];
        tfq::Unpack<BITS>::template run<2>(w, ua, ub, tfq::MAGIC, tfq::QP<BITS>::value, p2);
        for (int i = 0; i < 4; ++i) if (p2[2 * i] != p[i]) { printf("stride mismatch\n"); ++bad; }
        if constexpr (BITS >= 4 && BITS <= 6) {   // offset form: every pair holds 128 + c
            uint32_t p4[4];
            tfq::Unpack<BITS>::template run<1, true>(w, ua, ub, tfq::MAGIC, tfq::QP<BITS>::value, p4);
            for (int i = 0; i < 4; ++i) {
                int lo = bf16_int((uint16_t)(p4[i] & 0xFFFF)), hi = bf16_int((uint16_t)(p4[i] >> 16));
                int want_lo = 128 + (int)bit_code(w, BITS, sh, i), want_hi = 128 + (int)bit_code(w, BITS, sh, i + 4);
                if (lo != want_lo || hi != want_hi) {
                    if (bad < 5) printf("OFF BITS=%d sh=%d pair %d: got (%d,%d) want (%d,%d)\n", BITS, sh, i, lo, hi, want_lo, want_hi);
                    ++bad;
                }
            }
        }
        if (BITS == 6) {   // the two words in swapped order with flipped selectors
            uint32_t p3[4];
            tfq::Unpack<6>::template run_words<1>(w[1], w[0], ua ^ 0x4444u, ub ^ 0x4444u, tfq::MAGIC, 0u, p3);
            for (int i = 0; i < 4; ++i) if (p3[i] != p[i]) { printf("swapped words mismatch\n"); ++bad; }
        }
        for (int i = 0; i < 4; ++i) {
            int lo = bf16_int((uint16_t)(p[i] & 0xFFFF)), hi = bf16_int((uint16_t)(p[i] >> 16));
            int want_lo = (int)bit_code(w, BITS, sh, i), want_hi = (int)bit_code(w, BITS, sh, i + 4);
            if (lo != want_lo || hi != want_hi) {
                if (bad < 5) printf("BITS=%d sh=%d pair %d: got (%d,%d) want (%d,%d)\n", BITS, sh, i, lo, hi, want_lo, want_hi);
                ++bad;
            }
        }
    }
    return bad;
}

int main() {
    std::mt19937 rng(12345);
    int bad = 0;
    bad += check<2>(rng, 0) + check<2>(rng, 16);
    bad += check<4>(rng, 0);
    bad += check<8>(rng, 0);
    for (int sh = 0; sh < 32; sh += 8) bad += check<3>(rng, sh) + check<5>(rng, sh);
    bad += check<6>(rng, 0) + check<6>(rng, 16);
    // slot map: each step/slot covers the 16 codes of two runs exactly once
    int seen[16] = {0};
    for (int j = 0; j < 4; ++j) for (int e = 0; e < 4; ++e) seen[tfq::slot_code(j, e)]++;
    for (int i = 0; i < 16; ++i) if (seen[i] != 1) { printf("slot map hole at %d\n", i); ++bad; }
    printf(bad ? "FAIL %d\n" : "PASS\n", bad);
    return bad ? 1 : 0;
}
