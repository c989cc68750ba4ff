// unpack.cuh -- MLX-affine codes -> exact bf16 pairs for the tensor-core A operand.
//
// Codes are stored low code first in a row's little-endian bitstream
// (TensorFold PR #788, commit "every MLX affine width in the row kernel":
// 3- and 5-bit rows hold eight codes in three or five bytes).  The kernel
// reads a "run" of 8 consecutive codes (8*BITS bits) of one row and forms four
// bf16x2 registers holding the code pairs (c_i, c_{i+4}), i = 0..3, each code
// entering as its own exact integer value (PR #788, the 2-bit affine_mm commit:
// codes enter "as itself, with no offset").
//
// Method: a code sitting at bit p of a 16-bit half (p + BITS <= 7) is OR-ed
// into the mantissa of bf16 128.0 (0x4300), giving 128 + c*2^p exactly; one
// bf16x2 add of -128 (p = 0) or one bf16x2 FMA with (2^-p, -128*2^-p) then
// yields c exactly.  8-bit codes do not fit the 7 mantissa bits: the low 7
// bits enter that way and the top bit picks an addend of -128 or 0.
//
// The header compiles as CUDA device code and as plain host C++ (for the CPU
// unit test of the extraction); host builds emulate the three device
// primitives (byte permute, funnel shift, bf16x2 fma).
#pragma once
#include <stdint.h>
#include <string.h>
#if defined(__CUDACC__)
#include <cuda_bf16.h>
#endif

#if defined(__CUDACC__)
#define TF_HD __host__ __device__ __forceinline__
#else
#define TF_HD inline
#endif

namespace tfq {

// Byte permute: result byte i = byte (s >> 4i) & 7 of the 8-byte value {b:a};
// bit 3 of a selector nibble replicates that byte's top bit instead.
TF_HD uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
#if defined(__CUDA_ARCH__)
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
    return d;
#else
    uint64_t v = ((uint64_t)b << 32) | a;
    uint32_t d = 0;
    for (int i = 0; i < 4; ++i) {
        uint32_t sel = (s >> (4 * i)) & 0xF;
        uint32_t byte = (uint32_t)(v >> (8 * (sel & 7))) & 0xFF;
        if (sel & 8) byte = (byte & 0x80) ? 0xFF : 0x00;
        d |= byte << (8 * i);
    }
    return d;
#endif
}

// Low 32 bits of ({hi:lo} >> sh), 0 <= sh < 32.
TF_HD uint32_t funnel(uint32_t lo, uint32_t hi, uint32_t sh) {
#if defined(__CUDA_ARCH__)
    return __funnelshift_r(lo, hi, sh);
#else
    return (uint32_t)((((uint64_t)hi << 32) | lo) >> (sh & 31));
#endif
}

// (a & m) | o  -- one LOP3 on the device.
TF_HD uint32_t mask_or(uint32_t a, uint32_t m, uint32_t o) { return (a & m) | o; }

// Low half from a, high half from b -- one LOP3 on the device.
TF_HD uint32_t halves(uint32_t a, uint32_t b) { return (a & 0x0000FFFFu) | (b & 0xFFFF0000u); }

#if !defined(__CUDA_ARCH__)
inline float bf16_to_float_host(uint16_t h) {
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)h << 16;
    return c.f;
}
inline uint16_t float_to_bf16_host_exact(float f) {
    // Only used on exactly representable values (small integers).
    union { uint32_t u; float f; } c;
    c.f = f;
    return (uint16_t)(c.u >> 16);
}
#endif

// d = a * b + c on two bf16 lanes (round to nearest even); exact in every use here.
TF_HD uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
#if defined(__CUDA_ARCH__)
    __nv_bfloat162 A, B, C;   // bit copies (no type-punned pointers)
    memcpy(&A, &a, 4);
    memcpy(&B, &b, 4);
    memcpy(&C, &c, 4);
    const __nv_bfloat162 r = __hfma2(A, B, C);
    uint32_t d;
    memcpy(&d, &r, 4);
    return d;
#else
    uint32_t d = 0;
    for (int h = 0; h < 2; ++h) {
        float x = bf16_to_float_host((uint16_t)(a >> (16 * h)));
        float y = bf16_to_float_host((uint16_t)(b >> (16 * h)));
        float z = bf16_to_float_host((uint16_t)(c >> (16 * h)));
        d |= (uint32_t)float_to_bf16_host_exact(x * y + z) << (16 * h);
    }
    return d;
#endif
}

// d = a + b on two bf16 lanes (round to nearest even); exact in every use here.
TF_HD uint32_t hadd2(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
#else
    return hfma2(a, 0x3F803F80u, b);
#endif
}

// bf16x2 constants: 128.0 magic, and (scale, addend) per mantissa position p.
constexpr uint32_t MAGIC = 0x43004300u;            // 128.0 | 128.0
constexpr uint32_t NEG128 = 0xC300C300u;           // -128
constexpr uint32_t Q3 = 0x3E003E00u, NEG16 = 0xC180C180u;   // p=3: 1/8, -16
constexpr uint32_t Q4 = 0x3D803D80u, NEG8 = 0xC100C100u;    // p=4: 1/16, -8

// Two forms of a run's pairs: exact codes c (OFF = false), or, for the widths
// whose pairs all sit at p = 0 (4, 5, 6 bits), offset codes 128 + c (OFF =
// true; a product built on them takes 128 * sum(x) back through its bias).
// Code pair at mantissa position p = 0: (128 + c) - 128, or 128 + c itself.
template <bool OFF = false>
TF_HD uint32_t at0(uint32_t u, uint32_t m, uint32_t mg) {
    return OFF ? mask_or(u, m, mg) : hadd2(mask_or(u, m, mg), NEG128);
}
// Code pair at position p > 0: (128 + c*2^p) * 2^-p - 128*2^-p, with q = 2^-p
// passed in a register (QP<BITS>) like `mg`.
TF_HD uint32_t atp(uint32_t u, uint32_t m, uint32_t mg, uint32_t q, uint32_t neg) {
    return hfma2(mask_or(u, m, mg), q, neg);
}

// The 2^-p pair that Unpack<BITS> uses for its p > 0 pairs (0 when it has none).
template <int BITS>
struct QP {
    static constexpr uint32_t value = BITS == 2 ? Q4 : BITS == 3 ? Q3 : 0u;
};

// Run of 8 codes -> pairs p[i*ST] = (c_i | c_{i+4} << 16) as exact bf16 values.
// `w` points at the 32-bit word holding the run's first bit; `ua`/`ub` come
// from lane_args<BITS>(sh) with `sh` that bit's position in the word (they are
// per-lane constants, computed once).  `mg` is MAGIC and `mq` is QP<BITS>,
// both passed in registers so that each mask-and-insert stays one three-input
// logic operation and each FMA takes one immediate.  Reads at most w[0], w[1].
template <int BITS>
struct Unpack;

template <>
struct Unpack<2> {  // 16 bits; sh in {0, 16}
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t sh, uint32_t, uint32_t mg, uint32_t mq, uint32_t *p) {
        static_assert(!OFF, "2-bit codes enter exactly");
        uint32_t v = w[0] >> sh;
        uint32_t u = halves(v, v << 8);              // c0..c3 @0,2,4,6 | c4..c7 @16,18,20,22
        uint32_t u1 = u >> 2;                        // c1, c3 @0,4 | c5, c7 @16,20
        p[0 * ST] = at0(u, 0x00030003u, mg);
        p[1 * ST] = at0(u1, 0x00030003u, mg);
        p[2 * ST] = atp(u, 0x00300030u, mg, mq, NEG8);
        p[3 * ST] = atp(u1, 0x00300030u, mg, mq, NEG8);
    }
};

template <>
struct Unpack<4> {  // 32 bits; sh == 0
    // A 4-bit code fits the 7-bit mantissa only at p <= 3: every pair is moved to p = 0.
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t, uint32_t, uint32_t mg, uint32_t mq, uint32_t *p) {
        uint32_t v = w[0];                           // c0..c3 @0,4,8,12 | c4..c7 @16,20,24,28
        p[0 * ST] = at0<OFF>(v, 0x000F000Fu, mg);
        p[1 * ST] = at0<OFF>(v >> 4, 0x000F000Fu, mg);
        p[2 * ST] = at0<OFF>(v >> 8, 0x000F000Fu, mg);
        p[3 * ST] = at0<OFF>(v >> 12, 0x000F000Fu, mg);
    }
};

template <>
struct Unpack<8> {  // 64 bits; sh == 0
    static TF_HD uint32_t one(uint32_t t, uint32_t mg) {
        // t: code a in byte 0, code b in byte 2.
        uint32_t mant = mask_or(t, 0x007F007Fu, mg);        // 128 + (c & 127)
        uint32_t sgn = prmt(t, 0u, 0xA484u);                // 0xFF00 per half if c >= 128
        uint32_t add = ~sgn & NEG128;                       // -128 if c < 128, else 0
        return hadd2(mant, add);
    }
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t, uint32_t, uint32_t mg, uint32_t mq, uint32_t *p) {
        static_assert(!OFF, "8-bit codes have no offset form (128 + c needs 9 bits)");
        uint32_t lo = w[0], hi = w[1];
        p[0 * ST] = one(prmt(lo, hi, 0x0400u), mg);   // byte i of lo -> 0, byte i of hi -> 2
        p[1 * ST] = one(prmt(lo, hi, 0x0501u), mg);
        p[2 * ST] = one(prmt(lo, hi, 0x0602u), mg);
        p[3 * ST] = one(prmt(lo, hi, 0x0703u), mg);
    }
};

template <>
struct Unpack<3> {  // 24 bits; sh in {0, 8, 16, 24}
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t sh, uint32_t, uint32_t mg, uint32_t mq, uint32_t *p) {
        static_assert(!OFF, "3-bit codes enter exactly");
        uint32_t v = funnel(w[0], w[1], sh);
        uint32_t u = halves(v, v << 4);   // c0..c3 @0,3,6,9 | c4..c7 @16,19,22,25
        uint32_t u2 = u >> 6;             // c2 @0, c3 @3 | c6 @16, c7 @19
        p[0 * ST] = at0(u, 0x00070007u, mg);
        p[1 * ST] = atp(u, 0x00380038u, mg, mq, NEG16);
        p[2 * ST] = at0(u2, 0x00070007u, mg);
        p[3 * ST] = atp(u2, 0x00380038u, mg, mq, NEG16);
    }
};

template <>
struct Unpack<5> {  // 40 bits; sh in {0, 8, 16, 24}
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t sh, uint32_t, uint32_t mg, uint32_t mq, uint32_t *p) {
        uint32_t lo = funnel(w[0], w[1], sh);               // run bits 0..31
        uint32_t hi = w[1] >> sh;                           // run bits 32..39 at 0..7
        uint32_t u = halves(lo, funnel(lo, hi, 4));         // c0,c1,c2 @0,5,10 | c4,c5,c6 @16,21,26
        uint32_t u3 = halves(lo >> 15, funnel(lo, hi, 19)); // c3 @0 | c7 @16
        p[0 * ST] = at0<OFF>(u, 0x001F001Fu, mg);
        p[1 * ST] = at0<OFF>(u >> 5, 0x001F001Fu, mg);
        p[2 * ST] = at0<OFF>(u >> 10, 0x001F001Fu, mg);
        p[3 * ST] = at0<OFF>(u3, 0x001F001Fu, mg);
    }
};

template <>
struct Unpack<6> {  // 48 bits; sh in {0, 16}
    // Run bytes {0,1,3,4} and {1,2,4,5}; raw byte = run byte + sh/8 (sh = 0 or 16).
    template <int ST = 1, bool OFF = false>
    static TF_HD void run(const uint32_t *w, uint32_t s0, uint32_t s2, uint32_t mg, uint32_t mq, uint32_t *p) {
        run_words<ST, OFF>(w[0], w[1], s0, s2, mg, mq, p);
    }
    // The run's two words passed in (a, b) = (w[0], w[1]); the same pairs come
    // from (a, b) = (w[1], w[0]) with both selectors XOR 0x4444 (each selector
    // byte index then names the other operand's byte).
    template <int ST = 1, bool OFF = false>
    static TF_HD void run_words(uint32_t a, uint32_t b, uint32_t s0, uint32_t s2, uint32_t mg, uint32_t mq,
                                uint32_t *p) {
        uint32_t P0 = prmt(a, b, s0);   // c0 @0, c1 @6 | c4 @16, c5 @22
        uint32_t P2 = prmt(a, b, s2);   // c2 @4, c3 @10 | c6 @20, c7 @26
        p[0 * ST] = at0<OFF>(P0, 0x003F003Fu, mg);
        p[1 * ST] = at0<OFF>(P0 >> 6, 0x003F003Fu, mg);
        p[2 * ST] = at0<OFF>(P2 >> 4, 0x003F003Fu, mg);
        p[3 * ST] = at0<OFF>(P2 >> 10, 0x003F003Fu, mg);
    }
};

// Per-lane arguments of Unpack<BITS>::run for a run starting at bit `sh` of a word.
template <int BITS>
TF_HD void lane_args(uint32_t sh, uint32_t &ua, uint32_t &ub) {
    if (BITS == 6) {
        ua = sh ? 0x6532u : 0x4310u;
        ub = sh ? 0x7643u : 0x5421u;
    } else {
        ua = sh;
        ub = 0u;
    }
}

// Position of code (step j, slot e) inside a thread's quarter of a group:
// step j takes pairs 2*(j%2) and 2*(j%2)+1 of run j/2; slot e = 0,1 are the
// low/high code of the first pair (A/B register 0), e = 2,3 of the second.
TF_HD int slot_code(int j, int e) { return 8 * (j >> 1) + 2 * (j & 1) + (e >> 1) + 4 * (e & 1); }

}  // namespace tfq
