// mx_codec.cuh -- element codecs shared by the producer and the GEMM epilogue:
// the power-of-two block-scale rules (FLOOR, CEIL, NEAREST on exact
// significands) and the round-to-nearest-even, saturating conversions to E4M3
// and E2M1 codes.
#pragma once
#include <cstdint>

#include "mx.h"

namespace mx {

constexpr int kElemE4M3 = 0, kElemE2M1 = 1;

__host__ __device__ constexpr int elem_of(int fmt)
{
    return (fmt == MX_FMT_MXFP8_E4M3 || fmt == MX_FMT_MOSS_FP8) ? kElemE4M3 : kElemE2M1;
}

// ------------------------------------------------------------ scale rules
// b > 0 finite as (1 + mant * 2^-23) * 2^fb, exactly (subnormals normalised).
struct Norm {
    int fb;
    uint32_t mant;
};

__device__ __forceinline__ Norm normalize_pos(float b)
{
    const uint32_t u = __float_as_uint(b);
    const int E = static_cast<int>((u >> 23) & 0xFFu);
    const uint32_t m = u & 0x7FFFFFu;
    if (E != 0)
        return {E - 127, m};
    const int msb = 31 - __clz(m);  // b = m * 2^-149
    return {msb - 149, (m << (23 - msb)) & 0x7FFFFFu};
}

// Power-of-two exponent e of a block with max |y| = b: the block is scaled by
// 2^-e and its E8M0 byte is e + 127.  Q = 448 = 1.75 * 2^8 (E4M3) or
// 6 = 1.5 * 2^2 (E2M1).  All decisions are made on the exact significand.
template <int ELEM>
__device__ __forceinline__ int pow2_exponent(float b, int rule)
{
    constexpr int fq = ELEM == kElemE4M3 ? 8 : 2;              // floor(log2 Q) (= emax)
    constexpr uint32_t mq = ELEM == kElemE4M3 ? 0x600000u : 0x400000u;  // Q significand bits
    const uint32_t u = __float_as_uint(b);
    const int E = static_cast<int>((u >> 23) & 0xFFu);
    if (E != 0 && rule != MX_SCALE_NEAREST) {  // normal b: floor(log2 b) = E - 127
        const int e = E - 127 - fq + ((rule == MX_SCALE_CEIL && (u & 0x7FFFFFu) > mq) ? 1 : 0);
        return max(-127, e);
    }
    if (b == 0.0f)
        return 0;
    const Norm n = normalize_pos(b);
    int e;
    if (rule == MX_SCALE_FLOOR) {
        e = n.fb - fq;  // floor(log2 b) - emax
    } else if (rule == MX_SCALE_CEIL) {
        e = n.fb - fq + (n.mant > mq ? 1 : 0);  // smallest e with b * 2^-e <= Q
    } else {  // NEAREST: round(log2(b / Q)) decided on squared significands
        const uint64_t MB = (1ull << 23) | n.mant, MQ = (1ull << 23) | mq;
        if (n.mant >= mq)
            e = n.fb - fq + ((MB * MB >= 2 * MQ * MQ) ? 1 : 0);
        else
            e = n.fb - fq - 1 + ((2 * MB * MB >= MQ * MQ) ? 1 : 0);
    }
    return max(-127, min(127, e));
}

// 2^-e as an fp32 value, e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float exp2_neg(int e)
{
    const int x = 127 - e;
    return x > 0 ? __uint_as_float(static_cast<uint32_t>(x) << 23) : __uint_as_float(0x00400000u);
}

// ------------------------------------------------------------------ casts
// Round-to-nearest-even, saturating; `lo` lands in the low byte/nibble.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// E2M1 codes of 8 values packed into one word, element 2i in the low nibble
// of byte i (the K-major packing the MMA reads).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&a)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
    return r;
}

__device__ __forceinline__ float dec_e4m3_pos(uint32_t c)
{
    const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
    return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

}  // namespace mx
