// quantize.cu -- the fused quantize producer of the block-scaled linear layer.
//
//   amax_kernel        max |x| over a bf16 tensor (level-1 scale input of MOSS
//                      and NVFP4; "MOSS: 用微缩放和自动缩放实现无损 FP8 训练",
//                      section 两级缩放实现).
//   quant_row_kernel   bf16 [R, C] -> K-major operand [R, C]: each thread owns
//                      8 consecutive elements (one 16-byte load); the 2 or 4
//                      threads of a scale block combine their maxima with warp
//                      shuffles; codes leave as one coalesced 8- or 4-byte store.
//   quant_col_kernel   bf16 [R, C] -> transposed operand [C, R] (quantized along
//                      R): a CTA stages SEG x 256 of the input in shared memory
//                      with 16-byte loads, then each thread encodes one column's
//                      SEG values into 32 bytes of output codes.
//   quant_tile_kernel  TMA-pipelined 64-row tiles; rowwise, colwise or both
//                      operands from one read of x (the dual-direction pass);
//                      the automatic producer in both directions.  The row and
//                      col kernels serve NVFP4 with the Hadamard transform and
//                      the `direct` test choice.
// All write the block scales straight into the tensor core's scale-factor
// layout ("格式感知融合:让FP4预训练提速两倍的工程实践", section
// 格式感知融合的设计思路: the producer writes the consumer's layout), and all
// can apply the fixed-sign 32-point Hadamard transform (the tile producer for
// the MX formats) and Philox stochastic rounding (same page, section
// 两个关键的数值技巧).
//
// Bit-exactness: every step is an exactly specified fp32 operation (products
// with __fmul_rn, correctly rounded quotients, adds in a fixed butterfly order) or
// an integer decision, so the codes and scale bytes are a pure function of the
// input, independent of launch shape.
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>

#include "mx_codec.cuh"
#include "mx_internal.cuh"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;

// the source buffers of all but the most recent committed bulk store group may be reused
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Named barrier that also ORs a predicate over its nthreads threads.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& w, float* v)
{
    v[0] = bf16_lo(w.x), v[1] = bf16_hi(w.x), v[2] = bf16_lo(w.y), v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z), v[5] = bf16_hi(w.z), v[6] = bf16_lo(w.w), v[7] = bf16_hi(w.w);
}

// Stochastic rounding of 8 values onto the E2M1 grid {0, .5, 1, 1.5, 2, 3,
// 4, 6}: a value rounds up iff u16 < p * 2^16, p = (|s| - lo) / (hi - lo),
// saturating at 6; the codes come packed as cvt_e2m1x8 packs them.  lo is
// |s| cut down to the grid: the spacing above it is 2^(E - 1) (E the exponent
// of |s|, at least 0), so p * 2^16 = (|s| - lo) * 2^(17 - E) exactly.
//
// The grid helpers below keep the work on the FMA pipe where they can: the
// power of two 2^(17 - E) (2^(19 - E') for E4M3) comes from one integer
// subtraction and a minimum on the exponent field, and lo from adding
// c = spacing * 2^23 in round-toward-zero (the sum's unit in the last place is
// the spacing, so the sum is c + lo exactly) and subtracting c again.  For
// either format c's bit pattern is 0x92800000 minus that of the power of two.
// lo carries the sign of s into the hardware conversion; the round-up bit is
// added to the code's magnitude (at most 6 for E2M1, 0x7E - 1 for E4M3 when a
// round-up can happen, so nothing carries into the sign).  No branches: the
// whole warp takes one path whatever the values.
__device__ __forceinline__ float sr_floor(float a, uint32_t mult_bits)
{
    const float c = __uint_as_float(0x92800000u - mult_bits);
    return __fsub_rn(__fadd_rz(a, c), c);
}

__device__ __forceinline__ float with_sign_of(float l, float s)
{
    return __uint_as_float(__float_as_uint(l) | (__float_as_uint(s) & 0x80000000u));
}

__device__ __forceinline__ uint32_t e2m1_sr8(const float* s, const uint32_t (&u)[8])
{
    float lo[8];
    uint32_t ups = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = fminf(fabsf(s[i]), 6.0f);
        const uint32_t mb = min(0x87800000u - (__float_as_uint(a) & 0x7F800000u), 0x48000000u);  // 2^(17 - E)
        const float l = sr_floor(a, mb);
        const float t = __fmul_rn(__fsub_rn(a, l), __uint_as_float(mb));
        lo[i] = with_sign_of(l, s[i]);
        ups += static_cast<float>(u[i]) < t ? (1u << (4 * i)) : 0u;
    }
    return cvt_e2m1x8(lo) + ups;
}

// Stochastic rounding of 8 values onto the E4M3 grid with the same rule (up
// iff u16 < p * 2^16, p = (|s| - lo) / (hi - lo)), saturating at 448; codes
// packed one per byte, element 0 in the low byte of out[0].  The spacing
// above lo is 2^(E' - 3), E' the exponent of |s| but at least -6 (the
// subnormal range's spacing 2^-9), so p * 2^16 = (|s| - lo) * 2^(19 - E')
// exactly.  lo and the round-up bit as for E2M1 above.
__device__ __forceinline__ void e4m3_sr8(const float* s, const uint32_t (&u)[8], uint32_t* out)
{
    float lo[8];
    uint32_t ups[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = fminf(fabsf(s[i]), 448.0f);
        const uint32_t mb = min(0x88800000u - (__float_as_uint(a) & 0x7F800000u), 0x4C000000u);  // 2^(19 - E')
        const float l = sr_floor(a, mb);
        const float t = __fmul_rn(__fsub_rn(a, l), __uint_as_float(mb));
        lo[i] = with_sign_of(l, s[i]);
        ups[i >> 2] += static_cast<float>(u[i]) < t ? (1u << (8 * (i & 3))) : 0u;
    }
    out[0] = (cvt_e4m3x2(lo[0], lo[1]) | (cvt_e4m3x2(lo[2], lo[3]) << 16)) + ups[0];
    out[1] = (cvt_e4m3x2(lo[4], lo[5]) | (cvt_e4m3x2(lo[6], lo[7]) << 16)) + ups[1];
}

// ------------------------------------------------------------- Philox4x32-10
// Salmon et al., SC'11: two 32x32 -> 64 multiplies per round, ten rounds, the
// key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// The 8 random 16-bit draws of the 8 elements with linear index L8*8 .. L8*8+7.
__device__ __forceinline__ void sr_bits8(uint64_t seed, uint32_t sid, uint64_t L8, uint32_t (&u)[8])
{
    const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(L8), static_cast<uint32_t>(L8 >> 32), sid, 0u),
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    u[0] = w.x & 0xFFFFu; u[1] = w.x >> 16;
    u[2] = w.y & 0xFFFFu; u[3] = w.y >> 16;
    u[4] = w.z & 0xFFFFu; u[5] = w.z >> 16;
    u[6] = w.w & 0xFFFFu; u[7] = w.w >> 16;
}

// In-register butterflies of the fixed-sign Sylvester transform over N values
// (stages h = 1, 2, 4, ... < N): (x_j, x_j+h) <- (x_j + x_j+h, x_j - x_j+h).
template <int N>
__device__ __forceinline__ void fwht_local(float* v)
{
#pragma unroll
    for (int h = 1; h < N; h <<= 1)
#pragma unroll
        for (int j = 0; j < N; ++j)
            if ((j & h) == 0) {
                const float a = v[j], b = v[j + h];
                v[j] = __fadd_rn(a, b);
                v[j + h] = __fsub_rn(a, b);
            }
}

// Butterfly stage across lanes: partner lane = lane ^ mask; the lower lane
// keeps x_lo + x_hi, the upper one x_lo - x_hi.
__device__ __forceinline__ void fwht_lanes(float (&v)[8], int mask, bool upper)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float p = __shfl_xor_sync(0xFFFFFFFFu, v[i], mask);
        v[i] = upper ? __fsub_rn(p, v[i]) : __fadd_rn(v[i], p);
    }
}

// Quotient v / d, rounded to nearest as an IEEE division would, for a
// divisor d that many elements share.  From the correctly rounded reciprocal
// r = RN(1/d) (one __frcp_rn per block), q0 = RN(v r) is within 1.5 ulp of v/d;
// one residual correction q1 = RN(q0 + (v - q0 d) r) (the residual is exact
// with one FMA) brings it within 1 ulp, and a second one rounds correctly by
// Markstein's theorem (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  The
// theorem assumes no underflow or overflow, so the fast path is taken only
// when the divisor (r == 0 marks one outside [2^-100, 2^100]), the quotient
// and the numerator are all at least 2^-100 in magnitude, which keeps both
// residuals exactly representable; everything else takes the IEEE division.
__device__ __forceinline__ float recip_for_div(float d)
{
    return (d >= 0x1p-100f && d <= 0x1p100f) ? __frcp_rn(d) : 0.0f;
}

// The rare IEEE fallback of div_shared, out of line so that the many inlined
// copies of the fast path stay small.
__device__ __noinline__ float div_ieee(float v, float d) { return __fdiv_rn(v, d); }

__device__ __forceinline__ float div_shared(float v, float d, float r)
{
    const float q0 = __fmul_rn(v, r);
    const float a = fabsf(q0);
    if (a >= 0x1p-100f && a <= 0x1p100f && fabsf(v) >= 0x1p-100f) {
        const float q1 = __fmaf_rn(__fmaf_rn(-q0, d, v), r, q0);
        return __fmaf_rn(__fmaf_rn(-q1, d, v), r, q1);
    }
    return (v == 0.0f && r != 0.0f) ? q0 : div_ieee(v, d);
}

__device__ __forceinline__ float tensor_scale_of(int fmt, const float* amax)
{
    if (fmt == MX_FMT_MOSS_FP8 || fmt == MX_FMT_NVFP4) {
        const float am = *amax;
        return am == 0.0f ? 1.0f : __fdiv_rn(am, fmt == MX_FMT_MOSS_FP8 ? 448.0f : 2688.0f);
    }
    return 1.0f;
}

// ---------------------------------------------------------- block encoding
// Quotients by a tensor-dependent divisor D without division.  With the
// double-word reciprocal hi = RN(1/D), lo = RN((1 - D hi) / D) (1 - D hi is
// exact in fp32 for hi = RN(1/D)), q = fma(x, hi, x * lo) lies within 2^-46
// (relative) of x / D before its one rounding, so q = RN(x / D) unless x / D
// is that close to an fp32 rounding midpoint.  The quotient is only used
// through step functions (E2M1 or E4M3 codes, power-of-two scale rules)
// whose boundaries are mu * 2^k with significands mu = 1 + j / 16, and a
// rounding difference can move a step only where q or RN(x / D) is such a
// boundary, i.e. where x / D is next to (mu +- 2^-24) * 2^k (mu - 2^-25 below
// a power of two).  For bf16 x that requires a bf16 value within 2^-46 of
// W = (mu +- 2^-24) * D in some binade; the certificate checks every W once,
// with a 2^-44 margin (bf16 values are 2^-8 apart, so a random D fails with
// probability near 2^-30).  D must lie in
// [2^-100, 2^100], so that x near a boundary is a normal bf16 value and x * lo
// does not underflow there; callers guard the overflow side per block.  The
// argument needs x on the bf16 lattice: fp32 values (Hadamard-transformed
// blocks) could sit within 2^-46 of a midpoint, so those divide exactly.
struct Recip2 {
    float hi, lo;
};

__device__ __forceinline__ Recip2 recip2(float D)
{
    Recip2 r;
    r.hi = __frcp_rn(D);
    r.lo = __fmul_rn(__fmaf_rn(-D, r.hi, 1.0f), r.hi);
    return r;
}

__device__ __forceinline__ float quot2(float x, const Recip2& r) { return __fmaf_rn(x, r.hi, __fmul_rn(x, r.lo)); }

// Whether pattern mu = 1 + j / 2^NFRAC is clear of bf16 values on both
// sides.  W = mu * D + s * D (s = +-2^-24, or -2^-25 below a power of two) is
// held exactly as P_hi + P_lo + s * D (two-product of mu * D with an FMA);
// when a bf16 value b is close, P_hi - b is exact and small, so the three
// small terms sum to the distance with an error near 2^-48 W, well inside the
// factor-4 margin.
template <int NFRAC>
__device__ __forceinline__ bool quot2_pattern_clear(float D, int j)
{
    const float mu = 1.0f + static_cast<float>(j) / static_cast<float>(1 << NFRAC);
    const float p_hi = __fmul_rn(mu, D);
    const float p_lo = __fmaf_rn(mu, D, -p_hi);
    const float b = __bfloat162float(__float2bfloat16_rn(p_hi));
    const float base = __fadd_rn(__fsub_rn(p_hi, b), p_lo);
    const float up = __fadd_rn(base, __fmul_rn(D, 0x1p-24f));
    const float down = __fsub_rn(base, __fmul_rn(D, j == 0 ? 0x1p-25f : 0x1p-24f));
    const float tol = __fmul_rn(p_hi, 0x1p-44f);
    return fabsf(up) > tol && fabsf(down) > tol;
}

__device__ __forceinline__ bool in_quot2_range(float D) { return D >= 0x1p-100f && D <= 0x1p100f; }

// E2M1 element codes (boundaries 0.25 .. 5: significands 1, 1.25, 1.5, 1.75).
__device__ __forceinline__ bool quot2_certified_e2m1(float d)
{
    if (!in_quot2_range(d))
        return false;
    bool ok = true;
    for (int j = 0; j < 4; ++j)
        ok &= quot2_pattern_clear<2>(d, j);
    return ok;
}

// E4M3 codes and power-of-two rule edges (significands 1 + j / 16); the
// sixteen patterns are split over the lanes of the calling warp.
__device__ __forceinline__ bool quot2_certified_e4m3_warp(float D)
{
    const int lane = threadIdx.x & 31;
    const bool ok = lane >= 16 || quot2_pattern_clear<4>(D, lane);
    return __all_sync(0xFFFFFFFFu, ok) && in_quot2_range(D);
}

// Tensor-level constants of one producer pass.
//  NVFP4: a block's divisor d = fl32(dec(s_b) * s_t) takes one of 128 values
//  (one per UE4M3 scale byte s_b), so each CTA tabulates {d, RN(1/d)} for the
//  exact division and the certified double-word reciprocal of d ({0, 0} for
//  d == 0: sign-kept zero codes; hi < 0 when not certified: those blocks
//  divide).  The block scale divides the block max by fl32(6 s_t).
//  MOSS: the level-1 division x / s_t (FLOOR and CEIL rules).
struct ScaleCtx {
    float ts;              // tensor scale (1 for the MX formats)
    float rts;             // recip_for_div(ts) (MOSS exact path)
    float nv_denom;        // fl32(6 * ts) (NVFP4)
    float rden;            // recip_for_div(nv_denom)
    Recip2 den2;           // double-word reciprocal of nv_denom
    Recip2 ts2;            // double-word reciprocal of ts
    bool den2_ok;          // NVFP4 block scale certified
    bool ts2_ok;           // MOSS level-1 scaling certified
    const float2* nv_tab;  // [128] {d, recip_for_div(d)} per scale byte (NVFP4)
    const float2* nv_q;    // [128] certified {hi, lo} of 1/d per scale byte (NVFP4)
};

// Every thread calls this (whole warps); the caller synchronises before the
// tables are read.
template <int FMT>
__device__ __forceinline__ ScaleCtx make_scale_ctx(const float* amax, float2* tab_smem, float2* q_smem, int rule)
{
    ScaleCtx c;
    c.ts = tensor_scale_of(FMT, amax);
    c.rts = recip_for_div(c.ts);
    c.nv_denom = __fmul_rn(6.0f, c.ts);
    c.rden = recip_for_div(c.nv_denom);
    c.nv_tab = tab_smem;
    c.nv_q = q_smem;
    c.den2 = recip2(in_quot2_range(c.nv_denom) ? c.nv_denom : 1.0f);
    c.ts2 = recip2(in_quot2_range(c.ts) ? c.ts : 1.0f);
    c.den2_ok = false;
    c.ts2_ok = false;
    if constexpr (FMT == MX_FMT_NVFP4) {
        c.den2_ok = quot2_certified_e4m3_warp(c.nv_denom);
        for (int sb = threadIdx.x; sb < 128; sb += blockDim.x) {
            const float d = __fmul_rn(dec_e4m3_pos(static_cast<uint32_t>(sb)), c.ts);
            tab_smem[sb] = make_float2(d, recip_for_div(d));
            const Recip2 r = recip2(in_quot2_range(d) ? d : 1.0f);
            q_smem[sb] = d == 0.0f ? make_float2(0.0f, 0.0f)
                       : quot2_certified_e2m1(d) ? make_float2(r.hi, r.lo) : make_float2(-1.0f, 0.0f);
        }
    }
    if constexpr (FMT == MX_FMT_MOSS_FP8)
        c.ts2_ok = (rule == MX_SCALE_FLOOR || rule == MX_SCALE_CEIL) && quot2_certified_e4m3_warp(c.ts);
    return c;
}

// MOSS level-1 scaling of one block: v <- fl32(v / s_t) for bf16 inputs v
// whose max |v| is xmax; returns max |fl32(v / s_t)| (a correctly rounded
// division by a positive constant is monotone, so it is the scaled xmax).  The
// product path needs the certificate and a scaled block clear of the fp32
// subnormal and overflow ranges.
template <int N>
__device__ __forceinline__ float moss_block(float (&v)[N], float xmax, const ScaleCtx& sc)
{
    const float ymax = quot2(xmax, sc.ts2);
    if (sc.ts2_ok && (xmax == 0.0f || (ymax >= 0x1p-100f && ymax < 0x1p100f))) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = quot2(v[i], sc.ts2);
        return ymax;
    }
#pragma unroll
    for (int i = 0; i < N; ++i)
        v[i] = div_shared(v[i], sc.ts, sc.rts);
    return div_shared(xmax, sc.ts, sc.rts);
}

// NVFP4 block scale byte: UE4M3_RNE(fl32(bmax / fl32(6 s_t))).  A quotient of
// 2^100 or more saturates either way (clamping also absorbs an overflowed
// product).  The certified product holds for bmax a bf16 value; the maxima of
// Hadamard-transformed blocks (BF16_IN false) are fp32 and divide exactly.
template <bool BF16_IN = true>
__device__ __forceinline__ uint32_t nvfp4_scale_byte(float bmax, const ScaleCtx& sc)
{
    const float qb = (BF16_IN && sc.den2_ok) ? fminf(quot2(bmax, sc.den2), 0x1p100f)
                                             : div_shared(bmax, sc.nv_denom, sc.rden);
    return cvt_e4m3x2(qb, 0.0f) & 0x7Fu;
}

// Encodes one scale block held as N consecutive values in registers (the
// block's max |v| is `bmax`).  Produces the scale byte and N codes packed
// little-endian into `out` (E4M3: N bytes; E2M1: N/2 bytes).  `L8` is the
// Philox counter of the first 8 elements (used only for SR).  The certified
// NVFP4 products hold for bf16 values; BF16_IN false (Hadamard-transformed
// fp32 values) takes the exact division.
template <int FMT, bool SR, int N, bool BF16_IN = true>
__device__ __forceinline__ uint32_t encode_block(float (&v)[N], float bmax, const ScaleCtx& sc, int rule,
                                                 uint64_t seed, uint32_t sid, uint64_t L8, uint32_t* out)
{
    constexpr int ELEM = elem_of(FMT);
    uint32_t sfbyte;
    bool zero = false;
    if constexpr (FMT == MX_FMT_NVFP4) {
        const uint32_t sb = nvfp4_scale_byte<BF16_IN>(bmax, sc);
        const float2 drd = sc.nv_tab[sb];  // {fl32(dec(sb) * ts), RN(1/d)}
        const float2 q2 = sc.nv_q[sb];     // certified {hi, lo}, or hi < 0
        sfbyte = sb;
        if (drd.x == 0.0f) {
            zero = true;
        } else if (!SR && BF16_IN && q2.x > 0.0f && __fmul_rn(bmax, q2.x) < 0x1p100f) {  // certified
            const Recip2 r{q2.x, q2.y};
#pragma unroll
            for (int i = 0; i < N; ++i)
                v[i] = quot2(v[i], r);
        } else {  // exact quotient (SR always needs it)
#pragma unroll
            for (int i = 0; i < N; ++i)
                v[i] = div_shared(v[i], drd.x, drd.y);
        }
    } else {
        const int e = pow2_exponent<ELEM>(bmax, rule);
        const float s2 = exp2_neg(e);
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = __fmul_rn(v[i], s2);
        sfbyte = static_cast<uint32_t>(e + 127);
    }
    if constexpr (ELEM == kElemE4M3) {
        if constexpr (SR) {
#pragma unroll
            for (int g = 0; g < N / 8; ++g) {
                uint32_t u[8];
                sr_bits8(seed, sid, L8 + g, u);
                e4m3_sr8(&v[8 * g], u, &out[2 * g]);
            }
        } else {
#pragma unroll
            for (int w = 0; w < N / 4; ++w)
                out[w] = cvt_e4m3x2(v[4 * w], v[4 * w + 1]) | (cvt_e4m3x2(v[4 * w + 2], v[4 * w + 3]) << 16);
        }
    } else {
#pragma unroll
        for (int w = 0; w < N / 8; ++w) {
            uint32_t word = 0;
            if (zero) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    word |= ((__float_as_uint(v[8 * w + i]) >> 31) << 3) << (4 * i);
            } else if constexpr (SR) {
                uint32_t u[8];
                sr_bits8(seed, sid, L8 + w, u);
                word = e2m1_sr8(&v[8 * w], u);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    word |= cvt_e2m1x2(v[8 * w + 2 * i], v[8 * w + 2 * i + 1]) << (8 * i);
            }
            out[w] = word;
        }
    }
    return sfbyte;
}

// ---------------------------------------------------------------- kernels
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x, int64_t R,
                                                        int64_t C, int64_t ld, unsigned* __restrict__ out)
{
    const int64_t cpr = C / 8;
    uint32_t m2 = 0;  // two packed |bf16| maxima
    auto fold = [&](const uint4& w) {
        m2 = __vmaxu2(m2, w.x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w.y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w.z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w.w & 0x7FFF7FFFu);
    };
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (ld == C) {  // contiguous: one flat stream of 16-byte chunks, two loads in flight
        const uint4* p = reinterpret_cast<const uint4*>(x);
        const int64_t total = R * cpr;
        int64_t t = tid;
        for (; t + nthr < total; t += 2 * nthr) {
            const uint4 a = __ldg(p + t), b = __ldg(p + t + nthr);
            fold(a);
            fold(b);
        }
        if (t < total)
            fold(__ldg(p + t));
    } else {
        for (int64_t r = blockIdx.y; r < R; r += gridDim.y)
            for (int64_t c8 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c8 < cpr;
                 c8 += static_cast<int64_t>(gridDim.x) * blockDim.x)
                fold(__ldg(reinterpret_cast<const uint4*>(x + r * ld + c8 * 8)));
    }
    unsigned m = max(m2 & 0xFFFFu, m2 >> 16) << 16;  // bf16 bits -> fp32 bits of |x|
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ unsigned wmax[kThreads / 32];
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < kThreads / 32 ? wmax[threadIdx.x] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (threadIdx.x == 0)
            atomicMax(out, m);
    }
}

// Rowwise producer.  One work item = one row and 256*U consecutive 8-element
// chunks of it; a thread handles U chunks (U loads in flight).
// Tensor amax of the Hadamard-transformed operand (NVFP4 with the transform):
// max |H32 y| over every 32 consecutive operand elements along K, each group
// transformed with the same butterflies, in the same order, as the producers
// use, so the amax is the exact maximum of the values they encode.
//   ROWWISE (K along the columns of x, C % 32 == 0): a warp takes 32
//   consecutive 8-element chunks; four lanes hold one 32-element group and
//   transform it with in-thread stages h = 1, 2, 4 and lane stages h = 8, 16.
//   COLWISE (K along the rows, R % 32 == 0): a lane holds two adjacent columns
//   over 32 rows (a warp reads 128 contiguous bytes per row) and transforms
//   each column in registers.
__global__ void __launch_bounds__(kThreads) had_amax_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                            int64_t ld, int dir, unsigned* __restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    float m = 0.0f;
    if (dir == MX_ROWWISE) {
        const int64_t cpr = C / 8, total = R * cpr;  // 8-element chunks, 4 per group (cpr % 4 == 0)
        for (int64_t t0 = warp * 32; t0 < total; t0 += nwarps * 32) {  // warp-uniform bound
            const int64_t t = t0 + lane;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (t < total) {
                const int64_t r = t / cpr, c8 = t - r * cpr;
                w = __ldg(reinterpret_cast<const uint4*>(x + r * ld + c8 * 8));
            }
            float v[8];
            unpack8(w, v);
            fwht_local<8>(v);
            fwht_lanes(v, 1, (lane & 1) != 0);
            fwht_lanes(v, 2, (lane & 2) != 0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m = fmaxf(m, fabsf(v[i]));
        }
    } else {
        const int64_t cpairs = (C + 1) / 2, rgroups = R / 32;
        const int64_t ctasks = (cpairs + 31) / 32, tasks = rgroups * ctasks;
        for (int64_t task = warp; task < tasks; task += nwarps) {
            const int64_t rg = task / ctasks, cp = (task - rg * ctasks) * 32 + lane;
            const int64_t c = 2 * cp;
            if (c < C) {
                float v0[32], v1[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint16_t* src = x + (rg * 32 + i) * ld + c;
                    const uint32_t w = c + 1 < C ? *reinterpret_cast<const uint32_t*>(src) : static_cast<uint32_t>(*src);
                    v0[i] = bf16_lo(w);
                    v1[i] = bf16_hi(w);
                }
                fwht_local<32>(v0);
                fwht_local<32>(v1);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    m = fmaxf(m, fmaxf(fabsf(v0[i]), fabsf(v1[i])));
            }
        }
    }
    unsigned mu = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));  // m >= 0: bits order like values
    __shared__ unsigned wmax[kThreads / 32];
    if (lane == 0)
        wmax[threadIdx.x >> 5] = mu;
    __syncthreads();
    if (threadIdx.x < 32) {
        mu = threadIdx.x < kThreads / 32 ? wmax[threadIdx.x] : 0u;
        mu = __reduce_max_sync(0xFFFFFFFFu, mu);
        if (threadIdx.x == 0)
            atomicMax(out, mu);
    }
}

template <int FMT, bool SR, bool HAD>
__global__ void __launch_bounds__(kThreads) quant_row_kernel(QuantArgs a)
{
    constexpr int BLOCK = fmt_block(FMT);
    constexpr int LPB = BLOCK / 8;  // lanes per scale block
    constexpr int U = 4;
    constexpr bool FP4 = elem_of(FMT) == kElemE2M1;
    const int lane = threadIdx.x & 31;
    const int64_t C = a.C, cpr = C / 8;
    const int64_t kgroups = sf_kgroups(C / BLOCK);
    const int64_t items_per_row = (cpr + kThreads * U - 1) / (kThreads * U);
    const int64_t items = a.R * items_per_row;
    __shared__ float2 nv_tab[128];
    __shared__ float2 nv_q[128];
    const ScaleCtx sc = make_scale_ctx<FMT>(a.amax, nv_tab, nv_q, a.rule);
    const float ts = sc.ts;
    if (fmt_has_tensor_scale(FMT) && blockIdx.x == 0 && threadIdx.x == 0)
        *a.tensor_scale = ts;
    __syncthreads();

    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t r = item / items_per_row;
        const int64_t cbase = (item - r * items_per_row) * (kThreads * U) + threadIdx.x;
        const uint16_t* xr = a.x + r * a.ld;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c8 = cbase + u * kThreads;
            w[u] = c8 < cpr ? __ldg(reinterpret_cast<const uint4*>(xr + c8 * 8)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c8 = cbase + u * kThreads;
            // Whole scale blocks are either all in range or all out of range
            // (C % BLOCK == 0), so the shuffles below stay within valid groups.
            if (cbase - threadIdx.x + u * kThreads >= cpr)
                break;  // warp-uniform: the whole CTA slice is past the row end
            float v[8] = {bf16_lo(w[u].x), bf16_hi(w[u].x), bf16_lo(w[u].y), bf16_hi(w[u].y),
                          bf16_lo(w[u].z), bf16_hi(w[u].z), bf16_lo(w[u].w), bf16_hi(w[u].w)};
            if constexpr (HAD) {
                fwht_local<8>(v);
                fwht_lanes(v, 1, (lane & 1) != 0);
                fwht_lanes(v, 2, (lane & 2) != 0);
            }
            float bmax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                bmax = fmaxf(bmax, fabsf(v[i]));
#pragma unroll
            for (int m = 1; m < LPB; m <<= 1)
                bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, m));
            if constexpr (FMT == MX_FMT_MOSS_FP8)
                bmax = moss_block(v, bmax, sc);
            if (c8 < cpr) {
                uint32_t out[2];
                const uint32_t sfb = encode_block<FMT, SR, 8, !HAD>(v, bmax, sc, a.rule, a.seed,
                                                                    a.stream_id, r * cpr + c8, out);
                if constexpr (FP4)
                    *reinterpret_cast<uint32_t*>(a.codes + r * (C / 2) + c8 * 4) = out[0];
                else
                    *reinterpret_cast<uint2*>(a.codes + r * C + c8 * 8) = make_uint2(out[0], out[1]);
                if ((lane & (LPB - 1)) == 0)
                    a.sf[sf_offset(r, (c8 * 8) / BLOCK, kgroups)] = static_cast<uint8_t>(sfb);
            }
        }
    }
}

// Colwise producer: operand row c (= input column c), K = R.  A CTA stages a
// tile of SEG input rows x 256 input columns in shared memory with coalesced
// 16-byte loads; then each thread encodes one column's SEG values (32 bytes of
// output codes) and writes them as two 16-byte stores.
template <int FMT, bool SR, bool HAD>
__global__ void __launch_bounds__(kThreads) quant_col_kernel(QuantArgs a)
{
    constexpr int BLOCK = fmt_block(FMT);
    constexpr bool FP4 = elem_of(FMT) == kElemE2M1;
    constexpr int SEG = FP4 ? 64 : 32;   // K elements per thread
    constexpr int TC = kThreads;         // input columns per tile
    constexpr int CPR = TC / 8;          // 16-byte chunks per tile row
    __shared__ __align__(16) uint16_t tile[SEG][TC];
    __shared__ float2 nv_tab[128];
    __shared__ float2 nv_q[128];
    const int64_t R = a.R, C = a.C;
    const ScaleCtx sc = make_scale_ctx<FMT>(a.amax, nv_tab, nv_q, a.rule);
    const float ts = sc.ts;
    if (fmt_has_tensor_scale(FMT) && blockIdx.x == 0 && threadIdx.x == 0)
        *a.tensor_scale = ts;
    const int64_t kgroups = sf_kgroups(R / BLOCK);
    const int64_t row_bytes = FP4 ? R / 2 : R;
    const int64_t ctiles = (C + TC - 1) / TC, ktiles = (R + SEG - 1) / SEG;
    for (int64_t t = blockIdx.x; t < ctiles * ktiles; t += gridDim.x) {
        const int64_t kt = t / ctiles, ct = t - kt * ctiles;
        const int64_t k0 = kt * SEG, c0 = ct * TC;
        const int nk = static_cast<int>(R - k0 < SEG ? R - k0 : SEG);  // multiple of 32
#pragma unroll
        for (int j = 0; j < SEG * CPR / kThreads; ++j) {
            const int i = j * kThreads + threadIdx.x;
            const int r = i / CPR, cc = (i % CPR) * 8;
            uint4 w = make_uint4(0, 0, 0, 0);
            const int64_t col = c0 + cc;
            if (r < nk && col < C) {
                const uint16_t* src = a.x + (k0 + r) * a.ld + col;
                if (col + 8 <= C) {
                    w = __ldg(reinterpret_cast<const uint4*>(src));
                } else {
                    uint16_t h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    for (int e = 0; e < 8 && col + e < C; ++e)
                        h[e] = src[e];
                    w = make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                                   h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
                }
            }
            *reinterpret_cast<uint4*>(&tile[r][cc]) = w;
        }
        __syncthreads();
        const int64_t c = c0 + threadIdx.x;
        if (c < C) {
            uint32_t out[8];
            // the transform covers 32 rows: one MX block, two NVFP4 blocks
            constexpr int G = HAD ? 32 : BLOCK;
            float grp[G];
#pragma unroll
            for (int b = 0; b < SEG / BLOCK; ++b) {
                if (b % (G / BLOCK) == 0) {
#pragma unroll
                    for (int i = 0; i < G; ++i)
                        grp[i] = __uint_as_float(static_cast<uint32_t>(tile[b * BLOCK + i][threadIdx.x]) << 16);
                    if constexpr (HAD)
                        fwht_local<G>(grp);
                }
                float blk[BLOCK];
#pragma unroll
                for (int i = 0; i < BLOCK; ++i)
                    blk[i] = grp[(b % (G / BLOCK)) * BLOCK + i];
                float bmax = 0.0f;
#pragma unroll
                for (int i = 0; i < BLOCK; ++i)
                    bmax = fmaxf(bmax, fabsf(blk[i]));
                if constexpr (FMT == MX_FMT_MOSS_FP8)
                    bmax = moss_block(blk, bmax, sc);
                constexpr int WPB = FP4 ? BLOCK / 8 : BLOCK / 4;  // output words per block
                const uint64_t L8 = static_cast<uint64_t>(c) * (R / 8) + (k0 + b * BLOCK) / 8;
                const uint32_t sfb = encode_block<FMT, SR, BLOCK, !HAD>(blk, bmax, sc, a.rule, a.seed,
                                                                  a.stream_id, L8, out + b * WPB);
                if (b * BLOCK < nk)
                    a.sf[sf_offset(c, (k0 + b * BLOCK) / BLOCK, kgroups)] = static_cast<uint8_t>(sfb);
            }
            uint8_t* dst = a.codes + c * row_bytes + (FP4 ? k0 / 2 : k0);
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
            if (nk == SEG)
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ tile producer
// Persistent producer over 64-row tiles of x (128 or 256 columns, see
// TileShape) staged in shared memory by TMA through a three-stage mbarrier
// pipeline.  From each staged tile it emits the rowwise operand (blocks along
// the columns: a lane encodes one block of one row per step, its 16-byte
// chunks read in a lane-rotated order that keeps a quarter-warp's loads on
// distinct banks), the colwise operand (blocks along the 64 rows: a thread
// encodes two adjacent columns over 32 rows, one or two blocks per column,
// read as bf16 pairs with conflict-free 4-byte loads), or both: one read of x
// then serves the forward operand and the transposed operand a backward pass
// needs ("格式感知融合:让FP4预训练提速两倍的工程实践", section
// FP4加速为何常常"纸上富贵": operand packing, layout construction and saving
// backward state are the costs around the GEMM).  When the code arrays can be
// described by tensor maps, the codes are written over the consumed stage
// (after a CTA barrier) and leave through TMA tensor stores issued by one
// thread, which also refills the previous tile's stage once its stores have
// read it; otherwise each thread stores its codes and the last warp out of a
// stage refills it.  Scale bytes go straight to the consumer layout.
// Rounding is a compile-time choice per direction and the Hadamard transform
// is compiled only for the MX formats, so a kernel holds only the code it
// runs.
constexpr int kTR = 64, kTStages = 3;

// Tile width, threads and CTAs per SM of one tile-producer instance: 128
// columns with four CTAs of 128 threads per SM for the round-to-nearest
// passes (shorter barriers, four independent pipelines per SM), 256 columns
// with two CTAs of 256 threads for the arithmetic-heavy ones (stochastic
// rounding, NVFP4_LOCAL's exact divisions), where the per-tile costs weigh
// more.  One thread per tile column; three stages of kTR x cols bf16.
template <int FMT, bool ROW_SR, bool COL_SR>
struct TileShape {
    static constexpr int cols = (FMT == MX_FMT_NVFP4_LOCAL || ROW_SR || COL_SR) ? 256 : 128;
    static constexpr int threads = cols, ctas = cols == 128 ? 4 : 2;
    static constexpr int bytes = kTR * cols * 2;
};

// NVFP4 block encode under a region's own FP32 scale ts (NVFP4_LOCAL): the
// NVFP4 steps with IEEE quotients.  The scale differs from region to region,
// so no table of certified divisors is built per pass; instead each block
// certifies its own divisor d = fl32(dec(s_b) * ts) (the bf16 inputs make the
// double-word reciprocal product decide every E2M1 code as the exact quotient
// would, as for global NVFP4) and falls back to the shared-divisor division
// when the certificate or the range guard fails, or under stochastic rounding,
// which needs the exact quotient.  Produces the scale byte and N/8 words of
// codes; `v` is overwritten.
template <bool SR, int N>
__device__ __forceinline__ uint32_t nvfp4_local_encode(float (&v)[N], float bmax, float ts, uint64_t seed, uint32_t sid,
                                                       uint64_t L8, uint32_t* out)
{
    const float den = __fmul_rn(6.0f, ts);
    const uint32_t sb = cvt_e4m3x2(div_shared(bmax, den, recip_for_div(den)), 0.0f) & 0x7Fu;
    const float d = __fmul_rn(dec_e4m3_pos(sb), ts);
    if (d == 0.0f) {  // the block scale decodes to 0: sign-kept zero codes
#pragma unroll
        for (int w = 0; w < N / 8; ++w) {
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                word |= ((__float_as_uint(v[8 * w + i]) >> 31) << 3) << (4 * i);
            out[w] = word;
        }
        return sb;
    }
    bool fast = false;
    if constexpr (!SR) {
        if (quot2_certified_e2m1(d)) {
            const Recip2 r2 = recip2(d);
            if (__fmul_rn(bmax, r2.hi) < 0x1p100f) {
#pragma unroll
                for (int i = 0; i < N; ++i)
                    v[i] = quot2(v[i], r2);
                fast = true;
            }
        }
    }
    if (!fast) {
        const float r = recip_for_div(d);
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = div_shared(v[i], d, r);
    }
#pragma unroll
    for (int w = 0; w < N / 8; ++w) {
        if constexpr (SR) {
            uint32_t u[8];
            sr_bits8(seed, sid, L8 + w, u);
            out[w] = e2m1_sr8(&v[8 * w], u);
        } else {
            float q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                q[i] = v[8 * w + i];
            out[w] = cvt_e2m1x8(q);
        }
    }
    return sb;
}

// NVFP4 round-to-nearest-even encode of one block by certified double-word
// reciprocal products (no division, no branch).  Returns the scale byte and
// sets `redo` for a block whose divisor is not certified or whose quotients
// could overflow; the caller re-encodes such a block with encode_block.  `v`
// is left unchanged.
template <int N>
__device__ __forceinline__ uint32_t nvfp4_encode_fast(const float (&v)[N], float bmax, const ScaleCtx& sc,
                                                      uint32_t* out, bool& redo)
{
    const uint32_t sb = nvfp4_scale_byte(bmax, sc);
    const float2 q2 = sc.nv_q[sb];  // {0, 0} for d == 0 (sign-kept zeros), hi < 0 when not certified
    const Recip2 r{q2.x, q2.y};
    redo = q2.x < 0.0f || !(__fmul_rn(bmax, q2.x) < 0x1p100f);
#pragma unroll
    for (int w = 0; w < N / 8; ++w) {
        float q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            q[i] = quot2(v[8 * w + i], r);
        out[w] = cvt_e2m1x8(q);
    }
    return sb;
}

// ------------------------------------------------ packed-pair block encoding
// Round-to-nearest encodes of the MX formats in the tile producer, on element
// pairs: the block maxima come from the raw bf16 words by the bf16x2 absolute
// maximum (a compare, so exact), and the power-of-two scaling uses the paired
// FP32 multiply (two independent IEEE products, each rounded to nearest with
// no flushing, exactly as __fmul_rn rounds).  The codes are those of
// encode_block.  Both paired instructions issue at half the scalar rate, so
// they save issue slots, not pipe time: measured, this pays for the MX
// formats and not for NVFP4 and MOSS, whose products are dependent pairs.

// max(|a|, |b|) per bf16 half; the result's sign bits are the xor of the
// inputs' and are cleared by the caller.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max |x| per half over W words (W a power of two), sign bits cleared.
template <int W>
__device__ __forceinline__ uint32_t absmax_words(const uint32_t* w)
{
    uint32_t m[W / 2];
#pragma unroll
    for (int i = 0; i < W / 2; ++i)
        m[i] = absmax_bf16x2(w[i], w[i + W / 2]);
#pragma unroll
    for (int h = W / 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i)
            m[i] = absmax_bf16x2(m[i], m[i + h]);
    return m[0] & 0x7FFF7FFFu;
}

// {lo, hi} bf16 halves of w times {s.x, s.y}, by one paired multiply.
__device__ __forceinline__ float2 scale_pair(uint32_t w, float2 s)
{
    const float lo = bf16_lo(w), hi = bf16_hi(w);
    float2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(lo), "f"(hi), "f"(s.x), "f"(s.y));
    return d;
}

// One MX block of N consecutive elements given as N/2 bf16 words (element 2i
// in the low half of word i): its scale byte and codes (packed as
// encode_block packs them).
template <int FMT, int N>
__device__ __forceinline__ uint32_t row_encode_packed(const uint32_t (&w)[N / 2], int rule, uint32_t* out)
{
    const uint32_t mw = absmax_words<N / 2>(w);
    const int e = pow2_exponent<elem_of(FMT)>(fmaxf(bf16_lo(mw), bf16_hi(mw)), rule);
    const float2 s2 = make_float2(exp2_neg(e), exp2_neg(e));
    if constexpr (elem_of(FMT) == kElemE4M3) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float2 a = scale_pair(w[2 * i], s2), b = scale_pair(w[2 * i + 1], s2);
            out[i] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 8; ++i) {
            float q[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 a = scale_pair(w[4 * i + j], s2);
                q[2 * j] = a.x;
                q[2 * j + 1] = a.y;
            }
            out[i] = cvt_e2m1x8(q);
        }
    }
    return static_cast<uint32_t>(e + 127);
}

// Two MX colwise blocks at once: N words, word e holding row e of column A
// (low half) and of column B (high half).  Scale bytes and codes per column.
template <int FMT, int N>
__device__ __forceinline__ void col_encode_packed(const uint32_t* pk, int rule, uint32_t* outA, uint32_t* outB,
                                                  uint32_t& sfA, uint32_t& sfB)
{
    const uint32_t mw = absmax_words<N>(pk);
    const int eA = pow2_exponent<elem_of(FMT)>(bf16_lo(mw), rule);
    const int eB = pow2_exponent<elem_of(FMT)>(bf16_hi(mw), rule);
    const float2 s2 = make_float2(exp2_neg(eA), exp2_neg(eB));
    sfA = static_cast<uint32_t>(eA + 127);
    sfB = static_cast<uint32_t>(eB + 127);
    if constexpr (elem_of(FMT) == kElemE4M3) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            float2 q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                q[j] = scale_pair(pk[4 * i + j], s2);
            outA[i] = cvt_e4m3x2(q[0].x, q[1].x) | (cvt_e4m3x2(q[2].x, q[3].x) << 16);
            outB[i] = cvt_e4m3x2(q[0].y, q[1].y) | (cvt_e4m3x2(q[2].y, q[3].y) << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 8; ++i) {
            float qa[8], qb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 q = scale_pair(pk[8 * i + j], s2);
                qa[j] = q.x;
                qb[j] = q.y;
            }
            outA[i] = cvt_e2m1x8(qa);
            outB[i] = cvt_e2m1x8(qb);
        }
    }
}

template <int FMT, bool DO_ROW, bool DO_COL, bool ROW_SR, bool COL_SR>
__global__ void __launch_bounds__(TileShape<FMT, ROW_SR, COL_SR>::threads, TileShape<FMT, ROW_SR, COL_SR>::ctas)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmrow,
                      const __grid_constant__ CUtensorMap tmcol, const TileArgs a)
{
    using TS = TileShape<FMT, ROW_SR, COL_SR>;
    constexpr int kTC = TS::cols, kTT = TS::threads, kTileBytes = TS::bytes;
    constexpr int BLOCK = fmt_block(FMT);
    constexpr bool FP4 = elem_of(FMT) == kElemE2M1;
    constexpr bool HAD_OK = FMT == MX_FMT_MXFP8_E4M3 || FMT == MX_FMT_MXFP4_E2M1;
    // colwise task: two adjacent columns x 32 rows (one or two scale blocks per column)
    constexpr int CW = 2, CROWS = 32, GPB = CROWS / BLOCK;
    constexpr int kColGroups = kTC / CW;
    static_assert(kColGroups * (kTR / CROWS) == kTT, "one colwise task per encoding thread");
    constexpr int WPB = FP4 ? BLOCK / 8 : BLOCK / 4;  // 32-bit code words per scale block
    constexpr int CWW = GPB * WPB;                     // code words per column of a task
    constexpr int CBB = CROWS * (FP4 ? 1 : 2) / 2;     // code bytes per column of a task
    constexpr int RB_T = kTC * (FP4 ? 1 : 2) / 2;      // rowwise code bytes per tile row
    constexpr int ROWREG = kTR * RB_T;                 // staged rowwise codes of a tile
    static_assert(ROWREG + kTC * (kTR / CROWS) * CBB <= kTileBytes, "staged codes fit the stage");
    // MX round-to-nearest encodes without the transform take the packed-pair
    // path (measured: faster for the MX formats; NVFP4 and MOSS, whose
    // products are pairs of dependent operations, run faster on the scalar path)
    constexpr bool ROW_PACKED = HAD_OK && !ROW_SR;
    constexpr bool COL_PACKED = HAD_OK && !COL_SR;
    static_assert(CW == 2, "the packed colwise encode takes two columns");
    // rowwise task: one scale block of one tile row per lane and step
    constexpr int CH = BLOCK / 8;             // 8-element chunks per block
    constexpr int BPR = kTC / BLOCK;          // blocks per tile row
    constexpr int RPS = 32 / BPR;             // tile rows per warp step
    constexpr int STEPS = kTR / (RPS * (kTT / 32));
    constexpr int CB = FP4 ? 4 : 8;           // code bytes per chunk
    extern __shared__ uint8_t smem_raw[];
    // 128-byte aligned stage base, by pointer arithmetic on the shared array so
    // that the tile reads stay shared-memory loads
    uint8_t* base = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const uint32_t sbase = smem_u32(base);
    const uint32_t full0 = sbase + kTStages * kTileBytes;
    const uint32_t staged0 = full0 + 8u * kTStages;  // the stage holds the tile's codes (one arrival per warp)
    __shared__ float2 nv_tab[128];
    __shared__ float2 nv_q[128];
    __shared__ int stage_out[kTStages];  // warps done with the stage's current tile
    __shared__ int64_t issued;           // tiles whose copy has been issued
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t R = a.R, C = a.C;
    const bool tma_st = a.tma_st != 0;
    const ScaleCtx sc = make_scale_ctx<FMT>(a.amax, nv_tab, nv_q, a.rule);
    if ((FMT == MX_FMT_NVFP4 || FMT == MX_FMT_MOSS_FP8) && blockIdx.x == 0 && tid == 0) {
        *a.tensor_scale = sc.ts;
        if (a.tensor_scale_copy) {
            *a.tensor_scale_copy = sc.ts;
            *a.amax_copy = *a.amax;
        }
    }
    const int64_t ctiles = (C + kTC - 1) / kTC, tiles = ((R + kTR - 1) / kTR) * ctiles;
    const int64_t my_n = blockIdx.x < tiles ? (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto issue = [&](int64_t i) {  // copy tile i of this CTA into stage i % kTStages
        const int st = static_cast<int>(i % kTStages);
        const int64_t t = blockIdx.x + i * gridDim.x;
        const int64_t rt = t / ctiles, ct = t - rt * ctiles;
        mbar_arrive_expect_tx(full0 + 8u * st, kTileBytes);
        tma_load_2d(sbase + st * kTileBytes, &tmx, full0 + 8u * st, static_cast<int32_t>(ct * kTC),
                    static_cast<int32_t>(rt * kTR));
    };
    if (tid == 0) {
        for (int st = 0; st < kTStages; ++st) {
            mbar_init(full0 + 8u * st, 1);
            mbar_init(staged0 + 8u * st, kTT / 32);
            stage_out[st] = 0;
        }
        fence_mbar_init();
        prefetch_tmap(&tmx);
        if (tma_st) {
            if (DO_ROW)
                prefetch_tmap(&tmrow);
            if (DO_COL)
                prefetch_tmap(&tmcol);
        }
        const int64_t first = my_n < kTStages ? my_n : kTStages;
        for (int64_t i = 0; i < first; ++i)
            issue(i);
        issued = first;
    }
    __syncthreads();  // scale table, barriers and counters are ready

    // ---------------------------------------------------------- encoding warps
    const bool row_had = HAD_OK && a.row_had, col_had = HAD_OK && a.col_had;
    const int64_t kg_row = sf_kgroups(C / BLOCK), kg_col = sf_kgroups(R / BLOCK);
    const int64_t col_row_bytes = FP4 ? R / 2 : R;
    const int cg = tid % kColGroups, rh = tid / kColGroups;
    bool timed_out = false;
    for (int64_t i = 0; i < my_n; ++i) {
        const int st = static_cast<int>(i % kTStages);
        if (!mbar_wait_bounded(full0 + 8u * st, static_cast<uint32_t>(i / kTStages) & 1u, a.wait_ns) ||
            (i == a.fail_at && tid == kTT - 1)) {
            atomicExch(a.status, MX_ERR_TIMEOUT);
            timed_out = true;
        }
        // The staged path votes on timeouts at its CTA barrier below, so that
        // every thread leaves together (a thread that gave up encodes whatever
        // the stage holds: in-bounds stores of values the error status voids).
        if (!tma_st && timed_out)
            break;
        uint8_t* stage = base + st * kTileBytes;
        const uint16_t* tile = reinterpret_cast<const uint16_t*>(stage);  // [kTR][kTC]
        const int64_t t = blockIdx.x + i * gridDim.x;
        const int64_t rt = t / ctiles, ct = t - rt * ctiles;
        const int64_t r0 = rt * kTR, c0 = ct * kTC;
        // Scale-byte positions: a 64-bit base per tile (its 512-byte chunks)
        // plus small offsets.  Tiles start on 64 rows and 128 columns, so a
        // tile's K-blocks never cross a group of four and its rows stay in one
        // 128-row chunk.
        const int64_t kb_r0 = c0 / BLOCK, kb_c0 = r0 / BLOCK;  // first K-block: rowwise, colwise
        uint8_t* const row_sf_tile = DO_ROW ? a.row_sf + ((r0 >> 7) * kg_row + (kb_r0 >> 2)) * 512 : nullptr;
        uint8_t* const col_sf_tile = DO_COL ? a.col_sf + ((c0 >> 7) * kg_col + (kb_c0 >> 2)) * 512 + (kb_c0 & 3) : nullptr;
        const int row_q0 = static_cast<int>((r0 >> 5) & 3);  // 32-row quarter of the tile's first row

        // Rowwise: lane = one scale block of one tile row, read as CH 16-byte
        // chunks.  Plain round-to-nearest passes take the chunks in a
        // lane-rotated order (slot i holds chunk (i + rot) % CH), which makes
        // each quarter-warp's loads hit 32 distinct banks; the codes go back to
        // their own positions when stored.  SR and the Hadamard transform need
        // the natural order.
        const int kbl = lane % BPR;
        const int rot = (ROW_SR || row_had) ? 0 : (CH == 2 ? (lane >> 2) & 1 : (CH == 4 ? (lane >> 1) & 3 : 0));
        uint32_t rout[DO_ROW ? STEPS : 1][FP4 ? BLOCK / 8 : BLOCK / 4];
        if constexpr (DO_ROW) {
            const int64_t col = c0 + kbl * BLOCK;
            const int sf_in_row = (kbl >> 2) * 512 + (kbl & 3);
#pragma unroll
            for (int s2 = 0; s2 < STEPS; ++s2) {
                const int rr = (s2 * (kTT / 32) + warp) * RPS + lane / BPR;
                const int64_t row = r0 + rr;
                const uint16_t* src = tile + rr * kTC + kbl * BLOCK;
                uint32_t* out = rout[s2];
                uint32_t sfb = 0;
                bool scalar = true;  // encode on the scalar path (SR, the transform, or not an MX format)
                if constexpr (ROW_PACKED) {
                    if (!row_had) {
                        uint32_t w[BLOCK / 2];
#pragma unroll
                        for (int c = 0; c < CH; ++c) {
                            const uint4 q = *reinterpret_cast<const uint4*>(src + ((c + rot) & (CH - 1)) * 8);
                            w[4 * c] = q.x, w[4 * c + 1] = q.y, w[4 * c + 2] = q.z, w[4 * c + 3] = q.w;
                        }
                        sfb = row_encode_packed<FMT, BLOCK>(w, a.rule, out);
                        scalar = false;
                    }
                }
                if (scalar) {
                    float v[BLOCK];
                    uint32_t w[BLOCK / 2];
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        const uint4 q = *reinterpret_cast<const uint4*>(src + ((c + rot) & (CH - 1)) * 8);
                        w[4 * c] = q.x, w[4 * c + 1] = q.y, w[4 * c + 2] = q.z, w[4 * c + 3] = q.w;
                        unpack8(q, v + 8 * c);
                    }
                    float bmax = 0.0f;
                    if constexpr (FMT == MX_FMT_NVFP4) {  // from the bf16 words, two at a time (measured faster for NVFP4 only)
                        const uint32_t mw = absmax_words<BLOCK / 2>(w);
                        bmax = fmaxf(bf16_lo(mw), bf16_hi(mw));
                    } else {
                        if constexpr (HAD_OK) {
                            if (row_had)
                                fwht_local<BLOCK>(v);
                        }
#pragma unroll
                        for (int e = 0; e < BLOCK; ++e)
                            bmax = fmaxf(bmax, fabsf(v[e]));
                    }
                    if constexpr (FMT == MX_FMT_MOSS_FP8)
                        bmax = moss_block(v, bmax, sc);
                    const uint64_t L8 = static_cast<uint64_t>(row) * (C / 8) + col / 8;
                    if constexpr (FMT == MX_FMT_NVFP4_LOCAL) {
                        sfb = nvfp4_local_encode<ROW_SR, BLOCK>(v, bmax, a.row_ts_v[r0 >> 7], a.seed, a.stream_id, L8,
                                                                out);
                    } else if constexpr (FMT == MX_FMT_NVFP4 && !ROW_SR) {
                        bool redo;
                        sfb = nvfp4_encode_fast<BLOCK>(v, bmax, sc, out, redo);
                        if (redo)  // rare: this block's divisor is not certified
                            sfb = encode_block<FMT, false, BLOCK>(v, bmax, sc, a.rule, 0, 0, 0, out);
                    } else {
                        sfb = encode_block<FMT, ROW_SR, BLOCK>(v, bmax, sc, a.rule, a.seed, a.stream_id, L8, out);
                    }
                }
                if (row < R && col < C) {  // whole scale blocks are in or out (C % BLOCK == 0)
                    if (!tma_st) {
                        uint8_t* dst = a.row_codes + row * (FP4 ? C / 2 : C) + (FP4 ? col / 2 : col);
#pragma unroll
                        for (int c = 0; c < CH; ++c) {
                            const int cc = (c + rot) & (CH - 1);
                            if constexpr (FP4)
                                *reinterpret_cast<uint32_t*>(dst + cc * CB) = out[c];
                            else
                                *reinterpret_cast<uint2*>(dst + cc * CB) = make_uint2(out[2 * c], out[2 * c + 1]);
                        }
                    }
                    row_sf_tile[sf_in_row + (rr & 31) * 16 + (row_q0 + (rr >> 5)) * 4] = static_cast<uint8_t>(sfb);
                }
            }
        }

        // Colwise: thread = two adjacent columns x 32 rows.  Each shared-memory
        // load brings both columns of one row (a warp reads 128 contiguous bytes
        // of that row: no bank conflicts); each column's 32 values are one MX
        // block or two NVFP4 blocks, encoded in registers.
        const int64_t kabs = r0 + rh * CROWS;  // first row (K) of this task
        // scale byte of tile column ml, tile K-block lk
        auto col_sf_at = [&](int ml, int lk) {
            return col_sf_tile + ((ml >> 7) ? kg_col * 512 : 0) + ((ml & 31) * 16 + ((ml >> 5) & 3) * 4 + lk);
        };
        uint32_t cout[DO_COL ? CW : 1][CWW];
        if constexpr (DO_COL) {
            if (kabs < R) {  // R % 32 == 0: a task's rows are wholly in or out
                uint32_t pk[CROWS];  // bf16 pairs: columns 2 cg, 2 cg + 1 of row e
#pragma unroll
                for (int e = 0; e < CROWS; ++e)
                    pk[e] = *reinterpret_cast<const uint32_t*>(tile + (rh * CROWS + e) * kTC + cg * CW);
                const int64_t cbase = c0 + cg * CW;
                // blocks left to the scalar path: bit j * GPB + g (column j, block g)
                uint32_t scalar = (1u << (CW * GPB)) - 1u;
                if constexpr (COL_PACKED) {
                    if (!col_had) {
                        scalar = 0;
#pragma unroll
                        for (int g = 0; g < GPB; ++g) {
                            uint32_t sfA, sfB;
                            col_encode_packed<FMT, BLOCK>(&pk[g * BLOCK], a.rule, &cout[0][g * WPB], &cout[1][g * WPB],
                                                          sfA, sfB);
                            if (cbase < C)
                                *col_sf_at(cg * CW, rh * GPB + g) = static_cast<uint8_t>(sfA);
                            if (cbase + 1 < C)
                                *col_sf_at(cg * CW + 1, rh * GPB + g) = static_cast<uint8_t>(sfB);
                        }
                    }
                }
                // NVFP4: block maxima of both columns from the bf16 words, two at a time
                uint32_t mwg[GPB];
#pragma unroll
                for (int g = 0; g < GPB; ++g)
                    mwg[g] = FMT == MX_FMT_NVFP4 ? absmax_words<BLOCK>(&pk[g * BLOCK]) : 0u;
#pragma unroll
                for (int j = 0; j < CW; ++j) {
#pragma unroll
                    for (int g = 0; g < GPB; ++g) {
                        if (!((scalar >> (j * GPB + g)) & 1u))
                            continue;
                        float blk[BLOCK];
#pragma unroll
                        for (int e = 0; e < BLOCK; ++e)
                            blk[e] = j ? bf16_hi(pk[g * BLOCK + e]) : bf16_lo(pk[g * BLOCK + e]);
                        float bmax = j ? bf16_hi(mwg[g]) : bf16_lo(mwg[g]);
                        if constexpr (FMT != MX_FMT_NVFP4) {
                            if constexpr (HAD_OK) {
                                if (col_had)
                                    fwht_local<BLOCK>(blk);
                            }
#pragma unroll
                            for (int e = 0; e < BLOCK; ++e)
                                bmax = fmaxf(bmax, fabsf(blk[e]));
                        }
                        if constexpr (FMT == MX_FMT_MOSS_FP8)
                            bmax = moss_block(blk, bmax, sc);
                        const int64_t kblk = kabs + g * BLOCK;
                        const uint64_t L8 = static_cast<uint64_t>(cbase + j) * (R / 8) + kblk / 8;
                        uint32_t* out = &cout[j][g * WPB];
                        uint32_t sfb;
                        if constexpr (FMT == MX_FMT_NVFP4_LOCAL) {
                            const float ts = cbase < C ? a.col_ts_v[cbase >> 7] : 1.0f;  // past C: zero fill, not stored
                            sfb = nvfp4_local_encode<COL_SR, BLOCK>(blk, bmax, ts, a.seed, a.stream_id, L8, out);
                        } else if constexpr (FMT == MX_FMT_NVFP4 && !COL_SR) {
                            bool redo;
                            sfb = nvfp4_encode_fast<BLOCK>(blk, bmax, sc, out, redo);  // leaves blk unchanged
                            if (redo)  // rare: this block's divisor is not certified
                                sfb = encode_block<FMT, false, BLOCK>(blk, bmax, sc, a.rule, 0, 0, 0, out);
                        } else {
                            sfb = encode_block<FMT, COL_SR, BLOCK>(blk, bmax, sc, a.rule, a.seed, a.stream_id, L8, out);
                        }
                        if (cbase + j < C)
                            *col_sf_at(cg * CW + j, rh * GPB + g) = static_cast<uint8_t>(sfb);
                    }
                    if (!tma_st && cbase + j < C) {
                        uint8_t* dst = a.col_codes + (cbase + j) * col_row_bytes + (FP4 ? kabs / 2 : kabs);
#pragma unroll
                        for (int q = 0; q < CWW / 4; ++q)
                            reinterpret_cast<uint4*>(dst)[q] =
                                make_uint4(cout[j][4 * q], cout[j][4 * q + 1], cout[j][4 * q + 2], cout[j][4 * q + 3]);
                    }
                }
            }
        }

        if (tma_st) {
            // The codes of the tile go out through TMA tensor stores from the
            // stage the tile came in on: once every thread is done reading it
            // (a barrier of the CTA), the codes are written over it (rowwise
            // [64 rows][row bytes], then colwise [32-row half][tile columns]
            // [column bytes]) and each warp signals the stage's "staged"
            // barrier; thread 0 waits for it, stores, and refills the stage of
            // the previous tile, whose stores have had a tile's time to read it.
            if (named_barrier_or(1, kTT, timed_out))  // every thread is done reading the stage
                break;
            if constexpr (DO_ROW) {
#pragma unroll
                for (int s2 = 0; s2 < STEPS; ++s2) {
                    const int rr = (s2 * (kTT / 32) + warp) * RPS + lane / BPR;
                    uint8_t* dst = stage + rr * RB_T + kbl * BLOCK * (FP4 ? 1 : 2) / 2;
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        const int cc = (c + rot) & (CH - 1);
                        if constexpr (FP4)
                            *reinterpret_cast<uint32_t*>(dst + cc * CB) = rout[s2][c];
                        else
                            *reinterpret_cast<uint2*>(dst + cc * CB) = make_uint2(rout[s2][2 * c], rout[s2][2 * c + 1]);
                    }
                }
            }
            if constexpr (DO_COL) {
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    uint8_t* dst = stage + ROWREG + (rh * kTC + cg * CW + j) * CBB;
#pragma unroll
                    for (int q = 0; q < CWW / 4; ++q)
                        reinterpret_cast<uint4*>(dst)[q] =
                            make_uint4(cout[j][4 * q], cout[j][4 * q + 1], cout[j][4 * q + 2], cout[j][4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(staged0 + 8u * st);
            if (tid == 0) {
                if (!mbar_wait_bounded(staged0 + 8u * st, static_cast<uint32_t>(i / kTStages) & 1u, a.wait_ns)) {
                    atomicExch(a.status, MX_ERR_TIMEOUT);  // the CTA stops at the next tile's barrier vote
                    timed_out = true;
                } else {
                    const uint32_t s = sbase + st * kTileBytes;
                    if constexpr (DO_ROW)
                        tma_store_2d(&tmrow, s, static_cast<int32_t>(FP4 ? c0 / 2 : c0), static_cast<int32_t>(r0));
                    if constexpr (DO_COL)
                        for (int h = 0; h < kTR / CROWS; ++h)
                            if (r0 + h * CROWS < R)
                                tma_store_2d(&tmcol, s + ROWREG + h * kTC * CBB,
                                             static_cast<int32_t>(FP4 ? (r0 + h * CROWS) / 2 : r0 + h * CROWS),
                                             static_cast<int32_t>(c0));
                    bulk_commit();
                    // the previous tile's stores have read its stage: refill it
                    if (i >= 1 && i - 1 + kTStages < my_n) {
                        bulk_wait_read_1();
                        issue(i - 1 + kTStages);
                        issued = i - 1 + kTStages + 1;
                    }
                }
            }
        } else {
            __syncwarp();  // every lane of this warp is done reading the stage
            if (lane == 0) {
                __threadfence_block();  // release this warp's reads before counting out
                if (atomicAdd(&stage_out[st], 1) == kTT / 32 - 1) {  // last warp out refills
                    __threadfence_block();
                    stage_out[st] = 0;
                    if (i + kTStages < my_n) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue(i + kTStages);
                        atomicMax(reinterpret_cast<unsigned long long*>(&issued),
                                  static_cast<unsigned long long>(i + kTStages + 1));
                    }
                }
            }
        }
    }
    // Leave only when no copy into this CTA's shared memory can still be in
    // flight (after a timeout some issued tiles were never consumed) and the
    // TMA stores have completed.
    __syncthreads();
    if (tid == 0) {
        if (tma_st)
            bulk_wait_all();
        const int64_t n = issued;
        for (int64_t j = n > kTStages ? n - kTStages : 0; j < n; ++j)
            (void)mbar_wait_bounded(full0 + 8u * static_cast<int>(j % kTStages),
                                    static_cast<uint32_t>(j / kTStages) & 1u, kWaitLimitNs);
    }
}

// NVFP4_LOCAL region maxima.  CTA (x, y) covers input rows
// 128 y .. 128 y + 127 and columns 2048 x .. 2048 x + 2047: thread t owns the
// 8-column chunk t of every row (a warp reads 512 contiguous bytes per row),
// so its columns stay in one 128-column region; row and column maxima are
// combined in the CTA and land with one atomicMax each (|x| bits order like
// the values).
constexpr int kRegSlab = 2048;
__global__ void __launch_bounds__(kThreads) region_amax_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                               int64_t ld, unsigned* __restrict__ amax_rows,
                                                               unsigned* __restrict__ amax_cols)
{
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kLocalRegion;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * kRegSlab + threadIdx.x * 8;
    const int64_t r1 = r0 + kLocalRegion < R ? r0 + kLocalRegion : R;
    uint32_t m2 = 0;  // two packed |bf16| maxima
    if (c < C) {
        for (int64_t r = r0; r < r1; ++r) {
            const uint16_t* p = x + r * ld + c;
            if (c + 8 <= C) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
                m2 = __vmaxu2(m2, w.x & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, w.y & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, w.z & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, w.w & 0x7FFF7FFFu);
            } else {
                for (int64_t e = 0; c + e < C; ++e)
                    m2 = __vmaxu2(m2, static_cast<uint32_t>(p[e]) & 0x7FFFu);
            }
        }
    }
    unsigned m = max(m2 & 0xFFFFu, m2 >> 16) << 16;  // bf16 bits -> fp32 bits of |x|
    // columns: the 16 threads of a 128-column region are one half-warp
    unsigned mc = m;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1)
        mc = max(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, o));
    if (amax_cols && (threadIdx.x & 15) == 0 && c < C)
        atomicMax(amax_cols + (c >> 7), mc);
    if (amax_rows) {
        unsigned mr = __reduce_max_sync(0xFFFFFFFFu, m);
        __shared__ unsigned wmax[kThreads / 32];
        if ((threadIdx.x & 31) == 0)
            wmax[threadIdx.x >> 5] = mr;
        __syncthreads();
        if (threadIdx.x < 32) {
            mr = threadIdx.x < kThreads / 32 ? wmax[threadIdx.x] : 0u;
            mr = __reduce_max_sync(0xFFFFFFFFu, mr);
            if (threadIdx.x == 0)
                atomicMax(amax_rows + blockIdx.y, mr);
        }
    }
}

__global__ void local_scales_kernel(const float* __restrict__ amax, float* __restrict__ ts, int64_t n)
{
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x)
        ts[g] = amax[g] == 0.0f ? 1.0f : __fdiv_rn(amax[g], 2688.0f);
}

__global__ void __launch_bounds__(kThreads) dequant_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ sf,
                                                           const float* __restrict__ ts, int64_t rows,
                                                           int64_t k, int fmt, float* __restrict__ out)
{
    const int block = fmt_block(fmt);
    const int64_t kgroups = sf_kgroups(k / block);
    const float t = (fmt_has_tensor_scale(fmt) && ts) ? *ts : 1.0f;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows * k;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / k, j = i - r * k;
        float cv;
        if (fmt_is_fp4(fmt)) {
            const uint32_t byte = codes[r * (k / 2) + j / 2];
            const uint32_t n = (j & 1) ? (byte >> 4) : (byte & 0xFu);
            const float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
            cv = (n & 8u) ? -mags[n & 7u] : mags[n & 7u];
        } else {
            const uint32_t byte = codes[r * k + j];
            const float mag = dec_e4m3_pos(byte & 0x7Fu);
            cv = (byte & 0x80u) ? -mag : mag;
        }
        const uint32_t s = sf[sf_offset(r, j / block, kgroups)];
        const float sv = fmt == MX_FMT_NVFP4 ? dec_e4m3_pos(s) : exp2_neg(127 - static_cast<int>(s));
        out[i] = __fmul_rn(__fmul_rn(cv, sv), t);
    }
}

__global__ void __launch_bounds__(kThreads) divide_check_kernel(const float* __restrict__ v, const float* __restrict__ d,
                                                                int64_t n, float* __restrict__ fast,
                                                                float* __restrict__ ieee)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float dv = d[i];
        fast[i] = div_shared(v[i], dv, recip_for_div(dv));
        ieee[i] = __fdiv_rn(v[i], dv);
    }
}

__global__ void wait_selftest_kernel(uint64_t limit_ns, int* status)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        // Nothing ever arrives on `bar`: the wait must give up.
        if (!mbar_wait_bounded(b, 0, limit_ns))
            atomicExch(status, MX_ERR_TIMEOUT);
    }
}

template <int FMT, bool SR, bool HAD>
int launch_q(const QuantArgs& q, const Device& d, cudaStream_t s)
{
    if (q.dir == MX_ROWWISE) {
        const int64_t cpr = q.C / 8;
        const int64_t items = q.R * ((cpr + kThreads * 4 - 1) / (kThreads * 4));
        const int grid = static_cast<int>(std::min<int64_t>(items, static_cast<int64_t>(d.sms) * 8));
        quant_row_kernel<FMT, SR, HAD><<<grid, kThreads, 0, s>>>(q);
        count_launch();
    } else {
        constexpr int SEG = elem_of(FMT) == kElemE2M1 ? 64 : 32;
        const int64_t tiles = ((q.C + kThreads - 1) / kThreads) * ((q.R + SEG - 1) / SEG);
        const int grid = static_cast<int>(std::min<int64_t>(tiles, static_cast<int64_t>(d.sms) * 8));
        quant_col_kernel<FMT, SR, HAD><<<grid, kThreads, 0, s>>>(q);
        count_launch();
    }
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

using EncodeTiledFnQ = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnQ encode_fn_q()
{
    static EncodeTiledFnQ fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFnQ>(p);
    }();
    return fn;
}

// 2-D map over a row-major byte matrix [rows, row_bytes] for TMA stores of
// box_bytes x box_rows boxes; false where the map cannot describe it (row
// stride not a multiple of 16 bytes).
bool make_code_store_map(CUtensorMap* m, void* base, int64_t rows, int64_t row_bytes, int box_bytes, int box_rows)
{
    EncodeTiledFnQ enc = encode_fn_q();
    if (!enc || row_bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int FMT, bool DO_ROW, bool DO_COL, bool ROW_SR, bool COL_SR>
int launch_tile(const TileArgs& t_in, int64_t ld, const Device& d, cudaStream_t s)
{
    auto kernel = quant_tile_kernel<FMT, DO_ROW, DO_COL, ROW_SR, COL_SR>;
    using TS = TileShape<FMT, ROW_SR, COL_SR>;
    constexpr int kTC = TS::cols;
    constexpr int smem = kTStages * TS::bytes + 2 * kTStages * 8 + 128;
    constexpr bool FP4 = elem_of(FMT) == kElemE2M1;
    static int configured_device = -1;
    if (configured_device != d.id) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return MX_ERR_CUDA;
        configured_device = d.id;
    }
    EncodeTiledFnQ enc = encode_fn_q();
    if (!enc)
        return MX_ERR_CUDA;
    TileArgs t = t_in;
    CUtensorMap m;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(t.C), static_cast<cuuint64_t>(t.R)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {kTC, kTR};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(t.x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MX_ERR_CUDA;
    // The codes leave through TMA stores when both code arrays can be
    // described by tensor maps (row strides that are multiples of 16 bytes),
    // else through direct stores.
    CUtensorMap mrow = m, mcol = m;
    const int64_t row_bytes = FP4 ? t.C / 2 : t.C, col_bytes = FP4 ? t.R / 2 : t.R;
    bool ok = true;
    if (DO_ROW)
        ok = ok && make_code_store_map(&mrow, t.row_codes, t.R, row_bytes, FP4 ? kTC / 2 : kTC, kTR);
    if (DO_COL)
        ok = ok && make_code_store_map(&mcol, t.col_codes, t.C, col_bytes, FP4 ? 16 : 32, kTC);
    t.tma_st = ok ? 1 : 0;
    const int64_t tiles = ((t.R + kTR - 1) / kTR) * ((t.C + kTC - 1) / kTC);
    const int grid = static_cast<int>(std::min<int64_t>(tiles, static_cast<int64_t>(d.sms) * TS::ctas));
    kernel<<<grid, TS::threads, smem, s>>>(m, mrow, mcol, t);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

// Rounding is a compile-time choice per direction.
template <int FMT, bool DO_ROW, bool DO_COL>
int launch_tile_sr(const TileArgs& t, int64_t ld, const Device& d, cudaStream_t s)
{
    const bool rsr = DO_ROW && t.row_sr, csr = DO_COL && t.col_sr;
    if (rsr && csr)
        return launch_tile<FMT, DO_ROW, DO_COL, DO_ROW, DO_COL>(t, ld, d, s);
    if (rsr)
        return launch_tile<FMT, DO_ROW, DO_COL, DO_ROW, false>(t, ld, d, s);
    if (csr)
        return launch_tile<FMT, DO_ROW, DO_COL, false, DO_COL>(t, ld, d, s);
    return launch_tile<FMT, DO_ROW, DO_COL, false, false>(t, ld, d, s);
}

template <bool DO_ROW, bool DO_COL>
int launch_tile_fmt(const TileArgs& t, int64_t ld, const Device& d, cudaStream_t s)
{
    switch (t.fmt) {
    case MX_FMT_MXFP8_E4M3: return launch_tile_sr<MX_FMT_MXFP8_E4M3, DO_ROW, DO_COL>(t, ld, d, s);
    case MX_FMT_MXFP4_E2M1: return launch_tile_sr<MX_FMT_MXFP4_E2M1, DO_ROW, DO_COL>(t, ld, d, s);
    case MX_FMT_NVFP4: return launch_tile_sr<MX_FMT_NVFP4, DO_ROW, DO_COL>(t, ld, d, s);
    case MX_FMT_MOSS_FP8: return launch_tile_sr<MX_FMT_MOSS_FP8, DO_ROW, DO_COL>(t, ld, d, s);
    case MX_FMT_NVFP4_LOCAL: return launch_tile_sr<MX_FMT_NVFP4_LOCAL, DO_ROW, DO_COL>(t, ld, d, s);
    default: return MX_ERR_INVALID_ARG;
    }
}

}  // namespace

int launch_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax, const Device& d, cudaStream_t s)
{
    if (cudaMemsetAsync(amax, 0, sizeof(float), s) != cudaSuccess)
        return MX_ERR_CUDA;
    if (R == 0 || C == 0)
        return MX_OK;
    const int64_t chunks = R * (C / 8);
    dim3 grid;
    if (ld == C) {
        grid.x = static_cast<unsigned>(std::max<int64_t>(
            1, std::min<int64_t>((chunks + kThreads - 1) / kThreads, static_cast<int64_t>(d.sms) * 8)));
    } else {
        grid.x = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((C / 8 + kThreads - 1) / kThreads, 64)));
        grid.y = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(R, (static_cast<int64_t>(d.sms) * 8 + grid.x - 1) / grid.x)));
    }
    amax_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), R, C, ld, reinterpret_cast<unsigned*>(amax));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_had_amax(const void* x, int64_t R, int64_t C, int64_t ld, int dir, float* amax, const Device& d,
                    cudaStream_t s)
{
    if (cudaMemsetAsync(amax, 0, sizeof(float), s) != cudaSuccess)
        return MX_ERR_CUDA;
    if (R == 0 || C == 0)
        return MX_OK;
    const int64_t warps = dir == MX_ROWWISE ? (R * (C / 8) + 31) / 32 : (R / 32) * (((C + 1) / 2 + 31) / 32);
    const int grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((warps + kThreads / 32 - 1) / (kThreads / 32), static_cast<int64_t>(d.sms) * 8)));
    had_amax_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), R, C, ld, dir,
                                              reinterpret_cast<unsigned*>(amax));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_region_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax_rows, float* amax_cols,
                       const Device& d, cudaStream_t s)
{
    const int64_t gr = (R + kLocalRegion - 1) / kLocalRegion, gc = (C + kLocalRegion - 1) / kLocalRegion;
    if (amax_rows && cudaMemsetAsync(amax_rows, 0, sizeof(float) * std::max<int64_t>(gr, 1), s) != cudaSuccess)
        return MX_ERR_CUDA;
    if (amax_cols && cudaMemsetAsync(amax_cols, 0, sizeof(float) * std::max<int64_t>(gc, 1), s) != cudaSuccess)
        return MX_ERR_CUDA;
    if (R == 0 || C == 0)
        return MX_OK;
    const dim3 grid(static_cast<unsigned>((C + kRegSlab - 1) / kRegSlab), static_cast<unsigned>(gr));
    region_amax_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), R, C, ld,
                                                 reinterpret_cast<unsigned*>(amax_rows),
                                                 reinterpret_cast<unsigned*>(amax_cols));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_local_scales(const float* amax, float* ts, int64_t n, const Device& d, cudaStream_t s)
{
    if (n <= 0)
        return MX_OK;
    const int grid = static_cast<int>(std::min<int64_t>((n + kThreads - 1) / kThreads, d.sms));
    local_scales_kernel<<<grid, kThreads, 0, s>>>(amax, ts, n);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_quantize(const QuantArgs& q, const Device& d, cudaStream_t s)
{
    const bool sr = q.rounding == MX_ROUND_SR;
    const bool had = q.hadamard != 0;
    switch (q.fmt) {
    case MX_FMT_MXFP8_E4M3:
        if (sr)
            return had ? launch_q<MX_FMT_MXFP8_E4M3, true, true>(q, d, s)
                       : launch_q<MX_FMT_MXFP8_E4M3, true, false>(q, d, s);
        return had ? launch_q<MX_FMT_MXFP8_E4M3, false, true>(q, d, s)
                   : launch_q<MX_FMT_MXFP8_E4M3, false, false>(q, d, s);
    case MX_FMT_MXFP4_E2M1:
        if (sr)
            return had ? launch_q<MX_FMT_MXFP4_E2M1, true, true>(q, d, s)
                       : launch_q<MX_FMT_MXFP4_E2M1, true, false>(q, d, s);
        return had ? launch_q<MX_FMT_MXFP4_E2M1, false, true>(q, d, s)
                   : launch_q<MX_FMT_MXFP4_E2M1, false, false>(q, d, s);
    case MX_FMT_NVFP4:
        if (sr)
            return had ? launch_q<MX_FMT_NVFP4, true, true>(q, d, s) : launch_q<MX_FMT_NVFP4, true, false>(q, d, s);
        return had ? launch_q<MX_FMT_NVFP4, false, true>(q, d, s) : launch_q<MX_FMT_NVFP4, false, false>(q, d, s);
    case MX_FMT_MOSS_FP8:
        return sr ? launch_q<MX_FMT_MOSS_FP8, true, false>(q, d, s) : launch_q<MX_FMT_MOSS_FP8, false, false>(q, d, s);
    default:
        return MX_ERR_INVALID_ARG;
    }
}

int launch_quantize_tile(const TileArgs& t, int64_t ld, const Device& d, cudaStream_t s)
{
    if (t.R == 0 || t.C == 0)
        return MX_OK;
    const bool row = t.row_codes != nullptr, col = t.col_codes != nullptr;
    if (row && col)
        return launch_tile_fmt<true, true>(t, ld, d, s);
    if (row)
        return launch_tile_fmt<true, false>(t, ld, d, s);
    if (col)
        return launch_tile_fmt<false, true>(t, ld, d, s);
    return MX_ERR_INVALID_ARG;
}

int launch_dequantize(const mx_tensor* A, float* out, const Device& d, cudaStream_t s)
{
    const int64_t n = A->rows * A->k;
    if (n == 0)
        return MX_OK;
    const int grid = static_cast<int>(std::min<int64_t>((n + kThreads - 1) / kThreads, static_cast<int64_t>(d.sms) * 8));
    dequant_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(A->codes), A->sf, A->tensor_scale, A->rows,
                                             A->k, A->fmt, out);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_divide_check(const float* v, const float* dv, int64_t n, float* fast, float* ieee, const Device& d,
                        cudaStream_t s)
{
    if (n == 0)
        return MX_OK;
    const int grid = static_cast<int>(std::min<int64_t>((n + kThreads - 1) / kThreads, static_cast<int64_t>(d.sms) * 8));
    divide_check_kernel<<<grid, kThreads, 0, s>>>(v, dv, n, fast, ieee);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_wait_selftest(uint64_t limit_ns, const Device& d, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, d.status);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
