/*
 * mx_oracle.c -- plain, slow CPU oracle for the block-scaled (microscaling)
 * low-precision linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path.  Page citations: see mx_oracle.h.
 *
 * Arithmetic conventions
 *   - bf16 -> fp32 is exact; every fp32 step the method fixes (a product by a
 *     power of two, the MOSS and NVFP4 divisions, the Hadamard butterflies) is
 *     done in C `float`, which is IEEE binary32 with round-to-nearest-even and
 *     gradual underflow on the targets we build for (FLT_EVAL_METHOD == 0,
 *     compiled with -ffp-contract=off, no -ffast-math).
 *   - Grid searches, scale-rule decisions and the GEMM use fp64, where every
 *     comparison made here is exact.
 *   - Codes are found by searching the enumerated value grid, not by bit tricks.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py; the
 * quotients by the tensor scale (NVFP4 block-scale byte and element divisor,
 * MOSS level 1) also in tests/test_oracle_quotient_pins.py.
 */
#include "mx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                            */
/* ------------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t orc_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))  /* NaN */
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* Value grids, defined by their bit patterns.                              */
/* E4M3 ([COAT] FP8 量化最佳化器狀態的難點: largest value 448, smallest      */
/* 0.00195 = 2^-9): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent  */
/* field 0 is subnormal m*2^-9; S.1111.111 is NaN; no infinities.           */
/* E2M1 ([FAF] FP4加速为何常常"纸上富贵": 1 sign, 2 exponent, 1 mantissa):  */
/* bias 1, exponent 0 is subnormal m*0.5, no NaN/Inf.                       */
/* E8M0 (the MX block scale, an exponent-only byte): 2^(b-127), 0xFF = NaN. */
/* ------------------------------------------------------------------------ */

double orc_decode_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 0xfu, m = code & 7u;
    if (e == 15u && m == 7u)
        return NAN;
    double mag = (e == 0u) ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

double orc_decode_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0u) ? 0.5 * (double)m : ldexp(1.0 + (double)m / 2.0, (int)e - 1);
    return s ? -mag : mag;
}

double orc_decode_e8m0(unsigned code)
{
    if ((code & 0xffu) == 0xffu)
        return NAN;
    return ldexp(1.0, (int)(code & 0xffu) - 127);
}

/* The non-negative value grids, decoded once from the bit patterns above:
 * E4M3 codes 0x00..0x7E and E2M1 codes 0..7, strictly increasing. */
static double g_e4m3_grid[0x7f];
static double g_e2m1_grid[8];

__attribute__((constructor)) static void init_grids(void)
{
    for (unsigned c = 0; c <= 0x7eu; ++c)
        g_e4m3_grid[c] = orc_decode_e4m3(c);
    for (unsigned c = 0; c <= 7u; ++c)
        g_e2m1_grid[c] = orc_decode_e2m1(c);
}

/* Nearest point of an increasing non-negative grid g[0] = 0 < ... < g[maxcode]
 * to a >= 0.  Values at or above the largest point saturate to it.  The
 * nearest point is one of the two grid neighbours of a; an exact tie goes to
 * the code whose mantissa LSB (= code LSB) is 0. */
static unsigned nearest_grid_code(double a, const double* g, unsigned maxcode)
{
    if (a >= g[maxcode])
        return maxcode;
    unsigned lo = 0u, hi = maxcode; /* invariant: g[lo] <= a < g[hi] */
    while (hi - lo > 1u) {
        unsigned mid = (lo + hi) / 2u;
        if (g[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - g[lo], dhi = g[hi] - a;
    if (dlo < dhi)
        return lo;
    if (dhi < dlo)
        return hi;
    return (lo & 1u) ? hi : lo;
}

/* Round-to-nearest-even with saturation to the largest finite value (the
 * "就近舍入" of [FAF] 两个关键的数值技巧; the clamp before the cast in [MOSS]
 * 两级缩放实现).  The sign bit of v is kept, also when the result is zero. */
unsigned orc_encode_e4m3_rne(float v)
{
    unsigned s = signbit(v) ? 0x80u : 0u;
    return s | nearest_grid_code(fabs((double)v), g_e4m3_grid, 0x7eu);
}

unsigned orc_encode_e2m1_rne(float v)
{
    unsigned s = signbit(v) ? 0x8u : 0u;
    return s | nearest_grid_code(fabs((double)v), g_e2m1_grid, 0x7u);
}

/* Stochastic rounding onto the E2M1 grid ([FAF] 两个关键的数值技巧: round up
 * with probability proportional to the distance, unbiased in expectation).
 * u16 is a uniform 16-bit integer; the value rounds up iff u16 * 2^-16 < p,
 * p = (|v| - lo) / (hi - lo).  Both sides of the comparison are exact. */
unsigned orc_encode_e2m1_sr(float v, unsigned u16)
{
    unsigned s = signbit(v) ? 0x8u : 0u;
    double a = fabs((double)v);
    if (a >= orc_decode_e2m1(7u))
        return s | 7u;
    unsigned lo = 0u;
    for (unsigned c = 0u; c <= 7u; ++c)
        if (orc_decode_e2m1(c) <= a)
            lo = c;
    double glo = orc_decode_e2m1(lo), ghi = orc_decode_e2m1(lo + 1u);
    if (a == glo)
        return s | lo;
    double p = (a - glo) / (ghi - glo);
    return s | (((double)(u16 & 0xffffu) < p * 65536.0) ? lo + 1u : lo);
}

/* Stochastic rounding onto the E4M3 grid: the same rule as E2M1 (round up
 * iff u16 * 2^-16 < p, p = (|v| - lo) / (hi - lo), lo <= |v| < hi adjacent
 * grid values, 0 and the subnormals included), saturating at 448.  The pages
 * attach stochastic rounding to the E2M1 route only ([FAF] 两个关键的数值技巧);
 * this is the same rule on the E4M3 grid.                                   */
unsigned orc_encode_e4m3_sr(float v, unsigned u16)
{
    unsigned s = signbit(v) ? 0x80u : 0u;
    double a = fabs((double)v);
    if (a >= orc_decode_e4m3(0x7eu))
        return s | 0x7eu;
    unsigned lo = 0u;
    for (unsigned c = 0u; c <= 0x7eu; ++c)
        if (orc_decode_e4m3(c) <= a)
            lo = c;
    double glo = orc_decode_e4m3(lo), ghi = orc_decode_e4m3(lo + 1u);
    if (a == glo)
        return s | lo;
    double p = (a - glo) / (ghi - glo);
    return s | (((double)(u16 & 0xffffu) < p * 65536.0) ? lo + 1u : lo);
}

/* ------------------------------------------------------------------------ */
/* Power-of-two block scales ([MOSS] Power-of-Two 的关键优势: dequantising  */
/* by 2^k is an exact exponent shift).  Returns e so that the block is      */
/* scaled by 2^-e and the E8M0 byte is e + 127, clamped to [-127, 127].     */
/*   FLOOR   : e = floor(log2 b) - emax (the MX-standard rule, [FAF]).      */
/*   CEIL    : smallest e with b * 2^-e <= Q (never saturates).             */
/*   NEAREST : e = round(log2(b / Q)), the rounding of [MOSS] 两级缩放实现. */
/* with Q = 448, emax = 8 for E4M3 and Q = 6, emax = 2 for E2M1.            */
/* ------------------------------------------------------------------------ */

static int floor_log2_pos(double b)
{
    int e;
    (void)frexp(b, &e); /* b = m * 2^e, m in [0.5, 1): exact */
    return e - 1;
}

int orc_pow2_exponent(float block_amax, int rule, int elem)
{
    double b = fabs((double)block_amax);
    double Q = (elem == ORC_ELEM_E4M3) ? 448.0 : 6.0;
    int emax = (elem == ORC_ELEM_E4M3) ? 8 : 2;
    if (b == 0.0)
        return 0;
    int e = 0;
    int fb = floor_log2_pos(b), fq = floor_log2_pos(Q);
    if (rule == ORC_RULE_FLOOR) {
        e = fb - emax;
    } else if (rule == ORC_RULE_CEIL) {
        e = fb - fq - 1; /* b * 2^-e > Q here; at most two increments follow */
        while (ldexp(b, -e) > Q)
            ++e;
    } else { /* NEAREST */
        int ep = fb - fq - 1; /* Q * 2^ep <= b holds here */
        while (ldexp(Q, ep + 1) <= b)
            ++ep;
        /* log2(b/Q) in [ep, ep+1): round up iff b^2 >= 2 Q^2 4^ep (exact in fp64) */
        e = ep + ((b * b >= 2.0 * Q * Q * ldexp(1.0, 2 * ep)) ? 1 : 0);
    }
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as  */
/* easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with    */
/* the paper's multipliers and Weyl key increments.                         */
/* ------------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
        uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)p1;
        uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The 16 random bits that decide element L (its linear index r*K + k in the
 * K-major output operand): one Philox block per 8 elements, counter
 * (L>>3 low word, L>>35, stream_id, 0), key (seed low word, seed high word);
 * element L takes 32-bit word (L&7)>>1, low half for even L, high for odd. */
unsigned orc_sr_u16(uint64_t seed, uint32_t stream_id, uint64_t L)
{
    uint32_t ctr[4] = {(uint32_t)(L >> 3), (uint32_t)(L >> 35), stream_id, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t w = out[(L & 7u) >> 1];
    return (L & 1u) ? (w >> 16) : (w & 0xffffu);
}

/* ------------------------------------------------------------------------ */
/* Fixed-sign 32-point Hadamard ([FAF] 两个关键的数值技巧): y = H32 x with   */
/* the unnormalised Sylvester matrix H[i][j] = (-1)^popcount(i & j) and no  */
/* random sign vector.  Computed in fp32 as five butterfly stages h = 1, 2, */
/* 4, 8, 16; each pair (j, j+h), j & h == 0, becomes (x_j + x_j+h,          */
/* x_j - x_j+h).  This fixes the fp32 rounding order.                       */
/* ------------------------------------------------------------------------ */

void orc_fwht32(float x[32])
{
    for (int h = 1; h < 32; h <<= 1)
        for (int j = 0; j < 32; ++j)
            if ((j & h) == 0) {
                float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout the tensor core reads ([FAF] 格式感知融合的设计思路: */
/* the producer writes the consumer's layout).  Logical scales [rows, kb]   */
/* are stored in 512-byte tiles of 128 rows x 4 k-blocks; tiles ordered by  */
/* row tile, then k-block group; inside a tile row r, block kb sits at      */
/* (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4.                           */
/* ------------------------------------------------------------------------ */

int64_t orc_sf_index(int64_t r, int64_t kb, int64_t kblocks)
{
    int64_t kgroups = (kblocks + 3) / 4;
    return ((r / 128) * kgroups + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4);
}

int64_t orc_sf_bytes(int64_t rows, int64_t kblocks)
{
    return ((rows + 127) / 128) * ((kblocks + 3) / 4) * 512;
}

void orc_sf_swizzle(const uint8_t* sf_logical, int64_t rows, int64_t kblocks, uint8_t* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t kb = 0; kb < kblocks; ++kb)
            out[orc_sf_index(r, kb, kblocks)] = sf_logical[r * kblocks + kb];
}

/* ------------------------------------------------------------------------ */
/* Quantizer                                                                */
/* ------------------------------------------------------------------------ */

float orc_amax_bf16(const uint16_t* x, int64_t R, int64_t C, int64_t ld)
{
    float m = 0.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float a = fabsf(orc_bf16_to_f32(x[r * ld + c]));
            if (a > m)
                m = a;
        }
    return m;
}

static int fmt_elem(int fmt)
{
    return (fmt == ORC_FMT_MXFP8 || fmt == ORC_FMT_MOSS) ? ORC_ELEM_E4M3 : ORC_ELEM_E2M1;
}

static int fmt_block(int fmt) { return (fmt == ORC_FMT_NVFP4 || fmt == ORC_FMT_NVFP4_LOCAL) ? 16 : 32; }
static int fmt_is_nvfp4(int fmt) { return fmt == ORC_FMT_NVFP4 || fmt == ORC_FMT_NVFP4_LOCAL; }

static unsigned encode_elem(float s, int elem, int rounding, unsigned u16)
{
    if (elem == ORC_ELEM_E4M3)
        return rounding == ORC_ROUND_SR ? orc_encode_e4m3_sr(s, u16) : orc_encode_e4m3_rne(s);
    return rounding == ORC_ROUND_SR ? orc_encode_e2m1_sr(s, u16) : orc_encode_e2m1_rne(s);
}

static void put_code(uint8_t* codes, int64_t r, int64_t k, int64_t K, int elem, unsigned c)
{
    if (elem == ORC_ELEM_E4M3) {
        codes[r * K + k] = (uint8_t)c;
    } else {
        uint8_t* p = &codes[r * (K / 2) + k / 2];
        if ((k & 1) == 0)
            *p = (uint8_t)((*p & 0xf0u) | (c & 0xfu));
        else
            *p = (uint8_t)((*p & 0x0fu) | ((c & 0xfu) << 4));
    }
}

/* Quantize a bf16 matrix x [R, C] (row stride ld elements) into a K-major
 * operand.  ROWWISE: operand rows = R, K = C.  COLWISE: quantize along dim 0,
 * operand rows = C, K = R (element (r, k) of the operand is x[k, r]).
 *
 * Per block of B consecutive operand elements along K (B = 32 for MXFP8,
 * MXFP4 and MOSS; 16 for NVFP4):
 *   MXFP8 / MXFP4: y = H32 x (if hadamard), e = rule(max|y|), default FLOOR,
 *     code = cast(fl32(y * 2^-e)), scale byte e + 127.
 *   MOSS ([MOSS] 创新 1 and 两级缩放实现): s_t = fl32(amax / 448);
 *     y = fl32(x / s_t); e = rule(max|y|), default CEIL (the smallest
 *     power-of-two micro scale that avoids overflow); code = E4M3(fl32(y*2^-e)).
 *   NVFP4 (block scaling with a per-block scale and a global tensor scale,
 *     [FAF] FP4加速为何常常"纸上富贵" and 格式感知融合的设计思路):
 *     s_t = fl32(amax / (448 * 6)); sb = UE4M3_rne(fl32(b / fl32(6 * s_t)));
 *     d = fl32(dec(sb) * s_t); code = E2M1(fl32(x / d)), or sign-kept zero
 *     when d == 0.  With hadamard, every 32 consecutive operand elements
 *     along K (two scale blocks) are first replaced by y = H32 x, and amax is
 *     max |y| over the whole transformed operand ([FAF] 两个关键的数值技巧
 *     puts the transform before quantization; the tensor scale must then
 *     cover the transformed values, which can exceed max |x|).
 *   The tensor scale is 1 when amax == 0.
 * cast: RNE (E4M3 or E2M1) or stochastic rounding (E2M1 only) with the bits
 * of orc_sr_u16 for element index L = r*K + k.
 * Outputs: codes [rows, K] (E4M3 one byte; E2M1 two per byte, even k in the
 * low nibble), sf_logical [rows, K/B], amax_out and tensor_scale_out (either
 * may be NULL; the tensor scale is written for MOSS and NVFP4 only).         */
int orc_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int dir, int fmt,
                 int block, int rounding, int rule, uint64_t seed, uint32_t stream_id,
                 int hadamard, const float* amax_in, uint8_t* codes, uint8_t* sf_logical,
                 float* amax_out, float* tensor_scale_out)
{
    if (!x || !codes || !sf_logical || R < 0 || C < 0 || ld < C)
        return ORC_ERR_ARG;
    if (fmt < ORC_FMT_MXFP8 || fmt > ORC_FMT_NVFP4_LOCAL || (dir != ORC_ROWWISE && dir != ORC_COLWISE))
        return ORC_ERR_ARG;
    if (block != fmt_block(fmt))
        return ORC_ERR_UNSUPPORTED;
    const int elem = fmt_elem(fmt);
    if (hadamard && !(fmt == ORC_FMT_MXFP8 || fmt == ORC_FMT_MXFP4 || fmt == ORC_FMT_NVFP4))
        return ORC_ERR_UNSUPPORTED;
    if (fmt_is_nvfp4(fmt) && rule != ORC_RULE_DEFAULT)
        return ORC_ERR_UNSUPPORTED; /* NVFP4 block scales are E4M3, not powers of two */
    if (rule == ORC_RULE_DEFAULT)
        rule = (fmt == ORC_FMT_MOSS) ? ORC_RULE_CEIL : ORC_RULE_FLOOR;
    const int64_t rows = (dir == ORC_ROWWISE) ? R : C;
    const int64_t K = (dir == ORC_ROWWISE) ? C : R;
    if (K % block != 0 || (hadamard && K % 32 != 0))
        return ORC_ERR_ARG;
    const int64_t kblocks = K / block;
    /* Elements transformed together along K: 32 with the Hadamard transform
     * (one MX block, two NVFP4 blocks), else one scale block. */
    const int group = hadamard ? 32 : block;

    /* Tensor scales.  One per tensor, except ORC_FMT_NVFP4_LOCAL: one per
     * region of ORC_LOCAL_REGION consecutive operand rows (all of K), the
     * scale domain of the producer that writes that region ([FAF]
     * 格式感知融合的设计思路: "CTA-local" nvfp), amax and tensor scale then
     * being arrays of ceil(rows / ORC_LOCAL_REGION) entries.                 */
    const int local = fmt == ORC_FMT_NVFP4_LOCAL;
    const int64_t nreg = local ? (rows + ORC_LOCAL_REGION - 1) / ORC_LOCAL_REGION : 1;
    float* amaxv = (float*)calloc((size_t)(nreg > 0 ? nreg : 1), sizeof(float));
    float* tsv = (float*)malloc(sizeof(float) * (size_t)(nreg > 0 ? nreg : 1));
    if (!amaxv || !tsv) {
        free(amaxv);
        free(tsv);
        return ORC_ERR_ARG;
    }
    if (local) {
        for (int64_t g = 0; g < nreg; ++g) {
            if (amax_in) {
                amaxv[g] = amax_in[g];
                continue;
            }
            float m = 0.0f;
            const int64_t r1 = (g + 1) * ORC_LOCAL_REGION < rows ? (g + 1) * ORC_LOCAL_REGION : rows;
            for (int64_t rr = g * ORC_LOCAL_REGION; rr < r1; ++rr)
                for (int64_t k = 0; k < K; ++k) {
                    float v = fabsf(orc_bf16_to_f32((dir == ORC_ROWWISE) ? x[rr * ld + k] : x[k * ld + rr]));
                    if (v > m)
                        m = v;
                }
            amaxv[g] = m;
        }
    } else if (fmt == ORC_FMT_NVFP4 && hadamard && !amax_in) {
        /* max |H32 x| over every 32-element group of the operand along K */
        float m = 0.0f;
        for (int64_t rr = 0; rr < rows; ++rr)
            for (int64_t k0 = 0; k0 < K; k0 += 32) {
                float y[32];
                for (int i = 0; i < 32; ++i)
                    y[i] = orc_bf16_to_f32((dir == ORC_ROWWISE) ? x[rr * ld + k0 + i] : x[(k0 + i) * ld + rr]);
                orc_fwht32(y);
                for (int i = 0; i < 32; ++i)
                    if (fabsf(y[i]) > m)
                        m = fabsf(y[i]);
            }
        amaxv[0] = m;
    } else if (fmt == ORC_FMT_MOSS || fmt == ORC_FMT_NVFP4 || amax_out) {
        amaxv[0] = amax_in ? *amax_in : orc_amax_bf16(x, R, C, ld);
    }
    for (int64_t g = 0; g < (nreg > 0 ? nreg : 1); ++g) {
        float ts = 1.0f;
        if (fmt == ORC_FMT_MOSS && amaxv[g] != 0.0f)
            ts = amaxv[g] / 448.0f;
        if (fmt_is_nvfp4(fmt) && amaxv[g] != 0.0f)
            ts = amaxv[g] / 2688.0f;
        tsv[g] = ts;
        if (amax_out && (local || g == 0))
            amax_out[g] = amaxv[g];
        if (tensor_scale_out && (fmt == ORC_FMT_MOSS || fmt_is_nvfp4(fmt)) && (local || g == 0))
            tensor_scale_out[g] = ts;
    }

    int64_t r;
#pragma omp parallel for schedule(dynamic, 16)
    for (r = 0; r < rows; ++r) {
        float yg[32];
        for (int64_t kb = 0; kb < kblocks; ++kb) {
            const int64_t k0 = kb * block;
            if (k0 % group == 0) { /* load (and transform) the next group */
                for (int i = 0; i < group; ++i) {
                    int64_t k = k0 + i;
                    uint16_t h = (dir == ORC_ROWWISE) ? x[r * ld + k] : x[k * ld + r];
                    yg[i] = orc_bf16_to_f32(h);
                }
                if (hadamard)
                    orc_fwht32(yg);
            }
            float y[32];
            for (int i = 0; i < block; ++i)
                y[i] = yg[k0 % group + i];
            const float ts = tsv[local ? r / ORC_LOCAL_REGION : 0];
            const float nv_denom = 6.0f * ts;
            if (fmt == ORC_FMT_MOSS)
                for (int i = 0; i < block; ++i)
                    y[i] = y[i] / ts;
            float b = 0.0f;
            for (int i = 0; i < block; ++i)
                if (fabsf(y[i]) > b)
                    b = fabsf(y[i]);
            uint8_t sfb;
            if (fmt_is_nvfp4(fmt)) {
                unsigned sb = orc_encode_e4m3_rne(b / nv_denom); /* b >= 0: sign bit 0 */
                float d = (float)orc_decode_e4m3(sb) * ts;
                for (int i = 0; i < block; ++i) {
                    int64_t k = k0 + i;
                    unsigned c;
                    if (d == 0.0f) {
                        c = signbit(y[i]) ? 0x8u : 0u;
                    } else {
                        unsigned u = (rounding == ORC_ROUND_SR)
                                         ? orc_sr_u16(seed, stream_id, (uint64_t)(r * K + k)) : 0u;
                        c = encode_elem(y[i] / d, elem, rounding, u);
                    }
                    put_code(codes, r, k, K, elem, c);
                }
                sfb = (uint8_t)sb;
            } else {
                int e = orc_pow2_exponent(b, rule, elem);
                float s2 = ldexpf(1.0f, -e);
                for (int i = 0; i < block; ++i) {
                    int64_t k = k0 + i;
                    unsigned u = (rounding == ORC_ROUND_SR)
                                     ? orc_sr_u16(seed, stream_id, (uint64_t)(r * K + k)) : 0u;
                    put_code(codes, r, k, K, elem, encode_elem(y[i] * s2, elem, rounding, u));
                }
                sfb = (uint8_t)(e + 127);
            }
            sf_logical[r * kblocks + kb] = sfb;
        }
    }
    free(amaxv);
    free(tsv);
    return ORC_OK;
}

/* Rowwise MX quantization of an fp32 matrix x [R, C] (row stride ld): the
 * MXFP8 / MXFP4 steps of orc_quantize (FLOOR rule, round-to-nearest-even)
 * applied to fp32 values instead of bf16 ones: per block of 32 consecutive
 * elements of a row, e = FLOOR(max|y|), code = cast(fl32(y * 2^-e)), scale byte
 * e + 127.  This is what a GEMM epilogue that emits the next layer's operand
 * ([FAF] 格式感知融合的设计思路: the producer writes the consumer's layout)
 * must produce from its fp32 output.                                        */
int orc_quantize_rows_f32(const float* x, int64_t R, int64_t C, int64_t ld, int fmt,
                          uint8_t* codes, uint8_t* sf_logical)
{
    if (!x || !codes || !sf_logical || R < 0 || C < 0 || ld < C)
        return ORC_ERR_ARG;
    if (fmt != ORC_FMT_MXFP8 && fmt != ORC_FMT_MXFP4)
        return ORC_ERR_UNSUPPORTED;
    if (C % 32 != 0)
        return ORC_ERR_ARG;
    const int elem = fmt_elem(fmt);
    const int64_t kblocks = C / 32;
    int64_t r;
#pragma omp parallel for schedule(dynamic, 16)
    for (r = 0; r < R; ++r) {
        for (int64_t kb = 0; kb < kblocks; ++kb) {
            const float* y = x + r * ld + kb * 32;
            float b = 0.0f;
            for (int i = 0; i < 32; ++i)
                if (fabsf(y[i]) > b)
                    b = fabsf(y[i]);
            const int e = orc_pow2_exponent(b, ORC_RULE_FLOOR, elem);
            const float s2 = ldexpf(1.0f, -e);
            for (int i = 0; i < 32; ++i)
                put_code(codes, r, kb * 32 + i, C, elem, encode_elem(y[i] * s2, elem, ORC_ROUND_RNE, 0u));
            sf_logical[r * kblocks + kb] = (uint8_t)(e + 127);
        }
    }
    return ORC_OK;
}

static double dec_code(const uint8_t* codes, int64_t r, int64_t k, int64_t K, int elem)
{
    if (elem == ORC_ELEM_E4M3)
        return orc_decode_e4m3(codes[r * K + k]);
    uint8_t byte = codes[r * (K / 2) + k / 2];
    return orc_decode_e2m1((k & 1) ? (byte >> 4) : (byte & 0xfu));
}

static double dec_sf(uint8_t s, int fmt)
{
    return fmt_is_nvfp4(fmt) ? orc_decode_e4m3(s) : orc_decode_e8m0(s);
}

/* out[r, k] = dec(code) * dec(block scale), exact in fp64 (no tensor scale). */
void orc_dequantize(const uint8_t* codes, const uint8_t* sf_logical, int64_t rows, int64_t k,
                    int fmt, int block, double* out)
{
    const int elem = fmt_elem(fmt);
    const int64_t kblocks = k / block;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < k; ++j)
            out[r * k + j] = dec_code(codes, r, j, k, elem) * dec_sf(sf_logical[r * kblocks + j / block], fmt);
}

/* Epilogue factor ([MOSS] GEMM Kernel 优化: dequantise once, after the main
 * loop): alpha = fl32(fl32(s_tA * s_tB) * extra); a missing tensor scale is 1. */
float orc_gemm_alpha(const float* ts_a, const float* ts_b, float extra)
{
    float a = ts_a ? *ts_a : 1.0f, b = ts_b ? *ts_b : 1.0f;
    float ab = a * b;
    return ab * extra;
}

/* C[i, j] = alpha * sum_k dq(A)[rows[i], k] * dq(B)[cols[j], k], accumulated
 * in fp64 over the dequantised operands; Cabs is the same with |.| on every
 * product (the scale of the rounding-error bound).  rows/cols NULL = all. */
void orc_gemm_q(const uint8_t* a_codes, const uint8_t* a_sf, const uint8_t* b_codes,
                const uint8_t* b_sf, int fmt, int block, int64_t M, int64_t N, int64_t K,
                double alpha, const int64_t* rows, int64_t nrows, const int64_t* cols,
                int64_t ncols, double* C, double* Cabs)
{
    const int elem = fmt_elem(fmt);
    const int64_t kblocks = K / block;
    if (!rows)
        nrows = M;
    if (!cols)
        ncols = N;
    double* bq = (double*)malloc(sizeof(double) * (size_t)(ncols * K));
    if (!bq)
        return;
    int64_t jj;
#pragma omp parallel for schedule(static)
    for (jj = 0; jj < ncols; ++jj) {
        int64_t j = cols ? cols[jj] : jj;
        for (int64_t k = 0; k < K; ++k)
            bq[jj * K + k] = dec_code(b_codes, j, k, K, elem) * dec_sf(b_sf[j * kblocks + k / block], fmt);
    }
    int64_t ii;
#pragma omp parallel for schedule(dynamic, 4)
    for (ii = 0; ii < nrows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        double* aq = (double*)malloc(sizeof(double) * (size_t)K);
        if (!aq)
            continue;
        for (int64_t k = 0; k < K; ++k)
            aq[k] = dec_code(a_codes, i, k, K, elem) * dec_sf(a_sf[i * kblocks + k / block], fmt);
        for (int64_t j2 = 0; j2 < ncols; ++j2) {
            const double* bj = bq + j2 * K;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = aq[k] * bj[k];
                s += p;
                sa += fabs(p);
            }
            C[ii * ncols + j2] = alpha * s;
            if (Cabs)
                Cabs[ii * ncols + j2] = fabs(alpha) * sa;
        }
        free(aq);
    }
    free(bq);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
