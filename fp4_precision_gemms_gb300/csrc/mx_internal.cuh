// mx_internal.cuh -- declarations shared by the library's translation units.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "mx.h"

namespace mx {

// Element encodings and block sizes per format.
__host__ __device__ constexpr bool fmt_is_nvfp4(int fmt) { return fmt == MX_FMT_NVFP4 || fmt == MX_FMT_NVFP4_LOCAL; }
__host__ __device__ constexpr bool fmt_is_fp4(int fmt) { return fmt == MX_FMT_MXFP4_E2M1 || fmt_is_nvfp4(fmt); }
__host__ __device__ constexpr int fmt_block(int fmt) { return fmt_is_nvfp4(fmt) ? 16 : 32; }
__host__ __device__ constexpr bool fmt_has_tensor_scale(int fmt) { return fmt_is_nvfp4(fmt) || fmt == MX_FMT_MOSS_FP8; }
__host__ __device__ constexpr bool fmt_is_local(int fmt) { return fmt == MX_FMT_NVFP4_LOCAL; }
constexpr int kLocalRegion = MX_LOCAL_REGION;  // operand rows per FP32 scale (NVFP4_LOCAL)
__host__ __device__ inline int64_t scale_count(int fmt, int64_t rows)
{
    return fmt_is_local(fmt) ? (rows > 0 ? (rows + kLocalRegion - 1) / kLocalRegion : 1) : (fmt_has_tensor_scale(fmt) ? 1 : 0);
}

// Scale-factor layout of the tensor core: 512-byte tiles of 128 rows x 4 K-blocks.
__host__ __device__ inline int64_t sf_kgroups(int64_t kblocks) { return (kblocks + 3) / 4; }
__host__ __device__ inline int64_t sf_layout_bytes(int64_t rows, int64_t kblocks)
{
    return ((rows + 127) / 128) * sf_kgroups(kblocks) * 512;
}
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t kb, int64_t kgroups)
{
    return ((r >> 7) * kgroups + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

struct Device {
    int id = -1;
    int sms = 0;
    int* status = nullptr;  // device address of the per-device status word
};

// Current device after checking it is an sm_103 part; MX_OK or an error.
int current_device(Device* d);

// Default bound on every device-side wait (ns).  Healthy waits are microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct QuantArgs {
    const uint16_t* x;
    int64_t R, C, ld;
    int dir, fmt, rounding, rule, hadamard;
    uint64_t seed;
    uint32_t stream_id;
    const float* amax;     // device: tensor amax (NVFP4/MOSS), already final
    float* tensor_scale;   // device output (NVFP4/MOSS)
    uint8_t* codes;
    uint8_t* sf;
};

// One producer pass over x emitting the rowwise operand, the colwise operand or
// both (a null codes pointer skips that direction).
struct TileArgs {
    const void* x;
    int64_t R, C;
    int fmt, rule;
    uint64_t seed;
    uint32_t stream_id;
    const float* amax;
    float* tensor_scale;
    float* amax_copy;          // optional second amax / tensor-scale destination
    float* tensor_scale_copy;  // (the colwise operand of a dual pass)
    uint8_t* row_codes;
    uint8_t* row_sf;
    int row_sr, row_had;
    uint8_t* col_codes;
    uint8_t* col_sf;
    int col_sr, col_had;
    int* status;
    uint64_t wait_ns;
    // NVFP4_LOCAL: tensor-scale arrays of the rowwise and colwise operands, one
    // entry per 128 operand rows (rows of x for the rowwise operand, columns of
    // x for the colwise one).
    const float* row_ts_v;
    const float* col_ts_v;
    // set by the launcher: 1 when the codes leave through TMA tensor stores
    int tma_st;
    // test hook: on this tile (of each CTA) the CTA's last thread gives up its
    // stage wait as if its limit had run out; -1 never
    int64_t fail_at;
};

// Number of kernels this library has launched in the process.
extern std::atomic<uint64_t> g_kernel_launches;
inline void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

int launch_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax, const Device& d,
                cudaStream_t s);
// Tensor amax of the Hadamard-transformed operand of x along `dir` (max |H32 y|
// over every 32 consecutive operand elements along K); C % 32 == 0 rowwise,
// R % 32 == 0 colwise.
int launch_had_amax(const void* x, int64_t R, int64_t C, int64_t ld, int dir, float* amax, const Device& d,
                    cudaStream_t s);
// NVFP4_LOCAL region maxima of bf16 x [R, C]: amax_rows[g] = max |x| over rows
// 128 g .. 128 g + 127, amax_cols[g] over columns 128 g .. (either may be null).
int launch_region_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax_rows, float* amax_cols,
                       const Device& d, cudaStream_t s);
// NVFP4_LOCAL tensor scales: ts[g] = fl32(amax[g] / 2688), or 1 where amax[g] == 0.
int launch_local_scales(const float* amax, float* ts, int64_t n, const Device& d, cudaStream_t s);
int launch_quantize(const QuantArgs& q, const Device& d, cudaStream_t s);
int launch_quantize_tile(const TileArgs& t, int64_t ld, const Device& d, cudaStream_t s);
int launch_dequantize(const mx_tensor* A, float* out, const Device& d, cudaStream_t s);
// out_mode: MX_OUT_F32 / MX_OUT_BF16 into C (row stride ldc elements), or 2 / 3
// for C quantized in the epilogue into the rowwise MXFP8 / MXFP4 operand
// (codes at C, row stride ldc bytes; E8M0 scales at q_sf in the tensor-core
// layout; N % 32 == 0).  amax_out (F32 / BF16 output only): max |C| as
// written, reduced into the fp32 bit pattern there (the caller zeroes it).
int launch_gemm(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc, int out_mode,
                const Device& d, cudaStream_t s, uint8_t* q_sf = nullptr, unsigned* amax_out = nullptr);
int launch_wait_selftest(uint64_t limit_ns, const Device& d, cudaStream_t s);
int launch_divide_check(const float* v, const float* dv, int64_t n, float* fast, float* ieee, const Device& d,
                        cudaStream_t s);

}  // namespace mx
