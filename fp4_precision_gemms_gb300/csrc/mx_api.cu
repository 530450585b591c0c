// mx_api.cu -- the extern "C" entry points declared in include/mx.h: argument
// validation on the host, the per-device status word, and the composition of
// quantize + GEMM into a linear layer's forward, data-gradient and
// weight-gradient passes.
#include <cstring>
#include <mutex>

#include "mx_internal.cuh"

namespace mx {

// Per-device status word written by kernels whose bounded waits give up.
__device__ int g_status_word;

std::atomic<uint64_t> g_kernel_launches{0};

void set_gemm_variant(int v);
int last_gemm_variant();

int current_device(Device* d)
{
    static std::mutex mu;
    static Device cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return MX_ERR_NO_DEVICE;
    }
    if (dev >= 64)
        return MX_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].id == dev) {
        *d = cache[dev];
        return MX_OK;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MX_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3)
        return MX_ERR_UNSUPPORTED;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&status, g_status_word) != cudaSuccess)
        return MX_ERR_CUDA;
    cache[dev].id = dev;
    cache[dev].sms = sms;
    cache[dev].status = static_cast<int*>(status);
    *d = cache[dev];
    return MX_OK;
}

}  // namespace mx

using namespace mx;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_fmt(int fmt) { return fmt >= MX_FMT_MXFP8_E4M3 && fmt <= MX_FMT_NVFP4_LOCAL; }

int64_t codes_row_bytes(int fmt, int64_t k) { return fmt_is_fp4(fmt) ? k / 2 : k; }

// K granularity the GEMM consumes per pipeline stage.
int64_t gemm_k_multiple(int fmt) { return fmt_is_fp4(fmt) ? 256 : 128; }

int check_operand(const mx_tensor* t)
{
    if (!t || !valid_fmt(t->fmt) || t->rows < 0 || t->k < 0 || t->block != fmt_block(t->fmt))
        return MX_ERR_INVALID_ARG;
    if ((t->rows > 0 && t->k > 0) && (!t->codes || !t->sf))
        return MX_ERR_INVALID_ARG;
    if (fmt_has_tensor_scale(t->fmt) && !t->tensor_scale)
        return MX_ERR_INVALID_ARG;
    if (!aligned16(t->codes) || !aligned16(t->sf))
        return MX_ERR_ALIGNMENT;
    return MX_OK;
}

struct Operand {  // an mx_tensor carved out of a workspace
    mx_tensor t;
};

// Carves the buffers of one quantized operand out of `ws` (256-byte aligned
// pieces); returns the bytes used.  With ws == NULL only counts.
size_t carve(uint8_t* ws, int fmt, int64_t rows, int64_t k, mx_tensor* t)
{
    size_t off = 0;
    const size_t cb = round_up(mx_codes_bytes(fmt, rows, k), 256);
    const size_t sb = round_up(mx_sf_bytes(fmt, rows, k), 256);
    const size_t nb = round_up(sizeof(float) * std::max<int64_t>(scale_count(fmt, rows), 1), 128);
    if (t) {
        std::memset(t, 0, sizeof *t);
        t->codes = ws ? ws + off : nullptr;
        t->sf = ws ? ws + off + cb : nullptr;
        t->amax = ws ? reinterpret_cast<float*>(ws + off + cb + sb) : nullptr;
        t->tensor_scale = ws ? reinterpret_cast<float*>(ws + off + cb + sb + nb) : nullptr;
    }
    off += cb + sb + 2 * nb;
    return off;
}

// Producer implementation for tests and tuning: 0 automatic (direct loads
// rowwise, tile producer colwise), 1 direct loads, 2 tile producer.  Per host
// thread, like the GEMM variant override.
thread_local int g_quant_impl = 0;
thread_local int64_t g_tile_fail_at = -1;  // test hook: tile producer's forced wait failure

// The backward calls' gradient fork: with both gradients requested, the weight
// gradient runs on a side stream while the data gradient runs on the caller's
// stream, joined back by events (in graph capture these become the graph's
// fork and join edges), so each GEMM's last partial wave leaves SMs to the
// other.  One non-blocking side stream and two events per host thread and
// device, created on first use outside capture; a call captured before they
// exist runs on the caller's stream alone.  The results do not depend on it.
struct BwdFork {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool failed = false;
};
constexpr int kForkDevices = 64;
thread_local BwdFork g_fork[kForkDevices];
thread_local int g_bwd_fork = 1;

// A side stream whose next work follows everything issued to s so far, or
// nullptr (run on s).  Leaves no CUDA error behind either way.
cudaStream_t fork_begin(const Device& d, cudaStream_t s)
{
    if (!g_bwd_fork || d.id < 0 || d.id >= kForkDevices)
        return nullptr;
    BwdFork& f = g_fork[d.id];
    if (!f.side) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (f.failed || cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            (void)cudaGetLastError();
            return nullptr;
        }
        cudaStream_t side = nullptr;
        if (cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            if (side)  // release whatever was made; this thread runs on s from now on
                (void)cudaStreamDestroy(side);
            if (f.fork)
                (void)cudaEventDestroy(f.fork);
            if (f.join)
                (void)cudaEventDestroy(f.join);
            f.fork = f.join = nullptr;
            f.failed = true;
            return nullptr;
        }
        f.side = side;
    }
    if (cudaEventRecord(f.fork, s) != cudaSuccess || cudaStreamWaitEvent(f.side, f.fork, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return f.side;
}

// Makes s wait for everything issued to the side stream.
int fork_end(const Device& d, cudaStream_t side, cudaStream_t s)
{
    BwdFork& f = g_fork[d.id];
    return cudaEventRecord(f.join, side) == cudaSuccess && cudaStreamWaitEvent(s, f.join, 0) == cudaSuccess
               ? MX_OK
               : MX_ERR_CUDA;
}

// Shared argument checks of the single and dual producers.
int check_quantize_args(const void* x, int64_t R, int64_t C, int64_t ld, int fmt, int block, int rule)
{
    if (!valid_fmt(fmt) || R < 0 || C < 0 || ld < C)
        return MX_ERR_INVALID_ARG;
    if (rule < MX_SCALE_DEFAULT || rule > MX_SCALE_NEAREST)
        return MX_ERR_INVALID_ARG;
    if (block != fmt_block(fmt))
        return MX_ERR_UNSUPPORTED;
    if (fmt == MX_FMT_NVFP4 && rule != MX_SCALE_DEFAULT)
        return MX_ERR_UNSUPPORTED;
    if (ld % 8 != 0 || !aligned16(x))
        return MX_ERR_ALIGNMENT;
    if (R > 0 && C > 0 && !x)
        return MX_ERR_INVALID_ARG;
    return MX_OK;
}

int check_direction(int fmt, int rounding, int hadamard)
{
    if (rounding != MX_ROUND_RNE && rounding != MX_ROUND_SR)
        return MX_ERR_INVALID_ARG;
    if (hadamard && !(fmt == MX_FMT_MXFP8_E4M3 || fmt == MX_FMT_MXFP4_E2M1 || fmt == MX_FMT_NVFP4))
        return MX_ERR_UNSUPPORTED;
    return MX_OK;
}

int check_output(const mx_tensor* out, int fmt, int64_t R, int64_t C)
{
    if (!out)
        return MX_ERR_INVALID_ARG;
    if (!aligned16(out->codes))
        return MX_ERR_ALIGNMENT;
    if (R > 0 && C > 0 && (!out->codes || !out->sf))
        return MX_ERR_INVALID_ARG;
    if (fmt_has_tensor_scale(fmt) && (!out->amax || !out->tensor_scale))
        return MX_ERR_INVALID_ARG;
    return MX_OK;
}

void fill_meta(mx_tensor* out, int64_t rows, int64_t k, int fmt, int hadamard)
{
    out->rows = rows;
    out->k = k;
    out->fmt = fmt;
    out->block = fmt_block(fmt);
    out->hadamard = hadamard ? 1 : 0;
}

// Makes out->amax hold max|x| (copied from amax_in or reduced from x).
int prepare_amax(const void* x, int64_t R, int64_t C, int64_t ld, const float* amax_in, mx_tensor* out, int dir,
                 const Device& d, cudaStream_t s)
{
    if (fmt_is_local(out->fmt)) {  // region maxima of the operand's rows, then the scales
        const int64_t n = scale_count(out->fmt, out->rows);
        int rc = MX_OK;
        if (amax_in) {
            if (amax_in != out->amax && cudaMemcpyAsync(out->amax, amax_in, sizeof(float) * n,
                                                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
                return MX_ERR_CUDA;
        } else {
            const bool rowwise = dir == MX_ROWWISE;
            rc = launch_region_amax(x, R, C, ld, rowwise ? out->amax : nullptr, rowwise ? nullptr : out->amax, d, s);
        }
        return rc != MX_OK ? rc : launch_local_scales(out->amax, out->tensor_scale, n, d, s);
    }
    if (amax_in) {
        if (amax_in != out->amax &&
            cudaMemcpyAsync(out->amax, amax_in, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return MX_ERR_CUDA;
        return MX_OK;
    }
    if (out->hadamard)  // the tensor scale covers the transformed values
        return launch_had_amax(x, R, C, ld, dir, out->amax, d, s);
    return launch_amax(x, R, C, ld, out->amax, d, s);
}

int set_unit_scale(mx_tensor* out, cudaStream_t s)
{
    static const float one = 1.0f;  // the tensor scale of an empty tensor
    return cudaMemcpyAsync(out->tensor_scale, &one, sizeof one, cudaMemcpyHostToDevice, s) == cudaSuccess ? MX_OK
                                                                                                        : MX_ERR_CUDA;
}

int quantize_impl(const void* x, int64_t R, int64_t C, int64_t ld, int dir, int fmt, int block, int rounding,
                  int rule, uint64_t seed, uint32_t stream_id, int hadamard, const float* amax_in, mx_tensor* out,
                  const Device& d, cudaStream_t s)
{
    if (dir != MX_ROWWISE && dir != MX_COLWISE)
        return MX_ERR_INVALID_ARG;
    int rc = check_quantize_args(x, R, C, ld, fmt, block, rule);
    if (rc == MX_OK)
        rc = check_direction(fmt, rounding, hadamard);
    if (rc == MX_OK)
        rc = check_output(out, fmt, R, C);
    if (rc != MX_OK)
        return rc;
    const int64_t rows = dir == MX_ROWWISE ? R : C;
    const int64_t k = dir == MX_ROWWISE ? C : R;
    if (k % block != 0 || (dir == MX_COLWISE && R % 32 != 0) || (hadamard && k % 32 != 0))
        return MX_ERR_ALIGNMENT;
    if (rule == MX_SCALE_DEFAULT)
        rule = fmt == MX_FMT_MOSS_FP8 ? MX_SCALE_CEIL : MX_SCALE_FLOOR;
    fill_meta(out, rows, k, fmt, hadamard);
    const bool ts = fmt_has_tensor_scale(fmt);
    if (ts && (rc = prepare_amax(x, R, C, ld, amax_in, out, dir, d, s)) != MX_OK)
        return rc;
    if (R == 0 || C == 0)
        return (ts && !fmt_is_local(fmt)) ? set_unit_scale(out, s) : MX_OK;
    // The tile producer is the automatic choice in both directions (measured
    // faster than the direct producers for rowwise passes as well).  The direct
    // producers have no region scales: NVFP4_LOCAL always takes the tile
    // producer; the tile producer has no NVFP4 transform: NVFP4 with the
    // Hadamard transform always takes the direct producers.
    const bool nv_had = fmt == MX_FMT_NVFP4 && hadamard;
    const bool tile = (g_quant_impl != 1 || fmt_is_local(fmt)) && !nv_had;
    if (tile) {
        TileArgs t = {};
        t.x = x;
        t.R = R;
        t.C = C;
        t.fmt = fmt;
        t.rule = rule;
        t.seed = seed;
        t.stream_id = stream_id;
        t.amax = out->amax;
        t.tensor_scale = out->tensor_scale;
        (dir == MX_ROWWISE ? t.row_ts_v : t.col_ts_v) = out->tensor_scale;
        uint8_t* codes = static_cast<uint8_t*>(out->codes);
        if (dir == MX_ROWWISE) {
            t.row_codes = codes;
            t.row_sf = out->sf;
            t.row_sr = rounding == MX_ROUND_SR;
            t.row_had = hadamard ? 1 : 0;
        } else {
            t.col_codes = codes;
            t.col_sf = out->sf;
            t.col_sr = rounding == MX_ROUND_SR;
            t.col_had = hadamard ? 1 : 0;
        }
        t.status = d.status;
        t.wait_ns = kWaitLimitNs;
        t.fail_at = g_tile_fail_at;
        return launch_quantize_tile(t, ld, d, s);
    }
    QuantArgs q;
    q.x = static_cast<const uint16_t*>(x);
    q.R = R;
    q.C = C;
    q.ld = ld;
    q.dir = dir;
    q.fmt = fmt;
    q.rounding = rounding;
    q.rule = rule;
    q.hadamard = hadamard ? 1 : 0;
    q.seed = seed;
    q.stream_id = stream_id;
    q.amax = out->amax;
    q.tensor_scale = out->tensor_scale;
    q.codes = static_cast<uint8_t*>(out->codes);
    q.sf = out->sf;
    return launch_quantize(q, d, s);
}

int quantize_dual_impl(const void* x, int64_t R, int64_t C, int64_t ld, int fmt, int block, int rule,
                       uint64_t seed, uint32_t stream_id, int row_rounding, int row_hadamard, int col_rounding,
                       int col_hadamard, const float* amax_in, mx_tensor* row_out, mx_tensor* col_out,
                       const Device& d, cudaStream_t s)
{
    int rc = check_quantize_args(x, R, C, ld, fmt, block, rule);
    if (rc == MX_OK)
        rc = check_direction(fmt, row_rounding, row_hadamard);
    if (rc == MX_OK)
        rc = check_direction(fmt, col_rounding, col_hadamard);
    if (rc == MX_OK)
        rc = check_output(row_out, fmt, R, C);
    if (rc == MX_OK)
        rc = check_output(col_out, fmt, R, C);
    if (rc != MX_OK)
        return rc;
    if (C % block != 0 || R % 32 != 0)
        return MX_ERR_ALIGNMENT;
    if (fmt == MX_FMT_NVFP4 && (row_hadamard || col_hadamard)) {
        // A transformed direction has a tensor amax of its own (that of its
        // transformed values), so the two operands get separate scales, each
        // from its own pass over x; one caller amax cannot serve both.
        if (amax_in)
            return MX_ERR_UNSUPPORTED;
        rc = quantize_impl(x, R, C, ld, MX_ROWWISE, fmt, block, row_rounding, rule, seed, stream_id, row_hadamard,
                           nullptr, row_out, d, s);
        if (rc != MX_OK)
            return rc;
        return quantize_impl(x, R, C, ld, MX_COLWISE, fmt, block, col_rounding, rule, seed, stream_id, col_hadamard,
                             nullptr, col_out, d, s);
    }
    if (rule == MX_SCALE_DEFAULT)
        rule = fmt == MX_FMT_MOSS_FP8 ? MX_SCALE_CEIL : MX_SCALE_FLOOR;
    fill_meta(row_out, R, C, fmt, row_hadamard);
    fill_meta(col_out, C, R, fmt, col_hadamard);
    const bool ts = fmt_has_tensor_scale(fmt);
    if (fmt_is_local(fmt)) {
        // row regions of x for the rowwise operand, column regions for the colwise one,
        // both from one pass over x
        if (amax_in)
            return MX_ERR_UNSUPPORTED;
        if ((rc = launch_region_amax(x, R, C, ld, row_out->amax, col_out->amax, d, s)) != MX_OK ||
            (rc = launch_local_scales(row_out->amax, row_out->tensor_scale, scale_count(fmt, R), d, s)) != MX_OK ||
            (rc = launch_local_scales(col_out->amax, col_out->tensor_scale, scale_count(fmt, C), d, s)) != MX_OK)
            return rc;
        if (R == 0 || C == 0)
            return MX_OK;
    } else if (ts && (rc = prepare_amax(x, R, C, ld, amax_in, row_out, MX_ROWWISE, d, s)) != MX_OK) {
        return rc;
    }
    if (R == 0 || C == 0) {
        if (!ts)
            return MX_OK;
        if ((rc = set_unit_scale(row_out, s)) != MX_OK)
            return rc;
        if (cudaMemcpyAsync(col_out->amax, row_out->amax, sizeof(float), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return MX_ERR_CUDA;
        return set_unit_scale(col_out, s);
    }
    TileArgs t = {};
    t.x = x;
    t.R = R;
    t.C = C;
    t.fmt = fmt;
    t.rule = rule;
    t.seed = seed;
    t.stream_id = stream_id;
    t.amax = row_out->amax;
    t.tensor_scale = row_out->tensor_scale;
    if (ts && !fmt_is_local(fmt)) {
        t.amax_copy = col_out->amax;
        t.tensor_scale_copy = col_out->tensor_scale;
    }
    t.row_ts_v = row_out->tensor_scale;
    t.col_ts_v = col_out->tensor_scale;
    t.row_codes = static_cast<uint8_t*>(row_out->codes);
    t.row_sf = row_out->sf;
    t.row_sr = row_rounding == MX_ROUND_SR;
    t.row_had = row_hadamard ? 1 : 0;
    t.col_codes = static_cast<uint8_t*>(col_out->codes);
    t.col_sf = col_out->sf;
    t.col_sr = col_rounding == MX_ROUND_SR;
    t.col_had = col_hadamard ? 1 : 0;
    t.status = d.status;
    t.wait_ns = kWaitLimitNs;
    t.fail_at = g_tile_fail_at;
    return launch_quantize_tile(t, ld, d, s);
}

int gemm_impl(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc, int out_dtype,
              const Device& d, cudaStream_t s, float* amax_out = nullptr)
{
    int rc = check_operand(A);
    if (rc != MX_OK)
        return rc;
    rc = check_operand(B);
    if (rc != MX_OK)
        return rc;
    if (A->fmt != B->fmt || A->k != B->k || A->hadamard != B->hadamard)
        return MX_ERR_INVALID_ARG;
    if (out_dtype != MX_OUT_F32 && out_dtype != MX_OUT_BF16)
        return MX_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->k;
    if (amax_out) {  // zeroed first: an empty product has amax 0
        if (reinterpret_cast<uintptr_t>(amax_out) % 4 != 0)
            return MX_ERR_ALIGNMENT;
        if (cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess)
            return MX_ERR_CUDA;
    }
    if (M == 0 || N == 0)
        return MX_OK;
    if (!C || ldc < N)
        return MX_ERR_INVALID_ARG;
    if (ldc % 8 != 0 || !aligned16(C) || K % gemm_k_multiple(A->fmt) != 0)
        return MX_ERR_ALIGNMENT;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return MX_ERR_UNSUPPORTED;
    const size_t esz = out_dtype == MX_OUT_BF16 ? 2 : 4;
    if (K == 0)
        return cudaMemset2DAsync(C, ldc * esz, 0, N * esz, M, s) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
    const float extra = A->hadamard ? extra_alpha * (1.0f / 32.0f) : extra_alpha;
    return launch_gemm(A, B, extra, C, ldc, out_dtype, d, s, nullptr, reinterpret_cast<unsigned*>(amax_out));
}

// The GEMM with its output quantized in the epilogue into the rowwise MX
// operand `out` (rows M, K = N) that a following GEMM consumes.
int gemm_quantized_impl(const mx_tensor* A, const mx_tensor* B, float extra_alpha, mx_tensor* out, const Device& d,
                        cudaStream_t s)
{
    int rc = check_operand(A);
    if (rc == MX_OK)
        rc = check_operand(B);
    if (rc != MX_OK)
        return rc;
    if (A->fmt != B->fmt || A->k != B->k || A->hadamard != B->hadamard || !out)
        return MX_ERR_INVALID_ARG;
    if (out->fmt != MX_FMT_MXFP8_E4M3 && out->fmt != MX_FMT_MXFP4_E2M1)
        return MX_ERR_UNSUPPORTED;
    const int64_t M = A->rows, N = B->rows, K = A->k;
    if (N % 32 != 0 || K % gemm_k_multiple(A->fmt) != 0)
        return MX_ERR_ALIGNMENT;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return MX_ERR_UNSUPPORTED;
    if ((rc = check_output(out, out->fmt, M, N)) != MX_OK || !aligned16(out->sf))
        return rc != MX_OK ? rc : MX_ERR_ALIGNMENT;
    fill_meta(out, M, N, out->fmt, 0);
    if (M == 0 || N == 0)
        return MX_OK;
    if (K == 0)
        return MX_ERR_UNSUPPORTED;  // an all-zero product has no use as an operand here
    const float extra = A->hadamard ? extra_alpha * (1.0f / 32.0f) : extra_alpha;
    const int mode = out->fmt == MX_FMT_MXFP8_E4M3 ? 2 : 3;
    const int64_t row_bytes = out->fmt == MX_FMT_MXFP8_E4M3 ? N : N / 2;
    return launch_gemm(A, B, extra, out->codes, row_bytes, mode, d, s, out->sf);
}

}  // namespace

extern "C" {

size_t mx_codes_bytes(int fmt, int64_t rows, int64_t k)
{
    if (!valid_fmt(fmt) || rows < 0 || k < 0 || (fmt_is_fp4(fmt) && k % 2))
        return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(codes_row_bytes(fmt, k));
}

size_t mx_sf_bytes(int fmt, int64_t rows, int64_t k)
{
    if (!valid_fmt(fmt) || rows < 0 || k < 0 || k % fmt_block(fmt))
        return 0;
    return static_cast<size_t>(sf_layout_bytes(rows, k / fmt_block(fmt)));
}

int mx_amax(const void* x, int64_t R, int64_t C, int64_t ld, float* amax, void* stream)
{
    if (!amax || R < 0 || C < 0 || ld < C || (R > 0 && C > 0 && !x))
        return MX_ERR_INVALID_ARG;
    if (ld % 8 != 0 || C % 8 != 0 || !aligned16(x))
        return MX_ERR_ALIGNMENT;
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return launch_amax(x, R, C, ld, amax, d, static_cast<cudaStream_t>(stream));
}

int mx_quantize(const void* x, int64_t R, int64_t C, int64_t ld, int dir, int fmt, int block, int rounding,
                int scale_rule, uint64_t seed, uint32_t stream_id, int hadamard, const float* amax_in,
                mx_tensor* out, void* stream)
{
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return quantize_impl(x, R, C, ld, dir, fmt, block, rounding, scale_rule, seed, stream_id, hadamard, amax_in, out,
                         d, static_cast<cudaStream_t>(stream));
}

int mx_quantize_dual(const void* x, int64_t R, int64_t C, int64_t ld, int fmt, int block, int scale_rule,
                     uint64_t seed, uint32_t stream_id, int row_rounding, int row_hadamard, int col_rounding,
                     int col_hadamard, const float* amax_in, mx_tensor* row_out, mx_tensor* col_out, void* stream)
{
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return quantize_dual_impl(x, R, C, ld, fmt, block, scale_rule, seed, stream_id, row_rounding, row_hadamard,
                              col_rounding, col_hadamard, amax_in, row_out, col_out, d,
                              static_cast<cudaStream_t>(stream));
}

int mx_dequantize(const mx_tensor* A, float* out, void* stream)
{
    int rc = check_operand(A);
    if (rc != MX_OK)
        return rc;
    if (!out && A->rows * A->k > 0)
        return MX_ERR_INVALID_ARG;
    Device d;
    rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return launch_dequantize(A, out, d, static_cast<cudaStream_t>(stream));
}

int mx_gemm(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc, int out_dtype,
            void* stream)
{
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return gemm_impl(A, B, extra_alpha, C, ldc, out_dtype, d, static_cast<cudaStream_t>(stream));
}

int mx_gemm_amax(const mx_tensor* A, const mx_tensor* B, float extra_alpha, void* C, int64_t ldc, int out_dtype,
                 float* amax_out, void* stream)
{
    if (!amax_out)
        return MX_ERR_INVALID_ARG;
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return gemm_impl(A, B, extra_alpha, C, ldc, out_dtype, d, static_cast<cudaStream_t>(stream), amax_out);
}

int mx_gemm_quantized(const mx_tensor* A, const mx_tensor* B, float extra_alpha, mx_tensor* out, void* stream)
{
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    return gemm_quantized_impl(A, B, extra_alpha, out, d, static_cast<cudaStream_t>(stream));
}

size_t mx_scale_count(int fmt, int64_t rows)
{
    return valid_fmt(fmt) && rows >= 0 ? static_cast<size_t>(scale_count(fmt, rows)) : 0;
}

size_t mx_linear_workspace_bytes(int64_t T, int64_t Kin, int64_t Nout, int fmt, int pass)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return 0;
    if (pass == 0)
        return carve(nullptr, fmt, T, Kin, nullptr) + carve(nullptr, fmt, Nout, Kin, nullptr);
    if (pass == 2)  // mx_linear_bwd_saved: dY rowwise [T, Nout] and dY^T [Nout, T]
        return carve(nullptr, fmt, T, Nout, nullptr) + carve(nullptr, fmt, Nout, T, nullptr);
    if (pass != 1)
        return 0;
    // dgrad: dY rowwise [T, Nout], W^T [Kin, Nout]; wgrad: dY^T [Nout, T], X^T [Kin, T]
    return carve(nullptr, fmt, T, Nout, nullptr) + carve(nullptr, fmt, Kin, Nout, nullptr) +
           carve(nullptr, fmt, Nout, T, nullptr) + carve(nullptr, fmt, Kin, T, nullptr);
}

int mx_linear_fwd(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout, int fmt, void* Y,
                  int out_dtype, void* workspace, size_t ws_bytes, void* stream)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return MX_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < mx_linear_workspace_bytes(T, Kin, Nout, fmt, 0))
        return MX_ERR_WORKSPACE;
    Device d;
    int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mx_tensor xq, wq;
    const size_t off = carve(ws, fmt, T, Kin, &xq);
    carve(ws + off, fmt, Nout, Kin, &wq);
    const int block = fmt_block(fmt);
    rc = quantize_impl(X, T, Kin, Kin, MX_ROWWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0, 0, nullptr, &xq,
                       d, s);
    if (rc != MX_OK)
        return rc;
    rc = quantize_impl(W, Nout, Kin, Kin, MX_ROWWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0, 0, nullptr,
                       &wq, d, s);
    if (rc != MX_OK)
        return rc;
    return gemm_impl(&xq, &wq, 1.0f, Y, Nout, out_dtype, d, s);
}

int mx_linear_bwd(const void* dY, const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout, int fmt,
                  const mx_bwd_opts* opts, void* dX, int dx_dtype, void* dW, int dw_dtype, void* workspace,
                  size_t ws_bytes, void* stream)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return MX_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < mx_linear_workspace_bytes(T, Kin, Nout, fmt, 1))
        return MX_ERR_WORKSPACE;
    mx_bwd_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts)
        o = *opts;
    Device d;
    int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mx_tensor dyr, wt, dyt, xt;
    size_t off = carve(ws, fmt, T, Nout, &dyr);
    off += carve(ws + off, fmt, Kin, Nout, &wt);
    off += carve(ws + off, fmt, Nout, T, &dyt);
    carve(ws + off, fmt, Kin, T, &xt);
    const int block = fmt_block(fmt);
    if (dX && dW) {
        // one pass over dY emits both its dgrad (rowwise) and wgrad (colwise) operands
        rc = quantize_dual_impl(dY, T, Nout, Nout, fmt, block, MX_SCALE_DEFAULT, o.seed, o.stream_id, MX_ROUND_RNE, 0,
                                o.wgrad_dy_rounding, o.wgrad_hadamard, nullptr, &dyr, &dyt, d, s);
        if (rc != MX_OK)
            return rc;
    }
    // data gradient on s, weight gradient on the side stream when both are wanted
    cudaStream_t sw = dX && dW ? fork_begin(d, s) : nullptr;
    if (dX) {
        if (!dW)
            rc = quantize_impl(dY, T, Nout, Nout, MX_ROWWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0, 0,
                               nullptr, &dyr, d, s);
        if (rc == MX_OK)
            rc = quantize_impl(W, Nout, Kin, Kin, MX_COLWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0, 0,
                               nullptr, &wt, d, s);
        if (rc == MX_OK)
            rc = gemm_impl(&dyr, &wt, 1.0f, dX, Kin, dx_dtype, d, s);
    }
    if (dW && rc == MX_OK) {
        cudaStream_t s2 = sw ? sw : s;
        if (!dX)
            rc = quantize_impl(dY, T, Nout, Nout, MX_COLWISE, fmt, block, o.wgrad_dy_rounding, MX_SCALE_DEFAULT,
                               o.seed, o.stream_id, o.wgrad_hadamard, nullptr, &dyt, d, s2);
        if (rc == MX_OK)
            rc = quantize_impl(X, T, Kin, Kin, MX_COLWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0,
                               o.wgrad_hadamard, nullptr, &xt, d, s2);
        if (rc == MX_OK)
            rc = gemm_impl(&dyt, &xt, 1.0f, dW, Kin, dw_dtype, d, s2);
    }
    if (sw) {
        const int rj = fork_end(d, sw, s);
        if (rc == MX_OK)
            rc = rj;
    }
    return rc;
}

size_t mx_linear_saved_bytes(int64_t T, int64_t Kin, int64_t Nout, int fmt)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return 0;
    return carve(nullptr, fmt, Kin, T, nullptr) + carve(nullptr, fmt, Kin, Nout, nullptr);  // X^T, W^T
}

namespace {

// The saved backward state of one layer: the colwise operands X^T [Kin, T]
// (for the weight gradient) and W^T [Kin, Nout] (for the data gradient), in
// that order, carved like a workspace.
void carve_saved(uint8_t* saved, int64_t T, int64_t Kin, int64_t Nout, int fmt, int wgrad_hadamard, mx_tensor* xt,
                 mx_tensor* wt)
{
    const size_t off = carve(saved, fmt, Kin, T, xt);
    carve(saved + off, fmt, Kin, Nout, wt);
    fill_meta(xt, Kin, T, fmt, wgrad_hadamard);
    fill_meta(wt, Kin, Nout, fmt, 0);
}

}  // namespace

int mx_linear_fwd_save(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout, int fmt,
                       const float* x_amax, const float* w_amax, const mx_bwd_opts* opts, void* Y, int out_dtype,
                       void* workspace, size_t ws_bytes, void* saved, size_t saved_bytes, void* stream)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return MX_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < mx_linear_workspace_bytes(T, Kin, Nout, fmt, 0) || !saved ||
        saved_bytes < mx_linear_saved_bytes(T, Kin, Nout, fmt))
        return MX_ERR_WORKSPACE;
    if (fmt_is_local(fmt) && (x_amax || w_amax))
        return MX_ERR_UNSUPPORTED;  // the region maxima of both directions come from the pass itself
    mx_bwd_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts)
        o = *opts;
    Device d;
    int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mx_tensor xq, wq, xt, wt;
    const size_t off = carve(ws, fmt, T, Kin, &xq);
    carve(ws + off, fmt, Nout, Kin, &wq);
    carve_saved(static_cast<uint8_t*>(saved), T, Kin, Nout, fmt, o.wgrad_hadamard, &xt, &wt);
    const int block = fmt_block(fmt);
    // one read of X: the forward operand and X^T, transformed as the weight gradient will want it
    rc = quantize_dual_impl(X, T, Kin, Kin, fmt, block, MX_SCALE_DEFAULT, 0, 0, MX_ROUND_RNE, 0, MX_ROUND_RNE,
                            o.wgrad_hadamard, x_amax, &xq, &xt, d, s);
    if (rc != MX_OK)
        return rc;
    // one read of W: the forward operand and W^T for the data gradient
    rc = quantize_dual_impl(W, Nout, Kin, Kin, fmt, block, MX_SCALE_DEFAULT, 0, 0, MX_ROUND_RNE, 0, MX_ROUND_RNE, 0,
                            w_amax, &wq, &wt, d, s);
    if (rc != MX_OK)
        return rc;
    return gemm_impl(&xq, &wq, 1.0f, Y, Nout, out_dtype, d, s);
}

int mx_linear_bwd_saved(const void* dY, int64_t T, int64_t Kin, int64_t Nout, int fmt, const float* dy_amax,
                        const mx_bwd_opts* opts, const void* saved, size_t saved_bytes, void* dX, int dx_dtype,
                        void* dW, int dw_dtype, void* workspace, size_t ws_bytes, void* stream)
{
    if (!valid_fmt(fmt) || T < 0 || Kin < 0 || Nout < 0)
        return MX_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < mx_linear_workspace_bytes(T, Kin, Nout, fmt, 2) || !saved ||
        saved_bytes < mx_linear_saved_bytes(T, Kin, Nout, fmt))
        return MX_ERR_WORKSPACE;
    if (fmt_is_local(fmt) && dy_amax)
        return MX_ERR_UNSUPPORTED;
    mx_bwd_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts)
        o = *opts;
    Device d;
    int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mx_tensor dyr, dyt, xt, wt;
    const size_t off = carve(ws, fmt, T, Nout, &dyr);
    carve(ws + off, fmt, Nout, T, &dyt);
    carve_saved(static_cast<uint8_t*>(const_cast<void*>(saved)), T, Kin, Nout, fmt, o.wgrad_hadamard, &xt, &wt);
    const int block = fmt_block(fmt);
    if (dX && dW) {
        rc = quantize_dual_impl(dY, T, Nout, Nout, fmt, block, MX_SCALE_DEFAULT, o.seed, o.stream_id, MX_ROUND_RNE, 0,
                                o.wgrad_dy_rounding, o.wgrad_hadamard, dy_amax, &dyr, &dyt, d, s);
    } else if (dX) {
        rc = quantize_impl(dY, T, Nout, Nout, MX_ROWWISE, fmt, block, MX_ROUND_RNE, MX_SCALE_DEFAULT, 0, 0, 0, dy_amax,
                           &dyr, d, s);
    } else if (dW) {
        rc = quantize_impl(dY, T, Nout, Nout, MX_COLWISE, fmt, block, o.wgrad_dy_rounding, MX_SCALE_DEFAULT, o.seed,
                           o.stream_id, o.wgrad_hadamard, dy_amax, &dyt, d, s);
    }
    if (rc != MX_OK)
        return rc;
    // data gradient on s, weight gradient on the side stream when both are wanted
    cudaStream_t sw = dX && dW ? fork_begin(d, s) : nullptr;
    if (dX)
        rc = gemm_impl(&dyr, &wt, 1.0f, dX, Kin, dx_dtype, d, s);
    if (dW && rc == MX_OK)
        rc = gemm_impl(&dyt, &xt, 1.0f, dW, Kin, dw_dtype, d, sw ? sw : s);
    if (sw) {
        const int rj = fork_end(d, sw, s);
        if (rc == MX_OK)
            rc = rj;
    }
    return rc;
}

const char* mx_strerror(int status)
{
    switch (status) {
    case MX_OK: return "ok";
    case MX_ERR_INVALID_ARG: return "invalid argument";
    case MX_ERR_UNSUPPORTED: return "unsupported format, option or device";
    case MX_ERR_ALIGNMENT: return "alignment or size-multiple rule violated";
    case MX_ERR_CUDA: return "CUDA call failed";
    case MX_ERR_TIMEOUT: return "device-side bounded wait timed out";
    case MX_ERR_NO_DEVICE: return "no usable CUDA device";
    case MX_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

int mx_last_device_status(void* stream)
{
    Device d;
    const int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MX_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess)
        return MX_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess)
        return MX_ERR_CUDA;
    return v;
}

int mx_selftest_bounded_wait(uint64_t limit_ns, void* stream)
{
    Device d;
    int rc = current_device(&d);
    if (rc != MX_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_wait_selftest(limit_ns, d, s);
    if (rc != MX_OK)
        return rc;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MX_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess)
        return MX_ERR_CUDA;
    return v;
}

uint64_t mx_launch_count(void) { return g_kernel_launches.load(); }

int mx_debug_divide(const float* v, const float* d, int64_t n, float* q_fast, float* q_ieee, void* stream)
{
    if (n < 0 || (n > 0 && (!v || !d || !q_fast || !q_ieee)))
        return MX_ERR_INVALID_ARG;
    Device dev;
    const int rc = current_device(&dev);
    if (rc != MX_OK)
        return rc;
    return launch_divide_check(v, d, n, q_fast, q_ieee, dev, static_cast<cudaStream_t>(stream));
}

// Test hook: producer implementation (0 automatic, 1 direct loads, 2 tile producer).
void mx_debug_set_quant_impl(int impl) { g_quant_impl = (impl >= 0 && impl <= 2) ? impl : 0; }

void mx_debug_set_tile_fail_at(int64_t tile) { g_tile_fail_at = tile >= 0 ? tile : -1; }

void mx_debug_set_bwd_fork(int on) { g_bwd_fork = on ? 1 : 0; }

// Test hook: force one GEMM kernel variant (0 = automatic).
void mx_debug_set_gemm_variant(int variant) { set_gemm_variant(variant); }
int mx_debug_last_gemm_variant(void) { return last_gemm_variant(); }

}  // extern "C"
