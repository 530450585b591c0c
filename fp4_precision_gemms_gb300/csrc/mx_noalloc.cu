// mx_noalloc.cu -- a linear-layer forward for callers that cannot allocate
// device memory.
//
// mx_linear_fwd needs a workspace for the quantized copies of X and W.  Some
// callers have no way to provide one: code running where cudaMalloc is not
// allowed or not wanted (inside a custom allocator or a memory-pool callback,
// in a process whose device memory is fully reserved up front, or behind a
// plugin interface that hands over only input and output pointers).  For them
// mx_linear_fwd_noalloc keeps its workspace in a fixed file-scope device array
// and allocates nothing.
#include <cstring>
#include <mutex>

#include "mx_internal.cuh"

namespace {

// Largest workspace the no-allocation forward can use.  The array lives in
// the module's global memory, so every GPU that loads the library holds these
// bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int scratch_address(int device, void** out)
{
    static std::mutex mu;
    static void* addr[64];
    if (device < 0 || device >= 64)
        return MX_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MX_ERR_CUDA;
        }
        addr[device] = p;
    }
    *out = addr[device];
    return MX_OK;
}

}  // namespace

extern "C" int mx_linear_fwd_noalloc(const void* X, const void* W, int64_t T, int64_t Kin, int64_t Nout,
                                     int fmt, void* Y, int out_dtype, void* stream)
{
    if (fmt < MX_FMT_MXFP8_E4M3 || fmt > MX_FMT_NVFP4_LOCAL || T < 0 || Kin < 0 || Nout < 0)
        return MX_ERR_INVALID_ARG;
    const size_t need = mx_linear_workspace_bytes(T, Kin, Nout, fmt, 0);
    if (need == 0 || need > kNoAllocScratchBytes)
        return MX_ERR_WORKSPACE;  // the quantized operands do not fit the fixed array
    mx::Device d;
    int rc = mx::current_device(&d);
    if (rc != MX_OK)
        return rc;
    void* ws = nullptr;
    rc = scratch_address(d.id, &ws);
    if (rc != MX_OK)
        return rc;
    // The forward rewrites every workspace byte it later reads (codes, scale
    // bytes of real rows, tensor scales) and clears the amax words (the tensor
    // amax, or the region maxima of NVFP4_LOCAL) on the stream before reducing
    // into them, so the previous call's contents do not leak into this one.
    return mx_linear_fwd(X, W, T, Kin, Nout, fmt, Y, out_dtype, ws, kNoAllocScratchBytes, stream);
}
