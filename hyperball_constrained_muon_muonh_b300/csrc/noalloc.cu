// muonh_orthogonalize_static: Newton-Schulz with scratch in a fixed device
// array instead of a caller-supplied workspace, for callers that cannot call
// cudaMalloc.  It runs the same kernels as muonh_orthogonalize.

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/muonh.h"

namespace muonh {
int report_error(int code, const char* msg);
}

namespace {

constexpr size_t kScratchBytes = MUONH_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress (per device).
__device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int muonh_orthogonalize_static(const void* in, int in_dtype, void* out, int out_dtype, int64_t rows,
                                          int64_t cols, int ns_steps, const float ns_coeffs[3], float eps,
                                          uint32_t flags, void* stream) {
    if ((in_dtype != MUONH_DTYPE_F32 && in_dtype != MUONH_DTYPE_BF16) ||
        (out_dtype != MUONH_DTYPE_F32 && out_dtype != MUONH_DTYPE_BF16))
        return muonh::report_error(MUONH_ERR_UNSUPPORTED,
                                   "in_dtype/out_dtype must be MUONH_DTYPE_F32 or MUONH_DTYPE_BF16");
    size_t need = 0;
    int r = muonh_orthogonalize_workspace_size(rows, cols, flags, &need);
    if (r != MUONH_OK) return r;
    if (need > kScratchBytes)
        return muonh::report_error(MUONH_ERR_WORKSPACE,
                                   "muonh_orthogonalize_static: this shape needs more scratch than the "
                                   "library's fixed 96 MiB array; use muonh_orthogonalize with a workspace");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return muonh::report_error(MUONH_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return muonh::report_error(MUONH_ERR_UNSUPPORTED, "muonh_orthogonalize_static: device index >= 64");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess || !p)
                return muonh::report_error(MUONH_ERR_CUDA, "muonh_orthogonalize_static: cudaGetSymbolAddress failed");
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    return muonh_orthogonalize(in, in_dtype, out, out_dtype, rows, cols, ns_steps, ns_coeffs, eps, flags, scratch,
                               kScratchBytes, stream);
}
