// gn_static.cu -- gn_silu_rows_static(): GroupNorm(+SiLU) that allocates no
// device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured in global capture mode (allocation calls are illegal there),
// plug-ins and engine hooks whose host framework owns all device memory and
// forbids allocations behind its back, and real-time paths that must not
// risk an allocator's implicit device synchronisation.  For them this entry
// point takes its scratch (the per-segment partial statistics, the channel
// records and the grid-barrier words that gn_silu_rows keeps in a workspace)
// from one fixed array compiled into the library, so a call never allocates.
//
// The array is GN_STATIC_SCRATCH_BYTES long and sits in the memory of every
// GPU that loads the library until the process exits.  All calls on a GPU
// share it, and it keeps whatever the previous call left in it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gnsilu.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices];   // device address of g_static_scratch, per device

// Device address of the scratch array on device `dev` (which must be
// current).  The host-side name g_static_scratch is only a stand-in; the
// real address comes from cudaGetSymbolAddress, looked up once per device.
int static_scratch(int dev, void **out)
{
    if (dev < 0 || dev >= kMaxDevices) return GN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GN_ERR_CUDA;
        }
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return GN_OK;
}

}  // namespace

extern "C" int gn_silu_rows_static(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16,
                                   int64_t N, int64_t L, int64_t C, int64_t G, float eps, int apply_silu,
                                   float *mean_out, float *rstd_out, void *stream)
{
    // Argument and shape checks happen inside gn_silu_rows_ex; only the
    // scratch size is checked here, so the array is never asked for more
    // than it holds.
    const size_t need = gn_silu_workspace_bytes(N, L, C, G);
    if (need > static_cast<size_t>(GN_STATIC_SCRATCH_BYTES)) return GN_ERR_WORKSPACE;
    if (need == 0) {
        // Unsupported shape or no usable device: let the full validation say
        // which.  A zero-byte workspace is passed so that this path can
        // never fall back to the library's allocating workspace: any shape
        // that passes validation is then refused as GN_ERR_WORKSPACE before
        // the (never dereferenced) pointer is used.
        return gn_silu_rows_ex(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, apply_silu, mean_out,
                               rstd_out, reinterpret_cast<void *>(static_cast<uintptr_t>(256)), 0,
                               GN_VARIANT_AUTO, stream);
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_DEVICE;
    }
    void *scratch = nullptr;
    const int rc = static_scratch(dev, &scratch);
    if (rc != GN_OK) return rc;
    // The grid-barrier words at the start of the scratch must read zero when
    // a call starts; the previous call may have left them otherwise (only if
    // it failed), so clear them on the caller's stream.
    if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    return gn_silu_rows_ex(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, apply_silu, mean_out, rstd_out,
                           scratch, static_cast<size_t>(GN_STATIC_SCRATCH_BYTES), GN_VARIANT_AUTO, stream);
}
