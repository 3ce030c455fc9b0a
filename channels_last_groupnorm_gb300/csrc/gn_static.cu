// gn_static.cu -- gn_silu_rows_static(): GroupNorm(+SiLU) that allocates no
// device memory.
//
// Some callers cannot call cudaMalloc.  A plug-in that runs inside a host
// framework which owns every byte of device memory (through its own pool,
// with its own accounting) may not allocate behind the framework's back.  A
// latency-critical path cannot afford the device-wide synchronisation and
// the unbounded time an allocation or a free may take.  A process that runs
// under a fixed device-memory budget cannot count on a new allocation
// succeeding mid-run.  For such callers this entry point takes its scratch
// (the per-segment partial statistics, the channel records and the
// grid-barrier words that gn_silu_rows keeps in a workspace) from one fixed
// array compiled into the library, so a call never allocates.
//
// The array is GN_STATIC_SCRATCH_BYTES long and sits in the memory of every
// GPU that loads the library until the process exits.  All calls on a GPU
// share it, and it keeps whatever the previous call left in it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gnsilu.h"
#include "capi_util.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices];   // device address of g_static_scratch, per device

// Device address of the scratch array on device `dev` (which must be
// current).  The host-side name g_static_scratch is only a stand-in; the
// real address comes from cudaGetSymbolAddress, looked up once per device
// and kept until the process exits.
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
    // Every check the call will make runs first, so that a refused call
    // returns its status without touching the shared array.
    size_t need = 0;
    const int rc = gn_capi::check_rows_call(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, mean_out, rstd_out,
                                            &need);
    if (rc != GN_OK) return rc;
    if (need > static_cast<size_t>(GN_STATIC_SCRATCH_BYTES)) return GN_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_DEVICE;
    }
    void *scratch = nullptr;
    const int rs = static_scratch(dev, &scratch);
    if (rs != GN_OK) return rs;
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
