// tc_common.cuh -- what the tensor-core kernel files share: the bounded
// mbarrier wait and the teardown drain, the lookup of the driver's
// tensor-map encoder, and the number of CTA pairs that fit on the device.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gn_ptx.cuh"

namespace gn {
namespace tc {

// Waiting threads sleep in the try_wait (up to this long per round) rather
// than spin, so that the warps still working keep the issue slots.
constexpr uint32_t kSleepNs = 20000;

// Bounded wait on an mbarrier phase.  False once `timeout_ns` pass (the
// CTA's abort flag, the kernel file's status word and its host-visible copy
// are then set), or at once when another thread of the CTA has aborted.
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns,
                                     unsigned int *status, unsigned int *host_status)
{
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    const uint64_t deadline = global_ns() + timeout_ns;
#pragma unroll 1
    for (;;) {
        if (mbar_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort) return false;
        if (global_ns() > deadline) {
            *abort = 1;
            atomicOr(status, 1u);
            raise_host_status(host_status);
            return false;
        }
    }
}

// A wait during teardown after an abort: bounded, but not cut short by the
// abort flag (the copies and MMAs it waits for are still in flight).
__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t deadline = global_ns() + timeout_ns;
#pragma unroll 1
    while (!mbar_wait_sleep(bar, parity, kSleepNs)) {
        if (global_ns() > deadline) return;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself); null if unavailable.
inline EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// How many clusters of two CTAs of `kernel` (threads, dynamic shared
// memory) can be resident at once; half the SMs if the query fails.
template <typename Kernel>
int pair_clusters(Kernel kernel, int threads, size_t smem, int sm_count)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count / 2));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = sm_count / 2;
    }
    return n;
}

// Programmatic dependent launch.  A kernel launched by launch_pdl may start
// while the kernel ahead of it in the stream is still running, once every
// CTA of that kernel has called griddep_launch_dependents (or exited); it
// must call griddep_wait before its first access to global memory, which
// then returns once that kernel has finished and its writes are visible.
// Every kernel here signals only after its own griddep_wait has returned, so
// a kernel that starts early still starts after everything ahead of its
// predecessor has finished (the one-pass attention kernel reads q and k
// without waiting).  For a kernel launched without the attribute both are
// no-ops.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace tc
}  // namespace gn
