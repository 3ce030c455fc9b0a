// capi_util.h -- what the two C-ABI translation units share: the current
// device (checked to be an sm_103 part, kernel attributes set once), the
// bound on every in-kernel wait, the overlap test used by the aliasing
// checks, and the library-wide kernel-launch counter.
#pragma once

#include <cstddef>
#include <cstdint>

namespace gn_capi {

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;      // max dynamic shared memory per block
    int smem_per_sm = 0;
    int coop = 0;
    int major = 0, minor = 0;
    int cluster_cap[17] = {};   // co-resident clusters of each size (cluster schedule)
    unsigned int *status_word = nullptr;   // the GroupNorm kernels' sticky status (device address)
    unsigned int *status_host = nullptr;   // its mapped host copy (device address)
};

// GN_OK with the device's properties, or GN_ERR_DEVICE / GN_ERR_CUDA.
int current_device(int *dev_out, DeviceInfo *info_out);
// Timeout of every bounded wait inside the kernels (GN_WAIT_TIMEOUT_MS, default 2000).
uint64_t wait_timeout_ns();
bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb);
void count_launches(uint64_t n);
// True once a kernel on device `dev` has given up a bounded wait and the
// status has not been cleared since (read from mapped host memory, no
// synchronisation).
bool kernel_status_raised(int dev);
// Every check gn_silu_rows_ex() makes before it launches anything, for the
// automatic schedule and a caller workspace: GN_OK with the workspace bytes
// the call needs, or the status the call would return.
int check_rows_call(const void *x, const float *gamma, const float *beta, const void *y, int64_t N, int64_t L,
                    int64_t C, int64_t G, float eps, const float *mean_out, const float *rstd_out,
                    size_t *workspace_need);

}  // namespace gn_capi
