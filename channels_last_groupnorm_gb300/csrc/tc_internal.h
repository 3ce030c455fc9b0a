// tc_internal.h -- host-side declarations of the tensor-core kernels
// (upconv_kernels.cu, attn_kernels.cu) for the C ABI in tc_capi.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace gn {

// ---- fused nearest-2x upsample + 3x3 convolution (upconv_kernels.cu) ----
// The pixel box of one 128-pixel output tile of one parity: BW columns x BH
// rows x BNI images, and the tile counts along each axis.
struct UpconvTiling {
    int BW, BH, BNI;
    int tiles_w, tiles_h, tiles_n;
};
// false when (H, W) admits no such tiling: W a multiple of 128, or W a power
// of two below 128 with H a multiple of 128 / W or a power of two below it.
bool upconv_tiling(int64_t N, int64_t H, int64_t W, UpconvTiling *t);
cudaError_t launch_upconv_fold(const void *w, void *wf, int Cin, int Cout, int sm_count, cudaStream_t s);
// 0 = launched; 1 = shape not tileable; 2 = tensor-map encoding failed;
// 3 = the launch failed (*err holds the CUDA error).
int launch_upconv(const void *x, const void *wf, const void *bias, void *y, int N, int H, int W, int Cin,
                  int Cout, int sm_count, uint64_t timeout_ns, cudaStream_t s, cudaError_t *err);
cudaError_t read_upconv_status(unsigned int *status);
cudaError_t clear_upconv_status();
// Device address of the mapped host word that mirrors the status (current device).
cudaError_t set_upconv_status_host(unsigned int *host_word);

// ---- single-head attention with the output projection folded into V (attn_kernels.cu) ----
constexpr int kAttnMaxS = 32768;   // the longest sequence gn_attn_folded takes
cudaError_t launch_attn_fold(const void *wv, const void *bv, const void *wo, const void *bo, void *wf, float *bf,
                             int D, int sm_count, cudaStream_t s);
size_t attn_workspace_bytes(int64_t S, int64_t D);
// The one-pass schedule (scores on chip) handles widths up to 512.
inline bool attn_one_pass_ok(int64_t D) { return D <= 512; }
// The automatic choice: the one-pass schedule once there are 32 query tiles
// of 128 rows (S >= 4096); below that its CTA pairs leave most SMs idle (the
// minimum workspace holds too few pieces to split tiles finely) and the
// stored-weights schedule is faster (GB300, D = 512: 38 against 60 us at
// S = 2048, 69 against 64 us at S = 4096, 170 against 157 us at S = 8192).
inline bool attn_one_pass_preferred(int64_t S, int64_t D) { return attn_one_pass_ok(D) && S >= 4096; }
// 0 = launched (*launches kernels); 2 = tensor-map encoding failed; 3 = a
// launch failed (*err holds the CUDA error).  one_pass selects the schedule;
// it may use workspace beyond gn_attn_workspace_bytes() (workspace_bytes) for
// the pieces of tiles it splits between CTA pairs.
int launch_attn_folded(const void *q, const void *k, const void *xn, const void *wf, const float *bf,
                       const void *residual, void *out, int S, int D, void *workspace, size_t workspace_bytes,
                       bool one_pass, int sm_count, uint64_t timeout_ns, cudaStream_t s, cudaError_t *err,
                       int *launches);
cudaError_t read_attn_status(unsigned int *status);
cudaError_t clear_attn_status();
// Device address of the mapped host word that mirrors the status (current device).
cudaError_t set_attn_status_host(unsigned int *host_word);

}  // namespace gn
