// tc_capi.cu -- the extern "C" entries (declared in include/gnsilu.h) of the
// tensor-core operations: the fused nearest-2x upsample + 3x3 convolution
// and the single-head attention with the output projection folded into V.
// Argument validation here; the kernels are in upconv_kernels.cu and
// attn_kernels.cu.
#include <algorithm>
#include <cstdint>

#include "../../include/gnsilu.h"
#include "capi_util.h"
#include "tc_internal.h"

namespace {

using gn_capi::DeviceInfo;
using gn_capi::count_launches;
using gn_capi::current_device;
using gn_capi::ranges_overlap;
using gn_capi::wait_timeout_ns;

}  // namespace

extern "C" {

// ---- fused nearest-2x upsample + 3x3 convolution ----------------------------
int64_t gn_upconv_folded_bytes(int64_t Cin, int64_t Cout)
{
    if (Cin < 1 || Cout < 1 || Cin > (1 << 20) || Cout > (1 << 20)) return -1;
    return 16 * Cin * Cout * 2;
}

namespace {

int upconv_channels_ok(int64_t Cin, int64_t Cout)
{
    return Cin >= 64 && Cin <= 8192 && Cin % 64 == 0 && Cout >= 128 && Cout <= 8192 && Cout % 128 == 0;
}

}  // namespace

int gn_upconv_fold(const void *w, void *wf, int64_t Cin, int64_t Cout, void *stream)
{
    if (!w || !wf) return GN_ERR_NULL;
    if (!upconv_channels_ok(Cin, Cout)) return GN_ERR_CHANNELS;
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(w) % 2 || addr(wf) % 16) return GN_ERR_ALIGN;
    if (ranges_overlap(w, static_cast<size_t>(9 * Cin * Cout * 2), wf,
                       static_cast<size_t>(gn_upconv_folded_bytes(Cin, Cout))))
        return GN_ERR_ALIAS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(dev)) return GN_ERR_KERNEL;
    const cudaError_t e = gn::launch_upconv_fold(w, wf, static_cast<int>(Cin), static_cast<int>(Cout), d.sm_count,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    count_launches(1);
    return GN_OK;
}

int gn_upconv_nhwc(const void *x, const void *wf, const void *bias, void *y, int64_t N, int64_t H, int64_t W,
                   int64_t Cin, int64_t Cout, void *stream)
{
    if (!x || !wf || !y) return GN_ERR_NULL;
    if (N < 0 || H < 1 || W < 1 || H > (1 << 20) || W > (1 << 20)) return GN_ERR_SHAPE;
    if (!upconv_channels_ok(Cin, Cout)) return GN_ERR_CHANNELS;
    if (N > 0 && (N > (1 << 20) || N * H * W > INT64_MAX / (4 * 2 * std::max(Cin, Cout)))) return GN_ERR_SHAPE;
    gn::UpconvTiling t;
    if (N > 0 && !gn::upconv_tiling(N, H, W, &t)) return GN_ERR_SHAPE;
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(x) % 16 || addr(wf) % 16 || addr(y) % 16 || (bias && addr(bias) % 4)) return GN_ERR_ALIGN;
    const size_t xb = static_cast<size_t>(N * H * W * Cin * 2);
    const size_t yb = static_cast<size_t>(N * 4 * H * W * Cout * 2);
    if (ranges_overlap(y, yb, x, xb) || ranges_overlap(y, yb, wf, static_cast<size_t>(gn_upconv_folded_bytes(Cin, Cout))) ||
        (bias && ranges_overlap(y, yb, bias, static_cast<size_t>(2 * Cout))))
        return GN_ERR_ALIAS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(dev)) return GN_ERR_KERNEL;
    if (N == 0) return GN_OK;
    cudaError_t e = cudaSuccess;
    const int r = gn::launch_upconv(x, wf, bias, y, static_cast<int>(N), static_cast<int>(H), static_cast<int>(W),
                                    static_cast<int>(Cin), static_cast<int>(Cout), d.sm_count, wait_timeout_ns(),
                                    static_cast<cudaStream_t>(stream), &e);
    if (r == 1) return GN_ERR_SHAPE;
    if (r != 0) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    count_launches(1);
    return GN_OK;
}

// ---- single-head attention with the output projection folded into V --------
namespace {

bool attn_width_ok(int64_t D) { return D >= 128 && D <= 1024 && D % 128 == 0; }

bool attn_tokens_ok(int64_t S) { return S >= 128 && S <= gn::kAttnMaxS && S % 128 == 0; }

}  // namespace

int gn_attn_fold(const void *wv, const void *bv, const void *wo, const void *bo, void *wf, float *bf, int64_t D,
                 void *stream)
{
    if (!wv || !bv || !wo || !bo || !wf || !bf) return GN_ERR_NULL;
    if (!attn_width_ok(D)) return GN_ERR_CHANNELS;
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(wv) % 2 || addr(bv) % 2 || addr(wo) % 2 || addr(bo) % 2 || addr(wf) % 16 || addr(bf) % 16)
        return GN_ERR_ALIGN;
    const size_t wb = static_cast<size_t>(2 * D * D), bb = static_cast<size_t>(4 * D);
    for (const void *in : {wv, wo})
        if (ranges_overlap(wf, wb, in, wb) || ranges_overlap(bf, bb, in, wb)) return GN_ERR_ALIAS;
    for (const void *in : {bv, bo})
        if (ranges_overlap(wf, wb, in, static_cast<size_t>(2 * D)) ||
            ranges_overlap(bf, bb, in, static_cast<size_t>(2 * D)))
            return GN_ERR_ALIAS;
    if (ranges_overlap(wf, wb, bf, bb)) return GN_ERR_ALIAS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(dev)) return GN_ERR_KERNEL;
    const cudaError_t e = gn::launch_attn_fold(wv, bv, wo, bo, wf, bf, static_cast<int>(D), d.sm_count,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    count_launches(1);
    return GN_OK;
}

size_t gn_attn_workspace_bytes(int64_t S, int64_t D)
{
    if (!attn_tokens_ok(S) || !attn_width_ok(D)) return 0;
    return gn::attn_workspace_bytes(S, D);
}

int gn_attn_folded(const void *q, const void *k, const void *xn, const void *wf, const float *bf,
                   const void *residual, void *out, int64_t S, int64_t D, void *workspace, size_t workspace_bytes,
                   void *stream)
{
    return gn_attn_folded_ex(q, k, xn, wf, bf, residual, out, S, D, workspace, workspace_bytes, GN_ATTN_AUTO,
                             stream);
}

int gn_attn_folded_ex(const void *q, const void *k, const void *xn, const void *wf, const float *bf,
                      const void *residual, void *out, int64_t S, int64_t D, void *workspace, size_t workspace_bytes,
                      int schedule, void *stream)
{
    if (!q || !k || !xn || !wf || !bf || !out || !workspace) return GN_ERR_NULL;
    if (!attn_tokens_ok(S)) return GN_ERR_SHAPE;
    if (!attn_width_ok(D)) return GN_ERR_CHANNELS;
    if (schedule != GN_ATTN_AUTO && schedule != GN_ATTN_ONE_PASS && schedule != GN_ATTN_STORED_WEIGHTS)
        return GN_ERR_VARIANT;
    if (schedule == GN_ATTN_ONE_PASS && !gn::attn_one_pass_ok(D)) return GN_ERR_VARIANT;
    const bool one_pass = schedule == GN_ATTN_ONE_PASS ||
                          (schedule == GN_ATTN_AUTO && gn::attn_one_pass_preferred(S, D));
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(q) % 16 || addr(k) % 16 || addr(xn) % 16 || addr(wf) % 16 || addr(bf) % 16 || addr(out) % 16 ||
        addr(workspace) % 256 || (residual && addr(residual) % 16))
        return GN_ERR_ALIGN;
    const size_t need = gn::attn_workspace_bytes(S, D);
    if (workspace_bytes < need) return GN_ERR_WORKSPACE;
    const size_t act = static_cast<size_t>(2 * S * D);
    const struct {
        const void *p;
        size_t n;
    } ins[] = {{q, act}, {k, act}, {xn, act}, {wf, static_cast<size_t>(2 * D * D)}, {bf, static_cast<size_t>(4 * D)}};
    // the whole workspace the caller hands over may be used (the one-pass
    // schedule keeps the pieces of split tiles beyond the minimum)
    const size_t wsb = workspace_bytes;
    for (const auto &in : ins)
        if (ranges_overlap(out, act, in.p, in.n) || ranges_overlap(workspace, wsb, in.p, in.n)) return GN_ERR_ALIAS;
    if (ranges_overlap(out, act, workspace, wsb)) return GN_ERR_ALIAS;
    if (residual && residual != out &&
        (ranges_overlap(out, act, residual, act) || ranges_overlap(workspace, wsb, residual, act)))
        return GN_ERR_ALIAS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(dev)) return GN_ERR_KERNEL;
    cudaError_t e = cudaSuccess;
    int launches = 0;
    const int r = gn::launch_attn_folded(q, k, xn, wf, bf, residual, out, static_cast<int>(S), static_cast<int>(D),
                                         workspace, workspace_bytes, one_pass, d.sm_count, wait_timeout_ns(),
                                         static_cast<cudaStream_t>(stream), &e, &launches);
    count_launches(static_cast<uint64_t>(launches));
    if (r != 0) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    return GN_OK;
}

}  // extern "C"
