// gn_capi.cu -- the extern "C" boundary of libgnsilu (declared in
// include/gnsilu.h): argument validation, the per-shape launch plan, the
// library-owned workspaces, and dispatch to the kernels in gn_kernels.cu.
//
// The rejection contract follows the sglang PR #33451 page ("FLUX.2 VAE
// decoder fast path behind quality=high", section "Modifications", item 1):
// unsupported inputs (non-power-of-two C, C > 2048, ...) are refused so the
// caller can fall back; here they return a status code and nothing runs.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gnsilu.h"
#include "capi_util.h"
#include "gn_internal.h"
#include "tc_internal.h"

namespace gn_capi {

std::atomic<uint64_t> g_launches{0};

void count_launches(uint64_t n) { g_launches.fetch_add(n); }

}  // namespace gn_capi

namespace {

using gn::Args;
using gn::Geom;
using gn_capi::DeviceInfo;
using gn_capi::g_launches;
using gn_capi::current_device;
using gn_capi::ranges_overlap;
using gn_capi::wait_timeout_ns;

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;

// Library-owned workspaces, one per (device, stream) on which calls without
// a caller workspace arrive, at most kMaxStreamWorkspaces per device: the
// least recently used one is freed when a further stream arrives, so that a
// caller that creates streams per request does not leak one per stream.
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    uint64_t last_use = 0;
};
constexpr int kMaxStreamWorkspaces = 8;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;
uint64_t g_workspace_clock = 0;

// Host-visible copies of the kernels' sticky status, one word per device
// index, in page-locked host memory mapped into every device (registered
// on the first call that sets up a device).  A kernel whose bounded wait
// expires sets its device's word; every entry point reads it before it
// launches anything, without synchronising.
constexpr int kStatusWords = 16384;
alignas(65536) unsigned int g_status_words[kStatusWords];
bool g_status_registered = false;

uint64_t env_u64(const char *name, uint64_t dflt)
{
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    char *end = nullptr;
    const unsigned long long r = std::strtoull(v, &end, 0);
    return (end && *end == '\0') ? static_cast<uint64_t>(r) : dflt;
}


// L2 eviction hints of the bulk copies (bit meanings in gn_internal.h).
uint32_t l2_hints()
{
    static const uint32_t h = static_cast<uint32_t>(env_u64("GN_L2_HINTS", 0));
    return h;
}

// GN_DYNAMIC_PASS2=0 keeps the fused kernel's pass 2 on its static piece
// assignment everywhere (for comparisons).
bool dynamic_pass2_enabled()
{
    static const bool on = env_u64("GN_DYNAMIC_PASS2", 1) != 0;
    return on;
}


// Channel counts an entry point serves: the power-of-two entries take the
// page's contract (C a power of two in [8, 2048]); the general entries take
// any C that is a multiple of 8 (one 16-byte vector) up to 2048.  Either way
// G divides C.
bool channels_ok(int64_t C, int64_t G, bool general)
{
    if (C < 8 || C > 2048) return false;
    if (general ? (C % 8 != 0) : ((C & (C - 1)) != 0)) return false;
    return G >= 1 && C % G == 0;
}

// Pure host checks (no CUDA call), in a fixed order.
int validate(const void *x, const float *gamma, const float *beta, const void *y, int64_t N, int64_t L,
             int64_t C, int64_t G, float eps, const float *mean_out, const float *rstd_out, bool general)
{
    if (!x || !gamma || !beta || !y) return GN_ERR_NULL;
    if (N < 1 || L < 1) return GN_ERR_SHAPE;
    if (!channels_ok(C, G, general)) return GN_ERR_CHANNELS;
    if (N > INT64_MAX / L) return GN_ERR_SHAPE;
    const int64_t rows = N * L;
    if (rows > INT64_MAX / (2 * C)) return GN_ERR_SHAPE;
    if (N > INT64_MAX / (4 * G)) return GN_ERR_SHAPE;
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(x) % 16 || addr(y) % 16) return GN_ERR_ALIGN;
    if (addr(gamma) % 4 || addr(beta) % 4) return GN_ERR_ALIGN;
    if (addr(mean_out) % 4 || addr(rstd_out) % 4) return GN_ERR_ALIGN;
    if (!std::isfinite(eps) || eps < 0.f) return GN_ERR_EPS;
    const size_t bytes = static_cast<size_t>(rows) * static_cast<size_t>(2 * C);
    if (x != y && ranges_overlap(x, bytes, y, bytes)) return GN_ERR_ALIAS;
    const size_t cb = static_cast<size_t>(4 * C);
    if (ranges_overlap(y, bytes, gamma, cb) || ranges_overlap(y, bytes, beta, cb)) return GN_ERR_ALIAS;
    const size_t sb = static_cast<size_t>(4 * N * G);
    for (const float *s : {mean_out, rstd_out}) {
        if (!s) continue;
        if (ranges_overlap(s, sb, y, bytes) || ranges_overlap(s, sb, x, bytes) ||
            ranges_overlap(s, sb, gamma, cb) || ranges_overlap(s, sb, beta, cb))
            return GN_ERR_ALIAS;
    }
    if (mean_out && rstd_out && ranges_overlap(mean_out, sb, rstd_out, sb)) return GN_ERR_ALIAS;
    return GN_OK;
}


struct Plan {
    Geom g{};
    gn::ClusterPlan cl{};    // the cluster schedule's layout (kind GN_VARIANT_CLUSTER)
    int kind = 0;            // GN_VARIANT_TWO_PASS, GN_VARIANT_FUSED or GN_VARIANT_CLUSTER
    int grid = 0;
    size_t off_partial = 0, off_gstat = 0, off_st = 0, off_mean = 0, off_rstd = 0;
    size_t ws_bytes = 0;
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Geometry of one schedule: piece size, segments per batch entry, grid and
// ring depth; plus the workspace layout.
Plan make_plan(int64_t N, int64_t L, int64_t C, int64_t G, int kind, const DeviceInfo &d)
{
    Plan p;
    p.kind = kind;
    Geom &g = p.g;
    g.N = N;
    g.L = L;
    g.C = static_cast<int32_t>(C);
    g.G = static_cast<int32_t>(G);
    g.Cg = static_cast<int32_t>(C / G);
    g.V = static_cast<int32_t>(C / 8);
    g.A = (gn::kConsumers / g.V) * g.V;
    const int64_t row_bytes = 2 * C;
    const int64_t grid_target = d.sm_count;   // one CTA per SM (288 threads, most of shared memory)
    const int64_t total_bytes = N * L * row_bytes;
    // pieces of whole rows, as large as 32 KB and at most kMaxVecPerThread
    // vectors per data-carrying consumer thread; smaller when that leaves
    // fewer than about four pieces per CTA; never below one row
    const int64_t pb_cap = std::min<int64_t>(gn::kMaxPieceBytes, int64_t(g.A) * gn::kMaxVecPerThread * 16);
    int64_t pb = pb_cap / row_bytes * row_bytes;
    while (pb > row_bytes && pb > gn::kMinPieceBytes && total_bytes / pb < 4 * grid_target)
        pb = std::max<int64_t>(row_bytes, (pb / 2) / row_bytes * row_bytes);
    g.piece_bytes = static_cast<int32_t>(pb);
    g.rows_per_piece = static_cast<int32_t>(pb / row_bytes);
    g.pieces_per_n = (L + g.rows_per_piece - 1) / g.rows_per_piece;
    int64_t S = grid_target / N;
    if (S < 1) S = 1;
    if (S > g.pieces_per_n) S = g.pieces_per_n;
    const int64_t max_seg = (kind == GN_VARIANT_FUSED) ? gn::kFusedMaxSegments : gn::kMaxSegments;
    if (S > max_seg) S = max_seg;
    g.S = static_cast<int32_t>(S);
    g.seg32 = (g.pieces_per_n < (int64_t(1) << 32)) ? 1 : 0;
    g.base_pieces = (g.pieces_per_n - 1) / g.S;
    g.last_item = static_cast<int32_t>((g.pieces_per_n - 1) % g.S);
    g.tail_rows = static_cast<int32_t>(L - (g.pieces_per_n - 1) * g.rows_per_piece);
    g.inv_L = static_cast<float>(1.0 / static_cast<double>(L));
    g.inv_LCg = static_cast<float>(1.0 / (static_cast<double>(L) * static_cast<double>(g.Cg)));
    g.Cg_pow2 = (g.Cg & (g.Cg - 1)) == 0 ? 1 : 0;
    g.log2_Cg = 0;
    while ((1 << g.log2_Cg) < g.Cg) ++g.log2_Cg;
    // per-CTA merge of the fused kernel: enough lanes per group that each
    // holds at most kStatRecords records, and as many as the 256 consumer
    // threads allow for few groups
    int lanes = 1;
    while (lanes < 32 && (S + lanes - 1) / lanes > gn::kStatRecords) lanes *= 2;
    int spread = 1;
    while (spread < 32 && spread * 2 * G <= gn::kConsumers) spread *= 2;
    g.stat_lanes = std::max(lanes, spread);
    g.stat_log2 = 0;
    while ((1 << g.stat_log2) < g.stat_lanes) ++g.stat_log2;
    const int per_pass = gn::kConsumers / g.stat_lanes;
    g.stat_passes = static_cast<int32_t>((G + per_pass - 1) / per_pass);
    g.rows_lo = static_cast<float>(g.base_pieces * g.rows_per_piece);
    g.rows_hi = static_cast<float>((g.base_pieces + 1) * g.rows_per_piece);
    g.rows_short = static_cast<float>(g.rows_per_piece - g.tail_rows);
    g.items = N * S;
    p.grid = static_cast<int>(g.items < grid_target ? g.items : grid_target);
    // ring depth from the shared memory left next to the auxiliary arrays
    const int kind_smem = (kind == GN_VARIANT_FUSED) ? gn::kFused : gn::kPass1;
    const int64_t budget = d.smem_optin;
    int64_t ring = (budget - static_cast<int64_t>(gn::aux_smem_bytes(g, kind_smem))) / pb;
    if (ring > gn::kMaxRing) ring = gn::kMaxRing;
    g.ring = static_cast<int32_t>(ring);
    // the fused kernel deals out pass 2 at run time for one batch entry
    // with one item per CTA and at least eight ring-fulls of pieces per CTA
    // (measured: 512 MiB 254 -> 243 us, 256 MiB 127.0 -> 125.8 us, but 96-128
    // MiB 49.8 -> 52.7 and 65.7 -> 68.9 us, where the unequal streaming
    // rates of the SMs matter less than taking pieces from the counter)
    g.dyn_top = g.base_pieces - g.ring;
    g.dyn_p2 = (kind == GN_VARIANT_FUSED && N == 1 && g.items == p.grid && g.base_pieces >= 8 * ring &&
                dynamic_pass2_enabled())
                   ? 1
                   : 0;
    // workspace
    size_t off = 256;   // barrier words
    p.off_partial = off;
    off = align256(off + static_cast<size_t>(N) * G * S * sizeof(float2));
    p.off_gstat = off;
    off = align256(off + static_cast<size_t>(N) * G * sizeof(float2));
    p.off_st = off;
    off = align256(off + static_cast<size_t>(N) * C * sizeof(float2));
    p.off_mean = off;
    off = align256(off + static_cast<size_t>(N) * G * sizeof(float));
    p.off_rstd = off;
    off = align256(off + static_cast<size_t>(N) * G * sizeof(float));
    p.ws_bytes = off;
    return p;
}

bool fused_launchable(const Plan &p, const DeviceInfo &d)
{
    if (!d.coop || p.g.ring < 2) return false;
    int blocks = 0;
    const uint32_t smem = gn::make_layout(p.g, gn::kFused).total;
    if (smem > static_cast<uint32_t>(d.smem_optin)) return false;
    if (gn::fused_blocks_per_sm(true, smem, &blocks) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return blocks >= 1 && p.grid <= blocks * d.sm_count;
}

// Whether the automatic choice takes the cluster schedule's layout: one
// round of clusters, and few enough 16-byte vectors per CTA that copying
// its slice rows (16-64 bytes each, one request per row segment) costs less
// than the fused schedule's grid barrier and global merge.  Measured on a
// GB300 (graph of calls, inputs larger than L2): up to 2048 vectors per CTA
// the cluster schedule takes 6.8-8.5 us against 10.6-11.6 us; up to 8192
// vectors with 32-byte or wider row segments (rows copied by tensor-map
// boxes beyond 2048) it still wins (16 MiB, C = 512: 13.9 against 15.1 us;
// 8 MiB, C = 256: 11.0 against 12.0), with 16-byte ones only up to about
// 3072; at 10924 vectors (16 MiB, C = 128) it loses (15.7 against 15.1).
bool cluster_preferred(const gn::ClusterPlan &cp)
{
    const int64_t vectors = static_cast<int64_t>(cp.R) * (cp.SC / 8);
    return cp.waves == 1 && (vectors <= 2048 || (vectors <= 8192 && cp.SC >= 16) || vectors <= 3072);
}

// The automatic choice: the cluster schedule where it is the faster one
// (x read once, no grid barrier; cluster_preferred), else the fused
// cooperative schedule when it can launch, else two passes.
int resolve_variant(int variant, int64_t N, int64_t L, int64_t C, int64_t G, const DeviceInfo &d, Plan *out)
{
    if (variant == GN_VARIANT_CLUSTER || variant == GN_VARIANT_AUTO) {
        gn::ClusterPlan cp;
        const bool ok = gn::plan_cluster(N, L, static_cast<int>(C), static_cast<int>(G), d.cluster_cap,
                                         d.smem_optin, &cp);
        if (ok && (variant == GN_VARIANT_CLUSTER || cluster_preferred(cp))) {
            *out = Plan{};
            out->kind = GN_VARIANT_CLUSTER;
            out->cl = cp;
            return GN_OK;
        }
        if (variant == GN_VARIANT_CLUSTER) return GN_ERR_VARIANT;
    }
    if (variant == GN_VARIANT_TWO_PASS) {
        *out = make_plan(N, L, C, G, GN_VARIANT_TWO_PASS, d);
        return out->g.ring >= 2 ? GN_OK : GN_ERR_VARIANT;
    }
    if (variant == GN_VARIANT_FUSED || variant == GN_VARIANT_AUTO) {
        Plan f = make_plan(N, L, C, G, GN_VARIANT_FUSED, d);
        if (fused_launchable(f, d)) {
            *out = f;
            return GN_OK;
        }
        if (variant == GN_VARIANT_FUSED) return GN_ERR_VARIANT;
        *out = make_plan(N, L, C, G, GN_VARIANT_TWO_PASS, d);
        return out->g.ring >= 2 ? GN_OK : GN_ERR_VARIANT;
    }
    return GN_ERR_VARIANT;
}

size_t workspace_bytes_any(int64_t N, int64_t L, int64_t C, int64_t G, const DeviceInfo &d)
{
    const Plan a = make_plan(N, L, C, G, GN_VARIANT_TWO_PASS, d);
    const Plan b = make_plan(N, L, C, G, GN_VARIANT_FUSED, d);
    return a.ws_bytes > b.ws_bytes ? a.ws_bytes : b.ws_bytes;
}

// Frees one library workspace once no kernel can still be using it.
int free_workspace(Workspace &w)
{
    if (!w.ptr) return GN_OK;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaFree(w.ptr) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    w.ptr = nullptr;
    w.bytes = 0;
    return GN_OK;
}

// Library-owned workspace of (device, stream), grown on demand; a new
// stream beyond kMaxStreamWorkspaces on the device takes the place of the
// least recently used one.
int library_workspace(int dev, cudaStream_t stream, size_t bytes, void **ptr)
{
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_workspaces.find({dev, stream});
    if (it == g_workspaces.end()) {
        int count = 0;
        auto lru = g_workspaces.end();
        for (auto j = g_workspaces.begin(); j != g_workspaces.end(); ++j) {
            if (j->first.first != dev) continue;
            ++count;
            if (lru == g_workspaces.end() || j->second.last_use < lru->second.last_use) lru = j;
        }
        if (count >= kMaxStreamWorkspaces) {
            if (free_workspace(lru->second) != GN_OK) return GN_ERR_CUDA;
            g_workspaces.erase(lru);
        }
        it = g_workspaces.emplace(std::make_pair(dev, stream), Workspace{}).first;
    }
    Workspace &w = it->second;
    w.last_use = ++g_workspace_clock;
    if (w.bytes < bytes) {
        if (free_workspace(w) != GN_OK) return GN_ERR_CUDA;
        const size_t want = bytes + bytes / 4;   // headroom for nearby shapes
        void *p = nullptr;
        if (cudaMalloc(&p, want) != cudaSuccess || cudaMemset(p, 0, want) != cudaSuccess) {
            cudaGetLastError();
            if (p) cudaFree(p);
            return GN_ERR_CUDA;
        }
        w.ptr = p;
        w.bytes = want;
    }
    *ptr = w.ptr;
    return GN_OK;
}

// Every check a GroupNorm call makes before it launches: arguments, device,
// the sticky kernel status, and the schedule.
int plan_call(const void *x, const float *gamma, const float *beta, const void *y, int64_t N, int64_t L, int64_t C,
              int64_t G, float eps, const float *mean_out, const float *rstd_out, const void *workspace, int variant,
              bool general, int *dev, DeviceInfo *d, Plan *p)
{
    int rc = validate(x, gamma, beta, y, N, L, C, G, eps, mean_out, rstd_out, general);
    if (rc != GN_OK) return rc;
    if (variant < GN_VARIANT_AUTO || variant > GN_VARIANT_CLUSTER) return GN_ERR_VARIANT;
    if (workspace && reinterpret_cast<uintptr_t>(workspace) % 256) return GN_ERR_ALIGN;
    if ((rc = current_device(dev, d)) != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(*dev)) return GN_ERR_KERNEL;
    return resolve_variant(variant, N, L, C, G, *d, p);
}

int run(const void *x, const float *gamma, const float *beta, void *y, int64_t N, int64_t L, int64_t C,
        int64_t G, float eps, int apply_silu, float *mean_out, float *rstd_out, void *workspace,
        size_t workspace_bytes, int variant, void *stream, bool general = false)
{
    int dev = -1;
    DeviceInfo d;
    Plan p;
    int rc = plan_call(x, gamma, beta, y, N, L, C, G, eps, mean_out, rstd_out, workspace, variant, general, &dev,
                       &d, &p);
    if (rc != GN_OK) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (workspace && workspace_bytes < workspace_bytes_any(N, L, C, G, d)) return GN_ERR_WORKSPACE;
    if (p.kind == GN_VARIANT_CLUSTER) {
        // everything stays in the clusters' shared memory: no workspace
        const cudaError_t e = gn::launch_cluster(p.cl, static_cast<const uint16_t *>(x), static_cast<uint16_t *>(y),
                                                 gamma, beta, mean_out, rstd_out, eps, apply_silu != 0, N, L,
                                                 static_cast<int>(C), static_cast<int>(G), wait_timeout_ns(),
                                                 d.status_word, d.status_host, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GN_ERR_CUDA;
        }
        g_launches.fetch_add(1);
        return GN_OK;
    }
    void *ws = workspace;
    if (!ws && (rc = library_workspace(dev, s, workspace_bytes_any(N, L, C, G, d), &ws)) != GN_OK) return rc;
    uint8_t *base = static_cast<uint8_t *>(ws);
    Args a{};
    a.x = static_cast<const uint16_t *>(x);
    a.y = static_cast<uint16_t *>(y);
    a.gamma = gamma;
    a.beta = beta;
    a.eps = eps;
    a.l2_hints = l2_hints();
    a.g = p.g;
    a.partial = reinterpret_cast<float2 *>(base + p.off_partial);
    a.gstat = reinterpret_cast<float2 *>(base + p.off_gstat);
    a.st = reinterpret_cast<float2 *>(base + p.off_st);
    a.mean = mean_out ? mean_out : reinterpret_cast<float *>(base + p.off_mean);
    a.rstd = rstd_out ? rstd_out : reinterpret_cast<float *>(base + p.off_rstd);
    a.sync = reinterpret_cast<unsigned int *>(base);
    a.timeout_ns = wait_timeout_ns();
    const bool silu = apply_silu != 0;
    cudaError_t e;
    if (p.kind == GN_VARIANT_FUSED) {
        e = gn::launch_fused(a, p.grid, silu, s);
        if (e == cudaSuccess) g_launches.fetch_add(1);
    } else {
        e = gn::launch_pass1(a, p.grid, s);
        if (e == cudaSuccess) {
            g_launches.fetch_add(1);
            e = gn::launch_finalize(a, s);
        }
        if (e == cudaSuccess) {
            g_launches.fetch_add(1);
            e = gn::launch_pass2(a, p.grid, silu, s);
        }
        if (e == cudaSuccess) g_launches.fetch_add(1);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    return GN_OK;
}

}  // namespace

namespace gn_capi {

int check_rows_call(const void *x, const float *gamma, const float *beta, const void *y, int64_t N, int64_t L,
                    int64_t C, int64_t G, float eps, const float *mean_out, const float *rstd_out,
                    size_t *workspace_need)
{
    int dev = -1;
    DeviceInfo d;
    Plan p;
    const int rc = plan_call(x, gamma, beta, y, N, L, C, G, eps, mean_out, rstd_out, nullptr, GN_VARIANT_AUTO,
                             false, &dev, &d, &p);
    if (rc != GN_OK) return rc;
    *workspace_need = workspace_bytes_any(N, L, C, G, d);
    return GN_OK;
}

bool kernel_status_raised(int dev)
{
    if (dev < 0 || dev >= kStatusWords) return false;
    return reinterpret_cast<volatile unsigned int *>(g_status_words)[dev] != 0u;
}

// Timeout of every bounded wait inside the kernels.
uint64_t wait_timeout_ns()
{
    static const uint64_t t = env_u64("GN_WAIT_TIMEOUT_MS", 2000) * 1000000ull;
    return t;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// Current device, checked to be an sm_103 part; kernel attributes set once.
int current_device(int *dev_out, DeviceInfo *info_out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ||
            cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev)) {
            cudaGetLastError();
            return GN_ERR_DEVICE;
        }
        if (d.major != 10 || d.minor != 3 || dev >= kStatusWords) return GN_ERR_DEVICE;
        if (gn::prepare_kernels(static_cast<uint32_t>(d.smem_optin)) != cudaSuccess ||
            gn::prepare_cluster_kernels(d.smem_optin, d.cluster_cap) != cudaSuccess) {
            cudaGetLastError();
            return GN_ERR_CUDA;
        }
        // map this device's status word (registering the words once) and
        // hand its device address to the kernel files
        if (!g_status_registered) {
            if (cudaHostRegister(g_status_words, sizeof(g_status_words),
                                 cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
                cudaGetLastError();
                return GN_ERR_CUDA;
            }
            g_status_registered = true;
        }
        void *word = nullptr;
        if (cudaHostGetDevicePointer(&word, &g_status_words[dev], 0) != cudaSuccess || !word ||
            gn::set_device_status_host(static_cast<unsigned int *>(word)) != cudaSuccess ||
            gn::device_status_address(&d.status_word) != cudaSuccess ||
            gn::set_upconv_status_host(static_cast<unsigned int *>(word)) != cudaSuccess ||
            gn::set_attn_status_host(static_cast<unsigned int *>(word)) != cudaSuccess) {
            cudaGetLastError();
            return GN_ERR_CUDA;
        }
        d.status_host = static_cast<unsigned int *>(word);
        d.ready = true;
    }
    *dev_out = dev;
    *info_out = d;
    return GN_OK;
}

}  // namespace gn_capi

extern "C" {

int gn_silu_rows_ex(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16, int64_t N,
                    int64_t L, int64_t C, int64_t G, float eps, int apply_silu, float *mean_out,
                    float *rstd_out, void *workspace, size_t workspace_bytes, int variant, void *stream)
{
    return run(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, apply_silu, mean_out, rstd_out, workspace,
               workspace_bytes, variant, stream);
}

int gn_silu_rows_any(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16, int64_t N,
                     int64_t L, int64_t C, int64_t G, float eps, int apply_silu, float *mean_out,
                     float *rstd_out, void *workspace, size_t workspace_bytes, int variant, void *stream)
{
    return run(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, apply_silu, mean_out, rstd_out, workspace,
               workspace_bytes, variant, stream, true);
}

int gn_silu_ndhwc(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16, int64_t N,
                  int64_t D, int64_t H, int64_t W, int64_t C, int64_t G, float eps, int apply_silu,
                  void *stream)
{
    if (D < 1 || H < 1 || W < 1 || H > INT64_MAX / W || D > INT64_MAX / (H * W)) {
        if (!x_bf16 || !gamma || !beta || !y_bf16) return GN_ERR_NULL;
        return GN_ERR_SHAPE;
    }
    return run(x_bf16, gamma, beta, y_bf16, N, D * H * W, C, G, eps, apply_silu, nullptr, nullptr, nullptr, 0,
               GN_VARIANT_AUTO, stream, true);
}

int gn_silu_rows(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16, int64_t N,
                 int64_t L, int64_t C, int64_t G, float eps, int apply_silu, void *stream)
{
    return run(x_bf16, gamma, beta, y_bf16, N, L, C, G, eps, apply_silu, nullptr, nullptr, nullptr, 0,
               GN_VARIANT_AUTO, stream);
}

int gn_silu_nhwc(const void *x_bf16, const float *gamma, const float *beta, void *y_bf16, int64_t N,
                 int64_t H, int64_t W, int64_t C, int64_t G, float eps, int apply_silu, void *stream)
{
    if (H < 1 || W < 1 || H > INT64_MAX / W) {
        if (!x_bf16 || !gamma || !beta || !y_bf16) return GN_ERR_NULL;
        return GN_ERR_SHAPE;
    }
    return gn_silu_rows(x_bf16, gamma, beta, y_bf16, N, H * W, C, G, eps, apply_silu, stream);
}

size_t gn_silu_workspace_bytes(int64_t N, int64_t L, int64_t C, int64_t G)
{
    if (N < 1 || L < 1 || N > INT64_MAX / L || N * L > INT64_MAX / (2 * 2048)) return 0;
    if (!channels_ok(C, G, true)) return 0;
    int dev = -1;
    DeviceInfo d;
    if (current_device(&dev, &d) != GN_OK) return 0;
    return workspace_bytes_any(N, L, C, G, d);
}

int gn_silu_pick_variant(int64_t N, int64_t L, int64_t C, int64_t G)
{
    if (N < 1 || L < 1 || N > INT64_MAX / L) return -GN_ERR_SHAPE;
    if (!channels_ok(C, G, true)) return -GN_ERR_CHANNELS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return -rc;
    Plan p;
    const int r = resolve_variant(GN_VARIANT_AUTO, N, L, C, G, d, &p);
    return r == GN_OK ? p.kind : -r;
}

uint64_t gn_kernel_launch_count(void) { return g_launches.load(); }

int gn_device_status(int clear)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_DEVICE;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return GN_ERR_CUDA;
    unsigned int st = 0, st_uc = 0, st_at = 0;
    if (gn::read_device_status(&st) != cudaSuccess) return GN_ERR_CUDA;
    if (gn::read_upconv_status(&st_uc) != cudaSuccess) return GN_ERR_CUDA;
    if (gn::read_attn_status(&st_at) != cudaSuccess) return GN_ERR_CUDA;
    st |= st_uc | st_at;
    if (gn_capi::kernel_status_raised(dev)) st |= 1u;
    if (clear) {
        if (gn::clear_device_status() != cudaSuccess) return GN_ERR_CUDA;
        if (gn::clear_upconv_status() != cudaSuccess) return GN_ERR_CUDA;
        if (gn::clear_attn_status() != cudaSuccess) return GN_ERR_CUDA;
        if (dev < kStatusWords) reinterpret_cast<volatile unsigned int *>(g_status_words)[dev] = 0u;
        std::lock_guard<std::mutex> lock(g_mu);
        for (auto &kv : g_workspaces) {
            if (kv.first.first == dev && kv.second.ptr && cudaMemset(kv.second.ptr, 0, 256) != cudaSuccess)
                return GN_ERR_CUDA;
        }
    }
    return st ? GN_ERR_KERNEL : GN_OK;
}

int gn_release_workspaces(void)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto it = g_workspaces.begin(); it != g_workspaces.end();) {
        if (it->first.first != dev) {
            ++it;
            continue;
        }
        if (free_workspace(it->second) != GN_OK) return GN_ERR_CUDA;
        it = g_workspaces.erase(it);
    }
    return GN_OK;
}

int gn_library_workspaces(void)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -GN_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    int count = 0;
    for (const auto &kv : g_workspaces)
        if (kv.first.first == dev && kv.second.ptr) ++count;
    return count;
}

int gn_selftest_bounded_wait(int mode, int timeout_ms, int *done, int blocks, void *stream)
{
    if (mode < 0 || mode > 1 || timeout_ms < 0 || timeout_ms > 10000 || blocks < 1 || blocks > 1024)
        return GN_ERR_SHAPE;
    if (!done) return GN_ERR_NULL;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    const cudaError_t e = gn::launch_selftest_wait(mode, static_cast<uint64_t>(timeout_ms) * 1000000ull, done,
                                                   blocks, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    g_launches.fetch_add(1);
    return GN_OK;
}

const char *gn_status_string(int status)
{
    switch (status) {
    case GN_OK: return "GN_OK: success";
    case GN_ERR_NULL: return "GN_ERR_NULL: a required pointer is NULL";
    case GN_ERR_SHAPE: return "GN_ERR_SHAPE: N, L, H or W below 1, or the element count overflows";
    case GN_ERR_CHANNELS:
        return "GN_ERR_CHANNELS: C must be a power of two in [8, 2048] (a multiple of 8 up to 2048 for "
               "gn_silu_rows_any / gn_silu_ndhwc) and G must divide C";
    case GN_ERR_ALIGN: return "GN_ERR_ALIGN: x/y need 16-byte, gamma/beta/statistics 4-byte, workspace 256-byte alignment";
    case GN_ERR_EPS: return "GN_ERR_EPS: eps must be finite and non-negative";
    case GN_ERR_ALIAS: return "GN_ERR_ALIAS: y overlaps x (other than in place) or another argument";
    case GN_ERR_WORKSPACE: return "GN_ERR_WORKSPACE: workspace smaller than gn_silu_workspace_bytes()";
    case GN_ERR_CUDA: return "GN_ERR_CUDA: a CUDA call or kernel launch failed";
    case GN_ERR_DEVICE: return "GN_ERR_DEVICE: no CUDA device, or the device is not sm_103";
    case GN_ERR_VARIANT: return "GN_ERR_VARIANT: unknown variant, or it cannot be launched for this shape";
    case GN_ERR_KERNEL: return "GN_ERR_KERNEL: a kernel gave up a bounded wait";
    case GN_ERR_FORMAT: return "GN_ERR_FORMAT: the half format is neither bf16 (0) nor fp16 (1)";
    default: return "unknown gn status";
    }
}

int gn_residual_gate_add(const void *residual, const void *update, const void *gate, void *out, int64_t rows,
                         int64_t D, int format, void *stream)
{
    if (!residual || !update || !gate || !out) return GN_ERR_NULL;
    if (rows < 0) return GN_ERR_SHAPE;
    if (D < 8 || D % 8 != 0) return GN_ERR_CHANNELS;
    if (rows > 0 && rows > INT64_MAX / (2 * D)) return GN_ERR_SHAPE;
    const auto addr = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(residual) % 16 || addr(update) % 16 || addr(gate) % 16 || addr(out) % 16) return GN_ERR_ALIGN;
    if (format != GN_FORMAT_BF16 && format != GN_FORMAT_FP16) return GN_ERR_FORMAT;
    const size_t bytes = static_cast<size_t>(rows) * static_cast<size_t>(2 * D);
    const size_t gbytes = static_cast<size_t>(2 * D);
    if (out != residual && ranges_overlap(out, bytes, residual, bytes)) return GN_ERR_ALIAS;
    if (out != update && ranges_overlap(out, bytes, update, bytes)) return GN_ERR_ALIAS;
    if (ranges_overlap(out, bytes, gate, gbytes)) return GN_ERR_ALIAS;
    int dev = -1;
    DeviceInfo d;
    const int rc = current_device(&dev, &d);
    if (rc != GN_OK) return rc;
    if (gn_capi::kernel_status_raised(dev)) return GN_ERR_KERNEL;
    if (rows == 0) return GN_OK;
    // eight resident blocks per SM to keep HBM busy; a tensor with fewer
    // vectors gets one vector per thread, so that its blocks spread over the
    // SMs evenly (at 512 x 3072, 768 blocks took 3.43 us a call against
    // 3.65 us for 192 blocks of four vectors per thread, which left two
    // blocks' data on 40 SMs and one on the rest)
    const int64_t nvec = rows * (D / 8);
    const int64_t want = (nvec + gn::kRgaThreads - 1) / gn::kRgaThreads;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8LL * d.sm_count)));
    const cudaError_t e = gn::launch_residual_gate(residual, update, gate, out, rows, D, format == GN_FORMAT_BF16,
                                                   blocks, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GN_ERR_CUDA;
    }
    g_launches.fetch_add(1);
    return GN_OK;
}

int gn_abi_version(void) { return 7; }

}  // extern "C"
