// gn_cluster.cu -- the cluster schedule of channels-last GroupNorm (+SiLU),
// for tensors that fit in the SMs' shared memory.
//
// The computation is that of gn_kernels.cu (sglang PR #33451, "FLUX.2 VAE
// decoder fast path behind quality=high", section "Modifications", item 1:
// a per-(batch, group) reduction over (N, L, C) rows, a finalize to mean /
// rstd with the affine folded into per-channel scale / shift, and the
// elementwise apply with optional SiLU), scheduled so that no statistic
// crosses L2 and no grid-wide barrier is needed:
//  * The channels are cut into slices of whole groups (SC channels, a
//    multiple of Cg and of 8); one unit of work is one (batch entry, slice).
//  * Each unit belongs to one thread-block cluster of CL CTAs.  CTA r of the
//    cluster owns rows [r R, (r + 1) R) of the unit and copies that R x SC
//    block once from HBM into its shared memory, where it stays until its
//    outputs are written: x is read once.  Every thread copies (cp.async,
//    16 bytes) exactly the vectors it later reduces and applies, in boxes
//    of rows whose mbarriers complete when all threads' copies of the box
//    have landed.  (A slice row is only 16-512 bytes long; tensor-map copies
//    of such narrow boxes are issued one row request at a time and were
//    several times slower.)
//  * Pass 1 reduces the box to one (mean, M2) record per group.  After a
//    cluster barrier every CTA reads the CL records of each of the slice's
//    groups from the other CTAs' shared memory (distributed shared memory)
//    and merges them in rank order, so all CTAs of the cluster hold the same
//    mean and rstd, bit for bit.
//  * Pass 2 applies scale / shift (+ SiLU) to the resident box and writes y
//    with 16-byte stores.
//  * Waits on the copies are bounded: a timeout records the sticky status
//    (the word the other GroupNorm kernels share, and its mapped host copy)
//    and the CTA skips its work; a launch that finds the status set writes
//    nothing.
//    Every thread passes both cluster barriers on every path, and the
//    second one keeps each CTA's records in place until the whole cluster
//    has read them.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "gn_internal.h"
#include "gn_math.cuh"
#include "gn_ptx.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace gn {

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the kernel ahead of it in the stream has
// finished, once every CTA of that kernel has signalled (or exited); it
// touches no global memory before griddep_wait returns.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


namespace {

constexpr int kClThreads = 512;
constexpr int kClMaxBoxRows = 256;     // rows per box (one mbarrier each)

struct ClArgs {
    CUtensorMap map;           // x as [N L rows][C], boxes of BR rows x SC channels (tma only)
    const uint16_t *x;
    uint16_t *y;
    const float *gamma, *beta;
    float *mean, *rstd;        // [N][G] or null
    float eps;
    float inv_L, inv_LCg;      // 1 / L and 1 / (L Cg)
    int32_t L, C, G, Cg;
    int32_t SC, VS, slices;    // slice channels, 16-byte vectors per slice row, slices per row
    int32_t A, P;              // threads that carry data, rows per pass (A = P * VS)
    int32_t vs_pow2;           // VS is a power of two: channel sums reduce across a warp by shuffles
    int32_t R, BR, boxes;      // rows per CTA, rows per box, boxes per CTA
    int32_t cl;                // CTAs per cluster
    int32_t tma;               // copy the rows with tensor-map boxes (one thread) instead of 16-byte copies
    uint64_t timeout_ns;
    unsigned int *status;        // the GroupNorm kernels' sticky status word (device memory)
    unsigned int *status_host;   // its host-visible copy (mapped page-locked host memory)
};

// Shared memory of one CTA: the resident rows, the channel sums, the
// per-group records and statistics, gamma / beta of the slice, the box
// mbarriers and the abort flag.
struct ClLayout {
    uint32_t box, scratch, rec, gst, gb, bars, flag, total;
};

__host__ __device__ inline ClLayout cl_layout(int SC, int Cg, int BR, int boxes, int A)
{
    ClLayout l;
    uint32_t off = 0;
    l.box = off;
    off += static_cast<uint32_t>(boxes) * static_cast<uint32_t>(BR) * static_cast<uint32_t>(SC) * 2u;
    off = align_up(off, 128);
    l.scratch = off;
    off += static_cast<uint32_t>(A) * 8u * 8u;
    const uint32_t ngl = static_cast<uint32_t>(SC / Cg);
    l.rec = off;
    off += 8u * ngl;
    l.gst = off;
    off += 8u * ngl;
    l.gb = off;
    off += 8u * static_cast<uint32_t>(SC);
    off = align_up(off, 16);
    l.bars = off;
    off += 8u * static_cast<uint32_t>(boxes);
    l.flag = off;
    off += 16;
    l.total = off;
    return l;
}

// 16 bytes global -> shared through L2 only; completion tracked below
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The mbarrier receives one arrival from this thread once all its earlier
// cp.async copies have landed (its expected count includes that arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ void stg128(uint16_t *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

template <bool SILU>
__global__ void __launch_bounds__(kClThreads, 1)
    gn_cluster_kernel(const __grid_constant__ ClArgs a)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    const ClLayout lay = cl_layout(a.SC, a.Cg, a.BR, a.boxes, a.A);
    const uint32_t base = smem_addr(sm);
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int unit = static_cast<int>(blockIdx.x) / a.cl;
    const int n = unit / a.slices;
    const int s = unit - n * a.slices;
    const int row0 = static_cast<int>(rank) * a.R;
    const int rows = max(0, min(a.R, a.L - row0));   // rows of the unit this CTA owns
    const int issued = (rows + a.BR - 1) / a.BR;      // boxes it copies
    const uint32_t bars = base + lay.bars;
    volatile int *abort = reinterpret_cast<volatile int *>(sm + lay.flag);
    // shared memory only until the kernel ahead in the stream has finished;
    // then a kernel launched after this one the same way may start (it waits
    // the same way)
    if (tid == 0) {
        *abort = 0;
        for (int b = 0; b < issued; ++b) mbar_init(bars + 8u * b, a.tma ? 1 : kClThreads);
        mbar_init_fence();
    }
    griddep_wait();
    if (tid == 0) griddep_launch_dependents();
    // Loads whose values are needed only later go out first, so that their
    // latency hides behind the copies: the sticky status (checked before
    // anything is written) and gamma / beta of the slice.
    const unsigned int status0 = (tid == 0) ? *reinterpret_cast<volatile unsigned int *>(a.status) : 0u;
    float gam = 0.f, bet = 0.f;
    if (tid < a.SC) {
        gam = __ldg(a.gamma + s * a.SC + tid);
        bet = __ldg(a.beta + s * a.SC + tid);
    }
    __syncthreads();
    const int VS = a.VS;
    const bool carrier = tid < a.A;
    const int vslot = tid % VS;
    const int rk = tid / VS;
    const uint32_t row_bytes = static_cast<uint32_t>(a.SC) * 2u;
    const uint32_t vaddr = base + lay.box + static_cast<uint32_t>(vslot) * 16u;
    if (a.tma) {
        // one thread copies the CTA's rows, box by box: a box is BR rows of
        // the slice (the last one may run past the CTA's rows: those are read
        // and not used, and rows past the tensor arrive as zeros)
        if (tid == 0) {
            for (int b = 0; b < issued; ++b) {
                mbar_arrive_expect_tx(bars + 8u * b, static_cast<uint32_t>(a.BR) * row_bytes);
                tma_load_2d(base + lay.box + static_cast<uint32_t>(b * a.BR) * row_bytes, &a.map, s * a.SC,
                            n * a.L + row0 + b * a.BR, bars + 8u * b);
            }
        }
    } else {
        // the vectors this thread reduces and applies, box by box; every
        // thread arrives on every box's mbarrier
        const uint16_t *src = a.x + (static_cast<int64_t>(n) * a.L + row0) * a.C + s * a.SC + 8 * vslot;
        int lr = rk;
        for (int b = 0; b < issued; ++b) {
            const int end = min(rows, (b + 1) * a.BR);
            if (carrier) {
                for (; lr < end; lr += a.P)
                    cp_async16(vaddr + static_cast<uint32_t>(lr) * row_bytes, src + static_cast<int64_t>(lr) * a.C);
            }
            cp_async_arrive(bars + 8u * b);
        }
    }

    // ---- pass 1: per-channel sums of (x - K), K the group's first value ----
    f2_t s1[4], s2[4], K[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s1[i] = pk(0.f, 0.f);
        s2[i] = pk(0.f, 0.f);
        K[i] = pk(0.f, 0.f);
    }
    if (carrier && rk < rows && tc::wait(bars, 0, abort, a.timeout_ns, a.status, a.status_host)) {
        float kc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ch = 8 * vslot + i;
            kc[i] = __uint_as_float(lds_u16(base + lay.box + 2u * static_cast<uint32_t>((ch / a.Cg) * a.Cg)) << 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) K[i] = pk(kc[2 * i], kc[2 * i + 1]);
        int bound = a.BR;   // first row of the next box not yet waited for
        int b = 1;
#pragma unroll 4
        for (int lr = rk; lr < rows; lr += a.P) {
            while (lr >= bound) {
                if (!tc::wait(bars + 8u * b, 0, abort, a.timeout_ns, a.status, a.status_host)) break;
                ++b;
                bound += a.BR;
            }
            if (lr >= bound) break;
            const uint4 w = lds128(vaddr + static_cast<uint32_t>(lr) * row_bytes);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const f2_t d = sub2(bf2_to_f2(ws[i]), K[i]);
                s1[i] = add2(s1[i], d);
                s2[i] = fma2(d, d, s2[i]);
            }
        }
    }
    // per-channel partial sums in shared memory: with VS a power of two the
    // lanes of a warp that hold the same channels are first combined by
    // shuffles, leaving one entry per (warp, channel); otherwise one entry
    // per (thread, channel).  Entry of channel ch from row rank r (warp or
    // thread row): scratch[8 (ch / 8 + VS r) + ch % 8].
    float2 *scratch = reinterpret_cast<float2 *>(sm + lay.scratch);
    {
        float c1[8], c2[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            upk(s1[i], c1[2 * i], c1[2 * i + 1]);
            upk(s2[i], c2[2 * i], c2[2 * i + 1]);
        }
        if (a.vs_pow2) {
            for (int off = VS; off < 32; off <<= 1) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c1[j] += __shfl_xor_sync(0xffffffffu, c1[j], off);
                    c2[j] += __shfl_xor_sync(0xffffffffu, c2[j], off);
                }
            }
            if ((tid & 31) < VS) {
                const int e = 8 * (vslot + VS * (tid >> 5));
#pragma unroll
                for (int j = 0; j < 8; ++j) scratch[e + j] = make_float2(c1[j], c2[j]);
            }
        } else if (carrier) {
#pragma unroll
            for (int j = 0; j < 8; ++j) scratch[8 * tid + j] = make_float2(c1[j], c2[j]);
        }
    }
    float2 *gb = reinterpret_cast<float2 *>(sm + lay.gb);
    if (tid < a.SC) gb[tid] = make_float2(gam, bet);
    if (status0 != 0u) *abort = 1;
    __syncthreads();

    // ---- per-CTA record of each group of the slice: (mean, M2) over its rows ----
    const int ngl = a.SC / a.Cg;
    float2 *rec = reinterpret_cast<float2 *>(sm + lay.rec);
    {
        const int warp = tid >> 5, lane = tid & 31;
        const int ranks = a.vs_pow2 ? kClThreads / 32 : a.P;
        const int entries = ranks * a.Cg;
        for (int gl = warp; gl < ngl; gl += kClThreads / 32) {
            float t1 = 0.f, t2 = 0.f;
            for (int e = lane; e < entries; e += 32) {
                const int r = e / a.Cg;
                const int ch = gl * a.Cg + (e - r * a.Cg);
                const float2 v = scratch[8 * ((ch >> 3) + VS * r) + (ch & 7)];
                t1 += v.x;
                t2 += v.y;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                t1 += __shfl_xor_sync(0xffffffffu, t1, off);
                t2 += __shfl_xor_sync(0xffffffffu, t2, off);
            }
            if (lane == 0) {
                float2 r = make_float2(0.f, 0.f);
                if (rows > 0 && !*abort) {
                    const float cnt = static_cast<float>(rows) * static_cast<float>(a.Cg);
                    const float k = __uint_as_float(lds_u16(base + lay.box + 2u * static_cast<uint32_t>(gl * a.Cg)) << 16);
                    const float d = t1 / cnt;
                    r = make_float2(k + d, fmaxf(t2 - t1 * d, 0.f));
                }
                rec[gl] = r;
            }
        }
    }
    __syncwarp();
    cluster_arrive();
    cluster_wait();

    // ---- merge the cluster's records in rank order (identical in every CTA) ----
    float2 *gst = reinterpret_cast<float2 *>(sm + lay.gst);
    for (int gl = tid; gl < ngl; gl += kClThreads) {
        float2 r[kClusterMaxCtas];
        float rw[kClusterMaxCtas];
        const uint32_t own = base + lay.rec + 8u * static_cast<uint32_t>(gl);
#pragma unroll
        for (int q = 0; q < kClusterMaxCtas; ++q) {
            if (q < a.cl) {
                r[q] = ld_cluster_f2(mapa_shared(own, static_cast<uint32_t>(q)));
                rw[q] = static_cast<float>(max(0, min(a.R, a.L - q * a.R)));
            } else {
                r[q] = make_float2(0.f, 0.f);
                rw[q] = 0.f;
            }
        }
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < kClusterMaxCtas; ++q) acc = fmaf(rw[q], r[q].x, acc);
        const float mean = acc * a.inv_L;
        const float cgf = static_cast<float>(a.Cg);
        float m2 = 0.f;
#pragma unroll
        for (int q = 0; q < kClusterMaxCtas; ++q) {
            const float d = r[q].x - mean;
            m2 += fmaf(cgf * rw[q] * d, d, r[q].y);
        }
        const float rstd = rsqrtf(fmaxf(m2 * a.inv_LCg, 0.f) + a.eps);
        gst[gl] = make_float2(mean, rstd);
        if (rank == 0 && !*abort) {
            const int64_t o = static_cast<int64_t>(n) * a.G + static_cast<int64_t>(s) * ngl + gl;
            if (a.mean) a.mean[o] = mean;
            if (a.rstd) a.rstd[o] = rstd;
        }
    }
    // this CTA has read every record it needs from the others
    __syncwarp();
    cluster_arrive();
    __syncthreads();

    // ---- pass 2: y = x * scale + shift (+ SiLU) from the resident rows ----
    if (!*abort && carrier && rk < rows) {
        // scale / shift of the thread's eight channels, folded from the
        // group statistics and gamma / beta
        float sc[8], sh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ch = 8 * vslot + i;
            const float2 g = gst[ch / a.Cg];
            const float2 ab = gb[ch];
            sc[i] = ab.x * g.y;
            sh[i] = ab.y - g.x * sc[i];
        }
        f2_t S[4], T[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            S[i] = pk(sc[2 * i], sc[2 * i + 1]);
            T[i] = pk(sh[2 * i], sh[2 * i + 1]);
        }
        uint16_t *dst = a.y + (static_cast<int64_t>(n) * a.L + row0) * a.C + static_cast<int64_t>(s) * a.SC + 8 * vslot;
        const int64_t row_stride = static_cast<int64_t>(a.C);
#pragma unroll 4
        for (int lr = rk; lr < rows; lr += a.P) {
            const uint4 w = lds128(vaddr + static_cast<uint32_t>(lr) * row_bytes);
            uint4 o;
            o.x = apply_pair<SILU>(w.x, S[0], T[0]);
            o.y = apply_pair<SILU>(w.y, S[1], T[1]);
            o.z = apply_pair<SILU>(w.z, S[2], T[2]);
            o.w = apply_pair<SILU>(w.w, S[3], T[3]);
            stg128(dst + lr * row_stride, o);
        }
    }
    // after a failure, let the copies still in flight land before the CTA
    // (and its shared memory) goes away
    if (*abort && tid == 0) {
        for (int b = 0; b < issued; ++b) tc::drain(bars + 8u * b, 0, a.timeout_ns);
    }
    __syncwarp();
    cluster_wait();
}

const void *cluster_fn(bool silu)
{
    return silu ? reinterpret_cast<const void *>(gn_cluster_kernel<true>)
                : reinterpret_cast<const void *>(gn_cluster_kernel<false>);
}

// rows a pass of the CTA's threads covers: each row is VS vectors
int rows_per_pass(int VS) { return kClThreads / VS; }

}  // namespace

cudaError_t prepare_cluster_kernels(int max_smem, int (&cap)[kClusterMaxCtas + 1])
{
    for (int silu = 0; silu < 2; ++silu) {
        const void *fn = cluster_fn(silu != 0);
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cap[0] = 0;
    for (int cl = 1; cl <= kClusterMaxCtas; ++cl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cl);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(max_smem);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = cl;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, cluster_fn(true), &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cap[cl] = n;
    }
    return cudaSuccess;
}

// The cheapest (slice width, cluster size) for this shape: every unit's rows
// must fit one CTA's shared memory per cluster rank; the estimated time is
// rounds of clusters x (a fixed cost per round, worth about kFixedBytes of
// transfer per CTA, + the bytes one CTA moves).  Ties go to wider slices
// (longer contiguous row segments), then smaller clusters.
// GN_CLUSTER_PLAN="SC,CL" restricts the search to one slice width and
// cluster size, and "SC,CL,COPY" also the copy mode (0: 16-byte copies by
// every thread, 1: tensor-map boxes), for measuring the alternatives;
// unset, every layout is considered.
static void forced_plan(int *sc, int *cl, int *copy)
{
    static int f_sc = 0, f_cl = 0, f_copy = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char *v = std::getenv("GN_CLUSTER_PLAN");
        if (!v) return;
        const int got = std::sscanf(v, "%d,%d,%d", &f_sc, &f_cl, &f_copy);
        if (got < 2) {
            f_sc = f_cl = 0;
            f_copy = -1;
        } else if (got == 2) {
            f_copy = -1;
        }
    });
    *sc = f_sc;
    *cl = f_cl;
    *copy = f_copy;
}

bool plan_cluster(int64_t N, int64_t L, int C, int G, const int (&cap)[kClusterMaxCtas + 1], int max_smem,
                  ClusterPlan *out)
{
    constexpr int64_t kFixedBytes = 96 * 1024;
    int force_sc = 0, force_cl = 0, force_copy = -1;
    forced_plan(&force_sc, &force_cl, &force_copy);
    if (N < 1 || L < 1 || C % 8 != 0 || G < 1 || C % G != 0) return false;
    if (L > (int64_t(1) << 30) || N > (int64_t(1) << 30)) return false;
    const int Cg = C / G;
    int step = Cg;
    while (step % 8 != 0) step += Cg;   // lcm(Cg, 8)
    bool found = false;
    ClusterPlan best{};
    int64_t best_cost = 0;
    for (int SC = step; SC <= 256 && SC <= C; SC += step) {
        if (C % SC != 0 || (force_sc && SC != force_sc)) continue;
        const int VS = SC / 8;
        const int P = rows_per_pass(VS);
        if (P < 1) continue;
        const int A = P * VS;
        const int64_t units = N * (C / SC);
        for (int cl = 1; cl <= kClusterMaxCtas; ++cl) {
            if (cap[cl] < 1 || (force_cl && cl != force_cl)) continue;
            const int64_t R = (L + cl - 1) / cl;
            if (cl > 1 && (cl - 1) * R >= L) continue;   // a CTA with no rows
            // boxes of at most 256 rows (the granularity at which pass 1 can
            // start on rows that have landed), each a multiple of 8 rows
            const int64_t boxes = (R + kClMaxBoxRows - 1) / kClMaxBoxRows;
            const int64_t BR = ((R + boxes - 1) / boxes + 7) / 8 * 8;
            if (boxes * BR * SC * 2 > max_smem) continue;
            const ClLayout lay = cl_layout(SC, Cg, static_cast<int>(BR), static_cast<int>(boxes), A);
            if (lay.total > static_cast<uint32_t>(max_smem)) continue;
            const int64_t waves = (units + cap[cl] - 1) / cap[cl];
            // a row segment narrower than a 32-byte sector costs a whole sector
            // (measured: 16-byte segments ran 0.2-1.3 us slower than the
            // 32- or 64-byte plans of the same bytes per CTA)
            const int64_t row_cost = SC * 2 < 32 ? 32 : SC * 2;
            const int64_t cost = waves * (kFixedBytes + R * row_cost);
            const bool better = !found || cost < best_cost ||
                                (cost == best_cost && (SC > best.SC || (SC == best.SC && cl < best.CL)));
            if (!better) continue;
            found = true;
            best_cost = cost;
            best.SC = SC;
            best.CL = cl;
            best.R = static_cast<int>(R);
            best.BR = static_cast<int>(BR);
            best.boxes = static_cast<int>(boxes);
            best.units = units;
            best.waves = static_cast<int>(waves);
            best.smem = lay.total;
            // tensor-map boxes once a CTA holds more than 2048 vectors (one
            // thread then issues a box per up to 256 rows instead of every
            // thread issuing its 16-byte copies; measured: 16 MiB at
            // 16-channel slices 16.2 -> 13.7 us, up to 2048 vectors within 1 %)
            best.tma = R * (SC / 8) > 2048 ? 1 : 0;
        }
    }
    if (found && force_copy >= 0) best.tma = force_copy ? 1 : 0;
    if (found) *out = best;
    return found;
}

cudaError_t launch_cluster(const ClusterPlan &p, const uint16_t *x, uint16_t *y, const float *gamma,
                           const float *beta, float *mean, float *rstd, float eps, bool silu, int64_t N, int64_t L,
                           int C, int G, uint64_t timeout_ns, unsigned int *status, unsigned int *status_host,
                           cudaStream_t s)
{
    if (p.units * p.CL > 0x7fffffffLL) return cudaErrorInvalidValue;
    ClArgs a{};
    a.x = x;
    a.y = y;
    a.gamma = gamma;
    a.beta = beta;
    a.mean = mean;
    a.rstd = rstd;
    a.eps = eps;
    a.inv_L = static_cast<float>(1.0 / static_cast<double>(L));
    a.inv_LCg = static_cast<float>(1.0 / (static_cast<double>(L) * static_cast<double>(C / G)));
    a.L = static_cast<int32_t>(L);
    a.C = C;
    a.G = G;
    a.Cg = C / G;
    a.SC = p.SC;
    a.VS = p.SC / 8;
    a.slices = C / p.SC;
    a.P = rows_per_pass(a.VS);
    a.A = a.P * a.VS;
    a.vs_pow2 = (a.VS & (a.VS - 1)) == 0 ? 1 : 0;
    a.R = p.R;
    a.BR = p.BR;
    a.boxes = p.boxes;
    a.cl = p.CL;
    // tensor-map copies need a 16-byte aligned base
    a.tma = p.tma && reinterpret_cast<uintptr_t>(x) % 16 == 0 ? 1 : 0;
    if (a.tma) {
        // x as [N L rows][C] bf16, boxes of BR rows x SC channels, no swizzle
        // (the rows land as the dense [row][SC] block the kernel reads)
        tc::EncodeTiledFn enc = tc::encode_fn();
        if (!enc) return cudaErrorNotSupported;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N * L)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(C) * 2};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.SC), static_cast<cuuint32_t>(p.BR)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&a.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    a.timeout_ns = timeout_ns;
    a.status = status;
    a.status_host = status_host;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.units * p.CL));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    void *params[] = {&a};
    return cudaLaunchKernelExC(&cfg, cluster_fn(silu), params);
}

}  // namespace gn
