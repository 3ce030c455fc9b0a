// attn_kernels.cu -- the VAE mid-block's single-head attention with the
// output projection folded into the value projection, on the sm_103a tensor
// cores.
//
// Operation (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
// quality=high", section "Modifications", item 2, attention bullet): with
// the query / key projections q, k [S][D], the GroupNorm output xn [S][D]
// and the value / output projections (wv, bv), (wo, bo),
//   out = softmax(q k^T / sqrt(D)) (xn wv^T + bv) wo^T + bo + residual
//       = softmax(q k^T / sqrt(D)) (xn W'^T + b') + residual,
//   W' = wo wv, b' = wo bv + bo,
// the second form being exact because every softmax row sums to 1.  This
// file evaluates the second form, by one of two schedules after the fold:
//  * one pass (D <= 512): V'^T = W' xn^T + b' by gemm_kernel, then
//    attn_flash_kernel on CTA pairs keeps each block of scores in tensor
//    memory and accumulates softmax(...) V' without writing the scores or the
//    weights (described at the kernel), and attn_combine_kernel merges the
//    pieces of tiles that were split between pairs;
//  * stored weights (any D): the kernels below.
//   attn_fold_kernel   W' (fp32 sums over D, rounded once to bf16) and b'
//                      (fp32), once per weight;
//   gemm_kernel        C = alpha A B^T (+ a per-row or per-column bias, + a
//                      bf16 residual), A [M][K] and B [N][K] bf16 K-major,
//                      fp32 accumulation in tensor memory; its epilogue can
//                      instead reduce each row segment of alpha A B^T to a
//                      softmax (max, sum of exp) record, or write the softmax
//                      weights exp(alpha A B^T - max) / sum as bf16.  Run four
//                      times: V'^T = W' xn^T + b' ([D][S], bf16); the scores
//                      q k^T / sqrt(D) reduced to per-row-segment records;
//                      the scores again, written as P ([S][S], bf16); and
//                      out = P V' + residual ([S][D], bf16);
//   softmax_stats_kernel  merges each row's records into (max, 1 / sum).
// The fp32 scores are never stored: computing them twice costs 2 S^2 D
// tensor-core flops, far cheaper than writing and re-reading 4 S^2 bytes.
// (An fp32 128 x 512 output block alone fills the 512 tensor-memory columns
// of an SM, which is why the one-pass kernel puts the scores and the output
// on different CTAs of a pair.)
//
// gemm_kernel is persistent (one CTA per SM): warp 0 issues TMA tile loads
// (128-byte swizzle) into a STAGES-deep ring, warp 1 owns 2 BN tensor-memory
// columns and issues tcgen05.mma (M = 128, N = BN, K = 16), warps 2-9 (two
// per tensor-memory lane quarter, each half of the columns) drain the two
// accumulators alternately (tcgen05.ld, epilogue; fp32 results pass through
// a shared-memory tile so that each store writes whole 128-byte row
// segments) while the next tile's MMAs run.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "tc_internal.h"
#include "gn_ptx.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace gn {

__device__ unsigned int g_at_status;
// the host-visible copy of g_at_status (mapped page-locked host memory; null until set)
__device__ unsigned int *g_at_status_host;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kGemmThreads = 320;   // producer warp, MMA warp, 8 epilogue warps

struct GemmArgs {
    int M, N, K;
    int n_tiles, tiles, ksteps;
    float alpha;
    const float *bias_m;            // [M] or null
    const float *bias_n;            // [N] or null
    const __nv_bfloat16 *residual;  // [M][N] bf16 or null
    void *c;                        // [M][N] fp32 or bf16
    int out_f32;
    int mode;                       // kGemmPlain, kGemmRowStats or kGemmSoftmax
    float2 *stats;                  // kGemmRowStats: [M][2 n_tiles] (max, sum of exp) per row segment
    const float2 *row_ml;           // kGemmSoftmax: [M] (row max, 1 / row sum of exp)
    uint64_t timeout_ns;
};

// Epilogue modes: the plain product (+ bias, + residual); per-row softmax
// statistics of alpha A B^T over each half tile (nothing else is written);
// the softmax weights exp(alpha A B^T - max) / sum, rounded to bf16.
constexpr int kGemmPlain = 0;
constexpr int kGemmRowStats = 1;
constexpr int kGemmSoftmax = 2;
constexpr float kLog2e = 1.4426950408889634f;

template <int BN, int STAGES>
struct GemmLayout {
    static constexpr uint32_t kBBytes = static_cast<uint32_t>(BN) * kBK * 2;
    static constexpr uint32_t kStage = kABytes + kBBytes;
    static constexpr uint32_t kRing = kStage * STAGES;
    static constexpr uint32_t kTmemCols = 2 * BN;
    static constexpr uint32_t kBars = kRing;
    static constexpr uint32_t kTmemSlot = kBars + 8 * (2 * STAGES + 5);
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kConsumed = kAbort + 4;
    // fp32 epilogue staging: per epilogue warp 32 rows x 32 floats (4 KB), the
    // 16-byte chunks of row r stored at chunk index c ^ (r & 7)
    static constexpr uint32_t kStaging = (kConsumed + 4 + 15) & ~15u;
    static constexpr uint32_t kBytes = kStaging + 8 * 32 * 32 * 4;
    static constexpr uint32_t kDynamic = kBytes + 1024;
};



}  // namespace

// ---------------------------------------------------------------------------
// W'[e][i] = sum_c wo[e][c] wv[c][i] (fp32, rounded once to bf16) and
// b'[e] = sum_c wo[e][c] bv[c] + bo[e] (fp32), one thread per output.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) attn_fold_kernel(const __nv_bfloat16 *__restrict__ wv,
                                                        const __nv_bfloat16 *__restrict__ bv,
                                                        const __nv_bfloat16 *__restrict__ wo,
                                                        const __nv_bfloat16 *__restrict__ bo,
                                                        __nv_bfloat16 *__restrict__ wf, float *__restrict__ bf,
                                                        int D)
{
    const int64_t total = static_cast<int64_t>(D) * (D + 1);
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = static_cast<int>(idx / (D + 1));
        const int i = static_cast<int>(idx % (D + 1));   // i == D: the bias
        const __nv_bfloat16 *wrow = wo + static_cast<int64_t>(e) * D;
        float acc = 0.f;
        if (i < D) {
            for (int c = 0; c < D; ++c)
                acc = fmaf(__bfloat162float(wrow[c]), __bfloat162float(wv[static_cast<int64_t>(c) * D + i]), acc);
            wf[static_cast<int64_t>(e) * D + i] = __float2bfloat16_rn(acc);
        } else {
            for (int c = 0; c < D; ++c) acc = fmaf(__bfloat162float(wrow[c]), __bfloat162float(bv[c]), acc);
            bf[e] = acc + __bfloat162float(bo[e]);
        }
    }
}

// ---------------------------------------------------------------------------
// Row softmax statistics: merge a row's `parts` (max, sum of exp) segment
// records into (max, 1 / sum), one warp per row, in a fixed order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 merge_ml(float2 a, float2 b)
{
    const float m = fmaxf(a.x, b.x);
    if (m == -INFINITY) return make_float2(m, 0.f);
    return make_float2(m, a.y * exp2f((a.x - m) * kLog2e) + b.y * exp2f((b.x - m) * kLog2e));
}

__global__ void __launch_bounds__(256) softmax_stats_kernel(const float2 *__restrict__ parts_in, int parts,
                                                            float2 *__restrict__ row_ml, int rows)
{
    tc::griddep_wait();   // launched with programmatic serialization after the pass that writes the records
    if (threadIdx.x == 0) tc::griddep_launch_dependents();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const float2 *p = parts_in + static_cast<int64_t>(warp) * parts;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int i = lane; i < parts; i += 32) acc = merge_ml(acc, p[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 other;
        other.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
        other.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc = merge_ml(acc, other);
    }
    if (lane == 0) row_ml[warp] = make_float2(acc.x, 1.0f / acc.y);
}

// ---------------------------------------------------------------------------
// The epilogue of one finished accumulator for one warp: its 32 rows
// (m_warp0 + lane, tensor-memory lanes of its quarter from `tbase`) and one
// half of the BN columns; hands the accumulator back with one arrival on
// `acc_empty` (in the peer CTA when `remote`) once the last columns are in
// registers.
// ---------------------------------------------------------------------------
template <int BN>
__device__ __forceinline__ void gemm_epilogue(const GemmArgs &args, uint32_t tbase, int m_warp0, int n0, int n_t,
                                              int half, int lane, float4 *stage, uint32_t acc_empty, bool remote)
{
    const int m = m_warp0 + lane;
    const float bm = args.bias_m ? args.bias_m[m] : 0.f;
    float run_m = -INFINITY, run_l = 0.f;   // kGemmRowStats: this row segment's running max / sum
    float2 ml = make_float2(0.f, 0.f);
    if (args.mode == kGemmSoftmax) ml = args.row_ml[m];
#pragma unroll 1
    for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), v);
        tmem_wait_ld();
        if (c + 32 == (half + 1) * (BN / 2)) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (remote)
                    mbar_arrive_cluster(acc_empty);
                else
                    mbar_arrive(acc_empty);
            }
        }
        float f[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) f[k] = fmaf(__uint_as_float(v[k]), args.alpha, bm);
        if (args.mode == kGemmRowStats) {
            float cmax = f[0];
#pragma unroll
            for (int k = 1; k < 32; ++k) cmax = fmaxf(cmax, f[k]);
            const float m_new = fmaxf(run_m, cmax);
            const float mb = m_new * kLog2e;
            float acc = run_l * exp2f(fmaf(run_m, kLog2e, -mb));
#pragma unroll
            for (int k = 0; k < 32; ++k) acc += exp2f(fmaf(f[k], kLog2e, -mb));
            run_l = acc;
            run_m = m_new;
            continue;
        }
        if (args.mode == kGemmSoftmax) {
            const float mb = ml.x * kLog2e;
#pragma unroll
            for (int k = 0; k < 32; ++k) f[k] = exp2f(fmaf(f[k], kLog2e, -mb)) * ml.y;
        }
        if (args.bias_n) {
            const float4 *b4 = reinterpret_cast<const float4 *>(args.bias_n + n0 + c);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 b = __ldg(b4 + k);
                f[4 * k] += b.x;
                f[4 * k + 1] += b.y;
                f[4 * k + 2] += b.z;
                f[4 * k + 3] += b.w;
            }
        }
        const int64_t at = static_cast<int64_t>(m) * args.N + n0 + c;
        if (args.residual) {
            const uint4 *r4 = reinterpret_cast<const uint4 *>(args.residual + at);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 rr = r4[k];
                const uint32_t w[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    f[8 * k + 2 * h] += __uint_as_float(w[h] << 16);
                    f[8 * k + 2 * h + 1] += __uint_as_float(w[h] & 0xffff0000u);
                }
            }
        }
        if (args.out_f32) {
            // through shared memory, so that each store instruction of the
            // warp writes four whole 128-byte row segments
#pragma unroll
            for (int k = 0; k < 8; ++k)
                stage[lane * 8 + (k ^ (lane & 7))] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
            __syncwarp();
            float *crow = static_cast<float *>(args.c) +
                          static_cast<int64_t>(m_warp0) * args.N + n0 + c;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = (lane >> 3) + 4 * i;
                const float4 val = stage[r * 8 + ((lane & 7) ^ (r & 7))];
                reinterpret_cast<float4 *>(crow + static_cast<int64_t>(r) * args.N)[lane & 7] = val;
            }
            __syncwarp();
        } else {
            // bf16: the same staging, 64 bytes per row; each store
            // instruction writes eight whole 64-byte row segments
            uint4 *stage4 = reinterpret_cast<uint4 *>(stage);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(f[8 * k + 2 * h], f[8 * k + 2 * h + 1]);
                    o[h] = *reinterpret_cast<const uint32_t *>(&hb);
                }
                stage4[lane * 4 + (k ^ (lane & 3))] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            __syncwarp();
            __nv_bfloat16 *crow = static_cast<__nv_bfloat16 *>(args.c) +
                                  static_cast<int64_t>(m_warp0) * args.N + n0 + c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = (lane >> 2) + 8 * i;
                const uint4 val = stage4[r * 4 + ((lane & 3) ^ (r & 3))];
                reinterpret_cast<uint4 *>(crow + static_cast<int64_t>(r) * args.N)[lane & 3] = val;
            }
            __syncwarp();
        }
    }
    if (args.mode == kGemmRowStats)
        args.stats[static_cast<int64_t>(m) * (2 * args.n_tiles) + 2 * n_t + half] =
            make_float2(run_m, run_l);
}

// ---------------------------------------------------------------------------
// C = alpha A B^T (+ bias, + residual): persistent, one CTA per SM; tile t:
// the N tile varies fastest.
// ---------------------------------------------------------------------------
template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const GemmArgs args)
{
    using L = GemmLayout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + L::kTmemSlot);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + L::kAbort);
    volatile int *consumed_sh = reinterpret_cast<volatile int *>(gbase + L::kConsumed);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // launched with programmatic serialization (tc::launch_pdl): nothing
    // global before the kernel ahead in the stream has finished; then a
    // kernel launched after this one the same way may start on the SMs this
    // grid leaves free
    tc::griddep_wait();
    if (threadIdx.x == 0) tc::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, 8);   // one arrival per epilogue warp
        }
        mbar_init(bar_drain, 1);
        *abort = (*reinterpret_cast<volatile unsigned int *>(&g_at_status) != 0u) ? 1 : 0;
        *consumed_sh = 0;
        mbar_init_fence();
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc(base + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort != 0;

    int issued = 0;
    if (!skip && warp == 0 && lane == 0) {
        int q = 0;
        bool go = true;
        for (int t = blockIdx.x; go && t < args.tiles; t += gridDim.x) {
            const int m0 = (t / args.n_tiles) * kBM, n0 = (t % args.n_tiles) * BN;
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (q >= STAGES && !tc::wait(bar_empty + 8 * s, ((q / STAGES) - 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) {
                    go = false;
                    break;
                }
                const uint32_t sa = base + s * L::kStage;
                mbar_arrive_expect_tx(bar_full + 8 * s, L::kStage);
                tma_load_2d(sa, &map_a, kt * kBK, m0, bar_full + 8 * s);
                tma_load_2d(sa + kABytes, &map_b, kt * kBK, n0, bar_full + 8 * s);
                issued = q + 1;
            }
        }
    } else if (!skip && warp == 1 && lane == 0) {
        constexpr uint32_t idesc = umma_idesc_bf16_f32(kBM, BN);
        int q = 0, lt = 0;
        bool go = true;
        for (int t = blockIdx.x; go && t < args.tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            if (lt >= 2 && !tc::wait(bar_acc_empty + 8 * buf, ((lt >> 1) - 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (!tc::wait(bar_full + 8 * s, (q / STAGES) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) {
                    go = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sa = base + s * L::kStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    umma_f16(d, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sa + kABytes + kk * 32), idesc,
                             (kt > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar_empty + 8 * s);
                *consumed_sh = q + 1;
            }
            if (go) umma_commit(bar_acc_full + 8 * buf);
        }
        umma_commit(bar_drain);
    } else if (!skip && warp >= 2) {
        // two warps per tensor-memory lane quarter, each draining half the columns
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        float4 *const stage = reinterpret_cast<float4 *>(gbase + L::kStaging) + (warp - 2) * 32 * 8;
        int lt = 0;
        for (int t = blockIdx.x; t < args.tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            const bool done = tc::wait(bar_acc_full + 8 * buf, (lt >> 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host);
            tc_fence_after_sync();
            if (!__all_sync(0xffffffffu, done && !*abort)) break;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
            gemm_epilogue<BN>(args, tbase, (t / args.n_tiles) * kBM + quad * 32, (t % args.n_tiles) * BN,
                              t % args.n_tiles, half, lane, stage, bar_acc_empty + 8 * buf, false);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort && !skip) {
        if (warp == 0 && lane == 0) {
            for (int q = *consumed_sh; q < issued; ++q)
                tc::drain(bar_full + 8 * (q % STAGES), (q / STAGES) & 1, args.timeout_ns);
        }
        if (warp == 1 && lane == 0) tc::drain(bar_drain, 0, args.timeout_ns);
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// The same GEMM on CTA pairs (a cluster of two CTAs): one
// tcgen05.mma.cta_group::2 of M = 256 (128 rows per CTA), N = 256 per pair
// tile; each CTA stages its own A rows and half of the B rows, so per SM the
// operand traffic is 2/3 of the single-CTA kernel's.  Barriers as in the
// upsample-conv pair kernel: `full` in the even CTA counts both CTAs' bytes,
// the pair MMA's commits arrive on both CTAs' `empty` / `acc_full`, and all
// sixteen epilogue warps arrive on the even CTA's `acc_empty`.
// ---------------------------------------------------------------------------
template <int STAGES>
struct GemmPairLayout {
    static constexpr uint32_t kBHalf = 128u * kBK * 2;
    static constexpr uint32_t kStage = kABytes + kBHalf;   // 32 KB
    static constexpr uint32_t kRing = kStage * STAGES;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kBars = kRing;
    static constexpr uint32_t kTmemSlot = kBars + 8 * (2 * STAGES + 5);
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kConsumed = kAbort + 4;
    static constexpr uint32_t kStaging = (kConsumed + 4 + 15) & ~15u;
    static constexpr uint32_t kBytes = kStaging + 8 * 32 * 32 * 4;
    static constexpr uint32_t kDynamic = kBytes + 1024;
};

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const GemmArgs args)
{
    using L = GemmPairLayout<STAGES>;
    constexpr int BN = 256;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + L::kTmemSlot);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + L::kAbort);
    volatile int *consumed_sh = reinterpret_cast<volatile int *>(gbase + L::kConsumed);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    // launched with programmatic serialization, as gemm_kernel
    tc::griddep_wait();
    if (threadIdx.x == 0) tc::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, 16);   // 8 epilogue warps x 2 CTAs
        }
        mbar_init(bar_drain, 1);
        *abort = (*reinterpret_cast<volatile unsigned int *>(&g_at_status) != 0u) ? 1 : 0;
        *consumed_sh = 0;
        mbar_init_fence();
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(base + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncwarp();
    cluster_sync_all();   // both CTAs' barriers are initialised before any signal crosses the pair
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort != 0;
    const uint32_t full_lead = mapa_shared(bar_full, 0);
    const uint32_t acc_empty_lead = mapa_shared(bar_acc_empty, 0);

    int issued = 0;
    if (!skip && warp == 0 && lane == 0) {
        int q = 0;
        bool go = true;
        for (int T = pair; go && T < args.tiles; T += npairs) {
            const int m0 = (2 * (T / args.n_tiles) + rank) * kBM;
            const int nrow = (T % args.n_tiles) * BN + rank * 128;
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (q >= STAGES && !tc::wait(bar_empty + 8 * s, ((q / STAGES) - 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) {
                    go = false;
                    break;
                }
                const uint32_t sa = base + s * L::kStage;
                if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * L::kStage);
                tma_load_2d_pair(sa, &map_a, kt * kBK, m0, full_lead + 8 * s);
                tma_load_2d_pair(sa + kABytes, &map_b, kt * kBK, nrow, full_lead + 8 * s);
                issued = q + 1;
            }
        }
    } else if (!skip && leader && warp == 1 && lane == 0) {
        constexpr uint32_t idesc = umma_idesc_bf16_f32(2 * kBM, BN);
        int q = 0, lt = 0;
        bool go = true;
        for (int T = pair; go && T < args.tiles; T += npairs, ++lt) {
            const int buf = lt & 1;
            if (lt >= 2 && !tc::wait(bar_acc_empty + 8 * buf, ((lt >> 1) - 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (!tc::wait(bar_full + 8 * s, (q / STAGES) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host)) {
                    go = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sa = base + s * L::kStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    umma_f16_pair(d, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sa + kABytes + kk * 32),
                                  idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit_pair(bar_empty + 8 * s, 0x3);
                *consumed_sh = q + 1;
            }
            if (go) umma_commit_pair(bar_acc_full + 8 * buf, 0x3);
        }
        umma_commit_pair(bar_drain, 0x1);
    } else if (!skip && warp >= 2) {
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        float4 *const stage = reinterpret_cast<float4 *>(gbase + L::kStaging) + (warp - 2) * 32 * 8;
        int lt = 0;
        for (int T = pair; T < args.tiles; T += npairs, ++lt) {
            const int buf = lt & 1;
            const bool done = tc::wait(bar_acc_full + 8 * buf, (lt >> 1) & 1, abort, args.timeout_ns, &g_at_status, g_at_status_host);
            tc_fence_after_sync();
            if (!__all_sync(0xffffffffu, done && !*abort)) break;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
            gemm_epilogue<BN>(args, tbase, (2 * (T / args.n_tiles) + rank) * kBM + quad * 32,
                              (T % args.n_tiles) * BN, T % args.n_tiles, half, lane, stage,
                              acc_empty_lead + 8 * buf, true);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort && !skip) {
        if (leader && warp == 0 && lane == 0) {
            for (int q = *consumed_sh; q < issued; ++q)
                tc::drain(bar_full + 8 * (q % STAGES), (q / STAGES) & 1, args.timeout_ns);
        }
        if (leader && warp == 1 && lane == 0) tc::drain(bar_drain, 0, args.timeout_ns);
        if (!leader && warp == 0 && lane == 0) {
            // this CTA's copies signal the even CTA's barriers: give them time to land
            const uint64_t until = global_ns() + 200000;
            while (global_ns() < until) __nanosleep(1000);
        }
        __syncthreads();
    }
    __syncwarp();
    cluster_sync_all();   // neither CTA leaves while the pair's MMAs or signals may touch it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// The softmax and the weighted sum in one pass over the keys, on CTA pairs,
// for widths D <= 512 (see the file comment):
//   out = softmax(q k^T / sqrt(D)) V' + residual,  given V'^T [D][S].
// The work is split into (tile of 128 query rows, block of 128 keys) units,
// and each cluster of two CTAs takes an equal run of consecutive units: whole
// tiles, and at either end possibly a piece of a tile that another cluster
// finishes (or starts).  A whole tile is written out by its cluster; a piece
// leaves its unnormalised output with the rows' running maxima and sums in
// the workspace, and attn_combine_kernel merges the pieces afterwards.
//  * CTA 0, the score CTA, keeps the tile's q rows in tensor memory (the
//    A operand of its MMAs; its softmax warps load them, one row per
//    thread), streams k in blocks of 128 keys (128-dimension chunks through
//    a shared-memory ring) and has tcgen05.mma compute each block's scores
//    into tensor memory (two buffers, so a block's MMAs run while the
//    softmax warps read the one before).  Its four softmax warps (one
//    tensor-memory lane quarter, one query row per thread) turn the scores
//    into weights p = 2^(s log2e / sqrt(D) - m): m is a running maximum
//    that moves only when a block's maximum exceeds it by more than 8
//    (weights stay below 2^8, and the output is rarely rescaled).  The
//    weights are rounded to bf16 and the rounded values summed into the row
//    sum l.  They are written into a staging buffer, in the
//    128-byte-swizzled K-major layout the output CTA's MMA reads, with each
//    row's rescale factor 2^(m_old - m_new) and a flag when m moved; one
//    thread then ships the block with bulk copies into the output CTA's
//    shared memory (distributed shared memory), completing on the output
//    CTA's mbarrier.
//  * CTA 1, the output CTA, holds the 128 x D fp32 output in tensor memory
//    (D <= 512 columns: which is why the scores live in the other CTA),
//    streams V'^T in 64-key chunks and accumulates O += P V'.  Before a block
//    that came with a rescale its MMA thread asks the eight epilogue warps
//    to multiply O's rows by the factors (after the previous block's MMAs
//    have completed); at the tile's end they write out = O / l + residual.
//    A forwarder warp hands each weights buffer back to the score CTA as
//    soon as the MMAs that read it have completed.
//  * Per block both tensor pipes do 2 x 128 x 128 x D flops.
//  * Tile t visits the key blocks starting at block t (the softmax does not
//    depend on the order): clusters working at the same time then read
//    different key and value rows, instead of all asking L2 for the same
//    lines at once.  A tile's pieces cover disjoint runs of that order.
// Every wait is bounded; a timeout records the sticky status and both CTAs
// still meet at the final cluster barrier before either leaves.
// ---------------------------------------------------------------------------
// warps: 0 producer, 1 and 10 the two MMA issuers, 12 and 13 their waiters,
// 2-9 softmax (score CTA: 2-5) / epilogue (output CTA), 11 the output CTA's
// forwarder.  An issuing thread that touches shared memory (every mbarrier
// wait does, and so does a plain load by any lane of its warp) stalls until
// its own MMAs in flight have completed, about 0.5 us on a GB300 (measured),
// which leaves the tensor pipe idle between chunks.  So a separate waiter
// warp polls the mbarriers and passes each go-ahead (or a failure) to its
// issuer with a named barrier, which does not stall the issuer; and two
// issuers, on separate accumulators, keep the pipe fed while one waits for
// its next operands.
constexpr int kFlashThreads = 448;
constexpr int kFlashKStages = 6;     // score CTA: 128-dimension chunks of key blocks in flight
constexpr int kFlashVStages = 4;     // output CTA: 64 keys x D/2 of V'^T per stage
constexpr float kFlashRescaleLog2 = 8.0f;
constexpr int kFlashEnd = -1;        // mailbox: the tile is finished
constexpr uint32_t kFlashPBytes = 32768u + 512u + 16u;   // one block's weights, factors and flags

// barrier indices (8 bytes each)
enum FlashBar {
    // score CTA
    kQFull = 0, kQFree = 1, kKFull = 2, kKEmpty = kKFull + kFlashKStages, kSFull = kKEmpty + kFlashKStages,
    kSEmpty = kSFull + 2, kPEmpty = kSEmpty + 2, kSDrain = kPEmpty + 2,
    // output CTA
    kPFull = kSDrain + 1, kVFull = kPFull + 2, kVEmpty = kVFull + kFlashVStages, kPDone = kVEmpty + kFlashVStages,
    kRescaleReq = kPDone + 2, kORescaled = kRescaleReq + 1, kOFull = kORescaled + 1, kOFree = kOFull + 1,
    kLFull = kOFree + 1, kODrain = kLFull + 2,
    // score CTA: a row-sum buffer of the output CTA is free again (its 8 epilogue warps)
    kLEmpty = kODrain + 1, kFlashBars = kLEmpty + 2
};

struct FlashArgs {
    int S, D, tiles, nblocks;
    // The work is tiles x nblocks (tile, key block) units; cluster c takes
    // the units [flash_unit_begin(c), flash_unit_begin(c + 1)): with split
    // set, an equal share whose ends may fall inside a tile (that tile's
    // parts are merged by attn_combine_kernel), else whole tiles.
    int units, clusters, split;
    float scale_log2;                  // log2(e) / sqrt(D)
    const __nv_bfloat16 *q;            // [S][D]
    const __nv_bfloat16 *residual;     // [S][D] or null
    __nv_bfloat16 *out;                // [S][D]
    // split: two slots per cluster (its first and its last piece of a tile),
    // each [D][128] fp32 unnormalised output, then 128 row maxima m and 128
    // row sums l
    float *partial;
    uint64_t timeout_ns;
};

// 32-bit arithmetic: S <= kAttnMaxS gives at most 256 tiles and 65536 units,
// and c <= clusters <= the SM count, so c * units stays far below 2^32.
static_assert(static_cast<unsigned long long>(kAttnMaxS / 128) * (kAttnMaxS / 128) * 1024ull < (1ull << 32),
              "unit boundaries need 32 bits");
__host__ __device__ inline int flash_unit_begin(const FlashArgs &a, int c)
{
    const uint32_t uc = static_cast<uint32_t>(c), cl = static_cast<uint32_t>(a.clusters);
    if (a.split) return static_cast<int>(uc * static_cast<uint32_t>(a.units) / cl);
    return static_cast<int>(uc * static_cast<uint32_t>(a.tiles) / cl) * a.nblocks;
}

__host__ __device__ inline size_t flash_slot_floats(int D) { return static_cast<size_t>(D) * 128 + 256; }

// Shared-memory layout.  The score CTA uses q / kring, the output CTA
// p / vring / alpha / flags / lsum / mailbox; the barriers and the small
// words sit after both.  Both CTAs run the same kernel, so an offset names
// the same place in either CTA (distributed shared memory addresses are
// formed with mapa from the writer's own offsets).
struct FlashLayout {
    uint32_t kring, pstage, astage, fstage, lstage;      // score CTA
    uint32_t p, vring, alpha, flags, lsum, mailbox;      // output CTA
    uint32_t bars, tslot, abort, counters, total;
};

__host__ __device__ inline FlashLayout flash_layout(int D)
{
    FlashLayout l;
    l.kring = 0;                                         // two [128 keys][64] bf16 boxes per stage
    l.pstage = l.kring + kFlashKStages * 32768u;         // one block's weights, as the output CTA lays them out
    l.astage = l.pstage + 32768u;                        // 128 rescale factors
    l.fstage = l.astage + 512u;                          // 4 flags
    l.lstage = l.fstage + 16u;                           // 128 row sums, then 128 row maxima
    const uint32_t score_end = l.lstage + 1024u;
    l.p = 0;                                             // two buffers of two [128][64] subtiles
    l.vring = 2u * 32768u;
    l.alpha = l.vring + kFlashVStages * static_cast<uint32_t>(D) * 64u;
    l.flags = l.alpha + 2u * 128u * 4u;
    l.lsum = l.flags + 2u * 4u * 4u;
    l.mailbox = l.lsum + 2u * 256u * 4u;
    const uint32_t out_end = l.mailbox + 16u;
    l.bars = (score_end > out_end ? score_end : out_end);
    l.bars = (l.bars + 15u) & ~15u;
    l.tslot = l.bars + 8u * kFlashBars;
    l.abort = l.tslot + 4u;
    l.counters = l.abort + 4u;                           // issued / consumed copies, for the drain
    l.total = l.counters + 32u;
    return l;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity, uint32_t sleep_ns)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(sleep_ns)
        : "memory");
    return done != 0;
}

// tc::wait for a phase completed by arrivals from the other CTA: acquire at
// cluster scope, so that what that CTA wrote before arriving is visible.
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns)
{
    if (mbar_try_wait_cluster(bar, parity, 0)) return true;
    if (*abort) return false;
    const uint64_t deadline = global_ns() + timeout_ns;
#pragma unroll 1
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity, tc::kSleepNs)) return true;
        if (*abort) return false;
        if (global_ns() > deadline) {
            *abort = 1;
            atomicOr(&g_at_status, 1u);
            raise_host_status(g_at_status_host);
            return false;
        }
    }
}

__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns)
{
    return tc::wait(bar, parity, abort, timeout_ns, &g_at_status, g_at_status_host);
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bulk copy from this CTA's shared memory to the peer's (shared::cluster
// addresses), completing `bytes` on the peer's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_cluster)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst_cluster), "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M = 128 rows, one per tensor-memory
// lane, K packed two bf16 per 32-bit column) read from tensor memory.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// A barrier over `count` threads (named barrier `id`) that also returns
// whether any of them passed pred = true.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "barrier.cta.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;"
                 ::"r"(bar_cluster), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
          "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
          "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Rows 32 quarter .. 32 quarter + 31 of query tile t, 64-dimension chunks
// [c0, c1), into tensor memory (columns 256 + d/2 of the calling warp's lane
// quarter).  The loads are coalesced (eight lanes read one row's 128 bytes
// of a chunk; a lane reading its own row would make every 16-byte load a
// separate request) and go through 8 KB of staging shared memory, 16-byte
// pieces XOR-swizzled by the row so that neither the writes nor the
// row-wise reads meet in a bank; each lane then takes its own row.  NF
// chunks' loads are in flight at a time, staged in NF x 4 KB.
template <int NF>
__device__ __forceinline__ void flash_load_q(const FlashArgs &args, uint32_t tmem, uint32_t lane_base, int t,
                                             int quarter, int lane, uint32_t stage, int c0, int c1)
{
    const int D = args.D, piece = lane & 7;
    const __nv_bfloat16 *src =
        args.q + (static_cast<int64_t>(t) * 128 + quarter * 32 + (lane >> 3)) * D + piece * 8;
#pragma unroll 1
    for (int c = c0; c < c1; c += NF) {
        const int nh = c1 - c < NF ? c1 - c : NF;
        uint4 g[NF][8];
#pragma unroll
        for (int h = 0; h < NF; ++h) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                g[h][i] = h < nh ? __ldg(reinterpret_cast<const uint4 *>(src + static_cast<int64_t>(4 * i) * D + (c + h) * 64))
                                 : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int h = 0; h < NF; ++h) {
            if (h < nh) {
                const uint32_t st = stage + static_cast<uint32_t>(h) * 4096u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t r = static_cast<uint32_t>(4 * i + (lane >> 3));
                    sts128(st + r * 128u + ((static_cast<uint32_t>(piece) ^ (r & 7u)) << 4), g[h][i]);
                }
            }
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < NF; ++h) {
            if (h < nh) {
                const uint32_t st = stage + static_cast<uint32_t>(h) * 4096u;
                uint32_t v[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 x = lds128(st + static_cast<uint32_t>(lane) * 128u +
                                           ((static_cast<uint32_t>(k) ^ (static_cast<uint32_t>(lane) & 7u)) << 4));
                    v[4 * k] = x.x;
                    v[4 * k + 1] = x.y;
                    v[4 * k + 2] = x.z;
                    v[4 * k + 3] = x.w;
                }
                tmem_st_32x32b_x32(tmem + lane_base + 256u + static_cast<uint32_t>((c + h) * 32), v);
            }
        }
        __syncwarp();
    }
    tmem_wait_st();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFlashThreads, 1)
    attn_flash_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const FlashArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const FlashLayout lay = flash_layout(args.D);
    const uint32_t bars = base + lay.bars;
    const auto bar = [bars](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + lay.tslot);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + lay.abort);
    volatile int *counters = reinterpret_cast<volatile int *>(gbase + lay.counters);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool scorer = rank == 0;
    const int cl = blockIdx.x >> 1;   // this cluster's share of the work units
    const int D = args.D, half = D / 2, nb = args.nblocks;
    const int ub = flash_unit_begin(args, cl), ue = flash_unit_begin(args, cl + 1);
    // score CTA: two score buffers (columns 0-255) and the q rows (from 256);
    // output CTA: the output, D columns
    const uint32_t tmem_cols = scorer ? 512u : (D <= 128 ? 128u : (D <= 256 ? 256u : 512u));

    if (threadIdx.x == 0) {
        if (scorer) {
            mbar_init(bar(kQFull), 8);               // the eight softmax warps, once q is in tensor memory
            mbar_init(bar(kQFree), 2);               // both issuers, after a tile's MMAs
            for (int i = 0; i < kFlashKStages; ++i) {
                mbar_init(bar(kKFull + i), 1);
                mbar_init(bar(kKEmpty + i), 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar(kSFull + i), 1);
                mbar_init(bar(kSEmpty + i), 8);      // the eight softmax warps
                mbar_init(bar(kPEmpty + i), 1);      // the output CTA's forwarder
            }
            mbar_init(bar(kSDrain), 2);
            for (int i = 0; i < 2; ++i) mbar_init(bar(kLEmpty + i), 8);
        } else {
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar(kPFull + i), 1);       // armed here (plus the bytes the score CTA copies)
                mbar_init(bar(kPDone + i), 2);       // both issuers (one half of D each)
                mbar_init(bar(kLFull + i), 1);
            }
            for (int i = 0; i < kFlashVStages; ++i) {
                mbar_init(bar(kVFull + i), 1);
                mbar_init(bar(kVEmpty + i), 1);
            }
            mbar_init(bar(kRescaleReq), 1);
            mbar_init(bar(kORescaled), 8);           // the eight epilogue warps
            mbar_init(bar(kOFull), 2);
            mbar_init(bar(kOFree), 8);
            mbar_init(bar(kODrain), 2);
            // the first uses of the weights and row-sum buffers expect their bytes
            for (int i = 0; i < 2; ++i) {
                mbar_arrive_expect_tx(bar(kPFull + i), kFlashPBytes);
                mbar_arrive_expect_tx(bar(kLFull + i), 1024u);
            }
        }
        *abort = (*reinterpret_cast<volatile unsigned int *>(&g_at_status) != 0u) ? 1 : 0;
        for (int i = 0; i < 8; ++i) counters[i] = 0;
        mbar_init_fence();
        if (scorer) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_k);
        } else {
            prefetch_tensormap(&map_v);
        }
    }
    if (warp == 1) {
        tmem_alloc(base + lay.tslot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncwarp();
    cluster_sync_all();   // both CTAs' barriers exist before anything crosses the pair
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort != 0;

    if (scorer) {
        if (!skip && warp == 0 && lane == 0) {
            // ---- producer: k in 128-dimension chunks (two boxes each) ----
            int kq = 0;
            bool go = true;
            for (int u = ub, nu = 0; go && u < ue; u = nu) {
                const int t = u / nb, j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile t
                nu = u + (j1 - j0);
                for (int j = j0; go && j < j1; ++j) {
                    for (int c = 0; c < D / 128; ++c, ++kq) {
                        const int st = kq % kFlashKStages;
                        if (kq >= kFlashKStages &&
                            !fwait(bar(kKEmpty + st), ((kq / kFlashKStages) - 1) & 1, abort, args.timeout_ns)) {
                            go = false;
                            break;
                        }
                        const uint32_t dst = base + lay.kring + st * 32768u;
                        const int key0 = ((j + t) % nb) * 128;
                        mbar_arrive_expect_tx(bar(kKFull + st), 32768u);
                        tma_load_2d(dst, &map_k, c * 128, key0, bar(kKFull + st));
                        tma_load_2d(dst + 16384u, &map_k, c * 128 + 64, key0, bar(kKFull + st));
                        counters[1] = kq + 1;   // k chunks issued
                    }
                }
            }
        } else if (!skip && (warp == 1 || warp == 10 || warp >= 12)) {
            // ---- MMA: S = q k^T per block into alternate buffers; warp 1 issues
            // the even blocks, warp 10 the odd ones.  Warp 12 (13) does the
            // waiting for warp 1 (10) and hands each go-ahead over at named
            // barrier 3 (4), so that the issuing thread never polls ----
            constexpr uint32_t idesc = umma_idesc_bf16_f32(128, 128);
            const bool waiter = warp >= 12;
            const int mine = (warp == 1 || warp == 12) ? 0 : 1;
            const uint32_t hb = 3u + static_cast<uint32_t>(mine);   // hand-offs that carry a failure
            const uint32_t hs = 5u + static_cast<uint32_t>(mine);   // plain hand-offs
            const int cpb = D / 128;   // chunks per block
            int g = 0, tq = 0;
            bool go = true, bad = false;   // bad: a wait of the waiter failed (sticky)
            for (int u = ub, nu = 0; go && u < ue; u = nu, ++tq) {
                const int j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile u / nb
                nu = u + (j1 - j0);
                if (waiter && lane == 0) bad = bad || !fwait(bar(kQFull), tq & 1, abort, args.timeout_ns);
                __syncwarp();
                if (bar_any(hb, 64, bad)) break;
                for (int j = j0; go && j < j1; ++j, ++g) {
                    if ((g & 1) != mine) continue;
                    const int buf = g & 1;
                    const uint32_t d = tmem + static_cast<uint32_t>(buf * 128);
                    for (int c = 0; c < cpb; ++c) {
                        const int kq = g * cpb + c;
                        const int st = kq % kFlashKStages;
                        if (waiter && lane == 0) {
                            if (c == 0 && g >= 2)
                                bad = bad || !fwait(bar(kSEmpty + buf), ((g >> 1) - 1) & 1, abort, args.timeout_ns);
                            bad = bad || !fwait(bar(kKFull + st), (kq / kFlashKStages) & 1, abort, args.timeout_ns);
                        }
                        __syncwarp();
                        // a block's first chunk carries any failure so far; within the
                        // block a plain barrier, which costs the issuer less (a failure
                        // there lets the issuer run on stale operands until the next
                        // block: wrong scores, never a wrong address, and the status
                        // word reports the call as failed)
                        if (c == 0) {
                            if (bar_any(hb, 64, bad)) {
                                go = false;
                                break;
                            }
                        } else {
                            named_sync(hs, 64);
                        }
                        if (!waiter && lane == 0) {
                            tc_fence_after_sync();
                            const uint32_t qa = tmem + 256u + static_cast<uint32_t>(c * 64);
                            const uint32_t ka = base + lay.kring + st * 32768u;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                umma_f16_ta(d, qa + kk * 8, sw128_kmajor_desc(ka + (kk >> 2) * 16384u + (kk & 3) * 32),
                                            idesc, (c > 0 || kk > 0) ? 1u : 0u);
                            umma_commit(bar(kKEmpty + st));
                        }
                        __syncwarp();
                    }
                    if (go && !waiter && lane == 0) umma_commit(bar(kSFull + buf));
                }
                if (go && !waiter && lane == 0) umma_commit(bar(kQFree));
            }
            if (!waiter && lane == 0) umma_commit(bar(kSDrain));
        } else if (!skip && warp >= 2 && warp < 10) {
            // ---- softmax: two warps per quarter of the query rows (warps w and
            // w + 4 share a lane quarter of tensor memory), each with 64 of a
            // block's 128 key columns, one row per thread.  The two halves of a
            // row exchange their maxima at a barrier of the pair, so that both
            // take the same rescale decision and weigh against the same m ----
            const int quad = warp & 3, hc = (warp - 2) >> 2;
            const int row = quad * 32 + lane;
            const bool shipper = threadIdx.x == 64;   // issues the bulk copies to the output CTA
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            const uint32_t remote = mapa_shared(base, 1) - base;   // add to an offset for CTA 1's address
            // keys 64 hc .. 64 hc + 63 of the block: weights subtile hc
            const uint32_t prow = base + lay.pstage + static_cast<uint32_t>(hc) * 16384u + static_cast<uint32_t>(row) * 128u;
            const uint32_t sw = static_cast<uint32_t>(row & 7);
            const uint32_t pair = 7u + static_cast<uint32_t>(quad);   // named barrier of the two warps of a quarter
            float *astage = reinterpret_cast<float *>(gbase + lay.astage);
            unsigned int *fstage = reinterpret_cast<unsigned int *>(gbase + lay.fstage);
            float *lstage = reinterpret_cast<float *>(gbase + lay.lstage);
            // the half-row maxima go through the row-sum staging area, which
            // holds nothing from the copy of a piece's sums to the next piece's end
            float *xstage = lstage;
            int g = 0, tq = 0;
            bool go = true, pending = false;
            for (int u = ub, nu = 0; go && u < ue; u = nu, ++tq) {
                const int t = u / nb, j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile t
                nu = u + (j1 - j0);
                float m = -INFINITY, l = 0.f;   // l: this half's share of the row sum
                {
                    // the tile's q rows into tensor memory (columns 256 + d/2; each
                    // warp one half of the dimensions of its quarter's rows), once
                    // the previous tile's MMAs are done with them
                    const bool ok = tq == 0 || fwait(bar(kQFree), (tq - 1) & 1, abort, args.timeout_ns);
                    if (bar_any(1, 256, !ok || *abort)) break;
                    tc_fence_after_sync();
                    // (through the weights staging buffer: it holds no weights
                    // now, the previous piece ended with every copy out of it read)
                    flash_load_q<1>(args, tmem, lane_base, t, quad, lane,
                                    base + lay.pstage + static_cast<uint32_t>(quad) * 8192u + static_cast<uint32_t>(hc) * 4096u,
                                    hc * (D / 128), (hc + 1) * (D / 128));
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kQFull));
                }
                for (int j = j0; j < j1; ++j, ++g) {
                    const int buf = g & 1;
                    const bool ok = fwait(bar(kSFull + buf), (g >> 1) & 1, abort, args.timeout_ns);
                    tc_fence_after_sync();
                    // the staging buffer is free once the previous copy has read it
                    if (shipper && pending) {
                        bulk_wait_read_all();
                        pending = false;
                    }
                    // one decision for all eight warps, so that none is left at a barrier
                    if (bar_any(1, 256, !ok || *abort)) {
                        go = false;
                        break;
                    }
                    const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(buf * 128 + hc * 64);
                    // one pass with the running maximum m, redone with the block's
                    // maximum when that exceeds m by more than the threshold (a
                    // decision per warp pair: tensor-memory loads are warp-collective,
                    // and both halves of a row decide alike)
                    float m_new = m, lb = 0.f;
                    bool resc = false;
#pragma unroll 1
                    for (int pass = 0; pass < 2; ++pass) {
                        float mx = -INFINITY;
                        lb = 0.f;
                        uint32_t v0[32], v1[32];
                        tmem_ld_32x32b_x32(taddr, v0);
                        tmem_ld_32x32b_x32(taddr + 32u, v1);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t w[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const uint32_t x0 = c ? v1[2 * k] : v0[2 * k], x1 = c ? v1[2 * k + 1] : v0[2 * k + 1];
                                const float s0 = __uint_as_float(x0), s1 = __uint_as_float(x1);
                                mx = fmaxf(mx, fmaxf(s0, s1));
                                const float p0 = ex2_approx(fmaf(s0, args.scale_log2, -m_new));
                                const float p1 = ex2_approx(fmaf(s1, args.scale_log2, -m_new));
                                w[k] = pack_bf16(p0, p1);
                                lb += __uint_as_float(w[k] << 16) + __uint_as_float(w[k] & 0xffff0000u);
                            }
                            // keys 64 hc + 32c .. + 31: 16-byte chunks 4c .. 4c + 3 of the subtile row
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t chunk = static_cast<uint32_t>(c * 4 + q);
                                sts128(prow + ((chunk ^ sw) << 4), make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
                            }
                        }
                        if (pass == 0) {
                            xstage[hc * 128 + row] = mx;
                            named_sync(pair, 64);
                            mx = fmaxf(mx, xstage[(hc ^ 1) * 128 + row]);
                            mx *= args.scale_log2;
                            resc = mx > m + kFlashRescaleLog2;
                            if (resc) m_new = mx;
                            if (!__any_sync(0xffffffffu, resc)) break;
                        }
                    }
                    const float alpha = resc ? ex2_approx(m - m_new) : 1.0f;
                    l = l * alpha + lb;
                    m = m_new;
                    // the scores are read: the MMA may overwrite the buffer
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kSEmpty + buf));
                    const unsigned any = __any_sync(0xffffffffu, resc) ? 1u : 0u;
                    if (hc == 0) {
                        astage[row] = alpha;
                        if (lane == 0) fstage[quad] = any;
                    }
                    fence_proxy_async_smem();   // the staged block, visible to the bulk copy
                    named_sync(2, 256);
                    if (shipper) {
                        // once the output CTA's MMAs have consumed the buffer two blocks back
                        if (g < 2 || fwait(bar(kPEmpty + buf), ((g >> 1) - 1) & 1, abort, args.timeout_ns)) {
                            // (the output CTA armed its barrier for these bytes)
                            const uint32_t full = base + remote + lay.bars + 8u * (kPFull + buf);
                            bulk_copy_to_peer(base + remote + lay.p + static_cast<uint32_t>(buf) * 32768u,
                                              base + lay.pstage, 32768u, full);
                            bulk_copy_to_peer(base + remote + lay.alpha + static_cast<uint32_t>(buf) * 512u,
                                              base + lay.astage, 512u, full);
                            bulk_copy_to_peer(base + remote + lay.flags + static_cast<uint32_t>(buf) * 16u,
                                              base + lay.fstage, 16u, full);
                            bulk_commit();
                            pending = true;
                        }
                    }
                }
                if (!go) break;
                // the piece's row sums (the two halves added) and maxima, once the
                // output CTA has read the ones that went into the same buffer two
                // pieces back (a failed wait sets the abort flag, which every
                // softmax warp sees at the next block)
                if (hc == 1) lstage[row] = l;
                named_sync(2, 256);
                if (hc == 0) {
                    lstage[row] = l + lstage[row];
                    lstage[128 + row] = m;
                }
                fence_proxy_async_smem();
                named_sync(2, 256);
                if (shipper &&
                    (tq < 2 || fwait(bar(kLEmpty + (tq & 1)), ((tq >> 1) - 1) & 1, abort, args.timeout_ns))) {
                    const uint32_t full = base + remote + lay.bars + 8u * (kLFull + (tq & 1));
                    bulk_copy_to_peer(base + remote + lay.lsum + static_cast<uint32_t>(tq & 1) * 1024u,
                                      base + lay.lstage, 1024u, full);
                    bulk_commit();
                    bulk_wait_read_all();
                    pending = false;
                }
            }
            // every copy has landed in the output CTA before this CTA can leave
            if (shipper) bulk_wait_all();
        }
    } else {
        if (!skip && warp == 0 && lane == 0) {
            // ---- producer: V'^T, stages of 64 keys x one half of D ----
            // (V'^T is the output of the kernel launched before this one,
            // which may still be running: this CTA's only read of it)
            tc::griddep_wait();
            int vq = 0;
            bool go = true;
            const uint32_t stage_bytes = static_cast<uint32_t>(half) * 128u;
            for (int u = ub, nu = 0; go && u < ue; u = nu) {
                const int t = u / nb, j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile t
                nu = u + (j1 - j0);
                for (int j = j0; go && j < j1; ++j)
                    for (int kh = 0; kh < 4; ++kh, ++vq) {   // (64-key chunk, half) pairs
                        const int st = vq % kFlashVStages;
                        if (vq >= kFlashVStages &&
                            !fwait(bar(kVEmpty + st), ((vq / kFlashVStages) - 1) & 1, abort, args.timeout_ns)) {
                            go = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(kVFull + st), stage_bytes);
                        tma_load_2d(base + lay.vring + static_cast<uint32_t>(st) * stage_bytes, &map_v,
                                    ((j + t) % nb) * 128 + (kh >> 1) * 64, (kh & 1) * half, bar(kVFull + st));
                        counters[4] = vq + 1;   // V stages issued
                    }
            }
        } else if (!skip && (warp == 1 || warp == 10 || warp >= 12)) {
            // ---- MMA: O += P V' per block, one half of D per issuer (warp 1
            // the first, warp 10 the second).  Warp 12 (13) does the waiting
            // for warp 1 (10), including the rescale handshake with the
            // epilogue, and hands each go-ahead over at named barrier 3 (4) ----
            const bool waiter = warp >= 12;
            const int h = (warp == 1 || warp == 12) ? 0 : 1;
            const uint32_t hb = 3u + static_cast<uint32_t>(h);   // hand-offs that carry a failure
            const uint32_t hs = 5u + static_cast<uint32_t>(h);   // plain hand-offs
            const bool lead = h == 0;   // its waiter posts the rescale requests and the tile's end
            const uint32_t idesc = umma_idesc_bf16_f32(128, half);
            volatile int *mailbox = reinterpret_cast<volatile int *>(gbase + lay.mailbox);
            volatile int *flags = reinterpret_cast<volatile int *>(gbase + lay.flags);
            int g = 0, tq = 0, ro = 0;
            bool go = true, bad = false;   // bad: a wait of the waiter failed (sticky)
            for (int u = ub, nu = 0; go && u < ue; u = nu, ++tq) {
                const int j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile u / nb
                nu = u + (j1 - j0);
                for (int j = j0; j < j1; ++j, ++g) {
                    const int buf = g & 1;
                    for (int kc = 0; kc < 2; ++kc) {   // the two 64-key chunks of this half
                        const int vq = g * 4 + kc * 2 + h;
                        const int st = vq % kFlashVStages;
                        if (waiter && lane == 0) {
                            if (kc == 0) {
                                bad = bad || !wait_cluster(bar(kPFull + buf), (g >> 1) & 1, abort, args.timeout_ns);
                                if (!bad && j == j0) {
                                    // the previous tile's output has been written out
                                    bad = tq > 0 && !fwait(bar(kOFree), (tq - 1) & 1, abort, args.timeout_ns);
                                } else if (!bad && (flags[buf * 4] | flags[buf * 4 + 1] | flags[buf * 4 + 2] |
                                                    flags[buf * 4 + 3])) {
                                    // O (both halves) complete up to the previous block, then
                                    // its rows rescaled by the epilogue
                                    bad = !fwait(bar(kPDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort, args.timeout_ns);
                                    if (!bad && lead) {
                                        *mailbox = buf;
                                        mbar_arrive(bar(kRescaleReq));
                                    }
                                    bad = bad || !fwait(bar(kORescaled), ro & 1, abort, args.timeout_ns);
                                    ++ro;
                                }
                            }
                            bad = bad || !fwait(bar(kVFull + st), (vq / kFlashVStages) & 1, abort, args.timeout_ns);
                        }
                        __syncwarp();
                        // as on the score side: the block's first chunk carries failures
                        if (kc == 0) {
                            if (bar_any(hb, 64, bad)) {
                                go = false;
                                break;
                            }
                        } else {
                            named_sync(hs, 64);
                        }
                        if (!waiter && lane == 0) {
                            tc_fence_after_sync();
                            const uint32_t pa = base + lay.p + static_cast<uint32_t>(buf) * 32768u + kc * 16384u;
                            const uint32_t va = base + lay.vring + static_cast<uint32_t>(st * half) * 128u;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_f16(tmem + static_cast<uint32_t>(h * half), sw128_kmajor_desc(pa + kk * 32),
                                         sw128_kmajor_desc(va + kk * 32), idesc, (j > j0 || kc > 0 || kk > 0) ? 1u : 0u);
                            umma_commit(bar(kVEmpty + st));
                        }
                        __syncwarp();
                    }
                    if (!go) break;
                    if (!waiter && lane == 0) umma_commit(bar(kPDone + buf));
                }
                if (!go) break;
                if (!waiter && lane == 0) umma_commit(bar(kOFull));
                if (waiter && lead && lane == 0 && !bad) {
                    *mailbox = kFlashEnd;
                    mbar_arrive(bar(kRescaleReq));
                }
            }
            if (!waiter && lane == 0) umma_commit(bar(kODrain));
        } else if (!skip && warp == 11 && lane == 0) {
            // ---- forwarder: a weights buffer goes back to the score CTA once its MMAs are done ----
            const uint32_t peer = mapa_shared(base, 0) - base;
            int g = 0;
            bool go = true;
            for (int u = ub; go && u < ue; ++u, ++g) {   // one key block per unit
                if (!fwait(bar(kPDone + (g & 1)), (g >> 1) & 1, abort, args.timeout_ns)) {
                    go = false;
                    break;
                }
                // the buffer's next use expects its bytes; then it goes back
                mbar_arrive_expect_tx(bar(kPFull + (g & 1)), kFlashPBytes);
                mbar_arrive_cluster(base + peer + lay.bars + 8u * (kPEmpty + (g & 1)));
            }
        } else if (!skip && warp >= 2 && warp < 10) {
            // ---- epilogue warps: rescale O on request; out = O / l + residual at the tile's end ----
            const int quad = warp & 3, h = (warp - 2) >> 2;
            const int row = quad * 32 + lane;
            const uint32_t taddr0 = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(h * half);
            const uint32_t peer0 = mapa_shared(base, 0) - base;   // add to an offset for CTA 0's address
            volatile int *mailbox = reinterpret_cast<volatile int *>(gbase + lay.mailbox);
            const float *alpha = reinterpret_cast<const float *>(gbase + lay.alpha);
            const float *lsum = reinterpret_cast<const float *>(gbase + lay.lsum);
            int rr = 0, tq = 0;
            bool go = true;
            for (int u = ub, nu = 0; go && u < ue; u = nu, ++tq) {
                const int t = u / nb, j0 = u % nb, j1 = min(nb, j0 + (ue - u));   // a piece of tile t
                nu = u + (j1 - j0);
                for (;;) {
                    const bool ok = fwait(bar(kRescaleReq), rr & 1, abort, args.timeout_ns);
                    ++rr;
                    if (!__all_sync(0xffffffffu, ok && !*abort)) {
                        go = false;
                        break;
                    }
                    const int mb = *mailbox;
                    if (mb == kFlashEnd) break;
                    tc_fence_after_sync();
                    const float a = alpha[mb * 128 + row];
#pragma unroll 1
                    for (int c = 0; c < half; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr0 + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * a);
                        tmem_st_32x32b_x32(taddr0 + c, v);
                    }
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kORescaled));
                }
                if (!go) break;
                bool ok = fwait(bar(kOFull), tq & 1, abort, args.timeout_ns);
                ok = ok && wait_cluster(bar(kLFull + (tq & 1)), (tq >> 1) & 1, abort, args.timeout_ns);
                // the buffer's next use (at the end of the tile two on, long after
                // this tile's sums are read) expects its bytes
                if (ok && warp == 2 && lane == 0) mbar_arrive_expect_tx(bar(kLFull + (tq & 1)), 1024u);
                tc_fence_after_sync();
                if (!__all_sync(0xffffffffu, ok && !*abort)) break;
                const float lrow = lsum[(tq & 1) * 256 + row], mrow = lsum[(tq & 1) * 256 + 128 + row];
                __syncwarp();
                // the score CTA may ship the next sums into this buffer
                if (lane == 0) mbar_arrive_cluster(base + peer0 + lay.bars + 8u * (kLEmpty + (tq & 1)));
                if (j0 == 0 && j1 == nb) {
                    // the whole tile: out = O / l + residual
                    const float inv = 1.0f / lrow;
                    const int64_t orow = static_cast<int64_t>(t) * 128 + row;
                    __nv_bfloat16 *dst = args.out + orow * D + h * half;
                    const __nv_bfloat16 *res = args.residual ? args.residual + orow * D + h * half : nullptr;
#pragma unroll 1
                    for (int c = 0; c < half; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr0 + c, v);
                        tmem_wait_ld();
                        float f[32];
#pragma unroll
                        for (int k = 0; k < 32; ++k) f[k] = __uint_as_float(v[k]) * inv;
                        if (res) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint4 rr4 = *reinterpret_cast<const uint4 *>(res + c + 8 * q);
                                const uint32_t w[4] = {rr4.x, rr4.y, rr4.z, rr4.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    f[8 * q + 2 * e] += __uint_as_float(w[e] << 16);
                                    f[8 * q + 2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4 *>(dst + c + 8 * q) = make_uint4(
                                pack_bf16(f[8 * q], f[8 * q + 1]), pack_bf16(f[8 * q + 2], f[8 * q + 3]),
                                pack_bf16(f[8 * q + 4], f[8 * q + 5]), pack_bf16(f[8 * q + 6], f[8 * q + 7]));
                    }
                } else {
                    // a piece of the tile: the unnormalised O ([D][128], so that a
                    // warp's stores of one column are contiguous) with the row's m
                    // and l, for attn_combine_kernel
                    float *slot = args.partial + static_cast<size_t>(2 * cl + (u == ub ? 0 : 1)) * flash_slot_floats(D);
#pragma unroll 1
                    for (int c = 0; c < half; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr0 + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            slot[static_cast<size_t>(h * half + c + k) * 128 + row] = __uint_as_float(v[k]);
                    }
                    if (h == 0) {
                        slot[static_cast<size_t>(D) * 128 + row] = mrow;
                        slot[static_cast<size_t>(D) * 128 + 128 + row] = lrow;
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kOFree));
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort && !skip && threadIdx.x == 0) {
        // let every copy and MMA this CTA started land before it leaves
        if (scorer) {
            // the last loads of every stage (earlier phases of a stage are complete)
            for (int q = counters[1] > kFlashKStages ? counters[1] - kFlashKStages : 0; q < counters[1]; ++q)
                tc::drain(bar(kKFull + q % kFlashKStages), (q / kFlashKStages) & 1, args.timeout_ns);
            tc::drain(bar(kSDrain), 0, args.timeout_ns);
        } else {
            for (int q = counters[4] > kFlashVStages ? counters[4] - kFlashVStages : 0; q < counters[4]; ++q)
                tc::drain(bar(kVFull + q % kFlashVStages), (q / kFlashVStages) & 1, args.timeout_ns);
            tc::drain(bar(kODrain), 0, args.timeout_ns);
        }
    }
    __syncthreads();
    __syncwarp();
    cluster_sync_all();   // neither CTA leaves while the other may still write into it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// Merges the pieces of each tile that more than one cluster worked on: with
// M the largest of the pieces' row maxima m_i and w_i = 2^(m_i - M),
//   out = (sum_i w_i O_i) / (sum_i w_i l_i) + residual.
// Grid (split tiles, D / kCombineCols), 128 threads, one row per thread and
// kCombineCols columns.  The residual and every piece's row maximum, row sum
// and outputs are loaded before any of them is used, so the merge waits for
// one round of loads (pieces past kCombineHeld, which the usual splits do
// not make, are folded in afterwards one at a time); the register bound
// keeps eight CTAs on an SM, so that the usual grids run in one or two rounds.
constexpr int kCombineCols = 16;
constexpr int kCombineHeld = 2;
constexpr int kCombineMaxTiles = kAttnMaxS / 128;

// The split tiles of a launch, each by the cluster that holds its first unit.
struct CombineTiles {
    int n;
    uint16_t c_lo[kCombineMaxTiles];
};

__global__ void __launch_bounds__(128, 8) attn_combine_kernel(const FlashArgs a, const __grid_constant__ CombineTiles ct)
{
    tc::griddep_wait();   // the pieces come from the pair kernel launched before this one
    const int nb = a.nblocks, D = a.D;
    const int c_lo = ct.c_lo[blockIdx.x];
    const int t = flash_unit_begin(a, c_lo + 1) / nb;   // the tile's first inner boundary follows cluster c_lo
    int c_hi = c_lo + 1;                                // the cluster holding the tile's last unit
    while (c_hi + 1 < a.clusters && flash_unit_begin(a, c_hi + 1) < (t + 1) * nb) ++c_hi;
    const int np = c_hi - c_lo + 1;
    const int row = threadIdx.x, col0 = blockIdx.y * kCombineCols;
    const size_t sf = flash_slot_floats(D), ml = static_cast<size_t>(D) * 128;
    // a cluster's piece of tile t is its first one if its units begin in tile t, else its last
    const auto slot_of = [&](int c) {
        return a.partial + static_cast<size_t>(2 * c + (flash_unit_begin(a, c) / nb == t ? 0 : 1)) * sf;
    };
    const int64_t orow = static_cast<int64_t>(t) * 128 + row;
    uint4 r4[kCombineCols / 8];
#pragma unroll
    for (int q = 0; q < kCombineCols / 8; ++q) r4[q] = make_uint4(0u, 0u, 0u, 0u);
    if (a.residual) {
        const uint4 *res = reinterpret_cast<const uint4 *>(a.residual + orow * D + col0);
#pragma unroll
        for (int q = 0; q < kCombineCols / 8; ++q) r4[q] = res[q];
    }
    float m[kCombineHeld], l[kCombineHeld], o[kCombineHeld][kCombineCols];
#pragma unroll
    for (int i = 0; i < kCombineHeld; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int k = 0; k < kCombineCols; ++k) o[i][k] = 0.f;
        if (i < np) {
            const float *sl = slot_of(c_lo + i);
            m[i] = sl[ml + row];
            l[i] = sl[ml + 128 + row];
#pragma unroll
            for (int k = 0; k < kCombineCols; ++k) o[i][k] = sl[static_cast<size_t>(col0 + k) * 128 + row];
        }
    }
    float M = m[0];
#pragma unroll
    for (int i = 1; i < kCombineHeld; ++i) M = fmaxf(M, m[i]);
    for (int i = kCombineHeld; i < np; ++i) M = fmaxf(M, slot_of(c_lo + i)[ml + row]);
    float acc[kCombineCols];
#pragma unroll
    for (int k = 0; k < kCombineCols; ++k) acc[k] = 0.f;
    float L = 0.f;
#pragma unroll
    for (int i = 0; i < kCombineHeld; ++i) {
        const float w = exp2f(m[i] - M);   // 0 for the pieces past np (m = -inf)
        L += w * l[i];
#pragma unroll
        for (int k = 0; k < kCombineCols; ++k) acc[k] += w * o[i][k];
    }
    for (int i = kCombineHeld; i < np; ++i) {
        const float *sl = slot_of(c_lo + i);
        const float w = exp2f(sl[ml + row] - M);
        L += w * sl[ml + 128 + row];
#pragma unroll
        for (int k = 0; k < kCombineCols; ++k) acc[k] += w * sl[static_cast<size_t>(col0 + k) * 128 + row];
    }
    const float inv = 1.0f / L;
    __nv_bfloat16 *dst = a.out + orow * D + col0;
#pragma unroll
    for (int q = 0; q < kCombineCols / 8; ++q) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = acc[8 * q + e] * inv;
        if (a.residual) {
            const uint32_t w[4] = {r4[q].x, r4[q].y, r4[q].z, r4[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] += __uint_as_float(w[e] << 16);
                f[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        *reinterpret_cast<uint4 *>(dst + 8 * q) = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                                            pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {


// A bf16 [rows][K] K-major operand, boxes of {64, box_rows}, 128-byte swizzle.
bool encode_kmajor(tc::EncodeTiledFn enc, CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES>
cudaError_t launch_gemm_variant(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &a, int sm_count,
                                cudaStream_t s)
{
    using L = GemmLayout<BN, STAGES>;
    static_assert(L::kDynamic <= 227 * 1024, "gemm ring does not fit in shared memory");
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gemm_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::kDynamic));
    });
    if (attr != cudaSuccess) return attr;
    const int blocks = a.tiles < sm_count ? a.tiles : sm_count;
    const cudaError_t e = tc::launch_pdl(gemm_kernel<BN, STAGES>, dim3(blocks), dim3(kGemmThreads), L::kDynamic, s,
                                         ma, mb, a);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

bool gemm_pair_enabled()
{
    static const bool on = [] {
        const char *v = std::getenv("GN_GEMM_PAIR");
        return !(v && v[0] == '0');
    }();
    return on;
}

// The three GEMM schedules and a rough cost model to choose among them:
// time ~ rounds of tiles over the SMs (or SM pairs) x the per-SM work of one
// tile / its tensor-pipe efficiency (CTA pairs ~0.93, single CTA 128x256
// ~0.80, 128x128 ~0.70).  CTA pairs need 16 or more K steps per tile to pay
// off (at S = 16384 the weighted sum, K = S, runs 199 -> 173 us on pairs,
// while the 8-step score passes run slower).  Problems with few tiles take
// the 128-wide tiles so that more SMs work (the weighted sum at S = 4096
// has 32 pair tiles for 76 pairs).
enum GemmSchedule { kPair256 = 0, kSingle256 = 1, kSingle128 = 2 };

GemmSchedule choose_gemm(int M, int N, int K, int sm_count)
{
    const auto cost = [sm_count](int64_t units, bool pair, double area_over_eff) {
        const int64_t slots = pair ? sm_count / 2 : sm_count;
        return static_cast<double>((units + slots - 1) / slots) * area_over_eff;
    };
    GemmSchedule best = kSingle128;
    double best_cost = cost(static_cast<int64_t>(M / 128) * (N / 128), false, 128.0 * 128.0 / 0.70);
    if (N % 256 == 0) {
        const double c = cost(static_cast<int64_t>(M / 128) * (N / 256), false, 128.0 * 256.0 / 0.80);
        if (c <= best_cost) {
            best = kSingle256;
            best_cost = c;
        }
        if (M % 256 == 0 && K / kBK >= 16 && gemm_pair_enabled()) {
            const double cp = cost(static_cast<int64_t>(M / 256) * (N / 256), true, 128.0 * 256.0 / 0.93);
            if (cp < best_cost) best = kPair256;
        }
    }
    return best;
}

int schedule_bn(GemmSchedule g) { return g == kSingle128 ? 128 : 256; }


template <int STAGES>
cudaError_t launch_gemm_pair(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &a, int sm_count,
                             cudaStream_t s)
{
    using L = GemmPairLayout<STAGES>;
    static_assert(L::kDynamic <= 227 * 1024, "gemm pair ring does not fit in shared memory");
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    static int max_clusters = 0;
    std::call_once(once, [sm_count] {
        attr = cudaFuncSetAttribute(gemm_pair_kernel<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::kDynamic));
        if (attr != cudaSuccess) return;
        max_clusters = tc::pair_clusters(gemm_pair_kernel<STAGES>, kGemmThreads, L::kDynamic, sm_count);
    });
    if (attr != cudaSuccess) return attr;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int pairs = a.tiles < max_clusters ? a.tiles : max_clusters;
    const cudaError_t e = tc::launch_pdl(gemm_pair_kernel<STAGES>, dim3(2 * pairs), dim3(kGemmThreads), L::kDynamic, s,
                                         ma, mb, a);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

// C[M][N] = alpha A[M][K] B[N][K]^T (+ bias_m[M], + bias_n[N], + residual),
// or the softmax statistics / weights of alpha A B^T (mode)
int run_gemm(const void *A, const void *B, void *C, int M, int N, int K, float alpha, const float *bias_m,
             const float *bias_n, const void *residual, bool out_f32, int mode, float2 *stats,
             const float2 *row_ml, int sm_count, uint64_t timeout_ns, cudaStream_t s, cudaError_t *err)
{
    tc::EncodeTiledFn enc = tc::encode_fn();
    if (!enc) return 2;
    const GemmSchedule sched = choose_gemm(M, N, K, sm_count);
    const int BN = schedule_bn(sched);
    // CTA pairs take 256-row x 256-column tiles (each CTA 128 rows and half the columns' B rows)
    const bool pair = sched == kPair256;
    CUtensorMap ma, mb;
    if (!encode_kmajor(enc, &ma, A, M, K, kBM) || !encode_kmajor(enc, &mb, B, N, K, pair ? 128 : BN)) return 2;
    GemmArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.n_tiles = N / BN;
    a.tiles = (M / (pair ? 2 * kBM : kBM)) * a.n_tiles;
    a.ksteps = K / kBK;
    a.alpha = alpha;
    a.bias_m = bias_m;
    a.bias_n = bias_n;
    a.residual = static_cast<const __nv_bfloat16 *>(residual);
    a.c = C;
    a.out_f32 = out_f32 ? 1 : 0;
    a.mode = mode;
    a.stats = stats;
    a.row_ml = row_ml;
    a.timeout_ns = timeout_ns;
    if (pair) {
        *err = launch_gemm_pair<6>(ma, mb, a, sm_count, s);
        return *err == cudaSuccess ? 0 : 3;
    }
    *err = (BN == 256) ? launch_gemm_variant<256, 4>(ma, mb, a, sm_count, s)
                       : launch_gemm_variant<128, 6>(ma, mb, a, sm_count, s);
    return *err == cudaSuccess ? 0 : 3;
}

}  // namespace

cudaError_t launch_attn_fold(const void *wv, const void *bv, const void *wo, const void *bo, void *wf, float *bf,
                             int D, int sm_count, cudaStream_t s)
{
    const int64_t total = static_cast<int64_t>(D) * (D + 1);
    const int64_t want = (total + 255) / 256;
    const int blocks = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
    attn_fold_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(wv),
                                            static_cast<const __nv_bfloat16 *>(bv),
                                            static_cast<const __nv_bfloat16 *>(wo),
                                            static_cast<const __nv_bfloat16 *>(bo), static_cast<__nv_bfloat16 *>(wf),
                                            bf, D);
    return cudaGetLastError();
}

namespace {

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// workspace: V'^T [D][S] bf16 | segment statistics [S][2 S/128] float2 (room
// for the 128-wide tiles) | row (max, 1/sum) [S] float2 | P [S][S] bf16
struct AttnWorkspace {
    size_t vt, stats, row_ml, p, total;
};

AttnWorkspace attn_layout(int64_t S, int64_t D)
{
    AttnWorkspace w;
    w.vt = 0;
    w.stats = w.vt + up256(static_cast<size_t>(2 * D * S));
    w.row_ml = w.stats + up256(static_cast<size_t>(8 * S * 2 * (S / 128)));
    w.p = w.row_ml + up256(static_cast<size_t>(8 * S));
    w.total = w.p + up256(static_cast<size_t>(2 * S * S));
    return w;
}

}  // namespace

size_t attn_workspace_bytes(int64_t S, int64_t D) { return attn_layout(S, D).total; }

namespace {

// Co-resident CTA pairs of the one-pass kernel at this shared-memory size
// (the occupancy query, once per size and device SM count).
int flash_pair_capacity(uint32_t smem, int sm_count)
{
    static std::mutex mu;
    static std::map<std::pair<uint32_t, int>, int> known;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(smem, sm_count);
    const auto it = known.find(key);
    if (it != known.end()) return it->second;
    const int cap = tc::pair_clusters(attn_flash_kernel, kFlashThreads, smem, sm_count);
    known[key] = cap;
    return cap;
}

// How many CTA pairs, and whether they share the (tile, key block) units
// equally (runs may end inside a tile: its pieces are merged afterwards,
// which needs two workspace slots per pair -- at most `fit` pairs) or take
// whole tiles: the cheapest by an estimate calibrated on a GB300 at D = 512,
// ~2 us per key block on the busiest pair, ~9 us per piece of a tile a pair
// starts (pipeline fill and drain), ~5 us for the merge.  (Measured at
// S = 4096: 64 pairs with half a tile each 63 us, 67 pairs with runs that
// cross a tile boundary 73 us, 32 pairs with a tile each 91 us.)  The
// result is remembered per shape.
void choose_flash_pairs(int tiles, int nblocks, int cap, size_t fit, int *pairs, int *split)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, std::pair<int, int>> known;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(tiles, nblocks, cap, fit);
    const auto it = known.find(key);
    if (it != known.end()) {
        *pairs = it->second.first;
        *split = it->second.second;
        return;
    }
    FlashArgs t{};
    t.tiles = tiles;
    t.nblocks = nblocks;
    t.units = tiles * nblocks;
    int best_c = 1, best_split = 0;
    double best_cost = 0.0;
    for (int c = 1; c <= cap && c <= t.units; ++c) {
        t.clusters = c;
        t.split = (tiles % c != 0) ? 1 : 0;
        if (t.split && static_cast<size_t>(c) > fit) continue;   // no room for the pieces
        if (!t.split && c > tiles) continue;
        int max_blocks = 0, max_pieces = 0;
        for (int k = 0; k < c; ++k) {
            const int ub = flash_unit_begin(t, k), ue = flash_unit_begin(t, k + 1);
            if (ue <= ub) continue;
            max_blocks = max_blocks > ue - ub ? max_blocks : ue - ub;
            const int pieces = (ue - 1) / nblocks - ub / nblocks + 1;
            max_pieces = max_pieces > pieces ? max_pieces : pieces;
        }
        const double cost = 2.0 * max_blocks + 9.0 * max_pieces + (t.split ? 5.0 : 0.0);
        if (c == 1 || cost < best_cost) {
            best_cost = cost;
            best_c = c;
            best_split = t.split;
        }
    }
    if (known.size() >= 256) known.clear();   // callers with ever new workspace sizes
    known[key] = std::make_pair(best_c, best_split);
    *pairs = best_c;
    *split = best_split;
}

// The tiles that the clusters' runs of units split: a boundary between two
// runs that falls inside a tile splits it, and the first such boundary of
// the tile names it (by the cluster before it, which holds the tile's first
// unit).
CombineTiles split_tiles(const FlashArgs &a)
{
    CombineTiles ct;
    ct.n = 0;
    int last = -1;
    for (int c = 1; c < a.clusters; ++c) {
        const int b = flash_unit_begin(a, c);
        if (b % a.nblocks == 0 || b / a.nblocks == last) continue;
        last = b / a.nblocks;
        ct.c_lo[ct.n++] = static_cast<uint16_t>(c - 1);
    }
    return ct;
}

// 0 = launched (*launches kernels); 2 = tensor-map encoding failed; 3 = a
// launch failed.  partial / partial_bytes: workspace the pieces of split
// tiles may use.
int run_flash(const void *q, const void *k, const void *vt, const void *residual, void *out, int S, int D,
              void *partial, size_t partial_bytes, int sm_count, uint64_t timeout_ns, cudaStream_t s,
              cudaError_t *err, int *launches)
{
    tc::EncodeTiledFn enc = tc::encode_fn();
    if (!enc) return 2;
    CUtensorMap mq, mk, mv;
    if (!encode_kmajor(enc, &mq, q, S, D, 128) || !encode_kmajor(enc, &mk, k, S, D, 128) ||
        !encode_kmajor(enc, &mv, vt, D, S, D / 2))
        return 2;
    FlashArgs a;
    a.S = S;
    a.D = D;
    a.tiles = S / 128;
    a.nblocks = S / 128;
    a.units = a.tiles * a.nblocks;
    a.scale_log2 = kLog2e / sqrtf(static_cast<float>(D));
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.residual = static_cast<const __nv_bfloat16 *>(residual);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.partial = static_cast<float *>(partial);
    a.timeout_ns = timeout_ns;
    const uint32_t smem = flash_layout(D).total + 1024u;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(attn_flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(flash_layout(512).total + 1024u));
    });
    if (attr != cudaSuccess) {
        *err = attr;
        return 3;
    }
    // the number of CTA pairs and the split (choose_flash_pairs)
    const int cap = flash_pair_capacity(smem, sm_count);
    const size_t slot_bytes = flash_slot_floats(D) * sizeof(float);
    const size_t fit = partial_bytes / (2 * slot_bytes);   // pairs whose pieces fit
    int best_c = 1, best_split = 0;
    choose_flash_pairs(a.tiles, a.nblocks, cap, fit, &best_c, &best_split);
    a.clusters = best_c;
    a.split = best_split;
    // both launches with programmatic serialization: the pair kernel starts
    // (barriers, tensor memory, q rows, key blocks, scores) while the
    // value-row GEMM ahead of it finishes, and waits only before loading its
    // output; the merge waits at entry
    *err = tc::launch_pdl(attn_flash_kernel, dim3(2 * a.clusters), dim3(kFlashThreads), smem, s, mq, mk, mv, a);
    if (*err != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    ++*launches;
    const CombineTiles ct = split_tiles(a);
    if (a.split && ct.n > 0) {
        *err = tc::launch_pdl(attn_combine_kernel, dim3(ct.n, D / kCombineCols), dim3(128), 0, s, a, ct);
        if (*err != cudaSuccess) {
            cudaGetLastError();
            return 3;
        }
        ++*launches;
    }
    return 0;
}

}  // namespace

int launch_attn_folded(const void *q, const void *k, const void *xn, const void *wf, const float *bf,
                       const void *residual, void *out, int S, int D, void *workspace, size_t workspace_bytes,
                       bool one_pass, int sm_count, uint64_t timeout_ns, cudaStream_t s, cudaError_t *err,
                       int *launches)
{
    const AttnWorkspace lay = attn_layout(S, D);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *vt = ws + lay.vt;
    if (one_pass) {
        *launches = 0;
        // V'^T = W' xn^T + b', then the one-pass softmax and weighted sum
        int r = run_gemm(wf, xn, vt, D, S, D, 1.0f, bf, nullptr, nullptr, false, kGemmPlain, nullptr, nullptr,
                         sm_count, timeout_ns, s, err);
        if (r) return r;
        ++*launches;
        return run_flash(q, k, vt, residual, out, S, D, ws + lay.stats, workspace_bytes - lay.stats, sm_count,
                         timeout_ns, s, err, launches);
    }
    float2 *stats = reinterpret_cast<float2 *>(ws + lay.stats);
    float2 *row_ml = reinterpret_cast<float2 *>(ws + lay.row_ml);
    void *p = ws + lay.p;
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    *launches = 0;
    // V'^T = W' xn^T + b' (b' per row of V'^T)
    int r = run_gemm(wf, xn, vt, D, S, D, 1.0f, bf, nullptr, nullptr, false, kGemmPlain, nullptr, nullptr,
                     sm_count, timeout_ns, s, err);
    if (r) return r;
    ++*launches;
    // pass 1 over the scores q k^T / sqrt(D): per-row (max, sum of exp) of each half tile
    r = run_gemm(q, k, nullptr, S, S, D, scale, nullptr, nullptr, nullptr, false, kGemmRowStats, stats, nullptr,
                 sm_count, timeout_ns, s, err);
    if (r) return r;
    ++*launches;
    // the rows' (max, 1 / sum)
    const int parts = 2 * (S / schedule_bn(choose_gemm(S, S, D, sm_count)));   // as pass 1 runs
    *err = tc::launch_pdl(softmax_stats_kernel, dim3((S + 7) / 8), dim3(256), 0, s, stats, parts, row_ml, S);
    if (*err != cudaSuccess) {
        cudaGetLastError();
        return 3;
    }
    ++*launches;
    // pass 2: the scores again, written as softmax weights P (bf16)
    r = run_gemm(q, k, p, S, S, D, scale, nullptr, nullptr, nullptr, false, kGemmSoftmax, nullptr, row_ml,
                 sm_count, timeout_ns, s, err);
    if (r) return r;
    ++*launches;
    // out = P V' + residual
    r = run_gemm(p, vt, out, S, D, S, 1.0f, nullptr, nullptr, residual, false, kGemmPlain, nullptr, nullptr,
                 sm_count, timeout_ns, s, err);
    if (r) return r;
    ++*launches;
    return 0;
}

cudaError_t read_attn_status(unsigned int *status)
{
    return cudaMemcpyFromSymbol(status, g_at_status, sizeof(unsigned int));
}

cudaError_t clear_attn_status()
{
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_at_status, &zero, sizeof(unsigned int));
}

cudaError_t set_attn_status_host(unsigned int *host_word)
{
    return cudaMemcpyToSymbol(g_at_status_host, &host_word, sizeof(host_word));
}

}  // namespace gn
