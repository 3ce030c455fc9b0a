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
// file evaluates the second form:
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
// (A single-pass, flash-style kernel does not fit D = 512 well: an fp32
// 128 x 512 output block alone fills the 512 tensor-memory columns of an SM.)
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
#include <mutex>

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
    gemm_kernel<BN, STAGES><<<blocks, kGemmThreads, L::kDynamic, s>>>(ma, mb, a);
    return cudaGetLastError();
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
    gemm_pair_kernel<STAGES><<<2 * pairs, kGemmThreads, L::kDynamic, s>>>(ma, mb, a);
    return cudaGetLastError();
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

int launch_attn_folded(const void *q, const void *k, const void *xn, const void *wf, const float *bf,
                       const void *residual, void *out, int S, int D, void *workspace, int sm_count,
                       uint64_t timeout_ns, cudaStream_t s, cudaError_t *err, int *launches)
{
    const AttnWorkspace lay = attn_layout(S, D);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *vt = ws + lay.vt;
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
    softmax_stats_kernel<<<(S + 7) / 8, 256, 0, s>>>(stats, parts, row_ml, S);
    *err = cudaGetLastError();
    if (*err != cudaSuccess) return 3;
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
