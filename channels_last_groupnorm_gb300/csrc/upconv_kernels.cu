// upconv_kernels.cu -- the decoder's up-sampler, nearest-2x upsample fused
// with the following 3x3 convolution (padding 1), on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Operation (sglang PR #33451, "FLUX.2 VAE decoder fast path behind
// quality=high", section "Modifications", item 2): with x channels-last
// [N][H][W][Cin] and the convolution weight w [Cout][Cin][3][3],
//   y[n][P][Q][co] = bias[co] + sum_{ky,kx} sum_ci u[n][P+ky-1][Q+kx-1][ci] w[co][ci][ky][kx],
//   u[n][p][q] = x[n][p/2][q/2] inside the 2H x 2W image, 0 outside.
// Nearest upsampling copies each input pixel into a 2x2 block, so an output
// pixel P = 2i + a, Q = 2j + b (parity (a, b)) reads only the 2x2 input
// window rows i + a - 1 + r, columns j + b - 1 + s (r, s in {0, 1}), and each
// window tap carries the sum of the 3x3 taps whose upsampled pixel falls on
// it: kernel row ky belongs to window row r exactly when
// floor((a + ky - 1) / 2) = r + a - 1, and likewise for columns.  These are
// the summed taps of the equivalent transposed convolution (kernel 4,
// stride 2, padding 1) that the page describes.  Per parity the convolution
// is then a GEMM with K = 4 Cin:
//   Y_ab[pixel, co] = sum_{r,s,ci} x[n][i+a-1+r][j+b-1+s][ci] * Wf_ab[co][r][s][ci].
//
// upconv_fold_kernel computes Wf (fp32 sums of bf16 taps, rounded once to
// bf16) into [4 parities][Cout][4 taps][Cin].  upconv_kernel is persistent
// (one CTA per SM) and walks output tiles of 128 pixels of one parity x BN
// output channels:
//   warp 0 (one thread)  TMA producer: per K step of 64 input channels of one
//                        tap, a 4-D box {64 ch, BW, BH, BNI} of x at the
//                        tap's shifted coordinates (out-of-image rows and
//                        columns are zero-filled by the copy engine, which is
//                        the convolution's padding) and the matching
//                        {64, BN} box of Wf, into a STAGES-deep ring that
//                        runs on across tile boundaries;
//   warp 1               allocates 2 BN tensor-memory columns (two
//                        accumulators); one thread issues four tcgen05.mma
//                        (M=128, N=BN, K=16) per K step into the tile's
//                        accumulator and commits each ring slot back to the
//                        producer and each finished accumulator to the
//                        epilogue;
//   warps 2-9            epilogue, two warps per tensor-memory lane quarter
//                        (each half of the channels): tcgen05.ld of the fp32
//                        accumulator (one pixel per thread), hand the
//                        accumulator back, + bias, round to bf16, and through a
//                        small shared-memory tile store to y at (2i + a, 2j + b)
//                        in 64-byte channel runs -- while the MMAs of the next
//                        tile run into the other accumulator.
// Every wait is bounded (a timeout sets a device status word and the CTA
// drains its copies and frees its tensor memory before it returns).
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

__device__ unsigned int g_uc_status;
// the host-visible copy of g_uc_status (mapped page-locked host memory; null until set)
__device__ unsigned int *g_uc_status_host;

namespace {

constexpr int kBM = 128;                                // output pixels per tile (MMA M)
constexpr int kBK = 64;                                 // input channels per K step
constexpr uint32_t kABytes = kBM * kBK * 2;             // 16 KB
constexpr int kUcThreads = 320;   // producer warp, MMA warp, 8 epilogue warps

struct UcArgs {
    int N, H, W, Cin, Cout;
    int BW, BH, BNI;            // the pixel box of one tile: BW x BH x BNI = 128
    int tiles_w, tiles_h;
    int co_tiles, chunks, ksteps;
    int tiles;                  // output tiles in all (tile pairs for the pair kernel)
    const __nv_bfloat16 *bias;  // [Cout] or null
    __nv_bfloat16 *y;
    uint64_t timeout_ns;
};

template <int BN, int STAGES>
struct UcLayout {
    static constexpr uint32_t kBBytes = static_cast<uint32_t>(BN) * kBK * 2;
    static constexpr uint32_t kStage = kABytes + kBBytes;
    static constexpr uint32_t kRing = kStage * STAGES;
    static constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators (double buffer)
    // after the ring, 8-byte mbarriers: full[STAGES], empty[STAGES],
    // acc_full[2], acc_empty[2], drain; then the TMEM slot, the abort flag
    // and the MMA thread's consumed-step count
    static constexpr uint32_t kBars = kRing;
    static constexpr uint32_t kTmemSlot = kBars + 8 * (2 * STAGES + 5);
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kConsumed = kAbort + 4;
    static constexpr uint32_t kStaging = (kConsumed + 4 + 15) & ~15u;   // 8 epilogue warps x 2 KB
    static constexpr uint32_t kBytes = kStaging + 8 * 2048;
    static constexpr uint32_t kDynamic = kBytes + 1024;  // slack to align the ring to 1024 B
};

// Tile t -> coordinates: the Cout tile varies fastest, then the parity, then
// the pixel tile, so CTAs working at the same time share x rows and the
// folded weights in L2.
struct TileCoord {
    int parity, i0, j0, n0, co0;
};

template <int BN>
__device__ __forceinline__ TileCoord tile_coord(int t, const UcArgs &a)
{
    TileCoord c;
    const int co_t = t % a.co_tiles;
    t /= a.co_tiles;
    c.parity = t & 3;
    t >>= 2;
    const int tw = t % a.tiles_w;
    t /= a.tiles_w;
    const int th = t % a.tiles_h;
    const int tn = t / a.tiles_h;
    c.i0 = th * a.BH;
    c.j0 = tw * a.BW;
    c.n0 = tn * a.BNI;
    c.co0 = co_t * BN;
    return c;
}



__device__ __forceinline__ int floor_half(int v) { return (v + 2) / 2 - 1; }   // floor(v / 2) for v >= -2

}  // namespace

// ---------------------------------------------------------------------------
// Wf[p][co][t][ci], p = 2a + b, t = 2r + s: the sum of w[co][ci][ky][kx] over
// the 3x3 taps that land on window tap (r, s) of parity (a, b).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) upconv_fold_kernel(const __nv_bfloat16 *__restrict__ w,
                                                          __nv_bfloat16 *__restrict__ wf, int Cin, int Cout)
{
    const int64_t total = 16LL * Cout * Cin;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int ci = static_cast<int>(idx % Cin);
        int64_t t = idx / Cin;
        const int tap = static_cast<int>(t % 4);
        t /= 4;
        const int co = static_cast<int>(t % Cout);
        const int p = static_cast<int>(t / Cout);
        const int a = p >> 1, b = p & 1, r = tap >> 1, s = tap & 1;
        const __nv_bfloat16 *src = w + (static_cast<int64_t>(co) * Cin + ci) * 9;
        float acc = 0.f;
        for (int ky = 0; ky < 3; ++ky) {
            if (floor_half(a + ky - 1) != r + a - 1) continue;
            for (int kx = 0; kx < 3; ++kx) {
                if (floor_half(b + kx - 1) != s + b - 1) continue;
                acc += __bfloat162float(src[ky * 3 + kx]);
            }
        }
        wf[idx] = __float2bfloat16_rn(acc);
    }
}

// ---------------------------------------------------------------------------
// The epilogue of one finished accumulator for one warp: the 32 pixels of
// its tensor-memory lane quarter and one half of the BN channels.  Each
// 32-channel chunk gets the bias, is rounded to bf16 and goes through a
// swizzled 2 KB shared-memory tile, so that each store instruction writes
// eight pixels' 64-byte channel runs (instead of 32 pixels' 16 bytes); the
// accumulator is handed back (one arrival on `acc_empty`, in the peer CTA
// when `remote`) once the warp's last columns are in registers.
// ---------------------------------------------------------------------------
template <int BN>
__device__ __forceinline__ void upconv_epilogue(const UcArgs &args, const TileCoord &tc, uint32_t tbase, int quad,
                                                int half, int lane, uint4 *stage, uint32_t acc_empty, bool remote)
{
    const int pa = tc.parity >> 1, pb = tc.parity & 1;
    // this lane stores pixels (lane >> 2) + 8 i of the warp's 32, 16 bytes each
    __nv_bfloat16 *rowp[4];
    bool rowv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = quad * 32 + (lane >> 2) + 8 * i;
        const int wi = m % args.BW;
        const int hi = (m / args.BW) % args.BH;
        const int n = tc.n0 + m / (args.BW * args.BH);
        rowv[i] = n < args.N;
        const int64_t P = 2LL * (tc.i0 + hi) + pa, Q = 2LL * (tc.j0 + wi) + pb;
        rowp[i] = args.y + ((static_cast<int64_t>(rowv[i] ? n : 0) * 2 * args.H + P) * 2 * args.W + Q) * args.Cout +
                  tc.co0;
    }
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
        uint32_t o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            float lo = __uint_as_float(v[2 * k]), hi2 = __uint_as_float(v[2 * k + 1]);
            if (args.bias) {
                const __nv_bfloat162 bb = *reinterpret_cast<const __nv_bfloat162 *>(args.bias + tc.co0 + c + 2 * k);
                lo += __low2float(bb);
                hi2 += __high2float(bb);
            }
            const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi2);
            o[k] = *reinterpret_cast<const uint32_t *>(&h);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            stage[lane * 4 + (k ^ (lane & 3))] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i;
            const uint4 val = stage[r * 4 + ((lane & 3) ^ (r & 3))];
            if (rowv[i]) reinterpret_cast<uint4 *>(rowp[i] + c)[lane & 3] = val;
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// the implicit-GEMM convolution: a persistent CTA per SM walks the tiles
// t = blockIdx.x, + gridDim.x, ...; the ring of operand stages runs across
// tile boundaries and the two tensor-memory accumulators alternate, so the
// epilogue of one tile overlaps the MMAs of the next.
// ---------------------------------------------------------------------------
template <int BN, int STAGES>
__global__ void __launch_bounds__(kUcThreads, 1)
    upconv_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                  const UcArgs args)
{
    using L = UcLayout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;   // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16;       // [2]
    const uint32_t bar_drain = bar_acc_empty + 16;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + L::kTmemSlot);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + L::kAbort);
    volatile int *consumed_sh = reinterpret_cast<volatile int *>(gbase + L::kConsumed);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // launched with programmatic serialization (tc::launch_pdl): nothing
    // global before the kernel ahead in the stream has finished
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
        *abort = (*reinterpret_cast<volatile unsigned int *>(&g_uc_status) != 0u) ? 1 : 0;
        *consumed_sh = 0;
        mbar_init_fence();
        prefetch_tensormap(&map_x);
        prefetch_tensormap(&map_w);
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

    int issued = 0;   // producer: ring steps whose loads were issued
    if (!skip && warp == 0 && lane == 0) {
        // ---- producer ----
        int q = 0;    // ring step, counted across tiles
        bool go = true;
        for (int t = blockIdx.x; go && t < args.tiles; t += gridDim.x) {
            const TileCoord tc = tile_coord<BN>(t, args);
            const int pa = tc.parity >> 1, pb = tc.parity & 1;
            const int wrow = tc.parity * args.Cout + tc.co0;
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (q >= STAGES && !tc::wait(bar_empty + 8 * s, ((q / STAGES) - 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) {
                    go = false;
                    break;
                }
                const int tap = kt / args.chunks;
                const int c0 = (kt - tap * args.chunks) * kBK;
                const int r = tap >> 1, sx = tap & 1;
                const uint32_t sa = base + s * L::kStage;
                mbar_arrive_expect_tx(bar_full + 8 * s, L::kStage);
                tma_load_4d(sa, &map_x, c0, tc.j0 + sx + pb - 1, tc.i0 + r + pa - 1, tc.n0, bar_full + 8 * s);
                tma_load_2d(sa + kABytes, &map_w, kt * kBK, wrow, bar_full + 8 * s);
                issued = q + 1;
            }
        }
    } else if (!skip && warp == 1 && lane == 0) {
        // ---- MMA issue ----
        constexpr uint32_t idesc = umma_idesc_bf16_f32(kBM, BN);
        int q = 0;
        int lt = 0;   // this CTA's tile count
        bool go = true;
        for (int t = blockIdx.x; go && t < args.tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            // the epilogue has drained this accumulator (tile lt - 2)
            if (lt >= 2 && !tc::wait(bar_acc_empty + 8 * buf, ((lt >> 1) - 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (!tc::wait(bar_full + 8 * s, (q / STAGES) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) {
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
        umma_commit(bar_drain);   // arrives once every MMA issued above has completed
    } else if (!skip && warp >= 2) {
        // ---- epilogue: two warps per tensor-memory lane quarter, each half the columns ----
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        uint4 *const stage = reinterpret_cast<uint4 *>(gbase + L::kStaging) + (warp - 2) * 128;
        int lt = 0;
        for (int t = blockIdx.x; t < args.tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            const bool done = tc::wait(bar_acc_full + 8 * buf, (lt >> 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host);
            tc_fence_after_sync();
            // warp-uniform, as the tensor-memory loads below are warp-collective
            if (!__all_sync(0xffffffffu, done && !*abort)) break;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
            upconv_epilogue<BN>(args, tile_coord<BN>(t, args), tbase, quad, half, lane, stage,
                                bar_acc_empty + 8 * buf, false);
        }
    }

    // ---- teardown: drain what is still in flight, then free tensor memory ----
    tc_fence_before_sync();
    __syncthreads();
    if (*abort && !skip) {
        if (warp == 0 && lane == 0) {
            // loads issued but never consumed still write into the ring
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
// The same convolution on CTA pairs (a cluster of two CTAs on two SMs): one
// tcgen05.mma.cta_group::2 of M = 256, N = 256 covers two pixel tiles (one
// per CTA) of the same parity and 256 output channels.  Each CTA stages its
// own A tile (16 KB per K step) and HALF of B (128 channels, 16 KB), so per
// SM the operand traffic through shared memory and L2 is two thirds of the
// single-CTA kernel's for the same MMA work.
//   full[s]       in the even CTA: expects both CTAs' bytes of ring step s
//                 (the odd CTA's copies signal it across the pair)
//   empty[s]      in both CTAs: the pair MMA's commit arrives on both
//   acc_full[b]   in both CTAs: the pair MMA's commit at the end of a tile
//   acc_empty[b]  in the even CTA: one arrival per epilogue warp of both CTAs
// ---------------------------------------------------------------------------
template <int STAGES>
struct PairLayout {
    static constexpr uint32_t kBHalf = 128u * kBK * 2;   // 16 KB
    static constexpr uint32_t kStage = kABytes + kBHalf;
    static constexpr uint32_t kRing = kStage * STAGES;
    static constexpr uint32_t kTmemCols = 512;          // two 256-column accumulators
    static constexpr uint32_t kBars = kRing;
    static constexpr uint32_t kTmemSlot = kBars + 8 * (2 * STAGES + 5);
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kConsumed = kAbort + 4;
    static constexpr uint32_t kStaging = (kConsumed + 4 + 15) & ~15u;   // 8 epilogue warps x 2 KB
    static constexpr uint32_t kBytes = kStaging + 8 * 2048;
    static constexpr uint32_t kDynamic = kBytes + 1024;
};

// Pair tile T -> this CTA's tile: the 256-channel tile varies fastest, then
// the parity, then the pixel-tile pair; CTA `rank` takes pixel tile
// 2 pp + rank (a tile past the last one lies beyond the batch: its loads
// read zeros and its stores are skipped).
__device__ __forceinline__ TileCoord pair_tile_coord(int T, int rank, const UcArgs &a)
{
    TileCoord c;
    const int co_t = T % a.co_tiles;
    T /= a.co_tiles;
    c.parity = T & 3;
    int pt = 2 * (T >> 2) + rank;
    const int tw = pt % a.tiles_w;
    pt /= a.tiles_w;
    const int th = pt % a.tiles_h;
    const int tn = pt / a.tiles_h;
    c.i0 = th * a.BH;
    c.j0 = tw * a.BW;
    c.n0 = tn * a.BNI;
    c.co0 = co_t * 256;
    return c;
}

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kUcThreads, 1)
    upconv_pair_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                       const UcArgs args)
{
    using L = PairLayout<STAGES>;
    constexpr int BN = 256;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t bar_full = base + L::kBars;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;   // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16;       // [2]
    const uint32_t bar_drain = bar_acc_empty + 16;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + L::kTmemSlot);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + L::kAbort);
    volatile int *consumed_sh = reinterpret_cast<volatile int *>(gbase + L::kConsumed);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    // launched with programmatic serialization, as upconv_kernel
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
        *abort = (*reinterpret_cast<volatile unsigned int *>(&g_uc_status) != 0u) ? 1 : 0;
        *consumed_sh = 0;
        mbar_init_fence();
        prefetch_tensormap(&map_x);
        prefetch_tensormap(&map_w);
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
        // ---- producer (both CTAs): own A tile, own half of B ----
        int q = 0;
        bool go = true;
        for (int T = pair; go && T < args.tiles; T += npairs) {
            const TileCoord tc = pair_tile_coord(T, rank, args);
            const int pa = tc.parity >> 1, pb = tc.parity & 1;
            const int wrow = tc.parity * args.Cout + tc.co0 + rank * 128;
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (q >= STAGES && !tc::wait(bar_empty + 8 * s, ((q / STAGES) - 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) {
                    go = false;
                    break;
                }
                const int tap = kt / args.chunks;
                const int c0 = (kt - tap * args.chunks) * kBK;
                const int r = tap >> 1, sx = tap & 1;
                const uint32_t sa = base + s * L::kStage;
                if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * L::kStage);
                tma_load_4d_pair(sa, &map_x, c0, tc.j0 + sx + pb - 1, tc.i0 + r + pa - 1, tc.n0, full_lead + 8 * s);
                tma_load_2d_pair(sa + kABytes, &map_w, kt * kBK, wrow, full_lead + 8 * s);
                issued = q + 1;
            }
        }
    } else if (!skip && leader && warp == 1 && lane == 0) {
        // ---- MMA issue (even CTA only) ----
        constexpr uint32_t idesc = umma_idesc_bf16_f32(2 * kBM, BN);
        int q = 0;
        int lt = 0;
        bool go = true;
        for (int T = pair; go && T < args.tiles; T += npairs, ++lt) {
            const int buf = lt & 1;
            if (lt >= 2 && !tc::wait(bar_acc_empty + 8 * buf, ((lt >> 1) - 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
            for (int kt = 0; kt < args.ksteps; ++kt, ++q) {
                const int s = q % STAGES;
                if (!tc::wait(bar_full + 8 * s, (q / STAGES) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host)) {
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
        // ---- epilogue (both CTAs): own pixels, 256 channels, two warps per lane quarter ----
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        uint4 *const stage = reinterpret_cast<uint4 *>(gbase + L::kStaging) + (warp - 2) * 128;
        int lt = 0;
        for (int T = pair; T < args.tiles; T += npairs, ++lt) {
            const int buf = lt & 1;
            const bool done = tc::wait(bar_acc_full + 8 * buf, (lt >> 1) & 1, abort, args.timeout_ns, &g_uc_status, g_uc_status_host);
            tc_fence_after_sync();
            if (!__all_sync(0xffffffffu, done && !*abort)) break;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
            upconv_epilogue<BN>(args, pair_tile_coord(T, rank, args), tbase, quad, half, lane, stage,
                                acc_empty_lead + 8 * buf, true);
        }
    }

    // ---- teardown ----
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


template <int BN, int STAGES>
cudaError_t launch_variant(const CUtensorMap &mx, const CUtensorMap &mw, const UcArgs &a, int blocks,
                           cudaStream_t s)
{
    using L = UcLayout<BN, STAGES>;
    static_assert(L::kDynamic <= 227 * 1024, "upconv ring does not fit in shared memory");
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(upconv_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::kDynamic));
    });
    if (attr != cudaSuccess) return attr;
    const cudaError_t e = tc::launch_pdl(upconv_kernel<BN, STAGES>, dim3(blocks), dim3(kUcThreads), L::kDynamic, s,
                                         mx, mw, a);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

template <int STAGES>
cudaError_t launch_pair(const CUtensorMap &mx, const CUtensorMap &mw, const UcArgs &a, int sm_count, cudaStream_t s)
{
    using L = PairLayout<STAGES>;
    static_assert(L::kDynamic <= 227 * 1024, "upconv pair ring does not fit in shared memory");
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    static int max_clusters = 0;
    std::call_once(once, [sm_count] {
        attr = cudaFuncSetAttribute(upconv_pair_kernel<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::kDynamic));
        if (attr != cudaSuccess) return;
        max_clusters = tc::pair_clusters(upconv_pair_kernel<STAGES>, kUcThreads, L::kDynamic, sm_count);
    });
    if (attr != cudaSuccess) return attr;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int pairs = a.tiles < max_clusters ? a.tiles : max_clusters;
    const cudaError_t e = tc::launch_pdl(upconv_pair_kernel<STAGES>, dim3(2 * pairs), dim3(kUcThreads), L::kDynamic, s,
                                         mx, mw, a);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

bool pair_kernel_enabled()
{
    static const bool on = [] {
        const char *v = std::getenv("GN_UPCONV_PAIR");
        return !(v && v[0] == '0');
    }();
    return on;
}

}  // namespace

bool upconv_tiling(int64_t N, int64_t H, int64_t W, UpconvTiling *t)
{
    if (N < 1 || H < 1 || W < 1) return false;
    const auto pow2 = [](int64_t v) { return v > 0 && (v & (v - 1)) == 0; };
    UpconvTiling r{};
    if (W >= kBM) {
        if (W % kBM != 0) return false;
        r.BW = kBM;
        r.BH = 1;
        r.BNI = 1;
    } else {
        if (!pow2(W)) return false;
        r.BW = static_cast<int>(W);
        const int64_t rows = kBM / W;
        if (H >= rows) {
            if (H % rows != 0) return false;
            r.BH = static_cast<int>(rows);
            r.BNI = 1;
        } else {
            if (!pow2(H)) return false;
            r.BH = static_cast<int>(H);
            r.BNI = static_cast<int>(kBM / (W * H));
        }
    }
    r.tiles_w = static_cast<int>(W / r.BW);
    r.tiles_h = static_cast<int>(H / r.BH);
    r.tiles_n = static_cast<int>((N + r.BNI - 1) / r.BNI);
    *t = r;
    return true;
}

cudaError_t launch_upconv_fold(const void *w, void *wf, int Cin, int Cout, int sm_count, cudaStream_t s)
{
    const int64_t total = 16LL * Cout * Cin;
    const int64_t want = (total + 255) / 256;
    const int blocks = static_cast<int>(want < 4LL * sm_count ? want : 4LL * sm_count);
    upconv_fold_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w),
                                              static_cast<__nv_bfloat16 *>(wf), Cin, Cout);
    return cudaGetLastError();
}

int launch_upconv(const void *x, const void *wf, const void *bias, void *y, int N, int H, int W, int Cin,
                  int Cout, int sm_count, uint64_t timeout_ns, cudaStream_t s, cudaError_t *err)
{
    *err = cudaSuccess;
    UpconvTiling t;
    if (!upconv_tiling(N, H, W, &t)) return 1;
    tc::EncodeTiledFn enc = tc::encode_fn();
    if (!enc) return 2;
    const int BN = (Cout % 256 == 0) ? 256 : 128;
    const bool use_pair = BN == 256 && pair_kernel_enabled();

    CUtensorMap mx, mw;
    {
        // x as a 4-D tensor {Cin, W, H, N} (innermost first), boxes of
        // {64 channels, BW, BH, BNI} pixels, 128-byte swizzle, zero fill
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Cin), static_cast<cuuint64_t>(W),
                                    static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(Cin) * 2, static_cast<cuuint64_t>(W) * Cin * 2,
                                       static_cast<cuuint64_t>(H) * W * Cin * 2};
        const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(t.BW),
                                   static_cast<cuuint32_t>(t.BH), static_cast<cuuint32_t>(t.BNI)};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 2;
    }
    {
        // folded weights as a 2-D tensor {4 Cin, 4 Cout}, boxes of {64, BN}
        // channels (a CTA pair: 128 channels, the half of B one CTA stages)
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(4) * Cin, static_cast<cuuint64_t>(4) * Cout};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(4) * Cin * 2};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(use_pair ? 128 : BN)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(wf), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 2;
    }
    UcArgs a;
    a.N = N;
    a.H = H;
    a.W = W;
    a.Cin = Cin;
    a.Cout = Cout;
    a.BW = t.BW;
    a.BH = t.BH;
    a.BNI = t.BNI;
    a.tiles_w = t.tiles_w;
    a.tiles_h = t.tiles_h;
    a.co_tiles = Cout / BN;
    a.chunks = Cin / kBK;
    a.ksteps = 4 * a.chunks;
    a.bias = static_cast<const __nv_bfloat16 *>(bias);
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.timeout_ns = timeout_ns;
    const int64_t pixel_tiles = static_cast<int64_t>(t.tiles_n) * t.tiles_h * t.tiles_w;
    const int64_t tiles = (use_pair ? (pixel_tiles + 1) / 2 : pixel_tiles) * 4 * a.co_tiles;
    if (tiles > 0x7fffffffLL) return 1;
    a.tiles = static_cast<int>(tiles);
    if (use_pair) {
        *err = launch_pair<6>(mx, mw, a, sm_count, s);
        return *err == cudaSuccess ? 0 : 3;
    }
    // persistent: one CTA per SM (each holds all 512 tensor-memory columns or half of them)
    const int blocks = static_cast<int>(tiles < sm_count ? tiles : sm_count);
    *err = (BN == 256) ? launch_variant<256, 4>(mx, mw, a, blocks, s)
                       : launch_variant<128, 6>(mx, mw, a, blocks, s);
    return *err == cudaSuccess ? 0 : 3;
}

cudaError_t read_upconv_status(unsigned int *status)
{
    return cudaMemcpyFromSymbol(status, g_uc_status, sizeof(unsigned int));
}

cudaError_t clear_upconv_status()
{
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_uc_status, &zero, sizeof(unsigned int));
}

cudaError_t set_upconv_status_host(unsigned int *host_word)
{
    return cudaMemcpyToSymbol(g_uc_status_host, &host_word, sizeof(host_word));
}

}  // namespace gn
