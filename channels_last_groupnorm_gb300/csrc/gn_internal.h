// gn_internal.h -- geometry and launch interface shared by the kernels
// (gn_kernels.cu) and the C ABI layer (gn_capi.cu).  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gn {

constexpr int kConsumers = 256;                 // consumer threads per CTA (8 warps)
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 32;       // + one producer warp
constexpr int kMaxRing = 32;                    // ring slots (one bit each in a 32-bit mask)
constexpr int kMaxPieceBytes = 32768;
constexpr int kMaxVecPerThread = kMaxPieceBytes / 16 / kConsumers;   // 16-byte vectors per thread per piece
constexpr int kMinPieceBytes = 1024;
constexpr int kMaxSegments = 512;               // segments per batch entry
constexpr int kFusedMaxSegments = 160;          // ... in the fused kernel (5 records per lane)
constexpr int kScratchBytes = 16384;            // pass-1 CTA reduction scratch
constexpr int kStatRecords = 20;               // fused kernel: item records per lane in the per-CTA merge
constexpr int kOneBarrierRecords = 8192;        // fused kernel: every CTA merges all G*S item records
                                                // of its batch entry itself when there are at most this many
constexpr int kSyncWords = 64;                  // 256-byte workspace header

// The (N, L, C) tensor is cut into pieces of whole rows (one bulk copy
// each); the pieces of one batch entry are dealt out round-robin to S work
// items, a work item being one (n, s) pair: item s owns pieces s, s + S, ...
struct Geom {
    int64_t N, L;
    int32_t C, G, Cg, V;          // V = C / 8 sixteen-byte vectors per row
    int32_t A;                    // consumer threads that carry data: (kConsumers / V) * V
    int32_t rows_per_piece;
    int32_t piece_bytes;          // rows_per_piece * C * 2
    int64_t pieces_per_n;
    int32_t S;                    // segments per batch entry
    int32_t ring;                 // ring slots in shared memory
    int64_t items;                // N * S
    int32_t seg32;                // pieces_per_n < 2^32: piece counts in 32-bit math
    // pieces of item s: base_pieces + (s <= last_item); item last_item owns
    // the batch entry's last piece, which holds tail_rows rows
    int64_t base_pieces;          // (pieces_per_n - 1) / S
    int32_t last_item;            // (pieces_per_n - 1) % S
    int32_t tail_rows;            // L - (pieces_per_n - 1) * rows_per_piece
    float inv_L, inv_LCg;         // 1 / L and 1 / (L * Cg), rounded to fp32
    int32_t Cg_pow2, log2_Cg;     // Cg is a power of two: Cg = 1 << log2_Cg
    int32_t stat_lanes;           // fused kernel: lanes per group in the per-CTA merge (power of two <= 32)
    int32_t stat_log2, stat_passes;   // log2(stat_lanes); passes over the groups
    float rows_lo, rows_hi, rows_short;   // item rows (base_pieces, base_pieces + 1 pieces) and the
                                          // short last piece's missing rows, as floats
    // fused kernel, one batch entry and one item per CTA: pass 2 deals the
    // pieces not resident in a ring out at run time (gn_kernels.cu,
    // produce_pass2_dyn); dyn_top is the highest row of the item sequences
    // that holds such a piece (base_pieces - ring; negative: none)
    int32_t dyn_p2;
    int64_t dyn_top;
};

struct Args {
    const uint16_t *x;            // bf16 [N][L][C]
    uint16_t *y;                  // bf16 [N][L][C]
    const float *gamma, *beta;    // [C]
    float eps;
    uint32_t l2_hints;            // bit 0: pass-2 loads evict_first, bit 1: pass-2
                                  // stores evict_first, bit 2: pass-1 loads evict_last
    Geom g;
    float2 *partial;              // [N][G][S] group record per item (mean, M2); its rows
                                  // follow from the geometry (item_rows_f)
    float2 *gstat;                // [N][G]    group (mean, rstd)   (fused)
    float2 *st;                   // [N][C]    (scale, shift)       (two-pass)
    float *mean, *rstd;           // [N][G]
    unsigned int *sync;           // fused: [0] grid-barrier arrivals, [1] re-arm count, [2] pass-2
                                  // piece counter, [3] exits (the last CTA zeroes [2] and [3])
    uint64_t timeout_ns;          // bound on every wait
};

// Byte offsets inside a CTA's dynamic shared memory.  `gstat` (per-group
// mean / rstd of the fused kernel) shares the pass-1 scratch; `chs` (the
// per-channel (mean, M2) of one work item) shares `st` in the fused kernel.
struct Layout {
    uint32_t ring, scratch, kvec, chs, st, gb, gstat, bars, flags, tags, total;
};

enum Kind { kPass1 = 1, kPass2 = 2, kFused = 3 };

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(const Geom &g, int kind)
{
    Layout s;
    uint32_t off = static_cast<uint32_t>(g.ring) * static_cast<uint32_t>(g.piece_bytes);
    s.ring = 0;
    s.scratch = off;
    s.gstat = off;
    if (kind != kPass2) off += kScratchBytes;
    s.kvec = off;
    if (kind != kPass2) off += align_up(4u * g.C, 16);
    s.chs = off;
    if (kind == kPass1) off += 8u * g.C;
    s.st = off;
    if (kind == kFused) {
        s.chs = off;
        off += 8u * g.C;
    }
    s.gb = off;
    if (kind == kFused) off += 8u * g.C;
    s.bars = align_up(off, 16);
    off = s.bars + 16u * g.ring;
    s.flags = off;
    off += 16;
    s.tags = off;   // fused kernel: the piece each ring slot holds in a dynamic pass 2
    if (kind == kFused) off += 4u * kMaxRing;
    s.total = off;
    return s;
}

// Dynamic shared memory besides the ring, for a given kind.
inline uint32_t aux_smem_bytes(const Geom &g, int kind)
{
    Geom t = g;
    t.ring = 0;
    return make_layout(t, kind).total + 16u * kMaxRing;
}

constexpr int kRgaThreads = 256;   // threads per block of the residual-gate kernel

// Residual-gate update y = residual + gate * update (rga_kernels.cu):
// rows x D half-precision elements (D a multiple of 8), bf16 or fp16.
cudaError_t launch_residual_gate(const void *residual, const void *update, const void *gate, void *out,
                                 int64_t rows, int64_t D, bool bf16, int blocks, cudaStream_t s);

// Host-side launchers (gn_kernels.cu).  They return the first CUDA error.
cudaError_t launch_pass1(const Args &a, int grid, cudaStream_t s);
cudaError_t launch_finalize(const Args &a, cudaStream_t s);
cudaError_t launch_pass2(const Args &a, int grid, bool silu, cudaStream_t s);
cudaError_t launch_fused(const Args &a, int grid, bool silu, cudaStream_t s);
// Maximum co-resident CTAs per SM of the fused kernel with `smem` bytes.
cudaError_t fused_blocks_per_sm(bool silu, uint32_t smem, int *blocks);
cudaError_t prepare_kernels(uint32_t max_smem);
cudaError_t launch_selftest_wait(int mode, uint64_t timeout_ns, int *done, int blocks, cudaStream_t s);
// ---- cluster schedule for tensors that fit in shared memory (gn_cluster.cu) ----
constexpr int kClusterMaxCtas = 16;   // largest cluster the schedule uses (non-portable above 8)
struct ClusterPlan {
    int SC;            // channels per slice: whole groups, a multiple of 8
    int CL;            // CTAs per cluster
    int R;             // rows per CTA
    int BR;            // rows per tensor-map box (a multiple of 8, at most 256)
    int boxes;         // boxes per CTA
    int64_t units;     // clusters: (batch entry, slice) pairs
    int waves;         // rounds of clusters the device runs one after another
    uint32_t smem;     // dynamic shared memory per CTA
    int tma;           // rows copied by tensor-map boxes (else 16-byte copies by every thread)
};
// Kernel attributes, and the co-resident clusters of each size 1..16
// (cap[size]) at `max_smem` bytes of shared memory per CTA.
cudaError_t prepare_cluster_kernels(int max_smem, int (&cap)[kClusterMaxCtas + 1]);
// False when no cluster layout fits the shape.
bool plan_cluster(int64_t N, int64_t L, int C, int G, const int (&cap)[kClusterMaxCtas + 1], int max_smem,
                  ClusterPlan *out);
cudaError_t launch_cluster(const ClusterPlan &p, const uint16_t *x, uint16_t *y, const float *gamma,
                           const float *beta, float *mean, float *rstd, float eps, bool silu, int64_t N, int64_t L,
                           int C, int G, uint64_t timeout_ns, unsigned int *status, unsigned int *status_host,
                           cudaStream_t s);

cudaError_t read_device_status(unsigned int *status);
// Device address of the GroupNorm kernels' sticky status word (current device).
cudaError_t device_status_address(unsigned int **word);
cudaError_t clear_device_status();
// Device address of the mapped host word that mirrors the status (current device).
cudaError_t set_device_status_host(unsigned int *host_word);

}  // namespace gn
