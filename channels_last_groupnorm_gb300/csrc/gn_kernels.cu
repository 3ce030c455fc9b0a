// gn_kernels.cu -- sm_103a kernels for channels-last GroupNorm (+SiLU).
//
// The computation follows the two-pass structure of sglang PR #33451
// ("FLUX.2 VAE decoder fast path behind quality=high", section
// "Modifications", item 1): a pass-1 per-(batch, channel) partial reduction
// over (N, L, C) rows, a finalize step producing per-(batch, group) mean /
// rstd with the affine folded into per-(batch, channel) scale / shift, and a
// pass-2 elementwise apply with optional SiLU.
//
// GB300 design:
//  * The tensor is cut into "pieces" of whole rows (up to 32 KB); each CTA
//    streams its pieces through a ring of shared-memory slots filled by bulk
//    TMA copies (cp.async.bulk) issued by one producer thread, completion
//    tracked on mbarriers.  Eight consumer warps read 16-byte vectors from
//    shared memory; each consumer thread always sees the same eight
//    channels, and a full piece is a fixed number of vectors per thread, so
//    the piece loops are compiled per vector count.  Channel pairs use the
//    packed fp32x2 instructions of sm_100+ (add/sub/mul/fma .f32x2).
//  * Pass 1 keeps, per thread, fp32 sums of (x - K) and (x - K)^2, K being
//    the channel's group's first value in the work item's first row (one
//    shift per group, so sums of a group's channels add directly), then
//    reduces them per CTA (warp butterflies and shared memory) into one
//    (mean, M2) record per (batch entry, group, item).  The finalize merges
//    the records of each group (Chan's parallel formula, around a shift).
//  * Pass 2 loads pieces the same way, in the reverse of pass-1 order so the
//    most recently read rows (still in L2) come first; each consumer thread
//    computes and stores its outputs (coalesced 16-byte global stores) and
//    then releases the slot.
//  * The fused kernel does all three steps in one cooperative launch: after
//    one grid barrier every CTA merges the G*S records of its batch entry
//    itself (a second barrier is used only when there are very many
//    groups); pieces still in the ring after pass 1 are not re-read.
//  * Every wait (mbarrier phase, grid barrier) is bounded by a deadline on
//    the global timer, counted from the start of that wait; on expiry the
//    kernel records a sticky status, stops issuing work, drains its own
//    copies and returns.
#include <cuda_bf16.h>

#include "gn_internal.h"
#include "gn_math.cuh"
#include "gn_ptx.cuh"

namespace gn {

// Sticky device-side status: bit 0 = a bounded wait expired.
__device__ unsigned int g_status;
// Its host-visible copy (mapped page-locked host memory; null until set).
__device__ unsigned int *g_status_host;

// ---------------------------------------------------------------------------
// work-item cursor.  Work item (n, s) owns the pieces k = s, s + S, s + 2S, ...
// of batch entry n: interleaving spreads every CTA's reads over the whole
// address range, so no CTA is stuck with a slower stretch of memory.
// ---------------------------------------------------------------------------
struct Cursor {
    int64_t it;        // work item id (n * S + s)
    int64_t n;
    int32_t s;
    int64_t k_last;    // last piece of the item
    int64_t k;         // current piece
};

// pieces of item s in one batch entry (S <= pieces_per_n, so at least one)
__device__ __forceinline__ int64_t item_pieces(const Geom &g, int32_t s)
{
    return g.base_pieces + (s <= g.last_item ? 1 : 0);
}

// rows of item s (as a float, for the statistics)
__device__ __forceinline__ float item_rows_f(const Geom &g, int32_t s)
{
    const float rows = s <= g.last_item ? g.rows_hi : g.rows_lo;
    return s == g.last_item ? rows - g.rows_short : rows;
}

__device__ __forceinline__ void load_item(const Geom &g, Cursor &c, int64_t it)
{
    c.it = it;
    c.n = it / g.S;
    c.s = static_cast<int32_t>(it - c.n * g.S);
    c.k_last = c.s + (item_pieces(g, c.s) - 1) * g.S;
}


__device__ __forceinline__ int32_t piece_rows(const Geom &g, int64_t k)
{
    return static_cast<int32_t>(min(static_cast<int64_t>(g.rows_per_piece), g.L - k * g.rows_per_piece));
}

__device__ __forceinline__ int64_t piece_elem_offset(const Geom &g, int64_t n, int64_t k)
{
    return (n * g.L + k * g.rows_per_piece) * g.C;
}

// One work item as the consumers see it: batch entry n, segment s, its
// piece count, and whether it owns the batch entry's short last piece.
struct Item {
    int64_t n;
    int32_t s;
    int64_t np;
    bool tail;
};

__device__ __forceinline__ Item make_item(const Geom &g, int64_t it)
{
    Item m;
    m.n = (g.items < (int64_t(1) << 31)) ? static_cast<int64_t>(static_cast<uint32_t>(it) / static_cast<uint32_t>(g.S))
                                          : it / g.S;
    m.s = static_cast<int32_t>(it - m.n * g.S);
    m.np = item_pieces(g, m.s);
    m.tail = (m.s + (m.np - 1) * g.S) == g.pieces_per_n - 1;
    return m;
}

// rows covered by an item: whole pieces, less the short tail of the last
// piece of the batch entry if the item owns it
__device__ __forceinline__ int64_t rows_of(const Geom &g, const Item &m)
{
    const int64_t rows = m.np * g.rows_per_piece;
    return m.tail ? rows - (g.pieces_per_n * g.rows_per_piece - g.L) : rows;
}

// pieces this CTA processes, over all its items
__device__ __forceinline__ int64_t cta_piece_count(const Geom &g)
{
    if (g.items <= gridDim.x)   // one item per CTA (grids are never wider than the items)
        return item_pieces(g, static_cast<int32_t>(blockIdx.x % static_cast<uint32_t>(g.S)));
    int64_t t = 0;
    for (int64_t it = blockIdx.x; it < g.items; it += gridDim.x)
        t += item_pieces(g, static_cast<int32_t>(it % g.S));
    return t;
}

__device__ __forceinline__ void cursor_first(const Geom &g, Cursor &c)
{
    load_item(g, c, blockIdx.x);
    c.k = c.s;
}

// returns false when the CTA has no further piece
__device__ __forceinline__ bool cursor_next(const Geom &g, Cursor &c)
{
    if (c.k < c.k_last) {
        c.k += g.S;
        return true;
    }
    const int64_t it = c.it + gridDim.x;
    if (it >= g.items) return false;
    load_item(g, c, it);
    c.k = c.s;
    return true;
}

__device__ __forceinline__ void cursor_last(const Geom &g, Cursor &c)
{
    const int64_t last = blockIdx.x + ((g.items - 1 - blockIdx.x) / gridDim.x) * gridDim.x;
    load_item(g, c, last);
    c.k = c.k_last;
}

__device__ __forceinline__ bool cursor_prev(const Geom &g, Cursor &c)
{
    if (c.k > c.s) {
        c.k -= g.S;
        return true;
    }
    const int64_t it = c.it - gridDim.x;
    if (it < 0) return false;
    load_item(g, c, it);
    c.k = c.k_last;
    return true;
}

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
struct Ctl {
    volatile int *abort;   // CTA-wide: a wait expired or the status was set
    uint64_t timeout_ns;   // bound on each single wait
};

__device__ __forceinline__ void record_timeout(const Ctl &ctl)
{
    *ctl.abort = 1;
    atomicOr(&g_status, 1u);
    raise_host_status(g_status_host);
}

// Waiting threads sleep in the try_wait (up to kWaitSleepNs per round)
// rather than spin, so that warps still busy with the previous piece keep
// the issue slots.
constexpr uint32_t kWaitSleepNs = 20000;

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl &ctl)
{
    // a completed phase is safe to consume even after an abort elsewhere in
    // the CTA; the abort is noticed on the first wait that does not complete
    if (mbar_try_wait(bar, parity)) return true;
    if (*ctl.abort) return false;
    const uint64_t deadline = global_ns() + ctl.timeout_ns;
#pragma unroll 1
    for (;;) {
        if (mbar_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (*ctl.abort) return false;
        if (global_ns() > deadline) {
            record_timeout(ctl);
            return false;
        }
    }
}

// Grid-wide barrier for the cooperative fused kernel: one release-arrival
// per CTA on a gpu-scope counter, then a bounded acquire-spin until `target`
// arrivals.  The CTA barrier before the arrival orders every thread's
// earlier global writes before it.
__device__ __forceinline__ bool grid_sync(unsigned int *counter, unsigned int target, const Ctl &ctl)
{
    __syncthreads();
    if (threadIdx.x == 0 && !*ctl.abort) {
        atom_add_release_gpu(counter, 1u);
        uint64_t deadline = 0;
#pragma unroll 1
        for (uint32_t it = 0;; ++it) {
            if (ld_acquire_gpu(counter) >= target) break;
            if ((it & 63u) == 63u) {
                const uint64_t now = global_ns();
                if (deadline == 0) {
                    deadline = now + ctl.timeout_ns;
                } else if (now > deadline) {
                    record_timeout(ctl);
                    break;
                }
            }
        }
    }
    __syncthreads();
    return !*ctl.abort;
}

// ---------------------------------------------------------------------------
// shared memory view of one CTA
// ---------------------------------------------------------------------------
struct Smem {
    uint8_t *base;
    Layout lay;
    uint32_t ring_s;                       // shared address of the ring
    uint32_t bars_s;                       // shared address of the mbarriers
    __device__ uint32_t full(int slot) const { return bars_s + 16u * slot; }
    __device__ uint32_t empty(int slot) const { return bars_s + 16u * slot + 8u; }
    __device__ uint32_t slot_addr(int slot, int piece_bytes) const
    {
        return ring_s + static_cast<uint32_t>(slot) * static_cast<uint32_t>(piece_bytes);
    }
};

__device__ __forceinline__ int slot_of(int64_t q, int ring)
{
    return (q < (int64_t(1) << 31)) ? static_cast<int>(static_cast<uint32_t>(q) % static_cast<uint32_t>(ring))
                                    : static_cast<int>(q % ring);
}

// ---------------------------------------------------------------------------
// producer (one thread): pass-1 loads
// ---------------------------------------------------------------------------
struct ProducerState {
    uint32_t empty_par;     // parity of the next empty-barrier phase to wait, per slot
    uint32_t issued_par;    // parity of loads issued, per slot
    uint32_t loaded;        // slots that ever received a load
};

__device__ __forceinline__ void issue_load(const Args &a, const Smem &sm, const Cursor &c, int slot,
                                           ProducerState &ps, uint64_t pol, bool hint)
{
    const Geom &g = a.g;
    const uint32_t bytes = static_cast<uint32_t>(piece_rows(g, c.k)) * static_cast<uint32_t>(g.C) * 2u;
    const uint16_t *src = a.x + piece_elem_offset(g, c.n, c.k);
    mbar_arrive_expect_tx(sm.full(slot), bytes);
    if (hint)
        bulk_load_hint(sm.slot_addr(slot, g.piece_bytes), src, bytes, sm.full(slot), pol);
    else
        bulk_load(sm.slot_addr(slot, g.piece_bytes), src, bytes, sm.full(slot));
    ps.issued_par ^= 1u << slot;
    ps.loaded |= 1u << slot;
}

// `absorb_tail`: afterwards also wait for the consumption of the last pieces
// (those no later load waited for), so that in the fused kernel the empty
// barriers are in step before pass 2 starts consuming the same slots again.
__device__ void produce_pass1(const Args &a, const Smem &sm, int64_t T, ProducerState &ps, const Ctl &ctl,
                              bool absorb_tail)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const bool hint = (a.l2_hints & 4u) != 0;
    const uint64_t pol = hint ? policy_evict_last() : 0;
    Cursor c;
    cursor_first(g, c);
    int slot = 0;
    for (int64_t q = 0; q < T; ++q) {
        if (q >= g.ring) {
            if (!wait_phase(sm.empty(slot), (ps.empty_par >> slot) & 1u, ctl)) return;
            ps.empty_par ^= 1u << slot;
        }
        issue_load(a, sm, c, slot, ps, pol, hint);
        cursor_next(g, c);
        slot = (slot + 1 == g.ring) ? 0 : slot + 1;
    }
    if (!absorb_tail) return;
    const int64_t tail = min(T, static_cast<int64_t>(g.ring));
    slot = slot_of(T - tail, g.ring);
    for (int64_t q = T - tail; q < T; ++q) {
        if (!wait_phase(sm.empty(slot), (ps.empty_par >> slot) & 1u, ctl)) return;
        ps.empty_par ^= 1u << slot;
        slot = (slot + 1 == g.ring) ? 0 : slot + 1;
    }
}

// ---------------------------------------------------------------------------
// producer (one thread): pass-2 loads, pieces in reverse order.  `resident`
// pieces (the last ones of pass 1, fused kernel only) are still in their
// ring slots and are not loaded again.  A slot is refilled as soon as the
// consumers have read it (they write y straight to global memory).
// ---------------------------------------------------------------------------
__device__ void produce_pass2(const Args &a, const Smem &sm, int64_t T, int64_t resident,
                              ProducerState &ps, const Ctl &ctl)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const bool hint = (a.l2_hints & 1u) != 0;
    const uint64_t pol = hint ? policy_evict_first() : 0;
    Cursor ld;
    cursor_last(g, ld);
    int slot = slot_of(T - 1, g.ring);
    for (int64_t q = T - 1; q >= 0; --q) {
        if (q < T - resident) {
            if (q + g.ring < T) {
                // the slot still holds piece q + ring, processed earlier
                if (!wait_phase(sm.empty(slot), (ps.empty_par >> slot) & 1u, ctl)) return;
                ps.empty_par ^= 1u << slot;
            }
            issue_load(a, sm, ld, slot, ps, pol, hint);
        }
        cursor_prev(g, ld);
        slot = (slot == 0) ? g.ring - 1 : slot - 1;
    }
}

// After an abort, let every load this producer issued land before the CTA
// exits.  Bounded by its own two-second deadline, independent of the
// (possibly shortened) wait timeout, so in-flight copies always get time to
// complete.
__device__ void drain_loads(const Smem &sm, const ProducerState &ps, int ring)
{
    const uint64_t deadline = global_ns() + 2000000000ull;
    for (int slot = 0; slot < ring; ++slot) {
        if (!((ps.loaded >> slot) & 1u)) continue;
        const uint32_t par = ((ps.issued_par >> slot) & 1u) ^ 1u;   // phase of the last load
#pragma unroll 1
        for (uint32_t it = 0;; ++it) {
            if (mbar_try_wait(sm.full(slot), par)) break;
            if ((it & 31u) == 31u && global_ns() > deadline) break;
        }
    }
}

// ---------------------------------------------------------------------------
// dynamic pass 2 (fused kernel, one batch entry, one item per CTA).  A CTA
// first applies the pieces still in its ring; the others are dealt out at
// run time: the producers take kDynBatch entries at a time from a
// grid-wide counter over (row i of the item sequences from dyn_top down,
// item s from the last down) -- the reverse of the order pass 1 read them
// in, so the first ones are still in L2 -- skipping resident pieces.  SMs
// that stream faster apply more pieces (the per-SM rates on a GB300 differ
// by up to 1.5x between SMs, the same SMs slow from call to call).  The
// producer hands each piece's index to the consumers in a word per ring
// slot; -1 ends the pass.
// ---------------------------------------------------------------------------
// one entry per counter update (measured against 2 and 4 at 256-512 MiB:
// 0.4-0.9 % faster; the ring hides the update's round trip to L2)
constexpr uint32_t kDynBatch = 1;

// Piece of counter entry q: -1 past the last one, -2 for an entry with no
// piece to load (item s has no row i, or the piece is resident in its
// owner's ring: the last min(pieces, ring) of the item).
__device__ __forceinline__ int64_t dyn_piece(const Geom &g, uint32_t q)
{
    const uint32_t S = static_cast<uint32_t>(g.S);
    const int64_t i = g.dyn_top - static_cast<int64_t>(q / S);
    if (i < 0) return -1;
    const int32_t s = g.S - 1 - static_cast<int32_t>(q % S);
    const int64_t np = item_pieces(g, s);
    if (i >= np - min(np, static_cast<int64_t>(g.ring))) return -2;
    return s + i * g.S;
}

// The ring position j of pass 2 uses slot (T - 1 - j) mod ring: positions
// 0 .. resident - 1 are the CTA's last pass-1 pieces, still in place.
__device__ __forceinline__ int dyn_slot(int64_t T, int64_t j, int ring)
{
    const int64_t r = (T - 1 - j) % ring;
    return static_cast<int>(r < 0 ? r + ring : r);
}

__device__ void produce_pass2_dyn(const Args &a, const Smem &sm, int64_t T, int64_t resident,
                                  ProducerState &ps, const Ctl &ctl)
{
    const Geom &g = a.g;
    const bool hint = (a.l2_hints & 1u) != 0;
    const uint64_t pol = hint ? policy_evict_first() : 0;
    volatile int32_t *tags = reinterpret_cast<volatile int32_t *>(sm.base + sm.lay.tags);
    uint32_t q = 0, q_end = 0;   // the batch of counter entries in hand
    for (int64_t j = resident;; ++j) {
        int64_t k;
        do {
            if (q == q_end) {
                q = atomicAdd(a.sync + 2, kDynBatch);
                q_end = q + kDynBatch;
            }
            k = dyn_piece(g, q++);
        } while (k == -2);
        const int slot = dyn_slot(T, j, g.ring);
        if (j >= g.ring) {
            // the slot holds position j - ring of this pass
            if (!wait_phase(sm.empty(slot), (ps.empty_par >> slot) & 1u, ctl)) return;
            ps.empty_par ^= 1u << slot;
        }
        if (k < 0) {
            tags[slot] = -1;
            mbar_arrive(sm.full(slot));   // a phase without bytes: the end of the pass
            ps.issued_par ^= 1u << slot;
            return;
        }
        tags[slot] = static_cast<int32_t>(k);
        Cursor c;
        c.n = 0;
        c.k = k;
        issue_load(a, sm, c, slot, ps, pol, hint);
    }
}

// ---------------------------------------------------------------------------
// consumers: pass 1
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Vector-slot bookkeeping.  A thread's 16-byte vector v of a piece holds
// channels 8 * (v % V) .. + 7.  POW2: C is a power of two, so V divides the
// kConsumers threads and every one carries data (A = kConsumers) and the
// slot arithmetic is a mask and a shift.  Otherwise A = (kConsumers / V) * V threads
// carry data and the slot arithmetic divides.
template <bool POW2>
__device__ __forceinline__ int carriers(const Geom &g) { return POW2 ? kConsumers : g.A; }

template <bool POW2>
__device__ __forceinline__ int vec_slot(const Geom &g, int t) { return POW2 ? (t & (g.V - 1)) : (t % g.V); }

template <bool POW2>
__device__ __forceinline__ int vec_rank(const Geom &g, int t) { return POW2 ? (t >> (__ffs(g.V) - 1)) : (t / g.V); }

// Scratch layout of the CTA reduction: float4 [quad q = 0..3][entry][slot]
// (q = 0, 1: sums of x - K of channels 8*slot + 0..3, + 4..7; q = 2, 3: the
// sums of squares), so that consecutive threads (consecutive slots) touch
// consecutive 16-byte words: no bank conflicts, four stores per thread.
__device__ __forceinline__ float4 *scr_at(float4 *scr, int cap, const Geom &g, int q, int entry, int vs)
{
    return scr + ((q * cap + entry) * g.V + vs);
}

__device__ __forceinline__ void store_entry(float4 *scr, int cap, const Geom &g, int entry, int vs,
                                            const float (&v1)[8], const float (&v2)[8])
{
    *scr_at(scr, cap, g, 0, entry, vs) = make_float4(v1[0], v1[1], v1[2], v1[3]);
    *scr_at(scr, cap, g, 1, entry, vs) = make_float4(v1[4], v1[5], v1[6], v1[7]);
    *scr_at(scr, cap, g, 2, entry, vs) = make_float4(v2[0], v2[1], v2[2], v2[3]);
    *scr_at(scr, cap, g, 3, entry, vs) = make_float4(v2[4], v2[5], v2[6], v2[7]);
}

__device__ __forceinline__ float comp(const float4 &v, int j)
{
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// Any C (the path of C that are not powers of two): reduce the per-thread
// shifted sums of one work item into the item's per-group (mean, M2)
// records.  Threads that share a vector slot
// first combine by warp shuffles (when the slot repeats inside a warp), then
// through shared memory; when the scratch cannot hold every entry at once,
// the upper half of the entries is first added into the lower half.  The
// per-channel results are then merged into one record per group.
template <bool POW2>
__device__ void reduce_item_general(const Args &a, const Smem &sm, const Item &m, const f2_t (&s1p)[4],
                                    const f2_t (&s2p)[4])
{
    const Geom &g = a.g;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    float v1[8], v2[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        upk(s1p[i], v1[2 * i], v1[2 * i + 1]);
        upk(s2p[i], v2[2 * i], v2[2 * i + 1]);
    }
    const int vs_own = vec_slot<POW2>(g, tid);
    int entries, entry;
    bool holder;   // this thread holds one entry of its slot
    if (g.V < 32 && (32 % g.V) == 0) {
        for (int off = g.V; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v1[j] += __shfl_xor_sync(0xffffffffu, v1[j], off);
                v2[j] += __shfl_xor_sync(0xffffffffu, v2[j], off);
            }
        }
        entries = kConsumerWarps;
        entry = warp;
        holder = lane < g.V;
    } else {
        // slots repeat across warps (or irregularly inside them): one entry
        // per data-carrying thread
        entries = vec_rank<POW2>(g, carriers<POW2>(g));
        entry = vec_rank<POW2>(g, tid);
        holder = tid < carriers<POW2>(g);
    }
    float4 *scr = reinterpret_cast<float4 *>(sm.base + sm.lay.scratch);
    const int cap = (kScratchBytes / 64) / g.V;   // entries per slot the scratch holds (>= 1)
    int live = entries;
    while (live > cap) {
        const int half = (live + 1) >> 1;        // entries [half, live) fold into [0, live - half)
        if (holder && entry >= half) store_entry(scr, cap, g, entry - half, vs_own, v1, v2);
        named_sync(1, kConsumers);
        if (holder && entry + half < live) {
            const float4 a0 = *scr_at(scr, cap, g, 0, entry, vs_own);
            const float4 a1 = *scr_at(scr, cap, g, 1, entry, vs_own);
            const float4 b0 = *scr_at(scr, cap, g, 2, entry, vs_own);
            const float4 b1 = *scr_at(scr, cap, g, 3, entry, vs_own);
            v1[0] += a0.x; v1[1] += a0.y; v1[2] += a0.z; v1[3] += a0.w;
            v1[4] += a1.x; v1[5] += a1.y; v1[6] += a1.z; v1[7] += a1.w;
            v2[0] += b0.x; v2[1] += b0.y; v2[2] += b0.z; v2[3] += b0.w;
            v2[4] += b1.x; v2[5] += b1.y; v2[6] += b1.z; v2[7] += b1.w;
        }
        if (entry >= half) holder = false;
        named_sync(1, kConsumers);
        live = half;
    }
    if (holder) store_entry(scr, cap, g, entry, vs_own, v1, v2);
    named_sync(1, kConsumers);
    const float *kvec = reinterpret_cast<const float *>(sm.base + sm.lay.kvec);
    float2 *chs = reinterpret_cast<float2 *>(sm.base + sm.lay.chs);
    const float count = static_cast<float>(rows_of(g, m));
    const float inv_count = 1.0f / count;
    // per channel (mean, M2) of the item; thread t finishes channel
    // 8 * (t % V) + t / V: consecutive threads read consecutive slots
    for (int idx = tid; idx < g.C; idx += kConsumers) {
        const int vs = vec_slot<POW2>(g, idx), j = vec_rank<POW2>(g, idx);
        const int ch = 8 * vs + j;
        float S1 = 0.f, S2 = 0.f;
        for (int e = 0; e < live; ++e) {
            S1 += comp(*scr_at(scr, cap, g, j >> 2, e, vs), j & 3);
            S2 += comp(*scr_at(scr, cap, g, 2 + (j >> 2), e, vs), j & 3);
        }
        const float m = S1 * inv_count;
        chs[ch] = make_float2(kvec[ch] + m, fmaxf(S2 - S1 * m, 0.f));
    }
    named_sync(1, kConsumers);
    // channels -> one record per group (Chan with equal counts: the mean of
    // the channel means, then the within- plus between-channel squares).
    // With Cg <= 16 a warp takes two groups, one per half-warp.
    const float cgf = static_cast<float>(g.Cg);
    const int span = g.Cg <= 16 ? 16 : 32;                  // lanes per group
    const int sub = lane / span;                            // which group of the warp
    const int sl = lane & (span - 1);
    const int per_warp = 32 / span;
    for (int base = warp * per_warp; base < g.G; base += kConsumerWarps * per_warp) {
        const int grp = base + sub;
        const bool active = grp < g.G;
        const float2 *cr = chs + (active ? grp : 0) * g.Cg;
        float mu = 0.f;
        if (active)
            for (int j = sl; j < g.Cg; j += span) mu += cr[j].x;
        for (int off = span >> 1; off > 0; off >>= 1) mu += __shfl_xor_sync(0xffffffffu, mu, off);
        mu /= cgf;
        float M2 = 0.f;
        if (active)
            for (int j = sl; j < g.Cg; j += span) {
                const float d = cr[j].x - mu;
                M2 += fmaf(count * d, d, cr[j].y);
            }
        for (int off = span >> 1; off > 0; off >>= 1) M2 += __shfl_xor_sync(0xffffffffu, M2, off);
        if (active && sl == 0) a.partial[(m.n * g.G + grp) * g.S + m.s] = make_float2(mu, M2);
    }
    named_sync(1, kConsumers);
}

// Vectors per carrier thread of a full piece, when that is a power of two up
// to kMaxVecPerThread (the bodies below are compiled for those counts);
// 0 otherwise.
__device__ __forceinline__ int vec_kind(int nvec, int A)
{
#pragma unroll
    for (int k = kMaxVecPerThread; k >= 1; k >>= 1)
        if (nvec == k * A) return k;
    return 0;
}

// Shifted sums of the vectors tid, tid + A, ... of one piece.  VPT > 0: a
// full piece of exactly VPT vectors per carrier thread (no bounds checks);
// VPT == 0: a piece of any size (the short last piece of a batch entry).
template <int VPT>
__device__ __forceinline__ void p1_piece(uint32_t base, int tid, int A, int nvec, const f2_t (&K)[4], f2_t (&s1)[4],
                                         f2_t (&s2)[4])
{
    if (VPT > 0) {
        uint4 w[VPT > 0 ? VPT : 1];
#pragma unroll
        for (int i = 0; i < VPT; ++i) w[i] = lds128(base + 16u * static_cast<uint32_t>(tid + i * A));
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const f2_t d = sub2(bf2_to_f2(ws[j]), K[j]);
                s1[j] = add2(s1[j], d);
                s2[j] = fma2(d, d, s2[j]);
            }
        }
    } else {
#pragma unroll 1
        for (int v = tid; v < nvec; v += A) {
            const uint4 w = lds128(base + 16u * v);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const f2_t d = sub2(bf2_to_f2(ws[j]), K[j]);
                s1[j] = add2(s1[j], d);
                s2[j] = fma2(d, d, s2[j]);
            }
        }
    }
}

// Power-of-two C: the item's per-group (mean, M2) records straight
// from the per-thread sums, without per-channel statistics.  Every channel
// of a group shares the group's shift K_g, so sums of different channels
// of one group add directly.  U = max(1, 8 / Cg) groups per thread; a group
// covers spg = max(1, Cg / 8) vector slots.
//  1. each thread folds its eight channel sums into its U group sums;
//  2. a butterfly over the lane offsets that stay inside a group (offsets
//     below spg: neighbouring slots of the group; offsets of V and more:
//     the same slot in another row of the warp) gives every lane its
//     group's warp total;
//  3. one lane per (warp or row, group) writes that total to shared memory;
//  4. thread t adds the R partials of group t in a fixed order, so the
//     result is deterministic.
template <int U>
__device__ void reduce_item_pow2(const Args &a, const Smem &sm, const Item &m, const f2_t (&s1p)[4],
                                 const f2_t (&s2p)[4])
{
    const Geom &g = a.g;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int V = g.V, Cg = g.Cg;
    const int vslot = tid & (V - 1);
    const int spg = Cg >= 8 ? Cg >> 3 : 1;
    float c1[8], c2[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        upk(s1p[i], c1[2 * i], c1[2 * i + 1]);
        upk(s2p[i], c2[2 * i], c2[2 * i + 1]);
    }
    float u1[U], u2[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        constexpr int W = 8 / U;   // channels per group sum
        float x1 = 0.f, x2 = 0.f;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            x1 += c1[u * W + j];
            x2 += c2[u * W + j];
        }
        u1[u] = x1;
        u2[u] = x2;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        if (off < spg || off >= V) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                u1[u] += __shfl_xor_sync(0xffffffffu, u1[u], off);
                u2[u] += __shfl_xor_sync(0xffffffffu, u2[u], off);
            }
        }
    }
    float2 *scr = reinterpret_cast<float2 *>(sm.base + sm.lay.scratch);
    const int sub = spg > 32 ? spg >> 5 : 1;          // warps per group and row
    const int R = V <= 32 ? kConsumerWarps : (kConsumers / V) * sub;
    const bool rep = (V >= 32 || lane < V) && (spg > 32 ? lane == 0 : (vslot & (spg - 1)) == 0);
    if (rep) {
        const int p = V <= 32 ? warp : (tid / V) * sub + ((vslot & (spg - 1)) >> 5);
        const int t0 = (8 * vslot) / Cg;
#pragma unroll
        for (int u = 0; u < U; ++u) scr[p * g.G + t0 + u] = make_float2(u1[u], u2[u]);
    }
    named_sync(1, kConsumers);
    const float *kvec = reinterpret_cast<const float *>(sm.base + sm.lay.kvec);
    const float rows = static_cast<float>(rows_of(g, m));
    const float inv_n = 1.0f / (rows * static_cast<float>(Cg));
    for (int t = tid; t < g.G; t += kConsumers) {
        float S1 = 0.f, S2 = 0.f;
        for (int p = 0; p < R; ++p) {
            const float2 v = scr[p * g.G + t];
            S1 += v.x;
            S2 += v.y;
        }
        const float mo = S1 * inv_n;   // mean - K_g
        a.partial[(m.n * g.G + t) * g.S + m.s] = make_float2(kvec[t * Cg] + mo, fmaxf(S2 - S1 * mo, 0.f));
    }
    named_sync(1, kConsumers);
}

template <bool POW2>
__device__ __forceinline__ void reduce_item(const Args &a, const Smem &sm, const Item &m, const f2_t (&s1p)[4],
                                            const f2_t (&s2p)[4])
{
    if (POW2) {
        const int Cg = a.g.Cg;
        if (Cg >= 8)
            reduce_item_pow2<1>(a, sm, m, s1p, s2p);
        else if (Cg == 4)
            reduce_item_pow2<2>(a, sm, m, s1p, s2p);
        else if (Cg == 2)
            reduce_item_pow2<4>(a, sm, m, s1p, s2p);
        else
            reduce_item_pow2<8>(a, sm, m, s1p, s2p);
    } else {
        reduce_item_general<POW2>(a, sm, m, s1p, s2p);
    }
}

// Consumer-side ring position and wait state, carried from piece to piece.
struct RingPos {
    int slot;
    uint32_t base;        // shared address of the slot
    uint32_t full_par;    // parity of the next full-barrier phase, per slot
    bool ok;              // no wait has expired
};

// The shift K of the thread's eight channels: each channel's group's first
// channel in the item's first row (shared by the whole group), read from
// the item's first piece; threads tid < V also publish them per channel.
template <bool POW2>
__device__ __forceinline__ void item_shift(const Geom &g, const Smem &sm, uint32_t base, int vslot, f2_t (&K)[4])
{
    float kc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = 8 * vslot + i;
        const int c0 = POW2 ? (c & ~(g.Cg - 1)) : (c / g.Cg) * g.Cg;
        kc[i] = __uint_as_float(lds_u16(base + 2u * c0) << 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) K[i] = pk(kc[2 * i], kc[2 * i + 1]);
    if (static_cast<int>(threadIdx.x) < g.V) {
        float4 *kv = reinterpret_cast<float4 *>(sm.base + sm.lay.kvec) + 2 * vslot;
        kv[0] = make_float4(kc[0], kc[1], kc[2], kc[3]);
        kv[1] = make_float4(kc[4], kc[5], kc[6], kc[7]);
    }
}

// `count` consecutive pieces of an item in pass 1, each of nvec vectors
// (VPT per carrier thread when VPT > 0).  The first one sets the shift K
// when need_k.
template <bool POW2, int VPT>
__device__ __forceinline__ void p1_run(const Geom &g, const Smem &sm, const Ctl &ctl, int64_t count, int nvec, int A,
                                    bool carrier, int vslot, bool need_k, f2_t (&K)[4], f2_t (&s1)[4], f2_t (&s2)[4],
                                    RingPos &rp)
{
    const int tid = threadIdx.x;
    for (int64_t j = 0; j < count; ++j) {
        if (rp.ok) rp.ok = wait_phase(sm.full(rp.slot), (rp.full_par >> rp.slot) & 1u, ctl);
        rp.full_par ^= 1u << rp.slot;
        if (rp.ok) {
            if (need_k && j == 0) item_shift<POW2>(g, sm, rp.base, vslot, K);
            if (carrier) p1_piece<VPT>(rp.base, tid, A, nvec, K, s1, s2);
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(sm.empty(rp.slot));
        if (++rp.slot == g.ring) {
            rp.slot = 0;
            rp.base = sm.ring_s;
        } else {
            rp.base += static_cast<uint32_t>(g.piece_bytes);
        }
    }
}

template <bool POW2>
__device__ void consume_pass1(const Args &a, const Smem &sm, int64_t T, uint32_t &full_par, const Ctl &ctl)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const int tid = threadIdx.x;
    const int vslot = vec_slot<POW2>(g, tid);
    const int A = carriers<POW2>(g);
    const bool carrier = POW2 || tid < A;
    const int full_nvec = g.rows_per_piece * g.V;
    const int tail_nvec = g.tail_rows * g.V;
    const int kind_full = vec_kind(full_nvec, A);
    RingPos rp{0, sm.ring_s, full_par, !*ctl.abort};
    for (int64_t it = blockIdx.x; it < g.items; it += gridDim.x) {
        const Item m = make_item(g, it);
        f2_t K[4], s1[4], s2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) K[i] = s1[i] = s2[i] = 0ull;
        // the item's full pieces, then the batch entry's short last piece
        const int64_t full = m.np - (m.tail ? 1 : 0);
        if (full > 0) {
            switch (kind_full) {
            case 8: p1_run<POW2, 8>(g, sm, ctl, full, full_nvec, A, carrier, vslot, true, K, s1, s2, rp); break;
            case 4: p1_run<POW2, 4>(g, sm, ctl, full, full_nvec, A, carrier, vslot, true, K, s1, s2, rp); break;
            case 2: p1_run<POW2, 2>(g, sm, ctl, full, full_nvec, A, carrier, vslot, true, K, s1, s2, rp); break;
            case 1: p1_run<POW2, 1>(g, sm, ctl, full, full_nvec, A, carrier, vslot, true, K, s1, s2, rp); break;
            default: p1_run<POW2, 0>(g, sm, ctl, full, full_nvec, A, carrier, vslot, true, K, s1, s2, rp); break;
            }
        }
        if (m.tail) p1_run<POW2, 0>(g, sm, ctl, 1, tail_nvec, A, carrier, vslot, full == 0, K, s1, s2, rp);
        reduce_item<POW2>(a, sm, m, s1, s2);
    }
    full_par = rp.full_par;
}

// ---------------------------------------------------------------------------
// finalize pieces
// ---------------------------------------------------------------------------
// Chan merge, by one warp, of the S item records (mean, M2) of each of GB
// groups (grp0, grp0 + gstride, ...; groups at or past G give nothing).
// Record s covers item_rows_f(s) * Cg elements.  Lane l holds records
// l, l + 32, ... (S <= 32 * PER_LANE); records past S count zero rows,
// which leaves every sum unchanged.  All GB * PER_LANE loads are issued
// before the first is used, so a batch costs one L2 round trip.  Returns
// (mean, rstd) of every group in every lane.
template <int PER_LANE, int GB>
__device__ __forceinline__ void merge_groups_warp(const Args &a, int64_t n, int grp0, int gstride, float2 (&out)[GB])
{
    const Geom &g = a.g;
    const int lane = threadIdx.x & 31;
    float2 r[GB][PER_LANE];
    const float2 *src_n = a.partial + n * g.G * g.S;   // then grp * S fits 32 bits
#pragma unroll
    for (int b = 0; b < GB; ++b) {
        const int grp = grp0 + b * gstride;
        const float2 *src = src_n + (grp < g.G ? grp : 0) * g.S;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int s = lane + 32 * i;
            r[b][i] = (grp < g.G && s < g.S) ? __ldcg(src + s) : make_float2(0.f, 0.f);
        }
    }
    float rows[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int s = lane + 32 * i;
        rows[i] = s < g.S ? item_rows_f(g, s) : 0.f;
    }
    const float cgf = static_cast<float>(g.Cg);
    float acc[GB];
#pragma unroll
    for (int b = 0; b < GB; ++b) {
        acc[b] = 0.f;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) acc[b] = fmaf(rows[i], r[b][i].x, acc[b]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int b = 0; b < GB; ++b) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
    float mean[GB], acc2[GB];
#pragma unroll
    for (int b = 0; b < GB; ++b) {
        mean[b] = acc[b] * g.inv_L;
        acc2[b] = 0.f;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const float d = r[b][i].x - mean[b];
            acc2[b] += fmaf(cgf * rows[i] * d, d, r[b][i].y);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int b = 0; b < GB; ++b) acc2[b] += __shfl_xor_sync(0xffffffffu, acc2[b], off);
#pragma unroll
    for (int b = 0; b < GB; ++b) {
        const float var = fmaxf(acc2[b] * g.inv_LCg, 0.f);
        out[b] = make_float2(mean[b], rsqrtf(var + a.eps));
    }
}

template <int PER_LANE>
__device__ __forceinline__ float2 merge_items_warp(const Args &a, int64_t n, int grp)
{
    float2 r[1];
    merge_groups_warp<PER_LANE, 1>(a, n, grp, 0, r);
    return r[0];
}

// ---------------------------------------------------------------------------
// consumers: pass 2 (reverse order, in place in shared memory)
// ---------------------------------------------------------------------------
// Outputs of vectors tid, tid + A, ... of one piece, each stored as soon as
// it is computed; dst points at this thread's first vector (piece start +
// tid).  VPT > 0: a full piece of exactly VPT vectors per carrier thread,
// VPT == 0: any size up to kMaxVecPerThread vectors per thread (the short
// last piece).  When this returns, every shared-memory load of the thread
// has been consumed by a store that is already issued.
template <bool SILU, int VPT>
__device__ __forceinline__ void p2_piece(uint32_t base, uint4 *dst, int tid, int A, int nvec, const f2_t (&S)[4],
                                         const f2_t (&Tt)[4])
{
#pragma unroll
    for (int i = 0; i < (VPT > 0 ? VPT : kMaxVecPerThread); ++i) {
        const int v = tid + i * A;
        if (VPT > 0 || v < nvec) {
            const uint4 w = lds128(base + 16u * static_cast<uint32_t>(v));
            uint4 o;
            o.x = apply_pair<SILU>(w.x, S[0], Tt[0]);
            o.y = apply_pair<SILU>(w.y, S[1], Tt[1]);
            o.z = apply_pair<SILU>(w.z, S[2], Tt[2]);
            o.w = apply_pair<SILU>(w.w, S[3], Tt[3]);
            dst[i * A] = o;
        }
    }
}

// Scale / shift of batch entry n into shared memory (fused kernel): the
// G group records (mean, rstd) written by the finalize step of the whole
// grid come in with one small batch of loads, then every channel folds its
// gamma / beta (loaded at kernel start) with its group's statistics.
__device__ void fused_scale_shift(const Args &a, const Smem &sm, int64_t n)
{
    const Geom &g = a.g;
    float2 *st = reinterpret_cast<float2 *>(sm.base + sm.lay.st);
    const float2 *gb = reinterpret_cast<const float2 *>(sm.base + sm.lay.gb);
    float2 *gs = reinterpret_cast<float2 *>(sm.base + sm.lay.gstat);
    for (int grp = threadIdx.x; grp < g.G; grp += kConsumers) gs[grp] = __ldcg(a.gstat + n * g.G + grp);
    named_sync(1, kConsumers);
    for (int c = threadIdx.x; c < g.C; c += kConsumers) {
        const float2 r = gs[g.Cg_pow2 ? (c >> g.log2_Cg) : (c / g.Cg)];
        const float2 ab = gb[c];
        const float sc = ab.x * r.y;
        st[c] = make_float2(sc, ab.y - r.x * sc);
    }
    named_sync(1, kConsumers);
}

// Scale / shift of batch entry n when every CTA merges the group records
// itself (one-barrier fused schedule).  P = stat_lanes lanes (a power of
// two, at most a warp) take one group: lane `sub` loads records sub,
// sub + P, ... (at most kStatRecords of them, all loads in flight at
// once).  The records are merged around a shift K (record 0's mean, which
// is within a few standard errors of the group mean):
//   A1 = sum rows_s (m_s - K),  A2 = sum [M2_s + rows_s Cg (m_s - K)^2]
//   mean = K + A1 / L,          M2 = A2 - Cg A1^2 / L
// with one butterfly over the P lanes; those lanes then fold gamma / beta
// of the group's channels.  The CTA that owns item 0 of n writes the
// statistics outputs.
__device__ void fused_local_stats(const Args &a, const Smem &sm, int64_t n, bool write_stats)
{
    const Geom &g = a.g;
    const int tid = threadIdx.x;
    const int P = g.stat_lanes;
    const int sub = tid & (P - 1);
    const int src_lane = (tid & 31) & ~(P - 1);   // lane of sub 0 in this lane's P-group
    const int per_pass = kConsumers >> g.stat_log2;
    const int passes = g.stat_passes;
    float2 *st = reinterpret_cast<float2 *>(sm.base + sm.lay.st);
    const float2 *gb = reinterpret_cast<const float2 *>(sm.base + sm.lay.gb);
    const float2 *src_n = a.partial + n * g.G * g.S;   // then grp * S fits 32 bits
    const float cgf = static_cast<float>(g.Cg);
    for (int pass = 0; pass < passes; ++pass) {
        const int grp = (tid >> g.stat_log2) + pass * per_pass;
        const bool valid = grp < g.G;
        const float2 *src = src_n + (valid ? grp : 0) * g.S;
        float2 r[kStatRecords];
#pragma unroll
        for (int i = 0; i < kStatRecords; ++i) {
            const int s_ = sub + P * i;
            r[i] = (valid && s_ < g.S) ? __ldcg(src + s_) : make_float2(0.f, 0.f);
        }
        const float K = __shfl_sync(0xffffffffu, r[0].x, src_lane);
        float A1 = 0.f, A2 = 0.f;
#pragma unroll
        for (int i = 0; i < kStatRecords; ++i) {
            const int s_ = sub + P * i;
            const float rows = s_ < g.S ? item_rows_f(g, s_) : 0.f;
            const float d = r[i].x - K;
            A1 = fmaf(rows, d, A1);
            A2 += fmaf(rows * cgf * d, d, r[i].y);
        }
        for (int off = 1; off < P; off <<= 1) {
            A1 += __shfl_xor_sync(0xffffffffu, A1, off);
            A2 += __shfl_xor_sync(0xffffffffu, A2, off);
        }
        const float mo = A1 * g.inv_L;
        const float mean = K + mo;
        const float var = fmaxf((A2 - cgf * A1 * mo) * g.inv_LCg, 0.f);
        const float rstd = rsqrtf(var + a.eps);
        if (valid) {
            if (write_stats && sub == 0) {
                a.mean[n * g.G + grp] = mean;
                a.rstd[n * g.G + grp] = rstd;
            }
            for (int c = grp * g.Cg + sub; c < (grp + 1) * g.Cg; c += P) {
                const float2 ab = gb[c];
                const float sc = ab.x * rstd;
                st[c] = make_float2(sc, ab.y - mean * sc);
            }
        }
    }
    named_sync(1, kConsumers);
}

// Where a consumer thread starts pass 2: the CTA's last item, the ring slot
// of its last piece and that piece's y address.  Integer divisions only;
// the fused kernel works this out before pass 1, while the first bulk
// copies are in flight, so that none of it sits between the grid barrier
// and the first output.
struct P2Start {
    int64_t it;
    Item m;
    int slot;
    uint4 *dst;
};

__device__ __forceinline__ P2Start pass2_start(const Args &a, int64_t T)
{
    const Geom &g = a.g;
    P2Start p;
    p.it = (g.items <= gridDim.x) ? blockIdx.x : blockIdx.x + ((g.items - 1 - blockIdx.x) / gridDim.x) * gridDim.x;
    p.m = make_item(g, p.it);
    p.slot = T > 0 ? slot_of(T - 1, g.ring) : 0;
    p.dst = reinterpret_cast<uint4 *>(a.y + piece_elem_offset(g, p.m.n, p.m.s + (p.m.np - 1) * g.S)) + threadIdx.x;
    return p;
}

// `count` consecutive pieces of an item in pass 2, walked backwards, each of
// nvec vectors (VPT per carrier thread when VPT > 0).  The first
// `resident` pieces are still in their ring slots from pass 1.
template <bool SILU, int VPT>
__device__ __forceinline__ void p2_run(const Geom &g, const Smem &sm, const Ctl &ctl, int64_t count, int nvec, int A,
                                    bool carrier, int item_stride, const f2_t (&S)[4], const f2_t (&Tt)[4],
                                    int64_t &resident, uint4 *&dst, RingPos &rp)
{
    const int tid = threadIdx.x;
    for (int64_t j = 0; j < count; ++j) {
        if (resident > 0) {
            --resident;
        } else {
            if (rp.ok) rp.ok = wait_phase(sm.full(rp.slot), (rp.full_par >> rp.slot) & 1u, ctl);
            rp.full_par ^= 1u << rp.slot;
        }
        // Every loaded value is used by an issued store before the slot is
        // released, so no shared-memory load of any lane is still in flight
        // when the warp signals the producer, which may then overwrite it.
        if (rp.ok && carrier) p2_piece<SILU, VPT>(rp.base, dst, tid, A, nvec, S, Tt);
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(sm.empty(rp.slot));   // the slot may be refilled now
        dst -= item_stride;
        if (rp.slot == 0) {
            rp.slot = g.ring - 1;
            rp.base = sm.slot_addr(rp.slot, g.piece_bytes);
        } else {
            --rp.slot;
            rp.base -= static_cast<uint32_t>(g.piece_bytes);
        }
    }
}

template <bool SILU, bool FUSED, bool POW2>
__device__ void consume_pass2(const Args &a, const Smem &sm, int64_t T, int64_t resident, uint32_t &full_par,
                              const Ctl &ctl, const P2Start &start)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const int tid = threadIdx.x;
    const int vslot = vec_slot<POW2>(g, tid);
    const int A = carriers<POW2>(g);
    const bool carrier = POW2 || tid < A;   // threads past A carry no data
    const int full_nvec = g.rows_per_piece * g.V;
    const int tail_nvec = g.tail_rows * g.V;
    const int kind_full = vec_kind(full_nvec, A);
    // y vectors between consecutive pieces of an item (S pieces apart; at
    // most 512 * 2048)
    const int item_stride = g.S * (g.piece_bytes / 16);
    RingPos rp{start.slot, sm.slot_addr(start.slot, g.piece_bytes), full_par, !*ctl.abort};
    int64_t cur_n = -1;
    int64_t it = start.it;
    Item m = start.m;
    uint4 *dst = start.dst;   // y of the item's last piece, this thread's first vector
    for (;;) {
        // (scale, shift) of the thread's eight channels, as pairs
        f2_t S[4], Tt[4];
        {
            const float4 *src;
            if (FUSED) {
                if (m.n != cur_n) {
                    if (g.G * g.S <= kOneBarrierRecords)
                        fused_local_stats(a, sm, m.n, m.s == 0);
                    else
                        fused_scale_shift(a, sm, m.n);
                }
                src = reinterpret_cast<const float4 *>(sm.base + sm.lay.st) + 4 * vslot;
            } else {
                src = reinterpret_cast<const float4 *>(a.st + m.n * g.C + 8 * vslot);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 v = FUSED ? src[j] : __ldcg(src + j);   // (s, t) of channels 2j, 2j+1
                S[j] = pk(v.x, v.z);
                Tt[j] = pk(v.y, v.w);
            }
            cur_n = m.n;
        }
        // backwards: the batch entry's short last piece (if the item owns it), then the full ones
        if (m.tail) p2_run<SILU, 0>(g, sm, ctl, 1, tail_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp);
        const int64_t full = m.np - (m.tail ? 1 : 0);
        switch (kind_full) {
        case 8: p2_run<SILU, 8>(g, sm, ctl, full, full_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp); break;
        case 4: p2_run<SILU, 4>(g, sm, ctl, full, full_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp); break;
        case 2: p2_run<SILU, 2>(g, sm, ctl, full, full_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp); break;
        case 1: p2_run<SILU, 1>(g, sm, ctl, full, full_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp); break;
        default: p2_run<SILU, 0>(g, sm, ctl, full, full_nvec, A, carrier, item_stride, S, Tt, resident, dst, rp); break;
        }
        it -= gridDim.x;
        if (it < 0) break;
        m = make_item(g, it);
        dst = reinterpret_cast<uint4 *>(a.y + piece_elem_offset(g, m.n, m.s + (m.np - 1) * g.S)) + tid;
    }
    full_par = rp.full_par;
}

template <bool SILU, bool POW2>
__device__ void consume_pass2_dyn(const Args &a, const Smem &sm, int64_t T, int64_t resident, uint32_t &full_par,
                                  const Ctl &ctl)
{
    const Geom &g = a.g;
    const int tid = threadIdx.x;
    const int32_t s = static_cast<int32_t>(blockIdx.x);   // this CTA's item
    if (g.G * g.S <= kOneBarrierRecords)
        fused_local_stats(a, sm, 0, s == 0);
    else
        fused_scale_shift(a, sm, 0);
    const int vslot = vec_slot<POW2>(g, tid);
    const int A = carriers<POW2>(g);
    const bool carrier = POW2 || tid < A;
    const int full_nvec = g.rows_per_piece * g.V;
    const int tail_nvec = g.tail_rows * g.V;
    const int kind_full = vec_kind(full_nvec, A);
    f2_t Sc[4], Tt[4];
    {
        const float4 *src = reinterpret_cast<const float4 *>(sm.base + sm.lay.st) + 4 * vslot;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = src[j];
            Sc[j] = pk(v.x, v.z);
            Tt[j] = pk(v.y, v.w);
        }
    }
    const volatile int32_t *tags = reinterpret_cast<const volatile int32_t *>(sm.base + sm.lay.tags);
    const int64_t np = item_pieces(g, s);
    bool ok = !*ctl.abort;
    for (int64_t j = 0;; ++j) {
        const int slot = dyn_slot(T, j, g.ring);
        int64_t k;
        if (j < resident) {
            k = s + (np - 1 - j) * g.S;   // still in the ring from pass 1
        } else {
            if (ok) ok = wait_phase(sm.full(slot), (full_par >> slot) & 1u, ctl);
            full_par ^= 1u << slot;
            if (!ok) break;
            k = tags[slot];
            if (k < 0) break;
        }
        const uint32_t base = sm.slot_addr(slot, g.piece_bytes);
        uint4 *dst = reinterpret_cast<uint4 *>(a.y + piece_elem_offset(g, 0, k)) + tid;
        if (ok && carrier) {
            if (k == g.pieces_per_n - 1) {
                p2_piece<SILU, 0>(base, dst, tid, A, tail_nvec, Sc, Tt);
            } else {
                switch (kind_full) {
                case 8: p2_piece<SILU, 8>(base, dst, tid, A, full_nvec, Sc, Tt); break;
                case 4: p2_piece<SILU, 4>(base, dst, tid, A, full_nvec, Sc, Tt); break;
                case 2: p2_piece<SILU, 2>(base, dst, tid, A, full_nvec, Sc, Tt); break;
                case 1: p2_piece<SILU, 1>(base, dst, tid, A, full_nvec, Sc, Tt); break;
                default: p2_piece<SILU, 0>(base, dst, tid, A, full_nvec, Sc, Tt); break;
                }
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(sm.empty(slot));   // the slot may be refilled now
    }
}

// ---------------------------------------------------------------------------
// kernel prologue: shared memory carve-up, mbarrier init, status check
// ---------------------------------------------------------------------------
extern __shared__ __align__(1024) uint8_t g_smem[];

__device__ __forceinline__ bool prologue(const Args &a, int kind, Smem &sm, Ctl &ctl, int64_t &T)
{
    sm.base = g_smem;
    sm.lay = make_layout(a.g, kind);
    sm.ring_s = smem_addr(g_smem);
    sm.bars_s = sm.ring_s + sm.lay.bars;
    volatile int *flags = reinterpret_cast<volatile int *>(g_smem + sm.lay.flags);
    // With programmatic stream serialization (the fused launch) the kernel
    // ahead in the stream may still be running: shared memory only until
    // griddepcontrol.wait returns (for other launches it returns at once).
    // Then a kernel launched after this one the same way may start.
    if (threadIdx.x < 32) {
        for (int s = threadIdx.x; s < a.g.ring; s += 32) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), kConsumerWarps);
        }
        mbar_init_fence();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 32) {
        const unsigned int st = *reinterpret_cast<volatile unsigned int *>(&g_status);
        flags[0] = (st != 0u) ? 1 : 0;
    }
    T = cta_piece_count(a.g);
    __syncthreads();
    ctl.abort = flags;
    ctl.timeout_ns = a.timeout_ns;
    return *flags == 0;
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
template <bool POW2>
__global__ void __launch_bounds__(kThreads, 1) gn_pass1_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    int64_t T;
    if (!prologue(a, kPass1, sm, ctl, T)) return;
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            ProducerState ps{0u, 0u, 0u};
            produce_pass1(a, sm, T, ps, ctl, false);
            if (*ctl.abort) drain_loads(sm, ps, a.g.ring);
        }
        return;
    }
    uint32_t full_par = 0;
    consume_pass1<POW2>(a, sm, T, full_par, ctl);
}

// Two-pass schedule, step 2: one warp per (n, g) merges the group's item
// records, writes mean / rstd and the scale / shift of its Cg channels.
__global__ void __launch_bounds__(256) gn_finalize_kernel(const __grid_constant__ Args a)
{
    if (*reinterpret_cast<volatile unsigned int *>(&g_status) != 0u) return;
    const Geom &g = a.g;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (t >= g.N * g.G) return;
    const int64_t n = t / g.G;
    const int grp = static_cast<int>(t - n * g.G);
    const int lane = threadIdx.x & 31;
    const float2 r = merge_items_warp<kMaxSegments / 32>(a, n, grp);
    if (lane == 0) {
        a.mean[t] = r.x;
        a.rstd[t] = r.y;
    }
    for (int j = lane; j < g.Cg; j += 32) {
        const int c = grp * g.Cg + j;
        const float sc = a.gamma[c] * r.y;
        a.st[n * g.C + c] = make_float2(sc, a.beta[c] - r.x * sc);
    }
}

template <bool SILU, bool POW2>
__global__ void __launch_bounds__(kThreads, 1) gn_pass2_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    int64_t T;
    if (!prologue(a, kPass2, sm, ctl, T)) return;
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            ProducerState ps{0u, 0u, 0u};
            produce_pass2(a, sm, T, 0, ps, ctl);
            if (*ctl.abort) drain_loads(sm, ps, a.g.ring);
        }
        return;
    }
    uint32_t full_par = 0;
    consume_pass2<SILU, false, POW2>(a, sm, T, 0, full_par, ctl, pass2_start(a, T));
}

template <bool SILU, bool POW2>
__global__ void __launch_bounds__(kThreads, 1) gn_fused_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    int64_t T;
    if (!prologue(a, kFused, sm, ctl, T)) return;
    const Geom &g = a.g;
    const int64_t resident = min(T, static_cast<int64_t>(g.ring));
    const bool producer = threadIdx.x == kConsumers;
    ProducerState ps{0u, 0u, 0u};
    uint32_t full_par = 0;

    // gamma / beta into shared memory while the first pieces are in flight
    if (threadIdx.x < kConsumers) {
        float2 *gb = reinterpret_cast<float2 *>(g_smem + sm.lay.gb);
        for (int c = threadIdx.x; c < g.C; c += kConsumers) gb[c] = make_float2(a.gamma[c], a.beta[c]);
    }

    // pass 1 (the consumers first work out where pass 2 will start)
    P2Start start{};
    if (producer) {
        produce_pass1(a, sm, T, ps, ctl, true);
    } else if (threadIdx.x < kConsumers) {
        start = pass2_start(a, T);
        consume_pass1<POW2>(a, sm, T, full_par, ctl);
    }
    // every item record of the grid is written
    grid_sync(a.sync, gridDim.x, ctl);
    const bool one_barrier = g.G * g.S <= kOneBarrierRecords;
    if (!one_barrier) {
        // finalize, step 1 (many groups): one warp per (n, g) task, spread
        // over the grid, merges the group's item records and publishes
        // (mean, rstd); a second barrier makes them visible to every CTA
        if (!*ctl.abort && threadIdx.x < kConsumers) {
            const int64_t tasks = g.N * g.G;
            for (int64_t t = static_cast<int64_t>(blockIdx.x) * kConsumerWarps + (threadIdx.x >> 5); t < tasks;
                 t += static_cast<int64_t>(gridDim.x) * kConsumerWarps) {
                const int64_t n = t / g.G;
                const float2 r = merge_items_warp<kFusedMaxSegments / 32>(a, n, static_cast<int>(t - n * g.G));
                if ((threadIdx.x & 31) == 0) {
                    a.gstat[t] = r;
                    a.mean[t] = r.x;
                    a.rstd[t] = r.y;
                }
            }
        }
        grid_sync(a.sync, 2u * gridDim.x, ctl);
    }
    if (threadIdx.x == kConsumers + 1 && !*ctl.abort) {
        // the last CTA past the last barrier re-arms the counters (done by
        // an otherwise idle producer-warp lane, off the consumers' path)
        if (atomicAdd(a.sync + 1, 1u) == gridDim.x - 1) {
            atomicExch(a.sync, 0u);
            atomicExch(a.sync + 1, 0u);
        }
    }

    // group statistics / scale and shift (per CTA, in consume_pass2), pass 2
    if (producer) {
        if (g.dyn_p2)
            produce_pass2_dyn(a, sm, T, resident, ps, ctl);
        else
            produce_pass2(a, sm, T, resident, ps, ctl);
        if (*ctl.abort) drain_loads(sm, ps, g.ring);
    } else if (threadIdx.x < kConsumers) {
        if (g.dyn_p2)
            consume_pass2_dyn<SILU, POW2>(a, sm, T, resident, full_par, ctl);
        else
            consume_pass2<SILU, true, POW2>(a, sm, T, resident, full_par, ctl, start);
    }
    if (g.dyn_p2) {
        // every piece this CTA took is done; the last CTA out zeroes the
        // counter for the next call
        __syncthreads();
        if (threadIdx.x == 0 && atomicAdd(a.sync + 3, 1u) == gridDim.x - 1) {
            atomicExch(a.sync + 2, 0u);
            atomicExch(a.sync + 3, 0u);
        }
    }
}

// Diagnostic: waits that nothing will ever satisfy, so the bounded-wait
// machinery must expire, record the sticky status and return.  mode 0: an
// mbarrier phase no thread arrives on; mode 1: a grid-barrier count no CTA
// reaches (the counter lives in this CTA's shared memory, so no global
// state is involved).  Writes 1 to done[blockIdx.x] when the CTA returns.
__global__ void __launch_bounds__(32) gn_selftest_wait_kernel(int mode, uint64_t timeout_ns, int *done)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ unsigned int counter;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        counter = 0;
        mbar_init(smem_addr(&bar), 1);
        mbar_init_fence();
    }
    __syncthreads();
    Ctl ctl;
    ctl.abort = &abort_flag;
    ctl.timeout_ns = timeout_ns;
    if (threadIdx.x == 0) {
        if (mode == 0) {
            wait_phase(smem_addr(&bar), 0, ctl);
        } else {
            const uint64_t deadline = global_ns() + timeout_ns;
            while (*reinterpret_cast<volatile unsigned int *>(&counter) < 1u) {
                if (global_ns() > deadline) {
                    record_timeout(ctl);
                    break;
                }
            }
        }
        done[blockIdx.x] = abort_flag ? 1 : 2;
    }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
static uint32_t smem_for(const Args &a, int kind) { return make_layout(a.g, kind).total; }

// The POW2 instantiations serve every C whose vector slots divide the
// consumer threads (C a power of two); the others serve the rest.
static bool pow2_slots(const Geom &g) { return kConsumers % g.V == 0; }

static const void *pass1_fn(bool pow2)
{
    return pow2 ? reinterpret_cast<const void *>(gn_pass1_kernel<true>)
                : reinterpret_cast<const void *>(gn_pass1_kernel<false>);
}

static const void *pass2_fn(bool silu, bool pow2)
{
    if (silu)
        return pow2 ? reinterpret_cast<const void *>(gn_pass2_kernel<true, true>)
                    : reinterpret_cast<const void *>(gn_pass2_kernel<true, false>);
    return pow2 ? reinterpret_cast<const void *>(gn_pass2_kernel<false, true>)
                : reinterpret_cast<const void *>(gn_pass2_kernel<false, false>);
}

static const void *fused_fn(bool silu, bool pow2)
{
    if (silu)
        return pow2 ? reinterpret_cast<const void *>(gn_fused_kernel<true, true>)
                    : reinterpret_cast<const void *>(gn_fused_kernel<true, false>);
    return pow2 ? reinterpret_cast<const void *>(gn_fused_kernel<false, true>)
                : reinterpret_cast<const void *>(gn_fused_kernel<false, false>);
}

cudaError_t prepare_kernels(uint32_t max_smem)
{
    const int sz = static_cast<int>(max_smem);
    for (int pow2 = 0; pow2 < 2; ++pow2) {
        const void *fns[] = {pass1_fn(pow2), pass2_fn(true, pow2), pass2_fn(false, pow2), fused_fn(true, pow2),
                             fused_fn(false, pow2)};
        for (const void *fn : fns) {
            const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, sz);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

static cudaError_t launch_plain(const void *fn, const Args &a, int grid, uint32_t smem, cudaStream_t s)
{
    Args copy = a;
    void *params[] = {&copy};
    return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), params, smem, s);
}

cudaError_t launch_pass1(const Args &a, int grid, cudaStream_t s)
{
    return launch_plain(pass1_fn(pow2_slots(a.g)), a, grid, smem_for(a, kPass1), s);
}

cudaError_t launch_finalize(const Args &a, cudaStream_t s)
{
    gn_finalize_kernel<<<static_cast<unsigned>((a.g.N * a.g.G + 7) / 8), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pass2(const Args &a, int grid, bool silu, cudaStream_t s)
{
    return launch_plain(pass2_fn(silu, pow2_slots(a.g)), a, grid, smem_for(a, kPass2), s);
}

cudaError_t fused_blocks_per_sm(bool silu, uint32_t smem, int *blocks)
{
    // the smaller of the two instantiations' figures, so that the answer
    // holds whichever one a launch picks
    int b0 = 0, b1 = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, fused_fn(silu, false), kThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, fused_fn(silu, true), kThreads, smem);
    if (e != cudaSuccess) return e;
    *blocks = b0 < b1 ? b0 : b1;
    return cudaSuccess;
}

cudaError_t launch_fused(const Args &a, int grid, bool silu, cudaStream_t s)
{
    Args copy = a;
    void *params[] = {&copy};
    // cooperative (the grid barrier), and with programmatic serialization:
    // the CTAs may start while the kernel ahead in the stream finishes
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_for(a, kFused);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, fused_fn(silu, pow2_slots(a.g)), params);
}

cudaError_t launch_selftest_wait(int mode, uint64_t timeout_ns, int *done, int blocks, cudaStream_t s)
{
    gn_selftest_wait_kernel<<<blocks, 32, 0, s>>>(mode, timeout_ns, done);
    return cudaGetLastError();
}

cudaError_t read_device_status(unsigned int *status)
{
    return cudaMemcpyFromSymbol(status, g_status, sizeof(unsigned int));
}

cudaError_t clear_device_status()
{
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

cudaError_t device_status_address(unsigned int **word)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(word), g_status);
}

cudaError_t set_device_status_host(unsigned int *host_word)
{
    return cudaMemcpyToSymbol(g_status_host, &host_word, sizeof(host_word));
}

}  // namespace gn
