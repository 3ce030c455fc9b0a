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
//  * The tensor is cut into "pieces" of whole rows (up to 16 KB); each CTA
//    streams its pieces through a ring of shared-memory slots filled by bulk
//    TMA copies (cp.async.bulk) issued by one producer thread, completion
//    tracked on mbarriers.  Eight consumer warps read 16-byte vectors from
//    shared memory; with C a power of two each consumer thread always sees
//    the same eight channels.
//  * Pass 1 keeps, per thread, fp32 sums of (x - K) and (x - K)^2 with K a
//    per-(work item, channel) shift (the item's first row), then reduces
//    them per CTA with warp shuffles and shared memory into a per-segment
//    (mean, M2) record.  Segments are merged with Chan's parallel formula,
//    first over segments per channel, then over the channels of a group.
//  * Pass 2 rewrites each piece in place in shared memory and sends it back
//    with a bulk TMA store; pieces are visited in the reverse of pass-1 order
//    so the most recently read rows (still in L2) come first.
//  * The fused kernel does all three steps in one cooperative launch with two
//    grid barriers; pieces still in the ring after pass 1 are not re-read.
//  * Every wait (mbarrier phase, grid barrier) is bounded by a deadline on
//    the global timer, counted from the start of that wait; on expiry the
//    kernel records a sticky status, stops issuing work, drains its own
//    copies and returns.
#include <cuda_bf16.h>

#include "gn_internal.h"
#include "gn_ptx.cuh"

namespace gn {

// Sticky device-side status: bit 0 = a bounded wait expired.
__device__ unsigned int g_status;

// ---------------------------------------------------------------------------
// work-item cursor
// ---------------------------------------------------------------------------
struct Cursor {
    int64_t it;        // work item id (n * S + s)
    int64_t n;
    int32_t s;
    int64_t p0, p1;    // piece range of the item inside batch entry n
    int64_t k;         // current piece
};

__device__ __forceinline__ void load_item(const Geom &g, Cursor &c, int64_t it)
{
    c.it = it;
    c.n = it / g.S;
    c.s = static_cast<int32_t>(it - c.n * g.S);
    c.p0 = static_cast<int64_t>(c.s) * g.pieces_per_n / g.S;
    c.p1 = static_cast<int64_t>(c.s + 1) * g.pieces_per_n / g.S;
}

__device__ __forceinline__ int64_t segment_rows(const Geom &g, int32_t s)
{
    const int64_t p0 = static_cast<int64_t>(s) * g.pieces_per_n / g.S;
    const int64_t p1 = static_cast<int64_t>(s + 1) * g.pieces_per_n / g.S;
    const int64_t r0 = p0 * g.rows_per_piece;
    const int64_t r1 = min(p1 * g.rows_per_piece, g.L);
    return r1 - r0;
}

__device__ __forceinline__ int32_t piece_rows(const Geom &g, int64_t k)
{
    return static_cast<int32_t>(min(static_cast<int64_t>(g.rows_per_piece), g.L - k * g.rows_per_piece));
}

__device__ __forceinline__ int64_t piece_elem_offset(const Geom &g, int64_t n, int64_t k)
{
    return (n * g.L + k * g.rows_per_piece) * g.C;
}

// pieces this CTA processes, over all its items
__device__ __forceinline__ int64_t cta_piece_count(const Geom &g)
{
    int64_t t = 0;
    for (int64_t it = blockIdx.x; it < g.items; it += gridDim.x) {
        Cursor c;
        load_item(g, c, it);
        t += c.p1 - c.p0;
    }
    return t;
}

__device__ __forceinline__ void cursor_first(const Geom &g, Cursor &c)
{
    load_item(g, c, blockIdx.x);
    c.k = c.p0;
}

// returns false when the CTA has no further piece
__device__ __forceinline__ bool cursor_next(const Geom &g, Cursor &c)
{
    if (++c.k < c.p1) return true;
    const int64_t it = c.it + gridDim.x;
    if (it >= g.items) return false;
    load_item(g, c, it);
    c.k = c.p0;
    return true;
}

__device__ __forceinline__ void cursor_last(const Geom &g, Cursor &c)
{
    const int64_t last = blockIdx.x + ((g.items - 1 - blockIdx.x) / gridDim.x) * gridDim.x;
    load_item(g, c, last);
    c.k = c.p1 - 1;
}

__device__ __forceinline__ bool cursor_prev(const Geom &g, Cursor &c)
{
    if (--c.k >= c.p0) return true;
    const int64_t it = c.it - gridDim.x;
    if (it < 0) return false;
    load_item(g, c, it);
    c.k = c.p1 - 1;
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
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl &ctl)
{
    if (*ctl.abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = global_ns() + ctl.timeout_ns;
#pragma unroll 1
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 31u) {
            if (*ctl.abort) return false;
            if (global_ns() > deadline) {
                record_timeout(ctl);
                return false;
            }
        }
    }
}

// Grid-wide barrier for the cooperative fused kernel: one arrival per CTA on
// a gpu-scope counter, then a bounded spin until `target` arrivals.
__device__ __forceinline__ bool grid_sync(unsigned int *counter, unsigned int target, const Ctl &ctl)
{
    __syncthreads();
    if (threadIdx.x == 0 && !*ctl.abort) {
        __threadfence();
        atom_add_release_gpu(counter, 1u);
        const uint64_t deadline = global_ns() + ctl.timeout_ns;
#pragma unroll 1
        for (uint32_t it = 0;; ++it) {
            if (ld_acquire_gpu(counter) >= target) break;
            if ((it & 15u) == 15u && global_ns() > deadline) {
                record_timeout(ctl);
                break;
            }
            __nanosleep(40);
        }
        __threadfence();
    }
    __syncthreads();
    return !*ctl.abort;
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
    return *reinterpret_cast<const uint32_t *>(&h);
}

// SiLU(z) = z * sigmoid(z), sigmoid from one ex2 and one reciprocal (both
// hardware approximations, a few ulp in fp32).
__device__ __forceinline__ float silu(float z)
{
    const float e = ex2_approx(z * -1.4426950408889634f);   // exp(-z)
    return z * rcp_approx(1.0f + e);
}

// ---------------------------------------------------------------------------
// shared memory view of one CTA
// ---------------------------------------------------------------------------
struct Smem {
    uint8_t *base;
    Layout lay;
    uint32_t ring_s;                       // shared address of the ring
    __device__ uint32_t full(int slot) const { return smem_addr(base + lay.bars) + 16u * slot; }
    __device__ uint32_t empty(int slot) const { return full(slot) + 8u; }
    __device__ uint32_t slot_addr(int slot, int piece_bytes) const
    {
        return ring_s + static_cast<uint32_t>(slot) * static_cast<uint32_t>(piece_bytes);
    }
};

__device__ __forceinline__ int slot_of(int64_t q, int ring) { return static_cast<int>(q % ring); }

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
// producer (one thread): pass-2 loads and stores, pieces in reverse order.
// `resident` pieces (the last ones of pass 1, fused kernel only) are still
// in their ring slots and are not loaded again.
// ---------------------------------------------------------------------------
__device__ void produce_pass2(const Args &a, const Smem &sm, int64_t T, int64_t resident,
                              ProducerState &ps, const Ctl &ctl)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const bool hint_ld = (a.l2_hints & 1u) != 0;
    const bool hint_st = (a.l2_hints & 2u) != 0;
    const uint64_t pol = (hint_ld || hint_st) ? policy_evict_first() : 0;
    Cursor ld, st;
    cursor_last(g, ld);
    cursor_last(g, st);
    int slot = slot_of(T - 1, g.ring);        // slot of the load cursor's piece
    int st_slot = slot;                       // slot of the store cursor's piece
    bool ok = !*ctl.abort;

    auto store_next = [&]() {
        if (ok) ok = wait_phase(sm.empty(st_slot), (ps.empty_par >> st_slot) & 1u, ctl);
        if (ok) {
            ps.empty_par ^= 1u << st_slot;
            const uint32_t bytes =
                static_cast<uint32_t>(piece_rows(g, st.k)) * static_cast<uint32_t>(g.C) * 2u;
            uint16_t *dst = a.y + piece_elem_offset(g, st.n, st.k);
            if (hint_st)
                bulk_store_hint(dst, sm.slot_addr(st_slot, g.piece_bytes), bytes, pol);
            else
                bulk_store(dst, sm.slot_addr(st_slot, g.piece_bytes), bytes);
            bulk_commit();
        }
        cursor_prev(g, st);
        st_slot = (st_slot == 0) ? g.ring - 1 : st_slot - 1;
    };

    int64_t stored = 0;
    for (int64_t q = T - 1; q >= 0; --q) {
        if (q < T - resident) {
            if (q + g.ring < T) {
                store_next();
                ++stored;
                bulk_wait_read_all();     // the slot's bytes have left shared memory
            }
            if (ok) issue_load(a, sm, ld, slot, ps, pol, hint_ld);
        }
        cursor_prev(g, ld);
        slot = (slot == 0) ? g.ring - 1 : slot - 1;
    }
    for (; stored < T; ++stored) store_next();
    bulk_wait_all();
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
// consumers: pass 1
// ---------------------------------------------------------------------------
// Reduce the per-thread shifted sums of one work item into the item's
// per-channel (mean, M2) record.
__device__ void reduce_item(const Args &a, const Smem &sm, const Cursor &c, const float (&s1)[8],
                            const float (&s2)[8])
{
    const Geom &g = a.g;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    float v1[8], v2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        v1[j] = s1[j];
        v2[j] = s2[j];
    }
    int entries, entry;
    bool writer;
    if (g.V < 32) {
        for (int off = g.V; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v1[j] += __shfl_xor_sync(0xffffffffu, v1[j], off);
                v2[j] += __shfl_xor_sync(0xffffffffu, v2[j], off);
            }
        }
        entries = kConsumerWarps;
        entry = warp;
        writer = lane < g.V;
    } else {
        entries = kConsumers / g.V;
        entry = tid / g.V;
        writer = true;
    }
    float *scr = reinterpret_cast<float *>(sm.base + sm.lay.scratch);
    if (writer) {
        float4 *dst = reinterpret_cast<float4 *>(scr + (entry * g.V + (tid % g.V)) * 16);
        dst[0] = make_float4(v1[0], v1[1], v1[2], v1[3]);
        dst[1] = make_float4(v1[4], v1[5], v1[6], v1[7]);
        dst[2] = make_float4(v2[0], v2[1], v2[2], v2[3]);
        dst[3] = make_float4(v2[4], v2[5], v2[6], v2[7]);
    }
    named_sync(1, kConsumers);
    const float *kvec = reinterpret_cast<const float *>(sm.base + sm.lay.kvec);
    const int64_t r0 = c.p0 * g.rows_per_piece;
    const int64_t r1 = min(c.p1 * g.rows_per_piece, g.L);
    const float count = static_cast<float>(r1 - r0);
    for (int ch = tid; ch < g.C; ch += kConsumers) {
        const int vs = ch >> 3, j = ch & 7;
        float S1 = 0.f, S2 = 0.f;
        for (int e = 0; e < entries; ++e) {
            S1 += scr[(e * g.V + vs) * 16 + j];
            S2 += scr[(e * g.V + vs) * 16 + 8 + j];
        }
        const float m = S1 / count;
        const float M2 = fmaxf(S2 - S1 * m, 0.f);
        a.partial[(c.n * g.C + ch) * g.S + c.s] = make_float2(kvec[ch] + m, M2);
    }
    named_sync(1, kConsumers);
}

__device__ void consume_pass1(const Args &a, const Smem &sm, int64_t T, uint32_t &full_par, const Ctl &ctl)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const int tid = threadIdx.x;
    const int vslot = tid % g.V;
    float *kvec = reinterpret_cast<float *>(sm.base + sm.lay.kvec);
    Cursor c;
    cursor_first(g, c);
    int slot = 0;
    float K[8], s1[8], s2[8];
    bool ok = !*ctl.abort;
    for (int64_t q = 0; q < T; ++q) {
        const bool first = (c.k == c.p0);
        if (first) {
#pragma unroll
            for (int j = 0; j < 8; ++j) s1[j] = s2[j] = 0.f;
        }
        if (ok) ok = wait_phase(sm.full(slot), (full_par >> slot) & 1u, ctl);
        full_par ^= 1u << slot;
        const uint32_t base = sm.slot_addr(slot, g.piece_bytes);
        if (ok) {
            if (first) {
                const uint4 w = lds128(base + 16u * vslot);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    K[2 * i] = bf_lo(ws[i]);
                    K[2 * i + 1] = bf_hi(ws[i]);
                }
                if (tid < g.V) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) kvec[8 * vslot + j] = K[j];
                }
            }
            const int nvec = piece_rows(g, c.k) * g.V;
#pragma unroll 4
            for (int v = tid; v < nvec; v += kConsumers) {
                const uint4 w = lds128(base + 16u * v);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float d0 = bf_lo(ws[i]) - K[2 * i];
                    const float d1 = bf_hi(ws[i]) - K[2 * i + 1];
                    s1[2 * i] += d0;
                    s2[2 * i] = fmaf(d0, d0, s2[2 * i]);
                    s1[2 * i + 1] += d1;
                    s2[2 * i + 1] = fmaf(d1, d1, s2[2 * i + 1]);
                }
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(sm.empty(slot));
        if (c.k + 1 == c.p1) reduce_item(a, sm, c, s1, s2);
        cursor_next(g, c);
        slot = (slot + 1 == g.ring) ? 0 : slot + 1;
    }
}

// ---------------------------------------------------------------------------
// finalize pieces
// ---------------------------------------------------------------------------
// Chan merge of the S segment records of channel (n, c), by one warp.
__device__ __forceinline__ float2 combine_channel(const Args &a, int64_t n, int c)
{
    const Geom &g = a.g;
    const int lane = threadIdx.x & 31;
    const float2 *src = a.partial + (n * g.C + c) * g.S;
    float mu[kPartialsPerLane], m2[kPartialsPerLane], cnt[kPartialsPerLane];
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kPartialsPerLane; ++i) {
        const int s = lane + 32 * i;
        if (s < g.S) {
            const float2 v = __ldcg(src + s);
            mu[i] = v.x;
            m2[i] = v.y;
            cnt[i] = static_cast<float>(segment_rows(g, s));
            acc = fmaf(cnt[i], v.x, acc);
        } else {
            mu[i] = m2[i] = cnt[i] = 0.f;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const float mean = acc / static_cast<float>(g.L);
    float acc2 = 0.f;
#pragma unroll
    for (int i = 0; i < kPartialsPerLane; ++i) {
        const float d = mu[i] - mean;
        acc2 += fmaf(cnt[i] * d, d, m2[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc2 += __shfl_xor_sync(0xffffffffu, acc2, off);
    return make_float2(mean, acc2);
}

// Chan merge of the Cg channel records of group (n, g): (mean, rstd).
__device__ __forceinline__ float2 combine_group(const Args &a, const float2 *ch, int Cg)
{
    float mu = 0.f;
    for (int j = 0; j < Cg; ++j) mu += ch[j].x;
    mu /= static_cast<float>(Cg);
    const float Lf = static_cast<float>(a.g.L);
    float M2 = 0.f;
    for (int j = 0; j < Cg; ++j) {
        const float d = ch[j].x - mu;
        M2 += fmaf(Lf * d, d, ch[j].y);
    }
    const float var = fmaxf(M2 / (Lf * static_cast<float>(Cg)), 0.f);
    return make_float2(mu, 1.0f / sqrtf(var + a.eps));
}

// ---------------------------------------------------------------------------
// consumers: pass 2 (reverse order, in place in shared memory)
// ---------------------------------------------------------------------------
template <bool SILU>
__device__ __forceinline__ uint32_t apply_pair(uint32_t w, float s0, float t0, float s1, float t1)
{
    float z0 = fmaf(bf_lo(w), s0, t0);
    float z1 = fmaf(bf_hi(w), s1, t1);
    if (SILU) {
        z0 = silu(z0);
        z1 = silu(z1);
    }
    return pack_bf16x2(z0, z1);
}

// Scale / shift of group statistics for batch entry n into shared memory
// (fused kernel).  Written to the statistics outputs by the one CTA that
// owns segment 0 of n.
__device__ void fused_group_finalize(const Args &a, const Smem &sm, int64_t n, bool write_stats)
{
    const Geom &g = a.g;
    float2 *st = reinterpret_cast<float2 *>(sm.base + sm.lay.st);
    float2 *gs = reinterpret_cast<float2 *>(sm.base + sm.lay.gstat);
    const int tid = threadIdx.x;
    // channel records -> shared memory (st doubles as staging)
    for (int c = tid; c < g.C; c += kConsumers) st[c] = __ldcg(a.chstat + n * g.C + c);
    named_sync(1, kConsumers);
    for (int grp = tid; grp < g.G; grp += kConsumers) {
        const float2 r = combine_group(a, st + grp * g.Cg, g.Cg);
        gs[grp] = r;
        if (write_stats) {
            a.mean[n * g.G + grp] = r.x;
            a.rstd[n * g.G + grp] = r.y;
        }
    }
    named_sync(1, kConsumers);
    for (int c = tid; c < g.C; c += kConsumers) {
        const float2 r = gs[c / g.Cg];
        const float sc = a.gamma[c] * r.y;
        st[c] = make_float2(sc, a.beta[c] - r.x * sc);
    }
    named_sync(1, kConsumers);
}

template <bool SILU, bool FUSED>
__device__ void consume_pass2(const Args &a, const Smem &sm, int64_t T, int64_t resident, uint32_t &full_par,
                              const Ctl &ctl)
{
    const Geom &g = a.g;
    if (T == 0) return;
    const int tid = threadIdx.x;
    const int vslot = tid % g.V;
    Cursor c;
    cursor_last(g, c);
    int slot = slot_of(T - 1, g.ring);
    int64_t cur_item = -1, cur_n = -1;
    float sc[8], sh[8];
    bool ok = !*ctl.abort;
    for (int64_t q = T - 1; q >= 0; --q) {
        if (c.it != cur_item) {
            if (FUSED) {
                if (c.n != cur_n) fused_group_finalize(a, sm, c.n, c.s == 0);
                const float2 *st = reinterpret_cast<const float2 *>(sm.base + sm.lay.st);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 v = st[8 * vslot + j];
                    sc[j] = v.x;
                    sh[j] = v.y;
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(a.st + c.n * g.C + 8 * vslot);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = __ldcg(src + j);
                    sc[2 * j] = v.x;
                    sh[2 * j] = v.y;
                    sc[2 * j + 1] = v.z;
                    sh[2 * j + 1] = v.w;
                }
            }
            cur_item = c.it;
            cur_n = c.n;
        }
        if (q < T - resident) {
            if (ok) ok = wait_phase(sm.full(slot), (full_par >> slot) & 1u, ctl);
            full_par ^= 1u << slot;
        }
        if (ok) {
            const uint32_t base = sm.slot_addr(slot, g.piece_bytes);
            const int nvec = piece_rows(g, c.k) * g.V;
#pragma unroll 4
            for (int v = tid; v < nvec; v += kConsumers) {
                const uint32_t addr = base + 16u * v;
                const uint4 w = lds128(addr);
                uint4 o;
                o.x = apply_pair<SILU>(w.x, sc[0], sh[0], sc[1], sh[1]);
                o.y = apply_pair<SILU>(w.y, sc[2], sh[2], sc[3], sh[3]);
                o.z = apply_pair<SILU>(w.z, sc[4], sh[4], sc[5], sh[5]);
                o.w = apply_pair<SILU>(w.w, sc[6], sh[6], sc[7], sh[7]);
                sts128(addr, o);
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(sm.empty(slot));
        cursor_prev(g, c);
        slot = (slot == 0) ? g.ring - 1 : slot - 1;
    }
}

// ---------------------------------------------------------------------------
// kernel prologue: shared memory carve-up, mbarrier init, status check
// ---------------------------------------------------------------------------
extern __shared__ __align__(1024) uint8_t g_smem[];

__device__ __forceinline__ bool prologue(const Args &a, int kind, Smem &sm, Ctl &ctl)
{
    sm.base = g_smem;
    sm.lay = make_layout(a.g, kind);
    sm.ring_s = smem_addr(g_smem);
    volatile int *flags = reinterpret_cast<volatile int *>(g_smem + sm.lay.flags);
    if (threadIdx.x == 0) {
        flags[0] = (*reinterpret_cast<volatile unsigned int *>(&g_status) != 0u) ? 1 : 0;
        for (int s = 0; s < a.g.ring; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), kConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    ctl.abort = flags;
    ctl.timeout_ns = a.timeout_ns;
    return *flags == 0;
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) gn_pass1_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    if (!prologue(a, kPass1, sm, ctl)) return;
    const int64_t T = cta_piece_count(a.g);
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            ProducerState ps{0u, 0u, 0u};
            produce_pass1(a, sm, T, ps, ctl, false);
            if (*ctl.abort) drain_loads(sm, ps, a.g.ring);
        }
        return;
    }
    uint32_t full_par = 0;
    consume_pass1(a, sm, T, full_par, ctl);
}

__global__ void __launch_bounds__(256) gn_finalize_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(16) float2 fin_smem[];   // [Cg] channel records + 1
    if (*reinterpret_cast<volatile unsigned int *>(&g_status) != 0u) return;
    const Geom &g = a.g;
    const int64_t n = blockIdx.x / g.G;
    const int grp = static_cast<int>(blockIdx.x % g.G);
    const int warp = threadIdx.x >> 5;
    for (int j = warp; j < g.Cg; j += 8) {
        const float2 r = combine_channel(a, n, grp * g.Cg + j);
        if ((threadIdx.x & 31) == 0) fin_smem[j] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const float2 r = combine_group(a, fin_smem, g.Cg);
        fin_smem[g.Cg] = r;
        a.mean[n * g.G + grp] = r.x;
        a.rstd[n * g.G + grp] = r.y;
    }
    __syncthreads();
    const float2 r = fin_smem[g.Cg];
    for (int j = threadIdx.x; j < g.Cg; j += 256) {
        const int c = grp * g.Cg + j;
        const float sc = a.gamma[c] * r.y;
        a.st[n * g.C + c] = make_float2(sc, a.beta[c] - r.x * sc);
    }
}

template <bool SILU>
__global__ void __launch_bounds__(kThreads) gn_pass2_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    if (!prologue(a, kPass2, sm, ctl)) return;
    const int64_t T = cta_piece_count(a.g);
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            ProducerState ps{0u, 0u, 0u};
            produce_pass2(a, sm, T, 0, ps, ctl);
            if (*ctl.abort) drain_loads(sm, ps, a.g.ring);
        }
        return;
    }
    uint32_t full_par = 0;
    consume_pass2<SILU, false>(a, sm, T, 0, full_par, ctl);
}

template <bool SILU>
__global__ void __launch_bounds__(kThreads, 1) gn_fused_kernel(const __grid_constant__ Args a)
{
    Smem sm;
    Ctl ctl;
    if (!prologue(a, kFused, sm, ctl)) return;
    const Geom &g = a.g;
    const int64_t T = cta_piece_count(g);
    const int64_t resident = min(T, static_cast<int64_t>(g.ring));
    const bool producer = threadIdx.x == kConsumers;
    ProducerState ps{0u, 0u, 0u};
    uint32_t full_par = 0;

    // pass 1
    if (producer) {
        produce_pass1(a, sm, T, ps, ctl, true);
    } else if (threadIdx.x < kConsumers) {
        consume_pass1(a, sm, T, full_par, ctl);
    }
    // every segment record of the grid is written
    grid_sync(a.sync, gridDim.x, ctl);

    // finalize, step 1: channel records, (n, c) pairs spread over the grid
    if (!*ctl.abort && threadIdx.x < kConsumers) {
        const int64_t tasks = g.N * g.C;
        const int64_t per = (tasks + gridDim.x - 1) / gridDim.x;
        const int64_t t0 = blockIdx.x * per;
        const int64_t t1 = min(t0 + per, tasks);
        for (int64_t t = t0 + (threadIdx.x >> 5); t < t1; t += kConsumerWarps) {
            const int64_t n = t / g.C;
            const int c = static_cast<int>(t - n * g.C);
            const float2 r = combine_channel(a, n, c);
            if ((threadIdx.x & 31) == 0) a.chstat[t] = r;
        }
    }
    grid_sync(a.sync, 2u * gridDim.x, ctl);
    if (threadIdx.x == 0 && !*ctl.abort) {
        // the last CTA past the second barrier re-arms the counters
        if (atomicAdd(a.sync + 1, 1u) == gridDim.x - 1) {
            atomicExch(a.sync, 0u);
            atomicExch(a.sync + 1, 0u);
        }
    }

    // finalize step 2 (per CTA, in consume_pass2) and pass 2
    if (producer) {
        produce_pass2(a, sm, T, resident, ps, ctl);
        if (*ctl.abort) drain_loads(sm, ps, g.ring);
    } else if (threadIdx.x < kConsumers) {
        consume_pass2<SILU, true>(a, sm, T, resident, full_par, ctl);
    }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
static uint32_t smem_for(const Args &a, int kind) { return make_layout(a.g, kind).total; }

cudaError_t prepare_kernels(uint32_t max_smem)
{
    cudaError_t e;
    const int sz = static_cast<int>(max_smem);
    if ((e = cudaFuncSetAttribute(gn_pass1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sz))) return e;
    if ((e = cudaFuncSetAttribute(gn_pass2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sz)))
        return e;
    if ((e = cudaFuncSetAttribute(gn_pass2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sz)))
        return e;
    if ((e = cudaFuncSetAttribute(gn_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sz)))
        return e;
    if ((e = cudaFuncSetAttribute(gn_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sz)))
        return e;
    return cudaFuncSetAttribute(gn_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 * 2049 + 16);
}

cudaError_t launch_pass1(const Args &a, int grid, cudaStream_t s)
{
    gn_pass1_kernel<<<grid, kThreads, smem_for(a, kPass1), s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const Args &a, cudaStream_t s)
{
    const uint32_t smem = 8u * (a.g.Cg + 1);
    gn_finalize_kernel<<<static_cast<unsigned>(a.g.N * a.g.G), 256, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pass2(const Args &a, int grid, bool silu, cudaStream_t s)
{
    if (silu)
        gn_pass2_kernel<true><<<grid, kThreads, smem_for(a, kPass2), s>>>(a);
    else
        gn_pass2_kernel<false><<<grid, kThreads, smem_for(a, kPass2), s>>>(a);
    return cudaGetLastError();
}

cudaError_t fused_blocks_per_sm(bool silu, uint32_t smem, int *blocks)
{
    if (silu)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, gn_fused_kernel<true>, kThreads, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, gn_fused_kernel<false>, kThreads, smem);
}

cudaError_t launch_fused(const Args &a, int grid, bool silu, cudaStream_t s)
{
    Args copy = a;
    void *params[] = {&copy};
    const void *fn = silu ? reinterpret_cast<const void *>(gn_fused_kernel<true>)
                          : reinterpret_cast<const void *>(gn_fused_kernel<false>);
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), params, smem_for(a, kFused), s);
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

}  // namespace gn
