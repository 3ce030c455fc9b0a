// rga_kernels.cu -- sm_103a kernel of the residual-gate update
//
//     y = residual + gate * update        (residual, update, y: [rows][D]
//                                          half precision; gate: one [D] row)
//
// bit for bit equal to the eager evaluation of the prhub digest of sglang PR
// #33823 (FLUX.2 bit-exact residual-gate fusion, sections "Functions and
// motivation" and "Implementation breakdown", items 1-3): the product is
// its own half-precision tensor, then added to the residual, each step
// rounded once to the half format (round to nearest even).
//
// The product and the sum are the packed half instructions mul.rn and
// add.rn on bf16x2 / f16x2, which round the exact result once.  That is the
// eager result: the fp32 product of two half values is exact, and the fp32
// rounding of the sum before its rounding to half never changes the half
// value (the operands carry 8 or 11 significant bits, so the exact sum
// needs more than 24 bits only when the smaller operand lies far below the
// half format's rounding midpoints).  The two instructions are kept
// separate (an fma would round once instead of twice).
//
// The work is pure streaming (6 bytes per element against HBM): each thread
// takes 16-byte vectors v, v + stride, ... with four vectors in flight per
// iteration; residual and update are read with streaming (evict-first)
// loads, the gate row through the read-only path (it stays in L1).
#include <cstdint>

#include "gn_internal.h"

namespace gn {

template <bool BF16>
__device__ __forceinline__ uint32_t rga_pair(uint32_t r, uint32_t u, uint32_t g)
{
    uint32_t p, y;
    if (BF16) {
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p) : "r"(g), "r"(u));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(r), "r"(p));
    } else {
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(g), "r"(u));
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(r), "r"(p));
    }
    return y;
}

template <bool BF16>
__device__ __forceinline__ uint4 rga_vec(const uint4 &r, const uint4 &u, const uint4 &g)
{
    return make_uint4(rga_pair<BF16>(r.x, u.x, g.x), rga_pair<BF16>(r.y, u.y, g.y), rga_pair<BF16>(r.z, u.z, g.z),
                      rga_pair<BF16>(r.w, u.w, g.w));
}

// Programmatic dependent launch (see launch_residual_gate).
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// streaming load (cache-streaming: evict-first; every element is read once)
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }

// nvec = rows * V vectors of 8 elements, V = D / 8 per row.  `col` is the
// column vector of a thread's current vector, advanced by stride % V.
template <bool BF16>
__global__ void __launch_bounds__(kRgaThreads) rga_kernel(const uint4 *__restrict__ res,
                                                           const uint4 *__restrict__ upd,
                                                           const uint4 *__restrict__ gate, uint4 *out,
                                                           int64_t nvec, int V)
{
    griddep_wait();   // residual, update and gate may come from the kernel ahead in the stream
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int step = static_cast<int>(stride % V);
    int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    int col = static_cast<int>(v % V);
    auto advance = [&](int c) {
        c += step;
        return c >= V ? c - V : c;
    };
    for (; v + 3 * stride < nvec; v += 4 * stride) {
        int c[4];
        c[0] = col;
        c[1] = advance(c[0]);
        c[2] = advance(c[1]);
        c[3] = advance(c[2]);
        uint4 r[4], u[4], g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r[k] = ld_stream(res + v + k * stride);
            u[k] = ld_stream(upd + v + k * stride);
            g[k] = __ldg(gate + c[k]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) out[v + k * stride] = rga_vec<BF16>(r[k], u[k], g[k]);
        col = advance(c[3]);
    }
    for (; v < nvec; v += stride) {
        out[v] = rga_vec<BF16>(ld_stream(res + v), ld_stream(upd + v), __ldg(gate + col));
        col = advance(col);
    }
}

cudaError_t launch_residual_gate(const void *residual, const void *update, const void *gate, void *out,
                                 int64_t rows, int64_t D, bool bf16, int blocks, cudaStream_t s)
{
    const int64_t nvec = rows * (D / 8);
    const int V = static_cast<int>(D / 8);
    const auto *r = static_cast<const uint4 *>(residual);
    const auto *u = static_cast<const uint4 *>(update);
    const auto *g = static_cast<const uint4 *>(gate);
    auto *y = static_cast<uint4 *>(out);
    // launched with programmatic stream serialization: the blocks may start
    // while the kernel ahead in the stream finishes, and wait for it before
    // their first access to global memory; a kernel launched after this one
    // the same way may start once every block of this one has waited
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kRgaThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return bf16 ? cudaLaunchKernelEx(&cfg, rga_kernel<true>, r, u, g, y, nvec, V)
                : cudaLaunchKernelEx(&cfg, rga_kernel<false>, r, u, g, y, nvec, V);
}

}  // namespace gn
