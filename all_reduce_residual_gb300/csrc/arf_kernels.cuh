// arf_kernels.cuh: sm_103a kernels of the all-reduce fusion epilogue.
//
// Both kernels stream the W partials once from HBM with 128-bit loads (one
// 16-byte chunk = 8 elements per load), sum them in binary32 in the order of
// the device pointer array, and round once to the I/O type. The work is
// HBM-bound (about 0.5 flop per byte), so there is no tensor-core path: the
// design goals are coalesced 16-byte accesses, many bytes in flight per SM,
// no re-reads, and grids sized from the SM count.
//
//  * ar_flat_kernel (kAllReduce): grid-stride over the M*H/8 chunks of the
//    output; each thread owns U chunks per loop trip and issues all U*W loads
//    before it adds.
//  * rms_kernel (kARResidualRMSNorm): a row of H elements is owned by one CTA
//    (cs == 1) or split over a cluster of cs CTAs. Each thread keeps its
//    rounded residual_out chunks in registers, so residual_out is never read
//    back; the row's sum of squares goes warp shuffle -> shared memory ->
//    (cluster) distributed shared memory, always in a fixed order.
//
// Pattern names follow tokenspeed PR #1075 "route generic MNNVL AR patterns
// to upstream flashinfer" (Summary); the device-side pointer array follows
// flashinfer PR #1321 "Optimizations for TRTLLM MNNVL Allreduce"
// (Description, "GPU array to pass the uc pointers"); vectorised loads
// follow the same page's Highlights (vectorised Lamport polling loads).
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "arf_internal.h"

namespace arf {

namespace cg = cooperative_groups;

// ---------------------------------------------------------------------------
// 8 x 16-bit values in one 128-bit vector <-> 8 binary32 values.
// Widening is exact; narrowing is round-to-nearest-even (cvt.rn).
// ---------------------------------------------------------------------------
template <typename T>
struct Pack8;

template <>
struct Pack8<__nv_bfloat16> {
    static __device__ __forceinline__ void widen(const uint4& v, float f[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // bf16 is the upper half of a binary32 encoding
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ uint4 narrow(const float f[8]) {
        uint4 v;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        return v;
    }
};

template <>
struct Pack8<__half> {
    // -0.0f + h with the sm_100 mixed-precision add: h is exactly
    // representable in binary32, so the sum is h itself (+0 stays +0, -0
    // stays -0); one FMA-pipe instruction instead of a conversion.
    static __device__ __forceinline__ float widen1(unsigned short h) {
        float f = -0.0f;
        asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(f) : "h"(h));
        return f;
    }
    static __device__ __forceinline__ void widen(const uint4& v, float f[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = widen1((unsigned short)(w[j] & 0xffffu));
            f[2 * j + 1] = widen1((unsigned short)(w[j] >> 16));
        }
    }
    static __device__ __forceinline__ uint4 narrow(const float f[8]) {
        uint4 v;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        return v;
    }
};

// ---------------------------------------------------------------------------
// Memory access. Partials are read exactly once: the read-only path without
// L1 allocation. gamma is re-read by every row: the default cached read-only
// load.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_once(const uint4* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// ld_once whose issue order the compiler keeps (volatile).
__device__ __forceinline__ uint4 ld_once_ordered(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The residual may be overwritten by this kernel (residual_out == residual):
// a coherent load, issued by the thread that later writes the same chunk.
__device__ __forceinline__ uint4 ld_resid(const uint4* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_keep(const uint4* p) { return __ldg(p); }

__device__ __forceinline__ void st_out(uint4* p, const uint4& v) { *p = v; }

// Chunk k (of VPT) of this thread within a run of blockDim.x*VPT chunks:
// every warp owns VPT*32 consecutive chunks, so each warp reads 512*VPT
// contiguous bytes of every rank's tensor (DRAM row locality), and each warp
// instruction still covers 32 consecutive 16-byte chunks (coalescing).
template <int VPT>
__device__ __forceinline__ int warp_run_chunk(int k) {
    return ((((int)threadIdx.x >> 5) * VPT + k) << 5) + ((int)threadIdx.x & 31);
}

// acc[e] += f32(v[e]): the 16-bit value widened exactly, then one IEEE
// binary32 round-to-nearest add. sm_100+ does both in one mixed-precision
// instruction (add.rn.f32.bf16 / add.rn.f32.f16: 16-bit operand, f32
// accumulator and result).
template <typename T>
struct MixedAdd;

template <>
struct MixedAdd<__nv_bfloat16> {
    static __device__ __forceinline__ float add(float acc, unsigned short h) {
        asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(acc) : "h"(h));
        return acc;
    }
};

template <>
struct MixedAdd<__half> {
    static __device__ __forceinline__ float add(float acc, unsigned short h) {
        asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(h));
        return acc;
    }
};

template <typename T>
__device__ __forceinline__ void accumulate(float acc[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[2 * j] = MixedAdd<T>::add(acc[2 * j], (unsigned short)(w[j] & 0xffffu));
        acc[2 * j + 1] = MixedAdd<T>::add(acc[2 * j + 1], (unsigned short)(w[j] >> 16));
    }
}

// acc[e] += binary32 partial values held as two 16-byte vectors (8 floats).
__device__ __forceinline__ void accumulate_f32(float acc[8], const uint4& a, const uint4& b) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], __uint_as_float(w[e]));
}

// Sum of the W partials at one chunk, in rank order, into acc (acc starts at
// +0.0f); c is the chunk's vector index in every partial. WS > 0: W == WS is
// known at compile time and every load is issued before the first add.
// WS == 0: W is read at run time and handled in groups of 8 predicated loads.
// F32P: binary32 partials, two vectors per chunk (c and c + 1), run-time W.
template <typename T, int WS, bool F32P = false>
__device__ __forceinline__ void rank_sum(float acc[8], const uint4* const* s_ptr, int W, int64_t c) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    if constexpr (F32P) {
        static_assert(WS == 0, "binary32 partials use the run-time rank count");
        for (int r0 = 0; r0 < W; r0 += 4) {
            uint4 v[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (r0 + j < W) {
                    v[j][0] = ld_once(s_ptr[r0 + j] + c);
                    v[j][1] = ld_once(s_ptr[r0 + j] + c + 1);
                }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (r0 + j < W) accumulate_f32(acc, v[j][0], v[j][1]);
        }
    } else if constexpr (WS > 0) {
        uint4 v[WS];
#pragma unroll
        for (int r = 0; r < WS; ++r) v[r] = ld_once(s_ptr[r] + c);
#pragma unroll
        for (int r = 0; r < WS; ++r) accumulate<T>(acc, v[r]);
    } else {
        for (int r0 = 0; r0 < W; r0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < W) v[j] = ld_once(s_ptr[r0 + j] + c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < W) accumulate<T>(acc, v[j]);
        }
    }
}

// Kernel prologue. As a programmatic dependent launch (lc.pdl), first let
// the next kernel in the stream begin launching, then wait until every
// earlier kernel has completed and its writes are visible: no global memory
// is touched before that wait, so the kernel is correct after any
// predecessor. Then copy the W partial pointers to shared memory, from the
// device pointer array or (by_value) from the launch parameters.
__device__ __forceinline__ void prologue(const uint4** s_ptr, const LaunchCommon& lc, int W) {
    if (lc.pdl) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    if (lc.by_value) {
        if (threadIdx.x == 0) {
#pragma unroll
            for (int i = 0; i < ARF_MAX_W; ++i)
                if (i < W) s_ptr[i] = static_cast<const uint4*>(lc.ptrs[i]);
        }
    } else {
        for (int i = threadIdx.x; i < W; i += blockDim.x) s_ptr[i] = static_cast<const uint4*>(lc.partials[i]);
    }
}

// ---------------------------------------------------------------------------
// kAllReduce: out = rn(sum_r P_r). Rows contiguous: one flat range of M*C
// chunks in tiles of nthr*U chunks. Strided rows: tiles never cross a row
// (tiles_per_row tiles per row; one division per tile).
// ---------------------------------------------------------------------------
template <typename T, int WS, int U, bool F32P>
__device__ __forceinline__ void flat_tile(const FlatParams& p, const uint4* const* s_ptr, int64_t row, int64_t col0,
                                          int64_t col_end) {
    // chunk col of row `row`: partial vector row*ldp + col (x2 for binary32),
    // output vector row*ldo + col
    const int64_t pbase = row * p.ly.ldp, obase = row * p.ly.ldo;
    if constexpr (WS > 0 && !F32P) {
        uint4 v[U][WS];
        if constexpr (WS >= 8 && U > 1) {
            // tensor by tensor, pinned in this order (volatile): a warp's U
            // pieces of one partial are requested back to back
#pragma unroll
            for (int r = 0; r < WS; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = col0 + u * 32;
                    if (c < col_end) v[u][r] = ld_once_ordered(s_ptr[r] + pbase + c);
                }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = col0 + u * 32;
                if (c < col_end) {
#pragma unroll
                    for (int r = 0; r < WS; ++r) v[u][r] = ld_once(s_ptr[r] + pbase + c);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = col0 + u * 32;
            if (c < col_end) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int r = 0; r < WS; ++r) accumulate<T>(acc, v[u][r]);
                st_out(p.out + obase + c, Pack8<T>::narrow(acc));
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = col0 + u * 32;
            if (c < col_end) {
                float acc[8];
                rank_sum<T, 0, F32P>(acc, s_ptr, p.W, pbase + (F32P ? 2 * c : c));
                st_out(p.out + obase + c, Pack8<T>::narrow(acc));
            }
        }
    }
}

template <typename T, int WS, int U, bool F32P = false>
__global__ void __launch_bounds__(kMaxThreads) ar_flat_kernel(FlatParams p) {
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    prologue(s_ptr, p.lc, p.W);
    __syncthreads();

    const int64_t tile = (int64_t)blockDim.x * U;
    if (!p.strided) {
        // the whole [M, C] range as one row (ldp = C or 2C, ldo = C)
        for (int64_t t0 = (int64_t)blockIdx.x * tile; t0 < p.nchunks; t0 += (int64_t)gridDim.x * tile)
            flat_tile<T, WS, U, F32P>(p, s_ptr, 0, t0 + warp_run_chunk<U>(0), p.nchunks);
    } else {
        const int64_t tiles_per_row = (p.C + tile - 1) / tile;
        const int64_t ntiles = tiles_per_row * p.M;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int64_t row = t / tiles_per_row;
            const int64_t col0 = (t - row * tiles_per_row) * tile;
            flat_tile<T, WS, U, F32P>(p, s_ptr, row, col0 + warp_run_chunk<U>(0), p.C);
        }
    }
}

// ---------------------------------------------------------------------------
// kARResidualRMSNorm: residual_out = rn(sum_r P_r + residual);
// out = rn((x * rsqrt(mean(x^2) + eps)) * gamma), x = residual_out.
// A cluster of p.cs CTAs owns one row at a time (p.cs == 1: a single CTA,
// launched without a cluster); CTA q of the cluster owns chunks
// [q*slice, min(C, (q+1)*slice)) of the row, and thread t of it the chunks
// q*slice + t + k*blockDim.x for k < VPT.
//
// Bytes in flight: with W known at compile time and VPT*(W+1) <= 18, a
// thread issues the loads of all its chunks of a row at once (one HBM round
// trip per row), and issues the next row's loads before the row's
// reduction barrier, so HBM stays busy while the CTA reduces and normalises.
// ---------------------------------------------------------------------------
template <int WS, int VPT>
struct RmsShape {
    static constexpr bool kPrefetch = rms_prefetches(WS, VPT);
    static constexpr bool kGammaRegs = VPT <= 2;  // else gamma is re-read from L1 per row
};

// Issue every load of one row for this thread: L[k][0..WS-1] = partials,
// L[k][WS] = residual. volatile keeps them where they are written (before
// the reduction barrier), which is the point of prefetching.
template <int WS, int VPT>
__device__ __forceinline__ void issue_row(uint4 (&L)[VPT][WS + 1], const uint4* const* s_ptr,
                                          const uint4* residual, int64_t pbase, int64_t rbase, int c0, int c1) {
    if constexpr (WS >= 8) {
        // Tensor by tensor (partials, then the residual): a warp's VPT pieces
        // of one tensor (32*VPT contiguous chunks) are requested back to back.
        // Measured on GB300 (W = 8, H = 7168): M = 1024 27.2 -> 26.7 us,
        // M = 2048 47.7 -> 45.9 us.
#pragma unroll
        for (int r = 0; r <= WS; ++r) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    const uint4* src = r == WS ? residual + rbase + c : s_ptr[r] + pbase + c;
                    if (r == WS)
                        asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(L[k][r].x), "=r"(L[k][r].y), "=r"(L[k][r].z), "=r"(L[k][r].w)
                                     : "l"(src));
                    else
                        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(L[k][r].x), "=r"(L[k][r].y), "=r"(L[k][r].z), "=r"(L[k][r].w)
                                     : "l"(src));
                }
            }
        }
    } else {
        // Fewer ranks: chunk by chunk, residual first (measured faster there:
        // W = 4, 80 MiB: 84.2 us, against 85.0 us tensor by tensor).
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int c = c0 + warp_run_chunk<VPT>(k);
            if (c < c1) {
                const uint4* rp = residual + rbase + c;
                asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(L[k][WS].x), "=r"(L[k][WS].y), "=r"(L[k][WS].z), "=r"(L[k][WS].w)
                             : "l"(rp));
#pragma unroll
                for (int r = 0; r < WS; ++r) {
                    const uint4* pp = s_ptr[r] + pbase + c;
                    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(L[k][r].x), "=r"(L[k][r].y), "=r"(L[k][r].z), "=r"(L[k][r].w)
                                 : "l"(pp));
                }
            }
        }
    }
}

// Largest cluster the row-split kernels are launched with.
constexpr int kMaxCluster = 16;

// Cluster barrier halves (PTX barrier.cluster). The kernels arrive once at
// the start (relaxed: it only tells the peers this CTA is running) and wait
// before their first access to a peer's shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// The CTA's part of a row statistic: butterfly in the warp, then the warps'
// sums in warp-index order (unrolled and predicated, so the shared-memory
// reads issue together; the additions keep their order). Every thread ends
// with the same value. Shared slots alternate with the row parity `it`.
__device__ __forceinline__ float cta_sum_squares(float ss, float (*s_warp)[kMaxThreads / 32], int it) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_warp[it & 1][warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kMaxThreads / 32; ++w)
        if (w < nwarps) tot += s_warp[it & 1][w];
    return tot;
}

// Row statistic over a cluster of cs CTAs; this CTA is rank q. Each CTA
// pushes its part into slot q of every CTA's s_cta (itself included: threads
// 0..cs-1 store one value each through distributed shared memory), one
// cluster barrier (release / acquire) makes the stores visible, and every
// CTA adds its own slots in CTA-rank order. Nobody reads a peer's shared
// memory, so a CTA may exit as soon as it is done. Slots alternate with the
// row parity: a CTA writes parity it & 1 again only after the next row's
// barrier, which every peer reaches after reading this row's slots.
// *wait_pending: this CTA still has to wait on its start arrival before the
// first store into a peer.
__device__ __forceinline__ float row_sum_squares(float ss, float (*s_warp)[kMaxThreads / 32],
                                                 float (*s_cta)[kMaxCluster], int cs, int q, int it,
                                                 bool* wait_pending) {
    float tot = cta_sum_squares(ss, s_warp, it);
    if (cs > 1) {
        if (*wait_pending) {
            cluster_wait();  // every peer is running
            *wait_pending = false;
        }
        cg::cluster_group cluster = cg::this_cluster();
        if ((int)threadIdx.x < cs) *cluster.map_shared_rank(&s_cta[it & 1][q], (int)threadIdx.x) = tot;
        cluster.sync();
        tot = 0.0f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
            if (r < cs) tot += s_cta[it & 1][r];
    }
    return tot;
}

// One chunk: t = sum_r P_r + residual (binary32, rank order, one rounding),
// store residual_out, return the rounded value, accumulate its squares.
template <typename T>
__device__ __forceinline__ uint4 residual_chunk(float acc[8], const uint4& rv, uint4* dst, float& ss) {
    accumulate<T>(acc, rv);
    const uint4 xs = Pack8<T>::narrow(acc);
    st_out(dst, xs);
    float x[8];
    Pack8<T>::widen(xs, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    return xs;
}

template <typename T>
__device__ __forceinline__ void normalise_chunk(const uint4& xs, const uint4& gv, float inv, uint4* dst) {
    float x[8], gg[8], y[8];
    Pack8<T>::widen(xs, x);
    Pack8<T>::widen(gv, gg);
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), gg[e]);
    st_out(dst, Pack8<T>::narrow(y));
}

template <typename T, int WS, int VPT, bool F32P = false, bool ONE_ROW = false>
__global__ void __launch_bounds__(kMaxThreads) rms_kernel(RmsParams p) {
    using Shape = RmsShape<WS, VPT>;
    static_assert(!F32P || WS == 0, "binary32 partials use the run-time rank count");
    static_assert(!ONE_ROW || Shape::kPrefetch, "the one-row form is the prefetching form without its row loop");
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];  // per-warp partial sums, by row parity
    __shared__ float s_cta[2][kMaxCluster];        // the cluster's CTA partials, by row parity

    prologue(s_ptr, p.lc, p.W);

    const int cs = p.cs;
    const int q = cs > 1 ? (int)cg::this_cluster().block_rank() : 0;
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t nclusters = gridDim.x / cs;
    const int c0 = q * p.slice;
    const int c1 = min(p.C, c0 + p.slice);

    uint4 g[Shape::kGammaRegs ? VPT : 1];
    if constexpr (Shape::kGammaRegs) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int c = c0 + warp_run_chunk<VPT>(k);
            if (c < c1) g[k] = ld_keep(p.gamma + c);
        }
    }
    __syncthreads();
    bool wait_pending = cs > 1;
    if (cs > 1) cluster_arrive_relaxed();

    if constexpr (ONE_ROW) {
        // Every cluster owns at most one row (grid >= rows): the same work as
        // the first trip of the prefetching loop below, without the loop and
        // the next-row prefetch (less code to fetch on a cold call).
        const int64_t row = cluster_id;
        if (row < p.M) {  // uniform over the cluster
            uint4 L[VPT][WS + 1];
            issue_row<WS, VPT>(L, s_ptr, p.residual, row * p.ly.ldp, row * p.ly.ldr, c0, c1);
            const int64_t ob = row * p.ly.ldo, rob = row * p.ly.ldro;
            uint4 xs[VPT];
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                    for (int r = 0; r < WS; ++r) accumulate<T>(acc, L[k][r]);
                    xs[k] = residual_chunk<T>(acc, L[k][WS], p.residual_out + rob + c, ss);
                }
            }
            const float inv = rsqrtf(row_sum_squares(ss, s_warp, s_cta, cs, q, 0, &wait_pending) / (float)p.H + p.eps);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    uint4 gv;
                    if constexpr (Shape::kGammaRegs) gv = g[k];
                    else gv = ld_keep(p.gamma + c);
                    normalise_chunk<T>(xs[k], gv, inv, p.out + ob + c);
                }
            }
        }
    } else if constexpr (Shape::kPrefetch) {
        uint4 L[VPT][WS + 1];
        int64_t row = cluster_id;
        if (row < p.M) issue_row<WS, VPT>(L, s_ptr, p.residual, row * p.ly.ldp, row * p.ly.ldr, c0, c1);
        for (int it = 0; row < p.M; row += nclusters, ++it) {
            const int64_t ob = row * p.ly.ldo, rob = row * p.ly.ldro;
            uint4 xs[VPT];
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                    for (int r = 0; r < WS; ++r) accumulate<T>(acc, L[k][r]);
                    xs[k] = residual_chunk<T>(acc, L[k][WS], p.residual_out + rob + c, ss);
                }
            }
            const int64_t next = row + nclusters;
            if (next < p.M) issue_row<WS, VPT>(L, s_ptr, p.residual, next * p.ly.ldp, next * p.ly.ldr, c0, c1);
            const float inv = rsqrtf(row_sum_squares(ss, s_warp, s_cta, cs, q, it, &wait_pending) / (float)p.H + p.eps);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    uint4 gv;
                    if constexpr (Shape::kGammaRegs) gv = g[k];
                    else gv = ld_keep(p.gamma + c);
                    normalise_chunk<T>(xs[k], gv, inv, p.out + ob + c);
                }
            }
        }
    } else {
        int it = 0;
        for (int64_t row = cluster_id; row < p.M; row += nclusters, ++it) {
            const int64_t pb = row * p.ly.ldp, rb = row * p.ly.ldr, ob = row * p.ly.ldo, rob = row * p.ly.ldro;
            uint4 xs[VPT];
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    float acc[8];
                    const uint4 rv = ld_resid(p.residual + rb + c);
                    rank_sum<T, WS, F32P>(acc, s_ptr, p.W, pb + (F32P ? 2 * (int64_t)c : (int64_t)c));
                    xs[k] = residual_chunk<T>(acc, rv, p.residual_out + rob + c, ss);
                }
            }
            const float inv = rsqrtf(row_sum_squares(ss, s_warp, s_cta, cs, q, it, &wait_pending) / (float)p.H + p.eps);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int c = c0 + warp_run_chunk<VPT>(k);
                if (c < c1) {
                    uint4 gv;
                    if constexpr (Shape::kGammaRegs) gv = g[k];
                    else gv = ld_keep(p.gamma + c);
                    normalise_chunk<T>(xs[k], gv, inv, p.out + ob + c);
                }
            }
        }
    }
    // A cluster without rows never waited on its start arrival: complete
    // that barrier phase before leaving.
    if (wait_pending) cluster_wait();
}

// ---------------------------------------------------------------------------
// kARResidualRMSNorm, streaming form (ARF_PATH_ASYNC). One CTA of
// kAsyncThreads threads per SM walks its rows (blockIdx.x + i*gridDim.x) in
// column blocks of kAsyncThreads chunks; thread t owns chunk t of every block.
// For the work item `stages-1` items ahead, each thread copies its chunk's
// W+1 vectors (partials, residual) into its own slots of a shared-memory ring
// with cp.async (16 bytes, cached in L2 only). Copies therefore stay in
// flight across row boundaries and barriers without holding registers, which
// lets wide rank counts (W = 16) keep as many bytes in flight as narrow ones.
// A thread reads only the slots it filled, so the hardware wait on its own
// copy groups (cp.async.wait_group) is all the data synchronisation there is.
// The rounded residual_out of the row stays in shared memory (same thread
// reads it back) until the row's statistic is known.
// ---------------------------------------------------------------------------
constexpr int kAsyncThreads = kAsyncCtaThreads;

__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* gptr) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gptr) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most n of this thread's most recent copy groups are pending
// (n >= 7 waits down to 7, which is stricter and still correct).
__device__ __forceinline__ void cp_async_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

template <typename T, int WS>
__global__ void __launch_bounds__(kAsyncThreads, 1) rms_async_kernel(RmsParams p) {
    static_assert(WS > 0, "the streaming kernel needs the rank count at compile time");
    extern __shared__ __align__(16) uint4 dyn_smem[];
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];

    prologue(s_ptr, p.lc, p.W);
    __syncthreads();

    const int S = p.stages;
    const int C = p.C;
    const int tid = threadIdx.x;
    const int nb = (C + kAsyncThreads - 1) / kAsyncThreads;
    uint4* ring = dyn_smem;                                           // [S][WS+1][kAsyncThreads]
    uint4* xrow = dyn_smem + (size_t)S * (WS + 1) * kAsyncThreads;    // [C]
    const uint32_t ring_addr = (uint32_t)__cvta_generic_to_shared(ring);
    constexpr uint32_t kRankStride = kAsyncThreads * 16;              // bytes between ranks in a slot
    constexpr uint32_t kSlotStride = (WS + 1) * kRankStride;          // bytes between ring slots

    // The producer side walks work items (row, column block) `S-1` ahead of
    // the consumer side; both advance (row, block, slot) by counting, no
    // division. Every item commits one copy group (empty past the last row),
    // so "at most S-1 groups pending" always means "my oldest item landed".
    int64_t in_row = blockIdx.x;
    int in_b = 0, in_slot = 0;
    auto issue_next = [&]() {
        if (in_row < p.M) {
            const int c = in_b * kAsyncThreads + tid;
            if (c < C) {
                const int64_t poff = in_row * p.ly.ldp + c, roff = in_row * p.ly.ldr + c;
                const uint32_t slot = ring_addr + (uint32_t)in_slot * kSlotStride + (uint32_t)tid * 16u;
#pragma unroll
                for (int r = 0; r < WS; ++r) cp_async16(slot + r * kRankStride, s_ptr[r] + poff);
                cp_async16(slot + WS * kRankStride, p.residual + roff);
            }
            if (++in_b == nb) {
                in_b = 0;
                in_row += gridDim.x;
            }
            if (++in_slot == S) in_slot = 0;
        }
        cp_async_commit();
    };

    for (int j = 0; j < S - 1; ++j) issue_next();
    int slot_i = 0, it = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) {
        const int64_t ob = row * p.ly.ldo, rob = row * p.ly.ldro;
        float ss = 0.0f;
        for (int b = 0; b < nb; ++b) {
            issue_next();
            cp_async_wait(S - 1);  // this item has landed in this thread's slots
            const int c = b * kAsyncThreads + tid;
            if (c < C) {
                const uint4* slot = ring + (size_t)slot_i * (WS + 1) * kAsyncThreads + tid;
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int r = 0; r < WS; ++r) accumulate<T>(acc, slot[r * kAsyncThreads]);
                xrow[c] = residual_chunk<T>(acc, slot[WS * kAsyncThreads], p.residual_out + rob + c, ss);
            }
            if (++slot_i == S) slot_i = 0;
        }
        // the row is complete: normalise it
        const float inv = rsqrtf(cta_sum_squares(ss, s_warp, it) / (float)p.H + p.eps);
        for (int b = 0; b < nb; ++b) {
            const int c = b * kAsyncThreads + tid;
            if (c < C) normalise_chunk<T>(xrow[c], ld_keep(p.gamma + c), inv, p.out + ob + c);
        }
    }
    cp_async_wait(0);  // only empty groups can remain; leave with nothing in flight
}

// Writes the W partial pointers of a staging area laid out as W equal
// partials, `stride` bytes apart (host-buffer entry point).
__global__ void fill_pointer_array(const void** array, const char* first, int64_t stride, int W);

}  // namespace arf
