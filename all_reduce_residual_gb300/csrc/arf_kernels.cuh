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
    static __device__ __forceinline__ void widen(const uint4& v, float f[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
            float2 t = __half22float2(h);
            f[2 * j] = t.x;
            f[2 * j + 1] = t.y;
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

// acc[e] += f32(v[e]), one IEEE binary32 round-to-nearest add per element.
template <typename T>
__device__ __forceinline__ void accumulate(float acc[8], const uint4& v) {
    float f[8];
    Pack8<T>::widen(v, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
}

// Sum of the W partials at chunk c, in rank order, into acc (acc starts at
// +0.0f). WS > 0: W == WS is known at compile time and every load is issued
// before the first add. WS == 0: W is read at run time and handled in groups
// of 8 predicated loads.
template <typename T, int WS>
__device__ __forceinline__ void rank_sum(float acc[8], const uint4* const* s_ptr, int W, int64_t c) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    if constexpr (WS > 0) {
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

// Copy the W partial pointers of the device pointer array to shared memory.
__device__ __forceinline__ void load_pointers(const uint4** s_ptr, const void* const* partials, int W) {
    for (int i = threadIdx.x; i < W; i += blockDim.x) s_ptr[i] = static_cast<const uint4*>(partials[i]);
}

// ---------------------------------------------------------------------------
// kAllReduce: out = rn(sum_r P_r), flat over all M*H/8 chunks.
// ---------------------------------------------------------------------------
template <typename T, int WS, int U>
__global__ void __launch_bounds__(kMaxThreads) ar_flat_kernel(FlatParams p) {
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    load_pointers(s_ptr, p.partials, p.W);
    __syncthreads();

    const int64_t nthr = blockDim.x;
    const int64_t step = (int64_t)gridDim.x * nthr * U;
    for (int64_t base = (int64_t)blockIdx.x * nthr * U + threadIdx.x; base < p.nchunks; base += step) {
        if constexpr (WS > 0) {
            // all U*W loads first, then the adds
            uint4 v[U][WS];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = base + u * nthr;
                if (c < p.nchunks) {
#pragma unroll
                    for (int r = 0; r < WS; ++r) v[u][r] = ld_once(s_ptr[r] + c);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = base + u * nthr;
                if (c < p.nchunks) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                    for (int r = 0; r < WS; ++r) accumulate<T>(acc, v[u][r]);
                    st_out(p.out + c, Pack8<T>::narrow(acc));
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = base + u * nthr;
                if (c < p.nchunks) {
                    float acc[8];
                    rank_sum<T, 0>(acc, s_ptr, p.W, c);
                    st_out(p.out + c, Pack8<T>::narrow(acc));
                }
            }
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
// ---------------------------------------------------------------------------
template <typename T, int WS, int VPT>
__global__ void __launch_bounds__(kMaxThreads) rms_kernel(RmsParams p) {
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];  // per-warp partial sums, by row parity
    __shared__ float s_cta[2];                     // this CTA's partial, read by its peers

    load_pointers(s_ptr, p.partials, p.W);

    const int cs = p.cs;
    const int q = cs > 1 ? (int)cg::this_cluster().block_rank() : 0;
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t nclusters = gridDim.x / cs;
    const int c0 = q * p.slice;
    const int c1 = min(p.C, c0 + p.slice);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

    // gamma: the same chunks for every row this thread touches
    uint4 g[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int c = c0 + threadIdx.x + k * blockDim.x;
        if (c < c1) g[k] = ld_keep(p.gamma + c);
    }
    __syncthreads();

    int it = 0;
    for (int64_t row = cluster_id; row < p.M; row += nclusters, ++it) {
        const int64_t rbase = row * (int64_t)p.C;
        uint4 xs[VPT];  // rounded residual_out, kept for the normalisation pass
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int c = c0 + threadIdx.x + k * blockDim.x;
            if (c < c1) {
                float acc[8];
                const uint4 rv = ld_resid(p.residual + rbase + c);
                rank_sum<T, WS>(acc, s_ptr, p.W, rbase + c);
                float r[8];
                Pack8<T>::widen(rv, r);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], r[e]);
                xs[k] = Pack8<T>::narrow(acc);
                st_out(p.residual_out + rbase + c, xs[k]);
                float x[8];
                Pack8<T>::widen(xs[k], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
            }
        }

        // row sum of squares: butterfly in the warp, warps in index order,
        // then (cluster) CTAs in rank order; every thread ends with the same value
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_warp[it & 1][warp] = ss;
        __syncthreads();
        float tot = 0.0f;
        for (int w = 0; w < nwarps; ++w) tot += s_warp[it & 1][w];
        if (cs > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            if (threadIdx.x == 0) s_cta[it & 1] = tot;
            cluster.sync();
            tot = 0.0f;
            for (int r = 0; r < cs; ++r) tot += *cluster.map_shared_rank(&s_cta[it & 1], r);
        }
        const float inv = rsqrtf(tot / (float)p.H + p.eps);

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int c = c0 + threadIdx.x + k * blockDim.x;
            if (c < c1) {
                float x[8], gg[8], y[8];
                Pack8<T>::widen(xs[k], x);
                Pack8<T>::widen(g[k], gg);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), gg[e]);
                st_out(p.out + rbase + c, Pack8<T>::narrow(y));
            }
        }
    }
    // A peer may still be reading this CTA's s_cta: leave together.
    if (cs > 1) cg::this_cluster().sync();
}

// Writes the W partial pointers of a staging area laid out as W equal
// partials, `stride` bytes apart (host-buffer entry point).
__global__ void fill_pointer_array(const void** array, const char* first, int64_t stride, int W);

}  // namespace arf
