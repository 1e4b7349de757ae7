// arf_elem.cuh: elementwise kernels for layouts the 16-byte kernels cannot
// take: H not a multiple of 8, row strides not a multiple of 8 elements, or
// residual / gamma / outputs not 16-byte aligned (2-byte alignment suffices;
// binary32 partials need 4). One element per thread per step where the
// rows of the tensors start at different offsets within a 16-byte vector,
// else 16-byte vectors with per-row heads and tails; the same
// arithmetic as the vector kernels: binary32 rank-order sum with one
// round-to-nearest add per rank, the residual added to the unrounded sum,
// one rounding, the statistic of the stored residual_out.
#pragma once

#include "arf_kernels.cuh"

namespace arf {

template <typename T>
__device__ __forceinline__ float widen1(unsigned short h);
template <>
__device__ __forceinline__ float widen1<__nv_bfloat16>(unsigned short h) {
    return __uint_as_float((uint32_t)h << 16);
}
template <>
__device__ __forceinline__ float widen1<__half>(unsigned short h) {
    return __half2float(__ushort_as_half(h));
}

template <typename T>
__device__ __forceinline__ unsigned short narrow1(float f);
template <>
__device__ __forceinline__ unsigned short narrow1<__nv_bfloat16>(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <>
__device__ __forceinline__ unsigned short narrow1<__half>(float f) {
    return __half_as_ushort(__float2half_rn(f));
}

// Rank-order binary32 sum of element i of every partial (acc from +0.0f).
template <typename T, bool F32P>
__device__ __forceinline__ float elem_rank_sum(const uint4* const* s_ptr, int W, int64_t i) {
    float acc = 0.0f;
    if constexpr (F32P) {
        for (int r = 0; r < W; ++r) acc = __fadd_rn(acc, reinterpret_cast<const float*>(s_ptr[r])[i]);
    } else {
        for (int r = 0; r < W; ++r)
            acc = MixedAdd<T>::add(acc, reinterpret_cast<const unsigned short*>(s_ptr[r])[i]);
    }
    return acc;
}

// elem_rank_sum for the vector forms' head and tail elements: with W == WS
// compiled in, every partial's load is issued before the first add (the
// run-time loop waits out one load latency per rank).
template <typename T, int WS>
__device__ __forceinline__ float elem_rank_sum_w(const uint4* const* s_ptr, int W, int64_t i) {
    if constexpr (WS > 0) {
        unsigned short v[WS];
#pragma unroll
        for (int r = 0; r < WS; ++r) v[r] = reinterpret_cast<const unsigned short*>(s_ptr[r])[i];
        float acc = 0.0f;
#pragma unroll
        for (int r = 0; r < WS; ++r) acc = MixedAdd<T>::add(acc, v[r]);
        return acc;
    } else {
        return elem_rank_sum<T, false>(s_ptr, W, i);
    }
}

// The split of one row into 16-byte vectors. All tensors of the call start
// row r at the same offset modulo 8 elements (flat_ok != 0), so one split
// serves them all: nh head elements up to the first 16-byte boundary, nb
// whole chunks, nt tail elements (nh, nt < 8).
struct RowSplit {
    int nh, nb, nt;
};
__device__ __forceinline__ RowSplit row_split(int64_t first_elem, int H) {
    RowSplit r;
    r.nh = (int)((8 - (first_elem & 7)) & 7);
    if (r.nh > H) r.nh = H;
    r.nb = (H - r.nh) / 8;
    r.nt = H - r.nh - 8 * r.nb;
    return r;
}

// Whether the vector forms apply: the host's layout verdict, and every
// partial pointer 16-byte aligned (the same answer in every thread).
__device__ __forceinline__ bool vector_layout(const ElemParams& p, const uint4* const* s_ptr) {
    bool vec = p.flat_ok != 0;
    for (int r = 0; r < p.W && vec; ++r) vec = (reinterpret_cast<uintptr_t>(s_ptr[r]) & 15u) == 0;
    return vec;
}

// The vector forms' chunks per trip: two where the rank count is compiled in
// (WS > 0) and a thread's loads for both fit the 64-register budget without
// spilling (kAllReduce up to 8 vectors, W <= 4; kARResidualRMSNorm, which
// also holds the residual, up to 6, W <= 2), else one.
template <int WS, bool RMS>
__host__ __device__ constexpr int elem_chunks_per_trip() {
    return WS > 0 && 2 * (WS + (RMS ? 1 : 0)) <= (RMS ? 6 : 8) ? 2 : 1;
}

// acc[q] = the rank-order sum of the partials at chunk c[q], for each q < K
// with ok[q]. WS > 0 (W == WS): every load of the K chunks is issued before
// the first add; WS == 0: rank_sum's groups of run-time ranks, chunk by chunk.
template <typename T, int WS, int K>
__device__ __forceinline__ void rank_sum_chunks(float (&acc)[K][8], const uint4* const* s_ptr, int W,
                                                const int64_t (&c)[K], const bool (&ok)[K]) {
    if constexpr (WS > 0) {
        uint4 v[K][WS];
#pragma unroll
        for (int q = 0; q < K; ++q)
#pragma unroll
            for (int r = 0; r < WS; ++r)
                if (ok[q]) v[q][r] = ld_once(s_ptr[r] + c[q]);
#pragma unroll
        for (int q = 0; q < K; ++q) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[q][e] = 0.0f;
#pragma unroll
            for (int r = 0; r < WS; ++r)
                if (ok[q]) accumulate<T>(acc[q], v[q][r]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < K; ++q)
            if (ok[q]) rank_sum<T, 0, false>(acc[q], s_ptr, W, c[q]);
    }
}

// kAllReduce: tiles of blockDim.x elements, never crossing a row.
// Tensors whose rows share their 16-byte phase (flat_ok, partial pointers
// aligned) take 16-byte vectors: contiguous ones as one flat range of M*H
// elements (vectors over the first (M*H)/8 chunks, then the last (M*H)%8
// elements one by one), strided ones a row per CTA (rows grid-stride; the
// head and tail elements of a row one per thread, its whole chunks as
// vectors). The arithmetic is the same in every form (rank-order
// mixed-precision adds, one rounding per element). WS > 0: W == WS compiled
// in for the vector forms. At most 64 registers, so that 256-thread CTAs fit
// four to an SM.
template <typename T, bool F32P, int WS = 0>
__global__ void __launch_bounds__(kMaxThreads, 2) ar_elem_kernel(ElemParams p) {
    static_assert(!F32P || WS == 0, "binary32 partials use the run-time rank count");
    constexpr int K = elem_chunks_per_trip<WS, false>();
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    prologue(s_ptr, p.lc, p.W);
    __syncthreads();
    if constexpr (!F32P) {
        if (vector_layout(p, s_ptr) && p.flat_ok == 1) {
            const int64_t total = p.M * (int64_t)p.H, nch = total / 8;
            const int64_t stride = (int64_t)gridDim.x * blockDim.x;
            const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
            uint4* out16 = reinterpret_cast<uint4*>(p.out);
            for (int64_t c0 = first; c0 < nch; c0 += K * stride) {
                int64_t c[K];
                bool ok[K];
#pragma unroll
                for (int q = 0; q < K; ++q) {
                    c[q] = c0 + q * stride;
                    ok[q] = c[q] < nch;
                }
                float acc[K][8];
                rank_sum_chunks<T, WS, K>(acc, s_ptr, p.W, c, ok);
#pragma unroll
                for (int q = 0; q < K; ++q)
                    if (ok[q]) st_out(out16 + c[q], Pack8<T>::narrow(acc[q]));
            }
            for (int64_t e = nch * 8 + first; e < total; e += stride)
                p.out[e] = narrow1<T>(elem_rank_sum_w<T, WS>(s_ptr, p.W, e));
            return;
        }
        if (vector_layout(p, s_ptr)) {
            const int B = blockDim.x, tid = threadIdx.x;  // B >= 32 > nh + nt
            uint4* out16 = reinterpret_cast<uint4*>(p.out);
            for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
                const int64_t op = row * p.ldp, oo = row * p.ldo;
                const RowSplit sp = row_split(op, p.H);
                const int k = tid < sp.nh ? tid : (tid >= B - sp.nt ? sp.nh + 8 * sp.nb + (tid - (B - sp.nt)) : -1);
                if (k >= 0) p.out[oo + k] = narrow1<T>(elem_rank_sum_w<T, WS>(s_ptr, p.W, op + k));
                const int64_t cp = (op + sp.nh) / 8, co = (oo + sp.nh) / 8;
                for (int j0 = tid; j0 < sp.nb; j0 += K * B) {
                    int64_t c[K];
                    bool ok[K];
#pragma unroll
                    for (int q = 0; q < K; ++q) {
                        c[q] = cp + j0 + q * B;
                        ok[q] = j0 + q * B < sp.nb;
                    }
                    float acc[K][8];
                    rank_sum_chunks<T, WS, K>(acc, s_ptr, p.W, c, ok);
#pragma unroll
                    for (int q = 0; q < K; ++q)
                        if (ok[q]) st_out(out16 + co + j0 + q * B, Pack8<T>::narrow(acc[q]));
                }
            }
            return;
        }
    }
    const int64_t per_row = (p.H + blockDim.x - 1) / blockDim.x;
    const int64_t ntiles = per_row * p.M;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t row = t / per_row;
        const int64_t e = (t - row * per_row) * blockDim.x + threadIdx.x;
        if (e < p.H) {
            const float acc = elem_rank_sum<T, F32P>(s_ptr, p.W, row * p.ldp + e);
            p.out[row * p.ldo + e] = narrow1<T>(acc);
        }
    }
}

// One row of kARResidualRMSNorm on tensors whose rows share their 16-byte
// phase (flat_ok, partials checked by the caller): the row splits into a
// head of fewer than 8 elements up to the first 16-byte boundary (threads
// 0..), whole 16-byte chunks, and a tail of fewer than 8 elements (the last
// threads), at each tensor's own row offset. gamma is indexed from the row
// start and read from L1, as 16-byte vectors where the row's chunks start
// on a 16-byte boundary of an aligned gamma, else element by element. Same
// arithmetic as the elementwise rows; residual_out is re-read in the second
// pass by the thread that wrote it. WS > 0: W == WS compiled in.
template <typename T, int WS>
__device__ __forceinline__ void rms_flat_row(const ElemParams& p, const uint4* const* s_ptr, int64_t row, int it,
                                             float (*s_warp)[kMaxThreads / 32]) {
    constexpr int K = elem_chunks_per_trip<WS, true>();
    const int64_t op = row * p.ldp, orr = row * p.ldr, oro = row * p.ldro, oo = row * p.ldo;
    const RowSplit sp = row_split(op, p.H);
    const int B = blockDim.x, tid = threadIdx.x;  // B >= 32 > nh + nt
    const int k = tid < sp.nh ? tid : (tid >= B - sp.nt ? sp.nh + 8 * sp.nb + (tid - (B - sp.nt)) : -1);
    // chunk j of the row in each tensor, as a 16-byte index
    const int64_t cp = (op + sp.nh) / 8, cr = (orr + sp.nh) / 8, cro = (oro + sp.nh) / 8, co = (oo + sp.nh) / 8;
    const uint4* res16 = reinterpret_cast<const uint4*>(p.residual);
    uint4* ro16 = reinterpret_cast<uint4*>(p.residual_out);
    uint4* out16 = reinterpret_cast<uint4*>(p.out);
    float ss = 0.0f;
    if (k >= 0) {
        const unsigned short rk = p.residual[orr + k];  // read before residual_out (maybe the same) is written
        float acc = elem_rank_sum_w<T, WS>(s_ptr, p.W, op + k);
        acc = MixedAdd<T>::add(acc, rk);
        const unsigned short xs = narrow1<T>(acc);
        p.residual_out[oro + k] = xs;
        const float x = widen1<T>(xs);
        ss = fmaf(x, x, ss);
    }
    for (int j0 = tid; j0 < sp.nb; j0 += K * B) {
        int64_t c[K];
        bool ok[K];
        uint4 rv[K];
#pragma unroll
        for (int q = 0; q < K; ++q) {
            c[q] = cp + j0 + q * B;
            ok[q] = j0 + q * B < sp.nb;
            if (ok[q]) rv[q] = ld_resid(res16 + cr + j0 + q * B);
        }
        float acc[K][8];
        rank_sum_chunks<T, WS, K>(acc, s_ptr, p.W, c, ok);
#pragma unroll
        for (int q = 0; q < K; ++q)
            if (ok[q]) (void)residual_chunk<T>(acc[q], rv[q], ro16 + cro + j0 + q * B, ss);
    }
    const float inv = rsqrtf(cta_sum_squares(ss, s_warp, it) / (float)p.H + p.eps);
    if (k >= 0) {
        const float x = widen1<T>(p.residual_out[oro + k]);
        const float g = widen1<T>(p.gamma[k]);
        p.out[oo + k] = narrow1<T>(__fmul_rn(__fmul_rn(x, inv), g));
    }
    // Second pass: gamma is one 16-byte load where the row's chunks start on
    // a 16-byte boundary of an aligned gamma, else eight element loads.
    const bool g_vec = sp.nh == 0 && (reinterpret_cast<uintptr_t>(p.gamma) & 15u) == 0;
    const uint4* g16 = reinterpret_cast<const uint4*>(p.gamma);
    for (int j = tid; j < sp.nb; j += B) {
        uint4 gv;
        if (g_vec) {
            gv = ld_keep(g16 + j);
        } else {
            const unsigned short* gp = p.gamma + sp.nh + 8 * j;
            gv.x = (uint32_t)__ldg(gp + 0) | ((uint32_t)__ldg(gp + 1) << 16);
            gv.y = (uint32_t)__ldg(gp + 2) | ((uint32_t)__ldg(gp + 3) << 16);
            gv.z = (uint32_t)__ldg(gp + 4) | ((uint32_t)__ldg(gp + 5) << 16);
            gv.w = (uint32_t)__ldg(gp + 6) | ((uint32_t)__ldg(gp + 7) << 16);
        }
        normalise_chunk<T>(ro16[cro + j], gv, inv, out16 + co + j);
    }
}

// kARResidualRMSNorm: one CTA per row (rows grid-stride). The rounded
// residual_out goes to memory in the first pass and is read back in the
// second by the thread that wrote it. Tensors whose rows share their
// 16-byte phase (flat_ok, and every partial pointer aligned) take
// rms_flat_row instead.
template <typename T, bool F32P, int WS = 0>
__global__ void __launch_bounds__(kMaxThreads, 2) rms_elem_kernel(ElemParams p) {
    static_assert(!F32P || WS == 0, "binary32 partials use the run-time rank count");
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];
    prologue(s_ptr, p.lc, p.W);
    __syncthreads();
    if constexpr (!F32P) {
        if (vector_layout(p, s_ptr)) {  // the same answer in every thread of every CTA
            int it = 0;
            for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) rms_flat_row<T, WS>(p, s_ptr, row, it, s_warp);
            return;
        }
    }
    int it = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) {
        float ss = 0.0f;
        for (int64_t e = threadIdx.x; e < p.H; e += blockDim.x) {
            float acc = elem_rank_sum<T, F32P>(s_ptr, p.W, row * p.ldp + e);
            acc = MixedAdd<T>::add(acc, p.residual[row * p.ldr + e]);
            const unsigned short xs = narrow1<T>(acc);
            p.residual_out[row * p.ldro + e] = xs;
            const float x = widen1<T>(xs);
            ss = fmaf(x, x, ss);
        }
        const float inv = rsqrtf(cta_sum_squares(ss, s_warp, it) / (float)p.H + p.eps);
        for (int64_t e = threadIdx.x; e < p.H; e += blockDim.x) {
            const float x = widen1<T>(p.residual_out[row * p.ldro + e]);
            const float g = widen1<T>(p.gamma[e]);
            p.out[row * p.ldo + e] = narrow1<T>(__fmul_rn(__fmul_rn(x, inv), g));
        }
    }
}

}  // namespace arf
