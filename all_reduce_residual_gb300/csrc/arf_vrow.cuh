// arf_vrow.cuh: kARResidualRMSNorm on rows that do not start on 16-byte
// boundaries (H % 8 != 0, or row strides that are not multiples of 8), when
// every tensor's row r starts at the same offset within a 16-byte vector and
// every tensor is 16-byte aligned (the elementwise kernels' vector layout).
//
// The row kernel's design, on such rows: a CTA owns a row, every thread
// holds its NV vectors of it in registers, issues all their loads at once,
// and issues the next row's loads before the row's reduction barrier. The row
// covers nvec = ceil((phase + H) / 8) aligned vectors, phase = the row's
// offset within its first vector. Interior vectors are one 16-byte load or
// store; the first and last vectors, which hold elements of the neighbouring
// rows, are loaded and stored element by element for the row's own lanes.
// gamma is staged once per CTA in shared memory with eight zero elements on
// either side, so the eight gamma values of any vector, at any phase, are a
// funnel shift of two aligned 16-byte shared-memory loads. Same arithmetic as
// every other kernel: rank-order binary32 sum of the 16-bit partials, the
// residual added to the unrounded sum, one rounding, the statistic of the
// stored residual_out, out = rn((x * inv) * gamma).
#pragma once

#include "arf_elem.cuh"

namespace arf {

// Row r's geometry: its phase within a 16-byte vector and the vectors it
// spans; vector j covers row elements [8j - phase, 8j - phase + 8).
struct VRow {
    int phase;
    int nvec;
    __device__ __forceinline__ bool lane_in(int j, int e, int H) const {
        const int i = 8 * j + e - phase;
        return i >= 0 && i < H;
    }
    // whether vector j holds elements outside the row
    __device__ __forceinline__ bool edge(int j, int H) const {
        return (j == 0 && phase > 0) || 8 * j + 8 - phase > H;
    }
};

__device__ __forceinline__ VRow vrow_of(int64_t row, int64_t ldp, int H) {
    VRow v;
    v.phase = (int)((row * ldp) & 7);
    v.nvec = (v.phase + H + 7) >> 3;
    return v;
}

// The in-row lanes of vector j of a row starting at element `row0` (others 0).
__device__ __forceinline__ uint4 ld_edge(const unsigned short* t, int64_t row0, const VRow& g, int j, int H) {
    unsigned short h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = g.lane_in(j, e, H) ? t[row0 + 8 * j + e - g.phase] : (unsigned short)0;
    uint4 v;
    v.x = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
    v.y = (uint32_t)h[2] | ((uint32_t)h[3] << 16);
    v.z = (uint32_t)h[4] | ((uint32_t)h[5] << 16);
    v.w = (uint32_t)h[6] | ((uint32_t)h[7] << 16);
    return v;
}

__device__ __forceinline__ void st_edge(unsigned short* t, int64_t row0, const VRow& g, int j, int H, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (g.lane_in(j, e, H)) t[row0 + 8 * j + e - g.phase] = (unsigned short)(w[e >> 1] >> (16 * (e & 1)));
}

// Elements [8 - sh, 16 - sh) of the 16 elements a then b (0 <= sh < 8).
__device__ __forceinline__ uint4 shift_in(const uint4& a, const uint4& b, int sh) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t r[4];
    switch (sh) {  // uniform over the CTA (one row's phase)
#define ARF_VROW_EVEN(S)                                       \
    case S:                                                    \
        _Pragma("unroll") for (int i = 0; i < 4; ++i) r[i] = w[(8 - S) / 2 + i]; \
        break;
#define ARF_VROW_ODD(S)                                                                   \
    case S:                                                                               \
        _Pragma("unroll") for (int i = 0; i < 4; ++i) r[i] =                              \
            __funnelshift_r(w[(8 - S - 1) / 2 + i], w[(8 - S + 1) / 2 + i], 16);          \
        break;
        ARF_VROW_EVEN(0)
        ARF_VROW_ODD(1)
        ARF_VROW_EVEN(2)
        ARF_VROW_ODD(3)
        ARF_VROW_EVEN(4)
        ARF_VROW_ODD(5)
        ARF_VROW_EVEN(6)
        default:
        ARF_VROW_ODD(7)
#undef ARF_VROW_EVEN
#undef ARF_VROW_ODD
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Issue every load of one row for this thread: L[k][0..WS-1] = partials,
// L[k][WS] = residual, for its vectors j = warp_run_chunk<NV>(k) < nvec.
template <int WS, int NV>
__device__ __forceinline__ void vrow_issue(uint4 (&L)[NV][WS + 1], const ElemParams& p, const uint4* const* s_ptr,
                                           int64_t row, const VRow& g) {
    const int64_t p0 = row * p.ldp, r0 = row * p.ldr;
    const int64_t vp = (p0 - g.phase) >> 3, vr = (r0 - g.phase) >> 3;  // first vector of the row
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int j = warp_run_chunk<NV>(k);
        if (j < g.nvec) {
            if (g.edge(j, p.H)) {
#pragma unroll
                for (int r = 0; r < WS; ++r)
                    L[k][r] = ld_edge(reinterpret_cast<const unsigned short*>(s_ptr[r]), p0, g, j, p.H);
                L[k][WS] = ld_edge(p.residual, r0, g, j, p.H);
            } else {
                // residual first (the thread that reads it writes residual_out there)
                asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(L[k][WS].x), "=r"(L[k][WS].y), "=r"(L[k][WS].z), "=r"(L[k][WS].w)
                             : "l"(reinterpret_cast<const uint4*>(p.residual) + vr + j));
#pragma unroll
                for (int r = 0; r < WS; ++r)
                    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(L[k][r].x), "=r"(L[k][r].y), "=r"(L[k][r].z), "=r"(L[k][r].w)
                                 : "l"(s_ptr[r] + vp + j));
            }
        }
    }
}

template <typename T, int WS, int NV>
__global__ void __launch_bounds__(kMaxThreads) rms_vrow_kernel(ElemParams p) {
    static_assert(vrow_compiled(WS, NV), "no such instance");
    extern __shared__ __align__(16) uint4 vrow_smem_buf[];
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];
    prologue(s_ptr, p.lc, p.W);
    // gamma, with eight zero elements on either side
    unsigned short* s_g = reinterpret_cast<unsigned short*>(vrow_smem_buf);
    const int ng = (int)(vrow_smem(p.H) / 2);
    for (int i = threadIdx.x; i < ng; i += blockDim.x) s_g[i] = (i >= 8 && i < p.H + 8) ? p.gamma[i - 8] : 0;
    __syncthreads();
    if (!vector_layout(p, s_ptr)) {  // the same answer in every thread of every CTA
        rms_elem_rows<T, false>(p, s_ptr, s_warp);
        return;
    }
    const uint4* g16 = vrow_smem_buf;
    const int H = p.H;
    uint4 L[NV][WS + 1];
    int64_t row = blockIdx.x;
    VRow g = vrow_of(row, p.ldp, H);
    if (row < p.M) vrow_issue<WS, NV>(L, p, s_ptr, row, g);
    for (int it = 0; row < p.M; ++it) {
        const int64_t ro0 = row * p.ldro, o0 = row * p.ldo;
        const int64_t vro = (ro0 - g.phase) >> 3, vo = (o0 - g.phase) >> 3;
        uint4 xs[NV];
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = warp_run_chunk<NV>(k);
            if (j < g.nvec) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int r = 0; r < WS; ++r) accumulate<T>(acc, L[k][r]);
                accumulate<T>(acc, L[k][WS]);
                xs[k] = Pack8<T>::narrow(acc);
                float x[8];
                Pack8<T>::widen(xs[k], x);
                if (g.edge(j, H)) {
                    st_edge(p.residual_out, ro0, g, j, H, xs[k]);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (g.lane_in(j, e, H)) ss = fmaf(x[e], x[e], ss);
                } else {
                    st_out(reinterpret_cast<uint4*>(p.residual_out) + vro + j, xs[k]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                }
            }
        }
        // the next row's loads, in flight across this row's barrier
        const int64_t next = row + gridDim.x;
        const VRow gn = vrow_of(next, p.ldp, H);
        if (next < p.M) vrow_issue<WS, NV>(L, p, s_ptr, next, gn);
        const float inv = rsqrtf(cta_sum_squares(ss, s_warp, it) / (float)H + p.eps);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int j = warp_run_chunk<NV>(k);
            if (j < g.nvec) {
                const uint4 gv = shift_in(g16[j], g16[j + 1], g.phase);
                float x[8], gg[8], y[8];
                Pack8<T>::widen(xs[k], x);
                Pack8<T>::widen(gv, gg);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), gg[e]);
                const uint4 ov = Pack8<T>::narrow(y);
                if (g.edge(j, H)) st_edge(p.out, o0, g, j, H, ov);
                else st_out(reinterpret_cast<uint4*>(p.out) + vo + j, ov);
            }
        }
        row = next;
        g = gn;
    }
}

}  // namespace arf
