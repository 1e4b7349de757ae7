// arf_bulk.cuh: kARResidualRMSNorm staged through shared memory by the
// Tensor Memory Accelerator's bulk copies (ARF_PATH_BULK).
//
// Each CTA walks its rows (blockIdx.x + i*gridDim.x) in column blocks of B
// chunks (B = blockDim.x; a chunk is 16 bytes, 8 elements). A work item is
// one (row, column block): W + 1 contiguous segments of B*16 bytes, one per
// partial and one of the residual. One thread (thread 0) keeps `stages`
// items in flight: for each it arms the slot's mbarrier with the item's byte
// count and issues W + 1 one-dimensional bulk copies (cp.async.bulk) into the
// slot. The copies complete on the barrier by transaction count, so no
// thread holds registers for bytes in flight and the HBM queue stays full
// across the row statistic and the normalisation of the previous row. Every
// thread then sums its chunk from shared memory (rank order, binary32, the
// same arithmetic as the row kernels), stores residual_out and keeps the
// rounded value in a row buffer in shared memory until the statistic is known.
//
// Waits are bounded: a thread that has not seen its slot fill within
// p.spin_limit SM cycles reports it, the whole CTA stops at the next block
// barrier, thread 0 waits (bounded again, by at least the default limit) for
// the copies it issued and has not seen land, counts the event in *p.status,
// and the CTA returns.
#pragma once

#include "arf_kernels.cuh"

namespace arf {

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// One arrival (the producer's) plus `bytes` expected from bulk copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of parity `parity` to complete; false once `limit` SM
// cycles have passed without it.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// Global -> shared bulk copy of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// RMS = false: the kAllReduce form. Items carry the W partials only, every
// thread stores rn(sum) of its chunk, and there is no row buffer or row
// statistic; the ring, the producer and the bounded waits are the same.
template <typename T, int WS, bool RMS = true>
__global__ void __launch_bounds__(kMaxThreads) rms_bulk_kernel(RmsParams p) {
    extern __shared__ __align__(128) uint4 bulk_smem[];
    __shared__ const uint4* s_ptr[ARF_MAX_W];
    __shared__ float s_warp[2][kMaxThreads / 32];
    __shared__ __align__(8) unsigned long long s_bar[kBulkMaxStages];

    prologue(s_ptr, p.lc, p.W);

    const int W = WS > 0 ? WS : p.W;
    const int NT = RMS ? W + 1 : W;  // segments per item: the partials (and the residual)
    const int B = blockDim.x, tid = threadIdx.x;
    const int S = p.stages, C = p.C;
    const int nb = (C + B - 1) / B;  // column blocks per row
    uint4* ring = bulk_smem;                                   // [S][NT][B]
    uint4* xrow = bulk_smem + (size_t)S * NT * B;              // [C]: the row's rounded residual_out (RMS)
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(s_bar);
    const uint32_t ring0 = (uint32_t)__cvta_generic_to_shared(ring);
    const uint32_t rank_bytes = (uint32_t)B * 16u;             // one segment's slot space
    const uint32_t slot_bytes = (uint32_t)NT * rank_bytes;
    const long long limit = p.spin_limit;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bar0 + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();  // partial pointers and barriers ready

    // Producer state (thread 0 only): the next item to issue, counted
    // without division; `issued` items so far.
    int64_t in_row = blockIdx.x;
    int in_b = 0, in_slot = 0;
    int64_t issued = 0;
    auto issue_next = [&]() {
        if (in_row >= p.M) return;
        const int c0 = in_b * B;
        const uint32_t bytes = (uint32_t)min(B, C - c0) * 16u;
        const uint32_t bar = bar0 + 8u * (uint32_t)in_slot;
        const uint32_t dst = ring0 + (uint32_t)in_slot * slot_bytes;
        if (!(p.hold_first && issued == 0)) {
            mbar_arrive_expect_tx(bar, bytes * (uint32_t)NT);
            const int64_t poff = in_row * p.ly.ldp + c0;
            for (int r = 0; r < W; ++r) bulk_load(dst + (uint32_t)r * rank_bytes, s_ptr[r] + poff, bytes, bar);
            if constexpr (RMS) bulk_load(dst + (uint32_t)W * rank_bytes, p.residual + in_row * p.ly.ldr + c0, bytes, bar);
        }
        ++issued;
        if (++in_b == nb) {
            in_b = 0;
            in_row += gridDim.x;
        }
        if (++in_slot == S) in_slot = 0;
    };
    if (tid == 0)
        for (int j = 0; j < S; ++j) issue_next();

    int slot = 0;
    uint32_t phase = 0;
    int64_t consumed = 0;
    bool failed = false;
    int it = 0;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) {
        const int64_t ob = row * p.ly.ldo, rob = row * p.ly.ldro;
        float ss = 0.0f;
        for (int b = 0; b < nb; ++b) {
            const bool ok = mbar_wait_bounded(bar0 + 8u * (uint32_t)slot, phase, limit);
            const int c = b * B + tid;
            if (ok && c < C) {
                const uint4* src = ring + (size_t)slot * NT * B + tid;
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
                if constexpr (WS > 0) {
#pragma unroll
                    for (int r = 0; r < WS; ++r) accumulate<T>(acc, src[(size_t)r * B]);
                } else {
                    for (int r = 0; r < W; ++r) accumulate<T>(acc, src[(size_t)r * B]);
                }
                if constexpr (RMS) xrow[c] = residual_chunk<T>(acc, src[(size_t)W * B], p.residual_out + rob + c, ss);
                else st_out(p.out + ob + c, Pack8<T>::narrow(acc));
            }
            // every thread is done with this slot (or the CTA gives up)
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            ++consumed;
            if (tid == 0) {
                // the slot's generic-proxy reads are ordered before the
                // async-proxy writes that refill it
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_next();
            }
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (failed) break;
        if constexpr (RMS) {
            const float inv = rsqrtf(cta_sum_squares(ss, s_warp, it) / (float)p.H + p.eps);
            for (int c = tid; c < C; c += B) normalise_chunk<T>(xrow[c], ld_keep(p.gamma + c), inv, p.out + ob + c);
        }
    }
    if (failed && tid == 0) {
        // Leave with no copy in flight into this CTA's shared memory. The
        // drain waits at least the default limit, however short the caller's
        // limit was: a copy that has not landed by then is lost, and this CTA
        // may exit with it still in flight.
        const long long drain = limit > kBulkSpinLimit ? limit : kBulkSpinLimit;
        for (int64_t j = consumed; j < issued; ++j) {
            if (p.hold_first && j == 0) continue;  // never issued
            (void)mbar_wait_bounded(bar0 + 8u * (uint32_t)(j % S), (uint32_t)((j / S) & 1), drain);
        }
        atomicAdd(p.status, 1u);
    }
}

}  // namespace arf
