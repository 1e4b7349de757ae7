// arf_measure.cu: a read-only streaming pass, the measurement reference for
// read-dominated calls (arf_read_pass in arf.h). On GB300 reads alone stream
// slower than a copy's mix of reads and writes at the sizes the epilogue
// runs at, so a call that mostly reads is bounded by the time this pass
// takes over the same number of bytes, not by the copy rate.
#include <cuda_runtime.h>

#include "arf_internal.h"

namespace arf {

// One tile of 4 x 256 16-byte vectors per CTA: every thread issues its four
// loads together, folds them into a register and exits, and the grid has a
// CTA per tile, so the hardware block scheduler hands the tiles to whichever
// SM has room. On GB300 SMs do not all stream at the same rate; a fixed
// share of the buffer per CTA (a resident grid walking it at a grid stride)
// waits for the slowest SMs: 136 MiB cold took 28.6 us that way, with the
// CTAs finishing over 18.8-24.2 us, against 26.2 us with a CTA per tile
// (512 MiB: 88.7 against 77.2 us). Larger tiles per CTA measured slower
// (8, 16 and 64 vectors per thread: 31.9, 32.8 and 38.9 us at 136 MiB). One
// store, under a condition the data cannot be shown to avoid, keeps the
// loads alive.
constexpr int kReadUnroll = 4;
constexpr int kReadThreads = 256;

__global__ void __launch_bounds__(kReadThreads) read_pass_kernel(const uint4* a, int64_t n, unsigned int* sink) {
    const int64_t base = (int64_t)blockIdx.x * (kReadThreads * kReadUnroll) + threadIdx.x;
    uint4 v[kReadUnroll];
#pragma unroll
    for (int k = 0; k < kReadUnroll; ++k) {
        const int64_t i = base + (int64_t)k * kReadThreads;
        if (i < n)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                         : "l"(a + i));
        else
            v[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    unsigned int x = 0;
#pragma unroll
    for (int k = 0; k < kReadUnroll; ++k) x ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    if (x == 0x9e3779b9u) *sink = x;
}

cudaError_t launch_read_pass(const void* buf, int64_t bytes, unsigned int* sink, cudaStream_t s) {
    const int64_t n = bytes / 16;
    const int64_t tile = (int64_t)kReadThreads * kReadUnroll;
    const int64_t grid = (n + tile - 1) / tile;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    read_pass_kernel<<<(unsigned)grid, kReadThreads, 0, s>>>(static_cast<const uint4*>(buf), n, sink);
    return cudaGetLastError();
}

}  // namespace arf
