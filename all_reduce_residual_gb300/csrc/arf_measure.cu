// arf_measure.cu: a read-only streaming pass, the measurement reference for
// read-dominated calls (arf_read_pass in arf.h). On GB300 reads alone stream
// slower than a copy's mix of reads and writes at the sizes the epilogue
// runs at, so a call that mostly reads is bounded by the time this pass
// takes over the same number of bytes, not by the copy rate.
#include <cuda_runtime.h>

#include "arf_internal.h"

namespace arf {

// Every thread reads 16-byte vectors at a grid stride and folds them into a
// register; one store, under a condition the data cannot be shown to avoid,
// keeps the loads alive.
__global__ void __launch_bounds__(512) read_pass_kernel(const uint4* a, int64_t n, unsigned int* sink) {
    unsigned int x = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        uint4 v;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(a + i));
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (x == 0x9e3779b9u) *sink = x;
}

cudaError_t launch_read_pass(const void* buf, int64_t bytes, int grid, unsigned int* sink, cudaStream_t s) {
    read_pass_kernel<<<grid, 512, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16, sink);
    return cudaGetLastError();
}

}  // namespace arf
