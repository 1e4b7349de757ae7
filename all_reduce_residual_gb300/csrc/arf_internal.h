// arf_internal.h: declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "arf.h"

namespace arf {

// Every kernel is compiled for at most this many threads per CTA.
constexpr int kMaxThreads = 512;

// Rank counts with a kernel specialised at compile time (0 = generic): the
// pages' tensor-parallel sizes up to 16, TP12 included.
constexpr bool w_spec_compiled(int ws) {
    return ws == 0 || ws == 1 || ws == 2 || ws == 4 || ws == 8 || ws == 12 || ws == 16;
}
// Flat-kernel unroll factors compiled per rank count (registers: U*W vectors).
constexpr bool flat_unroll_compiled(int ws, int u) {
    return (u == 1) || (u == 2 && ws <= 8) || (u == 4 && ws <= 4);
}
// Chunks per thread compiled for the RMS kernel.
constexpr bool rms_vpt_compiled(int vpt) { return vpt == 1 || vpt == 2 || vpt == 4 || vpt == 8; }
// Whether the row/cluster RMS kernel instance (ws, vpt) holds a whole row of
// loads per thread in registers and issues the next row's before the row
// barrier: the rank count compiled in and VPT*(W+1) <= 18 vectors.
constexpr bool rms_prefetches(int ws, int vpt) { return ws > 0 && vpt * (ws + 1) <= 18; }

// How a kernel finds the W partial pointers and when it may start.
struct LaunchCommon {
    const void* const* partials;    // device array of W device pointers, or
    const void* ptrs[ARF_MAX_W];    // the pointers themselves (by_value)
    int by_value;                   // 1: read ptrs[] from the launch parameters
    int pdl;                        // 1: launched as a programmatic dependent
};

// Row layout shared by both kernels. A chunk is 8 elements; strides are in
// 16-byte vectors. 16-bit partials: chunk c of row m is vector m*ldp + c;
// binary32 partials (f32p): vectors m*ldp + 2c and m*ldp + 2c + 1.
struct RowLayout {
    int64_t ldp;   // partials row stride (vectors)
    int64_t ldr;   // residual row stride (vectors)
    int64_t ldo;   // out row stride (vectors)
    int64_t ldro;  // residual_out row stride (vectors)
};

struct FlatParams {
    LaunchCommon lc;
    RowLayout ly;
    uint4* out;
    int64_t nchunks;              // M*C
    int64_t M;
    int C;                        // chunks per row, H/8
    int strided;                  // 0: rows contiguous (a flat range of chunks)
    int W;
};

struct RmsParams {
    LaunchCommon lc;
    RowLayout ly;
    const uint4* residual;
    const uint4* gamma;
    uint4* out;
    uint4* residual_out;
    int64_t M;
    int C;      // 16-byte chunks per row, H/8
    int H;
    int W;
    int cs;     // CTAs per row (cluster size), 1 = no cluster
    int slice;  // chunks per CTA: ceil(C / cs)
    int stages; // streaming / bulk paths: work items in flight
    float eps;
    // bulk path (ARF_PATH_BULK) only
    unsigned int* status;  // device counter: CTAs whose wait gave up
    long long spin_limit;  // SM cycles a wait may take before giving up
    int hold_first;        // testing the bounded waits: never issue item 0
};

// Elementwise kernels (arf_elem.cuh): any H, 2-byte alignment.
struct ElemParams {
    LaunchCommon lc;
    const unsigned short* residual;
    const unsigned short* gamma;
    unsigned short* out;
    unsigned short* residual_out;
    int64_t M;
    int64_t ldp, ldr, ldo, ldro;  // row strides, elements
    int H;
    int W;
    float eps;
    // Whether 16-byte vectors can serve this layout: out (and, for the RMS
    // pattern, residual and residual_out) 16-byte aligned and every row
    // stride congruent to ldp modulo 8, so that row r of every tensor starts
    // at the same offset within a 16-byte vector. 1: the tensors are also
    // contiguous ([M,H], strides H), one flat range of M*H elements; 2: rows
    // apart; 0: neither. The kernels then take vectors if every partial
    // pointer is 16-byte aligned too (they check): per row, an elementwise
    // head up to the first 16-byte boundary, whole chunks, an elementwise
    // tail; kAllReduce on contiguous tensors runs the whole range as one.
    int flat_ok;
};

// Launchers, one per I/O type (arf_launch_bf16.cu / arf_launch_fp16.cu).
// They assume a plan that passed arf_plan_check. f32p: binary32 partials.
cudaError_t launch_flat_bf16(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p);
cudaError_t launch_flat_fp16(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p);
cudaError_t launch_rms_bf16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p);
cudaError_t launch_rms_fp16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p);
// kAllReduce on the bulk-copy kernel (ARF_PATH_BULK): RmsParams with the
// residual, gamma and residual_out unused.
cudaError_t launch_bulk_ar_bf16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s);
cudaError_t launch_bulk_ar_fp16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s);
cudaError_t bulk_ar_max_active_blocks_bf16(const arf_plan_t& plan, int W, int* n);
cudaError_t bulk_ar_max_active_blocks_fp16(const arf_plan_t& plan, int W, int* n);
cudaError_t launch_elem_bf16(const ElemParams& p, const arf_plan_t& plan, bool rms, cudaStream_t s, bool f32p);
cudaError_t launch_elem_fp16(const ElemParams& p, const arf_plan_t& plan, bool rms, cudaStream_t s, bool f32p);

// Per-device kernel attributes, set once at workspace creation: 16-CTA
// clusters for the cluster kernels (when the device has clusters) and
// `max_dyn_smem` bytes of dynamic shared memory for the streaming kernels.
cudaError_t configure_kernels_bf16(bool clusters, int max_dyn_smem);
cudaError_t configure_kernels_fp16(bool clusters, int max_dyn_smem);

// Threads per CTA and static shared memory of the streaming kernel.
constexpr int kAsyncCtaThreads = 256;
constexpr int kAsyncStaticSmem = 1024;  // upper bound, for the planner
// Dynamic shared memory of the streaming kernel for W ranks, `stages` ring
// slots and rows of C chunks.
constexpr size_t async_dyn_smem(int W, int stages, int C) {
    return (size_t)stages * (size_t)(W + 1) * kAsyncCtaThreads * 16u + (size_t)C * 16u;
}

// The bulk-copy kernel (arf_bulk.cuh): at most this many ring slots; its
// static shared memory; its dynamic shared memory for W ranks, `stages`
// slots of `threads` chunks per rank and rows of C chunks.
constexpr int kBulkMaxStages = 16;
// Its __shared__ arrays: s_ptr (8 * ARF_MAX_W bytes), s_warp (2 * kMaxThreads
// / 32 floats) and s_bar (8 * kBulkMaxStages bytes); the kAllReduce form
// drops s_warp. With the 1 KB the SM reserves per CTA, this is what decides
// whether two CTAs of long rows fit on one SM.
constexpr int kBulkStaticSmem = 8 * ARF_MAX_W + 2 * (kMaxThreads / 32) * 4 + 8 * kBulkMaxStages;
constexpr size_t bulk_dyn_smem(int W, int stages, int threads, int C) {
    return (size_t)stages * (size_t)(W + 1) * (size_t)threads * 16u + (size_t)C * 16u;
}
// ... and of its kAllReduce form (partials only, no row buffer).
constexpr size_t bulk_ar_dyn_smem(int W, int stages, int threads) {
    return (size_t)stages * (size_t)W * (size_t)threads * 16u;
}
// Default wait limit of the bulk kernel: 2^31 SM cycles, about a second.
constexpr long long kBulkSpinLimit = 1ll << 31;

// How many clusters of plan.cluster CTAs of plan.threads threads the RMS
// kernel instance of `plan` can keep resident at once (0 = cannot launch).
cudaError_t rms_max_active_clusters_bf16(const arf_plan_t& plan, int* n, bool f32p = false);
cudaError_t rms_max_active_clusters_fp16(const arf_plan_t& plan, int* n, bool f32p = false);
// How many CTAs of the RMS kernel instance of `plan` (rows of C chunks, W
// ranks) one SM can hold.
cudaError_t rms_max_active_blocks_bf16(const arf_plan_t& plan, int C, int W, int* n, bool f32p = false);
cudaError_t rms_max_active_blocks_fp16(const arf_plan_t& plan, int C, int W, int* n, bool f32p = false);

// Record a CUDA error as the workspace's last one (arf_last_cuda_error).
void note_cuda_error(arf_workspace_t ws, cudaError_t e);

// The staging array of arf_run_host_static (arf_static.cu): its device
// address on the current device (cudaGetSymbolAddress), and the address a
// workspace looked up at creation (or the error that lookup returned).
cudaError_t static_staging_address(void** out);
cudaError_t workspace_static_staging(arf_workspace_t ws, void** out);

// The read-only measurement pass (arf_measure.cu): a CTA per 16 KiB tile.
cudaError_t launch_read_pass(const void* buf, int64_t bytes, unsigned int* sink, cudaStream_t s);

// Host-buffer helper kernel launcher (arf_api.cu).
cudaError_t launch_fill_pointer_array(const void** array, const char* first, int64_t stride, int W,
                                      cudaStream_t s);

}  // namespace arf
