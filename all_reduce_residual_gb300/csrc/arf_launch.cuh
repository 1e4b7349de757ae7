// arf_launch.cuh: kernel tables and launchers for one I/O type. Included by
// arf_launch_bf16.cu and arf_launch_fp16.cu, which instantiate it once each.
#pragma once

#include "arf_bulk.cuh"
#include "arf_elem.cuh"

namespace arf {

using FlatFn = void (*)(FlatParams);
using RmsFn = void (*)(RmsParams);
using ElemFn = void (*)(ElemParams);

template <typename T, int WS>
FlatFn flat_by_unroll(int u) {
    switch (u) {
        case 1: return ar_flat_kernel<T, WS, 1>;
        case 2: if constexpr (flat_unroll_compiled(WS, 2)) return ar_flat_kernel<T, WS, 2>; else return nullptr;
        case 4: if constexpr (flat_unroll_compiled(WS, 4)) return ar_flat_kernel<T, WS, 4>; else return nullptr;
        default: return nullptr;
    }
}

template <typename T>
FlatFn flat_kernel_for(int ws, int u, bool f32p = false) {
    if (f32p) {  // binary32 partials: run-time rank count only
        if (ws != 0) return nullptr;
        switch (u) {
            case 1: return ar_flat_kernel<T, 0, 1, true>;
            case 2: return ar_flat_kernel<T, 0, 2, true>;
            case 4: return ar_flat_kernel<T, 0, 4, true>;
            default: return nullptr;
        }
    }
    switch (ws) {
        case 0: return flat_by_unroll<T, 0>(u);
        case 1: return flat_by_unroll<T, 1>(u);
        case 2: return flat_by_unroll<T, 2>(u);
        case 4: return flat_by_unroll<T, 4>(u);
        case 8: return flat_by_unroll<T, 8>(u);
        case 12: return flat_by_unroll<T, 12>(u);
        case 16: return flat_by_unroll<T, 16>(u);
        default: return nullptr;
    }
}

template <typename T, int WS>
RmsFn rms_by_vpt(int vpt) {
    switch (vpt) {
        case 1: return rms_kernel<T, WS, 1>;
        case 2: return rms_kernel<T, WS, 2>;
        case 4: return rms_kernel<T, WS, 4>;
        case 8: return rms_kernel<T, WS, 8>;
        default: return nullptr;
    }
}

template <typename T>
RmsFn rms_kernel_for(int ws, int vpt, bool f32p = false) {
    if (f32p) {  // binary32 partials: run-time rank count only
        if (ws != 0) return nullptr;
        switch (vpt) {
            case 1: return rms_kernel<T, 0, 1, true>;
            case 2: return rms_kernel<T, 0, 2, true>;
            case 4: return rms_kernel<T, 0, 4, true>;
            case 8: return rms_kernel<T, 0, 8, true>;
            default: return nullptr;
        }
    }
    switch (ws) {
        case 0: return rms_by_vpt<T, 0>(vpt);
        case 1: return rms_by_vpt<T, 1>(vpt);
        case 2: return rms_by_vpt<T, 2>(vpt);
        case 4: return rms_by_vpt<T, 4>(vpt);
        case 8: return rms_by_vpt<T, 8>(vpt);
        case 12: return rms_by_vpt<T, 12>(vpt);
        case 16: return rms_by_vpt<T, 16>(vpt);
        default: return nullptr;
    }
}

// The one-row form of the prefetching instances (grid covers every row).
template <typename T, int WS>
RmsFn one_row_by_vpt(int vpt) {
    switch (vpt) {
        case 1: if constexpr (rms_prefetches(WS, 1)) return rms_kernel<T, WS, 1, false, true>; else return nullptr;
        case 2: if constexpr (rms_prefetches(WS, 2)) return rms_kernel<T, WS, 2, false, true>; else return nullptr;
        case 4: if constexpr (rms_prefetches(WS, 4)) return rms_kernel<T, WS, 4, false, true>; else return nullptr;
        case 8: if constexpr (rms_prefetches(WS, 8)) return rms_kernel<T, WS, 8, false, true>; else return nullptr;
        default: return nullptr;
    }
}

template <typename T>
RmsFn one_row_kernel_for(int ws, int vpt) {
    switch (ws) {
        case 1: return one_row_by_vpt<T, 1>(vpt);
        case 2: return one_row_by_vpt<T, 2>(vpt);
        case 4: return one_row_by_vpt<T, 4>(vpt);
        case 8: return one_row_by_vpt<T, 8>(vpt);
        case 12: return one_row_by_vpt<T, 12>(vpt);
        case 16: return one_row_by_vpt<T, 16>(vpt);
        default: return nullptr;
    }
}

template <typename T>
RmsFn async_kernel_for(int ws) {
    switch (ws) {
        case 1: return rms_async_kernel<T, 1>;
        case 2: return rms_async_kernel<T, 2>;
        case 4: return rms_async_kernel<T, 4>;
        case 8: return rms_async_kernel<T, 8>;
        case 12: return rms_async_kernel<T, 12>;
        case 16: return rms_async_kernel<T, 16>;
        default: return nullptr;
    }
}

template <typename T>
RmsFn bulk_kernel_for(int ws) {
    switch (ws) {
        case 0: return rms_bulk_kernel<T, 0>;
        case 1: return rms_bulk_kernel<T, 1>;
        case 2: return rms_bulk_kernel<T, 2>;
        case 4: return rms_bulk_kernel<T, 4>;
        case 8: return rms_bulk_kernel<T, 8>;
        case 12: return rms_bulk_kernel<T, 12>;
        case 16: return rms_bulk_kernel<T, 16>;
        default: return nullptr;
    }
}

template <typename T>
RmsFn bulk_ar_kernel_for(int ws) {
    switch (ws) {
        case 0: return rms_bulk_kernel<T, 0, false>;
        case 1: return rms_bulk_kernel<T, 1, false>;
        case 2: return rms_bulk_kernel<T, 2, false>;
        case 4: return rms_bulk_kernel<T, 4, false>;
        case 8: return rms_bulk_kernel<T, 8, false>;
        case 12: return rms_bulk_kernel<T, 12, false>;
        case 16: return rms_bulk_kernel<T, 16, false>;
        default: return nullptr;
    }
}

template <typename T>
cudaError_t launch_bulk_ar_t(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s) {
    RmsFn fn = bulk_ar_kernel_for<T>(plan.w_spec);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.dynamicSmemBytes = bulk_ar_dyn_smem(p.W, plan.stages, plan.threads);
    cfg.stream = s;
    if (p.lc.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename T>
cudaError_t bulk_ar_max_active_blocks_t(const arf_plan_t& plan, int W, int* n) {
    RmsFn fn = bulk_ar_kernel_for<T>(plan.w_spec);
    if (!fn) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, fn, plan.threads, bulk_ar_dyn_smem(W, plan.stages, plan.threads));
}

// The RMS kernel of a plan and its dynamic shared memory (rows of C chunks,
// W ranks). one_row: every cluster of the grid owns at most one row, so the
// prefetching instances may use their one-row form.
template <typename T>
RmsFn rms_fn_for(const arf_plan_t& plan, bool f32p, bool one_row = false) {
    if (plan.path == ARF_PATH_ASYNC) return f32p ? nullptr : async_kernel_for<T>(plan.w_spec);
    if (plan.path == ARF_PATH_BULK) return f32p ? nullptr : bulk_kernel_for<T>(plan.w_spec);
    if (one_row && !f32p) {
        RmsFn fn = one_row_kernel_for<T>(plan.w_spec, plan.vpt);
        if (fn) return fn;
    }
    return rms_kernel_for<T>(plan.w_spec, plan.vpt, f32p);
}

inline size_t rms_dyn_smem(const arf_plan_t& plan, int C, int W) {
    if (plan.path == ARF_PATH_ASYNC) return async_dyn_smem(plan.w_spec, plan.stages, C);
    if (plan.path == ARF_PATH_BULK) return bulk_dyn_smem(W, plan.stages, plan.threads, C);
    return 0;
}

template <typename T>
cudaError_t launch_flat_t(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p) {
    FlatFn fn = flat_kernel_for<T>(plan.w_spec, plan.vpt, f32p);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.stream = s;
    if (p.lc.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename T>
cudaError_t launch_rms_t(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p) {
    const bool one_row = (int64_t)(plan.grid / plan.cluster) >= p.M;
    RmsFn fn = rms_fn_for<T>(plan, f32p, one_row);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.dynamicSmemBytes = rms_dyn_smem(plan, p.C, p.W);
    cfg.stream = s;
    unsigned n = 0;
    if (plan.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)plan.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (p.lc.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

// The elementwise instance for a call: binary32 partials, else the rank
// count compiled in where there is one (1, 2, 4, 8; the plan's w_spec does
// not apply to these kernels), else the run-time rank count.
template <typename T>
ElemFn elem_kernel_for(bool rms, bool f32p, int W) {
    if (f32p) return rms ? rms_elem_kernel<T, true> : ar_elem_kernel<T, true>;
    switch (W) {
        case 1: return rms ? rms_elem_kernel<T, false, 1> : ar_elem_kernel<T, false, 1>;
        case 2: return rms ? rms_elem_kernel<T, false, 2> : ar_elem_kernel<T, false, 2>;
        case 4: return rms ? rms_elem_kernel<T, false, 4> : ar_elem_kernel<T, false, 4>;
        case 8: return rms ? rms_elem_kernel<T, false, 8> : ar_elem_kernel<T, false, 8>;
        default: return rms ? rms_elem_kernel<T, false> : ar_elem_kernel<T, false>;
    }
}

template <typename T>
cudaError_t launch_elem_t(const ElemParams& p, const arf_plan_t& plan, bool rms, cudaStream_t s, bool f32p) {
    ElemFn fn = elem_kernel_for<T>(rms, f32p, p.W);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.stream = s;
    if (p.lc.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename T>
cudaError_t configure_kernels_t(bool clusters, int max_dyn_smem) {
    const int ws_list[] = {0, 1, 2, 4, 8, 12, 16};
    const int vpt_list[] = {1, 2, 4, 8};
    if (clusters)
        for (int ws : ws_list)
            for (int vpt : vpt_list)
                for (int f32p = 0; f32p < 3; ++f32p) {
                    RmsFn fn = f32p == 2 ? one_row_kernel_for<T>(ws, vpt) : rms_kernel_for<T>(ws, vpt, f32p != 0);
                    if (!fn) continue;
                    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (e != cudaSuccess) return e;
                }
    for (int ws : ws_list) {
        for (RmsFn fn : {async_kernel_for<T>(ws), bulk_kernel_for<T>(ws), bulk_ar_kernel_for<T>(ws)}) {
            if (!fn) continue;
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

template <typename T>
// Occupancy answers cover both forms a plan may launch (the row loop and,
// where it exists, the one-row form): the smaller of the two.
cudaError_t rms_max_active_clusters_t(const arf_plan_t& plan, int* n, bool f32p) {
    RmsFn fns[2] = {rms_kernel_for<T>(plan.w_spec, plan.vpt, f32p),
                    f32p ? nullptr : one_row_kernel_for<T>(plan.w_spec, plan.vpt)};
    if (!fns[0]) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int best = -1;
    for (RmsFn fn : fns) {
        if (!fn) continue;
        int k = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&k, fn, &cfg);
        if (e != cudaSuccess) return e;
        best = best < 0 || k < best ? k : best;
    }
    *n = best;
    return cudaSuccess;
}

template <typename T>
cudaError_t rms_max_active_blocks_t(const arf_plan_t& plan, int C, int W, int* n, bool f32p) {
    int best = -1;
    for (int one_row = 0; one_row < 2; ++one_row) {
        RmsFn fn = rms_fn_for<T>(plan, f32p, one_row != 0);
        if (!fn) return cudaErrorInvalidValue;
        int k = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, fn, plan.threads, rms_dyn_smem(plan, C, W));
        if (e != cudaSuccess) return e;
        best = best < 0 || k < best ? k : best;
    }
    *n = best;
    return cudaSuccess;
}

}  // namespace arf
