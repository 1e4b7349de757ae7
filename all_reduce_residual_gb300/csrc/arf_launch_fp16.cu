// fp16 instances of the epilogue kernels.
#include "arf_launch.cuh"

namespace arf {

cudaError_t launch_flat_fp16(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p) {
    return launch_flat_t<__half>(p, plan, s, f32p);
}
cudaError_t launch_rms_fp16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s, bool f32p) {
    return launch_rms_t<__half>(p, plan, s, f32p);
}
cudaError_t launch_elem_fp16(const ElemParams& p, const arf_plan_t& plan, bool rms, cudaStream_t s, bool f32p) {
    return launch_elem_t<__half>(p, plan, rms, s, f32p);
}
cudaError_t configure_kernels_fp16(bool clusters, int max_dyn_smem) {
    return configure_kernels_t<__half>(clusters, max_dyn_smem);
}
cudaError_t rms_max_active_clusters_fp16(const arf_plan_t& plan, int* n, bool f32p) {
    return rms_max_active_clusters_t<__half>(plan, n, f32p);
}

cudaError_t rms_max_active_blocks_fp16(const arf_plan_t& plan, int C, int W, int* n, bool f32p) {
    return rms_max_active_blocks_t<__half>(plan, C, W, n, f32p);
}

cudaError_t launch_bulk_ar_fp16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s) {
    return launch_bulk_ar_t<__half>(p, plan, s);
}
cudaError_t bulk_ar_max_active_blocks_fp16(const arf_plan_t& plan, int W, int* n) {
    return bulk_ar_max_active_blocks_t<__half>(plan, W, n);
}

}  // namespace arf
