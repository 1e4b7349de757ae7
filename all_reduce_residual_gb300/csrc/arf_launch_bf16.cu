// bf16 instances of the epilogue kernels.
#include "arf_launch.cuh"

namespace arf {

cudaError_t launch_flat_bf16(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s) {
    return launch_flat_t<__nv_bfloat16>(p, plan, s);
}
cudaError_t launch_rms_bf16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s) {
    return launch_rms_t<__nv_bfloat16>(p, plan, s);
}
cudaError_t allow_large_clusters_bf16() { return allow_large_clusters_t<__nv_bfloat16>(); }
cudaError_t rms_max_active_clusters_bf16(const arf_plan_t& plan, int* n) {
    return rms_max_active_clusters_t<__nv_bfloat16>(plan, n);
}

cudaError_t rms_max_active_blocks_bf16(const arf_plan_t& plan, int* n) {
    return rms_max_active_blocks_t<__nv_bfloat16>(plan, n);
}

}  // namespace arf
