// fp16 instances of the epilogue kernels.
#include "arf_launch.cuh"

namespace arf {

cudaError_t launch_flat_fp16(const FlatParams& p, const arf_plan_t& plan, cudaStream_t s) {
    return launch_flat_t<__half>(p, plan, s);
}
cudaError_t launch_rms_fp16(const RmsParams& p, const arf_plan_t& plan, cudaStream_t s) {
    return launch_rms_t<__half>(p, plan, s);
}
cudaError_t allow_large_clusters_fp16() { return allow_large_clusters_t<__half>(); }
cudaError_t rms_max_active_clusters_fp16(const arf_plan_t& plan, int* n) {
    return rms_max_active_clusters_t<__half>(plan, n);
}

cudaError_t rms_max_active_blocks_fp16(const arf_plan_t& plan, int* n) {
    return rms_max_active_blocks_t<__half>(plan, n);
}

}  // namespace arf
