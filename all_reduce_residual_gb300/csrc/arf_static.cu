// arf_static.cu: arf_run_host_static, the host-buffer entry point for callers
// that cannot allocate device memory.
//
// Who needs it: a caller that holds its data in host memory and is not
// allowed to call cudaMalloc or any other allocator on the device. Typical
// cases are a plugin living inside a framework or serving engine whose own
// allocator has reserved the device memory up front (an outside cudaMalloc
// would fail or break its accounting), and a latency-critical host thread
// that cannot afford cudaMalloc's implicit device-wide synchronisation. Such
// a caller cannot provide the device staging buffer that arf_run_host needs.
//
// Here that staging buffer is a file-scope device array compiled into the
// library, ARF_STATIC_STAGING_BYTES bytes. Host code cannot use the array's
// name as a device address (on the host it is only a stand-in symbol), so
// arf_workspace_create looks the address up with cudaGetSymbolAddress, with
// the workspace's device current, and the workspace keeps it. Under CUDA's
// lazy module loading (the default) that lookup is also what loads the array
// onto the device, so the array is taken when the first workspace on a device
// is created, never inside a call of this entry point; it stays until the
// process exits. A workspace lives in one CUDA context: after a device reset
// it must be destroyed and created again, which looks the address up anew.
#include "arf.h"
#include "arf_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_staging[ARF_STATIC_STAGING_BYTES];

}  // namespace

namespace arf {

cudaError_t static_staging_address(void** out) { return cudaGetSymbolAddress(out, g_static_staging); }

}  // namespace arf

extern "C" size_t arf_static_staging_bytes(void) { return (size_t)ARF_STATIC_STAGING_BYTES; }

extern "C" arf_status_t arf_run_host_static(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                            const void* const* partials_host, const void* residual_host,
                                            const void* gamma_host, float eps, void* out_host,
                                            void* residual_out_host, int64_t M, int64_t H, arf_dtype_t dtype,
                                            void* stream) {
    if (!ws) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(ws, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (M == 0) return ARF_OK;
    if (arf_host_staging_bytes(pattern, W, M, H, dtype) > (size_t)ARF_STATIC_STAGING_BYTES)
        return ARF_ERR_UNSUPPORTED;  // larger than the built-in staging array
    // the address the workspace looked up on its device at creation
    void* staging = nullptr;
    const cudaError_t e = arf::workspace_static_staging(ws, &staging);
    if (e != cudaSuccess) {
        arf::note_cuda_error(ws, e);
        return ARF_ERR_CUDA;
    }
    // The rest is arf_run_host on the built-in array: device checks (the
    // current device must be the workspace's, whose array this is), copies
    // in, the kernel, copies out. Every region the kernels read is written
    // earlier in the same call, so nothing in the array has to start at zero.
    return arf_run_host(ws, pattern, W, partials_host, residual_host, gamma_host, eps, out_host,
                        residual_out_host, M, H, dtype, staging, (size_t)ARF_STATIC_STAGING_BYTES, stream);
}
