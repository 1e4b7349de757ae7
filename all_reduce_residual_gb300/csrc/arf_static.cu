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
// library, ARF_STATIC_STAGING_BYTES bytes, which every GPU that loads the
// library keeps until the process exits. Host code cannot use the array's
// name as a device address (on the host it is only a stand-in symbol), so the
// address is obtained with cudaGetSymbolAddress once per device, with that
// device current, on the first call made on that device.
#include <mutex>

#include "arf.h"
#include "arf_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_staging[ARF_STATIC_STAGING_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_setup_mu;
void* g_staging_addr[kMaxDevices] = {};

// Device address of g_static_staging on the current device `device`,
// looked up once per device.
cudaError_t staging_address(int device, void** out) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_staging_addr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_staging);
        if (e != cudaSuccess) return e;
        g_staging_addr[device] = p;
    }
    *out = g_staging_addr[device];
    return cudaSuccess;
}

}  // namespace

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
    int device = -1;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess && (device < 0 || device >= kMaxDevices)) e = cudaErrorInvalidDevice;
    void* staging = nullptr;
    if (e == cudaSuccess) e = staging_address(device, &staging);
    if (e != cudaSuccess) {
        arf::note_cuda_error(ws, e);
        return ARF_ERR_CUDA;
    }
    // The rest is arf_run_host on the built-in array: device checks, copies
    // in, the kernel, copies out. Every region the kernels read is written
    // earlier in the same call, so nothing in the array has to start at zero.
    return arf_run_host(ws, pattern, W, partials_host, residual_host, gamma_host, eps, out_host,
                        residual_out_host, M, H, dtype, staging, (size_t)ARF_STATIC_STAGING_BYTES, stream);
}
