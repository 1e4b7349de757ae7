// arf_api.cu: the C ABI of include/arf.h: validation, launch planning,
// dispatch, and the host-buffer entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <climits>
#include <initializer_list>
#include <cstring>
#include <map>
#include <vector>
#include <mutex>
#include <new>
#include <tuple>

#include "arf.h"
#include "arf_internal.h"

struct arf_workspace {
    int device = 0;
    arf_device_caps_t caps = {};
    bool log = false;
    std::mutex mu;
    std::map<std::tuple<int, int, int64_t, int64_t, int>, arf_plan_t> plans;
    std::atomic<int> last_err{0};
    unsigned int* wait_timeouts = nullptr;  // device counter of the bulk kernel's given-up waits
    // Device address of the staging array of arf_run_host_static on this
    // workspace's device, looked up at creation (arf_static.cu), or the
    // error the lookup returned.
    void* static_staging = nullptr;
    cudaError_t static_staging_err = cudaErrorInvalidValue;
    // arf_run_host's pipelined form: a stream for the host-to-device copies
    // and one for the device-to-host copies, forked from and joined back into
    // the caller's stream with the events; host_mu keeps one call's records
    // and waits from interleaving with another's.
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_in = nullptr, ev_done = nullptr, ev_join = nullptr;
    std::mutex host_mu;
};

namespace {

using arf::kMaxThreads;
constexpr int kBulkMaxRanks = 12;  // the planner's bulk-path limit

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_pattern(int p) { return p == ARF_ALLREDUCE || p == ARF_AR_RESIDUAL_RMSNORM; }
bool valid_dtype(int d) { return d == ARF_BF16 || d == ARF_FP16; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

arf_status_t cuda_fail(arf_workspace_t ws, cudaError_t e) {
    if (ws) ws->last_err.store((int)e);
    return ARF_ERR_CUDA;
}

// The RMS plan for a given cluster size and chunks-per-thread count: threads
// cover the CTA's slice in whole warps; grid = rows (clusters) up to what the
// SMs can hold by thread count (the workspace refines this by occupancy).
arf_plan_t rms_plan(const arf_device_caps_t& caps, int w_spec, int64_t M, int64_t H, int cs, int vpt) {
    arf_plan_t pl = {};
    const int C = (int)(H / 8);
    const int slice = (int)ceil_div(C, cs);
    while (vpt < 8 && ceil_div(slice, vpt) > kMaxThreads) vpt *= 2;
    const int t = (int)ceil_div(ceil_div(slice, vpt), 32) * 32;
    pl.threads = t < 32 ? 32 : t;
    pl.vpt = vpt;
    pl.w_spec = w_spec;
    pl.cluster = cs;
    pl.path = cs == 1 ? ARF_PATH_ROW : ARF_PATH_CLUSTER;
    const int per_sm = caps.max_threads_per_sm / pl.threads > 0 ? caps.max_threads_per_sm / pl.threads : 1;
    int64_t max_clusters = (int64_t)caps.num_sms * per_sm / cs;
    if (max_clusters < 1) max_clusters = 1;
    const int64_t g = M < max_clusters ? M : max_clusters;
    pl.grid = (int)((g > 0 ? g : 1) * cs);
    return pl;
}

// Whether a row plan should launch one CTA per row (grid = M, the kernel's
// one-row form) rather than a resident grid looping over rows: W = 2 and 4
// at two chunks per thread, measured faster that way (the planner's RMS
// branch gives the numbers).
bool one_row_grid_wanted(const arf_plan_t& pl, int W) {
    return pl.path == ARF_PATH_ROW && pl.vpt == 2 && (W == 2 || W == 4) && pl.w_spec == W;
}

// One CTA per row with the fewest chunks per thread that keep it at <= 512
// threads (rows of up to 8 x 512 chunks).
arf_plan_t row_plan(const arf_device_caps_t& caps, int w_spec, int64_t M, int64_t H) {
    int vpt = 1;
    while (vpt < 8 && ceil_div(H / 8, vpt) > kMaxThreads) vpt *= 2;
    return rms_plan(caps, w_spec, M, H, 1, vpt);
}

// The bulk-copy plan (ARF_PATH_BULK) for rows of H elements and W ranks:
// column blocks of up to 512 chunks; as many CTAs per SM (up to 4, and at
// most 2048 threads) as fit with 2 ring slots each, or else one CTA per SM
// with up to 4 slots; narrower blocks if not even 2 slots fit. Measured on
// GB300: more CTAs with 2 slots beat fewer with deeper rings (W = 3:
// 29.4 us with 2 slots and 2 CTAs per SM, 30.7 us with 3 slots; W = 2,
// M = 3315: 3 CTAs per SM 36.3 us, 2 CTAs 38.7 us). False if nothing fits.
bool bulk_plan(const arf_device_caps_t& caps, int w_spec, int W, int64_t M, int64_t H, arf_plan_t* out) {
    const int64_t C = H / 8;
    const int64_t per_sm = (int64_t)caps.max_smem_per_block + 1024;  // the SM's shared memory
    const int64_t fixed = C * 16 + arf::kBulkStaticSmem;             // row buffer + static
    for (int B = (int)(C < kMaxThreads ? ceil_div(C, 32) * 32 : kMaxThreads); B >= 64; B /= 2) {
        const int64_t slot = (int64_t)(W + 1) * B * 16;
        for (int per = 4; per >= 1; --per) {
            if ((int64_t)per * B > caps.max_threads_per_sm) continue;
            const int64_t budget = per > 1 ? per_sm / per - 1024 : caps.max_smem_per_block;
            const int64_t s = (budget - fixed) / slot;
            if (s < 2) continue;
            arf_plan_t pl = {};
            pl.path = ARF_PATH_BULK;
            pl.threads = B;
            pl.vpt = 1;
            pl.cluster = 1;
            pl.w_spec = w_spec;
            pl.stages = per > 1 ? 2 : (int)(s < 4 ? s : 4);
            const int64_t g = (int64_t)caps.num_sms * per;
            pl.grid = (int)(M < g ? (M > 0 ? M : 1) : g);
            *out = pl;
            return true;
        }
    }
    return false;
}

const char* pattern_name(int p) { return p == ARF_ALLREDUCE ? "kAllReduce" : "kARResidualRMSNorm"; }
const char* path_name(int p) {
    switch (p) {
        case ARF_PATH_FLAT: return "flat";
        case ARF_PATH_ROW: return "row";
        case ARF_PATH_CLUSTER: return "cluster";
        case ARF_PATH_ASYNC: return "async";
        case ARF_PATH_ELEM: return "elem";
        case ARF_PATH_BULK: return "bulk";
        default: return "?";
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// status, workspace
// ---------------------------------------------------------------------------

extern "C" const char* arf_status_string(arf_status_t s) {
    switch (s) {
        case ARF_OK: return "ok";
        case ARF_ERR_INVALID_ARG: return "invalid argument";
        case ARF_ERR_UNSUPPORTED: return "unsupported size, alignment or plan";
        case ARF_ERR_CUDA: return "CUDA error";
        case ARF_ERR_DEVICE_MISMATCH: return "current device or stream device differs from the workspace device";
    }
    return "unknown status";
}

namespace {

// Free what a workspace holds on its device (the current device).
void release_device_resources(arf_workspace* ws) {
    if (ws->wait_timeouts) (void)cudaFree(ws->wait_timeouts);
    ws->wait_timeouts = nullptr;
    for (cudaStream_t* st : {&ws->h2d, &ws->d2h})
        if (*st) (void)cudaStreamDestroy(*st), *st = nullptr;
    for (cudaEvent_t* ev : {&ws->ev_fork, &ws->ev_in, &ws->ev_done, &ws->ev_join})
        if (*ev) (void)cudaEventDestroy(*ev), *ev = nullptr;
}

}  // namespace

extern "C" arf_status_t arf_workspace_create(int device, arf_workspace_t* ws_out) {
    if (!ws_out) return ARF_ERR_INVALID_ARG;
    *ws_out = nullptr;
    arf_workspace* ws = new (std::nothrow) arf_workspace();
    if (!ws) return ARF_ERR_CUDA;
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e == cudaSuccess && (device < 0 || device >= count)) e = cudaErrorInvalidDevice;
    if (e == cudaSuccess) e = cudaSetDevice(device);
    int sms = 0, thr = 0, cl = 0, smem = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&thr, cudaDevAttrMaxThreadsPerMultiProcessor, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e == cudaSuccess) {
        const int dyn = smem - arf::kAsyncStaticSmem;
        e = arf::configure_kernels_bf16(cl != 0, dyn);
        if (e == cudaSuccess) e = arf::configure_kernels_fp16(cl != 0, dyn);
    }
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&ws->wait_timeouts), 256);
    if (e == cudaSuccess) e = cudaMemset(ws->wait_timeouts, 0, 256);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ws->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ws->d2h, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&ws->ev_fork, &ws->ev_in, &ws->ev_done, &ws->ev_join})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        release_device_resources(ws);
        delete ws;
        (void)cudaGetLastError();
        return ARF_ERR_CUDA;
    }
    ws->device = device;
    ws->caps.num_sms = sms;
    ws->caps.max_threads_per_sm = thr;
    ws->caps.max_smem_per_block = smem;
    ws->caps.max_cluster = 1;
    if (cl) {
        // The largest cluster the row-split kernel can be launched with,
        // probed on a representative instance (128 threads).
        for (int cs = 16; cs >= 2; cs /= 2) {
            arf_plan_t probe = {};
            probe.path = ARF_PATH_CLUSTER;
            probe.threads = 128;
            probe.vpt = 1;
            probe.cluster = cs;
            probe.grid = cs;
            probe.w_spec = 8;
            int n = 0;
            if (arf::rms_max_active_clusters_bf16(probe, &n) == cudaSuccess && n > 0) {
                ws->caps.max_cluster = cs;
                break;
            }
            (void)cudaGetLastError();
        }
    }
    {
        // The built-in staging array of arf_run_host_static: its address on
        // this device, with the device current. Under lazy module loading this
        // lookup is what loads the array, so the array is taken here, at
        // set-up, and not inside a later call. A failure only disables that
        // entry point (it then returns ARF_ERR_CUDA with this error).
        void* addr = nullptr;
        const cudaError_t se = arf::static_staging_address(&addr);
        if (se == cudaSuccess) {
            ws->static_staging = addr;
            ws->static_staging_err = cudaSuccess;
        } else {
            ws->static_staging_err = se;
            (void)cudaGetLastError();
        }
    }
    const char* lg = std::getenv("ARF_LOG");
    ws->log = lg && lg[0] == '1';
    if (ws->log)
        std::fprintf(stderr, "[arf] device %d: %d SMs, %d threads/SM, %d B smem/CTA, max cluster %d\n", device,
                     sms, thr, smem, ws->caps.max_cluster);
    *ws_out = ws;
    return ARF_OK;
}

extern "C" arf_status_t arf_workspace_destroy(arf_workspace_t ws) {
    if (ws && ws->wait_timeouts) {
        int cur = -1;
        const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != ws->device &&
                              cudaSetDevice(ws->device) == cudaSuccess;
        release_device_resources(ws);
        if (switched) (void)cudaSetDevice(cur);
        (void)cudaGetLastError();
    }
    delete ws;
    return ARF_OK;
}

extern "C" arf_status_t arf_workspace_wait_timeouts(arf_workspace_t ws, unsigned int* count_out) {
    if (!ws || !count_out) return ARF_ERR_INVALID_ARG;
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e == cudaSuccess && cur != ws->device) e = cudaSetDevice(ws->device);
    unsigned int n = 0;
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&n, ws->wait_timeouts, sizeof n, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && n != 0) e = cudaMemset(ws->wait_timeouts, 0, sizeof n);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (cur >= 0 && cur != ws->device) (void)cudaSetDevice(cur);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    *count_out = n;
    return ARF_OK;
}

extern "C" arf_status_t arf_workspace_caps(arf_workspace_t ws, arf_device_caps_t* caps_out) {
    if (!ws || !caps_out) return ARF_ERR_INVALID_ARG;
    *caps_out = ws->caps;
    return ARF_OK;
}

extern "C" int arf_last_cuda_error(arf_workspace_t ws) { return ws ? ws->last_err.load() : 0; }

cudaError_t arf::workspace_static_staging(arf_workspace_t ws, void** out) {
    if (!ws->static_staging) return ws->static_staging_err;
    *out = ws->static_staging;
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// capability and planning
// ---------------------------------------------------------------------------

namespace {
// Longest kARResidualRMSNorm row a cluster of `max_cluster` CTAs can hold.
int64_t max_rms_row(int max_cluster) { return (int64_t)ARF_MAX_H_PER_CTA * (max_cluster < 1 ? 1 : max_cluster); }

// The elementwise kernels' plan: kAllReduce tiles of 256 elements, up to a
// device-full of CTAs; kARResidualRMSNorm one CTA per row, up to 512 threads.
arf_plan_t elem_plan(const arf_device_caps_t& caps, arf_pattern_t pattern, int64_t M, int64_t H) {
    arf_plan_t pl = {};
    pl.path = ARF_PATH_ELEM;
    pl.vpt = 1;
    pl.cluster = 1;
    if (pattern == ARF_ALLREDUCE) {
        pl.threads = 256;
        const int64_t tiles = ceil_div(H, 256) * M;
        const int64_t cap = (int64_t)caps.num_sms * (caps.max_threads_per_sm / 256 > 0 ? caps.max_threads_per_sm / 256 : 1);
        const int64_t g = tiles < cap ? tiles : cap;
        pl.grid = (int)(g > 0 ? g : 1);
    } else if (M >= 3 * (int64_t)caps.num_sms && H >= 1024) {
        // Many rows: narrower CTAs with several chunks per thread, more of
        // them per SM, hide a row's two dependent passes behind other rows
        // better than one wide CTA per row does. Measured on GB300 (cold,
        // 512 -> chosen threads): W = 2, H = 4098, M = 456 14.4 -> 12.3 us
        // (256), M = 4096 67.4 -> 43.1 us (128); W = 8, H = 7175, M = 456
        // 22.3 -> 18.9 us (256); 256 and 128 tie near M = 1024.
        const bool narrow = M >= 7 * (int64_t)caps.num_sms;
        pl.threads = narrow ? 128 : 256;
        const int64_t cap = (narrow ? 8 : 4) * (int64_t)caps.num_sms;
        pl.grid = (int)(M < cap ? M : cap);
    } else {
        int64_t t = ceil_div(H, 32) * 32;
        if (t > kMaxThreads) t = kMaxThreads;
        pl.threads = (int)t;
        const int per_sm = caps.max_threads_per_sm / pl.threads > 0 ? caps.max_threads_per_sm / pl.threads : 1;
        const int64_t cap = (int64_t)caps.num_sms * per_sm;
        const int64_t g = M < cap ? M : cap;
        pl.grid = (int)(g > 0 ? g : 1);
    }
    return pl;
}
}  // namespace

extern "C" arf_status_t arf_supports(arf_workspace_t ws, arf_pattern_t pattern, int W, int64_t M, int64_t H,
                                     arf_dtype_t dtype) {
    if (!valid_pattern(pattern) || !valid_dtype(dtype)) return ARF_ERR_INVALID_ARG;
    if (H <= 0 || M < 0) return ARF_ERR_INVALID_ARG;
    if (W < 1 || W > ARF_MAX_W) return ARF_ERR_UNSUPPORTED;
    if (H > ARF_MAX_H) return ARF_ERR_UNSUPPORTED;
    (void)ws;
    // [M,H] indices and the chunk count stay far inside int64
    if (M > ((int64_t)1 << 40) / H) return ARF_ERR_UNSUPPORTED;
    return ARF_OK;
}

namespace {

// The measured plan table (arf_plan_table.inc, written by plan_table.py
// from cold timings on one device): for a device with exactly these
// capabilities, a pattern, dtype, W, H and a range of M, a plan shape and a
// rule for its grid. Threads per block, cluster size and grid come from the
// device (flashinfer PR #1507 "update allreduce to match trtllm",
// Highlights), chosen per shape from measurements (vLLM PR #53318 "Tune
// FlashInfer all-reduce selection on SM103", Scope).
struct PlanTableRow {
    int num_sms, max_cluster, max_threads_per_sm, max_smem_per_block;
    int pattern, dtype, W;
    int64_t H, m_lo, m_hi;
    int path, threads, vpt, cluster, w_spec, stages;
    int grid_rule;  // PlanGridRule
    int per_sm;     // CTAs per SM (resident and tiles rules)
};

enum PlanGridRule {
    kGridRows = 0,      // M * cluster: one CTA (or cluster) per row
    kGridResident = 1,  // min(M, per_sm * SMs / cluster) * cluster
    kGridChunks = 2,    // ceil(M * H / 8 / (threads * vpt)): flat kAllReduce
    kGridTiles = 3,     // min(ceil(H / threads) * M, per_sm * SMs): elementwise kAllReduce
};

const PlanTableRow kPlanTable[] = {
#include "arf_plan_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0},  // end
};

// The table's plan for this call, if a row covers it and its plan passes
// arf_plan_check.
bool table_plan(const arf_device_caps_t& caps, arf_pattern_t pattern, int W, int64_t M, int64_t H,
                arf_dtype_t dtype, arf_plan_t* out) {
    for (const PlanTableRow& r : kPlanTable) {
        if (r.num_sms == 0) break;
        if (r.num_sms != caps.num_sms || r.max_cluster != caps.max_cluster ||
            r.max_threads_per_sm != caps.max_threads_per_sm || r.max_smem_per_block != caps.max_smem_per_block)
            continue;
        if (r.pattern != (int)pattern || r.dtype != (int)dtype || r.W != W || r.H != H || M < r.m_lo || M > r.m_hi)
            continue;
        arf_plan_t pl = {};
        pl.path = r.path;
        pl.threads = r.threads;
        pl.vpt = r.vpt;
        pl.cluster = r.cluster;
        pl.w_spec = r.w_spec;
        pl.stages = r.stages;
        const int64_t cs = r.cluster > 0 ? r.cluster : 1;
        int64_t g;
        switch (r.grid_rule) {
            case kGridRows: g = M * cs; break;
            case kGridResident: {
                int64_t n = (int64_t)r.per_sm * caps.num_sms / cs;
                if (n < 1) n = 1;
                g = (M < n ? M : n) * cs;
                break;
            }
            case kGridChunks: g = ceil_div(M * H / 8, (int64_t)r.threads * r.vpt); break;
            case kGridTiles: {
                g = ceil_div(H, r.threads) * M;
                const int64_t cap = (int64_t)r.per_sm * caps.num_sms;
                if (g > cap) g = cap;
                break;
            }
            default: return false;
        }
        const int64_t gmax = (int64_t)(INT32_MAX / cs) * cs;
        if (g < 1) g = 1;
        if (g > gmax) g = gmax;
        pl.grid = (int)g;
        if (arf_plan_check(&caps, &pl, pattern, W, M, H, dtype) != ARF_OK) return false;
        *out = pl;
        return true;
    }
    return false;
}

}  // namespace

extern "C" arf_status_t arf_plan_for_caps(const arf_device_caps_t* caps, arf_pattern_t pattern, int W,
                                          int64_t M, int64_t H, arf_dtype_t dtype, arf_plan_t* plan_out) {
    if (!caps || !plan_out) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(nullptr, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (caps->num_sms < 1 || caps->max_threads_per_sm < 32 || caps->max_cluster < 1) return ARF_ERR_INVALID_ARG;
    // A measured plan for this device and shape, where the table has one;
    // else the closed-form rules.
    if (table_plan(*caps, pattern, W, M, H, dtype, plan_out)) return ARF_OK;
    return arf_plan_rules(caps, pattern, W, M, H, dtype, plan_out);
}

extern "C" arf_status_t arf_plan_rules(const arf_device_caps_t* caps, arf_pattern_t pattern, int W, int64_t M,
                                       int64_t H, arf_dtype_t dtype, arf_plan_t* plan_out) {
    if (!caps || !plan_out) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(nullptr, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (caps->num_sms < 1 || caps->max_threads_per_sm < 32 || caps->max_cluster < 1) return ARF_ERR_INVALID_ARG;
    const int w_spec = arf::w_spec_compiled(W) ? W : 0;
    arf_plan_t pl = {};
    if (H % 8 != 0 || (pattern == ARF_AR_RESIDUAL_RMSNORM && H > max_rms_row(caps->max_cluster))) {
        // no 16-byte chunking possible, or a row longer than the device's
        // clusters hold: the elementwise kernels
        pl = elem_plan(*caps, pattern, M, H);
    } else if (pattern == ARF_ALLREDUCE) {
        // One pass over all chunks (no grid-stride trips). Bandwidth sizes:
        // 256-thread CTAs with 2 chunks per thread (4 for W <= 2) where the
        // rank count is compiled in with W <= 8; measured on GB300 for W = 8,
        // H = 7168: M = 1024 24.0 -> 23.0 us, M = 2048 40.0 -> 39.2 us against
        // one chunk per thread. Sizes below two device-fulls of chunks
        // (latency-bound): 128-thread CTAs with the same chunks per thread,
        // the fastest shape in measured sweeps of decode-size calls.
        const int64_t nchunks = M * H / 8;
        const bool small = nchunks < (int64_t)caps->num_sms * caps->max_threads_per_sm * 2;
        int u = 1;
        if (w_spec > 0) u = w_spec <= 2 ? 4 : 2;
        while (!arf::flat_unroll_compiled(w_spec, u)) u /= 2;
        pl.path = ARF_PATH_FLAT;
        pl.threads = small ? 128 : 256;
        pl.vpt = u;
        pl.cluster = 1;
        pl.w_spec = w_spec;
        const int64_t need = ceil_div(nchunks, (int64_t)pl.threads * u);
        pl.grid = (int)(need < 1 ? 1 : (need > INT32_MAX ? INT32_MAX : need));
    } else {
        // One CTA per row with the fewest 16-byte chunks per thread that keep
        // it at <= 512 threads (the kernel then keeps a whole row of loads in
        // flight per thread, and the next row's across the row barrier, when
        // VPT*(W+1) <= 18). Only decode-size batches of few, wide rows split a
        // row over a cluster: one chunk per thread, 4-8 CTAs per row, so that
        // the few rows still spread over several SMs.
        const int C = (int)(H / 8);
        int cs = 1, vpt = 1;
        while (vpt < 8 && ceil_div(C, vpt) > kMaxThreads) vpt *= 2;
        if (M > 0 && M < 16 && C >= 512 && caps->max_cluster > 1) {
            vpt = 1;
            cs = 2;
            while (cs < 8 && cs < caps->max_cluster && (int64_t)cs * M < 32) cs *= 2;
        }
        // Rows longer than one CTA holds (H > 32768): the smallest cluster
        // that keeps a CTA's slice at <= 2048 chunks (4 per thread), or the
        // largest the device has.
        if (C > kMaxThreads * 8) {
            int big = 2;
            while (big < caps->max_cluster && big < 16 && ceil_div(C, big) > kMaxThreads * 4) big *= 2;
            if (big > cs) cs = big;
            vpt = 1;
        }
        pl = rms_plan(*caps, w_spec, M, H, cs, vpt);
        // One CTA per row without the register prefetch (rank count not
        // compiled in, or too many vectors per thread): the bulk-copy ring
        // keeps the loads in flight instead, for up to 12 ranks (wider ring
        // slots leave too little shared memory for two of them). Measured on
        // GB300 (fraction of the copy peak, row kernel -> bulk): W = 3, M =
        // 2000: 0.49 -> 0.88; W = 5: 0.61 -> 0.85; W = 12: 0.61 -> 0.73;
        // W = 4, H = 32768: 0.65 -> 0.81. With the prefetch the row kernel
        // stays ahead (W = 4, M = 1989: 1.03 vs 0.93).
        // fp16 rows of 2 chunks per thread with few ranks, once every CTA
        // loops over several rows: the prefetching fp16 instances then stall
        // on their loads far more than the bf16 ones (W = 2, M = 3315: 50.4
        // vs 38.8 us, same instruction count and DRAM bytes, whatever the
        // data); with one row per CTA they match bf16. Measured crossover
        // (fp16, H = 7168, row -> bulk): W <= 2 ties from M = 2 SMs and wins
        // from M = 800 (W = 2, M = 1024: 20.2 -> 16.4 us); W = 4 loses at
        // M = 304 (10.4 vs 12.2 us), ties to M = 1500 and wins from 8 SMs'
        // worth (M = 2400: 40.8 -> 38.1 us; M = 5851: 99.9 -> 84.4 us).
        const int64_t sms = caps->num_sms;
        // W = 2 and 4 (two chunks per thread, prefetching): one CTA per row,
        // grid = M, in the one-row form. Its smaller register footprint lets
        // CTAs share an SM, which replaces the in-CTA prefetch, and it has no
        // fp16 penalty. Measured (H = 7168, cold): W = 2, M = 3315 bf16 39.1
        // -> 37.7 us, fp16 50.6 -> 38.7 us; W = 4, M = 5851 bf16 83.9 ->
        // 83.0 us, fp16 100.2 -> 83.3 us; W = 4, M = 1989 fp16 35.2 -> 29.0
        // us. W = 8 (53.8 vs 46.4 us) and W = 1 (49.1 vs 43.3 us) keep the
        // row loop.
        if (one_row_grid_wanted(pl, W)) pl.grid = (int)(M < INT32_MAX ? M : INT32_MAX);
        const bool fp16_rows = dtype == ARF_FP16 && pl.vpt == 2 && W == 1 && M >= 2 * sms;
        // Rows longer than one CTA holds (a cluster per row) once there are
        // rows for half the SMs: the bulk ring, where its row buffer and two
        // ring slots fit. Measured on GB300 (cold, cluster -> bulk): W = 2,
        // H = 32776, M = 76 19.2 -> 15.8 us, M = 2048 280.7 -> 107.6 us; W = 8,
        // M = 608 85.7 -> 77.1 us; W = 4, H = 65536, M = 152 31.6 -> 27.7 us,
        // but M = 512 84.1 -> 92.8 us (one CTA per SM). Fewer rows keep the
        // cluster (W = 4, H = 65536, M = 64: 16.5 vs 24.6 us). Those figures
        // are for blocks of 512 chunks; rows whose buffer leaves room only for
        // blocks narrower than 256 chunks keep the cluster too.
        const bool long_rows = pl.path == ARF_PATH_CLUSTER && C > kMaxThreads * 8 && 2 * M >= sms;
        if ((pl.path == ARF_PATH_ROW && (!arf::rms_prefetches(pl.w_spec, pl.vpt) || fp16_rows)) || long_rows) {
            arf_plan_t b;
            if (W <= kBulkMaxRanks && bulk_plan(*caps, w_spec, W, M, H, &b) && (!long_rows || b.threads >= 256))
                pl = b;
        }
        // The streaming kernel (ARF_PATH_ASYNC) is not chosen: measured on
        // GB300 it keeps fewer bytes in flight than the row kernel's register
        // prefetch (8 warps per SM issuing per-thread copies), e.g. 107 us vs
        // 83 us in-kernel for W=4, M=5851, H=7168. It stays available to
        // explicit plans.
    }
    *plan_out = pl;
    return ARF_OK;
}

extern "C" arf_status_t arf_plan_check(const arf_device_caps_t* caps, const arf_plan_t* pl, arf_pattern_t pattern,
                                       int W, int64_t M, int64_t H, arf_dtype_t dtype) {
    if (!caps || !pl) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(nullptr, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (pl->w_spec != 0 && pl->w_spec != W) return ARF_ERR_UNSUPPORTED;
    if (!arf::w_spec_compiled(pl->w_spec)) return ARF_ERR_UNSUPPORTED;
    if (pl->threads < 32 || pl->threads > kMaxThreads || pl->threads % 32 != 0) return ARF_ERR_UNSUPPORTED;
    if (pl->cluster < 1 || pl->grid < 1 || pl->grid % pl->cluster != 0) return ARF_ERR_UNSUPPORTED;
    if (pl->path == ARF_PATH_ELEM) {
        if (pl->cluster != 1 || pl->vpt != 1 || pl->stages != 0 || pl->w_spec != 0) return ARF_ERR_UNSUPPORTED;
        return ARF_OK;
    }
    // The 16-byte kernels need whole chunks. kAllReduce is elementwise, so
    // the flat kernel also takes H % 8 != 0 when M * H is a multiple of 8:
    // contiguous tensors are then one range of whole chunks (the call checks
    // the layout and takes the elementwise kernel otherwise).
    const bool flat_range = pattern == ARF_ALLREDUCE && pl->path == ARF_PATH_FLAT && (M * H) % 8 == 0;
    if (H % 8 != 0 && !flat_range) return ARF_ERR_UNSUPPORTED;
    if (pl->path == ARF_PATH_ASYNC) {
        if (pattern != ARF_AR_RESIDUAL_RMSNORM || pl->w_spec == 0 || pl->w_spec != W) return ARF_ERR_UNSUPPORTED;
        if (pl->threads != arf::kAsyncCtaThreads || pl->cluster != 1 || pl->vpt != 1) return ARF_ERR_UNSUPPORTED;
        if (pl->stages < 2 || pl->stages > 8) return ARF_ERR_UNSUPPORTED;
        const size_t need = arf::async_dyn_smem(W, pl->stages, (int)(H / 8)) + arf::kAsyncStaticSmem;
        if (need > (size_t)caps->max_smem_per_block) return ARF_ERR_UNSUPPORTED;
        return ARF_OK;
    }
    if (pl->path == ARF_PATH_BULK) {
        if (pl->cluster != 1 || pl->vpt != 1) return ARF_ERR_UNSUPPORTED;
        if (pl->stages < 2 || pl->stages > arf::kBulkMaxStages) return ARF_ERR_UNSUPPORTED;
        const size_t need = (pattern == ARF_ALLREDUCE ? arf::bulk_ar_dyn_smem(W, pl->stages, pl->threads)
                                                      : arf::bulk_dyn_smem(W, pl->stages, pl->threads, (int)(H / 8))) +
                            arf::kBulkStaticSmem;
        if (need > (size_t)caps->max_smem_per_block) return ARF_ERR_UNSUPPORTED;
        return ARF_OK;
    }
    if (pl->stages != 0) return ARF_ERR_UNSUPPORTED;
    if (pattern == ARF_ALLREDUCE) {
        if (pl->path != ARF_PATH_FLAT || pl->cluster != 1) return ARF_ERR_UNSUPPORTED;
        if (!(pl->vpt == 1 || pl->vpt == 2 || pl->vpt == 4) || !arf::flat_unroll_compiled(pl->w_spec, pl->vpt))
            return ARF_ERR_UNSUPPORTED;
    } else {
        if (pl->path == ARF_PATH_ROW) {
            if (pl->cluster != 1) return ARF_ERR_UNSUPPORTED;
        } else if (pl->path == ARF_PATH_CLUSTER) {
            const int c = pl->cluster;
            if (!(c == 2 || c == 4 || c == 8 || c == 16) || c > caps->max_cluster) return ARF_ERR_UNSUPPORTED;
        } else {
            return ARF_ERR_UNSUPPORTED;
        }
        if (!arf::rms_vpt_compiled(pl->vpt)) return ARF_ERR_UNSUPPORTED;
        const int64_t slice = ceil_div(H / 8, pl->cluster);
        if ((int64_t)pl->threads * pl->vpt < slice) return ARF_ERR_UNSUPPORTED;
    }
    return ARF_OK;
}

namespace {

cudaError_t max_active_clusters(arf_dtype_t dt, const arf_plan_t& pl, int* n, bool f32p = false) {
    return dt == ARF_BF16 ? arf::rms_max_active_clusters_bf16(pl, n, f32p)
                          : arf::rms_max_active_clusters_fp16(pl, n, f32p);
}

cudaError_t max_active_blocks(arf_dtype_t dt, const arf_plan_t& pl, int64_t H, int W, int* n) {
    const int C = (int)(H / 8);
    return dt == ARF_BF16 ? arf::rms_max_active_blocks_bf16(pl, C, W, n) : arf::rms_max_active_blocks_fp16(pl, C, W, n);
}

// The planner's plan, with the cluster size lowered until the cluster kernel
// instance can actually be made resident on this device. During stream
// capture no occupancy query is made: the plan then rests on the cluster
// limit probed at workspace creation, and it is not cached, so the next call
// outside a capture makes the checked plan for the same key.
arf_status_t device_plan(arf_workspace_t ws, arf_pattern_t pattern, int W, int64_t M, int64_t H,
                         arf_dtype_t dtype, arf_plan_t* out, bool capturing = false) {
    const auto key = std::make_tuple((int)pattern, W, M, H, (int)dtype);
    {
        std::lock_guard<std::mutex> lk(ws->mu);
        auto it = ws->plans.find(key);
        if (it != ws->plans.end()) {
            *out = it->second;
            return ARF_OK;
        }
    }
    arf_plan_t pl;
    arf_status_t st = arf_plan_for_caps(&ws->caps, pattern, W, M, H, dtype, &pl);
    if (st != ARF_OK) return st;
    // A plan from the measured table was timed as it stands on a device with
    // these capabilities: it is used without the refinements below.
    arf_plan_t tp;
    const bool refine = !capturing && !table_plan(ws->caps, pattern, W, M, H, dtype, &tp);
    if (refine && pl.path == ARF_PATH_ASYNC) {
        int b = 0;
        cudaError_t e = max_active_blocks(dtype, pl, H, W, &b);
        if (e != cudaSuccess || b < 1) {  // the ring does not fit: one CTA per row instead
            (void)cudaGetLastError();
            pl = row_plan(ws->caps, pl.w_spec, M, H);
        }
    }
    if (refine && pl.path == ARF_PATH_BULK) {
        int b = 0;
        cudaError_t e = max_active_blocks(dtype, pl, H, W, &b);
        if (e == cudaSuccess && b > 0) {
            const int64_t cap = (int64_t)ws->caps.num_sms * b;
            if (cap < pl.grid) pl.grid = (int)cap;
        } else {  // the ring does not fit after all: one CTA per row
            (void)cudaGetLastError();
            pl = row_plan(ws->caps, pl.w_spec, M, H);
        }
    }
    while (refine && pl.path == ARF_PATH_CLUSTER) {
        int n = 0;
        cudaError_t e = max_active_clusters(dtype, pl, &n);
        if (e == cudaSuccess && n > 0) {
            // no more clusters than can be resident at once (rows loop)
            if ((int64_t)n * pl.cluster < pl.grid) pl.grid = n * pl.cluster;
            break;
        }
        (void)cudaGetLastError();
        pl = rms_plan(ws->caps, pl.w_spec, M, H, pl.cluster / 2, pl.vpt);
    }
    // a fallback that cannot cover the row (a long row on a device that holds
    // only smaller clusters) is refused rather than launched
    st = arf_plan_check(&ws->caps, &pl, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (refine && pl.path == ARF_PATH_ROW && !one_row_grid_wanted(pl, W)) {
        int b = 0;
        cudaError_t e = max_active_blocks(dtype, pl, H, W, &b);
        if (e == cudaSuccess && b > 0) {
            const int64_t cap = (int64_t)ws->caps.num_sms * b;
            if (cap < pl.grid) pl.grid = (int)cap;
        } else {
            (void)cudaGetLastError();
        }
    }
    if (ws->log)
        std::fprintf(stderr, "[arf] plan %s W=%d M=%lld H=%lld %s: path=%s threads=%d vpt=%d cluster=%d grid=%d w_spec=%d stages=%d\n",
                     pattern_name(pattern), W, (long long)M, (long long)H, dtype == ARF_BF16 ? "bf16" : "fp16",
                     path_name(pl.path), pl.threads, pl.vpt, pl.cluster, pl.grid, pl.w_spec, pl.stages);
    if (!capturing) {
        std::lock_guard<std::mutex> lk(ws->mu);
        ws->plans[key] = pl;
    }
    *out = pl;
    return ARF_OK;
}

// Row strides in elements and the partial type of one call.
struct Layout {
    int64_t ldp, ldr, ldo, ldro;
    bool f32p;
    bool vec_ok;    // the 16-byte kernels can take it
    bool range_ok;  // kAllReduce: contiguous 16-bit tensors, M*H a multiple of 8 and out
                    // 16-byte aligned, so the flat kernel can run one range of chunks
};

bool odd(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; }

// Everything arf_run checks before it launches (sizes already supported),
// and whether the 16-byte kernels can take the layout.
arf_status_t check_call(arf_pattern_t pattern, const arf_run_opts_t* opts, bool by_value,
                        const void* const* partials, const void* residual, const void* gamma, float eps,
                        const void* out, const void* residual_out, int64_t M, int64_t H, Layout* ly) {
    if (!partials || !out) return ARF_ERR_INVALID_ARG;
    const bool rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
    ly->ldp = opts && opts->ld_partials ? opts->ld_partials : H;
    ly->ldr = opts && opts->ld_residual ? opts->ld_residual : H;
    ly->ldo = opts && opts->ld_out ? opts->ld_out : H;
    ly->ldro = opts && opts->ld_residual_out ? opts->ld_residual_out : H;
    ly->f32p = opts && opts->partials_f32;
    if (ly->ldp < H || ly->ldo < H) return ARF_ERR_INVALID_ARG;
    if (rms) {
        if (!residual || !gamma || !residual_out) return ARF_ERR_INVALID_ARG;
        if (!std::isfinite(eps) || eps < 0.0f) return ARF_ERR_INVALID_ARG;
        if (out == residual_out) return ARF_ERR_INVALID_ARG;
        if (ly->ldr < H || ly->ldro < H) return ARF_ERR_INVALID_ARG;
        if (residual == residual_out && ly->ldr != ly->ldro) return ARF_ERR_INVALID_ARG;
        if (odd(residual) || odd(gamma) || odd(residual_out)) return ARF_ERR_UNSUPPORTED;
    }
    // every tensor's extent, M rows of its stride, stays inside the bound
    // arf_supports puts on M*H, so that no index computation can overflow
    const int64_t max_ld = ((int64_t)1 << 40) / (M > 0 ? M : 1);
    if (ly->ldp > max_ld || ly->ldo > max_ld || (rms && (ly->ldr > max_ld || ly->ldro > max_ld)))
        return ARF_ERR_UNSUPPORTED;
    if (odd(out)) return ARF_ERR_UNSUPPORTED;
    if (!by_value && (reinterpret_cast<uintptr_t>(partials) & 7u) != 0) return ARF_ERR_UNSUPPORTED;
    bool v = H % 8 == 0 && ly->ldp % 8 == 0 && ly->ldo % 8 == 0 && aligned16(out);
    if (rms) v = v && ly->ldr % 8 == 0 && ly->ldro % 8 == 0 && aligned16(residual) && aligned16(gamma) &&
                 aligned16(residual_out);
    ly->vec_ok = v;
    ly->range_ok = !rms && !ly->f32p && ly->ldp == H && ly->ldo == H && (M * H) % 8 == 0 && aligned16(out);
    return ARF_OK;
}

// Whether the 16-byte kernel of plan `pl` can take this call's layout: the
// flat kAllReduce kernel on rows of H % 8 != 0 runs the whole contiguous
// [M,H] as one range; every other 16-byte kernel needs 16-byte rows.
bool layout_fits(const arf_plan_t& pl, arf_pattern_t pattern, int64_t H, const Layout& L) {
    if (pattern == ARF_ALLREDUCE && pl.path == ARF_PATH_FLAT && H % 8 != 0) return L.range_ok;
    return L.vec_ok;
}

// Current device and stream device must be the workspace's. While `stream`
// is being captured into a graph, only capture-safe queries are made (the
// stream's device cannot be queried then; *capturing reports it).
arf_status_t check_device(arf_workspace_t ws, cudaStream_t stream, bool* capturing) {
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    if (cur != ws->device) return ARF_ERR_DEVICE_MISMATCH;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    *capturing = cs != cudaStreamCaptureStatusNone;
    if (*capturing) return ARF_OK;
    int sdev = -1;
    e = cudaStreamGetDevice(stream, &sdev);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    if (sdev != ws->device) return ARF_ERR_DEVICE_MISMATCH;
    return ARF_OK;
}

void fill_common(arf::LaunchCommon& lc, const void* const* partials, int W, bool by_value, bool pdl) {
    if (by_value) {
        for (int r = 0; r < W; ++r) lc.ptrs[r] = partials[r];
        lc.partials = nullptr;
    } else {
        lc.partials = partials;
    }
    lc.by_value = by_value ? 1 : 0;
    lc.pdl = pdl ? 1 : 0;
}

arf_status_t launch(arf_workspace_t ws, const arf_plan_t& pl, arf_pattern_t pattern, int W,
                    const void* const* partials, bool by_value, bool pdl, const void* residual, const void* gamma,
                    float eps, void* out, void* residual_out, int64_t M, int64_t H, arf_dtype_t dtype,
                    const Layout& L, cudaStream_t stream, const arf_run_opts_t* opts) {
    cudaError_t e;
    const bool bf = dtype == ARF_BF16;
    if (pl.path == ARF_PATH_ELEM) {
        arf::ElemParams p = {};
        fill_common(p.lc, partials, W, by_value, pdl);
        p.residual = static_cast<const unsigned short*>(residual);
        p.gamma = static_cast<const unsigned short*>(gamma);
        p.out = static_cast<unsigned short*>(out);
        p.residual_out = static_cast<unsigned short*>(residual_out);
        p.M = M;
        p.ldp = L.ldp;
        p.ldr = L.ldr;
        p.ldo = L.ldo;
        p.ldro = L.ldro;
        p.H = (int)H;
        p.W = W;
        p.eps = eps;
        const bool rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
        // 16-byte vectors need every tensor's row r to start at the same
        // offset modulo 8 elements (strides congruent mod 8) from 16-byte
        // aligned bases; contiguous tensors are also one flat range.
        const int64_t res = ((L.ldp % 8) + 8) % 8;
        bool vec = !L.f32p && aligned16(out) && L.ldo % 8 == res;
        if (rms) vec = vec && aligned16(residual) && aligned16(residual_out) && L.ldr % 8 == res && L.ldro % 8 == res;
        const bool contiguous = L.ldp == H && L.ldo == H && (!rms || (L.ldr == H && L.ldro == H));
        p.flat_ok = !vec ? 0 : (contiguous ? 1 : 2);
        e = bf ? arf::launch_elem_bf16(p, pl, rms, stream, L.f32p) : arf::launch_elem_fp16(p, pl, rms, stream, L.f32p);
        if (e != cudaSuccess) return cuda_fail(ws, e);
        return ARF_OK;
    }
    // 16-byte vectors: 16-bit tensors have 8 elements per vector, binary32 partials 4
    arf::RowLayout rl;
    rl.ldp = L.f32p ? L.ldp / 4 : L.ldp / 8;
    rl.ldr = L.ldr / 8;
    rl.ldo = L.ldo / 8;
    rl.ldro = L.ldro / 8;
    if (pattern == ARF_ALLREDUCE && pl.path == ARF_PATH_BULK) {
        arf::RmsParams p = {};
        fill_common(p.lc, partials, W, by_value, pdl);
        p.ly = rl;
        p.out = static_cast<uint4*>(out);
        p.M = M;
        p.C = (int)(H / 8);
        p.H = (int)H;
        p.W = W;
        p.cs = 1;
        p.slice = p.C;
        p.stages = pl.stages;
        p.status = ws->wait_timeouts;
        p.spin_limit = opts && opts->wait_limit_cycles > 0 ? (long long)opts->wait_limit_cycles : arf::kBulkSpinLimit;
        p.hold_first = opts && opts->hold_first_copy ? 1 : 0;
        e = bf ? arf::launch_bulk_ar_bf16(p, pl, stream) : arf::launch_bulk_ar_fp16(p, pl, stream);
    } else if (pattern == ARF_ALLREDUCE) {
        arf::FlatParams p = {};
        fill_common(p.lc, partials, W, by_value, pdl);
        p.ly = rl;
        p.out = static_cast<uint4*>(out);
        p.nchunks = M * H / 8;
        p.M = M;
        p.C = (int)(H / 8);
        p.strided = (L.ldp != H || L.ldo != H) ? 1 : 0;
        p.W = W;
        e = bf ? arf::launch_flat_bf16(p, pl, stream, L.f32p) : arf::launch_flat_fp16(p, pl, stream, L.f32p);
    } else {
        arf::RmsParams p = {};
        fill_common(p.lc, partials, W, by_value, pdl);
        p.ly = rl;
        p.residual = static_cast<const uint4*>(residual);
        p.gamma = static_cast<const uint4*>(gamma);
        p.out = static_cast<uint4*>(out);
        p.residual_out = static_cast<uint4*>(residual_out);
        p.M = M;
        p.C = (int)(H / 8);
        p.H = (int)H;
        p.W = W;
        p.cs = pl.cluster;
        p.slice = (int)ceil_div(p.C, pl.cluster);
        p.stages = pl.stages;
        p.eps = eps;
        p.status = ws->wait_timeouts;
        p.spin_limit = opts && opts->wait_limit_cycles > 0 ? (long long)opts->wait_limit_cycles : arf::kBulkSpinLimit;
        p.hold_first = opts && opts->hold_first_copy ? 1 : 0;
        e = bf ? arf::launch_rms_bf16(p, pl, stream, L.f32p) : arf::launch_rms_fp16(p, pl, stream, L.f32p);
    }
    if (e != cudaSuccess) return cuda_fail(ws, e);
    return ARF_OK;
}

arf_status_t run_impl(arf_workspace_t ws, const arf_run_opts_t* opts, arf_pattern_t pattern, int W,
                      const void* const* partials, const void* residual, const void* gamma, float eps, void* out,
                      void* residual_out, int64_t M, int64_t H, arf_dtype_t dtype, void* stream_v) {
    if (!ws) return ARF_ERR_INVALID_ARG;
    const arf_plan_t* forced = opts ? opts->plan : nullptr;
    const bool by_value = opts && opts->partials_by_value;
    const int pdl_opt = opts ? opts->pdl : 0;
    if (pdl_opt < 0 || pdl_opt > 2) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(ws, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (forced) {
        st = arf_plan_check(&ws->caps, forced, pattern, W, M, H, dtype);
        if (st != ARF_OK) return st;
    }
    if (M == 0) return ARF_OK;
    Layout L;
    st = check_call(pattern, opts, by_value, partials, residual, gamma, eps, out, residual_out, M, H, &L);
    if (st != ARF_OK) return st;
    if (forced && forced->path != ARF_PATH_ELEM) {
        // an explicit 16-byte plan needs a layout those kernels take; binary32
        // partials exist only in the run-time-W instances of the row/flat kernels
        if (!layout_fits(*forced, pattern, H, L)) return ARF_ERR_UNSUPPORTED;
        if (L.f32p && (forced->w_spec != 0 || forced->path == ARF_PATH_ASYNC || forced->path == ARF_PATH_BULK))
            return ARF_ERR_UNSUPPORTED;
    }
    if (by_value) {
        for (int r = 0; r < W; ++r)
            if (!partials[r]) return ARF_ERR_INVALID_ARG;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    bool capturing = false;
    st = check_device(ws, stream, &capturing);
    if (st != ARF_OK) return st;
    arf_plan_t pl;
    if (forced) {
        pl = *forced;
        if (pl.path == ARF_PATH_CLUSTER && !capturing) {
            // a cluster shape must fit the device: no launch that cannot start
            int n = 0;
            cudaError_t e = max_active_clusters(dtype, pl, &n, L.f32p);
            if (e != cudaSuccess) return cuda_fail(ws, e);
            if (n < 1) return ARF_ERR_UNSUPPORTED;
        }
        if ((pl.path == ARF_PATH_ASYNC || pl.path == ARF_PATH_BULK) && !capturing) {
            int b = 0;
            cudaError_t e = pattern == ARF_ALLREDUCE
                                ? (dtype == ARF_BF16 ? arf::bulk_ar_max_active_blocks_bf16(pl, W, &b)
                                                     : arf::bulk_ar_max_active_blocks_fp16(pl, W, &b))
                                : max_active_blocks(dtype, pl, H, W, &b);
            if (e != cudaSuccess) return cuda_fail(ws, e);
            if (b < 1) return ARF_ERR_UNSUPPORTED;
        }
    } else {
        st = device_plan(ws, pattern, W, M, H, dtype, &pl, capturing);
        if (st != ARF_OK) return st;
        if (pl.path != ARF_PATH_ELEM) {
            if (!layout_fits(pl, pattern, H, L)) {
                pl = elem_plan(ws->caps, pattern, M, H);  // strides or alignment the vectors cannot take
            } else if (L.f32p) {
                // binary32 partials: the run-time W instances of the row and
                // flat kernels (the bulk ring holds 16-bit rows)
                if (pl.path == ARF_PATH_BULK) pl = row_plan(ws->caps, 0, M, H);
                pl.w_spec = 0;
                if (pl.path == ARF_PATH_CLUSTER && !capturing) {
                    int n = 0;
                    if (max_active_clusters(dtype, pl, &n, true) != cudaSuccess || n < 1) {
                        (void)cudaGetLastError();
                        pl = elem_plan(ws->caps, pattern, M, H);
                    }
                }
            }
        }
    }
    // Programmatic dependent launch: by default for latency-bound launches
    // (grid x threads at most 1/16 of the device's resident threads), where
    // overlapping this launch with the previous kernel's tail is the gain;
    // larger grids would hold SM slots with waiting CTAs.
    const bool pdl = pdl_opt == 1 || (pdl_opt == 0 && (int64_t)pl.grid * pl.threads * 16 <=
                                                          (int64_t)ws->caps.num_sms * ws->caps.max_threads_per_sm);
    return launch(ws, pl, pattern, W, partials, by_value, pdl, residual, gamma, eps, out, residual_out, M, H, dtype,
                  L, stream, opts);
}

}  // namespace

namespace {

// Candidate plans around the planner's: every compiled shape near it that
// arf_plan_check accepts on this device.
std::vector<arf_plan_t> tune_candidates(const arf_device_caps_t& caps, const arf_plan_t& base,
                                        arf_pattern_t pattern, int W, int64_t M, int64_t H, arf_dtype_t dtype) {
    std::vector<arf_plan_t> out;
    auto add = [&](const arf_plan_t& p) {
        if (arf_plan_check(&caps, &p, pattern, W, M, H, dtype) != ARF_OK) return;
        for (const auto& q : out)
            if (std::memcmp(&q, &p, sizeof p) == 0) return;
        out.push_back(p);
    };
    add(base);
    if (base.path == ARF_PATH_ELEM) {
        // each CTA width with the base grid, and with as many of its CTAs as
        // the SMs hold by thread count (capped at the rows, or kAllReduce's
        // row tiles): the shapes that won the measured sweeps were of the
        // second kind (128 x 8 SMs, 256 x 4 SMs, 512 x 2 SMs)
        for (int t : {64, 128, 256, 512}) {
            arf_plan_t p = base;
            p.threads = t;
            add(p);
            const int per_sm = caps.max_threads_per_sm / t > 0 ? caps.max_threads_per_sm / t : 1;
            const int64_t full = (int64_t)caps.num_sms * per_sm;
            const int64_t units = pattern == ARF_ALLREDUCE ? ceil_div(H, t) * M : M;
            const int64_t g = units < full ? units : full;
            p.grid = (int)(g > 0 ? g : 1);
            add(p);
        }
        return out;
    }
    const int w_specs[2] = {base.w_spec, 0};
    if (pattern == ARF_ALLREDUCE) {
        const int64_t nchunks = M * H / 8;
        for (int ws : w_specs)
            for (int t : {128, 256, 512})
                for (int u : {1, 2, 4}) {
                    arf_plan_t p = base;
                    p.w_spec = ws;
                    p.threads = t;
                    p.vpt = u;
                    const int64_t need = ceil_div(nchunks, (int64_t)t * u);
                    p.grid = (int)(need < 1 ? 1 : (need > INT32_MAX ? INT32_MAX : need));
                    add(p);
                }
        return out;
    }
    for (int ws : w_specs)
        for (int cs : {1, 2, 4, 8, 16}) {
            if (cs > caps.max_cluster) continue;
            for (int vpt : {1, 2, 4, 8}) {
                arf_plan_t p = rms_plan(caps, ws, M, H, cs, vpt);
                if (p.vpt != vpt) continue;  // rms_plan raised it: covered by a larger vpt
                add(p);
            }
        }
    // the bulk-copy ring: block widths, depths, one or two CTAs per SM
    for (int ws : w_specs)
        for (int t : {128, 256, 512})
            for (int s : {2, 3, 4})
                for (int per : {1, 2}) {
                    arf_plan_t p = {};
                    p.path = ARF_PATH_BULK;
                    p.threads = t;
                    p.vpt = 1;
                    p.cluster = 1;
                    p.w_spec = ws;
                    p.stages = s;
                    const int64_t g = (int64_t)caps.num_sms * per;
                    p.grid = (int)(M < g ? (M > 0 ? M : 1) : g);
                    add(p);
                }
    return out;
}

}  // namespace

extern "C" arf_status_t arf_workspace_autotune(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                               const void* const* partials_dev, const void* residual,
                                               const void* gamma, float eps, void* out, void* residual_out,
                                               int64_t M, int64_t H, arf_dtype_t dtype, int reps, void* stream,
                                               arf_plan_t* plan_out, float* us_out) {
    if (!ws) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(ws, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (reps <= 0) reps = 20;
    arf_plan_t base;
    st = device_plan(ws, pattern, W, M, H, dtype, &base);
    if (st != ARF_OK) return st;
    if (M == 0) {
        if (plan_out) *plan_out = base;
        if (us_out) *us_out = 0.0f;
        return ARF_OK;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return cuda_fail(ws, e);
    }
    arf_plan_t best = base;
    float best_us = -1.0f;
    for (const arf_plan_t& cand : tune_candidates(ws->caps, base, pattern, W, M, H, dtype)) {
        arf_run_opts_t o = {};
        o.plan = &cand;
        // warm-up; a plan this device cannot hold (UNSUPPORTED) is skipped
        st = run_impl(ws, &o, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype, stream);
        if (st == ARF_ERR_UNSUPPORTED) continue;
        if (st != ARF_OK) break;
        st = run_impl(ws, &o, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype, stream);
        if (st != ARF_OK) break;
        e = cudaEventRecord(e0, s);
        for (int i = 0; i < reps && e == cudaSuccess && st == ARF_OK; ++i)
            st = run_impl(ws, &o, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype,
                          stream);
        if (e == cudaSuccess) e = cudaEventRecord(e1, s);
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        float ms = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
        if (e != cudaSuccess || st != ARF_OK) break;
        const float us = ms * 1000.0f / (float)reps;
        if (best_us < 0.0f || us < best_us) {
            best_us = us;
            best = cand;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    if (st != ARF_OK && st != ARF_ERR_UNSUPPORTED) return st;
    {
        std::lock_guard<std::mutex> lk(ws->mu);
        ws->plans[std::make_tuple((int)pattern, W, M, H, (int)dtype)] = best;
    }
    if (ws->log)
        std::fprintf(stderr, "[arf] autotune %s W=%d M=%lld H=%lld: path=%s threads=%d vpt=%d cluster=%d grid=%d "
                     "w_spec=%d, %.3f us/call\n", pattern_name(pattern), W, (long long)M, (long long)H,
                     path_name(best.path), best.threads, best.vpt, best.cluster, best.grid, best.w_spec, best_us);
    if (plan_out) *plan_out = best;
    if (us_out) *us_out = best_us;
    return ARF_OK;
}

extern "C" arf_status_t arf_workspace_plan(arf_workspace_t ws, arf_pattern_t pattern, int W, int64_t M, int64_t H,
                                           arf_dtype_t dtype, arf_plan_t* plan_out) {
    if (!ws || !plan_out) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(ws, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    return device_plan(ws, pattern, W, M, H, dtype, plan_out);
}

// ---------------------------------------------------------------------------
// the epilogue
// ---------------------------------------------------------------------------

extern "C" arf_status_t arf_run(arf_workspace_t ws, arf_pattern_t pattern, int W, const void* const* partials_dev,
                                const void* residual, const void* gamma, float eps, void* out, void* residual_out,
                                int64_t M, int64_t H, arf_dtype_t dtype, void* stream) {
    return run_impl(ws, nullptr, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype,
                    stream);
}

extern "C" arf_status_t arf_run_ex(arf_workspace_t ws, const arf_run_opts_t* opts, arf_pattern_t pattern, int W,
                                   const void* const* partials, const void* residual, const void* gamma, float eps,
                                   void* out, void* residual_out, int64_t M, int64_t H, arf_dtype_t dtype,
                                   void* stream) {
    return run_impl(ws, opts, pattern, W, partials, residual, gamma, eps, out, residual_out, M, H, dtype, stream);
}

extern "C" arf_status_t arf_run_planned(arf_workspace_t ws, const arf_plan_t* plan, arf_pattern_t pattern, int W,
                                        const void* const* partials_dev, const void* residual, const void* gamma,
                                        float eps, void* out, void* residual_out, int64_t M, int64_t H,
                                        arf_dtype_t dtype, void* stream) {
    if (!plan) return ARF_ERR_INVALID_ARG;
    arf_run_opts_t opts = {};
    opts.plan = plan;
    return run_impl(ws, &opts, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype,
                    stream);
}

// ---------------------------------------------------------------------------
// host buffers
// ---------------------------------------------------------------------------

namespace arf {

void note_cuda_error(arf_workspace_t ws, cudaError_t e) { (void)cuda_fail(ws, e); }

__global__ void fill_pointer_array(const void** array, const char* first, int64_t stride, int W) {
    for (int r = threadIdx.x; r < W; r += blockDim.x) array[r] = first + (int64_t)r * stride;
}

cudaError_t launch_fill_pointer_array(const void** array, const char* first, int64_t stride, int W,
                                      cudaStream_t s) {
    fill_pointer_array<<<1, 64, 0, s>>>(array, first, stride, W);
    return cudaGetLastError();
}

}  // namespace arf

namespace {

// Staging layout, each region 256-byte aligned:
//   [pointer array: W x 8 B][P_0] ... [P_{W-1}][residual][gamma][out][residual_out]
struct Staging {
    size_t ptrs, p0, plane, residual, gamma, out, residual_out, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

Staging staging_layout(arf_pattern_t pattern, int W, int64_t M, int64_t H) {
    Staging s = {};
    const size_t plane = up256((size_t)M * (size_t)H * 2);
    const bool rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
    s.ptrs = 0;
    s.p0 = up256((size_t)W * sizeof(void*));
    s.plane = plane;
    size_t at = s.p0 + (size_t)W * plane;
    s.residual = at;
    if (rms) at += plane;
    s.gamma = at;
    if (rms) at += up256((size_t)H * 2);
    s.out = at;
    at += plane;
    s.residual_out = at;
    if (rms) at += plane;
    s.total = at;
    return s;
}

}  // namespace

namespace {

// Row blocks of arf_run_host's pipelined form: one per 4 MiB of an [M,H]
// tensor, at most 8; 1 = the plain form (copies in, kernel, copies out, all
// on the caller's stream). Host-to-device and device-to-host copies run at
// once only on separate streams; on GB300 (pinned memory over NVLink-C2C)
// one direction moves about 200 GB/s whatever the number of streams, both
// directions together 250-270 GB/s.
int host_pipeline_blocks(int64_t M, int64_t H) {
    const int64_t plane = M * H * 2;
    const int64_t b = plane / (4ll << 20);
    return (int)std::min<int64_t>(std::min<int64_t>(b, 8), M);
}

// Pipelined arf_run_host over `blocks` blocks of rows: block b's inputs are
// copied in on ws->h2d, its kernel runs on the caller's stream once they have
// landed, and its outputs are copied out on ws->d2h, so block b's outputs
// travel while block b+1's inputs do. The kernels take the partial pointers
// by value (each block's pointers are offsets into the staging planes). Both
// copy streams start after the caller's earlier work (ev_fork) and the
// caller's stream waits for the last copy out (ev_join), so the call is
// ordered with other work on `stream` as the plain form is, under stream
// capture too.
arf_status_t run_host_pipelined(arf_workspace_t ws, arf_pattern_t pattern, int W, const void* const* partials_host,
                                const void* residual_host, const void* gamma_host, float eps, void* out_host,
                                void* residual_out_host, int64_t M, int64_t H, arf_dtype_t dtype, char* base,
                                const Staging& L, int blocks, cudaStream_t stream) {
    const bool rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
    const size_t row = (size_t)H * 2;
    // whole multiples of 8 rows, so that every block starts on a 16-byte
    // boundary whatever H (the 16-byte kernels then take every block)
    const int64_t rows_per = ceil_div(ceil_div(M, blocks), 8) * 8;
    std::lock_guard<std::mutex> lock(ws->host_mu);
    cudaError_t e = cudaEventRecord(ws->ev_fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ws->h2d, ws->ev_fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ws->d2h, ws->ev_fork, 0);
    if (rms && e == cudaSuccess)
        e = cudaMemcpyAsync(base + L.gamma, gamma_host, row, cudaMemcpyHostToDevice, ws->h2d);
    arf_run_opts_t opts = {};
    opts.partials_by_value = 1;
    opts.pdl = 2;  // each kernel follows an event wait: nothing to overlap
    const void* ptrs[ARF_MAX_W];
    arf_status_t st = ARF_OK;
    for (int64_t r0 = 0; r0 < M && e == cudaSuccess && st == ARF_OK; r0 += rows_per) {
        const int64_t mb = std::min<int64_t>(rows_per, M - r0);
        const size_t off = (size_t)r0 * row, nb = (size_t)mb * row;
        for (int r = 0; r < W && e == cudaSuccess; ++r) {
            char* dst = base + L.p0 + (size_t)r * L.plane + off;
            e = cudaMemcpyAsync(dst, static_cast<const char*>(partials_host[r]) + off, nb, cudaMemcpyHostToDevice,
                                ws->h2d);
            ptrs[r] = dst;
        }
        if (rms && e == cudaSuccess)
            e = cudaMemcpyAsync(base + L.residual + off, static_cast<const char*>(residual_host) + off, nb,
                                cudaMemcpyHostToDevice, ws->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(ws->ev_in, ws->h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ws->ev_in, 0);
        if (e != cudaSuccess) break;
        st = run_impl(ws, &opts, pattern, W, ptrs, rms ? base + L.residual + off : nullptr,
                      rms ? base + L.gamma : nullptr, eps, base + L.out + off,
                      rms ? base + L.residual_out + off : nullptr, mb, H, dtype, stream);
        if (st != ARF_OK) break;
        e = cudaEventRecord(ws->ev_done, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ws->d2h, ws->ev_done, 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char*>(out_host) + off, base + L.out + off, nb, cudaMemcpyDeviceToHost,
                                ws->d2h);
        if (rms && e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char*>(residual_out_host) + off, base + L.residual_out + off, nb,
                                cudaMemcpyDeviceToHost, ws->d2h);
    }
    // Join both copy streams back into the caller's stream, also after a
    // failure part-way, so that no capture is left with an unjoined stream.
    cudaError_t j = cudaEventRecord(ws->ev_join, ws->h2d);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, ws->ev_join, 0);
    if (j == cudaSuccess) j = cudaEventRecord(ws->ev_join, ws->d2h);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, ws->ev_join, 0);
    if (e == cudaSuccess) e = j;
    if (st != ARF_OK) return st;
    if (e != cudaSuccess) return cuda_fail(ws, e);
    return ARF_OK;
}

}  // namespace

extern "C" size_t arf_host_staging_bytes(arf_pattern_t pattern, int W, int64_t M, int64_t H, arf_dtype_t dtype) {
    if (arf_supports(nullptr, pattern, W, M, H, dtype) != ARF_OK) return 0;
    return staging_layout(pattern, W, M, H).total;
}

extern "C" arf_status_t arf_run_host(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                     const void* const* partials_host, const void* residual_host,
                                     const void* gamma_host, float eps, void* out_host, void* residual_out_host,
                                     int64_t M, int64_t H, arf_dtype_t dtype, void* staging_dev,
                                     size_t staging_bytes, void* stream_v) {
    if (!ws) return ARF_ERR_INVALID_ARG;
    arf_status_t st = arf_supports(ws, pattern, W, M, H, dtype);
    if (st != ARF_OK) return st;
    if (M == 0) return ARF_OK;
    const bool rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
    if (!partials_host || !out_host) return ARF_ERR_INVALID_ARG;
    for (int r = 0; r < W; ++r)
        if (!partials_host[r]) return ARF_ERR_INVALID_ARG;
    if (rms) {
        if (!residual_host || !gamma_host || !residual_out_host) return ARF_ERR_INVALID_ARG;
        if (!std::isfinite(eps) || eps < 0.0f) return ARF_ERR_INVALID_ARG;
        if (out_host == residual_out_host) return ARF_ERR_INVALID_ARG;
    }
    const Staging L = staging_layout(pattern, W, M, H);
    if (!staging_dev || (reinterpret_cast<uintptr_t>(staging_dev) & 255u) != 0 || staging_bytes < L.total)
        return ARF_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    bool capturing = false;
    st = check_device(ws, stream, &capturing);
    if (st != ARF_OK) return st;

    char* base = static_cast<char*>(staging_dev);
    const size_t bytes = (size_t)M * (size_t)H * 2;
    const int blocks = host_pipeline_blocks(M, H);
    if (blocks > 1)
        return run_host_pipelined(ws, pattern, W, partials_host, residual_host, gamma_host, eps, out_host,
                                  residual_out_host, M, H, dtype, base, L, blocks, stream);
    cudaError_t e = arf::launch_fill_pointer_array(reinterpret_cast<const void**>(base + L.ptrs), base + L.p0,
                                                   (int64_t)L.plane, W, stream);
    for (int r = 0; r < W && e == cudaSuccess; ++r)
        e = cudaMemcpyAsync(base + L.p0 + (size_t)r * L.plane, partials_host[r], bytes, cudaMemcpyHostToDevice,
                            stream);
    if (rms && e == cudaSuccess)
        e = cudaMemcpyAsync(base + L.residual, residual_host, bytes, cudaMemcpyHostToDevice, stream);
    if (rms && e == cudaSuccess)
        e = cudaMemcpyAsync(base + L.gamma, gamma_host, (size_t)H * 2, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(ws, e);

    st = run_impl(ws, nullptr, pattern, W, reinterpret_cast<const void* const*>(base + L.ptrs),
                  rms ? base + L.residual : nullptr, rms ? base + L.gamma : nullptr, eps, base + L.out,
                  rms ? base + L.residual_out : nullptr, M, H, dtype, stream);
    if (st != ARF_OK) return st;

    e = cudaMemcpyAsync(out_host, base + L.out, bytes, cudaMemcpyDeviceToHost, stream);
    if (rms && e == cudaSuccess)
        e = cudaMemcpyAsync(residual_out_host, base + L.residual_out, bytes, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(ws, e);
    return ARF_OK;
}

extern "C" arf_status_t arf_read_pass(arf_workspace_t ws, const void* buf, int64_t bytes, void* stream) {
    if (!ws || bytes < 0 || bytes % 16 != 0) return ARF_ERR_INVALID_ARG;
    if (bytes == 0) return ARF_OK;
    if (!buf || !aligned16(buf)) return ARF_ERR_INVALID_ARG;
    // the sink is a spare word of the workspace's device allocation, past
    // the wait-timeout counter
    cudaError_t e = arf::launch_read_pass(buf, bytes, ws->wait_timeouts + 32, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(ws, e);
    return ARF_OK;
}
