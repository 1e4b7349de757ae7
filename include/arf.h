/*
 * arf.h: the all-reduce fusion epilogue on one GPU (C ABI).
 *
 * What the library computes. In tensor-parallel decode each of W ranks holds
 * a partial activation [M,H]; the all-reduce sums them, and a fused epilogue
 * may follow. tokenspeed PR #1075 "route generic MNNVL AR patterns to
 * upstream flashinfer" (description, Summary) names the two generic fusion
 * patterns built here:
 *   kAllReduce          out          = sum_r P_r
 *   kARResidualRMSNorm  residual_out = sum_r P_r + residual
 *                       out          = RMSNorm(residual_out) * gamma
 * Here all W partials sit in this GPU's own memory and are reached through a
 * device-resident array of W pointers, the form flashinfer PR #1321
 * "Optimizations for TRTLLM MNNVL Allreduce" (Description: "Use GPU array to
 * pass the uc pointers") gives for the per-rank buffers. Nothing crosses GPUs.
 *
 * Numeric contract (both dtypes, bf16 and fp16: flashinfer PR #1321,
 * Highlights, __nv_half support):
 *   acc = 0.0f; for r = 0..W-1 in array order: acc = acc + f32(P_r[m,i])
 *       binary32 round-to-nearest adds, no reassociation, no FMA, no FTZ;
 *   kAllReduce:  out[m,i] = rn(acc)                      (bitwise defined)
 *   kARResidualRMSNorm:
 *       residual_out[m,i] = rn(acc + f32(residual[m,i])) (one rounding;
 *                                                          bitwise defined)
 *       x_i = f32(residual_out[m,i])                      (the stored value)
 *       inv = rsqrt(sum_i x_i^2 / H + eps)                (mean over H, eps
 *                                                          inside the root)
 *       out[m,i] = rn((x_i * inv) * f32(gamma[i]))        (binary32, within
 *                                                          1 ulp of the exact
 *                                                          value rounded once)
 *   rn() = round to nearest even into the I/O dtype.
 * The sum of squares is reduced in a fixed tree for a given launch plan, so
 * repeated calls with the same plan are bitwise identical.
 *
 * Layout. Every [M,H] tensor is contiguous row-major (row stride H elements),
 * gamma is [H]. Element type is bf16 or fp16 (16-bit codes).
 *
 * Ownership. The caller owns every tensor and the pointer array; they must
 * stay valid until the stream work completes. The library keeps no tensor
 * pointer after a call returns. A workspace owns host state (device id, SM
 * count, cluster limits, plan cache), one 256-byte device word, the bulk
 * kernel's wait-timeout counter, and two copy streams with four events for
 * arf_run_host, all made at creation and released at destruction; no call
 * allocates device memory.
 *
 * Errors. Every entry point returns a status and never throws. On any error
 * nothing is launched and no output is written.
 */
#ifndef ARF_H
#define ARF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum arf_status {
    ARF_OK = 0,
    ARF_ERR_INVALID_ARG = 1,     /* NULL pointer, negative size, bad eps, aliasing */
    ARF_ERR_UNSUPPORTED = 2,     /* valid but outside what this build handles */
    ARF_ERR_CUDA = 3,            /* a CUDA call failed; see arf_last_cuda_error */
    ARF_ERR_DEVICE_MISMATCH = 4  /* current device or stream device != workspace device */
} arf_status_t;

/* Fusion patterns, named as in tokenspeed PR #1075 (Summary). */
typedef enum arf_pattern {
    ARF_ALLREDUCE = 0,           /* kAllReduce */
    ARF_AR_RESIDUAL_RMSNORM = 1  /* kARResidualRMSNorm */
} arf_pattern_t;

typedef enum arf_dtype {
    ARF_BF16 = 0,
    ARF_FP16 = 1
} arf_dtype_t;

/* Kernel shapes a plan can select. */
typedef enum arf_path {
    ARF_PATH_FLAT = 0,    /* kAllReduce: grid-stride over 16-byte chunks of [M,H] */
    ARF_PATH_ROW = 1,     /* kARResidualRMSNorm: one CTA owns a whole row */
    ARF_PATH_CLUSTER = 2, /* kARResidualRMSNorm: a row split over a thread-block
                             cluster, sum of squares exchanged through DSMEM */
    ARF_PATH_ASYNC = 3,   /* kARResidualRMSNorm, W in {1,2,4,8,16}: one CTA of
                             256 threads per SM streams its rows in column
                             blocks of 256 chunks through a ring of `stages`
                             asynchronous shared-memory copies (cp.async) */
    ARF_PATH_ELEM = 4,    /* either pattern, any layout (H not a multiple of 8,
                             row strides not a multiple of 8, tensors only 2-byte
                             aligned): 16-byte vectors with per-row heads and
                             tails where every tensor is 16-byte aligned and all
                             row strides agree modulo 8, else one element per
                             thread per step */
    ARF_PATH_BULK = 5     /* either pattern, 16-bit partials: each CTA walks
                             its rows in column blocks of `threads` chunks;
                             one thread keeps `stages` blocks in flight as TMA
                             bulk copies (cp.async.bulk) into a shared-memory
                             ring, completed on mbarriers by byte count. Its
                             waits are bounded: see
                             arf_workspace_wait_timeouts. */
} arf_path_t;

/* Limits of this build. */
#define ARF_MAX_W 64        /* ranks: the pages' world sizes {2,...,64}, plus 1 */
#define ARF_MAX_H 524288    /* hidden size */
#define ARF_MAX_H_PER_CTA 32768 /* kARResidualRMSNorm rows longer than this are
                                   split over a thread-block cluster (H up to
                                   ARF_MAX_H_PER_CTA x the cluster limit); longer
                                   still, or H not a multiple of 8, take the
                                   elementwise path */

/* What the planner needs to know about a device. */
typedef struct arf_device_caps {
    int num_sms;            /* streaming multiprocessors */
    int max_cluster;        /* largest usable cluster size (1, 2, 4, 8 or 16) */
    int max_threads_per_sm; /* resident threads per SM */
    int max_smem_per_block; /* opt-in shared memory per CTA, bytes */
} arf_device_caps_t;

/* A launch plan: which kernel shape and launch configuration one call uses. */
typedef struct arf_plan {
    int path;     /* arf_path_t */
    int threads;  /* threads per CTA, a multiple of 32 in [32, 512] */
    int vpt;      /* 16-byte chunks per thread per row (row/cluster paths) or
                     chunks per thread per loop trip (flat path): 1, 2, 4 or 8 */
    int cluster;  /* CTAs per row (cluster path: 2, 4, 8 or 16; else 1) */
    int grid;     /* CTAs launched; a multiple of `cluster` */
    int w_spec;   /* rank count compiled into the kernel, or 0 for the generic
                     kernel that reads W at run time */
    int stages;   /* async path: copies in flight per thread, in column
                     blocks (2..8); bulk path: ring slots, in column blocks
                     (2..16); 0 on the other paths */
} arf_plan_t;

typedef struct arf_workspace* arf_workspace_t;

/* ---- workspace -------------------------------------------------------- */

/* Create a workspace for CUDA device `device`: reads the SM count and the
 * resident-thread limit, and probes the largest cluster size the cluster
 * kernel can be launched with (the launch configuration is then derived
 * from these, as flashinfer PR #1507 "update allreduce to match trtllm",
 * Highlights, derives threads_per_block and cluster_size from the SM count).
 * Makes `device` current on the calling thread. Allocates the workspace's
 * only device memory here: 256 bytes holding the bulk kernel's wait-timeout
 * counter (arf_workspace_wait_timeouts); no later call allocates for it.
 * Also creates the two non-blocking streams and four events of
 * arf_run_host's pipelined form; arf_workspace_destroy releases them all.
 * Errors: ws_out NULL -> INVALID_ARG; no such device or a CUDA failure -> CUDA. */
arf_status_t arf_workspace_create(int device, arf_workspace_t* ws_out);

/* Destroy a workspace. NULL is accepted and returns ARF_OK. */
arf_status_t arf_workspace_destroy(arf_workspace_t ws);

/* The device capabilities the workspace plans with. */
arf_status_t arf_workspace_caps(arf_workspace_t ws, arf_device_caps_t* caps_out);

/* The cudaError_t of the workspace's last ARF_ERR_CUDA (0 if none). */
int arf_last_cuda_error(arf_workspace_t ws);

/* Every wait of the bulk kernel (ARF_PATH_BULK) on its shared-memory ring is
 * bounded (about a second by default, arf_run_opts_t.wait_limit_cycles): a
 * CTA whose copies have not landed by then stops, waits (bounded again) for
 * the copies it issued, adds 1 to a counter in the workspace's device memory
 * and returns, so the context stays usable; that call's outputs are then
 * incomplete. This waits for all work on the workspace's device
 * (cudaDeviceSynchronize), reads the counter into *count_out and resets it
 * to 0. Not during stream capture.
 * Errors: NULL argument -> INVALID_ARG; a CUDA failure -> CUDA. */
arf_status_t arf_workspace_wait_timeouts(arf_workspace_t ws, unsigned int* count_out);

/* Static text for a status code (never NULL). */
const char* arf_status_string(arf_status_t status);

/* ---- capability and planning (host only, no device work) --------------- */

/* Whether (pattern, W, M, H, dtype) is handled, judged on the sizes alone in
 * the manner of the supports()/dispatch contract of tokenspeed PR #1075
 * (Summary). ws may be NULL (shape rules only). Returns ARF_OK, or the status
 * arf_run would return for these sizes: W outside [1, ARF_MAX_W] or
 * H > ARF_MAX_H -> UNSUPPORTED; H <= 0 or M < 0 or a bad enum -> INVALID_ARG.
 * Sizes the 16-byte kernels cannot take (H % 8 != 0, kARResidualRMSNorm rows
 * longer than the device's clusters hold) run on the elementwise path. */
arf_status_t arf_supports(arf_workspace_t ws, arf_pattern_t pattern, int W,
                          int64_t M, int64_t H, arf_dtype_t dtype);

/* The plan the library picks for these sizes on a device with `caps`.
 * Pure function of its arguments. Threads per block, cluster size and grid
 * follow from the device (flashinfer PR #1507 "update allreduce to match
 * trtllm", Highlights), chosen per shape (vLLM PR #53318 "Tune FlashInfer
 * all-reduce selection on SM103", Scope): first from the library's measured
 * plan table, whose rows hold the fastest plan timed cold (L2 flushed) for
 * a device with exactly these capabilities, a pattern, dtype, W, H and a
 * range of M; for shapes and devices the table does not cover, from the
 * closed-form rules of arf_plan_rules. */
arf_status_t arf_plan_for_caps(const arf_device_caps_t* caps, arf_pattern_t pattern,
                               int W, int64_t M, int64_t H, arf_dtype_t dtype,
                               arf_plan_t* plan_out);

/* The closed-form planning rules alone, without the measured table: the plan
 * arf_plan_for_caps returns where the table has no row. Same arguments,
 * results and errors. No counterpart on the pages beyond the launch-
 * configuration remark cited above. */
arf_status_t arf_plan_rules(const arf_device_caps_t* caps, arf_pattern_t pattern,
                            int W, int64_t M, int64_t H, arf_dtype_t dtype,
                            arf_plan_t* plan_out);

/* The plan arf_run would use on this workspace (memoised per shape). */
arf_status_t arf_workspace_plan(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                int64_t M, int64_t H, arf_dtype_t dtype,
                                arf_plan_t* plan_out);

/* Whether `plan` is a legal plan for these sizes on `caps` (ARF_OK) or not
 * (UNSUPPORTED), the check arf_run_planned applies. */
arf_status_t arf_plan_check(const arf_device_caps_t* caps, const arf_plan_t* plan,
                            arf_pattern_t pattern, int W, int64_t M, int64_t H,
                            arf_dtype_t dtype);

/* ---- the epilogue ------------------------------------------------------ */

/* Run one pattern, asynchronously on `stream` (a cudaStream_t; NULL = the
 * legacy default stream). No allocation, no host synchronisation and no host
 * read of device data, so the call can be captured into a CUDA graph; a
 * captured graph bakes in the pointer values, so keep them stable. Make one
 * uncaptured call per shape first: it memoises the plan after checking on
 * the device that its cluster shape can be resident (a first call made under
 * capture skips that query and relies on the cluster limit probed when the
 * workspace was created). While capturing, the stream's device is not
 * checked (CUDA does not allow that query then).
 *
 *   partials_dev  DEVICE array of W device pointers, each to an [M,H] tensor;
 *                 ranks are summed in this array's order. Every pointer must
 *                 be 16-byte aligned (a precondition: it is not readable from
 *                 the host without a synchronisation).
 *   residual      [M,H] device, read      (kARResidualRMSNorm; else ignored)
 *   gamma         [H]   device, read      (kARResidualRMSNorm; else ignored)
 *   eps           finite, >= 0            (kARResidualRMSNorm; else ignored)
 *   out           [M,H] device, written
 *   residual_out  [M,H] device, written   (kARResidualRMSNorm; else ignored)
 *
 * Any buffer, and the pointer array, may also be page-locked host memory the
 * GPU can address (for example from cudaHostAlloc): the kernels then read and
 * write it in place over the host link, with no staging copies (on
 * Grace-Blackwell the NVLink-C2C link; measured about twice as fast as
 * arf_run_host's copies for decode-size calls).
 * Inputs are never modified. residual_out == residual is allowed (in place):
 * each element is read before the same thread overwrites it. out ==
 * residual_out is rejected (INVALID_ARG); other overlaps are undefined.
 * M == 0 returns ARF_OK and launches nothing.
 * Errors: see arf_supports; NULL required pointer, non-finite or negative eps
 * -> INVALID_ARG; residual, gamma, out or residual_out at an odd address ->
 * UNSUPPORTED (2-byte aligned but not 16-byte aligned: the elementwise path;
 * partial pointers must be 16-byte aligned when H % 8 == 0, 2-byte otherwise);
 * current device or stream device != workspace device -> DEVICE_MISMATCH;
 * launch failure -> CUDA (code in arf_last_cuda_error). */
arf_status_t arf_run(arf_workspace_t ws, arf_pattern_t pattern, int W,
                     const void* const* partials_dev,
                     const void* residual, const void* gamma, float eps,
                     void* out, void* residual_out,
                     int64_t M, int64_t H, arf_dtype_t dtype, void* stream);

/* Measure candidate launch plans for these sizes on the caller's buffers and
 * keep the fastest in the workspace: later arf_run calls of the same
 * (pattern, W, M, H, dtype) use it. Candidates: the planner's plan and its
 * neighbours (threads, chunks per thread, cluster size, compiled or run-time
 * rank count, bulk ring width and depth; for the elementwise path each CTA
 * width with the planner's grid and with a device-full grid) that pass
 * arf_plan_check and fit the device. Each runs `reps`
 * times (<= 0: 20) back to back on `stream`, timed with CUDA events after two
 * warm-up calls; the call synchronises the stream, so it cannot be captured.
 * Buffers and arguments are those of an arf_run call; the outputs are
 * overwritten (with the values arf_run would write). The chosen plan is
 * returned in plan_out and its mean time per call in us_out (either may be
 * NULL). Errors: as arf_run. */
arf_status_t arf_workspace_autotune(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                    const void* const* partials_dev,
                                    const void* residual, const void* gamma, float eps,
                                    void* out, void* residual_out,
                                    int64_t M, int64_t H, arf_dtype_t dtype, int reps,
                                    void* stream, arf_plan_t* plan_out, float* us_out);

/* arf_run with an explicit launch plan instead of the planner's (tuning
 * sweeps and tests of every kernel shape). The plan must pass
 * arf_plan_check for the workspace's caps, and a cluster plan must be one the
 * device can keep resident, else UNSUPPORTED. Same semantics
 * and results contract as arf_run; out may differ from arf_run's by the
 * reduction tree of the sum of squares (within the 1 ulp bound). */
arf_status_t arf_run_planned(arf_workspace_t ws, const arf_plan_t* plan,
                             arf_pattern_t pattern, int W,
                             const void* const* partials_dev,
                             const void* residual, const void* gamma, float eps,
                             void* out, void* residual_out,
                             int64_t M, int64_t H, arf_dtype_t dtype, void* stream);

/* Per-call options of arf_run_ex. Zero-initialise, then set what is needed
 * (all zero = arf_run). */
typedef struct arf_run_opts {
    const arf_plan_t* plan;  /* NULL: the planner's plan; else an explicit plan,
                                checked as by arf_run_planned */
    int partials_by_value;   /* 0: `partials` is a DEVICE array of W device
                                pointers (as arf_run). 1: `partials` is a HOST
                                array of W device pointers; the values are
                                copied into the kernel launch, so the kernel
                                reads no pointer array; a captured graph keeps
                                the values, and the host array may be reused
                                as soon as the call returns. Not faster: on
                                GB300 at decode sizes (W = 8, H = 7168,
                                M = 1..64) the launch's larger parameter block
                                (room for ARF_MAX_W pointers) costs more than
                                the pointer-array read it saves: cold level or
                                up to 0.8 us slower, warm in CUDA graphs
                                0.1-0.4 us slower. It is for callers that have
                                no device pointer array. */
    int pdl;                 /* programmatic dependent launch: the kernel may
                                be scheduled while the previous kernel in the
                                stream still runs, and waits
                                (griddepcontrol.wait) for it to complete before
                                it touches any memory, so results are the same;
                                what overlaps is launch latency.
                                0 = the library's choice (the default, also for
                                arf_run): on for latency-bound launches, whose
                                grid x threads is at most 1/16 of the threads
                                the device holds (decode sizes; measured on
                                GB300 in CUDA graphs: k3 TP8 M = 1..8
                                kARResidualRMSNorm 2.6-2.7 -> 2.2-2.4 us per
                                call), off for larger ones, where waiting CTAs
                                would hold SM slots; 1 = always; 2 = never.
                                Other values -> ARF_ERR_INVALID_ARG. */
    int64_t ld_partials;     /* row strides in elements (0 = H, contiguous): of */
    int64_t ld_residual;     /* every partial, the residual, out and            */
    int64_t ld_out;          /* residual_out. Each must be >= H                 */
    int64_t ld_residual_out; /* (ARF_ERR_INVALID_ARG) and M * stride <= 2^40
                                (ARF_ERR_UNSUPPORTED). Strides that are
                                multiples of 8 keep the 16-byte kernels. */
    int partials_f32;        /* 1: the partials are binary32 [M,H] tensors (the
                                I/O dtype still applies to residual, gamma and
                                the outputs); they enter the binary32 rank-order
                                sum exactly; 4-byte alignment required */
    int64_t wait_limit_cycles; /* bulk path: SM cycles a wait on a ring slot
                                  may take before the CTA gives up (0 = the
                                  default, 2^31, about a second) */
    int hold_first_copy;     /* TESTING ONLY; leave 0 in production code.
                                Bulk path: 1 = every CTA leaves its first ring
                                slot unfilled, so its first wait runs out (see
                                arf_workspace_wait_timeouts); the call then
                                produces NO complete output. It exists so that
                                a test can make a bounded wait give up without
                                faulting anything. */
} arf_run_opts_t;

/* arf_run with per-call options (NULL opts = arf_run). Same semantics,
 * results contract and errors; with partials_by_value, `partials` must point
 * to W readable host pointers (INVALID_ARG if any is NULL); a stride below H,
 * or residual_out == residual with different strides -> INVALID_ARG. Layouts
 * the 16-byte kernels cannot take (strides not multiples of 8, tensors only
 * 2-byte aligned) run on the elementwise path; odd addresses -> UNSUPPORTED. */
arf_status_t arf_run_ex(arf_workspace_t ws, const arf_run_opts_t* opts,
                        arf_pattern_t pattern, int W, const void* const* partials,
                        const void* residual, const void* gamma, float eps,
                        void* out, void* residual_out,
                        int64_t M, int64_t H, arf_dtype_t dtype, void* stream);

/* ---- host buffers ------------------------------------------------------ */

/* Bytes of device staging that arf_run_host needs for these sizes. */
size_t arf_host_staging_bytes(arf_pattern_t pattern, int W, int64_t M, int64_t H,
                              arf_dtype_t dtype);

/* The epilogue on HOST buffers: copies the inputs to `staging_dev`, runs
 * the pattern there and copies the outputs back, all ordered on `stream`
 * (returns before they finish; synchronise the stream before reading the
 * outputs). Copies overlap other work only from page-locked host memory.
 *
 * Tensors of 8 MiB or more are pipelined in blocks of rows (one per 4 MiB,
 * at most 8; rows per block a multiple of 8, so that each block starts on a
 * 16-byte boundary for any H): a block's inputs are copied in on a stream of the workspace,
 * its kernel runs on `stream` once they have landed, and its outputs are
 * copied out on a second stream of the workspace while later blocks' inputs
 * are still coming in. Both copy streams start after the work enqueued on
 * `stream` before the call, and `stream` waits for the last copy out (event
 * fork and join), so the call is ordered with other work on `stream` as a
 * single-stream call would be, under stream capture too. Calls on one
 * workspace are enqueued one at a time (the workspace holds a lock while
 * enqueuing) and share its copy streams. Rows of different blocks never
 * alias, so residual_out_host may be residual_host and out_host may be one
 * of the partials' buffers, as in the single-stream form.
 *
 *   partials_host  HOST array of W host pointers, each to an [M,H] tensor
 *   residual_host, gamma_host, out_host, residual_out_host: host buffers with
 *                  the roles and layouts of arf_run's arguments
 *   staging_dev    device buffer of at least arf_host_staging_bytes(...)
 *                  bytes, 256-byte aligned, owned by the caller, not used by
 *                  anything else until the stream work completes
 * Errors: as arf_run; staging_dev NULL, misaligned or too small -> INVALID_ARG. */
arf_status_t arf_run_host(arf_workspace_t ws, arf_pattern_t pattern, int W,
                          const void* const* partials_host,
                          const void* residual_host, const void* gamma_host, float eps,
                          void* out_host, void* residual_out_host,
                          int64_t M, int64_t H, arf_dtype_t dtype,
                          void* staging_dev, size_t staging_bytes, void* stream);

/* ---- host buffers, no device allocation ------------------------------- */

/* Size of the staging array built into the library for arf_run_host_static. */
#define ARF_STATIC_STAGING_BYTES (16u << 20) /* 16 MiB */

/* ARF_STATIC_STAGING_BYTES as the built library has it (for bindings that do
 * not read this header). No counterpart on the source pages. */
size_t arf_static_staging_bytes(void);

/* arf_run_host for callers that cannot allocate device memory. There is no
 * counterpart on the source pages: it exists for callers such as a plugin
 * inside a framework or serving engine whose allocator owns the device
 * memory, or a latency-critical host thread that cannot pay for cudaMalloc's
 * implicit synchronisation, neither of which can hand arf_run_host a staging
 * buffer. It allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library call): the staging lives in a file-scope device array of
 * ARF_STATIC_STAGING_BYTES bytes compiled into the library.
 *
 * When the array is taken: arf_workspace_create looks up its device address
 * (cudaGetSymbolAddress, with the workspace's device current) and keeps it in
 * the workspace. Under CUDA's lazy module loading (the default since CUDA
 * 12.2) that lookup loads the array, so its 16 MiB are taken on a device when
 * the first workspace there is created; with eager loading, when the library
 * is loaded. Either way never inside a call of this entry point, and the
 * array stays until the process exits. A workspace belongs to one CUDA
 * context: after cudaDeviceReset destroy it and create a new one. If the
 * lookup failed (for example the device had no memory left for the array)
 * this entry point returns ARF_ERR_CUDA with that error in
 * arf_last_cuda_error; the workspace's other entry points are unaffected.
 *
 * Arguments, results and errors are those of arf_run_host without the staging
 * arguments; the current device must be the workspace's. Sizes whose staging
 * (arf_host_staging_bytes) exceeds ARF_STATIC_STAGING_BYTES are rejected with
 * ARF_ERR_UNSUPPORTED before anything is enqueued. Every call on a device
 * shares the one array, which keeps the last call's contents (no call relies
 * on it starting at zero: each call writes every byte it reads). Calls whose
 * GPU work can overlap (other streams, other threads, other workspaces on the
 * same device) race on the array: serialise them, for example on one stream. */
arf_status_t arf_run_host_static(arf_workspace_t ws, arf_pattern_t pattern, int W,
                                 const void* const* partials_host,
                                 const void* residual_host, const void* gamma_host, float eps,
                                 void* out_host, void* residual_out_host,
                                 int64_t M, int64_t H, arf_dtype_t dtype, void* stream);

/* ---- measurement ----------------------------------------------------- */

/* Read `bytes` bytes at `buf` once, in 16-byte vectors, and discard them
 * (nothing is written but, with vanishing probability, one word of the
 * workspace's own device memory). A CTA per 16 KiB tile, each thread issuing
 * its four loads together, so the hardware block scheduler balances the SMs.
 * No counterpart on the source pages: it is the roofline reference for calls
 * that mostly read. On GB300 reads alone stream slower than a copy's mix of
 * reads and writes at the sizes the epilogue runs at (the copy's writes stay
 * in L2), so such a call is bounded by this pass over its reads.
 * Asynchronous on `stream`; time it with events.
 *   buf    device (or device-addressable host) memory, 16-byte aligned
 *   bytes  a multiple of 16; 0 launches nothing
 * Errors: NULL ws or buf (bytes > 0), misaligned buf, bytes < 0 or not a
 * multiple of 16 -> INVALID_ARG; launch failure -> CUDA. */
arf_status_t arf_read_pass(arf_workspace_t ws, const void* buf, int64_t bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ARF_H */
