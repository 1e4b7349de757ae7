/*
 * device_run.c: the epilogue driven from plain C99 through include/arf.h, on
 * device buffers from the CUDA runtime, checked against the CPU oracle
 * (oracle/arf_oracle.c, linked in: this is a test). For each case it makes
 * seeded inputs, runs arf_run on the default stream, copies the outputs back
 * and compares: kAllReduce out and residual_out bitwise, the normalised out
 * within one code of the oracle's (same sign, adjacent codes: at most one
 * unit in the last place of the larger magnitude). Prints one line per case
 * and exits non-zero on the first mismatch or error. Needs a GPU.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "arf.h"
#include "arf_oracle.h"

/* xorshift64*: the inputs' only source of randomness */
static uint64_t rng_state;
static uint32_t next_u32(void) {
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (uint32_t)((rng_state * 0x2545F4914F6CDD1DULL) >> 32);
}

/* A finite 16-bit code with magnitude in [2^-3, 2^3): random sign and
 * mantissa, exponent field from the format's bias. */
static uint16_t random_code(int dtype) {
    const uint32_t r = next_u32();
    const uint32_t sign = (r >> 31) & 1u;
    if (dtype == ARF_BF16) {
        const uint32_t e = 124u + (r >> 24) % 6u; /* bias 127 */
        return (uint16_t)((sign << 15) | (e << 7) | (r & 0x7fu));
    }
    const uint32_t e = 12u + (r >> 24) % 6u; /* bias 15 */
    return (uint16_t)((sign << 15) | (e << 10) | (r & 0x3ffu));
}

/* gamma: positive, magnitude in [0.5, 2) */
static uint16_t random_gamma(int dtype) {
    const uint32_t r = next_u32();
    if (dtype == ARF_BF16) return (uint16_t)(((126u + (r >> 24) % 2u) << 7) | (r & 0x7fu));
    return (uint16_t)(((14u + (r >> 24) % 2u) << 10) | (r & 0x3ffu));
}

static int within_one_code(uint16_t a, uint16_t b) {
    if (a == b) return 1;
    if (((a | b) & 0x7fffu) == 0) return 1; /* +0 and -0 */
    if ((a ^ b) & 0x8000u) return 0;
    const int d = (int)(a & 0x7fffu) - (int)(b & 0x7fffu);
    return d == 1 || d == -1;
}

#define CUDA_OK(x)                                                              \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            printf("FAIL cuda %s: %s\n", #x, cudaGetErrorString(e_));           \
            return 1;                                                           \
        }                                                                       \
    } while (0)

static int run_case(arf_workspace_t ws, int pattern, int W, int64_t M, int64_t H, int dtype, uint64_t seed) {
    const size_t n = (size_t)M * (size_t)H, bytes = n * 2;
    rng_state = seed * 0x9E3779B97F4A7C15ULL + 1;
    uint16_t** hp = (uint16_t**)calloc((size_t)W, sizeof *hp);
    void** dp = (void**)calloc((size_t)W, sizeof *dp);
    uint16_t *hr = malloc(bytes), *hg = malloc((size_t)H * 2), *out = malloc(bytes), *ro = malloc(bytes);
    uint16_t *ref_out = malloc(bytes), *ref_ro = malloc(bytes);
    if (!hp || !dp || !hr || !hg || !out || !ro || !ref_out || !ref_ro) return 1;
    for (int r = 0; r < W; ++r) {
        hp[r] = malloc(bytes);
        if (!hp[r]) return 1;
        for (size_t i = 0; i < n; ++i) hp[r][i] = random_code(dtype);
    }
    for (size_t i = 0; i < n; ++i) hr[i] = random_code(dtype);
    for (int64_t i = 0; i < H; ++i) hg[i] = random_gamma(dtype);
    const float eps = 1e-6f;

    void *dr = NULL, *dg = NULL, *dout = NULL, *dro = NULL, **dptrs = NULL;
    for (int r = 0; r < W; ++r) {
        CUDA_OK(cudaMalloc(&dp[r], bytes));
        CUDA_OK(cudaMemcpy(dp[r], hp[r], bytes, cudaMemcpyHostToDevice));
    }
    CUDA_OK(cudaMalloc((void**)&dptrs, (size_t)W * sizeof(void*)));
    CUDA_OK(cudaMemcpy(dptrs, dp, (size_t)W * sizeof(void*), cudaMemcpyHostToDevice));
    CUDA_OK(cudaMalloc(&dr, bytes));
    CUDA_OK(cudaMalloc(&dg, (size_t)H * 2));
    CUDA_OK(cudaMalloc(&dout, bytes));
    CUDA_OK(cudaMalloc(&dro, bytes));
    CUDA_OK(cudaMemcpy(dr, hr, bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dg, hg, (size_t)H * 2, cudaMemcpyHostToDevice));

    const int rms = pattern == ARF_AR_RESIDUAL_RMSNORM;
    const arf_status_t st = arf_run(ws, (arf_pattern_t)pattern, W, (const void* const*)dptrs, rms ? dr : NULL,
                                    rms ? dg : NULL, eps, dout, rms ? dro : NULL, M, H, (arf_dtype_t)dtype, NULL);
    if (st != ARF_OK) {
        printf("FAIL arf_run %s (cuda %d)\n", arf_status_string(st), arf_last_cuda_error(ws));
        return 1;
    }
    CUDA_OK(cudaDeviceSynchronize());
    CUDA_OK(cudaMemcpy(out, dout, bytes, cudaMemcpyDeviceToHost));
    if (rms) CUDA_OK(cudaMemcpy(ro, dro, bytes, cudaMemcpyDeviceToHost));

    if (arf_oracle_run(pattern, W, (const void* const*)hp, hr, hg, eps, ref_out, ref_ro, M, H, dtype) != 0) {
        printf("FAIL oracle\n");
        return 1;
    }
    size_t exact_bad = 0, near = 0, far = 0;
    for (size_t i = 0; i < n; ++i) {
        if (!rms) {
            exact_bad += out[i] != ref_out[i];
            continue;
        }
        exact_bad += ro[i] != ref_ro[i];
        if (out[i] != ref_out[i]) {
            if (within_one_code(out[i], ref_out[i])) ++near;
            else ++far;
        }
    }
    printf("%s pattern=%d W=%d M=%lld H=%lld dtype=%d bitwise_mismatches=%zu out_one_code=%zu out_beyond=%zu\n",
           exact_bad || far ? "FAIL" : "OK", pattern, W, (long long)M, (long long)H, dtype, exact_bad, near, far);

    for (int r = 0; r < W; ++r) {
        cudaFree(dp[r]);
        free(hp[r]);
    }
    cudaFree(dptrs);
    cudaFree(dr);
    cudaFree(dg);
    cudaFree(dout);
    cudaFree(dro);
    free(hp), free(dp), free(hr), free(hg), free(out), free(ro), free(ref_out), free(ref_ro);
    return exact_bad || far ? 1 : 0;
}

int main(void) {
    arf_workspace_t ws = NULL;
    const arf_status_t st = arf_workspace_create(0, &ws);
    if (st != ARF_OK) {
        printf("FAIL arf_workspace_create %s\n", arf_status_string(st));
        return 1;
    }
    static const struct { int pattern, W; long long M, H; int dtype; } cases[] = {
        {ARF_ALLREDUCE, 4, 37, 7168, ARF_BF16},         {ARF_AR_RESIDUAL_RMSNORM, 4, 37, 7168, ARF_BF16},
        {ARF_AR_RESIDUAL_RMSNORM, 16, 5, 4104, ARF_FP16}, {ARF_AR_RESIDUAL_RMSNORM, 8, 1, 7168, ARF_BF16},
        {ARF_ALLREDUCE, 3, 9, 1030, ARF_FP16},          {ARF_AR_RESIDUAL_RMSNORM, 3, 9, 1030, ARF_FP16},
        {ARF_AR_RESIDUAL_RMSNORM, 2, 3, 32776, ARF_BF16},
    };
    int bad = 0;
    for (int i = 0; i < (int)(sizeof cases / sizeof cases[0]) && !bad; ++i)
        bad = run_case(ws, cases[i].pattern, cases[i].W, cases[i].M, cases[i].H, cases[i].dtype, 1000u + (unsigned)i);
    arf_workspace_destroy(ws);
    return bad;
}
