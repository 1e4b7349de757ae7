/*
 * host_calls.c: drives the host-only part of the C ABI (include/arf.h) from
 * plain C99, without Python: status strings, the shape rules of
 * arf_supports, the planner for a given device description, the staging
 * sizes. Prints one line per result; tests/test_c_abi.py compares them with
 * the same calls made through the Python binding. Needs no GPU.
 */
#include <stdio.h>

#include "arf.h"

static void print_plan(const char* tag, arf_status_t st, const arf_plan_t* p) {
    printf("plan %s %d %d %d %d %d %d %d %d\n", tag, (int)st, p->path, p->threads, p->vpt, p->cluster, p->grid,
           p->w_spec, p->stages);
}

int main(void) {
    for (int s = 0; s <= 5; ++s) printf("status %d %s\n", s, arf_status_string((arf_status_t)s));

    static const struct { int pattern, W; long long M, H; int dtype; } shapes[] = {
        {ARF_ALLREDUCE, 4, 5851, 7168, ARF_BF16},        {ARF_AR_RESIDUAL_RMSNORM, 4, 5851, 7168, ARF_BF16},
        {ARF_AR_RESIDUAL_RMSNORM, 16, 585, 7168, ARF_FP16}, {ARF_AR_RESIDUAL_RMSNORM, 8, 1, 7168, ARF_BF16},
        {ARF_ALLREDUCE, 2, 4096, 4098, ARF_BF16},        {ARF_AR_RESIDUAL_RMSNORM, 3, 2000, 7168, ARF_BF16},
        {ARF_AR_RESIDUAL_RMSNORM, 65, 8, 1024, ARF_BF16}, {ARF_AR_RESIDUAL_RMSNORM, 2, 8, 0, ARF_BF16},
    };
    const int n = (int)(sizeof shapes / sizeof shapes[0]);
    /* a GB300 as the workspace reports it, and a smaller device */
    const arf_device_caps_t gb300 = {152, 16, 2048, 232448};
    const arf_device_caps_t small = {20, 1, 1536, 101376};
    for (int i = 0; i < n; ++i) {
        const arf_status_t sup = arf_supports(NULL, (arf_pattern_t)shapes[i].pattern, shapes[i].W, shapes[i].M,
                                              shapes[i].H, (arf_dtype_t)shapes[i].dtype);
        printf("supports %d %d\n", i, (int)sup);
        if (sup != ARF_OK) continue;
        char tag[32];
        arf_plan_t p = {0};
        arf_status_t st = arf_plan_for_caps(&gb300, (arf_pattern_t)shapes[i].pattern, shapes[i].W, shapes[i].M,
                                            shapes[i].H, (arf_dtype_t)shapes[i].dtype, &p);
        snprintf(tag, sizeof tag, "gb300_%d", i);
        print_plan(tag, st, &p);
        if (st == ARF_OK)
            printf("check %d %d\n", i,
                   (int)arf_plan_check(&gb300, &p, (arf_pattern_t)shapes[i].pattern, shapes[i].W, shapes[i].M,
                                       shapes[i].H, (arf_dtype_t)shapes[i].dtype));
        arf_plan_t q = {0};
        st = arf_plan_rules(&small, (arf_pattern_t)shapes[i].pattern, shapes[i].W, shapes[i].M, shapes[i].H,
                            (arf_dtype_t)shapes[i].dtype, &q);
        snprintf(tag, sizeof tag, "small_%d", i);
        print_plan(tag, st, &q);
        printf("staging %d %zu\n", i,
               arf_host_staging_bytes((arf_pattern_t)shapes[i].pattern, shapes[i].W, shapes[i].M, shapes[i].H,
                                      (arf_dtype_t)shapes[i].dtype));
    }
    printf("static_staging %zu\n", arf_static_staging_bytes());
    /* calls that need a workspace refuse NULL instead of crashing */
    printf("null_ws %d\n", (int)arf_run(NULL, ARF_ALLREDUCE, 2, NULL, NULL, NULL, 0.0f, NULL, NULL, 1, 8, ARF_BF16,
                                        NULL));
    return 0;
}
