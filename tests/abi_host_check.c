/* Plain-C client of include/fsdp.h: compiled with gcc -std=c11 -Wall -Werror
 * and linked against libfsdpreduce.so by tests/test_c_client.py. It calls
 * only host-side entry points and argument checks that return before any
 * CUDA work, so it runs without a GPU. Prints "ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fsdp.h"

#define CHECK(cond)                                                 \
    do {                                                            \
        if (!(cond)) {                                              \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                               \
        }                                                           \
    } while (0)

int main(void) {
    CHECK(fsdp_padded_numel(4099, 2) == 4100);
    CHECK(fsdp_padded_numel(855654400, 8) == 855654400);
    CHECK(fsdp_padded_numel(-1, 2) == -1);

    /* the tiny unit's layout: w[64,64], b[3] */
    const int64_t shapes[] = {64, 64, 3};
    const int32_t ndims[] = {2, 1};
    fsdp_view views[2];
    int64_t padded = 0;
    CHECK(fsdp_unflatten_views(shapes, ndims, 2, 2, views, &padded) == FSDP_OK);
    CHECK(padded == 4100);
    CHECK(views[0].offset == 0 && views[0].numel == 4096 && views[0].ndim == 2 && views[0].shape[1] == 64);
    CHECK(views[1].offset == 4096 && views[1].numel == 3 && views[1].shape[0] == 3);

    CHECK(strncmp(fsdp_status_string(FSDP_OK), "FSDP_OK", 7) == 0);
    CHECK(strncmp(fsdp_status_string(FSDP_ERR_ALIGNMENT), "FSDP_ERR_ALIGNMENT", 18) == 0);

    /* argument checks that fail on the host before any CUDA call */
    fsdp_adamw_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.0f, 0 /* step 0: invalid */, 1.0f};
    const void *grads[2] = {(const void *)0x100000, (const void *)0x200000};
    CHECK(fsdp_reduce_scatter_adam_cast(grads, FSDP_BF16, 2, 16, (float *)0x1000000, (float *)0x2000000,
                                        (float *)0x3000000, (void *)0x4000000, FSDP_BF16, &hp, 0, 2, NULL,
                                        NULL) == FSDP_ERR_INVALID_ARG);
    hp.step = 1;
    CHECK(fsdp_reduce_scatter_adam_cast(grads, (fsdp_dtype)7, 2, 16, (float *)0x1000000, (float *)0x2000000,
                                        (float *)0x3000000, (void *)0x4000000, FSDP_BF16, &hp, 0, 2, NULL,
                                        NULL) == FSDP_ERR_UNSUPPORTED_DTYPE);
    void *dst[1] = {(void *)0x5000001};
    CHECK(fsdp_all_gather((const void *)0x4000000, FSDP_BF16, 2, 16, dst, 1, NULL, NULL) == FSDP_ERR_ALIGNMENT);
    fsdp_step_config cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.optimizer = FSDP_OPT_SGD;
    cfg.reduce_dtype = FSDP_F32;
    cfg.lr = 1e-2f;
    cfg.step = 1;
    cfg.grad_scale = 1.0f;
    CHECK(fsdp_reduce_scatter_step(grads, FSDP_BF16, 2, 16, (void *)0x1000000, (void *)0x2000000,
                                   (void *)0x3000000 /* SGD takes one state */, FSDP_F32, (void *)0x4000000,
                                   FSDP_BF16, &cfg, 0, 2, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    /* the multi-unit step: nothing to do, then a unit rejected before launch */
    CHECK(fsdp_step_units(NULL, 0, &hp, 2, 0, NULL, NULL, NULL) == FSDP_OK);
    void *fulls[2] = {(void *)0x8000000, (void *)0x9000000};
    fsdp_unit u;
    memset(&u, 0, sizeof(u));
    u.grads = grads;
    u.full_bufs = fulls;
    u.master = (float *)0x1000000;
    u.exp_avg = (float *)0x2000000;
    u.exp_avg_sq = (float *)0x3000000;
    u.shard_out = (void *)0x4000000;
    u.padded_numel = 15; /* not a multiple of world */
    u.world = 2;
    u.grad_dtype = FSDP_BF16;
    u.out_dtype = FSDP_BF16;
    u.n_full = 2;
    CHECK(fsdp_step_units(&u, 1, &hp, 1, 1, NULL, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    u.padded_numel = 0; /* an empty unit is skipped */
    CHECK(fsdp_step_units(&u, 1, &hp, 1, 1, NULL, NULL, NULL) == FSDP_OK);
    /* the variant multi-unit step: SGD takes one state */
    fsdp_unit_ex v;
    memset(&v, 0, sizeof(v));
    v.grads = grads;
    v.full_bufs = fulls;
    v.param = (void *)0x1000000;
    v.state0 = (void *)0x2000000;
    v.state1 = (void *)0x3000000;
    v.shard_out = (void *)0x4000000;
    v.padded_numel = 16;
    v.world = 2;
    v.grad_dtype = FSDP_BF16;
    v.state_dtype = FSDP_F32;
    v.out_dtype = FSDP_BF16;
    v.n_full = 2;
    CHECK(fsdp_step_units_ex(&v, 1, &cfg, 1, NULL, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_units_ex(NULL, 0, &cfg, 1, NULL, NULL, NULL) == FSDP_OK);
    CHECK(fsdp_step_units_ex(&v, 1, NULL, 1, NULL, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    /* the launch-count query: an empty model makes none; no output, or an
     * invalid unit, is refused */
    int64_t launches = -1;
    CHECK(fsdp_step_units_launches(NULL, 0, &hp, 1, 0, &launches) == FSDP_OK && launches == 0);
    CHECK(fsdp_step_units_launches(NULL, 0, &hp, 1, 0, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_units_ex_launches(&v, 1, &cfg, 1, &launches) == FSDP_ERR_INVALID_ARG);
    /* the captured step: no handle to fill, no graph to launch */
    fsdp_step_graph *graph = (fsdp_step_graph *)&u; /* overwritten with NULL on error */
    CHECK(fsdp_step_graph_create(NULL, 1, 1, 0, NULL, NULL, &graph) == FSDP_ERR_INVALID_ARG && graph == NULL);
    CHECK(fsdp_step_graph_create(&u, 1, 1, 0, NULL, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_graph_launch(NULL, &hp, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_graph_destroy(NULL) == FSDP_OK);
    /* the validated plan: no handle to fill, no plan to launch */
    fsdp_step_plan *plan = (fsdp_step_plan *)&u; /* overwritten with NULL on error */
    CHECK(fsdp_step_plan_create(NULL, 1, 1, 0, NULL, NULL, &plan) == FSDP_ERR_INVALID_ARG && plan == NULL);
    CHECK(fsdp_step_plan_create(&u, 1, 1, 0, NULL, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_plan_create_ex(&v, 1, &cfg, 1, NULL, NULL, &plan) == FSDP_ERR_INVALID_ARG && plan == NULL);
    CHECK(fsdp_step_plan_launch(NULL, &hp, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_plan_launch_ex(NULL, &cfg, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_step_plan_destroy(NULL) == FSDP_OK);
    CHECK(fsdp_take_wait_timeouts(NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_check_bounded_wait(0, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_check_bounded_wait(((int64_t)1 << 31) + 1, NULL, NULL) == FSDP_ERR_INVALID_ARG);
    CHECK(fsdp_last_cuda_error() == 0);
    printf("ok\n");
    return 0;
}
