/* Plain-C GPU client of include/fsdp.h: no Python, no torch. Allocates the
 * buffers of one unit (N = 2, P = 4099, padded to 4100) with the CUDA runtime,
 * runs three steps through the C ABI on a stream it creates (flatten of the
 * master's two pieces; steps 1 and 2: the fused reduce-scatter + AdamW + cast
 * and an all-gather into both gathered buffers; step 3: the same unit as a
 * one-unit model validated once, fsdp_step_plan_create, and launched,
 * fsdp_step_plan_launch), and writes the results as raw bytes to the file
 * named by argv[1]: master, exp_avg, exp_avg_sq (fp32), shard_out and both
 * gathered buffers (bf16 bits), the non-finite count and the count of the
 * gathers' bounded waits that gave up (uint32 each). tests/test_c_client.py
 * compares them with the oracle. Inputs are exact in bf16/fp32 and defined
 * below, so the test can rebuild them. Prints "ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fsdp.h"

#define N 2
#define P 4099
#define PPAD 4100
#define STEPS 3

#define CK(x)                                                                          \
    do {                                                                               \
        if ((x) != cudaSuccess) {                                                      \
            fprintf(stderr, "CUDA call failed (line %d)\n", __LINE__);                 \
            return 1;                                                                  \
        }                                                                              \
    } while (0)
#define FS(x)                                                                          \
    do {                                                                               \
        fsdp_status s_ = (x);                                                          \
        if (s_ != FSDP_OK) {                                                           \
            fprintf(stderr, "%s (line %d)\n", fsdp_status_string(s_), __LINE__);       \
            return 1;                                                                  \
        }                                                                              \
    } while (0)

/* gradient of rank q at step t, element j: a multiple of 2^-10 in [-48, 48]
 * * 2^-10, exact in bf16; bf16 bits are the top half of the fp32 bits */
static uint16_t grad_bits(int q, int t, int j) {
    const float x = (float)((j * 7 + q * 13 + t * 29) % 97 - 48) / 1024.0f;
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

/* initial master, element j: a multiple of 2^-11 */
static float master0(int j) { return (float)((j * 5) % 201 - 100) / 2048.0f; }

int main(int argc, char **argv) {
    if (argc != 2) return 2;
    static float h_master[P];
    static uint16_t h_grad[N][PPAD];
    for (int j = 0; j < P; ++j) h_master[j] = master0(j);

    cudaStream_t stream;
    CK(cudaStreamCreate(&stream));
    float *piece[2], *master, *m, *v;
    void *grads_d[N], *shard, *full[2];
    uint32_t *nonfinite, *wait_timeouts;
    CK(cudaMalloc((void **)&piece[0], 4096 * 4));  /* the unit's two parameters: w[64,64], b[3] */
    CK(cudaMalloc((void **)&piece[1], 3 * 4));
    CK(cudaMalloc((void **)&master, PPAD * 4));
    CK(cudaMalloc((void **)&m, PPAD * 4));
    CK(cudaMalloc((void **)&v, PPAD * 4));
    for (int q = 0; q < N; ++q) CK(cudaMalloc(&grads_d[q], PPAD * 2));
    CK(cudaMalloc(&shard, PPAD * 2));
    for (int d = 0; d < 2; ++d) CK(cudaMalloc(&full[d], PPAD * 2));
    CK(cudaMalloc((void **)&nonfinite, 4));
    CK(cudaMalloc((void **)&wait_timeouts, 4));
    CK(cudaMemset(m, 0, PPAD * 4));
    CK(cudaMemset(v, 0, PPAD * 4));
    CK(cudaMemset(nonfinite, 0, 4));
    CK(cudaMemset(wait_timeouts, 0, 4));
    CK(cudaMemcpy(piece[0], h_master, 4096 * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(piece[1], h_master + 4096, 3 * 4, cudaMemcpyHostToDevice));

    /* the FlatParameter: flatten + zero pad, and the views of its parameters */
    const void *srcs[2] = {piece[0], piece[1]};
    const int64_t numels[2] = {4096, 3};
    fsdp_view views[2];
    FS(fsdp_flatten_pad(srcs, numels, 2, FSDP_F32, N, master, PPAD, views, stream));
    if (views[1].offset != 4096 || views[1].numel != 3) return 3;

    /* the same unit as a one-unit model, for the last step */
    fsdp_unit unit;
    memset(&unit, 0, sizeof(unit));
    unit.grads = (const void *const *)grads_d;
    unit.full_bufs = full;
    unit.master = master;
    unit.exp_avg = m;
    unit.exp_avg_sq = v;
    unit.shard_out = shard;
    unit.padded_numel = PPAD;
    unit.world = N;
    unit.grad_dtype = FSDP_BF16;
    unit.out_dtype = FSDP_BF16;
    unit.n_full = 2;
    fsdp_step_plan *plan = NULL;
    FS(fsdp_step_plan_create(&unit, 1, 1, 0, nonfinite, wait_timeouts, &plan));

    for (int t = 1; t <= STEPS; ++t) {
        for (int q = 0; q < N; ++q) {
            for (int j = 0; j < PPAD; ++j) h_grad[q][j] = j < P ? grad_bits(q, t, j) : 0;
            CK(cudaMemcpyAsync(grads_d[q], h_grad[q], PPAD * 2, cudaMemcpyHostToDevice, stream));
        }
        fsdp_adamw_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, t, 1.0f};
        if (t < STEPS) {
            FS(fsdp_reduce_scatter_adam_cast((const void *const *)grads_d, FSDP_BF16, N, PPAD, master, m, v, shard,
                                             FSDP_BF16, &hp, 0, N, nonfinite, stream));
            FS(fsdp_all_gather(shard, FSDP_BF16, N, PPAD, full, 2, wait_timeouts, stream));
        } else {
            FS(fsdp_step_plan_launch(plan, &hp, stream));
        }
        CK(cudaStreamSynchronize(stream)); /* the host gradient buffer is reused */
    }
    FS(fsdp_step_plan_destroy(plan));

    static float out_f[3][PPAD];
    static uint16_t out_h[3][PPAD];
    uint32_t nf = 0, wt = 0;
    CK(cudaMemcpy(out_f[0], master, PPAD * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_f[1], m, PPAD * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_f[2], v, PPAD * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_h[0], shard, PPAD * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_h[1], full[0], PPAD * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_h[2], full[1], PPAD * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&nf, nonfinite, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&wt, wait_timeouts, 4, cudaMemcpyDeviceToHost));

    FILE *f = fopen(argv[1], "wb");
    if (!f) return 4;
    fwrite(out_f, 4, 3 * PPAD, f);
    fwrite(out_h, 2, 3 * PPAD, f);
    fwrite(&nf, 4, 1, f);
    fwrite(&wt, 4, 1, f);
    fclose(f);
    printf("ok\n");
    return 0;
}
