// group.cuh -- argument blocks of the batched launches: one launch of the
// fused update, or of the all-gather, over many small units that share the
// world size and the dtypes. A model of many small FSDP units (RegNet vision
// models under VISSL are among FSDP's users: "Fully Sharded Data Parallel:
// faster AI training with fewer GPUs", "Adoption paths for FSDP", "Computer
// vision models in VISSL") would otherwise pay a kernel launch, a ramp-up and
// a tail per unit, which for units of a few hundred thousand parameters cost
// more than their bytes.
//
// The blocks travel by value as the kernel's only argument (kernel parameter
// space, at most 32,764 bytes), so a batched launch needs no device memory of
// its own. Each CTA finds its unit by a binary search over the units' first
// CTA indices and then runs the per-unit kernel's code on it unchanged.
#pragma once

#include "common.cuh"

namespace fsdp {

// Units per batched launch. 256 units' descriptors take 30.8 KB of the
// 32,764 bytes of kernel parameter space (the asserts below). Measured
// against 128 (the same results bit for bit): a model of 500 units of 20 k
// elements 0.104 against 0.121 ms per step (4 launches instead of 8); 200
// and 256 units of 50 k unchanged (their two groups of 128 already overlapped
// on the two side streams).
#ifndef FSDP_GROUP_MAX
#define FSDP_GROUP_MAX 256
#endif
constexpr int kGroupMax = FSDP_GROUP_MAX;
constexpr int kGroupMaxWorld = 8;                       // gradient / destination pointers per unit
#ifndef FSDP_GROUP_MAX_NUMEL_LOG2
#define FSDP_GROUP_MAX_NUMEL_LOG2 24
#endif
constexpr int64_t kGroupMaxNumel = int64_t(1) << FSDP_GROUP_MAX_NUMEL_LOG2;  // units up to this size are batched
constexpr int kGroupGatherTile = 16384;                 // bytes per CTA of the batched gather
// Threads per CTA of both batched updates. A unit's CTA count is sized from
// it on the host (group_update_ctas), so each batched kernel asserts that it
// launches exactly this many: a build that changed one kernel's block size
// alone would otherwise leave chunks of every unit unvisited.
constexpr int kGroupThreads = 256;

// One unit of a batched update: all ranks' blocks [0, numel), every base
// pointer 16-byte aligned, state in device memory.
struct GroupUnit {
    const void *grads[kGroupMaxWorld];  // world pointers used
    float *master;
    float *m;
    float *v;
    void *out;
    int64_t numel;      // padded_numel
    int64_t cta_begin;  // the unit's first CTA in the launch
    int32_t ncta;       // its CTAs: max(1, ceil(numel / 8 / threads per CTA))
    int32_t pad;
};

struct RsaGroupArgs {
    AdamScalars s;  // first member: the block a captured step rewrites per step
    uint32_t *nonfinite;
    int32_t n;      // units
    int32_t world;
    GroupUnit u[kGroupMax];
};

// One unit of a batched update with the first all-gather fused in (the
// update also stores every output word to the unit's gathered buffers):
// GroupUnit's fields and the gathered buffers' pointers. The descriptor is
// 184 bytes, so a launch takes up to kFusedGroupMax units (23.6 KB of
// parameter space).
constexpr int kFusedGroupMax = 128;

struct FusedGroupUnit {
    const void *grads[kGroupMaxWorld];  // world pointers used
    void *full[kGroupMaxWorld];         // n_full pointers used
    float *master;
    float *m;
    float *v;
    void *out;          // the compute-dtype shard (shard_out)
    int64_t numel;      // padded_numel
    int64_t cta_begin;  // the unit's first CTA in the launch
    int32_t ncta;       // its CTAs, as group_update_ctas counts them
    int32_t n_full;     // 1..kGroupMaxWorld
};

struct RsaFusedGroupArgs {
    AdamScalars s;  // first member: the block a captured step rewrites per step
    uint32_t *nonfinite;
    int32_t n;      // units
    int32_t world;
    FusedGroupUnit u[kFusedGroupMax];
};

// One unit of a batched all-gather: src and every destination 16-byte aligned.
struct GatherGroupUnit {
    const void *src;
    void *dst[kGroupMaxWorld];  // n_dst pointers used
    int64_t nbytes;
    int64_t tile_begin;  // the unit's first CTA (one tile per CTA)
    int32_t n_dst;
    int32_t pad;
};

struct GatherGroupArgs {
    int32_t n;
    int32_t pad;
    uint32_t *timeouts;  // the call's count of bounded waits that gave up (device, or NULL)
    GatherGroupUnit u[kGroupMax];
};

// One unit of a batched variant step (fsdp_reduce_scatter_step's update):
// all ranks' blocks [0, numel), every base pointer 16-byte aligned, the
// parameter in device memory.
struct StepGroupUnit {
    const void *grads[kGroupMaxWorld];  // world pointers used
    void *param;
    void *s0;
    void *s1;   // NULL for SGD
    void *out;  // NULL for bf16/fp16 state
    int64_t numel;
    int64_t cta_begin;
    int32_t ncta;
    int32_t pad;
};

struct StepGroupArgs {
    StepScalars k;        // first members: the block a captured step rewrites per step
    int32_t reduce_lowp;
    int32_t world;
    uint32_t *nonfinite;
    int32_t n;
    int32_t pad;
    StepGroupUnit u[kGroupMax];
};

static_assert(sizeof(RsaGroupArgs) < 32764, "kernel parameter space");
static_assert(sizeof(StepGroupArgs) < 32764, "kernel parameter space");
static_assert(sizeof(GatherGroupArgs) < 32764, "kernel parameter space");
static_assert(sizeof(RsaFusedGroupArgs) < 32764, "kernel parameter space");

// CTAs of one unit in a batched update (kGroupThreads chunks each), and
// tiles of one unit in a batched gather (at least one each: a CTA also takes
// the elements or bytes after the vector part).
int32_t group_update_ctas(int64_t numel);
int64_t group_gather_tiles(int64_t nbytes);

// Launch `grid` CTAs of the batched kernels on stream s.
fsdp_status launch_rsa_group(const RsaGroupArgs &g, int grad_dtype, int out_dtype, int64_t grid, cudaStream_t s);
fsdp_status launch_gather_group(const GatherGroupArgs &g, int64_t grid, cudaStream_t s);
// The batched update with the first gather fused in (rsa_group_fused.cu).
fsdp_status launch_rsa_fused_group(const RsaFusedGroupArgs &g, int grad_dtype, int out_dtype, int64_t grid,
                                   cudaStream_t s);

// The batched variant step, one translation unit per optimizer
// (step_group_<optimizer>.cu); (state, out) dtype pairs as the per-unit
// variant kernel: fp32 state with any compute dtype, or bf16/fp16 state that
// is its own shard.
fsdp_status launch_step_group_adamw(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype,
                                    int64_t grid, cudaStream_t s);
fsdp_status launch_step_group_sgd(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype,
                                  int64_t grid, cudaStream_t s);
fsdp_status launch_step_group_adamax(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype,
                                     int64_t grid, cudaStream_t s);
fsdp_status launch_step_group_adadelta(const StepGroupArgs &g, int grad_dtype, int out_dtype, int state_dtype,
                                       int64_t grid, cudaStream_t s);

}  // namespace fsdp
