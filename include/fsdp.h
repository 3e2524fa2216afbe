/*
 * fsdp.h -- C ABI of libfsdpreduce.so, the FSDP FlatParameter step on one
 * GB300 (sm_103a).
 *
 * One FSDP unit's step, as the sources describe it:
 *   "Fully Sharded Data Parallel: faster AI training with fewer GPUs"
 *   (techreport.ngo), "From all-reduce to sharded parameters": the DDP
 *   all-reduce splits into a reduce-scatter (gradients summed in equal blocks,
 *   block r to rank r) and an all-gather; each rank updates only its own
 *   shard of the weights; the result is identical to DDP.
 *   "FSDP (Fully Sharded Data Parallel)" (vanos001.github.io), "The Sharding
 *   Scheme", "The Per-Layer Communication", "Mixed Precision and FSDP":
 *   P/N parameter, gradient and fp32 Adam-state shards per rank; all-gather
 *   before forward and backward, reduce-scatter after backward; bf16 compute
 *   copy with fp32 master weights.
 *   "Data Parallelism" (vanos001.github.io), "The Basic Protocol":
 *   G_avg = (1/N) sum_i G_i; W = W - lr * Adam(G_avg, m, v).
 *   "fairseq ... FSDP 实战指南" (zskr.cn), "参数定义与底层实现" and
 *   "限制与兼容性说明": fp32 reduce-scatter option, fp16 compute dtype, and
 *   exactness for pointwise optimizers such as AdamW.
 *
 * Emulation. The N ranks of one unit live in one GPU's memory: rank q's
 * gradient is its own flat buffer; the fp32 master, exp_avg (m) and
 * exp_avg_sq (v) of all ranks are the concatenation of the N shards, so rank
 * r's shard is elements [r*S, (r+1)*S) of each, S = P_pad / N. A call may
 * emulate any contiguous subset of ranks [rank_begin, rank_end).
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device addresses of the current device;
 *    pointer arrays themselves (grads, srcs, full_bufs) are HOST arrays of
 *    device addresses. The caller owns every buffer; the library allocates
 *    no device memory and keeps no state besides launch caches (the SM
 *    count and kernel occupancies per device), the side streams of
 *    fsdp_step_units, one device counter of bounded waits that gave up
 *    (fsdp_take_wait_timeouts), and the host memory of the handles it
 *    returns (fsdp_step_graph, fsdp_step_plan).
 *  - Bounded waits. The all-gather's bulk-copy (TMA) pipeline waits on
 *    shared-memory barriers for its loads; each wait gives up after about
 *    one second of SM clocks. A wait that gives up makes its CTA return
 *    early (after one more bounded wait on each load it still has in flight,
 *    so that a copy that is only slow lands first): the gathered buffers of
 *    that call are then incomplete. Every entry point that launches a gather
 *    takes `wait_timeouts`, a device uint32 (or NULL) that each wait giving
 *    up increments; the caller zeroes it and reads it after the call's work,
 *    stream-ordered like nonfinite_count, with no device-wide
 *    synchronization. A non-zero count means that call's gathered buffers,
 *    and anything launched after it on the device, must not be trusted: a
 *    bulk copy that does not complete within a second is a fault of the
 *    device, not a slow copy. The count is 0 in normal operation.
 *  - Offload. Where an argument says "device or mapped host", the buffer
 *    may also be page-locked host memory mapped into the device's address
 *    space (cudaHostAlloc, or cudaHostRegister with mapping; the same
 *    address under unified addressing). The kernel then reads and writes it
 *    over the host link: the optimizer state and fp32 master kept in CPU
 *    memory ("FSDP (Fully Sharded Data Parallel)", "CPU Offloading";
 *    "fairseq ... FSDP 实战指南", --cpu-offload), updated by the same kernel.
 *    The other buffers must be device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Device work is enqueued on it and the call returns without
 *    synchronizing.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error status and enqueues nothing. A launch
 *    failure returns FSDP_ERR_CUDA; fsdp_last_cuda_error() then gives the
 *    cudaError_t value. The calls that take a whole model (fsdp_step_units*,
 *    the plans and the captured steps) keep host bookkeeping of their own;
 *    if the host cannot provide it they return FSDP_ERR_HOST_MEMORY, with
 *    nothing enqueued. Nothing aborts, traps or prints.
 *  - Element pointers must be aligned to their element size. Any such
 *    alignment works; 16-byte-aligned bases take the vectorised path.
 */
#ifndef FSDP_H
#define FSDP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FSDP_MAX_WORLD 64 /* largest N (emulated ranks) and largest all-gather fan-out */
#define FSDP_MAX_NDIM 8   /* largest rank of an original parameter's shape */

typedef enum {
    FSDP_OK = 0,
    FSDP_ERR_INVALID_ARG = 1,       /* null pointer, bad size, bad range, aliasing, ... */
    FSDP_ERR_ALIGNMENT = 2,         /* a pointer not aligned to its element size */
    FSDP_ERR_CUDA = 3,              /* a CUDA call or kernel launch failed */
    FSDP_ERR_UNSUPPORTED_DTYPE = 4, /* dtype not accepted by this entry point */
    FSDP_ERR_HOST_MEMORY = 5        /* host memory for the library's bookkeeping of a model ran out */
} fsdp_status;

typedef enum { FSDP_F32 = 0, FSDP_BF16 = 1, FSDP_F16 = 2 } fsdp_dtype;

/* Pointwise optimizers of fsdp_reduce_scatter_step ("fairseq ... FSDP
 * 实战指南", "限制与兼容性说明": FSDP works with Adam, AdamW, Adadelta,
 * Adamax, SGD and other pointwise optimizers). */
typedef enum {
    FSDP_OPT_ADAMW = 0,     /* states: exp_avg, exp_avg_sq */
    FSDP_OPT_SGD = 1,       /* state: momentum buffer (state1 unused) */
    FSDP_OPT_ADAMAX = 2,    /* states: exp_avg, exp_inf */
    FSDP_OPT_ADADELTA = 3   /* states: square_avg, acc_delta */
} fsdp_optimizer;

/* A view of one original parameter inside a FlatParameter ("FSDP (Fully
 * Sharded Data Parallel)", "Common Pitfalls": use_orig_params keeps
 * named-parameter access as views into the flat parameter). */
typedef struct {
    int32_t ndim;
    int32_t reserved;               /* 0 */
    int64_t shape[FSDP_MAX_NDIM];   /* dims beyond ndim are 0 */
    int64_t offset;                 /* first element inside the flat buffer */
    int64_t numel;                  /* product of shape[0..ndim) (1 for ndim 0) */
} fsdp_view;

/* AdamW hyperparameters of one step. One parameter group per unit: the same
 * values apply to every element, biases and norm weights included ("Fully
 * Sharded Data Parallel: ...", "Harnessing FSDP's full power", item 3). */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;  /* decoupled: p <- p * (1 - lr * weight_decay) */
    int64_t step;        /* t, 1 on the first step */
    float grad_scale;    /* static loss scale the gradients carry; 1 if none */
} fsdp_adamw_hparams;

/* Configuration of one variant step (fsdp_reduce_scatter_step). */
typedef struct {
    int32_t optimizer;     /* fsdp_optimizer */
    int32_t reduce_dtype;  /* fsdp_dtype: FSDP_F32 (fp32 reduce-scatter) or the gradient dtype */
    float lr;
    float beta1;           /* AdamW/Adamax beta1; SGD momentum; Adadelta rho */
    float beta2;           /* AdamW/Adamax beta2 (unused otherwise) */
    float eps;             /* AdamW/Adamax/Adadelta epsilon (unused by SGD) */
    float weight_decay;    /* AdamW: decoupled; SGD/Adamax/Adadelta: wd*p added to the gradient */
    int64_t step;          /* t, 1 on the first step */
    float grad_scale;      /* static loss scale the gradients carry; 1 if none */
} fsdp_step_config;

/* The buffers of one FSDP unit (one FlatParameter) for fsdp_step_units,
 * laid out as the single-unit entry points take them. Caller-owned. */
typedef struct {
    const void *const *grads;    /* host array of `world` pointers (device or mapped host), padded_numel each */
    void *const *full_bufs;      /* host array of n_full device pointers, padded_numel each (NULL if n_full == 0) */
    float *master;               /* fp32, device or mapped host, padded_numel */
    float *exp_avg;              /* fp32, device or mapped host, padded_numel */
    float *exp_avg_sq;           /* fp32, device or mapped host, padded_numel */
    void *shard_out;             /* device, padded_numel elements of out_dtype */
    int64_t padded_numel;        /* a multiple of world (0: the unit is skipped) */
    int32_t world;               /* N, 1..FSDP_MAX_WORLD */
    int32_t grad_dtype;          /* fsdp_dtype */
    int32_t out_dtype;           /* fsdp_dtype */
    int32_t n_full;              /* 0..FSDP_MAX_WORLD */
} fsdp_unit;

/* ceil(numel / world) * world: the FlatParameter length after zero padding
 * at the end, so that it splits into `world` equal shards. Returns -1 when
 * numel < 0 or world < 1. Host only. */
int64_t fsdp_padded_numel(int64_t numel, int world);

/* Layout of a FlatParameter, host only, touches no GPU.
 * shapes: the n_tensors shapes concatenated (ndims[k] entries for tensor k,
 * in registration order; ndims[k] in [0, FSDP_MAX_NDIM], negative dims are
 * invalid). Writes n_tensors views (offset = sum of the previous numels, no
 * gaps) to views_out and the padded length to *padded_numel_out.
 * Source: "Fully Sharded Data Parallel: ...", "Harnessing FSDP's full
 * power", item 3 (a unit's parameters are flattened into a single tensor);
 * "FSDP (Fully Sharded Data Parallel)", "Common Pitfalls" (views of the
 * original parameters). */
fsdp_status fsdp_unflatten_views(const int64_t *shapes, const int32_t *ndims, int n_tensors,
                                 int world, fsdp_view *views_out, int64_t *padded_numel_out);

/* Flatten and pad (device). Copies n_tensors contiguous device tensors of
 * `dtype` (srcs[k] holds numels[k] elements) back to back into dst_flat and
 * zero-fills the padding [sum(numels), dst_numel). dst_numel must equal
 * fsdp_padded_numel(sum(numels), world). Sources must not overlap dst_flat.
 * views_out (host, may be NULL) receives one 1-D view per tensor.
 * Same sources as fsdp_unflatten_views. */
fsdp_status fsdp_flatten_pad(const void *const *srcs, const int64_t *numels, int n_tensors,
                             fsdp_dtype dtype, int world, void *dst_flat, int64_t dst_numel,
                             fsdp_view *views_out, void *stream);

/* The fused reduce-scatter + AdamW + cast (device), for emulated ranks
 * r in [rank_begin, rank_end), i in [0, S), j = r*S + i:
 *   acc  = G_0[j] + G_1[j] + ... + G_{N-1}[j]   fp32, ranks in order 0..N-1
 *   g    = acc * c,            c = fp32(1 / (N * grad_scale))
 *   p    = master[j] * fp32(1 - lr*weight_decay)
 *   m    = beta1 * m[j] + fp32(1 - beta1) * g
 *   v    = beta2 * v[j] + fp32(1 - beta2) * (g * g)
 *   p    = p - alpha * (m / (sqrt(v) / b2s + eps)),
 *          alpha = fp32(lr / (1 - beta1^t)), b2s = fp32(sqrt(1 - beta2^t))
 *   master[j], exp_avg[j], exp_avg_sq[j] = p, m, v   (in place)
 *   shard_out[j] = p rounded to nearest even in out_dtype
 * every operation rounded to fp32 on its own (no fused multiply-add); the
 * scalars are computed in double and rounded once. Elements outside the
 * emulated ranks' blocks are not touched.
 * Sources: the reduce-scatter is "From all-reduce to sharded parameters"
 * (first figure caption) with the average of "The Basic Protocol" and the
 * fp32 accumulation of --fp32-reduce-scatter; the update is the pointwise
 * AdamW step on the local shard ("限制与兼容性说明", second figure caption
 * of "From all-reduce to sharded parameters"); the cast is the compute copy
 * of "Mixed Precision and FSDP". The AdamW formula, the reduction order and
 * the single multiply by c are this library's reading (the pages print none).
 *
 *   grads        host array of `world` pointers (device or mapped host),
 *                each padded_numel elements of grad_dtype (F32, BF16 or
 *                F16); read only.
 *   padded_numel P_pad, a multiple of world (0 is a no-op).
 *   master, exp_avg, exp_avg_sq   fp32 (device or mapped host),
 *                padded_numel each, in place.
 *   shard_out    device, padded_numel elements of out_dtype (F32, BF16,
 *                F16); must not overlap the gradients or the state.
 *   hp           host; step >= 1, grad_scale > 0.
 *   rank_begin, rank_end   0 <= rank_begin <= rank_end <= world.
 *   nonfinite_count  device uint32 or NULL: incremented by the number of
 *                elements whose averaged gradient g is not finite (reported,
 *                never skipped); the caller zeroes it.
 */
fsdp_status fsdp_reduce_scatter_adam_cast(const void *const *grads, fsdp_dtype grad_dtype,
                                          int world, int64_t padded_numel, float *master,
                                          float *exp_avg, float *exp_avg_sq, void *shard_out,
                                          fsdp_dtype out_dtype, const fsdp_adamw_hparams *hp,
                                          int rank_begin, int rank_end,
                                          uint32_t *nonfinite_count, void *stream);

/* The fused update with the all-gather fused in (device): everything
 * fsdp_reduce_scatter_adam_cast does for the emulated ranks [rank_begin,
 * rank_end), and every updated compute-dtype element is also stored to each
 * of the n_dst gathered buffers: full_k[j] = out[j] for j in those ranks'
 * blocks, k < n_dst. With all ranks emulated this equals
 * fsdp_reduce_scatter_adam_cast followed by fsdp_all_gather, without
 * reading shard_out back. shard_out may be NULL (not written): the
 * no-reshard mode keeps the gathered parameters instead of the shard
 * ("Fully Sharded Data Parallel: ...", "Adoption paths for FSDP":
 * --no-reshard-after-forward; "fairseq ... FSDP 实战指南", "参数定义与底层实现":
 * reshard_after_forward).
 *   full_bufs    host array of n_dst device pointers (1 <= n_dst <=
 *                FSDP_MAX_WORLD), padded_numel elements of out_dtype each;
 *                no written buffer may overlap another or the gradients.
 * Other arguments and errors as fsdp_reduce_scatter_adam_cast. */
fsdp_status fsdp_reduce_scatter_adam_cast_gather(const void *const *grads, fsdp_dtype grad_dtype,
                                                 int world, int64_t padded_numel, float *master,
                                                 float *exp_avg, float *exp_avg_sq, void *shard_out,
                                                 fsdp_dtype out_dtype, void *const *full_bufs, int n_dst,
                                                 const fsdp_adamw_hparams *hp, int rank_begin,
                                                 int rank_end, uint32_t *nonfinite_count, void *stream);

/* The variant steps (device): the fused reduce-scatter + optimizer step +
 * cast with a choice of optimizer, reduction precision and state precision,
 * for emulated ranks [rank_begin, rank_end), i in [0, S), j = r*S + i:
 *   acc = G_0[j]; acc = acc + G_q[j] for q = 1..N-1, in fp32; with
 *         reduce_dtype equal to the gradient dtype every partial sum is
 *         rounded to that dtype (the reduce-scatter without
 *         --fp32-reduce-scatter, "参数定义与底层实现"; the FP16 reduce-scatter of
 *         "Harnessing FSDP's full power", item 4)
 *   g   = acc * fp32(1 / (N * grad_scale))
 *   then, one fp32 rounding per operation (wd = weight_decay):
 *   AdamW:    as fsdp_reduce_scatter_adam_cast
 *   SGD:      d = g + wd*p; b = d if step == 1 else beta1*b + d; p = p - lr*b
 *   Adamax:   d = g + wd*p; m = beta1*m + fp32(1-beta1)*d;
 *             u = max(beta2*u, |d| + eps) (NaN if either side is NaN);
 *             p = p - fp32(lr/(1-beta1^t)) * (m/u)
 *   Adadelta: d = g + wd*p; s = beta1*s + fp32(1-beta1)*(d*d);
 *             delta = (sqrt(a + eps)/sqrt(s + eps))*d;
 *             a = beta1*a + fp32(1-beta1)*(delta*delta); p = p - lr*delta
 * The rules are the textbook ones; the pages name the optimizers only.
 *   state_dtype FSDP_F32: param is the fp32 master, state0/state1 fp32, and
 *     shard_out (out_dtype, required) receives p rounded to nearest even.
 *   state_dtype FSDP_BF16 / FSDP_F16: param, state0 and state1 hold that
 *     dtype with no fp32 master ("Mixed Precision and FSDP": pure bf16;
 *     "Harnessing FSDP's full power", item 4: FP16 master weights); each
 *     value is widened, updated in fp32 and rounded to nearest even when
 *     stored; param is itself the rank's compute-dtype shard, so shard_out
 *     must be NULL and out_dtype equal to state_dtype.
 *   grads        host array of `world` pointers (device or mapped host),
 *                padded_numel each.
 *   param, state0, state1   device or mapped host, padded_numel elements
 *                each, in place; state1 must be NULL for SGD and non-NULL
 *                otherwise.
 *   cfg          host; step >= 1, grad_scale > 0, optimizer and
 *                reduce_dtype as above.
 * Other arguments, in-place rules and errors as
 * fsdp_reduce_scatter_adam_cast. */
fsdp_status fsdp_reduce_scatter_step(const void *const *grads, fsdp_dtype grad_dtype, int world,
                                     int64_t padded_numel, void *param, void *state0, void *state1,
                                     fsdp_dtype state_dtype, void *shard_out, fsdp_dtype out_dtype,
                                     const fsdp_step_config *cfg, int rank_begin, int rank_end,
                                     uint32_t *nonfinite_count, void *stream);

/* All-gather (device): every destination receives the whole rank-ordered
 * concatenation of the shards, full_k[j] = shard_out[j] for j < padded_numel,
 * k < n_dst. Rank r's shard is shard_out[r*S, (r+1)*S), so the copy is the
 * all-gather of "From all-reduce to sharded parameters" (first figure
 * caption) and of "The Per-Layer Communication" (before forward and before
 * backward), one destination per emulated rank.
 *   shard_out    device, padded_numel elements of dtype (any of the three).
 *   full_bufs    host array of n_dst device pointers (1 <= n_dst <=
 *                FSDP_MAX_WORLD), padded_numel elements each; they must not
 *                overlap shard_out or each other. Host memory is refused
 *                (FSDP_ERR_INVALID_ARG) for shard_out and full_bufs alike:
 *                the copy uses bulk transfers between device buffers.
 *   world        N; padded_numel must be a multiple of it.
 *   wait_timeouts  device uint32 or NULL: incremented by each bounded wait
 *                of this call that gave up (see "Bounded waits" above). */
fsdp_status fsdp_all_gather(const void *shard_out, fsdp_dtype dtype, int world,
                            int64_t padded_numel, void *const *full_bufs, int n_dst,
                            uint32_t *wait_timeouts, void *stream);

/* The step of a whole model (device): its FSDP units in order, each one's
 * fused reduce-scatter + AdamW + cast over all its ranks followed by
 * `gathers` all-gathers of its shard_out into its n_full buffers, in the
 * order of `stream` -- the per-unit driver of "FSDP (Fully Sharded Data Parallel)",
 * "The Per-Layer Communication" (one unit per wrapped layer, each
 * reduce-scattered and gathered on its own) in one call. With
 * fuse_first_gather != 0 the first gather of each unit is written by its
 * update kernel (as fsdp_reduce_scatter_adam_cast_gather) and gathers - 1
 * separate gathers follow.
 *   units        host array of n_units descriptors (n_units >= 0).
 *   hp           host; the same hyperparameters for every unit (one
 *                optimizer over the model); step >= 1, grad_scale > 0.
 *   gathers      0..FSDP_MAX_WORLD; units with gathers > 0 need n_full >= 1.
 *   nonfinite_count  device uint32 or NULL, summed over all units.
 *   wait_timeouts    device uint32 or NULL, the bounded waits of all the
 *                units' gathers that gave up (see "Bounded waits" above).
 * Every unit is validated as the single-unit entry points validate it, and
 * no buffer written by one unit may overlap a buffer written or a gradient
 * read by another, before anything is enqueued: an invalid unit makes the
 * call return its status and enqueue nothing. FSDP_ERR_CUDA reports a launch that failed
 * after the units before it were enqueued.
 * Scheduling: the units share no written buffer, so with two or more of
 * them their kernels are spread round-robin over two streams the library
 * keeps per host thread and device (created on first use), which wait for
 * the work already on `stream` and which `stream` waits for afterwards; a
 * unit's kernels run in order on one of them and overlap the neighbouring
 * unit's. Work enqueued on `stream` after the call sees every unit done.
 * Batching: small units are stepped together, up to 256 per launch of each
 * kernel (128 when the first gather is fused into the update), when they
 * share N (1, 2, 4 or 8), the dtype pair and the gathers, and each has at most
 * 2^24 elements, at most 8 gathered buffers, 16-byte aligned buffers and
 * its state in device memory; every element sees the same operations as in
 * the unit's own launch, so the results are the same bits. Every other unit
 * keeps its own launches. */
fsdp_status fsdp_step_units(const fsdp_unit *units, int n_units, const fsdp_adamw_hparams *hp,
                            int gathers, int fuse_first_gather, uint32_t *nonfinite_count,
                            uint32_t *wait_timeouts, void *stream);

/* The buffers of one FSDP unit for fsdp_step_units_ex (the variant steps),
 * laid out as fsdp_reduce_scatter_step takes them. Caller-owned. */
typedef struct {
    const void *const *grads;    /* host array of `world` pointers (device or mapped host), padded_numel each */
    void *const *full_bufs;      /* host array of n_full device pointers, padded_numel elements of out_dtype */
    void *param;                 /* state_dtype, device or mapped host, padded_numel */
    void *state0;                /* state_dtype, device or mapped host, padded_numel */
    void *state1;                /* state_dtype, device or mapped host; NULL for SGD */
    void *shard_out;             /* device, out_dtype; fp32 state only (NULL for bf16/fp16 state) */
    int64_t padded_numel;        /* a multiple of world (0: the unit is skipped) */
    int32_t world;               /* N, 1..FSDP_MAX_WORLD */
    int32_t grad_dtype;          /* fsdp_dtype */
    int32_t state_dtype;         /* fsdp_dtype */
    int32_t out_dtype;           /* fsdp_dtype; equal to state_dtype for bf16/fp16 state */
    int32_t n_full;              /* 0..FSDP_MAX_WORLD */
    int32_t reserved;            /* must be 0 (FSDP_ERR_INVALID_ARG otherwise) */
} fsdp_unit_ex;

/* The multi-unit step with the variant update (device): as fsdp_step_units,
 * but each unit takes fsdp_reduce_scatter_step's update under the one `cfg`
 * (optimizer, reduction dtype, hyperparameters), followed by `gathers`
 * all-gathers of its compute-dtype shards -- shard_out for fp32 state, the
 * parameter itself for bf16/fp16 state -- into its n_full buffers. No gather
 * is fused. Validation (every unit as fsdp_reduce_scatter_step validates it,
 * no buffer written by two units or written by one and read by another,
 * nothing enqueued on error), scheduling
 * over the side streams, batching of small units (those that also share
 * the state dtype; the optimizer and reduction are the call's) and errors as
 * fsdp_step_units. */
fsdp_status fsdp_step_units_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                               int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                               void *stream);

/* How many kernel launches fsdp_step_units (and the step captured from the
 * same arguments) makes for these units, gathers and fusion, with the small
 * units batched as that call batches them: per unit or batch one update and
 * one launch per separate gather, nothing for empty units. The units are
 * validated as fsdp_step_units validates them (the same statuses); nothing
 * is enqueued and nothing runs on the device.
 *   hp             host; validated, not otherwise used.
 *   launches_out   host; receives the count. */
fsdp_status fsdp_step_units_launches(const fsdp_unit *units, int n_units, const fsdp_adamw_hparams *hp,
                                     int gathers, int fuse_first_gather, int64_t *launches_out);

/* The same for fsdp_step_units_ex. */
fsdp_status fsdp_step_units_ex_launches(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                        int gathers, int64_t *launches_out);

/* A model step captured as a CUDA graph (opaque; host memory owned by the
 * library, freed by fsdp_step_graph_destroy). */
typedef struct fsdp_step_graph fsdp_step_graph;

/* Capture the step fsdp_step_units would enqueue for these units, gathers,
 * fusion and counters into a CUDA graph, instantiated on the current device.
 * The units are validated as fsdp_step_units validates them; nothing runs.
 * The graph holds the buffers' addresses: they must stay allocated, and a
 * step launched from it touches exactly those buffers. Each launch writes
 * its own step's scalars, so one graph serves every step: one launch for
 * the whole model, batched launches included.
 *   graph_out    host; receives the handle (NULL on error). */
fsdp_status fsdp_step_graph_create(const fsdp_unit *units, int n_units, int gathers, int fuse_first_gather,
                                   uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                   fsdp_step_graph **graph_out);

/* Launch the captured step on `stream` with the scalars of hp (computed as
 * fsdp_reduce_scatter_adam_cast computes them, per unit for its world size).
 * Stream-ordered and asynchronous like the other entry points; results are
 * bit-identical to fsdp_step_units with the same hp. Not thread-safe for
 * one graph (each launch rewrites its update nodes). */
fsdp_status fsdp_step_graph_launch(fsdp_step_graph *graph, const fsdp_adamw_hparams *hp, void *stream);

/* The same for a model of variant units (fsdp_step_units_ex): captured with
 * cfg's optimizer, whose kernels the graph holds; cfg is validated as
 * fsdp_step_units_ex validates it. */
fsdp_status fsdp_step_graph_create_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                      int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                      fsdp_step_graph **graph_out);

/* Launch a captured variant step with cfg's scalars and reduction dtype.
 * cfg->optimizer must be the one the graph was captured with, and
 * reduce_dtype FSDP_F32 or every unit's gradient dtype; otherwise nothing
 * is launched. A graph from fsdp_step_graph_create takes
 * fsdp_step_graph_launch, one from fsdp_step_graph_create_ex this call. */
fsdp_status fsdp_step_graph_launch_ex(fsdp_step_graph *graph, const fsdp_step_config *cfg, void *stream);

/* Free a captured step (NULL is a no-op). Launches already enqueued complete. */
fsdp_status fsdp_step_graph_destroy(fsdp_step_graph *graph);

/* A model step validated once (opaque; host memory owned by the library,
 * freed by fsdp_step_plan_destroy). */
typedef struct fsdp_step_plan fsdp_step_plan;

/* Validate the units of fsdp_step_units once, for repeated steps: every
 * check fsdp_step_units makes on every call (arguments, alignment,
 * residency of the state and of the gathered buffers, overlaps between
 * units) runs here, together with the batching of small units; nothing is
 * enqueued. The plan holds the buffers' addresses, as a captured step does:
 * they must stay allocated, and a step launched from it touches exactly
 * those buffers. The eager counterpart of fsdp_step_graph_create, for
 * callers that do not capture graphs: the per-layer step of "FSDP (Fully
 * Sharded Data Parallel)", "The Per-Layer Communication", with one unit per
 * wrapped layer and the validation paid once per model, not once per step.
 * The plan belongs to the device that is current when it is made: a launch
 * with another device current is refused (FSDP_ERR_INVALID_ARG, nothing
 * enqueued), since the buffers' addresses are that device's.
 *   plan_out     host; receives the handle (NULL on error).
 * Other arguments and statuses as fsdp_step_units. */
fsdp_status fsdp_step_plan_create(const fsdp_unit *units, int n_units, int gathers, int fuse_first_gather,
                                  uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                  fsdp_step_plan **plan_out);

/* The same for the units of fsdp_step_units_ex, validated with cfg (its
 * optimizer is the plan's; its scalars are not kept). */
fsdp_status fsdp_step_plan_create_ex(const fsdp_unit_ex *units, int n_units, const fsdp_step_config *cfg,
                                     int gathers, uint32_t *nonfinite_count, uint32_t *wait_timeouts,
                                     fsdp_step_plan **plan_out);

/* Enqueue one step of a plan from fsdp_step_plan_create on `stream` with
 * the scalars of hp (step >= 1, grad_scale > 0, else FSDP_ERR_INVALID_ARG
 * and nothing enqueued): the launches fsdp_step_units would make with the
 * same arguments, bit-identical results, scheduling and errors as that
 * call. Only hp is checked per call. Not thread-safe for one plan (each
 * launch rewrites the plan's kernel arguments). */
fsdp_status fsdp_step_plan_launch(fsdp_step_plan *plan, const fsdp_adamw_hparams *hp, void *stream);

/* The same for a plan from fsdp_step_plan_create_ex: cfg->optimizer must be
 * the plan's and reduce_dtype FSDP_F32 or every unit's gradient dtype;
 * otherwise nothing is enqueued. */
fsdp_status fsdp_step_plan_launch_ex(fsdp_step_plan *plan, const fsdp_step_config *cfg, void *stream);

/* Free a plan (NULL is a no-op). Launches already enqueued complete. */
fsdp_status fsdp_step_plan_destroy(fsdp_step_plan *plan);

/* Human-readable name of a status. Never NULL. */
const char *fsdp_status_string(fsdp_status status);

/* cudaError_t value behind the calling thread's last FSDP_ERR_CUDA (0 if none). */
int fsdp_last_cuda_error(void);

/* Device-wide diagnostics of the bounded waits (see "Bounded waits" above):
 * every wait that gives up, in any call, is also counted on the current
 * device. This call synchronizes the current device, writes the count
 * accumulated since the previous call to *count_out (host) and resets it.
 * A caller that checks each call reads that call's wait_timeouts instead. */
fsdp_status fsdp_take_wait_timeouts(uint32_t *count_out);

/* Self-test of the failure path of those bounded waits, without a fault:
 * launches one CTA on `stream` (a cudaStream_t; NULL = the legacy default
 * stream) that waits, with the library's bounded wait, on a shared-memory
 * barrier that expects two arrivals and receives one. The wait gives up
 * after about `limit_cycles` SM clock cycles and is counted as a gather's
 * would be: on the device (fsdp_take_wait_timeouts) and in wait_timeouts
 * (device uint32 or NULL); the kernel then returns and the context stays
 * usable. Asynchronous. limit_cycles must be in [1, 2^31]
 * (FSDP_ERR_INVALID_ARG otherwise, nothing launched). */
fsdp_status fsdp_check_bounded_wait(int64_t limit_cycles, uint32_t *wait_timeouts, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_H */
