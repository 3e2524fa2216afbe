// gather.cu -- the all-gather of the compute-dtype shards.
//
// Rank r's shard is shard_out[r*S, (r+1)*S), so the concatenation of the N
// shards in rank order is shard_out itself, and every emulated rank's full
// buffer receives a copy of it ("Fully Sharded Data Parallel: faster AI
// training with fewer GPUs", "From all-reduce to sharded parameters", first
// figure caption; "FSDP (Fully Sharded Data Parallel)", "The Per-Layer
// Communication": gathered before forward and again before backward).
//
// The traffic is (1 + n_dst) * P_pad * sizeof(dtype) bytes: the source is
// read once and written n_dst times, so the copy is HBM-write bound.
//
// Main path (all pointers 16-byte aligned, at least kTmaMinBytes): a TMA
// pipeline. One thread per CTA loads a tile of the source into shared memory
// with a 1-D bulk copy (completion counted on an mbarrier), then issues one
// bulk store of that shared tile per destination; kStages tiles are in
// flight per CTA. One instruction moves a whole tile, so the store stream is
// not limited by per-thread store issue the way 16-byte stores from every
// thread are. Fallback (unaligned pointers, small copies): every thread loads
// one 16-byte word and stores it to every destination; a tail shorter than
// 16 bytes moves in 2-byte units.
#include "group.cuh"
#include "host.cuh"
#include "tma.cuh"

namespace fsdp {
namespace {

constexpr int kThreads = 256;

template <int ND>
__global__ void __launch_bounds__(kThreads)
    gather_kernel(const __grid_constant__ GatherArgs a, int64_t nvec, int64_t tail_units) {
    const int n = ND > 0 ? ND : a.n_dst;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const char *src = static_cast<const char *>(a.src);
    for (int64_t k = tid; k < nvec; k += stride) {
        const uint4 x = ld_stream(src + 16 * k);
        if constexpr (ND > 0) {
#pragma unroll
            for (int d = 0; d < ND; ++d) st_stream(static_cast<char *>(a.dst[d]) + 16 * k, x);
        } else {
            for (int d = 0; d < n; ++d) st_stream(static_cast<char *>(a.dst[d]) + 16 * k, x);
        }
    }
    // 2-byte units after the vector part
    const int64_t base = 16 * nvec;
    for (int64_t u = tid; u < tail_units; u += stride) {
        const uint16_t x = *reinterpret_cast<const uint16_t *>(src + base + 2 * u);
        for (int d = 0; d < n; ++d) *reinterpret_cast<uint16_t *>(static_cast<char *>(a.dst[d]) + base + 2 * u) = x;
    }
}

// ---------------------------------------------------------------- TMA path

#ifndef FSDP_GATHER_TILE
#define FSDP_GATHER_TILE 16384
#endif
#ifndef FSDP_GATHER_STAGES
#define FSDP_GATHER_STAGES 4
#endif
// Grid: up to FSDP_GATHER_GRID_MULT resident waves of CTAs (one tile per CTA
// for units up to ~1.9 GB of output dtype). Measured on the 70B unit, 2.21 ms
// per 8-way gather against 2.54 ms with a single persistent wave striding
// over all tiles.
#ifndef FSDP_GATHER_GRID_MULT
#define FSDP_GATHER_GRID_MULT 256
#endif
constexpr int kTile = FSDP_GATHER_TILE;      // bytes per bulk tile (multiple of 16)
constexpr int kStages = FSDP_GATHER_STAGES;  // tiles in flight per CTA
constexpr int kTmaThreads = 32;
constexpr int64_t kTmaMinBytes = 1 << 20;
constexpr long long kWaitLimitCycles = 1ll << 31;  // ~1 s at 2 GHz

// Bounded mbarrier waits that gave up (a kernel then returns early), over
// every call on this device since the last fsdp_take_wait_timeouts.
__device__ uint32_t g_gather_wait_timeouts;

// A bounded wait gave up: count it on the device and, when the caller asked
// for it, in the call's own counter.
__device__ __forceinline__ void count_timeout(uint32_t *per_call) {
    atomicAdd(&g_gather_wait_timeouts, 1u);
    if (per_call != nullptr) atomicAdd(per_call, 1u);
}

template <int ND>
__global__ void __launch_bounds__(kTmaThreads)
    gather_tma_kernel(const __grid_constant__ GatherArgs a, int64_t bulk_bytes) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar[kStages];
    const char *src = static_cast<const char *>(a.src);
    // bytes after the bulk part (< 16, a multiple of 2): lanes of CTA 0
    if (blockIdx.x == 0) {
        const int64_t tail_units = (a.nbytes - bulk_bytes) / 2;
        for (int64_t u = threadIdx.x; u < tail_units; u += blockDim.x) {
            const uint16_t x = *reinterpret_cast<const uint16_t *>(src + bulk_bytes + 2 * u);
            for (int d = 0; d < a.n_dst; ++d)
                *reinterpret_cast<uint16_t *>(static_cast<char *>(a.dst[d]) + bulk_bytes + 2 * u) = x;
        }
    }
    if (threadIdx.x != 0) return;
    const int n = ND > 0 ? ND : a.n_dst;
    const int64_t ntiles = (bulk_bytes + kTile - 1) / kTile;
    const int64_t first = blockIdx.x, step = gridDim.x;  // tiles first, first + step, ...
    const int64_t mine = ntiles > first ? (ntiles - first + step - 1) / step : 0;
    if (mine == 0) return;
#pragma unroll
    for (int s = 0; s < kStages; ++s) tma::mbar_init(&bar[s], 1);
    tma::fence_mbar_init();

    auto tile_bytes = [&](int64_t t) -> uint32_t {
        const int64_t left = bulk_bytes - t * kTile;
        return static_cast<uint32_t>(left < kTile ? left : kTile);
    };
    auto load = [&](int64_t it) {
        const int s = static_cast<int>(it % kStages);
        const int64_t t = first + it * step;
        const uint32_t bytes = tile_bytes(t);
        tma::mbar_arrive_expect_tx(&bar[s], bytes);
        tma::bulk_load(smem + s * kTile, src + t * kTile, bytes, &bar[s]);
    };

    int64_t issued = 0;  // loads issued: iterations [0, issued)
    for (; issued < mine && issued < kStages; ++issued) load(issued);
    uint32_t parity = 0;  // bit s: parity of stage s's next phase
    for (int64_t it = 0; it < mine; ++it) {
        const int s = static_cast<int>(it % kStages);
        if (!tma::mbar_wait_bounded(&bar[s], (parity >> s) & 1u, kWaitLimitCycles)) {
            count_timeout(a.timeouts);
            // The loads of iterations [it, issued) may still be writing this
            // CTA's shared memory: give each one more bounded wait (iteration
            // j completes phase j / kStages of its stage) so that a copy that
            // is only slow lands before the CTA exits, then drain the stores.
            for (int64_t j = it; j < issued; ++j)
                (void)tma::mbar_wait_bounded(&bar[j % kStages], static_cast<uint32_t>((j / kStages) & 1),
                                             kWaitLimitCycles);
            tma::bulk_wait<0>();
            return;
        }
        parity ^= 1u << s;
        const int64_t t = first + it * step;
        const uint32_t bytes = tile_bytes(t);
        if constexpr (ND > 0) {
#pragma unroll
            for (int d = 0; d < ND; ++d) tma::bulk_store(static_cast<char *>(a.dst[d]) + t * kTile, smem + s * kTile, bytes);
        } else {
            for (int d = 0; d < n; ++d) tma::bulk_store(static_cast<char *>(a.dst[d]) + t * kTile, smem + s * kTile, bytes);
        }
        tma::bulk_commit();
        // the previous tile's stores have read their stage once at most one
        // group (this tile's) still reads shared memory; refill that stage
        if (it >= 1 && it - 1 + kStages < mine) {
            tma::bulk_wait_read<1>();
            load(it - 1 + kStages);
            issued = it + kStages;
        }
    }
    tma::bulk_wait<0>();
}

// The batched all-gather (group.cuh): one CTA per 16 KB tile of one unit,
// the unit found by a binary search over the units' first tiles. Thread 0
// bulk-loads the tile into shared memory and bulk-stores it to each of the
// unit's destinations, as one CTA of gather_tma_kernel does for its tile;
// the unit's first CTA also copies the bytes after its last whole 16-byte
// word (2-byte units).
__global__ void __launch_bounds__(kTmaThreads) gather_group_kernel(const __grid_constant__ GatherGroupArgs g) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    const int64_t b = blockIdx.x;
    int lo = 0, hi = g.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g.u[mid].tile_begin <= b) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    const GatherGroupUnit &U = g.u[lo];
    const int64_t t = b - U.tile_begin;
    const int64_t bulk = U.nbytes / 16 * 16;
    const char *src = static_cast<const char *>(U.src);
    if (t == 0) {
        const int64_t tail_units = (U.nbytes - bulk) / 2;
        for (int64_t k = threadIdx.x; k < tail_units; k += blockDim.x) {
            const uint16_t x = *reinterpret_cast<const uint16_t *>(src + bulk + 2 * k);
            for (int d = 0; d < U.n_dst; ++d)
                *reinterpret_cast<uint16_t *>(static_cast<char *>(U.dst[d]) + bulk + 2 * k) = x;
        }
    }
    if (threadIdx.x != 0) return;
    const int64_t off = t * kGroupGatherTile;
    if (off >= bulk) return;
    const int64_t left = bulk - off;
    const uint32_t bytes = static_cast<uint32_t>(left < kGroupGatherTile ? left : kGroupGatherTile);
    tma::mbar_init(&bar, 1);
    tma::fence_mbar_init();
    tma::mbar_arrive_expect_tx(&bar, bytes);
    tma::bulk_load(smem, src + off, bytes, &bar);
    if (!tma::mbar_wait_bounded(&bar, 0, kWaitLimitCycles)) {
        count_timeout(g.timeouts);
        // one more bounded wait, so that a load that is only slow lands in
        // shared memory before the CTA exits
        (void)tma::mbar_wait_bounded(&bar, 0, kWaitLimitCycles);
        tma::bulk_wait<0>();
        return;
    }
    for (int d = 0; d < U.n_dst; ++d) tma::bulk_store(static_cast<char *>(U.dst[d]) + off, smem, bytes);
    tma::bulk_commit();
    tma::bulk_wait<0>();
}

// A bounded wait on a barrier that nothing completes (two arrivals expected,
// one made): it gives up after `limit` cycles and is counted like a gather's,
// on the device and in the call's counter. The failure path of the bounded
// waits, exercised without a fault.
__global__ void __launch_bounds__(32) stalled_wait_kernel(long long limit, uint32_t *per_call) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    tma::mbar_init(&bar, 2);
    tma::fence_mbar_init();
    tma::mbar_arrive(&bar);
    if (!tma::mbar_wait_bounded(&bar, 0, limit)) count_timeout(per_call);
}

template <int ND>
fsdp_status launch_tma(const GatherArgs &a, cudaStream_t stream) {
    static std::atomic<int> occupancy{0};
    static PerDeviceOnce configured;  // the opt-in is a per-device function attribute
    const int smem = kStages * kTile;
    const int dev = current_device();
    if (!configured.is_done(dev)) {
        cudaError_t e = cudaFuncSetAttribute(gather_tma_kernel<ND>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_status(e);
        configured.mark(dev);
    }
    int blocks_per_sm = 1;
    const fsdp_status so = cached_occupancy(occupancy, gather_tma_kernel<ND>, kTmaThreads, smem, &blocks_per_sm);
    if (so != FSDP_OK) return so;
    const int64_t bulk = a.nbytes / 16 * 16;
    const int64_t ntiles = (bulk + kTile - 1) / kTile;
    const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm * FSDP_GATHER_GRID_MULT;
    const int grid = static_cast<int>(ntiles < cap ? (ntiles > 0 ? ntiles : 1) : cap);
    gather_tma_kernel<ND><<<grid, kTmaThreads, smem, stream>>>(a, bulk);
    return check_launch();
}

// ---------------------------------------------------------------- vector path

template <int ND>
fsdp_status launch_nd(const GatherArgs &a, cudaStream_t stream) {
    static std::atomic<int> occupancy{0};
    int blocks_per_sm = 1;
    const fsdp_status so = cached_occupancy(occupancy, gather_kernel<ND>, kThreads, 0, &blocks_per_sm);
    if (so != FSDP_OK) return so;
    bool vec = aligned(a.src, 16);
    for (int d = 0; d < a.n_dst; ++d) vec = vec && aligned(a.dst[d], 16);
    if (vec && a.nbytes >= kTmaMinBytes) return launch_tma<ND>(a, stream);
    const int64_t nvec = vec ? a.nbytes / 16 : 0;
    const int64_t tail_units = (a.nbytes - 16 * nvec) / 2;
    const int64_t items = nvec + tail_units;
    const int64_t need = (items + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
    const int grid = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
    gather_kernel<ND><<<grid, kThreads, 0, stream>>>(a, nvec, tail_units);
    return check_launch();
}

}  // namespace

uint32_t take_gather_wait_timeouts() {
    uint32_t n = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&n, g_gather_wait_timeouts, sizeof(n)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_gather_wait_timeouts, &zero, sizeof(zero));
    return n;
}

int64_t group_gather_tiles(int64_t nbytes) {
    const int64_t n = (nbytes / 16 * 16 + kGroupGatherTile - 1) / kGroupGatherTile;
    return n > 0 ? n : 1;
}

fsdp_status launch_gather_group(const GatherGroupArgs &g, int64_t grid, cudaStream_t stream) {
    if (g.n < 1 || g.n > kGroupMax || grid < 1 || grid > 0x7fffffff) return FSDP_ERR_INVALID_ARG;
    gather_group_kernel<<<static_cast<unsigned>(grid), kTmaThreads, kGroupGatherTile, stream>>>(g);
    return check_launch();
}

fsdp_status launch_stalled_wait(long long limit_cycles, uint32_t *per_call, cudaStream_t stream) {
    stalled_wait_kernel<<<1, 32, 0, stream>>>(limit_cycles, per_call);
    return check_launch();
}

fsdp_status launch_gather(const GatherArgs &a, cudaStream_t stream) {
    switch (a.n_dst) {
        case 1: return launch_nd<1>(a, stream);
        case 2: return launch_nd<2>(a, stream);
        case 4: return launch_nd<4>(a, stream);
        case 8: return launch_nd<8>(a, stream);
        default: return launch_nd<0>(a, stream);
    }
}

}  // namespace fsdp
