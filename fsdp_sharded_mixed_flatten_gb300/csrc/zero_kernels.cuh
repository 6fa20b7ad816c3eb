// Kernel argument blocks and launcher declarations shared between the host
// API (zero_api.cu) and the kernel translation units.  Arguments travel by
// value in the launch (__grid_constant__), so the library needs no device
// allocation for its pointer tables.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "zero_common.cuh"

namespace zf {

constexpr int kMaxRanks = 512;        // must equal ZERO_MAX_RANKS
constexpr int kFlattenBatch = 64;     // tensors per flatten / unflatten launch

// Fused step and reduce-scatter.  `accum` doubles as the fp32 gradient-shard
// output of the reduce-scatter kernel.
template <int MAXR>
struct StepArgs {
    const uint16_t* grads[MAXR];
    float* master[MAXR];
    float* m[MAXR];
    float* v[MAXR];
    float* accum[MAXR];
    uint16_t* out[MAXR];
    int64_t S;
    int64_t P_pad;
    int32_t n_ranks;
    int32_t n_out;
    int32_t tiles_per_rank;
    float n_ranks_f;
    float inv_n;          // 1 / n_ranks (exact when n_ranks is a power of two)
    int32_t n_pow2;       // n_ranks is a power of two
    AdamConsts k;
};

// Unfused AdamW on the shards and all-gather of bf16 shards.
template <int MAXR>
struct ShardArgs {
    const float* grad_shards[MAXR];
    const uint16_t* param_shards_in[MAXR];
    float* master[MAXR];
    float* m[MAXR];
    float* v[MAXR];
    uint16_t* param_shards[MAXR];
    uint16_t* out[MAXR];
    int64_t S;
    int32_t n_ranks;
    int32_t n_out;
    int32_t tiles_per_rank;
    AdamConsts k;
};

// Flatten / unflatten of up to kFlattenBatch tensors covering the flat range
// [begin, end).  Tensor t occupies [off[t], off[t] + num[t]).
struct FlatArgs {
    const void* tensors[kFlattenBatch];
    int64_t off[kFlattenBatch];
    int64_t num[kFlattenBatch];
    void* flat[kMaxRanks];     // one flat buffer, or n_ranks shards
    int64_t begin;
    int64_t end;
    int64_t S;
    int32_t n_tensors;         // 0: zero-fill (the tail padding)
    int32_t split;             // flat[] holds n_ranks shards of S elements
};

// Bulk-copy staged kernels: argument block covering up to kMaxUnits units
// (FlatParameters) whose per-rank pointers live in one flat table.
constexpr int kStagedTile = 4096;   // shard elements per tile (512 consumers x 8)
constexpr int kMaxUnits = 64;
constexpr int kMaxPtrs = 3392;

struct UnitDesc {
    int64_t S;
    int64_t P_pad;
    int64_t P_valid;          // elements the buffers hold: P_pad, or numel when unpadded
    int32_t n_ranks;
    int32_t n_out;
    int32_t tile_begin;       // first tile of this unit in the launch's tile sequence
    int32_t tiles_per_rank;   // ceil(S / kStagedTile)
    int32_t off_grads;        // ptrs[off_grads + k]: rank k's bf16 gradient buffer
    int32_t off_master;       // ptrs[off_master + r] (and off_m, off_v): fp32 state shards
    int32_t off_m;
    int32_t off_v;
    int32_t off_accum;        // fp32 accumulator / gradient-shard output
    int32_t off_out;          // ptrs[off_out + o]: bf16 gathered parameters
    float n_ranks_f;
    float inv_n;
    int32_t n_pow2;
    int32_t tail_group;       // fused step with S mod kStagedTile in [1, kTailGroupMax]: every
                              // rank's last piece in one tile (the unit's last)
};
constexpr int kTailGroupMax = 8;   // elements per rank in a tail group (one thread's group)

// Launch-wide fields of a staged launch.
struct MultiHeader {
    int32_t n_units;
    int32_t total_tiles;
    int32_t grid;           // CTAs to launch; 0: the persistent grid for the kernel form
    int32_t sched_slot;     // dynamic tile scheduling slot (sched_slot), -1: fixed order
    AdamConsts k;
    // global gradient-norm clipping
    double* partials;       // per-CTA sums of squares of the averaged gradient
    int32_t partial_base;   // first slot a norm launch writes (one slot per CTA)
    int32_t n_partials;     // slots an update launch reduces (fixed order)
    double max_norm;        // clip threshold
    float* norm_out;        // optional: total norm written by CTA 0 of an update launch
};

// Argument block of one staged launch, in two capacities: the launch copies
// the whole block, so small launches use a small one (each launch pays for
// its argument bytes).
template <int UNITS, int PTRS>
struct MultiArgsT {
    static constexpr int kUnits = UNITS;
    static constexpr int kPtrs = PTRS;
    MultiHeader h;
    UnitDesc unit[UNITS];
    const void* ptrs[PTRS];
};
using MultiArgsS = MultiArgsT<4, 384>;
using MultiArgs = MultiArgsT<kMaxUnits, kMaxPtrs>;   // the host builds this one

static_assert(sizeof(MultiArgs) <= 32764, "launch argument block limit");

enum StepMode : int {
    kModePlain = 0,       // fused step from the gradients
    kModeAccumFinal = 1,  // fused last micro-step: g = (accum + mean) / K
    kModeRsStore = 2,     // reduce-scatter: accum = mean
    kModeRsAdd = 3,       // reduce-scatter: accum += mean
    kModeRsNorm = 4,      // clipping pass 1: accum = mean, per-CTA sum of mean^2
    kModeRsAvgNorm = 5,   // clipping pass 1, last micro-step: accum = (accum + mean) / K, sum
    kModeFromShard = 6,   // clipping pass 2: AdamW from accum * clip coefficient
    kModeMeanDiv = 7      // ZeRO-1 last step: fp32 full accumulators, g = mean / K
};

// Device-side status codes (g_zf_device_status); must match ZERO_DEVICE_*.
constexpr int kDeviceOk = 0;
constexpr int kDeviceTimeout = 1;
constexpr int kDeviceSchedConflict = 2;

// Launchers (return the launch status; grid sizes are chosen inside).
template <int MAXR>
cudaError_t launch_fused_step(const StepArgs<MAXR>& a, int mode, cudaStream_t stream);
template <int MAXR>
cudaError_t launch_reduce_scatter(const StepArgs<MAXR>& a, int accumulate, cudaStream_t stream);
template <int MAXR>
cudaError_t launch_adamw_shards(const ShardArgs<MAXR>& a, cudaStream_t stream);
template <int MAXR>
cudaError_t launch_all_gather(const ShardArgs<MAXR>& a, cudaStream_t stream);
cudaError_t launch_flatten(const FlatArgs& a, int elem_bytes, int unflatten, cudaStream_t stream);
// Bulk-copy staged fused step / reduce-scatter over the units of `a` (mode:
// StepMode); `n_ptrs` pointers of a.ptrs are in use (picks the block size).
// Sets a.h.sched_slot (the tile order) for the launch.
cudaError_t launch_staged_step(MultiArgs& a, int n_ptrs, int mode, cudaStream_t stream);
// The same, reading fp32 gradient buffers (ZeRO-1 full accumulators; mode
// kModeMeanDiv only).
cudaError_t launch_staged_step_f32(MultiArgs& a, int n_ptrs, cudaStream_t stream);
// ZeRO-1 local accumulation of each rank's bf16 gradient into its full fp32
// accumulator (a.grads -> a.accum, P_pad elements each).
template <int MAXR>
cudaError_t launch_zero1_accumulate(const StepArgs<MAXR>& a, int first, cudaStream_t stream);
// The same through the bulk-copy pipeline (the default; the register kernel
// above runs under ZERO_STEP_KERNEL=direct).
template <int MAXR>
cudaError_t launch_zero1_accumulate_staged(const StepArgs<MAXR>& a, int first, cudaStream_t stream);
// Persistent grid for a staged launch over `total_tiles` tiles (at most one
// CTA per SM).  A norm launch is given this many CTAs explicitly (h.grid) and
// writes exactly this many partial sums.
int staged_grid(int mode, int total_tiles);
// Dynamic tile-scheduling slot for a staged launch on `stream` (-1: the fixed
// tile order).
int sched_slot(cudaStream_t stream);
// One CTA waiting on a barrier that nothing completes (tests the bounded wait).
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);
// Read (and optionally clear) the device status word; synchronises `stream`.
cudaError_t read_device_status(int* status, int clear, cudaStream_t stream);

// Persistent grid size: resident CTAs per SM x SMs on the current device,
// capped by the work available.
int persistent_grid(const void* kernel, int threads, size_t smem, int64_t work_ctas);

}  // namespace zf
