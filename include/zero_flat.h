/*
 * zero_flat.h -- C ABI of the GB300 (sm_103a) ZeRO / FSDP sharded
 * mixed-precision step over a FlatParameter.
 *
 * The method (sources by page title and section):
 *   [L5] "Lesson 5: ZeRO and FSDP (including the FSDP2 architecture)",
 *        hpc.payai.win: section 2 (what ZeRO-1/2/3 shard), section 3 (one
 *        optimizer step = reduce-scatter of the gradients, local update of the
 *        1/N_d fp32 master/m/v shard and in-place cast to BF16, all-gather of
 *        the updated shards), section 7.1 (FlatParameter: a unit's tensors are
 *        flattened into one 1-D buffer, tail-padded to a multiple of the rank
 *        count, split along the data-parallel dimension).
 *   [LA] "FSDP", Latent Atlas (process-cxr.github.io): section 5.1 (every rank
 *        holds an equal contiguous slice of every unit), section 8.2 (bf16
 *        gradients, fp32 master update).
 *   [DZ] "Data parallelism and ZeRO memory sharding", jefxiong.cn: section 3.1
 *        (the synchronised gradient is the mean of the ranks' gradients),
 *        section 4.2 and the appendix simulator (bias-corrected Adam on each
 *        rank's slice, then the slices are concatenated).
 *
 * All N_d logical data-parallel ranks live in ONE GPU's memory as separate
 * buffers, so the "collectives" are HBM-streaming kernels, not network calls.
 *
 * Conventions shared by every entry point
 *   - bf16 values travel as uint16_t bit patterns; fp32 as float.
 *   - Every buffer is owned by the caller.  The library allocates no memory
 *     and keeps no state between calls except one device status word (see
 *     zero_device_status), the 32 KB scratch array of
 *     zero_step_units_clip_noalloc and 16 KB of tile-scheduling counters;
 *     only zero_device_status synchronises a stream.
 *   - Tile scheduling: the fused kernels stream tiles of 4096 elements of one
 *     rank's shard through persistent CTAs, one per SM.  When a launch runs
 *     at least 16 rounds of tiles (and is not a norm pass of the clipped
 *     step), each CTA takes its first tile by its index and then claims tiles
 *     from a counter instead of taking them in a fixed order, so that faster
 *     SMs take more (the SMs' speeds differ by up to 40 % when a tile takes
 *     one pass through the kernel's shared-memory ring).  Results do not
 *     depend on the order, nor on the grid: a shorter launch whose tiles
 *     span several passes (more than 8 ranks) runs as many CTAs as make
 *     every round of tiles full but the last.  Launches made directly use a
 *     counter per (device, stream), and per host thread on the per-thread
 *     default stream (cudaStreamPerThread);
 *     launches captured into a CUDA graph take one of 1023 capture counters
 *     in turn.  Each launch leaves its counter at zero; if two launches ever
 *     claim from one counter at the same time (a stream destroyed while its
 *     last launch runs and its handle reused at once, or more than 1023
 *     captured launches replayed concurrently), their results are wrong and
 *     ZERO_DEVICE_SCHED_CONFLICT is recorded (see zero_device_status).
 *   - Device-side calls are asynchronous on `stream` (a cudaStream_t, or NULL
 *     for the legacy default stream) and return after the launch.  The return
 *     code covers argument checks and launch errors; completion and any later
 *     kernel fault are observed by synchronising the stream.
 *   - Pointer arrays (`const T* const* x`) are HOST arrays of DEVICE pointers;
 *     they are copied into the launch, so they may be freed on return.
 *   - Every device pointer must be 16-byte aligned (ZERO_ERR_MISALIGNED).
 *   - Offsets and sizes are element counts (int64_t).
 *   - Elements [P, P_pad) -- the tail padding -- of the gradients, master, m
 *     and v must be zero on entry; they then stay zero.
 *   - Non-finite gradients propagate through the update: an element whose
 *     gradient is NaN or infinite on some rank averages to NaN (the error term
 *     of the compensated rank sum is inf - inf), and its master, m and v
 *     become NaN.  The clipped step reports a NaN norm then, and its NaN
 *     coefficient makes every gradient NaN; a caller checks the norm to skip
 *     such a step.
 *   - Arguments are checked before anything is queued: after ZERO_ERR_INVALID_ARG,
 *     ZERO_ERR_MISALIGNED or ZERO_ERR_SIZE nothing was launched or copied.  A
 *     call that needs several launches or copies may return ZERO_ERR_CUDA after
 *     queuing some of them.  zero_last_error() gives a message (per calling
 *     thread).
 *   - Failure injection, for tests of callers' error paths: while the
 *     environment variable ZERO_SCHED_SHARED is set (to anything but "0"),
 *     every dynamically scheduled launch claims its tiles from one counter
 *     kept for this purpose, so that launches on two streams at once collide.
 *     While the
 *     environment variable ZERO_INJECT_FAILURE is set, every CUDA call the
 *     library would make whose label contains its value (for example
 *     "clip update pass", "staged launch", "gradient copy to the device") is
 *     skipped and the entry point returns ZERO_ERR_CUDA, exactly as if that
 *     call had failed; the calls before it in the same entry point are queued
 *     as usual.  The variable is read at every call.
 */
#ifndef ZERO_FLAT_H
#define ZERO_FLAT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest supported number of logical ranks N_d and of all-gather outputs. */
#define ZERO_MAX_RANKS 512

enum {
    ZERO_OK = 0,
    ZERO_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad hyper-parameter */
    ZERO_ERR_MISALIGNED = -2,  /* a device pointer is not 16-byte aligned            */
    ZERO_ERR_SIZE = -3,        /* inconsistent layout, too many ranks, overflow       */
    ZERO_ERR_CUDA = -4         /* the CUDA runtime reported an error at launch        */
};

/* FlatParameter layout of one FSDP unit ([L5] section 7.1; [LA] section 5.1),
 * or (flags = ZERO_LAYOUT_UNPADDED, from zero_param_layout) the per-parameter
 * Shard(0) layout of one parameter. */
typedef struct zero_layout {
    int64_t n_tensors;    /* tensors flattened into the unit                   */
    int64_t numel;        /* P: sum of the tensors' element counts             */
    int64_t numel_padded; /* P_pad: P rounded up to a multiple of n_ranks      */
    int64_t shard_numel;  /* S = P_pad / n_ranks; rank r owns [r*S, (r+1)*S)   */
    int32_t n_ranks;      /* N_d logical data-parallel ranks                   */
    int32_t flags;        /* 0, or ZERO_LAYOUT_UNPADDED                        */
} zero_layout_t;

/* No padding exists in memory: gradient and parameter buffers hold numel
 * elements and rank r's state shard holds clamp(numel - r*S, 0, S). */
#define ZERO_LAYOUT_UNPADDED 1

/* AdamW hyper-parameters of one optimizer step ([DZ] section 4.2).  Doubles:
 * the library derives its fp32 kernel constants (bias corrections included)
 * in double precision.  Decoupled weight decay theta *= (1 - lr*wd). */
typedef struct zero_adamw {
    double lr;            /* >= 0                                   */
    double beta1;         /* in [0, 1)                              */
    double beta2;         /* in [0, 1)                              */
    double eps;           /* >= 0                                   */
    double weight_decay;  /* >= 0                                   */
    int64_t step;         /* t >= 1, counts optimizer steps         */
} zero_adamw_t;

/*
 * zero_flat_layout -- host only.  ([L5] section 7.1; [LA] section 5.1)
 * Offsets of the tensors in the flat buffer (prefix sums in the given order,
 * no gaps and no per-tensor alignment), P, the tail padding to a multiple of
 * n_ranks, and the shard size S.
 *   numels[n_tensors]       element count of each tensor (>= 0, sum > 0)
 *   offsets_out[n_tensors]  receives each tensor's first flat index
 *   layout_out              receives the layout
 * Errors: ZERO_ERR_INVALID_ARG (null, n_tensors < 1, n_ranks < 1, a negative
 * count, total 0), ZERO_ERR_SIZE (the total overflows int64).
 */
int zero_flat_layout(const int64_t* numels, int64_t n_tensors, int32_t n_ranks,
                     int64_t* offsets_out, zero_layout_t* layout_out);

/*
 * zero_param_layout -- host only.  FSDP2 per-parameter Shard(0) ([L5] section
 * 7.2: every parameter keeps its shape and is split along dim 0 over the
 * ranks, with no FlatParameter and no padding; [A03] section 4; [LA] section
 * 9.5).  A parameter of dim0 rows of row_numel elements is cut the way a tensor
 * is chunked into n_ranks pieces: S = ceil(dim0 / n_ranks) * row_numel, rank r
 * owns elements [r*S, min((r+1)*S, numel)) -- possibly none.  The layout has
 * flags = ZERO_LAYOUT_UNPADDED and numel_padded = n_ranks * S (a virtual size:
 * nothing of it beyond numel is allocated or touched).  Such layouts are
 * accepted by zero_step, zero_step_units(_clip) and zero_reduce_scatter (the
 * staged kernels); the other device entry points reject them.
 * Errors: ZERO_ERR_INVALID_ARG (non-positive sizes), ZERO_ERR_SIZE (overflow).
 */
int zero_param_layout(int64_t dim0, int64_t row_numel, int32_t n_ranks, zero_layout_t* layout_out);

/* Elements of rank `rank`'s shard under `layout` (S, fewer, or 0 at the end
 * of an unpadded layout). */
int zero_shard_numel(const zero_layout_t* layout, int32_t rank, int64_t* numel_out);

/*
 * zero_shard_segments -- host only.  ([LA] section 5.1: a rank's slice cuts
 * across the unit's tensors.)
 * The pieces of rank `rank`'s shard [r*S, (r+1)*S) in flat order: for piece j,
 * seg_tensor[j] is the tensor index (or -1 for the tail padding) and
 * [seg_begin[j], seg_end[j]) the element range inside that tensor (for the
 * padding: the flat range).  Tensors with zero elements yield no piece.
 *   cap      capacity of the three output arrays
 *   n_seg    receives the number of pieces (also when cap is too small)
 * Errors: ZERO_ERR_INVALID_ARG (null, rank out of range), ZERO_ERR_SIZE
 * (inconsistent layout, or cap < *n_seg: the arrays hold the first cap pieces).
 */
int zero_shard_segments(const zero_layout_t* layout, const int64_t* offsets,
                        const int64_t* numels, int32_t rank, int64_t* seg_tensor,
                        int64_t* seg_begin, int64_t* seg_end, int64_t cap, int64_t* n_seg);

/*
 * zero_flatten -- device.  ([L5] section 7.1: flatten a unit's parameters.)
 * Copies n_tensors device tensors (elem_bytes = 2 for bf16, 4 for fp32) into
 * the flat layout and zero-fills the tail padding [P, P_pad).
 *   src[n_tensors]  device pointers; tensor i has numels[i] elements (a null
 *                   pointer is allowed only for a tensor with 0 elements)
 *   offsets, numels HOST arrays as returned / given to zero_flat_layout
 *   dst             dst_split == 0: dst[0] is one flat buffer of P_pad elements;
 *                   dst_split == 1: dst[r] (r < n_ranks) is rank r's shard of
 *                   S elements (e.g. fp32 master weights per rank)
 * Errors: INVALID_ARG, MISALIGNED (dst only; sources may have any alignment
 * of their element type), SIZE, CUDA.
 */
int zero_flatten(const void* const* src, const int64_t* offsets, const int64_t* numels,
                 int32_t elem_bytes, void* const* dst, int32_t dst_split,
                 const zero_layout_t* layout, void* stream);

/*
 * zero_unflatten -- device.  The inverse view of zero_flatten: copies each
 * tensor's range of the flat buffer (or of the shards) back into dst[i].
 * Same arguments with src/dst roles exchanged; padding is not copied.
 */
int zero_unflatten(const void* const* src, int32_t src_split, const int64_t* offsets,
                   const int64_t* numels, int32_t elem_bytes, void* const* dst,
                   const zero_layout_t* layout, void* stream);

/*
 * zero_reduce_scatter -- device.  ([L5] section 3, step 1; [DZ] section 3.1.)
 * Reduce-scatter by averaging: for every rank r and i < S,
 *   mean = (1/N_d) * sum_{k=0}^{N_d-1} grads[k][r*S + i]
 * summed in rank order 0..N_d-1 with a compensated fp32 sum (error-free
 * two-sum), then
 *   accumulate == 0:  grad_shards[r][i] = mean
 *   accumulate == 1:  grad_shards[r][i] = grad_shards[r][i] + mean   (fp32)
 *   grads[n_ranks]        bf16, each P_pad elements (rank k's full gradient)
 *   grad_shards[n_ranks]  fp32, each S elements
 */
int zero_reduce_scatter(const uint16_t* const* grads, float* const* grad_shards,
                        const zero_layout_t* layout, int32_t accumulate, void* stream);

/*
 * zero_adamw_shard_step -- device.  ([L5] section 3, step 2; [DZ] section 4.2.)
 * Every rank's local AdamW update of its fp32 shard and cast to bf16:
 *   g = grad_shards[r][i] / grad_divisor          (grad_divisor = K averages K
 *                                                  accumulated micro-steps; 1 = none)
 *   m = b1*m + (1-b1)*g;   v = b2*v + (1-b2)*g^2
 *   theta = theta*(1 - lr*wd) - (lr/(1-b1^t)) * m / (sqrt(v)/sqrt(1-b2^t) + eps)
 *   param_shards[r][i] = bf16_rne(theta)
 *   master/m/v[n_ranks]    fp32, each S elements, updated in place
 *   grad_shards[n_ranks]   fp32, each S elements
 *   param_shards[n_ranks]  bf16, each S elements (output)
 */
int zero_adamw_shard_step(float* const* master, float* const* m, float* const* v,
                          const float* const* grad_shards, float grad_divisor,
                          uint16_t* const* param_shards, const zero_layout_t* layout,
                          const zero_adamw_t* hp, void* stream);

/*
 * zero_all_gather -- device.  ([L5] section 3, step 3; [DZ] appendix: the
 * updated slices are concatenated once.)
 *   full_params[o][r*S + i] = param_shards[r][i]   for every o < n_out
 *   param_shards[n_ranks]  bf16, each S elements
 *   full_params[n_out]     bf16, each P_pad elements (1 <= n_out <= ZERO_MAX_RANKS)
 */
int zero_all_gather(const uint16_t* const* param_shards, uint16_t* const* full_params,
                    int32_t n_out, const zero_layout_t* layout, void* stream);

/*
 * zero_step -- device, fused.  The whole step of [L5] section 3 in one pass
 * over HBM: reduce-scatter by averaging, AdamW on each rank's shard, bf16 cast
 * and all-gather; neither the fp32 gradient shard nor the bf16 shard is ever
 * written to memory.  Bit-identical to zero_reduce_scatter +
 * zero_adamw_shard_step + zero_all_gather on the same inputs.
 *
 * Micro-step accumulation ([L5] sections 2 and 3: ZeRO-2 reduce-scatters every
 * micro-batch into a sharded fp32 accumulator):
 *   accum == NULL:  micro_step = n_micro = 1; a plain step.
 *   accum != NULL:  1 <= micro_step <= n_micro;
 *     micro_step <  n_micro: accum[r] = (micro_step == 1 ? 0 : accum[r]) + mean;
 *                            no optimizer update, full_params untouched;
 *     micro_step == n_micro: g = (accum[r] + mean) / n_micro (accum[r] itself is
 *                            not rewritten), then the update as above
 *                            (n_micro == 1: g = mean, accum is not touched).
 *   grads[n_ranks]                 bf16, each P_pad
 *   master/m/v/accum[n_ranks]      fp32, each S
 *   full_params[n_out]             bf16, each P_pad
 *   hp                             read only when the optimizer runs
 */
int zero_step(const uint16_t* const* grads, float* const* master, float* const* m,
              float* const* v, float* const* accum, int32_t micro_step, int32_t n_micro,
              uint16_t* const* full_params, int32_t n_out, const zero_layout_t* layout,
              const zero_adamw_t* hp, void* stream);

/*
 * zero_device_status -- host, synchronous.  Failure detection for the kernels
 * that wait on shared-memory barriers (the bulk-copy staged fused step and
 * reduce-scatter): every such wait gives up after about 2 seconds, records
 * ZERO_DEVICE_TIMEOUT in a device status word, and the kernel returns early
 * (its outputs are then incomplete).  A dynamically scheduled launch that
 * found its tile counter used by another launch at the same time records
 * ZERO_DEVICE_SCHED_CONFLICT (its outputs are wrong; see "Tile scheduling"
 * above).  The first problem recorded stays.  This call synchronises
 * `stream`, stores the word in *status (ZERO_DEVICE_OK when nothing went
 * wrong) and, if clear != 0, resets it.  No counterpart on the pages: it
 * reports a launch that did not complete, instead of letting a wait hang the
 * GPU.
 * Errors: ZERO_ERR_INVALID_ARG (status NULL), ZERO_ERR_CUDA.
 */
enum { ZERO_DEVICE_OK = 0, ZERO_DEVICE_TIMEOUT = 1, ZERO_DEVICE_SCHED_CONFLICT = 2 };
int zero_device_status(void* stream, int32_t* status, int32_t clear);

/*
 * zero_selftest_wait_timeout -- device.  Launches one CTA that waits on a
 * shared-memory barrier nothing ever completes, with the same bounded wait the
 * staged kernels use but a limit of limit_ns nanoseconds (1 .. 1e9).  The wait
 * runs out, ZERO_DEVICE_TIMEOUT is recorded and the kernel returns; the
 * context stays usable.  Exists so that failure detection can be tested
 * without hanging or faulting the GPU.  No counterpart on the pages.
 */
int zero_selftest_wait_timeout(int64_t limit_ns, void* stream);

/*
 * zero_unit_t / zero_step_units -- device, fused, several FlatParameters per
 * launch.  FSDP wraps a model as many units (one per transformer block plus a
 * root unit, [LA] section 9.1; [DZ] section 5.5), each its own FlatParameter
 * with its own layout and buffers.  zero_step_units(units, n) computes exactly
 * what n calls of zero_step (one per unit, same micro_step / n_micro / hp)
 * compute, bit for bit, but packs the units into as few launches as the launch
 * argument block allows (up to 64 units and 3392 pointers per launch), so
 * small units do not each pay a launch, a pipeline fill and a tail.
 * Either every unit has an accumulator or none does.
 */
#define ZERO_UNITS_PER_LAUNCH 64      /* units packed into one launch at most          */
#define ZERO_POINTERS_PER_LAUNCH 3392 /* device pointers per launch: per unit 4*N_d +    */
                                      /* n_out (plain), 5*N_d + n_out (last micro-step), */
                                      /* 2*N_d (accumulation micro-step)                 */
typedef struct zero_unit {
    const zero_layout_t* layout;
    const uint16_t* const* grads;    /* [layout->n_ranks] bf16, each P_pad   */
    float* const* master;            /* [n_ranks] fp32, each S               */
    float* const* m;                 /* [n_ranks]                            */
    float* const* v;                 /* [n_ranks]                            */
    float* const* accum;             /* [n_ranks] or NULL                    */
    uint16_t* const* full_params;    /* [n_out] bf16, each P_pad             */
    int32_t n_out;
    int32_t reserved;
} zero_unit_t;

int zero_step_units(const zero_unit_t* units, int32_t n_units, int32_t micro_step,
                    int32_t n_micro, const zero_adamw_t* hp, void* stream);

/*
 * zero_step_units_clip -- device.  zero_step_units with global gradient-norm
 * clipping ([DZ] section 6: a norm over the whole model needs a reduction
 * across every shard).  Reading: the clip-by-total-L2-norm rule -- over every
 * element of every unit's averaged gradient g (the reduce-scatter mean, or at
 * the last micro-step the accumulated mean / n_micro),
 *   norm = sqrt(sum g^2),  coef = max_norm / (norm + 1e-6),
 *   g <- g * coef (fp32) when coef < 1,
 * then AdamW, bf16 cast and all-gather as in zero_step.
 *   Every unit needs `accum` (fp32, [n_ranks] x S): it receives the averaged,
 *   unclipped gradient of this step (at accumulation micro-steps it is the
 *   usual accumulator, and the call is the same as zero_step_units).
 *   workspace        caller-owned device scratch of at least the size
 *                    zero_clip_workspace_bytes reports, 16-byte aligned; it
 *                    holds per-CTA partial sums between the two passes
 *   norm_out         NULL, or a device float receiving the total norm
 * Two passes over HBM: the first reads the gradients and writes the averaged
 * gradient (2*N_d + 4 bytes per element, +4 at a last micro-step), the second
 * reads it with the state and writes state and parameters (30 bytes).
 * Deterministic: the partial sums are reduced in a fixed order.
 * Errors: as zero_step_units; ZERO_ERR_SIZE if the workspace is too small.
 */
int zero_step_units_clip(const zero_unit_t* units, int32_t n_units, int32_t micro_step,
                         int32_t n_micro, const zero_adamw_t* hp, double max_norm,
                         void* workspace, int64_t workspace_bytes, float* norm_out, void* stream);

/*
 * zero_clip_workspace_bytes -- host.  Workspace size zero_step_units_clip
 * needs for these units on the current device (one double per CTA of each
 * norm launch).
 */
int zero_clip_workspace_bytes(const zero_unit_t* units, int32_t n_units, int32_t n_micro,
                              int64_t* bytes);

/*
 * zero_step_units_host -- device, with host buffers.  zero_step_units for a
 * caller whose gradients arrive in host memory and who wants the gathered
 * parameters back in host memory: the end-to-end form of the step.  On one
 * GPU the host link carries what the pages' interconnect carries, the
 * reduce-scatter's input and the all-gather's output ([L5] section 3: one
 * reduce-scatter in, one all-gather out per step).
 *   host_grads[u][k]  pinned host memory: rank k's gradient of unit u, as
 *                     many bf16 elements as units[u].grads[k] holds
 *                     (numel_padded, or numel for an unpadded layout); copied
 *                     into units[u].grads[k] on h2d_stream
 *   host_params       NULL, or [n_units] pinned host buffers (NULL entries
 *                     allowed): when the optimizer runs (micro_step ==
 *                     n_micro), units[u].full_params[0] is copied into
 *                     host_params[u] on d2h_stream once the step is done
 *   flags             0 or any of ZERO_HOST_GRADS_FREE, ZERO_HOST_SM_COPY
 *                     (ZERO_ERR_INVALID_ARG for other bits).
 *                     ZERO_HOST_GRADS_FREE: by default the copies first
 *                     wait for the work already queued on compute_stream,
 *                     which may still read the device gradient buffers; with
 *                     the flag the caller guarantees those buffers are free
 *                     (for instance it alternates two sets of gradient buffers
 *                     and orders h2d_stream itself), so that the next step's
 *                     copies overlap this step's update; ZERO_HOST_SM_COPY:
 *                     rows in pinned, mapped host memory whose address is a
 *                     multiple of 16 bytes move through the SMs (a copy kernel
 *                     loading and storing through the host memory's device
 *                     mapping, CTAs of 1024 threads on a third of the SMs, on
 *                     h2d_stream and d2h_stream) instead of the copy engines,
 *                     and the step's launches size their grids for the other
 *                     SMs, so that a step runs beside the next step's copy;
 *                     other rows still take the copy engines.  Measured on
 *                     GB300: the same 211 GB/s host-to-device, without the
 *                     copy engines' periodic stalls.  The flags combine.
 * The step itself runs on compute_stream once every copy has landed and once
 * the parameter copies queued on d2h_stream by earlier calls are done (the
 * step overwrites the device parameters they read).  On the copy engines a
 * unit whose rank rows are evenly spaced in both memories moves with one 2D copy
 * when the runtime accepts one (rows of separate allocations may be rejected),
 * otherwise with one copy per rank.  The call returns when everything is
 * queued; synchronize d2h_stream (compute_stream if host_params is NULL)
 * before reading the results.  The library allocates no memory; it creates and
 * releases the events that order the three streams.
 * Errors: as zero_step_units; ZERO_ERR_INVALID_ARG for a NULL host_grads row;
 * ZERO_ERR_CUDA if a copy cannot be queued.
 */
#define ZERO_HOST_GRADS_FREE 1
#define ZERO_HOST_SM_COPY 2
int zero_step_units_host(const zero_unit_t* units, int32_t n_units,
                         const uint16_t* const* const* host_grads, uint16_t* const* host_params,
                         int32_t micro_step, int32_t n_micro, const zero_adamw_t* hp,
                         int32_t flags, void* h2d_stream, void* compute_stream, void* d2h_stream);

/*
 * zero_step_units_clip_noalloc -- device.  The same computation as
 * zero_step_units_clip for callers that cannot allocate device memory for the
 * workspace: a runtime that gives all device memory to its own pool at
 * start-up and allows no allocation on the side, or a deployment whose device
 * memory budget is fixed before the optimizer runs.  This call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine); the partial
 * sums live in a scratch array of ZERO_NOALLOC_CLIP_SLOTS doubles (32 KB) that
 * the library reserves on every GPU that loads it, until the process exits.
 * No counterpart on the pages: this is a deployment variant only.
 *   - The first call on a device sets up the array's device address (looked
 *     up with that device current); make that first call before any stream
 *     capture.  Later calls outside capture look the address up again, so a
 *     cudaDeviceReset between calls is harmless; a call captured after a
 *     reset, with no uncaptured call in between, would use the old address.
 *   - Every call shares the one array.  Each call writes every slot it later
 *     reads, so nothing needs clearing, but calls that overlap on the GPU
 *     (two streams at once) race on it: serialise them.
 *   - At most 256 units per call, and the units may need at most
 *     ZERO_NOALLOC_CLIP_SLOTS partial sums (one per CTA of each norm launch);
 *     larger calls are rejected with ZERO_ERR_SIZE before anything is
 *     launched -- use zero_step_units_clip with a workspace then.
 * Arguments and results otherwise as zero_step_units_clip.
 */
#define ZERO_NOALLOC_CLIP_SLOTS 4096
int zero_step_units_clip_noalloc(const zero_unit_t* units, int32_t n_units, int32_t micro_step,
                                 int32_t n_micro, const zero_adamw_t* hp, double max_norm,
                                 float* norm_out, void* stream);

/*
 * zero1_accumulate / zero1_step -- device.  The ZeRO-1 form of gradient
 * accumulation ([L5] section 3: with ZeRO-1 each rank still holds its full
 * gradient, so it can accumulate the micro-batches locally and reduce-scatter
 * once, at the last one; ZeRO-2 keeps only its shard and must reduce-scatter
 * every micro-batch, which is what zero_step's accumulator does; [L5]
 * section 2: the fp32 accumulator costs +4 Psi per rank under ZeRO-1 and
 * +4 Psi / N_d under ZeRO-2).
 *   zero1_accumulate: for every rank k and e < P_pad,
 *     full_accum[k][e] = (first ? 0 : full_accum[k][e]) + grads[k][e]   (fp32)
 *     grads[n_ranks]       bf16, each P_pad;   full_accum[n_ranks] fp32, each P_pad
 *   zero1_step: after n_micro micro-steps, the single reduce-scatter of the
 *     accumulators by averaging (compensated fp32 sum in rank order), divided
 *     by n_micro, then AdamW, bf16 cast and all-gather exactly as zero_step.
 * Per element and micro-step zero1_accumulate moves 6 (first) or 10 bytes per
 * rank and zero1_step 4*N_d + 26, against 2*N_d + 4..8 and 2*N_d + 30 for the
 * ZeRO-2 form: with every rank in one GPU the communication ZeRO-1 saves is
 * free and its local accumulation costs HBM traffic instead.
 */
int zero1_accumulate(const uint16_t* const* grads, float* const* full_accum, int32_t first,
                     const zero_layout_t* layout, void* stream);
int zero1_step(const float* const* full_accum, int32_t n_micro, float* const* master,
               float* const* m, float* const* v, uint16_t* const* full_params, int32_t n_out,
               const zero_layout_t* layout, const zero_adamw_t* hp, void* stream);

/* Message for the last non-OK return on the calling thread ("" if none). */
const char* zero_last_error(void);

/* ABI version of this header (bumped on any incompatible change). */
int32_t zero_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_FLAT_H */
