// Host side of the C ABI declared in include/zero_flat.h: argument checks,
// FlatParameter and per-parameter layouts, derivation of the fp32 kernel
// constants in double precision, packing of the per-rank pointer tables into
// the launch arguments, dispatch to the kernels, and the stream ordering of
// the host-buffer step.  The library allocates no memory.  Its only state is
// a per-thread error message, per-device caches of kernel attributes and
// occupancy, and (device side) the status word and the scratch array of the
// no-alloc clipped step.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <mutex>
#include <vector>

#include "zero_flat.h"
#include "zero_host.cuh"
#include "zero_kernels.cuh"

#define ZERO_API extern "C" __attribute__((visibility("default")))

static_assert(zf::kMaxRanks == ZERO_MAX_RANKS, "rank limit mismatch");
static_assert(zf::kMaxUnits == ZERO_UNITS_PER_LAUNCH && zf::kMaxPtrs == ZERO_POINTERS_PER_LAUNCH,
              "launch packing limits mismatch");
static_assert(zf::kDeviceOk == ZERO_DEVICE_OK && zf::kDeviceTimeout == ZERO_DEVICE_TIMEOUT &&
                  zf::kDeviceSchedConflict == ZERO_DEVICE_SCHED_CONFLICT,
              "device status codes mismatch");
// One unit always fits a launch: at most 5 pointers per rank (gradients,
// master, m, v, accumulator) plus one per gathered output.
static_assert(5 * ZERO_MAX_RANKS + ZERO_MAX_RANKS <= ZERO_POINTERS_PER_LAUNCH,
              "a unit with the most ranks and outputs must fit one launch");

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return ZERO_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool unpadded(const zero_layout_t* L) { return (L->flags & ZERO_LAYOUT_UNPADDED) != 0; }

int check_layout(const zero_layout_t* L) {
    if (L == nullptr) return fail(ZERO_ERR_INVALID_ARG, "layout is NULL");
    if (L->n_ranks < 1) return fail(ZERO_ERR_INVALID_ARG, "n_ranks = %d < 1", L->n_ranks);
    if (L->n_ranks > ZERO_MAX_RANKS)
        return fail(ZERO_ERR_SIZE, "n_ranks = %d exceeds %d", L->n_ranks, ZERO_MAX_RANKS);
    if (L->numel < 1) return fail(ZERO_ERR_INVALID_ARG, "numel = %lld < 1", (long long)L->numel);
    if (L->n_tensors < 1) return fail(ZERO_ERR_INVALID_ARG, "n_tensors < 1");
    if (L->flags != 0 && L->flags != ZERO_LAYOUT_UNPADDED)
        return fail(ZERO_ERR_INVALID_ARG, "unknown layout flags %d", L->flags);
    if (L->shard_numel < 1 || L->numel_padded / L->n_ranks != L->shard_numel ||
        L->numel_padded % L->n_ranks != 0)
        return fail(ZERO_ERR_SIZE, "numel_padded != n_ranks * shard_numel");
    if (L->numel_padded < L->numel)
        return fail(ZERO_ERR_SIZE, "numel_padded < numel");
    if (!unpadded(L) && L->numel_padded - L->numel >= L->n_ranks)
        return fail(ZERO_ERR_SIZE, "numel_padded is not numel rounded up to a multiple of n_ranks");
    const int64_t tiles = (L->shard_numel + zf::kTile - 1) / zf::kTile;
    if (tiles * L->n_ranks > std::numeric_limits<int32_t>::max())
        return fail(ZERO_ERR_SIZE, "flat buffer too large");
    return ZERO_OK;
}

// Entry points that only handle FlatParameter (padded) layouts.
int check_padded(const zero_layout_t* L, const char* what) {
    if (int rc = check_layout(L)) return rc;
    if (unpadded(L))
        return fail(ZERO_ERR_INVALID_ARG, "%s does not take unpadded per-parameter layouts", what);
    return ZERO_OK;
}

template <typename T>
int check_ptrs(const T* const* ptrs, int n, const char* name, bool allow_null_array = false) {
    if (ptrs == nullptr) {
        if (allow_null_array) return ZERO_OK;
        return fail(ZERO_ERR_INVALID_ARG, "%s is NULL", name);
    }
    for (int i = 0; i < n; ++i) {
        if (ptrs[i] == nullptr) return fail(ZERO_ERR_INVALID_ARG, "%s[%d] is NULL", name, i);
        if (!aligned16(ptrs[i]))
            return fail(ZERO_ERR_MISALIGNED, "%s[%d] is not 16-byte aligned", name, i);
    }
    return ZERO_OK;
}

int check_hp(const zero_adamw_t* hp) {
    if (hp == nullptr) return fail(ZERO_ERR_INVALID_ARG, "hyper-parameters are NULL");
    const double vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : vals)
        if (!std::isfinite(x)) return fail(ZERO_ERR_INVALID_ARG, "non-finite hyper-parameter");
    if (hp->lr < 0 || hp->eps < 0 || hp->weight_decay < 0)
        return fail(ZERO_ERR_INVALID_ARG, "lr, eps and weight_decay must be >= 0");
    if (hp->beta1 < 0 || hp->beta1 >= 1 || hp->beta2 < 0 || hp->beta2 >= 1)
        return fail(ZERO_ERR_INVALID_ARG, "betas must lie in [0, 1)");
    if (hp->step < 1) return fail(ZERO_ERR_INVALID_ARG, "step = %lld < 1", (long long)hp->step);
    return ZERO_OK;
}

// fp32 kernel constants from double-precision hyper-parameters: each derived
// quantity (1 - beta, bias corrections, lr*wd) is formed in double and rounded
// once; the moment coefficients are split into (hi, lo) fp32 pairs.
void split_f32(double x, float& hi, float& lo) {
    hi = static_cast<float>(x);
    lo = static_cast<float>(x - static_cast<double>(hi));
}

zf::AdamConsts derive_consts(const zero_adamw_t* hp, double divisor) {
    zf::AdamConsts k{};
    const double t = static_cast<double>(hp->step);
    const double bc1 = 1.0 - std::pow(hp->beta1, t);
    const double bc2 = 1.0 - std::pow(hp->beta2, t);
    split_f32(hp->beta1, k.beta1, k.beta1_lo);
    split_f32(1.0 - hp->beta1, k.one_minus_beta1, k.one_minus_beta1_lo);
    split_f32(hp->beta2, k.beta2, k.beta2_lo);
    split_f32(1.0 - hp->beta2, k.one_minus_beta2, k.one_minus_beta2_lo);
    k.eps = static_cast<float>(hp->eps);
    k.lr_wd = static_cast<float>(hp->lr * hp->weight_decay);
    k.step_size = static_cast<float>(hp->lr / bc1);
    k.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    k.divisor = static_cast<float>(divisor);
    return k;
}

int cuda_status(cudaError_t e, const char* what) {
    if (e != cudaSuccess)
        return fail(ZERO_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return ok();
}

// Host-side failure injection for tests of the error paths: while the
// environment variable ZERO_INJECT_FAILURE is set, a CUDA call (a launch, a
// copy, a stream ordering) whose label contains its value is not made, and
// the entry point returns ZERO_ERR_CUDA as it would for a failed call.  Read
// at every call.
bool injected(const char* what) {
    const char* v = std::getenv("ZERO_INJECT_FAILURE");
    return v != nullptr && v[0] != '\0' && std::strstr(what, v) != nullptr;
}

// One CUDA call with its status converted, unless a test injects its failure.
template <class F>
int cuda_call(const char* what, F&& call) {
    if (injected(what)) return fail(ZERO_ERR_CUDA, "%s: injected failure", what);
    return cuda_status(call(), what);
}

// Label of a staged launch, by mode.
const char* staged_label(int mode) {
    switch (mode) {
        case zf::kModePlain: return "staged launch: step";
        case zf::kModeAccumFinal: return "staged launch: accumulated step";
        case zf::kModeRsStore: return "staged launch: reduce-scatter";
        case zf::kModeRsAdd: return "staged launch: reduce-scatter add";
        case zf::kModeRsNorm: return "staged launch: clip norm pass";
        case zf::kModeRsAvgNorm: return "staged launch: clip norm pass, last micro-step";
        case zf::kModeFromShard: return "staged launch: clip update pass";
        case zf::kModeMeanDiv: return "staged launch: ZeRO-1 step";
        default: return "staged launch";
    }
}

// Which fused / reduce-scatter kernel runs: the bulk-copy staged one
// (default) or the direct-load one.  ZERO_STEP_KERNEL=direct selects the
// latter (both compute bit-identical results); read at every call.
bool use_staged() {
    const char* v = std::getenv("ZERO_STEP_KERNEL");
    return !(v != nullptr && std::strcmp(v, "direct") == 0);
}

int tiles_per_rank(const zero_layout_t* L) {
    return static_cast<int>((L->shard_numel + zf::kTile - 1) / zf::kTile);
}

template <int MAXR>
void fill_step_args(zf::StepArgs<MAXR>& a, const zero_layout_t* L) {
    a.S = L->shard_numel;
    a.P_pad = L->numel_padded;
    a.n_ranks = L->n_ranks;
    a.n_out = 0;
    a.tiles_per_rank = tiles_per_rank(L);
    a.n_ranks_f = static_cast<float>(L->n_ranks);
    a.inv_n = static_cast<float>(1.0 / static_cast<double>(L->n_ranks));
    a.n_pow2 = (L->n_ranks & (L->n_ranks - 1)) == 0 ? 1 : 0;
}

// Host view of one unit for the staged (multi-unit) launches.
struct UnitView {
    const zero_layout_t* L;
    const uint16_t* const* grads;
    float* const* master;
    float* const* m;
    float* const* v;
    float* const* accum;
    uint16_t* const* out;
    int32_t n_out;
};

bool mode_reads_grads(int mode) { return mode != zf::kModeFromShard; }
bool mode_updates(int mode) {
    return mode == zf::kModePlain || mode == zf::kModeAccumFinal || mode == zf::kModeFromShard ||
           mode == zf::kModeMeanDiv;
}
bool mode_uses_accum(int mode) { return mode != zf::kModePlain && mode != zf::kModeMeanDiv; }

int pointers_needed(const UnitView& u, int mode) {
    const int n = u.L->n_ranks;
    return (mode_reads_grads(mode) ? n : 0) + (mode_updates(mode) ? 3 * n + u.n_out : 0) +
           (mode_uses_accum(mode) ? n : 0);
}

// Global gradient-norm clipping bookkeeping: where the norm launches write
// their per-CTA partial sums and what the update launches reduce.
struct ClipPlan {
    double* partials = nullptr;
    int64_t capacity = 0;     // slots available
    int64_t slots_used = 0;   // written so far by norm launches
    int32_t n_partials = 0;   // slots the update launches reduce
    double max_norm = 0.0;
    float* norm_out = nullptr;
    bool dry_run = false;     // only count slots (no launch)
};

// Pack units into as few staged launches as the argument block allows
// (kMaxUnits units, kMaxPtrs pointers) and launch them in order.
int launch_units_staged(const UnitView* units, int n_units, int mode, const zf::AdamConsts& k,
                        cudaStream_t stream, ClipPlan* clip = nullptr) {
    static thread_local zf::MultiArgs a;
    int np = 0;
    a.h.n_units = 0;
    a.h.total_tiles = 0;
    a.h.grid = 0;
    a.h.sched_slot = -1;
    a.h.k = k;
    auto flush = [&]() -> int {
        if (a.h.n_units == 0) return ZERO_OK;
        int rc = ZERO_OK;
        if (clip != nullptr) {
            a.h.partials = clip->partials;
            a.h.partial_base = static_cast<int32_t>(clip->slots_used);
            a.h.n_partials = clip->n_partials;
            a.h.max_norm = clip->max_norm;
            a.h.norm_out = clip->norm_out;
            if (mode == zf::kModeRsNorm || mode == zf::kModeRsAvgNorm) {
                // The launch runs exactly `grid` CTAs, one partial sum each.
                const int grid = zf::staged_grid(mode, a.h.total_tiles);
                if (clip->slots_used + grid > clip->capacity && !clip->dry_run)
                    return fail(ZERO_ERR_SIZE, "clipping workspace too small: need %lld slots",
                                (long long)(clip->slots_used + grid));
                a.h.grid = grid;
                clip->slots_used += grid;
            }
        } else {
            a.h.partials = nullptr;
            a.h.norm_out = nullptr;
        }
        if (clip == nullptr || !clip->dry_run) {
            rc = cuda_call(staged_label(mode), [&] {
                return mode == zf::kModeMeanDiv ? zf::launch_staged_step_f32(a, np, stream)
                                                : zf::launch_staged_step(a, np, mode, stream);
            });
        }
        a.h.n_units = 0;
        a.h.total_tiles = 0;
        a.h.grid = 0;
        np = 0;
        return rc;
    };
    for (int i = 0; i < n_units; ++i) {
        const UnitView& u = units[i];
        const int n = u.L->n_ranks;
        const int need = pointers_needed(u, mode);
        const int64_t tpr = (u.L->shard_numel + zf::kStagedTile - 1) / zf::kStagedTile;
        // the fused step takes every rank's last piece of at most 8 elements as
        // one tile (the unit's tail group) instead of one tile per rank
        const int64_t tail = u.L->shard_numel % zf::kStagedTile;
        const bool group = mode == zf::kModePlain && tail > 0 && tail <= zf::kTailGroupMax &&
                           n <= zf::kMaxRanks;
        const int64_t tiles = group ? (tpr - 1) * n + 1 : tpr * n;
        if (a.h.n_units == zf::kMaxUnits || np + need > zf::kMaxPtrs ||
            static_cast<int64_t>(a.h.total_tiles) + tiles > std::numeric_limits<int32_t>::max()) {
            if (int rc = flush()) return rc;
        }
        zf::UnitDesc& d = a.unit[a.h.n_units];
        d.S = u.L->shard_numel;
        d.P_pad = u.L->numel_padded;
        d.P_valid = unpadded(u.L) ? u.L->numel : u.L->numel_padded;
        d.n_ranks = n;
        d.n_out = 0;
        d.tile_begin = a.h.total_tiles;
        d.tiles_per_rank = static_cast<int32_t>(tpr);
        d.n_ranks_f = static_cast<float>(n);
        d.inv_n = static_cast<float>(1.0 / static_cast<double>(n));
        d.n_pow2 = (n & (n - 1)) == 0 ? 1 : 0;
        d.tail_group = group ? 1 : 0;
        d.off_grads = d.off_master = d.off_m = d.off_v = d.off_accum = d.off_out = -1;
        if (mode_reads_grads(mode)) {
            d.off_grads = np;
            for (int r = 0; r < n; ++r) a.ptrs[np++] = u.grads[r];
        }
        if (mode_updates(mode)) {
            d.off_master = np;
            for (int r = 0; r < n; ++r) a.ptrs[np++] = u.master[r];
            d.off_m = np;
            for (int r = 0; r < n; ++r) a.ptrs[np++] = u.m[r];
            d.off_v = np;
            for (int r = 0; r < n; ++r) a.ptrs[np++] = u.v[r];
            d.n_out = u.n_out;
            d.off_out = np;
            for (int o = 0; o < u.n_out; ++o) a.ptrs[np++] = u.out[o];
        }
        if (mode_uses_accum(mode)) {
            d.off_accum = np;
            for (int r = 0; r < n; ++r) a.ptrs[np++] = u.accum[r];
        }
        a.h.total_tiles += static_cast<int32_t>(tiles);
        a.h.n_units += 1;
    }
    return flush();
}

// One unit's step with the direct-load kernels.
template <int MAXR>
int run_step_direct(const UnitView& u, int32_t micro_step, int32_t n_micro,
                    const zero_adamw_t* hp, cudaStream_t stream) {
    // Up to 24 KB: kept in per-thread static storage rather than on the stack.
    static thread_local zf::StepArgs<MAXR> args;
    std::memset(&args, 0, sizeof args);
    fill_step_args(args, u.L);
    const int n = u.L->n_ranks;
    for (int k = 0; k < n; ++k) args.grads[k] = u.grads[k];
    const bool micro = u.accum != nullptr && n_micro > 1;
    if (micro && micro_step < n_micro) {
        for (int r = 0; r < n; ++r) args.accum[r] = u.accum[r];
        return cuda_call("reduce-scatter launch", [&] {
            return zf::launch_reduce_scatter<MAXR>(args, micro_step > 1 ? 1 : 0, stream);
        });
    }
    for (int r = 0; r < n; ++r) {
        args.master[r] = u.master[r];
        args.m[r] = u.m[r];
        args.v[r] = u.v[r];
        if (micro) args.accum[r] = u.accum[r];
    }
    for (int o = 0; o < u.n_out; ++o) args.out[o] = u.out[o];
    args.n_out = u.n_out;
    args.k = derive_consts(hp, micro ? static_cast<double>(n_micro) : 1.0);
    return cuda_call("fused step launch", [&] {
        return zf::launch_fused_step<MAXR>(args, micro ? zf::kModeAccumFinal : zf::kModePlain,
                                           stream);
    });
}

// Validate one unit's arguments for zero_step / zero_step_units.
int check_unit(const UnitView& u, int32_t micro_step, int32_t n_micro, bool optimizer_runs) {
    if (int rc = check_layout(u.L)) return rc;
    const int n = u.L->n_ranks;
    if (int rc = check_ptrs(u.grads, n, "grads")) return rc;
    if (u.accum == nullptr) {
        if (micro_step != 1 || n_micro != 1)
            return fail(ZERO_ERR_INVALID_ARG, "micro-stepping needs an accumulator");
    } else {
        if (n_micro < 1 || micro_step < 1 || micro_step > n_micro)
            return fail(ZERO_ERR_INVALID_ARG, "need 1 <= micro_step <= n_micro");
        if (n_micro > 1) {
            if (int rc = check_ptrs(const_cast<const float* const*>(u.accum), n, "accum")) return rc;
        }
    }
    if (optimizer_runs) {
        if (u.n_out < 1 || u.n_out > ZERO_MAX_RANKS)
            return fail(ZERO_ERR_INVALID_ARG, "n_out must lie in [1, %d]", ZERO_MAX_RANKS);
        if (int rc = check_ptrs(const_cast<const float* const*>(u.master), n, "master")) return rc;
        if (int rc = check_ptrs(const_cast<const float* const*>(u.m), n, "m")) return rc;
        if (int rc = check_ptrs(const_cast<const float* const*>(u.v), n, "v")) return rc;
        if (int rc = check_ptrs(const_cast<const uint16_t* const*>(u.out), u.n_out, "full_params"))
            return rc;
    }
    return ZERO_OK;
}

// Every check run_units makes before it launches anything.
int validate_units(const UnitView* units, int n_units, int32_t micro_step, int32_t n_micro,
                   const zero_adamw_t* hp) {
    // Every unit shares micro_step / n_micro; the optimizer runs unless this is
    // an accumulation-only micro-step.
    const bool micro = units[0].accum != nullptr && n_micro > 1;
    const bool optimizer_runs = !(micro && micro_step < n_micro);
    if (optimizer_runs) {
        if (int rc = check_hp(hp)) return rc;
    }
    for (int i = 0; i < n_units; ++i) {
        if ((units[i].accum != nullptr) != (units[0].accum != nullptr))
            return fail(ZERO_ERR_INVALID_ARG, "either every unit has an accumulator or none");
        if (int rc = check_unit(units[i], micro_step, n_micro, optimizer_runs)) return rc;
    }
    if (!use_staged()) {
        for (int i = 0; i < n_units; ++i) {
            if (unpadded(units[i].L))
                return fail(ZERO_ERR_INVALID_ARG,
                            "unpadded per-parameter layouts need the staged kernels "
                            "(ZERO_STEP_KERNEL=direct is set)");
        }
    }
    return ZERO_OK;
}

int run_units(const UnitView* units, int n_units, int32_t micro_step, int32_t n_micro,
              const zero_adamw_t* hp, cudaStream_t stream) {
    if (int rc = validate_units(units, n_units, micro_step, n_micro, hp)) return rc;
    const bool micro = units[0].accum != nullptr && n_micro > 1;
    const bool optimizer_runs = !(micro && micro_step < n_micro);
    if (use_staged()) {
        int mode = zf::kModePlain;
        if (micro) mode = micro_step < n_micro ? (micro_step > 1 ? zf::kModeRsAdd : zf::kModeRsStore)
                                               : zf::kModeAccumFinal;
        zf::AdamConsts k{};
        if (optimizer_runs) k = derive_consts(hp, micro ? static_cast<double>(n_micro) : 1.0);
        return launch_units_staged(units, n_units, mode, k, stream);
    }
    for (int i = 0; i < n_units; ++i) {
        const UnitView& u = units[i];
        const int need = u.L->n_ranks > (optimizer_runs ? u.n_out : 0) ? u.L->n_ranks : u.n_out;
        const int rc = need <= 64 ? run_step_direct<64>(u, micro_step, n_micro, hp, stream)
                                  : run_step_direct<512>(u, micro_step, n_micro, hp, stream);
        if (rc) return rc;
    }
    return ok();
}

}  // namespace

// ------------------------------------------------------------------ API ----

ZERO_API int32_t zero_abi_version(void) { return 1; }

ZERO_API const char* zero_last_error(void) { return g_err; }

ZERO_API int zero_flat_layout(const int64_t* numels, int64_t n_tensors, int32_t n_ranks,
                              int64_t* offsets_out, zero_layout_t* layout_out) {
    if (numels == nullptr || offsets_out == nullptr || layout_out == nullptr)
        return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (n_tensors < 1) return fail(ZERO_ERR_INVALID_ARG, "n_tensors < 1");
    if (n_ranks < 1) return fail(ZERO_ERR_INVALID_ARG, "n_ranks < 1");
    int64_t total = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0) return fail(ZERO_ERR_INVALID_ARG, "numels[%lld] < 0", (long long)i);
        if (total > std::numeric_limits<int64_t>::max() - numels[i])
            return fail(ZERO_ERR_SIZE, "total element count overflows int64");
        offsets_out[i] = total;
        total += numels[i];
    }
    if (total < 1) return fail(ZERO_ERR_INVALID_ARG, "the tensors hold no elements");
    const int64_t shard = total / n_ranks + (total % n_ranks != 0 ? 1 : 0);
    if (shard > std::numeric_limits<int64_t>::max() / n_ranks)
        return fail(ZERO_ERR_SIZE, "padded size overflows int64");
    layout_out->n_tensors = n_tensors;
    layout_out->numel = total;
    layout_out->shard_numel = shard;
    layout_out->numel_padded = shard * n_ranks;
    layout_out->n_ranks = n_ranks;
    layout_out->flags = 0;
    return ok();
}

ZERO_API int zero_shard_segments(const zero_layout_t* L, const int64_t* offsets,
                                 const int64_t* numels, int32_t rank, int64_t* seg_tensor,
                                 int64_t* seg_begin, int64_t* seg_end, int64_t cap,
                                 int64_t* n_seg) {
    if (int rc = check_padded(L, "zero_shard_segments")) return rc;
    if (offsets == nullptr || numels == nullptr || n_seg == nullptr)
        return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (cap > 0 && (seg_tensor == nullptr || seg_begin == nullptr || seg_end == nullptr))
        return fail(ZERO_ERR_INVALID_ARG, "NULL output array");
    if (rank < 0 || rank >= L->n_ranks) return fail(ZERO_ERR_INVALID_ARG, "rank out of range");
    const int64_t lo = static_cast<int64_t>(rank) * L->shard_numel;
    const int64_t hi = lo + L->shard_numel;
    int64_t count = 0;
    int64_t expect = 0;
    for (int64_t t = 0; t < L->n_tensors; ++t) {
        if (offsets[t] != expect || numels[t] < 0)
            return fail(ZERO_ERR_SIZE, "offsets do not match numels");
        expect += numels[t];
        const int64_t b = offsets[t] > lo ? offsets[t] : lo;
        const int64_t e = offsets[t] + numels[t] < hi ? offsets[t] + numels[t] : hi;
        if (b < e) {
            if (count < cap) {
                seg_tensor[count] = t;
                seg_begin[count] = b - offsets[t];
                seg_end[count] = e - offsets[t];
            }
            ++count;
        }
    }
    if (expect != L->numel) return fail(ZERO_ERR_SIZE, "numels do not sum to the layout's numel");
    const int64_t pb = L->numel > lo ? L->numel : lo;
    if (pb < hi) {
        if (count < cap) {
            seg_tensor[count] = -1;
            seg_begin[count] = pb;
            seg_end[count] = hi;
        }
        ++count;
    }
    *n_seg = count;
    if (count > cap) return fail(ZERO_ERR_SIZE, "cap %lld < %lld pieces", (long long)cap,
                                 (long long)count);
    return ok();
}

static int flatten_impl(const void* const* tensors, const int64_t* offsets, const int64_t* numels,
                        int32_t elem_bytes, void* const* flat, int32_t split,
                        const zero_layout_t* L, void* stream, int unflatten) {
    if (int rc = check_padded(L, "zero_flatten / zero_unflatten")) return rc;
    if (tensors == nullptr || offsets == nullptr || numels == nullptr || flat == nullptr)
        return fail(ZERO_ERR_INVALID_ARG, "NULL argument");
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(ZERO_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
    if (split != 0 && split != 1) return fail(ZERO_ERR_INVALID_ARG, "split must be 0 or 1");
    const int n_flat = split ? L->n_ranks : 1;
    if (int rc = check_ptrs(const_cast<const void* const*>(flat), n_flat, "flat buffers")) return rc;
    int64_t expect = 0;
    for (int64_t t = 0; t < L->n_tensors; ++t) {
        if (offsets[t] != expect || numels[t] < 0)
            return fail(ZERO_ERR_SIZE, "offsets do not match numels");
        if (numels[t] > 0) {
            if (tensors[t] == nullptr)
                return fail(ZERO_ERR_INVALID_ARG, "tensor %lld is NULL", (long long)t);
            if ((reinterpret_cast<uintptr_t>(tensors[t]) % elem_bytes) != 0)
                return fail(ZERO_ERR_MISALIGNED, "tensor %lld is not element aligned", (long long)t);
        }
        expect += numels[t];
    }
    if (expect != L->numel) return fail(ZERO_ERR_SIZE, "numels do not sum to the layout's numel");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    static thread_local zf::FlatArgs a;
    std::memset(&a, 0, sizeof a);
    a.S = L->shard_numel;
    a.split = split;
    for (int i = 0; i < n_flat; ++i) a.flat[i] = flat[i];
    for (int64_t t0 = 0; t0 < L->n_tensors; t0 += zf::kFlattenBatch) {
        const int64_t t1 = t0 + zf::kFlattenBatch < L->n_tensors ? t0 + zf::kFlattenBatch
                                                                 : L->n_tensors;
        a.n_tensors = static_cast<int32_t>(t1 - t0);
        for (int64_t t = t0; t < t1; ++t) {
            a.tensors[t - t0] = tensors[t];
            a.off[t - t0] = offsets[t];
            a.num[t - t0] = numels[t];
        }
        a.begin = offsets[t0];
        a.end = offsets[t1 - 1] + numels[t1 - 1];
        if (a.end > a.begin) {
            if (int rc = cuda_call("flatten launch",
                                   [&] { return zf::launch_flatten(a, elem_bytes, unflatten, st); }))
                return rc;
        }
    }
    if (!unflatten && L->numel_padded > L->numel) {
        a.n_tensors = 0;
        a.begin = L->numel;
        a.end = L->numel_padded;
        if (int rc = cuda_call("padding launch",
                               [&] { return zf::launch_flatten(a, elem_bytes, 0, st); }))
            return rc;
    }
    return ok();
}

ZERO_API int zero_flatten(const void* const* src, const int64_t* offsets, const int64_t* numels,
                          int32_t elem_bytes, void* const* dst, int32_t dst_split,
                          const zero_layout_t* L, void* stream) {
    return flatten_impl(src, offsets, numels, elem_bytes, dst, dst_split, L, stream, 0);
}

ZERO_API int zero_unflatten(const void* const* src, int32_t src_split, const int64_t* offsets,
                            const int64_t* numels, int32_t elem_bytes, void* const* dst,
                            const zero_layout_t* L, void* stream) {
    // The per-tensor buffers are the destination here; the flat buffer(s) the source.
    return flatten_impl(const_cast<const void* const*>(dst), offsets, numels, elem_bytes,
                        const_cast<void* const*>(src), src_split, L, stream, 1);
}

template <int MAXR>
static int rs_impl(const uint16_t* const* grads, float* const* grad_shards, const zero_layout_t* L,
                   int32_t accumulate, cudaStream_t st) {
    static thread_local zf::StepArgs<MAXR> a;
    std::memset(&a, 0, sizeof a);
    fill_step_args(a, L);
    for (int k = 0; k < L->n_ranks; ++k) {
        a.grads[k] = grads[k];
        a.accum[k] = grad_shards[k];
    }
    return cuda_call("reduce-scatter launch",
                     [&] { return zf::launch_reduce_scatter<MAXR>(a, accumulate, st); });
}

ZERO_API int zero_reduce_scatter(const uint16_t* const* grads, float* const* grad_shards,
                                 const zero_layout_t* L, int32_t accumulate, void* stream) {
    if (int rc = check_layout(L)) return rc;
    const int n = L->n_ranks;
    if (int rc = check_ptrs(grads, n, "grads")) return rc;
    if (int rc = check_ptrs(const_cast<const float* const*>(grad_shards), n, "grad_shards"))
        return rc;
    if (accumulate != 0 && accumulate != 1)
        return fail(ZERO_ERR_INVALID_ARG, "accumulate must be 0 or 1");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_staged()) {
        const UnitView u{L, grads, nullptr, nullptr, nullptr, grad_shards, nullptr, 0};
        return launch_units_staged(&u, 1, accumulate ? zf::kModeRsAdd : zf::kModeRsStore,
                                   zf::AdamConsts{}, st);
    }
    if (unpadded(L))
        return fail(ZERO_ERR_INVALID_ARG, "unpadded layouts need the staged kernels");
    if (n <= 64) return rs_impl<64>(grads, grad_shards, L, accumulate, st);
    return rs_impl<512>(grads, grad_shards, L, accumulate, st);
}

template <int MAXR>
static int adamw_impl(float* const* master, float* const* m, float* const* v,
                      const float* const* grad_shards, float grad_divisor,
                      uint16_t* const* param_shards, const zero_layout_t* L,
                      const zero_adamw_t* hp, cudaStream_t st) {
    static thread_local zf::ShardArgs<MAXR> a;
    std::memset(&a, 0, sizeof a);
    a.S = L->shard_numel;
    a.n_ranks = L->n_ranks;
    a.tiles_per_rank = tiles_per_rank(L);
    for (int r = 0; r < L->n_ranks; ++r) {
        a.master[r] = master[r];
        a.m[r] = m[r];
        a.v[r] = v[r];
        a.grad_shards[r] = grad_shards[r];
        a.param_shards[r] = param_shards[r];
    }
    a.k = derive_consts(hp, static_cast<double>(grad_divisor));
    return cuda_call("adamw launch", [&] { return zf::launch_adamw_shards<MAXR>(a, st); });
}

ZERO_API int zero_adamw_shard_step(float* const* master, float* const* m, float* const* v,
                                   const float* const* grad_shards, float grad_divisor,
                                   uint16_t* const* param_shards, const zero_layout_t* L,
                                   const zero_adamw_t* hp, void* stream) {
    if (int rc = check_padded(L, "zero_adamw_shard_step")) return rc;
    if (int rc = check_hp(hp)) return rc;
    const int n = L->n_ranks;
    if (int rc = check_ptrs(const_cast<const float* const*>(master), n, "master")) return rc;
    if (int rc = check_ptrs(const_cast<const float* const*>(m), n, "m")) return rc;
    if (int rc = check_ptrs(const_cast<const float* const*>(v), n, "v")) return rc;
    if (int rc = check_ptrs(grad_shards, n, "grad_shards")) return rc;
    if (int rc = check_ptrs(const_cast<const uint16_t* const*>(param_shards), n, "param_shards"))
        return rc;
    if (!(grad_divisor > 0.0f) || !std::isfinite(grad_divisor))
        return fail(ZERO_ERR_INVALID_ARG, "grad_divisor must be a positive finite number");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n <= 64) return adamw_impl<64>(master, m, v, grad_shards, grad_divisor, param_shards, L, hp, st);
    return adamw_impl<512>(master, m, v, grad_shards, grad_divisor, param_shards, L, hp, st);
}

template <int MAXR>
static int gather_impl(const uint16_t* const* param_shards, uint16_t* const* full, int32_t n_out,
                       const zero_layout_t* L, cudaStream_t st) {
    static thread_local zf::ShardArgs<MAXR> a;
    std::memset(&a, 0, sizeof a);
    a.S = L->shard_numel;
    a.n_ranks = L->n_ranks;
    a.n_out = n_out;
    a.tiles_per_rank = tiles_per_rank(L);
    for (int r = 0; r < L->n_ranks; ++r) a.param_shards_in[r] = param_shards[r];
    for (int o = 0; o < n_out; ++o) a.out[o] = full[o];
    return cuda_call("all-gather launch", [&] { return zf::launch_all_gather<MAXR>(a, st); });
}

ZERO_API int zero_all_gather(const uint16_t* const* param_shards, uint16_t* const* full_params,
                             int32_t n_out, const zero_layout_t* L, void* stream) {
    if (int rc = check_padded(L, "zero_all_gather")) return rc;
    if (n_out < 1 || n_out > ZERO_MAX_RANKS)
        return fail(ZERO_ERR_INVALID_ARG, "n_out must lie in [1, %d]", ZERO_MAX_RANKS);
    const int n = L->n_ranks;
    if (int rc = check_ptrs(param_shards, n, "param_shards")) return rc;
    if (int rc = check_ptrs(const_cast<const uint16_t* const*>(full_params), n_out, "full_params"))
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n <= 64 && n_out <= 64) return gather_impl<64>(param_shards, full_params, n_out, L, st);
    return gather_impl<512>(param_shards, full_params, n_out, L, st);
}

ZERO_API int zero_step(const uint16_t* const* grads, float* const* master, float* const* m,
                       float* const* v, float* const* accum, int32_t micro_step, int32_t n_micro,
                       uint16_t* const* full_params, int32_t n_out, const zero_layout_t* L,
                       const zero_adamw_t* hp, void* stream) {
    const UnitView u{L, grads, master, m, v, accum, full_params, n_out};
    return run_units(&u, 1, micro_step, n_micro, hp, static_cast<cudaStream_t>(stream));
}

ZERO_API int zero_step_units(const zero_unit_t* units, int32_t n_units, int32_t micro_step,
                             int32_t n_micro, const zero_adamw_t* hp, void* stream) {
    if (units == nullptr || n_units < 1) return fail(ZERO_ERR_INVALID_ARG, "no units");
    if (n_units > 4096) return fail(ZERO_ERR_SIZE, "at most 4096 units per call");
    static thread_local std::vector<UnitView> views;
    views.resize(static_cast<size_t>(n_units));
    for (int i = 0; i < n_units; ++i) {
        const zero_unit_t& x = units[i];
        views[i] = UnitView{x.layout, x.grads, x.master, x.m, x.v, x.accum, x.full_params, x.n_out};
    }
    return run_units(views.data(), n_units, micro_step, n_micro, hp,
                     static_cast<cudaStream_t>(stream));
}

namespace {

// An event recorded on `from` that `to` waits for; released at once (the
// wait keeps what it needs).
int order_streams(cudaStream_t from, cudaStream_t to, const char* what) {
    if (injected(what)) return fail(ZERO_ERR_CUDA, "%s: injected failure", what);
    cudaEvent_t ev = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev, from);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
    if (ev != nullptr) {
        const cudaError_t d = cudaEventDestroy(ev);
        if (e == cudaSuccess) e = d;
    }
    return cuda_status(e, what);
}

// Rows r = 0..n-1 at base + r * pitch (pitch in bytes, at least `width`)?
template <class T>
bool evenly_spaced(const T* const* rows, int n, int64_t width, int64_t* pitch) {
    if (n < 2) {
        *pitch = width;
        return true;
    }
    const auto b0 = reinterpret_cast<uintptr_t>(rows[0]);
    const auto b1 = reinterpret_cast<uintptr_t>(rows[1]);
    if (b1 <= b0) return false;
    const uintptr_t p = b1 - b0;
    if (p < static_cast<uintptr_t>(width) ||
        p > static_cast<uintptr_t>(std::numeric_limits<int32_t>::max()))
        return false;
    for (int r = 2; r < n; ++r) {
        if (reinterpret_cast<uintptr_t>(rows[r]) != b0 + p * static_cast<uintptr_t>(r)) return false;
    }
    *pitch = static_cast<int64_t>(p);
    return true;
}

// The device address of pinned host memory at p (its device mapping), or
// nullptr when p is not in pinned, mapped host memory.
const void* host_mapping(const void* p) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

// Segments for the SM copy kernel, launched in batches of kHostCopySegs.
struct SmCopies {
    zf::HostCopyArgs a;
    cudaStream_t stream;
    const char* what;

    int add(const void* src, void* dst, int64_t bytes) {
        a.src[a.n] = src;
        a.dst[a.n] = dst;
        a.bytes[a.n] = bytes;
        return ++a.n == zf::kHostCopySegs ? flush() : ZERO_OK;
    }
    int flush() {
        if (a.n == 0) return ZERO_OK;
        const int rc = cuda_call(what, [&] { return zf::launch_host_copy(a, stream); });
        a.n = 0;
        return rc;
    }
};

}  // namespace

ZERO_API int zero_step_units_host(const zero_unit_t* units, int32_t n_units,
                                  const uint16_t* const* const* host_grads,
                                  uint16_t* const* host_params, int32_t micro_step,
                                  int32_t n_micro, const zero_adamw_t* hp, int32_t flags,
                                  void* h2d_stream, void* compute_stream, void* d2h_stream) {
    if (units == nullptr || n_units < 1) return fail(ZERO_ERR_INVALID_ARG, "no units");
    if (n_units > 4096) return fail(ZERO_ERR_SIZE, "at most 4096 units per call");
    if (host_grads == nullptr) return fail(ZERO_ERR_INVALID_ARG, "host_grads is NULL");
    if ((flags & ~(ZERO_HOST_GRADS_FREE | ZERO_HOST_SM_COPY)) != 0)
        return fail(ZERO_ERR_INVALID_ARG, "unknown flags");
    for (int i = 0; i < n_units; ++i) {
        const zero_unit_t& x = units[i];
        if (x.layout == nullptr || x.grads == nullptr || host_grads[i] == nullptr)
            return fail(ZERO_ERR_INVALID_ARG, "unit %d: NULL layout or gradient rows", i);
        if (int rc = check_layout(x.layout)) return rc;
        for (int k = 0; k < x.layout->n_ranks; ++k) {
            if (host_grads[i][k] == nullptr || x.grads[k] == nullptr)
                return fail(ZERO_ERR_INVALID_ARG, "unit %d rank %d: NULL gradient buffer", i, k);
        }
    }
    {
        // every check of the step itself, before any copy is queued
        static thread_local std::vector<UnitView> views;
        views.resize(static_cast<size_t>(n_units));
        for (int i = 0; i < n_units; ++i) {
            const zero_unit_t& x = units[i];
            views[i] = UnitView{x.layout, x.grads, x.master, x.m, x.v, x.accum, x.full_params,
                                x.n_out};
        }
        if (int rc = validate_units(views.data(), n_units, micro_step, n_micro, hp)) return rc;
    }
    const auto h2d = static_cast<cudaStream_t>(h2d_stream);
    const auto comp = static_cast<cudaStream_t>(compute_stream);
    const auto d2h = static_cast<cudaStream_t>(d2h_stream);
    if (!(flags & ZERO_HOST_GRADS_FREE)) {
        if (int rc = order_streams(comp, h2d, "ordering the gradient copies")) return rc;
    }
    const bool sm_copy = (flags & ZERO_HOST_SM_COPY) != 0;
    static thread_local SmCopies sm;
    sm.a.n = 0;
    sm.stream = h2d;
    sm.what = "gradient copy to the device";
    for (int i = 0; i < n_units; ++i) {
        if (injected("gradient copy to the device"))
            return fail(ZERO_ERR_CUDA, "gradient copy to the device: injected failure");
        const zero_unit_t& x = units[i];
        const int n = x.layout->n_ranks;
        const int64_t count = unpadded(x.layout) ? x.layout->numel : x.layout->numel_padded;
        const int64_t width = count * static_cast<int64_t>(sizeof(uint16_t));
        int64_t dpitch = 0, spitch = 0;
        cudaError_t e = cudaSuccess;
        bool done = false;
        if (sm_copy) {
            // rows in pinned, mapped host memory on the 16-byte grid go through
            // the SMs; any other row through a copy engine
            for (int k = 0; k < n && e == cudaSuccess; ++k) {
                const void* src = reinterpret_cast<uintptr_t>(host_grads[i][k]) % 16 == 0
                                      ? host_mapping(host_grads[i][k])
                                      : nullptr;
                if (src != nullptr) {
                    if (int rc = sm.add(src, const_cast<uint16_t*>(x.grads[k]), width)) return rc;
                } else {
                    e = cudaMemcpyAsync(const_cast<uint16_t*>(x.grads[k]), host_grads[i][k],
                                        static_cast<size_t>(width), cudaMemcpyHostToDevice, h2d);
                }
            }
            done = true;
        }
        if (!done && n > 1 && evenly_spaced(x.grads, n, width, &dpitch) &&
            evenly_spaced(host_grads[i], n, width, &spitch)) {
            // Evenly spaced rows need not lie in one allocation (separate
            // buffers can land at a regular stride): the runtime then rejects
            // the 2D copy before queuing anything, and the rows go one by one.
            e = cudaMemcpy2DAsync(const_cast<uint16_t*>(x.grads[0]), static_cast<size_t>(dpitch),
                                  host_grads[i][0], static_cast<size_t>(spitch),
                                  static_cast<size_t>(width), static_cast<size_t>(n),
                                  cudaMemcpyHostToDevice, h2d);
            done = e == cudaSuccess;
            if (e == cudaErrorInvalidValue) {
                (void)cudaGetLastError();
                e = cudaSuccess;
            }
        }
        if (!done) {
            for (int k = 0; k < n && e == cudaSuccess; ++k) {
                e = cudaMemcpyAsync(const_cast<uint16_t*>(x.grads[k]), host_grads[i][k],
                                    static_cast<size_t>(width), cudaMemcpyHostToDevice, h2d);
            }
        }
        if (int rc = cuda_status(e, "gradient copy to the device")) return rc;
    }
    if (int rc = sm.flush()) return rc;
    if (int rc = order_streams(h2d, comp, "ordering the step after the copies")) return rc;
    if (host_params != nullptr) {
        // the step overwrites the device parameters that earlier calls' copies
        // to the host may still be reading
        if (int rc = order_streams(d2h, comp, "ordering the step after earlier parameter copies"))
            return rc;
    }
    {
        // with SM transfers the step leaves their SMs free, so that it runs
        // beside the next step's gradient copy instead of behind it
        struct Reserve {
            explicit Reserve(int n) { zf::set_reserved_sms(n); }
            ~Reserve() { zf::set_reserved_sms(0); }
        } reserve(sm_copy ? zf::host_copy_ctas() : 0);
        if (int rc = zero_step_units(units, n_units, micro_step, n_micro, hp, compute_stream))
            return rc;
    }
    const bool optimizer_runs = units[0].accum == nullptr || n_micro <= 1 || micro_step == n_micro;
    if (host_params != nullptr && optimizer_runs) {
        if (int rc = order_streams(comp, d2h, "ordering the parameter copies")) return rc;
        sm.a.n = 0;
        sm.stream = d2h;
        sm.what = "parameter copy to the host";
        for (int i = 0; i < n_units; ++i) {
            const zero_unit_t& x = units[i];
            if (host_params[i] == nullptr || x.n_out < 1 || x.full_params == nullptr) continue;
            const int64_t count = unpadded(x.layout) ? x.layout->numel : x.layout->numel_padded;
            const int64_t bytes = count * static_cast<int64_t>(sizeof(uint16_t));
            void* dst = sm_copy && reinterpret_cast<uintptr_t>(host_params[i]) % 16 == 0
                            ? const_cast<void*>(host_mapping(host_params[i]))
                            : nullptr;
            if (dst != nullptr) {
                if (int rc = sm.add(x.full_params[0], dst, bytes)) return rc;
                continue;
            }
            if (int rc = cuda_call("parameter copy to the host", [&] {
                    return cudaMemcpyAsync(host_params[i], x.full_params[0],
                                           static_cast<size_t>(bytes), cudaMemcpyDeviceToHost,
                                           d2h);
                }))
                return rc;
        }
        if (int rc = sm.flush()) return rc;
    }
    return ok();
}

ZERO_API int zero_device_status(void* stream, int32_t* status, int32_t clear) {
    if (status == nullptr) return fail(ZERO_ERR_INVALID_ARG, "status is NULL");
    int v = 0;
    if (int rc = cuda_status(zf::read_device_status(&v, clear != 0, static_cast<cudaStream_t>(stream)),
                             "device status read"))
        return rc;
    *status = v;
    return ok();
}

ZERO_API int zero_selftest_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 1000000000) return fail(ZERO_ERR_INVALID_ARG, "limit_ns out of range");
    return cuda_status(zf::launch_wait_timeout_selftest(static_cast<uint64_t>(limit_ns),
                                                        static_cast<cudaStream_t>(stream)),
                       "self-test launch");
}

// ---------------------------------------------------- gradient clipping ----

namespace {

int clip_prepare(const zero_unit_t* units, int32_t n_units, int32_t micro_step, int32_t n_micro,
                 std::vector<UnitView>& views) {
    if (units == nullptr || n_units < 1) return fail(ZERO_ERR_INVALID_ARG, "no units");
    if (n_units > 4096) return fail(ZERO_ERR_SIZE, "at most 4096 units per call");
    views.resize(static_cast<size_t>(n_units));
    for (int i = 0; i < n_units; ++i) {
        const zero_unit_t& x = units[i];
        views[i] = UnitView{x.layout, x.grads, x.master, x.m, x.v, x.accum, x.full_params, x.n_out};
        if (x.accum == nullptr)
            return fail(ZERO_ERR_INVALID_ARG, "clipping needs every unit's accum (gradient shards)");
    }
    if (n_micro < 1 || micro_step < 1 || micro_step > n_micro)
        return fail(ZERO_ERR_INVALID_ARG, "need 1 <= micro_step <= n_micro");
    return ZERO_OK;
}

}  // namespace

ZERO_API int zero_clip_workspace_bytes(const zero_unit_t* units, int32_t n_units, int32_t n_micro,
                                       int64_t* bytes) {
    if (bytes == nullptr) return fail(ZERO_ERR_INVALID_ARG, "bytes is NULL");
    static thread_local std::vector<UnitView> views;
    if (int rc = clip_prepare(units, n_units, n_micro, n_micro, views)) return rc;
    for (const UnitView& u : views) {
        if (int rc = check_layout(u.L)) return rc;
    }
    ClipPlan plan;
    plan.dry_run = true;
    const int mode = n_micro > 1 ? zf::kModeRsAvgNorm : zf::kModeRsNorm;
    if (int rc = launch_units_staged(views.data(), n_units, mode, zf::AdamConsts{}, nullptr, &plan))
        return rc;
    *bytes = plan.slots_used * static_cast<int64_t>(sizeof(double));
    return ok();
}

ZERO_API int zero_step_units_clip(const zero_unit_t* units, int32_t n_units, int32_t micro_step,
                                  int32_t n_micro, const zero_adamw_t* hp, double max_norm,
                                  void* workspace, int64_t workspace_bytes, float* norm_out,
                                  void* stream) {
    static thread_local std::vector<UnitView> views;
    if (int rc = clip_prepare(units, n_units, micro_step, n_micro, views)) return rc;
    const bool accumulating = n_micro > 1 && micro_step < n_micro;
    for (const UnitView& u : views) {
        if (int rc = check_unit(u, micro_step, n_micro, !accumulating)) return rc;
        if (int rc = check_ptrs(const_cast<const float* const*>(u.accum), u.L->n_ranks, "accum"))
            return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (accumulating) {
        return launch_units_staged(views.data(), n_units,
                                   micro_step > 1 ? zf::kModeRsAdd : zf::kModeRsStore,
                                   zf::AdamConsts{}, st);
    }
    if (int rc = check_hp(hp)) return rc;
    if (!(max_norm > 0.0) || !std::isfinite(max_norm))
        return fail(ZERO_ERR_INVALID_ARG, "max_norm must be a positive finite number");
    if (workspace == nullptr) return fail(ZERO_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned16(workspace)) return fail(ZERO_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    if (norm_out != nullptr && (reinterpret_cast<uintptr_t>(norm_out) & 3u) != 0)
        return fail(ZERO_ERR_MISALIGNED, "norm_out is not 4-byte aligned");
    ClipPlan plan;
    plan.partials = static_cast<double*>(workspace);
    plan.capacity = workspace_bytes / static_cast<int64_t>(sizeof(double));
    plan.max_norm = max_norm;
    plan.norm_out = norm_out;
    const zf::AdamConsts k = derive_consts(hp, static_cast<double>(n_micro));
    // Pass 1: averaged gradient into accum, per-CTA sums of its squares.
    const int norm_mode = n_micro > 1 ? zf::kModeRsAvgNorm : zf::kModeRsNorm;
    if (int rc = launch_units_staged(views.data(), n_units, norm_mode, k, st, &plan)) return rc;
    // Pass 2: AdamW from the clipped averaged gradient, bf16 cast, all-gather.
    plan.n_partials = static_cast<int32_t>(plan.slots_used);
    return launch_units_staged(views.data(), n_units, zf::kModeFromShard, k, st, &plan);
}

// ------------------------------------------------ no-allocation variant ----
//
// zero_step_units_clip needs a small device workspace between its two passes.
// Some callers cannot allocate device memory for it: a runtime that hands all
// device memory to its own pool at start-up and lets no library allocate on
// the side, or a deployment whose device-memory budget is fixed before the
// optimizer runs.  zero_step_units_clip_noalloc keeps the partial sums in the
// array below instead, which the module reserves when it is loaded (every GPU
// that loads this library holds it, 32 KB, until the process exits).

static __device__ __align__(256) double g_noalloc_clip_partials[ZERO_NOALLOC_CLIP_SLOTS];

namespace {

constexpr int kNoAllocMaxDevices = 64;
constexpr int kNoAllocMaxUnits = 256;

// Device address of the scratch array for the current device.  Host code may
// not use the array's name as a device address (it is a host-side stand-in),
// so the address is looked up with that device current.  The first call on a
// device sets the address up.  Every later call made outside stream capture
// looks it up again (cheap once the module is loaded), so that a context torn
// down and recreated by cudaDeviceReset is given the new address rather than
// a stale one; a call being captured uses the last address looked up, and a
// capture on a device that has never been set up is refused.
int noalloc_scratch(cudaStream_t stream, double** out) {
    int dev = -1;
    if (int rc = cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return fail(ZERO_ERR_SIZE, "device index %d beyond %d", dev, kNoAllocMaxDevices);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (int rc = cuda_status(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing"))
        return rc;
    static std::mutex mu;
    static double* ptrs[kNoAllocMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        if (int rc = cuda_status(cudaGetSymbolAddress(&p, g_noalloc_clip_partials),
                                 "cudaGetSymbolAddress(clipping scratch)"))
            return rc;
        ptrs[dev] = static_cast<double*>(p);
    } else if (ptrs[dev] == nullptr) {
        return fail(ZERO_ERR_INVALID_ARG,
                    "the first zero_step_units_clip_noalloc call on a device must come before "
                    "any stream capture (it sets up the scratch address)");
    }
    *out = ptrs[dev];
    return ZERO_OK;
}

}  // namespace

ZERO_API int zero_step_units_clip_noalloc(const zero_unit_t* units, int32_t n_units,
                                          int32_t micro_step, int32_t n_micro,
                                          const zero_adamw_t* hp, double max_norm,
                                          float* norm_out, void* stream) {
    if (units == nullptr || n_units < 1) return fail(ZERO_ERR_INVALID_ARG, "no units");
    if (n_units > kNoAllocMaxUnits)
        return fail(ZERO_ERR_SIZE, "at most %d units per call without a workspace",
                    kNoAllocMaxUnits);
    if (n_micro < 1 || micro_step < 1 || micro_step > n_micro)
        return fail(ZERO_ERR_INVALID_ARG, "need 1 <= micro_step <= n_micro");
    UnitView views[kNoAllocMaxUnits];
    const bool accumulating = n_micro > 1 && micro_step < n_micro;
    for (int i = 0; i < n_units; ++i) {
        const zero_unit_t& x = units[i];
        views[i] = UnitView{x.layout, x.grads, x.master, x.m, x.v, x.accum, x.full_params, x.n_out};
        if (x.accum == nullptr)
            return fail(ZERO_ERR_INVALID_ARG, "clipping needs every unit's accum (gradient shards)");
        if (int rc = check_unit(views[i], micro_step, n_micro, !accumulating)) return rc;
        if (int rc = check_ptrs(const_cast<const float* const*>(x.accum), x.layout->n_ranks,
                                "accum"))
            return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (accumulating) {
        return launch_units_staged(views, n_units,
                                   micro_step > 1 ? zf::kModeRsAdd : zf::kModeRsStore,
                                   zf::AdamConsts{}, st);
    }
    if (int rc = check_hp(hp)) return rc;
    if (!(max_norm > 0.0) || !std::isfinite(max_norm))
        return fail(ZERO_ERR_INVALID_ARG, "max_norm must be a positive finite number");
    if (norm_out != nullptr && (reinterpret_cast<uintptr_t>(norm_out) & 3u) != 0)
        return fail(ZERO_ERR_MISALIGNED, "norm_out is not 4-byte aligned");
    const int norm_mode = n_micro > 1 ? zf::kModeRsAvgNorm : zf::kModeRsNorm;
    // Count the partial-sum slots first, so that an oversized call launches nothing.
    ClipPlan count;
    count.dry_run = true;
    if (int rc = launch_units_staged(views, n_units, norm_mode, zf::AdamConsts{}, st, &count))
        return rc;
    if (count.slots_used > ZERO_NOALLOC_CLIP_SLOTS)
        return fail(ZERO_ERR_SIZE,
                    "these units need %lld partial-sum slots; the built-in scratch holds %d "
                    "(use zero_step_units_clip with a workspace)",
                    (long long)count.slots_used, ZERO_NOALLOC_CLIP_SLOTS);
    double* scratch = nullptr;
    if (int rc = noalloc_scratch(st, &scratch)) return rc;
    ClipPlan plan;
    plan.partials = scratch;
    plan.capacity = ZERO_NOALLOC_CLIP_SLOTS;
    plan.max_norm = max_norm;
    plan.norm_out = norm_out;
    const zf::AdamConsts k = derive_consts(hp, static_cast<double>(n_micro));
    // Every partial slot the update pass reads is written by this call's norm
    // pass first, so the scratch needs no clearing.
    if (int rc = launch_units_staged(views, n_units, norm_mode, k, st, &plan)) return rc;
    plan.n_partials = static_cast<int32_t>(plan.slots_used);
    return launch_units_staged(views, n_units, zf::kModeFromShard, k, st, &plan);
}

// ------------------------------------------------ ZeRO-1 accumulation ------

ZERO_API int zero1_accumulate(const uint16_t* const* grads, float* const* full_accum,
                              int32_t first, const zero_layout_t* L, void* stream) {
    if (int rc = check_padded(L, "zero1_accumulate")) return rc;
    const int n = L->n_ranks;
    if (int rc = check_ptrs(grads, n, "grads")) return rc;
    if (int rc = check_ptrs(const_cast<const float* const*>(full_accum), n, "full_accum"))
        return rc;
    if (first != 0 && first != 1) return fail(ZERO_ERR_INVALID_ARG, "first must be 0 or 1");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto go = [&](auto& a) -> int {
        std::memset(&a, 0, sizeof a);
        fill_step_args(a, L);
        for (int k = 0; k < n; ++k) {
            a.grads[k] = grads[k];
            a.accum[k] = full_accum[k];
        }
        return ZERO_OK;
    };
    const bool staged = use_staged();
    if (n <= 64) {
        static thread_local zf::StepArgs<64> a;
        go(a);
        return cuda_call("ZeRO-1 accumulate launch", [&] {
            return staged ? zf::launch_zero1_accumulate_staged<64>(a, first, st)
                          : zf::launch_zero1_accumulate<64>(a, first, st);
        });
    }
    static thread_local zf::StepArgs<512> a;
    go(a);
    return cuda_call("ZeRO-1 accumulate launch", [&] {
        return staged ? zf::launch_zero1_accumulate_staged<512>(a, first, st)
                      : zf::launch_zero1_accumulate<512>(a, first, st);
    });
}

ZERO_API int zero1_step(const float* const* full_accum, int32_t n_micro, float* const* master,
                        float* const* m, float* const* v, uint16_t* const* full_params,
                        int32_t n_out, const zero_layout_t* L, const zero_adamw_t* hp,
                        void* stream) {
    if (int rc = check_padded(L, "zero1_step")) return rc;
    if (int rc = check_hp(hp)) return rc;
    if (n_micro < 1) return fail(ZERO_ERR_INVALID_ARG, "n_micro < 1");
    const int n = L->n_ranks;
    if (int rc = check_ptrs(full_accum, n, "full_accum")) return rc;
    // The staged kernel reads the accumulators through the gradient table.
    const UnitView u{L, reinterpret_cast<const uint16_t* const*>(full_accum), master, m, v,
                     nullptr, full_params, n_out};
    if (int rc = check_unit(u, 1, 1, true)) return rc;
    return launch_units_staged(&u, 1, zf::kModeMeanDiv,
                               derive_consts(hp, static_cast<double>(n_micro)),
                               static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------ per-parameter Shard(0) ----

ZERO_API int zero_param_layout(int64_t dim0, int64_t row_numel, int32_t n_ranks,
                               zero_layout_t* layout_out) {
    if (layout_out == nullptr) return fail(ZERO_ERR_INVALID_ARG, "layout_out is NULL");
    if (dim0 < 1 || row_numel < 1 || n_ranks < 1)
        return fail(ZERO_ERR_INVALID_ARG, "dim0, row_numel and n_ranks must be positive");
    if (dim0 > std::numeric_limits<int64_t>::max() / row_numel)
        return fail(ZERO_ERR_SIZE, "numel overflows int64");
    const int64_t chunk_rows = dim0 / n_ranks + (dim0 % n_ranks != 0 ? 1 : 0);
    if (chunk_rows > std::numeric_limits<int64_t>::max() / row_numel / n_ranks)
        return fail(ZERO_ERR_SIZE, "padded size overflows int64");
    layout_out->n_tensors = 1;
    layout_out->numel = dim0 * row_numel;
    layout_out->shard_numel = chunk_rows * row_numel;
    layout_out->numel_padded = layout_out->shard_numel * n_ranks;
    layout_out->n_ranks = n_ranks;
    layout_out->flags = ZERO_LAYOUT_UNPADDED;
    return ok();
}

ZERO_API int zero_shard_numel(const zero_layout_t* L, int32_t rank, int64_t* numel_out) {
    if (int rc = check_layout(L)) return rc;
    if (numel_out == nullptr) return fail(ZERO_ERR_INVALID_ARG, "numel_out is NULL");
    if (rank < 0 || rank >= L->n_ranks) return fail(ZERO_ERR_INVALID_ARG, "rank out of range");
    int64_t n = L->shard_numel;
    if (unpadded(L)) {
        const int64_t left = L->numel - static_cast<int64_t>(rank) * L->shard_numel;
        n = left < 0 ? 0 : (left < n ? left : n);
    }
    *numel_out = n;
    return ok();
}
