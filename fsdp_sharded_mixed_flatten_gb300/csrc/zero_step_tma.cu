// Bulk-copy (TMA) staged fused step and reduce-scatter, over one or many
// FlatParameters (FSDP units) per launch.
//
// Same arithmetic, element order and results as zero_step.cu (bit-identical);
// what changes is how the bytes reach the SM.  One producer lane per CTA
// streams every byte a tile reads -- the tile's fp32 state (master, m, v,
// accumulator) and, eight ranks per stage, the N_d gradient slices (bf16, or
// fp32 for the ZeRO-1 full accumulators, four per stage) --
// into a ring of shared-memory stages with cp.async.bulk (the Blackwell TMA
// engine: plain global->shared copies whose completion is counted in bytes on
// an mbarrier).  Sixteen consumer warps wait on a stage, read their 8 elements
// per rank from shared memory, release the stage and finally run AdamW and
// write the results.  A tile is 4096 elements of one rank's shard of one unit,
// so every gradient copy is an 8 KB contiguous run of one buffer; the ring of
// 3 x 64 KB stages keeps up to 192 KB in flight per SM independently of the
// consumers' registers, which the direct-load kernel cannot (its in-flight
// bytes are bounded by the loads it holds in registers).  Measured on GB300: with 8
// consumer warps per SM the kernel stayed issue/latency-bound near 70 % of
// the HBM bandwidth; 16 consumer warps reach it.
//
// One launch may cover several units (the tiles of all units form one global
// tile sequence), so small units do not each pay a launch, a pipeline fill
// and a tail.
//
// Copies must start on 16-byte boundaries: a rank's slice of a tile starts at
// flat element r*S + j0, so the copied range is widened down to a multiple of
// 8 elements and consumers realign in registers, exactly like the direct
// kernel.  The last partial 16-byte group of a buffer is never copied; the
// threads that own it read it from global memory.
//
// Every wait is bounded (kWaitLimitNs of wall time on %globaltimer).  A wait
// that runs out records kDeviceTimeout in g_zf_device_status, tells the rest
// of the CTA to stop, and the CTA waits (bounded again) for the copies it
// issued before it returns.
#include <atomic>
#include <cstdlib>
#include <limits>
#include <mutex>
#include <thread>
#include <vector>
#include <type_traits>

#include "zero_kernels.cuh"

namespace zf {

__device__ int g_zf_device_status = 0;

// Dynamic tile scheduling.  The persistent CTAs of a long launch claim tiles
// from one counter instead of striding through them in a fixed order:
// measured on GB300, the SMs of a launch whose tiles take one stage each
// (N_d <= 2, the clipped step's update pass) run at speeds up to 40 % apart,
// and with a fixed order the fast ones sat idle for the last 15 % of the
// launch; launches of multi-stage tiles gained 1-2 % as well.  Every
// element's result is the same whichever CTA computes it.  A slot is
// {next tile, CTAs finished}; the last CTA of a launch to finish puts it back
// to zero, so the slot is ready for the next launch on the same stream (the
// host gives every stream a slot of its own; see sched_slot).
// Slots [0, kStreamSlots): one per (device, stream) for launches made
// directly; [kStreamSlots, kSharedSlot): launches captured into CUDA graphs,
// one each in turn; kSharedSlot: every launch while ZERO_SCHED_SHARED is set
// (failure injection).
constexpr int kStreamSlots = 1024;
constexpr int kSchedSlots = 2048;
constexpr int kSharedSlot = kSchedSlots - 1;
constexpr int kDynamicMinRounds = 16;
__device__ unsigned int g_zf_sched[kSchedSlots][2];

namespace {

constexpr int kConsumerWarps = 16;                     // 512 consumers, 8 elements each
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;           // + 1 producer warp
// Gradient element types the staged kernel reads: bf16 gradients, or the fp32
// full accumulators of the ZeRO-1 variant.  kAlign elements make 16 bytes,
// the granularity of a bulk copy.
template <class GT>
struct GradTraits;
template <>
struct GradTraits<uint16_t> {
    static constexpr int kAlign = 8;
    static constexpr int kRanksPerStage = 8;
    __device__ static float widen(uint16_t x) { return bf16_to_float(x); }
};
template <>
struct GradTraits<float> {
    static constexpr int kAlign = 4;
    static constexpr int kRanksPerStage = 4;
    __device__ static float widen(float x) { return x; }
};
// A rank's copied slice of a tile: the tile widened down to the 16-byte grid.
template <class GT>
constexpr int slice_bytes() {
    return (kStagedTile + GradTraits<GT>::kAlign) * static_cast<int>(sizeof(GT));
}
constexpr int kSliceBytes = slice_bytes<uint16_t>();      // 8208
// The ring: 3 stages of 64 KB.  A tile's first stage holds its fp32 state
// arrays (16 KB each) and, when the whole tile fits, its gradient slices too
// (lead_ranks); every further stage holds the next 8 ranks' bf16 slices (4
// fp32 slices).  At N_d = 2 a tile is one stage (three tiles in flight); at
// N_d = 64 it spans 9.  (A ring of 12 x 16 KB stages was measured: it helped
// N_d = 2 but the 4x more barrier round trips per tile cost 20 % at N_d >= 8.)
constexpr int kStageBytes = 8 * kSliceBytes;               // 65664
constexpr int kStages = 3;
static_assert(GradTraits<uint16_t>::kRanksPerStage * slice_bytes<uint16_t>() <= kStageBytes &&
                  GradTraits<float>::kRanksPerStage * slice_bytes<float>() <= kStageBytes,
              "gradient slices must fit a stage");
constexpr int kStateArrayBytes = kStagedTile * 4;      // 16384
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;       // 0.2 s

static_assert(kConsumers * kVec == kStagedTile, "one thread owns 8 elements of a tile");
static_assert(kConsumers >= kMaxRanks && kTailGroupMax <= kVec && kMaxUnits <= 64,
              "a tail group gives every rank one consumer thread and one group of elements; "
              "a 64-bit mask names a launch's units");
static_assert(4 * kStateArrayBytes <= kStageBytes, "the state arrays must fit one stage");

// Ranks whose gradient slices share the first stage of a tile with its NS
// state arrays.
template <class GT>
__host__ __device__ constexpr int first_stage_ranks(int ns) {
    return (kStageBytes - ns * kStateArrayBytes) / slice_bytes<GT>() <
                   GradTraits<GT>::kRanksPerStage
               ? (kStageBytes - ns * kStateArrayBytes) / slice_bytes<GT>()
               : GradTraits<GT>::kRanksPerStage;
}
static_assert(kSliceBytes % 16 == 0, "bulk copies need 16-byte sizes");

// Gradient ranks carried by a tile's first stage.  Without state arrays the
// first stage is an ordinary gradient stage.  With them, the ranks join the
// state only in a LEAD launch, one whose every unit has few enough ranks that
// the whole tile fits that one stage (N_d <= 2 for the plain step): one
// barrier round trip per tile and up to three tiles in flight.  Otherwise the
// state travels alone.  The choice is a template parameter: measured on
// GB300, deciding it per tile at run time cost 2-3 % at N_d = 8 and splitting
// the ranks unevenly over a tile's stages (2 + 6 at N_d = 8) cost 7 %.
template <int NS, class GT, bool LEAD>
__device__ __forceinline__ int lead_ranks(int n_gr) {
    constexpr int R0 = first_stage_ranks<GT>(NS);
    if constexpr (NS == 0) return n_gr < R0 ? n_gr : R0;
    if constexpr (LEAD) return n_gr;
    return 0;
}

// Modes whose first stage has room for gradient slices next to the state.
template <int NS, class GT>
constexpr bool can_lead() {
    return NS > 0 && first_stage_ranks<GT>(NS) > 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Global -> shared bulk copy completing `bytes` on the mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Bounded wait on one phase of an mbarrier.  Returns false if the CTA has
// been told to stop or the limit ran out (then the CTA is told to stop and
// the device status records the timeout).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicCAS(&g_zf_device_status, kDeviceOk, kDeviceTimeout);
            return false;
        }
    }
}

// Unit of a global tile index: the last unit whose first tile is <= tile.
template <class A>
__device__ __forceinline__ int find_unit(const A& a, int tile) {
    int lo = 0, hi = a.h.n_units - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit[mid].tile_begin <= tile) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

// Geometry of one tile, identical for the producer and the consumers.
struct TileGeom {
    const UnitDesc* u;
    int r;            // rank whose shard the tile covers
    int64_t j0;       // first shard-local element of the tile
    int nvalid;       // valid elements in the tile (<= kStagedTile)
    int64_t e0;       // first flat element
    int mis;          // e0 mod kAlign (8 for bf16, 4 for fp32 gradients)
    int64_t a0;       // aligned start of every rank's copied slice
    int64_t a1;       // end of the copied slice (aligned, never past the last full 16 bytes)
    int state_valid;  // state elements copied (multiple of 4)
    bool group;       // the unit's tail group: every rank's short last piece (tail_group)
};

template <class A, class GT>
__device__ __forceinline__ TileGeom tile_geom(const A& a, int tile) {
    constexpr int64_t AL = GradTraits<GT>::kAlign;
    TileGeom g;
    g.u = &a.unit[find_unit(a, tile)];
    const int local = tile - g.u->tile_begin;
    const int64_t S = g.u->S;
    // A unit's tiles: first every rank's full tiles (rank by rank), then the
    // ranks' short last tiles.  A short tile costs a whole pass through the
    // pipeline, so the short ones go to the end of the unit, where they fill
    // the last round of the persistent CTAs instead of lengthening it.
    const int full = static_cast<int>(S / kStagedTile);
    const int n_full = full * g.u->n_ranks;
    g.group = false;
    if (local >= n_full && g.u->tail_group) {
        // One tile for every rank's last S mod 4096 (<= 8) elements: no stage
        // carries it; consumer thread r computes rank r's piece (tail_group).
        g.group = true;
        g.r = 0;
        g.j0 = static_cast<int64_t>(full) * kStagedTile;
        g.nvalid = g.u->n_ranks;
        g.e0 = g.j0;
        g.mis = 0;
        g.a0 = g.a1 = 0;
        g.state_valid = 0;
        return g;
    }
    if (local < n_full) {
        g.r = local / full;
        g.j0 = static_cast<int64_t>(local - g.r * full) * kStagedTile;
    } else {
        g.r = local - n_full;
        g.j0 = static_cast<int64_t>(full) * kStagedTile;
    }
    g.e0 = static_cast<int64_t>(g.r) * S + g.j0;
    // valid elements: the tile, the rank's shard and the buffers all bound it
    // (an unpadded per-parameter layout ends before its last shards do)
    int64_t rem = S - g.j0;
    if (g.u->P_valid - g.e0 < rem) rem = g.u->P_valid - g.e0;
    g.nvalid = static_cast<int>(rem < kStagedTile ? (rem > 0 ? rem : 0) : kStagedTile);
    g.mis = static_cast<int>(g.e0 & (AL - 1));
    g.a0 = g.e0 - g.mis;
    const int64_t a1 = (g.e0 + g.nvalid + AL - 1) & ~(AL - 1);
    const int64_t floor_al = g.u->P_valid & ~(AL - 1);
    g.a1 = a1 < floor_al ? a1 : floor_al;
    if (g.a1 < g.a0) g.a1 = g.a0;
    g.state_valid = g.nvalid & ~3;
    return g;
}

template <typename T, class A>
__device__ __forceinline__ T ptr_at(const A& a, int index) {
    return static_cast<T>(const_cast<void*>(a.ptrs[index]));
}

template <class GT, class A>
__device__ __forceinline__ const GT* grad_ptr(const A& a, const UnitDesc* u, int k) {
    return ptr_at<const GT*, A>(a, u->off_grads + k);
}

// Per mode: how many fp32 state arrays a tile's state block holds (master,
// m, v, accumulator in that order; the reduce-scatter modes only the
// accumulator), whether the gradients are read, and whether the mode writes
// the averaged gradient to the accumulator (a reduce-scatter) or updates.
template <int MODE>
struct ModeTraits {
    static constexpr bool kReduceScatter =
        MODE == kModeRsStore || MODE == kModeRsAdd || MODE == kModeRsNorm || MODE == kModeRsAvgNorm;
    static constexpr bool kNorm = MODE == kModeRsNorm || MODE == kModeRsAvgNorm;
    static constexpr bool kReadsGrads = MODE != kModeFromShard;
    static constexpr int kStateArrays = (MODE == kModePlain || MODE == kModeMeanDiv) ? 3
                                        : (MODE == kModeAccumFinal || MODE == kModeFromShard) ? 4
                                        : (MODE == kModeRsAdd || MODE == kModeRsAvgNorm) ? 1
                                                                                        : 0;
};

// State array `array` of rank r (order: master, m, v, accumulator; the
// reduce-scatter modes only have the accumulator).
template <int MODE, class A>
__device__ __forceinline__ float* state_ptr(const A& a, const UnitDesc* u, int array,
                                            int r) {
    if constexpr (ModeTraits<MODE>::kReduceScatter) {
        return ptr_at<float*, A>(a, u->off_accum + r);
    } else {
        const int off = array == 0 ? u->off_master
                        : array == 1 ? u->off_m
                        : array == 2 ? u->off_v
                                     : u->off_accum;
        return ptr_at<float*, A>(a, off + r);
    }
}

// Sum up to kRanksPerStage rank slices of one stage into (s, c) for a
// thread's 8 elements starting A elements into its aligned pair of words.
// first: the stage holds the tile's rank 0, whose values start the sums
// (first_rank: the bits a two-sum into (0, 0) leaves, in two packed additions
// instead of seven; measured on GB300 the 7.5B step 1.046 -> 1.055 of the
// copy peak, the clipped GPT-2-small step 0.977 -> 0.988, P = 4M+13 at
// N_d = 64 0.903 -> 0.920).
// fp32 gradient slices: a thread's 8 values start A words into its three
// aligned 16-byte words.
template <int A, int RMAX>
__device__ __forceinline__ void consume_stage_f32(const uint8_t* stage, int nk, int tid,
                                                  float2 (&s)[4], float2 (&c)[4], bool first) {
    constexpr int kSlice = slice_bytes<float>();
    const uint8_t* base = stage + tid * 32;
    auto rank = [&](int kk) {
        const float4* p = reinterpret_cast<const float4*>(base + kk * kSlice);
        const float4 x0 = p[0], x1 = p[1];
        const float4 x2 = (A != 0) ? p[2] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float W[12] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                             x2.x, x2.y, x2.z, x2.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 x = make_float2(W[A + 2 * q], W[A + 2 * q + 1]);
            if (kk == 0 && first) {
                first_rank2(s[q], c[q], x);
            } else {
                two_sum_add2(s[q], c[q], x);
            }
        }
    };
    if (nk == RMAX) {          // a full stage: no bound check per rank (as consume_stage)
#pragma unroll
        for (int kk = 0; kk < RMAX; ++kk) rank(kk);
        return;
    }
#pragma unroll 1
    for (int kk = 0; kk < nk; ++kk) rank(kk);
}

template <int A, int RMAX>
__device__ __forceinline__ void consume_stage(const uint8_t* stage, int nk, int tid,
                                              float2 (&s)[4], float2 (&c)[4], bool first) {
    const uint8_t* base = stage + tid * 16;
    if (nk == RMAX) {
        // A full stage (every stage of a tile but its last, and the last when
        // N_d is a multiple of 8) without a bound check per rank: the loads of
        // all its ranks then issue back to back ahead of the two-sums.
        // Measured on GB300: the 7.5B step 1.003 -> 1.047 of the copy peak, the
        // Llama layer 1.020 -> 1.059, the clipped GPT-2-small step 0.927 -> 0.970.
#pragma unroll
        for (int kk = 0; kk < RMAX; ++kk) {
            const uint4* p = reinterpret_cast<const uint4*>(base + kk * kSliceBytes);
            uint4 x = p[0];
            if constexpr (A != 0) x = align_shift<A>(x, p[1]);
            if (kk == 0 && first) first_rank_bf16x8(s, c, x);
            else two_sum_add_bf16x8(s, c, x);
        }
        return;
    }
    // A partial stage (the last of a tile when N_d is not a multiple of 8):
    // a rolled loop, so that the code of each misalignment stays small.  A
    // short launch whose shards hold fewer tiles than the grid has CTAs
    // that meet a different misalignment at every tile; with this path
    // unrolled too they ran from a twice larger instruction footprint and
    // measured 9 % slower (P = 4,194,317, N_d = 8).
#pragma unroll 1
    for (int kk = 0; kk < nk; ++kk) {
        const uint4* p = reinterpret_cast<const uint4*>(base + kk * kSliceBytes);
        uint4 x = p[0];
        if constexpr (A != 0) x = align_shift<A>(x, p[1]);
        if (kk == 0 && first) first_rank_bf16x8(s, c, x);
        else two_sum_add_bf16x8(s, c, x);
    }
}

// A unit's tail group (fused step only).  When every rank's shard ends in a
// piece of at most 8 elements (S mod 4096 <= 8), those N_d pieces form one
// tile instead of N_d: measured on GB300, each short tile otherwise cost
// nearly a full tile's pass through the pipeline (P = 4M+13 at N_d = 64 ran
// at 0.79 of the copy peak with its 64 one-element tiles and at 0.90 without
// them).  Consumer thread r computes rank r's piece straight from global
// memory: its gradients from every rank -- loaded KB ranks at a time, so that
// the loads are in flight together -- summed in rank order with the same
// two-sums, then the mean, AdamW, the bf16 cast and the gathered writes,
// operation for operation as in the tiles (the scalar forms round exactly as
// the packed ones), so the results are the same bits.
template <int KB, int QMAX, class A>
__device__ __forceinline__ void tail_group_sum(const A& a, const UnitDesc* u, int64_t e, int nv,
                                               float (&sm)[8], float (&cm)[8]) {
    // KB ranks x QMAX elements per batch, every load unconditional (indices
    // clamped into the buffers; what is not needed is not summed), so that a
    // batch's loads are in flight together
    const int n = u->n_ranks;
    for (int k0 = 0; k0 < n; k0 += KB) {
        uint16_t x[KB][QMAX];
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
            const uint16_t* src = grad_ptr<uint16_t, A>(a, u, min(k0 + kk, n - 1)) + e;
#pragma unroll
            for (int q = 0; q < QMAX; ++q) x[kk][q] = src[min(q, nv - 1)];
        }
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
            if (k0 + kk < n) {
#pragma unroll
                for (int q = 0; q < QMAX; ++q) {
                    if (q < nv) two_sum_add1(sm[q], cm[q], bf16_to_float(x[kk][q]));
                }
            }
        }
    }
}

template <class A>
__device__ __forceinline__ void tail_group_step(const A& a, const UnitDesc* u, int tid) {
    const int64_t j0 = (u->S / kStagedTile) * kStagedTile;
    const int r = tid;
    if (r >= u->n_ranks) return;
    const int64_t e = static_cast<int64_t>(r) * u->S + j0;
    int64_t rem = u->S - j0;
    if (u->P_valid - e < rem) rem = u->P_valid - e;
    const int nv = static_cast<int>(rem > 0 ? (rem < kVec ? rem : kVec) : 0);
    if (nv <= 0) return;
    float sm[8], cm[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) sm[q] = cm[q] = 0.0f;
    if (nv == 1) {
        tail_group_sum<16, 1>(a, u, e, nv, sm, cm);
    } else if (nv == 2) {
        tail_group_sum<8, 2>(a, u, e, nv, sm, cm);
    } else if (nv <= 4) {
        tail_group_sum<4, 4>(a, u, e, nv, sm, cm);
    } else {
        tail_group_sum<2, 8>(a, u, e, nv, sm, cm);
    }
    float* master = ptr_at<float*, A>(a, u->off_master + r) + j0;
    float* m = ptr_at<float*, A>(a, u->off_m + r) + j0;
    float* v = ptr_at<float*, A>(a, u->off_v + r) + j0;
    float th[8], mm[8], vv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int qq = min(q, nv - 1);
        th[q] = master[qq];
        mm[q] = m[qq];
        vv[q] = v[qq];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (q < nv) {
            const float g = u->n_pow2 ? __fmul_rn(__fadd_rn(sm[q], cm[q]), u->inv_n)
                                      : finish_mean(sm[q], cm[q], u->n_ranks_f, u->inv_n, false);
            adamw_update(a.h.k, g, th[q], mm[q], vv[q]);
            master[q] = th[q];
            m[q] = mm[q];
            v[q] = vv[q];
            const uint16_t b = float_to_bf16_rn(th[q]);
            for (int o = 0; o < u->n_out; ++o) ptr_at<uint16_t*, A>(a, u->off_out + o)[e + q] = b;
        }
    }
}

template <int MODE, class A, class GT, bool LEAD>
__device__ void producer_loop(const A& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                              volatile int* abort_flag, uint32_t* issued_out,
                              volatile int* tile_of) {
    constexpr int NS = ModeTraits<MODE>::kStateArrays;
    constexpr int RG = GradTraits<GT>::kRanksPerStage;
    const int slot_id = a.h.sched_slot;
    const bool dyn = slot_id >= 0;
    unsigned int* next_tile = dyn ? &g_zf_sched[slot_id][0] : nullptr;
    uint32_t it = 0;
    // Every CTA's first tile is its own index.  After it, in the fixed order,
    // CTA c takes c + G, c + 2G, ...; in the dynamic order it claims the next
    // tile (G + the counter) when its ring has room for it: the ring runs
    // ahead of the consumers, so the claim's round trip overlaps their work,
    // and no CTA holds a tile back while others run dry.
    const int total = a.h.total_tiles;
    const int G = static_cast<int>(gridDim.x);
    auto next_of = [&](int t) -> int {
        return dyn ? G + static_cast<int>(atomicAdd(next_tile, 1u)) : t + G;
    };
    int tile = static_cast<int>(blockIdx.x);
    while (tile < total) {
        const TileGeom g = tile_geom<A, GT>(a, tile);
        if (g.nvalid == 0) {              // past the end of an unpadded parameter
            tile = next_of(tile);
            continue;
        }
        if (g.group) {
            // A tail group reads nothing through the ring.  In the fixed order
            // the consumers find it themselves; in the dynamic order an empty
            // stage names it to them.
            if (dyn) {
                const uint32_t slot = it % kStages, parity = ((it / kStages) & 1) ^ 1;
                if (!mbar_wait_bounded(smem_u32(&empty[slot]), parity, abort_flag, kWaitLimitNs)) {
                    *issued_out = it;
                    return;
                }
                tile_of[slot] = tile;
                mbar_arrive(smem_u32(&full[slot]));
                ++it;
            }
            tile = next_of(tile);
            continue;
        }
        const int n_ranks = ModeTraits<MODE>::kReadsGrads ? g.u->n_ranks : 0;
        const uint32_t sbytes = static_cast<uint32_t>(g.state_valid) * 4;
        const uint32_t gbytes = static_cast<uint32_t>(g.a1 - g.a0) * sizeof(GT);
        // stage 0: state arrays + ranks [0, r0); then RG ranks per stage
        const int r0 = lead_ranks<NS, GT, LEAD>(n_ranks);
        const int n_stages = 1 + (n_ranks - r0 + RG - 1) / RG;
        bool stop = false;
        for (int st = 0; st < n_stages; ++st) {
            const uint32_t slot = it % kStages, parity = ((it / kStages) & 1) ^ 1;
            if (!mbar_wait_bounded(smem_u32(&empty[slot]), parity, abort_flag, kWaitLimitNs)) {
                stop = true;
                break;
            }
            // the consumers learn a dynamically claimed tile from its first
            // stage (published before the arrive, which releases it)
            if (st == 0) tile_of[slot] = tile;
            const int k0 = st == 0 ? 0 : r0 + (st - 1) * RG;
            const int nk = st == 0 ? r0 : min(RG, n_ranks - k0);
            const int ns = st == 0 ? NS : 0;
            const uint32_t bar = smem_u32(&full[slot]);
            mbar_arrive_expect_tx(bar, ns * sbytes + nk * gbytes);
            const uint32_t dst = smem_u32(smem + slot * kStageBytes);
            if (sbytes > 0) {
                for (int arr = 0; arr < ns; ++arr) {
                    bulk_copy_g2s(dst + arr * kStateArrayBytes,
                                  state_ptr<MODE, A>(a, g.u, arr, g.r) + g.j0, sbytes, bar);
                }
            }
            if (gbytes > 0 && nk > 0) {
                // the stage's gradient pointers first, as one batch of loads
                // from the argument block (measured +0.1-0.4 % over loading
                // each just before its copy)
                const uint32_t gdst = dst + ns * kStateArrayBytes;
                const GT* src[RG];
#pragma unroll
                for (int kk = 0; kk < RG; ++kk) {
                    src[kk] = grad_ptr<GT, A>(a, g.u, min(k0 + kk, n_ranks - 1));
                }
#pragma unroll
                for (int kk = 0; kk < RG; ++kk) {
                    if (kk < nk) bulk_copy_g2s(gdst + kk * slice_bytes<GT>(), src[kk] + g.a0, gbytes, bar);
                }
            }
            ++it;
        }
        if (stop || *abort_flag) {
            *issued_out = it;
            return;
        }
        tile = next_of(tile);
    }
    if (dyn) {
        // No tile left: an empty stage whose tile index is -1 tells the
        // consumers to stop.
        const uint32_t slot = it % kStages, parity = ((it / kStages) & 1) ^ 1;
        if (mbar_wait_bounded(smem_u32(&empty[slot]), parity, abort_flag, kWaitLimitNs)) {
            tile_of[slot] = -1;
            mbar_arrive(smem_u32(&full[slot]));
            ++it;
        }
    }
    *issued_out = it;
}

template <int MODE, class A, class GT, bool LEAD, bool ALIGNED>
__device__ void consumer_loop(const A& a, const uint8_t* smem, uint64_t* full,
                              uint64_t* empty, volatile int* abort_flag,
                              unsigned int* consumed_min, float clip_coef, double* warp_sq,
                              const volatile int* tile_of) {
    constexpr int NS = ModeTraits<MODE>::kStateArrays;
    const int tid = threadIdx.x;  // 0..kConsumers-1
    const int lane = tid & 31;
    uint32_t it = 0;
    bool ok = true;
    // compensated sums of squares (norm modes): two packed accumulators for
    // whole groups (element pairs 0, 2 and 1, 3: half the dependency chain of
    // one, measured +0.35 % on the clipped GPT-2-small step), a scalar pair
    // for the ragged end
    float2 sq2_s = make_float2(0.0f, 0.0f), sq2_c = make_float2(0.0f, 0.0f);
    float2 sq3_s = make_float2(0.0f, 0.0f), sq3_c = make_float2(0.0f, 0.0f);
    float sq_s = 0.0f, sq_c = 0.0f;
    constexpr int RG = GradTraits<GT>::kRanksPerStage;
    const bool dyn = a.h.sched_slot >= 0;
    int next_static = static_cast<int>(blockIdx.x);
    uint64_t groups = 0;   // units (of at most 64 per launch) whose tail group this CTA took
    while (ok) {
        // The next tile: in the fixed order, or (dynamic scheduling) the one
        // the producer names in the tile's first stage, -1 when none is left.
        const uint8_t* first_stage = nullptr;
        int tile;
        if (dyn) {
            const uint32_t slot = it % kStages, parity = (it / kStages) & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[slot]), parity,
                                                           abort_flag, kWaitLimitNs))) {
                ok = false;
                break;
            }
            tile = tile_of[slot];
            if (tile < 0) break;
            first_stage = smem + slot * kStageBytes;
        } else {
            tile = next_static;
            if (tile >= a.h.total_tiles) break;
            next_static += static_cast<int>(gridDim.x);
        }
        const TileGeom g = tile_geom<A, GT>(a, tile);
        if (g.nvalid == 0) continue;      // past the end of an unpadded parameter (uniform;
                                          // a dynamic producer never names such a tile)
        const UnitDesc* u = g.u;
        const int n_ranks = u->n_ranks;
        const int first = tid * kVec;
        const int nv = max(0, min(kVec, g.nvalid - first));
        const int64_t j = g.j0 + first;       // thread's first shard-local element
        const int64_t e = g.e0 + first;       // thread's first flat element

        float st[NS > 0 ? NS : 1][8];
        const bool from_smem = first + kVec <= g.state_valid;
        float2 s[4], c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s[q] = make_float2(0.0f, 0.0f);
            c[q] = make_float2(0.0f, 0.0f);
        }
        const bool vec = (nv == kVec) && (e + kVec <= g.a1);
        const int n_gr = ModeTraits<MODE>::kReadsGrads ? n_ranks : 0;
        // Ranks [k0, k0 + nk) of the tile from one stage into (s, c).
        // (rmax: a compile-time bound on nk, so that a LEAD launch's first
        // stage unrolls only the ranks it can hold)
        auto consume = [&](const uint8_t* stage, int k0, int nk, auto rmax) {
            constexpr int RM = decltype(rmax)::value;
            if (vec) {
                if constexpr (ALIGNED) {
                    consume_stage<0, RM>(stage, nk, tid, s, c, k0 == 0);
                } else if constexpr (sizeof(GT) == 4) {
                    switch (g.mis) {
                        case 0: consume_stage_f32<0, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 1: consume_stage_f32<1, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 2: consume_stage_f32<2, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        default: consume_stage_f32<3, RM>(stage, nk, tid, s, c, k0 == 0); break;
                    }
                } else {
                    switch (g.mis) {
                        case 0: consume_stage<0, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 1: consume_stage<1, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 2: consume_stage<2, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 3: consume_stage<3, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 4: consume_stage<4, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 5: consume_stage<5, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        case 6: consume_stage<6, RM>(stage, nk, tid, s, c, k0 == 0); break;
                        default: consume_stage<7, RM>(stage, nk, tid, s, c, k0 == 0); break;
                    }
                }
            } else if (nv > 0) {
                // Ragged end: scalar reads from global memory, the same two-sum
                // lane by lane (element 2q in .x, 2q+1 in .y).
                for (int kk = 0; kk < nk; ++kk) {
                    const GT* src = grad_ptr<GT, A>(a, u, k0 + kk) + e;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (2 * q < nv) {
                            two_sum_add1(s[q].x, c[q].x, GradTraits<GT>::widen(src[2 * q]));
                        }
                        if (2 * q + 1 < nv) {
                            two_sum_add1(s[q].y, c[q].y, GradTraits<GT>::widen(src[2 * q + 1]));
                        }
                    }
                }
            }
        };
        // Wait for the ring's next stage; the outcome is made warp-uniform so
        // that the warp's later shuffles see every lane.
        auto wait_full = [&]() -> const uint8_t* {
            const uint32_t slot = it % kStages, parity = (it / kStages) & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[slot]), parity,
                                                           abort_flag, kWaitLimitNs))) {
                return nullptr;
            }
            return smem + slot * kStageBytes;
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[it % kStages]));
            ++it;
        };

        if constexpr (MODE == kModePlain && sizeof(GT) == 2) {
            if (g.group) {
                // computed after the tile loop, whose registers are free then
                groups |= 1ull << static_cast<int>(u - a.unit);
                if (first_stage != nullptr) release();   // the empty stage that named it
                continue;
            }
        }
        // The tile's first stage: its state arrays, then ranks [0, r0).
        const int r0 = lead_ranks<NS, GT, LEAD>(n_gr);
        {
            const uint8_t* stage = first_stage != nullptr ? first_stage : wait_full();
            if (stage == nullptr) {
                ok = false;
                continue;
            }
#pragma unroll
            for (int arr = 0; arr < NS; ++arr) {
                if (from_smem) {
                    // A thread's 32 bytes are two 16-byte words; threads 4-7 of
                    // every 8 read their upper word first, so that each
                    // quarter-warp's 16-byte reads fall in distinct banks.
                    const float4* p =
                        reinterpret_cast<const float4*>(stage + arr * kStateArrayBytes + first * 4);
                    const int sw = (tid >> 2) & 1;
                    const float4 ya = p[sw], yb = p[sw ^ 1];
                    const float4 x0 = sw ? yb : ya, x1 = sw ? ya : yb;
                    st[arr][0] = x0.x; st[arr][1] = x0.y; st[arr][2] = x0.z; st[arr][3] = x0.w;
                    st[arr][4] = x1.x; st[arr][5] = x1.y; st[arr][6] = x1.z; st[arr][7] = x1.w;
                } else {
                    const float* src = state_ptr<MODE, A>(a, u, arr, g.r) + j;
#pragma unroll
                    for (int t = 0; t < kVec; ++t) st[arr][t] = (t < nv) ? src[t] : 0.0f;
                }
            }
            if constexpr (NS == 0 || LEAD) {
                constexpr int kFirstMax = NS == 0 ? RG : first_stage_ranks<GT>(NS);
                if (r0 > 0) {
                    consume(stage + NS * kStateArrayBytes, 0, r0,
                            std::integral_constant<int, kFirstMax>());
                }
            }
            release();
        }
        // Then RG ranks per stage (none left in a LEAD launch).
        if constexpr (NS == 0 || !LEAD) {
            for (int k0 = r0; k0 < n_gr; k0 += RG) {
                const uint8_t* stage = wait_full();
                if (stage == nullptr) {
                    ok = false;
                    break;
                }
                consume(stage, k0, min(RG, n_gr - k0), std::integral_constant<int, RG>());
                release();
            }
        }
        // every lane of this warp owns a full group (warp-uniform)
        const bool warp_full = (first - lane * kVec) + 32 * kVec <= g.nvalid;
        if (!ok || (nv == 0 && !warp_full)) continue;

        float mean[8];
        if (u->n_pow2) {
            // exact scaling, both lanes of a pair in one packed add and multiply
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 r = __fmul2_rn(__fadd2_rn(s[q], c[q]), splat2(u->inv_n));
                mean[2 * q] = r.x;
                mean[2 * q + 1] = r.y;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mean[2 * q] = finish_mean(s[q].x, c[q].x, u->n_ranks_f, u->inv_n, false);
                mean[2 * q + 1] = finish_mean(s[q].y, c[q].y, u->n_ranks_f, u->inv_n, false);
            }
        }

        if constexpr (ModeTraits<MODE>::kReduceScatter) {
            float out[8];
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                out[t] = mean[t];
                if constexpr (MODE == kModeRsAdd) out[t] = __fadd_rn(st[0][t], mean[t]);
                if constexpr (MODE == kModeRsAvgNorm) {
                    out[t] = __fdiv_rn(__fadd_rn(st[0][t], mean[t]), a.h.k.divisor);
                }
            }
            if constexpr (ModeTraits<MODE>::kNorm) {
                if (nv == kVec) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 o = make_float2(out[2 * q], out[2 * q + 1]);
                        if (q & 1) {
                            two_sum_add2(sq3_s, sq3_c, __fmul2_rn(o, o));
                        } else {
                            two_sum_add2(sq2_s, sq2_c, __fmul2_rn(o, o));
                        }
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < kVec; ++t) {
                        if (t < nv) two_sum_add1(sq_s, sq_c, __fmul_rn(out[t], out[t]));
                    }
                }
            }
            float* dst = state_ptr<MODE, A>(a, u, 0, g.r) + j;
            if (nv == kVec) {
                st_f32x8(dst, out);
            } else {
                for (int t = 0; t < nv; ++t) dst[t] = out[t];
            }
        } else {
            float gr[kVec];
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                gr[t] = mean[t];
                if constexpr (MODE == kModeAccumFinal) {
                    gr[t] = __fdiv_rn(__fadd_rn(st[3][t], mean[t]), a.h.k.divisor);
                }
                if constexpr (MODE == kModeFromShard) {
                    gr[t] = clip_coef == 1.0f ? st[3][t] : __fmul_rn(st[3][t], clip_coef);
                }
                if constexpr (MODE == kModeMeanDiv) gr[t] = __fdiv_rn(mean[t], a.h.k.divisor);
            }
#pragma unroll
            for (int t = 0; t < kVec; t += 2) {
                float2 th = make_float2(st[0][t], st[0][t + 1]);
                float2 mm = make_float2(st[1][t], st[1][t + 1]);
                float2 vv = make_float2(st[2][t], st[2][t + 1]);
                adamw_update2(a.h.k, make_float2(gr[t], gr[t + 1]), th, mm, vv);
                st[0][t] = th.x; st[0][t + 1] = th.y;
                st[1][t] = mm.x; st[1][t + 1] = mm.y;
                st[2][t] = vv.x; st[2][t + 1] = vv.y;
            }
            float* master = state_ptr<MODE, A>(a, u, 0, g.r) + j;
            float* m = state_ptr<MODE, A>(a, u, 1, g.r) + j;
            float* v = state_ptr<MODE, A>(a, u, 2, g.r) + j;
            if (nv == kVec) {
                st_f32x8(master, st[0]);
                st_f32x8(m, st[1]);
                st_f32x8(v, st[2]);
                const uint4 w = make_uint4(pack_bf16x2(st[0][0], st[0][1]),
                                           pack_bf16x2(st[0][2], st[0][3]),
                                           pack_bf16x2(st[0][4], st[0][5]),
                                           pack_bf16x2(st[0][6], st[0][7]));
                if constexpr (ALIGNED) {
                    for (int o = 0; o < u->n_out; ++o) {
                        *reinterpret_cast<uint4*>(ptr_at<uint16_t*, A>(a, u->off_out + o) + e) = w;
                    }
                } else {
                    const int mis = static_cast<int>(e & 7);
                    // An odd offset would leave store_bf16x8 eight 2-byte stores
                    // per lane; the warp then realigns through shuffles and
                    // issues one aligned 16-byte store per lane.  Even offsets
                    // keep the plain 4- or 8-byte stores (measured faster there).
                    const bool by_warp = warp_full && (mis & 1);
                    for (int o = 0; o < u->n_out; ++o) {
                        uint16_t* dst = ptr_at<uint16_t*, A>(a, u->off_out + o);
                        if (by_warp) {
                            store_bf16x8_warp(dst, e, mis, w, lane);
                        } else {
                            store_bf16x8(dst, e, mis, w);
                        }
                    }
                }
            } else {
                for (int t = 0; t < nv; ++t) {
                    master[t] = st[0][t];
                    m[t] = st[1][t];
                    v[t] = st[2][t];
                    const uint16_t b = float_to_bf16_rn(st[0][t]);
                    for (int o = 0; o < u->n_out; ++o) {
                        ptr_at<uint16_t*, A>(a, u->off_out + o)[e + t] = b;
                    }
                }
            }
        }
    }
    if constexpr (MODE == kModePlain && sizeof(GT) == 2) {
        while (ok && groups != 0) {
            const int ui = __ffsll(static_cast<long long>(groups)) - 1;
            groups &= groups - 1;
            tail_group_step<A>(a, &a.unit[ui], tid);
        }
    }
    if (lane == 0) atomicMin(consumed_min, it);
    if constexpr (ModeTraits<MODE>::kNorm) {
        // Warp sum of the threads' compensated sums, in double, fixed order.
        double w = static_cast<double>(sq3_s.x) + static_cast<double>(sq3_c.x) +
                   static_cast<double>(sq3_s.y) + static_cast<double>(sq3_c.y) +
                   static_cast<double>(sq2_s.x) + static_cast<double>(sq2_c.x) +
                   static_cast<double>(sq2_s.y) + static_cast<double>(sq2_c.y) +
                   static_cast<double>(sq_s) + static_cast<double>(sq_c);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) w += __shfl_down_sync(0xFFFFFFFFu, w, off);
        if (lane == 0) warp_sq[tid >> 5] = w;
    }
}

}  // namespace

// LEAD: every unit's whole tile fits the first stage (lead_ranks).  ALIGNED:
// every unit's shard length S is a multiple of 8, so every rank's slice and
// every thread's 8 elements start on the 16-byte grid and no realignment code
// is compiled in.
template <int MODE, class A, class GT = uint16_t, bool LEAD = false, bool ALIGNED = false>
__global__ void __launch_bounds__(kTmaThreads, 1)
staged_step_kernel(const __grid_constant__ A a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ int abort_flag;
    __shared__ uint32_t issued;
    __shared__ unsigned int consumed_min;
    __shared__ float clip_coef;
    __shared__ double warp_sq[kConsumerWarps];
    __shared__ int tile_of[kStages];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kConsumerWarps);
        }
        abort_flag = 0;
        issued = 0;
        consumed_min = 0xFFFFFFFFu;
        clip_coef = 1.0f;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if constexpr (MODE == kModeFromShard) {
        // Total norm from the norm launches' partial sums in a fixed order, so
        // that every CTA derives the same coefficient: lane l of warp 0 adds
        // slots l, l + 32, ... in turn, then a fixed shuffle tree (the lanes'
        // loads overlap instead of one thread walking every slot).
        if (threadIdx.x < 32) {
            double t = 0.0;
            for (int i = static_cast<int>(threadIdx.x); i < a.h.n_partials; i += 32) {
                t += a.h.partials[i];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_down_sync(0xFFFFFFFFu, t, off);
            if (threadIdx.x == 0) {
                const double norm = sqrt(t);
                const double coef = a.h.max_norm / (norm + 1e-6);
                clip_coef = coef >= 1.0 ? 1.0f : static_cast<float>(coef);
                if (blockIdx.x == 0 && a.h.norm_out != nullptr) {
                    *a.h.norm_out = static_cast<float>(norm);
                }
            }
        }
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            producer_loop<MODE, A, GT, LEAD>(a, smem, full, empty, &abort_flag, &issued,
                                                   tile_of);
        }
    } else {
        consumer_loop<MODE, A, GT, LEAD, ALIGNED>(a, smem, full, empty, &abort_flag,
                                                        &consumed_min, clip_coef, warp_sq,
                                                        tile_of);
    }
    __syncthreads();
    if constexpr (ModeTraits<MODE>::kNorm) {
        if (threadIdx.x == 0) {
            double total = 0.0;
            for (int w = 0; w < kConsumerWarps; ++w) total += warp_sq[w];
            a.h.partials[a.h.partial_base + blockIdx.x] = total;
        }
    }
    if (threadIdx.x == 0 && abort_flag) {
        // Let every copy this CTA issued land before shared memory goes away.
        for (uint32_t it = consumed_min; it < issued; ++it) {
            const uint32_t slot = it % kStages, parity = (it / kStages) & 1;
            int dummy = 0;
            mbar_wait_bounded(smem_u32(&full[slot]), parity, &dummy, kDrainLimitNs);
        }
    }
    if (threadIdx.x == 0 && a.h.sched_slot >= 0) {
        // Every claim of this CTA came before the barrier above; the last CTA
        // to get here puts the scheduling slot back to zero for the next
        // launch.  The counter hands out tiles G, G + 1, ... and every CTA
        // makes one claim past the end, so a slot used by this launch alone
        // ends at total_tiles (a dynamic launch has total_tiles >= G);
        // anything else means another launch claimed from it meanwhile (an
        // aborted launch has recorded its timeout already).
        unsigned int* sl = g_zf_sched[a.h.sched_slot];
        __threadfence();
        if (atomicAdd(&sl[1], 1u) == gridDim.x - 1) {
            const unsigned int claims = atomicExch(&sl[0], 0u);
            atomicExch(&sl[1], 0u);
            if (claims != static_cast<unsigned int>(a.h.total_tiles)) {
                atomicCAS(&g_zf_device_status, kDeviceOk, kDeviceSchedConflict);
            }
        }
    }
}

constexpr size_t kStagedSmem = static_cast<size_t>(kStages) * kStageBytes;

// Raise the kernel's dynamic shared-memory limit once per device.
template <int MODE, class A, class GT = uint16_t, bool LEAD = false, bool ALIGNED = false>
static cudaError_t prepare_kernel(const void* kfn) {
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (bit != 0 && (done_mask.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kStagedSmem));
    if (e == cudaSuccess && bit != 0) done_mask.fetch_or(bit, std::memory_order_release);
    return e;
}

template <int MODE, class A>
static int grid_for(int total_tiles) {
    const void* kfn = reinterpret_cast<const void*>(&staged_step_kernel<MODE, A>);
    prepare_kernel<MODE, A>(kfn);
    return persistent_grid(kfn, kTmaThreads, kStagedSmem, total_tiles);
}

template <int MODE, class A, class GT, bool LEAD, bool ALIGNED>
static cudaError_t launch_as(const A& a, cudaStream_t stream) {
    const void* kfn =
        reinterpret_cast<const void*>(&staged_step_kernel<MODE, A, GT, LEAD, ALIGNED>);
    cudaError_t e = prepare_kernel<MODE, A, GT, LEAD, ALIGNED>(kfn);
    if (e != cudaSuccess) return e;
    // h.grid when set: a norm launch runs exactly the CTAs whose partial-sum
    // slots were counted, a short multi-stage launch its balanced grid (never
    // more than the resident CTAs: the kernel has no inter-CTA dependence, and
    // CTAs beyond the resident ones would only run in a later wave).
    const int grid = a.h.grid > 0 ? a.h.grid
                                  : persistent_grid(kfn, kTmaThreads, kStagedSmem, a.h.total_tiles);
    staged_step_kernel<MODE, A, GT, LEAD, ALIGNED>
        <<<grid, kTmaThreads, kStagedSmem, stream>>>(a);
    return cudaGetLastError();
}

// Copy the used part of the host's full argument block into a smaller one.
template <class A>
static const A& shrink(const MultiArgs& big, int n_ptrs) {
    static thread_local A small;
    small.h = big.h;
    for (int i = 0; i < big.h.n_units; ++i) small.unit[i] = big.unit[i];
    for (int i = 0; i < n_ptrs; ++i) small.ptrs[i] = big.ptrs[i];
    return small;
}

// The smaller argument block when the launch fits it (a launch copies its
// whole block), else the full one.
template <int MODE, class GT, bool LEAD, bool ALIGNED>
static cudaError_t launch_form(const MultiArgs& a, int n_ptrs, cudaStream_t stream) {
    if (a.h.n_units <= MultiArgsS::kUnits && n_ptrs <= MultiArgsS::kPtrs) {
        return launch_as<MODE, MultiArgsS, GT, LEAD, ALIGNED>(
            shrink<MultiArgsS>(a, n_ptrs), stream);
    }
    return launch_as<MODE, MultiArgs, GT, LEAD, ALIGNED>(a, stream);
}

// Pick the kernel form: LEAD when every unit's whole tile fits one stage, the
// ALIGNED form when every unit's S is a multiple of 8; and
// the tile order (a.h.sched_slot).
template <int MODE, class GT = uint16_t>
static cudaError_t launch_sized(MultiArgs& a, int n_ptrs, cudaStream_t stream) {
    constexpr int NS = ModeTraits<MODE>::kStateArrays;
    constexpr bool kCanLead = can_lead<NS, GT>() && ModeTraits<MODE>::kReadsGrads;
    // every bf16-gradient mode has an ALIGNED form (the clipped step's norm
    // and update passes measured 2.5 % faster with it on GPT-2-small)
    constexpr bool kHasAligned = sizeof(GT) == 2;
    int max_ranks = 0;
    bool aligned = true;
    for (int i = 0; i < a.h.n_units; ++i) {
        if (a.unit[i].n_ranks > max_ranks) max_ranks = a.unit[i].n_ranks;
        if (a.unit[i].S % 8 != 0) aligned = false;
    }
    const bool lead = kCanLead && max_ranks <= first_stage_ranks<GT>(NS);
    // Dynamic tile order for launches that run many rounds of tiles: the SMs'
    // speeds differ (measured on GB300: up to 40 % where a tile takes one
    // stage) and a fixed order leaves the fast ones idle at the end.  Short
    // launches (fewer than kDynamicMinRounds rounds) measured about 1 % slower
    // with the claims and keep the fixed order.  The norm passes keep it too,
    // so that their per-CTA partial sums, and the norm, are reproducible bit
    // for bit.
    a.h.sched_slot = -1;
    if (!ModeTraits<MODE>::kNorm && a.h.grid == 0 &&
        a.h.total_tiles >= kDynamicMinRounds * grid_for<MODE, MultiArgsS>(a.h.total_tiles)) {
        a.h.sched_slot = sched_slot(stream);
    }
    // A short launch in the fixed order whose tiles span several stages (more
    // than 8 ranks): as many CTAs as make every round full but the last, whose
    // CTAs then finish together instead of a few of them running one more
    // multi-stage tile while the rest idle.  Measured on GB300, P = 1,048,589
    // and 4,194,304 at N_d = 64: 0.69 -> 0.71 and 0.92 -> 0.93 of the copy peak.
    if (!ModeTraits<MODE>::kNorm && a.h.grid == 0 && a.h.sched_slot < 0 &&
        ModeTraits<MODE>::kReadsGrads && !lead &&
        max_ranks > GradTraits<GT>::kRanksPerStage) {
        const int gmax = grid_for<MODE, MultiArgsS>(a.h.total_tiles);
        const int rounds = (a.h.total_tiles + gmax - 1) / gmax;
        a.h.grid = (a.h.total_tiles + rounds - 1) / rounds;
    }
    if constexpr (kHasAligned) {
        if (aligned) {
            if constexpr (kCanLead) {
                if (lead) return launch_form<MODE, GT, true, true>(a, n_ptrs, stream);
            }
            return launch_form<MODE, GT, false, true>(a, n_ptrs, stream);
        }
    }
    if constexpr (kCanLead) {
        if (lead) return launch_form<MODE, GT, true, false>(a, n_ptrs, stream);
    }
    return launch_form<MODE, GT, false, false>(a, n_ptrs, stream);
}

cudaError_t launch_staged_step_f32(MultiArgs& a, int n_ptrs, cudaStream_t stream) {
    if (a.h.total_tiles <= 0) return cudaSuccess;
    return launch_sized<kModeMeanDiv, float>(a, n_ptrs, stream);
}

// Scheduling slot of a launch on `stream` on the current device.  Launches
// made directly get their stream's slot, one per (device, stream): a stream
// runs its launches one after another and each launch leaves its slot at
// zero, so launches sharing a slot never overlap.  The per-thread default
// stream handle (cudaStreamPerThread) names a different stream in every host
// thread, so it gets a slot per (device, thread).  Launches captured into a
// CUDA graph take the capture slots in turn (a replay runs in whatever stream
// the graph is launched into).  -1 (the fixed order) once the stream slots
// are used up or when the stream's state cannot be read.  Two launches
// running at once on one slot -- a stream destroyed with a launch still
// running and its handle handed out again, or graphs holding more than
// kSharedSlot - kStreamSlots captured launches replayed at once -- are
// detected at the end of the launch (ZERO_DEVICE_SCHED_CONFLICT).
int sched_slot(cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (dev < 0 || dev >= 64) return -1;
    if (const char* f = std::getenv("ZERO_SCHED_SHARED")) {
        // failure injection for tests: every launch on one slot of its own
        if (f[0] != '\0' && f[0] != '0') return kSharedSlot;
    }
    struct Key {
        int dev;
        cudaStream_t stream;
        std::thread::id thread;   // only for cudaStreamPerThread
        int slot;
    };
    static std::mutex mu;
    static std::vector<Key> keys;
    static int used[64] = {};
    static unsigned int captured[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (cap != cudaStreamCaptureStatusNone) {
        return kStreamSlots + static_cast<int>(captured[dev]++ % (kSharedSlot - kStreamSlots));
    }
    const std::thread::id thread =
        stream == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
    for (const Key& k : keys) {
        if (k.dev == dev && k.stream == stream && k.thread == thread) return k.slot;
    }
    if (used[dev] >= kStreamSlots) return -1;
    keys.push_back(Key{dev, stream, thread, used[dev]++});
    return keys.back().slot;
}

int staged_grid(int mode, int total_tiles) {
    // The grid depends only on the kernel's resources, which every block size
    // and mode share; the smallest instantiation stands for all.
    (void)mode;
    return grid_for<kModePlain, MultiArgsS>(total_tiles);
}

cudaError_t launch_staged_step(MultiArgs& a, int n_ptrs, int mode, cudaStream_t stream) {
    if (a.h.total_tiles <= 0) return cudaSuccess;
    switch (mode) {
        case kModePlain: return launch_sized<kModePlain>(a, n_ptrs, stream);
        case kModeAccumFinal: return launch_sized<kModeAccumFinal>(a, n_ptrs, stream);
        case kModeRsStore: return launch_sized<kModeRsStore>(a, n_ptrs, stream);
        case kModeRsAdd: return launch_sized<kModeRsAdd>(a, n_ptrs, stream);
        case kModeRsNorm: return launch_sized<kModeRsNorm>(a, n_ptrs, stream);
        case kModeRsAvgNorm: return launch_sized<kModeRsAvgNorm>(a, n_ptrs, stream);
        default: return launch_sized<kModeFromShard>(a, n_ptrs, stream);
    }
}

// ---------------------------------------------------------------------------
// ZeRO-1 local accumulation through the same bulk-copy pipeline: rank k's full
// fp32 accumulator += rank k's bf16 gradient, element by element (no exchange
// between ranks).  A tile is 4096 elements of one rank's buffers; the producer
// lane copies the tile's gradient (8 KB) and, after the first micro-step, its
// accumulator (16 KB) into a ring of eight 24 KB stages, so that up to 192 KB
// per SM are in flight whatever the consumers' registers hold.  Consumers add
// in fp32 (one rounding per add, as the register kernel does) and store the
// accumulator with 16-byte streaming stores.
constexpr int kZ1Stages = 8;
constexpr int kZ1GradBytes = kStagedTile * 2;                  // 8192
constexpr int kZ1StageBytes = kZ1GradBytes + kStagedTile * 4;  // 24576
constexpr size_t kZ1Smem = static_cast<size_t>(kZ1Stages) * kZ1StageBytes;

// sched: dynamic tile-scheduling slot (as the fused step's), -1: fixed order.
// A tile here takes one stage, the form whose SMs ran at different speeds.
template <int MAXR, int FIRST>
__global__ void __launch_bounds__(kTmaThreads, 1)
zero1_accumulate_staged_kernel(const __grid_constant__ StepArgs<MAXR> a, int sched) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kZ1Stages];
    __shared__ __align__(8) uint64_t empty[kZ1Stages];
    __shared__ int abort_flag;
    __shared__ uint32_t issued;
    __shared__ unsigned int consumed_min;
    __shared__ int tile_of[kZ1Stages];
    const bool dyn = sched >= 0;
    const int64_t G = gridDim.x;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kZ1Stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kConsumerWarps);
        }
        abort_flag = 0;
        issued = 0;
        consumed_min = 0xFFFFFFFFu;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const int64_t tpr = (a.P_pad + kStagedTile - 1) / kStagedTile;
    const int64_t total = tpr * a.n_ranks;
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) {
            uint32_t it = 0;
            unsigned int* next_tile = dyn ? &g_zf_sched[sched][0] : nullptr;
            bool stop = false;
            for (int64_t tile = blockIdx.x; tile < total;
                 tile = dyn ? G + static_cast<int64_t>(atomicAdd(next_tile, 1u)) : tile + G) {
                const int k = static_cast<int>(tile / tpr);
                const int64_t e0 = (tile - k * tpr) * kStagedTile;
                const int64_t n = a.P_pad - e0 < kStagedTile ? a.P_pad - e0 : kStagedTile;
                const uint32_t gbytes = static_cast<uint32_t>(n & ~7LL) * 2;
                const uint32_t abytes = FIRST ? 0u : static_cast<uint32_t>(n & ~3LL) * 4;
                const uint32_t slot = it % kZ1Stages, parity = ((it / kZ1Stages) & 1) ^ 1;
                if (!mbar_wait_bounded(smem_u32(&empty[slot]), parity, &abort_flag, kWaitLimitNs)) {
                    stop = true;
                    break;
                }
                tile_of[slot] = static_cast<int>(tile);
                const uint32_t bar = smem_u32(&full[slot]);
                const uint32_t dst = smem_u32(smem + slot * kZ1StageBytes);
                mbar_arrive_expect_tx(bar, gbytes + abytes);
                if (gbytes > 0) bulk_copy_g2s(dst, a.grads[k] + e0, gbytes, bar);
                if (abytes > 0) bulk_copy_g2s(dst + kZ1GradBytes, a.accum[k] + e0, abytes, bar);
                ++it;
            }
            if (dyn && !stop) {
                // no tile left: an empty stage with tile index -1 stops the consumers
                const uint32_t slot = it % kZ1Stages, parity = ((it / kZ1Stages) & 1) ^ 1;
                if (mbar_wait_bounded(smem_u32(&empty[slot]), parity, &abort_flag, kWaitLimitNs)) {
                    tile_of[slot] = -1;
                    mbar_arrive(smem_u32(&full[slot]));
                    ++it;
                }
            }
            issued = it;
        }
    } else {
        const int tid = threadIdx.x;
        const int lane = tid & 31;
        const int first = tid * kVec;
        uint32_t it = 0;
        int64_t next_static = blockIdx.x;
        while (true) {
            // the next tile: in the fixed order, or the one the producer named
            // in the stage (-1: none left)
            if (!dyn && next_static >= total) break;
            const uint32_t slot = it % kZ1Stages, parity = (it / kZ1Stages) & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&full[slot]), parity,
                                                           &abort_flag, kWaitLimitNs)))
                break;
            int64_t tile = next_static;
            if (dyn) {
                tile = tile_of[slot];
                if (tile < 0) break;
            } else {
                next_static += G;
            }
            const int k = static_cast<int>(tile / tpr);
            const int64_t e0 = (tile - k * tpr) * kStagedTile;
            const int64_t n = a.P_pad - e0 < kStagedTile ? a.P_pad - e0 : kStagedTile;
            const int nv = static_cast<int>(n - first < kVec ? (n - first > 0 ? n - first : 0) : kVec);
            const uint8_t* stage = smem + slot * kZ1StageBytes;
            float* acc = a.accum[k] + e0 + first;
            float x[8];
            if (nv == kVec) {
                // a whole group lies inside both copied ranges
                const uint4 w = *reinterpret_cast<const uint4*>(stage + first * 2);
                const float2 p0 = bf16x2_to_float2(w.x), p1 = bf16x2_to_float2(w.y);
                const float2 p2 = bf16x2_to_float2(w.z), p3 = bf16x2_to_float2(w.w);
                x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y;
                x[4] = p2.x; x[5] = p2.y; x[6] = p3.x; x[7] = p3.y;
                if constexpr (!FIRST) {
                    // threads 4-7 of every 8 read their upper 16 bytes first, so
                    // that each quarter-warp's reads fall in distinct banks
                    const float4* p =
                        reinterpret_cast<const float4*>(stage + kZ1GradBytes + first * 4);
                    const int sw = (tid >> 2) & 1;
                    const float4 ya = p[sw], yb = p[sw ^ 1];
                    const float4 o0 = sw ? yb : ya, o1 = sw ? ya : yb;
                    x[0] = __fadd_rn(o0.x, x[0]); x[1] = __fadd_rn(o0.y, x[1]);
                    x[2] = __fadd_rn(o0.z, x[2]); x[3] = __fadd_rn(o0.w, x[3]);
                    x[4] = __fadd_rn(o1.x, x[4]); x[5] = __fadd_rn(o1.y, x[5]);
                    x[6] = __fadd_rn(o1.z, x[6]); x[7] = __fadd_rn(o1.w, x[7]);
                }
            } else {
                // the end of the buffer: plain reads of what the copies left out
                const uint16_t* g = a.grads[k] + e0 + first;
#pragma unroll
                for (int t = 0; t < kVec; ++t) {
                    x[t] = 0.0f;
                    if (t < nv) x[t] = FIRST ? bf16_to_float(g[t]) : __fadd_rn(acc[t], bf16_to_float(g[t]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
            ++it;
            if (nv == kVec) {
                st_f32x8(acc, x);
            } else {
#pragma unroll
                for (int t = 0; t < kVec; ++t) {
                    if (t < nv) acc[t] = x[t];
                }
            }
        }
        if (lane == 0) atomicMin(&consumed_min, it);
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        // Let every copy this CTA issued land before shared memory goes away.
        for (uint32_t it = consumed_min; it < issued; ++it) {
            const uint32_t slot = it % kZ1Stages, parity = (it / kZ1Stages) & 1;
            int dummy = 0;
            mbar_wait_bounded(smem_u32(&full[slot]), parity, &dummy, kDrainLimitNs);
        }
    }
    if (threadIdx.x == 0 && dyn) {
        // as in the fused step: the last CTA returns the slot to zero and
        // checks that it saw this launch's claims alone
        unsigned int* sl = g_zf_sched[sched];
        __threadfence();
        if (atomicAdd(&sl[1], 1u) == gridDim.x - 1) {
            const unsigned int claims = atomicExch(&sl[0], 0u);
            atomicExch(&sl[1], 0u);
            if (claims != static_cast<unsigned int>(total)) {
                atomicCAS(&g_zf_device_status, kDeviceOk, kDeviceSchedConflict);
            }
        }
    }
}

template <int MAXR>
cudaError_t launch_zero1_accumulate_staged(const StepArgs<MAXR>& a, int first,
                                           cudaStream_t stream) {
    const int64_t tiles = (a.P_pad + kStagedTile - 1) / kStagedTile * a.n_ranks;
    if (tiles <= 0) return cudaSuccess;
    const void* kfn = first ? reinterpret_cast<const void*>(&zero1_accumulate_staged_kernel<MAXR, 1>)
                            : reinterpret_cast<const void*>(&zero1_accumulate_staged_kernel<MAXR, 0>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kZ1Smem));
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(kfn, kTmaThreads, kZ1Smem, tiles);
    // dynamic order as for the fused step: launches of at least
    // kDynamicMinRounds rounds (tile indices within an int)
    const int sched = tiles >= static_cast<int64_t>(kDynamicMinRounds) * grid &&
                              tiles < std::numeric_limits<int32_t>::max()
                          ? sched_slot(stream)
                          : -1;
    if (first) {
        zero1_accumulate_staged_kernel<MAXR, 1><<<grid, kTmaThreads, kZ1Smem, stream>>>(a, sched);
    } else {
        zero1_accumulate_staged_kernel<MAXR, 0><<<grid, kTmaThreads, kZ1Smem, stream>>>(a, sched);
    }
    return cudaGetLastError();
}

template cudaError_t launch_zero1_accumulate_staged<64>(const StepArgs<64>&, int, cudaStream_t);
template cudaError_t launch_zero1_accumulate_staged<512>(const StepArgs<512>&, int, cudaStream_t);

// A barrier that nothing completes: the bounded wait must run out, record the
// timeout and let the kernel return.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns);
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t read_device_status(int* status, int clear, cudaStream_t stream) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_zf_device_status, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_zf_device_status, &zero, sizeof(int), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    *status = v;
    return e;
}

}  // namespace zf
