// Bulk-copy (TMA) staged fused step and reduce-scatter, over one or many
// FlatParameters (FSDP units) per launch.
//
// Same arithmetic, element order and results as zero_step.cu (bit-identical);
// what changes is how the bytes reach the SM.  One producer lane per CTA
// streams every byte a tile reads -- the tile's fp32 state (master, m, v,
// accumulator) and, eight ranks per stage, the N_d bf16 gradient slices --
// into a ring of shared-memory stages with cp.async.bulk (the Blackwell TMA
// engine: plain global->shared copies whose completion is counted in bytes on
// an mbarrier).  Sixteen consumer warps wait on a stage, read their 8 elements
// per rank from shared memory, release the stage and finally run AdamW and
// write the results.  A tile is 4096 elements of one rank's shard of one unit,
// so every gradient copy is an 8 KB contiguous run of one buffer; the ring
// keeps up to 3 x 64 KB in flight per SM independently of the consumers'
// registers, which the direct-load kernel cannot (its in-flight bytes are
// bounded by the loads it holds in registers).  Measured on GB300: with 8
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
#include "zero_kernels.cuh"

namespace zf {

__device__ int g_zf_device_status = 0;

namespace {

constexpr int kConsumerWarps = 16;                     // 512 consumers, 8 elements each
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;           // + 1 producer warp
constexpr int kSliceElems = kStagedTile + 8;           // aligned superset of a rank's tile slice
constexpr int kSliceBytes = kSliceElems * 2;           // 8208
constexpr int kRanksPerStage = 8;
constexpr int kStageBytes = kRanksPerStage * kSliceBytes;  // 65664 (>= 4 fp32 state arrays)
constexpr int kStages = 3;                             // ring depth: 3 x 64 KB per SM
constexpr int kStateArrayBytes = kStagedTile * 4;      // 16384
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;       // 0.2 s

static_assert(kConsumers * kVec == kStagedTile, "one thread owns 8 elements of a tile");
static_assert(4 * kStateArrayBytes <= kStageBytes, "state block must fit one stage");
static_assert(kSliceBytes % 16 == 0, "bulk copies need 16-byte sizes");

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
            atomicExch(&g_zf_device_status, kDeviceTimeout);
            return false;
        }
    }
}

// Unit of a global tile index: the last unit whose first tile is <= tile.
__device__ __forceinline__ int find_unit(const MultiArgs& a, int tile) {
    int lo = 0, hi = a.n_units - 1;
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
    int mis;          // e0 mod 8
    int64_t a0;       // aligned start of every rank's copied slice
    int64_t a1;       // end of the copied slice (aligned, never past the last full 8-group)
    int state_valid;  // state elements copied (multiple of 4)
};

__device__ __forceinline__ TileGeom tile_geom(const MultiArgs& a, int tile) {
    TileGeom g;
    g.u = &a.unit[find_unit(a, tile)];
    const int local = tile - g.u->tile_begin;
    const int64_t S = g.u->S;
    g.r = local / g.u->tiles_per_rank;
    g.j0 = static_cast<int64_t>(local - g.r * g.u->tiles_per_rank) * kStagedTile;
    const int64_t rem = S - g.j0;
    g.nvalid = static_cast<int>(rem < kStagedTile ? rem : kStagedTile);
    g.e0 = static_cast<int64_t>(g.r) * S + g.j0;
    g.mis = static_cast<int>(g.e0 & 7);
    g.a0 = g.e0 - g.mis;
    const int64_t a1 = (g.e0 + g.nvalid + 7) & ~static_cast<int64_t>(7);
    const int64_t floor8 = g.u->P_pad & ~static_cast<int64_t>(7);
    g.a1 = a1 < floor8 ? a1 : floor8;
    if (g.a1 < g.a0) g.a1 = g.a0;
    g.state_valid = g.nvalid & ~3;
    return g;
}

template <typename T>
__device__ __forceinline__ T ptr_at(const MultiArgs& a, int index) {
    return static_cast<T>(const_cast<void*>(a.ptrs[index]));
}

__device__ __forceinline__ const uint16_t* grad_ptr(const MultiArgs& a, const UnitDesc* u, int k) {
    return ptr_at<const uint16_t*>(a, u->off_grads + k);
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
    static constexpr int kStateArrays = MODE == kModePlain ? 3
                                        : (MODE == kModeAccumFinal || MODE == kModeFromShard) ? 4
                                        : (MODE == kModeRsAdd || MODE == kModeRsAvgNorm) ? 1
                                                                                        : 0;
};

// State array `array` of rank r (order: master, m, v, accumulator; the
// reduce-scatter modes only have the accumulator).
template <int MODE>
__device__ __forceinline__ float* state_ptr(const MultiArgs& a, const UnitDesc* u, int array,
                                            int r) {
    if constexpr (ModeTraits<MODE>::kReduceScatter) {
        return ptr_at<float*>(a, u->off_accum + r);
    } else {
        const int off = array == 0 ? u->off_master
                        : array == 1 ? u->off_m
                        : array == 2 ? u->off_v
                                     : u->off_accum;
        return ptr_at<float*>(a, off + r);
    }
}

// Sum up to kRanksPerStage rank slices of one stage into (s, c) for a
// thread's 8 elements starting A elements into its aligned pair of words.
template <int A>
__device__ __forceinline__ void consume_stage(const uint8_t* stage, int nk, int tid,
                                              float2 (&s)[4], float2 (&c)[4]) {
    const uint8_t* base = stage + tid * 16;
#pragma unroll
    for (int kk = 0; kk < kRanksPerStage; ++kk) {
        if (kk < nk) {
            const uint4* p = reinterpret_cast<const uint4*>(base + kk * kSliceBytes);
            uint4 x = p[0];
            if constexpr (A != 0) x = align_shift<A>(x, p[1]);
            two_sum_add_bf16x8(s, c, x);
        }
    }
}

template <int MODE>
__device__ void producer_loop(const MultiArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                              volatile int* abort_flag, uint32_t* issued_out) {
    constexpr int NS = ModeTraits<MODE>::kStateArrays;
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < a.total_tiles; tile += gridDim.x) {
        const TileGeom g = tile_geom(a, tile);
        const int n_ranks = g.u->n_ranks;
        if constexpr (NS > 0) {
            const uint32_t slot = it % kStages, parity = ((it / kStages) & 1) ^ 1;
            if (!mbar_wait_bounded(smem_u32(&empty[slot]), parity, abort_flag, kWaitLimitNs)) break;
            const uint32_t bytes = static_cast<uint32_t>(g.state_valid) * 4;
            const uint32_t bar = smem_u32(&full[slot]);
            mbar_arrive_expect_tx(bar, NS * bytes);
            if (bytes > 0) {
                const uint32_t dst = smem_u32(smem + slot * kStageBytes);
#pragma unroll
                for (int arr = 0; arr < NS; ++arr) {
                    bulk_copy_g2s(dst + arr * kStateArrayBytes,
                                  state_ptr<MODE>(a, g.u, arr, g.r) + g.j0, bytes, bar);
                }
            }
            ++it;
        }
        const uint32_t gbytes = static_cast<uint32_t>(g.a1 - g.a0) * 2;
        const int groups =
            ModeTraits<MODE>::kReadsGrads ? (n_ranks + kRanksPerStage - 1) / kRanksPerStage : 0;
        bool stop = false;
        for (int grp = 0; grp < groups; ++grp) {
            const uint32_t slot = it % kStages, parity = ((it / kStages) & 1) ^ 1;
            if (!mbar_wait_bounded(smem_u32(&empty[slot]), parity, abort_flag, kWaitLimitNs)) {
                stop = true;
                break;
            }
            const int k0 = grp * kRanksPerStage;
            const int nk = min(kRanksPerStage, n_ranks - k0);
            const uint32_t bar = smem_u32(&full[slot]);
            mbar_arrive_expect_tx(bar, nk * gbytes);
            if (gbytes > 0) {
                const uint32_t dst = smem_u32(smem + slot * kStageBytes);
                for (int kk = 0; kk < nk; ++kk) {
                    bulk_copy_g2s(dst + kk * kSliceBytes, grad_ptr(a, g.u, k0 + kk) + g.a0, gbytes,
                                  bar);
                }
            }
            ++it;
        }
        if (stop || *abort_flag) break;
    }
    *issued_out = it;
}

template <int MODE>
__device__ void consumer_loop(const MultiArgs& a, const uint8_t* smem, uint64_t* full,
                              uint64_t* empty, volatile int* abort_flag,
                              unsigned int* consumed_min, float clip_coef, double* warp_sq) {
    constexpr int NS = ModeTraits<MODE>::kStateArrays;
    const int tid = threadIdx.x;  // 0..kConsumers-1
    const int lane = tid & 31;
    uint32_t it = 0;
    bool ok = true;
    float sq_s = 0.0f, sq_c = 0.0f;   // compensated sum of squares (norm modes)
    for (int tile = blockIdx.x; tile < a.total_tiles && ok; tile += gridDim.x) {
        const TileGeom g = tile_geom(a, tile);
        const UnitDesc* u = g.u;
        const int n_ranks = u->n_ranks;
        const int first = tid * kVec;
        const int nv = max(0, min(kVec, g.nvalid - first));
        const int64_t j = g.j0 + first;       // thread's first shard-local element
        const int64_t e = g.e0 + first;       // thread's first flat element

        float st[NS > 0 ? NS : 1][8];
        if constexpr (NS > 0) {
            const uint32_t slot = it % kStages, parity = (it / kStages) & 1;
            if (!mbar_wait_bounded(smem_u32(&full[slot]), parity, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            const bool from_smem = first + kVec <= g.state_valid;
#pragma unroll
            for (int arr = 0; arr < NS; ++arr) {
                if (from_smem) {
                    const float4* p = reinterpret_cast<const float4*>(
                        smem + slot * kStageBytes + arr * kStateArrayBytes + first * 4);
                    const float4 x0 = p[0], x1 = p[1];
                    st[arr][0] = x0.x; st[arr][1] = x0.y; st[arr][2] = x0.z; st[arr][3] = x0.w;
                    st[arr][4] = x1.x; st[arr][5] = x1.y; st[arr][6] = x1.z; st[arr][7] = x1.w;
                } else {
                    const float* src = state_ptr<MODE>(a, u, arr, g.r) + j;
#pragma unroll
                    for (int t = 0; t < kVec; ++t) st[arr][t] = (t < nv) ? src[t] : 0.0f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
            ++it;
        }

        float2 s[4], c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s[q] = make_float2(0.0f, 0.0f);
            c[q] = make_float2(0.0f, 0.0f);
        }
        const bool vec = (nv == kVec) && (e + kVec <= g.a1);
        const int groups =
            ModeTraits<MODE>::kReadsGrads ? (n_ranks + kRanksPerStage - 1) / kRanksPerStage : 0;
        for (int grp = 0; grp < groups; ++grp) {
            const uint32_t slot = it % kStages, parity = (it / kStages) & 1;
            if (!mbar_wait_bounded(smem_u32(&full[slot]), parity, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            const int k0 = grp * kRanksPerStage;
            const int nk = min(kRanksPerStage, n_ranks - k0);
            const uint8_t* stage = smem + slot * kStageBytes;
            if (vec) {
                switch (g.mis) {
                    case 0: consume_stage<0>(stage, nk, tid, s, c); break;
                    case 1: consume_stage<1>(stage, nk, tid, s, c); break;
                    case 2: consume_stage<2>(stage, nk, tid, s, c); break;
                    case 3: consume_stage<3>(stage, nk, tid, s, c); break;
                    case 4: consume_stage<4>(stage, nk, tid, s, c); break;
                    case 5: consume_stage<5>(stage, nk, tid, s, c); break;
                    case 6: consume_stage<6>(stage, nk, tid, s, c); break;
                    default: consume_stage<7>(stage, nk, tid, s, c); break;
                }
            } else if (nv > 0) {
                // Ragged end: scalar reads from global memory, the same two-sum
                // lane by lane (element 2q in .x, 2q+1 in .y).
                for (int kk = 0; kk < nk; ++kk) {
                    const uint16_t* src = grad_ptr(a, u, k0 + kk) + e;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (2 * q < nv) two_sum_add1(s[q].x, c[q].x, bf16_to_float(src[2 * q]));
                        if (2 * q + 1 < nv) {
                            two_sum_add1(s[q].y, c[q].y, bf16_to_float(src[2 * q + 1]));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
            ++it;
        }
        if (!ok || nv == 0) continue;

        float mean[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mean[2 * q] = finish_mean(s[q].x, c[q].x, u->n_ranks_f, u->inv_n, u->n_pow2);
            mean[2 * q + 1] = finish_mean(s[q].y, c[q].y, u->n_ranks_f, u->inv_n, u->n_pow2);
        }

        if constexpr (ModeTraits<MODE>::kReduceScatter) {
            float out[8];
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                out[t] = mean[t];
                if constexpr (MODE == kModeRsAdd) out[t] = __fadd_rn(st[0][t], mean[t]);
                if constexpr (MODE == kModeRsAvgNorm) {
                    out[t] = __fdiv_rn(__fadd_rn(st[0][t], mean[t]), a.k.divisor);
                }
                if constexpr (ModeTraits<MODE>::kNorm) {
                    if (t < nv) two_sum_add1(sq_s, sq_c, __fmul_rn(out[t], out[t]));
                }
            }
            float* dst = state_ptr<MODE>(a, u, 0, g.r) + j;
            if (nv == kVec) {
                st_f32x8(dst, out);
            } else {
                for (int t = 0; t < nv; ++t) dst[t] = out[t];
            }
        } else {
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                float gr = mean[t];
                if constexpr (MODE == kModeAccumFinal) {
                    gr = __fdiv_rn(__fadd_rn(st[3][t], mean[t]), a.k.divisor);
                }
                if constexpr (MODE == kModeFromShard) {
                    gr = clip_coef == 1.0f ? st[3][t] : __fmul_rn(st[3][t], clip_coef);
                }
                adamw_update(a.k, gr, st[0][t], st[1][t], st[2][t]);
            }
            float* master = state_ptr<MODE>(a, u, 0, g.r) + j;
            float* m = state_ptr<MODE>(a, u, 1, g.r) + j;
            float* v = state_ptr<MODE>(a, u, 2, g.r) + j;
            if (nv == kVec) {
                st_f32x8(master, st[0]);
                st_f32x8(m, st[1]);
                st_f32x8(v, st[2]);
                const uint4 w = make_uint4(pack_bf16x2(st[0][0], st[0][1]),
                                           pack_bf16x2(st[0][2], st[0][3]),
                                           pack_bf16x2(st[0][4], st[0][5]),
                                           pack_bf16x2(st[0][6], st[0][7]));
                const int mis = static_cast<int>(e & 7);
                for (int o = 0; o < u->n_out; ++o) {
                    store_bf16x8(ptr_at<uint16_t*>(a, u->off_out + o), e, mis, w);
                }
            } else {
                for (int t = 0; t < nv; ++t) {
                    master[t] = st[0][t];
                    m[t] = st[1][t];
                    v[t] = st[2][t];
                    const uint16_t b = float_to_bf16_rn(st[0][t]);
                    for (int o = 0; o < u->n_out; ++o) {
                        ptr_at<uint16_t*>(a, u->off_out + o)[e + t] = b;
                    }
                }
            }
        }
    }
    if (lane == 0) atomicMin(consumed_min, it);
    if constexpr (ModeTraits<MODE>::kNorm) {
        // Warp sum of the threads' compensated sums, in double, fixed order.
        double w = static_cast<double>(sq_s) + static_cast<double>(sq_c);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) w += __shfl_down_sync(0xFFFFFFFFu, w, off);
        if (lane == 0) warp_sq[tid >> 5] = w;
    }
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kTmaThreads, 1)
staged_step_kernel(const __grid_constant__ MultiArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ int abort_flag;
    __shared__ uint32_t issued;
    __shared__ unsigned int consumed_min;
    __shared__ float clip_coef;
    __shared__ double warp_sq[kConsumerWarps];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kConsumerWarps);
        }
        abort_flag = 0;
        issued = 0;
        consumed_min = 0xFFFFFFFFu;
        clip_coef = 1.0f;
        if constexpr (MODE == kModeFromShard) {
            // Total norm from the norm launches' partial sums, in a fixed order,
            // so every CTA derives the same coefficient.
            double total = 0.0;
            for (int i = 0; i < a.n_partials; ++i) total += a.partials[i];
            const double norm = sqrt(total);
            const double coef = a.max_norm / (norm + 1e-6);
            clip_coef = coef >= 1.0 ? 1.0f : static_cast<float>(coef);
            if (blockIdx.x == 0 && a.norm_out != nullptr) *a.norm_out = static_cast<float>(norm);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) producer_loop<MODE>(a, smem, full, empty, &abort_flag, &issued);
    } else {
        consumer_loop<MODE>(a, smem, full, empty, &abort_flag, &consumed_min, clip_coef, warp_sq);
    }
    __syncthreads();
    if constexpr (ModeTraits<MODE>::kNorm) {
        if (threadIdx.x == 0) {
            double total = 0.0;
            for (int w = 0; w < kConsumerWarps; ++w) total += warp_sq[w];
            a.partials[a.partial_base + blockIdx.x] = total;
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
}

constexpr size_t kStagedSmem = static_cast<size_t>(kStages) * kStageBytes;

template <int MODE>
static int grid_for(int total_tiles) {
    const void* kfn = reinterpret_cast<const void*>(&staged_step_kernel<MODE>);
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kStagedSmem));
    return persistent_grid(kfn, kTmaThreads, kStagedSmem, total_tiles);
}

template <int MODE>
static cudaError_t launch_staged(const MultiArgs& a, cudaStream_t stream) {
    const void* kfn = reinterpret_cast<const void*>(&staged_step_kernel<MODE>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kStagedSmem));
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(kfn, kTmaThreads, kStagedSmem, a.total_tiles);
    staged_step_kernel<MODE><<<grid, kTmaThreads, kStagedSmem, stream>>>(a);
    return cudaGetLastError();
}

int staged_grid(int mode, int total_tiles) {
    switch (mode) {
        case kModePlain: return grid_for<kModePlain>(total_tiles);
        case kModeAccumFinal: return grid_for<kModeAccumFinal>(total_tiles);
        case kModeRsStore: return grid_for<kModeRsStore>(total_tiles);
        case kModeRsAdd: return grid_for<kModeRsAdd>(total_tiles);
        case kModeRsNorm: return grid_for<kModeRsNorm>(total_tiles);
        case kModeRsAvgNorm: return grid_for<kModeRsAvgNorm>(total_tiles);
        default: return grid_for<kModeFromShard>(total_tiles);
    }
}

cudaError_t launch_staged_step(const MultiArgs& a, int mode, cudaStream_t stream) {
    if (a.total_tiles <= 0) return cudaSuccess;
    switch (mode) {
        case kModePlain: return launch_staged<kModePlain>(a, stream);
        case kModeAccumFinal: return launch_staged<kModeAccumFinal>(a, stream);
        case kModeRsStore: return launch_staged<kModeRsStore>(a, stream);
        case kModeRsAdd: return launch_staged<kModeRsAdd>(a, stream);
        case kModeRsNorm: return launch_staged<kModeRsNorm>(a, stream);
        case kModeRsAvgNorm: return launch_staged<kModeRsAvgNorm>(a, stream);
        default: return launch_staged<kModeFromShard>(a, stream);
    }
}

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
