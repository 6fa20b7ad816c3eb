// Reduce-scatter by averaging and the fused step of the sharded
// mixed-precision FlatParameter update, with direct (register) loads.  These
// kernels run when ZERO_STEP_KERNEL=direct is set; by default the same
// computation runs in the bulk-copy staged kernel of zero_step_tma.cu, with
// bit-identical results.
//
// Method ("Lesson 5: ZeRO and FSDP (including the FSDP2 architecture)",
// section 3): the ranks' gradients are reduce-scattered, each rank updates
// its 1/N_d fp32 master/m/v shard and casts it to bf16 in place, and the bf16
// shards are all-gathered.  With all N_d logical ranks in one GPU's memory the
// three steps become one streaming pass: every CTA tile is kTile consecutive
// elements of one rank's shard, every thread 8 of them; the thread sums the N_d
// gradient values of its elements (rank order, compensated), updates the
// state and writes the bf16 parameters straight to their all-gathered
// position.  Per element the fused pass moves 2*N_d (gradients) + 24
// (master/m/v read and write) + 2*n_out (parameters) bytes, each once.
//
// Gradient loads are 16-byte, coalesced across the warp (512 contiguous bytes
// per rank per warp), cache-streaming.  When r*S is not a multiple of 8 the
// rank's flat slice is not 16-byte aligned: each thread then reads the two
// aligned vectors that cover its 8 elements and realigns them in registers.
#include <mutex>

#include "zero_host.cuh"
#include "zero_kernels.cuh"

namespace zf {

// Sum over ranks of the 8 aligned-to-A elements starting at flat index e0,
// from vector loads.  A = e0 mod 8 is a template parameter so that the
// realignment uses fixed register selections.
template <int MAXR, int A>
__device__ __forceinline__ void rank_sum_vec(const StepArgs<MAXR>& a, int64_t e0,
                                             float2 (&s)[4], float2 (&c)[4]) {
    const int64_t ea = e0 - A;
    constexpr int U = (A == 0) ? 8 : 4;
    const int n = a.n_ranks;
    int k = 0;
    for (; k + U <= n; k += U) {
        uint4 w0[U];
        uint4 w1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint16_t* p = a.grads[k + u] + ea;
            w0[u] = ld_stream(p);
            if constexpr (A != 0) w1[u] = ld_stream(p + 8);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint4 x;
            if constexpr (A != 0) {
                x = align_shift<A>(w0[u], w1[u]);
            } else {
                x = w0[u];
            }
            two_sum_add_bf16x8_c(s, c, x);
        }
    }
    for (; k < n; ++k) {
        const uint16_t* p = a.grads[k] + ea;
        uint4 x = ld_stream(p);
        if constexpr (A != 0) x = align_shift<A>(x, ld_stream(p + 8));
        two_sum_add_bf16x8_c(s, c, x);
    }
}

// Means over ranks of the nv (<= 8) flat elements starting at e0; entries past
// nv are set to 0.
template <int MAXR>
__device__ __forceinline__ void group_mean(const StepArgs<MAXR>& a, int64_t e0, int nv,
                                           float (&mean)[8]) {
    const int mis = static_cast<int>(e0 & 7);
    const bool vec = (nv == kVec) && (mis == 0 || e0 - mis + 16 <= a.P_pad);
    if (vec) {
        float2 s[4], c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s[q] = make_float2(0.0f, 0.0f);
            c[q] = make_float2(0.0f, 0.0f);
        }
        switch (mis) {
            case 0: rank_sum_vec<MAXR, 0>(a, e0, s, c); break;
            case 1: rank_sum_vec<MAXR, 1>(a, e0, s, c); break;
            case 2: rank_sum_vec<MAXR, 2>(a, e0, s, c); break;
            case 3: rank_sum_vec<MAXR, 3>(a, e0, s, c); break;
            case 4: rank_sum_vec<MAXR, 4>(a, e0, s, c); break;
            case 5: rank_sum_vec<MAXR, 5>(a, e0, s, c); break;
            case 6: rank_sum_vec<MAXR, 6>(a, e0, s, c); break;
            default: rank_sum_vec<MAXR, 7>(a, e0, s, c); break;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mean[2 * q] = finish_mean(s[q].x, c[q].x, a.n_ranks_f, a.inv_n, a.n_pow2);
            mean[2 * q + 1] = finish_mean(s[q].y, c[q].y, a.n_ranks_f, a.inv_n, a.n_pow2);
        }
    } else {
#pragma unroll
        for (int t = 0; t < kVec; ++t) {
            float s = 0.0f, c = 0.0f;
            if (t < nv) {
                for (int k = 0; k < a.n_ranks; ++k) {
                    two_sum_add1(s, c, bf16_to_float(a.grads[k][e0 + t]));
                }
                mean[t] = finish_mean(s, c, a.n_ranks_f, a.inv_n, a.n_pow2);
            } else {
                mean[t] = 0.0f;
            }
        }
    }
}

__device__ __forceinline__ void load_shard8(const float* p, int nv, float (&x)[8]) {
    if (nv == kVec) {
        ld_f32x8(p, x);
    } else {
#pragma unroll
        for (int t = 0; t < kVec; ++t) x[t] = (t < nv) ? p[t] : 0.0f;
    }
}

__device__ __forceinline__ void store_shard8(float* p, int nv, const float (&x)[8]) {
    if (nv == kVec) {
        st_f32x8(p, x);
    } else {
#pragma unroll
        for (int t = 0; t < kVec; ++t) {
            if (t < nv) p[t] = x[t];
        }
    }
}

template <int MAXR, int MODE>
__global__ void __launch_bounds__(kThreads)
fused_step_kernel(const __grid_constant__ StepArgs<MAXR> a) {
    const int n_tiles = a.tiles_per_rank * a.n_ranks;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int r = tile / a.tiles_per_rank;
        const int64_t j0 = static_cast<int64_t>(tile - r * a.tiles_per_rank) * kTile +
                           static_cast<int64_t>(threadIdx.x) * kVec;
        if (j0 >= a.S) continue;
        const int nv = static_cast<int>(min(static_cast<int64_t>(kVec), a.S - j0));
        const int64_t e0 = static_cast<int64_t>(r) * a.S + j0;

        float th[8], mm[8], vv[8], acc[8];
        load_shard8(a.master[r] + j0, nv, th);
        load_shard8(a.m[r] + j0, nv, mm);
        load_shard8(a.v[r] + j0, nv, vv);
        if constexpr (MODE == kModeAccumFinal) load_shard8(a.accum[r] + j0, nv, acc);

        float mean[8];
        group_mean(a, e0, nv, mean);

#pragma unroll
        for (int t = 0; t < kVec; ++t) {
            float g = mean[t];
            if constexpr (MODE == kModeAccumFinal) {
                g = __fdiv_rn(__fadd_rn(acc[t], mean[t]), a.k.divisor);
            }
            adamw_update(a.k, g, th[t], mm[t], vv[t]);
        }
        store_shard8(a.master[r] + j0, nv, th);
        store_shard8(a.m[r] + j0, nv, mm);
        store_shard8(a.v[r] + j0, nv, vv);

        if (nv == kVec) {
            const uint4 w = make_uint4(pack_bf16x2(th[0], th[1]), pack_bf16x2(th[2], th[3]),
                                       pack_bf16x2(th[4], th[5]), pack_bf16x2(th[6], th[7]));
            const int mis = static_cast<int>(e0 & 7);
            for (int o = 0; o < a.n_out; ++o) store_bf16x8(a.out[o], e0, mis, w);
        } else {
            for (int o = 0; o < a.n_out; ++o) {
#pragma unroll
                for (int t = 0; t < kVec; ++t) {
                    if (t < nv) a.out[o][e0 + t] = float_to_bf16_rn(th[t]);
                }
            }
        }
    }
}

template <int MAXR, int ACC>
__global__ void __launch_bounds__(kThreads)
reduce_scatter_kernel(const __grid_constant__ StepArgs<MAXR> a) {
    const int n_tiles = a.tiles_per_rank * a.n_ranks;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int r = tile / a.tiles_per_rank;
        const int64_t j0 = static_cast<int64_t>(tile - r * a.tiles_per_rank) * kTile +
                           static_cast<int64_t>(threadIdx.x) * kVec;
        if (j0 >= a.S) continue;
        const int nv = static_cast<int>(min(static_cast<int64_t>(kVec), a.S - j0));
        const int64_t e0 = static_cast<int64_t>(r) * a.S + j0;
        float acc[8];
        if constexpr (ACC) load_shard8(a.accum[r] + j0, nv, acc);
        float mean[8];
        group_mean(a, e0, nv, mean);
        if constexpr (ACC) {
#pragma unroll
            for (int t = 0; t < kVec; ++t) mean[t] = __fadd_rn(acc[t], mean[t]);
        }
        store_shard8(a.accum[r] + j0, nv, mean);
    }
}

// SMs this thread's launches leave free for the host-buffer step's SM
// transfers (set_reserved_sms): the persistent kernels then size their grids
// for the remaining SMs, so that a step runs beside the next step's copy
// instead of behind it.
thread_local int t_reserved_sms = 0;

void set_reserved_sms(int n) { t_reserved_sms = n > 0 ? n : 0; }

// Resident CTAs per SM for (kernel, threads, smem) on a device, and the SM
// count, looked up once and cached (the occupancy query is not free).
int persistent_grid(const void* kernel, int threads, size_t smem, int64_t work_ctas) {
    struct Entry {
        const void* kernel;
        int dev, threads;
        size_t smem;
        int sms, per_sm;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n_cached = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    int sms = 0, per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cached; ++i) {
            const Entry& e = cache[i];
            if (e.kernel == kernel && e.dev == dev && e.threads == threads && e.smem == smem) {
                sms = e.sms;
                per_sm = e.per_sm;
                break;
            }
        }
        if (sms == 0) {
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
            if (sms < 1) sms = 1;
            if (per_sm < 1) per_sm = 1;
            if (n_cached < 64) cache[n_cached++] = Entry{kernel, dev, threads, smem, sms, per_sm};
        }
    }
    const int usable = t_reserved_sms < sms ? sms - t_reserved_sms : 1;
    const int64_t cap = static_cast<int64_t>(usable) * per_sm;
    const int64_t g = work_ctas < cap ? work_ctas : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

template <int MAXR>
cudaError_t launch_fused_step(const StepArgs<MAXR>& a, int mode, cudaStream_t stream) {
    const int64_t n_tiles = static_cast<int64_t>(a.tiles_per_rank) * a.n_ranks;
    if (mode == kModeAccumFinal) {
        const void* kfn = reinterpret_cast<const void*>(&fused_step_kernel<MAXR, kModeAccumFinal>);
        const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
        fused_step_kernel<MAXR, kModeAccumFinal><<<grid, kThreads, 0, stream>>>(a);
    } else {
        const void* kfn = reinterpret_cast<const void*>(&fused_step_kernel<MAXR, kModePlain>);
        const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
        fused_step_kernel<MAXR, kModePlain><<<grid, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

template <int MAXR>
cudaError_t launch_reduce_scatter(const StepArgs<MAXR>& a, int accumulate, cudaStream_t stream) {
    const int64_t n_tiles = static_cast<int64_t>(a.tiles_per_rank) * a.n_ranks;
    if (accumulate) {
        const void* kfn = reinterpret_cast<const void*>(&reduce_scatter_kernel<MAXR, 1>);
        const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
        reduce_scatter_kernel<MAXR, 1><<<grid, kThreads, 0, stream>>>(a);
    } else {
        const void* kfn = reinterpret_cast<const void*>(&reduce_scatter_kernel<MAXR, 0>);
        const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
        reduce_scatter_kernel<MAXR, 0><<<grid, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

template cudaError_t launch_fused_step<64>(const StepArgs<64>&, int, cudaStream_t);
template cudaError_t launch_fused_step<512>(const StepArgs<512>&, int, cudaStream_t);
template cudaError_t launch_reduce_scatter<64>(const StepArgs<64>&, int, cudaStream_t);
template cudaError_t launch_reduce_scatter<512>(const StepArgs<512>&, int, cudaStream_t);

}  // namespace zf
