// Unfused pieces of the sharded step and the FlatParameter copies:
//   adamw_shard_kernel  every rank's AdamW update of its fp32 shard + bf16 cast
//                       ("Lesson 5: ZeRO and FSDP", section 3, step 2)
//   all_gather_kernel   bf16 shards -> full flat parameter buffer(s)
//                       (section 3, step 3)
//   flatten_kernel      per-tensor buffers <-> flat buffer / rank shards
//                       (section 7.1: FlatParameter flatten + tail padding)
//   zero1_accumulate_kernel  ZeRO-1 local fp32 accumulation of each rank's full
//                       gradient with register loads (section 3, on gradient
//                       accumulation); the default is the bulk-copy form in
//                       zero_step_tma.cu
#include "zero_kernels.cuh"

namespace zf {

template <int MAXR>
__global__ void __launch_bounds__(kThreads)
adamw_shard_kernel(const __grid_constant__ ShardArgs<MAXR> a) {
    const int n_tiles = a.tiles_per_rank * a.n_ranks;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int r = tile / a.tiles_per_rank;
        const int64_t j0 = static_cast<int64_t>(tile - r * a.tiles_per_rank) * kTile +
                           static_cast<int64_t>(threadIdx.x) * kVec;
        if (j0 >= a.S) continue;
        const int nv = static_cast<int>(min(static_cast<int64_t>(kVec), a.S - j0));
        float th[8], mm[8], vv[8], gs[8];
        if (nv == kVec) {
            ld_f32x8(a.master[r] + j0, th);
            ld_f32x8(a.m[r] + j0, mm);
            ld_f32x8(a.v[r] + j0, vv);
            ld_f32x8(a.grad_shards[r] + j0, gs);
        } else {
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                const bool in = t < nv;
                th[t] = in ? a.master[r][j0 + t] : 0.0f;
                mm[t] = in ? a.m[r][j0 + t] : 0.0f;
                vv[t] = in ? a.v[r][j0 + t] : 0.0f;
                gs[t] = in ? a.grad_shards[r][j0 + t] : 0.0f;
            }
        }
#pragma unroll
        for (int t = 0; t < kVec; ++t) {
            const float g = __fdiv_rn(gs[t], a.k.divisor);
            adamw_update(a.k, g, th[t], mm[t], vv[t]);
        }
        if (nv == kVec) {
            st_f32x8(a.master[r] + j0, th);
            st_f32x8(a.m[r] + j0, mm);
            st_f32x8(a.v[r] + j0, vv);
            *reinterpret_cast<uint4*>(a.param_shards[r] + j0) =
                make_uint4(pack_bf16x2(th[0], th[1]), pack_bf16x2(th[2], th[3]),
                           pack_bf16x2(th[4], th[5]), pack_bf16x2(th[6], th[7]));
        } else {
#pragma unroll
            for (int t = 0; t < kVec; ++t) {
                if (t < nv) {
                    a.master[r][j0 + t] = th[t];
                    a.m[r][j0 + t] = mm[t];
                    a.v[r][j0 + t] = vv[t];
                    a.param_shards[r][j0 + t] = float_to_bf16_rn(th[t]);
                }
            }
        }
    }
}

template <int MAXR>
__global__ void __launch_bounds__(kThreads)
all_gather_kernel(const __grid_constant__ ShardArgs<MAXR> a) {
    const int n_tiles = a.tiles_per_rank * a.n_ranks;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int r = tile / a.tiles_per_rank;
        const int64_t j0 = static_cast<int64_t>(tile - r * a.tiles_per_rank) * kTile +
                           static_cast<int64_t>(threadIdx.x) * kVec;
        if (j0 >= a.S) continue;
        const int nv = static_cast<int>(min(static_cast<int64_t>(kVec), a.S - j0));
        const int64_t e0 = static_cast<int64_t>(r) * a.S + j0;
        if (nv == kVec) {
            const uint4 w = __ldcs(reinterpret_cast<const uint4*>(a.param_shards_in[r] + j0));
            const int mis = static_cast<int>(e0 & 7);
            for (int o = 0; o < a.n_out; ++o) store_bf16x8(a.out[o], e0, mis, w);
        } else {
            for (int o = 0; o < a.n_out; ++o) {
                for (int t = 0; t < nv; ++t) a.out[o][e0 + t] = a.param_shards_in[r][j0 + t];
            }
        }
    }
}

// Index of the tensor that holds flat element e: the last t with off[t] <= e
// (zero-size tensors share their offset with the next tensor and lose the tie).
__device__ __forceinline__ int find_tensor(const FlatArgs& a, int64_t e) {
    int lo = 0, hi = a.n_tensors - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.off[mid] <= e) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

template <typename T, int UNFLATTEN>
__global__ void __launch_bounds__(kThreads) flatten_kernel(const __grid_constant__ FlatArgs a) {
    // The flat range is walked rank slice by rank slice, so that the shard
    // index needs no division.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t S = a.split ? a.S : (a.end - a.begin);
    const int64_t first = a.split ? (a.begin / S) : 0;
    const int64_t base0 = a.split ? 0 : a.begin;
    for (int64_t slice = first;; ++slice) {
        const int64_t s_begin = a.split ? slice * S : base0;
        const int64_t s_end = a.split ? s_begin + S : a.end;
        if (s_begin >= a.end) break;
        const int64_t lo = s_begin > a.begin ? s_begin : a.begin;
        const int64_t hi = s_end < a.end ? s_end : a.end;
        T* flat = static_cast<T*>(a.flat[a.split ? slice : 0]);
        const int64_t flat_origin = a.split ? s_begin : 0;
        for (int64_t e = lo + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < hi;
             e += stride) {
            if (a.n_tensors == 0) {
                if constexpr (!UNFLATTEN) flat[e - flat_origin] = T(0);
                continue;
            }
            const int t = find_tensor(a, e);
            const int64_t i = e - a.off[t];
            if constexpr (UNFLATTEN) {
                static_cast<T*>(const_cast<void*>(a.tensors[t]))[i] = flat[e - flat_origin];
            } else {
                flat[e - flat_origin] = static_cast<const T*>(a.tensors[t])[i];
            }
        }
        if (!a.split) break;
    }
}

template <int MAXR>
cudaError_t launch_adamw_shards(const ShardArgs<MAXR>& a, cudaStream_t stream) {
    const int64_t n_tiles = static_cast<int64_t>(a.tiles_per_rank) * a.n_ranks;
    const void* kfn = reinterpret_cast<const void*>(&adamw_shard_kernel<MAXR>);
    const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
    adamw_shard_kernel<MAXR><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int MAXR>
cudaError_t launch_all_gather(const ShardArgs<MAXR>& a, cudaStream_t stream) {
    const int64_t n_tiles = static_cast<int64_t>(a.tiles_per_rank) * a.n_ranks;
    const void* kfn = reinterpret_cast<const void*>(&all_gather_kernel<MAXR>);
    const int grid = persistent_grid(kfn, kThreads, 0, n_tiles);
    all_gather_kernel<MAXR><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_flatten(const FlatArgs& a, int elem_bytes, int unflatten, cudaStream_t stream) {
    const int64_t n = a.end - a.begin;
    if (n <= 0) return cudaSuccess;
    const int64_t ctas = (n + kThreads - 1) / kThreads;
#define ZF_FLATTEN_LAUNCH(T, U)                                                              \
    do {                                                                                     \
        const void* kfn = reinterpret_cast<const void*>(&flatten_kernel<T, U>);             \
        const int grid = persistent_grid(kfn, kThreads, 0, ctas);                           \
        flatten_kernel<T, U><<<grid, kThreads, 0, stream>>>(a);                             \
    } while (0)
    if (elem_bytes == 2) {
        if (unflatten) ZF_FLATTEN_LAUNCH(uint16_t, 1); else ZF_FLATTEN_LAUNCH(uint16_t, 0);
    } else {
        if (unflatten) ZF_FLATTEN_LAUNCH(uint32_t, 1); else ZF_FLATTEN_LAUNCH(uint32_t, 0);
    }
#undef ZF_FLATTEN_LAUNCH
    return cudaGetLastError();
}

// ZeRO-1 local accumulation: rank k's full fp32 accumulator (P_pad elements)
// plus its own bf16 gradient, element by element (no exchange between ranks).
// blockIdx.y is the rank; 8 elements per group, 16-byte loads and stores.
// Each thread issues the loads of kZ1Unroll groups before it adds and stores
// any of them, so that enough bytes are in flight to cover HBM latency.
constexpr int kZ1Unroll = 4;

template <int FIRST>
__device__ __forceinline__ void z1_group(const uint4 w, const float (&o)[8], float* dst) {
    float x[8];
    const float2 p0 = bf16x2_to_float2(w.x), p1 = bf16x2_to_float2(w.y);
    const float2 p2 = bf16x2_to_float2(w.z), p3 = bf16x2_to_float2(w.w);
    x[0] = p0.x; x[1] = p0.y; x[2] = p1.x; x[3] = p1.y;
    x[4] = p2.x; x[5] = p2.y; x[6] = p3.x; x[7] = p3.y;
    if constexpr (!FIRST) {
#pragma unroll
        for (int t = 0; t < kVec; ++t) x[t] = __fadd_rn(o[t], x[t]);
    }
    st_f32x8(dst, x);
}

template <int MAXR, int FIRST>
__global__ void __launch_bounds__(kThreads)
zero1_accumulate_kernel(const __grid_constant__ StepArgs<MAXR> a) {
    const int k = blockIdx.y;
    const uint16_t* g = a.grads[k];
    float* acc = a.accum[k];
    const int64_t groups = a.P_pad / kVec;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; q + (kZ1Unroll - 1) * stride < groups; q += kZ1Unroll * stride) {
        uint4 w[kZ1Unroll];
        float o[kZ1Unroll][8];
#pragma unroll
        for (int u = 0; u < kZ1Unroll; ++u) w[u] = ld_stream(g + (q + u * stride) * kVec);
        if constexpr (!FIRST) {
#pragma unroll
            for (int u = 0; u < kZ1Unroll; ++u) ld_f32x8(acc + (q + u * stride) * kVec, o[u]);
        }
#pragma unroll
        for (int u = 0; u < kZ1Unroll; ++u) z1_group<FIRST>(w[u], o[u], acc + (q + u * stride) * kVec);
    }
    for (; q < groups; q += stride) {
        const uint4 w = ld_stream(g + q * kVec);
        float o[8];
        if constexpr (!FIRST) ld_f32x8(acc + q * kVec, o);
        z1_group<FIRST>(w, o, acc + q * kVec);
    }
    const int64_t tail0 = groups * kVec;
    if (blockIdx.x == 0 && tail0 + threadIdx.x < a.P_pad) {
        const int64_t e = tail0 + threadIdx.x;
        const float x = bf16_to_float(g[e]);
        acc[e] = FIRST ? x : __fadd_rn(acc[e], x);
    }
}

template <int MAXR>
cudaError_t launch_zero1_accumulate(const StepArgs<MAXR>& a, int first, cudaStream_t stream) {
    const int64_t groups = a.P_pad / kVec;
    const void* kfn = first ? reinterpret_cast<const void*>(&zero1_accumulate_kernel<MAXR, 1>)
                            : reinterpret_cast<const void*>(&zero1_accumulate_kernel<MAXR, 0>);
    const int64_t want = (groups + kThreads - 1) / kThreads;
    int gx = persistent_grid(kfn, kThreads, 0, want * a.n_ranks) / a.n_ranks;
    if (gx < 1) gx = 1;
    if (gx > want && want > 0) gx = static_cast<int>(want);
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(a.n_ranks));
    if (first) {
        zero1_accumulate_kernel<MAXR, 1><<<grid, kThreads, 0, stream>>>(a);
    } else {
        zero1_accumulate_kernel<MAXR, 0><<<grid, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

template cudaError_t launch_zero1_accumulate<64>(const StepArgs<64>&, int, cudaStream_t);
template cudaError_t launch_zero1_accumulate<512>(const StepArgs<512>&, int, cudaStream_t);
template cudaError_t launch_adamw_shards<64>(const ShardArgs<64>&, cudaStream_t);
template cudaError_t launch_adamw_shards<512>(const ShardArgs<512>&, cudaStream_t);
template cudaError_t launch_all_gather<64>(const ShardArgs<64>&, cudaStream_t);
template cudaError_t launch_all_gather<512>(const ShardArgs<512>&, cudaStream_t);

}  // namespace zf
