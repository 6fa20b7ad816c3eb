// host_copy_kernel: the host-buffer step's gradient and parameter transfers
// through the SMs.  The host link carries the reduce-scatter's input and the
// all-gather's output ("Lesson 5: ZeRO and FSDP", section 3: one
// reduce-scatter in and one all-gather out per step).  On GB300 the copy
// engines' host-to-device copies come to stall for tens of milliseconds
// every few hundred milliseconds once a host has run a few jobs, while SM
// loads of the same pinned memory keep their 211 GB/s.  CTAs of 1024 threads
// with two 16-byte loads in flight per thread were the fastest of the shapes
// measured (128 to 1024 threads, 1 to 8 loads each); on a third of the SMs,
// beside a step kernel on the rest, they keep the link busy while the step
// runs (16 to 48 SMs measured; 48 best).
#include "zero_host.cuh"

namespace zf {

namespace {

constexpr int kCopyThreads = 1024;
constexpr int kCopyUnroll = 2;   // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads, 2)
host_copy_kernel(const __grid_constant__ HostCopyArgs a) {
    const uint32_t stride = gridDim.x * kCopyThreads;     // in 16-byte chunks
    for (int s = 0; s < a.n; ++s) {
        const int64_t bytes = a.bytes[s];
        const int64_t n16 = bytes / 16;
        const uint4* src = static_cast<const uint4*>(a.src[s]) + blockIdx.x * kCopyThreads +
                           threadIdx.x;
        uint4* dst = static_cast<uint4*>(a.dst[s]) + blockIdx.x * kCopyThreads + threadIdx.x;
        int64_t left = n16 - static_cast<int64_t>(blockIdx.x * kCopyThreads + threadIdx.x);
        for (; left > (kCopyUnroll - 1) * static_cast<int64_t>(stride);
             left -= kCopyUnroll * static_cast<int64_t>(stride)) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) v[u] = __ldcs(src + u * stride);
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) __stcs(dst + u * stride, v[u]);
            src += kCopyUnroll * stride;
            dst += kCopyUnroll * stride;
        }
        for (; left > 0; left -= stride, src += stride, dst += stride) __stcs(dst, __ldcs(src));
        // the last bytes % 16 bytes (an even count: bf16 rows), 2 bytes a thread
        const int tail = static_cast<int>(bytes - n16 * 16);
        if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail / 2) {
            const auto* s2 = reinterpret_cast<const uint16_t*>(static_cast<const uint4*>(a.src[s]) + n16);
            auto* d2 = reinterpret_cast<uint16_t*>(static_cast<uint4*>(a.dst[s]) + n16);
            d2[threadIdx.x] = s2[threadIdx.x];
        }
    }
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace

int host_copy_ctas() {
    const int sms = sm_count();
    return sms >= 3 ? sms / 3 : 1;
}

cudaError_t launch_host_copy(const HostCopyArgs& a, cudaStream_t stream) {
    if (a.n <= 0) return cudaSuccess;
    if (sm_count() <= 0) return cudaErrorInvalidDevice;
    host_copy_kernel<<<host_copy_ctas(), kCopyThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace zf
