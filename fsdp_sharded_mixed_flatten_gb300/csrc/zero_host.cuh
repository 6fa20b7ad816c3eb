// Copies between pinned host memory and device memory done by the SMs
// (loads and stores through the host memory's device mapping) instead of
// the copy engines: the host-buffer step's transport when the caller asks
// for it (ZERO_HOST_SM_COPY).
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace zf {

// Segments of one launch: segment s moves bytes[s] bytes from src[s] to
// dst[s]; both addresses are 16-byte aligned device addresses (a host buffer
// through its device mapping), bytes[s] is even.
constexpr int kHostCopySegs = 256;

struct HostCopyArgs {
    int32_t n;
    const void* src[kHostCopySegs];
    void* dst[kHostCopySegs];
    int64_t bytes[kHostCopySegs];
};

// One CTA of 1024 threads per SM, at most 32 registers a thread.  Its CTAs
// and those of the staged step kernel do not fit an SM together, so a step
// queued behind a running copy starts as the copy's CTAs finish.
cudaError_t launch_host_copy(const HostCopyArgs& a, cudaStream_t stream);

}  // namespace zf
