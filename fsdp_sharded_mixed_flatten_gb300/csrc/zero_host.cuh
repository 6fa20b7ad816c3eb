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

// One CTA of 1024 threads per SM on a third of the SMs (host_copy_ctas), at
// most 32 registers a thread.  Its CTAs and those of the staged step kernel
// do not fit an SM together, so the host-buffer step sizes its step launches
// for the other two thirds (set_reserved_sms) and the two run side by side.
cudaError_t launch_host_copy(const HostCopyArgs& a, cudaStream_t stream);

// CTAs (one per SM) of a transfer launch: a third of the SMs.
int host_copy_ctas();

// SMs that the calling thread's persistent step launches leave free (0: none);
// defined with the grid sizing in zero_step.cu.
void set_reserved_sms(int n);

}  // namespace zf
