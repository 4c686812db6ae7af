// probe.cu -- a streaming read of one device buffer, the read-only bandwidth
// ceiling the decode kernels are measured against (they read the cache and write
// almost nothing, so a copy benchmark, which also writes, understates what they can
// reach).  Every 16-byte vector is loaded once through the read-only path; a checksum
// goes to the caller's sink word so the loads cannot be dropped.
#include <algorithm>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeCtasPerSm = 8;
constexpr int kProbeUnroll = 4;

__global__ void __launch_bounds__(kProbeThreads) stream_read_kernel(const uint4* __restrict__ p,
                                                                    int64_t n, uint32_t* sink)
{
    const int64_t stride = (int64_t)gridDim.x * kProbeThreads;
    uint32_t acc = 0;
    int64_t i = (int64_t)blockIdx.x * kProbeThreads + threadIdx.x;
    // kProbeUnroll independent 16-byte loads in flight per thread, no per-load branch
    for (; i + (kProbeUnroll - 1) * stride < n; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u)
            v[u] = __ldg(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u)
            acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n; i += stride) {
        const uint4 v = __ldg(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    // one atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0)
        atomicXor(sink, acc);
}

}  // namespace

}  // namespace pa

extern "C" int pa_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream)
{
    if (!buf || !sink || bytes == 0 || bytes % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) != 0 || (reinterpret_cast<uintptr_t>(sink) & 3u))
        return PA_ERR_INVALID;
    const int sms = pa::device_sm_count();
    if (sms <= 0)
        return PA_ERR_CUDA;
    const int64_t n = (int64_t)(bytes / 16);
    const int64_t want = (n + pa::kProbeThreads - 1) / pa::kProbeThreads;
    const int grid = (int)std::min<int64_t>((int64_t)sms * pa::kProbeCtasPerSm, want);
    pa::stream_read_kernel<<<grid, pa::kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(buf), n, sink);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
