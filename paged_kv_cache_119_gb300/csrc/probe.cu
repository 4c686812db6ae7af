// probe.cu -- a streaming read of one device buffer, the read-only bandwidth
// ceiling the decode kernels are measured against (they read the cache and write
// almost nothing, so a copy benchmark, which also writes, understates what they can
// reach).  Every 16-byte vector is loaded once through the read-only path; a checksum
// goes to the caller's sink word so the loads cannot be dropped.  A second form reads
// fixed-size runs in a caller-given order: the ceiling for a paged cache whose blocks
// of one kv head are runs of block_size x head_dim x element-size bytes scattered
// through the pool.
#include <algorithm>
#include <cstdint>

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

// Random-run read: run order[i] (RUN bytes at order[i] * RUN) for every i, each CTA
// taking `per` consecutive entries of `order` and keeping four runs in flight, as a
// decode CTA walks its block table.  An index outside [0, nruns) is skipped and
// counted in *bad.
template <int RUN>
__global__ void __launch_bounds__(kProbeThreads)
    run_read_kernel(const uint4* __restrict__ p, const int32_t* __restrict__ order, int64_t num,
                    int64_t nruns, int64_t per, uint32_t* sink, uint32_t* bad)
{
    constexpr int V = RUN / 16;                               // 16-byte vectors per run
    constexpr int K = (V + kProbeThreads - 1) / kProbeThreads; // vectors per thread per run
    uint32_t acc = 0;
    const int64_t first = (int64_t)blockIdx.x * per;
    const int64_t last = first + per < num ? first + per : num;
    for (int64_t i = first; i < last; i += 4) {
        uint4 v[4][K];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int64_t id = i + j < last ? (int64_t)__ldg(order + i + j) : -1;
            if (id >= nruns) {
                if (threadIdx.x == 0)
                    atomicAdd(bad, 1u);
                id = -1;
            }
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int e = k * kProbeThreads + threadIdx.x;
                v[j][k] = (id >= 0 && e < V) ? __ldg(p + id * V + e) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int k = 0; k < K; ++k)
                acc ^= v[j][k].x ^ v[j][k].y ^ v[j][k].z ^ v[j][k].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0)
        atomicXor(sink, acc);
}

}  // namespace

}  // namespace pa

extern "C" int pa_stream_read_runs(const void* buf, size_t bytes, uint32_t run_bytes,
                                   const int32_t* order, int64_t num_runs, uint32_t* sink,
                                   void* stream)
{
    if (!buf || !order || !sink || num_runs <= 0 || (reinterpret_cast<uintptr_t>(buf) & 15u) != 0 ||
        (reinterpret_cast<uintptr_t>(order) & 3u) != 0 || (reinterpret_cast<uintptr_t>(sink) & 3u))
        return PA_ERR_INVALID;
    if (run_bytes != 1024 && run_bytes != 2048 && run_bytes != 4096 && run_bytes != 8192 &&
        run_bytes != 16384)
        return PA_ERR_INVALID;
    const int64_t nruns = (int64_t)(bytes / run_bytes);
    if (nruns <= 0 || nruns > INT32_MAX)
        return PA_ERR_INVALID;
    const int sms = pa::device_sm_count();
    if (sms <= 0)
        return PA_ERR_CUDA;
    const int64_t grid = std::min<int64_t>((int64_t)sms * pa::kProbeCtasPerSm, num_runs);
    const int64_t per = (num_runs + grid - 1) / grid;
    const int g = (int)((num_runs + per - 1) / per);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint4* p = static_cast<const uint4*>(buf);
    uint32_t* bad = sink + 1;
    switch (run_bytes) {
    case 1024: pa::run_read_kernel<1024><<<g, pa::kProbeThreads, 0, st>>>(p, order, num_runs, nruns, per, sink, bad); break;
    case 2048: pa::run_read_kernel<2048><<<g, pa::kProbeThreads, 0, st>>>(p, order, num_runs, nruns, per, sink, bad); break;
    case 4096: pa::run_read_kernel<4096><<<g, pa::kProbeThreads, 0, st>>>(p, order, num_runs, nruns, per, sink, bad); break;
    case 8192: pa::run_read_kernel<8192><<<g, pa::kProbeThreads, 0, st>>>(p, order, num_runs, nruns, per, sink, bad); break;
    default: pa::run_read_kernel<16384><<<g, pa::kProbeThreads, 0, st>>>(p, order, num_runs, nruns, per, sink, bad); break;
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

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
