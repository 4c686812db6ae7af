// decode_noalloc.cu -- pa_decode_noalloc: split-context paged decode whose
// scratch lives in a fixed, file-scope device array instead of a caller buffer.
//
// Who needs it: callers that cannot allocate device memory on the decode path.
// Examples are a plugin running inside a host runtime that owns all device
// memory and forbids cudaMalloc in its enqueue hook, and a plain C caller with
// no allocator.  cudaMalloc may synchronise the device, and it draws from
// memory the host has already budgeted.  Such callers still pass q, the caches,
// the tables and the output, but cannot hand over the workspace pa_decode's
// split path needs.
//
// Cost: every GPU that loads this module holds PA_NOALLOC_SCRATCH_BYTES of
// device memory for the life of the process.
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace {

// Partial rows, maxima and sums of the split passes (the same layout the
// caller-provided workspace of pa_decode has).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_address[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_noalloc_scratch on the current device.  Host code must not
// use the symbol itself: on the host it names a stand-in, not device memory.
// The address is looked up once per device, with that device current.
cudaError_t scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_address[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_address[dev] = ptr;
    }
    *out = g_scratch_address[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int pa_decode_noalloc(void* out, pa_dtype out_dtype, const void* q,
                                 const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                                 int64_t num_blocks, const int32_t* block_tables,
                                 int64_t block_table_stride, const int32_t* context_lens,
                                 int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 float scale, int32_t partition_size, void* stream)
{
    if (partition_size == 0)
        partition_size = pa::kAutoPartitionTokens;
    if (partition_size < 0)
        return PA_ERR_INVALID;                      // this entry point always splits
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                  max_context_len, block_size, partition_size);
    if (need > PA_NOALLOC_SCRATCH_BYTES)
        return PA_ERR_WORKSPACE;                    // larger than the static scratch
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return PA_ERR_CUDA;
    // Every partial the merge pass reads is written earlier in the same call, so
    // nothing left in the scratch by a previous call needs clearing.
    return pa_decode(out, out_dtype, q, k_cache, v_cache, kv_dtype, num_blocks, block_tables,
                     block_table_stride, context_lens, max_context_len, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, block_size, scale, partition_size, scratch,
                     PA_NOALLOC_SCRATCH_BYTES, stream);
}
