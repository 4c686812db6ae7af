// decode_bf16.cu -- paged decode attention, __nv_bfloat16 KV cache (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream)
{
    return launch_decode_typed<__nv_bfloat16>(p, head_dim, block_size, gc, stream);
}

}  // namespace pa
