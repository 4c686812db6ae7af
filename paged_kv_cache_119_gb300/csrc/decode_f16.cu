// decode_f16.cu -- paged decode attention, __half KV cache (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream)
{
    return launch_decode_typed<__half>(p, head_dim, block_size, gc, stream);
}

}  // namespace pa
