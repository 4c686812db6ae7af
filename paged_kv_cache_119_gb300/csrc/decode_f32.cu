// decode_f32.cu -- paged decode attention, float KV cache (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f32(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream)
{
    return launch_decode_typed<float>(p, head_dim, block_size, gc, stream);
}

int occupancy_decode_f32(int head_dim, int block_size, int gc)
{
    return occupancy_decode_typed<float>(head_dim, block_size, gc);
}

}  // namespace pa
