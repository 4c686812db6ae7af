// decode_bf16.cu -- paged decode attention, __nv_bfloat16 KV cache: the tensor-core kernel
// (decode_mma.cuh) when a CTA serves at least kMmaMinHeads query heads of one kv head, else the
// CUDA-core kernel (decode_kernel.cuh).
#include "decode_mma.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream)
{
    if (decode_kernel_for(PA_BF16, head_dim, gc) == DecodeKernel::kMmaSync)
        return launch_decode_mma<__nv_bfloat16>(p, head_dim, block_size, gc, stream);
    return launch_decode_typed<__nv_bfloat16>(p, head_dim, block_size, gc, stream);
}

int occupancy_decode_bf16(int head_dim, int block_size, int gc)
{
    if (decode_kernel_for(PA_BF16, head_dim, gc) == DecodeKernel::kMmaSync)
        return occupancy_decode_mma<__nv_bfloat16>(head_dim, block_size, gc);
    return occupancy_decode_typed<__nv_bfloat16>(head_dim, block_size, gc);
}

}  // namespace pa
