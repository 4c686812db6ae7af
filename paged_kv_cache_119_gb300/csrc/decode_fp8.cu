// decode_fp8.cu -- paged decode attention over E4M3 (FP8) caches with per-kv-head
// scales; queries and native outputs are fp16 or bf16.  head_dim 128 with up to 4 query
// heads per CTA runs on the E4M3 tcgen05 kernel (decode_tc8.cuh).  Otherwise the
// mma.sync kernel (decode_mma.cuh) serves at least kMmaMinHeadsFp8 query heads per CTA,
// the CUDA-core kernel (decode_kernel.cuh) the rest; all read one byte per cached element.
#include "decode_mma.cuh"

namespace pa {

namespace {

template <typename T>
cudaError_t launch_fp8(const DecodeParams& p, int head_dim, int block_size, int gc,
                       cudaStream_t stream)
{
    if (decode_kernel_for(PA_FP8_E4M3, head_dim, gc) == DecodeKernel::kMmaSync)
        return launch_decode_mma<T, __nv_fp8_e4m3>(p, head_dim, block_size, gc, stream);
    return launch_decode_typed<T, __nv_fp8_e4m3>(p, head_dim, block_size, gc, stream);
}

template <typename T>
int occupancy_fp8(int head_dim, int block_size, int gc)
{
    if (decode_kernel_for(PA_FP8_E4M3, head_dim, gc) == DecodeKernel::kMmaSync)
        return occupancy_decode_mma<T, __nv_fp8_e4m3>(head_dim, block_size, gc);
    return occupancy_decode_typed<T, __nv_fp8_e4m3>(head_dim, block_size, gc);
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeParams& p, pa_dtype q_dtype, int head_dim,
                              int block_size, int gc, cudaStream_t stream)
{
    if (decode_kernel_for(PA_FP8_E4M3, head_dim, gc) == DecodeKernel::kTc8)
        return launch_decode_tc8(p, q_dtype, block_size, gc, stream);
    if (q_dtype == PA_F16)
        return launch_fp8<__half>(p, head_dim, block_size, gc, stream);
    if (q_dtype == PA_BF16)
        return launch_fp8<__nv_bfloat16>(p, head_dim, block_size, gc, stream);
    return cudaErrorInvalidValue;
}

int occupancy_decode_fp8(pa_dtype q_dtype, int head_dim, int block_size, int gc)
{
    if (decode_kernel_for(PA_FP8_E4M3, head_dim, gc) == DecodeKernel::kTc8)
        return occupancy_decode_tc8(q_dtype, block_size, gc);
    if (q_dtype == PA_F16)
        return occupancy_fp8<__half>(head_dim, block_size, gc);
    if (q_dtype == PA_BF16)
        return occupancy_fp8<__nv_bfloat16>(head_dim, block_size, gc);
    return 0;
}

}  // namespace pa
