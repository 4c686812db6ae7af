// chunk_attn.cu -- host launchers of the chunk-attention kernel (chunk_attn.cuh)
// for f16 and bf16 caches: head_dim 64 / 128, block_size 16 / 32.
#include "chunk_attn.cuh"

namespace pa {

template <typename T, int D, int BS>
struct ChunkVariant {
    static constexpr int kStages = ChunkStages<D>::value;
    using Sm = ChunkSmem<D, kStages>;
    static constexpr auto kernel() { return chunk_attn_kernel<T, D, BS, kStages>; }
    static cudaError_t configure()
    {
        return configure_once(reinterpret_cast<const void*>(kernel()), Sm::kAlloc);
    }
    static cudaError_t launch(const ChunkParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream)
    {
        cudaError_t err = configure();
        if (err != cudaSuccess)
            return err;
        const bool split = p.partition_tokens > 0;
        const dim3 grid(split ? p.max_parts : 1, p.num_kv_heads * p.m_tiles, p.num_seqs);
        kernel()<<<grid, kChunkThreads, Sm::kAlloc, stream>>>(p, tk, tv);
        err = cudaGetLastError();
        if (err != cudaSuccess || !split)
            return err;
        chunk_reduce_kernel<T, D><<<dim3((unsigned)p.num_rows, p.num_q_heads), D, 0, stream>>>(p);
        return cudaGetLastError();
    }
    static int occupancy()
    {
        int n = 0;
        if (configure() != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel(), kChunkThreads, Sm::kAlloc) !=
                cudaSuccess)
            return 0;
        return n;
    }
};

#define PA_CHUNK_VARIANTS(X) X(128, 16) X(128, 32) X(64, 16) X(64, 32)

cudaError_t launch_chunk_attention(const ChunkParams& p, pa_dtype dtype, int head_dim,
                                   int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t stream)
{
#define PA_CHUNK_CASE(D_, BS_)                                                          \
    if (head_dim == D_ && block_size == BS_)                                            \
        return dtype == PA_BF16 ? ChunkVariant<__nv_bfloat16, D_, BS_>::launch(p, tk, tv, stream) \
                                : ChunkVariant<__half, D_, BS_>::launch(p, tk, tv, stream);
    if (dtype == PA_BF16 || dtype == PA_F16) {
        PA_CHUNK_VARIANTS(PA_CHUNK_CASE)
    }
#undef PA_CHUNK_CASE
    return cudaErrorInvalidValue;
}

int occupancy_chunk_attention(pa_dtype dtype, int head_dim, int block_size)
{
#define PA_CHUNK_OCC(D_, BS_)                                                  \
    if (head_dim == D_ && block_size == BS_)                                   \
        return dtype == PA_BF16 ? ChunkVariant<__nv_bfloat16, D_, BS_>::occupancy() \
                                : ChunkVariant<__half, D_, BS_>::occupancy();
    if (dtype == PA_BF16 || dtype == PA_F16) {
        PA_CHUNK_VARIANTS(PA_CHUNK_OCC)
    }
#undef PA_CHUNK_OCC
    return 0;
}

}  // namespace pa
