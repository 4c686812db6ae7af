// chunk_attn.cu -- host launchers of chunk attention (head_dim 64 / 128, block_size
// 16 / 32): the tcgen05 kernel of chunk_attn.cuh for long chunks (f16 and bf16 caches,
// and E4M3 caches at head_dim 128 through an f16 conversion stage), and the decode
// kernels' chunk-row modes when a kv head has only a few (token, head) rows.
#include "chunk_attn.cuh"
#include "decode_mma.cuh"

namespace pa {

// F8: E4M3 caches (head_dim 128): three 16-bit stages and four raw one-byte stages.
// E4M3 and bf16 caches add the four converter warps.
template <typename T, int D, int BS, bool F8 = false>
struct ChunkVariant {
    static constexpr int kStages = F8 ? 3 : ChunkStages<D>::value;
    static constexpr int kRaw = F8 ? 4 : 0;
    static constexpr int kThreads =
        (F8 || std::is_same_v<T, __nv_bfloat16>) ? kChunkThreadsConv : kChunkThreads;
    using Sm = ChunkSmem<D, kStages, kRaw>;
    static constexpr auto kernel() { return chunk_attn_kernel<T, D, BS, kStages, kRaw>; }
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
        kernel()<<<grid, kThreads, Sm::kAlloc, stream>>>(p, tk, tv);
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
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel(), kThreads, Sm::kAlloc) !=
                cudaSuccess)
            return 0;
        return n;
    }
};

// Chunk rows on the mma.sync decode kernel: NH rows per CTA, the split merged by
// chunk_reduce_kernel (the same partial-row layout).  T: query / native output type;
// TK: cache element type (T, or __nv_fp8_e4m3 for a quantised cache).
template <typename T, int D, int BS, int NH, typename TK = T>
struct ChunkRowsVariant {
    static constexpr int kBPT = mma_blocks_per_tile<TK, D, BS>();
    static constexpr int kStages = MmaStages<TK, D, BS * kBPT>::value;
    using Sm = MmaSmem<TK, D, BS * kBPT, kStages>;
    static constexpr auto kernel() { return decode_mma_kernel<T, TK, D, BS, NH, kStages, true, kBPT>; }
    static cudaError_t configure()
    {
        return configure_once(reinterpret_cast<const void*>(kernel()), Sm::kAlloc);
    }
    static cudaError_t launch(const DecodeParams& p, const ChunkParams& cp, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream)
    {
        cudaError_t err = configure();
        if (err != cudaSuccess)
            return err;
        const bool split = p.partition_tokens > 0;
        const dim3 grid(split ? p.max_parts : 1, p.num_kv_heads * p.chunks, p.num_seqs);
        kernel()<<<grid, kDecodeThreads, Sm::kAlloc, stream>>>(p, tk, tv);
        err = cudaGetLastError();
        if (err != cudaSuccess || !split)
            return err;
        chunk_reduce_kernel<T, D><<<dim3((unsigned)cp.num_rows, cp.num_q_heads), D, 0, stream>>>(cp);
        return cudaGetLastError();
    }
    static int occupancy()
    {
        return configure() == cudaSuccess
                   ? kernel_occupancy(reinterpret_cast<const void*>(kernel()), Sm::kAlloc)
                   : 0;
    }
};

#define PA_CHUNK_ROWS_VARIANTS(X) \
    X(128, 16, 8) X(128, 16, 4) X(128, 32, 8) X(128, 32, 4) X(64, 16, 8) X(64, 16, 4) \
    X(64, 32, 8) X(64, 32, 4)

cudaError_t launch_chunk_rows(const DecodeParams& p, const ChunkParams& cp, pa_dtype dtype,
                              int head_dim, int block_size, int nh, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream)
{
#define PA_CHUNK_ROWS_CASE(D_, BS_, NH_)                                                    \
    if (head_dim == D_ && block_size == BS_ && nh == NH_)                                   \
        return dtype == PA_BF16                                                             \
                   ? ChunkRowsVariant<__nv_bfloat16, D_, BS_, NH_>::launch(p, cp, tk, tv, stream) \
                   : ChunkRowsVariant<__half, D_, BS_, NH_>::launch(p, cp, tk, tv, stream);
    if (dtype == PA_BF16 || dtype == PA_F16) {
        PA_CHUNK_ROWS_VARIANTS(PA_CHUNK_ROWS_CASE)
    }
#undef PA_CHUNK_ROWS_CASE
    return cudaErrorInvalidValue;
}

// E4M3 caches on the chunk-row path (q_dtype F16 or BF16; p.k_scale, p.v_scale set);
// the E4M3 tcgen05 kernel where use_tc8 says so, else the mma.sync kernel.
cudaError_t launch_chunk_rows_fp8(const DecodeParams& p, const ChunkParams& cp, pa_dtype q_dtype,
                                  int head_dim, int block_size, int nh, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t stream)
{
    if (use_tc8(head_dim, nh))
        return launch_chunk_rows_tc8(p, cp, q_dtype, block_size, nh, tk, tv, stream);
#define PA_CHUNK_ROWS_CASE(D_, BS_, NH_)                                                     \
    if (head_dim == D_ && block_size == BS_ && nh == NH_)                                    \
        return q_dtype == PA_BF16                                                            \
                   ? ChunkRowsVariant<__nv_bfloat16, D_, BS_, NH_, __nv_fp8_e4m3>::launch(    \
                         p, cp, tk, tv, stream)                                              \
                   : ChunkRowsVariant<__half, D_, BS_, NH_, __nv_fp8_e4m3>::launch(p, cp, tk, tv, \
                                                                                  stream);
    if (q_dtype == PA_BF16 || q_dtype == PA_F16) {
        PA_CHUNK_ROWS_VARIANTS(PA_CHUNK_ROWS_CASE)
    }
#undef PA_CHUNK_ROWS_CASE
    return cudaErrorInvalidValue;
}

int occupancy_chunk_rows_fp8(pa_dtype q_dtype, int head_dim, int block_size, int nh)
{
    if (use_tc8(head_dim, nh))
        return occupancy_chunk_rows_tc8(q_dtype, block_size, nh);
#define PA_CHUNK_ROWS_OCC(D_, BS_, NH_)                                                       \
    if (head_dim == D_ && block_size == BS_ && nh == NH_)                                     \
        return q_dtype == PA_BF16                                                             \
                   ? ChunkRowsVariant<__nv_bfloat16, D_, BS_, NH_, __nv_fp8_e4m3>::occupancy() \
                   : ChunkRowsVariant<__half, D_, BS_, NH_, __nv_fp8_e4m3>::occupancy();
    if (q_dtype == PA_BF16 || q_dtype == PA_F16) {
        PA_CHUNK_ROWS_VARIANTS(PA_CHUNK_ROWS_OCC)
    }
#undef PA_CHUNK_ROWS_OCC
    return 0;
}

int occupancy_chunk_rows(pa_dtype dtype, int head_dim, int block_size, int nh)
{
#define PA_CHUNK_ROWS_OCC(D_, BS_, NH_)                                          \
    if (head_dim == D_ && block_size == BS_ && nh == NH_)                        \
        return dtype == PA_BF16 ? ChunkRowsVariant<__nv_bfloat16, D_, BS_, NH_>::occupancy() \
                                : ChunkRowsVariant<__half, D_, BS_, NH_>::occupancy();
    if (dtype == PA_BF16 || dtype == PA_F16) {
        PA_CHUNK_ROWS_VARIANTS(PA_CHUNK_ROWS_OCC)
    }
#undef PA_CHUNK_ROWS_OCC
    return 0;
}

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

cudaError_t launch_chunk_attention_fp8(const ChunkParams& p, pa_dtype q_dtype, int block_size,
                                       const CUtensorMap& tk, const CUtensorMap& tv,
                                       cudaStream_t stream)
{
#define PA_CHUNK_F8_CASE(BS_)                                                                   \
    if (block_size == BS_)                                                                     \
        return q_dtype == PA_BF16                                                              \
                   ? ChunkVariant<__nv_bfloat16, 128, BS_, true>::launch(p, tk, tv, stream)    \
                   : ChunkVariant<__half, 128, BS_, true>::launch(p, tk, tv, stream);
    if (q_dtype == PA_BF16 || q_dtype == PA_F16) {
        PA_CHUNK_F8_CASE(16) PA_CHUNK_F8_CASE(32)
    }
#undef PA_CHUNK_F8_CASE
    return cudaErrorInvalidValue;
}

int occupancy_chunk_attention_fp8(pa_dtype q_dtype, int block_size)
{
#define PA_CHUNK_F8_OCC(BS_)                                                    \
    if (block_size == BS_)                                                     \
        return q_dtype == PA_BF16 ? ChunkVariant<__nv_bfloat16, 128, BS_, true>::occupancy() \
                                  : ChunkVariant<__half, 128, BS_, true>::occupancy();
    if (q_dtype == PA_BF16 || q_dtype == PA_F16) {
        PA_CHUNK_F8_OCC(16) PA_CHUNK_F8_OCC(32)
    }
#undef PA_CHUNK_F8_OCC
    return 0;
}

}  // namespace pa
