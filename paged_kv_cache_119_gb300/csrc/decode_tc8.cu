// decode_tc8.cu -- host launchers of the E4M3 tensor-core decode (decode_tc8.cuh),
// head_dim 128: decode (R = 1, 2 or 4 query heads per CTA) and chunk rows (R = 4 (token,
// head) rows per CTA).  Split launches are merged by the decode or the chunk reduce kernel (the
// same partial-row layout).
#include "chunk_attn.cuh"
#include "decode_kernel.cuh"
#include "decode_tc8.cuh"

namespace pa {

namespace {

// Ring depth: two 32 KB K + V stages, so that three CTAs fit on an SM.
template <int R>
struct Tc8Stages {
    static constexpr int value = 2;
};

template <typename T, int BS, int R, bool CH>
struct Tc8Variant {
    static constexpr int kStages = Tc8Stages<R>::value;
    using Sm = Tc8Smem<R, kStages>;
    static constexpr auto kernel() { return decode_tc8_kernel<T, BS, R, kStages, CH>; }
    static cudaError_t configure()
    {
        return configure_once(reinterpret_cast<const void*>(kernel()), Sm::kAlloc);
    }
    static cudaError_t launch(const DecodeParams& p, const ChunkParams* cp, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream)
    {
        cudaError_t err = configure();
        if (err != cudaSuccess)
            return err;
        const bool split = p.partition_tokens > 0;
        const dim3 grid(split ? p.max_parts : 1, p.num_kv_heads * p.chunks, p.num_seqs);
        kernel()<<<grid, kTc8Threads, Sm::kAlloc, stream>>>(p, tk, tv);
        err = cudaGetLastError();
        if (err != cudaSuccess || !split)
            return err;
        if constexpr (CH)
            chunk_reduce_kernel<T, 128><<<dim3((unsigned)cp->num_rows, cp->num_q_heads), 128, 0, stream>>>(*cp);
        else
            reduce_kernel<T, 128><<<dim3(p.num_q_heads, p.num_seqs), 128, 0, stream>>>(p);
        return cudaGetLastError();
    }
    static int occupancy()
    {
        int n = 0;
        if (configure() != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel(), kTc8Threads, Sm::kAlloc) !=
                cudaSuccess)
            return 0;
        return n;
    }
};

template <typename T, bool CH>
cudaError_t launch_typed(const DecodeParams& p, const ChunkParams* cp, int block_size, int rows,
                         const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream)
{
#define PA_TC8_CASE(BS_, R_)                                                       \
    if (block_size == BS_ && rows == R_)                                           \
        return Tc8Variant<T, BS_, R_, CH>::launch(p, cp, tk, tv, stream);
    PA_TC8_CASE(16, 4) PA_TC8_CASE(32, 4)
    if constexpr (!CH) {
        PA_TC8_CASE(16, 2) PA_TC8_CASE(16, 1) PA_TC8_CASE(32, 2) PA_TC8_CASE(32, 1)
    }
#undef PA_TC8_CASE
    return cudaErrorInvalidValue;
}

template <typename T, bool CH>
int occupancy_typed(int block_size, int rows)
{
#define PA_TC8_OCC(BS_, R_)                                  \
    if (block_size == BS_ && rows == R_)                     \
        return Tc8Variant<T, BS_, R_, CH>::occupancy();
    PA_TC8_OCC(16, 4) PA_TC8_OCC(32, 4)
    if constexpr (!CH) {
        PA_TC8_OCC(16, 2) PA_TC8_OCC(16, 1) PA_TC8_OCC(32, 2) PA_TC8_OCC(32, 1)
    }
#undef PA_TC8_OCC
    return 0;
}

}  // namespace

cudaError_t launch_decode_tc8(const DecodeParams& p, pa_dtype q_dtype, int block_size, int rows,
                              cudaStream_t stream)
{
    CUtensorMap tk{}, tv{};
    cudaError_t e = kv_tensor_map(&tk, p.k_cache, p.num_blocks, p.num_kv_heads, block_size, 128,
                                  PA_FP8_E4M3);
    if (e == cudaSuccess)
        e = kv_tensor_map(&tv, p.v_cache, p.num_blocks, p.num_kv_heads, block_size, 128, PA_FP8_E4M3);
    if (e != cudaSuccess)
        return e;
    if (q_dtype == PA_BF16)
        return launch_typed<__nv_bfloat16, false>(p, nullptr, block_size, rows, tk, tv, stream);
    if (q_dtype == PA_F16)
        return launch_typed<__half, false>(p, nullptr, block_size, rows, tk, tv, stream);
    return cudaErrorInvalidValue;
}

int occupancy_decode_tc8(pa_dtype q_dtype, int block_size, int rows)
{
    if (q_dtype == PA_BF16)
        return occupancy_typed<__nv_bfloat16, false>(block_size, rows);
    if (q_dtype == PA_F16)
        return occupancy_typed<__half, false>(block_size, rows);
    return 0;
}

cudaError_t launch_chunk_rows_tc8(const DecodeParams& p, const ChunkParams& cp, pa_dtype q_dtype,
                                  int block_size, int rows, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t stream)
{
    if (q_dtype == PA_BF16)
        return launch_typed<__nv_bfloat16, true>(p, &cp, block_size, rows, tk, tv, stream);
    if (q_dtype == PA_F16)
        return launch_typed<__half, true>(p, &cp, block_size, rows, tk, tv, stream);
    return cudaErrorInvalidValue;
}

int occupancy_chunk_rows_tc8(pa_dtype q_dtype, int block_size, int rows)
{
    if (q_dtype == PA_BF16)
        return occupancy_typed<__nv_bfloat16, true>(block_size, rows);
    if (q_dtype == PA_F16)
        return occupancy_typed<__half, true>(block_size, rows);
    return 0;
}

}  // namespace pa
