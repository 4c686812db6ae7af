// pa_internal.h -- declarations shared by the library's translation units
// (kernel parameter blocks and per-dtype launchers).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "pa.h"

namespace pa {

// Consumer warps per decode CTA; one more warp issues the bulk copies.
constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeThreads = (kDecodeConsumerWarps + 1) * 32;
// 16-bit caches use the tensor-core decode when a CTA serves at least this many
// query heads, else the CUDA-core decode.
constexpr int kMmaMinHeads = 4;
// E4M3 caches: the same threshold (the tensor-core kernel's exact one-instruction
// E4M3 -> f16 conversion is measured against the CUDA-core kernel's E4M3 -> f32).
constexpr int kMmaMinHeadsFp8 = 4;
// Partition length the automatic split uses (a multiple of every block size).
constexpr int kAutoPartitionTokens = 512;

struct DecodeParams {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    // one-pass CUDA-core decode, optional: CTA row z serves sequence seq_order[z].x,
    // whose context length is seq_order[z].y (the longest-first order seq_order.cu
    // builds); null: row z serves sequence z
    const int2* seq_order;
    float* part_o;       // [S][Hq][max_parts][D] normalised partial outputs (split only)
    float* part_ml;      // [S][Hq][max_parts][2] (running max in log2 units, sum)
    const float* k_scale;  // [Hkv] per-head scales of a quantised (E4M3) cache, else null
    const float* v_scale;
    unsigned* err;       // device error word
    int64_t num_blocks;
    int64_t bt_stride;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;           // num_q_heads / num_kv_heads
    int chunks;          // group / heads-per-CTA
    int max_context_len;
    int partition_tokens;  // 0: one CTA covers the whole context
    int max_parts;
    int out_f32;
    float scale_log2;    // scale * log2(e): scores are kept in base-2 units
    // chunk rows (decode_mma_kernel's CH mode only; null / 0 for decode)
    const int32_t* query_start;
    int64_t num_rows;
    int max_query_len;
    // test hook of the CUDA-core decode (0 = off): CTA (linear block index) fault_cta - 1
    // issues no copy and waits fault_wait_ns at most, so its bounded waits give up
    int fault_cta;
    uint32_t fault_wait_ns;
};

// Longest-first dispatch of a one-pass CUDA-core decode with more CTAs than one wave:
// a CTA that starts late on a long context stretches the kernel's tail.  seq_order.cu
// sorts the sequences into kOrderClasses length classes, longest class first, stably
// (index order within a class, so neighbouring sequences, e.g. ones sharing a prefix,
// stay close).  The order takes 8 bytes per sequence of the call's workspace.
// (Measured on the LLaMA-13B batch: 4 classes 412.3 us, 8 classes 409.7, 16 classes
// 407.6; 16 is what the order kernel's 64 registers a thread hold.)
constexpr int kOrderClasses = 16;
inline size_t seq_order_bytes(int64_t num_seqs)
{
    return (size_t)((num_seqs * 8 + 255) / 256 * 256);
}
cudaError_t launch_seq_order(const int32_t* context_lens, int num_seqs, int max_context_len,
                             int2* order, cudaStream_t stream);

// Per-dtype decode launchers (one translation unit each).  `gc` is the number of
// query heads one CTA serves (1, 2, 4 or 8).  Return cudaErrorInvalidValue for
// an unsupported (head_dim, block_size, gc) combination.
cudaError_t launch_decode_f32(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream);
cudaError_t launch_decode_f16(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int block_size, int gc,
                               cudaStream_t stream);

// E4M3 caches (decode_fp8.cu): q_dtype PA_F16 or PA_BF16; p.k_scale / p.v_scale set.
cudaError_t launch_decode_fp8(const DecodeParams& p, pa_dtype q_dtype, int head_dim,
                              int block_size, int gc, cudaStream_t stream);
int occupancy_decode_fp8(pa_dtype q_dtype, int head_dim, int block_size, int gc);
// Whether an E4M3 call with this head_dim and rows per CTA (query heads, or chunk rows)
// runs on the E4M3 tcgen05 kernel (decode_tc8.cuh).  At 8 rows per CTA the mma.sync
// kernel streams faster (measured on GB300: its four consumer warps work on separate
// blocks and free each block on its own, against one 128-token tile chain per CTA).
inline bool use_tc8(int head_dim, int rows) { return head_dim == 128 && rows <= 4; }

// The attention kernel a decode call runs, from the cache type, head_dim and the query
// heads one CTA serves (gc).  The per-dtype launchers route by this function, and
// pa_decode_kernel_name reports it, so the two cannot disagree.
enum class DecodeKernel { kCudaCore, kMmaSync, kTc8 };
inline DecodeKernel decode_kernel_for(pa_dtype kv_dtype, int head_dim, int gc)
{
    if (kv_dtype == PA_FP8_E4M3) {
        if (use_tc8(head_dim, gc))
            return DecodeKernel::kTc8;
        return gc >= kMmaMinHeadsFp8 ? DecodeKernel::kMmaSync : DecodeKernel::kCudaCore;
    }
    if (kv_dtype != PA_F32 && gc >= kMmaMinHeads)
        return DecodeKernel::kMmaSync;
    return DecodeKernel::kCudaCore;
}
// The E4M3 tensor-core decode at head_dim 128 (decode_tc8.cu): `rows` = query heads per
// CTA (1, 2, 4 or 8); makes its own tensor maps.
cudaError_t launch_decode_tc8(const DecodeParams& p, pa_dtype q_dtype, int block_size, int rows,
                              cudaStream_t stream);
int occupancy_decode_tc8(pa_dtype q_dtype, int block_size, int rows);

// Resident decode CTAs per SM for this dtype / shape / heads-per-CTA (0 if unknown).
int occupancy_decode_f32(int head_dim, int block_size, int gc);
int occupancy_decode_f16(int head_dim, int block_size, int gc);
int occupancy_decode_bf16(int head_dim, int block_size, int gc);

struct ReshapeParams {
    const uint4* k;
    const uint4* v;
    uint4* k_cache;
    uint4* v_cache;
    const int64_t* slot_mapping;
    unsigned* err;
    int64_t num_tokens;
    int64_t num_blocks;
    int num_kv_heads;
    int row_vecs;       // 16-byte vectors per head row (head_dim * elem_size / 16)
    int block_size;
};
cudaError_t launch_reshape_and_cache(const ReshapeParams& p, cudaStream_t stream);

// Quantising cache write into E4M3 caches: codes e4m3(fp32(x) / scale[h]).
struct ReshapeFp8Params {
    const void* k;
    const void* v;
    unsigned char* k_cache;
    unsigned char* v_cache;
    const float* k_scale;
    const float* v_scale;
    const int64_t* slot_mapping;
    unsigned* err;
    int64_t num_tokens;
    int64_t num_blocks;
    int num_kv_heads;
    int head_dim;       // a multiple of 16
    int block_size;
};
cudaError_t launch_reshape_and_cache_fp8(const ReshapeFp8Params& p, pa_dtype src_dtype,
                                         cudaStream_t stream);

// One copy_blocks launch covers up to kCopyMaxLayers layers and kCopyMaxPairs
// pairs; the parameter block stays under the classic 4 KB kernel-parameter limit.
constexpr int kCopyMaxLayers = 8;
constexpr int kCopyMaxPairs = 480;
struct CopyParams {
    uint4* k[kCopyMaxLayers];
    uint4* v[kCopyMaxLayers];
    int2 pairs[kCopyMaxPairs];
    int64_t block_vecs;  // 16-byte vectors per block
    int num_layers;
    int num_pairs;
};
cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream);

// Block moves between two pools of each cache (swapping to and from a pinned host
// pool).  Up to kSwapMaxCaches caches and kSwapMaxPairs pairs per launch: about
// 9 KB of kernel parameters (sm_70 and later take up to 32 KB).
constexpr int kSwapMaxCaches = 64;
constexpr int kSwapMaxPairs = 1024;
struct SwapParams {
    const uint4* src[kSwapMaxCaches];
    uint4* dst[kSwapMaxCaches];
    int2 pairs[kSwapMaxPairs];   // (source block, destination block)
    int64_t block_vecs;          // 16-byte vectors per block
    int num_caches;
    int num_pairs;
};
cudaError_t launch_swap_blocks(const SwapParams& p, cudaStream_t stream);

// Tensor map over a [num_blocks][num_kv_heads][block_size][head_dim] cache, as
// 3-D (head_dim, block_size, num_blocks * num_kv_heads) with 128-byte swizzle and
// a box of 128-byte rows x block_size tokens (64 dims of a 16-bit dtype, or 128
// E4M3 codes; E4M3 needs head_dim 128).  Encoded maps are cached per (base,
// shape, dtype).
cudaError_t kv_tensor_map(CUtensorMap* map, const void* base, int64_t num_blocks, int num_kv_heads,
                          int block_size, int head_dim, pa_dtype dtype);

// (query token, query head) rows one chunk-attention CTA serves (two 128-row tiles).
constexpr int kChunkCtaRows = 256;

// Causal attention of chunks of new query tokens over the paged cache (the
// tensor-core kernel of chunk_attn.cuh).  Rows of q / out are (query token, query
// head) pairs, [num_rows][num_q_heads][head_dim].
struct ChunkParams {
    void* out;                   // [num_rows][Hq][D], fp32 or the cache dtype
    const void* q;               // [num_rows][Hq][D], the cache dtype
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;  // [num_seqs + 1]
    float* part_o;               // [num_rows][Hq][max_parts][D] (split only)
    float* part_ml;              // [num_rows][Hq][max_parts][2]
    const float* k_scale;        // [Hkv] scales of E4M3 caches, else null
    const float* v_scale;
    unsigned* err;
    int64_t num_blocks;
    int64_t bt_stride;
    int64_t num_rows;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;                   // num_q_heads / num_kv_heads (<= 128)
    int rows_tokens;             // chunk tokens per CTA: kChunkCtaRows / group
    int m_tiles;                 // row tiles per (sequence, kv head)
    int max_query_len;
    int max_context_len;
    int partition_tokens;        // 0: one pass; else a multiple of 64
    int max_parts;
    int out_f32;
    float scale_log2;
};
cudaError_t launch_chunk_attention(const ChunkParams& p, pa_dtype dtype, int head_dim,
                                   int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t stream);
// Resident chunk-attention CTAs per SM (0 if unknown).
int occupancy_chunk_attention(pa_dtype dtype, int head_dim, int block_size);
// The same kernel over E4M3 caches (head_dim 128; q_dtype F16 or BF16; p.k_scale and
// p.v_scale set): the tiles are converted to f16 in shared memory; tk / tv are the
// E4M3 tensor maps.
cudaError_t launch_chunk_attention_fp8(const ChunkParams& p, pa_dtype q_dtype, int block_size,
                                       const CUtensorMap& tk, const CUtensorMap& tv,
                                       cudaStream_t stream);
int occupancy_chunk_attention_fp8(pa_dtype q_dtype, int block_size);
// Few rows per kv head: the mma.sync decode kernel in chunk-row mode, `nh` (4 or 8)
// rows per CTA; p carries the chunk fields (query_start, num_rows, max_query_len)
// and p.chunks = row chunks per kv head; cp describes the same call for the merge.
// Rows per kv head at or below this use it.
constexpr int kChunkRowsMax = 32;
cudaError_t launch_chunk_rows(const DecodeParams& p, const ChunkParams& cp, pa_dtype dtype,
                              int head_dim, int block_size, int nh, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream);
int occupancy_chunk_rows(pa_dtype dtype, int head_dim, int block_size, int nh);
// E4M3 caches, chunk rows: short chunks at head_dim 128 and every chunk at head_dim 64
// (long chunks at 128 take launch_chunk_attention_fp8).
cudaError_t launch_chunk_rows_fp8(const DecodeParams& p, const ChunkParams& cp, pa_dtype q_dtype,
                                  int head_dim, int block_size, int nh, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t stream);
int occupancy_chunk_rows_fp8(pa_dtype q_dtype, int head_dim, int block_size, int nh);
// E4M3 chunk rows at head_dim 128 on the E4M3 tensor-core decode (decode_tc8.cu), `rows`
// (4 or 8) rows per CTA; tk / tv are the E4M3 tensor maps of the caches.
cudaError_t launch_chunk_rows_tc8(const DecodeParams& p, const ChunkParams& cp, pa_dtype q_dtype,
                                  int block_size, int rows, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t stream);
int occupancy_chunk_rows_tc8(pa_dtype q_dtype, int block_size, int rows);

// Sets the dynamic shared-memory limit of a kernel once per device and process.
inline cudaError_t configure_once(const void* kernel, int smem_bytes)
{
    static std::mutex mu;
    static std::vector<std::pair<const void*, int>> done;   // (kernel, device)
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& d : done)
        if (d.first == kernel && d.second == dev)
            return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (err == cudaSuccess)
        done.emplace_back(kernel, dev);
    return err;
}

// The calling device's error word (device address), or nullptr on failure.
unsigned* device_error_word();
// SM count of the calling device (cached), or 0 on failure.
int device_sm_count();

}  // namespace pa
