// cache_ops.cu -- the cache-maintenance kernels: reshape_and_cache (and its E4M3
// quantising form), copy_blocks and swap_blocks.  All but the E4M3 write are bit-exact
// 16-byte vector copies that touch no value.
//
// reshape_and_cache ("PagedAttention 完全拆解", section 原理详解（三）：kernel 实现,
// item 1, fused reshape and block write; Figure 6 decode steps): the row of each
// new token and kv head moves to the pool slot its slot_mapping entry names, in
// the pool's [block][head][slot][dim] order, in one launch.
//
// copy_blocks (same section, item 3, fused block copy; section 内存共享, Figure 8):
// many non-contiguous whole-block copies in one launch instead of one
// cudaMemcpyAsync per block.  The (src, dst) pairs and per-layer pool pointers
// travel in the kernel parameter block, so nothing is allocated or uploaded.
//
// swap_blocks (same page, section 调度与抢占, 换出 (Swapping); Figure 19a: many small
// per-block transfers leave the link idle): the same gather between two pools in
// different memories -- device and pinned host memory, which the GPU reads and
// writes directly over NVLink-C2C -- so swapping a sequence group out or in is one
// launch whatever its block count.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One thread per 16-byte vector of a (token, head) row, for K and for V.
// Consecutive threads cover consecutive vectors of one row, so both the read of
// k[i][h][:] and the write to the cache slot are fully coalesced.  64-bit grid-stride
// form, for calls of more than 2^31 - 1 vectors per tensor.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const ReshapeParams p)
{
    const int64_t per_tensor = p.num_tokens * p.num_kv_heads * p.row_vecs;
    const int64_t total = 2 * per_tensor;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const bool is_v = i >= per_tensor;
        const int64_t j = is_v ? i - per_tensor : i;
        const int c = (int)(j % p.row_vecs);
        const int64_t th = j / p.row_vecs;           // token * num_kv_heads + head
        const int h = (int)(th % p.num_kv_heads);
        const int64_t tok = th / p.num_kv_heads;
        const int64_t slot = p.slot_mapping[tok];
        if (slot < 0)
            continue;                                // padding token
        if (slot >= p.num_blocks * p.block_size) {
            if (c == 0 && h == 0 && !is_v)
                atomicOr(p.err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t off = slot - blk * p.block_size;
        const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.row_vecs + c;
        if (is_v)
            p.v_cache[dst] = p.v[j];
        else
            p.k_cache[dst] = p.k[j];
    }
}

// The usual form: one thread per 16-byte vector i of the step's (token, head) rows,
// moving vector i of K and vector i of V.  Index arithmetic is 32-bit (the launcher
// takes this form when the vector count fits), both source loads are issued before
// the slot is read, and a decode step's rows fit one resident wave (256 new tokens x
// 40 heads of LLaMA-13B: 640 CTAs).
__global__ void __launch_bounds__(256) reshape_and_cache_pair_kernel(const ReshapeParams p,
                                                                     int items)
{
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= items)
        return;
    const uint4 kx = p.k[i];
    const uint4 vx = p.v[i];
    const int th = i / p.row_vecs;                   // token * num_kv_heads + head
    const int c = i - th * p.row_vecs;
    const int tok = th / p.num_kv_heads;
    const int h = th - tok * p.num_kv_heads;
    const int64_t slot = p.slot_mapping[tok];
    if (slot < 0)
        return;                                      // padding token
    if (slot >= p.num_blocks * p.block_size) {
        if (c == 0 && h == 0)
            atomicOr(p.err, PA_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / p.block_size;
    const int64_t off = slot - blk * p.block_size;
    const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.row_vecs + c;
    p.k_cache[dst] = kx;
    p.v_cache[dst] = vx;
}

cudaError_t launch_reshape_and_cache(const ReshapeParams& p, cudaStream_t stream)
{
    const int64_t items = p.num_tokens * p.num_kv_heads * p.row_vecs;
    if (items == 0)
        return cudaSuccess;
    if (items <= INT32_MAX) {
        reshape_and_cache_pair_kernel<<<(int)((items + 255) / 256), 256, 0, stream>>>(p,
                                                                                     (int)items);
        return cudaGetLastError();
    }
    const int64_t total = 2 * items;
    const int sms = device_sm_count();
    const int64_t want = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
    const int blocks = (int)(want < cap ? want : cap);
    reshape_and_cache_kernel<<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// Quantising cache write: one thread per 16 consecutive elements of a (token, head)
// row, for K and for V; each element becomes e4m3(fp32(x) / scale[head]) (IEEE fp32
// division, round to nearest even, saturating at +-448) and the 16 codes are stored
// with one 16-byte store.  (One thread for K and V together, as in the 16-bit write,
// measured slower here: the fp32 divisions make each thread's work long, and half as
// many threads hide less of it.)
template <typename TS>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(const ReshapeFp8Params p)
{
    const int groups = p.head_dim / 16;
    const int64_t per_tensor = p.num_tokens * p.num_kv_heads * groups;
    const int64_t total = 2 * per_tensor;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const bool is_v = i >= per_tensor;
        const int64_t j = is_v ? i - per_tensor : i;
        const int grp = (int)(j % groups);
        const int64_t th = j / groups;                       // token * num_kv_heads + head
        const int h = (int)(th % p.num_kv_heads);
        const int64_t tok = th / p.num_kv_heads;
        const int64_t slot = p.slot_mapping[tok];
        if (slot < 0)
            continue;
        if (slot >= p.num_blocks * p.block_size) {
            if (grp == 0 && h == 0 && !is_v)
                atomicOr(p.err, PA_DEVERR_SLOT);
            continue;
        }
        const TS* src = reinterpret_cast<const TS*>(is_v ? p.v : p.k) + th * p.head_dim + grp * 16;
        const float scale = (is_v ? p.v_scale : p.k_scale)[h];
        float x[16];
        Load<TS, 4>::run(src, *reinterpret_cast<float(*)[4]>(&x[0]));
        Load<TS, 4>::run(src + 4, *reinterpret_cast<float(*)[4]>(&x[4]));
        Load<TS, 4>::run(src + 8, *reinterpret_cast<float(*)[4]>(&x[8]));
        Load<TS, 4>::run(src + 12, *reinterpret_cast<float(*)[4]>(&x[12]));
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(x[4 * k] / scale, x[4 * k + 1] / scale), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(x[4 * k + 2] / scale, x[4 * k + 3] / scale), __NV_SATFINITE, __NV_E4M3);
            w[k] = lo | (hi << 16);
        }
        const int64_t blk = slot / p.block_size;
        const int64_t off = slot - blk * p.block_size;
        unsigned char* dst = (is_v ? p.v_cache : p.k_cache) +
                             ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_dim + grp * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_reshape_and_cache_fp8(const ReshapeFp8Params& p, pa_dtype src_dtype,
                                         cudaStream_t stream)
{
    const int64_t total = 2 * p.num_tokens * p.num_kv_heads * (p.head_dim / 16);
    if (total == 0)
        return cudaSuccess;
    const int sms = device_sm_count();
    const int64_t want = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
    const int blocks = (int)(want < cap ? want : cap);
    switch (src_dtype) {
    case PA_F32: reshape_and_cache_fp8_kernel<float><<<blocks, 256, 0, stream>>>(p); break;
    case PA_F16: reshape_and_cache_fp8_kernel<__half><<<blocks, 256, 0, stream>>>(p); break;
    case PA_BF16: reshape_and_cache_fp8_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// grid = (pairs, 2 * layers, splits): CTA (p, l2, s) copies the s-th slice of
// block pairs[p].src of pool l2 (K pools first, then V pools) to pairs[p].dst.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyParams p)
{
    const int pair = blockIdx.x;
    const int layer = blockIdx.y >> 1;
    uint4* pool = (blockIdx.y & 1) ? p.v[layer] : p.k[layer];
    const int64_t src = (int64_t)p.pairs[pair].x * p.block_vecs;
    const int64_t dst = (int64_t)p.pairs[pair].y * p.block_vecs;
    const int64_t slice = (p.block_vecs + gridDim.z - 1) / gridDim.z;
    const int64_t lo = blockIdx.z * slice;
    const int64_t hi = min(p.block_vecs, lo + slice);
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x)
        pool[dst + i] = pool[src + i];
}

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream)
{
    if (p.num_pairs == 0 || p.num_layers == 0)
        return cudaSuccess;
    // about 8 vectors per thread per CTA; large blocks are split across CTAs
    int64_t splits = (p.block_vecs + 2047) / 2048;
    if (splits > 64)
        splits = 64;
    dim3 grid(p.num_pairs, 2 * p.num_layers, (unsigned)splits);
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// grid = (pairs, caches, slices): CTA (p, c, s) moves the s-th slice of block
// pairs[p].x of src[c] to block pairs[p].y of dst[c].  Four independent 16-byte
// loads per thread are in flight before the stores, to cover the latency of the
// host link.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const SwapParams p)
{
    const int pair = blockIdx.x;
    const uint4* src = p.src[blockIdx.y] + (int64_t)p.pairs[pair].x * p.block_vecs;
    uint4* dst = p.dst[blockIdx.y] + (int64_t)p.pairs[pair].y * p.block_vecs;
    const int64_t slice = (p.block_vecs + gridDim.z - 1) / gridDim.z;
    const int64_t lo = blockIdx.z * slice;
    const int64_t hi = min(p.block_vecs, lo + slice);
    int64_t i = lo + threadIdx.x;
    for (; i + 3 * 256 < hi; i += 4 * 256) {
        const uint4 a = src[i], b = src[i + 256], c = src[i + 512], d = src[i + 768];
        dst[i] = a;
        dst[i + 256] = b;
        dst[i + 512] = c;
        dst[i + 768] = d;
    }
    for (; i < hi; i += 256)
        dst[i] = src[i];
}

cudaError_t launch_swap_blocks(const SwapParams& p, cudaStream_t stream)
{
    if (p.num_pairs == 0 || p.num_caches == 0)
        return cudaSuccess;
    // about 16 vectors per thread per CTA; large blocks are split across CTAs
    int64_t splits = (p.block_vecs + 4095) / 4096;
    if (splits > 64)
        splits = 64;
    dim3 grid(p.num_pairs, p.num_caches, (unsigned)splits);
    swap_blocks_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
