// pa_api.cu -- the C ABI of libpa.so (declared in include/pa.h): argument
// validation, the split-context and dispatch-order decisions, workspace carving and
// kernel dispatch.
// Everything here is host code except the device error word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

// Device error word (PA_DEVERR_* bits); one per device, set by the kernels.
__device__ unsigned g_device_error;

namespace {

constexpr int kMaxDevices = 64;
unsigned* g_error_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(int dt) { return dt == PA_F32 ? 4 : (dt == PA_FP8_E4M3 ? 1 : 2); }

bool valid_dtype(int dt) { return dt == PA_F32 || dt == PA_F16 || dt == PA_BF16; }

// [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Whether [ws, ws + n) shares a byte with any of the buffers: a workspace the kernels
// write while they read the call's inputs must be disjoint from all of them.
struct Span {
    const void* p;
    size_t n;
};
bool overlaps_any(const void* ws, size_t n, std::initializer_list<Span> bufs)
{
    for (const Span& b : bufs)
        if (overlaps(ws, n, b.p, b.n))
            return true;
    return false;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Query heads served by one decode CTA: the largest of 8, 4, 2, 1 dividing the group.
int heads_per_cta(int group)
{
    for (int gc : {8, 4, 2, 1})
        if (group % gc == 0)
            return gc;
    return 1;
}

// Partition length in tokens, or 0 for one pass per (sequence, kv head).
// partition_size < 0: never split; > 0: that length whenever it splits anything.
// 0 (automatic): with units = sequences x kv heads x head chunks (CTAs per
// partition) and slots = SMs x resident decode CTAs per SM, keep one pass when
// units > slots / 2 (the unsplit grid already fills at least half the GPU).
// Otherwise split into parts = min(slots / units, max_context_len / 512) so that
// one wave of CTAs fills the resident slots: concurrent CTAs share the HBM
// bandwidth, so a single full wave of long partitions beats several waves of
// short ones (measured on GB300: 8 x 32768 tokens, 64 CTAs per partition,
// 166 us at 8 parts vs 171 us at 19 and 194 us at 64).
int choose_partition(int partition_size, int max_context_len, int64_t units, int64_t slots,
                     int block_size)
{
    if (partition_size < 0)
        return 0;
    if (partition_size > 0)
        return max_context_len > partition_size ? partition_size : 0;
    const int pmin = kAutoPartitionTokens;
    if (max_context_len <= pmin)
        return 0;
    if (slots <= 0)
        slots = 2 * 148;
    if (2 * units > slots)
        return 0;
    const int64_t max_parts = (max_context_len + pmin - 1) / pmin;
    const int64_t parts = std::min<int64_t>(slots / units, max_parts);
    if (parts <= 1)
        return 0;
    const int per = (int)((max_context_len + parts - 1) / parts);
    const int P = (per + block_size - 1) / block_size * block_size;
    return P >= max_context_len ? 0 : P;
}

// Partition length of the chunk-attention kernel (a multiple of its 64-token K/V
// tile), or 0 for one pass; the same one-wave rule as choose_partition.
int choose_chunk_partition(int partition_size, int max_context_len, int64_t units, int64_t slots)
{
    if (partition_size < 0)
        return 0;
    if (partition_size > 0)
        return max_context_len > partition_size ? partition_size : 0;
    const int pmin = kAutoPartitionTokens;
    if (max_context_len <= pmin)
        return 0;
    if (slots <= 0)
        slots = 148;
    if (2 * units > slots)
        return 0;
    const int64_t max_parts = (max_context_len + pmin - 1) / pmin;
    const int64_t parts = std::min<int64_t>(slots / units, max_parts);
    if (parts <= 1)
        return 0;
    const int per = (int)((max_context_len + parts - 1) / parts);
    const int P = (per + 63) / 64 * 64;
    return P >= max_context_len ? 0 : P;
}

// Partition length of the E4M3 tensor-core decode (decode_tc8.cuh), or 0 for one pass.
// A CTA of that kernel keeps about one 32 KB tile load in flight, so the grid needs many
// CTAs to cover the memory latency: with units = CTAs per partition and slots = SMs x
// resident CTAs per SM, contexts are cut until the grid holds about four CTAs per slot,
// into whole 128-token tiles of at least 512 tokens.  An explicit partition_size is
// used as in choose_partition.
int choose_partition_tc8(int partition_size, int max_context_len, int64_t units, int64_t slots)
{
    if (partition_size < 0)
        return 0;
    if (partition_size > 0)
        return max_context_len > partition_size ? partition_size : 0;
    if (slots <= 0)
        slots = 3 * 148;
    const int64_t want = 4 * slots;
    if (units >= want || max_context_len <= 512)
        return 0;
    const int64_t max_parts = (max_context_len + 511) / 512;
    const int64_t parts = std::min<int64_t>((want + units - 1) / units, max_parts);
    if (parts <= 1)
        return 0;
    const int per = (int)((max_context_len + parts - 1) / parts);
    const int P = (per + 127) / 128 * 128;
    return P >= max_context_len ? 0 : P;
}

size_t workspace_layout(int64_t rows, int max_parts, int head_dim, size_t* ml_offset)
{
    const size_t o_bytes = align_up((size_t)rows * max_parts * head_dim * sizeof(float), 256);
    if (ml_offset)
        *ml_offset = o_bytes;
    return o_bytes + (size_t)rows * max_parts * 2 * sizeof(float);
}

}  // namespace

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

struct MapKey {
    const void* base;
    int64_t num_blocks;
    int num_kv_heads, block_size, head_dim, dtype;
    bool operator==(const MapKey& o) const
    {
        return base == o.base && num_blocks == o.num_blocks && num_kv_heads == o.num_kv_heads &&
               block_size == o.block_size && head_dim == o.head_dim && dtype == o.dtype;
    }
};

constexpr int kMapCache = 16;
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};
MapEntry g_map_cache[kMapCache];
int g_map_next = 0;
std::mutex g_map_mutex;

}  // namespace

cudaError_t kv_tensor_map(CUtensorMap* map, const void* base, int64_t num_blocks, int num_kv_heads,
                          int block_size, int head_dim, pa_dtype dtype)
{
    const MapKey key{base, num_blocks, num_kv_heads, block_size, head_dim, (int)dtype};
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (const MapEntry& e : g_map_cache)
        if (e.used && e.key == key) {
            *map = e.map;
            return cudaSuccess;
        }
    EncodeTiledFn fn = encode_tiled_fn();
    const bool fp8 = dtype == PA_FP8_E4M3;
    if (!fn || (!fp8 && elem_size(dtype) != 2) || (fp8 && head_dim != 128))
        return cudaErrorNotSupported;
    if (num_blocks * (int64_t)num_kv_heads >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;           // the TMA z coordinate is a signed 32-bit int
    const cuuint64_t esz = fp8 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)block_size,
                                (cuuint64_t)num_blocks * (cuuint64_t)num_kv_heads};
    const cuuint64_t strides[2] = {head_dim * esz, (cuuint64_t)block_size * head_dim * esz};
    const cuuint32_t box[3] = {fp8 ? 128u : 64u, (cuuint32_t)block_size, 1};   // 128-byte rows
    const cuuint32_t estride[3] = {1, 1, 1};
    CUtensorMap m;
    const CUresult r = fn(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : (dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16),
                          3, const_cast<void*>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    g_map_cache[g_map_next] = MapEntry{key, m, true};
    g_map_next = (g_map_next + 1) % kMapCache;
    *map = m;
    return cudaSuccess;
}

unsigned* device_error_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    if (!g_error_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess)
            return nullptr;
        g_error_ptr[dev] = static_cast<unsigned*>(ptr);
    }
    return g_error_ptr[dev];
}

int device_sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim/block_size/dtype not built";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: split-context workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime or launch failure";
    default: return "unknown pa_status";
    }
}

const char* pa_version(void) { return "paged_kv_cache_119_gb300 0.1 sm_103a"; }

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t block_size,
                                 int32_t partition_size)
{
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        block_size <= 0 || partition_size < 0)
        return 0;
    // an automatic one-pass call's dispatch order
    const size_t order = partition_size == 0 ? seq_order_bytes(num_seqs) : 0;
    const int P = partition_size > 0 ? partition_size : kAutoPartitionTokens;
    if (max_context_len <= P)
        return order;
    const int max_parts = (max_context_len + P - 1) / P;
    return std::max(order, workspace_layout((int64_t)num_seqs * num_q_heads, max_parts,
                                            head_dim, nullptr));
}

}  // extern "C"

namespace {

// The partition length pa_decode uses for these arguments (0: one pass).  *order_out
// (optional): whether a one-pass call builds the longest-first dispatch order -- an
// automatic call on the CUDA-core decode kernel whose grid holds more CTAs than one
// wave.  Measured on GB300: the LLaMA-13B and OPT-13B batches decode 2.5 % faster in
// that order.  The other kernels are slower in it: the E4M3 tcgen05 decode by 8-10 %
// (its CTAs' fixed start-up and epilogue work no longer hides behind long streams once
// only short sequences are left), the shared-prefix mma.sync batch by 2.5 % (sequences
// that share prefix blocks no longer run side by side).
int decode_partition(pa_dtype q_dtype, pa_dtype kv_dtype, int num_seqs, int num_kv_heads,
                     int group, int head_dim, int block_size, int max_context_len,
                     int partition_size, bool* order_out = nullptr)
{
    const int gc = heads_per_cta(group);
    int occ = 0;
    if (partition_size == 0) {
        switch (kv_dtype) {
        case PA_F32: occ = occupancy_decode_f32(head_dim, block_size, gc); break;
        case PA_F16: occ = occupancy_decode_f16(head_dim, block_size, gc); break;
        case PA_BF16: occ = occupancy_decode_bf16(head_dim, block_size, gc); break;
        case PA_FP8_E4M3: occ = occupancy_decode_fp8(q_dtype, head_dim, block_size, gc); break;
        }
    }
    const int64_t units = (int64_t)num_seqs * num_kv_heads * (group / gc);
    const int64_t slots = (int64_t)device_sm_count() * occ;
    const DecodeKernel kernel = decode_kernel_for(kv_dtype, head_dim, gc);
    if (order_out)
        *order_out = partition_size == 0 && kernel == DecodeKernel::kCudaCore && slots > 0 &&
                     units > slots;
    if (kernel == DecodeKernel::kTc8)
        return choose_partition_tc8(partition_size, max_context_len, units, slots);
    return choose_partition(partition_size, max_context_len, units, slots, block_size);
}

// How pa_chunk_attention runs a call: few (token, head) rows per kv head go to a decode
// kernel in chunk-row mode (nh rows per CTA), longer chunks to the tcgen05 chunk kernel
// (rows_tokens chunk tokens per CTA; over E4M3 caches with an f16 conversion stage, at
// head_dim 128 -- E4M3 at head_dim 64 always takes the chunk-row path); partition =
// split length.
struct ChunkPlan {
    bool rows_path;
    int nh;          // rows per CTA on the decode kernel
    int chunks;      // CTAs per (sequence, kv head, partition)
    int rows_tokens; // tcgen05 kernel: chunk tokens per CTA
    int partition;
};

ChunkPlan chunk_plan(pa_dtype q_dtype, pa_dtype kv_dtype, int num_seqs, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_query_len,
                     int max_context_len, int partition_size)
{
    ChunkPlan c{};
    const int group = num_q_heads / num_kv_heads;
    const int64_t rows = (int64_t)max_query_len * group;
    const bool fp8 = kv_dtype == PA_FP8_E4M3;
    if (rows <= kChunkRowsMax || (fp8 && head_dim != 128)) {
        c.rows_path = true;
        c.nh = rows <= 4 ? 4 : 8;
        c.chunks = (int)std::min<int64_t>((rows + c.nh - 1) / c.nh, INT32_MAX);
        int occ = 0;
        if (partition_size == 0)
            occ = fp8 ? occupancy_chunk_rows_fp8(q_dtype, head_dim, block_size, c.nh)
                      : occupancy_chunk_rows(kv_dtype, head_dim, block_size, c.nh);
        const int64_t units = (int64_t)num_seqs * num_kv_heads * c.chunks;
        const int64_t slots = (int64_t)device_sm_count() * occ;
        c.partition = (fp8 && use_tc8(head_dim, c.nh))
                          ? choose_partition_tc8(partition_size, max_context_len, units, slots)
                          : choose_partition(partition_size, max_context_len, units, slots,
                                             block_size);
        return c;
    }
    c.rows_tokens = kChunkCtaRows / group;
    c.chunks = (max_query_len + c.rows_tokens - 1) / c.rows_tokens;
    int occ = 0;
    if (partition_size == 0)
        occ = fp8 ? occupancy_chunk_attention_fp8(q_dtype, block_size)
                  : occupancy_chunk_attention(kv_dtype, head_dim, block_size);
    c.partition = choose_chunk_partition(partition_size, max_context_len,
                                         (int64_t)num_seqs * num_kv_heads * c.chunks,
                                         (int64_t)device_sm_count() * occ);
    return c;
}

// One-shot wait-timeout test hook armed by pa_test_arm_wait_timeout, consumed by the
// calling thread's next decode call: (chosen CTA's linear index + 1, wait limit in ns).
thread_local int g_fault_cta = 0;
thread_local uint32_t g_fault_wait_ns = 0;

// Shared body of pa_decode and pa_decode_fp8.  q_dtype is the type of q (and of a
// native out); kv_dtype the cache's, PA_FP8_E4M3 with k_scale / v_scale.
int decode_impl(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                const float* k_scale, const float* v_scale, int64_t num_blocks,
                const int32_t* block_tables, int64_t block_table_stride,
                const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                float scale, int32_t partition_size, void* workspace, size_t workspace_bytes,
                void* stream)
{
    const bool fp8 = kv_dtype == PA_FP8_E4M3;
    const int fault_cta = g_fault_cta;           // the test hook lasts one call
    const uint32_t fault_wait_ns = g_fault_wait_ns;
    g_fault_cta = 0;
    g_fault_wait_ns = 0;
    if (!valid_dtype(q_dtype) || !(out_dtype == PA_F32 || out_dtype == q_dtype))
        return PA_ERR_INVALID;
    if (num_seqs < 0 || num_seqs > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return PA_ERR_INVALID;
    if (!(head_dim == 64 || head_dim == 128) || !(block_size == 16 || block_size == 32))
        return PA_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_table_stride <= 0 ||
        max_context_len < 0 || (int64_t)max_context_len > block_table_stride * block_size ||
        !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (partition_size > 0 && partition_size % block_size != 0)
        return PA_ERR_INVALID;
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID;
    if (fp8 && (!k_scale || !v_scale))
        return PA_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID;

    const int group = num_q_heads / num_kv_heads;
    const int gc = heads_per_cta(group);
    const int chunks = group / gc;
    if ((int64_t)num_kv_heads * chunks > 65535)
        return PA_ERR_INVALID;
    const size_t q_bytes = (size_t)num_seqs * num_q_heads * head_dim * elem_size(q_dtype);
    const size_t out_bytes = (size_t)num_seqs * num_q_heads * head_dim * elem_size(out_dtype);
    const size_t pool_bytes =
        (size_t)num_blocks * num_kv_heads * block_size * head_dim * elem_size(kv_dtype);
    if (overlaps(out, out_bytes, q, q_bytes) || overlaps(out, out_bytes, k_cache, pool_bytes) ||
        overlaps(out, out_bytes, v_cache, pool_bytes))
        return PA_ERR_INVALID;
    const std::initializer_list<Span> inputs = {
        {out, out_bytes}, {q, q_bytes}, {k_cache, pool_bytes}, {v_cache, pool_bytes},
        {block_tables, (size_t)num_seqs * (size_t)block_table_stride * 4},
        {context_lens, (size_t)num_seqs * 4}};

    bool order_seqs = false;
    const int P = decode_partition(q_dtype, kv_dtype, num_seqs, num_kv_heads, group, head_dim,
                                   block_size, max_context_len, partition_size, &order_seqs);
    DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.k_scale = fp8 ? k_scale : nullptr;
    p.v_scale = fp8 ? v_scale : nullptr;
    p.num_blocks = num_blocks;
    p.bt_stride = block_table_stride;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.chunks = chunks;
    p.max_context_len = max_context_len;
    p.partition_tokens = P;
    p.max_parts = 1;
    p.out_f32 = out_dtype == PA_F32 ? 1 : 0;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);  // log2(e)
    p.fault_cta = fault_cta;
    p.fault_wait_ns = fault_wait_ns;
    if (P > 0) {
        p.max_parts = (max_context_len + P - 1) / P;
        size_t ml_off = 0;
        const size_t need = workspace_layout((int64_t)num_seqs * num_q_heads, p.max_parts,
                                             head_dim, &ml_off);
        if (!workspace || workspace_bytes < need || !aligned16(workspace))
            return PA_ERR_WORKSPACE;
        if (overlaps_any(workspace, need, inputs))
            return PA_ERR_INVALID;
        p.part_o = static_cast<float*>(workspace);
        p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off);
    }
    p.err = device_error_word();
    if (!p.err)
        return PA_ERR_CUDA;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // a one-pass CUDA-core grid of several waves starts the longest sequences first, when
    // the workspace has room for the order and touches none of the inputs it is built from
    const size_t order_bytes = seq_order_bytes(num_seqs);
    if (P == 0 && order_seqs && workspace && aligned16(workspace) &&
        workspace_bytes >= order_bytes && !overlaps_any(workspace, order_bytes, inputs)) {
        int2* order = static_cast<int2*>(workspace);
        if (launch_seq_order(context_lens, num_seqs, max_context_len, order, st) != cudaSuccess)
            return PA_ERR_CUDA;
        p.seq_order = order;
    }
    cudaError_t e = cudaErrorInvalidValue;
    switch (kv_dtype) {
    case PA_F32: e = launch_decode_f32(p, head_dim, block_size, gc, st); break;
    case PA_F16: e = launch_decode_f16(p, head_dim, block_size, gc, st); break;
    case PA_BF16: e = launch_decode_bf16(p, head_dim, block_size, gc, st); break;
    case PA_FP8_E4M3: e = launch_decode_fp8(p, q_dtype, head_dim, block_size, gc, st); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
              const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
              const int32_t* block_tables, int64_t block_table_stride,
              const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
              float scale, int32_t partition_size, void* workspace, size_t workspace_bytes,
              void* stream)
{
    if (!valid_dtype(kv_dtype))
        return PA_ERR_INVALID;
    return decode_impl(out, out_dtype, q, kv_dtype, k_cache, v_cache, kv_dtype, nullptr, nullptr,
                       num_blocks, block_tables, block_table_stride, context_lens,
                       max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, scale, partition_size, workspace, workspace_bytes, stream);
}

int pa_decode_fp8(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                  const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, int64_t num_blocks, const int32_t* block_tables,
                  int64_t block_table_stride, const int32_t* context_lens,
                  int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float scale,
                  int32_t partition_size, void* workspace, size_t workspace_bytes, void* stream)
{
    if (!(q_dtype == PA_F16 || q_dtype == PA_BF16))
        return PA_ERR_UNSUPPORTED;
    return decode_impl(out, out_dtype, q, q_dtype, k_cache, v_cache, PA_FP8_E4M3, k_scale,
                       v_scale, num_blocks, block_tables, block_table_stride, context_lens,
                       max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, scale, partition_size, workspace, workspace_bytes, stream);
}

int32_t pa_decode_partition_tokens(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t max_context_len,
                                   int32_t partition_size)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || max_context_len < 0 || block_size <= 0)
        return PA_ERR_INVALID;
    if (partition_size > 0 && partition_size % block_size != 0)
        return PA_ERR_INVALID;
    if (partition_size == 0 && device_sm_count() <= 0)
        return PA_ERR_CUDA;
    return decode_partition(q_dtype, kv_dtype, num_seqs, num_kv_heads, num_q_heads / num_kv_heads,
                            head_dim, block_size, max_context_len, partition_size);
}

int32_t pa_decode_orders_sequences(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t max_context_len,
                                   int32_t partition_size)
{
    const int32_t P = pa_decode_partition_tokens(q_dtype, kv_dtype, num_seqs, num_q_heads,
                                                 num_kv_heads, head_dim, block_size,
                                                 max_context_len, partition_size);
    if (P != 0)
        return P < 0 ? P : 0;
    bool order_seqs = false;
    decode_partition(q_dtype, kv_dtype, num_seqs, num_kv_heads, num_q_heads / num_kv_heads,
                     head_dim, block_size, max_context_len, partition_size, &order_seqs);
    return order_seqs && num_seqs > 0 ? 1 : 0;
}

int32_t pa_chunk_partition_tokens(pa_dtype kv_dtype, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t max_query_len, int32_t max_context_len,
                                  int32_t partition_size)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 128 ||
        max_context_len < 0 || max_query_len < 0)
        return PA_ERR_INVALID;
    if (partition_size > 0 && partition_size % 64 != 0)
        return PA_ERR_INVALID;
    if (partition_size == 0 && device_sm_count() <= 0)
        return PA_ERR_CUDA;
    return chunk_plan(kv_dtype == PA_FP8_E4M3 ? PA_BF16 : kv_dtype, kv_dtype, num_seqs,
                      num_q_heads, num_kv_heads, head_dim, block_size, max_query_len,
                      max_context_len, partition_size)
        .partition;
}

int pa_test_arm_wait_timeout(int32_t cta_index, uint32_t wait_limit_us)
{
    if (cta_index < 0 || cta_index == INT32_MAX || wait_limit_us < 1 || wait_limit_us > 1000000)
        return PA_ERR_INVALID;
    g_fault_cta = cta_index + 1;
    g_fault_wait_ns = wait_limit_us * 1000u;
    return PA_OK;
}

const char* pa_decode_kernel_name(pa_dtype kv_dtype, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim)
{
    if (!(valid_dtype(kv_dtype) || kv_dtype == PA_FP8_E4M3) || num_q_heads <= 0 ||
        num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        !(head_dim == 64 || head_dim == 128))
        return nullptr;
    switch (decode_kernel_for(kv_dtype, head_dim, heads_per_cta(num_q_heads / num_kv_heads))) {
    case DecodeKernel::kTc8: return "decode_tc8_kernel";
    case DecodeKernel::kMmaSync: return "decode_mma_kernel";
    default: return "decode_kernel";
    }
}

const char* pa_chunk_kernel_name(pa_dtype kv_dtype, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_query_len)
{
    if (!(kv_dtype == PA_F16 || kv_dtype == PA_BF16 || kv_dtype == PA_FP8_E4M3) ||
        num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        num_q_heads / num_kv_heads > 128 || !(head_dim == 64 || head_dim == 128) ||
        max_query_len <= 0)
        return nullptr;
    // the route does not depend on the split: a never-split plan needs no device query
    const ChunkPlan plan = chunk_plan(kv_dtype == PA_FP8_E4M3 ? PA_BF16 : kv_dtype, kv_dtype, 1,
                                      num_q_heads, num_kv_heads, head_dim, 16, max_query_len,
                                      max_query_len, -1);
    if (plan.rows_path)
        return kv_dtype == PA_FP8_E4M3 && use_tc8(head_dim, plan.nh)
                   ? "decode_tc8_kernel (chunk rows)"
                   : "decode_mma_kernel (chunk rows)";
    return kv_dtype == PA_FP8_E4M3 ? "chunk_attn_kernel (E4M3 tiles converted to f16)"
                                   : "chunk_attn_kernel";
}

size_t pa_chunk_workspace_bytes(int64_t num_query_tokens, int32_t num_q_heads, int32_t head_dim,
                                int32_t max_context_len, int32_t partition_size)
{
    if (num_query_tokens < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        partition_size < 0)
        return 0;
    const int P = partition_size > 0 ? partition_size : kAutoPartitionTokens;
    if (max_context_len <= P)
        return 0;
    const int max_parts = (max_context_len + P - 1) / P;
    return workspace_layout(num_query_tokens * num_q_heads, max_parts, head_dim, nullptr);
}

// Shared body of pa_chunk_attention and pa_chunk_attention_fp8: q_dtype is the type of
// q (and of a native out), kv_dtype the cache's (PA_FP8_E4M3 with k_scale / v_scale).
static int chunk_impl(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                      const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                      const float* k_scale, const float* v_scale, int64_t num_blocks,
                      const int32_t* block_tables, int64_t block_table_stride,
                      const int32_t* context_lens, const int32_t* query_start,
                      int64_t num_query_tokens, int32_t max_query_len, int32_t max_context_len,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, float scale, int32_t partition_size,
                      void* workspace, size_t workspace_bytes, void* stream)
{
    const bool fp8 = kv_dtype == PA_FP8_E4M3;
    if (!(q_dtype == PA_F16 || q_dtype == PA_BF16)) {
        return (q_dtype == PA_F32 || q_dtype == PA_FP8_E4M3) ? PA_ERR_UNSUPPORTED
                                                             : PA_ERR_INVALID;
    }
    if (!(out_dtype == PA_F32 || out_dtype == q_dtype))
        return PA_ERR_INVALID;
    if (fp8 && (!k_scale || !v_scale))
        return PA_ERR_INVALID;
    if (num_seqs < 0 || num_seqs > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 128)
        return PA_ERR_INVALID;
    if (!(head_dim == 64 || head_dim == 128) || !(block_size == 16 || block_size == 32))
        return PA_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_table_stride <= 0 ||
        max_context_len < 0 || (int64_t)max_context_len > block_table_stride * block_size ||
        max_query_len < 0 || max_query_len > max_context_len || num_query_tokens < 0 ||
        num_query_tokens > INT32_MAX || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (partition_size > 0 && partition_size % 64 != 0)
        return PA_ERR_INVALID;
    if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return PA_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID;
    const int group = num_q_heads / num_kv_heads;
    const ChunkPlan plan = chunk_plan(q_dtype, kv_dtype, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, max_query_len, max_context_len,
                                      partition_size);
    if ((int64_t)num_kv_heads * plan.chunks > 65535)
        return PA_ERR_INVALID;
    const size_t row_elems = (size_t)num_query_tokens * num_q_heads * head_dim;
    const size_t q_bytes = row_elems * elem_size(q_dtype);
    const size_t out_bytes = row_elems * elem_size(out_dtype);
    const size_t pool_bytes =
        (size_t)num_blocks * num_kv_heads * block_size * head_dim * elem_size(kv_dtype);
    if (overlaps(out, out_bytes, q, q_bytes) || overlaps(out, out_bytes, k_cache, pool_bytes) ||
        overlaps(out, out_bytes, v_cache, pool_bytes))
        return PA_ERR_INVALID;
    const std::initializer_list<Span> inputs = {
        {out, out_bytes}, {q, q_bytes}, {k_cache, pool_bytes}, {v_cache, pool_bytes},
        {block_tables, (size_t)num_seqs * (size_t)block_table_stride * 4},
        {context_lens, (size_t)num_seqs * 4}, {query_start, (size_t)(num_seqs + 1) * 4}};

    const int P = plan.partition;
    ChunkParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = query_start;
    p.num_blocks = num_blocks;
    p.bt_stride = block_table_stride;
    p.num_rows = num_query_tokens;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.rows_tokens = plan.rows_tokens;
    p.m_tiles = plan.chunks;
    p.max_query_len = max_query_len;
    p.max_context_len = max_context_len;
    p.partition_tokens = P;
    p.max_parts = 1;
    p.out_f32 = out_dtype == PA_F32 ? 1 : 0;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);  // log2(e)
    if (P > 0) {
        p.max_parts = (max_context_len + P - 1) / P;
        size_t ml_off = 0;
        const size_t need = workspace_layout(num_query_tokens * num_q_heads, p.max_parts,
                                             head_dim, &ml_off);
        if (!workspace || workspace_bytes < need || !aligned16(workspace))
            return PA_ERR_WORKSPACE;
        if (overlaps_any(workspace, need, inputs))
            return PA_ERR_INVALID;
        p.part_o = static_cast<float*>(workspace);
        p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off);
    }
    p.k_scale = fp8 ? k_scale : nullptr;
    p.v_scale = fp8 ? v_scale : nullptr;
    p.err = device_error_word();
    if (!p.err)
        return PA_ERR_CUDA;
    CUtensorMap tk{}, tv{};
    cudaError_t e = cudaSuccess;
    if (!fp8 || head_dim == 128) {               // E4M3 at head_dim 64 moves by 1-D bulk copies
        e = kv_tensor_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim, kv_dtype);
        if (e == cudaSuccess)
            e = kv_tensor_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim,
                              kv_dtype);
    }
    if (e == cudaErrorInvalidValue)
        return PA_ERR_INVALID;
    if (e != cudaSuccess)
        return PA_ERR_CUDA;
    if (plan.rows_path) {
        DecodeParams d{};
        d.out = out;
        d.q = q;
        d.k_cache = k_cache;
        d.v_cache = v_cache;
        d.block_tables = block_tables;
        d.context_lens = context_lens;
        d.part_o = p.part_o;
        d.part_ml = p.part_ml;
        d.err = p.err;
        d.num_blocks = num_blocks;
        d.bt_stride = block_table_stride;
        d.num_seqs = num_seqs;
        d.num_q_heads = num_q_heads;
        d.num_kv_heads = num_kv_heads;
        d.group = group;
        d.chunks = plan.chunks;
        d.max_context_len = max_context_len;
        d.partition_tokens = P;
        d.max_parts = p.max_parts;
        d.out_f32 = p.out_f32;
        d.scale_log2 = p.scale_log2;
        d.query_start = query_start;
        d.num_rows = num_query_tokens;
        d.max_query_len = max_query_len;
        d.k_scale = fp8 ? k_scale : nullptr;
        d.v_scale = fp8 ? v_scale : nullptr;
        e = fp8 ? launch_chunk_rows_fp8(d, p, q_dtype, head_dim, block_size, plan.nh, tk, tv,
                                        static_cast<cudaStream_t>(stream))
                : launch_chunk_rows(d, p, kv_dtype, head_dim, block_size, plan.nh, tk, tv,
                                    static_cast<cudaStream_t>(stream));
    } else if (fp8) {
        e = launch_chunk_attention_fp8(p, q_dtype, block_size, tk, tv,
                                       static_cast<cudaStream_t>(stream));
    } else {
        e = launch_chunk_attention(p, kv_dtype, head_dim, block_size, tk, tv,
                                   static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_chunk_attention(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                       const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                       const int32_t* block_tables, int64_t block_table_stride,
                       const int32_t* context_lens, const int32_t* query_start,
                       int64_t num_query_tokens, int32_t max_query_len, int32_t max_context_len,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, float scale, int32_t partition_size,
                       void* workspace, size_t workspace_bytes, void* stream)
{
    if (kv_dtype == PA_FP8_E4M3)
        return PA_ERR_UNSUPPORTED;               // E4M3 caches: pa_chunk_attention_fp8
    return chunk_impl(out, out_dtype, q, kv_dtype, k_cache, v_cache, kv_dtype, nullptr, nullptr,
                      num_blocks, block_tables, block_table_stride, context_lens, query_start,
                      num_query_tokens, max_query_len, max_context_len, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, scale, partition_size, workspace,
                      workspace_bytes, stream);
}

int pa_chunk_attention_fp8(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                           const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, int64_t num_blocks, const int32_t* block_tables,
                           int64_t block_table_stride, const int32_t* context_lens,
                           const int32_t* query_start, int64_t num_query_tokens,
                           int32_t max_query_len, int32_t max_context_len, int32_t num_seqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, float scale, int32_t partition_size,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    return chunk_impl(out, out_dtype, q, q_dtype, k_cache, v_cache, PA_FP8_E4M3, k_scale, v_scale,
                      num_blocks, block_tables, block_table_stride, context_lens, query_start,
                      num_query_tokens, max_query_len, max_context_len, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, block_size, scale, partition_size, workspace,
                      workspace_bytes, stream);
}

int pa_reshape_and_cache_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_cache,
                             void* v_cache, const float* k_scale, const float* v_scale,
                             const int64_t* slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, void* stream)
{
    if (!valid_dtype(src_dtype) || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID;
    if (head_dim % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
        return PA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID;
    const size_t pool_bytes = (size_t)num_blocks * num_kv_heads * block_size * head_dim;
    if (overlaps(k_cache, pool_bytes, v_cache, pool_bytes))
        return PA_ERR_INVALID;
    ReshapeFp8Params p{};
    p.k = k;
    p.v = v;
    p.k_cache = static_cast<unsigned char*>(k_cache);
    p.v_cache = static_cast<unsigned char*>(v_cache);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.slot_mapping = slot_mapping;
    p.err = device_error_word();
    if (!p.err)
        return PA_ERR_CUDA;
    p.num_tokens = num_tokens;
    p.num_blocks = num_blocks;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    return launch_reshape_and_cache_fp8(p, src_dtype, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         pa_dtype dtype, void* stream)
{
    if (!valid_dtype(dtype) || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID;
    const size_t row_bytes = (size_t)head_dim * elem_size(dtype);
    if (row_bytes % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return PA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID;
    const size_t pool_bytes = (size_t)num_blocks * num_kv_heads * block_size * row_bytes;
    if (overlaps(k_cache, pool_bytes, v_cache, pool_bytes))
        return PA_ERR_INVALID;
    ReshapeParams p{};
    p.k = static_cast<const uint4*>(k);
    p.v = static_cast<const uint4*>(v);
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.slot_mapping = slot_mapping;
    p.err = device_error_word();
    if (!p.err)
        return PA_ERR_CUDA;
    p.num_tokens = num_tokens;
    p.num_blocks = num_blocks;
    p.num_kv_heads = num_kv_heads;
    p.row_vecs = (int)(row_bytes / 16);
    p.block_size = block_size;
    return launch_reshape_and_cache(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                   const int64_t* src_dst_pairs_host, int64_t num_pairs, int64_t block_bytes,
                   int64_t num_blocks, void* stream)
{
    if (num_layers < 0 || num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 != 0 ||
        num_blocks <= 0 || num_blocks > INT32_MAX)
        return PA_ERR_INVALID;
    if (num_layers == 0 || num_pairs == 0)
        return PA_OK;
    if (!k_caches || !v_caches || !src_dst_pairs_host)
        return PA_ERR_INVALID;
    for (int l = 0; l < num_layers; ++l)
        if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
            return PA_ERR_INVALID;
    std::vector<int64_t> dst(num_pairs), src(num_pairs);
    for (int64_t i = 0; i < num_pairs; ++i) {
        src[i] = src_dst_pairs_host[2 * i];
        dst[i] = src_dst_pairs_host[2 * i + 1];
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks)
            return PA_ERR_INVALID;
    }
    std::sort(dst.begin(), dst.end());
    if (std::adjacent_find(dst.begin(), dst.end()) != dst.end())
        return PA_ERR_INVALID;                       // two pairs write one block
    for (int64_t s : src)
        if (std::binary_search(dst.begin(), dst.end(), s))
            return PA_ERR_INVALID;                   // a destination is also a source

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int l0 = 0; l0 < num_layers; l0 += kCopyMaxLayers) {
        for (int64_t p0 = 0; p0 < num_pairs; p0 += kCopyMaxPairs) {
            CopyParams p{};
            p.num_layers = std::min<int>(kCopyMaxLayers, num_layers - l0);
            p.num_pairs = (int)std::min<int64_t>(kCopyMaxPairs, num_pairs - p0);
            p.block_vecs = block_bytes / 16;
            for (int l = 0; l < p.num_layers; ++l) {
                p.k[l] = static_cast<uint4*>(k_caches[l0 + l]);
                p.v[l] = static_cast<uint4*>(v_caches[l0 + l]);
            }
            for (int i = 0; i < p.num_pairs; ++i)
                p.pairs[i] = make_int2((int)src_dst_pairs_host[2 * (p0 + i)],
                                       (int)src_dst_pairs_host[2 * (p0 + i) + 1]);
            if (launch_copy_blocks(p, st) != cudaSuccess)
                return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}

int pa_swap_blocks(void* const* src_caches, void* const* dst_caches, int32_t num_caches,
                   const int64_t* src_dst_pairs_host, int64_t num_pairs, int64_t block_bytes,
                   int64_t src_num_blocks, int64_t dst_num_blocks, void* stream)
{
    if (num_caches < 0 || num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 != 0 ||
        src_num_blocks <= 0 || src_num_blocks > INT32_MAX || dst_num_blocks <= 0 ||
        dst_num_blocks > INT32_MAX)
        return PA_ERR_INVALID;
    if (num_caches == 0 || num_pairs == 0)
        return PA_OK;
    if (!src_caches || !dst_caches || !src_dst_pairs_host)
        return PA_ERR_INVALID;
    std::vector<int64_t> dst(num_pairs);
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t s = src_dst_pairs_host[2 * i], d = src_dst_pairs_host[2 * i + 1];
        if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks)
            return PA_ERR_INVALID;
        dst[i] = d;
    }
    std::sort(dst.begin(), dst.end());
    if (std::adjacent_find(dst.begin(), dst.end()) != dst.end())
        return PA_ERR_INVALID;                       // two pairs write one block
    const size_t src_bytes = (size_t)src_num_blocks * block_bytes;
    const size_t dst_bytes = (size_t)dst_num_blocks * block_bytes;
    std::vector<const uint4*> srcp(num_caches);
    std::vector<uint4*> dstp(num_caches);
    for (int c = 0; c < num_caches; ++c) {
        void* pools[2] = {src_caches[c], dst_caches[c]};
        if (!pools[0] || !pools[1] || !aligned16(pools[0]) || !aligned16(pools[1]) ||
            overlaps(pools[0], src_bytes, pools[1], dst_bytes))
            return PA_ERR_INVALID;
        void* dev[2] = {nullptr, nullptr};
        for (int k = 0; k < 2; ++k) {
            // device memory, or pinned host memory the device can address
            cudaPointerAttributes a{};
            if (cudaPointerGetAttributes(&a, pools[k]) != cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_INVALID;
            }
            if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeHost &&
                a.type != cudaMemoryTypeManaged)
                return PA_ERR_INVALID;
            dev[k] = a.devicePointer ? a.devicePointer : pools[k];
        }
        srcp[c] = static_cast<const uint4*>(dev[0]);
        dstp[c] = static_cast<uint4*>(dev[1]);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SwapParams p{};
    for (int c0 = 0; c0 < num_caches; c0 += kSwapMaxCaches) {
        for (int64_t p0 = 0; p0 < num_pairs; p0 += kSwapMaxPairs) {
            p.num_caches = std::min<int>(kSwapMaxCaches, num_caches - c0);
            p.num_pairs = (int)std::min<int64_t>(kSwapMaxPairs, num_pairs - p0);
            p.block_vecs = block_bytes / 16;
            for (int c = 0; c < p.num_caches; ++c) {
                p.src[c] = srcp[c0 + c];
                p.dst[c] = dstp[c0 + c];
            }
            for (int i = 0; i < p.num_pairs; ++i)
                p.pairs[i] = make_int2((int)src_dst_pairs_host[2 * (p0 + i)],
                                       (int)src_dst_pairs_host[2 * (p0 + i) + 1]);
            if (launch_swap_blocks(p, st) != cudaSuccess)
                return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}

int pa_get_device_error(uint32_t* flags, void* stream)
{
    if (!flags)
        return PA_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned value = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbolAsync(&value, g_device_error, sizeof value, 0,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PA_ERR_CUDA;
    *flags = value;
    return PA_OK;
}

}  // extern "C"
