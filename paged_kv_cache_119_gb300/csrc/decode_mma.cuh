// decode_mma.cuh -- paged decode attention for grouped-query heads on the tensor
// cores (sm_103a), over fp16/bf16 caches and E4M3 caches (codes converted exactly to
// the 16-bit operand type).
//
// Same result as decode_kernel (the block-wise attention of "PagedAttention
// 完全拆解", section 原理详解（二）, evaluated with a running max), organised for
// GQA: one CTA serves NH (4 or 8) query heads that share a kv head, so a K/V tile
// is read once for all of them and q.K^T, P.V become small dense contractions
// (4 multiply-adds per K/V byte at group 8, more than the CUDA cores sustain at
// HBM speed).
//
//   * Producer warp: per tile, D/64 tensor-map TMA copies of K and of V
//     (cp.async.bulk.tensor, box = 64 dims x B tokens, 128-byte swizzle) into an
//     mbarrier ring; the tensor map's third coordinate is block * Hkv + kv head,
//     so the block-table entry is the only address input.
//   * Consumer warps (tile i -> warp i % 4, each stage owned by one warp):
//       S^T[16 tok x 8 heads] = K[16 x D] . Q^T  -- mma.sync m16n8k16, K from
//         ldmatrix on the swizzled tile, Q^T fragments held in registers;
//       running max / sum per head in fp32 (base 2); the accumulator is rescaled
//         only when some head's max rose (a warp vote);
//       P^T is split into hi + lo halves of the cache dtype (P = hi + lo to
//         ~2^-16 relative), and each 8x8 block is transposed in registers with
//         movmatrix into the B operand of the second product;
//       O^T[D x 8 heads] += V^T . P^T  -- mma.sync, V^T from ldmatrix.trans.
//   * Tokens past the context in the last tile: scores become -inf by select,
//     and their V fragments are zeroed before the product (unused slots may
//     hold NaN, and 0 * NaN is NaN).
//   * Warps merge through shared memory (reusing the ring) in a fixed order.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode_kernel.cuh"

namespace pa {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // packs (lo, hi) into one 32-bit register, rounding to nearest even
    __device__ __forceinline__ static uint32_t pack(float lo, float hi)
    {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w)
    {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
    }
};

template <>
struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi)
    {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w)
    {
        return __half22float2(*reinterpret_cast<__half2*>(&w));
    }
};

// Converts one raw E4M3 tile [B][D] (row-major bytes) into the 128-byte-swizzled
// 16-bit layout the tensor-map TMA produces: D/64 regions of B rows x 128 bytes,
// the 16-byte chunk j of row r stored at chunk position j ^ (r & 7).  One lane per
// 64-element half row; E4M3 -> f16 is exact and so is f16 -> bf16 for these values.
template <typename T, int D, int BS>
__device__ __forceinline__ void convert_e4m3_tile(const unsigned char* src, unsigned char* dst,
                                                  int lane)
{
    constexpr int HALVES = D / 64;
#pragma unroll
    for (int hr = lane; hr < BS * HALVES; hr += 32) {
        const int r = hr / HALVES;
        const int h = hr - r * HALVES;
        const uint4* in = reinterpret_cast<const uint4*>(src + r * D + h * 64);
        unsigned char* out_row = dst + h * (BS * 128) + r * 128;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            const uint4 w = in[q];                         // 16 codes -> chunks 2q, 2q+1
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {                  // 2 codes per packed 32-bit word
                const __half2_raw hv =
                    __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(words[i / 2] >> (16 * (i % 2))),
                                               __NV_E4M3);
                if constexpr (DType<T>::id == PA_F16) {
                    packed[i] = *reinterpret_cast<const uint32_t*>(&hv);
                } else {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv));
                    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
                    packed[i] = *reinterpret_cast<const uint32_t*>(&b);
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int j = 2 * q + k;
                *reinterpret_cast<uint4*>(out_row + ((j ^ (r & 7)) << 4)) =
                    make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
            }
        }
    }
}

// Shared memory of the tensor-core kernel.  16-bit caches: the ring holds the
// swizzled K and V tiles the tensor-map TMA writes.  E4M3 caches: the ring holds
// the raw one-byte tiles (1-D bulk copies) and each consumer warp owns a staging
// pair of 16-bit swizzled tiles, in the same layout, that it converts them into.
template <typename TK, int D, int BS, int NSTAGE>
struct MmaSmem {
    static constexpr bool kFp8 = sizeof(TK) == 1;
    // E4M3 with head_dim 128: a tile row is 128 bytes, so the raw tile arrives by
    // tensor-map TMA with 128-byte swizzle and fragments are read from it directly
    static constexpr bool kDirect = kFp8 && D == 128;
    static constexpr int kHalfBytes = BS * 128;                // one 64-dim box: B rows x 128 B
    static constexpr int kTileBytes = (D / 64) * kHalfBytes;   // one 16-bit K (or V) tile
    static constexpr int kScratchBytes =
        (kFp8 && !kDirect) ? kDecodeConsumerWarps * 2 * kTileBytes : 0;
    static constexpr int kFp8TileBytes = BS * D;               // one E4M3 K (or V) tile
    static constexpr int kStageBytes = kFp8 ? 2 * kFp8TileBytes : 2 * kTileBytes;
    static constexpr int kRingOffset = kScratchBytes;
    static constexpr int kRingBytes = NSTAGE * kStageBytes;
    static constexpr int kBarOffset = kRingOffset + kRingBytes;
    static constexpr int kOkOffset = kBarOffset + 2 * NSTAGE * 8;
    static constexpr int kFlagOffset = kOkOffset + NSTAGE * 4;
    static constexpr int kBytes = kFlagOffset + 16;
    static constexpr int kAlloc = kBytes + 1024;                 // room to align the ring to 1 KB
    // merge area at offset 0 (the ring, or the staging tiles), reused once every tile
    // is consumed
    static constexpr int kMergeAcc = kDecodeConsumerWarps * 8 * D * 4;
    static constexpr int kMergeBytes = kMergeAcc + kDecodeConsumerWarps * 8 * 2 * 4;
    static_assert(kMergeBytes <= ((kFp8 && !kDirect) ? kScratchBytes : kRingBytes),
                  "merge area must fit");
    static_assert(kHalfBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

// Four CTAs per SM (at most 96 registers a thread) keep the 16-bit and block-size-16
// E4M3 forms resident; the block-size-32 E4M3 form converts wider tiles and runs
// faster at 128 registers and three CTAs.
template <typename TK, int BS>
constexpr int mma_min_blocks() { return (sizeof(TK) == 1 && BS == 32) ? 3 : 4; }

// T: query / native output type (the mma operand type).  TK: cache element type,
// T itself (tiles by tensor-map TMA) or __nv_fp8_e4m3 (raw tiles by 1-D bulk copy,
// converted exactly to T in shared memory; the value is code * per-kv-head scale).
// CH (chunk rows): the NH B-operand columns are rows R0 .. R0+NH-1 of the
// (chunk token, query head) rows of one kv head -- several new query tokens of a
// sequence attended causally, each row masked at its own position (speculative
// verification, short chunks) -- instead of NH query heads of one token.
// BPT: cache blocks per tile (a ring stage); the tile is TB = BS * BPT tokens.
template <typename T, typename TK, int D, int BS, int NH, int NSTAGE, bool CH = false, int BPT = 1>
__global__ void __launch_bounds__(kDecodeThreads, mma_min_blocks<TK, BS * BPT>())
    decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv)
{
    constexpr int TB = BS * BPT;      // tokens per tile
    using Sm = MmaSmem<TK, D, TB, NSTAGE>;
    constexpr bool kFp8 = Sm::kFp8;
    // tensor-core operand type: the query type for 16-bit caches; f16 for E4M3 caches
    // (an E4M3 code converts to f16 exactly in one instruction per pair)
    using TM = std::conditional_t<kFp8, __half, T>;
    constexpr bool kDirect = Sm::kDirect;
    constexpr int NCW = kDecodeConsumerWarps;
    constexpr int KS = D / 16;        // k-steps of the score product / m-blocks of P.V
    constexpr int MB = TB / 16;       // 16-token row blocks per tile
    static_assert(BPT == 1 || (BPT == 2 && Sm::kDirect), "two blocks per tile: direct E4M3 tiles");
    static_assert(NH == 1 || NH == 2 || NH == 4 || NH == 8, "1, 2, 4 or 8 query heads per CTA");
    static_assert(NSTAGE % NCW == 0, "each ring stage must belong to one consumer warp");
    static_assert(BS % 16 == 0 && D % 64 == 0, "block_size 16/32, head_dim 64/128");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOffset);
    uint64_t* empty = full + NSTAGE;
    int* stage_ok = reinterpret_cast<int*>(smem + Sm::kOkOffset);
    int* poison = reinterpret_cast<int*>(smem + Sm::kFlagOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y / p.chunks;
    const int h0 = kvh * p.group + (blockIdx.y % p.chunks) * NH;
    const int part = blockIdx.x;
    const bool split = p.partition_tokens > 0;

    const int L = p.context_lens[seq];
    // chunk rows: the sequence's rows of q / out are query_start[seq] .. + n - 1
    int qs0 = 0, n = 1, R0 = 0;
    if constexpr (CH) {
        qs0 = p.query_start[seq];
        n = p.query_start[seq + 1] - qs0;
        R0 = (blockIdx.y % p.chunks) * NH;
    }
    const bool rows_sane = !CH || (qs0 >= 0 && n >= 0 && (int64_t)qs0 + n <= p.num_rows);
    if (L < 0 || L > p.max_context_len || !rows_sane ||
        (CH && (n > L || n > p.max_query_len))) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);
        if (!split && rows_sane) {
            for (int idx = threadIdx.x; idx < NH * D; idx += blockDim.x) {
                if constexpr (CH) {
                    const int R = R0 + idx / D;
                    const int j = R / p.group;
                    if (j < n)
                        store_out<T>(p, ((int64_t)(qs0 + j) * p.num_q_heads + kvh * p.group +
                                         (R - j * p.group)) * D + idx % D,
                                     __int_as_float(0x7fc00000));
                } else {
                    store_out<T>(p, ((int64_t)seq * p.num_q_heads + h0) * D + idx,
                                 __int_as_float(0x7fc00000));
                }
            }
        }
        return;
    }
    int t_end = L;
    if constexpr (CH) {
        if (seq == p.num_seqs - 1 && part == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
            (int64_t)qs0 + n != p.num_rows)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);   // rows after the last chunk belong to no one
        if (R0 / p.group >= n)
            return;                                // no chunk token in this row chunk
        t_end = L - n + min(n - 1, (R0 + NH - 1) / p.group) + 1;   // last row's position + 1
    }
    int t0 = 0, t1 = t_end;
    if (split) {
        t0 = part * p.partition_tokens;
        if (t0 >= t_end)
            return;
        t1 = min(t_end, t0 + p.partition_tokens);
    }
    const int jb = t0 / BS;                       // first cache block (partitions start on one)
    const int nblk = (t1 > t0) ? (t1 + BS - 1) / BS - jb : 0;
    const int ntiles = (nblk + BPT - 1) / BPT;    // tile it: blocks jb + BPT it .. + BPT - 1

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *poison = 0;
        fence_mbar_init();
    }
    if ((!kFp8 || kDirect) && warp == NCW && lane == 0) {
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------------------------ producer
        const int32_t* bt_row = p.block_tables + (int64_t)seq * p.bt_stride + jb;
        const uint64_t policy = l2_evict_first_policy();
        int next = (lane < nblk) ? __ldg(bt_row + lane) : 0;
        bool aborted = false;
        // block-table entries 32 at a time (BPT divides 32, so no tile straddles two
        // batches), the next 32 in flight while the current ones are used
        for (int base = 0; base < nblk && !aborted; base += 32) {
            const int cur = next;
            if (base + 32 + lane < nblk)
                next = __ldg(bt_row + base + 32 + lane);
            const int cnt = min(32, nblk - base);
            for (int i = 0; i < cnt; i += BPT) {
                int pbn[BPT];
#pragma unroll
                for (int b = 0; b < BPT; ++b)
                    pbn[b] = __shfl_sync(kFullMask, cur, i + b);   // i + b <= 31
                const int nb = min(BPT, cnt - i);                  // blocks of the tile in range
                const int it = (base + i) / BPT;
                const int stage = it % NSTAGE;
                int ok = 1;
                if (lane == 0) {
                    if (it >= NSTAGE && !mbar_wait(&empty[stage], ((it / NSTAGE) - 1) & 1)) {
                        atomicOr(p.err, PA_DEVERR_TIMEOUT);
                        ok = 0;
                    }
                    if (ok) {
                        bool all_valid = true;
                        uint32_t tx = 0;
#pragma unroll
                        for (int b = 0; b < BPT; ++b) {
                            const bool valid = b < nb && pbn[b] >= 0 && (int64_t)pbn[b] < p.num_blocks;
                            all_valid = all_valid && (b >= nb || valid);
                            tx += valid ? 2u * (kFp8 ? BS * D : BS * D * 2) : 0u;
                        }
                        stage_ok[stage] = all_valid ? 1 : 0;
                        if (!all_valid)
                            atomicOr(p.err, PA_DEVERR_BLOCK_ID);
                        if (tx == 0) {
                            mbar_arrive(&full[stage]);
                        } else {
                            unsigned char* dst = smem + Sm::kRingOffset + stage * Sm::kStageBytes;
                            mbar_arrive_expect_tx(&full[stage], tx);
#pragma unroll
                            for (int b = 0; b < BPT; ++b) {
                                if (b >= nb || pbn[b] < 0 || (int64_t)pbn[b] >= p.num_blocks)
                                    continue;
                                unsigned char* bdst = dst + b * (BS * 128);   // rows of block b
                                if constexpr (kDirect) {
                                    const int z = pbn[b] * p.num_kv_heads + kvh;
                                    tma_load_3d(bdst, &tk, 0, 0, z, &full[stage], policy);
                                    tma_load_3d(bdst + Sm::kFp8TileBytes, &tv, 0, 0, z, &full[stage],
                                                policy);
                                } else if constexpr (kFp8) {
                                    const int64_t off =
                                        ((int64_t)pbn[b] * p.num_kv_heads + kvh) * Sm::kFp8TileBytes;
                                    bulk_g2s(dst, reinterpret_cast<const unsigned char*>(p.k_cache) + off,
                                             Sm::kFp8TileBytes, &full[stage], policy);
                                    bulk_g2s(dst + Sm::kFp8TileBytes,
                                             reinterpret_cast<const unsigned char*>(p.v_cache) + off,
                                             Sm::kFp8TileBytes, &full[stage], policy);
                                } else {
                                    const int z = pbn[b] * p.num_kv_heads + kvh;   // < 2^31 (checked on the host)
#pragma unroll
                                    for (int h = 0; h < D / 64; ++h) {
                                        tma_load_3d(bdst + h * Sm::kHalfBytes, &tk, 64 * h, 0, z,
                                                    &full[stage], policy);
                                        tma_load_3d(bdst + Sm::kTileBytes + h * Sm::kHalfBytes, &tv,
                                                    64 * h, 0, z, &full[stage], policy);
                                    }
                                }
                            }
                        }
                    }
                }
                if (!__shfl_sync(kFullMask, ok, 0)) {
                    aborted = true;
                    break;
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------------- consumers
    const int g = lane >> 2;          // fragment row group
    const int c = lane & 3;           // fragment column pair
    // Q^T fragments: b0 = q[head g][16ks + 2c, +1], b1 = q[head g][16ks + 2c + 8, +9]
    uint32_t qb[KS][2];
    float q_unscale = 1.f;            // for E4M3 caches: q was scaled by 2^-e to fit f16
    {
        bool live = g < NH;
        int64_t qr = (int64_t)seq * p.num_q_heads + h0 + (live ? g : 0);
        if constexpr (CH) {
            const int R = R0 + g;
            const int j = R / p.group;
            live = live && j < n;
            qr = live ? (int64_t)(qs0 + j) * p.num_q_heads + kvh * p.group + (R - j * p.group) : 0;
        }
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(p.q) + qr * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            // k-indices 2c, 2c+1 | 2c+8, 2c+9 of step ks are head dims 16ks + 2c.. | +8..,
            // or, reading E4M3 bytes directly, 16ks + 4c, +1 | +2, +3 (the same
            // permutation of the summed dimension is applied to K)
            const int d0 = kDirect ? 16 * ks + 4 * c : 16 * ks + 2 * c;
            const int d1 = kDirect ? d0 + 2 : d0 + 8;
            qb[ks][0] = live ? __ldg(qrow + d0 / 2) : 0u;
            qb[ks][1] = live ? __ldg(qrow + d1 / 2) : 0u;
        }
        if constexpr (kFp8 && !std::is_same_v<T, __half>) {
            // bf16 queries become f16 operands: scale by a power of two 2^-e so that the
            // largest |q| of the CTA's heads stays below 2^15 (no overflow; the scaling
            // is exact), and fold 2^e back into the scores
            float amax = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 f = Mma<T>::unpack(qb[ks][j]);
                    amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
#pragma unroll
            for (int msk = 16; msk >= 1; msk >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, msk));
            int e = 0;
            if (amax >= 32768.f)
                e = ((__float_as_int(amax) >> 23) & 0xff) - 127 - 14;   // 2^-e * amax < 2^15
            const float down = __int_as_float((127 - e) << 23);
            q_unscale = __int_as_float((127 + e) << 23);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 f = Mma<T>::unpack(qb[ks][j]);
                    qb[ks][j] = Mma<__half>::pack(f.x * down, f.y * down);
                }
        }
    }
    // per-thread statistics for heads 2c and 2c+1 (base-2 units)
    float m[2] = {-INFINITY, -INFINITY};
    float lsum[2] = {0.f, 0.f};
    float o[KS][4];                   // O^T fragments: (d = 16mb + g (+8), heads 2c, 2c+1)
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[i][j] = 0.f;
    bool poisoned = false;
    // scores carry the softmax scale (base 2) and, for a quantised cache, the K scale
    const float sl2 = kFp8 ? p.scale_log2 * p.k_scale[kvh] * q_unscale : p.scale_log2;
    // chunk rows: the last visible position of rows 2c and 2c+1 (-1: padding row)
    int lim[2] = {0, 0};
    if constexpr (CH) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int R = R0 + 2 * c + j;
            const int tk = R / p.group;
            lim[j] = (2 * c + j < NH && tk < n) ? L - n + tk : -1;
        }
    }

    for (int it = warp; it < ntiles; it += NCW) {
        const int stage = it % NSTAGE;
        if (!mbar_wait(&full[stage], (it / NSTAGE) & 1)) {
            if (lane == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            poisoned = true;
            break;
        }
        if (!stage_ok[stage]) {
            poisoned = true;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
            continue;
        }
        uint32_t kbase, vbase;
        if constexpr (kDirect) {
            kbase = smem_addr(smem + Sm::kRingOffset + stage * Sm::kStageBytes);
            vbase = kbase + Sm::kFp8TileBytes;
        } else if constexpr (kFp8) {
            // convert the raw tiles into this warp's swizzled 16-bit staging tiles
            // (E4M3 -> T is exact), then hand the stage back to the producer
            unsigned char* stg = smem + warp * 2 * Sm::kTileBytes;
            const unsigned char* raw = smem + Sm::kRingOffset + stage * Sm::kStageBytes;
            __syncwarp();                      // the previous tile's ldmatrix reads are done
            convert_e4m3_tile<TM, D, TB>(raw, stg, lane);
            convert_e4m3_tile<TM, D, TB>(raw + Sm::kFp8TileBytes, stg + Sm::kTileBytes, lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
            kbase = smem_addr(stg);
            vbase = kbase + Sm::kTileBytes;
        } else {
            kbase = smem_addr(smem + stage * Sm::kStageBytes);
            vbase = kbase + Sm::kTileBytes;
        }
        const int nvalid = min(TB, t1 - (jb * BS + it * TB));

#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
            if (16 * mb >= nvalid)
                break;                         // the rest of the tile lies past the context
            // ---- S^T = K . Q^T for tokens 16mb .. 16mb+15
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (kDirect) {
                // rows 16mb+g and +8; the 4 codes at head dims 16ks + 4c .. +3 of a row
                // (16-byte chunk ks, swizzled by row) give a0 / a2 (and a1 / a3)
                const int r0 = 16 * mb + g, r1 = r0 + 8;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const uint32_t w0 = lds_u32(kbase + r0 * 128 + ((ks ^ (r0 & 7)) << 4) + 4 * c);
                    const uint32_t w1 = lds_u32(kbase + r1 * 128 + ((ks ^ (r1 & 7)) << 4) + 4 * c);
                    const uint32_t a[4] = {e4m3x2_to_f16x2(w0), e4m3x2_to_f16x2(w1),
                                           e4m3x2_to_f16x2(w0 >> 16), e4m3x2_to_f16x2(w1 >> 16)};
                    Mma<TM>::run(s, a, qb[ks][0], qb[ks][1]);
                }
            } else {
                const int r = 16 * mb + (lane & 7) + 8 * ((lane >> 3) & 1);   // token row
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int chunk = 2 * ks + (lane >> 4);                   // 16-byte column
                    const uint32_t addr = kbase + (chunk >> 3) * Sm::kHalfBytes + r * 128 +
                                          (((chunk & 7) ^ (r & 7)) << 4);
                    uint32_t a[4];
                    ldsm_x4(addr, a);
                    Mma<TM>::run(s, a, qb[ks][0], qb[ks][1]);
                }
            }
            // ---- online softmax: s[0], s[1] = token 16mb+g; s[2], s[3] = token 16mb+g+8
            const int tok_a = 16 * mb + g, tok_b = tok_a + 8;
            float x[4];
            x[0] = tok_a < nvalid ? s[0] * sl2 : -INFINITY;
            x[1] = tok_a < nvalid ? s[1] * sl2 : -INFINITY;
            x[2] = tok_b < nvalid ? s[2] * sl2 : -INFINITY;
            x[3] = tok_b < nvalid ? s[3] * sl2 : -INFINITY;
            if constexpr (CH) {
                // causal within the chunk: token t is visible to a row at position >= t
                const int abs_a = jb * BS + it * TB + tok_a, abs_b = abs_a + 8;
                x[0] = abs_a <= lim[0] ? x[0] : -INFINITY;
                x[1] = abs_a <= lim[1] ? x[1] : -INFINITY;
                x[2] = abs_b <= lim[0] ? x[2] : -INFINITY;
                x[3] = abs_b <= lim[1] ? x[3] : -INFINITY;
            }
            float alpha[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float tmax = fmaxf(x[j], x[j + 2]);
                tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 4));
                tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 8));
                tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 16));
                const float mnew = fmaxf(m[j], tmax);       // -inf only for padded heads
                alpha[j] = (mnew == m[j]) ? 1.f : ex2_approx(m[j] - mnew);   // 1: max unchanged
                m[j] = mnew;
                const float pa = (mnew == -INFINITY) ? 0.f : ex2_approx(x[j] - mnew);
                const float pb = (mnew == -INFINITY) ? 0.f : ex2_approx(x[j + 2] - mnew);
                x[j] = pa;
                x[j + 2] = pb;
                lsum[j] = fmaf(lsum[j], alpha[j], pa + pb);
            }
            // once the running maxima settle (most tiles of a long context) no row of the
            // warp rescales, and the 4 x KS multiplies by 1 are skipped
            if (__any_sync(kFullMask, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int i = 0; i < KS; ++i) {
                    o[i][0] *= alpha[0];
                    o[i][1] *= alpha[1];
                    o[i][2] *= alpha[0];
                    o[i][3] *= alpha[1];
                }
            }
            // ---- P^T (hi + lo) into B fragments: transpose each 8x8 block in registers
            const uint32_t hi_a = Mma<TM>::pack(x[0], x[1]);
            const uint32_t hi_b = Mma<TM>::pack(x[2], x[3]);
            const float2 fa = Mma<TM>::unpack(hi_a), fb = Mma<TM>::unpack(hi_b);
            const uint32_t lo_a = Mma<TM>::pack(x[0] - fa.x, x[1] - fa.y);
            const uint32_t lo_b = Mma<TM>::pack(x[2] - fb.x, x[3] - fb.y);
            const uint32_t bh0 = movmatrix_trans(hi_a), bh1 = movmatrix_trans(hi_b);
            const uint32_t bl0 = movmatrix_trans(lo_a), bl1 = movmatrix_trans(lo_b);
            // ---- O^T += V^T . P^T over tokens 16mb .. 16mb+15
            const int vr = 16 * mb + (lane & 7) + 8 * (lane >> 4);            // token row
            const bool ragged = nvalid < 16 * (mb + 1);
            uint32_t vpair[8];   // direct E4M3: the two m-blocks 2j, 2j+1 read together
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                uint32_t a[4];
                if constexpr (kDirect) {
                    // m-block i = 2j + q holds head dims 32j + 4g + 2q (m = g) and +1
                    // (m = g + 8): token pairs (2c, 2c+1) and (2c+8, 2c+9) of those dims
                    // come from 4-byte loads of the four rows, interleaved by byte_perm
                    if (i % 2 == 0) {
                        const int j = i / 2;
                        const int t0 = 16 * mb + 2 * c;
                        const int chunk = 2 * j + (g >> 2);
                        const int off = 4 * (g & 3);
                        const uint32_t w0 = lds_u32(vbase + t0 * 128 + ((chunk ^ (t0 & 7)) << 4) + off);
                        const uint32_t w1 = lds_u32(vbase + (t0 + 1) * 128 +
                                                    ((chunk ^ ((t0 + 1) & 7)) << 4) + off);
                        const uint32_t w8 = lds_u32(vbase + (t0 + 8) * 128 +
                                                    ((chunk ^ ((t0 + 8) & 7)) << 4) + off);
                        const uint32_t w9 = lds_u32(vbase + (t0 + 9) * 128 +
                                                    ((chunk ^ ((t0 + 9) & 7)) << 4) + off);
                        const uint32_t e01 = __byte_perm(w0, w1, 0x5140);   // dims +0, +1
                        const uint32_t e23 = __byte_perm(w0, w1, 0x7362);   // dims +2, +3
                        const uint32_t f01 = __byte_perm(w8, w9, 0x5140);
                        const uint32_t f23 = __byte_perm(w8, w9, 0x7362);
                        vpair[0] = e4m3x2_to_f16x2(e01);
                        vpair[1] = e4m3x2_to_f16x2(e01 >> 16);
                        vpair[2] = e4m3x2_to_f16x2(f01);
                        vpair[3] = e4m3x2_to_f16x2(f01 >> 16);
                        vpair[4] = e4m3x2_to_f16x2(e23);
                        vpair[5] = e4m3x2_to_f16x2(e23 >> 16);
                        vpair[6] = e4m3x2_to_f16x2(f23);
                        vpair[7] = e4m3x2_to_f16x2(f23 >> 16);
                    }
                    const int b = 4 * (i % 2);
                    a[0] = vpair[b];
                    a[1] = vpair[b + 1];
                    a[2] = vpair[b + 2];
                    a[3] = vpair[b + 3];
                } else {
                    const int chunk = 2 * i + ((lane >> 3) & 1);
                    const uint32_t addr = vbase + (chunk >> 3) * Sm::kHalfBytes + vr * 128 +
                                          (((chunk & 7) ^ (vr & 7)) << 4);
                    ldsm_x4_trans(addr, a);
                }
                if (ragged) {
                    // a0, a1 hold tokens 16mb + 2c, +1; a2, a3 tokens 16mb + 2c + 8, +9
                    const int t = 16 * mb + 2 * c;
                    const uint32_t m01 = (t < nvalid ? 0x0000ffffu : 0u) | (t + 1 < nvalid ? 0xffff0000u : 0u);
                    const uint32_t m23 = (t + 8 < nvalid ? 0x0000ffffu : 0u) |
                                         (t + 9 < nvalid ? 0xffff0000u : 0u);
                    a[0] &= m01;
                    a[1] &= m01;
                    a[2] &= m23;
                    a[3] &= m23;
                }
                Mma<TM>::run(o[i], a, bh0, bh1);
                Mma<TM>::run(o[i], a, bl0, bl1);
            }
        }
        if constexpr (!kFp8 || kDirect) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
        }
    }

    // ------------------------------------------------------------- merge the warps
    named_barrier(1, NCW * 32);            // every tile consumed: the ring / staging is free
    float* mrg_acc = reinterpret_cast<float*>(smem);                    // [NCW][8][D]
    float* mrg_ml = mrg_acc + NCW * 8 * D;                               // [NCW][8][2]
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        float l = lsum[j];
        l += __shfl_xor_sync(kFullMask, l, 4);
        l += __shfl_xor_sync(kFullMask, l, 8);
        l += __shfl_xor_sync(kFullMask, l, 16);
        if (g == 0) {
            mrg_ml[(warp * 8 + 2 * c + j) * 2 + 0] = m[j];
            mrg_ml[(warp * 8 + 2 * c + j) * 2 + 1] = l;
        }
    }
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        // head dims of m-block i's rows g and g + 8
        const int d = kDirect ? 32 * (i / 2) + 4 * g + 2 * (i % 2) : 16 * i + g;
        const int d8 = kDirect ? d + 1 : d + 8;
        mrg_acc[(warp * 8 + 2 * c) * D + d] = o[i][0];
        mrg_acc[(warp * 8 + 2 * c + 1) * D + d] = o[i][1];
        mrg_acc[(warp * 8 + 2 * c) * D + d8] = o[i][2];
        mrg_acc[(warp * 8 + 2 * c + 1) * D + d8] = o[i][3];
    }
    if (poisoned)
        *poison = 1;
    named_barrier(1, NCW * 32);

    const bool bad = *poison != 0;
    for (int idx = threadIdx.x; idx < NH * D; idx += NCW * 32) {
        const int h = idx / D;
        const int d = idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w)
            M = fmaxf(M, mrg_ml[(w * 8 + h) * 2]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float cw = exp2f(mrg_ml[(w * 8 + h) * 2] - M);
                num = fmaf(cw, mrg_acc[(w * 8 + h) * D + d], num);
                den = fmaf(cw, mrg_ml[(w * 8 + h) * 2 + 1], den);
            }
        }
        float out = den > 0.f ? num / den : 0.f;
        if constexpr (kFp8)
            out *= p.v_scale[kvh];
        if (bad)
            out = __int_as_float(0x7fc00000);
        int64_t row = (int64_t)seq * p.num_q_heads + h0 + h;
        if constexpr (CH) {
            const int R = R0 + h;
            const int j = R / p.group;
            if (j >= n)
                continue;                          // padding row
            row = (int64_t)(qs0 + j) * p.num_q_heads + kvh * p.group + (R - j * p.group);
        }
        if (split) {
            const int64_t prow = row * p.max_parts + part;
            p.part_o[prow * D + d] = out;
            if (d == 0) {
                p.part_ml[prow * 2 + 0] = M;
                p.part_ml[prow * 2 + 1] = den;
            }
        } else {
            store_out<T>(p, row * D + d, out);
        }
    }
}

// Ring depth of the tensor-core kernel: one stage per consumer warp for 16-bit
// caches (the consumers need little time per tile, so a shallow ring and more
// resident CTAs per SM beat a deeper ring: measured on GB300, 75 vs 95 us for the
// shared-prefix decode and 175 vs 194 us for the 8 x 32768-token decode), two for
// E4M3 caches, whose stages are half the size.
template <typename TK, int D, int TB>
struct MmaStages {
    static constexpr int value = kDecodeConsumerWarps * (sizeof(TK) == 1 ? 2 : 1);
};

// Cache blocks per tile: two for E4M3 tiles read directly at block size 16, so that a
// tile (an 8 KB stage, 32 tokens) spreads each consumer's per-tile softmax and
// hand-over work over as many bytes as at block size 32 (one block of 16 tokens is
// 4 KB of K + V).
template <typename TK, int D, int BS>
constexpr int mma_blocks_per_tile() { return (sizeof(TK) == 1 && D == 128 && BS == 16) ? 2 : 1; }

template <typename T, typename TK, int D, int BS, int NH>
struct MmaVariant {
    static constexpr int kBPT = mma_blocks_per_tile<TK, D, BS>();
    static constexpr int kStages = MmaStages<TK, D, BS * kBPT>::value;
    using Sm = MmaSmem<TK, D, BS * kBPT, kStages>;
    static constexpr auto kernel() { return decode_mma_kernel<T, TK, D, BS, NH, kStages, false, kBPT>; }
    static cudaError_t configure()
    {
        return configure_once(reinterpret_cast<const void*>(kernel()), Sm::kAlloc);
    }
    static cudaError_t launch(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream)
    {
        cudaError_t err = configure();
        if (err != cudaSuccess)
            return err;
        const bool split = p.partition_tokens > 0;
        dim3 grid(split ? p.max_parts : 1, p.num_kv_heads * p.chunks, p.num_seqs);
        kernel()<<<grid, kDecodeThreads, Sm::kAlloc, stream>>>(p, tk, tv);
        err = cudaGetLastError();
        if (err != cudaSuccess || !split)
            return err;
        reduce_kernel<T, D><<<dim3(p.num_q_heads, p.num_seqs), D, 0, stream>>>(p);
        return cudaGetLastError();
    }
};

// Tensor-core path (4 or 8 query heads per CTA; the kernel also takes 1 or 2, but
// the CUDA-core kernel serves those, as measured faster for MHA).  T: the 16-bit query type;
// TK: T, or __nv_fp8_e4m3 for a quantised cache (no tensor maps needed then).
#define PA_MMA_VARIANTS(X)                                                                    \
    X(128, 16, 8) X(128, 16, 4) X(128, 32, 8) X(128, 32, 4) X(64, 16, 8) X(64, 16, 4)           \
    X(64, 32, 8) X(64, 32, 4)
#define PA_MMA_VARIANTS_SMALL(X) \
    X(128, 16, 2) X(128, 16, 1) X(128, 32, 2) X(128, 32, 1) X(64, 16, 2) X(64, 16, 1) X(64, 32, 2) X(64, 32, 1)

template <typename T, typename TK = T>
cudaError_t launch_decode_mma(const DecodeParams& p, int head_dim, int block_size, int gc,
                              cudaStream_t stream)
{
    CUtensorMap tk{}, tv{};
    if (sizeof(TK) == 2 || head_dim == 128) {      // 16-bit tiles, or direct E4M3 tiles
        cudaError_t e = kv_tensor_map(&tk, p.k_cache, p.num_blocks, p.num_kv_heads, block_size,
                                      head_dim, DType<TK>::id);
        if (e == cudaSuccess)
            e = kv_tensor_map(&tv, p.v_cache, p.num_blocks, p.num_kv_heads, block_size, head_dim,
                              DType<TK>::id);
        if (e != cudaSuccess)
            return e;
    }
#define PA_MMA_CASE(D_, BS_, NH_)                                  \
    if (head_dim == D_ && block_size == BS_ && gc == NH_)          \
        return MmaVariant<T, TK, D_, BS_, NH_>::launch(p, tk, tv, stream);
    PA_MMA_VARIANTS(PA_MMA_CASE)
    if constexpr (sizeof(TK) == 1) {
        PA_MMA_VARIANTS_SMALL(PA_MMA_CASE)
    }
#undef PA_MMA_CASE
    return cudaErrorInvalidValue;
}

// Resident CTAs per SM of the tensor-core kernel for this shape (0 if unknown).
template <typename T, typename TK = T>
int occupancy_decode_mma(int head_dim, int block_size, int gc)
{
#define PA_MMA_OCC(D_, BS_, NH_)                                   \
    if (head_dim == D_ && block_size == BS_ && gc == NH_) {        \
        using V = MmaVariant<T, TK, D_, BS_, NH_>;                 \
        return V::configure() == cudaSuccess                       \
                   ? kernel_occupancy(reinterpret_cast<const void*>(V::kernel()), V::Sm::kAlloc) \
                   : 0;                                            \
    }
    PA_MMA_VARIANTS(PA_MMA_OCC)
    if constexpr (sizeof(TK) == 1) {
        PA_MMA_VARIANTS_SMALL(PA_MMA_OCC)
    }
#undef PA_MMA_OCC
    return 0;
}

}  // namespace pa
