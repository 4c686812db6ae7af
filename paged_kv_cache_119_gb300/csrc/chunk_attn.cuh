// chunk_attn.cuh -- causal attention of a chunk of new query tokens per sequence
// over the paged KV cache, on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// What it computes (the chunked-prefill / speculative-verification use of the
// paged cache: "PagedAttention 完全拆解", section "局限与未解决的问题" item 6;
// "PagedAttention 与 vLLM 推理加速", section "一图总结"): sequence s owns query rows
// query_start[s] .. query_start[s+1]-1; with n of them and context L, chunk token
// j sits at position L - n + j and attends to cached tokens 0 .. L - n + j, i.e.
// the softmax attention of section "背景" over that prefix, read through the
// block table.
//
// Organisation.  A CTA owns 256 (query token, query head) rows that share a kv
// head -- TT = 256 / G consecutive chunk tokens x the G heads of the group, row
// r = token * G + head -- as two 128-row query tiles.  K and V stream through the
// block table in tiles of 64 tokens, each tile serving both query tiles:
//   S_q[128 x 64]  = Q_q[128 x D] . K^T      (tcgen05.mma kind::f16, fp32 in TMEM)
//   O_q[128 x D]  += P_q[128 x 64] . V        (P in f16, A operand read from tensor
//                                              memory; V in f16)
//   * warp 0 (producer): block-table entries and tensor-map TMA of the tile's K
//     and V boxes (64 dims x B tokens, 128-byte swizzle) into an mbarrier ring;
//   * warps 1 and 10: one thread each issues the MMAs of one query tile (warp 1 also
//     allocates all 512 tensor-memory columns): the scores of the next tile go out
//     before P.V of the current one, into a second S buffer.  Each issuer waits only
//     on its own query tile's completions, so the tensor core takes work from the
//     other while one waits;
//   * warps 2-5 (query tile 0) and 6-9 (query tile 1), one thread per row = TMEM
//     lane: read S, mask (causal within the chunk, end of context), online softmax
//     in base 2, write P back over the S buffer it came from (packed f16 pairs),
//     keep O up to date;
//   * over bf16 caches, warps 11-14 rewrite each V tile in place as f16 (below).
// The S/P buffers alternate between tiles, so the softmax of tile i+1 never waits
// for P.V of tile i; the scores of tile i+2 reuse a buffer only once P.V of tile i
// has read it.
// Two softmax warps per SM sub-partition hide each other's latency; the MUFU work
// (one exp2 per score) stays below the tensor-core time of a tile.
// Rescaling O is lazy: a row's reference maximum moves only when a tile's maximum
// exceeds it by more than 2^8 in probability, so p = 2^(x - m_ref) <= 256 and most
// tiles need no tensor-memory round trip.  O / l is exact for any reference, as O
// and l share it.
// P enters P.V as one f16 term, 2^7 p (at most 2^15, and normal down to p = 2^-21),
// rounded to nearest: up to 2^-11 relative per weight, so the output is off by at
// most 2^-11 of the largest |v| the row weighs (fp32 accumulation), a quarter of the
// bf16 output's own rounding step; one bf16 rounding of p would cost 2^-9, and a
// second (lo) term would cost as much tensor and softmax work again.  The 2^7 is
// carried by the exponent (p = 2^(x - m_ref + 7)) and cancels against the row sum.
// So V must be f16 too: f16 caches are, E4M3 caches convert to f16 anyway, and over
// bf16 caches four converter warps rewrite each V tile in place (same swizzled
// layout, bf16 -> f16 is exact for 2^-14 <= |v| <= 65280) and zero its rows past the
// range.  A value without an f16 value (|v| >= 65536, infinite or NaN) becomes
// infinite or NaN; the epilogue sets PA_DEVERR_RANGE for a row whose probabilities are
// finite but whose O is not.  K stays bf16 (the score product is bf16 x bf16).
// Long contexts with few CTAs are split into partitions merged by
// chunk_reduce_kernel, as in the decode path.
// The epilogue reads O once its issuer's one-phase completion barrier has fired (P.V of
// the last two tiles may be pending or done in any combination when a warp gets there,
// which a wait on the per-tile parity barrier cannot tell apart).
//
// E4M3 caches (NRAW > 0, head_dim 128): the producer's TMA fills a ring of raw one-byte
// K + V tiles, and four converter warps (11-14) turn each into the f16 swizzled tiles of
// the ring above (E4M3 -> f16 is exact), then hand it to the issuers and release the raw
// slot.  The operands are f16: a bf16 query row is scaled into f16 range by a power of
// two (exact) that joins the row's score scale together with the kv head's K scale, and
// the V scale multiplies the output.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"

namespace pa {

constexpr int kChunkQTiles = 2;      // 128-row query tiles per CTA
constexpr int kChunkRows = 128;      // M of the tensor-core tile
constexpr int kChunkTileTok = 64;    // tokens per K/V tile (N of the score product)
constexpr int kChunkSoftmaxWarps = 4 * kChunkQTiles;
// warps: 0 producer, 1 tensor-memory allocator + MMA issuer of query tile 0, 2-9
// softmax, 10 MMA issuer of query tile 1; over E4M3 and bf16 caches, 11-14 convert
// tiles to f16
constexpr int kChunkThreads = 64 + 32 * kChunkSoftmaxWarps + 32;
constexpr int kChunkConvWarps = 4;
constexpr int kChunkThreadsConv = kChunkThreads + 32 * kChunkConvWarps;
// P.V takes P as 2^kChunkPExp p: p <= 2^8 (the lazy rescale), so 2^15 at most in f16
constexpr float kChunkPExp = 7.f;

// NRAW > 0 (E4M3 caches): a ring of NRAW raw one-byte K + V tiles that the converter
// warps turn into the 16-bit tiles of the NST-stage ring.
template <int D, int NST, int NRAW = 0>
struct ChunkSmem {
    static constexpr int kHalves = D / 64;                       // 128-byte column groups
    static constexpr int kQHalf = kChunkRows * 128;              // 16 KB
    static constexpr int kQTile = kHalves * kQHalf;              // one 128-row query tile
    static constexpr int kKVHalf = kChunkTileTok * 128;          // 8 KB
    static constexpr int kKBytes = kHalves * kKVHalf;
    static constexpr int kStageBytes = 2 * kKBytes;              // K then V
    static constexpr int kQOff = 0;
    static constexpr int kStageOff = kQOff + kChunkQTiles * kQTile;
    static constexpr int kRawTile = kChunkTileTok * D;           // one E4M3 K (or V) tile
    static constexpr int kRawStage = 2 * kRawTile;
    static constexpr int kRawOff = kStageOff + NST * kStageBytes;
    static constexpr int kBarOff = kRawOff + NRAW * kRawStage;
    // full[NST], empty[NST], s_full[2][2], p_full[2][2], pv_done[2], q_full, mma_done[2],
    // v_zero, raw_full[NRAW], raw_empty[NRAW], vconv[NST]
    static constexpr int kNumBars = 3 * NST + 14 + 2 * NRAW;
    static constexpr int kOkOff = kBarOff + 8 * kNumBars;        // stage_ok[NST], raw_ok[NRAW]
    static constexpr int kSlotOff = kOkOff + 4 * (NST + NRAW);   // TMEM address
    static constexpr int kBytes = kSlotOff + 16;
    static constexpr int kAlloc = kBytes + 1024;                 // 1 KB alignment slack
    // tensor memory: O of query tile q at column 128 q, its two S/P buffers at
    // 256 + 128 q and 256 + 128 q + 64 (P: f16 pairs in the first 32 columns)
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 256;
    static_assert(D <= 128, "O must fit in 128 columns");
    static_assert(NRAW == 0 || D == 128, "E4M3 tiles need 128-byte rows");
    static_assert(kRawTile % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Stages of the K/V ring: as many as fit next to the query tiles.
template <int D>
struct ChunkStages {
    static constexpr int value = D == 128 ? 5 : 8;
};

// Stores 32 consecutive outputs v[i] * mul (NaN when nan_out) at base + idx as
// fp32 (which = 0), f16 (1) or bf16 (2); idx is a multiple of 32.
__device__ __forceinline__ void store_row32(void* base, int64_t idx, const float (&v)[32], float mul,
                                            bool nan_out, int which)
{
    const float qnan = __int_as_float(0x7fc00000);
    if (which == 0) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = nan_out ? make_float4(qnan, qnan, qnan, qnan)
                             : make_float4(v[4 * i] * mul, v[4 * i + 1] * mul, v[4 * i + 2] * mul,
                                           v[4 * i + 3] * mul);
        return;
    }
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = nan_out ? qnan : v[2 * i] * mul;
        const float b = nan_out ? qnan : v[2 * i + 1] * mul;
        if (which == 1) {
            __half2 h = __floats2half2_rn(a, b);
            packed[i] = *reinterpret_cast<uint32_t*>(&h);
        } else {
            __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            packed[i] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
}

// max(a, b, c) in one instruction (NaN operands are ignored, as by fmaxf).
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// grid = (partitions, num_kv_heads * m_tiles, num_seqs); kChunkThreads threads over
// f16 caches, kChunkThreadsConv over E4M3 (NRAW > 0) and bf16 caches.  T: query /
// native output type.  Over E4M3 caches (value = code * per-kv-head scale) the
// tensor-core operands are f16: the codes convert exactly, a bf16 query row is scaled
// into f16 range by a power of two (exact), and the scales fold into the scores and
// the output.
template <typename T, int D, int BS, int NST, int NRAW = 0>
__global__ void __launch_bounds__((NRAW > 0 || std::is_same_v<T, __nv_bfloat16>) ? kChunkThreadsConv
                                                                                 : kChunkThreads,
                                  1)
    chunk_attn_kernel(const __grid_constant__ ChunkParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv)
{
    using Sm = ChunkSmem<D, NST, NRAW>;
    constexpr bool kF8 = NRAW > 0;
    constexpr bool kVConv = !kF8 && std::is_same_v<T, __nv_bfloat16>;   // bf16 V -> f16 in place
    using TM = std::conditional_t<kF8, __half, T>;   // operand type of the score product
    constexpr int NT = kChunkTileTok;
    constexpr int BPT = NT / BS;                 // cache blocks per K/V tile
    constexpr int KS = D / 16;                   // k-steps of the score product
    constexpr bool kBf16 = DType<TM>::id == PA_BF16;
    static_assert(NT % BS == 0 && D % 64 == 0, "block_size 16/32, head_dim 64/128");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);
    uint64_t* empty = full + NST;
    uint64_t* s_full = empty + NST;              // [query tile][S/P buffer]
    uint64_t* p_full = s_full + 4;               // [query tile][S/P buffer]
    uint64_t* pv_done = p_full + 4;              // [query tile]
    uint64_t* q_full = pv_done + 2;
    uint64_t* mma_done = q_full + 1;             // [query tile]
    uint64_t* v_zero = mma_done + 2;             // the last tile's V rows past the range are 0
    uint64_t* raw_full = v_zero + 1;             // [raw slot] (E4M3 caches)
    uint64_t* raw_empty = raw_full + NRAW;
    uint64_t* vconv = raw_empty + NRAW;          // [stage] (bf16 caches: V tile is f16)
    int* stage_ok = reinterpret_cast<int*>(smem + Sm::kOkOff);
    int* raw_ok = stage_ok + NST;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Sm::kSlotOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y / p.m_tiles;
    const int mt = blockIdx.y - kvh * p.m_tiles;
    const int part = blockIdx.x;
    const bool split = p.partition_tokens > 0;
    const int G = p.group;
    const int TT = p.rows_tokens;

    const int qs0 = p.query_start[seq];
    const int qs1 = p.query_start[seq + 1];
    const int n = qs1 - qs0;
    const int L = p.context_lens[seq];
    const bool rows_sane = qs0 >= 0 && n >= 0 && (int64_t)qs1 <= p.num_rows;
    if (!rows_sane || L < 0 || L > p.max_context_len || n > L || n > p.max_query_len) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);
        if (!split && rows_sane && part == 0 && mt == 0) {
            // the sequence's rows of this kv head's query heads become NaN
            const int64_t cnt = (int64_t)n * G * D;
            for (int64_t i = threadIdx.x; i < cnt; i += blockDim.x) {
                const int64_t tok = i / ((int64_t)G * D);
                const int rem = (int)(i - tok * G * D);
                const int64_t idx = ((qs0 + tok) * p.num_q_heads + kvh * G) * D + rem;
                if (p.out_f32)
                    store_as(static_cast<float*>(p.out) + idx, __int_as_float(0x7fc00000));
                else
                    store_as(static_cast<T*>(p.out) + idx, __int_as_float(0x7fc00000));
            }
        }
        return;
    }
    if (seq == p.num_seqs - 1 && part == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
        (int64_t)qs1 != p.num_rows)
        atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);   // rows after the last chunk belong to no one
    const int j0 = mt * TT;
    if (j0 >= n)
        return;                                  // no chunk token in this row tile
    const int ntok = min(TT, n - j0);
    const int pos_first = L - n + j0;            // position of the tile's first token
    const int t_end = pos_first + ntok;          // tokens [0, t_end) are seen by some row
    int t0 = 0, t1 = t_end;
    if (split) {
        t0 = part * p.partition_tokens;
        if (t0 >= t_end)
            return;
        t1 = min(t_end, t0 + p.partition_tokens);
    }
    const int ntiles = (t1 - t0 + NT - 1) / NT;  // >= 1

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], kF8 ? kChunkConvWarps : 1);   // converters, or the TMA
            mbar_init(&empty[s], kChunkQTiles);          // one commit per issuer
        }
#pragma unroll
        for (int s = 0; s < NRAW; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kChunkConvWarps);
        }
#pragma unroll
        for (int s = 0; s < NST; ++s)
            mbar_init(&vconv[s], kChunkConvWarps);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
        }
#pragma unroll
        for (int q = 0; q < kChunkQTiles; ++q) {
            mbar_init(&pv_done[q], 1);
            mbar_init(&mma_done[q], 1);
        }
        mbar_init(q_full, kChunkSoftmaxWarps);
        mbar_init(v_zero, kChunkSoftmaxWarps);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, Sm::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        const int32_t* bt_row = p.block_tables + (int64_t)seq * p.bt_stride;
        const uint64_t policy = l2_evict_first_policy();
        const int blk_end = (t1 + BS - 1) / BS;
        // 16-bit caches fill the MMA ring directly; E4M3 caches fill the raw ring
        constexpr int NP = kF8 ? NRAW : NST;
        uint64_t* pfull = kF8 ? raw_full : full;
        uint64_t* pempty = kF8 ? raw_empty : empty;
        int* pok = kF8 ? raw_ok : stage_ok;
        int issued = 0;
        for (int it = 0; it < ntiles; ++it) {
            const int st = it % NP;
            const int b0 = (t0 + it * NT) / BS;
            const int nb = min(BPT, blk_end - b0);
            int pbn = -1;
            bool valid = false;
            if (lane < nb) {
                pbn = __ldg(bt_row + b0 + lane);
                valid = pbn >= 0 && (int64_t)pbn < p.num_blocks;
            }
            const unsigned vmask = __ballot_sync(kFullMask, valid);
            int ok = 1;
            if (lane == 0) {
                if (it >= NP && !mbar_wait(&pempty[st], ((it / NP) - 1) & 1)) {
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                    ok = 0;
                } else {
                    const int nvalid = __popc(vmask);
                    pok[st] = nvalid == nb ? 1 : 0;
                    if (nvalid != nb)
                        atomicOr(p.err, PA_DEVERR_BLOCK_ID);
                    // a block is one 128-byte-row box per 64 dims (16-bit) or per 128 codes
                    mbar_arrive_expect_tx(&pfull[st],
                                          (uint32_t)nvalid * 2u * (kF8 ? 1 : Sm::kHalves) * BS * 128u);
                }
            }
            if (!__shfl_sync(kFullMask, ok, 0))
                break;
            if (kF8 && valid) {
                unsigned char* kdst = smem + Sm::kRawOff + st * Sm::kRawStage + lane * (BS * 128);
                const int z = pbn * p.num_kv_heads + kvh;     // < 2^31 (checked on the host)
                tma_load_3d(kdst, &tk, 0, 0, z, &pfull[st], policy);
                tma_load_3d(kdst + Sm::kRawTile, &tv, 0, 0, z, &pfull[st], policy);
            } else if (valid) {
                unsigned char* kdst = smem + Sm::kStageOff + st * Sm::kStageBytes + lane * (BS * 128);
                const int z = pbn * p.num_kv_heads + kvh;     // < 2^31 (checked on the host)
#pragma unroll
                for (int h = 0; h < Sm::kHalves; ++h) {
                    tma_load_3d(kdst + h * Sm::kKVHalf, &tk, 64 * h, 0, z, &full[st], policy);
                    tma_load_3d(kdst + Sm::kKBytes + h * Sm::kKVHalf, &tv, 64 * h, 0, z, &full[st],
                                policy);
                }
            }
            issued = it + 1;
        }
        // no copy may still be in flight into this CTA's shared memory at exit
        if (lane == 0)
            for (int it = max(0, issued - NP); it < issued; ++it)
                mbar_wait(&pfull[it % NP], (it / NP) & 1);
        __syncwarp();
    } else if ((kF8 || kVConv) && warp > 2 + kChunkSoftmaxWarps) {
        // ------------------------------------------------ E4M3 -> f16 tile conversion
        // A raw tile row is 128 codes in 128-byte-swizzled order (16-byte chunk c of row
        // t at c ^ (t & 7)); the f16 tile is two 64-dim halves of 128-byte rows in the
        // same swizzle.  Each (token, 16-code chunk) item becomes two f16 chunks.
        if constexpr (kF8) {
            const int ct = threadIdx.x - kChunkThreads;      // 0 .. 32 * kChunkConvWarps - 1
            constexpr int kItems = NT * 8;                   // per K (or V) tile
            for (int it = 0; it < ntiles; ++it) {
                const int r = it % NRAW;
                const int st = it % NST;
                bool ok = mbar_wait(&raw_full[r], (it / NRAW) & 1);
                if (ok && it >= NST)
                    ok = mbar_wait(&empty[st], ((it / NST) - 1) & 1);   // both issuers' P.V
                if (!ok) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT);
                    break;
                }
                const unsigned char* raw = smem + Sm::kRawOff + r * Sm::kRawStage;
                unsigned char* dst = smem + Sm::kStageOff + st * Sm::kStageBytes;
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
#pragma unroll 4
                    for (int item = ct; item < kItems; item += 32 * kChunkConvWarps) {
                        const int t = item >> 3;
                        const int c = item & 7;
                        const uint4 w = *reinterpret_cast<const uint4*>(
                            raw + kv * Sm::kRawTile + t * 128 + ((c ^ (t & 7)) << 4));
                        unsigned char* row =
                            dst + kv * Sm::kKBytes + (c >> 2) * Sm::kKVHalf + t * 128;
                        const int c0 = 2 * (c & 3);
                        *reinterpret_cast<uint4*>(row + ((c0 ^ (t & 7)) << 4)) =
                            make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16),
                                       e4m3x2_to_f16x2(w.y), e4m3x2_to_f16x2(w.y >> 16));
                        *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (t & 7)) << 4)) =
                            make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16),
                                       e4m3x2_to_f16x2(w.w), e4m3x2_to_f16x2(w.w >> 16));
                    }
                }
                fence_proxy_async_smem();                    // f16 tiles -> tensor core
                __syncwarp();
                if (lane == 0) {
                    if (warp == 3 + kChunkSoftmaxWarps)
                        stage_ok[st] = raw_ok[r];
                    mbar_arrive(&full[st]);
                    mbar_arrive(&raw_empty[r]);
                }
            }
        } else if constexpr (kVConv) {
            // bf16 -> f16 of each V tile in place, once its bytes are in (the K half is
            // left to the score product meanwhile); rows past the range become 0, so
            // that 0 * V stays 0 whatever an unused slot holds.  The stage is refilled
            // only after both P.V of the tile, which wait for this hand-over.  A value
            // without an f16 value becomes infinite (or stays NaN); the epilogue reports
            // the rows it reaches.
            const int ct = threadIdx.x - kChunkThreads;      // 0 .. 32 * kChunkConvWarps - 1
            constexpr int kItems = NT * 8 * Sm::kHalves;     // 16-byte chunks of a V tile
            constexpr int kPer = kItems / (32 * kChunkConvWarps);
            static_assert(kItems % (32 * kChunkConvWarps) == 0, "whole chunks per thread");
            for (int it = 0; it < ntiles; ++it) {
                const int st = it % NST;
                if (!mbar_wait(&full[st], (it / NST) & 1)) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT);
                    break;
                }
                const int nv = min(NT, t1 - (t0 + it * NT));  // rows inside the range
                unsigned char* vt = smem + Sm::kStageOff + st * Sm::kStageBytes + Sm::kKBytes;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int item = ct + i * 32 * kChunkConvWarps;
                    const int w = item % (NT * 8);           // chunk within a 64-dim half
                    uint4* chunk = reinterpret_cast<uint4*>(vt + (item / (NT * 8)) * Sm::kKVHalf +
                                                            w * 16);
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if ((w >> 3) < nv) {
                        const uint4 b = *chunk;
                        const uint32_t in[4] = {b.x, b.y, b.z, b.w};
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __half2 h = __floats2half2_rn(__uint_as_float(in[j] << 16),
                                                                __uint_as_float(in[j] & 0xffff0000u));
                            o[j] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        v = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    *chunk = v;
                }
                fence_proxy_async_smem();                    // f16 V -> tensor core
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&vconv[st]);
            }
        }
    } else if (warp == 1 || warp == 2 + kChunkSoftmaxWarps) {
        // ------------------------------------------- MMA issue, one query tile per warp
        const int q = warp == 1 ? 0 : 1;
        if (lane == 0) {
            const uint32_t sq = smem_addr(smem + Sm::kQOff + q * Sm::kQTile);
            const uint32_t idesc_s = mma_idesc_f16(kBf16, kChunkRows, NT, false);
            const uint32_t idesc_o = mma_idesc_f16(false, kChunkRows, D, true);   // f16 P, V
            bool ok = mbar_wait(q_full, 0);
            // S of tile it into this query tile's S buffer it & 1
            auto issue_scores = [&](int it) {
                const uint32_t kb = smem_addr(smem + Sm::kStageOff + (it % NST) * Sm::kStageBytes);
                const uint32_t dcol = tbase + Sm::kSCol + q * 128 + (it & 1) * NT;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint64_t a = sw128_desc(sq + (kk / 4) * Sm::kQHalf + (kk % 4) * 32, 16, 1024);
                    const uint64_t b =
                        sw128_desc(kb + (kk / 4) * Sm::kKVHalf + (kk % 4) * 32, 16, 1024);
                    tc_mma_f16(dcol, a, b, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[q * 2 + (it & 1)]);
            };
            if (ok)
                ok = mbar_wait(&full[0], 0);
            if (ok) {
                tc_fence_after();
                issue_scores(0);
            }
            for (int it = 0; it < ntiles && ok; ++it) {
                if (it + 1 < ntiles) {
                    ok = mbar_wait(&full[(it + 1) % NST], ((it + 1) / NST) & 1);
                    // S/P buffer (it+1)&1 holds P of tile it-1 until its P.V completes
                    if (ok && it >= 1)
                        ok = mbar_wait(&pv_done[q], (it - 1) & 1);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_scores(it + 1);
                }
                ok = mbar_wait(&p_full[q * 2 + (it & 1)], (it >> 1) & 1);
                if constexpr (kVConv) {
                    if (ok)                           // V in f16, rows past the range zeroed
                        ok = mbar_wait(&vconv[it % NST], (it / NST) & 1);
                } else {
                    if (ok && t0 + (it + 1) * NT > t1)
                        ok = mbar_wait(v_zero, 0);   // last tile: V rows past the range zeroed
                }
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t vb =
                    smem_addr(smem + Sm::kStageOff + (it % NST) * Sm::kStageBytes + Sm::kKBytes);
                const uint32_t pcol = tbase + Sm::kSCol + q * 128 + (it & 1) * NT;
#pragma unroll
                for (int kk = 0; kk < NT / 16; ++kk) {        // 16 tokens = 8 columns of P
                    const uint64_t b = sw128_desc(vb + kk * 16 * 128, Sm::kKVHalf, 1024);
                    tc_mma_f16_ts(tbase + q * 128, pcol + kk * 8, b, idesc_o,
                                  (it > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&pv_done[q]);
                tc_commit(&empty[it % NST]);
            }
            if (!ok)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            tc_commit(&mma_done[q]);          // every MMA above completes before TMEM is freed
            mbar_wait(&mma_done[q], 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        const int q = (warp - 2) >> 2;                   // query tile of this warp
        const int wq = warp & 3;                         // TMEM lane quarter of this warp
        const int rr = 32 * wq + lane;                   // row within the query tile = TMEM lane
        const int r = q * kChunkRows + rr;               // row within the CTA
        const int tok = r / G;
        const int g = r - tok * G;
        const bool row_valid = tok < ntok;               // (r >= TT * G gives tok >= TT)
        const int pos = pos_first + tok;
        const int64_t qrow = (int64_t)(qs0 + j0 + tok) * p.num_q_heads + (int64_t)kvh * G + g;
        // scores are used as s * sl2 with sl2 > 0: a negative scale flips the sign of q
        // (exact), a zero scale makes q zero (every score 0); over E4M3 caches the K scale
        // of the kv head joins the softmax scale
        const float sl2_raw = kF8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
        const uint32_t qflip = sl2_raw < 0.f ? 0x80008000u : 0u;
        const bool qzero = sl2_raw == 0.f;
        float sl2 = qzero ? 1.f : fabsf(sl2_raw);
        {
            // Q rows into the 128-byte-swizzled operand layout; rows past the chunk are 0
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                              (row_valid ? qrow : 0) * D);
            unsigned char* qdst = smem + Sm::kQOff + q * Sm::kQTile + rr * 128;
            constexpr bool kToF16 = kF8 && DType<T>::id == PA_BF16;
            float down = 1.f;
            if constexpr (kToF16) {
                // a bf16 row becomes f16 operands: a power of two 2^-e puts its largest
                // |q| in [2^14, 2^15), so the 8-bit mantissas convert exactly; 2^e goes
                // into the row's score scale
                float amax = 0.f;
                if (row_valid && !qzero) {
#pragma unroll 4
                    for (int c = 0; c < D / 8; ++c) {
                        const uint4 v = __ldg(src + c);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                                     fabsf(__uint_as_float(w[j] & 0xffff0000u))));
                    }
                }
                const int ex = (__float_as_int(amax) >> 23) & 0xff;   // biased exponent
                // amax in [2^(ex-127), 2^(ex-126)): scale by 2^(141 - ex); rows of zeros,
                // tiny rows and a NaN / infinite row keep the scale 1
                const int sh = (ex == 0 || ex == 255) ? 0 : max(-100, min(100, 141 - ex));
                down = __int_as_float((127 + sh) << 23);
                sl2 *= __int_as_float((127 - sh) << 23);
            }
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (row_valid && !qzero) {
                    v = __ldg(src + c);
                    if constexpr (kToF16) {
                        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                                                __uint_as_float(w[j] & 0xffff0000u) * down);
                            w[j] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        v = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    v.x ^= qflip;
                    v.y ^= qflip;
                    v.z ^= qflip;
                    v.w ^= qflip;
                }
                *reinterpret_cast<uint4*>(qdst + (c / 8) * Sm::kQHalf + (((c & 7) ^ (rr & 7)) << 4)) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(q_full);

        const bool warp_live = __any_sync(kFullMask, row_valid);
        const uint32_t lane_t = tbase + ((uint32_t)(32 * wq) << 16);
        const uint32_t o_col = lane_t + q * 128;
        float m_ref = -INFINITY, lsum = 0.f;
        bool poisoned = false;
        for (int it = 0; it < ntiles; ++it) {
            const int b = it & 1;
            const int st = it % NST;
            const int tb = t0 + it * NT;
            bool ok = mbar_wait(&s_full[q * 2 + b], (it >> 1) & 1);
            ok = ok && mbar_wait(&full[st], (it / NST) & 1);   // stage_ok and the tile's bytes
            if (!ok) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                poisoned = true;
                break;
            }
            if (!stage_ok[st])
                poisoned = true;
            tc_fence_after();
            const uint32_t sp_col = lane_t + Sm::kSCol + q * 128 + b * NT;   // this row's S/P buffer
            float s[NT];
            if (warp_live)
                tmem_ld64(sp_col, s);
            if (warp_live) {
                const int lim = row_valid ? pos - tb : -1;   // columns c <= lim are visible
                if (lim < NT - 1) {
#pragma unroll
                    for (int c = 0; c < NT; ++c)
                        s[c] = c <= lim ? s[c] : -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mx[i] = s[i];
#pragma unroll
                for (int c = 8; c + 16 <= NT; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mx[i] = max3f(mx[i], s[c + i], s[c + 8 + i]);
#pragma unroll
                for (int c = 8 + (NT - 8) / 16 * 16; c < NT; ++c)
                    mx[c & 7] = fmaxf(mx[c & 7], s[c]);
                const float smax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7]));
                const float tmax = smax == -INFINITY ? -INFINITY : smax * sl2;
                const bool need = tmax > m_ref + 8.f;
                if (it > 0 && __any_sync(kFullMask, need)) {
                    // O holds P.V of tiles 0 .. it-1: wait for the last, then rescale the
                    // rows whose reference maximum moves
                    if (!mbar_wait(&pv_done[q], (it - 1) & 1)) {
                        if (lane == 0)
                            atomicOr(p.err, PA_DEVERR_TIMEOUT);
                        poisoned = true;
                    }
                    tc_fence_after();
                    const float alpha = need ? ex2_approx(m_ref - tmax) : 1.f;
#pragma unroll 1
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        float o[32];
                        tmem_ld32(o_col + 32 * c4, o);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 v = fmul2(make_float2(o[i], o[i + 1]), make_float2(alpha, alpha));
                            o[i] = v.x;
                            o[i + 1] = v.y;
                        }
                        tmem_st32(o_col + 32 * c4, o);
                    }
                }
                if (need) {
                    lsum *= ex2_approx(m_ref - tmax);
                    m_ref = tmax;
                }
                // 2^7 p = 2^(s * sl2 - m_ref + 7), in place; 0 where masked (s = -inf) or no
                // reference; the row sum carries the same 2^7
                const float nm = (m_ref == -INFINITY ? 0.f : -m_ref) + kChunkPExp;
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < NT; c += 2) {
                    const float2 x = ffma2(make_float2(s[c], s[c + 1]), make_float2(sl2, sl2),
                                           make_float2(nm, nm));
                    s[c] = ex2_approx(x.x);
                    s[c + 1] = ex2_approx(x.y);
                    acc[(c >> 1) & 3] = ffma2(make_float2(s[c], s[c + 1]), make_float2(1.f, 1.f),
                                              acc[(c >> 1) & 3]);
                }
                lsum += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                        ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
            }
            if (warp_live) {
                // P over the first 32 columns of the S buffer, as f16 pairs
                uint32_t ph[NT / 2];
#pragma unroll
                for (int k = 0; k < NT / 2; ++k) {
                    const __half2 h = __floats2half2_rn(s[2 * k], s[2 * k + 1]);
                    ph[k] = *reinterpret_cast<const uint32_t*>(&h);
                }
                tmem_st32_raw(sp_col, ph);
            }
            if (!kVConv && tb + NT > t1) {
                // V rows past the range may hold anything (unused slots, stale tiles):
                // zero them so that 0 * V stays 0; both issuers wait for v_zero before
                // their last P.V
                const int v0 = t1 - tb;
                const int rows = NT - v0;
                unsigned char* vbase = smem + Sm::kStageOff + st * Sm::kStageBytes + Sm::kKBytes;
                for (int idx = threadIdx.x - 64; idx < Sm::kHalves * rows * 8;
                     idx += 32 * kChunkSoftmaxWarps) {
                    const int h = idx / (rows * 8);
                    const int w = idx - h * rows * 8;
                    *reinterpret_cast<uint4*>(vbase + h * Sm::kKVHalf + (v0 + w / 8) * 128 +
                                              (w % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(v_zero);
            }
            tc_fence_before();                           // the P store precedes P.V
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[q * 2 + b]);
        }

        // ---------------------------------------------------------------- epilogue
        // every MMA of this query tile has completed once its issuer's final commit has
        // (one phase, so no parity wait can alias: P.V of the last two tiles may be pending
        // or done in any combination when a warp gets here)
        if (!mbar_wait(&mma_done[q], 0)) {
            if (lane == 0)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            poisoned = true;
        }
        tc_fence_after();
        if (warp_live) {
            // over E4M3 caches the V scale of the kv head multiplies the output
            const float inv = lsum > 0.f ? (kF8 ? p.v_scale[kvh] : 1.f) / lsum : 0.f;
            const int which = (split || p.out_f32) ? 0 : (DType<T>::id == PA_F16 ? 1 : 2);
            // over a bf16 cache, O that is not finite while the probabilities and their
            // sum are means the row weighed a V element without an f16 value (O itself
            // cannot overflow: |O| <= l max|v|, far inside fp32)
            const bool watch = kVConv && row_valid && !poisoned && lsum > 0.f && lsum < INFINITY;
            bool unconvertible = false;
#pragma unroll 1
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float o[32];
                tmem_ld32(o_col + 32 * c4, o);
                if (!row_valid)
                    continue;
                if (watch)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        unconvertible |= !(fabsf(o[i]) < INFINITY);
                if (split) {
                    const int64_t prw = qrow * p.max_parts + part;
                    store_row32(p.part_o, prw * D + 32 * c4, o, inv, poisoned, 0);
                    if (c4 == 0) {
                        p.part_ml[prw * 2 + 0] = poisoned ? __int_as_float(0x7fc00000) : m_ref;
                        p.part_ml[prw * 2 + 1] = lsum;
                    }
                } else {
                    store_row32(p.out, qrow * D + 32 * c4, o, inv, poisoned, which);
                }
            }
            if (kVConv && __any_sync(kFullMask, unconvertible) && lane == 0)
                atomicOr(p.err, PA_DEVERR_RANGE);
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, Sm::kTmemCols);
    }
}

// Merges the partitions of a split chunk launch: one CTA of D threads per
// (query row, query head); grid = (rows, num_q_heads).
template <typename T, int D>
__global__ void __launch_bounds__(D) chunk_reduce_kernel(const ChunkParams p)
{
    const int64_t row = blockIdx.x;
    const int h = blockIdx.y;
    const int d = threadIdx.x;
    // the sequence owning the row: query_start[s] <= row < query_start[s + 1]
    int lo = 0, hi = p.num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.query_start[mid] <= row)
            lo = mid;
        else
            hi = mid;
    }
    const int s = lo;
    const int qs0 = p.query_start[s], qs1 = p.query_start[s + 1];
    const int n = qs1 - qs0;
    const int L = p.context_lens[s];
    const int64_t idx = (row * p.num_q_heads + h) * D + d;
    float out;
    if (row < qs0 || row >= qs1 || n > L || L < 0 || L > p.max_context_len || n > p.max_query_len) {
        out = __int_as_float(0x7fc00000);
        if (d == 0 && h == 0)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);
    } else {
        const int pos = L - n + (int)(row - qs0);
        const int nparts = min(p.max_parts, (pos + p.partition_tokens) / p.partition_tokens);
        const int64_t prow0 = (row * p.num_q_heads + h) * p.max_parts;
        float M = -INFINITY;
        for (int k = 0; k < nparts; ++k)
            M = fmaxf(M, p.part_ml[(prow0 + k) * 2]);
        float num = 0.f, den = 0.f;
        for (int k = 0; k < nparts; ++k) {
            const float mk = p.part_ml[(prow0 + k) * 2];
            const float w = mk == -INFINITY ? 0.f : exp2f(mk - M) * p.part_ml[(prow0 + k) * 2 + 1];
            num = fmaf(w, p.part_o[(prow0 + k) * D + d], num);
            den += w;
        }
        // a poisoned partition (NaN) makes the row NaN; no visible token gives 0
        out = den > 0.f ? num / den : (den == 0.f ? 0.f : __int_as_float(0x7fc00000));
    }
    if (p.out_f32)
        store_as(static_cast<float*>(p.out) + idx, out);
    else
        store_as(static_cast<T*>(p.out) + idx, out);
}

}  // namespace pa
