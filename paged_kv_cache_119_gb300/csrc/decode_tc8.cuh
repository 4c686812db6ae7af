// decode_tc8.cuh -- paged decode attention over E4M3 (FP8) caches on the 5th-generation
// tensor cores (tcgen05.mma kind::f8f6f4, sm_103a), head_dim 128.
//
// What it computes: the block-wise attention of "PagedAttention 完全拆解", section
// 原理详解（二）, over a quantised cache (value = code * per-kv-head scale), the same
// result as the CUDA-core and mma.sync decode kernels; with CH, the chunk-row form
// (several new query tokens of a sequence, each masked at its own position).
//
// Why a separate kernel: at one byte per element, converting every cached code to a
// float on the CUDA cores costs more issue slots than HBM time allows, most of all
// for multi-head attention (one query row per kv head).  Here the codes go into the
// tensor core as they are, and the products are transposed so that the 128 tokens
// of a K/V tile sit on the 128 tensor-memory lanes:
//   S^T[128 tok x N] = K[128 tok x 128 dims] . Qt^T    A = the K tile as the TMA wrote
//                                                      it (K-major, 128-byte swizzle)
//   O^T[128 dims x N] = V^T[128 dims x 128 tok] . Pt^T A = the same V tile read
//                                                      MN-major (tokens along K)
// kind::f8f6f4 multiplies E4M3 by E4M3, so the other operand is E4M3 too: query row r
// is written as four E4M3 terms, q * sigma_r = Q0 + Q1/16 + Q2/256 + Q3/4096 (sigma_r a
// power of two that puts max |q| in [128, 256)), in columns 4r .. 4r+3 of Qt; each
// term is the previous remainder times 16, rounded to nearest even, so the four carry
// about 16 significant bits; the last resolves 2^-21 of the scaled row, so a query
// element is exact down to about 2^-21 (bf16) or 2^-18 (f16) of the row's largest, and
// smaller ones keep an error below 2^-29 of it.  The probabilities are
// split the same way, 256 p = P0 + P1/16 + P2/256 + P3/4096, in rows 4r .. 4r+3 of Pt.
// The fp32 results of the term columns are combined with the same weights.
//
// Roles (224 threads):
//   * warps 0 and 6, producers of K and of V: block-table entries and tensor-map TMA of
//     the tile's blocks (box = B tokens x 128 bytes, 128-byte swizzle; the tensor map's
//     third coordinate is block * Hkv + kv head) into rings of NST slots.  A K slot is
//     released when the scores of its tile are computed, a V slot when P.V has read it,
//     so the K loads of later tiles are in flight while a tile is still being softmaxed;
//   * warp 1: allocates the tensor memory; one thread issues the MMAs, whichever is
//     ready: S of the next tile once its K is in, P.V of a tile once its P is written
//     and its V is in;
//   * warps 2-5, one thread per tensor-memory lane: read the scores of their token,
//     exchange per-row tile maxima through shared memory and an mbarrier, online
//     softmax in base 2, write the four P terms, zero the V rows past the range on the
//     last tile (unused slots may hold NaN, and 0 * NaN is NaN); then, as head dim d,
//     read the P.V result of the previous tile and fold it into their accumulators.
// S and O tensor-memory buffers and the Pt buffers alternate between tiles, so the
// softmax of tile i+1 overlaps P.V of tile i.  Every wait is bounded; an invalid
// block id makes the CTA's rows NaN, decided after the final CTA barrier.
#pragma once

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"

namespace pa {

constexpr int kTc8Tok = 128;        // tokens per K/V tile (M of the score product)
constexpr int kTc8Terms = 4;        // E4M3 terms per query row and per probability
constexpr int kTc8Threads = 224;    // K producer, MMA issuer, 4 softmax warps, V producer

template <int R, int NST>
struct Tc8Smem {
    static constexpr int N = kTc8Terms * R < 16 ? 16 : kTc8Terms * R;   // MMA N (16 or 32)
    static constexpr int kTile = kTc8Tok * 128;                         // one K or V tile
    static constexpr int kStage = 2 * kTile;                            // K then V
    static constexpr int kQOff = NST * kStage;                          // Qt: N rows x 128 B
    static constexpr int kPOff = kQOff + N * 128;                       // Pt: 2 x N rows x 128 B
    static constexpr int kRedOff = kPOff + 2 * N * 128;                 // red_max[2][4][R]
    static constexpr int kLOff = kRedOff + 2 * 4 * R * 4;               // red_l[4][R]
    static constexpr int kBarOff = (kLOff + 4 * R * 4 + 7) / 8 * 8;
    // kfull[NST], vfull[NST], kempty[NST], vempty[NST], s_full[2], p_full[2], pv_done[2],
    // red[2], mma_done
    static constexpr int kNumBars = 4 * NST + 9;
    static constexpr int kSlotOff = kBarOff + 8 * kNumBars;             // TMEM address
    static constexpr int kPoisonOff = kSlotOff + 4;
    static constexpr int kBytes = kPoisonOff + 4;
    static constexpr int kAlloc = kBytes + 1024;                        // 1 KB alignment slack
    // tensor memory: S buffers at columns 0 and N, O buffers at 2N and 3N
    static constexpr int kTmemCols = 4 * N < 32 ? 32 : 4 * N;
    static_assert(N == 16 || N == 32, "R = 1, 2, 4 or 8 rows per CTA");
    static_assert((N * 128) % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

// Instruction descriptor of tcgen05.mma kind::f8f6f4, E4M3 x E4M3, fp32 accumulator:
// bits 4-5 accumulator format (1 = f32), 7-9 / 10-12 A / B format (0 = E4M3), bit 15
// A major-ness (1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t mma_idesc_e4m3(int M, int N, bool a_mn_major)
{
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[tmem] = A . B (+ D when accumulate != 0), E4M3 operands in shared memory; one
// k-step covers 32 elements (32 bytes of a K-major row).
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive fp32 columns of this thread's lane, waited for in the same statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[N])
{
    if constexpr (N == 16)
        tmem_ld16(taddr, v);
    else
        tmem_ld32(taddr, v);
}

// (a, b) -> E4M3 codes, round to nearest even, saturating to +-448 (NaN stays NaN):
// a in the low byte, b in the high byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// The values of the two E4M3 codes in the low 16 bits (low byte -> .x); exact.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two_codes)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)(two_codes & 0xffffu)));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Four E4M3 terms of a and of b (|a|, |b| <= 256): x = T0 + T1/16 + T2/256 + T3/4096,
// each term the nearest E4M3 value of 16 x the previous remainder (the remainders are
// exact in fp32).  ta[k] / tb[k] = term k's code.
__device__ __forceinline__ void e4m3_terms(float a, float b, uint32_t (&ta)[kTc8Terms],
                                           uint32_t (&tb)[kTc8Terms])
{
#pragma unroll
    for (int k = 0; k < kTc8Terms; ++k) {
        const uint32_t c = f32x2_to_e4m3x2(a, b);
        ta[k] = c & 0xffu;
        tb[k] = c >> 8;
        if (k + 1 < kTc8Terms) {
            const float2 v = e4m3x2_value(c);
            a = 16.f * (a - v.x);
            b = 16.f * (b - v.y);
        }
    }
}

// Weighted sum of four term columns: c0 + c1/16 + c2/256 + c3/4096 (smallest first).
__device__ __forceinline__ float combine_terms(float c0, float c1, float c2, float c3)
{
    return fmaf(fmaf(fmaf(c3, 0.0625f, c2), 0.0625f, c1), 0.0625f, c0);
}

// Byte offset of element (row, col) of a 128-byte-swizzled operand with 128-byte rows.
__device__ __forceinline__ int sw128_byte(int row, int col)
{
    return row * 128 + ((((col >> 4) ^ row) & 7) << 4) + (col & 15);
}

// T: query / native output type (f16 or bf16).  BS: block size.  R: query rows per CTA
// (decode: R query heads of one kv head; CH: R (chunk token, head) rows of one kv head,
// row R0 + r = token (R0 + r) / group, head (R0 + r) % group).
// grid = (partitions, num_kv_heads * chunks, num_seqs); kTc8Threads threads.
template <typename T, int BS, int R, int NST, bool CH>
__global__ void __launch_bounds__(kTc8Threads, 3)
    decode_tc8_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv)
{
    using Sm = Tc8Smem<R, NST>;
    constexpr int D = 128;
    constexpr int N = Sm::N;
    constexpr int BPT = kTc8Tok / BS;           // cache blocks per tile
    static_assert(BS == 16 || BS == 32, "block_size 16 or 32");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);   // [stage]
    uint64_t* vfull = kfull + NST;
    uint64_t* kempty = vfull + NST;
    uint64_t* vempty = kempty + NST;
    uint64_t* s_full = vempty + NST;            // [S buffer]
    uint64_t* p_full = s_full + 2;              // [P buffer]
    uint64_t* pv_done = p_full + 2;             // [O buffer]
    uint64_t* red_bar = pv_done + 2;            // [exchange buffer]
    uint64_t* mma_done = red_bar + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Sm::kSlotOff);
    int* poison = reinterpret_cast<int*>(smem + Sm::kPoisonOff);
    float* red_max = reinterpret_cast<float*>(smem + Sm::kRedOff);   // [2][4][R]
    float* red_l = reinterpret_cast<float*>(smem + Sm::kLOff);       // [4][R]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y / p.chunks;
    const int R0 = (blockIdx.y - kvh * p.chunks) * R;
    const int part = blockIdx.x;
    const bool split = p.partition_tokens > 0;

    const int L = p.context_lens[seq];
    int qs0 = 0, n = 1;
    if constexpr (CH) {
        qs0 = p.query_start[seq];
        n = p.query_start[seq + 1] - qs0;
    }
    // the q / out row of CTA row r, or -1 for a padding row
    auto out_row = [&](int r) -> int64_t {
        if constexpr (CH) {
            const int rr = R0 + r;
            const int j = rr / p.group;
            return j < n ? (int64_t)(qs0 + j) * p.num_q_heads + (int64_t)kvh * p.group + (rr - j * p.group)
                         : -1;
        } else {
            return (int64_t)seq * p.num_q_heads + (int64_t)kvh * p.group + R0 + r;
        }
    };
    const bool rows_sane = !CH || (qs0 >= 0 && n >= 0 && (int64_t)qs0 + n <= p.num_rows);
    if (L < 0 || L > p.max_context_len || !rows_sane || (CH && (n > L || n > p.max_query_len))) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);
        if (!split && rows_sane) {
            for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
                const int64_t row = out_row(idx / D);
                if (row >= 0)
                    store_out<T>(p, row * D + idx % D, __int_as_float(0x7fc00000));
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
        t_end = L - n + min(n - 1, (R0 + R - 1) / p.group) + 1;   // last row's position + 1
    }
    int t0 = 0, t1 = t_end;
    if (split) {
        t0 = part * p.partition_tokens;
        if (t0 >= t_end)
            return;
        t1 = min(t_end, t0 + p.partition_tokens);
    }
    const int ntiles = (t1 - t0 + kTc8Tok - 1) / kTc8Tok;   // 0 only for an empty context

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&vfull[s], 1);
            mbar_init(&kempty[s], 1);
            mbar_init(&vempty[s], 1);
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);
            mbar_init(&pv_done[b], 1);
            mbar_init(&red_bar[b], 4);
        }
        mbar_init(mma_done, 1);
        *poison = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
    }
    __syncthreads();

    // per-row results of the softmax warps, stored after the final CTA barrier
    int64_t orow_e[R];
    float acc_e[R], m_e[R], l_e[R];

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------- producers: K (warp 0), V (warp 6)
        // They start at once (they need neither the tensor memory nor the query terms) and
        // run separately: a K slot is free again as soon as its scores are computed, a V
        // slot only once P.V has read it, so K loads run ahead of V loads.
        const bool is_k = warp == 0;
        const CUtensorMap* map = is_k ? &tk : &tv;
        uint64_t* fullb = is_k ? kfull : vfull;
        uint64_t* emptyb = is_k ? kempty : vempty;
        const int half = is_k ? 0 : Sm::kTile;
        const int32_t* bt_row = p.block_tables + (int64_t)seq * p.bt_stride;
        const uint64_t policy = l2_evict_first_policy();
        const int blk_first = t0 / BS;             // partitions start on block boundaries
        const int nblk = (t1 + BS - 1) / BS - blk_first;
        // block-table entries 32 at a time (4 or 8 tiles), the next 32 in flight while the
        // current ones are used
        int cur = lane < nblk ? __ldg(bt_row + blk_first + lane) : -1;
        int nxt = 32 + lane < nblk ? __ldg(bt_row + blk_first + 32 + lane) : -1;
        int issued = 0;
        for (int it = 0; it < ntiles; ++it) {
            const int st = it % NST;
            const int lb = it * BPT;               // first block of the tile, CTA-relative
            if (it > 0 && (lb & 31) == 0) {
                cur = nxt;
                nxt = lb + 32 + lane < nblk ? __ldg(bt_row + blk_first + lb + 32 + lane) : -1;
            }
            const int nb = min(BPT, nblk - lb);
            const int e = __shfl_sync(kFullMask, cur, ((lb & 31) + lane) & 31);
            int pbn = -1;
            bool valid = false;
            if (lane < nb) {
                pbn = e;
                valid = pbn >= 0 && (int64_t)pbn < p.num_blocks;
            }
            const unsigned vmask = __ballot_sync(kFullMask, valid);
            int ok = 1;
            if (lane == 0) {
                if (it >= NST && !mbar_wait(&emptyb[st], ((it / NST) - 1) & 1)) {
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                    ok = 0;
                } else {
                    const int nvalid = __popc(vmask);
                    if (nvalid != nb) {                // the CTA's rows become NaN
                        atomicOr(p.err, PA_DEVERR_BLOCK_ID);
                        *poison = 1;
                    }
                    mbar_arrive_expect_tx(&fullb[st], (uint32_t)nvalid * BS * 128u);
                }
            }
            if (!__shfl_sync(kFullMask, ok, 0)) {
                if (lane == 0)
                    *poison = 1;
                break;
            }
            if (valid) {
                const int z = pbn * p.num_kv_heads + kvh;     // < 2^31 (checked on the host)
                tma_load_3d(smem + st * Sm::kStage + half + lane * (BS * 128), map, 0, 0, z,
                            &fullb[st], policy);
            }
            issued = it + 1;
        }
        // no copy may still be in flight into this CTA's shared memory at exit
        if (lane == 0)
            for (int it = max(0, issued - NST); it < issued; ++it)
                mbar_wait(&fullb[it % NST], (it / NST) & 1);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        tmem_alloc(tslot, Sm::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
        named_barrier(1, 160);               // tensor memory allocated; Qt written
        tc_fence_after();
        const uint32_t tbase = *tslot;
        if (lane == 0) {
            const uint32_t idesc_s = mma_idesc_e4m3(kTc8Tok, N, false);
            const uint32_t idesc_o = mma_idesc_e4m3(D, N, true);
            const uint32_t qaddr = smem_addr(smem + Sm::kQOff);
            auto issue_scores = [&](int it) {
                const uint32_t kb = smem_addr(smem + (it % NST) * Sm::kStage);
                const uint32_t dcol = tbase + (it & 1) * N;
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk)
                    tc_mma_e4m3(dcol, sw128_desc(kb + kk * 32, 16, 1024),
                                sw128_desc(qaddr + kk * 32, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                tc_commit(&s_full[it & 1]);
                tc_commit(&kempty[it % NST]);  // K of the stage is consumed
            };
            auto issue_pv = [&](int it) {
                const uint32_t vb = smem_addr(smem + (it % NST) * Sm::kStage + Sm::kTile);
                const uint32_t pb = smem_addr(smem + Sm::kPOff + (it & 1) * N * 128);
                const uint32_t ocol = tbase + 2 * N + (it & 1) * N;
#pragma unroll
                for (int kk = 0; kk < kTc8Tok / 32; ++kk)
                    // V^T: 32 tokens per k-step = four 8-token swizzle atoms of 1 KB
                    tc_mma_e4m3(ocol, sw128_desc(vb + kk * 4096, 16, 1024),
                                sw128_desc(pb + kk * 32, 16, 1024), idesc_o, kk > 0 ? 1u : 0u);
                tc_commit(&pv_done[it & 1]);
                tc_commit(&vempty[it % NST]);  // V of the stage is consumed
            };
            // Issue whichever product is ready: the scores of tile ns once its K is in,
            // P.V of tile np once its P is written and its V is in (non-blocking tests:
            // a suspended try_wait on one barrier would hide the other's completion).  P.V never waits for the next
            // tile's data, so a stage goes back to the producer as soon as it is used.
            // S buffer ns&1 is free once P of tile ns-2 was handed over (ns <= np + 1);
            // the O buffer of tile np was read back before P of tile np was.
            bool ok = true;
            int ns = 0, np = 0;
            uint64_t t_last = 0;
            uint32_t spins = 0;
            while (np < ntiles) {
                if (ns < ntiles && ns <= np + 1 && mbar_test_wait(&kfull[ns % NST], (ns / NST) & 1)) {
                    tc_fence_after();
                    issue_scores(ns);
                    ++ns;
                    spins = 0;
                } else if (np < ns && mbar_test_wait(&p_full[np & 1], (np >> 1) & 1) &&
                           mbar_test_wait(&vfull[np % NST], (np / NST) & 1)) {
                    tc_fence_after();
                    issue_pv(np);
                    ++np;
                    spins = 0;
                } else if ((++spins & 255u) == 1u) {
                    const uint64_t now = global_timer_ns();
                    if (spins == 1u)
                        t_last = now;
                    else if (now - t_last > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            tc_commit(mma_done);             // every MMA above completes before TMEM is freed
            mbar_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax and output warps
        const int sw = warp - 2;                     // 0..3
        const int wq = warp & 3;                     // TMEM lane quarter of this warp
        const int tl = 32 * wq + lane;               // TMEM lane: token of a tile / head dim
        int64_t orow[R];
        int lim[R];                                  // last visible position of row r (-1: none)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            orow[r] = out_row(r);
            if constexpr (CH)
                lim[r] = orow[r] >= 0 ? L - n + (R0 + r) / p.group : -1;
            else
                lim[r] = L - 1;
        }
        // ---- query terms into Qt: this thread is head dim tl of every row
        float mult[R];                               // score multiplier (base 2) per row
        {
            float qv[R], am[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                qv[r] = orow[r] >= 0 ? static_cast<float>(reinterpret_cast<const T*>(p.q)[orow[r] * D + tl])
                                     : 0.f;
                am[r] = fabsf(qv[r]);
#pragma unroll
                for (int msk = 16; msk >= 1; msk >>= 1)
                    am[r] = fmaxf(am[r], __shfl_xor_sync(kFullMask, am[r], msk));
                if (lane == 0)
                    red_l[sw * R + r] = am[r];
            }
            named_barrier(2, 128);
            const float ks = p.k_scale[kvh] * p.scale_log2;
            float sg[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float a = fmaxf(fmaxf(red_l[r], red_l[R + r]), fmaxf(red_l[2 * R + r], red_l[3 * R + r]));
                const int e = (__float_as_int(a) >> 23) & 0xff;
                // sigma = 2^(134 - e) puts max |q| in [128, 256) (e >= 8: a row below
                // 2^-119 keeps sigma = 2^126); a NaN or infinite q makes every term NaN,
                // and the row NaN, as in the exact attention
                const int ec = max(e, 8);
                sg[r] = e == 255 ? __int_as_float(0x7fc00000) : __int_as_float((261 - ec) << 23);
                mult[r] = ks * __int_as_float((ec - 7) << 23);                 // ks / sigma
            }
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                uint32_t ta[kTc8Terms], tb[kTc8Terms];
                e4m3_terms(qv[r] * sg[r], r + 1 < R ? qv[r + 1] * sg[r + 1] : 0.f, ta, tb);
#pragma unroll
                for (int k = 0; k < kTc8Terms; ++k) {
                    smem[Sm::kQOff + sw128_byte(kTc8Terms * r + k, tl)] = (unsigned char)ta[k];
                    if (r + 1 < R)
                        smem[Sm::kQOff + sw128_byte(kTc8Terms * (r + 1) + k, tl)] = (unsigned char)tb[k];
                }
            }
            // rows past 4R of Qt and of both Pt buffers stay zero
#pragma unroll
            for (int row = kTc8Terms * R; row < N; ++row) {
                smem[Sm::kQOff + sw128_byte(row, tl)] = 0;
                smem[Sm::kPOff + sw128_byte(row, tl)] = 0;
                smem[Sm::kPOff + N * 128 + sw128_byte(row, tl)] = 0;
            }
        }
        fence_proxy_async_smem();
        named_barrier(1, 160);
        tc_fence_after();
        const uint32_t tbase = *tslot;
        const uint32_t lane_t = tbase + ((uint32_t)(32 * wq) << 16);

        float m[R], lsum[R], acc[R], apend[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            m[r] = -INFINITY;
            lsum[r] = 0.f;
            acc[r] = 0.f;
            apend[r] = 1.f;
        }
        bool poisoned = false, aborted = false;
        // folds P.V of tile i (O^T, this thread = head dim tl) into acc with the
        // rescale factor of that tile
        auto read_back = [&](int i, const float (&al)[R]) {
            if (!mbar_wait(&pv_done[i & 1], (i >> 1) & 1)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                poisoned = aborted = true;
                return;
            }
            tc_fence_after();
            float ov[N];
            tmem_ldn<N>(lane_t + 2 * N + (i & 1) * N, ov);
#pragma unroll
            for (int r = 0; r < R; ++r)
                acc[r] = fmaf(acc[r], al[r],
                              combine_terms(ov[4 * r], ov[4 * r + 1], ov[4 * r + 2], ov[4 * r + 3]));
        };
        for (int it = 0; it < ntiles; ++it) {
            const int b = it & 1;
            const int st = it % NST;
            const int tb = t0 + it * kTc8Tok;
            // the scores imply the tile's K (the K slot may already hold a later tile:
            // neither kfull nor any per-stage word is read here)
            if (!mbar_wait(&s_full[b], (it >> 1) & 1)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                poisoned = aborted = true;
                break;
            }
            tc_fence_after();
            float sv[N];
            tmem_ldn<N>(lane_t + b * N, sv);
            const int pos = tb + tl;                 // this thread's token
            float x[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float s = combine_terms(sv[4 * r], sv[4 * r + 1], sv[4 * r + 2], sv[4 * r + 3]);
                x[r] = (pos < t1 && pos <= lim[r]) ? s * mult[r] : -INFINITY;
                float wmx = x[r];
#pragma unroll
                for (int msk = 16; msk >= 1; msk >>= 1)
                    wmx = fmaxf(wmx, __shfl_xor_sync(kFullMask, wmx, msk));
                if (lane == 0)
                    red_max[(b * 4 + sw) * R + r] = wmx;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&red_bar[b]);
            if (!mbar_wait(&red_bar[b], (it >> 1) & 1)) {
                if (lane == 0)
                    atomicOr(p.err, PA_DEVERR_TIMEOUT);
                poisoned = aborted = true;
                break;
            }
            float al[R];
            uint32_t pt[R][kTc8Terms];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float* rm = red_max + b * 4 * R + r;
                const float tmax = fmaxf(fmaxf(rm[0], rm[R]), fmaxf(rm[2 * R], rm[3 * R]));
                const float mnew = fmaxf(m[r], tmax);
                al[r] = mnew == -INFINITY ? 1.f : ex2_approx(m[r] - mnew);   // 0 on the first tile
                m[r] = mnew;
                // p in [0, 1]; 0 while the row has seen no visible token, NaN for a NaN score
                x[r] = (mnew == -INFINITY && x[r] == -INFINITY) ? 0.f : ex2_approx(x[r] - mnew);
                lsum[r] = fmaf(lsum[r], al[r], x[r]);
            }
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                uint32_t tb2[kTc8Terms];
                e4m3_terms(256.f * x[r], r + 1 < R ? 256.f * x[r + 1] : 0.f, pt[r], tb2);
                if (r + 1 < R)
#pragma unroll
                    for (int k = 0; k < kTc8Terms; ++k)
                        pt[r + 1][k] = tb2[k];
            }
            // byte tl of swizzled row n of Pt: n * 128 + (tl ^ ((n & 7) << 4)) for tl < 128,
            // the same place as sw128_byte(n, tl)
            unsigned char* pbuf = smem + Sm::kPOff + b * N * 128;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int k = 0; k < kTc8Terms; ++k) {
                    const int n = kTc8Terms * r + k;
                    pbuf[n * 128 + (tl ^ ((n & 7) << 4))] = (unsigned char)pt[r][k];
                }
            if (tb + kTc8Tok > t1) {
                // last tile: V rows of tokens past the range (unused slot, missing block,
                // stale tile) become 0, once the tile's V is in (its slot is not reused
                // before this tile's P.V)
                if (!mbar_wait(&vfull[st], (it / NST) & 1)) {
                    if (lane == 0)
                        atomicOr(p.err, PA_DEVERR_TIMEOUT);
                    poisoned = aborted = true;
                    break;
                }
                // rows nv .. 127 are one contiguous span: the 128 threads zero it together,
                // consecutive 16-byte stores (no bank conflicts)
                const int nv = t1 - tb;                  // 1 .. 127 rows of the range
                uint4* vz = reinterpret_cast<uint4*>(smem + st * Sm::kStage + Sm::kTile + nv * 128);
                for (int j = tl; j < (kTc8Tok - nv) * 8; j += kTc8Tok)
                    vz[j] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[b]);
            if (it >= 1) {
                read_back(it - 1, apend);
                if (aborted)
                    break;
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
                apend[r] = al[r];
        }
        if (ntiles > 0 && !aborted)
            read_back(ntiles - 1, apend);

        // ---------------------------------------------------------------- epilogue
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float l = lsum[r];
#pragma unroll
            for (int msk = 16; msk >= 1; msk >>= 1)
                l += __shfl_xor_sync(kFullMask, l, msk);
            lsum[r] = l;
        }
        if (lane == 0)                               // red_l: the query maxima were read before barrier 1
#pragma unroll
            for (int r = 0; r < R; ++r)
                red_l[sw * R + r] = lsum[r];
        if (poisoned)
            *poison = 1;
        named_barrier(2, 128);
        const float vs = p.v_scale[kvh] * (1.f / 256.f);   // P carried 256 p
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float l = (red_l[r] + red_l[R + r]) + (red_l[2 * R + r] + red_l[3 * R + r]);
            orow_e[r] = orow[r];
            m_e[r] = m[r];
            l_e[r] = l;
            acc_e[r] = l == 0.f ? 0.f : acc[r] / l * vs;    // NaN scores keep l NaN
        }
        tc_fence_before();
    }
    // every role is done: the producers' invalid-block flags are visible, the tensor
    // memory is no longer read
    __syncthreads();
    if (warp >= 2 && warp < 6) {
        const bool bad = *poison != 0;
        const int tl = 32 * (warp & 3) + lane;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (orow_e[r] < 0)
                continue;                            // padding row
            const float out = bad ? __int_as_float(0x7fc00000) : acc_e[r];
            if (split) {
                const int64_t prow = orow_e[r] * p.max_parts + part;
                p.part_o[prow * D + tl] = out;
                if (tl == 0) {
                    p.part_ml[prow * 2 + 0] = m_e[r];
                    p.part_ml[prow * 2 + 1] = l_e[r];
                }
            } else {
                store_out<T>(p, orow_e[r] * D + tl, out);
            }
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(*tslot, Sm::kTmemCols);
    }
}

}  // namespace pa
