// decode_kernel.cuh -- paged decode attention kernels (sm_103a).
//
// What is computed ("PagedAttention 完全拆解", section 原理详解（二）：块式注意力的数学):
// for sequence s and query head h, with kv head h / group,
//     a_t = exp(scale q.k_t) / sum_u exp(scale q.k_u),   o = sum_t a_t v_t,
// where k_t, v_t are read from physical block block_tables[s][t / B], slot t % B
// (iaim.asia/ai-infra/182, section KV Cache 如何按块分配).  The block-wise form
// on the first page shows the sum may be taken block by block with no
// approximation; we use the running-max form (online softmax, iaim.asia page,
// section vLLM 内核里的缓解写法) so every K/V byte is read exactly once.
//
// GB300 design:
//   * CTA = (partition, kv head x query-head chunk, sequence).  All GC query
//     heads of a chunk share one pass over the kv head's blocks, so with GQA a
//     K/V tile is read from HBM once per group, not once per query head.  A
//     one-pass grid of several waves may take its sequences from a longest-first
//     order (seq_order.cu): CTA row z then serves the z-th sequence of it.
//   * Warp NCW is the producer: it prefetches the CTA's block-table slice
//     (int32, 32 entries per coalesced load, one round ahead), turns each entry
//     into an int64 address and issues one 1-D bulk TMA copy per K tile and per
//     V tile ([B][D] is contiguous in the pool) into an NSTAGE-deep shared-memory
//     ring guarded by full/empty mbarriers.  No register staging, no address
//     arithmetic in the consumers.
//   * Warps 0..NCW-1 consume tiles round-robin (tile i -> warp i % NCW).  Each
//     lane owns D/32 contiguous head dims.  Scores: per-token partial dots
//     reduced by a transposed butterfly (one shuffle per value per halving step,
//     instead of a full warp reduction per token).  Online softmax in base 2
//     (scale * log2 e is folded into q), fp32 everywhere.  P is published through
//     shared memory and P.V accumulates in registers.
//   * Each warp keeps its own (max, sum, acc); the warps are merged through
//     shared memory at the end in a fixed order, so the result depends only on
//     logical token positions, never on physical block ids.
//   * Split contexts write a normalised partial row plus (max, sum) per
//     partition; reduce_kernel merges them.
//   * Masking of the ragged last block is done by select (score = -inf, and the
//     P.V loop stops at the last valid token) so NaN-filled unused slots never
//     reach the arithmetic.
#pragma once

#include <math.h>

#include <mutex>
#include <utility>
#include <vector>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Sums v[0..N-1] over the 32 lanes of the warp.  On return, lane l holds the
// full sum of value index (l >> (5 - log2 N)).  Each halving step exchanges
// half of the remaining values with the partner lane, so N values cost
// N - 1 + (5 - log2 N) shuffles instead of 5N.
template <int N>
__device__ __forceinline__ float butterfly_sum(float (&v)[N], int lane)
{
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
    int mask = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1) {
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, mask);
        }
        mask >>= 1;
    }
    float r = v[0];
#pragma unroll
    for (; mask >= 1; mask >>= 1)
        r += __shfl_xor_sync(kFullMask, r, mask);
    return r;
}

template <int N>
struct Log2 {
    static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

template <typename T, int D, int BS, int GC, int NSTAGE>
struct DecodeSmem {
    static constexpr int kTile = BS * D;                       // elements of one K or V tile
    static constexpr int kTileBytes = kTile * (int)sizeof(T);
    static constexpr int kRingBytes = NSTAGE * 2 * kTileBytes;
    static constexpr int kBarOffset = kRingBytes;              // full[NSTAGE], empty[NSTAGE]
    static constexpr int kOkOffset = kBarOffset + 2 * NSTAGE * 8;
    static constexpr int kFlagOffset = kOkOffset + NSTAGE * 4;
    static constexpr int kPOffset = (kFlagOffset + 4 + 15) / 16 * 16;
    static constexpr int kPBytes = kDecodeConsumerWarps * GC * BS * 4;
    static constexpr int kAccOffset = kPOffset + kPBytes;
    static constexpr int kAccBytes = kDecodeConsumerWarps * GC * D * 4;
    static constexpr int kMlOffset = kAccOffset + kAccBytes;
    static constexpr int kMlBytes = kDecodeConsumerWarps * GC * 2 * 4;
    static constexpr int kBytes = kMlOffset + kMlBytes;
    static_assert(kTileBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
};

template <typename T>
__device__ __forceinline__ void store_out(const DecodeParams& p, int64_t idx, float x)
{
    if (p.out_f32)
        store_as(reinterpret_cast<float*>(p.out) + idx, x);
    else
        store_as(reinterpret_cast<T*>(p.out) + idx, x);
}

// The sequence a decode CTA serves (x) and its context length (y): CTA row z serves
// sequence z, or the z-th of the longest-first order when the call built one.
__device__ __forceinline__ int2 decode_seq(const DecodeParams& p)
{
    if (p.seq_order) {
        const int2 e = p.seq_order[blockIdx.z];
        if ((unsigned)e.x < (unsigned)p.num_seqs)   // always, unless the lengths were
            return e;                               // changed while the order was built
    }
    return make_int2((int)blockIdx.z, p.context_lens[blockIdx.z]);
}

// T: query / native output type.  TK: cache element type (T itself, or
// __nv_fp8_e4m3 for a quantised cache whose value is code * per-kv-head scale).
template <typename T, typename TK, int D, int BS, int GC, int NSTAGE>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_kernel(const DecodeParams p)
{
    using Smem = DecodeSmem<TK, D, BS, GC, NSTAGE>;
    constexpr bool kFp8 = sizeof(TK) == 1;
    constexpr int NCW = kDecodeConsumerWarps;
    constexpr int E = D / 32;                  // head dims per lane
    constexpr int TC = BS < 8 ? BS : 8;        // tokens per butterfly
    constexpr int NCH = BS / TC;               // butterflies per tile
    constexpr int TOK_SHIFT = 5 - Log2<TC>::value;
    constexpr int kTile = Smem::kTile;
    static_assert(D % 32 == 0 && (E == 2 || E == 4), "head_dim must be 64 or 128");
    static_assert(NSTAGE % NCW == 0, "each ring stage must belong to one consumer warp");
    // copy a tile to registers and release its stage early when K + V take <= 64 registers
    constexpr bool kEarlyRelease = 2 * BS * E * (int)sizeof(TK) / 4 <= 64;

    extern __shared__ __align__(128) unsigned char smem[];
    TK* ring = reinterpret_cast<TK*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NSTAGE;
    int* stage_ok = reinterpret_cast<int*>(smem + Smem::kOkOffset);
    int* poison = reinterpret_cast<int*>(smem + Smem::kFlagOffset);
    float* pbuf = reinterpret_cast<float*>(smem + Smem::kPOffset);
    float* mrg_acc = reinterpret_cast<float*>(smem + Smem::kAccOffset);
    float* mrg_ml = reinterpret_cast<float*>(smem + Smem::kMlOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int2 seq_len = decode_seq(p);
    const int seq = seq_len.x;
    const int kvh = blockIdx.y / p.chunks;
    const int h0 = kvh * p.group + (blockIdx.y % p.chunks) * GC;
    const int part = blockIdx.x;
    const bool split = p.partition_tokens > 0;

    const int L = seq_len.y;
    if (L < 0 || L > p.max_context_len) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(p.err, PA_DEVERR_CONTEXT_LEN);
        if (!split) {                             // the reduce pass handles split calls
            for (int idx = threadIdx.x; idx < GC * D; idx += blockDim.x)
                store_out<T>(p, ((int64_t)seq * p.num_q_heads + h0) * D + idx,
                             __int_as_float(0x7fc00000));
        }
        return;
    }
    int t0 = 0, t1 = L;
    if (split) {
        t0 = part * p.partition_tokens;
        if (t0 >= L)
            return;                               // this partition lies past the context
        t1 = min(L, t0 + p.partition_tokens);
    }
    const int jb = t0 / BS;                       // partitions start on block boundaries
    const int ntiles = (t1 > t0) ? (t1 + BS - 1) / BS - jb : 0;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *poison = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // test hook (off unless armed on the host): the chosen CTA's producer issues no copy
    // at all, so nothing is ever in flight for it, and its consumers' waits give up after
    // fault_wait_ns; every other CTA runs as usual
    const bool fault = p.fault_cta > 0 &&
                       (int64_t)blockIdx.x + (int64_t)gridDim.x *
                                                 ((int64_t)blockIdx.y + (int64_t)gridDim.y * blockIdx.z) ==
                           (int64_t)p.fault_cta - 1;
    const uint64_t wait_limit = fault ? (uint64_t)p.fault_wait_ns : kWaitLimitNs;

    if (warp == NCW) {
        // ------------------------------------------------------------------ producer
        if (fault)
            return;
        const int32_t* bt_row = p.block_tables + (int64_t)seq * p.bt_stride + jb;
        const TK* kpool = reinterpret_cast<const TK*>(p.k_cache) + (int64_t)kvh * kTile;
        const TK* vpool = reinterpret_cast<const TK*>(p.v_cache) + (int64_t)kvh * kTile;
        const int64_t blk_stride = (int64_t)p.num_kv_heads * kTile;
        const uint64_t policy = l2_evict_first_policy();
        int next = (lane < ntiles) ? __ldg(bt_row + lane) : 0;
        bool aborted = false;
        for (int base = 0; base < ntiles && !aborted; base += 32) {
            const int cur = next;
            if (base + 32 + lane < ntiles)
                next = __ldg(bt_row + base + 32 + lane);   // next round, in flight meanwhile
            const int cnt = min(32, ntiles - base);
            for (int i = 0; i < cnt; ++i) {
                const int pbn = __shfl_sync(kFullMask, cur, i);
                const int it = base + i;
                const int stage = it % NSTAGE;
                int ok = 1;
                if (lane == 0) {
                    if (it >= NSTAGE && !mbar_wait(&empty[stage], ((it / NSTAGE) - 1) & 1)) {
                        atomicOr(p.err, PA_DEVERR_TIMEOUT);
                        ok = 0;
                    }
                    if (ok) {
                        const bool valid = pbn >= 0 && (int64_t)pbn < p.num_blocks;
                        stage_ok[stage] = valid ? 1 : 0;
                        if (valid) {
                            const int64_t off = (int64_t)pbn * blk_stride;
                            TK* dst = ring + stage * 2 * kTile;
                            mbar_arrive_expect_tx(&full[stage], 2u * Smem::kTileBytes);
                            bulk_g2s(dst, kpool + off, Smem::kTileBytes, &full[stage], policy);
                            bulk_g2s(dst + kTile, vpool + off, Smem::kTileBytes, &full[stage], policy);
                        } else {
                            atomicOr(p.err, PA_DEVERR_BLOCK_ID);
                            mbar_arrive(&full[stage]);
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
    // q carries the softmax scale (base 2) and, for a quantised cache, the K scale
    const float qscale = kFp8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
    float qf[GC][E];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        const T* qp = reinterpret_cast<const T*>(p.q) + ((int64_t)seq * p.num_q_heads + h0 + g) * D +
                      lane * E;
        Load<T, E>::run(qp, qf[g]);
#pragma unroll
        for (int e = 0; e < E; ++e)
            qf[g][e] *= qscale;
    }
    float m[GC], lsum[GC], acc[GC][E];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        m[g] = -INFINITY;
        lsum[g] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[g][e] = 0.f;
    }
    bool poisoned = false;
    float* my_p = pbuf + warp * GC * BS;
    const int mytok = lane >> TOK_SHIFT;

    for (int it = warp; it < ntiles; it += NCW) {
        const int stage = it % NSTAGE;
        if (!mbar_wait(&full[stage], (it / NSTAGE) & 1, wait_limit)) {
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
        const TK* Ks = ring + stage * 2 * kTile;
        const TK* Vs = Ks + kTile;
        const int nvalid = min(BS, t1 - (jb + it) * BS);

        // Small tiles are copied to registers and the stage is released at once, so
        // the producer refills it while this warp computes (the stage would
        // otherwise be held through the whole tile's arithmetic).
        Raw<TK, E> kr[kEarlyRelease ? BS : 1], vr[kEarlyRelease ? BS : 1];
        if constexpr (kEarlyRelease) {
#pragma unroll
            for (int t = 0; t < BS; ++t) {
                load_raw<TK, E>(Ks + t * D + lane * E, kr[t]);
                load_raw<TK, E>(Vs + t * D + lane * E, vr[t]);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
        }
        auto k_row = [&](int t, float (&f)[E]) {
            if constexpr (kEarlyRelease)
                raw_to_float<TK, E>(kr[t], f);
            else
                Load<TK, E>::run(Ks + t * D + lane * E, f);
        };
        auto v_row = [&](int t, float (&f)[E]) {
            if constexpr (kEarlyRelease)
                raw_to_float<TK, E>(vr[t], f);
            else
                Load<TK, E>::run(Vs + t * D + lane * E, f);
        };

        // scores s[g][c] for token c * TC + mytok, base-2 units
        float s[GC][NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float kf[TC][E];
#pragma unroll
            for (int tt = 0; tt < TC; ++tt)
                k_row(c * TC + tt, kf[tt]);
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                float part_dot[TC];
#pragma unroll
                for (int tt = 0; tt < TC; ++tt) {
                    // pairs of head dims accumulate in packed fp32, then the two halves add
                    float2 a2 = fmul2(make_float2(qf[g][0], qf[g][1]),
                                      make_float2(kf[tt][0], kf[tt][1]));
#pragma unroll
                    for (int e = 2; e < E; e += 2)
                        a2 = ffma2(make_float2(qf[g][e], qf[g][e + 1]),
                                   make_float2(kf[tt][e], kf[tt][e + 1]), a2);
                    part_dot[tt] = a2.x + a2.y;
                }
                s[g][c] = butterfly_sum<TC>(part_dot, lane);
            }
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c)
            if (c * TC + mytok >= nvalid) {
#pragma unroll
                for (int g = 0; g < GC; ++g)
                    s[g][c] = -INFINITY;
            }

        // online softmax update per head
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            float tmax = s[g][0];
#pragma unroll
            for (int c = 1; c < NCH; ++c)
                tmax = fmaxf(tmax, s[g][c]);
#pragma unroll
            for (int msk = 16; msk >= (1 << TOK_SHIFT); msk >>= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, msk));
            const float mnew = fmaxf(m[g], tmax);        // finite: nvalid >= 1
            const float alpha = exp2f(m[g] - mnew);       // 0 on the first tile
            m[g] = mnew;
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                s[g][c] = exp2f(s[g][c] - mnew);
                psum += s[g][c];
            }
            lsum[g] = fmaf(lsum[g], alpha, psum);
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                const float2 r = fmul2(make_float2(acc[g][e], acc[g][e + 1]),
                                       make_float2(alpha, alpha));
                acc[g][e] = r.x;
                acc[g][e + 1] = r.y;
            }
            if ((lane & ((1 << TOK_SHIFT) - 1)) == 0) {
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    my_p[g * BS + c * TC + mytok] = s[g][c];
            }
        }
        __syncwarp();

        // acc += P . V over the valid tokens of the tile
#pragma unroll
        for (int t4 = 0; t4 < BS; t4 += 4) {
            if (t4 < nvalid) {
                float4 pv[GC];
#pragma unroll
                for (int g = 0; g < GC; ++g)
                    pv[g] = *reinterpret_cast<const float4*>(my_p + g * BS + t4);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (t4 + u < nvalid) {
                        float vf[E];
                        v_row(t4 + u, vf);
#pragma unroll
                        for (int g = 0; g < GC; ++g) {
                            const float pt = u == 0 ? pv[g].x : u == 1 ? pv[g].y : u == 2 ? pv[g].z : pv[g].w;
#pragma unroll
                            for (int e = 0; e < E; e += 2) {
                                const float2 r = ffma2(make_float2(pt, pt),
                                                       make_float2(vf[e], vf[e + 1]),
                                                       make_float2(acc[g][e], acc[g][e + 1]));
                                acc[g][e] = r.x;
                                acc[g][e + 1] = r.y;
                            }
                        }
                    }
                }
            }
        }
        if constexpr (!kEarlyRelease) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
        }
    }

    // ------------------------------------------------------------- merge the warps
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        float l = lsum[g];
#pragma unroll
        for (int msk = 16; msk >= (1 << TOK_SHIFT); msk >>= 1)
            l += __shfl_xor_sync(kFullMask, l, msk);
        if (lane == 0) {
            mrg_ml[(warp * GC + g) * 2 + 0] = m[g];
            mrg_ml[(warp * GC + g) * 2 + 1] = l;
        }
#pragma unroll
        for (int e = 0; e < E; ++e)
            mrg_acc[(warp * GC + g) * D + lane * E + e] = acc[g][e];
    }
    if (poisoned)
        *poison = 1;
    named_barrier(1, NCW * 32);

    const bool bad = *poison != 0;
    const float oscale = kFp8 ? p.v_scale[kvh] : 1.f;     // V scale of a quantised cache
    for (int idx = threadIdx.x; idx < GC * D; idx += NCW * 32) {
        const int g = idx / D;
        const int d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w)
            M = fmaxf(M, mrg_ml[(w * GC + g) * 2]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float c = exp2f(mrg_ml[(w * GC + g) * 2] - M);
                num = fmaf(c, mrg_acc[(w * GC + g) * D + d], num);
                den = fmaf(c, mrg_ml[(w * GC + g) * 2 + 1], den);
            }
        }
        float o = den > 0.f ? num / den : 0.f;
        if constexpr (kFp8)
            o *= oscale;
        if (bad)
            o = __int_as_float(0x7fc00000);
        const int64_t row = (int64_t)seq * p.num_q_heads + h0 + g;
        if (split) {
            const int64_t prow = row * p.max_parts + part;
            p.part_o[prow * D + d] = o;
            if (d == 0) {
                p.part_ml[prow * 2 + 0] = M;
                p.part_ml[prow * 2 + 1] = den;
            }
        } else {
            store_out<T>(p, row * D + d, o);
        }
    }
}

// Second pass of a split call: merges the partitions of one (sequence, query
// head).  With per-partition maxima m_p, sums l_p and normalised rows o_p:
//   M = max m_p,  w_p = 2^(m_p - M) l_p,  o = sum w_p o_p / sum w_p.
// Launched with D threads per CTA, grid (num_q_heads, num_seqs).
template <typename T, int D>
__global__ void __launch_bounds__(D) reduce_kernel(const DecodeParams p)
{
    const int h = blockIdx.x;
    const int seq = blockIdx.y;
    const int d = threadIdx.x;
    const int64_t row = (int64_t)seq * p.num_q_heads + h;
    const int L = p.context_lens[seq];
    if (L < 0 || L > p.max_context_len) {
        store_out<T>(p, row * D + d, __int_as_float(0x7fc00000));
        return;
    }
    const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
    const float* ml = p.part_ml + row * p.max_parts * 2;
    const float* po = p.part_o + row * p.max_parts * D + d;
    float M = -INFINITY;
    for (int i = 0; i < nparts; ++i)
        M = fmaxf(M, ml[2 * i]);
    float num = 0.f, den = 0.f;
    for (int i = 0; i < nparts; ++i) {
        const float w = exp2f(ml[2 * i] - M) * ml[2 * i + 1];
        num = fmaf(w, po[(int64_t)i * D], num);
        den += w;
    }
    // no visible token gives 0; a NaN partition (poisoned, or NaN scores) makes the row NaN
    store_out<T>(p, row * D + d, den > 0.f ? num / den : (den == 0.f ? 0.f : __int_as_float(0x7fc00000)));
}

// Ring depth: a multiple of the consumer-warp count (about 64 KB of K/V per CTA,
// 1 to 3 stages per warp).  Because tile i uses stage i % NSTAGE and is consumed
// by warp i % NCW, NCW | NSTAGE makes every stage belong to exactly one warp,
// which consumes its rounds in order.  So a consumer never waits on a phase more
// than one ahead of its barrier, and parity waits are exact.  (With NSTAGE not a
// multiple of NCW, two warps can hold different rounds of one stage at once and
// a parity wait can succeed a full phase early.)
template <typename T, int D, int BS>
struct DecodeStages {
    static constexpr int kStageBytes = 2 * BS * D * (int)sizeof(T);   // T: cache element type
    static constexpr int kPerWarp = 65536 / (kDecodeConsumerWarps * kStageBytes);
    static constexpr int value =
        kDecodeConsumerWarps * (kPerWarp < 1 ? 1 : (kPerWarp > 3 ? 3 : kPerWarp));
};

// Resident CTAs per SM for a decode kernel with this dynamic shared memory.
inline int kernel_occupancy(const void* kernel, int smem_bytes)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kDecodeThreads, smem_bytes) !=
        cudaSuccess)
        return 0;
    return n;
}

template <typename T, typename TK, int D, int BS, int GC>
struct CoreVariant {
    static constexpr int kStages = DecodeStages<TK, D, BS>::value;
    using Smem = DecodeSmem<TK, D, BS, GC, kStages>;
    static constexpr auto kernel() { return decode_kernel<T, TK, D, BS, GC, kStages>; }
    static cudaError_t configure()
    {
        return configure_once(reinterpret_cast<const void*>(kernel()), Smem::kBytes);
    }
    static cudaError_t launch(const DecodeParams& p, cudaStream_t stream)
    {
        cudaError_t err = configure();
        if (err != cudaSuccess)
            return err;
        const bool split = p.partition_tokens > 0;
        dim3 grid(split ? p.max_parts : 1, p.num_kv_heads * p.chunks, p.num_seqs);
        kernel()<<<grid, kDecodeThreads, Smem::kBytes, stream>>>(p);
        err = cudaGetLastError();
        if (err != cudaSuccess || !split)
            return err;
        reduce_kernel<T, D><<<dim3(p.num_q_heads, p.num_seqs), D, 0, stream>>>(p);
        return cudaGetLastError();
    }
};

#define PA_CORE_VARIANTS(X)                                                              \
    X(128, 16, 1) X(128, 16, 2) X(128, 16, 4) X(128, 16, 8) X(128, 32, 1) X(128, 32, 2) \
    X(128, 32, 4) X(128, 32, 8) X(64, 16, 1) X(64, 16, 2) X(64, 16, 4) X(64, 16, 8)     \
    X(64, 32, 1) X(64, 32, 2) X(64, 32, 4) X(64, 32, 8)

// Whether the CUDA-core kernel serves this many heads per CTA for cache type TK:
// 16-bit and E4M3 caches use the tensor-core kernel from kMmaMinHeads heads on,
// so those variants are never built.
template <typename TK, int GC>
constexpr bool core_serves() { return sizeof(TK) == 4 || GC < kMmaMinHeads; }

template <typename T, typename TK, int D, int BS, int GC>
cudaError_t launch_core(const DecodeParams& p, cudaStream_t stream)
{
    if constexpr (core_serves<TK, GC>())
        return CoreVariant<T, TK, D, BS, GC>::launch(p, stream);
    else
        return cudaErrorInvalidValue;
}

template <typename T, typename TK, int D, int BS, int GC>
int occupancy_core()
{
    if constexpr (core_serves<TK, GC>()) {
        using V = CoreVariant<T, TK, D, BS, GC>;
        return V::configure() == cudaSuccess
                   ? kernel_occupancy(reinterpret_cast<const void*>(V::kernel()), V::Smem::kBytes)
                   : 0;
    } else {
        return 0;
    }
}

template <typename T, typename TK = T>
cudaError_t launch_decode_typed(const DecodeParams& p, int head_dim, int block_size, int gc,
                                cudaStream_t stream)
{
#define PA_CORE_CASE(D_, BS_, GC_)                                   \
    if (head_dim == D_ && block_size == BS_ && gc == GC_)            \
        return launch_core<T, TK, D_, BS_, GC_>(p, stream);
    PA_CORE_VARIANTS(PA_CORE_CASE)
#undef PA_CORE_CASE
    return cudaErrorInvalidValue;
}

// Resident CTAs per SM of the CUDA-core kernel for this shape (0 if unknown).
template <typename T, typename TK = T>
int occupancy_decode_typed(int head_dim, int block_size, int gc)
{
#define PA_CORE_OCC(D_, BS_, GC_)                                    \
    if (head_dim == D_ && block_size == BS_ && gc == GC_)            \
        return occupancy_core<T, TK, D_, BS_, GC_>();
    PA_CORE_VARIANTS(PA_CORE_OCC)
#undef PA_CORE_OCC
    return 0;
}

}  // namespace pa
