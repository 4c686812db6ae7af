// seq_order.cu -- the longest-first dispatch order of a one-pass decode.
//
// A decode grid runs one CTA row per sequence, and the hardware starts CTA rows in
// index order.  When the grid holds several waves, a long context whose CTAs start in
// the last wave keeps a few SMs streaming after the rest are idle.  This kernel sorts
// the sequences into kOrderClasses classes of context length, longest class first, and
// writes order[z] = (sequence, context length) for CTA row z.  The sort is stable:
// within a class, sequences keep their index order, so neighbours (e.g. sequences that
// share a prefix and read the same blocks through L2) stay close together.
//
// One CTA of 1024 threads.  Thread t owns the index range [t * per, (t + 1) * per)
// (per = ceil(n / 1024)).  It counts its sequences per class.  A block-wide exclusive
// scan per class gives it the first slot of each class, and it then writes its
// sequences in index order.  Results of the decode do not depend on the order: each
// (sequence, head) is still computed by one CTA.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kOrderThreads = 1024;
constexpr int kOrderWarps = kOrderThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// class 0 holds the longest contexts (within max_len / kOrderClasses of max_len);
// lengths outside [0, max_len] are clamped here and flagged by the decode kernel
__device__ __forceinline__ int length_class(int L, int max_len)
{
    const int64_t c = min(max(L, 0), max_len);
    return (int)((int64_t)(max_len - c) * kOrderClasses / ((int64_t)max_len + 1));
}

__device__ __forceinline__ int warp_inclusive_scan(int x, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFull, x, d);
        if (lane >= d)
            x += y;
    }
    return x;
}

__global__ void __launch_bounds__(kOrderThreads)
    seq_order_kernel(const int32_t* __restrict__ lens, int n, int max_len, int2* __restrict__ order)
{
    static_assert(kOrderClasses <= kOrderWarps, "one warp scans each class");
    static_assert(kOrderWarps <= 32, "one lane per warp total");
    __shared__ int warp_base[kOrderClasses][kOrderWarps];
    __shared__ int class_base[kOrderClasses];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int per = (n + kOrderThreads - 1) / kOrderThreads;
    const int i0 = min(n, t * per), i1 = min(n, i0 + per);

    int cnt[kOrderClasses];
#pragma unroll
    for (int k = 0; k < kOrderClasses; ++k)
        cnt[k] = 0;
    for (int i = i0; i < i1; ++i) {
        const int c = length_class(lens[i], max_len);
#pragma unroll
        for (int k = 0; k < kOrderClasses; ++k)
            cnt[k] += (c == k);
    }
    // slot of this thread's first sequence of class k =
    //   (sequences of longer classes) + (class-k sequences of lower threads)
    int slot[kOrderClasses];
#pragma unroll
    for (int k = 0; k < kOrderClasses; ++k) {
        const int x = warp_inclusive_scan(cnt[k], lane);
        slot[k] = x - cnt[k];
        if (lane == 31)
            warp_base[k][warp] = x;
    }
    __syncthreads();
    if (warp < kOrderClasses) {                    // warp k: the warp totals of class k
        const bool mine = lane < kOrderWarps;      // lanes past the warp count add 0
        const int own = mine ? warp_base[warp][lane] : 0;
        const int x = warp_inclusive_scan(own, lane);
        if (mine)
            warp_base[warp][lane] = x - own;
        if (lane == 31)
            class_base[warp] = x;                  // the class total, for now
    }
    __syncthreads();
    if (t == 0) {
        int s = 0;
        for (int k = 0; k < kOrderClasses; ++k) {
            const int c = class_base[k];
            class_base[k] = s;
            s += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kOrderClasses; ++k)
        slot[k] += class_base[k] + warp_base[k][warp];

    for (int i = i0; i < i1; ++i) {
        const int L = lens[i];
        const int c = length_class(L, max_len);
        int pos = 0;
#pragma unroll
        for (int k = 0; k < kOrderClasses; ++k)
            if (c == k)
                pos = slot[k]++;
        if (pos < n)                               // always, unless lens changes meanwhile
            order[pos] = make_int2(i, L);
    }
}

}  // namespace

cudaError_t launch_seq_order(const int32_t* context_lens, int num_seqs, int max_context_len,
                             int2* order, cudaStream_t stream)
{
    if (num_seqs <= 0)
        return cudaSuccess;
    seq_order_kernel<<<1, kOrderThreads, 0, stream>>>(context_lens, num_seqs, max_context_len,
                                                      order);
    return cudaGetLastError();
}

}  // namespace pa
