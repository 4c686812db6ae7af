// pa_device.cuh -- device-side helpers shared by the library's kernels:
// mbarrier and bulk-copy (TMA) PTX wrappers, bounded waits, dtype loads/stores.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr unsigned kFullMask = 0xffffffffu;

// A bounded pipeline wait gives up after this many nanoseconds of %globaltimer.
// No legitimate wait in these kernels comes near it (a whole launch takes well
// under a millisecond); it only turns a lost completion into an error flag.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// (the arrival's phase state is not needed: the sink operand `_` discards it)
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of the phase with the given parity (try_wait may suspend the
// thread for a while, which delays a loop that polls several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// stops waiting) once limit_ns (by default kWaitLimitNs) has passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_timer_ns() - t0 > limit_ns)
            return false;
    }
}

// L2 policy for data read exactly once per launch (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared through the TMA unit; completion is counted in
// bytes on `bar`.  dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tensor-map TMA load into shared memory, completion counted in bytes on `bar`
// (for the caches: x = head dim, y = token in block, z = block * Hkv + head).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// Packed fp32 pair arithmetic (one instruction for two IEEE fp32 operations, each
// rounded to nearest even as its scalar form would be).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 2^x on the MUFU unit, one instruction (relative error about 2^-22, far inside the
// attention tolerance; results below 2^-126 flush to zero, and 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ----------------------------------------------------------------------------- dtypes

template <typename T>
struct DType;
template <>
struct DType<float> {
    static constexpr pa_dtype id = PA_F32;
};
template <>
struct DType<__half> {
    static constexpr pa_dtype id = PA_F16;
};
template <>
struct DType<__nv_bfloat16> {
    static constexpr pa_dtype id = PA_BF16;
};
template <>
struct DType<__nv_fp8_e4m3> {
    static constexpr pa_dtype id = PA_FP8_E4M3;
};

// Two E4M3 codes (low byte first) as two fp32 values; exact.
// Two E4M3 codes (low 16 bits, low byte first) as an f16x2 operand word; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu),
                                                     __NV_E4M3);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_codes, __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads N consecutive elements (N * sizeof(T) bytes, naturally aligned) as fp32.
template <typename T, int N>
struct Load;

template <>
struct Load<__nv_bfloat16, 4> {
    __device__ __forceinline__ static void run(const __nv_bfloat16* p, float (&f)[4])
    {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    }
};
template <>
struct Load<__nv_bfloat16, 2> {
    __device__ __forceinline__ static void run(const __nv_bfloat16* p, float (&f)[2])
    {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        f[0] = bf16_lo(w); f[1] = bf16_hi(w);
    }
};
template <>
struct Load<__half, 4> {
    __device__ __forceinline__ static void run(const __half* p, float (&f)[4])
    {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
};
template <>
struct Load<__half, 2> {
    __device__ __forceinline__ static void run(const __half* p, float (&f)[2])
    {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
        f[0] = a.x; f[1] = a.y;
    }
};
template <>
struct Load<float, 4> {
    __device__ __forceinline__ static void run(const float* p, float (&f)[4])
    {
        const float4 w = *reinterpret_cast<const float4*>(p);
        f[0] = w.x; f[1] = w.y; f[2] = w.z; f[3] = w.w;
    }
};
template <>
struct Load<float, 2> {
    __device__ __forceinline__ static void run(const float* p, float (&f)[2])
    {
        const float2 w = *reinterpret_cast<const float2*>(p);
        f[0] = w.x; f[1] = w.y;
    }
};

template <int N>
struct Load<__nv_fp8_e4m3, N>;   // defined after Raw below

// N consecutive elements of T held as raw 32-bit words (N * sizeof(T) / 4 of them),
// loaded with one vector load and converted to fp32 later.
template <typename T, int N>
struct Raw {
    static constexpr int kBytes = N * (int)sizeof(T);
    static constexpr int W = (kBytes + 3) / 4;
    uint32_t w[W];
};

template <typename T, int N>
__device__ __forceinline__ void load_raw(const T* p, Raw<T, N>& r)
{
    if constexpr (Raw<T, N>::kBytes == 2) {
        r.w[0] = *reinterpret_cast<const uint16_t*>(p);
    } else if constexpr (Raw<T, N>::W == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    } else if constexpr (Raw<T, N>::W == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        r.w[0] = v.x; r.w[1] = v.y;
    } else {
        r.w[0] = *reinterpret_cast<const uint32_t*>(p);
    }
}

template <typename T, int N>
__device__ __forceinline__ void raw_to_float(const Raw<T, N>& r, float (&f)[N])
{
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            f[i] = __uint_as_float(r.w[i]);
    } else if constexpr (sizeof(T) == 1) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 v = e4m3x2_to_float2(r.w[i / 2] >> (16 * (i % 2)));
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    } else if constexpr (DType<T>::id == PA_BF16) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            f[2 * i] = bf16_lo(r.w[i]);
            f[2 * i + 1] = bf16_hi(r.w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&r.w[i]));
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

template <int N>
struct Load<__nv_fp8_e4m3, N> {
    __device__ __forceinline__ static void run(const __nv_fp8_e4m3* p, float (&f)[N])
    {
        Raw<__nv_fp8_e4m3, N> r;
        load_raw<__nv_fp8_e4m3, N>(p, r);
        raw_to_float<__nv_fp8_e4m3, N>(r, f);
    }
};

// Stores one fp32 value as T, rounding to nearest even.
__device__ __forceinline__ void store_as(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

}  // namespace pa
