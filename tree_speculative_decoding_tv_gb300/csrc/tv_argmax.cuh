// Vocab-argmax building blocks of the acceptance kernels (tv_accept.cu).
//
// A row's argmax is the position of its largest logit, NaN counting above every value,
// equal values to the smaller index (the acceptance rule's target token).  Every partial
// result is one 64-bit key whose unsigned order is that order, so partials combine with
// max (and with a 64-bit atomicMax across CTAs).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tv {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Streaming 16-byte load (evict-first); volatile so a batch of them is issued back to back.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 64-bit key whose unsigned order is the argmax order: the value's rank in the
// high half (every NaN ranks highest, -0 ranks with +0), then 0xFFFFFFFF - index
// so that equal values favour the smaller index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int i)
{
    const uint32_t u = __float_as_uint(v);
    uint32_t rank;
    if (v != v)
        rank = 0xFFFFFFFFu;
    else if (v == 0.f)
        rank = 0x80000000u;
    else
        rank = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)rank << 32) | (0xFFFFFFFFu - (uint32_t)i);
}

// max with a NaN counting as the largest value
__device__ __forceinline__ float max_nan(float a, float b) { return (a != a) ? a : ((b != b) ? b : fmaxf(a, b)); }

// Order-preserving 32-bit rank of a value (the high half of its key): every NaN
// on top, -0 with +0, never 0.
__device__ __forceinline__ uint32_t value_rank(float v) { return (uint32_t)(argmax_key(v, 0) >> 32); }

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) { return *reinterpret_cast<__nv_bfloat162 *>(&w); }

__device__ __forceinline__ __nv_bfloat162 vec_max2(const uint4 &v)
{
    return __hmax2_nan(__hmax2_nan(as_bf2(v.x), as_bf2(v.y)), __hmax2_nan(as_bf2(v.z), as_bf2(v.w)));
}

}  // namespace tv
