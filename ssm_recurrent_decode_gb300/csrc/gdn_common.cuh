// gdn_common.cuh -- device helpers shared by the decode kernels (internal to libgdn_decode.so).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_decode.h"

namespace gdn {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------------------------
// element conversion
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// four consecutive elements -> float4 (the pointer is 4-element aligned)
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const bf16 *p)
{
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    float4 r;
    r.x = __uint_as_float(raw.x << 16);
    r.y = __uint_as_float(raw.x & 0xFFFF0000u);
    r.z = __uint_as_float(raw.y << 16);
    r.w = __uint_as_float(raw.y & 0xFFFF0000u);
    return r;
}

template <typename T> __device__ __forceinline__ void store4(T *p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *p, float4 v)
{
    *reinterpret_cast<float4 *>(p) = v;
}
template <> __device__ __forceinline__ void store4<bf16>(bf16 *p, float4 v)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&lo);
    raw.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// ---------------------------------------------------------------------------------------------
// streaming state access: the state is touched once per call, so it should not displace the
// small, reused inputs in L1/L2 (evict-first policy on both loads and stores)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ void st_stream(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

// bf16 state storage: four consecutive values as one 8-byte access, widened to / rounded from fp32
__device__ __forceinline__ float4 ld_stream(const bf16 *p)
{
    const uint2 raw = __ldcs(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}
__device__ __forceinline__ void st_stream(bf16 *p, float4 v)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&lo);
    raw.y = *reinterpret_cast<uint32_t *>(&hi);
    __stcs(reinterpret_cast<uint2 *>(p), raw);
}

// ---------------------------------------------------------------------------------------------
// small vector arithmetic
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float dot4(float4 a, float4 b)
{
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float4 scale4(float4 a, float s)
{
    return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b)
{
    return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}
// s * a + d * k, elementwise
__device__ __forceinline__ float4 axpby4(float s, float4 a, float d, float4 k)
{
    return make_float4(fmaf(d, k.x, s * a.x), fmaf(d, k.y, s * a.y), fmaf(d, k.z, s * a.z),
                       fmaf(d, k.w, s * a.w));
}
// a * x + d * k, elementwise with a per-element decay a
__device__ __forceinline__ float4 decay_update4(float4 a, float4 x, float d, float4 k)
{
    return make_float4(fmaf(d, k.x, a.x * x.x), fmaf(d, k.y, a.y * x.y), fmaf(d, k.z, a.z * x.z),
                       fmaf(d, k.w, a.w * x.w));
}

// sum over aligned groups of LANES consecutive lanes (LANES a power of two <= 32)
template <int LANES> __device__ __forceinline__ float group_sum(float x)
{
#pragma unroll
    for (int off = LANES / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    return x;
}

// ---------------------------------------------------------------------------------------------
// scalar gate functions
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float softplus_f(float x)
{
    // log(1 + e^x) without overflow: max(x, 0) + log1p(e^-|x|)
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ void raise_flag(int32_t *err, int32_t bit)
{
    if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------------------------
// index checks of the debug build (-DGDN_DEBUG): GDN_IN(err, i, n) is true when 0 <= i < n;
// otherwise it ORs GDN_DEVERR_RANGE into err and is false, and the caller skips the access. In
// the release build it is the constant true and costs nothing.
// ---------------------------------------------------------------------------------------------
#ifdef GDN_DEBUG
__device__ __forceinline__ bool index_in_range(int32_t *err, long long i, long long n)
{
    if (i >= 0 && i < n) return true;
    raise_flag(err, GDN_DEVERR_RANGE);
    return false;
}
#define GDN_IN(err, i, n) (::gdn::index_in_range((err), (long long)(i), (long long)(n)))
#else
#define GDN_IN(err, i, n) (true)
#endif

}  // namespace gdn
