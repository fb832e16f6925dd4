// sdm_rows.cuh -- row helpers of the DW and backward kernels: a lane's 4 or 8 columns of a row (f32 or bf16),
// per-lane cp.async copies into shared memory, and the lane tree that sums a dot's 32 lane partials.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace sdm {
namespace rows {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }

// a lane's 4 columns of a row as floats (read-only data: the non-coherent path)
__device__ __forceinline__ void ld4(const float* p, float (&o)[4]) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
    o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
// a row the same launch rewrites: the coherent L2 path
__device__ __forceinline__ void ld4cg(const float* p, float (&o)[4]) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void ld4cg(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 v = __ldcg(reinterpret_cast<const uint2*>(p));
    o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
    o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
// 4 columns from shared memory
__device__ __forceinline__ void get4(const float* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void get4(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
    o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
// A lane's 4 columns kept in the storage type until used (8 bytes bf16 / 16 bytes f32 of registers).
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
    float4 v;
    __device__ __forceinline__ void zero() { v = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void ld(const float* p) { v = __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ void ld_cg(const float* p) { v = __ldcg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ void get(float (&o)[4]) const { o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w; }
    __device__ __forceinline__ float operator[](int i) const { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct Raw4<__nv_bfloat16> {
    uint2 v;
    __device__ __forceinline__ void zero() { v = make_uint2(0u, 0u); }
    __device__ __forceinline__ void ld(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ void ld_cg(const __nv_bfloat16* p) { v = __ldcg(reinterpret_cast<const uint2*>(p)); }
    __device__ __forceinline__ void get(float (&o)[4]) const {
        o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
        o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
    __device__ __forceinline__ float operator[](int i) const {
        const uint32_t w = i < 2 ? v.x : v.y;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};
// A lane's 8 columns kept in the storage type (16 bytes bf16 / 32 bytes f32 of registers): one
// 16-byte vector access per lane for bfloat16 rows, two for float32.
template <typename T>
struct Raw8;
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void ld(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void ld_cg(const float* p) {
        a = __ldcg(reinterpret_cast<const float4*>(p));
        b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void st(float* p) const {
        reinterpret_cast<float4*>(p)[0] = a;
        reinterpret_cast<float4*>(p)[1] = b;
    }
    __device__ __forceinline__ float operator[](int i) const {
        const float4& q = i < 4 ? a : b;
        const int j = i & 3;
        return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
    }
};
template <>
struct Raw8<__nv_bfloat16> {
    uint4 v;
    __device__ __forceinline__ void ld(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ void ld_cg(const __nv_bfloat16* p) { v = __ldcg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ void st(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = v; }
    __device__ __forceinline__ float operator[](int i) const {
        const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};

// store: f32 as is, bf16 rounded to nearest even
__device__ __forceinline__ void st4(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float (&o)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// store with the streaming hint (evict-first in L2): f32 as is, bf16 rounded to nearest even
__device__ __forceinline__ void st4cs(float* p, const float (&o)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(o[0], o[1], o[2], o[3]));
}
__device__ __forceinline__ void st4cs(__nv_bfloat16* p, const float (&o)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o[2], o[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    __stcs(reinterpret_cast<uint2*>(p), u);
}

// store 8 columns: f32 as is, bf16 rounded to nearest even
__device__ __forceinline__ void st8(float* p, const float (&o)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&o)[8]) {
    uint4 u;
    uint32_t* const w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 x = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&x);
    }
    *reinterpret_cast<uint4*>(p) = u;
}

// Per-lane asynchronous copy of a lane's 4 columns (16 bytes f32, 8 bytes bf16) into shared memory;
// the lane later reads back only what it copied, after cp_wait.
template <typename T>
__device__ __forceinline__ void cp4(T* smem_dst, const T* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    if constexpr (sizeof(T) == 4)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem_src) : "memory");
}
// The same with a zero fill: a lane with `on` false reads nothing and writes zeros.
template <typename T>
__device__ __forceinline__ void cp4z(T* smem_dst, const T* gmem_src, bool on) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    const int n = on ? static_cast<int>(4 * sizeof(T)) : 0;
    if constexpr (sizeof(T) == 4)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem_src), "r"(n) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(d), "l"(gmem_src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A lane's partial of a dot over its 4 columns: one fmaf chain in column order.
__device__ __forceinline__ float dot4(const float (&x)[4], const float (&y)[4]) {
    return fmaf(x[3], y[3], fmaf(x[2], y[2], fmaf(x[1], y[1], x[0] * y[0])));
}

// The sum of x over the 32 lanes, in every lane: lanes paired l, l ^ h for h = 1, 2, 4, 8, 16 (both
// partners add the same two values, so every lane holds the same bits).
__device__ __forceinline__ float allsum(float x) {
#pragma unroll
    for (int k = 1; k <= 16; k <<= 1) x += __shfl_xor_sync(kFull, x, k);
    return x;
}

// 16 values per lane, each summed over the 32 lanes by the tree of allsum, transposed: at level h a
// lane keeps the values whose index bit matches its lane bit and adds its partner's copy, so each
// level halves the values. Lane l returns the sum of value (l & 15): 16 shuffles for 16 sums.
__device__ __forceinline__ float tsum16(const float (&v)[16], int lane) {
    float a[8], b[4], c[2];
    const bool h1 = lane & 1, h2 = lane & 2, h4 = lane & 4, h8 = lane & 8;
#pragma unroll
    for (int m = 0; m < 8; ++m) {   // a[m]: index 2m + (lane & 1)
        const float keep = h1 ? v[2 * m + 1] : v[2 * m], send = h1 ? v[2 * m] : v[2 * m + 1];
        a[m] = keep + __shfl_xor_sync(kFull, send, 1);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {   // b[m]: index 4m + (lane & 3)
        const float keep = h2 ? a[2 * m + 1] : a[2 * m], send = h2 ? a[2 * m] : a[2 * m + 1];
        b[m] = keep + __shfl_xor_sync(kFull, send, 2);
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {   // c[m]: index 8m + (lane & 7)
        const float keep = h4 ? b[2 * m + 1] : b[2 * m], send = h4 ? b[2 * m] : b[2 * m + 1];
        c[m] = keep + __shfl_xor_sync(kFull, send, 4);
    }
    const float keep = h8 ? c[1] : c[0], send = h8 ? c[0] : c[1];
    float x = keep + __shfl_xor_sync(kFull, send, 8);   // index lane & 15
    x += __shfl_xor_sync(kFull, x, 16);
    return x;
}

}  // namespace rows
}  // namespace sdm
