// pkv_common.cuh -- device helpers shared by the pkv kernels (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Per-device error word: the first device-data error seen since the last
// pkv_last_device_error() sets flag = 1 and detail = the offending value.
struct DevErr {
    int flag;
    int pad;
    long long detail;
};

__device__ __forceinline__ void record_error(DevErr *e, long long detail) {
    if (atomicCAS(&e->flag, 0, 1) == 0) e->detail = detail;
}

// bf16 pair in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy through L2 only (cp.async.cg); src_bytes = 0
// fills the destination with zeros without reading memory.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes = 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Partial stores with L2 evict_last priority: the merge reads the split-K
// partials after a K/V stream that is usually larger than L2 and would
// otherwise push the early ones out to DRAM.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_keep(float *addr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;\n" ::"l"(addr), "f"(v), "l"(pol) : "memory");
}
// 16-byte aligned float4 store with the same policy
__device__ __forceinline__ void st_keep4(float *addr, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(addr), "f"(a),
                 "f"(b), "f"(c), "f"(d), "l"(pol)
                 : "memory");
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int bytes = 4;
    __device__ static float to_f(float x) { return x; }
    __device__ static float from_f(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int bytes = 2;
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Load N consecutive elements starting at p (N*sizeof(T) is 4, 8 or 16
// bytes and p is aligned to that) and widen to float.
template <typename T, int N>
__device__ __forceinline__ void load_widen(const T *p, float (&out)[N]);

template <>
__device__ __forceinline__ void load_widen<__nv_bfloat16, 2>(const __nv_bfloat16 *p, float (&o)[2]) {
    uint32_t w = *reinterpret_cast<const uint32_t *>(p);
    o[0] = bf16lo(w);
    o[1] = bf16hi(w);
}
template <>
__device__ __forceinline__ void load_widen<__nv_bfloat16, 4>(const __nv_bfloat16 *p, float (&o)[4]) {
    uint2 w = *reinterpret_cast<const uint2 *>(p);
    o[0] = bf16lo(w.x); o[1] = bf16hi(w.x); o[2] = bf16lo(w.y); o[3] = bf16hi(w.y);
}
template <>
__device__ __forceinline__ void load_widen<__nv_bfloat16, 8>(const __nv_bfloat16 *p, float (&o)[8]) {
    uint4 w = *reinterpret_cast<const uint4 *>(p);
    o[0] = bf16lo(w.x); o[1] = bf16hi(w.x); o[2] = bf16lo(w.y); o[3] = bf16hi(w.y);
    o[4] = bf16lo(w.z); o[5] = bf16hi(w.z); o[6] = bf16lo(w.w); o[7] = bf16hi(w.w);
}
template <>
__device__ __forceinline__ void load_widen<float, 2>(const float *p, float (&o)[2]) {
    float2 w = *reinterpret_cast<const float2 *>(p);
    o[0] = w.x; o[1] = w.y;
}
template <>
__device__ __forceinline__ void load_widen<float, 4>(const float *p, float (&o)[4]) {
    float4 w = *reinterpret_cast<const float4 *>(p);
    o[0] = w.x; o[1] = w.y; o[2] = w.z; o[3] = w.w;
}

}  // namespace pkv
