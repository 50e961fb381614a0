// Device helpers shared by the scan and state-update kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// compile-time bool tag (selects a code variant inside a generic lambda)
template <bool V> struct BoolC { static constexpr bool value = V; };

// 2^x on the MUFU unit (ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the MUFU unit.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v), passing v through for v > 20 (beta = 1).
// For v <= 20: softplus(v) = max(v, 0) + log1p(e), e = exp(-|v|) in (0, 1]. log1p(e) is
// evaluated from the identity log1p(e) = 2*atanh(s), s = e / (2 + e) in (0, 1/3], as the
// odd series 2*s*(1 + s^2/3 + s^4/5 + ... + s^12/13); the first omitted term is below
// 1.6e-8 relative at s = 1/3, under half an fp32 ulp.
__device__ __forceinline__ float softplus_of(float v, float e) {   // e = exp(-|v|)
    const float s = e * rcp_approx(2.0f + e);
    const float s2 = s * s;
    float p = 1.0f / 13.0f;
    p = fmaf(p, s2, 1.0f / 11.0f);
    p = fmaf(p, s2, 1.0f / 9.0f);
    p = fmaf(p, s2, 1.0f / 7.0f);
    p = fmaf(p, s2, 1.0f / 5.0f);
    p = fmaf(p, s2, 1.0f / 3.0f);
    p = fmaf(p, s2, 1.0f);
    const float r = fmaxf(v, 0.0f) + 2.0f * s * p;
    return v > 20.0f ? v : r;
}
__device__ __forceinline__ float softplus_f(float v) { return softplus_of(v, ex2(-fabsf(v) * kLog2e)); }

// softplus(v) and its derivative sigmoid(v) from one exponential e = exp(-|v|):
// sigmoid(v) = 1/(1+e) for v >= 0, e/(1+e) for v < 0.
__device__ __forceinline__ float softplus_sigmoid(float v, float &sg) {
    const float e = ex2(-fabsf(v) * kLog2e);
    const float r = rcp_approx(1.0f + e);
    sg = v >= 0.0f ? r : e * r;
    return softplus_of(v, e);
}

// SiLU(z) = z * sigmoid(z) = z / (1 + e^-z).
__device__ __forceinline__ float silu_f(float z) {
    const float e = ex2(-z * kLog2e);
    return z * rcp_approx(1.0f + e);
}

// phi(x) = (e^x - 1)/x, the factor that turns dt*B into the zero-order-hold B_bar
// ((exp(dt*A) - 1)/A * B); x = dt*A, abar = exp(x) already computed. For |x| < 1/8 a cubic
// Taylor polynomial (truncation <= 2e-6 relative), else (abar - 1)/x (cancellation in
// abar - 1 <= 2e-6 relative there). phi(0) = 1: the Euler step.
__device__ __forceinline__ float zoh_phi(float x, float abar) {
    float p = fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f);
    p = fmaf(p, x, 0.5f);
    p = fmaf(p, x, 1.0f);
    return fabsf(x) < 0.125f ? p : (abar - 1.0f) * rcp_approx(x);
}

// a - b on packed pairs (f32x2, round to nearest)
__device__ __forceinline__ float2 fsub2_rn(float2 a, float2 b) {
    float2 r;
    asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
        " sub.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// --- io conversions ---------------------------------------------------------------------
template <typename IO> struct io_traits;
template <> struct io_traits<float> {
    static constexpr int kSize = 4;
    __device__ __forceinline__ static float to_f(float v) { return v; }
};
template <> struct io_traits<__nv_bfloat16> {
    static constexpr int kSize = 2;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Unpack 16 bytes of io data into 16/sizeof(IO) floats.
__device__ __forceinline__ void unpack16(const uint4 v, float *out, float) {
    out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4 v, float *out, __nv_bfloat16) {
    out[0] = bf16lo(v.x); out[1] = bf16hi(v.x); out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
    out[4] = bf16lo(v.z); out[5] = bf16hi(v.z); out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
}

// Pack 16/sizeof(IO) floats into 16 bytes of io data (bf16: round to nearest even).
__device__ __forceinline__ uint4 pack16(const float *in, float) {
    return make_uint4(__float_as_uint(in[0]), __float_as_uint(in[1]), __float_as_uint(in[2]),
                      __float_as_uint(in[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack16(const float *in, __nv_bfloat16) {
    return make_uint4(pack_bf16x2(in[0], in[1]), pack_bf16x2(in[2], in[3]),
                      pack_bf16x2(in[4], in[5]), pack_bf16x2(in[6], in[7]));
}

__device__ __forceinline__ void store_io(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// --- async global->shared copies (16-byte granules, zero-fill beyond src_bytes) ---------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Transposed butterfly over the G lanes of a channel: on entry v[i] is this lane's partial
// for timestep tb+i (i < G); on exit v[0] is the full sum for timestep tb + (lane % G).
template <int G>
__device__ __forceinline__ float group_reduce_transpose(float (&v)[G], int lane) {
#pragma unroll
    for (int h = G / 2; h >= 1; h /= 2) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float lo = v[i], hi = v[i + h];
            const float send = upper ? lo : hi;
            const float keep = upper ? hi : lo;
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    return v[0];
}

}  // namespace ssm
