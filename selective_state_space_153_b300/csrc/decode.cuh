// Recurrent single-token step (section 5.3 of "From RNN to Mamba", lmnt.cn: inference
// advances one fixed-size fp32 state per channel token by token; the update is the body
// of the section 3.2 loop for one timestep):
//   state = exp(dt*A) * state + dt*B*x ;  y = (sum_n C*state + D*x) * SiLU(z).
// Memory-bound: the fp32 state is read and written once. Vector path (N % 4 == 0): one
// thread per (b, d, 4 consecutive states) with 16-byte state loads/stores, the y partials
// reduced across the N/4 lanes of a channel with shuffles (N/4 must divide 32, i.e.
// N in {4, 8, 16, 32, 64, 128}); otherwise one thread per (b, d) walking all states.
#pragma once
#include "check.cuh"
#include "common.cuh"

namespace ssm {

// four consecutive io elements (8-byte aligned for bf16, 16 for fp32) as floats
__device__ __forceinline__ void load_io4(const __nv_bfloat16 *src, float *out) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(src));
    out[0] = bf16lo(v.x); out[1] = bf16hi(v.x); out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
}
__device__ __forceinline__ void load_io4(const float *src, float *out) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}

struct DecodeParams {
    float *state;
    const void *x, *dt, *B, *C, *z;
    const float *A, *D;
    void *y;
    int64_t Bt, Dm, N;
    int zoh;   // nonzero: launch the zero-order-hold variant (B_bar = (exp(dt*A) - 1)/A * B)
};

// Checked build: the addresses a thread of channel row cl (= b*Dm + d) touches -- `cnt`
// states from `n0` and the B, C elements of the same states, x, dt, z, y at cl, A and D of
// channel d -- lie inside their arrays. Always true in the normal build.
template <typename IO>
__device__ __forceinline__ bool decode_addrs_ok(const DecodeParams &p, int64_t cl, int64_t b, int64_t d, int64_t n0,
                                                int64_t cnt) {
#ifdef SSM_CHECK
    const uint64_t es = sizeof(IO), BD = (uint64_t)p.Bt * p.Dm, BN = (uint64_t)p.Bt * p.N;
    bool ok = SSM_CHK_G(p.state, BD * p.N * 4, p.state + cl * p.N + n0, cnt * 4) &&
              SSM_CHK_G(p.A, (uint64_t)p.Dm * p.N * 4, p.A + d * p.N + n0, cnt * 4) &&
              SSM_CHK_G(p.x, BD * es, reinterpret_cast<const IO *>(p.x) + cl, es) &&
              SSM_CHK_G(p.dt, BD * es, reinterpret_cast<const IO *>(p.dt) + cl, es) &&
              SSM_CHK_G(p.y, BD * es, reinterpret_cast<const IO *>(p.y) + cl, es) &&
              SSM_CHK_G(p.B, BN * es, reinterpret_cast<const IO *>(p.B) + b * p.N + n0, cnt * es) &&
              SSM_CHK_G(p.C, BN * es, reinterpret_cast<const IO *>(p.C) + b * p.N + n0, cnt * es);
    if (p.z != nullptr) ok = ok && SSM_CHK_G(p.z, BD * es, reinterpret_cast<const IO *>(p.z) + cl, es);
    if (p.D != nullptr) ok = ok && SSM_CHK_G(p.D, (uint64_t)p.Dm * 4, p.D + d, 4);
    return ok;
#else
    (void)p; (void)cl; (void)b; (void)d; (void)n0; (void)cnt;
    return true;
#endif
}


// Vector path: lane l of a warp owns the 16-byte piece q = l % LPC of channel
// d = warp*(32/LPC) + l/LPC of batch row b = blockIdx.y (LPC = N/4 lanes per channel), so
// every warp-wide load or store covers 512 contiguous bytes of the state and the index
// arithmetic is shifts (no 64-bit division). B and C of the row are read as 4-element
// vectors (the caller checks their alignment); the y partials are summed across the LPC
// lanes of a channel.
template <typename IO, int LPC, bool ZOH = false>
__global__ void __launch_bounds__(256) decode_wide_kernel(const DecodeParams p) {
    const int b = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int q = t % LPC;
    const int d = t / LPC;
    const bool valid = d < p.Dm && decode_addrs_ok<IO>(p, (int64_t)b * p.Dm + d, b, d, 4 * q, 4);
    float acc = 0.0f, xv = 0.0f, zv = 0.0f;
    if (valid) {
        const int64_t cl = (int64_t)b * p.Dm + d;
        float4 *sp = reinterpret_cast<float4 *>(p.state + cl * p.N) + q;
        float4 v = __ldcs(sp);
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p.A + (int64_t)d * p.N) + q);
        xv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.x)[cl]);
        const float dt = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.dt)[cl]);
        if (p.z != nullptr) zv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.z)[cl]);
        float bv[4], cv[4];
        load_io4(reinterpret_cast<const IO *>(p.B) + (int64_t)b * p.N + 4 * q, bv);
        load_io4(reinterpret_cast<const IO *>(p.C) + (int64_t)b * p.N + 4 * q, cv);
        const float dx = dt * xv, dl = dt * kLog2e;
        if constexpr (ZOH) {
            const float ab[4] = {ex2(dl * a.x), ex2(dl * a.y), ex2(dl * a.z), ex2(dl * a.w)};
            const float av[4] = {a.x, a.y, a.z, a.w};
            float wv[4] = {dx * bv[0], dx * bv[1], dx * bv[2], dx * bv[3]};
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] *= zoh_phi(dt * av[i], ab[i]);
            v.x = fmaf(ab[0], v.x, wv[0]);
            v.y = fmaf(ab[1], v.y, wv[1]);
            v.z = fmaf(ab[2], v.z, wv[2]);
            v.w = fmaf(ab[3], v.w, wv[3]);
        } else {
            v.x = fmaf(ex2(dl * a.x), v.x, dx * bv[0]);
            v.y = fmaf(ex2(dl * a.y), v.y, dx * bv[1]);
            v.z = fmaf(ex2(dl * a.z), v.z, dx * bv[2]);
            v.w = fmaf(ex2(dl * a.w), v.w, dx * bv[3]);
        }
        __stcs(sp, v);
        acc = fmaf(cv[0], v.x, fmaf(cv[1], v.y, fmaf(cv[2], v.z, cv[3] * v.w)));
    }
#pragma unroll
    for (int o = LPC / 2; o >= 1; o /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (valid && q == 0) {
        float yv = acc + (p.D != nullptr ? p.D[d] * xv : 0.0f);
        if (p.z != nullptr) yv *= silu_f(zv);
        store_io(reinterpret_cast<IO *>(p.y) + (int64_t)b * p.Dm + d, yv);
    }
}

template <typename IO, int LPC, bool ZOH = false>  // LPC: lanes per channel = N/4
__global__ void __launch_bounds__(256) decode_vec_kernel(const DecodeParams p) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t chan = gid / LPC;   // b*Dm + d
    const int q = (int)(gid % LPC);
    const int64_t cl = chan < p.Bt * p.Dm ? chan : 0;
    const int64_t b = cl / p.Dm, d = cl % p.Dm;
    const bool valid = chan < p.Bt * p.Dm && decode_addrs_ok<IO>(p, cl, b, d, 4 * q, 4);
    float acc = 0.0f;
    float xv = 0.0f, zv = 0.0f;
    if (valid) {
        const IO *X = reinterpret_cast<const IO *>(p.x);
        const IO *DT = reinterpret_cast<const IO *>(p.dt);
        const IO *Bm = reinterpret_cast<const IO *>(p.B);
        const IO *Cm = reinterpret_cast<const IO *>(p.C);
        xv = io_traits<IO>::to_f(X[cl]);
        const float dt = io_traits<IO>::to_f(DT[cl]);
        if (p.z != nullptr) zv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.z)[cl]);
        float4 *sp = reinterpret_cast<float4 *>(p.state + cl * p.N) + q;
        float4 s = __ldcs(sp);
        const float4 a4 = __ldg(reinterpret_cast<const float4 *>(p.A + d * p.N) + q);
        const int64_t nb = b * p.N + 4 * q;
        const float b0 = io_traits<IO>::to_f(Bm[nb]), b1 = io_traits<IO>::to_f(Bm[nb + 1]);
        const float b2 = io_traits<IO>::to_f(Bm[nb + 2]), b3 = io_traits<IO>::to_f(Bm[nb + 3]);
        const float c0 = io_traits<IO>::to_f(Cm[nb]), c1 = io_traits<IO>::to_f(Cm[nb + 1]);
        const float c2 = io_traits<IO>::to_f(Cm[nb + 2]), c3 = io_traits<IO>::to_f(Cm[nb + 3]);
        const float dx = dt * xv, dl = dt * kLog2e;
        const float ab[4] = {ex2(dl * a4.x), ex2(dl * a4.y), ex2(dl * a4.z), ex2(dl * a4.w)};
        float wv[4] = {dx * b0, dx * b1, dx * b2, dx * b3};
        if constexpr (ZOH) {
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] *= zoh_phi(dt * av[i], ab[i]);
        }
        s.x = fmaf(ab[0], s.x, wv[0]);
        s.y = fmaf(ab[1], s.y, wv[1]);
        s.z = fmaf(ab[2], s.z, wv[2]);
        s.w = fmaf(ab[3], s.w, wv[3]);
        __stcs(sp, s);
        acc = fmaf(c0, s.x, fmaf(c1, s.y, fmaf(c2, s.z, c3 * s.w)));
    }
#pragma unroll
    for (int o = LPC / 2; o >= 1; o /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (valid && q == 0) {
        float yv = acc + (p.D != nullptr ? p.D[d] * xv : 0.0f);
        if (p.z != nullptr) yv *= silu_f(zv);
        store_io(reinterpret_cast<IO *>(p.y) + cl, yv);
    }
}

template <typename IO, bool ZOH = false>
__global__ void __launch_bounds__(256) decode_scalar_kernel(const DecodeParams p) {
    const int64_t cl = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (cl >= p.Bt * p.Dm) return;
    const int64_t b = cl / p.Dm, d = cl % p.Dm;
    if (!decode_addrs_ok<IO>(p, cl, b, d, 0, p.N)) return;   // no shuffles in this kernel
    const IO *Bm = reinterpret_cast<const IO *>(p.B);
    const IO *Cm = reinterpret_cast<const IO *>(p.C);
    const float xv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.x)[cl]);
    const float dt = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.dt)[cl]);
    const float dx = dt * xv, dl = dt * kLog2e;
    float acc = 0.0f;
    for (int64_t n = 0; n < p.N; ++n) {
        float s = p.state[cl * p.N + n];
        const float an = p.A[d * p.N + n], ab = ex2(dl * an);
        float w = dx * io_traits<IO>::to_f(Bm[b * p.N + n]);
        if constexpr (ZOH) w *= zoh_phi(dt * an, ab);
        s = fmaf(ab, s, w);
        p.state[cl * p.N + n] = s;
        acc = fmaf(io_traits<IO>::to_f(Cm[b * p.N + n]), s, acc);
    }
    float yv = acc + (p.D != nullptr ? p.D[d] * xv : 0.0f);
    if (p.z != nullptr) yv *= silu_f(io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.z)[cl]));
    store_io(reinterpret_cast<IO *>(p.y) + cl, yv);
}

}  // namespace ssm
