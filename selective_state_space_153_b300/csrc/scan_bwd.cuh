// Selective scan backward: gradients of sum(y*dy) (+ sum(h_last*dlast)) with respect to u,
// delta, A, B, C, D, z and the dt bias, for the per-timestep loop of section 3.2 of
// "From RNN to Mamba: state-space model principles and long-sequence modelling in practice"
// (lmnt.cn). Training differentiates through the recurrence (section 2.2 of that page); the
// adjoint of h_t = a_t*h_{t-1} + dt_t*u_t*B_t, y_t = (sum_n C_t*h_t + D*u_t)*SiLU(z_t) is the
// reverse recurrence
//     lambda_t = dyhat_t * C_t + c_t,   c_{t-1} = a_t * lambda_t,   c_{L-1} = dlast,
// with dyhat_t = dy_t * SiLU(z_t), from which (per channel d, state n, step t)
//     dB_t += lambda_t dt_t u_t         dC_t += dyhat_t h_t          (summed over channels)
//     du_t  = sum_n lambda_t dt_t B_t + dyhat_t D
//     ddt_t = sum_n lambda_t (u_t B_t + A a_t h_{t-1}),   ddelta_t = ddt_t * sigmoid(v_t)
//     dA   += lambda_t dt_t a_t h_{t-1}   dD += dyhat_t u_t   dz_t = dy_t yhat_t SiLU'(z_t)
// (v = delta + bias; sigmoid is the softplus derivative; without softplus ddelta = ddt).
//
// Work decomposition: a thread owns Q states n = g + G*q of one channel (G lanes per
// channel, a power of two <= 32; the batch row is grid.y so a warp never spans two rows).
// Pass 1 (scan_bwd_ckpt_kernel) runs the recurrence forward and stores h at the start of
// every S-step segment. Pass 2 (scan_bwd_kernel) walks the segments backwards: it recomputes
// the segment's S states into registers from the checkpoint, then runs the adjoint over the
// segment in reverse. Sums over the states of a channel use shuffles across its G lanes; sums
// over channels (dB, dC) are pre-reduced across the warp's channels with shuffles, staged
// per warp for the whole segment in shared memory, summed over the CTA's warps after the
// segment and added with one fp32 atomic per (CTA, state, step); dA, dD and the dt bias are
// summed over the sequence in the thread and added once at the end.
#pragma once
#include "common.cuh"

namespace ssm {

constexpr int kBwdS = 16;        // steps per checkpoint segment
constexpr int kBwdThreads = 128;
// dynamic shared memory of scan_bwd_kernel<., G, Q> beyond its input tile: the dB/dC
// partials [2][warps][kBwdS][G*Q] floats
constexpr size_t bwd_smem_bytes(int G, int Q) { return (size_t)2 * (kBwdThreads / 32) * kBwdS * G * Q * sizeof(float); }

struct BwdParams {
    const void *u, *delta, *z, *B, *C, *dy;
    const float *A, *D, *bias, *dlast;
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *dbias;
    float *ckpt;                  // [Bt*Dm][nseg][G*Q]: h before each segment's first step
    int64_t Bt, Dm, L, N;
    int softplus, nseg;
};

__device__ __forceinline__ float bwd_dt(float v, int softplus) { return softplus ? softplus_f(v) : v; }

// sum over the G lanes of a channel (lanes g = lane % G are consecutive)
template <int G>
__device__ __forceinline__ float sum_lanes(float v) {
#pragma unroll
    for (int o = G / 2; o >= 1; o /= 2) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// sum over the 32/G channels of a warp (lanes with the same g)
template <int G>
__device__ __forceinline__ float sum_channels(float v) {
#pragma unroll
    for (int o = G; o < 32; o *= 2) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inputs of one S-step segment, staged by the whole CTA with coalesced loads: B and C rows of
// the batch row ([G*Q][S], zero beyond N or L) and, per channel of the CTA, dt, the softplus
// derivative, u, dy and z ([kCpb][S]); dt = softplus(delta + bias) is formed once per
// (channel, step) here rather than in every lane.
template <typename IO, int G, int Q>
struct BwdTile {
    static constexpr int kCpb = kBwdThreads / G;
    static constexpr int kFloats = 2 * G * Q * kBwdS + 5 * kCpb * kBwdS;
    float *B, *C, *dt, *sg, *u, *dy, *z;
    __device__ BwdTile(float *base) {
        B = base; C = B + G * Q * kBwdS; dt = C + G * Q * kBwdS; sg = dt + kCpb * kBwdS;
        u = sg + kCpb * kBwdS; dy = u + kCpb * kBwdS; z = dy + kCpb * kBwdS;
    }
    // full = false: only what the forward recompute needs (B, dt, u)
    __device__ void load(const BwdParams &p, int64_t b, int64_t t0, bool full) {
        const int tid = threadIdx.x;
        const IO *Bm = reinterpret_cast<const IO *>(p.B) + b * p.N * p.L;
        const IO *Cm = reinterpret_cast<const IO *>(p.C) + b * p.N * p.L;
        for (int e = tid; e < (full ? 2 : 1) * G * Q * kBwdS; e += kBwdThreads) {
            const int which = e / (G * Q * kBwdS), r = e % (G * Q * kBwdS), n = r / kBwdS, i = r % kBwdS;
            const int64_t t = t0 + i;
            float v = 0.0f;
            if (n < p.N && t < p.L) v = io_traits<IO>::to_f((which ? Cm : Bm)[n * p.L + t]);
            (which ? C : B)[r] = v;
        }
        for (int e = tid; e < kCpb * kBwdS; e += kBwdThreads) {
            const int cc = e / kBwdS, i = e % kBwdS;
            const int64_t d = (int64_t)blockIdx.x * kCpb + cc, t = t0 + i;
            float dtv = 0.0f, sgv = 0.0f, uv = 0.0f, dyv = 0.0f, zv = 0.0f;
            if (d < p.Dm && t < p.L) {
                const int64_t idx = (b * p.Dm + d) * p.L + t;
                const float v = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.delta)[idx]) +
                                (p.bias ? p.bias[d] : 0.0f);
                dtv = bwd_dt(v, p.softplus);
                sgv = p.softplus ? 1.0f / (1.0f + ex2(-v * kLog2e)) : 1.0f;
                uv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.u)[idx]);
                if (full) {
                    dyv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.dy)[idx]);
                    if (p.z) zv = io_traits<IO>::to_f(reinterpret_cast<const IO *>(p.z)[idx]);
                }
            }
            dt[e] = dtv; sg[e] = sgv; u[e] = uv; dy[e] = dyv; z[e] = zv;
        }
    }
};

template <int G, int Q>
constexpr size_t bwd_tile_bytes() { return (size_t)BwdTile<float, G, Q>::kFloats * sizeof(float); }

template <typename IO, int G, int Q>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_ckpt_kernel(const BwdParams p) {
    constexpr int kCpb = kBwdThreads / G;
    extern __shared__ float smemf[];
    BwdTile<IO, G, Q> tile(smemf);
    const int tid = threadIdx.x, g = tid % G, cc = tid / G;
    const int64_t b = blockIdx.y, d = (int64_t)blockIdx.x * kCpb + cc;
    const bool valid = d < p.Dm;                 // every thread takes part in the tile loads
    const int64_t bd = b * p.Dm + (valid ? d : 0);
    float Ap[Q], h[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int n = g + G * q;
        Ap[q] = (valid && n < p.N) ? p.A[(valid ? d : 0) * p.N + n] * kLog2e : 0.0f;
        h[q] = 0.0f;
    }
    float *ck = p.ckpt + bd * (int64_t)p.nseg * (G * Q);
    for (int seg = 0; seg < p.nseg; ++seg) {
        if (valid) {
#pragma unroll
            for (int q = 0; q < Q; ++q) ck[(int64_t)seg * (G * Q) + g + G * q] = h[q];
        }
        __syncthreads();
        tile.load(p, b, (int64_t)seg * kBwdS, false);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kBwdS; ++i) {
            const float dt = tile.dt[cc * kBwdS + i];
            const float x = dt * tile.u[cc * kBwdS + i];
#pragma unroll
            for (int q = 0; q < Q; ++q) h[q] = fmaf(ex2(dt * Ap[q]), h[q], x * tile.B[(g + G * q) * kBwdS + i]);
        }
    }
}

template <typename IO, int G, int Q>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_kernel(const BwdParams p) {
    constexpr int kCpb = kBwdThreads / G;
    constexpr int kWarps = kBwdThreads / 32;
    // staged segment inputs, then per warp and step the channel-summed dB and dC partials
    // for the G*Q states ([2][kWarps][kBwdS][G*Q])
    extern __shared__ float smemf[];
    BwdTile<IO, G, Q> tile(smemf);
    float *sPartBuf = smemf + BwdTile<IO, G, Q>::kFloats;
    auto sPart = [&](int which, int w, int i, int n) -> float & {
        return sPartBuf[(((size_t)which * kWarps + w) * kBwdS + i) * (G * Q) + n];
    };
    const int tid = threadIdx.x, g = tid % G, warp = tid >> 5, cc = tid / G;
    const int64_t b = blockIdx.y, d = (int64_t)blockIdx.x * kCpb + cc;
    const bool valid = d < p.Dm;                // invalid lanes still take part in the shuffles
    const int64_t dd = valid ? d : 0;
    const int64_t bd = b * p.Dm + dd;
    const float Dv = (valid && p.D) ? p.D[dd] : 0.0f;
    float An[Q], Ap[Q], c[Q], dA[Q];
    bool nv[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int n = g + G * q;
        nv[q] = valid && n < p.N;
        An[q] = nv[q] ? p.A[dd * p.N + n] : 0.0f;
        Ap[q] = An[q] * kLog2e;
        c[q] = (nv[q] && p.dlast) ? p.dlast[bd * p.N + n] : 0.0f;
        dA[q] = 0.0f;
    }
    float dD = 0.0f, dbias = 0.0f;
    const float *ck = p.ckpt + bd * (int64_t)p.nseg * (G * Q);
    for (int seg = p.nseg - 1; seg >= 0; --seg) {
        const int64_t t0 = (int64_t)seg * kBwdS;
        __syncthreads();                        // the previous segment is done with the tile
        tile.load(p, b, t0, true);
        __syncthreads();
        float hs[Q][kBwdS + 1];                 // hs[q][0]: h before the segment; hs[q][i+1]: after step t0+i
#pragma unroll
        for (int q = 0; q < Q; ++q) hs[q][0] = valid ? ck[(int64_t)seg * (G * Q) + g + G * q] : 0.0f;
#pragma unroll
        for (int i = 0; i < kBwdS; ++i) {
            const float dt = tile.dt[cc * kBwdS + i];
            const float x = dt * tile.u[cc * kBwdS + i];
#pragma unroll
            for (int q = 0; q < Q; ++q)
                hs[q][i + 1] = fmaf(ex2(dt * Ap[q]), hs[q][i], x * tile.B[(g + G * q) * kBwdS + i]);
        }
#pragma unroll
        for (int i = kBwdS - 1; i >= 0; --i) {
            const int64_t t = t0 + i;
            if (t >= p.L) {                     // uniform across the block (same t everywhere)
                if ((threadIdx.x & 31) < G) {
#pragma unroll
                    for (int q = 0; q < Q; ++q) sPart(0, warp, i, g + G * q) = sPart(1, warp, i, g + G * q) = 0.0f;
                }
                continue;
            }
            const float dt = tile.dt[cc * kBwdS + i];
            const float uu = tile.u[cc * kBwdS + i];
            float bq[Q], cq[Q], yh = 0.0f;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                bq[q] = tile.B[(g + G * q) * kBwdS + i];
                cq[q] = tile.C[(g + G * q) * kBwdS + i];
                yh = fmaf(cq[q], hs[q][i + 1], yh);
            }
            yh = sum_lanes<G>(yh) + Dv * uu;    // yhat_t, before the gate
            const float dyv = tile.dy[cc * kBwdS + i];
            float dyh = dyv, dzv = 0.0f;
            if (p.z) {
                const float zz = tile.z[cc * kBwdS + i];
                const float sg = 1.0f / (1.0f + ex2(-zz * kLog2e));
                dyh = dyv * zz * sg;            // dy * SiLU(z)
                dzv = dyv * yh * sg * (1.0f + zz * (1.0f - sg));
            }
            float du = 0.0f, ddt = 0.0f;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const float a = ex2(dt * Ap[q]);
                const float lam = fmaf(dyh, cq[q], c[q]);
                const float hp = hs[q][i];
                du = fmaf(lam * dt, bq[q], du);
                ddt = fmaf(lam, fmaf(uu, bq[q], An[q] * a * hp), ddt);
                dA[q] = fmaf(lam * dt * a, hp, dA[q]);
                c[q] = a * lam;
                // sums over the warp's channels, staged for the CTA-wide sum after the segment
                const float gb = sum_channels<G>(nv[q] ? lam * dt * uu : 0.0f);
                const float gc = sum_channels<G>(nv[q] ? dyh * hs[q][i + 1] : 0.0f);
                if ((threadIdx.x & 31) < G) {
                    sPart(0, warp, i, g + G * q) = gb;
                    sPart(1, warp, i, g + G * q) = gc;
                }
            }
            du = sum_lanes<G>(du);
            ddt = sum_lanes<G>(ddt);
            if (valid && g == 0) {
                const float ddl = ddt * tile.sg[cc * kBwdS + i];
                p.du[bd * p.L + t] = fmaf(dyh, Dv, du);
                p.ddelta[bd * p.L + t] = ddl;
                if (p.dz) p.dz[bd * p.L + t] = dzv;
                dD = fmaf(dyh, uu, dD);
                dbias += ddl;
            }
        }
        // dB, dC of the segment: sum the warps' partials, one atomic per (state, step)
        __syncthreads();
        for (int e = tid; e < 2 * kBwdS * G * Q; e += kBwdThreads) {
            const int which = e / (kBwdS * G * Q), r = e % (kBwdS * G * Q);
            const int i = r / (G * Q), n = r % (G * Q);
            const int64_t t = t0 + i;
            if (n >= p.N || t >= p.L) continue;
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) acc += sPart(which, w, i, n);
            atomicAdd((which ? p.dC : p.dB) + (b * p.N + n) * p.L + t, acc);
        }
    }
    if (!valid) return;
#pragma unroll
    for (int q = 0; q < Q; ++q)
        if (nv[q]) atomicAdd(p.dA + dd * p.N + g + G * q, dA[q]);
    if (g == 0) {
        if (p.dD) atomicAdd(p.dD + dd, dD);
        if (p.dbias) atomicAdd(p.dbias + dd, dbias);
    }
}

}  // namespace ssm
