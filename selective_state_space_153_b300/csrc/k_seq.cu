// Sequential-lane scan launches (scan_seq.cuh), the chunk-carry combine and a zero fill.
#include <algorithm>

#include "launch.h"

namespace ssm {

// Incoming state of every chunk from the chunk aggregates, sequentially over chunks:
//   hin[0] = 0,  hin[k+1] = exp(A * sum_dt[k]) * hin[k] + hlocal_end[k].
// One thread per (channel, state).
__global__ void chunk_combine_kernel(const float *__restrict__ A, const float *__restrict__ agg_h,
                                     const float *__restrict__ agg_s, float *__restrict__ hin,
                                     int64_t BD, int64_t Dm, int64_t N, int npad, int nchunks) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BD * npad) return;
    const int64_t bd = i / npad;
    const int n = (int)(i % npad);
    const int64_t d = bd % Dm;
    const float Ap = n < N ? A[d * N + n] * kLog2e : 0.0f;
    float h = 0.0f;
    for (int k = 0; k < nchunks; ++k) {
        hin[((int64_t)k * BD + bd) * npad + n] = h;
        if (k + 1 < nchunks) {
            const float P = ex2(Ap * agg_s[(int64_t)k * BD + bd]);
            h = fmaf(P, h, agg_h[((int64_t)k * BD + bd) * npad + n]);
        }
    }
}

// The same incoming states for many chunks, in three phases of one CTA per 32 (channel,
// state) pairs: thread (pair, group g) composes the aggregates of chunk group g (kCombGroups
// groups of consecutive chunks; the group's decay is exp(A * its summed dt)), one thread per
// pair then chains the group aggregates, and every thread replays its group from the group's
// incoming state. The sequential depth is about 2*nchunks/kCombGroups + kCombGroups steps
// instead of nchunks (the composition of affine maps is associative).
constexpr int kCombPairs = 32, kCombGroups = 16;
__global__ void __launch_bounds__(kCombPairs * kCombGroups)
    chunk_combine_grouped_kernel(const float *__restrict__ A, const float *__restrict__ agg_h,
                                 const float *__restrict__ agg_s, float *__restrict__ hin, int64_t BD, int64_t Dm,
                                 int64_t N, int npad, int nchunks) {
    __shared__ float sS[kCombGroups][kCombPairs], sH[kCombGroups][kCombPairs];
    const int pl = threadIdx.x % kCombPairs, g = threadIdx.x / kCombPairs;
    const int64_t i = (int64_t)blockIdx.x * kCombPairs + pl;
    const bool valid = i < BD * npad;
    const int64_t bd = valid ? i / npad : 0;
    const int n = valid ? (int)(i % npad) : 0;
    const float Ap = (valid && n < N) ? A[(bd % Dm) * N + n] * kLog2e : 0.0f;
    const int cpg = (nchunks + kCombGroups - 1) / kCombGroups;
    const int k0 = min(g * cpg, nchunks), k1 = min(k0 + cpg, nchunks);
    // group aggregate of the chunks k0..k1-1 that have one (all but the last chunk)
    float h = 0.0f, S = 0.0f;
    if (valid) {
        for (int k = k0; k < min(k1, nchunks - 1); ++k) {
            const float sdt = agg_s[(int64_t)k * BD + bd];
            h = fmaf(ex2(Ap * sdt), h, agg_h[((int64_t)k * BD + bd) * npad + n]);
            S += sdt;
        }
    }
    sS[g][pl] = S;
    sH[g][pl] = h;
    __syncthreads();
    if (g == 0) {   // incoming state of every group
        float x = 0.0f;
        for (int gg = 0; gg < kCombGroups; ++gg) {
            const float hg = sH[gg][pl];
            sH[gg][pl] = x;
            x = fmaf(ex2(Ap * sS[gg][pl]), x, hg);
        }
    }
    __syncthreads();
    if (!valid) return;
    float x = sH[g][pl];
    for (int k = k0; k < k1; ++k) {
        hin[((int64_t)k * BD + bd) * npad + n] = x;
        if (k + 1 < nchunks) x = fmaf(ex2(Ap * agg_s[(int64_t)k * BD + bd]), x, agg_h[((int64_t)k * BD + bd) * npad + n]);
    }
}

// Rows of `len` io elements at stride src_ld copied to stride dst_ld, elements len..dst_ld-1
// of each destination row zeroed: puts rows whose byte length is not a multiple of 16 on
// 16-byte boundaries for the channel-pair kernel (and takes its y rows back). A thread moves
// one 16-byte piece of a destination row: 16-byte loads and stores on whichever side is
// aligned, element by element on the other. Rows on blockIdx.y (+ k*gridDim.y).
template <typename IO>
__global__ void restride_kernel(const IO *__restrict__ src, int64_t src_ld, IO *__restrict__ dst, int64_t dst_ld,
                                int64_t rows, int64_t len) {
    constexpr int E = 16 / (int)sizeof(IO);
    const int64_t pieces = (dst_ld + E - 1) / E;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const IO *s = src + r * src_ld;
        IO *d = dst + r * dst_ld;
        const bool dvec = (reinterpret_cast<uintptr_t>(d) & 15u) == 0;
        for (int64_t pc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; pc < pieces;
             pc += (int64_t)gridDim.x * blockDim.x) {
            const int64_t t0 = pc * E;
            union {
                uint4 q;
                IO e[E];
            } v;
            if ((reinterpret_cast<uintptr_t>(s + t0) & 15u) == 0 && t0 + E <= len) {
                v.q = __ldg(reinterpret_cast<const uint4 *>(s + t0));
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k) v.e[k] = t0 + k < len ? s[t0 + k] : IO(0.0f);
            }
            if (dvec && t0 + E <= dst_ld) {
                *reinterpret_cast<uint4 *>(d + t0) = v.q;
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (t0 + k < dst_ld) d[t0 + k] = v.e[k];
            }
        }
    }
}

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, int NPER, int G, bool AGG, bool AL>
cudaError_t launch_seq_t(const SeqParams &prm, int grid_y, cudaStream_t s) {
    using Cfg = SeqCfg<IO, NPER, G, kSeqWarps, kSeqTile>;
    auto k = scan_seq_kernel<IO, NPER, G, kSeqWarps, kSeqTile, AGG, AL>;
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    });
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(prm.Bt * prm.chan_blocks), (unsigned)grid_y);
    k<<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO, int NPER, int G>
cudaError_t launch_seq_g(const SeqParams &prm, bool agg, bool aligned, int grid_y, cudaStream_t s) {
    if (agg) return aligned ? launch_seq_t<IO, NPER, G, true, true>(prm, grid_y, s)
                            : launch_seq_t<IO, NPER, G, true, false>(prm, grid_y, s);
    return aligned ? launch_seq_t<IO, NPER, G, false, true>(prm, grid_y, s)
                   : launch_seq_t<IO, NPER, G, false, false>(prm, grid_y, s);
}

#define SSM_SEQ_CASES(X) X(4, 1) X(8, 1) X(16, 1) X(4, 4) X(16, 2) X(16, 4) X(16, 8)

template <typename IO>
cudaError_t launch_seq_io(int nper, int g, bool agg, bool aligned, const SeqParams &prm, int grid_y, cudaStream_t s) {
    switch (nper * 100 + g) {
#define SSM_SEQ_LAUNCH(NP, GG) case NP * 100 + GG: return launch_seq_g<IO, NP, GG>(prm, agg, aligned, grid_y, s);
        SSM_SEQ_CASES(SSM_SEQ_LAUNCH)
#undef SSM_SEQ_LAUNCH
        default: return cudaErrorInvalidConfiguration;
    }
}

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0.0f;
}
}  // namespace

cudaError_t launch_seq(ssm_dtype_t io, int nper, int g, bool agg, bool aligned, const SeqParams &prm,
                       int grid_y, cudaStream_t s) {
    return io == SSM_BF16 ? launch_seq_io<bf16>(nper, g, agg, aligned, prm, grid_y, s)
                          : launch_seq_io<float>(nper, g, agg, aligned, prm, grid_y, s);
}

bool seq_plan_supported(int nper, int g) {
    switch (nper * 100 + g) {
#define SSM_SEQ_OK(NP, GG) case NP * 100 + GG: return true;
        SSM_SEQ_CASES(SSM_SEQ_OK)
#undef SSM_SEQ_OK
        default: return false;
    }
}

cudaError_t launch_chunk_combine(const float *A, const float *agg_h, const float *agg_s, float *hin,
                                 int64_t BD, int64_t Dm, int64_t N, int npad, int nchunks, cudaStream_t s) {
    const int64_t total = BD * npad;
    // deep chains over few (channel, state) pairs: grouped (sequential depth ~2*nchunks/16 + 16).
    // Measured on B300, 1 x 48 x 131072 x 64 (444 chunks, 3072 pairs): 75 -> 8 us; with many
    // pairs the plain kernel is faster (1 x 1536 x 131072 x 64, 54 chunks: 18 vs 64 us;
    // 1 x 384 x 131072 x 64: 16 vs 21 us).
    if (nchunks > 2 * kCombGroups && total < 8192)
        chunk_combine_grouped_kernel<<<(unsigned)((total + kCombPairs - 1) / kCombPairs), kCombPairs * kCombGroups, 0,
                                       s>>>(A, agg_h, agg_s, hin, BD, Dm, N, npad, nchunks);
    else
        chunk_combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(A, agg_h, agg_s, hin, BD, Dm, N, npad,
                                                                              nchunks);
    return cudaGetLastError();
}

cudaError_t launch_restride(ssm_dtype_t io, const void *src, int64_t src_ld, void *dst, int64_t dst_ld, int64_t rows,
                            int64_t len, cudaStream_t s) {
    if (rows <= 0 || dst_ld <= 0) return cudaSuccess;
    const int64_t pieces = (dst_ld * (int64_t)(io == SSM_BF16 ? 2 : 4) + 15) / 16;
    const dim3 grid((unsigned)std::min<int64_t>((pieces + 255) / 256, 64), (unsigned)std::min<int64_t>(rows, 65535));
    if (io == SSM_BF16)
        restride_kernel<bf16><<<grid, 256, 0, s>>>(static_cast<const bf16 *>(src), src_ld, static_cast<bf16 *>(dst),
                                                   dst_ld, rows, len);
    else
        restride_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(src), src_ld, static_cast<float *>(dst),
                                                    dst_ld, rows, len);
    return cudaGetLastError();
}

cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t s) {
    zero_f32_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, s>>>(p, n);
    return cudaGetLastError();
}

}  // namespace ssm
