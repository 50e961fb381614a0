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
    chunk_combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(A, agg_h, agg_s, hin, BD, Dm, N, npad,
                                                                          nchunks);
    return cudaGetLastError();
}

cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t s) {
    zero_f32_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, s>>>(p, n);
    return cudaGetLastError();
}

}  // namespace ssm
