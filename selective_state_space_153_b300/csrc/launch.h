// Host-side launch functions of the kernels, one translation unit per kernel family (so the
// library builds in parallel). Each returns the launch's cudaError_t; none allocates memory.
// The host logic in ssm_api.cu plans a call and picks one of these.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "ssm_scan.h"
#include "scan_seq.cuh"
#include "decode.cuh"
#include "scan_bwd.cuh"
#include "scan_tc.cuh"

namespace ssm {

// Runs `set` (a kernel's attribute calls) once per device: bit i of `done` records that it
// succeeded on device i (devices from 64 on: every time). Safe to call from several threads;
// a race only repeats the calls.
template <typename F>
cudaError_t once_per_device(std::atomic<unsigned long long> &done, F &&set) {
    int dev = 0;
    if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    if (dev < 64 && (done.load(std::memory_order_acquire) >> dev & 1ull)) return cudaSuccess;
    const cudaError_t e = set();
    if (e == cudaSuccess && dev < 64) done.fetch_or(1ull << dev, std::memory_order_acq_rel);
    return e;
}

// channel-pair scan (scan_pair.cuh). variant: 0 = Euler, 1 = zero-order hold, 2 = conv front
#ifndef SSM_PAIR_T
#define SSM_PAIR_T 16
#endif
constexpr int kPairT = SSM_PAIR_T;   // timesteps per tile of the channel-pair kernel
enum PairVariant { kPairEuler = 0, kPairZoh = 1, kPairConv = 2 };
cudaError_t launch_pair(ssm_dtype_t io, int variant, int ks, int gp, bool agg, const SeqParams &prm,
                        int grid_y, cudaStream_t s);
// dynamic shared memory per CTA of a channel-pair launch (0: no such kernel)
size_t pair_smem(ssm_dtype_t io, int ks, int gp, bool conv, bool agg);
// warps per CTA of a channel-pair launch
int pair_warps_of(int ks, int gp, bool agg);
// resident CTAs per SM that the launch bounds allow (register budget)
int pair_min_blocks_of(int ks, int gp, bool agg);

// sequential-lane scan (scan_seq.cuh) and the chunk-carry combine
constexpr int kSeqTile = 32;    // timesteps per tile
constexpr int kSeqWarps = 4;    // warps per CTA
cudaError_t launch_seq(ssm_dtype_t io, int nper, int g, bool agg, bool aligned, const SeqParams &prm,
                       int grid_y, cudaStream_t s);
bool seq_plan_supported(int nper, int g);
cudaError_t launch_chunk_combine(const float *A, const float *agg_h, const float *agg_s, float *hin,
                                 int64_t BD, int64_t Dm, int64_t N, int npad, int nchunks, cudaStream_t s);
// rows of `len` io elements from stride src_ld to stride dst_ld (destination tails zeroed)
cudaError_t launch_restride(ssm_dtype_t io, const void *src, int64_t src_ld, void *dst, int64_t dst_ld, int64_t rows,
                            int64_t len, cudaStream_t s);
cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t s);

// persistent time-split scans (scan_tc.cuh / scan_tp.cuh): B/C preparation, then the kernel
cudaError_t launch_bc_prep(ssm_dtype_t io, const void *B, const void *C, float *bc, int64_t N, int64_t L,
                           int64_t Lp, int np, int64_t batch, cudaStream_t s);
cudaError_t launch_tc(ssm_dtype_t io, bool pipelined, int G, const TcParams &prm, cudaStream_t s);

// recurrent single-token step (decode.cuh). kind: 0 = wide (16-byte B/C), 1 = vector,
// 2 = scalar (N % 4 != 0)
cudaError_t launch_decode(ssm_dtype_t io, int kind, int lpc, bool zoh, const DecodeParams &p, cudaStream_t s);

// backward (scan_bwd.cuh): checkpoint pass then adjoint pass; G lanes per channel
// backward: G lanes per channel, Q (2 or 4) states per lane
cudaError_t launch_bwd(ssm_dtype_t io, int G, int Q, const BwdParams &p, cudaStream_t s);

}  // namespace ssm
