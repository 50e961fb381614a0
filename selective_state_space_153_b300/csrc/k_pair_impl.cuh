// Launches of the channel-pair scan kernel (scan_pair.cuh) for one io type and one variant
// (Euler / zero-order hold / conv front). Each k_pair_*.cu instantiates one combination, so
// the kernels build in parallel.
#pragma once
#include "launch.h"
#include "scan_pair.cuh"

namespace ssm {

// the lane splits built: (states per lane KS, lanes per channel pair GP)
#define SSM_PAIR_CASES(X) X(4, 1) X(4, 2) X(4, 4) X(8, 1) X(8, 2) X(8, 4) X(8, 8) X(8, 16) X(16, 4)

template <typename IO, int KS, int GP, bool AGG, bool ZOH, bool CONV>
cudaError_t launch_pair_t(const SeqParams &prm, int grid_y, cudaStream_t s) {
    constexpr int W = pair_warps(KS, GP, AGG);
    using Cfg = PairCfg<IO, KS, GP, W, kPairT, CONV>;
    auto k = scan_pair_kernel<IO, KS, GP, W, kPairT, AGG, ZOH, CONV>;
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    });
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(prm.Bt * prm.chan_blocks), (unsigned)grid_y);
    k<<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO, bool ZOH, bool CONV>
cudaError_t launch_pair_variant(int ks, int gp, bool agg, const SeqParams &prm, int grid_y, cudaStream_t s) {
    switch (ks * 100 + gp) {
#define SSM_PAIR_LAUNCH(KS, GP)                                                                  \
    case KS * 100 + GP:                                                                          \
        return agg ? launch_pair_t<IO, KS, GP, true, ZOH, CONV>(prm, grid_y, s)                  \
                   : launch_pair_t<IO, KS, GP, false, ZOH, CONV>(prm, grid_y, s);
        SSM_PAIR_CASES(SSM_PAIR_LAUNCH)
#undef SSM_PAIR_LAUNCH
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace ssm

// one translation unit: launch_pair_<tag>(...) for io type IO_T, zero-order hold ZOH_V,
// conv front CONV_V
#define SSM_DEFINE_PAIR_TU(tag, IO_T, ZOH_V, CONV_V)                                               \
    namespace ssm {                                                                              \
    cudaError_t launch_pair_##tag(int ks, int gp, bool agg, const SeqParams &prm, int grid_y,     \
                                  cudaStream_t s) {                                              \
        return launch_pair_variant<IO_T, ZOH_V, CONV_V>(ks, gp, agg, prm, grid_y, s);            \
    }                                                                                            \
    }
