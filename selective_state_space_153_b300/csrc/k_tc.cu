// Persistent time-split scan launches (scan_tc.cuh / scan_tp.cuh) and their B/C preparation.
#include "launch.h"
#include "scan_tp.cuh"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

int sm_count_dev() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

template <typename IO, int G>
cudaError_t launch_tc_t(const TcParams &prm, cudaStream_t s) {
    using Cfg = TcCfg<IO, G>;
    auto k = scan_tc_kernel<IO, G>;
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
        if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        return r;
    });
    if (e != cudaSuccess) return e;
    k<<<(unsigned)sm_count_dev(), Cfg::W * 32, Cfg::SMEM, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO, int G>
cudaError_t launch_tp_t(const TcParams &prm, cudaStream_t s) {
    using Cfg = TpCfg<IO, G>;
    auto k = scan_tp_kernel<IO, G>;
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
        if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        return r;
    });
    if (e != cudaSuccess) return e;
    k<<<(unsigned)sm_count_dev(), Cfg::W * 32, Cfg::SMEM, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_tc_io(bool pipelined, int G, const TcParams &prm, cudaStream_t s) {
    if (pipelined) {
        switch (G) {
            case 1:
                if constexpr (tp_bytes<IO, 1>(2) <= kSmemLimit) return launch_tp_t<IO, 1>(prm, s);
                return cudaErrorInvalidConfiguration;
            case 2: return launch_tp_t<IO, 2>(prm, s);
            case 4: return launch_tp_t<IO, 4>(prm, s);
            case 8: return launch_tp_t<IO, 8>(prm, s);
            default: return cudaErrorInvalidConfiguration;
        }
    }
    switch (G) {
        case 1: return launch_tc_t<IO, 1>(prm, s);
        case 2: return launch_tc_t<IO, 2>(prm, s);
        case 4: return launch_tc_t<IO, 4>(prm, s);
        case 8: return launch_tc_t<IO, 8>(prm, s);
        default: return cudaErrorInvalidConfiguration;
    }
}
}  // namespace

cudaError_t launch_bc_prep(ssm_dtype_t io, const void *B, const void *C, float *bc, int64_t N, int64_t L,
                           int64_t Lp, int np, int64_t batch, cudaStream_t s) {
    const dim3 pg((unsigned)(Lp / 32), (unsigned)batch);
    const size_t psm = (size_t)2 * np * 33 * 4;
    if (io == SSM_BF16)
        bc_prep_kernel<bf16><<<pg, 256, psm, s>>>(static_cast<const bf16 *>(B), static_cast<const bf16 *>(C), bc,
                                                  N, L, Lp, np);
    else
        bc_prep_kernel<float><<<pg, 256, psm, s>>>(static_cast<const float *>(B), static_cast<const float *>(C), bc,
                                                   N, L, Lp, np);
    return cudaGetLastError();
}

cudaError_t launch_tc(ssm_dtype_t io, bool pipelined, int G, const TcParams &prm, cudaStream_t s) {
    return io == SSM_BF16 ? launch_tc_io<bf16>(pipelined, G, prm, s) : launch_tc_io<float>(pipelined, G, prm, s);
}

}  // namespace ssm
