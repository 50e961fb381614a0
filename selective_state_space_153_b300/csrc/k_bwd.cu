// Selective scan backward launches (scan_bwd.cuh): checkpoint pass, then the adjoint pass.
#include "launch.h"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, int G>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t s) {
    constexpr size_t ck = bwd_ckpt_smem_bytes<G>(), sm = bwd_smem_bytes<G>();
    const dim3 grid((unsigned)((p.Dm + BwdCfg<G>::kCpb - 1) / BwdCfg<G>::kCpb), (unsigned)p.Bt);
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(scan_bwd_kernel<IO, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_ckpt_kernel<IO, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck);
        return r;
    });
    if (e != cudaSuccess) return e;
    scan_bwd_ckpt_kernel<IO, G><<<grid, kBwdThreads, ck, s>>>(p);
    scan_bwd_kernel<IO, G><<<grid, kBwdThreads, sm, s>>>(p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(int G, const BwdParams &p, cudaStream_t s) {
    switch (G) {
        case 1: return launch_bwd_t<IO, 1>(p, s);
        case 2: return launch_bwd_t<IO, 2>(p, s);
        case 4: return launch_bwd_t<IO, 4>(p, s);
        case 8: return launch_bwd_t<IO, 8>(p, s);
        case 16: return launch_bwd_t<IO, 16>(p, s);
        case 32: return launch_bwd_t<IO, 32>(p, s);
        default: return cudaErrorInvalidConfiguration;
    }
}
}  // namespace

cudaError_t launch_bwd(ssm_dtype_t io, int G, const BwdParams &p, cudaStream_t s) {
    return io == SSM_BF16 ? launch_bwd_io<bf16>(G, p, s) : launch_bwd_io<float>(G, p, s);
}

}  // namespace ssm
