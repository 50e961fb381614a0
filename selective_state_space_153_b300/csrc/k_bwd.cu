// Selective scan backward launches (scan_bwd.cuh): checkpoint pass, then the adjoint pass.
#include "launch.h"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, int G, int Q>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t s) {
    constexpr size_t ck = bwd_ckpt_smem_bytes<IO, G, Q>(), sm = bwd_smem_bytes<IO, G, Q>();
    constexpr int kCpb = BwdCfg<G, Q>::kCpb;
    const dim3 grid((unsigned)((p.Dm + kCpb - 1) / kCpb), (unsigned)p.Bt);
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(scan_bwd_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_ckpt_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck);
        return r;
    });
    if (e != cudaSuccess) return e;
    scan_bwd_ckpt_kernel<IO, G, Q><<<grid, kBwdThreads, ck, s>>>(p);
    scan_bwd_kernel<IO, G, Q><<<grid, kBwdThreads, sm, s>>>(p);
    return cudaGetLastError();
}

// lane splits built: four states per lane with 1-32 lanes per channel, two states per lane
// with 2-16
template <typename IO>
cudaError_t launch_bwd_io(int G, int Q, const BwdParams &p, cudaStream_t s) {
    switch (Q * 100 + G) {
        case 401: return launch_bwd_t<IO, 1, 4>(p, s);
        case 402: return launch_bwd_t<IO, 2, 4>(p, s);
        case 404: return launch_bwd_t<IO, 4, 4>(p, s);
        case 408: return launch_bwd_t<IO, 8, 4>(p, s);
        case 416: return launch_bwd_t<IO, 16, 4>(p, s);
        case 432: return launch_bwd_t<IO, 32, 4>(p, s);
        case 202: return launch_bwd_t<IO, 2, 2>(p, s);
        case 204: return launch_bwd_t<IO, 4, 2>(p, s);
        case 208: return launch_bwd_t<IO, 8, 2>(p, s);
        case 216: return launch_bwd_t<IO, 16, 2>(p, s);
        default: return cudaErrorInvalidConfiguration;
    }
}
}  // namespace

cudaError_t launch_bwd(ssm_dtype_t io, int G, int Q, const BwdParams &p, cudaStream_t s) {
    return io == SSM_BF16 ? launch_bwd_io<bf16>(G, Q, p, s) : launch_bwd_io<float>(G, Q, p, s);
}

}  // namespace ssm
