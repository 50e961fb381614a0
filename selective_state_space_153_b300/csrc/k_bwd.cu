// Selective scan backward launches (scan_bwd.cuh): checkpoint pass, then the adjoint pass.
#include "launch.h"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, int G, int Q>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t s) {
    constexpr size_t tb = bwd_tile_bytes<G, Q>(), sm = tb + bwd_smem_bytes(G, Q);
    const dim3 grid((unsigned)((p.Dm + kBwdThreads / G - 1) / (kBwdThreads / G)), (unsigned)p.Bt);
    static unsigned long long attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sm);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    scan_bwd_ckpt_kernel<IO, G, Q><<<grid, kBwdThreads, tb, s>>>(p);
    scan_bwd_kernel<IO, G, Q><<<grid, kBwdThreads, sm, s>>>(p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(int G, int Q, const BwdParams &p, cudaStream_t s) {
    switch (G * 10 + Q) {
#define SSM_BWD(GG, QQ) case GG * 10 + QQ: return launch_bwd_t<IO, GG, QQ>(p, s);
        SSM_BWD(1, 1) SSM_BWD(1, 2) SSM_BWD(2, 2) SSM_BWD(4, 2) SSM_BWD(8, 2) SSM_BWD(16, 2)
        SSM_BWD(32, 2) SSM_BWD(32, 4)
#undef SSM_BWD
        default: return cudaErrorInvalidConfiguration;
    }
}
}  // namespace

cudaError_t launch_bwd(ssm_dtype_t io, int G, int Q, const BwdParams &p, cudaStream_t s) {
    return io == SSM_BF16 ? launch_bwd_io<bf16>(G, Q, p, s) : launch_bwd_io<float>(G, Q, p, s);
}

}  // namespace ssm
