// Selective scan backward launches (scan_bwd.cuh): checkpoint pass (with a time split, in one
// launch with the adjoint aggregate pass, then the chunk combine); then the adjoint pass.
#include <algorithm>

#include "launch.h"

namespace ssm {

// Time split, combine: one thread per (batch row and channel, state slot n < np). Walks the
// chunks forwards with the state entering each (H_0 = 0, H_{k+1} = exp(A*sdt_k) H_k + hloc_k),
// leaving H_k in place of hloc_k, then backwards with the adjoint carry entering each chunk's
// last step (cin_{last} = dlast, cin_{k-1} = exp(A*sdt_k) cin_k + cloc_k).
__global__ void __launch_bounds__(256) bwd_chunk_combine_kernel(const BwdParams p, int np) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.Bt * p.Dm * np) return;
    const int64_t bd = idx / np, d = bd % p.Dm;
    const int n = (int)(idx % np);
    const float Ap = n < p.N ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + d * p.N + n) * kLog2e : 0.0f;
    const uint64_t cb = bwd_chunk_bytes(p, np), sb = bwd_chunk_bytes(p, 1);
    // every address is read (through the read-only path) before this thread writes it, and no
    // other thread touches it, so the loads of later chunks may run ahead of the stores
    auto ldro = [](const float *base, uint64_t total, const float *q) {
        return SSM_CHK_G(base, total, q, 4) ? __ldg(q) : 0.0f;
    };
    float H = 0.0f;
#pragma unroll 8
    for (int kc = 0; kc < p.nchunk; ++kc) {
        float *hl = p.hloc + (bd * p.nchunk + kc) * np + n;
        const float loc = ldro(p.hloc, cb, hl);
        const float a = ex2(Ap * ldro(p.sdt, sb, p.sdt + bd * p.nchunk + kc));
        st_chk_g(p.hloc, cb, hl, H);
        H = fmaf(a, H, loc);
    }
    float c = (n < p.N && p.dlast) ? ld_chk_g(p.dlast, (uint64_t)(p.Bt * p.Dm * p.N) * 4, p.dlast + bd * p.N + n) : 0.0f;
#pragma unroll 8
    for (int kc = p.nchunk - 1; kc >= 0; --kc) {
        st_chk_g(p.cin, cb, p.cin + (bd * p.nchunk + kc) * np + n, c);
        if (kc > 0)
            c = fmaf(ex2(Ap * ldro(p.sdt, sb, p.sdt + bd * p.nchunk + kc)), c,
                     ldro(p.cloc, cb, p.cloc + (bd * p.nchunk + kc) * np + n));
    }
}

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, int G, int Q>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t s) {
    constexpr size_t ck = bwd_ckpt_smem_bytes<IO, G, Q>(), sm = bwd_smem_bytes<IO, G, Q, false>();
    constexpr size_t sms = bwd_smem_bytes<IO, G, Q, true>();
    constexpr size_t ag = bwd_agg_smem_bytes<IO, G, Q>(), fr = ck > ag ? ck : ag;
    constexpr int kCpb = BwdCfg<G, Q>::kCpb;
    const dim3 grid((unsigned)((p.Dm + kCpb - 1) / kCpb), (unsigned)p.Bt, (unsigned)p.nchunk);
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(scan_bwd_kernel<IO, G, Q, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_kernel<IO, G, Q, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sms);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_ckpt_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_split_front_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)fr);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (p.nchunk > 1) {   // time split: chunk-local checkpoints and adjoint carries, both combines
        scan_bwd_split_front_kernel<IO, G, Q><<<dim3(grid.x, grid.y, 2 * grid.z - 1), kBwdThreads, fr, s>>>(p);
        const int64_t threads = p.Bt * p.Dm * (int64_t)(G * Q);
        bwd_chunk_combine_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p, G * Q);
        scan_bwd_kernel<IO, G, Q, true><<<grid, kBwdThreads, sms, s>>>(p);
    } else {
        scan_bwd_ckpt_kernel<IO, G, Q><<<grid, kBwdThreads, ck, s>>>(p);
        scan_bwd_kernel<IO, G, Q, false><<<grid, kBwdThreads, sm, s>>>(p);
    }
    return cudaGetLastError();
}

// CTAs of the split adjoint pass that fit one SM: its launch bound, or what its shared memory
// allows (228 KB per SM, 1 KB of it reserved per CTA)
template <typename IO, int G, int Q>
int split_adjoint_ctas_t() {
    constexpr int by_smem = (int)(233472 / (bwd_smem_bytes<IO, G, Q, true>() + 1024));
    return std::min(Q == 4 ? 3 : 4, by_smem);
}

// lane splits built: four states per lane with 1-32 lanes per channel, two states per lane
// with 2-16
template <typename IO>
int split_adjoint_ctas_io(int G, int Q) {
    switch (Q * 100 + G) {
        case 401: return split_adjoint_ctas_t<IO, 1, 4>();
        case 402: return split_adjoint_ctas_t<IO, 2, 4>();
        case 404: return split_adjoint_ctas_t<IO, 4, 4>();
        case 408: return split_adjoint_ctas_t<IO, 8, 4>();
        case 416: return split_adjoint_ctas_t<IO, 16, 4>();
        case 432: return split_adjoint_ctas_t<IO, 32, 4>();
        case 202: return split_adjoint_ctas_t<IO, 2, 2>();
        case 204: return split_adjoint_ctas_t<IO, 4, 2>();
        case 208: return split_adjoint_ctas_t<IO, 8, 2>();
        case 216: return split_adjoint_ctas_t<IO, 16, 2>();
        default: return 1;
    }
}

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

int bwd_split_adjoint_ctas_per_sm(ssm_dtype_t io, int G, int Q) {
    return io == SSM_BF16 ? split_adjoint_ctas_io<bf16>(G, Q) : split_adjoint_ctas_io<float>(G, Q);
}

}  // namespace ssm
