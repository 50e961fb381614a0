// Selective scan backward launches (scan_bwd.cuh): checkpoint pass; with a time split the
// adjoint aggregate pass, the chunk combine and the checkpoint correction; then the adjoint
// pass.
#include "launch.h"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

// Time split, combine: one thread per (batch row and channel, state slot n < np). Walks the
// chunks forwards with the state entering each (H_0 = 0, H_{k+1} = exp(A*sdt_k) H_k + hloc_k),
// leaving H_k in place of hloc_k, then backwards with the adjoint carry entering each chunk's
// last step (cin_{last} = dlast, cin_{k-1} = exp(A*sdt_k) cin_k + cloc_k).
__global__ void __launch_bounds__(256) bwd_chunk_combine_kernel(const BwdParams p, int np) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.Bt * p.Dm * np) return;
    const int64_t bd = idx / np, d = bd % p.Dm;
    const int n = (int)(idx % np);
    const float Ap = n < p.N ? p.A[d * p.N + n] * kLog2e : 0.0f;
    float H = 0.0f;
    for (int kc = 0; kc < p.nchunk; ++kc) {
        float *hl = p.hloc + (bd * p.nchunk + kc) * np + n;
        const float loc = *hl;
        *hl = H;
        H = fmaf(ex2(Ap * p.sdt[bd * p.nchunk + kc]), H, loc);
    }
    float c = (n < p.N && p.dlast) ? p.dlast[bd * p.N + n] : 0.0f;
    for (int kc = p.nchunk - 1; kc >= 0; --kc) {
        p.cin[(bd * p.nchunk + kc) * np + n] = c;
        if (kc > 0) c = fmaf(ex2(Ap * p.sdt[bd * p.nchunk + kc]), c, p.cloc[(bd * p.nchunk + kc) * np + n]);
    }
}

// Time split, checkpoints of chunks 1..: the checkpoint pass took the state from 0 at the
// chunk; add exp(A*cumdt) H_k, H_k the state entering the chunk. One thread per four state
// slots of one (batch row and channel, segment).
__global__ void __launch_bounds__(256) bwd_ckpt_fix_kernel(const BwdParams p, int np) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int nq = np / 4;
    if (idx >= p.Bt * p.Dm * p.nseg * nq) return;
    const int64_t row = idx / nq, bd = row / p.nseg, d = bd % p.Dm;
    const int seg = (int)(row % p.nseg), n = 4 * (int)(idx % nq), kc = seg / p.seg_per_chunk;
    if (kc == 0) return;
    const float e = p.cumdt[bd * p.nseg + seg] * kLog2e;
    const float4 H = *reinterpret_cast<const float4 *>(p.hloc + (bd * p.nchunk + kc) * np + n);
    float4 *q = reinterpret_cast<float4 *>(p.ckpt + row * np + n);
    float4 v = *q;
    v.x = fmaf(n + 0 < p.N ? ex2(p.A[d * p.N + n + 0] * e) : 1.0f, H.x, v.x);
    v.y = fmaf(n + 1 < p.N ? ex2(p.A[d * p.N + n + 1] * e) : 1.0f, H.y, v.y);
    v.z = fmaf(n + 2 < p.N ? ex2(p.A[d * p.N + n + 2] * e) : 1.0f, H.z, v.z);
    v.w = fmaf(n + 3 < p.N ? ex2(p.A[d * p.N + n + 3] * e) : 1.0f, H.w, v.w);
    *q = v;
}

template <typename IO, int G, int Q>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t s) {
    constexpr size_t ck = bwd_ckpt_smem_bytes<IO, G, Q>(), sm = bwd_smem_bytes<IO, G, Q>();
    constexpr size_t ag = bwd_agg_smem_bytes<IO, G, Q>();
    constexpr int kCpb = BwdCfg<G, Q>::kCpb;
    const dim3 grid((unsigned)((p.Dm + kCpb - 1) / kCpb), (unsigned)p.Bt, (unsigned)p.nchunk);
    static std::atomic<unsigned long long> attr_set{0};
    const cudaError_t e = once_per_device(attr_set, [&] {
        cudaError_t r = cudaFuncSetAttribute(scan_bwd_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_ckpt_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(scan_bwd_agg_kernel<IO, G, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ag);
        return r;
    });
    if (e != cudaSuccess) return e;
    scan_bwd_ckpt_kernel<IO, G, Q><<<grid, kBwdThreads, ck, s>>>(p);
    if (p.nchunk > 1) {   // time split: the adjoint carries of chunks 1.., then both combines
        scan_bwd_agg_kernel<IO, G, Q><<<dim3(grid.x, grid.y, grid.z - 1), kBwdThreads, ag, s>>>(p);
        const int64_t threads = p.Bt * p.Dm * (int64_t)(G * Q);
        bwd_chunk_combine_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p, G * Q);
        const int64_t fix = p.Bt * p.Dm * (int64_t)p.nseg * (G * Q / 4);
        bwd_ckpt_fix_kernel<<<(unsigned)((fix + 255) / 256), 256, 0, s>>>(p, G * Q);
    }
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
