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

// The same combine with the chunks spread over a warp (nchunk <= 64): lane l owns chunks 2l and
// 2l+1, and the chains become scans of affine maps (x -> m*x + c; "x then y" composes to
// (m_y m_x, m_y c_x + c_y)), forwards over the states entering the chunks and backwards over
// the adjoint carries, in five shuffle steps each. One warp per (row, state slot).
__device__ __forceinline__ float2 affine_then(float2 x, float2 y) {   // apply x, then y
    return make_float2(y.x * x.x, fmaf(y.x, x.y, y.y));
}
__global__ void __launch_bounds__(256) bwd_chunk_combine_warp_kernel(const BwdParams p, int np) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= p.Bt * p.Dm * np) return;                 // whole warps leave together
    const int64_t bd = w / np, d = bd % p.Dm;
    const int n = (int)(w % np), K = p.nchunk;
    const float Ap = n < p.N ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + d * p.N + n) * kLog2e : 0.0f;
    const uint64_t cb = bwd_chunk_bytes(p, np), sb = bwd_chunk_bytes(p, 1);
    const int k0 = 2 * lane, k1 = k0 + 1;
    // chunk k's decay product over its steps, its state from 0 and its adjoint carry from 0
    auto decay = [&](int k) { return ex2(Ap * ld_chk_g(p.sdt, sb, p.sdt + bd * K + k)); };
    const float P0 = k0 < K ? decay(k0) : 1.0f, P1 = k1 < K ? decay(k1) : 1.0f;
    float *hl0 = p.hloc + (bd * K + k0) * np + n, *hl1 = p.hloc + (bd * K + k1) * np + n;
    const float h0 = k0 < K ? ld_chk_g(p.hloc, cb, hl0) : 0.0f, h1 = k1 < K ? ld_chk_g(p.hloc, cb, hl1) : 0.0f;
    // forward: exclusive scan of the lanes' maps (chunk k0 then k1) over lower lanes
    const float2 f0 = make_float2(P0, h0), f1 = make_float2(P1, h1);
    float2 inc = affine_then(f0, f1);
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
        const float2 up = make_float2(__shfl_up_sync(0xffffffffu, inc.x, o), __shfl_up_sync(0xffffffffu, inc.y, o));
        if (lane >= o) inc = affine_then(up, inc);
    }
    const float prev = __shfl_up_sync(0xffffffffu, inc.y, 1);
    const float Hin = lane > 0 ? prev : 0.0f;                          // applied to H_0 = 0
    if (k0 < K) st_chk_g(p.hloc, cb, hl0, Hin);                    // state entering chunk k0
    if (k1 < K) st_chk_g(p.hloc, cb, hl1, fmaf(P0, Hin, h0));      // entering chunk k1
    // backward: carry into chunk k-1 = P_k * (carry into chunk k) + cloc_k, chunk 0's map unused
    auto cl = [&](int k) { return ld_chk_g(p.cloc, cb, p.cloc + (bd * K + k) * np + n); };
    const float2 g0 = (k0 >= 1 && k0 < K) ? make_float2(P0, cl(k0)) : make_float2(1.0f, 0.0f);
    const float2 g1 = k1 < K ? make_float2(P1, cl(k1)) : make_float2(1.0f, 0.0f);
    float2 suf = affine_then(g1, g0);                                 // chunk k1's map, then k0's
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
        const float2 dn = make_float2(__shfl_down_sync(0xffffffffu, suf.x, o), __shfl_down_sync(0xffffffffu, suf.y, o));
        if (lane + o < 32) suf = affine_then(dn, suf);                // higher chunks act first
    }
    float2 ex = make_float2(__shfl_down_sync(0xffffffffu, suf.x, 1), __shfl_down_sync(0xffffffffu, suf.y, 1));
    if (lane == 31) ex = make_float2(1.0f, 0.0f);
    const float dl = (n < p.N && p.dlast) ? ld_chk_g(p.dlast, (uint64_t)(p.Bt * p.Dm * p.N) * 4, p.dlast + bd * p.N + n) : 0.0f;
    const float c1 = fmaf(ex.x, dl, ex.y);                           // carry into chunk k1
    if (k1 < K) st_chk_g(p.cin, cb, p.cin + (bd * K + k1) * np + n, c1);
    if (k0 < K) st_chk_g(p.cin, cb, p.cin + (bd * K + k0) * np + n, k1 < K ? fmaf(g1.x, c1, g1.y) : c1);
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
        const int64_t rows = p.Bt * p.Dm * (int64_t)(G * Q);
        // the warp scan from 32 chunks: below, the loop's coalesced accesses (consecutive
        // threads, consecutive states) beat a warp of mostly idle lanes (measured on B300:
        // 11-26 chunks 1.4-2.5x slower with the scan, 32-37 chunks 1.1-1.7x faster)
        if (p.nchunk >= 32 && p.nchunk <= 64)
            bwd_chunk_combine_warp_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, s>>>(p, G * Q);
        else
            bwd_chunk_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p, G * Q);
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
