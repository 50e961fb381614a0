// Host side of the C ABI declared in include/ssm_scan.h: argument checks, launch planning,
// kernel dispatch, workspace handling and the host-buffer pipeline.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "ssm_scan.h"
#include "common.cuh"
#include "decode.cuh"
#include "scan_seq.cuh"

namespace {

using bf16 = __nv_bfloat16;
using namespace ssm;

constexpr int kTile = 32;
constexpr int kWarps = 4;

__device__ int g_device_status = 0;  // written only by bounded device-side waits

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t io_size(ssm_dtype_t t) { return t == SSM_BF16 ? 2 : 4; }

ssm_status_t check_dims(const ssm_dims_t *dims, bool need_L) {
    if (dims == nullptr) return SSM_ERR_NULL;
    if (dims->batch < 0 || dims->dim < 0 || dims->seqlen < 0 || dims->dstate < 1) return SSM_ERR_SHAPE;
    if (dims->io_dtype != SSM_F32 && dims->io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (dims->dstate > SSM_MAX_DSTATE) return SSM_ERR_UNSUPPORTED;
    // overflow guard: every tensor must have < 2^62 bytes
    const double lim = 4.0e18;
    const double bdl = (double)dims->batch * (double)dims->dim * (double)(need_L ? std::max<int64_t>(dims->seqlen, 1) : 1);
    if (bdl * 4.0 > lim || (double)dims->batch * dims->dstate * (need_L ? std::max<int64_t>(dims->seqlen, 1) : 1) * 4.0 > lim ||
        (double)dims->batch * dims->dim * dims->dstate * 4.0 > lim)
        return SSM_ERR_SHAPE;
    return SSM_OK;
}

// ---- launch plan for the scan ------------------------------------------------------------
struct ScanPlan {
    int nper, g;   // states per lane, lanes per channel
    int nchunks;
    int64_t chunk_len;
};

int sm_count() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

ScanPlan plan_scan(const ssm_dims_t &d) {
    ScanPlan p{16, 1, 1, d.seqlen};
    const int64_t N = d.dstate, chans = d.batch * d.dim;
    const int64_t sms = sm_count();
    if (N <= 4) { p.nper = 4; p.g = 1; }
    else if (N <= 8) { p.nper = 8; p.g = 1; }
    else if (N <= 16) {
        // one lane per channel when that fills the GPU, else four lanes of four states
        if (chans >= sms * 16 * 32) { p.nper = 16; p.g = 1; } else { p.nper = 4; p.g = 4; }
    } else if (N <= 32) { p.nper = 16; p.g = 2; }
    else if (N <= 64) { p.nper = 16; p.g = 4; }
    else { p.nper = 16; p.g = 8; }
    const int64_t warps = (chans * p.g + 31) / 32;
    const int64_t want = sms * 12;
    if (warps < sms * 8 && d.seqlen >= 4 * kTile) {
        int64_t nc = (want + warps - 1) / warps;
        nc = std::min<int64_t>(nc, d.seqlen / (4 * kTile));
        nc = std::max<int64_t>(std::min<int64_t>(nc, 4096), 1);
        p.nchunks = (int)nc;
    }
    if (const char *env = std::getenv("SSM_PLAN")) {  // "nper,g,nchunks" (experiments)
        int a = 0, b = 0, c = 0;
        if (std::sscanf(env, "%d,%d,%d", &a, &b, &c) == 3 && a > 0 && b > 0 && c > 0) {
            p.nper = a; p.g = b; p.nchunks = std::min(c, 4096);
        }
    }
    if (p.nper * p.g < N) p.nper = (int)((N + p.g - 1) / p.g + 3) / 4 * 4;
    int64_t cl = (d.seqlen + p.nchunks - 1) / p.nchunks;
    cl = (cl + kTile - 1) / kTile * kTile;
    p.chunk_len = std::max<int64_t>(cl, kTile);
    p.nchunks = (int)((d.seqlen + p.chunk_len - 1) / p.chunk_len);
    if (p.nchunks < 1) p.nchunks = 1;
    return p;
}

size_t scan_workspace_bytes(const ssm_dims_t &d, const ScanPlan &p) {
    if (p.nchunks <= 1) return 0;
    const size_t BD = (size_t)(d.batch * d.dim), npad = (size_t)(p.nper * p.g);
    const size_t agg_h = (size_t)p.nchunks * BD * npad * 4, agg_s = (size_t)p.nchunks * BD * 4;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    return up(agg_h) + up(agg_s) + up(agg_h);
}

// ---- kernel dispatch -------------------------------------------------------------------
template <typename IO, int NPER, int G, bool AGG, bool AL>
cudaError_t launch_seq_t(const SeqParams &prm, int grid_y, cudaStream_t s) {
    using Cfg = SeqCfg<IO, NPER, G, kWarps, kTile>;
    auto k = scan_seq_kernel<IO, NPER, G, kWarps, kTile, AGG, AL>;
    static unsigned long long attr_set = 0;  // per instantiation: bit i = set on device i
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
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

template <typename IO>
cudaError_t launch_seq(const ScanPlan &pl, const SeqParams &prm, bool agg, bool aligned, int grid_y, cudaStream_t s) {
    switch (pl.nper * 100 + pl.g) {
        case 401: return launch_seq_g<IO, 4, 1>(prm, agg, aligned, grid_y, s);
        case 801: return launch_seq_g<IO, 8, 1>(prm, agg, aligned, grid_y, s);
        case 1601: return launch_seq_g<IO, 16, 1>(prm, agg, aligned, grid_y, s);
        case 404: return launch_seq_g<IO, 4, 4>(prm, agg, aligned, grid_y, s);
        case 1602: return launch_seq_g<IO, 16, 2>(prm, agg, aligned, grid_y, s);
        case 1604: return launch_seq_g<IO, 16, 4>(prm, agg, aligned, grid_y, s);
        case 1608: return launch_seq_g<IO, 16, 8>(prm, agg, aligned, grid_y, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

int channels_per_cta(const ScanPlan &pl) { return kWarps * 32 / pl.g; }

bool plan_supported(const ScanPlan &pl) {
    switch (pl.nper * 100 + pl.g) {
        case 401: case 801: case 1601: case 404: case 1602: case 1604: case 1608: return true;
        default: return false;
    }
}

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) p[i] = 0.0f;
}

ssm_status_t scan_checks(const ssm_dims_t *dims, const void *u, const void *delta, const float *A,
                         const void *B, const void *C, const float *D, const void *z,
                         const float *delta_bias, void *y, float *last_state) {
    ssm_status_t st = check_dims(dims, true);
    if (st != SSM_OK) return st;
    const bool empty = dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0;
    if (!empty && (!u || !delta || !A || !B || !C || !y)) return SSM_ERR_NULL;
    const void *ptrs[] = {u, delta, B, C, z, y, last_state};   // read/written with 16-byte accesses
    for (const void *q : ptrs)
        if (q != nullptr && !aligned16(q)) return SSM_ERR_ALIGN;
    const void *scal[] = {A, D, delta_bias};                    // read element by element
    for (const void *q : scal)
        if (q != nullptr && !aligned_to(q, 4)) return SSM_ERR_ALIGN;
    return SSM_OK;
}

ssm_status_t run_scan(const ssm_dims_t *dims, const void *u, const void *delta, const float *A,
                      const void *B, const void *C, const float *D, const void *z,
                      const float *delta_bias, int delta_softplus, void *y, float *last_state,
                      void *workspace, size_t ws_bytes, bool own_ws, cudaStream_t s) {
    const ssm_dims_t d = *dims;
    if (d.batch == 0 || d.dim == 0) return SSM_OK;
    if (d.seqlen == 0) {
        if (last_state) {
            const int64_t n = d.batch * d.dim * d.dstate;
            zero_f32_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, s>>>(last_state, n);
            if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const ScanPlan pl = plan_scan(d);
    if (!plan_supported(pl)) return SSM_ERR_UNSUPPORTED;
    const size_t need = scan_workspace_bytes(d, pl);
    bool allocated = false;
    if (need > 0) {
        if (workspace == nullptr || ws_bytes < need) {
            if (!own_ws) return SSM_ERR_WORKSPACE;
            if (cudaMallocAsync(&workspace, need, s) != cudaSuccess) return SSM_ERR_CUDA;
            allocated = true;
        } else if (!aligned16(workspace)) {
            return SSM_ERR_ALIGN;
        }
    }
    SeqParams prm{};
    prm.u = u; prm.delta = delta; prm.z = z; prm.B = B; prm.C = C;
    prm.A = A; prm.D = D; prm.bias = delta_bias; prm.y = y; prm.last_state = last_state;
    prm.Bt = d.batch; prm.Dm = d.dim; prm.L = d.seqlen; prm.N = d.dstate;
    prm.softplus = delta_softplus ? 1 : 0;
    prm.chunk_len = pl.chunk_len; prm.nchunks = pl.nchunks;
    const int cpc = channels_per_cta(pl);
    prm.chan_blocks = (int)((d.dim + cpc - 1) / cpc);
    prm.npad = pl.nper * pl.g;
    const size_t esz = io_size(d.io_dtype);
    const bool aligned = ((size_t)d.seqlen * esz) % 16 == 0;
    cudaError_t e = cudaSuccess;
    if (pl.nchunks > 1) {
        const size_t BD = (size_t)(d.batch * d.dim), npad = (size_t)prm.npad;
        auto up = [](size_t x) { return (x + 255) / 256 * 256; };
        char *w = static_cast<char *>(workspace);
        prm.agg_h = reinterpret_cast<float *>(w);
        prm.agg_s = reinterpret_cast<float *>(w + up((size_t)pl.nchunks * BD * npad * 4));
        float *hin = reinterpret_cast<float *>(w + up((size_t)pl.nchunks * BD * npad * 4) + up((size_t)pl.nchunks * BD * 4));
        e = d.io_dtype == SSM_BF16 ? launch_seq<bf16>(pl, prm, true, aligned, pl.nchunks - 1, s)
                                   : launch_seq<float>(pl, prm, true, aligned, pl.nchunks - 1, s);
        if (e == cudaSuccess) {
            const int64_t total = (int64_t)BD * prm.npad;
            chunk_combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
                A, prm.agg_h, prm.agg_s, hin, (int64_t)BD, d.dim, d.dstate, prm.npad, pl.nchunks);
            e = cudaGetLastError();
        }
        prm.hin = hin;
    }
    if (e == cudaSuccess)
        e = d.io_dtype == SSM_BF16 ? launch_seq<bf16>(pl, prm, false, aligned, pl.nchunks, s)
                                   : launch_seq<float>(pl, prm, false, aligned, pl.nchunks, s);
    if (allocated) cudaFreeAsync(workspace, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" {

ssm_status_t ssm_selective_scan_fwd(const ssm_dims_t *dims, const void *u, const void *delta,
                                    const float *A, const void *B, const void *C, const float *D,
                                    const void *z, const float *delta_bias, int delta_softplus,
                                    void *y, float *last_state, void *stream) {
    ssm_status_t st = scan_checks(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                    nullptr, 0, true, static_cast<cudaStream_t>(stream));
}

size_t ssm_selective_scan_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    return scan_workspace_bytes(*dims, plan_scan(*dims));
}

ssm_status_t ssm_selective_scan_fwd_ws(const ssm_dims_t *dims, const void *u, const void *delta,
                                       const float *A, const void *B, const void *C,
                                       const float *D, const void *z, const float *delta_bias,
                                       int delta_softplus, void *y, float *last_state,
                                       void *workspace, size_t workspace_bytes, void *stream) {
    ssm_status_t st = scan_checks(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    if (workspace != nullptr && !aligned16(workspace)) return SSM_ERR_ALIGN;
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                    workspace, workspace_bytes, false, static_cast<cudaStream_t>(stream));
}

ssm_status_t ssm_state_update(const ssm_dims_t *dims, float *state, const void *x, const void *dt,
                              const float *A, const void *B, const void *C, const float *D,
                              const void *z, void *y, void *stream) {
    ssm_status_t st = check_dims(dims, false);
    if (st != SSM_OK) return st;
    if (dims->batch == 0 || dims->dim == 0) return SSM_OK;
    if (!state || !x || !dt || !A || !B || !C || !y) return SSM_ERR_NULL;
    // state and A: 16-byte aligned (vector path); per-token vectors: element-aligned, so
    // they may be rows of a [steps][batch][dim] array
    if (!aligned16(state) || !aligned16(A)) return SSM_ERR_ALIGN;
    const size_t esz = io_size(dims->io_dtype);
    const void *tok[] = {x, dt, B, C, z, y};
    for (const void *q : tok)
        if (q != nullptr && !aligned_to(q, esz)) return SSM_ERR_ALIGN;
    if (D != nullptr && !aligned_to(D, 4)) return SSM_ERR_ALIGN;
    DecodeParams p{state, x, dt, B, C, z, A, D, y, dims->batch, dims->dim, dims->dstate};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t N = dims->dstate, chans = dims->batch * dims->dim;
    const bool bf = dims->io_dtype == SSM_BF16;
    const int lpc = (int)(N / 4);
    if (N % 4 == 0 && lpc >= 1 && lpc <= 32 && (32 % lpc) == 0) {
        const int64_t threads = chans * lpc;
        const unsigned grid = (unsigned)((threads + 255) / 256);
#define SSM_DEC(L) \
    case L: bf ? decode_vec_kernel<bf16, L><<<grid, 256, 0, s>>>(p) : decode_vec_kernel<float, L><<<grid, 256, 0, s>>>(p); break;
        switch (lpc) { SSM_DEC(1) SSM_DEC(2) SSM_DEC(4) SSM_DEC(8) SSM_DEC(16) SSM_DEC(32) default: return SSM_ERR_UNSUPPORTED; }
#undef SSM_DEC
    } else {
        const unsigned grid = (unsigned)((chans + 255) / 256);
        if (bf) decode_scalar_kernel<bf16><<<grid, 256, 0, s>>>(p);
        else decode_scalar_kernel<float><<<grid, 256, 0, s>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status_t ssm_selective_scan_fwd_host(const ssm_dims_t *dims, const void *u, const void *delta,
                                         const float *A, const void *B, const void *C,
                                         const float *D, const void *z, const float *delta_bias,
                                         int delta_softplus, void *y, float *last_state,
                                         void *stream) {
    ssm_status_t st = check_dims(dims, true);
    if (st != SSM_OK) return st;
    const ssm_dims_t d = *dims;
    if (d.batch == 0 || d.dim == 0) return SSM_OK;
    if (d.seqlen > 0 && (!u || !delta || !A || !B || !C || !y)) return SSM_ERR_NULL;
    if (d.seqlen == 0) {
        if (last_state) std::memset(last_state, 0, sizeof(float) * (size_t)(d.batch * d.dim * d.dstate));
        return SSM_OK;
    }
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    const size_t esz = io_size(d.io_dtype);
    const size_t L = (size_t)d.seqlen, N = (size_t)d.dstate, Dm = (size_t)d.dim;
    // blocks of channels within a batch row; two pipelines alternate
    const size_t nblk_per_row = std::max<size_t>(1, std::min<size_t>(Dm, 4));
    // blocks start on multiples of 4 channels so that A + d0*N, D + d0 and bias + d0 stay
    // 16-byte aligned; each batch row of B and C gets its own 256-byte aligned slot
    const size_t blk = ((Dm + nblk_per_row - 1) / nblk_per_row + 3) / 4 * 4;
    const size_t bc_row = (N * L * esz + 255) / 256 * 256;
    cudaStream_t ss[2] = {nullptr, nullptr};
    cudaEvent_t ev_in = nullptr;
    ssm_status_t rc = SSM_OK;
    void *dA = nullptr, *dD = nullptr, *dbias = nullptr, *dB = nullptr, *dC = nullptr;
    void *bu[2] = {nullptr, nullptr}, *bdl[2] = {nullptr, nullptr}, *bz[2] = {nullptr, nullptr};
    void *by[2] = {nullptr, nullptr}, *bst[2] = {nullptr, nullptr};
    const size_t row_bytes = blk * L * esz;
    auto CK = [&](cudaError_t e) { if (e != cudaSuccess && rc == SSM_OK) rc = SSM_ERR_CUDA; return e == cudaSuccess; };
    CK(cudaStreamCreateWithFlags(&ss[0], cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&ss[1], cudaStreamNonBlocking));
    CK(cudaEventCreateWithFlags(&ev_in, cudaEventDisableTiming));
    if (rc == SSM_OK) {
        CK(cudaMallocAsync(&dA, Dm * N * 4, s0));
        if (D) CK(cudaMallocAsync(&dD, Dm * 4, s0));
        if (delta_bias) CK(cudaMallocAsync(&dbias, Dm * 4, s0));
        CK(cudaMallocAsync(&dB, (size_t)d.batch * bc_row, s0));
        CK(cudaMallocAsync(&dC, (size_t)d.batch * bc_row, s0));
        for (int i = 0; i < 2; ++i) {
            CK(cudaMallocAsync(&bu[i], row_bytes, s0));
            CK(cudaMallocAsync(&bdl[i], row_bytes, s0));
            if (z) CK(cudaMallocAsync(&bz[i], row_bytes, s0));
            CK(cudaMallocAsync(&by[i], row_bytes, s0));
            if (last_state) CK(cudaMallocAsync(&bst[i], blk * N * 4, s0));
        }
    }
    if (rc == SSM_OK) {
        CK(cudaMemcpyAsync(dA, A, Dm * N * 4, cudaMemcpyHostToDevice, s0));
        if (D) CK(cudaMemcpyAsync(dD, D, Dm * 4, cudaMemcpyHostToDevice, s0));
        if (delta_bias) CK(cudaMemcpyAsync(dbias, delta_bias, Dm * 4, cudaMemcpyHostToDevice, s0));
        for (int64_t b = 0; b < d.batch; ++b) {
            CK(cudaMemcpyAsync(static_cast<char *>(dB) + b * bc_row, static_cast<const char *>(B) + b * N * L * esz,
                               N * L * esz, cudaMemcpyHostToDevice, s0));
            CK(cudaMemcpyAsync(static_cast<char *>(dC) + b * bc_row, static_cast<const char *>(C) + b * N * L * esz,
                               N * L * esz, cudaMemcpyHostToDevice, s0));
        }
        CK(cudaEventRecord(ev_in, s0));
        CK(cudaStreamWaitEvent(ss[0], ev_in, 0));
        CK(cudaStreamWaitEvent(ss[1], ev_in, 0));
    }
    size_t it = 0;
    for (int64_t b = 0; b < d.batch && rc == SSM_OK; ++b) {
        for (size_t d0 = 0; d0 < Dm && rc == SSM_OK; d0 += blk, ++it) {
            const int k = (int)(it & 1);
            cudaStream_t s = ss[k];
            const size_t nd = std::min(blk, Dm - d0);
            const size_t off = ((size_t)b * Dm + d0) * L * esz;
            CK(cudaMemcpyAsync(bu[k], static_cast<const char *>(u) + off, nd * L * esz, cudaMemcpyHostToDevice, s));
            CK(cudaMemcpyAsync(bdl[k], static_cast<const char *>(delta) + off, nd * L * esz, cudaMemcpyHostToDevice, s));
            if (z) CK(cudaMemcpyAsync(bz[k], static_cast<const char *>(z) + off, nd * L * esz, cudaMemcpyHostToDevice, s));
            ssm_dims_t sub{1, (int64_t)nd, d.seqlen, d.dstate, d.io_dtype};
            const size_t boff = (size_t)b * bc_row;
            ssm_status_t r = ssm_selective_scan_fwd(
                &sub, bu[k], bdl[k], static_cast<float *>(dA) + d0 * N, static_cast<char *>(dB) + boff,
                static_cast<char *>(dC) + boff, D ? static_cast<float *>(dD) + d0 : nullptr, z ? bz[k] : nullptr,
                delta_bias ? static_cast<float *>(dbias) + d0 : nullptr, delta_softplus, by[k],
                last_state ? static_cast<float *>(bst[k]) : nullptr, s);
            if (r != SSM_OK) { rc = r; break; }
            CK(cudaMemcpyAsync(static_cast<char *>(y) + off, by[k], nd * L * esz, cudaMemcpyDeviceToHost, s));
            if (last_state)
                CK(cudaMemcpyAsync(last_state + ((size_t)b * Dm + d0) * N, bst[k], nd * N * 4, cudaMemcpyDeviceToHost, s));
        }
    }
    for (int i = 0; i < 2; ++i)
        if (ss[i]) CK(cudaStreamSynchronize(ss[i]));
    // release everything on s0 after both pipelines finished
    void *all[] = {dA, dD, dbias, dB, dC, bu[0], bu[1], bdl[0], bdl[1], bz[0], bz[1], by[0], by[1], bst[0], bst[1]};
    for (void *q : all)
        if (q) cudaFreeAsync(q, s0);
    CK(cudaStreamSynchronize(s0));
    for (int i = 0; i < 2; ++i)
        if (ss[i]) cudaStreamDestroy(ss[i]);
    if (ev_in) cudaEventDestroy(ev_in);
    return rc;
}

ssm_status_t ssm_stream_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
        return static_cast<ssm_status_t>(v);
    }
    return SSM_OK;
}

const char *ssm_status_string(ssm_status_t status) {
    switch (status) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_NULL: return "SSM_ERR_NULL: a required pointer is NULL";
        case SSM_ERR_SHAPE: return "SSM_ERR_SHAPE: invalid dimensions";
        case SSM_ERR_DTYPE: return "SSM_ERR_DTYPE: unknown io dtype";
        case SSM_ERR_ALIGN: return "SSM_ERR_ALIGN: pointer not aligned as required";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: unsupported configuration";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA: CUDA runtime error";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT: a bounded device-side wait gave up";
        case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE: workspace missing or too small";
        default: return "SSM_ERR_UNKNOWN";
    }
}

int ssm_version(void) { return (1 << 16) | 0; }

}  // extern "C"
