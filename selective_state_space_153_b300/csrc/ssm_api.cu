// Host side of the C ABI declared in include/ssm_scan.h: argument checks, launch planning,
// kernel dispatch, workspace handling and the host-buffer pipeline.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <atomic>
#include <mutex>

#include "ssm_scan.h"
#include "common.cuh"
#include "ptx.cuh"
#include "decode.cuh"
#include "scan_seq.cuh"
#include "scan_tc.cuh"
#include "scan_tp.cuh"
#include "scan_pair.cuh"
#include "scan_bwd.cuh"

namespace {

using bf16 = __nv_bfloat16;
using namespace ssm;

constexpr int kTile = 32;
constexpr int kWarps = 4;

// structured-A detection in the forward scans (ssm_set_structured_a): 1 = on, 0 = off
std::atomic<int> g_structured_a{0};


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

size_t seq_workspace_bytes(const ssm_dims_t &d, const ScanPlan &p) {
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

// ---- persistent TMEM-replay path ---------------------------------------------------------
struct TcPlan {
    bool use = false;
    bool pipelined = true;   // scan_tp_kernel (default, dstate <= 64) or scan_tc_kernel
    int T = kTpT;
    int cpw = 8, np = 64;    // channels per group, padded states
    int G = 4, NG = 0, groups_per_b = 0, nseg = 1, seg_tiles = 1, ntiles = 0;
    int64_t Lp = 0;
    size_t off_carry = 0, off_bc = 0, bytes = 0, ctrl_bytes = 0;
};

bool env_is(const char *name, const char *val) {
    const char *e = std::getenv(name);
    return e != nullptr && std::strcmp(e, val) == 0;
}

TcPlan plan_tc(const ssm_dims_t &d) {
    TcPlan t;
    if (env_is("SSM_KERNEL", "seq")) return t;
    const size_t esz = io_size(d.io_dtype);
    if (((size_t)d.seqlen * esz) % 16 != 0) return t;                       // TMA row strides
    if (d.seqlen >= (int64_t)1 << 30 || d.dim >= (int64_t)1 << 30 || d.batch >= (int64_t)1 << 30) return t;
    const int64_t N = d.dstate;
    // pipelined kernel: GP = 8-state groups per channel pair (N <= 64), 64/GP channels per group;
    // otherwise the barrier-phased kernel: G = 16-state groups per channel, 32/G channels
    // (fp32 with N <= 8 would need 64-channel groups whose tiles do not fit shared memory)
    t.pipelined = !env_is("SSM_KERNEL", "tc") && N <= 64 && !(N <= 8 && d.io_dtype == SSM_F32);
    if (t.pipelined) {
        t.G = N <= 8 ? 1 : (N <= 16 ? 2 : (N <= 32 ? 4 : 8));
        t.cpw = 64 / t.G;
        t.np = 8 * t.G;
    } else {
        t.G = N <= 16 ? 1 : (N <= 32 ? 2 : (N <= 64 ? 4 : 8));
        t.cpw = 32 / t.G;
        t.np = 16 * t.G;
    }
    const int cpw = t.cpw;
    t.groups_per_b = (int)((d.dim + cpw - 1) / cpw);
    const int64_t ng = d.batch * t.groups_per_b;
    t.T = t.pipelined ? kTpT : kTcT;
    t.ntiles = (int)((d.seqlen + t.T - 1) / t.T);
    const int64_t sms = sm_count();
    const bool forced = env_is("SSM_KERNEL", "tc") || env_is("SSM_KERNEL", "tp");
    if (ng >= (int64_t)1 << 24) return t;
    if (!forced && (ng < sms || t.ntiles < 4)) return t;
    t.NG = (int)ng;
    int64_t nseg = (16 * sms + ng - 1) / ng;
    nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, t.ntiles));
    t.seg_tiles = (int)((t.ntiles + nseg - 1) / nseg);
    t.nseg = (t.ntiles + t.seg_tiles - 1) / t.seg_tiles;
    t.Lp = (int64_t)t.ntiles * t.T;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    t.ctrl_bytes = up((size_t)(1 + t.NG) * 4);
    t.off_carry = t.ctrl_bytes;
    t.off_bc = t.off_carry + up((size_t)t.NG * 2 * 512 * 4);
    t.bytes = t.off_bc + up((size_t)d.batch * t.Lp * 2 * t.np * 4);
    t.use = true;
    return t;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [Bt][Dm][L] io tensor, box [1][CPW][box_t]
bool make_map(CUtensorMap *m, const void *base, const ssm_dims_t &d, int cpw, int box_t) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const size_t esz = io_size(d.io_dtype);
    const cuuint64_t dims[3] = {(cuuint64_t)d.seqlen, (cuuint64_t)d.dim, (cuuint64_t)d.batch};
    const cuuint64_t strides[2] = {(cuuint64_t)(d.seqlen * esz), (cuuint64_t)(d.seqlen * d.dim * esz)};
    const cuuint32_t box[3] = {(cuuint32_t)box_t, (cuuint32_t)cpw, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, d.io_dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename IO, int G>
cudaError_t launch_tc_t(const TcParams &prm, cudaStream_t s) {
    using Cfg = TcCfg<IO, G>;
    auto k = scan_tc_kernel<IO, G>;
    static unsigned long long attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    k<<<(unsigned)sm_count(), Cfg::W * 32, Cfg::SMEM, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO, int G>
cudaError_t launch_tp_t(const TcParams &prm, cudaStream_t s) {
    using Cfg = TpCfg<IO, G>;
    auto k = scan_tp_kernel<IO, G>;
    static unsigned long long attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    k<<<(unsigned)sm_count(), Cfg::W * 32, Cfg::SMEM, s>>>(prm);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_tc(bool pipelined, int G, const TcParams &prm, cudaStream_t s) {
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

ssm_status_t run_scan_tc(const ssm_dims_t &d, const TcPlan &t, const void *u, const void *delta, const float *A,
                         const void *B, const void *C, const float *D, const void *z, const float *delta_bias,
                         int delta_softplus, void *y, float *last_state, char *ws, cudaStream_t s) {
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int cpw = t.cpw;
    if (!make_map(&prm.map_u, u, d, cpw, t.T) || !make_map(&prm.map_delta, delta, d, cpw, t.T) ||
        !make_map(&prm.map_z, z ? z : u, d, cpw, t.T) || !make_map(&prm.map_y, y, d, cpw, t.T) ||
        !make_map(&prm.map_y8, y, d, cpw, 8))
        return SSM_ERR_CUDA;
    prm.bc = reinterpret_cast<const float *>(ws + t.off_bc);
    prm.A = A; prm.D = D; prm.bias = delta_bias; prm.last_state = last_state;
    prm.ctrl = reinterpret_cast<int *>(ws);
    prm.carry = reinterpret_cast<float *>(ws + t.off_carry);
    prm.Bt = d.batch; prm.Dm = d.dim; prm.L = d.seqlen; prm.N = d.dstate; prm.Lp = t.Lp;
    prm.NG = t.NG; prm.groups_per_b = t.groups_per_b; prm.nseg = t.nseg; prm.seg_tiles = t.seg_tiles;
    prm.ntiles = t.ntiles; prm.has_z = z != nullptr; prm.softplus = delta_softplus ? 1 : 0;
    prm.cpw = t.cpw;
    prm.np = t.np;
    prm.spin_limit = 1u << 24;
    prm.force_timeout = 0;
    if (env_is("SSM_TEST_FORCE_TIMEOUT", "1")) { prm.force_timeout = 1; prm.spin_limit = 256; }
    if (cudaMemsetAsync(ws, 0, t.ctrl_bytes, s) != cudaSuccess) return SSM_ERR_CUDA;
    const int NP = t.np;
    float *bc = reinterpret_cast<float *>(ws + t.off_bc);
    const dim3 pg((unsigned)(t.Lp / 32), (unsigned)d.batch);
    const size_t psm = (size_t)2 * NP * 33 * 4;
    if (d.io_dtype == SSM_BF16)
        bc_prep_kernel<bf16><<<pg, 256, psm, s>>>(static_cast<const bf16 *>(B), static_cast<const bf16 *>(C), bc,
                                                  d.dstate, d.seqlen, t.Lp, NP);
    else
        bc_prep_kernel<float><<<pg, 256, psm, s>>>(static_cast<const float *>(B), static_cast<const float *>(C), bc,
                                                   d.dstate, d.seqlen, t.Lp, NP);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    const cudaError_t e = d.io_dtype == SSM_BF16 ? launch_tc<bf16>(t.pipelined, t.G, prm, s)
                                                 : launch_tc<float>(t.pipelined, t.G, prm, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
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

// ---- channel-pair sequential path (default for 16-byte aligned rows) ----------------------
#ifndef SSM_PAIR_T
#define SSM_PAIR_T 16
#endif
constexpr int kPairT = SSM_PAIR_T;   // timesteps per tile of the channel-pair kernel

struct PairPlan {
    bool use = false;
    int ks = 8, gp = 8;          // states per lane per channel, lanes per channel pair
    int nchunks = 1;
    int64_t chunk_len = 0;
    int cb_agg = 0, cb_full = 0;         // channel blocks per batch row, aggregate / full pass
    int np = 0;                  // padded states = ks * gp
    size_t smem_agg = 0, smem_full = 0;  // dynamic shared memory per CTA of each pass
};

// smallest power-of-two lane count gp with gp * ks >= N states
int pair_gp(int64_t N, int ks) {
    int gp = 1;
    while ((int64_t)gp * ks < N) gp *= 2;
    return gp;
}

template <typename IO, int KS, int GP, bool AGG, bool ZOH, bool CONV = false>
cudaError_t launch_pair_t(const SeqParams &prm, int grid_y, cudaStream_t s) {
    constexpr int W = pair_warps(KS, GP, AGG);
    using Cfg = PairCfg<IO, KS, GP, W, kPairT, CONV>;
    auto k = scan_pair_kernel<IO, KS, GP, W, kPairT, AGG, ZOH, CONV>;
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

template <typename IO, int KS, int GP>
cudaError_t launch_pair_g(const SeqParams &prm, bool agg, int grid_y, cudaStream_t s) {
    if (prm.conv_w != nullptr)   // conv front (Euler discretisation)
        return agg ? launch_pair_t<IO, KS, GP, true, false, true>(prm, grid_y, s)
                   : launch_pair_t<IO, KS, GP, false, false, true>(prm, grid_y, s);
    if (prm.zoh)
        return agg ? launch_pair_t<IO, KS, GP, true, true>(prm, grid_y, s)
                   : launch_pair_t<IO, KS, GP, false, true>(prm, grid_y, s);
    return agg ? launch_pair_t<IO, KS, GP, true, false>(prm, grid_y, s)
               : launch_pair_t<IO, KS, GP, false, false>(prm, grid_y, s);
}

#define SSM_PAIR_CASES(X) X(4, 1) X(4, 2) X(4, 4) X(8, 1) X(8, 2) X(8, 4) X(8, 8) X(8, 16) X(16, 4)

template <typename IO>
cudaError_t launch_pair(const PairPlan &pl, const SeqParams &prm, bool agg, int grid_y, cudaStream_t s) {
    switch (pl.ks * 100 + pl.gp) {
#define SSM_PAIR_LAUNCH(KS, GP) case KS * 100 + GP: return launch_pair_g<IO, KS, GP>(prm, agg, grid_y, s);
        SSM_PAIR_CASES(SSM_PAIR_LAUNCH)
#undef SSM_PAIR_LAUNCH
        default: return cudaErrorInvalidConfiguration;
    }
}

size_t pair_smem(ssm_dtype_t io, int ks, int gp, bool conv, bool agg) {
    switch (ks * 100 + gp) {
#define SSM_PAIR_SMEM(KS, GP) \
    case KS * 100 + GP: \
        if (agg) { \
            if (conv) return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, true), kPairT, true>::kSmem \
                                            : PairCfg<float, KS, GP, pair_warps(KS, GP, true), kPairT, true>::kSmem; \
            return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, true), kPairT>::kSmem \
                                  : PairCfg<float, KS, GP, pair_warps(KS, GP, true), kPairT>::kSmem; \
        } \
        if (conv) return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, false), kPairT, true>::kSmem \
                                        : PairCfg<float, KS, GP, pair_warps(KS, GP, false), kPairT, true>::kSmem; \
        return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, false), kPairT>::kSmem \
                              : PairCfg<float, KS, GP, pair_warps(KS, GP, false), kPairT>::kSmem;
        SSM_PAIR_CASES(SSM_PAIR_SMEM)
#undef SSM_PAIR_SMEM
        default: return 0;
    }
}

PairPlan plan_pair(const ssm_dims_t &d, bool conv = false) {
    PairPlan p;
    if (env_is("SSM_KERNEL", "seq") || env_is("SSM_KERNEL", "tc") || env_is("SSM_KERNEL", "tp")) return p;
    const size_t esz = io_size(d.io_dtype);
    if (((size_t)d.seqlen * esz) % 16 != 0 || d.dstate > 128) return p;   // rows move in 16-byte pieces
    const int64_t N = d.dstate, BD = d.batch * d.dim, sms = sm_count();
    // eight states per lane and channel, unless four give the GPU at least one warp per SM
    // sub-partition where eight do not (few channels with few states)
    p.ks = 8;
    p.gp = pair_gp(N, 8);
    if (N <= 16 && (BD * p.gp + 63) / 64 < 4 * sms) { p.ks = 4; p.gp = pair_gp(N, 4); }
    // sixteen states per lane for 33..64 states where a long sequence (>= 65536 steps) will
    // be chunked (eight states per lane give fewer than two warps per SM sub-partition): the y
    // reduction and the per-step dt loads are shared by twice the states, at 3 CTAs per SM
    // instead of 16 warps. Measured on B300 against eight states per lane: 1 x 1536 x 131072
    // x 64 4.77 vs 4.89 ms, 1 x 768 x 131072 2.41 vs 2.50, 1 x 2560 x 65536 3.95 vs 4.09,
    // 2 x 1536 x 65536 equal; shorter sequences lost (4 x 1536 x 16384 2.54 vs 2.37 ms,
    // 1 x 5120 x 32768 4.08 vs 4.04). Not with the conv front, whose per-channel window work
    // does not shrink with it (5.34 -> 5.63 ms on the first shape).
    if (!conv && N > 32 && N <= 64 && d.seqlen >= 65536 && BD * p.gp / 64 < 8 * sms) {
        p.ks = 16;
        p.gp = pair_gp(N, 16);
    }
    if (env_is("SSM_PAIR_KS", "4") && N <= 16) { p.ks = 4; p.gp = pair_gp(N, 4); }   // experiments, tests
    if (env_is("SSM_PAIR_KS", "8")) { p.ks = 8; p.gp = pair_gp(N, 8); }
    if (env_is("SSM_PAIR_KS", "16") && N > 32 && N <= 64) { p.ks = 16; p.gp = pair_gp(N, 16); }
    p.np = p.ks * p.gp;
    p.smem_agg = pair_smem(d.io_dtype, p.ks, p.gp, conv, true);
    p.smem_full = pair_smem(d.io_dtype, p.ks, p.gp, conv, false);
    if (p.smem_agg == 0 || p.smem_full == 0) return p;
    const int64_t wa = pair_warps(p.ks, p.gp, true), wf = pair_warps(p.ks, p.gp, false);
    p.cb_agg = (int)((d.dim + wa * 64 / p.gp - 1) / (wa * 64 / p.gp));
    p.cb_full = (int)((d.dim + wf * 64 / p.gp - 1) / (wf * 64 / p.gp));
    // CTAs of the full pass resident per SM: shared memory (228 KB, 1 KB reserved per CTA),
    // threads (2048) and the registers the launch bounds allow.
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(
        std::min<int64_t>((228 * 1024) / (int64_t)(p.smem_full + 1024), 2048 / (wf * 32)),
        pair_min_blocks((int)wf, p.ks, p.gp)));
    // The sequence is cut into chunks (aggregate pass + combine + full pass) when the channels
    // alone give fewer than two warps per SM sub-partition: the latency-bound recurrence gains
    // more from the extra warps than the aggregate pass (up to 1.9x the work) costs. The chunk
    // count is up to four waves of resident CTAs, as long as a chunk keeps 2048 steps: more
    // waves even out the tails of the waves (measured on B300 for 1 x 1536 x 131072 x 64);
    // chunks of a few hundred steps lose to their fixed costs.
    const int64_t slots = sms * per_sm, base = d.batch * p.cb_full;
    int64_t nc = 1;
    if (base * wf < 8 * sms) {
        const int64_t wave = std::max<int64_t>(1, slots / base);
        int64_t w = 4;
        while (w > 1 && d.seqlen < wave * w * 2048) --w;
        nc = wave * w;
    }
    if (const char *env = std::getenv("SSM_PAIR_CHUNKS")) nc = std::max(1, std::atoi(env));   // experiments
    nc = std::min<int64_t>(nc, std::max<int64_t>(1, d.seqlen / (4 * kPairT)));
    nc = std::min<int64_t>(nc, 4096);
    int64_t cl = (d.seqlen + nc - 1) / nc;
    cl = (cl + kPairT - 1) / kPairT * kPairT;
    p.chunk_len = std::max<int64_t>(cl, kPairT);
    p.nchunks = (int)((d.seqlen + p.chunk_len - 1) / p.chunk_len);
    p.use = true;
    return p;
}

size_t pair_workspace_bytes(const ssm_dims_t &d, const PairPlan &p) {
    if (!p.use || p.nchunks <= 1) return 0;
    const size_t BD = (size_t)(d.batch * d.dim);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t agg_h = (size_t)p.nchunks * BD * p.np * 4, agg_s = (size_t)p.nchunks * BD * 4;
    return up(agg_h) + up(agg_s) + up(agg_h);
}

ssm_status_t run_scan_pair(const ssm_dims_t &d, const PairPlan &pl, const void *u, const void *delta, const float *A,
                           const void *B, const void *C, const float *D, const void *z, const float *delta_bias,
                           int delta_softplus, void *y, float *last_state, void *workspace, size_t ws_bytes,
                           bool own_ws, cudaStream_t s, int zoh, const float *conv_w = nullptr,
                           const float *conv_b = nullptr, int conv_k = 0) {
    const size_t need = pair_workspace_bytes(d, pl);
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
    prm.npad = pl.np;
    prm.zoh = zoh ? 1 : 0;
    prm.conv_w = conv_w; prm.conv_b = conv_b; prm.conv_k = conv_k;
    prm.structured = g_structured_a.load();
    cudaError_t e = cudaSuccess;
    const bool bf = d.io_dtype == SSM_BF16;
    if (pl.nchunks > 1) {
        const size_t BD = (size_t)(d.batch * d.dim), np = (size_t)pl.np;
        auto up = [](size_t x) { return (x + 255) / 256 * 256; };
        char *w = static_cast<char *>(workspace);
        prm.agg_h = reinterpret_cast<float *>(w);
        prm.agg_s = reinterpret_cast<float *>(w + up((size_t)pl.nchunks * BD * np * 4));
        float *hin = reinterpret_cast<float *>(w + up((size_t)pl.nchunks * BD * np * 4) + up((size_t)pl.nchunks * BD * 4));
        prm.chan_blocks = pl.cb_agg;
        e = bf ? launch_pair<bf16>(pl, prm, true, pl.nchunks - 1, s) : launch_pair<float>(pl, prm, true, pl.nchunks - 1, s);
        if (e == cudaSuccess) {
            const int64_t total = (int64_t)BD * pl.np;
            chunk_combine_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
                A, prm.agg_h, prm.agg_s, hin, (int64_t)BD, d.dim, d.dstate, pl.np, pl.nchunks);
            e = cudaGetLastError();
        }
        prm.hin = hin;
    }
    prm.chan_blocks = pl.cb_full;
    if (e == cudaSuccess)
        e = bf ? launch_pair<bf16>(pl, prm, false, pl.nchunks, s) : launch_pair<float>(pl, prm, false, pl.nchunks, s);
    if (allocated) cudaFreeAsync(workspace, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status_t run_scan(const ssm_dims_t *dims, const void *u, const void *delta, const float *A,
                      const void *B, const void *C, const float *D, const void *z,
                      const float *delta_bias, int delta_softplus, void *y, float *last_state,
                      void *workspace, size_t ws_bytes, bool own_ws, cudaStream_t s, int zoh = 0) {
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
    const PairPlan pp = plan_pair(d);
    if (pp.use)
        return run_scan_pair(d, pp, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, workspace,
                             ws_bytes, own_ws, s, zoh);
    if (zoh) return SSM_ERR_UNSUPPORTED;   // the zero-order hold runs on the channel-pair kernel only
    const TcPlan tp = plan_tc(d);
    if (tp.use) {
        char *w = static_cast<char *>(workspace);
        bool alloc = false;
        if (w == nullptr || ws_bytes < tp.bytes) {
            if (!own_ws) return SSM_ERR_WORKSPACE;
            if (cudaMallocAsync(reinterpret_cast<void **>(&w), tp.bytes, s) != cudaSuccess) return SSM_ERR_CUDA;
            alloc = true;
        }
        const ssm_status_t r = run_scan_tc(d, tp, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w, s);
        if (alloc) cudaFreeAsync(w, s);
        return r;
    }
    const ScanPlan pl = plan_scan(d);
    if (!plan_supported(pl)) return SSM_ERR_UNSUPPORTED;
    const size_t need = seq_workspace_bytes(d, pl);
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

// ---- fixed scratch for ssm_selective_scan_fwd_noalloc -------------------------------------
// Callers that cannot allocate device memory at call time (their memory is held by another
// allocator's pool, their device has no stream-ordered pools, or they are plain C code with
// nothing to own a workspace) get the chunk carries, control words and prepared B/C from this
// array instead. One copy exists per device, in the module's own global memory; it is only
// ever passed to run_scan as a caller workspace, so no code path allocates on its behalf.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_SCRATCH_MAX_BYTES];

constexpr int kScratchDevices = 64;   // devices whose scratch address is cached
std::mutex g_scratch_mu;
void *g_scratch_addr[kScratchDevices] = {};

// Device address of the current device's scratch, resolved with cudaGetSymbolAddress at
// first use on that device (which may load the module: outside any stream capture).
ssm_status_t scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    const bool cached = dev >= 0 && dev < kScratchDevices;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cached && g_scratch_addr[dev] != nullptr) {
        *out = g_scratch_addr[dev];
        return SSM_OK;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();   // do not leave the error for the next launch check to find
        return SSM_ERR_CUDA;
    }
    if (cached) g_scratch_addr[dev] = p;
    *out = p;
    return SSM_OK;
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
    const PairPlan pp = plan_pair(*dims);
    if (pp.use) return pair_workspace_bytes(*dims, pp);
    const TcPlan tp = plan_tc(*dims);
    if (tp.use) return tp.bytes;
    return seq_workspace_bytes(*dims, plan_scan(*dims));
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

ssm_status_t ssm_selective_scan_fwd_noalloc(const ssm_dims_t *dims, const void *u, const void *delta,
                                            const float *A, const void *B, const void *C,
                                            const float *D, const void *z, const float *delta_bias,
                                            int delta_softplus, void *y, float *last_state,
                                            void *stream) {
    ssm_status_t st = scan_checks(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    const size_t need = ssm_selective_scan_workspace_bytes(dims);
    if (need > SSM_SCRATCH_MAX_BYTES) return SSM_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        st = scratch_address(&scratch);
        if (st != SSM_OK) return st;
    }
    // own_ws = false: run_scan may only use the scratch, never allocate a replacement
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                    scratch, need > 0 ? SSM_SCRATCH_MAX_BYTES : 0, false,
                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
ssm_status_t state_update_impl(const ssm_dims_t *dims, float *state, const void *x, const void *dt,
                               const float *A, const void *B, const void *C, const float *D,
                               const void *z, void *y, void *stream, int zoh) {
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
    DecodeParams p{state, x, dt, B, C, z, A, D, y, dims->batch, dims->dim, dims->dstate, zoh ? 1 : 0};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t N = dims->dstate, chans = dims->batch * dims->dim;
    const bool bf = dims->io_dtype == SSM_BF16;
    const int lpc = (int)(N / 4);
    // batch rows on grid.y and 16-byte B/C reads when B and C rows are 4-element aligned;
    // the row's channels must fit a 32-bit thread index and grid.y (65535 rows)
    const bool wide = aligned_to(B, 4 * esz) && aligned_to(C, 4 * esz) && dims->batch <= 65535 &&
                      dims->dim * lpc < (int64_t)1 << 30 && !env_is("SSM_DEC_OLD", "1");
    if (wide && N % 4 == 0 && lpc >= 1 && lpc <= 32 && (32 % lpc) == 0) {
        const dim3 grid((unsigned)((dims->dim * lpc + 255) / 256), (unsigned)dims->batch);
#define SSM_DECW(L)                                                                                    \
    case L:                                                                                            \
        if (zoh) bf ? decode_wide_kernel<bf16, L, true><<<grid, 256, 0, s>>>(p) : decode_wide_kernel<float, L, true><<<grid, 256, 0, s>>>(p); \
        else bf ? decode_wide_kernel<bf16, L><<<grid, 256, 0, s>>>(p) : decode_wide_kernel<float, L><<<grid, 256, 0, s>>>(p);                \
        break;
        switch (lpc) { SSM_DECW(1) SSM_DECW(2) SSM_DECW(4) SSM_DECW(8) SSM_DECW(16) SSM_DECW(32) default: return SSM_ERR_UNSUPPORTED; }
#undef SSM_DECW
    } else if (N % 4 == 0 && lpc >= 1 && lpc <= 32 && (32 % lpc) == 0) {
        const int64_t threads = chans * lpc;
        const unsigned grid = (unsigned)((threads + 255) / 256);
#define SSM_DEC(L)                                                                                     \
    case L:                                                                                            \
        if (zoh) bf ? decode_vec_kernel<bf16, L, true><<<grid, 256, 0, s>>>(p) : decode_vec_kernel<float, L, true><<<grid, 256, 0, s>>>(p); \
        else bf ? decode_vec_kernel<bf16, L><<<grid, 256, 0, s>>>(p) : decode_vec_kernel<float, L><<<grid, 256, 0, s>>>(p);                \
        break;
        switch (lpc) { SSM_DEC(1) SSM_DEC(2) SSM_DEC(4) SSM_DEC(8) SSM_DEC(16) SSM_DEC(32) default: return SSM_ERR_UNSUPPORTED; }
#undef SSM_DEC
    } else {
        const unsigned grid = (unsigned)((chans + 255) / 256);
        if (zoh) {
            if (bf) decode_scalar_kernel<bf16, true><<<grid, 256, 0, s>>>(p);
            else decode_scalar_kernel<float, true><<<grid, 256, 0, s>>>(p);
        } else {
            if (bf) decode_scalar_kernel<bf16><<<grid, 256, 0, s>>>(p);
            else decode_scalar_kernel<float><<<grid, 256, 0, s>>>(p);
        }
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
}  // namespace

extern "C" {

ssm_status_t ssm_state_update(const ssm_dims_t *dims, float *state, const void *x, const void *dt,
                              const float *A, const void *B, const void *C, const float *D,
                              const void *z, void *y, void *stream) {
    return state_update_impl(dims, state, x, dt, A, B, C, D, z, y, stream, 0);
}

ssm_status_t ssm_state_update_disc(const ssm_dims_t *dims, float *state, const void *x, const void *dt,
                                   const float *A, const void *B, const void *C, const float *D,
                                   const void *z, int discretization, void *y, void *stream) {
    if (discretization != SSM_DISC_EULER && discretization != SSM_DISC_ZOH) return SSM_ERR_UNSUPPORTED;
    return state_update_impl(dims, state, x, dt, A, B, C, D, z, y, stream, discretization == SSM_DISC_ZOH);
}

ssm_status_t ssm_selective_scan_fwd_disc(const ssm_dims_t *dims, const void *u, const void *delta,
                                         const float *A, const void *B, const void *C, const float *D,
                                         const void *z, const float *delta_bias, int delta_softplus,
                                         int discretization, void *y, float *last_state, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    ssm_status_t st = scan_checks(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    if (discretization != SSM_DISC_EULER && discretization != SSM_DISC_ZOH) return SSM_ERR_UNSUPPORTED;
    if (workspace != nullptr && !aligned16(workspace)) return SSM_ERR_ALIGN;
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, workspace,
                    workspace_bytes, workspace == nullptr, static_cast<cudaStream_t>(stream),
                    discretization == SSM_DISC_ZOH);
}

ssm_status_t ssm_conv_selective_scan_fwd(const ssm_dims_t *dims, const void *x, const float *conv_w,
                                         const float *conv_b, int conv_width, const void *delta, const float *A,
                                         const void *B, const void *C, const float *D, const void *z,
                                         const float *delta_bias, int delta_softplus, void *y, float *last_state,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    ssm_status_t st = scan_checks(dims, x, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    if (conv_width < 1 || conv_width > 4) return SSM_ERR_UNSUPPORTED;
    if (conv_b != nullptr && !aligned_to(conv_b, 4)) return SSM_ERR_ALIGN;
    if (workspace != nullptr && !aligned16(workspace)) return SSM_ERR_ALIGN;
    const ssm_dims_t d = *dims;
    if (d.batch == 0 || d.dim == 0 || d.seqlen == 0)
        return run_scan(dims, x, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, workspace,
                        workspace_bytes, workspace == nullptr, static_cast<cudaStream_t>(stream));
    if (conv_w == nullptr) return SSM_ERR_NULL;
    if (!aligned_to(conv_w, 4)) return SSM_ERR_ALIGN;
    const PairPlan pp = plan_pair(d, true);
    if (!pp.use) return SSM_ERR_UNSUPPORTED;   // the conv front runs on the channel-pair kernel only
    return run_scan_pair(d, pp, x, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, workspace,
                         workspace_bytes, workspace == nullptr, static_cast<cudaStream_t>(stream), 0, conv_w, conv_b,
                         conv_width);
}

size_t ssm_conv_selective_scan_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    return pair_workspace_bytes(*dims, plan_pair(*dims, true));
}

}  // extern "C"

namespace {
// backward lane split: Q <= 4 states per lane, G lanes per channel (a power of two, <= 32)
// Q states per thread, G lanes per channel (G * Q >= N). Two states per thread up to 64
// states: the 16-step state history then fits in registers with 4 CTAs per SM (measured on
// 8 x 1536 x 2048 x 16: 3.86 ms at four states per thread, 3.23 ms at two).
void bwd_split(int64_t N, int *G, int *Q) {
    *Q = N <= 1 ? 1 : (N <= 64 ? 2 : 4);
    int g = 1;
    while (g < 32 && (int64_t)g * *Q < N) g *= 2;
    *G = g;
}
}  // namespace

extern "C" {

size_t ssm_selective_scan_bwd_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    int G, Q;
    bwd_split(dims->dstate, &G, &Q);
    const int64_t nseg = (dims->seqlen + kBwdS - 1) / kBwdS;
    return (size_t)(dims->batch * dims->dim) * (size_t)nseg * (size_t)(G * Q) * sizeof(float);
}

ssm_status_t ssm_selective_scan_bwd(const ssm_dims_t *dims, const void *u, const void *delta, const float *A,
                                    const void *B, const void *C, const float *D, const void *z,
                                    const float *delta_bias, int delta_softplus, const void *dy,
                                    const float *dlast_state, float *du, float *ddelta, float *dA, float *dB,
                                    float *dC, float *dD, float *dz, float *ddelta_bias, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    ssm_status_t st = check_dims(dims, true);
    if (st != SSM_OK) return st;
    const ssm_dims_t d = *dims;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d.batch == 0 || d.dim == 0) return SSM_OK;
    if (!A || !dA) return SSM_ERR_NULL;
    const bool empty = d.seqlen == 0;
    if (!empty && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)) return SSM_ERR_NULL;
    const size_t esz = io_size(d.io_dtype);
    const void *io_ptrs[] = {u, delta, B, C, z, dy};
    for (const void *q : io_ptrs)
        if (q != nullptr && !aligned_to(q, esz)) return SSM_ERR_ALIGN;
    const void *f_ptrs[] = {A, D, delta_bias, dlast_state, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias};
    for (const void *q : f_ptrs)
        if (q != nullptr && !aligned_to(q, 4)) return SSM_ERR_ALIGN;
    if (d.batch > 65535) return SSM_ERR_UNSUPPORTED;
    // gradients summed over the sequence, the batch or the channels start at zero
    const size_t BD = (size_t)(d.batch * d.dim), NL = (size_t)(d.dstate * d.seqlen);
    if (cudaMemsetAsync(dA, 0, (size_t)(d.dim * d.dstate) * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    if (dD && cudaMemsetAsync(dD, 0, (size_t)d.dim * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)d.dim * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    if (empty) return SSM_OK;
    if (cudaMemsetAsync(dB, 0, (size_t)d.batch * NL * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    if (cudaMemsetAsync(dC, 0, (size_t)d.batch * NL * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    if (dz && !z && cudaMemsetAsync(dz, 0, BD * (size_t)d.seqlen * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    const size_t need = ssm_selective_scan_bwd_workspace_bytes(dims);
    bool allocated = false;
    if (workspace == nullptr) {
        if (cudaMallocAsync(&workspace, need, s) != cudaSuccess) return SSM_ERR_CUDA;
        allocated = true;
    } else if (workspace_bytes < need) {
        return SSM_ERR_WORKSPACE;
    } else if (!aligned16(workspace)) {
        return SSM_ERR_ALIGN;
    }
    BwdParams p{u, delta, z, B, C, dy, A, D, delta_bias, dlast_state, du, ddelta, dA, dB, dC, dD,
                z ? dz : nullptr, ddelta_bias, static_cast<float *>(workspace), d.batch, d.dim, d.seqlen,
                d.dstate, delta_softplus ? 1 : 0, (int)((d.seqlen + kBwdS - 1) / kBwdS)};
    int G, Q;
    bwd_split(d.dstate, &G, &Q);
    const dim3 grid((unsigned)((d.dim + kBwdThreads / G - 1) / (kBwdThreads / G)), (unsigned)d.batch);
    const bool bf = d.io_dtype == SSM_BF16;
#define SSM_BWD(GG, QQ)                                                                                \
    case GG * 10 + QQ: {                                                                               \
        constexpr size_t tb = bwd_tile_bytes<GG, QQ>(), sm = tb + bwd_smem_bytes(GG, QQ);             \
        if (bf) {                                                                                      \
            cudaFuncSetAttribute(scan_bwd_kernel<bf16, GG, QQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm); \
            scan_bwd_ckpt_kernel<bf16, GG, QQ><<<grid, kBwdThreads, tb, s>>>(p);                      \
            scan_bwd_kernel<bf16, GG, QQ><<<grid, kBwdThreads, sm, s>>>(p);                           \
        } else {                                                                                       \
            cudaFuncSetAttribute(scan_bwd_kernel<float, GG, QQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm); \
            scan_bwd_ckpt_kernel<float, GG, QQ><<<grid, kBwdThreads, tb, s>>>(p);                     \
            scan_bwd_kernel<float, GG, QQ><<<grid, kBwdThreads, sm, s>>>(p);                          \
        }                                                                                              \
        break;                                                                                         \
    }
    switch (G * 10 + Q) {
        SSM_BWD(1, 1) SSM_BWD(1, 2) SSM_BWD(2, 2) SSM_BWD(4, 2) SSM_BWD(8, 2) SSM_BWD(16, 2)
        SSM_BWD(32, 2) SSM_BWD(32, 4)
        default:
            if (allocated) cudaFreeAsync(workspace, s);
            return SSM_ERR_UNSUPPORTED;
    }
#undef SSM_BWD
    const cudaError_t e = cudaGetLastError();
    if (allocated) cudaFreeAsync(workspace, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
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
    if (cudaMemcpyFromSymbol(&v, ssm::g_ssm_status, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(ssm::g_ssm_status, &zero, sizeof(int)) != cudaSuccess) return SSM_ERR_CUDA;
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

int ssm_set_structured_a(int enable) { return g_structured_a.exchange(enable ? 1 : 0); }

int ssm_version(void) { return (1 << 16) | 0; }

}  // extern "C"
