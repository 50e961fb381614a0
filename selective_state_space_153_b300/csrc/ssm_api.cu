// Host side of the C ABI declared in include/ssm_scan.h: argument checks, launch planning,
// kernel dispatch (launch.h; the kernels live in the k_*.cu translation units), workspace
// handling and the host-buffer pipeline.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "ssm_scan.h"
#include "launch.h"
#include "scan_tp.cuh"

namespace ssm {
// the device status word that bounded waits set (declared in ptx.cuh)
__device__ int g_ssm_status = 0;
}  // namespace ssm

namespace {

using bf16 = __nv_bfloat16;
using namespace ssm;

// structured-A detection in the forward scans (ssm_set_structured_a): 1 = on, 0 = off
std::atomic<int> g_structured_a{0};

// ---- launch-plan override (ssm_set_plan_override): process-wide, all zero = the planner ----
std::mutex g_override_mu;
ssm_plan_override_t g_override{};

ssm_plan_override_t plan_override() {
    std::lock_guard<std::mutex> lock(g_override_mu);
    return g_override;
}

// ---- the CUDA error behind the last SSM_ERR_CUDA of this thread (ssm_last_cuda_error) -----
thread_local int t_last_cuda_error = 0;

// SSM_OK for cudaSuccess; otherwise records `e` for ssm_last_cuda_error, clears the runtime's
// last-error slot (so that the next launch check does not find it) and returns SSM_ERR_CUDA.
ssm_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SSM_OK;
    t_last_cuda_error = (int)e;
    cudaGetLastError();
    return SSM_ERR_CUDA;
}

// ---- registered default workspace (ssm_set_workspace), one per device --------------------
constexpr int kMaxDevices = 64;
std::mutex g_ws_mu;
void *g_ws_ptr[kMaxDevices] = {};
size_t g_ws_bytes[kMaxDevices] = {};

// The current device's registered workspace, or {nullptr, 0}.
void registered_workspace(void **ptr, size_t *bytes) {
    *ptr = nullptr;
    *bytes = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return;
    }
    std::lock_guard<std::mutex> lock(g_ws_mu);
    *ptr = g_ws_ptr[dev];
    *bytes = g_ws_bytes[dev];
}

// How an entry point without a workspace argument (or given NULL) gets its workspace:
// the registered one if there is one (then it must be large enough: no allocation), else a
// stream-ordered allocation by the library.
struct WsChoice {
    void *ptr;
    size_t bytes;
    bool may_alloc;
};
WsChoice default_workspace() {
    WsChoice c{nullptr, 0, true};
    registered_workspace(&c.ptr, &c.bytes);
    if (c.ptr != nullptr) c.may_alloc = false;
    return c;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t io_size(ssm_dtype_t t) { return t == SSM_BF16 ? 2 : 4; }
size_t up256(size_t x) { return (x + 255) / 256 * 256; }

ssm_status_t check_dims(const ssm_dims_t *dims, bool need_L) {
    if (dims == nullptr) return SSM_ERR_NULL;
    if (dims->batch < 0 || dims->dim < 0 || dims->seqlen < 0 || dims->dstate < 1) return SSM_ERR_SHAPE;
    if (dims->io_dtype != SSM_F32 && dims->io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (dims->dstate > SSM_MAX_DSTATE) return SSM_ERR_UNSUPPORTED;
    // overflow guard: every tensor must have < 2^62 bytes
    const double lim = 4.0e18;
    const double Lf = (double)(need_L ? std::max<int64_t>(dims->seqlen, 1) : 1);
    if ((double)dims->batch * dims->dim * Lf * 4.0 > lim || (double)dims->batch * dims->dstate * Lf * 4.0 > lim ||
        (double)dims->batch * dims->dim * dims->dstate * 4.0 > lim)
        return SSM_ERR_SHAPE;
    return SSM_OK;
}

int sm_count() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    else cudaGetLastError();   // no device (planning on a host without one): the B300's count
    return n;
}

// ---- sequential-lane kernel plan (rows that are not 16-byte multiples) ---------------------
struct ScanPlan {
    int nper, g;   // states per lane, lanes per channel
    int nchunks;
    int64_t chunk_len;
};

ScanPlan plan_scan(const ssm_dims_t &d, const ssm_plan_override_t &ov) {
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
    if (warps < sms * 8 && d.seqlen >= 4 * kSeqTile) {
        int64_t nc = (want + warps - 1) / warps;
        nc = std::min<int64_t>(nc, d.seqlen / (4 * kSeqTile));
        nc = std::max<int64_t>(std::min<int64_t>(nc, 4096), 1);
        p.nchunks = (int)nc;
    }
    if (ov.seq_states_per_lane > 0 && ov.seq_lanes_per_channel > 0) {
        p.nper = ov.seq_states_per_lane;
        p.g = ov.seq_lanes_per_channel;
    }
    if (ov.chunks > 0) p.nchunks = std::min(ov.chunks, 4096);
    if (p.nper * p.g < N) p.nper = (int)((N + p.g - 1) / p.g + 3) / 4 * 4;
    int64_t cl = (d.seqlen + p.nchunks - 1) / p.nchunks;
    cl = (cl + kSeqTile - 1) / kSeqTile * kSeqTile;
    p.chunk_len = std::max<int64_t>(cl, kSeqTile);
    p.nchunks = (int)((d.seqlen + p.chunk_len - 1) / p.chunk_len);
    if (p.nchunks < 1) p.nchunks = 1;
    return p;
}

size_t seq_workspace_bytes(const ssm_dims_t &d, const ScanPlan &p) {
    if (p.nchunks <= 1) return 0;
    const size_t BD = (size_t)(d.batch * d.dim), npad = (size_t)(p.nper * p.g);
    const size_t agg_h = (size_t)p.nchunks * BD * npad * 4, agg_s = (size_t)p.nchunks * BD * 4;
    return up256(agg_h) + up256(agg_s) + up256(agg_h);
}

// ---- persistent time-split kernels (selected only through the plan override) --------------
struct TcPlan {
    bool use = false;
    bool pipelined = true;   // scan_tp_kernel (dstate <= 64) or scan_tc_kernel
    int T = kTpT;
    int cpw = 8, np = 64;    // channels per group, padded states
    int G = 4, NG = 0, groups_per_b = 0, nseg = 1, seg_tiles = 1, ntiles = 0;
    int64_t Lp = 0;
    size_t off_carry = 0, off_bc = 0, bytes = 0, ctrl_bytes = 0;
};

TcPlan plan_tc(const ssm_dims_t &d, const ssm_plan_override_t &ov) {
    TcPlan t;
    if (ov.kernel != SSM_KERNEL_TC && ov.kernel != SSM_KERNEL_TP) return t;
    const size_t esz = io_size(d.io_dtype);
    if (((size_t)d.seqlen * esz) % 16 != 0) return t;                       // TMA row strides
    if (d.seqlen >= (int64_t)1 << 30 || d.dim >= (int64_t)1 << 30 || d.batch >= (int64_t)1 << 30) return t;
    const int64_t N = d.dstate;
    // pipelined kernel: GP = 8-state groups per channel pair (N <= 64), 64/GP channels per group;
    // otherwise the barrier-phased kernel: G = 16-state groups per channel, 32/G channels
    // (fp32 with N <= 8 would need 64-channel groups whose tiles do not fit shared memory)
    t.pipelined = ov.kernel == SSM_KERNEL_TP && N <= 64 && !(N <= 8 && d.io_dtype == SSM_F32);
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
    if (ng >= (int64_t)1 << 24) return t;
    t.NG = (int)ng;
    int64_t nseg = (16 * sms + ng - 1) / ng;
    nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, t.ntiles));
    t.seg_tiles = (int)((t.ntiles + nseg - 1) / nseg);
    t.nseg = (t.ntiles + t.seg_tiles - 1) / t.seg_tiles;
    t.Lp = (int64_t)t.ntiles * t.T;
    t.ctrl_bytes = up256((size_t)(1 + t.NG) * 4);
    t.off_carry = t.ctrl_bytes;
    t.off_bc = t.off_carry + up256((size_t)t.NG * 2 * 512 * 4);
    t.bytes = t.off_bc + up256((size_t)d.batch * t.Lp * 2 * t.np * 4);
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

ssm_status_t run_scan_tc(const ssm_dims_t &d, const TcPlan &t, const ssm_plan_override_t &ov, const void *u,
                         const void *delta, const float *A, const void *B, const void *C, const float *D,
                         const void *z, const float *delta_bias, int delta_softplus, void *y, float *last_state,
                         char *ws, cudaStream_t s) {
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int cpw = t.cpw;
    if (!make_map(&prm.map_u, u, d, cpw, t.T) || !make_map(&prm.map_delta, delta, d, cpw, t.T) ||
        !make_map(&prm.map_z, z ? z : u, d, cpw, t.T) || !make_map(&prm.map_y, y, d, cpw, t.T) ||
        !make_map(&prm.map_y8, y, d, cpw, 8))
        return cuda_status(cudaErrorInvalidValue);
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
    if (ov.force_timeout) { prm.force_timeout = 1; prm.spin_limit = 256; }
    cudaError_t e = cudaMemsetAsync(ws, 0, t.ctrl_bytes, s);
    if (e == cudaSuccess)
        e = launch_bc_prep(d.io_dtype, B, C, reinterpret_cast<float *>(ws + t.off_bc), d.dstate, d.seqlen, t.Lp, t.np,
                           d.batch, s);
    if (e == cudaSuccess) e = launch_tc(d.io_dtype, t.pipelined, t.G, prm, s);
    return cuda_status(e);
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

// restrided = the rows will be copied to a padded stride first (rows that are not 16-byte
// multiples), so their own length need not be one
PairPlan plan_pair(const ssm_dims_t &d, const ssm_plan_override_t &ov, bool conv = false, bool restrided = false) {
    PairPlan p;
    if (ov.kernel == SSM_KERNEL_SEQ || ov.kernel == SSM_KERNEL_TC || ov.kernel == SSM_KERNEL_TP) return p;
    const size_t esz = io_size(d.io_dtype);
    if (d.dstate > 128) return p;
    if (((size_t)d.seqlen * esz) % 16 != 0) {   // rows move in 16-byte pieces
        // a forced sequential-lane split keeps ragged rows on that kernel
        if (!restrided || ov.seq_states_per_lane != 0 || ov.seq_lanes_per_channel != 0) return p;
    }
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
    if (ov.pair_states_per_lane == 4 && N <= 16) { p.ks = 4; p.gp = pair_gp(N, 4); }
    if (ov.pair_states_per_lane == 8) { p.ks = 8; p.gp = pair_gp(N, 8); }
    if (ov.pair_states_per_lane == 16 && N > 32 && N <= 64) { p.ks = 16; p.gp = pair_gp(N, 16); }
    p.np = p.ks * p.gp;
    p.smem_agg = pair_smem(d.io_dtype, p.ks, p.gp, conv, true);
    p.smem_full = pair_smem(d.io_dtype, p.ks, p.gp, conv, false);
    if (p.smem_agg == 0 || p.smem_full == 0) return p;
    const int64_t wa = pair_warps_of(p.ks, p.gp, true), wf = pair_warps_of(p.ks, p.gp, false);
    p.cb_agg = (int)((d.dim + wa * 64 / p.gp - 1) / (wa * 64 / p.gp));
    p.cb_full = (int)((d.dim + wf * 64 / p.gp - 1) / (wf * 64 / p.gp));
    // CTAs of the full pass resident per SM: shared memory (228 KB, 1 KB reserved per CTA),
    // threads (2048) and the registers the launch bounds allow.
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(
        std::min<int64_t>((228 * 1024) / (int64_t)(p.smem_full + 1024), 2048 / (wf * 32)),
        pair_min_blocks_of(p.ks, p.gp, false)));
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
    if (ov.chunks > 0) nc = ov.chunks;
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
    const size_t agg_h = (size_t)p.nchunks * BD * p.np * 4, agg_s = (size_t)p.nchunks * BD * 4;
    return up256(agg_h) + up256(agg_s) + up256(agg_h);
}

// A workspace of at least `need` bytes for one call: the caller's, or a stream-ordered
// allocation when allowed. `allocated` tells the caller to free it stream-ordered.
ssm_status_t acquire_workspace(void **ws, size_t ws_bytes, size_t need, bool may_alloc, cudaStream_t s,
                               bool *allocated) {
    *allocated = false;
    if (need == 0) return SSM_OK;
    if (*ws == nullptr || ws_bytes < need) {
        if (!may_alloc) return SSM_ERR_WORKSPACE;
        if (const cudaError_t e = cudaMallocAsync(ws, need, s); e != cudaSuccess) return cuda_status(e);
        *allocated = true;
    } else if (!aligned16(*ws)) {
        return SSM_ERR_ALIGN;
    }
    return SSM_OK;
}

ssm_status_t run_scan_pair(const ssm_dims_t &d, const PairPlan &pl, const void *u, const void *delta, const float *A,
                           const void *B, const void *C, const float *D, const void *z, const float *delta_bias,
                           int delta_softplus, void *y, float *last_state, void *workspace, size_t ws_bytes,
                           bool may_alloc, cudaStream_t s, int zoh, const float *conv_w = nullptr,
                           const float *conv_b = nullptr, int conv_k = 0, int64_t ld = 0) {
    bool allocated = false;
    ssm_status_t st = acquire_workspace(&workspace, ws_bytes, pair_workspace_bytes(d, pl), may_alloc, s, &allocated);
    if (st != SSM_OK) return st;
    SeqParams prm{};
    prm.u = u; prm.delta = delta; prm.z = z; prm.B = B; prm.C = C;
    prm.A = A; prm.D = D; prm.bias = delta_bias; prm.y = y; prm.last_state = last_state;
    prm.Bt = d.batch; prm.Dm = d.dim; prm.L = d.seqlen; prm.N = d.dstate;
    prm.ld = ld > 0 ? ld : d.seqlen;
    prm.softplus = delta_softplus ? 1 : 0;
    prm.chunk_len = pl.chunk_len; prm.nchunks = pl.nchunks;
    prm.npad = pl.np;
    prm.zoh = zoh ? 1 : 0;
    prm.conv_w = conv_w; prm.conv_b = conv_b; prm.conv_k = conv_k;
    prm.structured = g_structured_a.load();
    prm.check_probe = plan_override().check_probe;
    const int variant = conv_w != nullptr ? kPairConv : (zoh ? kPairZoh : kPairEuler);
    cudaError_t e = cudaSuccess;
    if (pl.nchunks > 1) {
        const size_t BD = (size_t)(d.batch * d.dim), np = (size_t)pl.np;
        char *w = static_cast<char *>(workspace);
        prm.agg_h = reinterpret_cast<float *>(w);
        prm.agg_s = reinterpret_cast<float *>(w + up256((size_t)pl.nchunks * BD * np * 4));
        float *hin = reinterpret_cast<float *>(w + up256((size_t)pl.nchunks * BD * np * 4) +
                                               up256((size_t)pl.nchunks * BD * 4));
        prm.chan_blocks = pl.cb_agg;
        e = launch_pair(d.io_dtype, variant, pl.ks, pl.gp, true, prm, pl.nchunks - 1, s);
        if (e == cudaSuccess)
            e = launch_chunk_combine(A, prm.agg_h, prm.agg_s, hin, (int64_t)BD, d.dim, d.dstate, pl.np, pl.nchunks, s);
        prm.hin = hin;
    }
    prm.chan_blocks = pl.cb_full;
    if (e == cudaSuccess) e = launch_pair(d.io_dtype, variant, pl.ks, pl.gp, false, prm, pl.nchunks, s);
    if (allocated) cudaFreeAsync(workspace, s);
    return cuda_status(e);
}

// Rows whose byte length is not a multiple of 16: the channel-pair kernel runs on copies of
// u, delta, z, B, C at the padded stride ld (L rounded up to 16 bytes) in the workspace, and
// its y comes back through a padded buffer. The workspace holds [u | delta | z | B | C | y |
// chunk carries]; the z slot is kept even without z, so the size depends on the shape only.
struct RaggedPlan {
    int64_t ld = 0;
    size_t off_dl = 0, off_z = 0, off_b = 0, off_c = 0, off_y = 0, off_carry = 0, bytes = 0;
};
RaggedPlan plan_ragged(const ssm_dims_t &d, const PairPlan &pp) {
    RaggedPlan r;
    const size_t esz = io_size(d.io_dtype), epp = 16 / esz;
    r.ld = (int64_t)(((size_t)d.seqlen + epp - 1) / epp * epp);
    const size_t io = up256((size_t)(d.batch * d.dim) * (size_t)r.ld * esz);
    const size_t bc = up256((size_t)(d.batch * d.dstate) * (size_t)r.ld * esz);
    r.off_dl = io;
    r.off_z = 2 * io;
    r.off_b = 3 * io;
    r.off_c = r.off_b + bc;
    r.off_y = r.off_c + bc;
    r.off_carry = r.off_y + io;
    r.bytes = r.off_carry + pair_workspace_bytes(d, pp);
    return r;
}

ssm_status_t run_scan_ragged(const ssm_dims_t &d, const PairPlan &pp, const RaggedPlan &rg, const void *u,
                             const void *delta, const float *A, const void *B, const void *C, const float *D,
                             const void *z, const float *delta_bias, int delta_softplus, void *y, float *last_state,
                             void *workspace, size_t ws_bytes, bool may_alloc, cudaStream_t s, int zoh,
                             const float *conv_w = nullptr, const float *conv_b = nullptr, int conv_k = 0) {
    bool allocated = false;
    ssm_status_t st = acquire_workspace(&workspace, ws_bytes, rg.bytes, may_alloc, s, &allocated);
    if (st != SSM_OK) return st;
    char *w = static_cast<char *>(workspace);
    const int64_t BD = d.batch * d.dim, BN = d.batch * d.dstate, L = d.seqlen;
    cudaError_t e = launch_restride(d.io_dtype, u, L, w, rg.ld, BD, L, s);
    if (e == cudaSuccess) e = launch_restride(d.io_dtype, delta, L, w + rg.off_dl, rg.ld, BD, L, s);
    if (e == cudaSuccess && z) e = launch_restride(d.io_dtype, z, L, w + rg.off_z, rg.ld, BD, L, s);
    if (e == cudaSuccess) e = launch_restride(d.io_dtype, B, L, w + rg.off_b, rg.ld, BN, L, s);
    if (e == cudaSuccess) e = launch_restride(d.io_dtype, C, L, w + rg.off_c, rg.ld, BN, L, s);
    if (e == cudaSuccess) {
        st = run_scan_pair(d, pp, w, w + rg.off_dl, A, w + rg.off_b, w + rg.off_c, D, z ? w + rg.off_z : nullptr,
                           delta_bias, delta_softplus, w + rg.off_y, last_state, w + rg.off_carry,
                           rg.bytes - rg.off_carry, false, s, zoh, conv_w, conv_b, conv_k, rg.ld);
        if (st == SSM_OK) e = launch_restride(d.io_dtype, w + rg.off_y, rg.ld, y, L, BD, L, s);
    }
    if (allocated) cudaFreeAsync(workspace, s);
    if (st != SSM_OK) return st;
    return cuda_status(e);
}

// The restrided channel-pair plan for `d` when its rows are not 16-byte multiples and the
// workspace allows it (the library may allocate, or the given workspace is large enough).
bool use_ragged(const ssm_dims_t &d, const ssm_plan_override_t &ov, bool conv, void *workspace, size_t ws_bytes,
                bool may_alloc, PairPlan *pp, RaggedPlan *rg) {
    if (((size_t)d.seqlen * io_size(d.io_dtype)) % 16 == 0) return false;
    *pp = plan_pair(d, ov, conv, true);
    if (!pp->use) return false;
    *rg = plan_ragged(d, *pp);
    return may_alloc || (workspace != nullptr && ws_bytes >= rg->bytes);
}

// Workspace bytes the scan of `d` needs under the current plan (0 if none).
// small = the plan without the restrided rows (what a workspace too small for them gets).
size_t scan_workspace_bytes(const ssm_dims_t &d, bool small = false) {
    if (d.batch == 0 || d.dim == 0 || d.seqlen == 0) return 0;
    const ssm_plan_override_t ov = plan_override();
    const PairPlan pp = plan_pair(d, ov);
    if (pp.use) return pair_workspace_bytes(d, pp);
    if (!small) {
        const PairPlan pr = plan_pair(d, ov, false, true);
        if (pr.use) return plan_ragged(d, pr).bytes;
    }
    const TcPlan tp = plan_tc(d, ov);
    if (tp.use) return tp.bytes;
    return seq_workspace_bytes(d, plan_scan(d, ov));
}

ssm_status_t run_scan(const ssm_dims_t *dims, const void *u, const void *delta, const float *A,
                      const void *B, const void *C, const float *D, const void *z,
                      const float *delta_bias, int delta_softplus, void *y, float *last_state,
                      void *workspace, size_t ws_bytes, bool may_alloc, cudaStream_t s, int zoh = 0) {
    const ssm_dims_t d = *dims;
    if (d.batch == 0 || d.dim == 0) return SSM_OK;
    if (d.seqlen == 0) {
        if (last_state) return cuda_status(launch_zero_f32(last_state, d.batch * d.dim * d.dstate, s));
        return SSM_OK;
    }
    const ssm_plan_override_t ov = plan_override();
    const PairPlan pp = plan_pair(d, ov);
    if (pp.use)
        return run_scan_pair(d, pp, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, workspace,
                             ws_bytes, may_alloc, s, zoh);
    PairPlan pr;
    RaggedPlan rg;
    if (use_ragged(d, ov, false, workspace, ws_bytes, may_alloc, &pr, &rg))
        return run_scan_ragged(d, pr, rg, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                               workspace, ws_bytes, may_alloc, s, zoh);
    if (zoh) return SSM_ERR_UNSUPPORTED;   // the zero-order hold runs on the channel-pair kernel only
    const TcPlan tp = plan_tc(d, ov);
    if (tp.use) {
        bool alloc = false;
        ssm_status_t st = acquire_workspace(&workspace, ws_bytes, tp.bytes, may_alloc, s, &alloc);
        if (st != SSM_OK) return st;
        st = run_scan_tc(d, tp, ov, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                         static_cast<char *>(workspace), s);
        if (alloc) cudaFreeAsync(workspace, s);
        return st;
    }
    const ScanPlan pl = plan_scan(d, ov);
    if (!seq_plan_supported(pl.nper, pl.g)) return SSM_ERR_UNSUPPORTED;
    bool allocated = false;
    ssm_status_t st = acquire_workspace(&workspace, ws_bytes, seq_workspace_bytes(d, pl), may_alloc, s, &allocated);
    if (st != SSM_OK) return st;
    SeqParams prm{};
    prm.u = u; prm.delta = delta; prm.z = z; prm.B = B; prm.C = C;
    prm.A = A; prm.D = D; prm.bias = delta_bias; prm.y = y; prm.last_state = last_state;
    prm.Bt = d.batch; prm.Dm = d.dim; prm.L = d.seqlen; prm.N = d.dstate; prm.ld = d.seqlen;
    prm.softplus = delta_softplus ? 1 : 0;
    prm.chunk_len = pl.chunk_len; prm.nchunks = pl.nchunks;
    const int cpc = kSeqWarps * 32 / pl.g;
    prm.chan_blocks = (int)((d.dim + cpc - 1) / cpc);
    prm.npad = pl.nper * pl.g;
    const bool aligned = ((size_t)d.seqlen * io_size(d.io_dtype)) % 16 == 0;
    cudaError_t e = cudaSuccess;
    if (pl.nchunks > 1) {
        const size_t BD = (size_t)(d.batch * d.dim), npad = (size_t)prm.npad;
        char *w = static_cast<char *>(workspace);
        prm.agg_h = reinterpret_cast<float *>(w);
        prm.agg_s = reinterpret_cast<float *>(w + up256((size_t)pl.nchunks * BD * npad * 4));
        float *hin = reinterpret_cast<float *>(w + up256((size_t)pl.nchunks * BD * npad * 4) +
                                               up256((size_t)pl.nchunks * BD * 4));
        e = launch_seq(d.io_dtype, pl.nper, pl.g, true, aligned, prm, pl.nchunks - 1, s);
        if (e == cudaSuccess)
            e = launch_chunk_combine(A, prm.agg_h, prm.agg_s, hin, (int64_t)BD, d.dim, d.dstate, prm.npad,
                                     pl.nchunks, s);
        prm.hin = hin;
    }
    if (e == cudaSuccess) e = launch_seq(d.io_dtype, pl.nper, pl.g, false, aligned, prm, pl.nchunks, s);
    if (allocated) cudaFreeAsync(workspace, s);
    return cuda_status(e);
}

// ---- fixed scratch for ssm_selective_scan_fwd_noalloc -------------------------------------
// Callers that cannot allocate device memory at call time (their memory is held by another
// allocator's pool, their device has no stream-ordered pools, or they are plain C code with
// nothing to own a workspace) get the chunk carries, control words and prepared B/C from this
// array instead. One copy exists per device, in the module's own global memory; it is only
// ever passed to run_scan as a caller workspace, so no code path allocates on its behalf.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_SCRATCH_MAX_BYTES];

// Identity of the current context (cuCtxGetId), so that a scratch address cached for a
// device is re-resolved after the device's primary context was torn down and re-created
// (cudaDeviceReset), when the module and its array move. 0 when the query is unavailable.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur == nullptr || get_id == nullptr || get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of the current device's scratch, resolved with cudaGetSymbolAddress on the
// first use in each context of the device (which may load the module: outside any stream
// capture) and cached for the later calls in the same context.
ssm_status_t scratch_address(void **out) {
    int dev = 0;
    if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_status(e);
    const bool cached = dev >= 0 && dev < kMaxDevices;
    // establishes the primary context if the call is the first CUDA work of this thread
    if (const cudaError_t e = cudaFree(nullptr); e != cudaSuccess) return cuda_status(e);
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cached && ctx != 0 && g_scratch_addr[dev] != nullptr && g_scratch_ctx[dev] == ctx) {
        *out = g_scratch_addr[dev];
        return SSM_OK;
    }
    void *p = nullptr;
    if (const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch); e != cudaSuccess || p == nullptr)
        return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    if (cached) {
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
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
    const WsChoice w = default_workspace();
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w.ptr, w.bytes,
                    w.may_alloc, static_cast<cudaStream_t>(stream));
}

size_t ssm_selective_scan_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    return scan_workspace_bytes(*dims);
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

ssm_status_t ssm_set_workspace(void *dev_ptr, size_t bytes) {
    if (dev_ptr == nullptr && bytes != 0) return SSM_ERR_NULL;
    if (dev_ptr != nullptr && bytes == 0) return SSM_ERR_WORKSPACE;
    if (dev_ptr != nullptr && !aligned16(dev_ptr)) return SSM_ERR_ALIGN;
    int dev = 0;
    if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return SSM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    g_ws_ptr[dev] = dev_ptr;
    g_ws_bytes[dev] = dev_ptr != nullptr ? bytes : 0;
    return SSM_OK;
}

ssm_status_t ssm_selective_scan_fwd_noalloc(const ssm_dims_t *dims, const void *u, const void *delta,
                                            const float *A, const void *B, const void *C,
                                            const float *D, const void *z, const float *delta_bias,
                                            int delta_softplus, void *y, float *last_state,
                                            void *stream) {
    ssm_status_t st = scan_checks(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
    if (st != SSM_OK) return st;
    size_t need = scan_workspace_bytes(*dims);
    if (need > SSM_SCRATCH_MAX_BYTES) need = scan_workspace_bytes(*dims, true);   // without restrided rows
    if (need > SSM_SCRATCH_MAX_BYTES) return SSM_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        st = scratch_address(&scratch);
        if (st != SSM_OK) return st;
    }
    // may_alloc = false: run_scan may only use the scratch, never allocate a replacement
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
    const int64_t N = dims->dstate;
    const int lpc = (int)(N / 4);
    const bool vec = N % 4 == 0 && lpc >= 1 && lpc <= 32 && (32 % lpc) == 0;
    // batch rows on grid.y and 16-byte B/C reads when B and C rows are 4-element aligned;
    // the row's channels must fit a 32-bit thread index and grid.y (65535 rows)
    const bool wide = aligned_to(B, 4 * esz) && aligned_to(C, 4 * esz) && dims->batch <= 65535 &&
                      dims->dim * lpc < (int64_t)1 << 30 && !plan_override().decode_elementwise;
    const int kind = vec ? (wide ? 0 : 1) : 2;
    const cudaError_t e = launch_decode(dims->io_dtype, kind, lpc, zoh != 0, p, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidConfiguration) {
        cudaGetLastError();
        return SSM_ERR_UNSUPPORTED;
    }
    return cuda_status(e);
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
    WsChoice w{workspace, workspace_bytes, false};
    if (workspace == nullptr) w = default_workspace();
    return run_scan(dims, u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w.ptr, w.bytes,
                    w.may_alloc, static_cast<cudaStream_t>(stream), discretization == SSM_DISC_ZOH);
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
    WsChoice w{workspace, workspace_bytes, false};
    if (workspace == nullptr) w = default_workspace();
    const ssm_dims_t d = *dims;
    if (d.batch == 0 || d.dim == 0 || d.seqlen == 0)
        return run_scan(dims, x, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w.ptr, w.bytes,
                        w.may_alloc, static_cast<cudaStream_t>(stream));
    if (conv_w == nullptr) return SSM_ERR_NULL;
    if (!aligned_to(conv_w, 4)) return SSM_ERR_ALIGN;
    const ssm_plan_override_t ov = plan_override();
    const PairPlan pp = plan_pair(d, ov, true);
    if (pp.use)
        return run_scan_pair(d, pp, x, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w.ptr,
                             w.bytes, w.may_alloc, static_cast<cudaStream_t>(stream), 0, conv_w, conv_b, conv_width);
    PairPlan pr;
    RaggedPlan rg;
    if (use_ragged(d, ov, true, w.ptr, w.bytes, w.may_alloc, &pr, &rg))   // x goes into the u slot
        return run_scan_ragged(d, pr, rg, x, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state, w.ptr,
                               w.bytes, w.may_alloc, static_cast<cudaStream_t>(stream), 0, conv_w, conv_b,
                               conv_width);
    // the conv front runs on the channel-pair kernel only
    return ((size_t)d.seqlen * io_size(d.io_dtype)) % 16 != 0 && plan_pair(d, ov, true, true).use ? SSM_ERR_WORKSPACE
                                                                                                   : SSM_ERR_UNSUPPORTED;
}

size_t ssm_conv_selective_scan_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    const ssm_plan_override_t ov = plan_override();
    const PairPlan pp = plan_pair(*dims, ov, true);
    if (pp.use) return pair_workspace_bytes(*dims, pp);
    const PairPlan pr = plan_pair(*dims, ov, true, true);
    return pr.use ? plan_ragged(*dims, pr).bytes : 0;
}

}  // extern "C"

namespace {
// Backward plan. Lane split: Q states per thread, G lanes per channel (the smallest power of
// two with Q*G >= N: 1-32 at four states, 2-16 at two), 128/G channels per CTA. Time split:
// with fewer than two CTAs per SM, the sequence is cut into K chunks of whole 8-step segments
// (at least 16 segments each, K <= 64), each a CTA of the checkpoint, aggregate and adjoint
// passes; K gives the adjoint at least two waves and, among those counts, the fullest last
// wave (1 x 1536 x 16384 x 16: 25 chunks 1.24 ms, 18 1.17, 37 1.15). Q = 2 for N <= 8, else 4; without a possible
// time split, also Q = 2 when four states per lane give fewer than half a warp per SM
// sub-partition. Measured on B300 (bf16, gate, ms; the planner's choice first; K = chunks):
//   8 x 1536 x 2048 x 16:   Q4 unsplit 1.08; Q4 K4 1.30; Q2 unsplit 1.29
//   4 x 1536 x 2048 x 16:   Q4 K16 0.59; Q2 unsplit 0.67; Q4 unsplit 0.89
//   1 x 768 x 8192 x 16:    Q4 K37 0.31; Q4 K32 0.35; Q2 unsplit 1.89
//   1 x 1536 x 4096 x 32:   Q4 K23 0.55; Q4 unsplit 1.27
//   2 x 512 x 4096 x 8:     Q2 K32 0.16; Q4 K74 0.28; Q2 unsplit 1.30
//   1 x 5120 x 4096 x 16:   Q4 K11 0.94; Q4 K8 0.97; Q2 unsplit 1.32
//   2 x 1536 x 16384 x 16:  Q4 K37 2.21; Q4 K13 2.35; Q2 unsplit 4.38
struct BwdPlan {
    int G, Q, nchunk, seg_per_chunk;
    int64_t nseg;
};
BwdPlan bwd_plan(const ssm_dims_t &d) {
    const int64_t N = d.dstate, nseg = (d.seqlen + kBwdS - 1) / kBwdS, sms = sm_count();
    auto lanes = [&](int q) {
        int g = q == 2 ? 2 : 1;
        while (g < 32 && (int64_t)g * q < N) g *= 2;
        return g;
    };
    auto ctas = [&](int q) {
        const int64_t cpb = 128 / lanes(q);
        return (d.dim + cpb - 1) / cpb * d.batch;
    };
    const ssm_plan_override_t ov = plan_override();
    auto chunks = [&](int q) -> int64_t {
        int64_t k = 1;
        if (ov.bwd_chunks > 0) {
            k = ov.bwd_chunks;
        } else if (ctas(q) < 2 * sms) {
            // the adjoint's CTAs are equal and latency-bound, so its time goes with whole waves:
            // from at least two waves up, the chunk count whose last wave is fullest
            const int64_t slots = (int64_t)bwd_split_adjoint_ctas_per_sm(d.io_dtype, lanes(q), q) * sms;
            const int64_t hi = std::min<int64_t>(nseg / 16, 64), lo = std::min(hi, (2 * slots + ctas(q) - 1) / ctas(q));
            double best = -1.0;
            for (int64_t c = std::max<int64_t>(lo, 1); c <= hi; ++c) {
                const int64_t cta = ctas(q) * c, waves = (cta + slots - 1) / slots;
                const double fill = (double)cta / (double)(waves * slots);
                if (fill > best + 1e-9) best = fill, k = c;
            }
        }
        return std::max<int64_t>(1, std::min<int64_t>({k, nseg, 65535}));
    };
    int q = 4;
    if (ov.bwd_states_per_lane == 2 && N <= 32) q = 2;
    else if (ov.bwd_states_per_lane == 0 && N <= 8) q = 2;
    else if (ov.bwd_states_per_lane == 0 && N <= 32 && chunks(4) == 1 && d.batch * d.dim * lanes(4) < 64 * sms)
        q = 2;
    if (nseg == 0) return BwdPlan{lanes(q), q, 1, 0, 0};
    const int64_t k = chunks(q), spc = (nseg + k - 1) / k;
    return BwdPlan{lanes(q), q, (int)((nseg + spc - 1) / spc), (int)spc, nseg};
}
// workspace floats of a backward plan: the checkpoints, and with a time split the per-segment
// dt sums and the per-chunk states and carries (hloc, sdt, cloc, cin); the two per-row arrays
// are padded to 4 floats so that every array starts on a 16-byte boundary
int64_t round4(int64_t x) { return (x + 3) / 4 * 4; }
int64_t bwd_workspace_floats(const ssm_dims_t &d, const BwdPlan &pl) {
    const int64_t BD = d.batch * d.dim, np = pl.G * pl.Q;
    int64_t f = BD * pl.nseg * np;
    if (pl.nchunk > 1) f += round4(BD * pl.nseg) + round4(BD * pl.nchunk) + 3 * BD * pl.nchunk * np;
    return f;
}
}  // namespace

extern "C" {

size_t ssm_selective_scan_bwd_workspace_bytes(const ssm_dims_t *dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    return (size_t)bwd_workspace_floats(*dims, bwd_plan(*dims)) * sizeof(float);
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
    if (workspace != nullptr && !aligned16(workspace)) return SSM_ERR_ALIGN;
    if (d.batch > 65535) return SSM_ERR_UNSUPPORTED;
    const size_t need = ssm_selective_scan_bwd_workspace_bytes(dims);
    WsChoice w{workspace, workspace_bytes, false};
    if (workspace == nullptr) w = default_workspace();
    if (!empty && need > 0 && !w.may_alloc && (w.ptr == nullptr || w.bytes < need)) return SSM_ERR_WORKSPACE;
    // gradients summed over the sequence, the batch or the channels start at zero
    const size_t BD = (size_t)(d.batch * d.dim), NL = (size_t)(d.dstate * d.seqlen);
    cudaError_t ez = cudaMemsetAsync(dA, 0, (size_t)(d.dim * d.dstate) * 4, s);
    if (ez == cudaSuccess && dD) ez = cudaMemsetAsync(dD, 0, (size_t)d.dim * 4, s);
    if (ez == cudaSuccess && ddelta_bias) ez = cudaMemsetAsync(ddelta_bias, 0, (size_t)d.dim * 4, s);
    if (ez != cudaSuccess || empty) return cuda_status(ez);
    ez = cudaMemsetAsync(dB, 0, (size_t)d.batch * NL * 4, s);
    if (ez == cudaSuccess) ez = cudaMemsetAsync(dC, 0, (size_t)d.batch * NL * 4, s);
    if (ez == cudaSuccess && dz && !z) ez = cudaMemsetAsync(dz, 0, BD * (size_t)d.seqlen * 4, s);
    if (ez != cudaSuccess) return cuda_status(ez);
    void *ws = w.ptr;
    bool allocated = false;
    st = acquire_workspace(&ws, w.bytes, need, w.may_alloc, s, &allocated);
    if (st != SSM_OK) return st;
    const BwdPlan pl = bwd_plan(d);
    BwdParams p{u, delta, z, B, C, dy, A, D, delta_bias, dlast_state, du, ddelta, dA, dB, dC, dD,
                z ? dz : nullptr, ddelta_bias, static_cast<float *>(ws), d.batch, d.dim, d.seqlen,
                d.dstate, delta_softplus ? 1 : 0, (int)pl.nseg, 0, 0, pl.nchunk, pl.seg_per_chunk,
                nullptr, nullptr, nullptr, nullptr, nullptr};
    if (pl.nchunk > 1) {   // after the checkpoints: cumdt, hloc, sdt, cloc, cin
        const int64_t BD = d.batch * d.dim, np = pl.G * pl.Q, K = pl.nchunk;
        float *q = static_cast<float *>(ws) + BD * pl.nseg * np;
        p.cumdt = q;
        q += round4(BD * pl.nseg);
        p.hloc = q;
        q += BD * K * np;
        p.sdt = q;
        q += round4(BD * K);
        p.cloc = q;
        q += BD * K * np;
        p.cin = q;
    }
    // rows read two steps per load: an even length and every row base on a 2-element boundary
    bool pair2 = d.seqlen % 2 == 0;
    for (const void *q : io_ptrs)
        if (q != nullptr && !aligned_to(q, 2 * esz)) pair2 = false;
    p.pair2 = pair2 ? 1 : 0;
    // rows staged by 16-byte asynchronous copies: rows of whole 16-byte pieces, aligned bases
    bool ring = (d.seqlen * (int64_t)esz) % 16 == 0;
    for (const void *q : io_ptrs)
        if (q != nullptr && !aligned16(q)) ring = false;
    p.ring = ring ? 1 : 0;
    const cudaError_t e = launch_bwd(d.io_dtype, pl.G, pl.Q, p, s);
    if (allocated) cudaFreeAsync(ws, s);
    if (e == cudaErrorInvalidConfiguration) {
        cudaGetLastError();
        return SSM_ERR_UNSUPPORTED;
    }
    return cuda_status(e);
}

// Channel blocks of the host-buffer entry: up to kHostBlocks per call, each with at least
// kHostBlockBytes of input. More blocks shorten the exposed head (the first block's input
// copy) and tail (the last block's scan and output copy). Measured on B300 for
// 1 x 1536 x 131072 x 64 bf16 (839 MB in, 403 MB out per call; both directions copied
// concurrently alone take 18.6 ms): 4 / 8 / 16 / 24 / 32 blocks 23.7 / 21.5 / 20.3 / 19.9 /
// 19.7 ms per call.
#ifndef SSM_HOST_BLOCKS
#define SSM_HOST_BLOCKS 32
#endif
constexpr int kHostBlocks = SSM_HOST_BLOCKS;
constexpr size_t kHostBlockBytes = (size_t)8 << 20;

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
    // Channel blocks (at least one per batch row) flow through three streams: copies in,
    // scans, copies out. Three buffer sets rotate, so block k's input
    // copy overlaps block k-1's scan and block k-2's output copy; the first block's input
    // copy and the last block's scan and output copy are the exposed head and tail.
    // Blocks start on multiples of 4 channels so that A + d0*N, D + d0 and bias + d0 stay
    // 16-byte aligned; each batch row of B and C gets its own 256-byte aligned slot.
    constexpr int kBufs = 3;
    const size_t row_in_bytes = Dm * L * esz * (z ? 3 : 2);
    const size_t per_row = std::max<size_t>(
        1, std::min<size_t>({(Dm + 3) / 4, (row_in_bytes + kHostBlockBytes - 1) / kHostBlockBytes,
                             (size_t)std::max<int64_t>(1, kHostBlocks / d.batch)}));
    const size_t blk = ((Dm + per_row - 1) / per_row + 3) / 4 * 4;
    const size_t bc_row = up256(N * L * esz);
    const size_t row_bytes = blk * L * esz;
    enum { kIn = 0, kScan = 1, kOut = 2 };
    cudaStream_t ss[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t ev_start = nullptr, ev_const = nullptr;
    cudaEvent_t ev_in[kBufs] = {}, ev_scan[kBufs] = {}, ev_out[kBufs] = {};
    ssm_status_t rc = SSM_OK;
    void *dA = nullptr, *dD = nullptr, *dbias = nullptr, *dB = nullptr, *dC = nullptr;
    void *bu[kBufs] = {}, *bdl[kBufs] = {}, *bz[kBufs] = {}, *by[kBufs] = {}, *bst[kBufs] = {};
    auto CK = [&](cudaError_t e) { if (e != cudaSuccess && rc == SSM_OK) rc = cuda_status(e); return e == cudaSuccess; };
    for (auto &q : ss) CK(cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking));
    CK(cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&ev_const, cudaEventDisableTiming));
    for (int i = 0; i < kBufs; ++i) {
        CK(cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming));
        CK(cudaEventCreateWithFlags(&ev_scan[i], cudaEventDisableTiming));
        CK(cudaEventCreateWithFlags(&ev_out[i], cudaEventDisableTiming));
    }
    if (rc == SSM_OK) {
        CK(cudaMallocAsync(&dA, Dm * N * 4, s0));
        if (D) CK(cudaMallocAsync(&dD, Dm * 4, s0));
        if (delta_bias) CK(cudaMallocAsync(&dbias, Dm * 4, s0));
        CK(cudaMallocAsync(&dB, (size_t)d.batch * bc_row, s0));
        CK(cudaMallocAsync(&dC, (size_t)d.batch * bc_row, s0));
        for (int i = 0; i < kBufs; ++i) {
            CK(cudaMallocAsync(&bu[i], row_bytes, s0));
            CK(cudaMallocAsync(&bdl[i], row_bytes, s0));
            if (z) CK(cudaMallocAsync(&bz[i], row_bytes, s0));
            CK(cudaMallocAsync(&by[i], row_bytes, s0));
            if (last_state) CK(cudaMallocAsync(&bst[i], blk * N * 4, s0));
        }
        // the pipeline starts after the allocations and whatever the caller queued on `stream`
        CK(cudaEventRecord(ev_start, s0));
        for (auto &q : ss) CK(cudaStreamWaitEvent(q, ev_start, 0));
    }
    if (rc == SSM_OK) {
        cudaStream_t si = ss[kIn];
        CK(cudaMemcpyAsync(dA, A, Dm * N * 4, cudaMemcpyHostToDevice, si));
        if (D) CK(cudaMemcpyAsync(dD, D, Dm * 4, cudaMemcpyHostToDevice, si));
        if (delta_bias) CK(cudaMemcpyAsync(dbias, delta_bias, Dm * 4, cudaMemcpyHostToDevice, si));
        for (int64_t b = 0; b < d.batch; ++b) {
            CK(cudaMemcpyAsync(static_cast<char *>(dB) + b * bc_row, static_cast<const char *>(B) + b * N * L * esz,
                               N * L * esz, cudaMemcpyHostToDevice, si));
            CK(cudaMemcpyAsync(static_cast<char *>(dC) + b * bc_row, static_cast<const char *>(C) + b * N * L * esz,
                               N * L * esz, cudaMemcpyHostToDevice, si));
        }
        CK(cudaEventRecord(ev_const, si));
        CK(cudaStreamWaitEvent(ss[kScan], ev_const, 0));
    }
    size_t k = 0;
    for (int64_t b = 0; b < d.batch && rc == SSM_OK; ++b) {
        for (size_t d0 = 0; d0 < Dm && rc == SSM_OK; d0 += blk, ++k) {
            const int j = (int)(k % kBufs);
            const size_t nd = std::min(blk, Dm - d0);
            const size_t off = ((size_t)b * Dm + d0) * L * esz;
            // copies in: buffer j is free once block k-3's scan has read it
            if (k >= kBufs) CK(cudaStreamWaitEvent(ss[kIn], ev_scan[j], 0));
            CK(cudaMemcpyAsync(bu[j], static_cast<const char *>(u) + off, nd * L * esz, cudaMemcpyHostToDevice, ss[kIn]));
            CK(cudaMemcpyAsync(bdl[j], static_cast<const char *>(delta) + off, nd * L * esz, cudaMemcpyHostToDevice,
                               ss[kIn]));
            if (z) CK(cudaMemcpyAsync(bz[j], static_cast<const char *>(z) + off, nd * L * esz, cudaMemcpyHostToDevice,
                                      ss[kIn]));
            CK(cudaEventRecord(ev_in[j], ss[kIn]));
            // scan: after its inputs, and after block k-3's output copy has read y and the state
            CK(cudaStreamWaitEvent(ss[kScan], ev_in[j], 0));
            if (k >= kBufs) CK(cudaStreamWaitEvent(ss[kScan], ev_out[j], 0));
            if (rc != SSM_OK) break;
            ssm_dims_t sub{1, (int64_t)nd, d.seqlen, d.dstate, d.io_dtype};
            const size_t boff = (size_t)b * bc_row;
            // the scans are queued on one stream; their chunk carries are stream-ordered
            // allocations (never the registered workspace)
            const ssm_status_t r = run_scan(
                &sub, bu[j], bdl[j], static_cast<float *>(dA) + d0 * N, static_cast<char *>(dB) + boff,
                static_cast<char *>(dC) + boff, D ? static_cast<float *>(dD) + d0 : nullptr, z ? bz[j] : nullptr,
                delta_bias ? static_cast<float *>(dbias) + d0 : nullptr, delta_softplus, by[j],
                last_state ? static_cast<float *>(bst[j]) : nullptr, nullptr, 0, true, ss[kScan]);
            if (r != SSM_OK) { rc = r; break; }
            CK(cudaEventRecord(ev_scan[j], ss[kScan]));
            // copies out
            CK(cudaStreamWaitEvent(ss[kOut], ev_scan[j], 0));
            CK(cudaMemcpyAsync(static_cast<char *>(y) + off, by[j], nd * L * esz, cudaMemcpyDeviceToHost, ss[kOut]));
            if (last_state)
                CK(cudaMemcpyAsync(last_state + ((size_t)b * Dm + d0) * N, bst[j], nd * N * 4, cudaMemcpyDeviceToHost,
                                   ss[kOut]));
            CK(cudaEventRecord(ev_out[j], ss[kOut]));
        }
    }
    for (auto &q : ss)
        if (q) CK(cudaStreamSynchronize(q));
    // release everything on s0 after the pipeline finished
    void *all[] = {dA, dD, dbias, dB, dC, bu[0], bu[1], bu[2], bdl[0], bdl[1], bdl[2], bz[0], bz[1], bz[2],
                   by[0], by[1], by[2], bst[0], bst[1], bst[2]};
    for (void *q : all)
        if (q) cudaFreeAsync(q, s0);
    CK(cudaStreamSynchronize(s0));
    for (auto &q : ss)
        if (q) cudaStreamDestroy(q);
    cudaEvent_t evs[] = {ev_start, ev_const, ev_in[0], ev_in[1], ev_in[2], ev_scan[0], ev_scan[1], ev_scan[2],
                         ev_out[0], ev_out[1], ev_out[2]};
    for (cudaEvent_t e : evs)
        if (e) cudaEventDestroy(e);
    return rc;
}

ssm_status_t ssm_stream_status(void *stream) {
    if (const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream)); e != cudaSuccess)
        return cuda_status(e);
    int v = 0;
    if (const cudaError_t e = cudaMemcpyFromSymbol(&v, ssm::g_ssm_status, sizeof(int)); e != cudaSuccess)
        return cuda_status(e);
    if (v != 0) {
        const int zero = 0;
        if (const cudaError_t e = cudaMemcpyToSymbol(ssm::g_ssm_status, &zero, sizeof(int)); e != cudaSuccess)
            return cuda_status(e);
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
        case SSM_ERR_CHECK: return "SSM_ERR_CHECK: a bounds check of the checked build failed";
        default: return "SSM_ERR_UNKNOWN";
    }
}

int ssm_last_cuda_error(void) { return t_last_cuda_error; }

const char *ssm_cuda_error_string(int code) {
    const char *t = cudaGetErrorString(static_cast<cudaError_t>(code));
    return t ? t : "unknown CUDA error";
}

int ssm_set_structured_a(int enable) { return g_structured_a.exchange(enable ? 1 : 0); }

ssm_status_t ssm_set_plan_override(const ssm_plan_override_t *ov) {
    ssm_plan_override_t v{};
    if (ov != nullptr) {
        v = *ov;
        if (v.kernel < SSM_KERNEL_AUTO || v.kernel > SSM_KERNEL_TP) return SSM_ERR_UNSUPPORTED;
        if (v.pair_states_per_lane != 0 && v.pair_states_per_lane != 4 && v.pair_states_per_lane != 8 &&
            v.pair_states_per_lane != 16)
            return SSM_ERR_UNSUPPORTED;
        if (v.chunks < 0 || v.seq_states_per_lane < 0 || v.seq_lanes_per_channel < 0) return SSM_ERR_SHAPE;
        if (v.bwd_states_per_lane != 0 && v.bwd_states_per_lane != 2 && v.bwd_states_per_lane != 4)
            return SSM_ERR_UNSUPPORTED;
        if (v.bwd_chunks < 0) return SSM_ERR_SHAPE;
        if ((v.seq_states_per_lane != 0 || v.seq_lanes_per_channel != 0) &&
            !seq_plan_supported(v.seq_states_per_lane, v.seq_lanes_per_channel))
            return SSM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_override_mu);
    g_override = v;
    return SSM_OK;
}

ssm_status_t ssm_get_plan_override(ssm_plan_override_t *out) {
    if (out == nullptr) return SSM_ERR_NULL;
    *out = plan_override();
    return SSM_OK;
}

int ssm_version(void) { return (1 << 16) | 3; }

}  // extern "C"
