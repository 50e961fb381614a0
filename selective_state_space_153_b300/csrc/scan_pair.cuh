// Selective scan, channel-pair kernel: each lane walks the sequence for TWO channels and KS
// of their states, so one shared-memory read of B[t, n..n+3] (and of C) serves two channels
// and every arithmetic step runs on packed pairs (f32x2): per (channel, state, timestep) one
// MUFU ex2 and four FP32 operations -- dt*A, dt*u*B, the recurrence FMA and the readout FMA.
//
// Source of the computation: the per-timestep loop of section 3.2 of "From RNN to Mamba:
// state-space model principles and long-sequence modelling in practice" (lmnt.cn):
// A_bar = exp(dt*A), B_bar = dt*B_t, h = A_bar*h + B_bar*x_t, y_t = sum_n h*C_t, then
// y + x*D and the SiLU(z) gate; dt = softplus(delta + bias) (sections 3.2-3.3).
//
// Work decomposition (one CTA): batch row b, kCh = WARPS*2*(32/GP) consecutive channels,
// one chunk [l_begin, l_end) of the sequence walked in tiles of T timesteps. KS is 4, 8 or
// 16 states per lane and channel; the planner picks it and the CTA width per pass.
//   lane (warp w, lane l): pair P = w*(32/GP) + l/GP -> channels 2P and 2P+1 of the block;
//   state group g = l%GP owns the states n = 4*(GP*q + g) + j (q < KS/4, j < 4), so the GP
//   groups of a pair read GP adjacent 16-byte pieces of a B/C row (one wavefront per
//   LDS.128, broadcast to the 32/GP pairs of the warp).
//   y: per channel each lane keeps its partial sum over its KS states; every GP timesteps
//   the GP lanes exchange partials with a transposed butterfly (lane g ends with the sum for
//   timestep tb+g), add D*u, apply the gate and store y.
// Rows of u, delta, z, y, B, C are addressed with the row stride p.ld: L, or the padded
// stride of rows the host copied onto 16-byte boundaries (rows that are not 16-byte
// multiples); the scan itself covers the L steps.
// Pipeline per tile: raw io rows (u, delta, z, B, C) arrive by cp.async three tiles deep;
// one barrier per tile; then tile j+1 is converted (softplus, dt*u per (channel, t); B, C to
// fp32, transposed to [t][n]) while tile j is scanned from the previous conversion.
//
// Discretisation: B_bar*u = dt*u*B (the lmnt.cn loop) or, with ZOH, the exact zero-order
// hold (exp(dt*A) - 1)/A * B * u of "Mamba architecture principles and industrial long-text
// practice" (jsqmd.com), section 2.3, from a = exp(dt*A) already computed for the
// recurrence (no extra exponential per element). In a tile where |dt*A| is above a threshold
// at every step for every state of the warp's channels it is (a - 1) * (u*B/A); otherwise
// u*B * dt*phi(dt*A), phi(x) = (e^x - 1)/x, with a cubic Taylor polynomial for |x| < 1/8
// (truncation <= 2e-6 relative) and (a - 1)/A above it.
//
// Structured A: where every state of a warp's channels has A[d, n] = (n + 1) * A[d, 0] (the
// S4D-real initialisation A_log = log(1..N) of section 3.3 of the lmnt.cn page, before
// training moves it), exp(dt*A[d, n]) = r^(n+1) with r = exp(dt*A[d, 0]). Such a warp
// (detected at run time with a warp vote, unless the host switches detection off) takes
// the decays of a quad of states n0..n0+3 as e, e*r, e*r^2, e*r^3 with e = exp(dt*A[d, n0]):
// one ex2 per quad and one per channel for r instead of one per state.
//
// Modes: FULL computes y (and the final state of the last chunk); AGG computes only the
// chunk's end state from h = 0 and the chunk's sum of dt, from which chunk_combine_kernel
// forms each chunk's incoming state (the recurrence is a composition of affine maps --
// section 2.2 of the lmnt.cn page, section 3.4 of "Mamba architecture principles and
// industrial long-text practice", jsqmd.com -- so chunk end states compose exactly).
#pragma once
#include "check.cuh"
#include "common.cuh"
#include "scan_seq.cuh"

namespace ssm {

template <typename IO, int KS, int GP, int WARPS, int T, bool CONV = false>
struct PairCfg {
    static constexpr int kThreads = WARPS * 32;
    static constexpr int kPairsW = 32 / GP;            // pairs per warp
    static constexpr int kPairs = WARPS * kPairsW;     // pairs per CTA
    static constexpr int kCh = 2 * kPairs;             // channels per CTA
    static constexpr int kQN = KS / 4;                 // float4 quads of states per lane
    static constexpr int kNP = 4 * GP * kQN;           // padded state count
    static constexpr int kEpr = 16 / (int)sizeof(IO);  // io elements per 16-byte piece
    static constexpr int kRS = T;                      // raw row stride (io elements)
    static constexpr int kRawRows = 3 * kCh + 2 * kNP;  // u, delta, z rows, then B, C rows
    static constexpr size_t kRawBytes = (size_t)kRawRows * kRS * sizeof(IO);
    static constexpr size_t kDxBytes = (size_t)T * kPairs * sizeof(float4);
    static constexpr size_t kBcBytes = (size_t)T * 2 * kNP * sizeof(float);
    static constexpr size_t kYsBytes = (size_t)kCh * kRS * sizeof(IO);   // y tile staging, rows like raw
    static constexpr size_t kOffDx = 3 * kRawBytes;
    static constexpr size_t kOffBc = kOffDx + 2 * kDxBytes;
    static constexpr size_t kOffYs = kOffBc + 2 * kBcBytes;
    static constexpr size_t kOffBias = kOffYs + 2 * kYsBytes;
    // steps per conversion item (8, or 4 when 8 would leave threads idle) and the aggregate
    // pass's per-item sums of dt, [2][kCh][T / kSI]
    static constexpr int kSI = (kCh * (T / 8) >= kThreads) ? 8 : 4;
    static constexpr size_t kOffTs = kOffBias + (size_t)kCh * sizeof(float);
    static constexpr size_t kTsBytes = (size_t)2 * kCh * (T / kSI) * sizeof(float);
    // the zero-order hold's per-item smallest dt of the in-range steps, [2][kCh][T / kSI]
    static constexpr size_t kOffTm = kOffTs + kTsBytes;
    static constexpr size_t kTmBytes = kTsBytes;
    // conv front: the conv + SiLU output u [2][kCh][T] fp32, the right-aligned taps [kCh][4],
    // the conv bias [kCh] and the chunk's first-tile halo [kCh][4] (three steps used)
    static constexpr size_t kOffSu = kOffTm + kTmBytes;
    static constexpr size_t kSuBytes = CONV ? (size_t)2 * kCh * T * sizeof(float) : 0;
    static constexpr size_t kOffCw = kOffSu + kSuBytes;
    static constexpr size_t kCwBytes = CONV ? (size_t)kCh * 9 * sizeof(float) : 0;
    static constexpr size_t kSmem = kOffCw + kCwBytes;
    static_assert(KS == 4 || KS == 8 || KS == 16, "states per lane per channel: 4, 8 or 16");
    static_assert(GP == 1 || GP == 2 || GP == 4 || GP == 8 || GP == 16, "lanes per pair");
    static_assert(T % 8 == 0 && T % GP == 0 && T % kEpr == 0, "tile: whole 16-byte pieces and reduce groups");
    static_assert((kRS * sizeof(IO)) % 16 == 0 && kRawBytes % 16 == 0, "16-byte aligned raw rows");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Warps per CTA for a lane split and pass: SSM_PAIR_WARPS (at most 64 channels per CTA) for
// four or more lanes per pair, fewer for GP < 4; the full pass of the 8-states x 8-lanes
// split (dstate 33..64) runs SSM_PAIR_WARPS_WIDE warps, so a CTA's B/C conversion and copies
// serve twice the channels (measured faster for that pass only; narrower CTAs win for the
// aggregate pass and for the other splits).
#ifndef SSM_PAIR_WARPS
#define SSM_PAIR_WARPS 4
#endif
#ifndef SSM_PAIR_WARPS_WIDE
#define SSM_PAIR_WARPS_WIDE 8
#endif
constexpr int pair_warps(int ks, int gp, bool agg) {
    return gp >= 4 ? ((!agg && ks == 8 && gp == 8) ? SSM_PAIR_WARPS_WIDE : SSM_PAIR_WARPS) : gp;
}
// Registers per thread the kernels are held to (launch bounds), so that residency per SM
// follows from the block size alone: 128, or 168 for sixteen lanes per pair and for sixteen
// states per lane (whose 32 states and 32 decay factors per lane spill under 128).
// Groups of GP steps of a tile unrolled into one loop body (1: a GP-step body walked T/GP
// times; larger bodies save loop and address work but the kernel's code outgrows the
// instruction cache). The Euler aggregate pass, whose body has no readout, unrolls the
// whole tile. Measured on B300, 1 x 1536 x 131072 x 64 bf16: full pass 2634 us (1) vs
// 2691 us (whole tile); aggregate 1955 vs 1909 us; the zero-order hold 6.94 vs 9.6 ms per
// call, where the whole-tile bodies stalled on instruction fetch.
#ifndef SSM_PAIR_TILE_UNROLL
#define SSM_PAIR_TILE_UNROLL 1
#endif
constexpr int kPairTileUnroll = SSM_PAIR_TILE_UNROLL;
// (Measured alternatives on B300 for 1 x 1536 x 131072 x 64: the full pass at 255 registers,
// 2 CTAs per SM, took 2.99 ms against 2.69 ms at 168 registers, 3 CTAs per SM.)
constexpr int pair_reg_budget(int ks, int gp) { return (gp >= 16 || ks >= 16) ? 168 : 128; }
constexpr int pair_min_blocks(int warps, int ks, int gp) { return 65536 / (warps * 32 * pair_reg_budget(ks, gp)); }

// S (4 or 8) consecutive io elements from shared memory as floats; the source is aligned to
// S elements (8 or 16 bytes for bf16, 16 or 32 for fp32)
template <int S>
__device__ __forceinline__ void load_steps(const __nv_bfloat16 *src, float (&out)[S]) {
    if constexpr (S == 8) {
        unpack16(*reinterpret_cast<const uint4 *>(src), out, __nv_bfloat16(0.0f));
    } else {
        const uint2 v = *reinterpret_cast<const uint2 *>(src);
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x); out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
    }
}
template <int S>
__device__ __forceinline__ void load_steps(const float *src, float (&out)[S]) {
#pragma unroll
    for (int q = 0; q < S / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4 *>(src + 4 * q);
        out[4 * q] = v.x; out[4 * q + 1] = v.y; out[4 * q + 2] = v.z; out[4 * q + 3] = v.w;
    }
}

// dt*phi(x), phi(x) = (e^x - 1)/x, for the pair (x0, x1) with x = dt*A given in log2 units
// (xl2 = x * log2(e)) and a = exp(x) from the recurrence: for |x| < 1/8 the cubic Taylor
// polynomial of phi written in xl2 (truncation <= 2e-6 relative) times dt; else (a - 1) * (1/A)
// (the cancellation in a - 1 is then <= 2e-6 relative). ninv_a = -1/A of the states (0 where
// A = 0, where the polynomial branch applies).
__device__ __forceinline__ float2 zoh_psi2(float2 xl2, float2 a, float2 dt, float2 ninv_a) {
    constexpr float c1 = 0.34657359027997264f;    // ln2 / 2
    constexpr float c2 = 0.080075118466603945f;   // ln2^2 / 6
    constexpr float c3 = 0.013876131297784016f;   // ln2^3 / 24
    constexpr float kSmall = 0.18033688011112042f;   // 1/8 in log2 units
    float2 poly = __ffma2_rn(xl2, make_float2(c3, c3), make_float2(c2, c2));
    poly = __ffma2_rn(poly, xl2, make_float2(c1, c1));
    poly = __ffma2_rn(poly, xl2, make_float2(1.0f, 1.0f));
    const float2 small = __fmul2_rn(poly, dt);
    const float2 big = __fmul2_rn(fsub2_rn(make_float2(1.0f, 1.0f), a), ninv_a);
    return make_float2(fabsf(xl2.x) < kSmall ? small.x : big.x, fabsf(xl2.y) < kSmall ? small.y : big.y);
}

// Zero-order hold, fast path: in a tile where |dt*A| >= the threshold at every step for every
// state of a warp's channels (log2 units; chosen per io type so that the relative error of
// exp(x) - 1, about 2e-7 / |x|, stays below the tolerance's scale: 1/8 for fp32 io, 2^-12 for
// bf16 io), B_bar*u = (a - 1) * (u*B/A) without the polynomial branch.
template <typename IO> struct ZohFast;
template <> struct ZohFast<float> { static constexpr float kMinXl2 = 0.18033688011112042f; };
template <> struct ZohFast<__nv_bfloat16> { static constexpr float kMinXl2 = 3.5221e-4f; };

template <typename IO, int KS, int GP, int WARPS, int T, bool AGG, bool ZOH = false, bool CONV = false>
__global__ void __launch_bounds__(WARPS * 32, pair_min_blocks(WARPS, KS, GP))
scan_pair_kernel(const SeqParams p) {
    using Cfg = PairCfg<IO, KS, GP, WARPS, T, CONV>;
    constexpr int kCh = Cfg::kCh, kPairs = Cfg::kPairs, kQN = Cfg::kQN, kNP = Cfg::kNP, kRS = Cfg::kRS;
    constexpr int kEpr = Cfg::kEpr, kPieces = T / kEpr;
    extern __shared__ __align__(16) unsigned char smem[];
    float4 *sDX0 = reinterpret_cast<float4 *>(smem + Cfg::kOffDx);   // [T][kPairs] (dt0, dt0*u0, dt1, dt1*u1)
    float *sBC0 = reinterpret_cast<float *>(smem + Cfg::kOffBc);     // [T][2*kNP]  B | C
    IO *sYS0 = reinterpret_cast<IO *>(smem + Cfg::kOffYs);           // [kCh][kRS]  y tile, io type
    float *sBias = reinterpret_cast<float *>(smem + Cfg::kOffBias);  // [kCh]
    float *sTS0 = reinterpret_cast<float *>(smem + Cfg::kOffTs);     // [2][kCh][T/kSI] sums of dt
    float *sTM0 = reinterpret_cast<float *>(smem + Cfg::kOffTm);     // [2][kCh][T/kSI] smallest dt (ZOH)
    float *sSu0 = reinterpret_cast<float *>(smem + Cfg::kOffSu);     // conv front: [2][kCh][T] u
    float *sCw = reinterpret_cast<float *>(smem + Cfg::kOffCw);      // conv front: [kCh][4] taps
    float *sCb = sCw + 4 * kCh;                                      // [kCh] conv bias
    float *sHalo = sCb + kCh;                                        // [kCh][4] steps before the chunk
    auto raw_of = [&](int j) { return reinterpret_cast<IO *>(smem + (size_t)(j % 3) * Cfg::kRawBytes); };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b = blockIdx.x / p.chan_blocks;
    const int64_t d0 = (int64_t)(blockIdx.x % p.chan_blocks) * kCh;
    const int k = blockIdx.y;
    const int64_t l_begin = (int64_t)k * p.chunk_len;
    const int64_t l_end = min(p.L, l_begin + p.chunk_len);
    const int ntiles = (int)((l_end - l_begin + T - 1) / T);
    const int N = (int)p.N;
    const int64_t BD = p.Bt * p.Dm;
    SSM_POISON_SMEM(smem);
    // array extents in bytes (used by the checked build's bounds checks; dead code otherwise)
    const uint64_t kIoB = (uint64_t)p.Bt * p.Dm * p.ld * sizeof(IO), kBcB = (uint64_t)p.Bt * p.N * p.ld * sizeof(IO);
    const uint64_t kAB = (uint64_t)p.Dm * p.N * 4, kDB = (uint64_t)p.Dm * 4;
    const uint64_t kCarryB = (uint64_t)p.nchunks * BD * p.npad * 4, kSumB = (uint64_t)p.nchunks * BD * 4;
    (void)kIoB; (void)kBcB; (void)kAB; (void)kDB; (void)kCarryB; (void)kSumB;
    auto ldA = [&](int64_t i) -> float { return ld_chk_g(p.A, kAB, p.A + i); };
#ifdef SSM_CHECK
    // test of the checks themselves: one load one element past A, which the check must skip
    if (p.check_probe && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) (void)ldA((int64_t)p.Dm * p.N);
#endif

    const int pr = warp * Cfg::kPairsW + lane / GP;   // pair within the block
    const int g = lane % GP;
    const int c0 = 2 * pr;                             // first channel of the pair (block-relative)
    const int64_t dch[2] = {d0 + c0, d0 + c0 + 1};
    const bool cv[2] = {dch[0] < p.Dm, dch[1] < p.Dm};

    // A * log2(e) for the lane's states, as (n, n+1) pairs; zero for padded states
    float2 Ap[2][kQN][2];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int q = 0; q < kQN; ++q)
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                const int n = 4 * (GP * q + g) + 2 * pp;
                const float a0 = (cv[ch] && n < N) ? ldA(dch[ch] * p.N + n) * kLog2e : 0.0f;
                const float a1 = (cv[ch] && n + 1 < N) ? ldA(dch[ch] * p.N + n + 1) * kLog2e : 0.0f;
                Ap[ch][q][pp] = make_float2(a0, a1);
            }
    // structured-A test for the lane's states; padded states (n >= N) never qualify
    float Ap0[2];
    bool lane_st = p.structured != 0;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const float A0 = cv[ch] ? ldA(dch[ch] * p.N) : 0.0f;
        Ap0[ch] = A0 * kLog2e;
#pragma unroll
        for (int q = 0; q < kQN; ++q)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int n = 4 * (GP * q + g) + jj;
                if (n >= N) lane_st = false;
                else if (cv[ch] && ldA(dch[ch] * p.N + n) != (float)(n + 1) * A0) lane_st = false;
            }
    }
    const bool st = __all_sync(0xffffffffu, lane_st);
    // -1/A of the lane's states (ZOH; zero where A = 0, where phi's polynomial branch applies)
    float2 iA[2][kQN][2];
    if constexpr (ZOH) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int q = 0; q < kQN; ++q)
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const float a0 = Ap[ch][q][pp].x, a1 = Ap[ch][q][pp].y;   // A*log2(e)
                    iA[ch][q][pp] = make_float2(a0 != 0.0f ? -kLog2e / a0 : 0.0f, a1 != 0.0f ? -kLog2e / a1 : 0.0f);
                }
    }
    // ZOH fast-path test: the smallest |A*log2(e)| over the lane's real states, per channel
    // (padded states carry no input, so they do not count; an invalid channel never blocks)
    float zmin[2] = {0.0f, 0.0f};
    if constexpr (ZOH) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            float m = 3.0e38f;
#pragma unroll
            for (int q = 0; q < kQN; ++q)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int n = 4 * (GP * q + g) + jj;
                    if (cv[ch] && n < N) m = fminf(m, fabsf(ldA(dch[ch] * p.N + n) * kLog2e));
                }
            zmin[ch] = m;
        }
    }
    float2 h[2][kQN][2];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int q = 0; q < kQN; ++q) {
            h[ch][q][0] = make_float2(0.f, 0.f);
            h[ch][q][1] = make_float2(0.f, 0.f);
            if (!AGG && p.hin != nullptr && cv[ch]) {
                const float4 v = ld_chk_g(p.hin, kCarryB, reinterpret_cast<const float4 *>(
                    p.hin + ((int64_t)k * BD + b * p.Dm + dch[ch]) * p.npad + 4 * (GP * q + g)));
                h[ch][q][0] = make_float2(v.x, v.y);
                h[ch][q][1] = make_float2(v.z, v.w);
            }
        }
    const float Dd[2] = {(!AGG && p.D != nullptr && cv[0]) ? ld_chk_g(p.D, kDB, p.D + dch[0]) : 0.0f,
                         (!AGG && p.D != nullptr && cv[1]) ? ld_chk_g(p.D, kDB, p.D + dch[1]) : 0.0f};

    const IO *gU = reinterpret_cast<const IO *>(p.u);
    const IO *gDelta = reinterpret_cast<const IO *>(p.delta);
    const IO *gZ = reinterpret_cast<const IO *>(p.z);
    const IO *gB = reinterpret_cast<const IO *>(p.B);
    const IO *gC = reinterpret_cast<const IO *>(p.C);
    const bool has_z = !AGG && p.z != nullptr;

    // raw rows: [0,kCh) u, [kCh,2kCh) delta, then (full pass) [2kCh,3kCh) z, then kNP B rows
    // and (full pass) kNP C rows; padded state rows are never copied (converted as zeros).
    // Copy item i of a tile is row i / kPieces, piece i % kPieces. A thread's items are the
    // same in every tile, so where it has few of them their global sources (at the chunk's
    // first step; null for an item with nothing to copy) are computed once and a tile adds
    // its time offset; the shared destinations are a fixed stride apart.
    constexpr int kRowB = AGG ? 2 * kCh : 3 * kCh;
    constexpr int kRows = AGG ? 2 * kCh + kNP : 3 * kCh + 2 * kNP;
    constexpr int kItems = (kRows * kPieces + Cfg::kThreads - 1) / Cfg::kThreads;
    constexpr bool kPre = kItems <= 6;
    constexpr uint32_t kItemStride = (uint32_t)((Cfg::kThreads / kPieces) * kRS * sizeof(IO));
    const int e0_me = (tid % kPieces) * kEpr;   // the thread's piece: kThreads is a multiple of kPieces
    const uint32_t idst0 = (uint32_t)(((tid / kPieces) * kRS + e0_me) * sizeof(IO));
    auto item_src = [&](int row) -> const IO * {   // source at the chunk's first step, or null
        if (row < kRowB) {
            const int kind = row / kCh, cc = row % kCh;
            if (d0 + cc >= p.Dm || (kind == 2 && !has_z)) return nullptr;
            const IO *base = kind == 0 ? gU : (kind == 1 ? gDelta : gZ);
            return base + ((b * p.Dm + d0 + cc) * p.ld + l_begin + e0_me);
        }
        if (row >= kRows) return nullptr;
        const int r = row - kRowB, kind = r / kNP, n = r % kNP;
        if (n >= N) return nullptr;
        return (kind == 0 ? gB : gC) + ((b * p.N + n) * p.ld + l_begin + e0_me);
    };
    const IO *isrc[kPre ? kItems : 1];
    if constexpr (kPre) {
#pragma unroll
        for (int k = 0; k < kItems; ++k) isrc[k] = item_src((tid + k * Cfg::kThreads) / kPieces);
    }
    // checked build: a copy source must lie inside u, delta, z, B or C
    auto src_ok = [&](const IO *src, int bytes) -> bool {
#ifdef SSM_CHECK
        auto in = [&](const IO *base, uint64_t total) {
            const uint64_t a = reinterpret_cast<uint64_t>(src), b0 = reinterpret_cast<uint64_t>(base);
            return base != nullptr && a >= b0 && a + (uint64_t)bytes <= b0 + total;
        };
        const bool ok = in(gU, kIoB) || in(gDelta, kIoB) || in(gZ, kIoB) || in(gB, kBcB) || in(gC, kBcB);
        if (!ok) set_status(kStatusCheck);
        return ok;
#else
        (void)src; (void)bytes;
        return true;
#endif
    };
    auto cp_chk = [&](uint32_t dst, const IO *src, int bytes) {
        if (src_ok(src, bytes) && SSM_CHK_SU(smem_u32(smem), dst, 16u)) cp_async16(dst, src, bytes);
    };
    auto issue_tile = [&](int j) {
        const uint32_t raw_s = smem_u32(raw_of(j));
        const int64_t toff = (int64_t)j * T;
        const int len = (int)min((int64_t)T, l_end - l_begin - toff);
        const int avail = max(0, min(kEpr, len - e0_me));
        if constexpr (kPre) {
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                if (isrc[k] != nullptr)
                    cp_chk(raw_s + idst0 + k * kItemStride, avail > 0 ? isrc[k] + toff : gU, avail * (int)sizeof(IO));
            }
        } else {
            for (int i = tid; i < kRows * kPieces; i += Cfg::kThreads) {
                const IO *src = item_src(i / kPieces);
                if (src != nullptr)
                    cp_chk(raw_s + (uint32_t)(((i / kPieces) * kRS + e0_me) * sizeof(IO)), avail > 0 ? src + toff : gU,
                           avail * (int)sizeof(IO));
            }
        }
        cp_async_commit();
    };

    // tile j's raw rows -> (dt, dt*u) per (channel, t), fp32 B, C as [t][n] and (aggregate
    // pass) the sums of dt over each item's steps. Items and their per-thread counts are
    // compile-time; a FULL tile has all T steps, so only the last tile checks its length.
    // Eight timesteps per item, or four when eight would leave threads without work.
    constexpr int kSI = Cfg::kSI;
    constexpr int kDXItems = kCh * (T / kSI);
    constexpr int kDXIter = (kDXItems + Cfg::kThreads - 1) / Cfg::kThreads;
    constexpr int kBCKinds = AGG ? 1 : 2;
    constexpr int kBCItems = kBCKinds * kNP * kPieces;
    constexpr int kBCIter = (kBCItems + Cfg::kThreads - 1) / Cfg::kThreads;
    auto convert = [&](int j, auto full_c) {
        constexpr bool FULL = decltype(full_c)::value;
        const IO *raw = raw_of(j);
        float4 *sDX = sDX0 + (size_t)(j & 1) * T * kPairs;
        float *sBC = sBC0 + (size_t)(j & 1) * T * 2 * kNP;
        const int len = FULL ? T : (int)min((int64_t)T, l_end - (l_begin + (int64_t)j * T));
#pragma unroll
        for (int it = 0; it < kDXIter; ++it) {
            const int i = tid + it * Cfg::kThreads;
            if (kDXItems % Cfg::kThreads != 0 && i >= kDXItems) break;
            const int cc = i % kCh, tq = (i / kCh) * kSI;
            float uu[kSI] = {}, dl[kSI] = {};
            if (SSM_CHK_S(smem, raw + (size_t)cc * kRS + tq, kSI * sizeof(IO)))
                load_steps<kSI>(raw + (size_t)cc * kRS + tq, uu);
            if (SSM_CHK_S(smem, raw + (size_t)(kCh + cc) * kRS + tq, kSI * sizeof(IO)))
                load_steps<kSI>(raw + (size_t)(kCh + cc) * kRS + tq, dl);
            if constexpr (CONV) {
                // u = SiLU(bias + sum_k w[k] x[t-3+k]) over the window x[tq-3 .. tq+kSI-1]; the
                // three steps before the tile come from this tile's row, the previous tile's
                // raw row (still resident) or, for the chunk's first tile, the halo
                float xw[kSI + 3];
#pragma unroll
                for (int e = 0; e < kSI; ++e) xw[3 + e] = uu[e];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    if (tq > 0) xw[i] = io_traits<IO>::to_f(ld_chk_s(smem, raw + (size_t)cc * kRS + tq - 3 + i));
                    else if (j > 0) xw[i] = io_traits<IO>::to_f(ld_chk_s(smem, raw_of(j - 1) + (size_t)cc * kRS + T - 3 + i));
                    else xw[i] = ld_chk_s(smem, sHalo + cc * 4 + i);
                }
                float *su = sSu0 + (size_t)(j & 1) * kCh * T + (size_t)cc * T + tq;
#pragma unroll
                for (int e = 0; e < kSI; ++e) {
                    float acc = ld_chk_s(smem, sCb + cc);
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc = fmaf(ld_chk_s(smem, sCw + cc * 4 + k), xw[e + k], acc);
                    uu[e] = silu_f(acc);
                    st_chk_s(smem, su + e, uu[e]);
                }
            }
            const bool ok = d0 + cc < p.Dm;
            const float bb = ld_chk_s(smem, sBias + cc);
            float dt[kSI];
#pragma unroll
            for (int e = 0; e < kSI; ++e) dt[e] = dl[e] + bb;
            if (p.softplus) {
#pragma unroll
                for (int e = 0; e < kSI; ++e) dt[e] = softplus_f(dt[e]);
            }
            float2 *dst = reinterpret_cast<float2 *>(sDX) + (size_t)tq * kPairs * 2 + cc;
            float ts = 0.0f, tm = 3.0e38f;
            (void)tm;
#pragma unroll
            for (int e = 0; e < kSI; ++e) {
                const bool in = ok && (FULL || tq + e < len);
                const float d = in ? dt[e] : 0.0f;
                ts += d;
                if constexpr (ZOH) tm = in ? fminf(tm, d) : tm;
                // (dt, dt*u) for the Euler step; (dt, u) for the zero-order hold, which forms
                // u*B*dt*phi or (a - 1)*u*B/A
                st_chk_s(smem, dst + (size_t)e * kPairs * 2, make_float2(d, in ? (ZOH ? uu[e] : d * uu[e]) : 0.0f));
            }
            if constexpr (AGG) st_chk_s(smem, sTS0 + (j & 1) * kDXItems + cc * (T / kSI) + tq / kSI, ts);
            if constexpr (ZOH) st_chk_s(smem, sTM0 + (j & 1) * kDXItems + cc * (T / kSI) + tq / kSI, tm);
        }
#pragma unroll
        for (int it = 0; it < kBCIter; ++it) {
            const int i = tid + it * Cfg::kThreads;
            if (kBCItems % Cfg::kThreads != 0 && i >= kBCItems) break;
            const int n = i % kNP, r = i / kNP, kind = r % kBCKinds, tq = (r / kBCKinds) * kEpr;
            float v[kEpr];
            if (n < N) {
                unpack16(ld_chk_s(smem, reinterpret_cast<const uint4 *>(raw + (size_t)(kRowB + kind * kNP + n) * kRS + tq)),
                         v, IO(0.0f));
            } else {
#pragma unroll
                for (int e = 0; e < kEpr; ++e) v[e] = 0.0f;
            }
            float *dst = sBC + (size_t)tq * 2 * kNP + kind * kNP + n;
#pragma unroll
            for (int e = 0; e < kEpr; ++e) st_chk_s(smem, dst + (size_t)e * 2 * kNP, v[e]);
        }
    };
    auto convert_tile = [&](int j) {
        if (l_end - (l_begin + (int64_t)j * T) >= T) convert(j, BoolC<true>{});
        else convert(j, BoolC<false>{});
    };

    float dsum[2] = {0.f, 0.f}, dsum_c[2] = {0.f, 0.f};   // compensated sums of dt (AGG)
    IO *gY = reinterpret_cast<IO *>(p.y);

    // coalesced store of tile j's staged y rows (16-byte pieces; element-wise on a ragged
    // tail); the thread's pieces are fixed, with their global destination at the chunk's
    // first step computed once (null past the last channel)
    constexpr int kYItems = (kCh * kPieces + Cfg::kThreads - 1) / Cfg::kThreads;
    IO *ydst[kYItems <= 2 ? kYItems : 1];
    if constexpr (kYItems <= 2) {
#pragma unroll
        for (int k = 0; k < kYItems; ++k) {
            const int i = tid + k * Cfg::kThreads, cc = i / kPieces;
            ydst[k] = (!AGG && i < kCh * kPieces && d0 + cc < p.Dm)
                          ? gY + ((b * p.Dm + d0 + cc) * p.ld + l_begin + e0_me) : nullptr;
        }
    }
    auto store_y = [&](int j) {
        const IO *ys = sYS0 + (size_t)(j & 1) * kCh * kRS;
        const int64_t toff = (int64_t)j * T;
        const int len = (int)min((int64_t)T, l_end - l_begin - toff);
        if (e0_me >= len) return;
        auto put = [&](IO *dst, const IO *src) {
            if (e0_me + kEpr <= len) {
                st_chk_g(gY, kIoB, reinterpret_cast<uint4 *>(dst), ld_chk_s(smem, reinterpret_cast<const uint4 *>(src)));
            } else {
                for (int e = 0; e < len - e0_me; ++e) st_chk_g(gY, kIoB, dst + e, ld_chk_s(smem, src + e));
            }
        };
        if constexpr (kYItems <= 2) {
#pragma unroll
            for (int k = 0; k < kYItems; ++k) {
                const int cc = (tid + k * Cfg::kThreads) / kPieces;
                if (ydst[k] != nullptr) put(ydst[k] + toff, ys + (size_t)cc * kRS + e0_me);
            }
        } else {
            for (int i = tid; i < kCh * kPieces; i += Cfg::kThreads) {
                const int cc = i / kPieces;
                if (d0 + cc >= p.Dm) continue;
                put(gY + ((b * p.Dm + d0 + cc) * p.ld + l_begin + e0_me) + toff, ys + (size_t)cc * kRS + e0_me);
            }
        }
    };

    for (int i = tid; i < kCh; i += Cfg::kThreads)
        st_chk_s(smem, sBias + i, (p.bias != nullptr && d0 + i < p.Dm) ? ld_chk_g(p.bias, kDB, p.bias + d0 + i) : 0.0f);
    if constexpr (CONV) {
        for (int i = tid; i < kCh; i += Cfg::kThreads) {
            const bool okc = d0 + i < p.Dm;
            for (int k = 0; k < 4; ++k) {   // taps right-aligned: the last tap meets x[t]
                const int kk = k - (4 - p.conv_k);
                st_chk_s(smem, sCw + i * 4 + k, (okc && kk >= 0)
                                                    ? ld_chk_g(p.conv_w, (uint64_t)p.Dm * p.conv_k * 4, p.conv_w + (d0 + i) * p.conv_k + kk)
                                                    : 0.0f);
            }
            st_chk_s(smem, sCb + i, (okc && p.conv_b != nullptr) ? ld_chk_g(p.conv_b, kDB, p.conv_b + d0 + i) : 0.0f);
            for (int k = 0; k < 3; ++k) {
                const int64_t s = l_begin - 3 + k;
                st_chk_s(smem, sHalo + i * 4 + k,
                         (okc && s >= 0) ? io_traits<IO>::to_f(ld_chk_g(gU, kIoB, gU + (b * p.Dm + d0 + i) * p.ld + s)) : 0.0f);
            }
        }
    }
    if (ntiles > 0) {
        issue_tile(0);
        cp_async_wait<0>();
        __syncthreads();
        convert_tile(0);
        if (ntiles > 1) issue_tile(1);
    }
    for (int j = 0; j < ntiles; ++j) {
        cp_async_wait<0>();   // tile j+1's raw rows (issued one tile ago)
        __syncthreads();      // conversion of tile j done; scan of tile j-1 done everywhere
        if (j + 2 < ntiles) issue_tile(j + 2);
        if (!AGG && j > 0) store_y(j - 1);
        if (j + 1 < ntiles) convert_tile(j + 1);

        const float4 *sDX = sDX0 + (size_t)(j & 1) * T * kPairs;
        const float *sBC = sBC0 + (size_t)(j & 1) * T * 2 * kNP;
        const IO *raw = raw_of(j);
        IO *ys = sYS0 + (size_t)(j & 1) * kCh * kRS;
        // per-lane bases: with the tile fully unrolled every step's offset is a constant
        const float4 *dxl = sDX + pr;
        const float *bcl = sBC + 4 * g;
        // y of the GP steps tb..tb+GP-1: the GP lanes of a pair exchange their partials (lane g
        // ends with timestep tb+g, both channels), add D*u, apply the gate and stage y for a
        // coalesced store after the next barrier (rows past the last channel are never stored)
        auto finish_group = [&](int tb, float (&yp)[2][GP]) {
            const int t = tb + g;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const float ysum = group_reduce_transpose<GP>(yp[ch], lane);
                const int cc = c0 + ch;
                const float uv = CONV ? ld_chk_s(smem, sSu0 + (size_t)(j & 1) * kCh * T + (size_t)cc * T + t)
                                      : io_traits<IO>::to_f(ld_chk_s(smem, raw + (size_t)cc * kRS + t));
                float yv = fmaf(Dd[ch], uv, ysum);
                if (has_z) yv *= silu_f(io_traits<IO>::to_f(ld_chk_s(smem, raw + (size_t)(2 * kCh + cc) * kRS + t)));
                if (SSM_CHK_S(smem, ys + (size_t)cc * kRS + t, sizeof(IO))) store_io(ys + (size_t)cc * kRS + t, yv);
            }
        };
        auto scan_tile = [&](auto st_c, auto zf_c) {
            constexpr bool ST = decltype(st_c)::value;
            constexpr bool zfast = decltype(zf_c)::value;   // zero-order hold: no polynomial branch
            (void)zfast;
#pragma unroll((AGG && !ZOH && !CONV) ? T / GP : kPairTileUnroll)
            for (int tb = 0; tb < T; tb += GP) {
                float yp[2][GP];
#pragma unroll
                for (int s = 0; s < GP; ++s) {
                    const int t = tb + s;
                    const float4 dx = ld_chk_s(smem, dxl + t * kPairs);
                    const float2 dd[2] = {make_float2(dx.x, dx.x), make_float2(dx.z, dx.z)};
                    const float2 xx[2] = {make_float2(dx.y, dx.y), make_float2(dx.w, dx.w)};
                    // structured A: r = exp(dt*A[d, 0]) and (r^2, r^2) per channel
                    float r[2] = {1.0f, 1.0f};
                    float2 r2[2] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
                    if constexpr (ST) {
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch) {
                            r[ch] = ex2(dd[ch].x * Ap0[ch]);
                            r2[ch] = __fmul2_rn(make_float2(r[ch], r[ch]), make_float2(r[ch], r[ch]));
                        }
                    }
                    float2 ya[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int q = 0; q < kQN; ++q) {
                        const float4 bq = ld_chk_s(smem, reinterpret_cast<const float4 *>(bcl + t * 2 * kNP + 4 * GP * q));
                        float4 cq = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (!AGG) cq = ld_chk_s(smem, reinterpret_cast<const float4 *>(bcl + t * 2 * kNP + kNP + 4 * GP * q));
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch) {
                            float2 e0, e1, a0, a1;
                            if constexpr (ST) {
                                const float e = ex2(dd[ch].x * Ap[ch][q][0].x);   // first state of the quad
                                a0 = make_float2(e, e * r[ch]);
                                a1 = __fmul2_rn(a0, r2[ch]);
                                if constexpr (ZOH) {
                                    e0 = __fmul2_rn(dd[ch], Ap[ch][q][0]);
                                    e1 = __fmul2_rn(dd[ch], Ap[ch][q][1]);
                                }
                            } else {
                                e0 = __fmul2_rn(dd[ch], Ap[ch][q][0]);
                                e1 = __fmul2_rn(dd[ch], Ap[ch][q][1]);
                                a0 = make_float2(ex2(e0.x), ex2(e0.y));
                                a1 = make_float2(ex2(e1.x), ex2(e1.y));
                            }
                            float2 w0, w1;
                            if constexpr (ZOH) {
                                // xx holds u here (see the conversion)
                                const float2 ub0 = __fmul2_rn(xx[ch], make_float2(bq.x, bq.y));
                                const float2 ub1 = __fmul2_rn(xx[ch], make_float2(bq.z, bq.w));
                                if constexpr (zfast) {
                                    // h = a*h + (a - 1)*K = a*(h + K) - K with K = u*B/A, from
                                    // nK = -K: one subtraction and one FMA (the state is updated
                                    // here; w stays unused)
                                    const float2 nk0 = __fmul2_rn(ub0, iA[ch][q][0]);
                                    const float2 nk1 = __fmul2_rn(ub1, iA[ch][q][1]);
                                    h[ch][q][0] = __ffma2_rn(a0, fsub2_rn(h[ch][q][0], nk0), nk0);
                                    h[ch][q][1] = __ffma2_rn(a1, fsub2_rn(h[ch][q][1], nk1), nk1);
                                } else {
                                    w0 = __fmul2_rn(ub0, zoh_psi2(e0, a0, dd[ch], iA[ch][q][0]));
                                    w1 = __fmul2_rn(ub1, zoh_psi2(e1, a1, dd[ch], iA[ch][q][1]));
                                }
                            } else {
                                w0 = __fmul2_rn(xx[ch], make_float2(bq.x, bq.y));
                                w1 = __fmul2_rn(xx[ch], make_float2(bq.z, bq.w));
                            }
                            if (!(ZOH && zfast)) {
                                h[ch][q][0] = __ffma2_rn(a0, h[ch][q][0], w0);
                                h[ch][q][1] = __ffma2_rn(a1, h[ch][q][1], w1);
                            }
                            if (!AGG) {
                                ya[ch] = __ffma2_rn(make_float2(cq.x, cq.y), h[ch][q][0], ya[ch]);
                                ya[ch] = __ffma2_rn(make_float2(cq.z, cq.w), h[ch][q][1], ya[ch]);
                            }
                        }
                    }
                    if (!AGG) {
                        yp[0][s] = ya[0].x + ya[0].y;
                        yp[1][s] = ya[1].x + ya[1].y;
                    }
                }
                if (!AGG) finish_group(tb, yp);
            }
        };
        // zero-order hold: the one-FMA form for the whole tile when |dt*A| stays above the
        // threshold at every step for every state of the warp's channels (a warp vote on the
        // tile's smallest dt per channel, recorded by the conversion)
        bool zf = false;
        if constexpr (ZOH) {
            const float *tm = sTM0 + (j & 1) * kDXItems;
            bool ok = true;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                float m = 3.0e38f;
#pragma unroll
                for (int r = 0; r < T / kSI; ++r) m = fminf(m, tm[(c0 + ch) * (T / kSI) + r]);
                ok = ok && (!cv[ch] || m * zmin[ch] >= ZohFast<IO>::kMinXl2);
            }
            zf = __all_sync(0xffffffffu, ok);
        }
        if constexpr (ZOH) {
            // (the structured-A power form keeps the general zero-order-hold form: two tile
            // bodies instead of four keep the kernel's code within the instruction cache)
            if (st) scan_tile(BoolC<true>{}, BoolC<false>{});
            else if (zf) scan_tile(BoolC<false>{}, BoolC<true>{});
            else scan_tile(BoolC<false>{}, BoolC<false>{});
        } else {
            if (st) scan_tile(BoolC<true>{}, BoolC<false>{});
            else scan_tile(BoolC<false>{}, BoolC<false>{});
        }
        if (AGG) {
            // this tile's sum of dt per channel, from the conversion's per-item sums
            const float *ts = sTS0 + (j & 1) * kDXItems;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                float tsum = 0.0f;
#pragma unroll
                for (int r = 0; r < T / kSI; ++r) tsum += ts[(c0 + ch) * (T / kSI) + r];
                const float yk = tsum - dsum_c[ch];
                const float tk = dsum[ch] + yk;
                dsum_c[ch] = (tk - dsum[ch]) - yk;
                dsum[ch] = tk;
            }
        }
    }
    cp_async_wait<0>();
    if (!AGG && ntiles > 0) {
        __syncthreads();
        store_y(ntiles - 1);
    }

#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        if (!cv[ch]) continue;
        const int64_t bd = b * p.Dm + dch[ch];
        if (AGG) {
            float *dst = p.agg_h + ((int64_t)k * BD + bd) * p.npad;
#pragma unroll
            for (int q = 0; q < kQN; ++q)
                st_chk_g(p.agg_h, kCarryB, reinterpret_cast<float4 *>(dst + 4 * (GP * q + g)),
                         make_float4(h[ch][q][0].x, h[ch][q][0].y, h[ch][q][1].x, h[ch][q][1].y));
            if (g == 0) st_chk_g(p.agg_s, kSumB, p.agg_s + (int64_t)k * BD + bd, dsum[ch]);
        } else if (p.last_state != nullptr && k == p.nchunks - 1) {
            float *dst = p.last_state + bd * p.N;
#pragma unroll
            for (int q = 0; q < kQN; ++q) {
                const float v[4] = {h[ch][q][0].x, h[ch][q][0].y, h[ch][q][1].x, h[ch][q][1].y};
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int n = 4 * (GP * q + g) + jj;
                    if (n < N) st_chk_g(p.last_state, (uint64_t)BD * p.N * 4, dst + n, v[jj]);
                }
            }
        }
    }
}

}  // namespace ssm
