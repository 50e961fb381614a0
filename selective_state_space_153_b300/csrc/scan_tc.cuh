// Selective scan, persistent kernel with the sequence split across warps and a tensor-memory
// replay (sm_100 family: TMA, mbarriers, tcgen05 tensor memory).
//
// The computation is the section 3.2 loop of "From RNN to Mamba" (lmnt.cn):
//   h = exp(dt*A)*h + dt*B_t*u_t,  y_t = sum_n C_t*h + D*u_t, gated by SiLU(z_t).
// It is a composition of affine maps h -> a*h + w (section 2.2 there; section 3.4 of the
// jsqmd.com page), so a stretch of timesteps can be run from h = 0 and corrected afterwards:
// with P = prod(a) over the stretch and e its end state from zero, the true end state is
// P*h_in + e.
//
// Work decomposition
//   * group  = CPW = 32/G consecutive channels of one batch row (a warp covers one group:
//              lane = (channel c, state group g), 16 states per lane, interleaved n).
//   * tile   = T = W*K timesteps; warp w owns steps [w*K, w*K+K) of every tile.
//   * unit   = one group x one segment of consecutive tiles. A CTA (one per SM, persistent)
//              takes units in segment-major ticket order; a unit needs the final state of
//              the same group's previous segment, published by whichever CTA ran it. With
//              more groups than CTAs that unit was dispatched a whole round earlier, so the
//              state is normally ready; the wait is bounded and reports SSM_ERR_TIMEOUT.
// Inside a tile (carry h known on entry):
//   warp 0      runs its K steps exactly from the carry (1 ex2 + 4 FP32 per element) and
//               writes its end state;
//   warps 1..W-2 run their steps from zero, keep a = exp2(dt*A*log2e) and w = dt*B*u in
//               tensor memory (tcgen05.st), and publish P = exp2(A*log2e*sum dt) and their
//               end state from zero;
//   warp W-1    keeps a, w in tensor memory only;
//   then every warp w >= 1 forms its exact incoming state from warp 0's end state and the
//   aggregates of warps 1..w-1, replays h = a*h + w from tensor memory (tcgen05.ld) and
//   reads out y. Warp W-1's final state is the next tile's carry. Only the middle warps pay
//   the extra FFMA of the local run; no exponential is recomputed.
// Data movement: u, delta (and z) tiles [CPW x T] by 3-D TMA tensor loads (zero fill beyond
// the tensor), B/C by one 1-D bulk copy per tile from a prepared fp32 [t][B|C][n] array,
// double-buffered on mbarriers; y tiles by TMA tensor stores (clipped at the tensor edge).
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ssm {

constexpr int kTcWarps = 8;   // W
constexpr int kTcK = 8;       // steps per warp per tile
constexpr int kTcT = kTcWarps * kTcK;

struct TcParams {
    CUtensorMap map_u, map_delta, map_z, map_y;   // 3-D [Bt][Dm][L] io-dtype tensors, box [1][CPW][T]
    CUtensorMap map_y8;                            // y with a box of 8 steps (per-warp stores)
    const float *bc;                               // [Bt][Lp][2*NP] fp32: B row then C row
    const float *A, *D, *bias;
    float *last_state;
    int *ctrl;                                     // [0] ticket, [1 + group] published segments
    float *carry;                                  // [NG][2][4][32][4]
    int64_t Bt, Dm, L, N, Lp;
    int NG, groups_per_b, nseg, seg_tiles, ntiles;
    int has_z, softplus;
    uint32_t spin_limit;
    int force_timeout;                             // test hook: wait for a flag nothing sets
    int cpw, np;                                   // geometry the host planned (checked on entry)
};

// Status recorded when a launch's planned geometry does not match the kernel's
constexpr int kStatusBadGeometry = 5;   // SSM_ERR_UNSUPPORTED

template <typename IO, int G>
struct TcCfg {
    static constexpr int W = kTcWarps, K = kTcK, T = kTcT;
    static constexpr int CPW = 32 / G, NP = 16 * G, BCROW = 2 * NP;
    static constexpr size_t RAW_ARR = (size_t)CPW * T * sizeof(IO);
    static constexpr size_t up128(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr size_t OFF_RAW = 0;                                    // [2][3][CPW][T] io
    static constexpr size_t OFF_BC = up128(OFF_RAW + 6 * RAW_ARR);          // [2][T][BCROW] f32
    static constexpr size_t OFF_Y = up128(OFF_BC + 2ull * T * BCROW * 4);   // [2][CPW][T] io
    static constexpr size_t OFF_DX = up128(OFF_Y + 2 * RAW_ARR);            // [W][K][CPW] float2
    static constexpr size_t OFF_AGG = up128(OFF_DX + (size_t)W * K * CPW * 8);  // [W][8][32] float4
    static constexpr size_t OFF_CARRY = OFF_AGG + (size_t)W * 8 * 32 * 16;      // [4][32] float4
    static constexpr size_t OFF_MISC = OFF_CARRY + 4 * 32 * 16;                 // mbar[2], ticket, tmem
    static constexpr size_t BYTES = OFF_MISC + 64;
    // one CTA per SM: the kernel owns all 512 tensor-memory columns
    static constexpr size_t SMEM = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "G");
    // every shared-memory buffer a TMA tensor copy reads or writes starts on 128 bytes
    static_assert(RAW_ARR % 128 == 0 && OFF_RAW % 128 == 0 && OFF_Y % 128 == 0, "TMA smem alignment");
};

// B, C [Bt][N][L] io -> bc [Bt][Lp][2*NP] fp32 (zero beyond N and L), 32 timesteps per block.
template <typename IO>
__global__ void __launch_bounds__(256) bc_prep_kernel(const IO *__restrict__ B, const IO *__restrict__ C,
                                                      float *__restrict__ bc, int64_t N, int64_t L, int64_t Lp,
                                                      int NP) {
    extern __shared__ float tile[];   // [2][NP][33]
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * 32;
    for (int i = threadIdx.x; i < 2 * NP * 32; i += blockDim.x) {
        const int arr = i / (NP * 32), n = (i / 32) % NP, tt = i % 32;
        const int64_t t = t0 + tt;
        float v = 0.0f;
        if (n < N && t < L) v = io_traits<IO>::to_f((arr ? C : B)[(b * N + n) * L + t]);
        tile[(arr * NP + n) * 33 + tt] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * 2 * NP; i += blockDim.x) {
        const int tt = i / (2 * NP), col = i % (2 * NP);
        const int arr = col / NP, n = col % NP;
        bc[((b * Lp) + t0 + tt) * (2 * NP) + col] = tile[(arr * NP + n) * 33 + tt];
    }
}

template <typename IO, int G>
__global__ void __launch_bounds__(kTcWarps * 32, 1) scan_tc_kernel(const __grid_constant__ TcParams p) {
    using Cfg = TcCfg<IO, G>;
    constexpr int W = Cfg::W, K = Cfg::K, T = Cfg::T, CPW = Cfg::CPW, NP = Cfg::NP, BCROW = Cfg::BCROW;
    extern __shared__ __align__(1024) unsigned char smem[];
    IO *raw = reinterpret_cast<IO *>(smem + Cfg::OFF_RAW);         // [buf][arr][CPW][T]
    float *sbc = reinterpret_cast<float *>(smem + Cfg::OFF_BC);     // [buf][T][BCROW]
    IO *ybuf = reinterpret_cast<IO *>(smem + Cfg::OFF_Y);           // [buf][CPW][T]
    float2 *sdx = reinterpret_cast<float2 *>(smem + Cfg::OFF_DX);   // [W][K][CPW]
    float4 *agg = reinterpret_cast<float4 *>(smem + Cfg::OFF_AGG);  // [W][8][32]
    float4 *scarry = reinterpret_cast<float4 *>(smem + Cfg::OFF_CARRY);  // [4][32]
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_MISC);
    int *s_ticket = reinterpret_cast<int *>(smem + Cfg::OFF_MISC + 16);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC + 20);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane / G, g = lane % G;
    constexpr size_t ARR = (size_t)CPW * T;
    if (p.cpw != CPW || p.np != NP) {   // tile sizes of the TMA boxes would not match expect_tx
        if (tid == 0) set_status(kStatusBadGeometry);
        return;
    }

    if (warp == 0) tmem_alloc(s_tmem, 512);
    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t my_tmem = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 256);
    uint32_t phase[2] = {0u, 0u};
    int jt = 0;
    const int total_units = p.NG * p.nseg;
    const uint32_t tile_bytes = (uint32_t)((p.has_z ? 3 : 2) * ARR * sizeof(IO) + (size_t)T * BCROW * 4);

    for (;;) {
        if (tid == 0) *s_ticket = atomicAdd(&p.ctrl[0], 1);
        __syncthreads();
        const int ticket = *s_ticket;
        __syncthreads();
        if (ticket >= total_units) break;
        const int s = ticket / p.NG, gi = ticket % p.NG;
        const int64_t b = gi / p.groups_per_b;
        const int64_t d0 = (int64_t)(gi % p.groups_per_b) * CPW;
        const int j0 = s * p.seg_tiles, j1 = min(j0 + p.seg_tiles, p.ntiles);
        const int64_t d = d0 + c;
        const bool cvalid = d < p.Dm;
        const int N = (int)p.N;

        auto issue = [&](int j, int buf) {
            IO *r = raw + (size_t)buf * 3 * ARR;
            mbar_arrive_expect_tx(&mbar[buf], tile_bytes);
            tma_load_3d(r, &p.map_u, j * T, (int)d0, (int)b, &mbar[buf]);
            tma_load_3d(r + ARR, &p.map_delta, j * T, (int)d0, (int)b, &mbar[buf]);
            if (p.has_z) tma_load_3d(r + 2 * ARR, &p.map_z, j * T, (int)d0, (int)b, &mbar[buf]);
            bulk_g2s(sbc + (size_t)buf * T * BCROW, p.bc + ((int64_t)b * p.Lp + (int64_t)j * T) * BCROW,
                     (uint32_t)(T * BCROW * 4), &mbar[buf]);
        };
        if (tid == 0) issue(j0, jt & 1);

        // per-lane constants of this unit
        float Ap[16];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int n = 4 * (G * q + g) + jj;
                Ap[4 * q + jj] = (cvalid && n < N) ? p.A[d * p.N + n] * kLog2e : 0.0f;
            }
        const float Dd = (p.D != nullptr && cvalid) ? p.D[d] : 0.0f;

        float h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = 0.0f;
        if (warp == 0 && s > 0) {
            if (lane == 0) {
                if (p.force_timeout) wait_flag_geq(&p.ctrl[1 + gi], 0x7fffffff, p.spin_limit);
                else wait_flag_geq(&p.ctrl[1 + gi], s, p.spin_limit);
            }
            __syncwarp();
            const float4 *src = reinterpret_cast<const float4 *>(p.carry + ((int64_t)gi * 2 + ((s - 1) & 1)) * 512);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldcg(src + q * 32 + lane);
                h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
            }
        }

        for (int j = j0; j < j1; ++j, ++jt) {
            const int buf = jt & 1;
            if (tid == 0 && j + 1 < j1) issue(j + 1, buf ^ 1);
            mbar_wait(&mbar[buf], phase[buf]);
            phase[buf] ^= 1u;
            const IO *ru = raw + (size_t)buf * 3 * ARR;
            const IO *rdl = ru + ARR;
            const IO *rz = ru + 2 * ARR;
            const float *bct = sbc + (size_t)buf * T * BCROW;
            IO *yb = ybuf + (size_t)buf * ARR;
            const int64_t t0 = (int64_t)j * T;

            // (1) dt and dt*u of this warp's steps
            float2 *mydx = sdx + (size_t)warp * K * CPW;
            for (int i = lane; i < CPW * K; i += 32) {
                const int cc = i % CPW, kk = i / CPW, tt = warp * K + kk;
                float dt = 0.0f, x = 0.0f;
                if (t0 + tt < p.L && d0 + cc < p.Dm) {
                    const float uu = io_traits<IO>::to_f(ru[cc * T + tt]);
                    dt = io_traits<IO>::to_f(rdl[cc * T + tt]) + (p.bias != nullptr ? p.bias[d0 + cc] : 0.0f);
                    if (p.softplus) dt = softplus_f(dt);
                    x = dt * uu;
                }
                mydx[kk * CPW + cc] = make_float2(dt, x);
            }
            __syncwarp();

            // y epilogue for one (channel, step) owned by this lane after the group reduction
            auto emit = [&](int tt, float ys) {
                float yv = 0.0f;
                if (cvalid && t0 + tt < p.L) {
                    yv = fmaf(Dd, io_traits<IO>::to_f(ru[c * T + tt]), ys);
                    if (p.has_z) yv *= silu_f(io_traits<IO>::to_f(rz[c * T + tt]));
                }
                store_io(yb + c * T + tt, yv);
            };

            if (warp == 0) {
                // exact run of steps [0, K) from the carry
                float ypart[G];
#pragma unroll
                for (int kk = 0; kk < K; ++kk) {
                    const float2 dx = mydx[kk * CPW + c];
                    const float *row = bct + (size_t)kk * BCROW;
                    float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 bq = *reinterpret_cast<const float4 *>(row + 4 * (G * q + g));
                        const float4 cq = *reinterpret_cast<const float4 *>(row + NP + 4 * (G * q + g));
                        const float2 dd = make_float2(dx.x, dx.x), xx = make_float2(dx.y, dx.y);
                        float2 e0 = __fmul2_rn(dd, make_float2(Ap[4 * q], Ap[4 * q + 1]));
                        float2 e1 = __fmul2_rn(dd, make_float2(Ap[4 * q + 2], Ap[4 * q + 3]));
                        const float2 a0 = make_float2(ex2(e0.x), ex2(e0.y));
                        const float2 a1 = make_float2(ex2(e1.x), ex2(e1.y));
                        const float2 w0 = __fmul2_rn(xx, make_float2(bq.x, bq.y));
                        const float2 w1 = __fmul2_rn(xx, make_float2(bq.z, bq.w));
                        const float2 h0 = __ffma2_rn(a0, make_float2(h[4 * q], h[4 * q + 1]), w0);
                        const float2 h1 = __ffma2_rn(a1, make_float2(h[4 * q + 2], h[4 * q + 3]), w1);
                        h[4 * q] = h0.x; h[4 * q + 1] = h0.y; h[4 * q + 2] = h1.x; h[4 * q + 3] = h1.y;
                        y2 = __ffma2_rn(make_float2(cq.x, cq.y), h0, y2);
                        y2 = __ffma2_rn(make_float2(cq.z, cq.w), h1, y2);
                    }
                    ypart[kk % G] = y2.x + y2.y;
                    if (kk % G == G - 1) {
                        const float ys = group_reduce_transpose<G>(ypart, lane);
                        emit(kk - (G - 1) + g, ys);
                    }
                }
                float4 *dst = agg;   // slot 4..7 of warp 0 = end state
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[(4 + q) * 32 + lane] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            } else {
                // run from zero; keep a, w in tensor memory
                const bool mid = warp < W - 1;
                float hl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) hl[i] = 0.0f;
                float sdt = 0.0f;
#pragma unroll
                for (int kk = 0; kk < K; ++kk) {
                    const float2 dx = mydx[kk * CPW + c];
                    sdt += dx.x;
                    const float *row = bct + (size_t)(warp * K + kk) * BCROW;
                    float r[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 bq = *reinterpret_cast<const float4 *>(row + 4 * (G * q + g));
                        const float2 dd = make_float2(dx.x, dx.x), xx = make_float2(dx.y, dx.y);
                        float2 e0 = __fmul2_rn(dd, make_float2(Ap[4 * q], Ap[4 * q + 1]));
                        float2 e1 = __fmul2_rn(dd, make_float2(Ap[4 * q + 2], Ap[4 * q + 3]));
                        const float2 a0 = make_float2(ex2(e0.x), ex2(e0.y));
                        const float2 a1 = make_float2(ex2(e1.x), ex2(e1.y));
                        const float2 w0 = __fmul2_rn(xx, make_float2(bq.x, bq.y));
                        const float2 w1 = __fmul2_rn(xx, make_float2(bq.z, bq.w));
                        r[4 * q] = a0.x; r[4 * q + 1] = a0.y; r[4 * q + 2] = a1.x; r[4 * q + 3] = a1.y;
                        r[16 + 4 * q] = w0.x; r[16 + 4 * q + 1] = w0.y; r[16 + 4 * q + 2] = w1.x; r[16 + 4 * q + 3] = w1.y;
                        if (mid) {
                            const float2 h0 = __ffma2_rn(a0, make_float2(hl[4 * q], hl[4 * q + 1]), w0);
                            const float2 h1 = __ffma2_rn(a1, make_float2(hl[4 * q + 2], hl[4 * q + 3]), w1);
                            hl[4 * q] = h0.x; hl[4 * q + 1] = h0.y; hl[4 * q + 2] = h1.x; hl[4 * q + 3] = h1.y;
                        }
                    }
                    tmem_st32(my_tmem + (uint32_t)(32 * kk), r);
                }
                if (mid) {
                    float4 *dst = agg + (size_t)warp * 8 * 32;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        dst[q * 32 + lane] = make_float4(ex2(Ap[4 * q] * sdt), ex2(Ap[4 * q + 1] * sdt),
                                                         ex2(Ap[4 * q + 2] * sdt), ex2(Ap[4 * q + 3] * sdt));
                        dst[(4 + q) * 32 + lane] = make_float4(hl[4 * q], hl[4 * q + 1], hl[4 * q + 2], hl[4 * q + 3]);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();   // end states and aggregates visible
            tc_fence_after();

            if (warp != 0) {
                // exact incoming state: warp 0's end state through the aggregates of 1..warp-1
                float hin[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = agg[(4 + q) * 32 + lane];
                    hin[4 * q] = v.x; hin[4 * q + 1] = v.y; hin[4 * q + 2] = v.z; hin[4 * q + 3] = v.w;
                }
                for (int v = 1; v < warp; ++v) {
                    const float4 *src = agg + (size_t)v * 8 * 32;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 P = src[q * 32 + lane], e = src[(4 + q) * 32 + lane];
                        const float2 r0 = __ffma2_rn(make_float2(P.x, P.y), make_float2(hin[4 * q], hin[4 * q + 1]), make_float2(e.x, e.y));
                        const float2 r1 = __ffma2_rn(make_float2(P.z, P.w), make_float2(hin[4 * q + 2], hin[4 * q + 3]), make_float2(e.z, e.w));
                        hin[4 * q] = r0.x; hin[4 * q + 1] = r0.y; hin[4 * q + 2] = r1.x; hin[4 * q + 3] = r1.y;
                    }
                }
                // replay from tensor memory
                float ra[32], rb[32];
                float ypart[G];
                tmem_ld32(my_tmem, ra);
                tmem_wait_ld(ra);
                auto step = [&](int kk, const float(&cur)[32]) {
                    const float *row = bct + (size_t)(warp * K + kk) * BCROW;
                    float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 cq = *reinterpret_cast<const float4 *>(row + NP + 4 * (G * q + g));
                        const float2 h0 = __ffma2_rn(make_float2(cur[4 * q], cur[4 * q + 1]),
                                                     make_float2(hin[4 * q], hin[4 * q + 1]),
                                                     make_float2(cur[16 + 4 * q], cur[16 + 4 * q + 1]));
                        const float2 h1 = __ffma2_rn(make_float2(cur[4 * q + 2], cur[4 * q + 3]),
                                                     make_float2(hin[4 * q + 2], hin[4 * q + 3]),
                                                     make_float2(cur[16 + 4 * q + 2], cur[16 + 4 * q + 3]));
                        hin[4 * q] = h0.x; hin[4 * q + 1] = h0.y; hin[4 * q + 2] = h1.x; hin[4 * q + 3] = h1.y;
                        y2 = __ffma2_rn(make_float2(cq.x, cq.y), h0, y2);
                        y2 = __ffma2_rn(make_float2(cq.z, cq.w), h1, y2);
                    }
                    ypart[kk % G] = y2.x + y2.y;
                    if (kk % G == G - 1) {
                        const float ys = group_reduce_transpose<G>(ypart, lane);
                        emit(warp * K + kk - (G - 1) + g, ys);
                    }
                };
#pragma unroll
                for (int kk = 0; kk < K; kk += 2) {
                    tmem_ld32(my_tmem + (uint32_t)(32 * (kk + 1)), rb);
                    step(kk, ra);
                    tmem_wait_ld(rb);
                    if (kk + 2 < K) tmem_ld32(my_tmem + (uint32_t)(32 * (kk + 2)), ra);
                    step(kk + 1, rb);
                    if (kk + 2 < K) tmem_wait_ld(ra);
                }
                if (warp == W - 1) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        scarry[q * 32 + lane] = make_float4(hin[4 * q], hin[4 * q + 1], hin[4 * q + 2], hin[4 * q + 3]);
                }
            } else if (tid == 0) {
                bulk_wait_read0();   // the previous tile's y store has finished reading its buffer
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();   // y tile and carry complete
            tc_fence_after();
            if (warp == 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = scarry[q * 32 + lane];
                    h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
                }
            }
            if (tid == 0) {
                tma_store_3d(&p.map_y, yb, (int)t0, (int)d0, (int)b);
                bulk_commit();
            }
        }

        // unit end: publish the segment's final state, or write the final state of the scan
        if (warp == 0) {
            if (s + 1 < p.nseg) {
                float4 *dst = reinterpret_cast<float4 *>(p.carry + ((int64_t)gi * 2 + (s & 1)) * 512);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    __stcg(dst + q * 32 + lane, make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]));
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release(&p.ctrl[1 + gi], s + 1);
            } else if (p.last_state != nullptr && cvalid) {
                float *dst = p.last_state + (b * p.Dm + d) * p.N;
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int n = 4 * (G * q + g) + jj;
                        if (n < N) dst[n] = h[4 * q + jj];
                    }
            }
        }
    }
    if (tid == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace ssm
