// Selective scan, persistent and warp-pipelined (sm_100 family: TMA, mbarriers, tensor memory).
//
// The computation is the section 3.2 loop of "From RNN to Mamba" (lmnt.cn):
//   h = exp(dt*A)*h + dt*B_t*u_t,  y_t = sum_n C_t*h + D*u_t, gated by SiLU(z_t),
// split along the sequence through the affine-map composition of its section 2.2 (and of
// section 3.4 of the jsqmd.com page): a stretch run from h = 0 with P = prod exp(dt*A) and end
// state e maps an incoming state h_in to P*h_in + e.
//
// Lanes. A lane owns TWO channels (c0 = 2p, c1 = 2p+1) and 8 states of each,
// n = 4*(GP*q + g) + j (q < 2, j < 4), GP = padded states / 8 lanes per channel pair. Every
// B/C value a lane reads from shared memory serves both channels, which halves the shared-
// memory bytes per element (shared-memory delivery, not arithmetic, would otherwise cap the
// scan at half the exp2 rate). A warp covers CPW = 64/GP channels; the GP lanes of a pair
// combine y with a transposed butterfly.
//
// Work. Units = (CPW-channel group, segment of tiles), taken by persistent CTAs (one per SM)
// in segment-major ticket order; a unit starts from the previous segment's final state
// (global carry ring, release/acquire flag, bounded wait). A tile is 64 steps; warp w of 8
// owns steps [8w, 8w+8). All warps run the same pipeline:
//   * local pass of tile j+1: a = exp2(dt*A*log2e), w = dt*u*B into tensor memory
//     (tcgen05.st), running end state from zero, P = exp2(A*log2e*sum dt) -> aggregate;
//   * replay of tile j from tensor memory (tcgen05.ld) from the exact incoming state
//     carry(j) composed with the aggregates of warps < w, with the readout y = C.h;
//   the two are fused step by step (tile j+1's local step kk overwrites the columns that
//   tile j's replay step kk has just read), so MUFU and FMA work share one stream.
//   Warp 0 also composes carry(j+1) = carry(j) through all eight aggregates of tile j and
//   feeds the TMA input ring (u, delta, z tiles by 3-D tensor loads; B/C as one bulk copy of
//   a prepared fp32 [t][B row | C row] tile); y leaves per warp by TMA tensor stores.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"
#include "scan_tc.cuh"

namespace ssm {

constexpr int kTpWarps = 8;
constexpr int kTpK = 8;
constexpr int kTpT = kTpWarps * kTpK;   // 64 steps per tile

// shared-memory bytes of the layout of TpCfg for S input stages
template <typename IO, int GP>
constexpr size_t tp_bytes(int S) {
    constexpr int W = kTpWarps, K = kTpK, T = kTpT, CPW = 64 / GP, BCROW = 16 * GP;
    auto up = [](size_t x) { return (x + 127) / 128 * 128; };
    const size_t raw = (size_t)CPW * T * sizeof(IO);
    size_t o = up((size_t)S * 3 * raw);
    o = up(o + (size_t)S * T * BCROW * 4);
    o = up(o + (size_t)W * 2 * K * CPW * 8);
    o = o + (size_t)2 * W * 8 * 32 * 16;
    o = up(o + (size_t)W * 2 * up((size_t)CPW * K * sizeof(IO)));
    o = o + (size_t)3 * 4 * 32 * 16;
    return o + 16 * 8 + 64;
}
constexpr size_t kSmemLimit = 232448;   // opt-in shared memory per CTA on sm_100-family parts

template <typename IO, int GP>
struct TpCfg {
    static_assert(GP == 1 || GP == 2 || GP == 4 || GP == 8, "8-state groups per channel pair");
    // input stages: as many as fit (the producer runs two tiles ahead)
    static constexpr int S = tp_bytes<IO, GP>(4) <= kSmemLimit ? 4 : (tp_bytes<IO, GP>(3) <= kSmemLimit ? 3 : 2);
    static constexpr int W = kTpWarps, K = kTpK, T = kTpT;
    static constexpr int PAIRS = 32 / GP, CPW = 2 * PAIRS, NP = 8 * GP, BCROW = 2 * NP;
    static constexpr size_t RAW_ARR = (size_t)CPW * T * sizeof(IO);
    static constexpr size_t up128(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr size_t OFF_RAW = 0;                                           // [S][3][CPW][T] io
    static constexpr size_t OFF_BC = up128((size_t)S * 3 * RAW_ARR);               // [S][T][BCROW] f32
    static constexpr size_t OFF_DX = up128(OFF_BC + (size_t)S * T * BCROW * 4);    // [W][2][K][CPW] float2
    static constexpr size_t OFF_AGG = up128(OFF_DX + (size_t)W * 2 * K * CPW * 8); // [2][W][8][32] float4
    static constexpr size_t Y_SLOT = up128((size_t)CPW * K * sizeof(IO));          // TMA store source
    static constexpr size_t OFF_Y = OFF_AGG + (size_t)2 * W * 8 * 32 * 16;         // [W][2] slots [CPW][K] io
    static constexpr size_t OFF_CARRY = up128(OFF_Y + (size_t)W * 2 * Y_SLOT);     // [3][4][32] float4
    static constexpr size_t OFF_BAR = OFF_CARRY + (size_t)3 * 4 * 32 * 16;
    static constexpr size_t OFF_MISC = OFF_BAR + 16 * 8;
    static constexpr size_t BYTES = OFF_MISC + 64;
    static constexpr size_t SMEM = BYTES > 120 * 1024 ? BYTES : 120 * 1024;        // one CTA per SM
    static_assert(BYTES == tp_bytes<IO, GP>(S) && BYTES <= kSmemLimit, "shared-memory layout");
    static_assert(RAW_ARR % 128 == 0 && OFF_Y % 128 == 0 && Y_SLOT % 128 == 0, "TMA smem alignment");
    static_assert(OFF_BC % 16 == 0 && ((size_t)T * BCROW * 4) % 16 == 0, "bulk copy alignment");
};

template <typename IO, int GP>
__global__ void __launch_bounds__(kTpWarps * 32, 1) scan_tp_kernel(const __grid_constant__ TcParams p) {
    using Cfg = TpCfg<IO, GP>;
    constexpr int W = Cfg::W, K = Cfg::K, T = Cfg::T, S = Cfg::S, CPW = Cfg::CPW, NP = Cfg::NP, BCROW = Cfg::BCROW;
    constexpr size_t ARR = (size_t)CPW * T;
    extern __shared__ __align__(1024) unsigned char smem[];
    IO *raw = reinterpret_cast<IO *>(smem + Cfg::OFF_RAW);
    float *sbc = reinterpret_cast<float *>(smem + Cfg::OFF_BC);
    float2 *sdx = reinterpret_cast<float2 *>(smem + Cfg::OFF_DX);
    float4 *agg = reinterpret_cast<float4 *>(smem + Cfg::OFF_AGG);     // [2][W][8][32]: P (4 slots), end state (4)
    unsigned char *ybase = smem + Cfg::OFF_Y;
    float4 *cbuf = reinterpret_cast<float4 *>(smem + Cfg::OFF_CARRY);  // [3][4][32]: carry into tile (2), unit end (1)
    uint64_t *bar_full = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);   // [S], 1 arrival + tx
    uint64_t *bar_empty = bar_full + S;                                         // [S], W arrivals
    uint64_t *bar_c = bar_empty + S;                                            // [2], 1 arrival
    uint64_t *bar_agg = bar_c + 2;                                              // [2], W arrivals
    int *s_ticket = reinterpret_cast<int *>(smem + Cfg::OFF_MISC);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pr = lane / GP, g = lane % GP;   // channel pair, 8-state group
    const int c0 = 2 * pr;                     // channels c0, c0 + 1 of the group
    if (p.cpw != CPW || p.np != NP) {          // tile sizes of the TMA boxes would not match expect_tx
        if (tid == 0) set_status(kStatusBadGeometry);
        return;
    }

    if (warp == 0) tmem_alloc(s_tmem, 512);
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], W);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_c[i], 1);
            mbar_init(&bar_agg[i], W);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // 256 columns of this warp's lane quarter (warps w and w+4 share a quarter)
    const uint32_t my_tmem = *s_tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 256);
    const uint32_t tile_bytes = (uint32_t)((p.has_z ? 3 : 2) * ARR * sizeof(IO) + (size_t)T * BCROW * 4);
    const int total_units = p.NG * p.nseg;
    int jt_base = 0;

    for (;;) {
        if (tid == 0) *s_ticket = atomicAdd(&p.ctrl[0], 1);
        __syncthreads();
        const int ticket = *s_ticket;
        __syncthreads();
        if (ticket >= total_units) break;
        const int s = ticket / p.NG, gi = ticket % p.NG;
        const int64_t b = gi / p.groups_per_b;
        const int64_t d0 = (int64_t)(gi % p.groups_per_b) * CPW;
        const int jfirst = s * p.seg_tiles;
        const int nt = min(jfirst + p.seg_tiles, p.ntiles) - jfirst;
        const int N = (int)p.N;
        const bool cv0 = d0 + c0 < p.Dm, cv1 = d0 + c0 + 1 < p.Dm;

        // chain pair ia = 4*ch + 2*q + jj/2  <->  channel c0+ch, states 4*(GP*q + g) + jj, +1
        float2 Ap[8];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int jj = 0; jj < 4; jj += 2) {
                    const int n = 4 * (GP * q + g) + jj;
                    const bool cv = ch ? cv1 : cv0;
                    const int64_t dd = d0 + c0 + ch;
                    Ap[4 * ch + 2 * q + jj / 2] =
                        make_float2((cv && n < N) ? p.A[dd * p.N + n] * kLog2e : 0.0f,
                                    (cv && n + 1 < N) ? p.A[dd * p.N + n + 1] * kLog2e : 0.0f);
                }
        const float Dd0 = (p.D != nullptr && cv0) ? p.D[d0 + c0] : 0.0f;
        const float Dd1 = (p.D != nullptr && cv1) ? p.D[d0 + c0 + 1] : 0.0f;
        // element e = lane + 32*m of a conversion belongs to channel (lane + 32*m) % CPW: one
        // channel per lane when CPW divides 32, two (alternating with m) when CPW = 64
        int conv_c[2];
        bool conv_valid[2];
        float conv_bias[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            conv_c[m] = (lane + 32 * m) % CPW;
            conv_valid[m] = d0 + conv_c[m] < p.Dm;
            conv_bias[m] = (p.bias != nullptr && conv_valid[m]) ? p.bias[d0 + conv_c[m]] : 0.0f;
        }

        auto stage_of = [&](int i) { return (jt_base + i) % S; };
        auto sphase = [&](int i) { return (uint32_t)(((jt_base + i) / S) & 1); };
        auto slot_of = [&](int i) { return (jt_base + i) & 1; };
        auto lphase = [&](int i) { return (uint32_t)(((jt_base + i) >> 1) & 1); };

        // producer (warp 0, lane 0): tile i of this unit into its stage
        auto issue = [&](int i) {
            const int st = stage_of(i);
            mbar_wait(&bar_empty[st], sphase(i) ^ 1u);
            IO *r = raw + (size_t)st * 3 * ARR;
            const int x = (jfirst + i) * T;
            mbar_arrive_expect_tx(&bar_full[st], tile_bytes);
            tma_load_3d(r, &p.map_u, x, (int)d0, (int)b, &bar_full[st]);
            tma_load_3d(r + ARR, &p.map_delta, x, (int)d0, (int)b, &bar_full[st]);
            if (p.has_z) tma_load_3d(r + 2 * ARR, &p.map_z, x, (int)d0, (int)b, &bar_full[st]);
            bulk_g2s(sbc + (size_t)st * T * BCROW, p.bc + ((int64_t)b * p.Lp + (int64_t)x) * BCROW,
                     (uint32_t)(T * BCROW * 4), &bar_full[st]);
        };
        // dt and dt*u of this warp's 8 steps of tile i -> sdx[warp][slot][kk][channel]
        auto convert = [&](int i) {
            const int st = stage_of(i);
            const IO *ru = raw + (size_t)st * 3 * ARR;
            const IO *rdl = ru + ARR;
            float2 *dst = sdx + ((size_t)warp * 2 + slot_of(i)) * K * CPW;
            const int64_t t0 = (int64_t)(jfirst + i) * T;
#pragma unroll
            for (int m = 0; m < CPW * K / 32; ++m) {
                const int e = lane + 32 * m, kk = e / CPW, tt = warp * K + kk, cc = conv_c[m & 1];
                float dt = 0.0f, x = 0.0f;
                if (t0 + tt < p.L && conv_valid[m & 1]) {
                    const float uu = io_traits<IO>::to_f(ru[cc * T + tt]);
                    dt = io_traits<IO>::to_f(rdl[cc * T + tt]) + conv_bias[m & 1];
                    if (p.softplus) dt = softplus_f(dt);
                    x = dt * uu;
                }
                dst[kk * CPW + cc] = make_float2(dt, x);
            }
            __syncwarp();
        };
        auto emit = [&](int i, int kk, int ch, float ys, IO *yb) {
            const IO *ru = raw + (size_t)stage_of(i) * 3 * ARR;
            const int tt = warp * K + kk, cc = c0 + ch;
            const int64_t t0 = (int64_t)(jfirst + i) * T;
            float yv = 0.0f;
            if ((ch ? cv1 : cv0) && t0 + tt < p.L) {
                yv = fmaf(ch ? Dd1 : Dd0, io_traits<IO>::to_f(ru[cc * T + tt]), ys);
                if (p.has_z) yv *= silu_f(io_traits<IO>::to_f(ru[2 * ARR + cc * T + tt]));
            }
            store_io(yb + cc * K + kk, yv);
        };
        auto y_buffer = [&](int i) {
            IO *yb = reinterpret_cast<IO *>(ybase + ((size_t)warp * 2 + slot_of(i)) * Cfg::Y_SLOT);
            if (lane == 0) bulk_wait_read1();
            __syncwarp();
            return yb;
        };
        auto y_store = [&](int i, IO *yb) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&p.map_y8, yb, (jfirst + i) * T + warp * K, (int)d0, (int)b);
                bulk_commit();
            }
        };
        // h <- P*h + e through the aggregates of warps [v0, v0 + nv) of `slot`, nv <= 2,
        // loads of the batch first
        auto compose2 = [&](float2 (&h)[8], int slot, int v0, int nv) {
            float4 Pv[2][4], Ev[2][4];
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (k < nv) {
                    const float4 *src = agg + ((size_t)slot * W + v0 + k) * 8 * 32;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        Pv[k][q] = src[q * 32 + lane];
                        Ev[k][q] = src[(4 + q) * 32 + lane];
                    }
                }
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (k < nv) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        h[2 * q] = __ffma2_rn(make_float2(Pv[k][q].x, Pv[k][q].y), h[2 * q], make_float2(Ev[k][q].x, Ev[k][q].y));
                        h[2 * q + 1] = __ffma2_rn(make_float2(Pv[k][q].z, Pv[k][q].w), h[2 * q + 1], make_float2(Ev[k][q].z, Ev[k][q].w));
                    }
                }
        };
        auto load_state = [&](float2 (&h)[8], const float4 *src) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = src[q * 32 + lane];
                h[2 * q] = make_float2(v.x, v.y);
                h[2 * q + 1] = make_float2(v.z, v.w);
            }
        };
        auto store_state = [&](float4 *dst, const float2 (&h)[8]) {
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q * 32 + lane] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
        };
        // local pass of step kk of tile i (both channels)
        auto local_step = [&](int i, int kk, float2 (&hl)[8], float2 &sdt) {
            const float4 dx = *reinterpret_cast<const float4 *>(sdx + (((size_t)warp * 2 + slot_of(i)) * K + kk) * CPW + c0);
            sdt.x += dx.x;   // channel c0: (dt, x) = (dx.x, dx.y); channel c1: (dx.z, dx.w)
            sdt.y += dx.z;
            const float *row = sbc + (size_t)stage_of(i) * T * BCROW + (size_t)(warp * K + kk) * BCROW;
            float r[32];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float4 bq = *reinterpret_cast<const float4 *>(row + 4 * (GP * q + g));
                const float2 b01 = make_float2(bq.x, bq.y), b23 = make_float2(bq.z, bq.w);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const float dtv = ch ? dx.z : dx.x, xv = ch ? dx.w : dx.y;
                    const float2 dd = make_float2(dtv, dtv), xx = make_float2(xv, xv);
                    const int ia = 4 * ch + 2 * q;          // pair index
                    const float2 e0 = __fmul2_rn(dd, Ap[ia]), e1 = __fmul2_rn(dd, Ap[ia + 1]);
                    const float2 a0 = make_float2(ex2(e0.x), ex2(e0.y));
                    const float2 a1 = make_float2(ex2(e1.x), ex2(e1.y));
                    const float2 w0 = __fmul2_rn(xx, b01), w1 = __fmul2_rn(xx, b23);
                    const int ri = 8 * ch + 4 * q;
                    r[ri] = a0.x; r[ri + 1] = a0.y; r[ri + 2] = a1.x; r[ri + 3] = a1.y;
                    r[16 + ri] = w0.x; r[16 + ri + 1] = w0.y; r[16 + ri + 2] = w1.x; r[16 + ri + 3] = w1.y;
                    hl[ia] = __ffma2_rn(a0, hl[ia], w0);
                    hl[ia + 1] = __ffma2_rn(a1, hl[ia + 1], w1);
                }
            }
            tmem_st32(my_tmem + (uint32_t)(32 * kk), r);
        };
        auto publish = [&](int i, const float2 (&hl)[8], float2 sdt) {
            tmem_wait_st();
            float4 *dst = agg + ((size_t)slot_of(i) * W + warp) * 8 * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 ss = (q < 2) ? make_float2(sdt.x, sdt.x) : make_float2(sdt.y, sdt.y);
                const float2 l0 = __fmul2_rn(Ap[2 * q], ss), l1 = __fmul2_rn(Ap[2 * q + 1], ss);
                dst[q * 32 + lane] = make_float4(ex2(l0.x), ex2(l0.y), ex2(l1.x), ex2(l1.y));
                dst[(4 + q) * 32 + lane] = make_float4(hl[2 * q].x, hl[2 * q].y, hl[2 * q + 1].x, hl[2 * q + 1].y);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_agg[slot_of(i)]);
        };
        float2 hin[8];
        float yp0[GP], yp1[GP];
        auto replay_step = [&](int i, int kk, const float (&cur)[32], IO *yb) {
            const float *row = sbc + (size_t)stage_of(i) * T * BCROW + (size_t)(warp * K + kk) * BCROW + NP;
            float2 y0a = make_float2(0.f, 0.f), y0b = y0a, y1a = y0a, y1b = y0a;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float4 cq = *reinterpret_cast<const float4 *>(row + 4 * (GP * q + g));
                const float2 c01 = make_float2(cq.x, cq.y), c23 = make_float2(cq.z, cq.w);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int ia = 4 * ch + 2 * q, ri = 8 * ch + 4 * q;
                    hin[ia] = __ffma2_rn(make_float2(cur[ri], cur[ri + 1]), hin[ia], make_float2(cur[16 + ri], cur[16 + ri + 1]));
                    hin[ia + 1] = __ffma2_rn(make_float2(cur[ri + 2], cur[ri + 3]), hin[ia + 1],
                                             make_float2(cur[16 + ri + 2], cur[16 + ri + 3]));
                    if (ch == 0) {
                        y0a = __ffma2_rn(c01, hin[ia], y0a);
                        y0b = __ffma2_rn(c23, hin[ia + 1], y0b);
                    } else {
                        y1a = __ffma2_rn(c01, hin[ia], y1a);
                        y1b = __ffma2_rn(c23, hin[ia + 1], y1b);
                    }
                }
            }
            yp0[kk % GP] = (y0a.x + y0a.y) + (y0b.x + y0b.y);
            yp1[kk % GP] = (y1a.x + y1a.y) + (y1b.x + y1b.y);
            if (kk % GP == GP - 1) {
                const float ys0 = group_reduce_transpose<GP>(yp0, lane);
                const float ys1 = group_reduce_transpose<GP>(yp1, lane);
                emit(i, kk - (GP - 1) + g, 0, ys0, yb);
                emit(i, kk - (GP - 1) + g, 1, ys1, yb);
            }
        };

        // carry into the unit's first tile (warp 0): zero, or the previous segment's final state
        if (warp == 0) {
            float2 carry[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) carry[q] = make_float2(0.f, 0.f);
            if (lane == 0) {
                issue(0);
                if (nt > 1) issue(1);
            }
            if (s > 0) {
                if (lane == 0) {
                    if (p.force_timeout) wait_flag_geq(&p.ctrl[1 + gi], 0x7fffffff, p.spin_limit);
                    else wait_flag_geq(&p.ctrl[1 + gi], s, p.spin_limit);
                }
                __syncwarp();
                const float4 *src = reinterpret_cast<const float4 *>(p.carry + ((int64_t)gi * 2 + ((s - 1) & 1)) * 512);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = __ldcg(src + q * 32 + lane);
                    carry[2 * q] = make_float2(v.x, v.y);
                    carry[2 * q + 1] = make_float2(v.z, v.w);
                }
            }
            store_state(cbuf + (size_t)slot_of(0) * 4 * 32, carry);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_c[slot_of(0)]);
        }
        // local pass of the unit's first tile
        {
            mbar_wait(&bar_full[stage_of(0)], sphase(0));
            convert(0);
            float2 hl[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) hl[q] = make_float2(0.f, 0.f);
            float2 sdt = make_float2(0.f, 0.f);
#pragma unroll
            for (int kk = 0; kk < K; ++kk) local_step(0, kk, hl, sdt);
            publish(0, hl, sdt);
        }
        for (int i = 0; i < nt; ++i) {
            const int buf = slot_of(i);
            mbar_wait(&bar_agg[buf], lphase(i));
            mbar_wait(&bar_c[buf], lphase(i));
            if (warp == 0) {
                // carry out of tile i through all eight aggregates; the carry out of the unit's
                // last tile goes to slot 2 (no barrier phase: read back by this warp below)
                float2 carry[8];
                load_state(carry, cbuf + (size_t)buf * 4 * 32);
#pragma unroll
                for (int v = 0; v < W; v += 2) compose2(carry, buf, v, 2);
                store_state(cbuf + (size_t)(i + 1 < nt ? (buf ^ 1) : 2) * 4 * 32, carry);
                __syncwarp();
                if (lane == 0 && i + 1 < nt) mbar_arrive(&bar_c[buf ^ 1]);
                // with three or more stages, tile i+2's stage held tile i+2-S <= i-1, already released
                if (S >= 3 && lane == 0 && i + 2 < nt) issue(i + 2);
            }
            // exact incoming state of this warp's sub-chunk
            load_state(hin, cbuf + (size_t)buf * 4 * 32);
#pragma unroll
            for (int v = 0; v < W - 1; v += 2)
                if (v < warp) compose2(hin, buf, v, min(warp - v, 2));
            const bool nxt = i + 1 < nt;
            if (nxt) {
                mbar_wait(&bar_full[stage_of(i + 1)], sphase(i + 1));
                convert(i + 1);
            }
            IO *yb = y_buffer(i);
            float2 hl[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) hl[q] = make_float2(0.f, 0.f);
            float2 sdt = make_float2(0.f, 0.f);
            // one register buffer: step kk's replay consumes it, the load of step kk+1 is issued,
            // and tile i+1's local step kk (which overwrites step kk's columns) covers its latency
            float ra[32];
            tmem_ld32(my_tmem, ra);
            tmem_wait_ld(ra);
#pragma unroll
            for (int kk = 0; kk < K; ++kk) {
                replay_step(i, kk, ra, yb);
                if (kk + 1 < K) tmem_ld32(my_tmem + (uint32_t)(32 * (kk + 1)), ra);
                if (nxt) local_step(i + 1, kk, hl, sdt);
                if (kk + 1 < K) tmem_wait_ld(ra);
            }
            y_store(i, yb);
            if (nxt) publish(i + 1, hl, sdt);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[stage_of(i)]);
            // with two stages, tile i+2 reuses tile i's stage: issue after releasing it
            if (S == 2 && warp == 0 && lane == 0 && i + 2 < nt) issue(i + 2);
        }
        // unit end: publish the segment's final state, or write the scan's final state
        if (warp == 0) {
            float2 carry[8];
            load_state(carry, cbuf + (size_t)2 * 4 * 32);
            if (s + 1 < p.nseg) {
                float4 *dst = reinterpret_cast<float4 *>(p.carry + ((int64_t)gi * 2 + (s & 1)) * 512);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    __stcg(dst + q * 32 + lane, make_float4(carry[2 * q].x, carry[2 * q].y, carry[2 * q + 1].x, carry[2 * q + 1].y));
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release(&p.ctrl[1 + gi], s + 1);
            } else if (p.last_state != nullptr) {
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    if (!(ch ? cv1 : cv0)) continue;
                    float *dst = p.last_state + (b * p.Dm + d0 + c0 + ch) * p.N;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int n = 4 * (GP * q + g) + jj;
                            const float2 v = carry[4 * ch + 2 * q + jj / 2];
                            if (n < N) dst[n] = (jj & 1) ? v.y : v.x;
                        }
                }
            }
        }
        jt_base += nt;
        __syncthreads();   // unit boundary
    }
    if (lane == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(*s_tmem, 512);
}

}  // namespace ssm
