// Selective scan, sequential-lane kernel: each lane walks the sequence for one channel and
// NPER of its states, so the recurrence h = exp(dt*A)*h + dt*B*u costs exactly one MUFU ex2
// and four FP32 operations per (channel, state, timestep).
//
// Source of the computation: the per-timestep loop of section 3.2 of "From RNN to Mamba:
// state-space model principles and long-sequence modelling in practice" (lmnt.cn):
// A_bar = exp(dt*A), B_bar = dt*B_t, h = A_bar*h + B_bar*x_t, y_t = sum_n h*C_t, then
// y + x*D and the SiLU(z) gate; dt = softplus(delta + bias) (sections 3.2-3.3).
//
// Work decomposition (one CTA):
//   * batch row b, a block of kCh = WARPS*32/G consecutive channels, one chunk of the
//     sequence [l_begin, l_end) walked in tiles of T timesteps;
//   * lane (warp w, lane l): channel c = w*(32/G) + l/G, state group g = l%G owning the
//     NPER states n = 4*(G*q + g) + j (q < NPER/4, j < 4). This interleaving makes the G
//     groups of a warp read G adjacent 16-byte pieces of a B/C row: one shared-memory
//     wavefront per LDS.128, broadcast to the 32/G channels.
//   * y: each lane accumulates its partial sum over its NPER states; every G timesteps the
//     G lanes of a channel exchange partials with a transposed butterfly (lane g ends with
//     the full sum for timestep tb+g), apply D*u and the gate, and stage y in shared memory
//     for one coalesced store per tile.
// Tiles are fetched with cp.async (double-buffered raw io data), converted once per
// (channel, timestep) -- softplus, dt*u -- and once per (state, timestep) -- B, C to fp32 --
// into shared memory.
//
// Modes: FULL computes y (and the final state of the last chunk); AGG computes only the
// chunk's end state from h = 0 and the chunk's sum of dt, which a combine kernel turns into
// each chunk's incoming state (the recurrence is a composition of affine maps -- section 2.2
// of the lmnt.cn page, section 3.4 of "Mamba architecture principles and industrial
// long-text practice", jsqmd.com -- so chunk end states compose exactly).
#pragma once
#include "check.cuh"
#include "common.cuh"

namespace ssm {

struct SeqParams {
    const void *u, *delta, *z, *B, *C;
    const float *A, *D, *bias;
    void *y;
    float *last_state;
    int64_t Bt, Dm, L, N;
    int64_t ld;         // channel-pair kernel: row stride (elements) of u, delta, z, y, B, C (>= L)
    int softplus;
    int64_t chunk_len;  // multiple of the tile length except possibly the last chunk
    int nchunks;
    int chan_blocks;    // channel blocks per batch row
    float *agg_h;       // [nchunks][Bt*Dm][Npad]   (AGG writes)
    float *agg_s;       // [nchunks][Bt*Dm]          (AGG writes)
    const float *hin;   // [nchunks][Bt*Dm][Npad] or null (FULL reads)
    int npad;           // NPER*G of the launched kernel
    int zoh;            // channel-pair kernel only: zero-order-hold B_bar (set by the host)
    const float *conv_w;   // channel-pair kernel with the conv front: [Dm][conv_k] fp32
    const float *conv_b;   // [Dm] fp32 or null
    int conv_k;            // 1..4
    int structured;        // channel-pair kernel: 1 = detect structured A per warp, 0 = never
    int check_probe;       // checked build: one deliberately out-of-range checked load (test)
};

template <typename IO, int NPER, int G, int WARPS, int T>
struct SeqCfg {
    static constexpr int kThreads = WARPS * 32;
    static constexpr int kCPW = 32 / G;
    static constexpr int kCh = WARPS * kCPW;
    static constexpr int kNpad = NPER * G;
    static constexpr int kBS = kNpad + 4;        // B/C row stride (floats): [T][kBS]
    static constexpr int kYS = T + 4;            // y staging row stride (floats): [kCh][kYS]
    static constexpr int kEpr = 16 / (int)sizeof(IO);
    static constexpr int kRowChunks = T / kEpr;  // 16-byte pieces per tile row
    static constexpr int kRawRows = 3 * kCh + 2 * kNpad;  // u, delta, z rows + B, C rows
    // shared memory, in bytes
    static constexpr size_t kRawBytes = (size_t)kRawRows * T * sizeof(IO);
    static constexpr size_t kOffDX = 2 * kRawBytes;
    static constexpr size_t kOffB = kOffDX + (size_t)T * kCh * sizeof(float2);
    static constexpr size_t kOffC = kOffB + (size_t)T * kBS * sizeof(float);
    static constexpr size_t kOffY = kOffC + (size_t)T * kBS * sizeof(float);
    static constexpr size_t kSmem = kOffY + (size_t)kCh * kYS * sizeof(float);
    static_assert(NPER % 4 == 0 && NPER >= 4, "NPER must be a multiple of 4");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "G must be 1, 2, 4 or 8");
    static_assert(T % 8 == 0 && T % G == 0, "tile must hold whole 16-byte pieces and G-steps");
    static_assert(kRawBytes % 16 == 0, "raw buffers must stay 16-byte aligned");
};

template <typename IO, int NPER, int G, int WARPS, int T, bool AGG, bool ALIGNED>
__global__ void __launch_bounds__(WARPS * 32)
scan_seq_kernel(const SeqParams p) {
    using Cfg = SeqCfg<IO, NPER, G, WARPS, T>;
    constexpr int kCh = Cfg::kCh, kNpad = Cfg::kNpad, kBS = Cfg::kBS, kYS = Cfg::kYS;
    extern __shared__ __align__(16) unsigned char smem[];
    IO *raw0 = reinterpret_cast<IO *>(smem);
    IO *raw1 = reinterpret_cast<IO *>(smem + Cfg::kRawBytes);
    float2 *sDX = reinterpret_cast<float2 *>(smem + Cfg::kOffDX);   // [T][kCh]
    float *sB = reinterpret_cast<float *>(smem + Cfg::kOffB);       // [T][kBS]
    float *sC = reinterpret_cast<float *>(smem + Cfg::kOffC);       // [T][kBS]
    float *sY = reinterpret_cast<float *>(smem + Cfg::kOffY);       // [kCh][kYS]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b = blockIdx.x / p.chan_blocks;
    const int64_t d0 = (int64_t)(blockIdx.x % p.chan_blocks) * kCh;
    const int k = blockIdx.y;
    const int64_t l_begin = (int64_t)k * p.chunk_len;
    const int64_t l_end = min(p.L, l_begin + p.chunk_len);
    const int ntiles = (int)((l_end - l_begin + T - 1) / T);
    const int N = (int)p.N;
    SSM_POISON_SMEM(smem);
    // array extents in bytes (the checked build's bounds checks; dead code otherwise)
    const uint64_t kIoB = (uint64_t)p.Bt * p.Dm * p.L * sizeof(IO), kBcB = (uint64_t)p.Bt * p.N * p.L * sizeof(IO);
    const uint64_t kAB = (uint64_t)p.Dm * p.N * 4, kDB = (uint64_t)p.Dm * 4;
    const uint64_t kCarryB = (uint64_t)p.nchunks * p.Bt * p.Dm * p.npad * 4, kSumB = (uint64_t)p.nchunks * p.Bt * p.Dm * 4;
    (void)kIoB; (void)kBcB; (void)kAB; (void)kDB; (void)kCarryB; (void)kSumB;

    const int c = warp * Cfg::kCPW + lane / G;   // this lane's channel within the block
    const int g = lane % G;
    const int64_t d = d0 + c;
    const bool cvalid = d < p.Dm;
    const int64_t bd = b * p.Dm + d;

    // per-lane constants: A*log2(e) for the lane's states (0 for padded states)
    float Ap[NPER];
#pragma unroll
    for (int q = 0; q < NPER / 4; ++q)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 4 * (G * q + g) + j;
            Ap[4 * q + j] = (cvalid && n < N) ? ld_chk_g(p.A, kAB, p.A + d * p.N + n) * kLog2e : 0.0f;
        }
    float h[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) h[i] = 0.0f;
    if (!AGG && p.hin != nullptr && cvalid) {
        const float *src = p.hin + ((int64_t)k * p.Bt * p.Dm + bd) * p.npad;
#pragma unroll
        for (int q = 0; q < NPER / 4; ++q) {
            const float4 v = ld_chk_g(p.hin, kCarryB, reinterpret_cast<const float4 *>(src + 4 * (G * q + g)));
            h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
        }
    }
    const float Dd = (!AGG && p.D != nullptr && cvalid) ? ld_chk_g(p.D, kDB, p.D + d) : 0.0f;
    const float bias_d = (p.bias != nullptr && cvalid) ? ld_chk_g(p.bias, kDB, p.bias + d) : 0.0f;

    // zero the padded B/C columns once (never overwritten)
    for (int i = tid; i < T * (kNpad - N); i += Cfg::kThreads) {
        const int t = i / (kNpad - N), n = N + i % (kNpad - N);
        st_chk_s(smem, sB + t * kBS + n, 0.0f);
        st_chk_s(smem, sC + t * kBS + n, 0.0f);
    }

    const IO *gU = reinterpret_cast<const IO *>(p.u);
    const IO *gDelta = reinterpret_cast<const IO *>(p.delta);
    const IO *gZ = reinterpret_cast<const IO *>(p.z);
    const IO *gB = reinterpret_cast<const IO *>(p.B);
    const IO *gC = reinterpret_cast<const IO *>(p.C);
    const bool has_z = !AGG && p.z != nullptr;

    // raw tile layout: rows [0,kCh) u, [kCh,2kCh) delta, [2kCh,3kCh) z, then kNpad B rows,
    // kNpad C rows; each row T io elements.
    auto issue_tile = [&](int j, IO *raw) {
        const int64_t t0 = l_begin + (int64_t)j * T;
        const int len = (int)min((int64_t)T, l_end - t0);
        const int nrows_ch = AGG ? 2 * kCh : (has_z ? 3 * kCh : 2 * kCh);
        const int nrows_n = AGG ? N : 2 * N;
        const int total = (nrows_ch + nrows_n) * Cfg::kRowChunks;
        for (int i = tid; i < total; i += Cfg::kThreads) {
            const int row = i / Cfg::kRowChunks, piece = i % Cfg::kRowChunks;
            const int e0 = piece * Cfg::kEpr;
            const IO *src;
            IO *dst;
            bool ok;
            if (row < nrows_ch) {
                const int kind = row / kCh, cc = row % kCh;
                const IO *base = kind == 0 ? gU : (kind == 1 ? gDelta : gZ);
                ok = (d0 + cc) < p.Dm;
                src = base + ((b * p.Dm + d0 + cc) * p.L + t0 + e0);
                dst = raw + (kind * kCh + cc) * T + e0;
            } else {
                const int r = row - nrows_ch, kind = r / N, n = r % N;
                const IO *base = kind == 0 ? gB : gC;
                ok = true;
                src = base + ((b * p.N + n) * p.L + t0 + e0);
                dst = raw + (3 * kCh + kind * kNpad + n) * T + e0;
            }
            const int avail = ok ? max(0, min(Cfg::kEpr, len - e0)) : 0;
            const uint64_t total = row < nrows_ch ? kIoB : kBcB;
            const void *sbase = row < nrows_ch ? (const void *)(row / kCh == 0 ? gU : (row / kCh == 1 ? gDelta : gZ))
                                               : (const void *)((row - nrows_ch) / N == 0 ? gB : gC);
            (void)total; (void)sbase;
            if (ALIGNED) {
                if (SSM_CHK_S(smem, dst, 16) && (avail == 0 || SSM_CHK_G(sbase, total, src, avail * sizeof(IO))))
                    cp_async16(dst, avail > 0 ? (const void *)src : (const void *)gU, avail * (int)sizeof(IO));
            } else {
#pragma unroll
                for (int e = 0; e < Cfg::kEpr; ++e)
                    st_chk_s(smem, dst + e, e < avail ? ld_chk_g(sbase, total, src + e) : IO(0.0f));
            }
        }
    };

    // Kahan-compensated sum of dt over the chunk (AGG)
    float dsum = 0.0f, dsum_c = 0.0f;

    if (ntiles > 0) issue_tile(0, raw0);
    cp_async_commit();
    for (int j = 0; j < ntiles; ++j) {
        IO *raw = (j & 1) ? raw1 : raw0;
        if (j + 1 < ntiles) issue_tile(j + 1, (j & 1) ? raw0 : raw1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int64_t t0 = l_begin + (int64_t)j * T;
        const int len = (int)min((int64_t)T, l_end - t0);
        // ---- convert: dt and dt*u per (channel, t); B, C per (state, t)
        for (int i = tid; i < kCh * T; i += Cfg::kThreads) {
            const int t = i % T, cc = i / T;
            float dt = 0.0f, x = 0.0f;
            if (t < len && d0 + cc < p.Dm) {
                const float uu = io_traits<IO>::to_f(ld_chk_s(smem, raw + cc * T + t));
                const float bb = (p.bias != nullptr) ? ld_chk_g(p.bias, kDB, p.bias + d0 + cc) : 0.0f;
                dt = io_traits<IO>::to_f(ld_chk_s(smem, raw + (kCh + cc) * T + t)) + bb;
                if (p.softplus) dt = softplus_f(dt);
                x = dt * uu;
            }
            st_chk_s(smem, sDX + t * kCh + cc, make_float2(dt, x));
        }
        for (int i = tid; i < N * T; i += Cfg::kThreads) {
            const int t = i % T, n = i / T;
            st_chk_s(smem, sB + t * kBS + n, io_traits<IO>::to_f(ld_chk_s(smem, raw + (3 * kCh + n) * T + t)));
            if (!AGG)
                st_chk_s(smem, sC + t * kBS + n, io_traits<IO>::to_f(ld_chk_s(smem, raw + (3 * kCh + kNpad + n) * T + t)));
        }
        __syncthreads();
        // ---- recurrence over the tile
        float tsum = 0.0f;
        float ypart[G];
#pragma unroll 1
        for (int tb = 0; tb < T; tb += G) {
#pragma unroll
            for (int s = 0; s < G; ++s) {
                const int t = tb + s;
                const float2 dx = ld_chk_s(smem, sDX + t * kCh + c);
                tsum += dx.x;
                float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
                for (int q = 0; q < NPER / 4; ++q) {
                    const float4 bv = ld_chk_s(smem, reinterpret_cast<const float4 *>(sB + t * kBS + 4 * (G * q + g)));
                    const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
                    float cc4[4] = {0.f, 0.f, 0.f, 0.f};
                    if (!AGG) {
                        const float4 cv = ld_chk_s(smem, reinterpret_cast<const float4 *>(sC + t * kBS + 4 * (G * q + g)));
                        cc4[0] = cv.x; cc4[1] = cv.y; cc4[2] = cv.z; cc4[3] = cv.w;
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int i = 4 * q + jj;
                        const float a = ex2(dx.x * Ap[i]);
                        h[i] = fmaf(a, h[i], dx.y * bb[jj]);
                        if (!AGG) {
                            if (jj & 1) y1 = fmaf(cc4[jj], h[i], y1);
                            else y0 = fmaf(cc4[jj], h[i], y0);
                        }
                    }
                }
                ypart[s] = y0 + y1;
            }
            if (!AGG) {
                const float ys = group_reduce_transpose<G>(ypart, lane);
                const int t = tb + g;  // the timestep this lane finished
                if (t < len && cvalid) {
                    const float uu = io_traits<IO>::to_f(ld_chk_s(smem, raw + c * T + t));
                    float yv = fmaf(Dd, uu, ys);
                    if (has_z) yv *= silu_f(io_traits<IO>::to_f(ld_chk_s(smem, raw + (2 * kCh + c) * T + t)));
                    st_chk_s(smem, sY + c * kYS + t, yv);
                }
            }
        }
        if (AGG) {  // compensated accumulation of the tile's dt sum
            const float yk = tsum - dsum_c;
            const float tk = dsum + yk;
            dsum_c = (tk - dsum) - yk;
            dsum = tk;
        }
        if (!AGG) {
            __syncthreads();
            // ---- store the y tile
            IO *gY = reinterpret_cast<IO *>(p.y);
            if (ALIGNED) {
                for (int i = tid; i < kCh * Cfg::kRowChunks; i += Cfg::kThreads) {
                    const int cc = i / Cfg::kRowChunks, e0 = (i % Cfg::kRowChunks) * Cfg::kEpr;
                    if (d0 + cc >= p.Dm || e0 >= len) continue;
                    IO *dst = gY + (b * p.Dm + d0 + cc) * p.L + t0 + e0;
                    const float *srcf = sY + cc * kYS + e0;
                    if (e0 + Cfg::kEpr <= len) {
                        float tmp[Cfg::kEpr];
#pragma unroll
                        for (int e = 0; e < Cfg::kEpr; ++e) tmp[e] = ld_chk_s(smem, srcf + e);
                        st_chk_g(gY, kIoB, reinterpret_cast<uint4 *>(dst), pack16(tmp, IO(0.0f)));
                    } else {
                        for (int e = 0; e < len - e0; ++e)
                            if (SSM_CHK_G(gY, kIoB, dst + e, sizeof(IO))) store_io(dst + e, ld_chk_s(smem, srcf + e));
                    }
                }
            } else {
                for (int i = tid; i < kCh * T; i += Cfg::kThreads) {
                    const int cc = i / T, t = i % T;
                    if (d0 + cc >= p.Dm || t >= len) continue;
                    if (SSM_CHK_G(gY, kIoB, gY + (b * p.Dm + d0 + cc) * p.L + t0 + t, sizeof(IO)))
                        store_io(gY + (b * p.Dm + d0 + cc) * p.L + t0 + t, ld_chk_s(smem, sY + cc * kYS + t));
                }
            }
        }
    }
    cp_async_wait<0>();

    if (!cvalid) return;
    if (AGG) {
        float *dst = p.agg_h + ((int64_t)k * p.Bt * p.Dm + bd) * p.npad;
#pragma unroll
        for (int q = 0; q < NPER / 4; ++q)
            st_chk_g(p.agg_h, kCarryB, reinterpret_cast<float4 *>(dst + 4 * (G * q + g)),
                     make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]));
        if (g == 0) st_chk_g(p.agg_s, kSumB, p.agg_s + (int64_t)k * p.Bt * p.Dm + bd, dsum);
    } else if (p.last_state != nullptr && k == p.nchunks - 1) {
        float *dst = p.last_state + bd * p.N;
#pragma unroll
        for (int q = 0; q < NPER / 4; ++q)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int n = 4 * (G * q + g) + jj;
                if (n < N) st_chk_g(p.last_state, (uint64_t)p.Bt * p.Dm * p.N * 4, dst + n, h[4 * q + jj]);
            }
    }
}

}  // namespace ssm
