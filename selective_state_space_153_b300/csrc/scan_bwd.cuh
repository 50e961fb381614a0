// Selective scan backward: gradients of sum(y*dy) (+ sum(h_last*dlast)) with respect to u,
// delta, A, B, C, D, z and the dt bias, for the per-timestep loop of section 3.2 of
// "From RNN to Mamba: state-space model principles and long-sequence modelling in practice"
// (lmnt.cn). Training differentiates through the recurrence (section 2.2 of that page); the
// adjoint of h_t = a_t*h_{t-1} + dt_t*u_t*B_t, y_t = (sum_n C_t*h_t + D*u_t)*SiLU(z_t) is the
// reverse recurrence
//     lambda_t = dyhat_t * C_t + c_t,   c_{t-1} = a_t * lambda_t,   c_{L-1} = dlast,
// with dyhat_t = dy_t * SiLU(z_t), from which (per channel d, state n, step t)
//     dB_t += lambda_t dt_t u_t         dC_t += dyhat_t h_t          (summed over channels)
//     du_t  = dt_t sum_n lambda_t B_t + dyhat_t D
//     ddt_t = u_t sum_n lambda_t B_t + sum_n lambda_t A a_t h_{t-1},   ddelta_t = ddt_t sigmoid(v_t)
//     dA   += lambda_t dt_t a_t h_{t-1}   dD += dyhat_t u_t   dz_t = dy_t yhat_t SiLU'(z_t)
// (v = delta + bias; sigmoid is the softplus derivative; without softplus ddelta = ddt).
//
// Work decomposition: a thread owns Q states n = g + G*q (q < Q; Q = 4, or 2 for small N or
// where four states per lane leave the GPU short of warps) of one channel, G lanes per
// channel (a power of two, QG >= N), 32/G channels per warp, 128/G per CTA; the batch row is
// grid.y and the time-split chunk grid.z. Pass 1 (scan_bwd_ckpt_kernel) runs the recurrence
// forward and stores h at the start of every S-step segment. With a time split (chunks of
// whole segments, each a CTA), pass 1 starts every chunk from 0, an aggregate pass
// (scan_bwd_agg_kernel) runs the adjoint of each chunk but the first from a zero carry, and a
// combine forms each chunk's incoming state and carry from those chunk-local results (the
// recurrences are linear in their initial values). Pass 2 (scan_bwd_kernel) walks the
// segments backwards (a split chunk from its incoming carry, correcting each chunk-local
// checkpoint by exp(A*cum) times the chunk's incoming state):
//   * the CTA stages the segment's B, C rows (as [t][g][q], so a lane's states are one
//     16-byte read) and, once per (channel, step), dt, the softplus derivative, u,
//     dyhat = dy*SiLU(z) and the gate derivative factor dy*SiLU'(z). The raw inputs of the
//     next segments are in flight while the current one computes: copied by cp.async into a
//     shared-memory ring where every row is a multiple of 16 bytes long and 16-byte aligned,
//     else fetched into registers (two steps of a row per load where the length is even and
//     the rows start on 2-element boundaries);
//   * each lane recomputes its states' S steps from the checkpoint, then runs the adjoint in
//     reverse;
//   * sums over the states of a channel (yhat, sum lambda*B, sum lambda*A*a*h) are kept per
//     step and combined over the G lanes with a transposed butterfly every G steps, after
//     which lane g holds (and writes) step g of the group: one exchange per lane and step
//     instead of a butterfly per value and step;
//   * the per-element dB and dC terms are collected per state as 4-step vectors in shared
//     memory, summed over the CTA's channels after the segment and added with one vector
//     atomic per (state, 4 steps);
//   * dA, dD and the dt bias are summed in registers and added once at the end.
#pragma once
#include "check.cuh"
#include "common.cuh"

namespace ssm {

constexpr int kBwdS = 8;         // steps per checkpoint segment
constexpr int kBwdThreads = 128;
constexpr int kBwdQ = 4;         // states per thread (the default; 2 is also built)

// 4-byte asynchronous global->shared copy (through L1)
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}

struct BwdParams {
    const void *u, *delta, *z, *B, *C, *dy;
    const float *A, *D, *bias, *dlast;
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *dbias;
    float *ckpt;                  // [Bt*Dm][nseg][Q*G]: h before each segment's first step
    int64_t Bt, Dm, L, N;
    int softplus, nseg;
    int pair2;                    // 1: rows read two steps at a time (L even, bases 2-element aligned)
    int ring;                     // 1: rows staged by asynchronous 16-byte copies (L*esz % 16 == 0,
                                  //    16-byte aligned bases)
    // time split: chunk k covers segments [k*seg_per_chunk, min(nseg, (k+1)*seg_per_chunk));
    // with nchunk > 1 (the arrays below are then in the workspace after ckpt):
    int nchunk, seg_per_chunk;
    float *cumdt;                 // [Bt*Dm][nseg]: sum of dt from the chunk's first step to the segment's
    float *hloc;                  // [Bt*Dm][nchunk][Q*G]: chunk-end state of the recurrence from 0;
                                  //    after the combine, the state entering the chunk
    float *sdt;                   // [Bt*Dm][nchunk]: sum of dt over the chunk
    float *cloc;                  // [Bt*Dm][nchunk][Q*G]: adjoint carry out of the chunk's start, from 0
    float *cin;                   // [Bt*Dm][nchunk][Q*G]: adjoint carry into the chunk's last step
};

// The backward kernels' dynamic shared memory (one declaration for all of them).
extern __shared__ float4 smem_bwd4[];

// Extents in bytes of the backward's arrays, for the checked build's bounds checks
// (-DSSM_CHECK; in the normal build the checks are the constant `true` and these go unused).
__device__ __forceinline__ uint64_t bwd_rows_bytes(const BwdParams &p, int esz) {   // [Bt][Dm][L]
    return (uint64_t)(p.Bt * p.Dm * p.L) * (uint64_t)esz;
}
__device__ __forceinline__ uint64_t bwd_bc_bytes(const BwdParams &p, int esz) {     // [Bt][N][L]
    return (uint64_t)(p.Bt * p.N * p.L) * (uint64_t)esz;
}
__device__ __forceinline__ uint64_t bwd_ck_bytes(const BwdParams &p, int np) {      // checkpoints
    return (uint64_t)(p.Bt * p.Dm * p.nseg) * (uint64_t)np * 4;
}
__device__ __forceinline__ uint64_t bwd_cum_bytes(const BwdParams &p) {             // cumdt
    return (uint64_t)(p.Bt * p.Dm * p.nseg) * 4;
}
__device__ __forceinline__ uint64_t bwd_chunk_bytes(const BwdParams &p, int np) {   // hloc, cloc, cin
    return (uint64_t)(p.Bt * p.Dm * p.nchunk) * (uint64_t)np * 4;
}
__device__ __forceinline__ uint64_t bwd_dn_bytes(const BwdParams &p) { return (uint64_t)(p.Dm * p.N) * 4; }
__device__ __forceinline__ uint64_t bwd_d_bytes(const BwdParams &p) { return (uint64_t)p.Dm * 4; }

// Shared-memory layout (floats) of the backward kernels for G lanes per channel and Q states
// per lane (2 or 4: one or two packed pairs).
template <int G, int Q = kBwdQ>
struct BwdCfg {
    static constexpr int kQ = Q, kNP = G * kQ, kS = kBwdS, kP = Q / 2;
    static_assert(Q == 2 || Q == 4, "2 or 4 states per lane");
    static constexpr int kCpb = kBwdThreads / G;          // channels per CTA
    static constexpr int kTileBC = kS * kNP;              // B or C: [S][G][Q]
    static constexpr int kChan = kCpb * kS;               // per-channel arrays [kCpb][S]
    // dB/dC partials: per kind and channel, one row of S steps per state, padded so that the
    // 16-byte stores of a warp's lanes fall into distinct banks
    static constexpr int kRow = kS + 4;
    static constexpr int kPartCh = kNP * kRow + 16;
    static constexpr int kOffB = 0, kOffC = kTileBC, kOffDt = 2 * kTileBC;
    static constexpr int kOffSg = kOffDt + kChan, kOffU = kOffSg + kChan, kOffDyh = kOffU + kChan;
    static constexpr int kOffGz = kOffDyh + kChan, kOffPart = kOffGz + kChan;
    static constexpr int kFloats = kOffPart + 2 * kCpb * kPartCh;
    static_assert(kS % 4 == 0 && (kOffPart % 4) == 0 && (kPartCh % 4) == 0 && (kRow % 4) == 0, "16-byte rows");
};
// what a copy-ring slot holds: the checkpoint pass's rows (B, delta, u), the adjoint's (B, C,
// delta, u, dy, z), or the adjoint aggregate pass's (C, delta, dy, z)
enum : int { kRingCkpt = 0, kRingFull = 1, kRingAgg = 2 };
template <typename IO, int G, int Q, int MODE, bool CK, bool CUM>
struct BwdRing;

// Raw inputs of one segment [t0, t0+S) of batch row b for the CTA's channels d0 .. d0+kCpb-1,
// fetched into registers one segment ahead (the loads are in flight while the previous
// segment computes) and then staged into shared memory (stage). FULL = false: only B, dt
// and u (the checkpoint pass).
template <typename IO, int G, int Q, bool FULL>
struct BwdFetch {
    using Cfg = BwdCfg<G, Q>;
    static constexpr int kS = Cfg::kS, kNP = Cfg::kNP, kCpb = Cfg::kCpb;
    // register slots per thread: an even count, so that reading two steps per item also covers
    // every element
    static constexpr int kBC = (FULL ? 2 : 1) * kNP * kS, kBCI = 2 * ((kBC + 2 * kBwdThreads - 1) / (2 * kBwdThreads));
    static constexpr int kCH = kCpb * kS, kCHI = 2 * ((kCH + 2 * kBwdThreads - 1) / (2 * kBwdThreads));
    static_assert(kS % 2 == 0, "two steps per item stay in one row");
    float bc[kBCI];
    float dl[kCHI], uu[kCHI], dy[kCHI], zz[kCHI];

    // two io elements (8 bytes for fp32, 4 for bf16) as floats
    __device__ __forceinline__ static float2 ld2(const IO *q) {
        if constexpr (sizeof(IO) == 4) {
            return __ldg(reinterpret_cast<const float2 *>(q));
        } else {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(q));
            return make_float2(bf16lo(w), bf16hi(w));
        }
    }

    __device__ __forceinline__ void fetch(const BwdParams &p, int64_t b, int64_t t0, int64_t d0) {
        const int tid = threadIdx.x;
        const IO *Bm = reinterpret_cast<const IO *>(p.B) + b * p.N * p.L;
        const IO *Cm = reinterpret_cast<const IO *>(p.C) + b * p.N * p.L;
        if (p.pair2) {   // item k2 of a thread: two consecutive steps of one row (slots 2*k2, 2*k2+1)
#pragma unroll
            for (int k2 = 0; k2 < kBCI / 2; ++k2) {
                const int e = 2 * (tid + k2 * kBwdThreads);
                const int kind = e / (kNP * kS), r = e % (kNP * kS), n = r / kS, i = r % kS;
                const int64_t t = t0 + i;
                float2 v = make_float2(0.f, 0.f);
                const IO *q = (kind ? Cm : Bm) + n * p.L + t;
                if (e < kBC && n < p.N && t < p.L &&
                    SSM_CHK_G(kind ? p.C : p.B, bwd_bc_bytes(p, sizeof(IO)), q, 2 * sizeof(IO)))
                    v = ld2(q);
                bc[2 * k2] = v.x;
                bc[2 * k2 + 1] = v.y;
            }
#pragma unroll
            for (int k2 = 0; k2 < kCHI / 2; ++k2) {
                const int e = 2 * (tid + k2 * kBwdThreads);
                const int cc = e / kS, i = e % kS;
                const int64_t d = d0 + cc, t = t0 + i;
                float2 a = make_float2(0.f, 0.f), c = a, f = a, g = a;
                if (e < kCH && d < p.Dm && t < p.L) {
                    const int64_t idx = (b * p.Dm + d) * p.L + t;
                    const uint64_t rb = bwd_rows_bytes(p, sizeof(IO));
                    auto row2 = [&](const void *base) {
                        const IO *q = reinterpret_cast<const IO *>(base) + idx;
                        return SSM_CHK_G(base, rb, q, 2 * sizeof(IO)) ? ld2(q) : make_float2(0.f, 0.f);
                    };
                    a = row2(p.delta);
                    c = row2(p.u);
                    if (FULL) {
                        f = row2(p.dy);
                        if (p.z) g = row2(p.z);
                    }
                }
                dl[2 * k2] = a.x; dl[2 * k2 + 1] = a.y;
                uu[2 * k2] = c.x; uu[2 * k2 + 1] = c.y;
                dy[2 * k2] = f.x; dy[2 * k2 + 1] = f.y;
                zz[2 * k2] = g.x; zz[2 * k2 + 1] = g.y;
            }
            return;
        }
#pragma unroll
        for (int k = 0; k < kBCI; ++k) {   // consecutive e: consecutive steps of one row
            const int e = tid + k * kBwdThreads;
            const int kind = e / (kNP * kS), r = e % (kNP * kS), n = r / kS, i = r % kS;
            const int64_t t = t0 + i;
            const IO *q = (kind ? Cm : Bm) + n * p.L + t;
            bc[k] = (e < kBC && n < p.N && t < p.L &&
                     SSM_CHK_G(kind ? p.C : p.B, bwd_bc_bytes(p, sizeof(IO)), q, sizeof(IO)))
                        ? io_traits<IO>::to_f(*q) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kCHI; ++k) {
            const int e = tid + k * kBwdThreads;
            const int cc = e / kS, i = e % kS;
            const int64_t d = d0 + cc, t = t0 + i;
            dl[k] = uu[k] = dy[k] = zz[k] = 0.0f;
            if (e < kCH && d < p.Dm && t < p.L) {
                const int64_t idx = (b * p.Dm + d) * p.L + t;
                const uint64_t rb = bwd_rows_bytes(p, sizeof(IO));
                auto row1 = [&](const void *base) {
                    const IO *q = reinterpret_cast<const IO *>(base) + idx;
                    return SSM_CHK_G(base, rb, q, sizeof(IO)) ? io_traits<IO>::to_f(*q) : 0.0f;
                };
                dl[k] = row1(p.delta);
                uu[k] = row1(p.u);
                if (FULL) {
                    dy[k] = row1(p.dy);
                    if (p.z) zz[k] = row1(p.z);
                }
            }
        }
    }

    // dt, the softplus derivative, u and (FULL) dyhat = dy*SiLU(z), dy*SiLU'(z) once per
    // (channel, step); B, C as [t][g][q] (state n = g + G*q), zeros beyond N, L or Dm
    // element of register slot k: tid + k*128 (one step per item), or 2*(tid + (k/2)*128) + k%2
    // (two steps per item)
    __device__ __forceinline__ static int slot_elem(const BwdParams &p, int tid, int k) {
        return p.pair2 ? 2 * (tid + (k / 2) * kBwdThreads) + (k & 1) : tid + k * kBwdThreads;
    }

    __device__ __forceinline__ void stage(const BwdParams &p, float *sm, const float *sbias, int64_t t0,
                                          int64_t d0) const {
        const int tid = threadIdx.x;
#pragma unroll
        for (int k = 0; k < kBCI; ++k) {
            const int e = slot_elem(p, tid, k);
            if (e >= kBC) break;
            const int kind = e / (kNP * kS), r = e % (kNP * kS), n = r / kS, i = r % kS;
            st_chk_s(smem_bwd4, sm + (kind ? Cfg::kOffC : Cfg::kOffB) + (i * G + n % G) * Cfg::kQ + n / G, bc[k]);
        }
#pragma unroll
        for (int k = 0; k < kCHI; ++k) {
            const int e = slot_elem(p, tid, k);
            if (e >= kCH) continue;
            const int cc = e / kS, i = e % kS;
            const int64_t d = d0 + cc, t = t0 + i;
            float dtv = 0.0f, sgv = 0.0f, dyh = 0.0f, gz = 0.0f;
            if (d < p.Dm && t < p.L) {
                const float v = dl[k] + sbias[cc];
                if (!FULL) dtv = p.softplus ? softplus_f(v) : v;
                else if (p.softplus) dtv = softplus_sigmoid(v, sgv);
                else dtv = v, sgv = 1.0f;
                if (FULL) {
                    if (p.z) {
                        const float sz = rcp_approx(1.0f + ex2(-zz[k] * kLog2e));
                        dyh = dy[k] * zz[k] * sz;                            // dy * SiLU(z)
                        gz = dy[k] * sz * (1.0f + zz[k] * (1.0f - sz));      // dy * SiLU'(z)
                    } else {
                        dyh = dy[k];
                    }
                }
            }
            st_chk_s(smem_bwd4, sm + Cfg::kOffDt + e, dtv);
            st_chk_s(smem_bwd4, sm + Cfg::kOffU + e, uu[k]);
            if (FULL) {
                st_chk_s(smem_bwd4, sm + Cfg::kOffSg + e, sgv);
                st_chk_s(smem_bwd4, sm + Cfg::kOffDyh + e, dyh);
                st_chk_s(smem_bwd4, sm + Cfg::kOffGz + e, gz);
            }
        }
    }
};

// Raw inputs of one segment copied into a shared-memory ring by cp.async, kStages - 1 segments
// ahead, where every row is a multiple of 16 bytes long and starts on a 16-byte boundary. A
// slot holds the segment's rows as [row][S] io elements -- the B and/or C rows n < kNP of the
// mode, then its channel rows (delta, u, dy, z, or a subset) of the CTA's channels -- and (CK)
// the checkpoints of the CTA's channels as [channel][kNP] floats, then (CUM, time split) their
// dt sums from the chunk's first step as [channel] floats. Pieces of rows beyond N, Dm or L
// are not copied; stage() reads zeros in their place.
template <typename IO, int G, int Q, int MODE, bool CK = (MODE == kRingFull), bool CUM = false>
struct BwdRing {
    using Cfg = BwdCfg<G, Q>;
    static constexpr int kS = Cfg::kS, kNP = Cfg::kNP, kCpb = Cfg::kCpb, kQ = Cfg::kQ;
    static constexpr int kStepsPerPiece = 16 / (int)sizeof(IO);
    static constexpr int kGran = kS / kStepsPerPiece;                 // pieces per row segment
    static constexpr bool FULL = MODE == kRingFull, AGG = MODE == kRingAgg;
    static constexpr int kRowsBC = (FULL ? 2 : 1) * kNP, kRowsCH = (FULL ? 4 : AGG ? 3 : 2) * kCpb;
    // B/C row block -> 0 B, 1 C; channel row block -> 0 delta, 1 u, 2 dy, 3 z
    __device__ __forceinline__ static int bc_kind(int blk) { return AGG ? 1 : blk; }
    __device__ __forceinline__ static int ch_array(int blk) { return AGG && blk > 0 ? blk + 1 : blk; }
    static constexpr int kRows = kRowsBC + kRowsCH;
    static constexpr int kCkFloats = CK ? kCpb * kNP : 0, kCumFloats = CUM ? kCpb : 0;
    // measured on B300: deeper rings change neither pass (adjoint 3 stages, checkpoint 6); a
    // 2-stage checkpoint ring is 8-35% slower
    static constexpr int kStages = FULL ? 2 : 4;
    static constexpr int kSlotBytes = kRows * kS * (int)sizeof(IO) + (kCkFloats + kCumFloats) * 4;
    static constexpr int kRowPieces = kRows * kGran, kCkEnd = kRowPieces + kCkFloats / 4;
    static constexpr int kPieces = kCkEnd + kCumFloats;    // the dt sums: one 4-byte copy each
    static constexpr int kPerThread = (kPieces + kBwdThreads - 1) / kBwdThreads;
    static_assert(kS % kStepsPerPiece == 0 && kNP % 4 == 0 && kSlotBytes % 16 == 0 && kCpb % 4 == 0, "16-byte pieces");
    static constexpr size_t bytes() { return (size_t)kStages * kSlotBytes; }

    // copies of segment seg into its slot (seg % kStages); the caller commits the group
    __device__ __forceinline__ static void issue(const BwdParams &p, unsigned char *ring, int64_t b, int seg,
                                                 int64_t d0) {
        unsigned char *slot = ring + (seg % kStages) * kSlotBytes;
        const int64_t t0 = (int64_t)seg * kS;
#pragma unroll
        for (int m = 0; m < kPerThread; ++m) {
            const int j = threadIdx.x + m * kBwdThreads;
            if (j >= kPieces) break;
            const void *src = nullptr, *sbase = nullptr;   // the piece and its array
            uint64_t stotal = 0;
            if (j < kRowPieces) {
                const int row = j / kGran, part = j % kGran;
                const int64_t t = t0 + part * kStepsPerPiece;
                if (t < p.L) {
                    if (row < kRowsBC) {
                        const int kind = bc_kind(row / kNP), n = row % kNP;
                        sbase = kind ? p.C : p.B;
                        stotal = bwd_bc_bytes(p, sizeof(IO));
                        if (n < p.N) src = reinterpret_cast<const IO *>(sbase) + (b * p.N + n) * p.L + t;
                    } else {
                        const int r = row - kRowsBC, arr = ch_array(r / kCpb), cc = r % kCpb;
                        const int64_t d = d0 + cc;
                        sbase = arr == 0 ? p.delta : arr == 1 ? p.u : arr == 2 ? p.dy : p.z;
                        stotal = bwd_rows_bytes(p, sizeof(IO));
                        if (d < p.Dm && sbase != nullptr)
                            src = reinterpret_cast<const IO *>(sbase) + (b * p.Dm + d) * p.L + t;
                    }
                }
            } else if (j < kCkEnd) {
                const int r = j - kRowPieces, cc = r / (kNP / 4), part = r % (kNP / 4);
                const int64_t d = d0 + cc;
                sbase = p.ckpt;
                stotal = bwd_ck_bytes(p, kNP);
                if (d < p.Dm) src = p.ckpt + ((b * p.Dm + d) * p.nseg + seg) * kNP + 4 * part;
            } else {
                const int cc = j - kCkEnd;
                const int64_t d = d0 + cc;
                const float *q = p.cumdt + (b * p.Dm + d) * p.nseg + seg;
                if (p.nchunk > 1 && d < p.Dm && SSM_CHK_G(p.cumdt, bwd_cum_bytes(p), q, 4) &&
                    SSM_CHK_S(smem_bwd4, slot + 16 * kCkEnd + 4 * cc, 4))
                    cp_async4(slot + 16 * kCkEnd + 4 * cc, q);
                continue;
            }
            if (src != nullptr && SSM_CHK_G(sbase, stotal, src, 16) && SSM_CHK_S(smem_bwd4, slot + 16 * j, 16))
                cp_async16(slot + 16 * j, src, 16);
        }
    }

    // converted segment into the compute layout (as BwdFetch::stage); (CK) ckn: this lane's
    // checkpoint pairs, cum: its channel's dt sum from the chunk's first step (time split)
    __device__ __forceinline__ static void stage(const BwdParams &p, const unsigned char *ring, float *sm,
                                                 const float *sbias, int seg, int64_t d0, float2 (&ckn)[Cfg::kP],
                                                 float &cum) {
        const int tid = threadIdx.x;
        const IO *raw = reinterpret_cast<const IO *>(ring + (seg % kStages) * kSlotBytes);
        const int64_t t0 = (int64_t)seg * kS;
        constexpr int kBC = kRowsBC * kS, kCH = kCpb * kS;
        for (int e = tid; e < kBC; e += kBwdThreads) {
            const int kind = bc_kind(e / (kNP * kS)), r = e % (kNP * kS), n = r / kS, i = r % kS;
            const float v = (n < p.N && t0 + i < p.L) ? io_traits<IO>::to_f(ld_chk_s(smem_bwd4, raw + e)) : 0.0f;
            st_chk_s(smem_bwd4, sm + (kind ? Cfg::kOffC : Cfg::kOffB) + (i * G + n % G) * kQ + n / G, v);
        }
        for (int e = tid; e < kCH; e += kBwdThreads) {
            const int cc = e / kS, i = e % kS;
            const int64_t d = d0 + cc, t = t0 + i;
            float dtv = 0.0f, sgv = 0.0f, dyh = 0.0f, gz = 0.0f, uu = 0.0f;
            // the channel row blocks of this mode: delta first, then u (not AGG), dy, z (not CKPT)
            constexpr int kU = 1, kDy = AGG ? 1 : 2, kZ = AGG ? 2 : 3;
            if (d < p.Dm && t < p.L) {
                const float dl = io_traits<IO>::to_f(ld_chk_s(smem_bwd4, raw + kBC + e));
                if (!AGG) uu = io_traits<IO>::to_f(ld_chk_s(smem_bwd4, raw + kBC + kU * kCH + e));
                const float v = dl + sbias[cc];
                if (!FULL) dtv = p.softplus ? softplus_f(v) : v;
                else if (p.softplus) dtv = softplus_sigmoid(v, sgv);
                else dtv = v, sgv = 1.0f;
                if (FULL || AGG) {
                    const float dy = io_traits<IO>::to_f(ld_chk_s(smem_bwd4, raw + kBC + kDy * kCH + e));
                    if (p.z) {
                        const float zz = io_traits<IO>::to_f(ld_chk_s(smem_bwd4, raw + kBC + kZ * kCH + e));
                        const float sz = rcp_approx(1.0f + ex2(-zz * kLog2e));
                        dyh = dy * zz * sz;                            // dy * SiLU(z)
                        if (FULL) gz = dy * sz * (1.0f + zz * (1.0f - sz));   // dy * SiLU'(z)
                    } else {
                        dyh = dy;
                    }
                }
            }
            st_chk_s(smem_bwd4, sm + Cfg::kOffDt + e, dtv);
            if (!AGG) st_chk_s(smem_bwd4, sm + Cfg::kOffU + e, uu);
            if (AGG) st_chk_s(smem_bwd4, sm + Cfg::kOffDyh + e, dyh);
            if (FULL) {
                st_chk_s(smem_bwd4, sm + Cfg::kOffSg + e, sgv);
                st_chk_s(smem_bwd4, sm + Cfg::kOffDyh + e, dyh);
                st_chk_s(smem_bwd4, sm + Cfg::kOffGz + e, gz);
            }
        }
        if (CK) {
            const int g = tid % G, cc = tid / G;
            const float *cks = reinterpret_cast<const float *>(reinterpret_cast<const unsigned char *>(raw) +
                                                               kRows * kS * sizeof(IO));
            const float *ck = cks + cc * kNP;
            const bool valid = d0 + cc < p.Dm;
#pragma unroll
            for (int k = 0; k < Cfg::kP; ++k)
                ckn[k] = valid ? make_float2(ld_chk_s(smem_bwd4, ck + g + G * 2 * k), ld_chk_s(smem_bwd4, ck + g + G * (2 * k + 1)))
                               : make_float2(0.f, 0.f);
            if (CUM) cum = (valid && p.nchunk > 1) ? ld_chk_s(smem_bwd4, cks + kCpb * kNP + cc) : 0.0f;
        }
    }
};

// Checkpoint pass: the forward recurrence, h stored before every S-step segment; the next
// segments' raw inputs are in flight (in registers, or in the copy ring) while the current one
// computes. SPLIT (a time-split chunk, launched with the aggregate pass): 64 registers, for
// eight CTAs per SM, the density the time split aims at (one lane per channel keeps 128
// channels' staging slots per thread and gets more); the unsplit kernel (at least two CTAs
// per SM, at most a few) keeps the registers for the prefetch: 8% faster on
// 8 x 1536 x 2048 x 16.
template <typename IO, int G, int Q>
constexpr size_t bwd_ckpt_smem_bytes() {
    return (size_t)(BwdCfg<G, Q>::kOffU + BwdCfg<G, Q>::kChan + BwdCfg<G, Q>::kCpb) * sizeof(float) +
           BwdRing<IO, G, Q, kRingCkpt>::bytes();
}
// the adjoint aggregate pass: the adjoint's staging without the partial sums or checkpoints
template <typename IO, int G, int Q>
constexpr size_t bwd_agg_smem_bytes() {
    return (size_t)(BwdCfg<G, Q>::kOffPart + BwdCfg<G, Q>::kCpb) * sizeof(float) + BwdRing<IO, G, Q, kRingAgg>::bytes();
}
// the adjoint pass; SPLIT: a time-split chunk (the incoming-state table, the dt sums in the ring)
template <typename IO, int G, int Q, bool SPLIT>
constexpr size_t bwd_smem_bytes() {
    return (size_t)(BwdCfg<G, Q>::kFloats + BwdCfg<G, Q>::kCpb * (1 + (SPLIT ? BwdCfg<G, Q>::kNP : 0))) * sizeof(float) +
           BwdRing<IO, G, Q, kRingFull, true, SPLIT>::bytes();
}

// A lane's Q consecutive floats at p (16-byte or 8-byte aligned) as Q/2 packed pairs.
template <int P>
__device__ __forceinline__ void load_pairs(const float *p, float2 (&out)[P]) {
    if constexpr (P == 2) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        out[0] = make_float2(v.x, v.y);
        out[1] = make_float2(v.z, v.w);
    } else {
        out[0] = *reinterpret_cast<const float2 *>(p);
    }
}

template <typename IO, int G, int Q, bool SPLIT>
__device__ __forceinline__ void bwd_ckpt_body(const BwdParams &p, int kc) {
    using Cfg = BwdCfg<G, Q>;
    constexpr int kS = Cfg::kS, kNP = Cfg::kNP, kQ = Cfg::kQ, kCpb = Cfg::kCpb, kP = Cfg::kP;
    float *sm = reinterpret_cast<float *>(smem_bwd4);
    SSM_POISON_SMEM(smem_bwd4);
    const int tid = threadIdx.x, g = tid % G, cc = tid / G;
    const int64_t b = blockIdx.y, d0 = (int64_t)blockIdx.x * kCpb, d = d0 + cc;
    const bool valid = d < p.Dm;                 // every thread takes part in the staging
    const int64_t bd = b * p.Dm + (valid ? d : 0);
    float2 Ap2[kP], h2[kP];
#pragma unroll
    for (int k = 0; k < kP; ++k) {
        const int n0 = g + G * 2 * k, n1 = n0 + G;
        Ap2[k] = make_float2((valid && n0 < p.N) ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + (valid ? d : 0) * p.N + n0) * kLog2e : 0.0f,
                             (valid && n1 < p.N) ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + (valid ? d : 0) * p.N + n1) * kLog2e : 0.0f);
        h2[k] = make_float2(0.f, 0.f);
    }
    float *ck = p.ckpt + bd * (int64_t)p.nseg * kNP;
    // this CTA's chunk of segments; the state starts from 0 at the chunk (time split: the
    // true state is added to these checkpoints once the chunks' end states are combined)
    const int s0 = kc * p.seg_per_chunk, s1 = min(p.nseg, s0 + p.seg_per_chunk);
    float cum = 0.0f;                               // sum of dt from the chunk's first step
    using Ring = BwdRing<IO, G, Q, kRingCkpt>;
    float *sbias = sm + Cfg::kOffU + Cfg::kChan;    // the CTA's channels' dt bias (0 without one)
    unsigned char *ring = reinterpret_cast<unsigned char *>(sbias + kCpb);
    for (int c = tid; c < kCpb; c += kBwdThreads)   // read after the loop's first barrier
        st_chk_s(smem_bwd4, sbias + c, (p.bias && d0 + c < p.Dm) ? ld_chk_g(p.bias, bwd_d_bytes(p), p.bias + d0 + c) : 0.0f);
    BwdFetch<IO, G, Q, false> f;
    float2 ck_unused[kP];
    float cum_unused;
    if (p.ring) {
#pragma unroll
        for (int s = 0; s < Ring::kStages - 1; ++s) {
            if (s0 + s < s1) Ring::issue(p, ring, b, s0 + s, d0);
            cp_async_commit();
        }
    } else {
        f.fetch(p, b, (int64_t)s0 * kS, d0);
    }
    for (int seg = s0; seg < s1; ++seg) {
        if (valid) {
#pragma unroll
            for (int k = 0; k < kP; ++k) {
                st_chk_g(p.ckpt, bwd_ck_bytes(p, kNP), ck + (int64_t)seg * kNP + g + G * 2 * k, h2[k].x);
                st_chk_g(p.ckpt, bwd_ck_bytes(p, kNP), ck + (int64_t)seg * kNP + g + G * (2 * k + 1), h2[k].y);
            }
            if (SPLIT && g == 0) st_chk_g(p.cumdt, bwd_cum_bytes(p), p.cumdt + bd * p.nseg + seg, cum);
        }
        if (p.ring) cp_async_wait<Ring::kStages - 2>();
        __syncthreads();
        if (p.ring) Ring::stage(p, ring, sm, sbias, seg, d0, ck_unused, cum_unused);
        else f.stage(p, sm, sbias, (int64_t)seg * kS, d0);
        __syncthreads();
        if (p.ring) {            // the slot of segment seg - 1, staged before the barriers above
            if (seg + Ring::kStages - 1 < s1) Ring::issue(p, ring, b, seg + Ring::kStages - 1, d0);
            cp_async_commit();
        } else if (seg + 1 < s1) {
            f.fetch(p, b, (int64_t)(seg + 1) * kS, d0);   // in flight during this segment
        }
#pragma unroll
        for (int i = 0; i < kS; ++i) {
            const float dt = sm[Cfg::kOffDt + cc * kS + i];
            const float x = dt * sm[Cfg::kOffU + cc * kS + i];
            cum += dt;
            float2 bv[kP];
            load_pairs<kP>(sm + Cfg::kOffB + (i * G + g) * kQ, bv);
#pragma unroll
            for (int k = 0; k < kP; ++k) {
                const float2 e = __fmul2_rn(make_float2(dt, dt), Ap2[k]);
                h2[k] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), h2[k], __fmul2_rn(make_float2(x, x), bv[k]));
            }
        }
    }
    if (SPLIT && valid) {                   // the chunk's end state from 0 and its dt sum
        float *hl = p.hloc + (bd * p.nchunk + kc) * kNP;
#pragma unroll
        for (int k = 0; k < kP; ++k) {
            st_chk_g(p.hloc, bwd_chunk_bytes(p, kNP), hl + g + G * 2 * k, h2[k].x);
            st_chk_g(p.hloc, bwd_chunk_bytes(p, kNP), hl + g + G * (2 * k + 1), h2[k].y);
        }
        if (g == 0) st_chk_g(p.sdt, bwd_chunk_bytes(p, 1), p.sdt + bd * p.nchunk + kc, cum);
    }
}

// Time split, adjoint aggregate pass (chunks 1 .. nchunk-1): the reverse recurrence
// c_{t-1} = a_t (dyhat_t C_t + c_t) over the chunk from c = 0 at its last step; stores the
// carry leaving its first step (cloc). The carry that actually enters each chunk is then
// cin_{k-1} = (prod of a_t over chunk k) cin_k + cloc_k, with cin_{last} = dlast.
template <typename IO, int G, int Q>
__device__ __forceinline__ void bwd_agg_body(const BwdParams &p, int kc) {
    using Cfg = BwdCfg<G, Q>;
    constexpr int kS = Cfg::kS, kNP = Cfg::kNP, kQ = Cfg::kQ, kCpb = Cfg::kCpb, kP = Cfg::kP;
    float *sm = reinterpret_cast<float *>(smem_bwd4);
    SSM_POISON_SMEM(smem_bwd4);
    const int tid = threadIdx.x, g = tid % G, cc = tid / G;
    const int64_t b = blockIdx.y, d0 = (int64_t)blockIdx.x * kCpb, d = d0 + cc;
    const bool valid = d < p.Dm;
    const int64_t bd = b * p.Dm + (valid ? d : 0);
    const int s0 = kc * p.seg_per_chunk, s1 = min(p.nseg, s0 + p.seg_per_chunk);
    float2 Ap2[kP], c2[kP];
#pragma unroll
    for (int k = 0; k < kP; ++k) {
        const int n0 = g + G * 2 * k, n1 = n0 + G;
        Ap2[k] = make_float2((valid && n0 < p.N) ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + (valid ? d : 0) * p.N + n0) * kLog2e : 0.0f,
                             (valid && n1 < p.N) ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + (valid ? d : 0) * p.N + n1) * kLog2e : 0.0f);
        c2[k] = make_float2(0.f, 0.f);
    }
    using Ring = BwdRing<IO, G, Q, kRingAgg>;
    float *sbias = sm + Cfg::kOffPart;
    unsigned char *ring = reinterpret_cast<unsigned char *>(sbias + kCpb);
    for (int c = tid; c < kCpb; c += kBwdThreads)   // read after the loop's first barrier
        st_chk_s(smem_bwd4, sbias + c, (p.bias && d0 + c < p.Dm) ? ld_chk_g(p.bias, bwd_d_bytes(p), p.bias + d0 + c) : 0.0f);
    BwdFetch<IO, G, Q, true> f;
    float2 ck_unused[kP];
    float cum_unused;
    if (p.ring) {
#pragma unroll
        for (int s = 0; s < Ring::kStages - 1; ++s) {
            if (s1 - 1 - s >= s0) Ring::issue(p, ring, b, s1 - 1 - s, d0);
            cp_async_commit();
        }
    } else {
        f.fetch(p, b, (int64_t)(s1 - 1) * kS, d0);
    }
    for (int seg = s1 - 1; seg >= s0; --seg) {
        if (p.ring) cp_async_wait<Ring::kStages - 2>();
        __syncthreads();
        if (p.ring) Ring::stage(p, ring, sm, sbias, seg, d0, ck_unused, cum_unused);
        else f.stage(p, sm, sbias, (int64_t)seg * kS, d0);
        __syncthreads();
        if (p.ring) {
            if (seg - (Ring::kStages - 1) >= s0) Ring::issue(p, ring, b, seg - (Ring::kStages - 1), d0);
            cp_async_commit();
        } else if (seg > s0) {
            f.fetch(p, b, (int64_t)(seg - 1) * kS, d0);
        }
#pragma unroll
        for (int i = kS - 1; i >= 0; --i) {
            const float dt = sm[Cfg::kOffDt + cc * kS + i], dyh = sm[Cfg::kOffDyh + cc * kS + i];
            float2 cv[kP];
            load_pairs<kP>(sm + Cfg::kOffC + (i * G + g) * kQ, cv);
#pragma unroll
            for (int k = 0; k < kP; ++k) {
                const float2 e = __fmul2_rn(make_float2(dt, dt), Ap2[k]);
                const float2 lam = __ffma2_rn(make_float2(dyh, dyh), cv[k], c2[k]);
                c2[k] = __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)), lam);
            }
        }
    }
    if (valid) {
        float *cl = p.cloc + (bd * p.nchunk + kc) * kNP;
#pragma unroll
        for (int k = 0; k < kP; ++k) {
            st_chk_g(p.cloc, bwd_chunk_bytes(p, kNP), cl + g + G * 2 * k, c2[k].x);
            st_chk_g(p.cloc, bwd_chunk_bytes(p, kNP), cl + g + G * (2 * k + 1), c2[k].y);
        }
    }
}

// Unsplit checkpoint pass: one CTA per channel block and batch row.
template <typename IO, int G, int Q>
__global__ void __launch_bounds__(kBwdThreads, 1) scan_bwd_ckpt_kernel(const BwdParams p) {
    bwd_ckpt_body<IO, G, Q, false>(p, 0);
}

// Time split, the two passes that need no combined carry, in one launch: grid.z < nchunk are
// the checkpoint pass's chunks, the rest the aggregate pass's chunks 1 .. nchunk-1. The two
// roles read the same rows and are both latency-bound; sharing the SMs evens out each one's
// partial last wave. Held to 64 registers (eight CTAs per SM).
template <typename IO, int G, int Q>
__global__ void __launch_bounds__(kBwdThreads, G >= 2 ? 8 : 4) scan_bwd_split_front_kernel(const BwdParams p) {
    if ((int)blockIdx.z < p.nchunk) bwd_ckpt_body<IO, G, Q, true>(p, (int)blockIdx.z);
    else bwd_agg_body<IO, G, Q>(p, (int)blockIdx.z - p.nchunk + 1);
}

template <typename IO, int G, int Q, bool SPLIT>
__global__ void __launch_bounds__(kBwdThreads, Q == 4 ? 3 : 4) scan_bwd_kernel(const BwdParams p) {
    using Cfg = BwdCfg<G, Q>;
    constexpr int kS = Cfg::kS, kNP = Cfg::kNP, kQ = Cfg::kQ, kCpb = Cfg::kCpb, kP = Cfg::kP;
    // sums over a channel's states: transposed butterfly every G steps (G <= S), else a
    // butterfly per step
    constexpr bool kTransposed = G <= kS;
    constexpr int kGrp = kTransposed ? G : 1;
    float *sm = reinterpret_cast<float *>(smem_bwd4);
    SSM_POISON_SMEM(smem_bwd4);
    const int tid = threadIdx.x, lane = tid & 31, g = tid % G, cc = tid / G;
    const int64_t b = blockIdx.y, d0 = (int64_t)blockIdx.x * kCpb, d = d0 + cc;
    const bool valid = d < p.Dm;                // invalid lanes still take part in the exchanges
    const int64_t dd = valid ? d : 0;
    const int64_t bd = b * p.Dm + dd;
    const float Dv = (valid && p.D) ? ld_chk_g(p.D, bwd_d_bytes(p), p.D + dd) : 0.0f;
    float An[kQ], c[kQ];
    bool nv[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
        const int n = g + G * q;
        nv[q] = valid && n < p.N;
        An[q] = nv[q] ? ld_chk_g(p.A, bwd_dn_bytes(p), p.A + dd * p.N + n) : 0.0f;
        c[q] = !nv[q] ? 0.0f
               : p.nchunk > 1 ? ld_chk_g(p.cin, bwd_chunk_bytes(p, kNP), p.cin + (bd * p.nchunk + blockIdx.z) * kNP + n)
               : p.dlast ? ld_chk_g(p.dlast, (uint64_t)(p.Bt * p.Dm * p.N) * 4, p.dlast + bd * p.N + n) : 0.0f;
    }
    // as state pairs (q = 2k, 2k+1) for the packed arithmetic
    float2 An2[kP], Ap2[kP], c2[kP], dA2[kP];
#pragma unroll
    for (int k = 0; k < kP; ++k) {
        An2[k] = make_float2(An[2 * k], An[2 * k + 1]);
        Ap2[k] = make_float2(An[2 * k] * kLog2e, An[2 * k + 1] * kLog2e);
        c2[k] = make_float2(c[2 * k], c[2 * k + 1]);
        dA2[k] = make_float2(0.f, 0.f);
    }
    float dD = 0.0f, dbias = 0.0f;
    const float *ck = p.ckpt + bd * (int64_t)p.nseg * kNP;
    const float *sB = sm + Cfg::kOffB + g * kQ, *sC = sm + Cfg::kOffC + g * kQ;
    const float *sDt = sm + Cfg::kOffDt + cc * kS, *sU = sm + Cfg::kOffU + cc * kS;
    const float *sDyh = sm + Cfg::kOffDyh + cc * kS, *sGz = sm + Cfg::kOffGz + cc * kS;
    const float *sSg = sm + Cfg::kOffSg + cc * kS;
    float *myPart = sm + Cfg::kOffPart + cc * Cfg::kPartCh;     // dB kind; dC at + kCpb * kPartCh

    // the three per-step sums of a channel for the step this lane finishes: outputs
    auto finish = [&](int i, int64_t t0, float yhs, float dus, float dds) {
        const int64_t t = t0 + i;
        if (!valid || t >= p.L) return;
        const float dt = sDt[i], uu = sU[i], dyh = sDyh[i];
        const float ddl = fmaf(uu, dus, dds) * sSg[i];
        st_chk_g(p.du, bwd_rows_bytes(p, 4), p.du + bd * p.L + t, fmaf(dyh, Dv, dt * dus));
        st_chk_g(p.ddelta, bwd_rows_bytes(p, 4), p.ddelta + bd * p.L + t, ddl);
        if (p.dz) st_chk_g(p.dz, bwd_rows_bytes(p, 4), p.dz + bd * p.L + t, sGz[i] * fmaf(Dv, uu, yhs));
        dD = fmaf(dyh, uu, dD);
        dbias += ddl;
    };

    using Ring = BwdRing<IO, G, Q, kRingFull, true, SPLIT>;
    float *sbias = sm + Cfg::kFloats;               // the CTA's channels' dt bias (0 without one)
    // time split: the state entering this chunk, [channel][kNP]; the checkpoint pass took the
    // chunk's checkpoints from 0, so each is corrected by exp(A*cum) times this state
    float *shin = sbias + kCpb;
    unsigned char *ring = reinterpret_cast<unsigned char *>(shin + (SPLIT ? kCpb * kNP : 0));
    const bool fold = SPLIT && blockIdx.z > 0;
    for (int c = tid; c < kCpb; c += kBwdThreads)   // read after the loop's first barrier
        st_chk_s(smem_bwd4, sbias + c, (p.bias && d0 + c < p.Dm) ? ld_chk_g(p.bias, bwd_d_bytes(p), p.bias + d0 + c) : 0.0f);
    if (fold) {
        for (int e = tid; e < kCpb * kNP; e += kBwdThreads) {
            const int64_t dc = d0 + e / kNP;
            st_chk_s(smem_bwd4, shin + e,
                     dc < p.Dm ? ld_chk_g(p.hloc, bwd_chunk_bytes(p, kNP), p.hloc + ((b * p.Dm + dc) * p.nchunk + blockIdx.z) * kNP + e % kNP)
                               : 0.0f);
        }
    }
    BwdFetch<IO, G, Q, true> f;
    // the segment's checkpoint (and time split: its dt sum from the chunk's first step),
    // fetched with its inputs one segment ahead
    auto fetch_ck = [&](int seg, float2 (&out)[kP], float &cm) {
#pragma unroll
        for (int k = 0; k < kP; ++k)
            out[k] = valid ? make_float2(ld_chk_g(p.ckpt, bwd_ck_bytes(p, kNP), ck + (int64_t)seg * kNP + g + G * 2 * k),
                                         ld_chk_g(p.ckpt, bwd_ck_bytes(p, kNP), ck + (int64_t)seg * kNP + g + G * (2 * k + 1)))
                           : make_float2(0.f, 0.f);
        cm = (valid && fold) ? ld_chk_g(p.cumdt, bwd_cum_bytes(p), p.cumdt + bd * p.nseg + seg) : 0.0f;
    };
    // dB, dC of the segment starting at t0: sum the CTA's channels, one vector atomic per
    // (state, 4 steps). Run for the previous segment between the next one's barriers (the
    // staging touches other shared memory), which saves a barrier per segment.
    auto reduce_dbc = [&](int64_t t0) {
        constexpr int kItems = 2 * kNP * (kS / 4);
        for (int e = tid; e < kItems; e += kBwdThreads) {
            const int kind = e / (kNP * (kS / 4)), r = e % (kNP * (kS / 4)), n = r / (kS / 4), tq = r % (kS / 4);
            if (n >= p.N) continue;
            const float *src = sm + Cfg::kOffPart + kind * kCpb * Cfg::kPartCh + n * Cfg::kRow + 4 * tq;
            float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll 8
            for (int ch = 0; ch < kCpb; ++ch) {
                const float4 v = ld_chk_s(smem_bwd4, reinterpret_cast<const float4 *>(src + ch * Cfg::kPartCh));
                lo = __fadd2_rn(lo, make_float2(v.x, v.y));
                hi = __fadd2_rn(hi, make_float2(v.z, v.w));
            }
            const float4 acc = make_float4(lo.x, lo.y, hi.x, hi.y);
            const int64_t t = t0 + 4 * tq;
            float *dst = (kind ? p.dC : p.dB) + (b * p.N + n) * p.L + t;
            if (t + 3 < p.L && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
                if (SSM_CHK_G(kind ? p.dC : p.dB, bwd_bc_bytes(p, 4), dst, 16))
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(acc.x), "f"(acc.y),
                                 "f"(acc.z), "f"(acc.w)
                                 : "memory");
            } else {
                const float av[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (t + k < p.L && SSM_CHK_G(kind ? p.dC : p.dB, bwd_bc_bytes(p, 4), dst + k, 4))
                        atomicAdd(dst + k, av[k]);
            }
        }
    };
    float2 ckn[kP];
    float cumn = 0.0f;
    // this CTA's chunk of segments, walked backwards from its last
    const int s0 = blockIdx.z * p.seg_per_chunk, s1 = min(p.nseg, s0 + p.seg_per_chunk);
    if (p.ring) {
#pragma unroll
        for (int s = 0; s < Ring::kStages - 1; ++s) {
            if (s1 - 1 - s >= s0) Ring::issue(p, ring, b, s1 - 1 - s, d0);
            cp_async_commit();
        }
    } else {
        f.fetch(p, b, (int64_t)(s1 - 1) * kS, d0);
        fetch_ck(s1 - 1, ckn, cumn);
    }
    for (int seg = s1 - 1; seg >= s0; --seg) {
        const int64_t t0 = (int64_t)seg * kS;
        if (p.ring) cp_async_wait<Ring::kStages - 2>();
        __syncthreads();                        // the previous segment is done with shared memory
        if (seg < s1 - 1) reduce_dbc(t0 + kS);   // the previous (later) segment's terms
        if (p.ring) Ring::stage(p, ring, sm, sbias, seg, d0, ckn, cumn);
        else f.stage(p, sm, sbias, t0, d0);
        __syncthreads();
        // states as pairs (q = 2k, 2k+1): hs[k][0] before the segment, hs[k][i+1] after step t0+i
        float2 hs[kP][kS + 1];
#pragma unroll
        for (int k = 0; k < kP; ++k) {
            hs[k][0] = ckn[k];
            if (fold) {
                const float2 e = __fmul2_rn(make_float2(cumn, cumn), Ap2[k]);
                const float2 H = make_float2(shin[cc * kNP + g + G * 2 * k], shin[cc * kNP + g + G * (2 * k + 1)]);
                hs[k][0] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), H, ckn[k]);
            }
        }
        if (p.ring) {   // into the slot of segment seg + 1, staged before the barriers above
            if (seg - (Ring::kStages - 1) >= s0) Ring::issue(p, ring, b, seg - (Ring::kStages - 1), d0);
            cp_async_commit();
        } else if (seg > s0) {   // the next segment's inputs and checkpoint, in flight meanwhile
            f.fetch(p, b, t0 - kS, d0);
            fetch_ck(seg - 1, ckn, cumn);
        }
#pragma unroll
        for (int i = 0; i < kS; ++i) {
            const float dt = sDt[i];
            const float x = dt * sU[i];
            float2 bv[kP];
            load_pairs<kP>(sB + i * G * kQ, bv);
#pragma unroll
            for (int k = 0; k < kP; ++k) {
                const float2 e = __fmul2_rn(make_float2(dt, dt), Ap2[k]);
                hs[k][i + 1] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), hs[k][i], __fmul2_rn(make_float2(x, x), bv[k]));
            }
        }
        float pb[kQ][4], pc[kQ][4];              // dB / dC terms of the current four steps
#pragma unroll
        for (int grp = kS / kGrp - 1; grp >= 0; --grp) {
            float red[3][kGrp];
#pragma unroll
            for (int s = kGrp - 1; s >= 0; --s) {
                const int i = grp * kGrp + s;
                const float dt = sDt[i], dyh = sDyh[i];
                const float x = dt * sU[i];
                float2 cv[kP], bv[kP];
                load_pairs<kP>(sC + i * G * kQ, cv);
                load_pairs<kP>(sB + i * G * kQ, bv);
                const float2 dt2 = make_float2(dt, dt), dyh2 = make_float2(dyh, dyh), x2 = make_float2(x, x);
                float2 yh2 = make_float2(0.f, 0.f), du2 = make_float2(0.f, 0.f), dd22 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < kP; ++k) {
                    const float2 e = __fmul2_rn(dt2, Ap2[k]);
                    const float2 a = make_float2(ex2(e.x), ex2(e.y));
                    const float2 lam = __ffma2_rn(dyh2, cv[k], c2[k]);
                    yh2 = __ffma2_rn(cv[k], hs[k][i + 1], yh2);
                    du2 = __ffma2_rn(lam, bv[k], du2);
                    const float2 P = __fmul2_rn(lam, __fmul2_rn(a, hs[k][i]));
                    dd22 = __ffma2_rn(An2[k], P, dd22);
                    dA2[k] = __ffma2_rn(dt2, P, dA2[k]);
                    c2[k] = __fmul2_rn(a, lam);
                    const float2 vb = __fmul2_rn(lam, x2), vc = __fmul2_rn(dyh2, hs[k][i + 1]);
                    pb[2 * k][i & 3] = vb.x;
                    pb[2 * k + 1][i & 3] = vb.y;
                    pc[2 * k][i & 3] = vc.x;
                    pc[2 * k + 1][i & 3] = vc.y;
                }
                const float yh = yh2.x + yh2.y, du = du2.x + du2.y, dd2 = dd22.x + dd22.y;
                if ((i & 3) == 0) {             // a full 4-step vector per state: to shared memory
#pragma unroll
                    for (int q = 0; q < kQ; ++q) {
                        const int n = g + G * q;
                        st_chk_s(smem_bwd4, reinterpret_cast<float4 *>(myPart + n * Cfg::kRow + i),
                                 make_float4(pb[q][0], pb[q][1], pb[q][2], pb[q][3]));
                        st_chk_s(smem_bwd4, reinterpret_cast<float4 *>(myPart + kCpb * Cfg::kPartCh + n * Cfg::kRow + i),
                                 make_float4(pc[q][0], pc[q][1], pc[q][2], pc[q][3]));
                    }
                }
                if constexpr (kTransposed) {
                    red[0][s] = yh;
                    red[1][s] = du;
                    red[2][s] = dd2;
                } else {
                    // butterfly over the G lanes of the channel; lane g == 0 writes the step
                    float ys = yh, us = du, ds = dd2;
#pragma unroll
                    for (int o = G / 2; o >= 1; o /= 2) {
                        ys += __shfl_xor_sync(0xffffffffu, ys, o);
                        us += __shfl_xor_sync(0xffffffffu, us, o);
                        ds += __shfl_xor_sync(0xffffffffu, ds, o);
                    }
                    if (g == 0) finish(i, t0, ys, us, ds);
                }
            }
            if constexpr (kTransposed) {
                // lane g ends with the sums of step grp*G + g
                const float yhs = group_reduce_transpose<kGrp>(red[0], lane);
                const float dus = group_reduce_transpose<kGrp>(red[1], lane);
                const float dds = group_reduce_transpose<kGrp>(red[2], lane);
                finish(grp * kGrp + g, t0, yhs, dus, dds);
            }
        }
    }
    __syncthreads();                            // the last segment's dB/dC terms are complete
    reduce_dbc((int64_t)s0 * kS);
    // dA per state; dD and the dt bias summed over the channel's lanes first
#pragma unroll
    for (int o = G / 2; o >= 1; o /= 2) {
        dD += __shfl_xor_sync(0xffffffffu, dD, o);
        dbias += __shfl_xor_sync(0xffffffffu, dbias, o);
    }
    if (!valid) return;
    float dA[kQ];
#pragma unroll
    for (int k = 0; k < kP; ++k) {
        dA[2 * k] = dA2[k].x;
        dA[2 * k + 1] = dA2[k].y;
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q)
        if (nv[q] && SSM_CHK_G(p.dA, bwd_dn_bytes(p), p.dA + dd * p.N + g + G * q, 4))
            atomicAdd(p.dA + dd * p.N + g + G * q, dA[q]);
    if (g == 0) {
        if (p.dD && SSM_CHK_G(p.dD, bwd_d_bytes(p), p.dD + dd, 4)) atomicAdd(p.dD + dd, dD);
        if (p.dbias && SSM_CHK_G(p.dbias, bwd_d_bytes(p), p.dbias + dd, 4)) atomicAdd(p.dbias + dd, dbias);
    }
}

// CTAs of the time-split adjoint pass that fit one SM (launch bound and shared memory); in
// k_bwd.cu
int bwd_split_adjoint_ctas_per_sm(ssm_dtype_t io, int G, int Q);

}  // namespace ssm
