// Channel-pair scan: dispatch over io type and variant, and the per-launch geometry the
// planner needs (shared memory, warps, register-bound residency).
#include "k_pair_impl.cuh"

namespace ssm {

cudaError_t launch_pair_bf16_euler(int, int, bool, const SeqParams &, int, cudaStream_t);
cudaError_t launch_pair_bf16_zoh(int, int, bool, const SeqParams &, int, cudaStream_t);
cudaError_t launch_pair_bf16_conv(int, int, bool, const SeqParams &, int, cudaStream_t);
cudaError_t launch_pair_f32_euler(int, int, bool, const SeqParams &, int, cudaStream_t);
cudaError_t launch_pair_f32_zoh(int, int, bool, const SeqParams &, int, cudaStream_t);
cudaError_t launch_pair_f32_conv(int, int, bool, const SeqParams &, int, cudaStream_t);

cudaError_t launch_pair(ssm_dtype_t io, int variant, int ks, int gp, bool agg, const SeqParams &prm,
                        int grid_y, cudaStream_t s) {
    const bool bf = io == SSM_BF16;
    switch (variant) {
        case kPairEuler: return bf ? launch_pair_bf16_euler(ks, gp, agg, prm, grid_y, s)
                                   : launch_pair_f32_euler(ks, gp, agg, prm, grid_y, s);
        case kPairZoh: return bf ? launch_pair_bf16_zoh(ks, gp, agg, prm, grid_y, s)
                                 : launch_pair_f32_zoh(ks, gp, agg, prm, grid_y, s);
        case kPairConv: return bf ? launch_pair_bf16_conv(ks, gp, agg, prm, grid_y, s)
                                  : launch_pair_f32_conv(ks, gp, agg, prm, grid_y, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

size_t pair_smem(ssm_dtype_t io, int ks, int gp, bool conv, bool agg) {
    using bf16 = __nv_bfloat16;
    switch (ks * 100 + gp) {
#define SSM_PAIR_SMEM(KS, GP)                                                                               \
    case KS * 100 + GP:                                                                                     \
        if (agg) {                                                                                          \
            if (conv) return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, true), kPairT, true>::kSmem \
                                            : PairCfg<float, KS, GP, pair_warps(KS, GP, true), kPairT, true>::kSmem; \
            return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, true), kPairT>::kSmem             \
                                  : PairCfg<float, KS, GP, pair_warps(KS, GP, true), kPairT>::kSmem;           \
        }                                                                                                   \
        if (conv) return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, false), kPairT, true>::kSmem \
                                        : PairCfg<float, KS, GP, pair_warps(KS, GP, false), kPairT, true>::kSmem; \
        return io == SSM_BF16 ? PairCfg<bf16, KS, GP, pair_warps(KS, GP, false), kPairT>::kSmem                \
                              : PairCfg<float, KS, GP, pair_warps(KS, GP, false), kPairT>::kSmem;
        SSM_PAIR_CASES(SSM_PAIR_SMEM)
#undef SSM_PAIR_SMEM
        default: return 0;
    }
}

int pair_warps_of(int ks, int gp, bool agg) { return pair_warps(ks, gp, agg); }

int pair_min_blocks_of(int ks, int gp, bool agg) { return pair_min_blocks(pair_warps(ks, gp, agg), ks, gp); }

}  // namespace ssm
