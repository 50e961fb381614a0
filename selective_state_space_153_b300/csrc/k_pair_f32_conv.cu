// Channel-pair scan launches: f32 io, conv variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(f32_conv, float, false, true)
