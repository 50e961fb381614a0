// Channel-pair scan launches: f32 io, zoh variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(f32_zoh, float, true, false)
