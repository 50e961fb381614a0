// Channel-pair scan launches: f32 io, euler variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(f32_euler, float, false, false)
