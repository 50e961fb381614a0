// Channel-pair scan launches: bf16 io, euler variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(bf16_euler, __nv_bfloat16, false, false)
