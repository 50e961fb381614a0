// Channel-pair scan launches: bf16 io, zoh variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(bf16_zoh, __nv_bfloat16, true, false)
