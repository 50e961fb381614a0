// Channel-pair scan launches: bf16 io, conv variant.
#include "k_pair_impl.cuh"
SSM_DEFINE_PAIR_TU(bf16_conv, __nv_bfloat16, false, true)
