// Recurrent single-token step launches (decode.cuh).
#include "launch.h"

namespace ssm {

namespace {
using bf16 = __nv_bfloat16;

template <typename IO, bool ZOH>
cudaError_t launch_decode_io(int kind, int lpc, const DecodeParams &p, cudaStream_t s) {
    const int64_t chans = p.Bt * p.Dm;
    if (kind == 0) {   // batch rows on grid.y, 16-byte B/C reads
        const dim3 grid((unsigned)((p.Dm * lpc + 255) / 256), (unsigned)p.Bt);
        switch (lpc) {
#define SSM_DECW(L) case L: decode_wide_kernel<IO, L, ZOH><<<grid, 256, 0, s>>>(p); break;
            SSM_DECW(1) SSM_DECW(2) SSM_DECW(4) SSM_DECW(8) SSM_DECW(16) SSM_DECW(32)
#undef SSM_DECW
            default: return cudaErrorInvalidConfiguration;
        }
    } else if (kind == 1) {   // element-wise B/C reads
        const unsigned grid = (unsigned)((chans * lpc + 255) / 256);
        switch (lpc) {
#define SSM_DEC(L) case L: decode_vec_kernel<IO, L, ZOH><<<grid, 256, 0, s>>>(p); break;
            SSM_DEC(1) SSM_DEC(2) SSM_DEC(4) SSM_DEC(8) SSM_DEC(16) SSM_DEC(32)
#undef SSM_DEC
            default: return cudaErrorInvalidConfiguration;
        }
    } else {   // one thread per channel
        decode_scalar_kernel<IO, ZOH><<<(unsigned)((chans + 255) / 256), 256, 0, s>>>(p);
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode(ssm_dtype_t io, int kind, int lpc, bool zoh, const DecodeParams &p, cudaStream_t s) {
    if (io == SSM_BF16)
        return zoh ? launch_decode_io<bf16, true>(kind, lpc, p, s) : launch_decode_io<bf16, false>(kind, lpc, p, s);
    return zoh ? launch_decode_io<float, true>(kind, lpc, p, s) : launch_decode_io<float, false>(kind, lpc, p, s);
}

}  // namespace ssm
