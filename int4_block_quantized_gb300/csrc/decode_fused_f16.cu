// decode_fused_f16.cu -- the one-kernel decode layer for fp16 activations:
// instantiations of decode_fused.cuh.
#include "decode_fused.cuh"

namespace qmoe {

cudaError_t launch_fused_f16(const FusedParams& f, int scale_dtype, bool has_zp, cudaStream_t st, bool pdl,
                             bool check_only) {
#define QMOE_FU(TS) return has_zp ? launch_fused_me<TS, __half, true>(f, st, pdl, check_only) \
                                  : launch_fused_me<TS, __half, false>(f, st, pdl, check_only)
  if (scale_dtype == 1) QMOE_FU(__nv_bfloat16);
  QMOE_FU(__half);
#undef QMOE_FU
}

}  // namespace qmoe
