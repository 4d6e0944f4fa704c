// decode_fused_bf16.cu -- the one-kernel decode layer for bf16 activations:
// instantiations of decode_fused.cuh, and the dispatch on the activation dtype.
#include "decode_fused.cuh"

namespace qmoe {

cudaError_t launch_fused_bf16(const FusedParams& f, int scale_dtype, bool has_zp, cudaStream_t st, bool pdl,
                             bool check_only) {
#define QMOE_FU(TS) return has_zp ? launch_fused_me<TS, __nv_bfloat16, true>(f, st, pdl, check_only) \
                                  : launch_fused_me<TS, __nv_bfloat16, false>(f, st, pdl, check_only)
  if (scale_dtype == 1) QMOE_FU(__nv_bfloat16);
  QMOE_FU(__half);
#undef QMOE_FU
}

cudaError_t launch_fused(const FusedParams& f, int act_dtype, int scale_dtype, bool has_zp, cudaStream_t st,
                         bool pdl, bool check_only) {
  return act_dtype == 1 ? launch_fused_bf16(f, scale_dtype, has_zp, st, pdl, check_only)
                        : launch_fused_f16(f, scale_dtype, has_zp, st, pdl, check_only);
}

}  // namespace qmoe
