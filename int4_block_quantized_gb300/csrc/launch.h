// launch.h -- internal host-side declarations: kernel launchers and the
// cudaLaunchKernelEx helper (programmatic dependent launch attribute).
#pragma once

#include <cuda_runtime.h>

#include "layout.h"

namespace qmoe {

template <typename... Args>
static inline cudaError_t launch_kernel(void (*fn)(Args...), dim3 grid, dim3 block, size_t smem,
                                        cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

// number of SMs of the current device (cached per device)
int device_sm_count();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per function, device
// and size (not a stream operation; cached so graph capture sees no calls)
cudaError_t ensure_smem_ptr(const void* fn, size_t bytes);
template <typename F>
static inline cudaError_t ensure_smem(F* fn, size_t bytes) {
  return ensure_smem_ptr(reinterpret_cast<const void*>(fn), bytes);
}

cudaError_t launch_route(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl);

// decode path: returns cudaErrorInvalidValue if the shape does not fit the
// kernel's shared-memory plan (the caller then reports UNSUPPORTED)
cudaError_t launch_decode(DecodeParams p, int mode, int act_dtype, int scale_dtype, bool has_zp,
                          cudaStream_t st, bool pdl);
bool decode_fits(int mode, int T, int N, int K, int bs, bool has_zp, int k);
// weight-format adapters (formats.cu)
cudaError_t launch_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int E, int K,
                               int N, int bs, int offset, const int32_t* offset_dev, uint8_t* w_out,
                               void* scales_out, uint8_t* zp_out, uint32_t* status, cudaStream_t st);
cudaError_t launch_gptq_zero_offset(const int32_t* qzeros, size_t n_words, int32_t* offset_out, cudaStream_t st);
cudaError_t launch_unpack_zp(const uint8_t* in, uint8_t* out, int rows, int nb, cudaStream_t st);
// fused decode layer (T <= kTokGroup): cudaErrorInvalidValue if the plan
// does not fit; check_only: plan only, nothing launched
cudaError_t launch_fused(const FusedParams& f, int act_dtype, int scale_dtype, bool has_zp, cudaStream_t st,
                         bool pdl, bool check_only);
cudaError_t launch_fused_f16(const FusedParams& f, int scale_dtype, bool has_zp, cudaStream_t st, bool pdl,
                             bool check_only);
cudaError_t launch_fused_bf16(const FusedParams& f, int scale_dtype, bool has_zp, cudaStream_t st, bool pdl,
                              bool check_only);

// prefill path: token gather + tile table, the two grouped GEMMs (mode 0
// gate-up with SwiGLU, mode 1 down with the weighted scatter-add), and the
// final fp32 -> act_dtype conversion (plus residual)
bool prefill_fits(int H, int I, int bs, int act_dtype, int scale_dtype, bool has_zp_gu, bool has_zp_d);
// dense MatMulNBits on the grouped GEMM (down mode, one expert): N outputs, K inputs
bool dense_fits(int N, int K, int bs, int act_dtype, int scale_dtype, bool has_zp);
// true if the GEMM's operands are fp16 while x is bf16 (x converted on gather)
bool prefill_x_to_f16(int act_dtype, int scale_dtype);
cudaError_t launch_dense_setup(const PrefillParams& p, const void* x, cudaStream_t st, bool pdl);
cudaError_t launch_prefill_permute(const PrefillParams& p, const void* x, int act_dtype, cudaStream_t st,
                                   bool pdl);
cudaError_t launch_prefill_gemm(const PrefillParams& p, int mode, int act_dtype, int scale_dtype, bool dense,
                                cudaStream_t st, bool pdl);
cudaError_t launch_prefill_convert(const PrefillParams& p, void* out, int act_dtype, cudaStream_t st,
                                   bool pdl);

cudaError_t launch_dequant(const uint8_t* w, const void* s, int scale_dtype, const uint8_t* zp,
                           int N, int K, int bs, float* out, cudaStream_t st);
cudaError_t launch_rmsnorm(const void* x, void* out, int act_dtype, int T, int H, float eps,
                           cudaStream_t st);

}  // namespace qmoe
