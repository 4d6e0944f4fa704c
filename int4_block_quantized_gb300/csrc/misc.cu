// misc.cu -- small kernels: standalone DequantizeLinear (fp32 out) and the
// layer stack's RMSNorm.
//
// Sources: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34): local fix A1
// (DequantizeLinear with block_size: extui -> uitofp -> subf -> mulf) and IR
// guide section 1 (RMSNorm: x / sqrt(mean(x^2) + eps) in f32, cast back).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

cudaError_t ensure_smem_ptr(const void* fn, size_t bytes) {
  struct Entry {
    const void* fn;
    int dev;
    size_t bytes;
  };
  static Entry table[256];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].dev == dev) {
      table[i].bytes = bytes;
      return cudaSuccess;
    }
  if (n < 256) table[n++] = Entry{fn, dev, bytes};
  return cudaSuccess;
}

// One thread per 8 codes (one 32-bit word of a row).  (q - zp) * scale is
// computed as float(q - zp) * scale: the integer difference and the product
// of a <=5-bit integer with a 16-bit float are exact in fp32.
template <typename TS, bool HAS_ZP>
__global__ void dequant_kernel(const uint8_t* __restrict__ w, const uint16_t* __restrict__ s,
                               const uint8_t* __restrict__ zp, int N, int K, int bs,
                               float* __restrict__ out) {
  const long long words = (long long)N * (K / 8);
  const int nb = K / bs;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < words;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i / (K / 8));
    const int k0 = (int)(i - (long long)n * (K / 8)) * 8;
    const uint32_t v = *reinterpret_cast<const uint32_t*>(w + (size_t)n * (K / 2) + k0 / 2);
    const int b = k0 / bs;  // 8 | bs, so all 8 codes share one block
    const float sc = Half<TS>::to_float(s[(size_t)n * nb + b]);
    const int z = HAS_ZP ? (int)zp[(size_t)n * nb + b] : 8;
    float r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = (float)((int)((v >> (4 * j)) & 15u) - z) * sc;
    float4* o = reinterpret_cast<float4*>(out + (size_t)n * K + k0);
    o[0] = make_float4(r[0], r[1], r[2], r[3]);
    o[1] = make_float4(r[4], r[5], r[6], r[7]);
  }
}

cudaError_t launch_dequant(const uint8_t* w, const void* s, int scale_dtype, const uint8_t* zp,
                           int N, int K, int bs, float* out, cudaStream_t st) {
  const long long words = (long long)N * (K / 8);
  const int threads = 256;
  long long blocks = (words + threads - 1) / threads;
  const long long cap = (long long)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const uint16_t* sp = static_cast<const uint16_t*>(s);
  if (scale_dtype == 1) {
    if (zp) dequant_kernel<__nv_bfloat16, true><<<(int)blocks, threads, 0, st>>>(w, sp, zp, N, K, bs, out);
    else dequant_kernel<__nv_bfloat16, false><<<(int)blocks, threads, 0, st>>>(w, sp, zp, N, K, bs, out);
  } else {
    if (zp) dequant_kernel<__half, true><<<(int)blocks, threads, 0, st>>>(w, sp, zp, N, K, bs, out);
    else dequant_kernel<__half, false><<<(int)blocks, threads, 0, st>>>(w, sp, zp, N, K, bs, out);
  }
  return cudaGetLastError();
}

// One CTA per token row; sum of squares in fp32 (fixed reduction order),
// then x * (1 / sqrt(mean + eps)) rounded to the activation type.
template <typename TA>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* x, uint16_t* out, int H, float eps) {
  pdl_wait();
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * H;
  float ss = 0.f;
  for (int h = threadIdx.x; h < H; h += 256) {
    const float v = Half<TA>::to_float(xr[h]);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  pdl_trigger();
  uint16_t* orow = out + (size_t)t * H;
  for (int h = threadIdx.x; h < H; h += 256) orow[h] = Half<TA>::from_float(Half<TA>::to_float(xr[h]) * inv);
}

cudaError_t launch_rmsnorm(const void* x, void* out, int act_dtype, int T, int H, float eps,
                           cudaStream_t st) {
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  uint16_t* op = static_cast<uint16_t*>(out);
  if (act_dtype == 1)
    return launch_kernel(rmsnorm_kernel<__nv_bfloat16>, dim3(T), dim3(256), 0, st, true, xp, op, H, eps);
  return launch_kernel(rmsnorm_kernel<__half>, dim3(T), dim3(256), 0, st, true, xp, op, H, eps);
}

}  // namespace qmoe
