// formats.cu -- weight-format adapters: GPTQ checkpoints and packed 4-bit
// zero points into the library's canonical layout, on the device.
//
// Source: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), "Bugs/Issues
// Found", item 1: GPTQ zero points are stored with an offset of +1
// (auto_gptq: 7 for a symmetric model) or +0 (8), told apart by the median
// stored zero.  The GPTQ bit layout is not on the pages; the one read here:
//   qweight [K/8, N] int32, bits 4j..4j+3 of word (i, n) = q[8i + j, n]
//   qzeros  [K/bs, N/8] int32, bits 4j..4j+3 of word (g, i) = stored zero of
//           block g, column 8i + j
//   scales  [K/bs, N] 16-bit
// Canonical: w [N, K/2] u8 (element 2j in the low nibble of byte j),
// scales [N, K/bs], zp [N, K/bs] u8.
//
// Byte b of qweight word (i, n) holds q[8i + 2b, n] in its low nibble and
// q[8i + 2b + 1, n] in its high nibble, which is canonical byte 4i + b of
// row n.  So the weight conversion is a transpose of the [K/8, N] matrix of
// 32-bit words into [N, K/8], and the scales a transpose of 16-bit values:
// both are shared-memory tiled transposes (coalesced 128-byte reads and
// writes), bound by HBM.  Zero points are unpacked from their words in the
// same tiled way.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

constexpr int kTile = 32;   // transpose tile (elements)
constexpr int kRowsPerPass = 8;  // block 32 x 8 threads

// out[e][c][r] = in[e][r][c], 32 x 32 tiles through shared memory
template <typename T>
__global__ void __launch_bounds__(kTile * kRowsPerPass) transpose_kernel(const T* __restrict__ in, T* __restrict__ out,
                                                                         int R, int C) {
  __shared__ T tile[kTile][kTile + 1];
  const size_t plane = (size_t)R * C;
  const T* src = in + blockIdx.z * plane;
  T* dst = out + blockIdx.z * plane;
  const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
  const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
  for (int i = 0; i < kTile; i += kRowsPerPass) {
    const int r = r0 + ty + i, c = c0 + tx;
    if (r < R && c < C) tile[ty + i][tx] = src[(size_t)r * C + c];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kTile; i += kRowsPerPass) {
    const int c = c0 + ty + i, r = r0 + tx;
    if (r < R && c < C) dst[(size_t)c * R + r] = tile[tx][ty + i];
  }
}

// zp[e][n][g] = stored(g, n) + offset from qzeros[e][g][n / 8]: a tile of
// 32 blocks x 32 words (256 columns) per CTA.  A zero point above 15 (a
// stored 15 with offset 1) is outside the 4-bit format: it is written as 15
// and reported as QMOE_ST_RANGE in *status (when given), because the
// weights of that block then differ from the checkpoint's.
__global__ void __launch_bounds__(kTile * kRowsPerPass) gptq_zeros_kernel(const uint32_t* __restrict__ qz,
                                                                          uint8_t* __restrict__ zp, int nb, int N,
                                                                          int offset, const int32_t* offset_dev,
                                                                          uint32_t* status) {
  __shared__ uint32_t tile[kTile][kTile + 1];
  const int NW = N / 8;
  const uint32_t* src = qz + (size_t)blockIdx.z * nb * NW;
  uint8_t* dst = zp + (size_t)blockIdx.z * N * nb;
  const int w0 = blockIdx.x * kTile, g0 = blockIdx.y * kTile;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int off = offset_dev ? *offset_dev : offset;
#pragma unroll
  for (int i = 0; i < kTile; i += kRowsPerPass) {
    const int g = g0 + ty + i, w = w0 + tx;
    if (g < nb && w < NW) tile[ty + i][tx] = src[(size_t)g * NW + w];
  }
  __syncthreads();
  // thread (tx, ty): block g0 + tx, columns n0 + ty + 8 m
  const int g = g0 + tx;
  bool over = false;
  for (int m = 0; m < kTile; ++m) {
    const int nl = ty + kRowsPerPass * m;  // 0 .. 255
    const int n = w0 * 8 + nl;
    if (g < nb && n < N) {
      const uint32_t word = tile[tx][nl >> 3];
      const int v = (int)((word >> (4 * (nl & 7))) & 15u) + off;
      over |= v > 15;
      dst[(size_t)n * nb + g] = (uint8_t)(v > 15 ? 15 : v);
    }
  }
  if (over && status) atomicOr(status, QMOE_ST_RANGE);
}

// offset_out = 1 if the lower median of all stored zero points is 7, else 0
// (one CTA: a 16-bin histogram in shared memory)
__global__ void __launch_bounds__(1024) gptq_zero_offset_kernel(const uint32_t* __restrict__ qz, size_t n_words,
                                                                int32_t* offset_out) {
  __shared__ unsigned long long hist[16];
  if (threadIdx.x < 16) hist[threadIdx.x] = 0;
  __syncthreads();
  unsigned long long local[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) local[v] = 0;
  for (size_t i = threadIdx.x; i < n_words; i += blockDim.x) {
    const uint32_t w = qz[i];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t v = (w >> (4 * j)) & 15u;
#pragma unroll
      for (int b = 0; b < 16; ++b) local[b] += (v == (uint32_t)b);
    }
  }
#pragma unroll
  for (int b = 0; b < 16; ++b)
    if (local[b]) atomicAdd(&hist[b], local[b]);
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long total = 0;
    for (int b = 0; b < 16; ++b) total += hist[b];
    const unsigned long long half = (total + 1) / 2;
    unsigned long long run = 0;
    int med = 0;
    for (int b = 0; b < 16; ++b) {
      run += hist[b];
      if (run >= half) {
        med = b;
        break;
      }
    }
    *offset_out = (total > 0 && med == 7) ? 1 : 0;
  }
}

// out[r][b] = nibble (b mod 2) of in[r][b / 2]
__global__ void unpack_zp_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, int rows, int nb) {
  const int pb = (nb + 1) / 2;
  const size_t total = (size_t)rows * nb;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / nb;
    const int b = (int)(i - r * nb);
    out[i] = (in[r * pb + (b >> 1)] >> (4 * (b & 1))) & 15;
  }
}

// ------------------------------------------------------------------- host

static dim3 tgrid(int rows, int cols, int E) {
  return dim3((cols + kTile - 1) / kTile, (rows + kTile - 1) / kTile, E);
}

cudaError_t launch_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int E, int K,
                               int N, int bs, int offset, const int32_t* offset_dev, uint8_t* w_out,
                               void* scales_out, uint8_t* zp_out, uint32_t* status, cudaStream_t st) {
  const dim3 blk(kTile, kRowsPerPass);
  const int nb = K / bs;
  // weights: [E][K/8][N] words -> [E][N][K/8] words
  transpose_kernel<uint32_t><<<tgrid(K / 8, N, E), blk, 0, st>>>(reinterpret_cast<const uint32_t*>(qweight),
                                                                  reinterpret_cast<uint32_t*>(w_out), K / 8, N);
  // scales: [E][nb][N] -> [E][N][nb]
  transpose_kernel<uint16_t><<<tgrid(nb, N, E), blk, 0, st>>>(static_cast<const uint16_t*>(scales),
                                                               static_cast<uint16_t*>(scales_out), nb, N);
  if (qzeros)
    gptq_zeros_kernel<<<tgrid(nb, N / 8, E), blk, 0, st>>>(reinterpret_cast<const uint32_t*>(qzeros), zp_out, nb,
                                                            N, offset, offset_dev, status);
  return cudaGetLastError();
}

cudaError_t launch_gptq_zero_offset(const int32_t* qzeros, size_t n_words, int32_t* offset_out, cudaStream_t st) {
  gptq_zero_offset_kernel<<<1, 1024, 0, st>>>(reinterpret_cast<const uint32_t*>(qzeros), n_words, offset_out);
  return cudaGetLastError();
}

cudaError_t launch_unpack_zp(const uint8_t* in, uint8_t* out, int rows, int nb, cudaStream_t st) {
  const size_t total = (size_t)rows * nb;
  const int threads = 256;
  size_t blocks = (total + threads - 1) / threads;
  const size_t cap = (size_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  unpack_zp_kernel<<<(unsigned)blocks, threads, 0, st>>>(in, out, rows, nb);
  return cudaGetLastError();
}

}  // namespace qmoe
