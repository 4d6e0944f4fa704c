// route.cu -- fused router: fp32 gate GEMV, softmax over all experts, top-k,
// and the token->expert grouping (histogram, prefix sum, stable permutation).
//
// Source: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), IR guide
// section 3 "MoE Block", Router (TopK via extern GPU kernel): gate linear
// hidden[T,H] x W_gate[H,E], softmax in f32 over the E logits, then the top-k
// probabilities best-first (kernel internals steps 1-3); grouping of the
// flattened assignments by expert from "Optimization Opportunities" item 9
// step 1 ("sort tokens by expert").
//
// GB300 design (not the pages' one-thread-per-token kernel): a CTA owns 8
// tokens; each warp streams a strided subset of router rows with coalesced
// 16-bit loads (lane = expert) and accumulates fp32 for all 8 tokens; the H
// reduction is split over up to 16 CTAs for small T, partial sums combined in
// a fixed order by the last CTA of each token tile (deterministic).  One warp
// per token then does the softmax and k rounds of warp-shuffle argmax.  The
// last CTA overall groups assignments by expert with __match_any_sync ranks:
// a stable counting sort, no global atomics besides the completion tickets.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

template <typename TA, int ME>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  extern __shared__ __align__(16) float smem_f[];
  pdl_wait();  // x may be the previous kernel's output
  pdl_trigger();
  const int split = blockIdx.x;
  const int tile = blockIdx.y;
  const int tiles = gridDim.y;
  const int t0 = tile * kRouteTokens;
  const int nt = min(kRouteTokens, p.T - t0);
  const int E = p.E, H = p.H, k = p.k;
  const int rps = p.rows_per_split;
  const int h0 = split * rps;
  const int rows = max(0, min(H, h0 + rps) - h0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = p.ctl + kCtlStatus;

  float* xs = smem_f;                           // [8][rps]
  float* red = smem_f + kRouteTokens * rps;     // [8 warps][8 tokens][E]
  __shared__ int sh_last;

  const uint16_t* x = static_cast<const uint16_t*>(p.x);
  const uint16_t* rw = static_cast<const uint16_t*>(p.router_w);

  for (int i = tid; i < kRouteTokens * rows; i += kRouteThreads) {
    const int t = i / rows, h = i - t * rows;
    xs[t * rps + h] = (t < nt) ? Half<TA>::to_float(x[(size_t)(t0 + t) * H + h0 + h]) : 0.f;
  }
  __syncthreads();

  // ---- partial logits over this CTA's rows, fp32 accumulate
  float acc[kRouteTokens][ME];
#pragma unroll
  for (int t = 0; t < kRouteTokens; ++t)
#pragma unroll
    for (int m = 0; m < ME; ++m) acc[t][m] = 0.f;
#pragma unroll 4
  for (int h = warp; h < rows; h += kRouteThreads / 32) {
    const uint16_t* row = rw + (size_t)(h0 + h) * E;
    float wv[ME];
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      wv[m] = (e < E) ? Half<TA>::to_float(__ldg(row + e)) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) {
      const float xv = xs[t * rps + h];
#pragma unroll
      for (int m = 0; m < ME; ++m) acc[t][m] = fmaf(xv, wv[m], acc[t][m]);
    }
  }
#pragma unroll
  for (int t = 0; t < kRouteTokens; ++t)
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      if (e < E) red[(warp * kRouteTokens + t) * E + e] = acc[t][m];
    }
  __syncthreads();

  // ---- combine the 8 warps in a fixed order
  const int nlog = kRouteTokens * E;
  for (int i = tid; i < nlog; i += kRouteThreads) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteThreads / 32; ++w) v += red[w * nlog + i];
    if (p.split > 1)
      p.partial[((size_t)split * tiles + tile) * nlog + i] = v;
    else
      red[i] = v;
  }

  if (p.split > 1) {
    // the last of this tile's split CTAs combines the partials (fixed order)
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t ticket = atomicAdd(p.ctl + kCtlTileTicket0 + tile, 1u);
      sh_last = (ticket == (uint32_t)(p.split - 1));
    }
    __syncthreads();
    if (!sh_last) return;
    __threadfence();
    if (tid == 0) p.ctl[kCtlTileTicket0 + tile] = 0u;
    for (int i = tid; i < nlog; i += kRouteThreads) {
      float v = 0.f;
      for (int s = 0; s < p.split; ++s) v += __ldcg(p.partial + ((size_t)s * tiles + tile) * nlog + i);
      red[i] = v;
    }
  }
  __syncthreads();

  // ---- softmax + top-k: one warp per token
  if (warp < nt) {
    const int t = t0 + warp;
    float lg[ME];
    float mx = -INFINITY;
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      lg[m] = (e < E) ? red[warp * E + e] + (p.bias ? p.bias[e] : 0.f) : -INFINITY;
      mx = fmaxf(mx, lg[m]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float ex[ME], sum = 0.f;
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      ex[m] = (lane + 32 * m < E) ? expf(lg[m] - mx) : 0.f;
      sum += ex[m];
    }
    sum = warp_sum(sum);
    float pr[ME];
#pragma unroll
    for (int m = 0; m < ME; ++m) pr[m] = ex[m] / sum;
    uint32_t chosen = 0;
    for (int j = 0; j < k; ++j) {
      float bp = -1.f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int m = 0; m < ME; ++m) {
        const int e = lane + 32 * m;
        if (e < E && !((chosen >> m) & 1u) && pr[m] > bp) {
          bp = pr[m];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (op > bp || (op == bp && oi < bi)) {
          bp = op;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) chosen |= 1u << (bi >> 5);
      if (lane == 0) {
        const size_t a = (size_t)t * k + j;
        p.topk_ids[a] = bi;
        p.topk_w[a] = bp;
        if (p.user_ids) p.user_ids[a] = bi;
        if (p.user_w) p.user_w[a] = bp;
      }
    }
  }

  // ---- the last tile to finish groups all assignments by expert
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicAdd(p.ctl + kCtlGroupTicket, 1u);
    sh_last = (ticket == (uint32_t)(tiles - 1));
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  if (tid == 0) p.ctl[kCtlGroupTicket] = 0u;

  const int A = p.T * k;
  int* cntw = reinterpret_cast<int*>(smem_f);                 // [8 warps][E]
  int* tot = cntw + (kRouteThreads / 32) * E;                 // [256]
  int* scan = tot + kRouteThreads;                            // [256]
  for (int i = tid; i < (kRouteThreads / 32) * E; i += kRouteThreads) cntw[i] = 0;
  __syncthreads();
  const int slab = (A + 7) / 8;
  const int a_beg = warp * slab, a_end = min(A, a_beg + slab);
  // pass 1: per-warp counts
  for (int base = a_beg; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int id = valid ? __ldcg(p.topk_ids + a) : -1;
    if (valid && (id < 0 || id >= E)) {
      set_status(status, QMOE_ST_INDEX);
      id = -1;
    }
    const uint32_t mask = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(mask) - 1) cntw[warp * E + id] += __popc(mask);
    __syncwarp();
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < kRouteThreads / 32; ++w) {
      const int c = cntw[w * E + tid];
      cntw[w * E + tid] = run;
      run += c;
    }
    tot[tid] = run;
  } else {
    tot[tid] = 0;
  }
  scan[tid] = tot[tid];
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {  // inclusive scan over experts
    const int v = (tid >= o) ? scan[tid - o] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int excl = scan[tid] - tot[tid];
  if (tid < E) {
    p.offsets[tid] = excl;
    if (p.user_offsets) p.user_offsets[tid] = excl;
    for (int w = 0; w < kRouteThreads / 32; ++w) cntw[w * E + tid] += excl;
  }
  if (tid == 0) {
    p.offsets[E] = A;
    if (p.user_offsets) p.user_offsets[E] = A;
  }
  __syncthreads();
  // active experts, increasing id: scan of (count > 0) flags
  scan[tid] = (tid < E && tot[tid] > 0) ? 1 : 0;
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {
    const int v = (tid >= o) ? scan[tid - o] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  if (tid < E && tot[tid] > 0) p.active[scan[tid]] = tid;  // slot 1 + exclusive rank
  if (tid == kRouteThreads - 1) p.active[0] = scan[tid];
  // pass 2: stable positions
  for (int base = a_beg; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int id = valid ? __ldcg(p.topk_ids + a) : -1;
    if (id >= E) id = -1;
    const uint32_t mask = __match_any_sync(0xffffffffu, id);
    if (id >= 0) {
      const int pos = cntw[warp * E + id] + __popc(mask & ((1u << lane) - 1u));
      p.perm[pos] = a;
      if (p.user_perm) p.user_perm[pos] = a;
    }
    __syncwarp();
    if (id >= 0 && lane == __ffs(mask) - 1) cntw[warp * E + id] += __popc(mask);
    __syncwarp();
  }
}

template <typename TA>
static cudaError_t launch_route_t(const RouteParams& p, cudaStream_t st, bool pdl) {
  const int tiles = (p.T + kRouteTokens - 1) / kRouteTokens;
  dim3 grid(p.split, tiles);
  size_t smem = sizeof(float) * ((size_t)kRouteTokens * p.rows_per_split +
                                 (size_t)(kRouteThreads / 32) * kRouteTokens * p.E);
  const size_t grp = sizeof(int) * ((size_t)(kRouteThreads / 32) * p.E + 2 * kRouteThreads);
  if (smem < grp) smem = grp;
  const int me = (p.E + 31) / 32;
  void (*fn)(RouteParams) = nullptr;
  if (me <= 1) fn = route_kernel<TA, 1>;
  else if (me <= 2) fn = route_kernel<TA, 2>;
  else if (me <= 4) fn = route_kernel<TA, 4>;
  else fn = route_kernel<TA, 8>;
  cudaError_t err = cudaSuccess;
  if (me <= 1) err = ensure_smem(route_kernel<TA, 1>, smem);
  else if (me <= 2) err = ensure_smem(route_kernel<TA, 2>, smem);
  else if (me <= 4) err = ensure_smem(route_kernel<TA, 4>, smem);
  else err = ensure_smem(route_kernel<TA, 8>, smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(fn, grid, dim3(kRouteThreads), smem, st, pdl, p);
}

cudaError_t launch_route(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl) {
  return act_dtype == 1 ? launch_route_t<__nv_bfloat16>(p, st, pdl)
                        : launch_route_t<__half>(p, st, pdl);
}

}  // namespace qmoe
