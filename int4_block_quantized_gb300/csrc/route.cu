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
// 16-bit loads (lane = expert) and accumulates fp32 for all 8 tokens.  For
// small T the H reduction is split over a thread-block cluster of up to 8
// CTAs whose partial logits are summed, in a fixed order, by the cluster's
// first CTA through distributed shared memory (no global round trip).  One
// warp per token then does the softmax and k rounds of warp-shuffle argmax.
// Grouping by expert is a stable counting sort ranked with __match_any_sync:
// one warp when there are at most 256 assignments, else all warps of the
// last CTA to finish.  Deterministic: no floating-point atomics.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t addr = smem_u32(local), raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}

// Warp-wide exclusive scan of `v` over lanes.
__device__ __forceinline__ int warp_excl_scan(int v, int lane) {
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}

// One warp groups A <= 256 assignments by expert (stable).  ids: expert of
// each assignment (shared or global memory); cnt / run: shared int[E].
__device__ void group_one_warp(const int32_t* ids, bool ids_global, int A, int E, int* cnt, int* run,
                               const RouteParams& p, int lane, uint32_t* status) {
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  for (int base = 0; base < A; base += 32) {
    const int a = base + lane;
    int id = -1;
    if (a < A) id = ids_global ? __ldcg(ids + a) : ids[a];
    if (a < A && (id < 0 || id >= E)) {
      set_status(status, QMOE_ST_INDEX);
      id = -1;
    }
    const uint32_t m = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(m) - 1) cnt[id] += __popc(m);
    __syncwarp();
  }
  // exclusive prefix over experts: lane owns experts [8*lane, 8*lane + 8)
  int c[8], f[8], sc = 0, sf = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane * 8 + j;
    c[j] = e < E ? cnt[e] : 0;
    f[j] = c[j] > 0;
    sc += c[j];
    sf += f[j];
  }
  int oc = warp_excl_scan(sc, lane), of = warp_excl_scan(sf, lane);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane * 8 + j;
    if (e < E) {
      run[e] = oc;
      p.offsets[e] = oc;
      if (p.user_offsets) p.user_offsets[e] = oc;
      if (f[j]) p.active[1 + of] = e;
    }
    oc += c[j];
    of += f[j];
  }
  if (lane == 31) {
    p.offsets[E] = A;
    if (p.user_offsets) p.user_offsets[E] = A;
    p.active[0] = of;
  }
  __syncwarp();
  for (int base = 0; base < A; base += 32) {
    const int a = base + lane;
    int id = -1;
    if (a < A) id = ids_global ? __ldcg(ids + a) : ids[a];
    if (id >= E) id = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, id);
    if (id >= 0) {
      const int pos = run[id] + __popc(m & ((1u << lane) - 1u));
      p.perm[pos] = a;
      if (p.user_perm) p.user_perm[pos] = a;
    }
    __syncwarp();
    if (id >= 0 && lane == __ffs(m) - 1) run[id] += __popc(m);
    __syncwarp();
  }
}

// All 8 warps of one CTA group A assignments (any size; stable).
__device__ void group_block(int A, int E, int* smem_i, const RouteParams& p, int tid,
                           uint32_t* status) {
  const int warp = tid >> 5, lane = tid & 31;
  int* cntw = smem_i;                                  // [8 warps][E]
  int* tot = cntw + (kRouteThreads / 32) * E;         // [256]
  int* scan = tot + kRouteThreads;                    // [256]
  for (int i = tid; i < (kRouteThreads / 32) * E; i += kRouteThreads) cntw[i] = 0;
  __syncthreads();
  const int slab = (A + 7) / 8;
  const int a_beg = warp * slab, a_end = min(A, a_beg + slab);
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
    int r = 0;
    for (int w = 0; w < kRouteThreads / 32; ++w) {
      const int c = cntw[w * E + tid];
      cntw[w * E + tid] = r;
      r += c;
    }
    tot[tid] = r;
  } else {
    tot[tid] = 0;
  }
  scan[tid] = tot[tid];
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {
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

// CLUSTER: gridDim.x H-splits form one cluster per token tile.
template <typename TA, int ME, bool CLUSTER>
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

  float* xs = smem_f;                                // [8][rps]
  float* red = smem_f + kRouteTokens * rps;          // [8 warps][8 tokens][E]
  __shared__ int sh_last;
  __shared__ int s_ids[kRouteTokens * kMaxTopk];

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
#pragma unroll 8
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

  // ---- combine the 8 warps in a fixed order (into red[0 .. 8E))
  const int nlog = kRouteTokens * E;
  for (int i = tid; i < nlog; i += kRouteThreads) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteThreads / 32; ++w) v += red[w * nlog + i];
    red[i] = v;
  }

  if (CLUSTER) {
    // the cluster's first CTA sums all splits' partials through DSMEM
    cluster_sync_all();
    const uint32_t rank = cluster_ctarank();
    if (rank == 0) {
      for (int i = tid; i < nlog; i += kRouteThreads) {
        float v = red[i];
        for (int r = 1; r < p.split; ++r) v += ld_dsmem_f32(red + i, (uint32_t)r);
        red[i] = v;
      }
    }
    cluster_sync_all();  // peers keep their shared memory until the reads are done
    if (rank != 0) return;
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
        s_ids[warp * k + j] = bi;
        if (p.user_ids) p.user_ids[a] = bi;
        if (p.user_w) p.user_w[a] = bp;
      }
    }
  }

  const int A = p.T * k;
  int* smem_i = reinterpret_cast<int*>(smem_f);
  if (tiles == 1) {
    // this CTA routed every token: group straight from shared memory
    __syncthreads();
    if (warp == 0) group_one_warp(s_ids, false, A, E, smem_i, smem_i + E, p, lane, status);
    return;
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
  if (A <= 256) {
    if (warp == 0) group_one_warp(p.topk_ids, true, A, E, smem_i, smem_i + E, p, lane, status);
  } else {
    group_block(A, E, smem_i, p, tid, status);
  }
}

template <typename TA, int ME>
static cudaError_t launch_route_me(const RouteParams& p, cudaStream_t st, bool pdl, size_t smem) {
  const int tiles = (p.T + kRouteTokens - 1) / kRouteTokens;
  dim3 grid(p.split, tiles);
  if (p.split > 1) {
    auto fn = route_kernel<TA, ME, true>;
    cudaError_t err = ensure_smem(fn, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
  }
  auto fn = route_kernel<TA, ME, false>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(fn, grid, dim3(kRouteThreads), smem, st, pdl, p);
}

template <typename TA>
static cudaError_t launch_route_t(const RouteParams& p, cudaStream_t st, bool pdl) {
  size_t smem = sizeof(float) * ((size_t)kRouteTokens * p.rows_per_split +
                                 (size_t)(kRouteThreads / 32) * kRouteTokens * p.E);
  const size_t grp = sizeof(int) * ((size_t)(kRouteThreads / 32) * p.E + 2 * kRouteThreads);
  if (smem < grp) smem = grp;
  const int me = (p.E + 31) / 32;
  if (me <= 1) return launch_route_me<TA, 1>(p, st, pdl, smem);
  if (me <= 2) return launch_route_me<TA, 2>(p, st, pdl, smem);
  if (me <= 4) return launch_route_me<TA, 4>(p, st, pdl, smem);
  return launch_route_me<TA, 8>(p, st, pdl, smem);
}

cudaError_t launch_route(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl) {
  return act_dtype == 1 ? launch_route_t<__nv_bfloat16>(p, st, pdl)
                        : launch_route_t<__half>(p, st, pdl);
}

}  // namespace qmoe
