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

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tmap.h"

namespace qmoe {

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

// The whole CTA groups A assignments (any size) by a stable counting sort:
// thread c < CH owns the contiguous chunk [c*L, (c+1)*L) of assignments;
// per-(expert, chunk) counts are scanned in expert-major order, which gives
// each chunk its first position inside every expert; the chunks then
// scatter in order.  Up to kRouteStageIds ids are first staged with
// coalesced loads in a chunk-transposed layout (element i of chunk c at
// i*(CH+1) + c: conflict-free both ways).
__device__ void group_chunked(int A, int E, int* smem_i, const RouteParams& p, int tid, uint32_t* status) {
  const int CH = route_group_chunks(E);
  const int L = (A + CH - 1) / CH;
  int* cnt = smem_i;                   // [E][CH]
  int* tsum = cnt + E * CH;            // [256]
  int* flag = tsum + kRouteThreads;    // [256]
  int* sids = flag + kRouteThreads;    // [L][CH + 1] when staged
  const bool staged = A <= kRouteStageIds;
  if (staged)
    for (int a = tid; a < A; a += kRouteThreads) sids[(a % L) * (CH + 1) + a / L] = __ldcg(p.topk_ids + a);
  for (int i = tid; i < E * CH; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();
  const int a0 = tid * L, a1 = tid < CH ? min(A, a0 + L) : a0;
  auto id_of = [&](int a) { return staged ? sids[(a - a0) * (CH + 1) + tid] : __ldcg(p.topk_ids + a); };
  for (int a = a0; a < a1; ++a) {
    const int id = id_of(a);
    if (id < 0 || id >= E)
      set_status(status, QMOE_ST_INDEX);
    else
      cnt[id * CH + tid] += 1;
  }
  __syncthreads();
  // exclusive scan over the flattened [E][CH] counts
  const int ntot = E * CH;
  const int seg = (ntot + kRouteThreads - 1) / kRouteThreads;
  const int s0 = min(ntot, tid * seg), s1 = min(ntot, s0 + seg);
  int local = 0;
  for (int i = s0; i < s1; ++i) local += cnt[i];
  tsum[tid] = local;
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {
    const int v = tid >= o ? tsum[tid - o] : 0;
    __syncthreads();
    tsum[tid] += v;
    __syncthreads();
  }
  int run = tsum[tid] - local;
  for (int i = s0; i < s1; ++i) {
    const int c = cnt[i];
    cnt[i] = run;
    run += c;
  }
  const int total = tsum[kRouteThreads - 1];
  __syncthreads();
  // expert offsets and the list of experts with at least one assignment
  int present = 0;
  if (tid < E) {
    const int off = cnt[tid * CH];
    const int next = tid + 1 < E ? cnt[(tid + 1) * CH] : total;
    p.offsets[tid] = off;
    if (p.user_offsets) p.user_offsets[tid] = off;
    present = next > off;
  }
  if (tid == 0) {
    p.offsets[E] = total;
    if (p.user_offsets) p.user_offsets[E] = total;
  }
  flag[tid] = present;
  __syncthreads();
  for (int o = 1; o < kRouteThreads; o <<= 1) {
    const int v = tid >= o ? flag[tid - o] : 0;
    __syncthreads();
    flag[tid] += v;
    __syncthreads();
  }
  if (present) p.active[flag[tid]] = tid;  // slot 1 + exclusive rank
  if (tid == kRouteThreads - 1) p.active[0] = flag[tid];
  // scatter, each chunk in assignment order
  for (int a = a0; a < a1; ++a) {
    const int id = id_of(a);
    if (id < 0 || id >= E) continue;
    const int pos = cnt[id * CH + tid]++;
    p.perm[pos] = a;
    if (p.user_perm) p.user_perm[pos] = a;
  }
}

// One thread-block cluster of kMaxSplit CTAs per tile of TOK tokens.  CTA s
// owns rows [s*rps, (s+1)*rps) of H.  The raw x rows and the router rows are
// copied into shared memory with cp.async (all 16-byte pieces in flight at
// once), x is transposed to [row][token] fp32, and each warp accumulates 8
// tokens over every NRG-th row (NRG = 8 / (TOK / 8)) in fp32.  The row
// groups are summed in a fixed order, then, after a cluster barrier, CTA s
// sums the 8 CTAs' partial logits of its own TOK/8 tokens in rank order
// (distributed shared memory; deterministic) and runs softmax + top-k, one
// warp per token.
template <typename TA, int ME, int TOK>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  constexpr int NW = kRouteThreads / 32;
  constexpr int NTG = TOK / 8;   // token groups of 8
  constexpr int NRG = NW / NTG;  // row groups
  constexpr int TPC = TOK / NW;  // tokens per CTA in the softmax phase
  extern __shared__ __align__(16) float smem_f[];
  pdl_wait();  // x may be the previous kernel's output
  pdl_trigger();
  const uint32_t rank = cluster_ctarank();
  const int t0 = blockIdx.y * TOK;
  const int nt = min(TOK, p.T - t0);
  const int E = p.E, H = p.H, k = p.k;
  const int rps = p.rows_per_split;
  const int h0 = (int)rank * rps;
  const int rows = max(0, min(H, h0 + rps) - h0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp % NRG, tg = warp / NRG;
  uint32_t* status = p.ctl + kCtlStatus;

  const int rc = route_chunk_rows(H, E, TOK);
  float* xs = smem_f;                                               // [rps][TOK]
  uint16_t* wch = reinterpret_cast<uint16_t*>(xs + (size_t)rps * TOK);  // [rc][E]
  float* part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(wch) + route_align16((size_t)2 * rc * E));
  uint16_t* xraw = reinterpret_cast<uint16_t*>(part);              // [TOK][rps + 8], before the partials
  const int xstride = rps + 8;
  __shared__ int sh_last;

  const uint16_t* x = static_cast<const uint16_t*>(p.x);
  const uint16_t* rw = static_cast<const uint16_t*>(p.router_w);
  // rows start on 8-row boundaries, so with 16-byte-aligned bases every
  // 16-byte piece of a chunk or an x row stays aligned
  const bool vecw = (reinterpret_cast<uintptr_t>(rw) & 15) == 0;
  const bool vecx = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (H & 7) == 0;

  auto stage_rows = [&](int r0, int nr) {
    const uint16_t* src = rw + (size_t)(h0 + r0) * E;
    const int nel = nr * E;
    if (vecw) {
      const int n16 = nel >> 3;
      for (int i = tid; i < n16; i += kRouteThreads) cp_async16(wch + 8 * i, src + 8 * i);
      for (int i = (n16 << 3) + tid; i < nel; i += kRouteThreads) wch[i] = __ldg(src + i);
    } else {
      for (int i = tid; i < nel; i += kRouteThreads) wch[i] = __ldg(src + i);
    }
  };

  // ---- raw x rows and the first router chunk, all in flight together
  if (vecx) {
    const int n16 = rows >> 3;  // rows is a multiple of 8 when H is
    for (int i = tid; i < nt * n16; i += kRouteThreads) {
      const int t = i / n16, c = i - t * n16;
      cp_async16(xraw + t * xstride + 8 * c, x + (size_t)(t0 + t) * H + h0 + 8 * c);
    }
  } else {
    for (int i = tid; i < nt * rows; i += kRouteThreads) {
      const int t = i / rows, h = i - t * rows;
      xraw[t * xstride + h] = x[(size_t)(t0 + t) * H + h0 + h];
    }
  }
  stage_rows(0, min(rc, rows));
  cp_async_wait_all();
  __syncthreads();
  for (int i = tid; i < rows * TOK; i += kRouteThreads) {
    const int h = i / TOK, t = i % TOK;
    xs[i] = t < nt ? Half<TA>::to_float(xraw[t * xstride + h]) : 0.f;
  }
  __syncthreads();  // xs complete; the raw x region is free for the partials

  // ---- partial logits: 8 tokens per warp over every NRG-th row
  float acc[8][ME];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int m = 0; m < ME; ++m) acc[j][m] = 0.f;
  for (int r0 = 0; r0 < rows; r0 += rc) {
    const int nr = min(rc, rows - r0);
    if (r0 > 0) {
      __syncthreads();  // the previous chunk is consumed
      stage_rows(r0, nr);
      cp_async_wait_all();
      __syncthreads();
    }
#pragma unroll 4
    for (int h = rg; h < nr; h += NRG) {
      float wv[ME];
#pragma unroll
      for (int m = 0; m < ME; ++m) {
        const int e = lane + 32 * m;
        wv[m] = (e < E) ? Half<TA>::to_float(wch[h * E + e]) : 0.f;
      }
      const float4* xr = reinterpret_cast<const float4*>(xs + (size_t)(r0 + h) * TOK + tg * 8);
      const float4 xa = xr[0], xb = xr[1];
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int m = 0; m < ME; ++m) acc[j][m] = fmaf(xv[j], wv[m], acc[j][m]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      if (e < E) part[((size_t)rg * TOK + tg * 8 + j) * E + e] = acc[j][m];
    }
  __syncthreads();
  if (NRG > 1)  // row groups summed in a fixed order
    for (int i = tid; i < TOK * E; i += kRouteThreads) {
      float v = part[i];
#pragma unroll
      for (int g = 1; g < NRG; ++g) v += part[(size_t)g * TOK * E + i];
      part[i] = v;
    }
  cluster_sync_all();  // every CTA's partials are complete

  // ---- this CTA's tokens: rank-ordered sum of the partials, softmax, top-k
  if (warp < TPC) {
    const int tl = (int)rank * TPC + warp;
    if (tl < nt) {
      const int t = t0 + tl;
      float lg[ME];
#pragma unroll
      for (int m = 0; m < ME; ++m) {
        const int e = lane + 32 * m;
        if (e < E) {
          float pv[kMaxSplit];
#pragma unroll
          for (int r = 0; r < kMaxSplit; ++r) pv[r] = ld_dsmem_f32(part + tl * E + e, (uint32_t)r);
          float v = 0.f;
#pragma unroll
          for (int r = 0; r < kMaxSplit; ++r) v += pv[r];
          lg[m] = v + (p.bias ? p.bias[e] : 0.f);
        } else {
          lg[m] = -INFINITY;
        }
      }
      int ids[kMaxTopk];
      float wts[kMaxTopk];
      softmax_topk<ME>(lg, E, k, p.gate_sigmoid != 0, lane, ids, wts);
      if (lane < k) {
        int bi = 0;
        float bp = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxTopk; ++q)
          if (q == lane) {
            bi = ids[q];
            bp = wts[q];
          }
        const size_t a = (size_t)t * k + lane;
        p.topk_ids[a] = bi;
        p.topk_w[a] = bp;
        if (p.user_ids) p.user_ids[a] = bi;
        if (p.user_w) p.user_w[a] = bp;
      }
    }
  }
  // peers keep their shared memory until the reads above are done; the
  // barrier's release/acquire also publishes the top-k writes cluster-wide
  cluster_sync_all();

  const int A = p.T * k;
  int* smem_i = reinterpret_cast<int*>(smem_f);
  if (gridDim.y == 1) {
    // one cluster routed every token: its first CTA groups them
    if (rank == 0 && warp == 0) {
      group_one_warp(p.topk_ids, true, A, E, smem_i, smem_i + E, p, lane, status);
    }
    return;
  }

  // ---- the last CTA to finish groups all assignments by expert
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicAdd(p.ctl + kCtlGroupTicket, 1u);
    sh_last = (ticket == gridDim.x * gridDim.y - 1);
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  if (tid == 0) p.ctl[kCtlGroupTicket] = 0u;
  if (A <= 256) {
    if (warp == 0) group_one_warp(p.topk_ids, true, A, E, smem_i, smem_i + E, p, lane, status);
  } else {
    group_chunked(A, E, smem_i, p, tid, status);
  }
}

// ------------------------------------------------------------ many tokens
// Tensor-core router for T > 16: one cluster of kMaxSplit CTAs per tile of
// 128 tokens.  CTA s reduces its share of H in 64-wide K chunks with
// tcgen05.mma (M = 128 tokens, N = E rounded up to 16, fp32 accumulation in
// TMEM): the x tile arrives by TMA (128-byte swizzle, rows past T read as
// zero) and the CTA's threads transpose the router rows into the K-major
// operand.  The router weight is read once per 128 tokens instead of once
// per 8.  Products of two 16-bit values are exact in fp32; the sums are
// fp32 (tensor-core accumulation order).  The kMaxSplit partial-logit tiles
// are summed in rank order through distributed shared memory, then softmax
// + top-k per token and the grouping, as in the small-T kernel.
constexpr int kRtTok = 128;
QMOE_HD int rt_np(int E) { return (E + 15) & ~15; }
QMOE_HD uint32_t rt_stage_bytes(int E) { return 16384u + (uint32_t)rt_np(E) * 128u; }
QMOE_HD size_t rt_smem_bytes(int T, int E, int k) {
  // [barriers][2 stages: x tile 16 KB + router operand NP x 128 B][partials 128 x (NP + 1) fp32]
  const size_t compute = 1024 + 2 * (size_t)rt_stage_bytes(E) + (size_t)kRtTok * (rt_np(E) + 1) * 4 + 1024;
  const size_t A = (size_t)T * k;
  const size_t group = A > 256 ? 4 * route_group_ints((int)A, E) + 2048 : 0;  // after the 1 KB header, + alignment
  return compute > group ? compute : group;
}

template <typename TA, int ME>
__global__ void __launch_bounds__(kRouteThreads) route_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                                 RouteParams p) {
  extern __shared__ __align__(1024) uint8_t rsm_raw[];
  uint8_t* sm = rsm_raw + ((1024u - (smem_u32(rsm_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);  // [2] x tile landed
  uint64_t* mmad = full + 2;                         // [2] MMAs done with the stage
  uint64_t* acc_done = full + 4;                     // all MMAs done
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 5);
  __shared__ int sh_last;
  const int E = p.E, H = p.H, k = p.k, NP = rt_np(E), PS = NP + 1;
  const uint32_t SB = rt_stage_bytes(E);
  uint8_t* stages = sm + 1024;
  float* part = reinterpret_cast<float*>(stages + 2 * SB);  // [128][PS]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = p.ctl + kCtlStatus;
  const uint32_t rank = cluster_ctarank();
  const int t0 = blockIdx.y * kRtTok;
  const int nkc = H / 64, cpr = (nkc + kMaxSplit - 1) / kMaxSplit;
  const int c0 = (int)rank * cpr, nc = max(0, min(nkc, c0 + cpr) - c0);
  const uint32_t tcols = NP > 64 ? 128u : NP > 32 ? 64u : 32u;
  const uint16_t* rw = static_cast<const uint16_t*>(p.router_w);
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *s_tmem;
  pdl_wait();  // x may be the previous kernel's output
  pdl_trigger();
  bool ok = true;
  const uint32_t idesc = idesc_f16(128, NP, std::is_same<TA, __nv_bfloat16>::value);
  for (int c = 0; c < nc; ++c) {
    const int s = c & 1;
    uint8_t* st = stages + s * SB;
    if (c >= 2) ok = mbar_wait(&mmad[s], ((c - 2) >> 1) & 1, status) && ok;  // stage free
    if (tid == 0) {
      mbar_arrive_expect_tx(&full[s], 16384u);
      tma_load_2d(st, &tm_x, (c0 + c) * 64, t0, &full[s]);
    }
    // router rows k0 .. k0 + 63 as the K-major operand [NP][64]: 16-byte
    // group g of row n at (n / 8) * 1024 + (n % 8) * 128 + (g ^ (n % 8)) * 16
    const int k0 = (c0 + c) * 64;
    for (int idx = tid; idx < 8 * NP; idx += kRouteThreads) {
      const int n = idx % NP, g = idx / NP;
      uint32_t w4[4] = {0u, 0u, 0u, 0u};
      if (n < E) {
        const uint16_t* src = rw + (size_t)(k0 + 8 * g) * E + n;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w4[i] = (uint32_t)__ldg(src + (size_t)(2 * i) * E) | ((uint32_t)__ldg(src + (size_t)(2 * i + 1) * E) << 16);
      }
      *reinterpret_cast<uint4*>(st + 16384 + (n >> 3) * 1024 + (n & 7) * 128 + ((g ^ (n & 7)) << 4)) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the MMA reads these through the async proxy
    __syncthreads();
    if (warp == 0) {
      ok = mbar_wait(&full[s], (c >> 1) & 1, status) && ok;
      tc_fence_after();
      if (ok) {
        const uint64_t ad = sw128_desc(smem_u32(st)), bd = sw128_desc(smem_u32(st + 16384));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16_ss_elect(tb, ad + 2 * kk, bd + 2 * kk, idesc, (c | kk) != 0);
      }
      mma_commit_elect(&mmad[s]);
    }
  }
  if (warp == 0) mma_commit_elect(acc_done);
  ok = mbar_wait(acc_done, 0, status) && ok;
  tc_fence_after();
  // partial logits of this CTA's share of H: warp w < 4 reads TMEM lanes
  // (tokens) 32w .. 32w + 31
  if (warp < 4) {
    const int tl = warp * 32 + lane;
    for (int c16 = 0; c16 < NP; c16 += 16) {
      uint32_t v[16];
      if (nc > 0 && ok) {
        tmem_ld16(tb + ((uint32_t)(warp * 32) << 16) + (uint32_t)c16, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) part[tl * PS + c16 + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  cluster_sync_all();  // every CTA's partials are complete
  // ---- this CTA's 16 tokens: rank-ordered sum of the partials, softmax, top-k
  for (int q = 0; q < kRtTok / kMaxSplit / (kRouteThreads / 32); ++q) {
    const int tl = (int)rank * (kRtTok / kMaxSplit) + q * (kRouteThreads / 32) + warp;
    const int t = t0 + tl;
    if (t < p.T) {
      float lg[ME];
#pragma unroll
      for (int m = 0; m < ME; ++m) {
        const int e = lane + 32 * m;
        if (e < E) {
          float v = 0.f;
#pragma unroll
          for (int r = 0; r < kMaxSplit; ++r) v += ld_dsmem_f32(part + tl * PS + e, (uint32_t)r);
          lg[m] = v + (p.bias ? p.bias[e] : 0.f);
        } else {
          lg[m] = -INFINITY;
        }
      }
      int ids[kMaxTopk];
      float wts[kMaxTopk];
      softmax_topk<ME>(lg, E, k, p.gate_sigmoid != 0, lane, ids, wts);
      if (lane < k) {
        int bi = 0;
        float bp = 0.f;
#pragma unroll
        for (int qq = 0; qq < kMaxTopk; ++qq)
          if (qq == lane) {
            bi = ids[qq];
            bp = wts[qq];
          }
        const size_t a = (size_t)t * k + lane;
        p.topk_ids[a] = bi;
        p.topk_w[a] = bp;
        if (p.user_ids) p.user_ids[a] = bi;
        if (p.user_w) p.user_w[a] = bp;
      }
    }
  }
  cluster_sync_all();  // peers keep their partials until the reads above are done
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, tcols);
  }
  const int A = p.T * k;
  int* smem_i = reinterpret_cast<int*>(sm + 1024);
  // ---- the last CTA to finish groups all assignments by expert
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicAdd(p.ctl + kCtlGroupTicket, 1u);
    sh_last = (ticket == gridDim.x * gridDim.y - 1);
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  if (tid == 0) p.ctl[kCtlGroupTicket] = 0u;
  if (A <= 256) {
    if (warp == 0) group_one_warp(p.topk_ids, true, A, E, smem_i, smem_i + E, p, lane, status);
  } else {
    group_chunked(A, E, smem_i, p, tid, status);
  }
}

bool route_tc_fits(int T, int H, int E, int k) {
  return T > kDecodeMaxTokens && H % 64 == 0 && H >= 64 && E >= 1 && E <= 128 &&
         rt_smem_bytes(T, E, k) <= 227 * 1024;
}

template <typename TA, int ME>
static cudaError_t launch_route_tc_me(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl) {
  CUtensorMap m;
  if (!make_map(&m, p.x, act_dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                (uint64_t)p.H, (uint64_t)p.T, 64, kRtTok, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  const size_t smem = rt_smem_bytes(p.T, p.E, p.k);
  auto fn = route_tc_kernel<TA, ME>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxSplit, (p.T + kRtTok - 1) / kRtTok);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kMaxSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fn, m, p);
}

template <typename TA>
static cudaError_t launch_route_tc(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl) {
  const int me = (p.E + 31) / 32;
  if (me <= 1) return launch_route_tc_me<TA, 1>(p, act_dtype, st, pdl);
  if (me <= 2) return launch_route_tc_me<TA, 2>(p, act_dtype, st, pdl);
  return launch_route_tc_me<TA, 4>(p, act_dtype, st, pdl);
}

template <typename TA, int ME, int TOK>
static cudaError_t launch_route_me(const RouteParams& p, cudaStream_t st, bool pdl, size_t smem) {
  const int tiles = (p.T + TOK - 1) / TOK;
  auto fn = route_kernel<TA, ME, TOK>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxSplit, tiles);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kMaxSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename TA>
static cudaError_t launch_route_t(const RouteParams& p, cudaStream_t st, bool pdl) {
  const size_t smem = route_smem_bytes(p.T, p.H, p.E, p.k);
  const int me = (p.E + 31) / 32;
  if (route_tokens(p.T, p.E) == 32) {
    if (me <= 1) return launch_route_me<TA, 1, 32>(p, st, pdl, smem);
    return launch_route_me<TA, 2, 32>(p, st, pdl, smem);
  }
  if (me <= 1) return launch_route_me<TA, 1, 8>(p, st, pdl, smem);
  if (me <= 2) return launch_route_me<TA, 2, 8>(p, st, pdl, smem);
  if (me <= 4) return launch_route_me<TA, 4, 8>(p, st, pdl, smem);
  return launch_route_me<TA, 8, 8>(p, st, pdl, smem);
}

cudaError_t launch_route(const RouteParams& p, int act_dtype, cudaStream_t st, bool pdl) {
  if (route_tc_fits(p.T, p.H, p.E, p.k) && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0)
    return act_dtype == 1 ? launch_route_tc<__nv_bfloat16>(p, act_dtype, st, pdl)
                          : launch_route_tc<__half>(p, act_dtype, st, pdl);
  return act_dtype == 1 ? launch_route_t<__nv_bfloat16>(p, st, pdl)
                        : launch_route_t<__half>(p, st, pdl);
}

}  // namespace qmoe
