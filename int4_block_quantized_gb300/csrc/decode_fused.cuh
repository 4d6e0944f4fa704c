// decode_fused.cuh -- the whole decode layer (router, gate-up with SwiGLU,
// down with the routing-weighted sum) in one cooperative launch, on the
// building blocks of decode_core.cuh.  The kernel and its host plan are
// templates here; decode_fused_f16.cu and decode_fused_bf16.cu instantiate
// them for each activation dtype (two translation units built in parallel).
//
// Sources: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), IR guide
// section 3 (MoE block: router TopK, Expert Computation steps 4-7) and the
// "Fused MoE Extern Kernels" update (kernel 1: gate + up with SwiGLU and
// the INT4 dequantisation inside the dot product; kernel 2: down with the
// routing-weighted reduce).
#pragma once

#include "decode_core.cuh"

namespace qmoe {
// ------------------------------------------------------------ fused layer
// The whole layer in one cooperative launch for T <= kTokGroup tokens:
//  1. router: a cluster of CL CTAs covers the router's 8 row splits of H
//     (kMaxSplit / CL splits per CTA) with the same fp32 operation order as
//     the router kernel (row groups h mod 8 summed in order, splits summed
//     in rank order through distributed shared memory), so every cluster
//     computes bit-identical logits and top-k, and no routing round trip
//     through global memory is needed;
//  2. gate-up + SwiGLU over the CTA's share of the selected experts' rows
//     (as the gate-up kernel), while the producer already streams this
//     CTA's down-projection weights into a second ring;
//  3. a grid barrier (all CTAs co-resident: cooperative launch) publishes
//     every SwiGLU output; the producer then fetches the activation rows of
//     the down stages and the down projection with the weighted sum over the
//     k experts finishes as in the down kernel.
constexpr uint32_t kFOffActive = 512;                                // bars: 4 rings x 8 + 1
constexpr uint32_t kFOffOff = kFOffActive + 4 * (kMaxExperts + 2);
constexpr uint32_t kFOffIds = kFOffOff + 4 * (kMaxExperts + 2);
constexpr uint32_t kFOffPerm = kFOffIds + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffWt = kFOffPerm + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffCnt = kFOffWt + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffMisc = kFOffCnt + 4 * kMaxExperts;
constexpr uint32_t kFFixed = (kFOffMisc + 16 + 127) & ~127u;
constexpr int kFusedCluster = 4;

template <typename TS, typename TA, bool HAS_ZP, int ME, int CL>
__global__ void __launch_bounds__(kDecodeThreads, 1) fused_decode_kernel(FusedParams f, FusedPlan P) {
  constexpr int VR = kMaxSplit / CL;  // router splits per CTA
  constexpr int NT = kDecodeThreads;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full_g = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_g = full_g + kMaxSlots;
  uint64_t* full_d = full_g + 2 * kMaxSlots;
  uint64_t* empty_d = full_g + 3 * kMaxSlots;
  uint64_t* gbar = full_g + 4 * kMaxSlots;
  int* s_active = reinterpret_cast<int*>(smem + kFOffActive);
  int* s_off = reinterpret_cast<int*>(smem + kFOffOff);
  int* s_ids = reinterpret_cast<int*>(smem + kFOffIds);
  int* s_perm = reinterpret_cast<int*>(smem + kFOffPerm);
  float* s_wt = reinterpret_cast<float*>(smem + kFOffWt);
  int* s_cnt = reinterpret_cast<int*>(smem + kFOffCnt);
  int* s_misc = reinterpret_cast<int*>(smem + kFOffMisc);  // nsg, nsd, abort
  float* res = reinterpret_cast<float*>(smem + P.res_off);
  StageEnt* stg = reinterpret_cast<StageEnt*>(smem + P.stg_off);
  StageEnt* std_ = reinterpret_cast<StageEnt*>(smem + P.std_off);
  uint8_t* ring_g = smem + P.ring_g;
  uint8_t* ring_d = smem + P.ring_d;
  // router scratch (xs, part, wch) inside the rings: no copy lands there
  // before routing ends
  float* xs = reinterpret_cast<float*>(smem + P.xs_off);        // [VR*rps][4]
  float* part = reinterpret_cast<float*>(smem + P.part_off);    // [VR][8][4][E]
  float* vpart = reinterpret_cast<float*>(smem + P.vpart_off);  // [VR][4][E], read by the cluster (own region)
  uint16_t* wch = reinterpret_cast<uint16_t*>(smem + P.wch_off);  // [pass_rows][E]

  const DecodeParams& g = f.g;
  const DecodeParams& d = f.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = g.ctl + kCtlStatus;
  const int T = g.T, H = g.K, E = g.E, k = g.k, A = T * k;
  const int NSg = P.g.nslots, NSd = P.d.nslots;
  // launched in clusters of CL covering the grid, or not at all: every CTA
  // sees the same values, so all return together before any cluster access
  if (CL > 1 && (cluster_nctarank() != (uint32_t)CL || cluster_count_x() * CL != gridDim.x)) {
    if (tid == 0) set_status(g.ctl + kCtlStatus, QMOE_ST_INDEX);
    return;
  }
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int rps = f.rps;
  const int hc0 = (int)rank * VR * rps;
  const int rows = max(0, min(H, hc0 + VR * rps) - hc0);

  if (tid == 0) {
    for (int i = 0; i < NSg; ++i) {
      mbar_init(&full_g[i], 32);
      mbar_init(&empty_g[i], kCW);
    }
    for (int i = 0; i < NSd; ++i) {
      mbar_init(&full_d[i], 32);
      mbar_init(&empty_d[i], kCW);
    }
    mbar_init(gbar, 1);
    fence_barrier_init();
  }

  // ---- 1. router.  The weight rows do not depend on the previous grid:
  //         the first pass is in flight before waiting for it.
  const uint16_t* rw = static_cast<const uint16_t*>(f.router_w);
  const bool vecw = (reinterpret_cast<uintptr_t>(rw) & 15) == 0;  // rows start on 8-row boundaries
  auto stage_rows = [&](int p0, int np) {
    const uint16_t* src = rw + (size_t)(hc0 + p0) * E;
    const int nel = np * E;
    const int n16 = vecw ? nel >> 3 : 0;
    for (int i = tid; i < n16; i += NT) cp_async16(wch + 8 * i, src + 8 * i);
    for (int i = (n16 << 3) + tid; i < nel; i += NT) wch[i] = __ldg(src + i);
  };
  if (rows > 0) stage_rows(0, min(P.pass_rows, rows));
  pdl_wait();  // x may be the previous kernel's output
  const uint16_t* x = static_cast<const uint16_t*>(f.x);
  for (int i = tid; i < rows * 4; i += NT) {
    const int h = i >> 2, t = i & 3;
    xs[i] = t < T ? Half<TA>::to_float(x[(size_t)t * H + hc0 + h]) : 0.f;
  }
  load_x_dec<TA>(f.x, T, H, res, tid, NT);
  cp_async_wait_all();
  __syncthreads();

  // partial logits: warp w < 8 is row group w (rows = w mod 8, ascending);
  // the accumulators are flushed at each split boundary
  {
    float acc[4][ME];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int m = 0; m < ME; ++m) acc[t][m] = 0.f;
    int cur = 0;
    auto flush = [&]() {
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int m = 0; m < ME; ++m) {
          const int e = lane + 32 * m;
          if (e < E) part[(((size_t)cur * 8 + warp) * 4 + t) * E + e] = acc[t][m];
          acc[t][m] = 0.f;
        }
      ++cur;
    };
    for (int p0 = 0; p0 < rows; p0 += P.pass_rows) {
      const int np = min(P.pass_rows, rows - p0);
      if (p0 > 0) {
        __syncthreads();  // the previous pass is consumed
        stage_rows(p0, np);
        cp_async_wait_all();
        __syncthreads();
      }
      // splits outermost: no division and no flush inside the row loop
      // (passes and splits start on multiples of 8 rows, so row j of the
      // pass belongs to row group j mod 8 = warp)
      if (warp < 8)
        for (int vr = p0 / rps; vr * rps < p0 + np; ++vr) {
          while (cur < vr) flush();
          const int j0 = max(p0, vr * rps) - p0, j1 = min(p0 + np, (vr + 1) * rps) - p0;
#pragma unroll 4
          for (int j = j0 + warp; j < j1; j += 8) {
            const int rel = p0 + j;
            float wv[ME];
#pragma unroll
            for (int m = 0; m < ME; ++m) {
              const int e = lane + 32 * m;
              wv[m] = (e < E) ? Half<TA>::to_float(wch[j * E + e]) : 0.f;
            }
            const float4 xv4 = reinterpret_cast<const float4*>(xs)[rel];
            const float xv[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
              for (int m = 0; m < ME; ++m) acc[t][m] = fmaf(xv[t], wv[m], acc[t][m]);
          }
        }
    }
    if (warp < 8)
      while (cur < VR) flush();
  }
  __syncthreads();
  for (int i = tid; i < VR * 4 * E; i += NT) {  // row groups summed in order
    const int vr = i / (4 * E), r = i - vr * 4 * E;
    const float* pp = part + (size_t)vr * 8 * 4 * E + r;
    float v = pp[0];
#pragma unroll
    for (int gi = 1; gi < 8; ++gi) v += pp[(size_t)gi * 4 * E];
    vpart[i] = v;
  }
  if (CL > 1) cluster_sync_all();
  else __syncthreads();
  if (warp < T) {
    float lg[ME];
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      if (e < E) {
        float pv[kMaxSplit];
#pragma unroll
        for (int r = 0; r < kMaxSplit; ++r) {
          const float* src = vpart + ((size_t)(r % VR) * 4 + warp) * E + e;
          pv[r] = CL > 1 ? ld_dsmem_f32(src, (uint32_t)(r / VR)) : *src;
        }
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxSplit; ++r) v += pv[r];
        lg[m] = v + (f.bias ? f.bias[e] : 0.f);
      } else {
        lg[m] = -INFINITY;
      }
    }
    int ids[kMaxTopk];
    float wts[kMaxTopk];
    softmax_topk<ME>(lg, E, k, f.gate_sigmoid != 0, lane, ids, wts);
    if (lane < k) {
      int bi = 0;
      float bp = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxTopk; ++q)
        if (q == lane) {
          bi = ids[q];
          bp = wts[q];
        }
      const int a = warp * k + lane;
      s_ids[a] = bi;
      s_wt[a] = bp;
      if (blockIdx.x == 0) {
        f.ws_ids[a] = bi;
        f.ws_w[a] = bp;
        if (f.user_ids) f.user_ids[a] = bi;
        if (f.user_w) f.user_w[a] = bp;
      }
    }
  }
  // No second cluster barrier: the split sums peers read sit in a region of
  // their own that nothing overwrites, and no CTA can exit before the grid
  // barrier, which every peer reaches only after its reads.
  __syncthreads();

  // grouping by expert (stable), one warp: A <= 32 assignments
  if (warp == 0) {
    for (int e = lane; e < E; e += 32) s_cnt[e] = 0;
    __syncwarp();
    int id = -1;
    if (lane < A) {
      id = s_ids[lane];
      if (id < 0 || id >= E) {
        set_status(status, QMOE_ST_INDEX);
        id = -1;
      }
    }
    const uint32_t mm = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(mm) - 1) s_cnt[id] = __popc(mm);
    __syncwarp();
    int c[8], fl[8], sc = 0, sf = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      c[j] = e < E ? s_cnt[e] : 0;
      fl[j] = c[j] > 0;
      sc += c[j];
      sf += fl[j];
    }
    int oc = sc, of = sf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y1 = __shfl_up_sync(0xffffffffu, oc, o), y2 = __shfl_up_sync(0xffffffffu, of, o);
      if (lane >= o) {
        oc += y1;
        of += y2;
      }
    }
    oc -= sc;
    of -= sf;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      if (e < E) {
        s_off[e] = oc;
        if (fl[j]) s_active[1 + of] = e;
      }
      oc += c[j];
      of += fl[j];
    }
    if (lane == 31) {
      s_off[E] = A;
      s_active[0] = of;
    }
    __syncwarp();
    if (id >= 0) s_perm[s_off[id] + __popc(mm & ((1u << lane) - 1u))] = lane;
    __syncwarp();
    if (blockIdx.x == 0) {  // the routing, also in the workspace
      for (int i = lane; i <= E; i += 32) f.ws_offsets[i] = s_off[i];
      for (int i = lane; i <= s_active[0]; i += 32) f.ws_active[i] = s_active[i];
      for (int i = lane; i < A; i += 32) f.ws_perm[i] = s_perm[i];
    }
  }
  __syncthreads();
  if (warp == kCW) {
    const int nsg = build_stages<kModeGateUp>(g, P.g, s_active, s_off, stg, blockIdx.x, gridDim.x, lane);
    const int nsd = build_stages<kModeDown>(d, P.d, s_active, s_off, std_, blockIdx.x, gridDim.x, lane);
    if (lane == 0) {
      s_misc[0] = nsg;
      s_misc[1] = nsd;
      s_misc[2] = 0;
    }
  }
  __syncthreads();
  const int nsg = s_misc[0], nsd = s_misc[1];
  const SlotLayout SLg = slot_layout(kModeGateUp, P.g.slot_rows, g.K, g.nb, HAS_ZP, g.src_row_floats, T);
  const SlotLayout SLd = slot_layout(kModeDown, P.d.slot_rows, d.K, d.nb, HAS_ZP, d.src_row_floats, T);

  if (warp == kCW) {
    // ============================================================ producer
    // Gate-up bytes first: they are on the critical path to the grid
    // barrier.  The down weights follow once the gate-up copies in flight
    // have landed (or, with more stages than slots, once the ring has
    // turned over), so that they do not share the CTA's HBM bandwidth with
    // the gate-up stream; they still land while the barrier is pending.
    const int n0g = min(NSg, nsg), n0d = min(NSd, nsd);
    issue_copies<kModeGateUp, HAS_ZP>(g, SLg, P.slot_g, stg, s_perm, ring_g, full_g, NSg, 0, n0g, true, true, lane);
    arrive_range(full_g, NSg, 0, n0g);
    bool ok = true;
    bool down_w = false;
    int ig = n0g;
    for (; ig < nsg; ++ig) {
      if (!(ok = mbar_wait(&empty_g[ig % NSg], ((ig / NSg) - 1) & 1, status))) break;
      if (!down_w) {
        issue_copies<kModeDown, HAS_ZP>(d, SLd, P.slot_d, std_, s_perm, ring_d, full_d, NSd, 0, n0d, true, false, lane);
        down_w = true;
      }
      issue_copies<kModeGateUp, HAS_ZP>(g, SLg, P.slot_g, stg, s_perm, ring_g, full_g, NSg, ig, ig + 1, true, true, lane);
      arrive_range(full_g, NSg, ig, ig + 1);
    }
    if (!down_w) {
      if (ok && nsg > 0) ok = mbar_wait(&full_g[(nsg - 1) % NSg], ((nsg - 1) / NSg) & 1, status);
      issue_copies<kModeDown, HAS_ZP>(d, SLd, P.slot_d, std_, s_perm, ring_d, full_d, NSd, 0, n0d, true, false, lane);
    }
    // down activations: only after the grid barrier (a consumer signals it)
    bool acts = ok && mbar_wait(gbar, 0, status);
    acts = acts && *reinterpret_cast<volatile int*>(s_misc + 2) == 0;
    if (acts) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      issue_copies<kModeDown, HAS_ZP>(d, SLd, P.slot_d, std_, s_perm, ring_d, full_d, NSd, 0, n0d, false, true, lane);
    }
    arrive_range(full_d, NSd, 0, n0d);  // always, so that the drain can see the weight copies land
    int id_ = n0d;
    if (acts)
      for (; id_ < nsd; ++id_) {
        if (!mbar_wait(&empty_d[id_ % NSd], ((id_ / NSd) - 1) & 1, status)) break;
        issue_copies<kModeDown, HAS_ZP>(d, SLd, P.slot_d, std_, s_perm, ring_d, full_d, NSd, id_, id_ + 1, true, true, lane);
        arrive_range(full_d, NSd, id_, id_ + 1);
      }
    // drain: no exit while bulk copies into this CTA's smem are in flight
    for (int s2 = max(0, ig - NSg); s2 < ig; ++s2)
      if (!mbar_wait(&full_g[s2 % NSg], (s2 / NSg) & 1, status)) break;
    for (int s2 = max(0, id_ - NSd); s2 < id_; ++s2)
      if (!mbar_wait(&full_d[s2 % NSd], (s2 / NSd) & 1, status)) break;
    return;
  }

  // ============================================================== consumers
  bool ok = consume_stages<kModeGateUp, TS, TA, HAS_ZP>(g, SLg, P.slot_g, stg, nsg, s_perm, res, nullptr, ring_g,
                                                        full_g, empty_g, NSg, warp, lane, status);
  // publish this CTA's SwiGLU outputs to every CTA's bulk copies
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
  if (tid == 0) {
    const bool gb = grid_barrier(g.ctl + kCtlGridCount, gridDim.x, status, kWaitLimitCycles);
    if (!gb || !ok) s_misc[2] = 1;
    mbar_arrive(gbar);
    pdl_trigger();
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
  if (*reinterpret_cast<volatile int*>(s_misc + 2) != 0) return;
  ok = consume_stages<kModeDown, TS, TA, HAS_ZP>(d, SLd, P.slot_d, std_, nsd, s_perm, res, res, ring_d, full_d,
                                                 empty_d, NSd, warp, lane, status);
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
  if (!ok) return;
  const int r0 = (int)(((long long)blockIdx.x * d.N) / gridDim.x);
  const int r1 = (int)(((long long)(blockIdx.x + 1) * d.N) / gridDim.x);
  down_combine<TA>(d, std_, nsd, s_perm, s_wt, res, r0, r1, tid, kCW * 32);
}

// ------------------------------------------------------------ fused host

// Shared-memory plan of the fused layer for `grid` CTAs in clusters of `cl`.
static bool plan_fused(int T, int H, int I, int E, int k, int bs, bool has_zp, int grid, int cl, FusedPlan* out) {
  if (T < 1 || T > kTokGroup || T * k > 32 || grid < 1 || cl < 1 || kMaxSplit % cl) return false;
  FusedPlan P = {};
  const int A = T * k, dmax = A < E ? A : E;
  const int VR = kMaxSplit / cl, rps = route_rows_per_split(H);
  // down: every CTA a fixed slice of output rows, all of it in the ring at once if it fits
  P.d.rows_cta = (H + grid - 1) / grid;
  P.d.slot_rows = P.d.rows_cta;
  P.d.max_stages = dmax + (A - dmax + kTokGroup - 1) / kTokGroup;
  const int nd_max = P.d.max_stages < 2 ? 2 : (P.d.max_stages > 4 ? 4 : P.d.max_stages);
  P.slot_d = slot_layout(kModeDown, P.d.slot_rows, I, I / bs, has_zp, dec_row_floats(I), T).bytes;
  // gate-up: the CTA's range of the flattened (expert, row) space
  const long long F = (long long)dmax * I;
  P.g.rows_cta = (int)((F + grid - 1) / grid);
  if (P.g.rows_cta < 1) P.g.rows_cta = 1;
  uint32_t res = (uint32_t)T * dec_row_floats(H) * 4;
  const uint32_t part_d = (uint32_t)P.d.max_stages * kTokGroup * P.d.rows_cta * 4;
  if (part_d > res) res = part_d;
  P.res_off = kFFixed;
  const uint32_t xs_b = (uint32_t)VR * rps * 16, part_b = (uint32_t)VR * 8 * 4 * E * 4,
                 vpart_b = (uint32_t)VR * 4 * E * 4;
  // Choose the ring shapes that keep the most gate-up rows in flight (the
  // stream that gates the grid barrier); among equals, fewer and larger
  // stages (two slots of half the CTA's rows streamed faster than four of
  // a quarter), then the deeper down ring.
  FusedPlan best = {};
  int best_rows = 0, best_ns = 0;
  for (int nd = nd_max; nd >= 2; --nd)
    for (int ns = 2; ns <= 4; ++ns) {
      P.d.nslots = nd;
      int sr = (P.g.rows_cta + ns - 1) / ns;
      if (sr > 64) sr = 64;
      for (; sr >= 1; sr = sr > 8 ? sr * 3 / 4 : sr - 1) {
        const int nst_min = (P.g.rows_cta + sr - 1) / sr;
        P.g.slot_rows = sr;
        P.g.max_stages = nst_min + (P.g.rows_cta + I - 1) / I + 1;
        P.g.nslots = ns < P.g.max_stages ? ns : P.g.max_stages;
        if (P.g.nslots < 2) P.g.nslots = 2;
        P.slot_g = slot_layout(kModeGateUp, sr, H, H / bs, has_zp, 0, T).bytes;
        P.stg_off = P.res_off + al16(res);
        P.std_off = P.stg_off + 48u * P.g.max_stages;
        // the split sums peers read: outside the rings, never overwritten
        P.vpart_off = al16(P.std_off + 48u * P.d.max_stages);
        P.ring_g = (P.vpart_off + vpart_b + 1023u) & ~1023u;
        P.ring_d = P.ring_g + P.g.nslots * P.slot_g;
        P.smem = P.ring_d + P.d.nslots * P.slot_d;
        if (P.smem > kSmemBudget) continue;
        // router scratch inside the rings; small rings (few rows per CTA)
        // are extended until it fits with at least 8 router rows per pass
        uint32_t room = P.smem - P.ring_g;
        P.xs_off = P.ring_g;
        P.part_off = P.xs_off + al16(xs_b);
        P.wch_off = P.part_off + al16(part_b);
        const uint32_t used = P.wch_off - P.ring_g;
        if (room < used + 16u * E) {
          room = (used + 16u * E + 127u) & ~127u;
          P.smem = P.ring_g + room;
          if (P.smem > kSmemBudget) continue;
        }
        int pr = (int)(((room - used) / (2u * E)) & ~7u);
        if (pr > VR * rps) pr = VR * rps;
        if (pr < 8) continue;
        P.pass_rows = pr;
        const int rows = min(P.g.nslots * sr, P.g.rows_cta);
        if (rows > best_rows || (rows == best_rows && ns < best_ns)) {
          best = P;
          best_rows = rows;
          best_ns = ns;
        }
        break;  // the largest slot that fits for this (nd, ns)
      }
    }
  if (best_rows == 0) return false;
  *out = best;
  return true;
}

// CTAs of a cooperative launch in clusters of kFusedCluster at one CTA per
// SM (cached per device and kernel)
template <typename F>
static int fused_grid(F* fn) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    if (ensure_smem(fn, kSmemBudget) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kFusedCluster * 64);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = kSmemBudget;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kFusedCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = n * kFusedCluster;
  }
  return cached[dev];
}

template <typename TS, typename TA, bool Z, int ME>
static cudaError_t launch_fused_t(const FusedParams& f, cudaStream_t st, bool pdl, bool check_only) {
  auto fn = fused_decode_kernel<TS, TA, Z, ME, kFusedCluster>;
  const int grid = fused_grid(fn);
  FusedPlan P;
  if (grid < kFusedCluster ||
      !plan_fused(f.g.T, f.g.K, f.g.N, f.g.E, f.g.k, f.g.bs, Z, grid, kFusedCluster, &P))
    return cudaErrorInvalidValue;
  if (check_only) return cudaSuccess;
  cudaError_t err = ensure_smem(fn, P.smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFusedCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
  attr[1].val.cooperative = 1;
  attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[2].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 3 : 2;
  return cudaLaunchKernelEx(&cfg, fn, f, P);
}

template <typename TS, typename TA, bool Z>
static cudaError_t launch_fused_me(const FusedParams& f, cudaStream_t st, bool pdl, bool check_only) {
  if (f.g.E <= 64) return launch_fused_t<TS, TA, Z, 2>(f, st, pdl, check_only);
  return launch_fused_t<TS, TA, Z, 8>(f, st, pdl, check_only);
}

}  // namespace qmoe
