// decode_fused.cuh -- the whole decode layer (router, gate-up with SwiGLU,
// down with the routing-weighted sum) in one launch, on the building blocks
// of decode_core.cuh.  The kernel and its host plan are templates here;
// decode_fused_f16.cu and decode_fused_bf16.cu instantiate them for each
// activation dtype (two translation units built in parallel).
//
// Sources: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), IR guide
// section 3 (MoE block: router TopK, Expert Computation steps 4-7) and the
// "Fused MoE Extern Kernels" update (kernel 1: gate + up with SwiGLU and
// the INT4 dequantisation inside the dot product; kernel 2: down with the
// routing-weighted reduce).
//
// GB300 design.  The distinct selected experts' intermediate rows, flattened
// expert-major into D*I rows, are cut into equal windows of whole 32-row
// units, one window per cluster of 4 CTAs.  The down projection is split
// along its reduction (I) at these windows, so no cluster waits for another
// cluster's SwiGLU output.  A CTA
//   1. computes the routing with the other CTAs of its cluster (each CTA
//      reduces a quarter of H for all experts, in the router kernel's fp32
//      order; the splits are summed in rank order through distributed shared
//      memory, so every cluster has the same bit-identical top-k);
//   2. issues, at once, bulk copies of all of its quarter of the window's
//      gate and up rows (codes, block scales, zero points) stage by stage,
//      and TMA tensor copies of the down codes it needs: its quarter of the
//      H output rows, over the whole window (16 bytes = one 32-code unit per
//      row per box), plus an L2 prefetch of their block scales/zero points;
//   3. computes gate and up for its rows as the stages land, then SwiGLU;
//   4. exchanges SwiGLU outputs with its cluster through distributed shared
//      memory, so every CTA holds the window's SwiGLU slice;
//   5. multiplies that slice into its down codes (one 32-code unit of one
//      output row per work item), sums each row over the units in order
//      times the routing weights, and adds it to an output accumulator in
//      the workspace control block as a 2^-32 fixed-point integer; the last
//      cluster to finish a quarter of H (a counter in the control block)
//      converts that quarter to the output and clears the accumulator.
// Every floating-point sum is in a fixed order and the cross-cluster sum is
// an integer one: results are bit-reproducible.  There is no
// grid-wide wait, so the launch needs no co-residency guarantee, and it
// triggers its dependents at entry so the next launch's CTAs start on the
// SMs this one leaves.
#pragma once

#include <cuda.h>

#include "decode_core.cuh"
#include "tmap.h"

namespace qmoe {

// One segment of a cluster window: rows [i0, i1) of expert e's intermediate
// dimension (multiples of 32), serving assignments perm[pbase .. pbase +
// ntok) (token tok[n], routing weight w[n]); window units [u0, u0 + (i1 -
// i0) / 32).
struct SegEnt {
  int e, pbase, ntok, i0, i1, u0, tok[4];
  float w[4];
  int pad[2];
};
static_assert(sizeof(SegEnt) == 64, "segment entry is 64 bytes");
// One 32-row unit of a cluster window: expert, first row, segment, and
// the expert's index among the distinct selected experts.
struct UnitEnt {
  int e, i, seg, pad;
};

constexpr int kFStageRows = 8;   // intermediate rows per gate-up stage
constexpr int kFMaxStages = 16;
constexpr int kFMaxSegs = 4;
constexpr int kFMaxUnits = 8;    // 32-row units per cluster window
constexpr int kFMaxItems = 12;   // down items (unit, row) per thread
constexpr int kFusedCluster = 4;
constexpr int kFusedThreads = kDecodeThreads;

// fixed shared-memory carve (bytes)
constexpr uint32_t kFOffBars = 0;                                   // kFMaxStages + 2 mbarriers
constexpr uint32_t kFOffMisc = 192;                                 // 16 ints
constexpr uint32_t kFOffActive = 256;
constexpr uint32_t kFOffOff = kFOffActive + 4 * (kMaxExperts + 2);
constexpr uint32_t kFOffIds = kFOffOff + 4 * (kMaxExperts + 2);
constexpr uint32_t kFOffPerm = kFOffIds + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffWt = kFOffPerm + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffCnt = kFOffWt + 4 * kTokGroup * kMaxTopk;
constexpr uint32_t kFOffStg = (kFOffCnt + 4 * kMaxExperts + 127) & ~127u;
constexpr uint32_t kFOffSeg = kFOffStg + 48 * kFMaxStages;
constexpr uint32_t kFOffUnit = kFOffSeg + 64 * kFMaxSegs;
constexpr uint32_t kFFixed = (kFOffUnit + 16 * kFMaxUnits + 127) & ~127u;
// misc slots
constexpr int kMiscNst = 0, kMiscNseg = 1, kMiscAbort = 2, kMiscLast = 3, kMiscNunit = 4, kMiscC0 = 5,
              kMiscC1 = 6, kMiscRng = 7;  // kMiscRng..+CL: the cluster CTAs' first window rows

// Shared-memory plan of the fused layer (host and device agree on it).
struct FusedPlan {
  int crows_max;    // rows per cluster window (multiple of 32, <= 32 * kFMaxUnits)
  int rows_max;     // gate-up rows per CTA (multiple of 8)
  int max_stages, max_segs;
  int slice, box_r, nboxes;  // down rows per CTA, TMA box rows, boxes per column group
  int box_w;        // TMA box width in bytes: 16 (a box per unit) or 16 * units (a box per segment)
  int pass_rows;    // router rows staged per pass
  uint32_t vpart_off, gu_off, acto_off, acta_off, xdec_off, dsc_off, dzp_off, dn_off, ring_off, smem;
  uint32_t xs_off, part_off, wch_off;  // router scratch, inside the ring (as are the
                                       // down phase's per-unit dot products later)
};

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// L2 prefetch of [p, p + bytes), shrunk inward to 16-byte boundaries
__device__ __forceinline__ void prefetch_range(const void* p, size_t bytes) {
  const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 15) & ~(uintptr_t)15;
  const uintptr_t b = (reinterpret_cast<uintptr_t>(p) + bytes) & ~(uintptr_t)15;
  for (uintptr_t c = a; c < b; c += (1u << 20)) {
    const uintptr_t n = (b - c) < (1u << 20) ? (b - c) : (1u << 20);
    prefetch_l2_bulk(reinterpret_cast<const void*>(c), (uint32_t)n);
  }
}

// 8 codes of one 32-bit word as (q - zp) * 16^j pairs (j = nibble position
// in its half-word), the 8-code form of dequant_chunk.
__device__ __forceinline__ void dequant_word(uint32_t q, const ZConst zc, uint32_t magic, f2 (&wv)[4]) {
  const uint32_t hi = q >> 16;
  wv[0] = fadd2(make_float2(or_masked<0xFu>(q, magic), or_masked<0xF0u>(q, magic)), zc.c01);
  wv[1] = fadd2(make_float2(or_masked<0xF00u>(q, magic), or_masked<0xF000u>(q, magic)), zc.c23);
  wv[2] = fadd2(make_float2(or_masked<0xFu>(hi, magic), or_masked<0xF0u>(hi, magic)), zc.c01);
  wv[3] = fadd2(make_float2(or_masked<0xF00u>(hi, magic), or_masked<0xF000u>(hi, magic)), zc.c23);
}

// Gate-up stage layout: one stage's rows of gate then up, as a decode slot.
__host__ __device__ inline SlotLayout fused_stage_layout(int nrows, int H, int nb, bool has_zp) {
  return slot_layout(kModeGateUp, nrows, H, nb, has_zp, 0, 1);
}

// The cluster window, its segments and units, and this CTA's gate-up stages
// (one warp).  Window of cluster q: 32-row units [q*U/NC, (q+1)*U/NC) of
// the flattened space; CTA r of the cluster: 8-row units [r*n8/CL,
// (r+1)*n8/CL) of the window.  Segment (expert) boundaries fall on 32-row
// units, so every stage is exactly 8 rows.  Returns false (all lanes) if a
// table would overflow.
template <bool HAS_ZP, bool T1>
__device__ bool build_fused_tables(const FusedPlan& P, int I, int H, int nbH, int k, int CL, int rank,
                                   const int* s_active, const int* s_off, const int* s_perm, const float* s_wt,
                                   SegEnt* seg, UnitEnt* unit, StageEnt* stg, int* misc, int cid, int ncl, int lane) {
  const int D = s_active[0];
  const int U = D * (I / 32);
  const int uc0 = (cid * U) / ncl, uc1 = ((cid + 1) * U) / ncl;  // U * ncl < 2^31 (host check)
  const int nwu = uc1 - uc0;
  if (nwu > kFMaxUnits) return false;
  // units (lane u) and segment starts (a unit at window start or at row 0 of its expert)
  int e = 0, i = 0, dd = 0;
  bool start = false;
  if (lane < nwu) {
    const int f = 32 * (uc0 + lane);
    dd = f / I;
    i = f - dd * I;
    e = s_active[1 + dd];
    start = lane == 0 || i == 0;
  }
  const uint32_t starts = __ballot_sync(0xffffffffu, start);
  const int nseg = __popc(starts);
  if (nseg > P.max_segs) return false;
  if (lane < nwu) {
    const int sidx = __popc(starts & ((2u << lane) - 1u)) - 1;
    unit[lane].e = e;
    unit[lane].i = i;
    unit[lane].seg = sidx;
    unit[lane].pad = dd;
    if (start) {
      SegEnt& sg = seg[sidx];
      sg.e = e;
      sg.pbase = T1 ? dd : s_off[e];
      sg.ntok = T1 ? 1 : s_off[e + 1] - s_off[e];
      sg.i0 = i;
      sg.u0 = lane;
      for (int n = 0; n < 4; ++n) {
        const int a = n < sg.ntok ? s_perm[sg.pbase + n] : 0;
        sg.tok[n] = n < sg.ntok ? a / k : -1;
        sg.w[n] = n < sg.ntok ? s_wt[a] : 0.f;
      }
    }
  }
  __syncwarp();
  if (lane < nwu && (lane + 1 == nwu || ((starts >> (lane + 1)) & 1u))) seg[unit[lane].seg].i1 = i + 32;
  // this CTA's gate-up rows [c0, c1) of the window, stage s = rows [c0 + 8s, c0 + 8s + 8)
  const int n8 = 4 * nwu;
  if (lane < CL) misc[kMiscRng + lane] = 8 * ((lane * n8) / CL);
  const int c0 = 8 * ((rank * n8) / CL), c1 = 8 * (((rank + 1) * n8) / CL);
  const int nst = (c1 - c0) / kFStageRows;
  if (nst > P.max_stages) return false;
  const uint32_t sb = fused_stage_layout(kFStageRows, H, nbH, HAS_ZP).bytes;
  __syncwarp();
  if (lane < nst) {
    const int c = c0 + kFStageRows * lane;
    const UnitEnt& un = unit[c >> 5];
    StageEnt& st = stg[lane];
    st.e = un.e;
    st.pbase = T1 ? un.pad : s_off[un.e];
    st.ntok = T1 ? 1 : s_off[un.e + 1] - s_off[un.e];
    st.row0 = un.i + (c & 31);
    st.nrows = kFStageRows;
    st.pad[0] = un.seg;
    st.pad[1] = (int)(lane * sb);
    st.pad[2] = c;  // window row of the stage's first row
  }
  if (lane == 0) {
    misc[kMiscNst] = nst;
    misc[kMiscNseg] = nseg;
    misc[kMiscNunit] = nwu;
    misc[kMiscC0] = c0;
    misc[kMiscC1] = c1;
  }
  return true;
}

// Bulk copies of gate-up stages [0, nst) (producer warp, jobs spread over the
// lanes), each stage at its own offset of the ring; then every lane arrives
// on every stage's barrier (count 32).
template <bool HAS_ZP>
__device__ void issue_fused_stages(const DecodeParams& g, StageEnt* stg, int nst, uint8_t* ring, uint64_t* full,
                                   int lane) {
  const int H = g.K, nb = g.nb;
  for (int jid = lane; jid < nst * 6; jid += 32) {
    const int s = jid / 6, job = jid % 6, m = job / 3, kind = job % 3;
    if (kind == 2 && !HAS_ZP) continue;
    StageEnt& st = stg[s];
    const SlotLayout SL = fused_stage_layout(st.nrows, H, nb, HAS_ZP);
    uint8_t* sb = ring + st.pad[1];
    const size_t row0 = (size_t)st.e * g.N + st.row0;
    if (kind == 0) {
      copy_bulk(sb + (m ? SL.w[1] : SL.w[0]), (m ? g.w[1] : g.w[0]) + row0 * (H / 2), (uint32_t)st.nrows * (H / 2),
                &full[s]);
    } else if (kind == 1) {
      const int ph = copy_ragged(sb + (m ? SL.s[1] : SL.s[0]),
                                 static_cast<const uint8_t*>(m ? g.s[1] : g.s[0]) + row0 * nb * 2,
                                 (uint32_t)st.nrows * nb * 2, &full[s]);
      if (m) st.ph[1] = ph; else st.ph[0] = ph;
    } else {
      const int ph = copy_ragged(sb + (m ? SL.z[1] : SL.z[0]), (m ? g.z[1] : g.z[0]) + row0 * nb,
                                 (uint32_t)st.nrows * nb, &full[s]);
      if (m) st.ph[3] = ph; else st.ph[2] = ph;
    }
  }
  __syncwarp();
  for (int s = 0; s < nst; ++s) mbar_arrive(&full[s]);
}

template <typename TS, typename TA, bool HAS_ZP, int ME, int CL, int CPL>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_decode_kernel(const __grid_constant__ CUtensorMap tm_d, FusedParams f, FusedPlan P) {
  constexpr int VR = kMaxSplit / CL;  // router splits per CTA
  constexpr int NTH = kFusedThreads;
  constexpr int NWP = NTH / 32;
  constexpr int NTR = CPL > 0 ? 1 : kTokGroup;  // tokens the router computes
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFOffBars);
  uint64_t* rbar = full + kFMaxStages;
  uint64_t* dbar = rbar + 1;
  int* s_misc = reinterpret_cast<int*>(smem + kFOffMisc);
  int* s_active = reinterpret_cast<int*>(smem + kFOffActive);
  int* s_off = reinterpret_cast<int*>(smem + kFOffOff);
  int* s_ids = reinterpret_cast<int*>(smem + kFOffIds);
  int* s_perm = reinterpret_cast<int*>(smem + kFOffPerm);
  float* s_wt = reinterpret_cast<float*>(smem + kFOffWt);
  int* s_cnt = reinterpret_cast<int*>(smem + kFOffCnt);
  StageEnt* stg = reinterpret_cast<StageEnt*>(smem + kFOffStg);
  SegEnt* seg = reinterpret_cast<SegEnt*>(smem + kFOffSeg);
  UnitEnt* unit = reinterpret_cast<UnitEnt*>(smem + kFOffUnit);
  float* vpart = reinterpret_cast<float*>(smem + P.vpart_off);   // [VR][4][E], read by the cluster (own region)
  float* gu = reinterpret_cast<float*>(smem + P.gu_off);         // [window row][2] gate, up (T = 1 path)
  float* act_own = reinterpret_cast<float*>(smem + P.acto_off);  // [4][crows_max] this CTA's rows, pre-scaled
  float* act_all = reinterpret_cast<float*>(smem + P.acta_off);  // [4][crows_max] the whole window's
  float* xdec = reinterpret_cast<float*>(smem + P.xdec_off);     // [T][dec_row_floats(H)] (general path)
  uint8_t* dn = smem + P.dn_off;  // down codes [column group][slice row][box_w bytes]; a column
                                  // group is a unit (box_w 16) or a segment of units
  uint16_t* dsc = reinterpret_cast<uint16_t*>(smem + P.dsc_off);  // [unit][slice row] down block scales
  uint8_t* dzp = smem + P.dzp_off;                                 // [unit][slice row] down zero points
  uint8_t* ring = smem + P.ring_off;
  // router scratch and, at the end, the final sum's partial sums: inside
  // the ring, used only while no gate-up copy can land there
  float* xs = reinterpret_cast<float*>(smem + P.xs_off);          // [VR*rps][4]
  float* part = reinterpret_cast<float*>(smem + P.part_off);      // [VR][8][4][E]
  uint16_t* wch = reinterpret_cast<uint16_t*>(smem + P.wch_off);  // [pass_rows][E]

  const DecodeParams& g = f.g;
  const DecodeParams& d = f.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = g.ctl + kCtlStatus;
  const int T = g.T, H = g.K, I = g.N, E = g.E, k = g.k, A = T * k;
  const int nbH = g.nb, nbI = d.nb;
  const int cmax = P.crows_max;
  // launched in clusters of CL covering the grid, or not at all: every CTA
  // sees the same values, so all return together before any cluster access
  if (CL > 1 && (cluster_nctarank() != (uint32_t)CL || cluster_count_x() * CL != gridDim.x)) {
    if (tid == 0) set_status(status, QMOE_ST_INDEX);
    return;
  }
  // the next launch may start its CTAs as soon as SMs free up; its own
  // griddepcontrol.wait still waits for this whole grid to complete
  pdl_trigger();
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
  const int rps = f.rps;
  const int hc0 = (int)rank * VR * rps;
  const int rows = max(0, min(H, hc0 + VR * rps) - hc0);
  const int hs0 = (int)rank * P.slice;  // this CTA's down output rows [hs0, hs0 + slice)

  if (tid == 0) {
    for (int i = 0; i < kFMaxStages + 2; ++i) mbar_init(&full[i], i < kFMaxStages ? 32 : 1);
    fence_barrier_init();
    s_misc[kMiscAbort] = 0;
  }
  __syncthreads();

  // ---- 1. router.  The weight rows do not depend on the previous grid:
  //         the first pass is in flight before waiting for it.
  const uint16_t* rw = static_cast<const uint16_t*>(f.router_w);
  const bool bulkw = (reinterpret_cast<uintptr_t>(rw) & 15) == 0;  // pass starts are 8-row multiples
  auto stage_rows = [&](int p0, int np) {
    const uint16_t* src = rw + (size_t)(hc0 + p0) * E;
    if (bulkw) {
      // four copies in flight (each a multiple of 8 rows = 16 * E bytes)
      if (tid < 32) {
        const int c8 = np >> 3, per = (c8 + 3) >> 2;
        if (tid == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier passes: generic proxy
          mbar_arrive_expect_tx(rbar, (uint32_t)np * E * 2);
        }
        __syncwarp();
        if (tid < 4) {
          const int a = min(c8, tid * per), b = min(c8, (tid + 1) * per);
          if (b > a) bulk_g2s(wch + (size_t)a * 8 * E, src + (size_t)a * 8 * E, (uint32_t)(b - a) * 16 * E, rbar);
        }
      }
    } else {
      for (int i = tid; i < np * E; i += NTH) wch[i] = __ldg(src + i);
    }
  };
  int npass = 0;
  bool ok = true;
  auto wait_rows = [&]() {
    if (bulkw) ok = mbar_wait(rbar, (uint32_t)(npass & 1), status) && ok;
    ++npass;
  };
  if (rows > 0) stage_rows(0, min(P.pass_rows, rows));
  pdl_wait();  // x may be the previous kernel's output
  const uint16_t* x = static_cast<const uint16_t*>(f.x);
  // router slice of x: xs[h][t] fp32, 8 rows per thread from one 16-byte load
  for (int i = tid; i < (rows >> 3) * kTokGroup; i += NTH) {
    const int t = i % kTokGroup, h8 = (i / kTokGroup) * 8;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (t < T) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + hc0 + h8));
      const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = Half<TA>::to_float((uint16_t)(qq[j >> 1] >> ((j & 1) * 16)));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) xs[(h8 + j) * 4 + t] = v[j];
  }
  if (CPL == 0) load_x_dec<TA>(f.x, T, H, xdec, tid, NTH);
  if (rows > 0) wait_rows();
  __syncthreads();

  // partial logits: warp w < 8 is row group w (rows = w mod 8, ascending);
  // the accumulators are flushed at each split boundary.  One token with an
  // even E <= 64: a lane owns experts (2 lane, 2 lane + 1), one 32-bit word
  // of a staged row, with a paired fma (each half the same fmaf as the
  // general form below).
  if (NTR == 1 && ME == 2 && (E & 1) == 0) {
    f2 acc2 = make_float2(0.f, 0.f);
    int cur = 0;
    const int e0 = 2 * lane;
    auto flush2 = [&]() {
      if (e0 < E) {
        part[((size_t)cur * 8 + warp) * 4 * E + e0] = acc2.x;
        part[((size_t)cur * 8 + warp) * 4 * E + e0 + 1] = acc2.y;
      }
      acc2 = make_float2(0.f, 0.f);
      ++cur;
    };
    for (int p0 = 0; p0 < rows; p0 += P.pass_rows) {
      const int np = min(P.pass_rows, rows - p0);
      if (p0 > 0) {
        __syncthreads();  // the previous pass is consumed
        stage_rows(p0, np);
        wait_rows();
        __syncthreads();
      }
      if (warp < 8)
        for (int vr = p0 / rps; vr * rps < p0 + np; ++vr) {
          while (cur < vr) flush2();
          const int j0 = max(p0, vr * rps) - p0, j1 = min(p0 + np, (vr + 1) * rps) - p0;
#pragma unroll 8
          for (int j = j0 + warp; j < j1; j += 8) {
            const uint32_t wbits = e0 < E ? *reinterpret_cast<const uint32_t*>(wch + (size_t)j * E + e0) : 0u;
            const float xv = xs[(p0 + j) * 4];
            acc2 = ffma2(make_float2(xv, xv),
                         make_float2(Half<TA>::to_float((uint16_t)(wbits & 0xFFFFu)),
                                     Half<TA>::to_float((uint16_t)(wbits >> 16))),
                         acc2);
          }
        }
    }
    if (warp < 8)
      while (cur < VR) flush2();
  } else {
    float acc[NTR][ME];
#pragma unroll
    for (int t = 0; t < NTR; ++t)
#pragma unroll
      for (int m = 0; m < ME; ++m) acc[t][m] = 0.f;
    int cur = 0;
    auto flush = [&]() {
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int m = 0; m < ME; ++m) {
          const int e = lane + 32 * m;
          if (e < E) part[(((size_t)cur * 8 + warp) * 4 + t) * E + e] = t < NTR ? acc[t < NTR ? t : 0][m] : 0.f;
        }
#pragma unroll
      for (int t = 0; t < NTR; ++t)
#pragma unroll
        for (int m = 0; m < ME; ++m) acc[t][m] = 0.f;
      ++cur;
    };
    for (int p0 = 0; p0 < rows; p0 += P.pass_rows) {
      const int np = min(P.pass_rows, rows - p0);
      if (p0 > 0) {
        __syncthreads();  // the previous pass is consumed
        stage_rows(p0, np);
        wait_rows();
        __syncthreads();
      }
      // splits outermost (passes and splits start on multiples of 8 rows,
      // so row j of the pass belongs to row group j mod 8 = warp)
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
            for (int t = 0; t < NTR; ++t)
#pragma unroll
              for (int m = 0; m < ME; ++m) acc[t][m] = fmaf(xv[t], wv[m], acc[t][m]);
          }
        }
    }
    if (warp < 8)
      while (cur < VR) flush();
  }
  __syncthreads();
  for (int i = tid; i < VR * NTR * E; i += NTH) {  // row groups summed in order
    const int vr = i / (NTR * E), r = i - vr * NTR * E;
    const float* pp = part + (size_t)vr * 8 * 4 * E + r;
    float v = pp[0];
#pragma unroll
    for (int gi = 1; gi < 8; ++gi) v += pp[(size_t)gi * 4 * E];
    vpart[(size_t)vr * 4 * E + r] = v;
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
  // Peers read vpart (a region nothing overwrites) before the window
  // exchange's cluster barriers, which this CTA also reaches.
  __syncthreads();

  // grouping by expert (stable), one warp: A <= 32 assignments; then the
  // window and stage tables
  if (warp == 0) {
    if (NTR == 1) {
      // one token: the stable grouping of its k distinct experts is their
      // ascending order; rank each by the others' ids
      int id = lane < k ? s_ids[lane] : 0x7fffffff;
      if (lane < k && (id < 0 || id >= E)) {
        set_status(status, QMOE_ST_INDEX);
        id = 0;
      }
      int rnk = 0;
      for (int q = 0; q < k; ++q) rnk += __shfl_sync(0xffffffffu, id, q) < id;
      if (lane < k) {
        s_active[1 + rnk] = id;
        s_perm[rnk] = lane;
      }
      if (lane == 0) s_active[0] = k;
      __syncwarp();
      if (blockIdx.x == 0) {  // the routing, also in the workspace
        for (int e = lane; e <= E; e += 32) {
          int c = 0;
          for (int q = 0; q < k; ++q) c += s_active[1 + q] < e;
          f.ws_offsets[e] = c;
        }
        if (lane <= k) f.ws_active[lane] = s_active[lane];
        if (lane < k) f.ws_perm[lane] = s_perm[lane];
      }
    } else {
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
    __syncwarp();
    if (!build_fused_tables<HAS_ZP, NTR == 1>(P, I, H, nbH, k, CL, (int)rank, s_active, s_off, s_perm, s_wt, seg,
                                               unit, stg, s_misc, cid, ncl, lane) &&
        lane == 0) {
      set_status(status, QMOE_ST_INDEX);  // no work for this CTA
      s_misc[kMiscNst] = s_misc[kMiscNseg] = s_misc[kMiscNunit] = s_misc[kMiscC0] = s_misc[kMiscC1] = 0;
      for (int r = 0; r < CL; ++r) s_misc[kMiscRng + r] = 0;
    }
  }
  __syncthreads();
  const int nst = s_misc[kMiscNst], nwu = s_misc[kMiscNunit];
  const int c0 = s_misc[kMiscC0], c1 = s_misc[kMiscC1];

  // ---- 2. every copy of the CTA's share, in flight at once.  First the
  //         block scale and zero point of every down item (unit u, output
  //         row hs0 + r), loaded with lanes running over the units of a row
  //         (a row's units share a sector), so that these small loads go out
  //         ahead of the bulk traffic; stored to shared memory as item
  //         u * slice + r once they return.
  const int ns_d = P.slice, nit_d = nwu * ns_d;
  uint16_t sv[kFMaxItems];
  uint8_t zv[kFMaxItems];
  {
    const uint16_t* s16 = static_cast<const uint16_t*>(d.s[0]);
    const int lbs_d = g.bs == 32 ? 5 : (g.bs == 64 ? 6 : 7);
#pragma unroll
    for (int j = 0; j < kFMaxItems; ++j) {
      const int idx = tid + j * NTH;  // row-major: idx = r * nwu + u
      if (idx < nit_d) {
        const int r = idx / nwu, u = idx - r * nwu;
        const size_t o = ((size_t)unit[u].e * H + hs0 + r) * nbI + (unit[u].i >> lbs_d);
        sv[j] = __ldg(s16 + o);
        zv[j] = HAS_ZP ? __ldg(d.z[0] + o) : (uint8_t)8;
      }
    }
  }
  // Then one warp issues the gate-up stages (the TMA unit serves them in
  // order), the down codes (rows [hs0, hs0 + slice) of each column group's
  // expert, box_w bytes from the group's first unit, box_r rows per box) and
  // an L2 prefetch of the whole rows of block scales / zero points around
  // this CTA's (the clusters on the neighbouring windows read the rest).
  if (warp == NWP - 1) {
    // the ring held the router scratch, written and read through the generic proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    issue_fused_stages<HAS_ZP>(g, stg, nst, ring, full, lane);
    const bool wide = P.box_w > 16;
    const int ncg = wide ? s_misc[kMiscNseg] : nwu;
    if (lane == 0) mbar_arrive_expect_tx(dbar, (uint32_t)ncg * P.nboxes * P.box_r * P.box_w);
    __syncwarp();
    for (int j = lane; j < ncg * P.nboxes; j += 32) {
      const int cg = j / P.nboxes, b = j - cg * P.nboxes;
      const int e = wide ? seg[cg].e : unit[cg].e, i0 = wide ? seg[cg].i0 : unit[cg].i;
      tma_load_2d(dn + ((size_t)cg * P.slice + (size_t)b * P.box_r) * P.box_w, &tm_d, i0 / 2,
                  e * H + hs0 + b * P.box_r, dbar);
    }
    const int nseg = s_misc[kMiscNseg];
    for (int s = lane; s < nseg; s += 32) {
      const size_t row0 = (size_t)seg[s].e * H + hs0;
      prefetch_range(static_cast<const uint16_t*>(d.s[0]) + row0 * nbI, (size_t)P.slice * nbI * 2);
      if (HAS_ZP) prefetch_range(d.z[0] + row0 * nbI, (size_t)P.slice * nbI);
    }
    // this CTA's 1/G share of the selected experts' down codes into L2 as one
    // sequential range: the strips the TMA boxes take are scattered 80-byte
    // pieces of whole expert matrices that the clusters read between them
    if (lane < 2) {
      const size_t per = (size_t)H * (I / 2), tot = (size_t)s_active[0] * per;
      const size_t a = (tot * blockIdx.x) / gridDim.x, b = (tot * (blockIdx.x + 1)) / gridDim.x;
      const size_t d0 = a / per, d1 = (b - 1) / per;
      const size_t dd = d0 + lane;
      if (b > a && dd <= d1) {
        const size_t lo = dd == d0 ? a - d0 * per : 0, hi = dd == d1 ? b - d1 * per : per;
        prefetch_range(d.w[0] + (size_t)s_active[1 + dd] * per + lo, hi - lo);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kFMaxItems; ++j) {
    const int idx = tid + j * NTH;
    if (idx < nit_d) {
      const int r = idx / nwu, u = idx - r * nwu;
      dsc[u * ns_d + r] = sv[j];
      if (HAS_ZP) dzp[u * ns_d + r] = zv[j];
    }
  }

  // ---- 3. gate-up + SwiGLU as the stages land
  const uint32_t magic = opaque(0x4B000000u);      // 2^23
  const uint32_t neg_magic = opaque(0xCB000000u);  // -2^23
  const ZConst zfixed = zconst(8u, neg_magic);     // no zero-point tensor: zp = 8
  const int lbs = g.bs == 32 ? 5 : (g.bs == 64 ? 6 : 7);
  bool wok = true;
  if (CPL > 0) {
    // T = 1, H = 1024 * CPL: lane owns chunks c = 32 u + lane of every row and
    // keeps their 32 activations in registers; a work item is one row of one
    // matrix (gate or up), dealt round-robin over all warps in stage order
    XChunk xr[CPL > 0 ? CPL : 1];
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(32 * u + lane) * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 q = __ldg(src + v);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float a0 = Half<TA>::to_float((uint16_t)(qq[2 * p] & 0xFFFFu));
          const float a1 = Half<TA>::to_float((uint16_t)(qq[2 * p] >> 16)) * 0.0625f;
          const float a2 = Half<TA>::to_float((uint16_t)(qq[2 * p + 1] & 0xFFFFu)) * 0.00390625f;
          const float a3 = Half<TA>::to_float((uint16_t)(qq[2 * p + 1] >> 16)) * 0.000244140625f;
          xr[u].v[2 * v + p] = make_float4(a0, a1, a2, a3);
        }
      }
    }
    // items: (stage s, row r) = rows of gate and up; stage s holds items
    // [8 s, 8 s + 8) (every stage is 8 rows)
    int waited = -1;
    for (int it = warp; it < kFStageRows * nst; it += NWP) {
      const int s = it / kFStageRows, r = it - s * kFStageRows;
      if (waited != s) {
        if (!mbar_wait(&full[s], 0u, status)) {
          wok = false;
          break;
        }
        waited = s;
      }
      const StageEnt& st = stg[s];
      const SlotLayout SL = fused_stage_layout(kFStageRows, H, nbH, HAS_ZP);
      const uint8_t* sb = ring + st.pad[1];
      uint4 q[2][CPL > 0 ? CPL : 1];
      float sc[2][CPL > 0 ? CPL : 1];
      uint32_t zz[2][CPL > 0 ? CPL : 1];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint8_t* wrow = sb + SL.w[m] + (size_t)r * (H / 2);
        const uint16_t* srow = reinterpret_cast<const uint16_t*>(sb + SL.s[m] + st.ph[m]) + (size_t)r * nbH;
        const uint8_t* zrow = sb + SL.z[m] + st.ph[2 + m] + (size_t)r * nbH;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          const int c = 32 * u + lane;
          q[m][u] = *reinterpret_cast<const uint4*>(wrow + c * 16);
          const int blk = (c * 32) >> lbs;
          sc[m][u] = Half<TS>::to_float(srow[blk]);
          zz[m][u] = HAS_ZP ? (uint32_t)zrow[blk] : 8u;
        }
      }
      float acc[2] = {0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          f2 wv[16];
          dequant_chunk(q[m][u], HAS_ZP ? zconst(zz[m][u], neg_magic) : zfixed, magic, wv);
          acc[m] = fmaf(sc[m][u], chunk_dot(wv, xr[u]), acc[m]);
        }
      // lanes < 16 keep gate and receive the other half's gate; lanes >= 16 up
      const bool lo = lane < 16;
      float v = (lo ? acc[0] : acc[1]) + __shfl_xor_sync(0xffffffffu, lo ? acc[1] : acc[0], 16);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if ((lane & 15) == 0) gu[(st.pad[2] + r) * 2 + (lane >> 4)] = v;
    }
    if (!wok) s_misc[kMiscAbort] = 1;
    __syncthreads();
    for (int c = c0 + tid; c < c1; c += NTH) {
      const int i = unit[c >> 5].i + (c & 31);
      const float gv = gu[2 * c], uv = gu[2 * c + 1];
      act_own[c] = gv / (1.f + expf(-gv)) * uv * dec_prescale(i);
    }
  } else {
    // general T <= 4: activations in shared memory (decode layout); a work
    // item is a group of rows of gate and up for every token of the stage
    const int kdec = dec_row_floats(H);
    const int bshift = lbs - 5;
    int item_base = 0;
    for (int s = 0; s < nst && wok; ++s) {
      const StageEnt& st = stg[s];
      const int nt = st.ntok, rg = rows_per_item(nt, 2);
      const int nitems = (st.nrows + rg - 1) / rg;
      int i = ((warp - item_base) % NWP + NWP) % NWP;
      item_base += nitems;
      if (i >= nitems) continue;
      if (!mbar_wait(&full[s], 0u, status)) {
        wok = false;
        break;
      }
      const SlotLayout SL = fused_stage_layout(st.nrows, H, nbH, HAS_ZP);
      const uint8_t* sb = ring + st.pad[1];
      const float4* xr[kTokGroup];
#pragma unroll
      for (int j = 0; j < kTokGroup; ++j) {
        const int jj = j < nt ? j : 0;
        xr[j] = reinterpret_cast<const float4*>(xdec) + (size_t)(s_perm[st.pbase + jj] / k) * (kdec / 4);
      }
      for (; i < nitems; i += NWP) {
        auto epi = [&](auto& acc_, auto ntc, auto rgc) {
          constexpr int NTC = decltype(ntc)::value, RGC = decltype(rgc)::value;
          const int rb = i * RGC, nr = min(RGC, st.nrows - rb);
          item_dot<2, NTC, RGC, TS, HAS_ZP>(sb, SL, st, rb, nr, xr, H, nbH, bshift, magic, neg_magic, zfixed, lane,
                                            acc_);
          const int r = lane / NTC, j = lane - r * NTC;
          if (r < nr && r < RGC) {
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int rr = 0; rr < RGC; ++rr)
#pragma unroll
              for (int jj = 0; jj < NTC; ++jj)
                if (rr == r && jj == j) {
                  v0 = acc_[0][rr][jj];
                  v1 = acc_[1][rr][jj];
                }
            const int ii = st.row0 + rb + r;
            act_own[(size_t)j * cmax + st.pad[2] + rb + r] = v0 / (1.f + expf(-v0)) * v1 * dec_prescale(ii);
          }
        };
        switch (nt) {
          case 1: { float a_[2][rows_per_item(1, 2)][1]; epi(a_, std::integral_constant<int, 1>(), std::integral_constant<int, rows_per_item(1, 2)>()); break; }
          case 2: { float a_[2][rows_per_item(2, 2)][2]; epi(a_, std::integral_constant<int, 2>(), std::integral_constant<int, rows_per_item(2, 2)>()); break; }
          case 3: { float a_[2][rows_per_item(3, 2)][3]; epi(a_, std::integral_constant<int, 3>(), std::integral_constant<int, rows_per_item(3, 2)>()); break; }
          default: { float a_[2][rows_per_item(4, 2)][4]; epi(a_, std::integral_constant<int, 4>(), std::integral_constant<int, rows_per_item(4, 2)>()); break; }
        }
      }
    }
    if (!wok) s_misc[kMiscAbort] = 1;
  }
  // no reuse of the ring (or exit) while bulk copies into it are in flight
  if (tid == 0)
    for (int s = 0; s < nst; ++s)
      if (!mbar_wait(&full[s], 0u, status)) {
        s_misc[kMiscAbort] = 1;
        break;
      }

  // ---- 4. the window's SwiGLU slice from the cluster: window row c is
  //         owned by the CTA whose 8-row range holds it
  if (CL > 1) cluster_sync_all();
  else __syncthreads();
  const int crows = 32 * nwu;
  for (int idx = tid; idx < T * crows; idx += NTH) {
    const int n = idx / crows, c = idx - n * crows;
    int owner = 0;
#pragma unroll
    for (int r = 1; r < CL; ++r)
      if (c >= s_misc[kMiscRng + r]) owner = r;
    const float* src = act_own + (size_t)n * cmax + c;
    act_all[(size_t)n * cmax + c] = CL > 1 ? ld_dsmem_f32(src, (uint32_t)owner) : *src;
  }
  if (CL > 1) cluster_sync_all();  // peers are done reading this CTA's shared memory
  else __syncthreads();
  if (tid == 0 && !mbar_wait(dbar, 0u, status)) s_misc[kMiscAbort] = 1;
  __syncthreads();
  const bool abort = s_misc[kMiscAbort] != 0;

  // ---- 5. down: item (unit u, output row hs0 + r) is the dot product of
  //         the unit's 16 bytes (32 codes) of that row with the unit's 32
  //         SwiGLU values, per assignment, times the block scale.  A second
  //         pass sums each row over the units in order, weighted by the
  //         routing weights, and adds it, in 2^-32 fixed point, to the
  //         output accumulator (integer adds: the sum over clusters does not
  //         depend on their order).
  {
    const int ns = P.slice, nit = nwu * ns;
    float* dpart = reinterpret_cast<float*>(ring);  // [unit][4][ns]: the ring is free now
    const bool wide = P.box_w > 16;
    // work item: (unit u, 32 rows) = one row per lane; each warp takes a
    // contiguous range of these (mostly one unit) and keeps the unit's 32
    // SwiGLU values per assignment in registers
    const int rg_per_u = (ns + 31) >> 5, ng = nwu * rg_per_u;
    const int g0 = (warp * ng) / NWP, g1 = ((warp + 1) * ng) / NWP;
    int ucur = -1, ntok = 0;
    XChunk xa;  // one token: the unit's SwiGLU values, reloaded when the unit changes
    for (int gi = g0; gi < g1 && !abort; ++gi) {
      const int u = gi / rg_per_u, r = (gi - u * rg_per_u) * 32 + lane;
      if (u != ucur) {
        ucur = u;
        ntok = seg[unit[u].seg].ntok;
        if (NTR == 1) {
          const float4* ap = reinterpret_cast<const float4*>(act_all + 32 * u);
#pragma unroll
          for (int v = 0; v < 8; ++v) xa.v[v] = ap[v];
        }
      }
      if (r >= ns) continue;  // a slice that is not a multiple of 32 rows
      const int item = u * ns + r;
      const uint32_t zp = HAS_ZP ? (uint32_t)dzp[item] : 8u;
      const float sc = Half<TS>::to_float(dsc[item]);
      const int cg = wide ? unit[u].seg : u;
      const uint4 qv = *reinterpret_cast<const uint4*>(
          dn + ((size_t)cg * ns + r) * P.box_w + (wide ? (u - seg[cg].u0) * 16 : 0));
      f2 wv[16];
      dequant_chunk(qv, HAS_ZP ? zconst(zp, neg_magic) : zfixed, magic, wv);
      if (NTR == 1) {
        dpart[(size_t)u * 4 * ns + r] = sc * chunk_dot(wv, xa);
      } else {
#pragma unroll
        for (int n = 0; n < NTR; ++n)
          if (n < ntok) {
            XChunk xn;
            const float4* ap = reinterpret_cast<const float4*>(act_all + (size_t)n * cmax + 32 * u);
#pragma unroll
            for (int v = 0; v < 8; ++v) xn.v[v] = ap[v];
            dpart[((size_t)u * 4 + n) * ns + r] = sc * chunk_dot(wv, xn);
          }
      }
    }
    __syncthreads();
    for (int idx = tid; idx < T * ns; idx += NTH) {
      const int t = idx / ns, rr = idx - t * ns;
      float v = 0.f;
      if (!abort)
        for (int uu = 0; uu < nwu; ++uu) {
          const SegEnt& sg = seg[unit[uu].seg];
#pragma unroll
          for (int n = 0; n < NTR; ++n)
            if (n < sg.ntok && sg.tok[n] == t) v = fmaf(sg.w[n], dpart[((size_t)uu * 4 + n) * ns + rr], v);
        }
      if (!(fabsf(v) < 1073741824.f)) set_status(status, QMOE_ST_RANGE);  // beyond the fixed-point range (or NaN)
      if (v != 0.f)
        atomicAdd(reinterpret_cast<unsigned long long*>(f.acc + (size_t)t * H + hs0 + rr),
                  (unsigned long long)__float2ll_rn(v * 4294967296.f));
    }
  }

  // ---- 6. the last cluster to finish this quarter of H converts it to the
  //         output (plus the residual) and clears the accumulator
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t old = atomicAdd(g.ctl + kCtlSliceDone + rank, 1u);
    s_misc[kMiscLast] = old == (uint32_t)(ncl - 1);
  }
  __syncthreads();
  if (!s_misc[kMiscLast]) return;
  __threadfence();
  {
    const int ns = P.slice;
    uint16_t* out = static_cast<uint16_t*>(d.out);
    for (int idx = tid; idx < T * ns / 2; idx += NTH) {
      const int t = (2 * idx) / ns, h = hs0 + 2 * idx - t * ns;
      long long* ap = f.acc + (size_t)t * H + h;
      const longlong2 a = __ldcg(reinterpret_cast<const longlong2*>(ap));
      float v0 = __ll2float_rn(a.x) * 2.3283064365386963e-10f;  // 2^-32
      float v1 = __ll2float_rn(a.y) * 2.3283064365386963e-10f;
      uint32_t* op = reinterpret_cast<uint32_t*>(out + (size_t)t * H + h);
      if (d.accumulate) {
        const uint32_t o = *op;
        v0 += Half<TA>::to_float((uint16_t)(o & 0xFFFFu));
        v1 += Half<TA>::to_float((uint16_t)(o >> 16));
      }
      *op = (uint32_t)Half<TA>::from_float(v0) | ((uint32_t)Half<TA>::from_float(v1) << 16);
      *reinterpret_cast<longlong2*>(ap) = make_longlong2(0, 0);
    }
  }
  if (tid == 0) atomicExch(g.ctl + kCtlSliceDone + rank, 0u);
}

// ------------------------------------------------------------ fused host

// Shared-memory plan of the fused layer for `grid` CTAs in clusters of `cl`;
// cpl > 0: the T = 1 path with activations in registers (H = 1024 * cpl).
static bool plan_fused(int T, int H, int I, int E, int k, int bs, bool has_zp, int grid, int cl, int cpl,
                       FusedPlan* out) {
  if (T < 1 || T > kTokGroup || T * k > 32 || grid < cl || cl < 1 || kMaxSplit % cl || grid % cl) return false;
  if (H % 32 || I % 32 || E > kMaxExperts || T * H > kCtlAccElems) return false;
  if (cpl > 0 && (T != 1 || H != 1024 * cpl)) return false;
  FusedPlan P = {};
  const int A = T * k, dmax = A < E ? A : E;
  const int ncl = grid / cl;
  const int U = dmax * (I / 32);
  const int cunits = (U + ncl - 1) / ncl;
  if (cunits > kFMaxUnits || (long long)U * ncl >= (1LL << 31)) return false;
  P.crows_max = 32 * (cunits < 1 ? 1 : cunits);
  P.rows_max = 8 * ((P.crows_max / 8 + cl - 1) / cl);
  P.max_segs = P.crows_max / I + 2;
  if (P.max_segs > kFMaxSegs) P.max_segs = kFMaxSegs;
  P.max_stages = P.rows_max / kFStageRows;  // every stage is exactly 8 rows
  if (P.max_stages > kFMaxStages) return false;
  // down: this CTA's quarter of H, boxes of at most 256 rows
  P.slice = H / cl;
  P.box_r = P.slice <= 256 ? P.slice : 256;
  if (P.slice % P.box_r || cunits * P.slice > kFMaxItems * kFusedThreads) return false;
  P.nboxes = P.slice / P.box_r;
  const int nbH = H / bs;
  // gate-up ring: every stage of the CTA resident at once
  const uint32_t ring = P.max_stages * fused_stage_layout(kFStageRows, H, nbH, has_zp).bytes;
  const int VR = kMaxSplit / cl, rps = route_rows_per_split(H);
  uint32_t o = kFFixed;
  P.vpart_off = o;
  o = al16(o + (uint32_t)VR * 4 * E * 4);
  P.gu_off = o;
  o = al16(o + (uint32_t)P.crows_max * 2 * 4);
  P.acto_off = o;
  o = al16(o + (uint32_t)kTokGroup * P.crows_max * 4);
  P.acta_off = o;
  o = al16(o + (uint32_t)kTokGroup * P.crows_max * 4);
  P.xdec_off = o;
  if (cpl == 0) o = al16(o + (uint32_t)T * dec_row_floats(H) * 4);
  P.dsc_off = o;
  o = al16(o + (uint32_t)cunits * P.slice * 2);
  P.dzp_off = o;
  o = al16(o + (uint32_t)cunits * P.slice);
  P.dn_off = (o + 127u) & ~127u;
  // down codes: a box per segment (box_w = the window's width) if that fits
  // the budget, else a box per 32-code unit
  const uint32_t dn_narrow = (uint32_t)cunits * P.slice * 16;
  const uint32_t dn_wide = (uint32_t)P.max_segs * P.slice * 16 * cunits;
  P.box_w = 16;
  uint32_t dn_b = dn_narrow;
  if (cunits > 1 && 16 * cunits <= 256) {
    // the least the ring must hold: the gate-up stages, the router scratch
    // with 8 staged rows, the down phase's per-unit dot products
    const uint32_t xs_b0 = (uint32_t)(kMaxSplit / cl) * route_rows_per_split(H) * 16;
    const uint32_t part_b0 = (uint32_t)(kMaxSplit / cl) * 8 * 4 * E * 4;
    uint32_t room_min = ring;
    const uint32_t router_min = al16(xs_b0) + al16(part_b0) + al16(16u * E);
    if (router_min > room_min) room_min = router_min;
    if ((uint32_t)cunits * 4 * P.slice * 4 > room_min) room_min = (uint32_t)cunits * 4 * P.slice * 4;
    const uint32_t ring_w = (((P.dn_off + dn_wide) + 1023u) & ~1023u);
    if (ring_w + ((room_min + 127u) & ~127u) <= kSmemBudget) {
      P.box_w = 16 * cunits;
      dn_b = dn_wide;
    }
  }
  o = P.dn_off + dn_b;
  P.ring_off = (o + 1023u) & ~1023u;
  if (P.ring_off > kSmemBudget) return false;
  // router scratch inside the ring: all of the CTA's router rows in one
  // pass if the budget allows, else passes of a multiple of 8 rows
  const uint32_t xs_b = (uint32_t)VR * rps * 16, part_b = (uint32_t)VR * 8 * 4 * E * 4;
  P.xs_off = P.ring_off;
  P.part_off = P.xs_off + al16(xs_b);
  P.wch_off = P.part_off + al16(part_b);
  const uint32_t used = P.wch_off - P.ring_off;
  const uint32_t avail = kSmemBudget - P.ring_off;
  if (avail < used + 16u * E || avail < ring) return false;
  int pr = (int)(((avail - used) / (2u * E)) & ~7u);
  if (pr > VR * rps) pr = VR * rps;
  P.pass_rows = pr;
  uint32_t room = ring;
  const uint32_t router_b = used + al16((uint32_t)pr * E * 2);
  if (router_b > room) room = router_b;
  // the down phase's per-unit dot products
  const uint32_t dpart_b = (uint32_t)cunits * 4 * P.slice * 4;
  if (dpart_b > room) room = dpart_b;
  P.smem = P.ring_off + ((room + 127u) & ~127u);
  if (P.smem > kSmemBudget) return false;
  *out = P;
  return true;
}

// CTAs of a launch in clusters of kFusedCluster at one CTA per SM (cached
// per device and kernel)
template <typename F>
static int fused_grid(F* fn) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    if (ensure_smem(fn, kSmemBudget) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kFusedCluster * 64);
    cfg.blockDim = dim3(kFusedThreads);
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

template <typename TS, typename TA, bool Z, int ME, int CPL>
static cudaError_t launch_fused_t(const FusedParams& f, cudaStream_t st, bool pdl, bool check_only) {
  auto fn = fused_decode_kernel<TS, TA, Z, ME, kFusedCluster, CPL>;
  const int grid = fused_grid(fn);
  FusedPlan P;
  if (grid < kFusedCluster ||
      !plan_fused(f.g.T, f.g.K, f.g.N, f.g.E, f.g.k, f.g.bs, Z, grid, kFusedCluster, CPL, &P))
    return cudaErrorInvalidValue;
  if (check_only) return encode_fn() ? cudaSuccess : cudaErrorInvalidValue;
  // down codes [E * H rows, I / 2 bytes]: boxes of box_w bytes by box_r
  // rows; 256-byte L2 promotion also fetches the neighbouring units, which
  // the clusters next to this one read
  CUtensorMap tm;
  if (!make_map(&tm, f.d.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)f.d.K / 2, (uint64_t)f.d.E * f.d.N,
                (uint32_t)P.box_w, (uint32_t)P.box_r, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  cudaError_t err = ensure_smem(fn, P.smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFusedCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fn, tm, f, P);
}

template <typename TS, typename TA, bool Z>
static cudaError_t launch_fused_me(const FusedParams& f, cudaStream_t st, bool pdl, bool check_only) {
  const bool fast = f.g.T == 1 && f.g.K == 2048;
  if (f.g.E <= 64)
    return fast ? launch_fused_t<TS, TA, Z, 2, 2>(f, st, pdl, check_only)
                : launch_fused_t<TS, TA, Z, 2, 0>(f, st, pdl, check_only);
  return fast ? launch_fused_t<TS, TA, Z, 8, 2>(f, st, pdl, check_only)
              : launch_fused_t<TS, TA, Z, 8, 0>(f, st, pdl, check_only);
}

}  // namespace qmoe
