// decode.cu -- small-T path of the layer (T <= 16 tokens): int4 weight rows
// are streamed from HBM with bulk TMA copies into a shared-memory ring,
// dequantised in registers and reduced with warp shuffles.  Also the dense
// MatMulNBits GEMV (E = 1).
//
// Sources: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), IR guide
// update "Fused MoE Extern Kernels": kernel 1 (gate + up projection with the
// SwiGLU fused, INT4 dequantisation inside the dot-product loop) and kernel 2
// (down projection with the routing-weighted reduce over the k experts fused);
// DequantizeLinear with block_size from local fix A1: w = (q - zp) * scale;
// SwiGLU act = silu(gate) * up from IR guide 3, Expert Computation step 5.
//
// GB300 design.  The pages' kernels give one warp per output row and read
// 4-byte words.  Here every CTA (one per SM) owns a contiguous slice of
// output rows and walks all selected experts for that slice, so each SM
// streams the same number of bytes whatever the routing.  A producer warp
// issues cp.async.bulk copies of whole row slices (contiguous in the
// [E, N, K/2] layout) plus their scales / zero points into a ring of shared
// memory stages guarded by mbarriers, so all of a CTA's bytes can be in
// flight at once.  Consumer warps read 16-byte chunks (32 codes = one 32-wide
// block), turn nibble j of each 16-bit half into the exact float
// (q - zp) * 16^j with one LOP3 and one packed subtract (magic exponent
// 2^23), and FMA with activations pre-scaled by 16^-j (fma.rn.f32x2), all
// in fp32.  Work is grouped per distinct expert, so every weight byte is
// read once per call even when several tokens chose the same expert.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

constexpr int kCW = 16;                         // consumer warps
constexpr int kDecodeThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kMaxSlots = 16;
constexpr uint32_t kFixedSmem = 3584;           // barriers, stage headers, routing copy
constexpr uint32_t kSmemBudget = 232448;        // 227 KB dynamic shared memory

struct SlotHdr {
  int e, ntok, ph[4];  // ph: alignment phase of scales0, scales1, zp0, zp1 images
  int a[kTokGroup], t[kTokGroup];
};
static_assert(sizeof(SlotHdr) <= 64, "stage header must fit 64 bytes");

struct SlotLayout {
  uint32_t w[2], s[2], z[2], act, bytes;
};

__host__ __device__ inline uint32_t al16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline SlotLayout slot_layout(int mode, int rows, int K, int nb, bool has_zp,
                                                  int act_row_floats, int T) {
  SlotLayout L;
  const int nmat = (mode == kModeGateUp) ? 2 : 1;
  uint32_t o = 0;
  for (int m = 0; m < 2; ++m) {
    L.w[m] = o;
    if (m < nmat) o += (uint32_t)rows * (K / 2);
  }
  for (int m = 0; m < 2; ++m) {
    L.s[m] = o;
    if (m < nmat) o = al16(o + (uint32_t)rows * nb * 2 + 16);
  }
  for (int m = 0; m < 2; ++m) {
    L.z[m] = o;
    if (m < nmat && has_zp) o = al16(o + (uint32_t)rows * nb + 16);
  }
  L.act = o;
  if (mode == kModeDown) o += (uint32_t)(T < kTokGroup ? T : kTokGroup) * act_row_floats * 4;
  L.bytes = (o + 127u) & ~127u;
  return L;
}

// Producer-warp copy of `bytes` global bytes into shared memory at
// dst_base + (src mod 16): the 16-byte-aligned middle goes by bulk copy
// (counted on `bar`), the ragged head / tail bytes by plain loads.
// Returns the phase (src mod 16).  Lane 0 must have added body bytes to the
// barrier's expected transaction count (see body_bytes()).
__device__ __forceinline__ uint32_t body_bytes(const void* src, uint32_t bytes) {
  const uint32_t ph = (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u);
  const uint32_t head = min(bytes, (16u - ph) & 15u);
  return (bytes - head) & ~15u;
}
__device__ __forceinline__ int stage_bytes(uint8_t* dst_base, const uint8_t* src, uint32_t bytes,
                                           uint64_t* bar, int lane) {
  const uint32_t ph = (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u);
  const uint32_t head = min(bytes, (16u - ph) & 15u);
  const uint32_t body = (bytes - head) & ~15u;
  const uint32_t tail = bytes - head - body;
  uint8_t* dst = dst_base + ph;
  if (lane == 0 && body) bulk_g2s(dst + head, src + head, body, bar);
  if ((uint32_t)lane < head) dst[lane] = __ldg(src + lane);
  if ((uint32_t)lane < tail) dst[head + body + lane] = __ldg(src + head + body + lane);
  return (int)ph;
}

// One output row against up to kTokGroup activation rows (decode layout).
// wrow: 16-byte chunks of packed codes; srow / zrow: the row's block scales
// and zero points; xs[j]: activation row j.  acc[j] += row . x_j (fp32).
template <typename TS, bool HAS_ZP>
__device__ __forceinline__ void row_dot(const uint8_t* wrow, const uint16_t* srow,
                                        const uint8_t* zrow, int nchunks, int bshift,
                                        const float* const* xs, int ntok, float* acc, int lane) {
  constexpr uint32_t kMagic = 0x4B000000u;  // 2^23
  for (int c = lane; c < nchunks; c += 32) {
    const uint4 q = *reinterpret_cast<const uint4*>(wrow + c * 16);
    const int blk = c >> bshift;
    const float s = Half<TS>::to_float(srow[blk]);
    const float z = HAS_ZP ? (float)zrow[blk] : 8.f;
    const f2 c01 = {8388608.f + z, fmaf(z, 16.f, 8388608.f)};
    const f2 c23 = {fmaf(z, 256.f, 8388608.f), fmaf(z, 4096.f, 8388608.f)};
    f2 wv[16];
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = qw[i], vh = qw[i] >> 16;
      wv[4 * i + 0] = fsub2({__uint_as_float(kMagic | (v & 0xFu)), __uint_as_float(kMagic | (v & 0xF0u))}, c01);
      wv[4 * i + 1] = fsub2({__uint_as_float(kMagic | (v & 0xF00u)), __uint_as_float(kMagic | (v & 0xF000u))}, c23);
      wv[4 * i + 2] = fsub2({__uint_as_float(kMagic | (vh & 0xFu)), __uint_as_float(kMagic | (vh & 0xF0u))}, c01);
      wv[4 * i + 3] = fsub2({__uint_as_float(kMagic | (vh & 0xF00u)), __uint_as_float(kMagic | (vh & 0xF000u))}, c23);
    }
    const int xo = ((c >> 5) * 8) * 32 + (c & 31);  // float4 index of f = 0
#pragma unroll
    for (int j = 0; j < kTokGroup; ++j) {
      if (j < ntok) {
        const float4* xr = reinterpret_cast<const float4*>(xs[j]) + xo;
        f2 d0 = {0.f, 0.f}, d1 = {0.f, 0.f}, d2 = {0.f, 0.f}, d3 = {0.f, 0.f};
#pragma unroll
        for (int f = 0; f < 8; f += 2) {
          const float4 xa = xr[f * 32];
          const float4 xb = xr[(f + 1) * 32];
          d0 = ffma2(wv[2 * f], {xa.x, xa.y}, d0);
          d1 = ffma2(wv[2 * f + 1], {xa.z, xa.w}, d1);
          d2 = ffma2(wv[2 * f + 2], {xb.x, xb.y}, d2);
          d3 = ffma2(wv[2 * f + 3], {xb.z, xb.w}, d3);
        }
        const float dot = ((d0.x + d0.y) + (d1.x + d1.y)) + ((d2.x + d2.y) + (d3.x + d3.y));
        acc[j] = fmaf(s, dot, acc[j]);
      }
    }
  }
}

// Stage iterator: (d-th active expert, first token of the group).
struct StageIt {
  int d, g0;
};

template <int MODE, typename TS, typename TA, bool HAS_ZP>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxSlots;
  SlotHdr* hdr = reinterpret_cast<SlotHdr*>(smem + 256);
  int* s_active = reinterpret_cast<int*>(smem + 256 + 64 * kMaxSlots);  // [0]=D, [1..D]
  int* s_off = s_active + (kMaxExperts + 2);                             // [E+1]
  float* res = reinterpret_cast<float*>(smem + kFixedSmem);
  uint8_t* slots = smem + p.slot_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = p.ctl ? p.ctl + kCtlStatus : nullptr;
  const int N = p.N, K = p.K, nb = p.nb;
  const int r0 = (int)(((long long)blockIdx.x * N) / gridDim.x);
  const int r1 = (int)(((long long)(blockIdx.x + 1) * N) / gridDim.x);
  const int nrows = r1 - r0;
  const int NS = p.nslots;
  const SlotLayout SL = slot_layout(MODE, p.rows_per_cta_max, K, nb, HAS_ZP, p.src_row_floats, p.T);
  const int kdec = dec_row_floats(K);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 32);
      mbar_init(&empty[i], kCW);
    }
    fence_barrier_init();
  }
  // activations resident for the whole kernel (gate-up / dense)
  if (MODE != kModeDown) {
    const uint16_t* x = static_cast<const uint16_t*>(p.x16);
    const int n = p.T * K;
    for (int i = tid; i < n; i += kDecodeThreads) {
      const int t = i / K, kk = i - t * K;
      res[t * kdec + dec_index(kk)] = Half<TA>::to_float(x[i]) * dec_prescale(kk);
    }
  } else {
    for (int i = tid; i < p.T * p.rows_per_cta_max; i += kDecodeThreads) res[i] = 0.f;
  }
  // routing (written by the router; for down, complete before this grid starts)
  if (MODE == kModeGateUp) pdl_wait();
  if (MODE == kModeDense) {
    if (tid == 0) {
      s_active[0] = 1;
      s_active[1] = 0;
      s_off[0] = 0;
      s_off[1] = p.T;
    }
  } else {
    for (int i = tid; i <= p.E; i += kDecodeThreads) s_off[i] = p.offsets[i];
    const int D = p.active[0];
    for (int i = tid; i <= D; i += kDecodeThreads) s_active[i] = p.active[i];
  }
  __syncthreads();
  if (MODE == kModeGateUp) pdl_trigger();
  const int D = s_active[0];

  auto n_of = [&](int d) {
    const int e = s_active[1 + d];
    return s_off[e + 1] - s_off[e];
  };

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    const int nmat = (MODE == kModeGateUp) ? 2 : 1;
    bool waited = (MODE != kModeDown);
    StageIt it = {0, 0};
    int stage = 0;
    // Down: weights of the first ring-full of stages go out before the
    // previous grid (gate-up, which writes act) has finished.
    int deferred_begin = -1, deferred_end = -1;
    StageIt deferred_it = it;
    for (; it.d < D; ++stage) {
      const int slot = stage % NS;
      const int round = stage / NS;
      if (round > 0) {
        if (!waited) {
          // flush the deferred activation copies before reusing a slot
          pdl_wait();
          waited = true;
          StageIt jt = deferred_it;
          for (int s2 = deferred_begin; s2 < deferred_end; ++s2) {
            const int sl = s2 % NS;
            const int n = n_of(jt.d), nt = min(kTokGroup, n - jt.g0);
            for (int j = 0; j < nt; ++j)
              if (lane == 0)
                bulk_g2s(slots + sl * SL.bytes + SL.act + (uint32_t)j * p.src_row_floats * 4,
                         p.src + (size_t)hdr[sl].a[j] * p.src_row_floats, p.src_row_floats * 4u,
                         &full[sl]);
            __syncwarp();
            mbar_arrive(&full[sl]);
            jt.g0 += kTokGroup;
            if (jt.g0 >= n) { ++jt.d; jt.g0 = 0; }
          }
        }
        if (!mbar_wait(&empty[slot], (round - 1) & 1, status)) break;
      }
      const int e = s_active[1 + it.d];
      const int n = n_of(it.d);
      const int ntok = min(kTokGroup, n - it.g0);
      uint8_t* sb = slots + slot * SL.bytes;
      // stage header
      if (lane == 0) {
        hdr[slot].e = e;
        hdr[slot].ntok = ntok;
      }
      if (lane < ntok) {
        const int a = (MODE == kModeDense) ? (it.g0 + lane) : p.perm[s_off[e] + it.g0 + lane];
        hdr[slot].a[lane] = a;
        hdr[slot].t[lane] = (MODE == kModeDense) ? a : a / p.k;
      }
      // expected transaction bytes
      uint32_t tx = 0;
      const size_t row0 = (size_t)e * N + r0;
      for (int m = 0; m < nmat; ++m) {
        tx += (uint32_t)nrows * (K / 2);
        tx += body_bytes(static_cast<const uint8_t*>(p.s[m]) + row0 * nb * 2, (uint32_t)nrows * nb * 2);
        if (HAS_ZP) tx += body_bytes(p.z[m] + row0 * nb, (uint32_t)nrows * nb);
      }
      if (MODE == kModeDown) tx += (uint32_t)ntok * p.src_row_floats * 4;
      if (lane == 0) asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&full[slot])), "r"(tx) : "memory");
      __syncwarp();
      for (int m = 0; m < nmat; ++m) {
        if (lane == 0) bulk_g2s(sb + SL.w[m], p.w[m] + row0 * (K / 2), (uint32_t)nrows * (K / 2), &full[slot]);
        const int phs = stage_bytes(sb + SL.s[m], static_cast<const uint8_t*>(p.s[m]) + row0 * nb * 2,
                                    (uint32_t)nrows * nb * 2, &full[slot], lane);
        int phz = 0;
        if (HAS_ZP) phz = stage_bytes(sb + SL.z[m], p.z[m] + row0 * nb, (uint32_t)nrows * nb, &full[slot], lane);
        if (lane == 0) {
          hdr[slot].ph[m] = phs;
          hdr[slot].ph[2 + m] = phz;
        }
      }
      __syncwarp();
      if (MODE == kModeDown && !waited) {
        if (deferred_begin < 0) {
          deferred_begin = stage;
          deferred_it = it;
        }
        deferred_end = stage + 1;
      } else {
        if (MODE == kModeDown) {
          for (int j = 0; j < ntok; ++j)
            if (lane == 0)
              bulk_g2s(sb + SL.act + (uint32_t)j * p.src_row_floats * 4,
                       p.src + (size_t)hdr[slot].a[j] * p.src_row_floats, p.src_row_floats * 4u,
                       &full[slot]);
          __syncwarp();
        }
        mbar_arrive(&full[slot]);
      }
      it.g0 += kTokGroup;
      if (it.g0 >= n) { ++it.d; it.g0 = 0; }
    }
    if (!waited) {
      pdl_wait();
      StageIt jt = deferred_it;
      for (int s2 = deferred_begin; s2 >= 0 && s2 < deferred_end; ++s2) {
        const int sl = s2 % NS;
        const int n = n_of(jt.d), nt = min(kTokGroup, n - jt.g0);
        for (int j = 0; j < nt; ++j)
          if (lane == 0)
            bulk_g2s(slots + sl * SL.bytes + SL.act + (uint32_t)j * p.src_row_floats * 4,
                     p.src + (size_t)hdr[sl].a[j] * p.src_row_floats, p.src_row_floats * 4u, &full[sl]);
        __syncwarp();
        mbar_arrive(&full[sl]);
        jt.g0 += kTokGroup;
        if (jt.g0 >= n) { ++jt.d; jt.g0 = 0; }
      }
    }
    // drain: do not exit while bulk copies into this CTA's smem are in flight
    for (int s2 = max(0, stage - NS); s2 < stage; ++s2)
      if (!mbar_wait(&full[s2 % NS], (s2 / NS) & 1, status)) break;
    return;
  }

  // -------------------------------------------------------------- consumers
  const int nchunks = K / 32;
  const int bshift = (p.bs == 32) ? 0 : (p.bs == 64 ? 1 : 2);
  StageIt it = {0, 0};
  int stage = 0;
  bool ok = true;
  for (; it.d < D; ++stage) {
    const int slot = stage % NS;
    if (!mbar_wait(&full[slot], (stage / NS) & 1, status)) { ok = false; break; }
    const SlotHdr h = hdr[slot];
    const uint8_t* sb = slots + slot * SL.bytes;
    const float* xs[kTokGroup];
#pragma unroll
    for (int j = 0; j < kTokGroup; ++j) {
      const int jj = j < h.ntok ? j : 0;
      if (MODE == kModeDown)
        xs[j] = reinterpret_cast<const float*>(sb + SL.act) + (size_t)jj * p.src_row_floats;
      else
        xs[j] = res + (size_t)h.t[jj] * kdec;
    }
    // rows of this stage: gate-up rotates the warp order per stage so all
    // warps stay busy; down keeps row ownership fixed (deterministic sums).
    const int first = (MODE == kModeGateUp) ? ((warp - (stage * nrows) % kCW) % kCW + kCW) % kCW : warp;
    for (int r = first; r < nrows; r += kCW) {
      float acc0[kTokGroup] = {0.f, 0.f, 0.f, 0.f};
      row_dot<TS, HAS_ZP>(sb + SL.w[0] + (size_t)r * (K / 2),
                          reinterpret_cast<const uint16_t*>(sb + SL.s[0] + h.ph[0]) + (size_t)r * nb,
                          sb + SL.z[0] + h.ph[2] + (size_t)r * nb, nchunks, bshift, xs, h.ntok, acc0, lane);
      if (MODE == kModeGateUp) {
        float acc1[kTokGroup] = {0.f, 0.f, 0.f, 0.f};
        row_dot<TS, HAS_ZP>(sb + SL.w[1] + (size_t)r * (K / 2),
                            reinterpret_cast<const uint16_t*>(sb + SL.s[1] + h.ph[1]) + (size_t)r * nb,
                            sb + SL.z[1] + h.ph[3] + (size_t)r * nb, nchunks, bshift, xs, h.ntok, acc1, lane);
        const int i = r0 + r;
        const int di = dec_index(i);
        const float pre = dec_prescale(i);
#pragma unroll
        for (int j = 0; j < kTokGroup; ++j) {
          if (j < h.ntok) {
            const float g = warp_sum(acc0[j]);
            const float u = warp_sum(acc1[j]);
            if (lane == 0) {
              const float act = g / (1.f + expf(-g)) * u;
              p.act_out[(size_t)h.a[j] * p.act_row_floats + di] = act * pre;
            }
          }
        }
      } else if (MODE == kModeDown) {
#pragma unroll
        for (int j = 0; j < kTokGroup; ++j) {
          if (j < h.ntok) {
            const float y = warp_sum(acc0[j]);
            if (lane == 0) res[h.t[j] * p.rows_per_cta_max + r] += p.topk_w[h.a[j]] * y;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < kTokGroup; ++j) {
          if (j < h.ntok) {
            const float y = warp_sum(acc0[j]);
            if (lane == 0)
              static_cast<uint16_t*>(p.out)[(size_t)h.t[j] * N + r0 + r] = Half<TA>::from_float(y);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    it.g0 += kTokGroup;
    if (it.g0 >= n_of(it.d)) { ++it.d; it.g0 = 0; }
  }
  if (MODE == kModeDown) {
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    if (!ok) return;
    uint16_t* out = static_cast<uint16_t*>(p.out);
    for (int i = tid; i < p.T * nrows; i += kCW * 32) {
      const int t = i / nrows, r = i - t * nrows;
      float v = res[t * p.rows_per_cta_max + r];
      const size_t o = (size_t)t * N + r0 + r;
      if (p.accumulate) v += Half<TA>::to_float(out[o]);
      out[o] = Half<TA>::from_float(v);
    }
  }
}

// ------------------------------------------------------------------- host

struct DecodePlan {
  int grid, rows_max, nslots;
  uint32_t slot_base, smem;
};

static bool plan_decode(int mode, int T, int N, int K, int bs, bool has_zp, int k, int E, int sms,
                        DecodePlan* out) {
  DecodePlan P;
  P.grid = N < sms ? N : sms;
  P.rows_max = (N + P.grid - 1) / P.grid;
  const int nb = K / bs;
  const int act_row = dec_row_floats(K);
  const SlotLayout SL = slot_layout(mode, P.rows_max, K, nb, has_zp, act_row, T);
  const uint32_t res = (mode == kModeDown) ? (uint32_t)T * P.rows_max * 4 : (uint32_t)T * act_row * 4;
  P.slot_base = (kFixedSmem + res + 1023u) & ~1023u;
  if (P.slot_base + 2 * SL.bytes > kSmemBudget) return false;
  int ns = (int)((kSmemBudget - P.slot_base) / SL.bytes);
  // no more slots than stages a CTA can have: sum over experts of
  // ceil(n_e / kTokGroup) with sum n_e = A, at most min(A, E) experts
  const int A = T * k;
  const int dmax = A < E ? A : E;
  const int max_stages = (mode == kModeDense) ? (T + kTokGroup - 1) / kTokGroup
                                              : dmax + (A - dmax + kTokGroup - 1) / kTokGroup;
  if (ns > max_stages) ns = max_stages < 2 ? 2 : max_stages;
  if (ns > kMaxSlots) ns = kMaxSlots;
  P.nslots = ns;
  P.smem = P.slot_base + ns * SL.bytes;
  *out = P;
  return true;
}

bool decode_fits(int mode, int T, int N, int K, int bs, bool has_zp, int k) {
  DecodePlan P;
  return T >= 1 && T <= kDecodeMaxTokens &&
         plan_decode(mode, T, N, K, bs, has_zp, k, kMaxExperts, device_sm_count(), &P);
}

template <int MODE, typename TS, typename TA, bool HAS_ZP>
static cudaError_t launch_decode_t(DecodeParams p, cudaStream_t st, bool pdl) {
  DecodePlan P;
  const int E = (MODE == kModeDense) ? 1 : p.E;
  if (!plan_decode(MODE, p.T, p.N, p.K, p.bs, HAS_ZP, p.k, E, device_sm_count(), &P))
    return cudaErrorInvalidValue;
  p.rows_per_cta_max = P.rows_max;
  p.nslots = P.nslots;
  p.slot_base = P.slot_base;
  auto fn = decode_kernel<MODE, TS, TA, HAS_ZP>;
  cudaError_t err = ensure_smem(decode_kernel<MODE, TS, TA, HAS_ZP>, P.smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(fn, dim3(P.grid), dim3(kDecodeThreads), (size_t)P.smem, st, pdl, p);
}

template <int MODE>
static cudaError_t dispatch_decode(const DecodeParams& p, int act_dtype, int scale_dtype, bool has_zp,
                                   cudaStream_t st, bool pdl) {
  const bool abf = act_dtype == 1, sbf = scale_dtype == 1;
#define QMOE_DEC(TS, TA, Z) return launch_decode_t<MODE, TS, TA, Z>(p, st, pdl)
  if (abf) {
    if (sbf) { if (has_zp) QMOE_DEC(__nv_bfloat16, __nv_bfloat16, true); QMOE_DEC(__nv_bfloat16, __nv_bfloat16, false); }
    if (has_zp) QMOE_DEC(__half, __nv_bfloat16, true);
    QMOE_DEC(__half, __nv_bfloat16, false);
  }
  if (sbf) { if (has_zp) QMOE_DEC(__nv_bfloat16, __half, true); QMOE_DEC(__nv_bfloat16, __half, false); }
  if (has_zp) QMOE_DEC(__half, __half, true);
  QMOE_DEC(__half, __half, false);
#undef QMOE_DEC
}

cudaError_t launch_decode(DecodeParams p, int mode, int act_dtype, int scale_dtype, bool has_zp,
                          cudaStream_t st, bool pdl) {
  if (mode == kModeGateUp) return dispatch_decode<kModeGateUp>(p, act_dtype, scale_dtype, has_zp, st, pdl);
  if (mode == kModeDown) return dispatch_decode<kModeDown>(p, act_dtype, scale_dtype, has_zp, st, pdl);
  return dispatch_decode<kModeDense>(p, act_dtype, scale_dtype, has_zp, st, pdl);
}

}  // namespace qmoe
