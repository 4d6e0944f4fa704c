// decode_core.cuh -- device building blocks shared by the decode kernels
// (decode.cu) and the one-kernel decode layer (decode_fused.cu): the
// shared-memory slot layout, the in-register dequantisation and dot
// products, the bulk-copy producer, the stage tables and the consumers.
// Everything here is a template or an inline function.
#pragma once
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace qmoe {

constexpr int kCW = 11;                         // consumer warps
constexpr int kDecodeThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kMaxSlots = 8;
// rows per work item for NT tokens and NMAT matrices (register budget:
// at most 4 rows x tokens x matrices partial sums, x chunks in registers)
__host__ __device__ constexpr int rows_per_item(int nt, int nmat) {
  return nmat == 2 ? (nt == 1 ? 2 : 1) : (nt == 1 ? 4 : (nt == 2 ? 2 : 1));
}
constexpr int kJobsPerStage = 10;               // W,S,Z of two matrices + 4 activation rows
constexpr uint32_t kSmemBudget = 232448;        // 227 KB dynamic shared memory

// One stage: rows [row0, row0 + nrows) of expert e's matrices and the
// tokens (assignments perm[pbase .. pbase + ntok)) they serve.
struct StageEnt {
  int e, pbase, ntok, row0, nrows;
  int ph[4];  // alignment phase of the scales0, scales1, zp0, zp1 images
  int pad[3];
};
static_assert(sizeof(StageEnt) == 48, "stage entry is 48 bytes");

// fixed shared-memory carve (bytes); the stage table follows at kFixedSmem
constexpr uint32_t kOffActive = 256;
constexpr uint32_t kOffOff = kOffActive + 4 * (kMaxExperts + 2);
constexpr uint32_t kOffPerm = kOffOff + 4 * (kMaxExperts + 2);
constexpr uint32_t kOffWt = kOffPerm + 4 * kDecodeMaxTokens * kMaxTopk;
constexpr uint32_t kFixedSmem = (kOffWt + 4 * kDecodeMaxTokens * kMaxTopk + 127) & ~127u;

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

// Shared-memory plan of one launch (host and device agree on it).
struct DecodePlan {
  int grid;        // CTAs
  int rows_cta;    // gate-up / dense: rows of the flattened space per CTA (max); down: slice rows (max)
  int slot_rows;   // rows per stage slot
  int max_stages;  // stage-table entries per CTA
  int nslots;
  uint32_t res_off, stage_off, slot_base, smem;
};

// ---------------------------------------------------------------- dequant
// A register the compiler cannot fold back into an immediate, so that
// (v & MASK) | magic is a single three-input LOP3.
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
  asm volatile("mov.b32 %0, %1;" : "=r"(v) : "r"(v));
  return v;
}
template <uint32_t MASK>
__device__ __forceinline__ float or_masked(uint32_t v, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(MASK), "r"(magic));  // (v & m) | c
  return __uint_as_float(d);
}

// -(2^23 + zp * 16^j) for nibble positions j = 0..3 of a half-word.
struct ZConst {
  f2 c01, c23;
};
__device__ __forceinline__ ZConst zconst(uint32_t zp, uint32_t neg_magic) {
  const uint32_t z = zp * 0x1111u;
  return ZConst{make_float2(or_masked<0xFu>(z, neg_magic), or_masked<0xF0u>(z, neg_magic)),
                make_float2(or_masked<0xF00u>(z, neg_magic), or_masked<0xF000u>(z, neg_magic))};
}

// Dequantise one 16-byte chunk (32 codes) into 16 float pairs holding
// (q - zp) * 16^j, j = position of the nibble in its 16-bit half-word:
// 2^23 + q * 16^j is the nibble OR-ed into the mantissa of 2^23 (one LOP3),
// and 2^23 + zp * 16^j is subtracted by a packed add.  Every value is an
// exact integer times a power of two.
__device__ __forceinline__ void dequant_chunk(const uint4 q, const ZConst zc, uint32_t magic,
                                              f2 (&wv)[16]) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = qw[i], hi = qw[i] >> 16;
    wv[4 * i + 0] = fadd2(make_float2(or_masked<0xFu>(lo, magic), or_masked<0xF0u>(lo, magic)), zc.c01);
    wv[4 * i + 1] = fadd2(make_float2(or_masked<0xF00u>(lo, magic), or_masked<0xF000u>(lo, magic)), zc.c23);
    wv[4 * i + 2] = fadd2(make_float2(or_masked<0xFu>(hi, magic), or_masked<0xF0u>(hi, magic)), zc.c01);
    wv[4 * i + 3] = fadd2(make_float2(or_masked<0xF00u>(hi, magic), or_masked<0xF000u>(hi, magic)), zc.c23);
  }
}

// 32 activations of one chunk (decode layout: 8 float4 strided by 32).
struct XChunk {
  float4 v[8];
};
__device__ __forceinline__ void load_x(const float4* xr, XChunk& x) {
#pragma unroll
  for (int f = 0; f < 8; ++f) x.v[f] = xr[f * 32];
}
// fp32 dot of a dequantised chunk with its activations (4 packed chains).
__device__ __forceinline__ float chunk_dot(const f2 (&wv)[16], const XChunk& x) {
  f2 d0 = make_float2(0.f, 0.f), d1 = d0, d2 = d0, d3 = d0;
#pragma unroll
  for (int f = 0; f < 8; f += 2) {
    d0 = ffma2(wv[2 * f], make_float2(x.v[f].x, x.v[f].y), d0);
    d1 = ffma2(wv[2 * f + 1], make_float2(x.v[f].z, x.v[f].w), d1);
    d2 = ffma2(wv[2 * f + 2], make_float2(x.v[f + 1].x, x.v[f + 1].y), d2);
    d3 = ffma2(wv[2 * f + 3], make_float2(x.v[f + 1].z, x.v[f + 1].w), d3);
  }
  const f2 d = fadd2(fadd2(d0, d1), fadd2(d2, d3));
  return d.x + d.y;
}

// Dense `Rows` x NT dot products of one work item: rows [rb, rb + nr) of the
// stage's matrices (NMAT = 2: gate and up) against NT activation rows.
// acc[m][r][j] gets lane-partial sums (fp32) to be reduced across the warp.
// A lane owns chunks c = 64 s + 2 lane + u (u = 0, 1) and sums them in
// ascending c.  Per step s every code, scale and zero point of the item is
// loaded before any arithmetic (a fully unrolled body with the loads in
// flight together; a loop over single chunks left each load's latency
// exposed), then dequantised and dotted.
template <int NMAT, int NT, int RG, typename TS, bool HAS_ZP>
__device__ __forceinline__ void item_dot(const uint8_t* slot, const SlotLayout& SL, const StageEnt& st,
                                         int rb, int nr, const float4* const (&xr)[kTokGroup],
                                         int K, int nb, int bshift, uint32_t magic, uint32_t neg_magic,
                                         const ZConst zfixed, int lane, float (&acc)[NMAT][RG][NT]) {
  const int nchunks = K / 32;
  const int row_bytes = K / 2;
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RG; ++r)
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[m][r][j] = 0.f;
  const uint8_t* wbase[NMAT];
  const uint16_t* sbase[NMAT];
  const uint8_t* zbase[NMAT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m) {
    wbase[m] = slot + SL.w[m] + (size_t)rb * row_bytes;
    sbase[m] = reinterpret_cast<const uint16_t*>(slot + SL.s[m] + st.ph[m]) + (size_t)rb * nb;
    zbase[m] = slot + SL.z[m] + st.ph[2 + m] + (size_t)rb * nb;
  }
  // Rows past the item's end (a ragged last item) load the last valid row
  // again and their sums are discarded by the caller; a missing second chunk
  // (odd chunk count) reloads the first with a zero scale, adding exactly
  // zero.  No load is predicated, so they all issue back to back.
  int roff[RG];
#pragma unroll
  for (int r = 0; r < RG; ++r) roff[r] = min(r, nr - 1);
  for (int c0 = 2 * lane; c0 < nchunks; c0 += 64) {
    const bool has1 = c0 + 1 < nchunks;
    uint4 q[2][RG][NMAT];
    float sc[2][RG][NMAT];
    uint32_t zz[2][RG][NMAT];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int r = 0; r < RG; ++r)
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const int c = (u == 1 && has1) ? c0 + 1 : c0;
          const int blk = c >> bshift;
          const size_t ro = (size_t)roff[r];
          q[u][r][m] = *reinterpret_cast<const uint4*>(wbase[m] + ro * row_bytes + c * 16);
          const float sv = Half<TS>::to_float(sbase[m][ro * nb + blk]);
          sc[u][r][m] = (u == 0 || has1) ? sv : 0.f;
          zz[u][r][m] = HAS_ZP ? (uint32_t)zbase[m][ro * nb + blk] : 8u;
        }
    const int xo0 = (c0 >> 6) * 512 + lane;  // float4 index of (s, u = 0, f = 0)
    if (NT == 1) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        XChunk xa;
        load_x(xr[0] + xo0 + (has1 ? u * 256 : 0), xa);
#pragma unroll
        for (int r = 0; r < RG; ++r)
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            f2 wv[16];
            dequant_chunk(q[u][r][m], HAS_ZP ? zconst(zz[u][r][m], neg_magic) : zfixed, magic, wv);
            acc[m][r][0] = fmaf(sc[u][r][m], chunk_dot(wv, xa), acc[m][r][0]);
          }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < RG; ++r)
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            f2 wv[16];
            dequant_chunk(q[u][r][m], HAS_ZP ? zconst(zz[u][r][m], neg_magic) : zfixed, magic, wv);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              XChunk xj;
              load_x(xr[j] + xo0 + (has1 ? u * 256 : 0), xj);
              acc[m][r][j] = fmaf(sc[u][r][m], chunk_dot(wv, xj), acc[m][r][j]);
            }
          }
    }
  }
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RG; ++r)
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[m][r][j] = warp_sum(acc[m][r][j]);
}

// ---------------------------------------------------------------- producer
// Copy `bytes` global bytes into shared memory at dst_base + (src mod 16):
// the 16-byte-aligned middle by bulk copy (expected bytes registered on `bar`
// first), the ragged head / tail (< 16 bytes each) by plain loads.  One
// lane does all of it; returns src mod 16.
__device__ __forceinline__ int copy_ragged(uint8_t* dst_base, const uint8_t* src, uint32_t bytes,
                                           uint64_t* bar) {
  const uint32_t ph = (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u);
  const uint32_t head = min(bytes, (16u - ph) & 15u);
  const uint32_t body = (bytes - head) & ~15u;
  const uint32_t tail = bytes - head - body;
  uint8_t* dst = dst_base + ph;
  if (body) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(body) : "memory");
    bulk_g2s(dst + head, src + head, body, bar);
  }
  for (uint32_t i = 0; i < head; ++i) dst[i] = __ldg(src + i);
  for (uint32_t i = 0; i < tail; ++i) dst[head + body + i] = __ldg(src + head + body + i);
  return (int)ph;
}

__device__ __forceinline__ void copy_bulk(uint8_t* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
  bulk_g2s(dst, src, bytes, bar);
}

template <int MODE, int NT, typename TS, typename TA, bool HAS_ZP>
__device__ __forceinline__ void run_item(const DecodeParams& p, const uint8_t* slot, const SlotLayout& SL,
                                         const StageEnt& st, int s, int g, int tg, const int* s_perm,
                                         const float* res, float* partial, int kdec, int bshift,
                                         uint32_t magic, uint32_t neg_magic, const ZConst zfixed,
                                         int lane) {
  constexpr int NMAT = (MODE == kModeGateUp) ? 2 : 1;
  constexpr int RG = rows_per_item(NT, NMAT);
  const int rb = g * RG;
  const int nr = min(RG, st.nrows - rb);
  const int j0 = tg * kTokGroup;
  // activation rows of the item's tokens
  const float4* xr[kTokGroup];
#pragma unroll
  for (int j = 0; j < kTokGroup; ++j) {
    const int jj = j < NT ? j : 0;
    if (MODE == kModeDown) {
      xr[j] = reinterpret_cast<const float4*>(slot + SL.act) + (size_t)(j0 + jj) * (p.src_row_floats / 4);
    } else {
      const int a = (MODE == kModeDense) ? (st.pbase + j0 + jj) : s_perm[st.pbase + j0 + jj];
      const int t = (MODE == kModeDense) ? a : a / p.k;
      xr[j] = reinterpret_cast<const float4*>(res) + (size_t)t * (kdec / 4);
    }
  }
  float acc[NMAT][RG][NT];
  item_dot<NMAT, NT, RG, TS, HAS_ZP>(slot, SL, st, rb, nr, xr, p.K, p.nb, bshift, magic, neg_magic,
                                     zfixed, lane, acc);
  // epilogue: one output per lane (lane = r * NT + j)
  const int r = lane / NT, j = lane - r * NT;
  if (r < nr && r < RG) {
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int rr = 0; rr < RG; ++rr)
#pragma unroll
      for (int jj = 0; jj < NT; ++jj)
        if (rr == r && jj == j) {
          v0 = acc[0][rr][jj];
          v1 = acc[NMAT - 1][rr][jj];
        }
    if (MODE == kModeGateUp) {
      const int a = s_perm[st.pbase + j0 + j];
      const int i = st.row0 + rb + r;
      const float act = v0 / (1.f + expf(-v0)) * v1;
      p.act_out[(size_t)a * p.act_row_floats + dec_index(i)] = act * dec_prescale(i);
    } else if (MODE == kModeDense) {
      const int t = st.pbase + j0 + j;
      static_cast<uint16_t*>(p.out)[(size_t)t * p.N + st.row0 + rb + r] = Half<TA>::from_float(v0);
    } else {
      partial[((size_t)s * kTokGroup + j) * st.nrows + rb + r] = v0;
    }
  }
}

// ---------------------------------------------------- kernel building blocks

// Stage table of one CTA (producer warp, all lanes): gate-up / dense take
// an equal contiguous range of the flattened (expert, row) space, cut at
// expert boundaries and at slot_rows; down takes output rows [r0, r1) of
// every selected expert, one stage per (expert, up to kTokGroup of its
// assignments).  Returns the number of stages (<= P.max_stages).
template <int MODE>
__device__ int build_stages(const DecodeParams& p, const DecodePlan& P, const int* s_active, const int* s_off,
                            StageEnt* s_stage, int cta, int ncta, int lane) {
  const int N = p.N;
  int nst = 0;
  if (MODE == kModeDown) {
    const int r0 = (int)(((long long)cta * N) / ncta);
    const int r1 = (int)(((long long)(cta + 1) * N) / ncta);
    const int D = r1 > r0 ? s_active[0] : 0;
    for (int d0 = 0; d0 < D; d0 += 32) {
      const int d = d0 + lane;
      int e = 0, n = 0, g = 0;
      if (d < D) {
        e = s_active[1 + d];
        n = s_off[e + 1] - s_off[e];
        g = (n + kTokGroup - 1) / kTokGroup;
      }
      int incl = g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int base = nst + incl - g;
      for (int gi = 0; gi < g && base + gi < P.max_stages; ++gi) {
        StageEnt& se = s_stage[base + gi];
        se.e = e;
        se.pbase = s_off[e] + gi * kTokGroup;
        se.ntok = min(kTokGroup, n - gi * kTokGroup);
        se.row0 = r0;
        se.nrows = r1 - r0;
      }
      nst += __shfl_sync(0xffffffffu, incl, 31);
    }
  } else if (lane == 0) {
    const int D = (MODE == kModeDense) ? 1 : s_active[0];
    const long long F = (long long)D * N;
    const long long f0 = (long long)cta * F / ncta, f1 = (long long)(cta + 1) * F / ncta;
    for (long long f = f0; f < f1 && nst < P.max_stages;) {
      const int d = (int)(f / N), i0 = (int)(f - (long long)d * N);
      const int n = (int)min((long long)min(N - i0, P.slot_rows), f1 - f);
      StageEnt& se = s_stage[nst++];
      se.e = (MODE == kModeDense) ? 0 : s_active[1 + d];
      se.pbase = (MODE == kModeDense) ? 0 : s_off[se.e];
      se.ntok = (MODE == kModeDense) ? p.T : s_off[se.e + 1] - s_off[se.e];
      se.row0 = i0;
      se.nrows = n;
      f += n;
    }
  }
  nst = __shfl_sync(0xffffffffu, nst, 0);
  return min(nst, P.max_stages);
}

// Copies of stages [sa, sb) into their ring slots (producer warp, jobs =
// (stage, kind) spread over the lanes): weights, scales and zero points if
// `weights`, the activation rows of down stages if `acts`.
template <int MODE, bool HAS_ZP>
__device__ void issue_copies(const DecodeParams& p, const SlotLayout& SL, uint32_t slot_bytes, StageEnt* s_stage,
                             const int* s_perm, uint8_t* slots, uint64_t* full, int NS, int sa, int sb,
                             bool weights, bool acts, int lane) {
  const int N = p.N, K = p.K, nb = p.nb;
  constexpr int nmat = (MODE == kModeGateUp) ? 2 : 1;
  const int total = (sb - sa) * kJobsPerStage;
  for (int jid = lane; jid < total; jid += 32) {
    const int s = sa + jid / kJobsPerStage, job = jid % kJobsPerStage;
    const int slot = s % NS;
    StageEnt& st = s_stage[s];
    uint8_t* sb_ = slots + slot * slot_bytes;
    uint64_t* bar = &full[slot];
    const size_t row0 = (size_t)st.e * N + st.row0;
    if (job < 6) {
      const int m = job / 3, kind = job % 3;
      if (!weights || m >= nmat || (kind == 2 && !HAS_ZP)) continue;
      // (select, not index: a runtime index would put the layout in local memory)
      const uint32_t ow = m ? SL.w[1] : SL.w[0], os = m ? SL.s[1] : SL.s[0], oz = m ? SL.z[1] : SL.z[0];
      if (kind == 0) {
        copy_bulk(sb_ + ow, (m ? p.w[1] : p.w[0]) + row0 * (K / 2), (uint32_t)st.nrows * (K / 2), bar);
      } else if (kind == 1) {
        st.ph[m] = copy_ragged(sb_ + os, static_cast<const uint8_t*>(m ? p.s[1] : p.s[0]) + row0 * nb * 2,
                               (uint32_t)st.nrows * nb * 2, bar);
      } else {
        st.ph[2 + m] = copy_ragged(sb_ + oz, (m ? p.z[1] : p.z[0]) + row0 * nb, (uint32_t)st.nrows * nb, bar);
      }
    } else if (MODE == kModeDown && acts) {
      const int j = job - 6;
      if (j >= st.ntok) continue;
      const int a = s_perm[st.pbase + j];
      copy_bulk(sb_ + SL.act + (uint32_t)j * p.src_row_floats * 4, p.src + (size_t)a * p.src_row_floats,
                p.src_row_floats * 4u, bar);
    }
  }
}

__device__ __forceinline__ void arrive_range(uint64_t* full, int NS, int sa, int sb) {
  __syncwarp();
  for (int s = sa; s < sb; ++s) mbar_arrive(&full[s % NS]);
}

// Consumer warps: every stage of the ring in order; the work items of a
// stage (token group x row group) are dealt round-robin over the warps,
// continuing the rotation across stages.  Returns false on a timeout.
template <int MODE, typename TS, typename TA, bool HAS_ZP>
__device__ bool consume_stages(const DecodeParams& p, const SlotLayout& SL, uint32_t slot_bytes,
                               const StageEnt* s_stage, int nst, const int* s_perm, const float* res, float* partial,
                               const uint8_t* slots, uint64_t* full, uint64_t* empty, int NS, int warp, int lane,
                               uint32_t* status) {
  const int kdec = dec_row_floats(p.K);
  const uint32_t magic = opaque(0x4B000000u);      // 2^23
  const uint32_t neg_magic = opaque(0xCB000000u);  // -2^23
  const ZConst zfixed = zconst(8u, neg_magic);     // no zero-point tensor: zp = 8
  const int bshift = (p.bs == 32) ? 0 : (p.bs == 64 ? 1 : 2);
  constexpr int NMAT = (MODE == kModeGateUp) ? 2 : 1;
  int item_base = 0;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % NS;
    // every warp waits for every stage in order (a waiter must never be two
    // phases ahead of an mbarrier)
    if (!mbar_wait(&full[slot], (s / NS) & 1, status)) return false;
    const StageEnt st = s_stage[s];
    const uint8_t* sb = slots + slot * slot_bytes;
    const int ntg = (st.ntok + kTokGroup - 1) / kTokGroup;
    int nitems = 0;
    for (int tg = 0; tg < ntg; ++tg) {
      const int rg = rows_per_item(min(kTokGroup, st.ntok - tg * kTokGroup), NMAT);
      nitems += (st.nrows + rg - 1) / rg;
    }
    for (int i = ((warp - item_base) % kCW + kCW) % kCW; i < nitems; i += kCW) {
      int tg = 0, g = i, nt = 0;
      for (;; ++tg) {
        nt = min(kTokGroup, st.ntok - tg * kTokGroup);
        const int ngr = (st.nrows + rows_per_item(nt, NMAT) - 1) / rows_per_item(nt, NMAT);
        if (g < ngr) break;
        g -= ngr;
      }
      switch (nt) {
        case 1: run_item<MODE, 1, TS, TA, HAS_ZP>(p, sb, SL, st, s, g, tg, s_perm, res, partial, kdec, bshift, magic, neg_magic, zfixed, lane); break;
        case 2: run_item<MODE, 2, TS, TA, HAS_ZP>(p, sb, SL, st, s, g, tg, s_perm, res, partial, kdec, bshift, magic, neg_magic, zfixed, lane); break;
        case 3: run_item<MODE, 3, TS, TA, HAS_ZP>(p, sb, SL, st, s, g, tg, s_perm, res, partial, kdec, bshift, magic, neg_magic, zfixed, lane); break;
        default: run_item<MODE, 4, TS, TA, HAS_ZP>(p, sb, SL, st, s, g, tg, s_perm, res, partial, kdec, bshift, magic, neg_magic, zfixed, lane); break;
      }
    }
    item_base += nitems;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  return true;
}

// Down: weighted sum over the selected experts of the CTA's output rows
// [r0, r1), in stage order (deterministic), plus the residual if asked.
template <typename TA>
__device__ void down_combine(const DecodeParams& p, const StageEnt* s_stage, int nst, const int* s_perm,
                             const float* s_wt, const float* partial, int r0, int r1, int tid, int nthreads) {
  const int nrows = r1 - r0;
  uint16_t* out = static_cast<uint16_t*>(p.out);
  for (int idx = tid; idx < p.T * nrows; idx += nthreads) {
    const int t = idx / nrows, r = idx - t * nrows;
    float v = 0.f;
    for (int s = 0; s < nst; ++s) {
      const StageEnt& st = s_stage[s];
      for (int j = 0; j < st.ntok; ++j) {
        const int a = s_perm[st.pbase + j];
        if (a / p.k == t) v = fmaf(s_wt[a], partial[((size_t)s * kTokGroup + j) * nrows + r], v);
      }
    }
    const size_t o = (size_t)t * p.N + r0 + r;
    if (p.accumulate) v += Half<TA>::to_float(out[o]);
    out[o] = Half<TA>::from_float(v);
  }
}

// x [T, K] 16-bit -> fp32 rows in decode layout, pre-scaled (gate-up / dense).
template <typename TA>
__device__ void load_x_dec(const void* x16, int T, int K, float* res, int tid, int nthreads) {
  const int kdec = dec_row_floats(K);
  const uint4* x8 = static_cast<const uint4*>(x16);
  const int n8 = T * K / 8;
  constexpr int kPer = 4;
  for (int i0 = tid; i0 < n8; i0 += nthreads * kPer) {
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + u * nthreads;
      if (i < n8) v[u] = __ldg(x8 + i);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + u * nthreads;
      if (i < n8) {
        const int t = (i * 8) / K, k0 = i * 8 - t * K;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int kk = k0 + e;
          const uint16_t b = (uint16_t)(w[e >> 1] >> ((e & 1) * 16));
          res[t * kdec + dec_index(kk)] = Half<TA>::to_float(b) * dec_prescale(kk);
        }
      }
    }
  }
}

}  // namespace qmoe
