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
// 4-byte words.  Here one CTA per SM streams an equal share of the selected
// experts' bytes:
//  * gate-up and the dense GEMV split the flattened (expert, row) space into
//    equal contiguous ranges, so a CTA's rows are one or two large
//    contiguous slices ("stages") of the [E, N, K/2] tensors;
//  * down gives each CTA a fixed slice of output rows across every selected
//    expert, so the weighted sum over the k experts stays inside the CTA
//    (deterministic, no atomics).
// A producer warp issues cp.async.bulk copies of each stage's rows, block
// scales and zero points into a ring of shared-memory slots guarded by
// mbarriers, the copies of a whole ring-full at once across its lanes.
// Consumer warps take (stage, 4-row group) work items, so different warps
// work on different stages concurrently.  A lane owns two adjacent 16-byte
// chunks (64 codes) of a row; nibble j of each 16-bit half-word becomes the
// exact float (q - zp) * 16^j with one three-input LOP3 (nibble OR-ed into
// the mantissa of 2^23) and half a packed subtract, and is multiplied with
// activations pre-scaled by 16^-j in packed fp32 FMAs (fma.rn.f32x2); all
// accumulation is fp32.  Work is grouped per distinct expert, so every
// weight byte is read once per call even when several tokens chose the
// same expert.
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

// Shared-memory plan of the fused layer: the two phases' rings (gate-up,
// down) side by side, the router's scratch laid over them.
struct FusedPlan {
  DecodePlan g, d;           // slot_rows, max_stages, nslots per phase
  uint32_t res_off;          // x in decode layout (gate-up), then the down partials
  uint32_t stg_off, std_off;  // stage tables
  uint32_t ring_g, ring_d, smem;
  uint32_t slot_g, slot_d;   // slot strides
  int pass_rows;             // router rows staged per pass
  uint32_t xs_off, part_off, vpart_off, wch_off;
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

template <int MODE, typename TS, typename TA, bool HAS_ZP>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(DecodeParams p, DecodePlan P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxSlots;
  uint64_t* route_bar = empty + kMaxSlots;
  int* s_nst = reinterpret_cast<int*>(route_bar + 1);
  int* s_active = reinterpret_cast<int*>(smem + kOffActive);  // [0]=D, [1..D]
  int* s_off = reinterpret_cast<int*>(smem + kOffOff);        // [E+1]
  int* s_perm = reinterpret_cast<int*>(smem + kOffPerm);      // [T*k]
  float* s_wt = reinterpret_cast<float*>(smem + kOffWt);      // [T*k] routing weights (down)
  float* res = reinterpret_cast<float*>(smem + P.res_off);    // x rows (gate-up / dense) or partials (down)
  StageEnt* s_stage = reinterpret_cast<StageEnt*>(smem + P.stage_off);
  uint8_t* slots = smem + P.slot_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = p.ctl ? p.ctl + kCtlStatus : nullptr;
  const int NS = P.nslots;
  const SlotLayout SL = slot_layout(MODE, P.slot_rows, p.K, p.nb, HAS_ZP, p.src_row_floats, p.T);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 32);
      mbar_init(&empty[i], kCW);
    }
    mbar_init(route_bar, 32);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ================================================================ producer
    // 1. routing -> shared memory (one round trip), then the stage table
    if (MODE == kModeGateUp) pdl_wait();
    if (MODE != kModeDense) {
      const int A = p.T * p.k;
      for (int i = lane; i <= p.E; i += 32) s_off[i] = __ldcg(p.offsets + i);
      for (int i = lane; i <= p.E; i += 32) s_active[i] = __ldcg(p.active + i);
      for (int i = lane; i < A; i += 32) s_perm[i] = __ldcg(p.perm + i);
      if (MODE == kModeDown)
        for (int i = lane; i < A; i += 32) s_wt[i] = __ldcg(p.topk_w + i);
      __syncwarp();
    }
    const int nst = build_stages<MODE>(p, P, s_active, s_off, s_stage, blockIdx.x, gridDim.x, lane);
    if (lane == 0) *s_nst = nst;
    __syncwarp();
    mbar_arrive(route_bar);  // release: routing and stage table
    if (MODE == kModeGateUp) pdl_trigger();

    // 2. first ring-full: every copy in flight at once.  For down, the
    //    activation rows come from the previous grid (gate-up): the weights
    //    go out before waiting for it.
    const int n0 = min(NS, nst);
    issue_copies<MODE, HAS_ZP>(p, SL, SL.bytes, s_stage, s_perm, slots, full, NS, 0, n0, true, MODE != kModeDown, lane);
    if (MODE == kModeDown) {
      pdl_wait();
      issue_copies<MODE, HAS_ZP>(p, SL, SL.bytes, s_stage, s_perm, slots, full, NS, 0, n0, false, true, lane);
    }
    arrive_range(full, NS, 0, n0);
    // 3. refill slots as consumers release them
    bool ok = true;
    for (int s = n0; s < nst; ++s) {
      ok = mbar_wait(&empty[s % NS], ((s / NS) - 1) & 1, status);
      if (!ok) break;
      issue_copies<MODE, HAS_ZP>(p, SL, SL.bytes, s_stage, s_perm, slots, full, NS, s, s + 1, true, true, lane);
      arrive_range(full, NS, s, s + 1);
    }
    // drain: do not exit while bulk copies into this CTA's smem are in flight
    if (ok)
      for (int s = max(0, nst - NS); s < nst; ++s)
        if (!mbar_wait(&full[s % NS], (s / NS) & 1, status)) break;
    return;
  }

  // ================================================================ consumers
  // gate-up / dense: activations resident for the whole kernel (the layer
  // input is complete before this grid starts: the router, the previous
  // grid, starts dependents only after its own wait)
  if (MODE != kModeDown) load_x_dec<TA>(p.x16, p.T, p.K, res, tid, kCW * 32);
  asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
  if (!mbar_wait(route_bar, 0, status)) return;
  const int nst = *s_nst;
  const bool ok = consume_stages<MODE, TS, TA, HAS_ZP>(p, SL, SL.bytes, s_stage, nst, s_perm, res, res, slots, full,
                                                       empty, NS, warp, lane, status);
  if (MODE == kModeDown) {
    asm volatile("bar.sync 1, %0;" ::"r"(kCW * 32) : "memory");
    if (!ok) return;
    const int r0 = (int)(((long long)blockIdx.x * p.N) / gridDim.x);
    const int r1 = (int)(((long long)(blockIdx.x + 1) * p.N) / gridDim.x);
    down_combine<TA>(p, s_stage, nst, s_perm, s_wt, res, r0, r1, tid, kCW * 32);
  }
}

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

// ------------------------------------------------------------------- host

static bool plan_decode(int mode, int T, int N, int K, int bs, bool has_zp, int k, int E, int sms,
                        DecodePlan* out) {
  DecodePlan P = {};
  const int nb = K / bs;
  const int act_row = dec_row_floats(K);
  const int A = T * k;
  const int dmax = (mode == kModeDense) ? 1 : (A < E ? A : E);
  // a CTA of the previous grid (gate-up) may still occupy the SM while
  // down streams its first weights: at small T keep both under one SM
  const uint32_t cap = (T <= kTokGroup) ? (mode == kModeDown ? 100u << 10 : 124u << 10) : kSmemBudget;
  if (mode == kModeDown) {
    P.grid = N < sms ? N : sms;
    P.rows_cta = (N + P.grid - 1) / P.grid;
    P.slot_rows = P.rows_cta;
    P.max_stages = dmax + (A - dmax + kTokGroup - 1) / kTokGroup;
  } else {
    P.grid = sms;
    const long long F = (long long)dmax * N;
    P.rows_cta = (int)((F + P.grid - 1) / P.grid);
    if (P.rows_cta < 1) P.rows_cta = 1;
  }
  P.res_off = kFixedSmem;
  uint32_t res = 0;
  if (mode == kModeDown) res = (uint32_t)P.max_stages * kTokGroup * P.rows_cta * 4;
  else res = (uint32_t)T * act_row * 4;
  if (mode != kModeDown) {
    // rows per slot: the CTA's range in as few stages as fit three slots
    const uint32_t per_row = slot_layout(mode, 1, K, nb, has_zp, act_row, T).bytes;
    const uint32_t fixed = kFixedSmem + al16(res) + 48 * 64 + 1024;
    if (fixed + 2 * per_row > cap) return false;
    int rcap = (int)((cap - fixed) / 3 / (per_row + 16));
    if (rcap > 64) rcap = 64;
    if (rcap < 1) rcap = 1;
    const int nst_min = (P.rows_cta + rcap - 1) / rcap;
    P.slot_rows = (P.rows_cta + nst_min - 1) / nst_min;
    if (P.slot_rows > N) P.slot_rows = N;
    // expert boundaries inside a CTA's range add at most one stage each
    P.max_stages = nst_min + (P.rows_cta + N - 1) / N + 1;
    if (mode == kModeDense) P.max_stages = nst_min + 1;
  }
  const SlotLayout SL = slot_layout(mode, P.slot_rows, K, nb, has_zp, act_row, T);
  P.stage_off = P.res_off + al16(res);
  P.slot_base = (P.stage_off + 48u * P.max_stages + 1023u) & ~1023u;
  if (P.slot_base + 2 * SL.bytes > kSmemBudget) return false;
  uint32_t avail = (cap > P.slot_base + 2 * SL.bytes ? cap : P.slot_base + 2 * SL.bytes) - P.slot_base;
  int ns = (int)(avail / SL.bytes);
  if (ns > P.max_stages) ns = P.max_stages;
  if (ns > kMaxSlots) ns = kMaxSlots;
  if (ns < 2) ns = 2;
  P.nslots = ns;
  P.smem = P.slot_base + ns * SL.bytes;
  if (P.smem > kSmemBudget) return false;
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
  auto fn = decode_kernel<MODE, TS, TA, HAS_ZP>;
  cudaError_t err = ensure_smem(fn, P.smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(fn, dim3(P.grid), dim3(kDecodeThreads), (size_t)P.smem, st, pdl, p, P);
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
  int best_rows = 0, best_ns = 0, best_nd = 0;
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
          best_nd = nd;
        }
        break;  // the largest slot that fits for this (nd, ns)
      }
    }
  (void)best_nd;
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

cudaError_t launch_fused(const FusedParams& f, int act_dtype, int scale_dtype, bool has_zp, cudaStream_t st,
                         bool pdl, bool check_only) {
  const bool abf = act_dtype == 1, sbf = scale_dtype == 1;
#define QMOE_FU(TS, TA) return has_zp ? launch_fused_me<TS, TA, true>(f, st, pdl, check_only) \
                                      : launch_fused_me<TS, TA, false>(f, st, pdl, check_only)
  if (abf) {
    if (sbf) QMOE_FU(__nv_bfloat16, __nv_bfloat16);
    QMOE_FU(__half, __nv_bfloat16);
  }
  if (sbf) QMOE_FU(__nv_bfloat16, __half);
  QMOE_FU(__half, __half);
#undef QMOE_FU
}

}  // namespace qmoe
