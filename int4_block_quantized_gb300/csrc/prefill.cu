// prefill.cu -- large-T path of the layer: tokens grouped by expert, then a
// grouped expert GEMM on the 5th-generation tensor cores (tcgen05) with the
// int4 weights dequantised on chip, SwiGLU fused into the gate-up epilogue
// and the routing-weighted scatter-add fused into the down epilogue.
//
// Sources: "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34), IR guide
// "Optimization Opportunities" item 9 (sort tokens by expert, one grouped
// GEMM over all experts using the grouping as a gather index, weighted
// un-permute) and item 6 (DequantizeLinear fused into the MatMul);
// DequantizeLinear with block_size from local fix A1; SwiGLU and the
// weighted sum from IR guide 3, Expert Computation steps 5-7.
//
// GB300 design.  Swap-AB: the weight rows are the MMA's M = 128 operand and
// an expert's tokens (up to 160 per tile) its N, so small experts still fill
// the tensor core's M dimension.  A gate-up tile stacks 64 gate rows over
// the same 64 up rows, so gate and up land in one TMEM accumulator and the
// SwiGLU pairs them in the epilogue.  Per CTA (one per SM, persistent):
//   a weight producer streams packed int4 tiles (TMA) and each tile's block
//           scales / zero points (bulk copies) through a deep ring;
//   a token producer streams token tiles (TMA, 128-byte swizzle);
//   eight dequantiser warps turn the codes into exact operands in
//           registers and store them into tensor memory (tcgen05.st): the
//           MMA reads the weight operand from TMEM, so shared memory only
//           carries the codes and the token tiles;
//   one thread issues tcgen05.mma (A from TMEM, B from shared memory) into
//           a double-buffered TMEM accumulator;
//   four epilogue warps tcgen05.ld it and apply SwiGLU or the weighted
//           fp32 scatter-add.
// Operands are exact (the rule is stated at gemm_ops below): a dequantised
// weight enters as one fp16 operand or as hi = RN(w) plus lo = w - hi; the
// SwiGLU output enters the down GEMM as hi + lo.  K is permuted inside every
// group of 8 (order 0,4,1,5,2,6,3,7) identically for weights and
// activations so one LOP3 yields two operands from a 32-bit word.
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "tmap.h"
#include "launch.h"

namespace qmoe {

constexpr int kGemmThreads = 512;  // 16 warps (roles listed at the kernel)
constexpr int kBN = 160;           // max tokens per tile (TMEM columns per accumulator)
// Token tiles of an expert with n assignments: one tile when n <= kBN (its
// weights dequantised once, wide MMAs), else ceil(n / 128) tiles of
// balanced size: splitting a large expert finer keeps the per-CTA work of
// the persistent schedule even.
__host__ __device__ inline int token_tiles(int n) { return n <= kBN ? (n > 0 ? 1 : 0) : (n + 127) / 128; }
constexpr int kBoxRows = 32;       // token rows per B TMA box
constexpr int kModeGU = 0, kModeDN = 1;

// position of element j (0..7) of a group of 8 in the permuted K order
__host__ __device__ __forceinline__ int kperm_pos(int j) { return (j & 3) * 2 + (j >> 2); }


// Eight bf16 values to fp16 (exact inside fp16's range; a value beyond it
// sets QMOE_ST_RANGE).
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 v, uint32_t* status) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool big = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
    big |= !(fabsf(a) <= 65504.f) || !(fabsf(b) <= 65504.f);
    w[i] = (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
  }
  if (big) set_status(status, QMOE_ST_RANGE);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- permute
// xp[r] = x[token of sorted assignment r] with K permuted inside each group
// of 8; out_acc = 0; block 0 also writes the token tile table: an expert
// with n assignments gets ceil(n/128) tiles of balanced size.
__global__ void __launch_bounds__(256) permute_kernel(const uint16_t* __restrict__ x, PrefillParams p) {
  pdl_wait();
  const int H = p.H, A = p.T * p.k;
  if (blockIdx.x == 0) {
    __shared__ int s_scan[kMaxExperts];
    const int e = threadIdx.x;
    int n = 0, tl = 0;
    if (e < p.E) {
      n = __ldcg(p.offsets + e + 1) - __ldcg(p.offsets + e);
      tl = token_tiles(n);
    }
    s_scan[e] = tl;
    __syncthreads();
    for (int o = 1; o < kMaxExperts; o <<= 1) {  // inclusive scan
      const int v = e >= o ? s_scan[e - o] : 0;
      __syncthreads();
      s_scan[e] += v;
      __syncthreads();
    }
    if (tl > 0) {
      const int base = s_scan[e] - tl;
      const int rows = (n + tl - 1) / tl;
      const int off = __ldcg(p.offsets + e);
      for (int i = 0; i < tl; ++i) {
        int32_t* d = p.tiles + 4 * (base + i);
        d[0] = e;
        d[1] = off + i * rows;
        d[2] = min(rows, n - i * rows);
        d[3] = 0;
      }
    }
    if (e == kMaxExperts - 1) p.ctl[kCtlNtiles] = (uint32_t)s_scan[e];
  }
  const int groups = H / 8;  // 16 bytes = one group of 8 per step
  for (int r = blockIdx.x; r < A; r += gridDim.x) {
    const int t = __ldcg(p.perm + r) / p.k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(p.xp + (size_t)r * H);
    for (int g = threadIdx.x; g < groups; g += blockDim.x) {
      uint4 v = __ldg(src + g);
      if (p.x_to_f16) v = bf16x8_to_f16(v, p.ctl + kCtlStatus);
      uint4 o;  // (e0,e1,..,e7) -> (e0,e4,e1,e5,e2,e6,e3,e7)
      o.x = __byte_perm(v.x, v.z, 0x5410);
      o.y = __byte_perm(v.x, v.z, 0x7632);
      o.z = __byte_perm(v.y, v.w, 0x5410);
      o.w = __byte_perm(v.y, v.w, 0x7632);
      dst[g] = o;
    }
  }
  const size_t n4 = (size_t)p.T * H / 4;
  float4* acc = reinterpret_cast<float4*>(p.out_acc);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_trigger();
}

// ---------------------------------------------------------- dense matmul
// MatMulNBits through the grouped GEMM's down mode: one "expert", token r
// is assignment r with weight 1.  Here p.T = M rows of x, p.I = K, p.H = N.
// Writes the trivial routing and token tiles (block 0), x with K permuted in
// groups of 8 into p.act, zeros into p.act_lo (x is exact in 16 bits) and
// into the fp32 accumulator.
__global__ void __launch_bounds__(256) dense_setup_kernel(const uint16_t* __restrict__ x, PrefillParams p) {
  pdl_wait();
  const int M = p.T, K = p.I;
  if (blockIdx.x == 0) {
    int32_t* perm = const_cast<int32_t*>(p.perm);
    float* w = const_cast<float*>(p.topk_w);
    int32_t* off = const_cast<int32_t*>(p.offsets);
    for (int r = threadIdx.x; r < M; r += blockDim.x) {
      perm[r] = r;
      w[r] = 1.f;
    }
    const int nt = token_tiles(M), rows = (M + nt - 1) / nt;
    for (int i = threadIdx.x; i < nt; i += blockDim.x) {
      int32_t* d = p.tiles + 4 * i;
      d[0] = 0;
      d[1] = i * rows;
      d[2] = min(rows, M - i * rows);
      d[3] = 0;
    }
    if (threadIdx.x == 0) {
      off[0] = 0;
      off[1] = M;
      p.ctl[kCtlNtiles] = (uint32_t)nt;
    }
  }
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t t0 = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t ng = (size_t)M * (K / 8);
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(p.act);
  uint4* dlo = reinterpret_cast<uint4*>(p.act_lo);
  for (size_t i = t0; i < ng; i += stride) {
    uint4 v = __ldg(src + i);
    if (p.x_to_f16) v = bf16x8_to_f16(v, p.ctl + kCtlStatus);
    uint4 o;  // (e0,e1,..,e7) -> (e0,e4,e1,e5,e2,e6,e3,e7)
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    dst[i] = o;
    if (dlo) dlo[i] = make_uint4(0, 0, 0, 0);
  }
  float4* acc = reinterpret_cast<float4*>(p.out_acc);
  const size_t n4 = (size_t)M * p.H / 4;
  for (size_t i = t0; i < n4; i += stride) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_trigger();
}

// ---------------------------------------------------------------- convert
// out = act_dtype(out_acc (+ out if accumulating)), 4 elements per step
template <typename TA>
__global__ void __launch_bounds__(256) convert_kernel(PrefillParams p, uint16_t* __restrict__ out) {
  pdl_wait();
  const size_t n4 = (size_t)p.T * p.H / 4;
  const float4* acc = reinterpret_cast<const float4*>(p.out_acc);
  uint2* o = reinterpret_cast<uint2*>(out);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    float4 v = __ldcg(acc + i);
    if (p.accumulate) {
      const uint2 r = o[i];
      v.x += Half<TA>::to_float((uint16_t)(r.x & 0xFFFFu));
      v.y += Half<TA>::to_float((uint16_t)(r.x >> 16));
      v.z += Half<TA>::to_float((uint16_t)(r.y & 0xFFFFu));
      v.w += Half<TA>::to_float((uint16_t)(r.y >> 16));
    }
    uint2 w;
    w.x = (uint32_t)Half<TA>::from_float(v.x) | ((uint32_t)Half<TA>::from_float(v.y) << 16);
    w.y = (uint32_t)Half<TA>::from_float(v.z) | ((uint32_t)Half<TA>::from_float(v.w) << 16);
    o[i] = w;
  }
}

// ------------------------------------------------------------ dequant core
// Two codes (the 4-bit fields at bits [0,4) and [16,20) of v) of one scale
// block to packed operand pairs.  w = (q - zp) * s is exact in fp32 (at most
// 4 + 11 significant bits); hi = RN_OT(w) and lo = w - hi, which OT holds
// exactly (the remainder has at most 7 significant bits), so hi + lo == w.
// "Magic" constants: 0x4300 | q is the bf16 number 128 + q and 0x6400 | q
// the fp16 number 1024 + q, so (magic | q) - (magic | zp) = q - zp exactly.
template <uint32_t MAGIC>
__device__ __forceinline__ uint32_t magic_pair(uint32_t v) {
  uint32_t h;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(h) : "r"(v), "n"(MAGIC));
  return h;
}
__device__ __forceinline__ uint32_t u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ uint32_t u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t v) { return *reinterpret_cast<__nv_bfloat162*>(&v); }
__device__ __forceinline__ __half2 h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

template <typename OT, typename TS>
struct Deq;
// bf16 operands, bf16 scales: qz * s has <= 12 significant bits
template <>
struct Deq<__nv_bfloat16, __nv_bfloat16> {
  __nv_bfloat162 zc, sc;
  __device__ __forceinline__ void set(uint32_t zp, uint16_t s) {
    zc = __bfloat162bfloat162(__ushort_as_bfloat16((uint16_t)(0x4300u | zp)));
    sc = __bfloat162bfloat162(__ushort_as_bfloat16(s));
  }
  __device__ __forceinline__ uint32_t hi(uint32_t v) const {
    return u32(__hmul2(__hsub2(bf2(magic_pair<0x43004300u>(v)), zc), sc));
  }
  __device__ __forceinline__ void both(uint32_t v, uint32_t& h, uint32_t& l) const {
    const __nv_bfloat162 qz = __hsub2(bf2(magic_pair<0x43004300u>(v)), zc);
    const __nv_bfloat162 hv = __hmul2(qz, sc);
    h = u32(hv);
    l = u32(__hfma2(qz, sc, __hneg2(hv)));
  }
};
// bf16 operands, fp16 scales: s = sh + sl with sh = RN_bf16(s) and sl exact
// (<= 3 bits); c = qz * sl is exact, hi = RN(qz * sh + c) = RN(w),
// d = qz * sh - hi and lo = d + c = w - hi are exact.
template <>
struct Deq<__nv_bfloat16, __half> {
  __nv_bfloat162 zc, shc, slc;
  __device__ __forceinline__ void set(uint32_t zp, uint16_t s) {
    zc = __bfloat162bfloat162(__ushort_as_bfloat16((uint16_t)(0x4300u | zp)));
    const float sf = __half2float(__ushort_as_half(s));
    const __nv_bfloat16 sh = __float2bfloat16_rn(sf);
    shc = __bfloat162bfloat162(sh);
    slc = __bfloat162bfloat162(__float2bfloat16_rn(sf - __bfloat162float(sh)));
  }
  __device__ __forceinline__ uint32_t hi(uint32_t v) const {
    const __nv_bfloat162 qz = __hsub2(bf2(magic_pair<0x43004300u>(v)), zc);
    return u32(__hfma2(qz, shc, __hmul2(qz, slc)));
  }
  __device__ __forceinline__ void both(uint32_t v, uint32_t& h, uint32_t& l) const {
    const __nv_bfloat162 qz = __hsub2(bf2(magic_pair<0x43004300u>(v)), zc);
    const __nv_bfloat162 c = __hmul2(qz, slc);
    const __nv_bfloat162 hv = __hfma2(qz, shc, c);
    h = u32(hv);
    l = u32(__hadd2(__hfma2(qz, shc, __hneg2(hv)), c));
  }
};
// fp16 operands (fp16 scales, or bf16 scales converted exactly to fp16):
// qz * s has <= 15 significant bits; exact split for scales >= 2^-14
template <typename TS>
struct DeqF16 {
  __half2 zc, sc;
  __device__ __forceinline__ void set(uint32_t zp, uint16_t s) {
    zc = __half2half2(__ushort_as_half((uint16_t)(0x6400u | zp)));
    sc = __half2half2(__float2half_rn(Half<TS>::to_float(s)));
  }
  __device__ __forceinline__ uint32_t hi(uint32_t v) const {
    return u32(__hmul2(__hsub2(h2(magic_pair<0x64006400u>(v)), zc), sc));
  }
  __device__ __forceinline__ void both(uint32_t v, uint32_t& h, uint32_t& l) const {
    const __half2 qz = __hsub2(h2(magic_pair<0x64006400u>(v)), zc);
    const __half2 hv = __hmul2(qz, sc);
    h = u32(hv);
    l = u32(__hfma2(qz, sc, __hneg2(hv)));
  }
};
template <> struct Deq<__half, __half> : DeqF16<__half> {};
template <> struct Deq<__half, __nv_bfloat16> : DeqF16<__nv_bfloat16> {};

// fp32 -> (hi, lo) operand pair of the activation (split path)
template <typename OT>
__device__ __forceinline__ void split_act(float a, uint16_t& h, uint16_t& l) {
  h = Half<OT>::from_float(a);
  l = Half<OT>::from_float(a - Half<OT>::to_float(h));
}

// ------------------------------------------------------------ grouped GEMM
constexpr uint32_t kTileOp = kBN * 128;    // 16-bit token tile: up to kBN rows x 64 K (SW128)
constexpr uint32_t kPkBytes = 128 * 32;    // packed codes: 128 rows x 64 codes
constexpr int kMaxPk = 24;                 // packed-code ring slots (at most)
constexpr int kMaxSt = 4;                  // operand stages (at most; 3 with hi + lo weights)
constexpr uint32_t kGbufFloats = 64 * 17;  // gate values of one 16-column chunk (padded rows)
constexpr uint32_t kTmemCols = 512;        // the whole TMEM of the SM (one CTA per SM)
constexpr uint32_t kAccCols = 2 * kBN;     // two 160-column accumulators, then the weight stages
constexpr uint32_t kSmemLimit = 232448;    // 227 KB per CTA
constexpr uint32_t kNapNs = 256;          // poll interval of the off-critical-path waits
constexpr uint32_t kMmaNapNs = 32;        // poll interval of the MMA issuer's waits (see the issuer)
constexpr int kDeqWarps = 8;               // two per sub-partition: row = warp%4*32+lane, half = warp/4

// Warp roles (kGemmThreads = 512; warp w issues from SM sub-partition w % 4
// and may touch TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31):
//   0-7    dequantisers (TMEM lane quadrant = warp % 4, K half = warp / 4)
//   8      TMEM owner and tcgen05.mma issuer (converged warp, elected lane)
//   9      token-tile producer (TMA, L2-resident gathered tokens / SwiGLU output)
//   10     weight producer: packed codes (deep ring) and each tile's scales / zero points
//   11     idle
//   12-15  epilogue (TMEM lane quadrant = warp % 4)
// TMEM columns: [0, 320) the two accumulators (token tiles of up to 160
// columns: an expert with up to 160 assignments is one tile, so its weights
// are dequantised once and each MMA is wide); from 320 one weight operand
// stage per 64-wide K chunk: 32 columns (64 16-bit values per row), twice
// that with hi + lo, so 4 stages, or 3 with hi + lo.  (Measured: 160-column
// tiles with 3 hi + lo stages beat 192 with 2 and 128 with 4 on the
// 2048-token stack layer.)
// Shared memory: [barriers][scale buffers][token stages: B hi, B lo][packed ring][exchange]
struct GemmSmem {
  uint32_t b_lo, stage;  // offset of the low tile inside a token stage, stage size
  uint32_t sz_bytes, sz_off, stage_off, pk_off, gbuf_off, total;
};
// as: activations (down: SwiGLU output) as hi + lo
__host__ __device__ inline GemmSmem gemm_smem(int mode, bool as, int nb, bool has_zp, int nst, int nsz, int npk) {
  GemmSmem S;
  S.b_lo = kTileOp;
  S.stage = (as ? 2u : 1u) * kTileOp;
  S.sz_bytes = ((uint32_t)128 * nb * 2 + (has_zp ? (uint32_t)128 * nb : 0u) + 1023u) & ~1023u;
  S.sz_off = 1024;
  S.stage_off = S.sz_off + nsz * S.sz_bytes;
  S.pk_off = S.stage_off + nst * S.stage;
  S.gbuf_off = S.pk_off + npk * kPkBytes;
  S.total = S.gbuf_off + (mode == kModeGU ? 2 * kGbufFloats * 4 : 0) + 1024;  // + base alignment slack
  return S;
}
// Pipeline plan.  Two tile-scale buffers first (with one, the weight
// producer cannot start the next tile's codes until the current tile is
// dequantised), then as many operand stages as TMEM holds (4, or 3 with hi
// + lo weights) down to 2 while at least 12 packed slots remain; the packed
// ring takes the rest (<= 24 slots).  Long reductions with small blocks
// (large whole-K scale buffers) fall back to one scale buffer and as few as
// 4 packed slots.
__host__ __device__ constexpr int gemm_max_stages(bool ws) {
  return (int)((512u - kAccCols) / (ws ? 64u : 32u)) < kMaxSt ? (int)((512u - kAccCols) / (ws ? 64u : 32u)) : kMaxSt;
}
__host__ inline bool gemm_plan(int mode, bool ws, bool as, int nb, bool has_zp, int& nst, int& nsz, int& npk) {
  for (int sz = 2; sz >= 1; --sz)
    for (int st = gemm_max_stages(ws); st >= 2; --st) {
      const int pmin = sz == 1 && st == 2 ? 4 : 12;
      int pk = kMaxPk;
      while (pk >= pmin && gemm_smem(mode, as, nb, has_zp, st, sz, pk).total > kSmemLimit) --pk;
      if (pk >= pmin) {
        nst = st;
        nsz = sz;
        npk = pk;
        return true;
      }
    }
  return false;
}

// bounded wait that also gives up once another role has aborted.  nap_ns >
// 0 (roles whose waits are long and off the critical path: the producers
// and the epilogue's wait for a finished accumulator) sleeps between polls,
// so that the waiting warps leave the issue slots to the dequantisers and
// the MMA issuer; the others poll with try_wait's own suspend hint.
// `limit` (SM cycles) is the control block's kCtlWaitLimit x 1024 when that
// is set, else kWaitLimitCycles: a test shortens it to drive every role's
// give-up and drain path.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort, long long limit, uint32_t nap_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!(nap_ns ? mbar_try_wait(bar, parity) : mbar_try_wait_sleep(bar, parity, 20000u))) {
    if (nap_ns) __nanosleep(nap_ns);
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      set_status(status, QMOE_ST_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// ring position: slot index and the parity of its current use
struct Ring {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// drain helper for the abort path: wait (bounded) for the last use of each
// slot of a ring whose `issued` uses went round-robin over n slots
__device__ __forceinline__ void drain_ring(uint64_t* full, int n, int issued) {
  for (int s = 0; s < n; ++s)
    if (issued > s) mbar_wait(&full[s], ((issued - 1 - s) / n) & 1, nullptr);
}

// One persistent CTA per SM.  Work item t = (weight row block mb, token
// tile nt), nt fastest, so the token tiles of one expert run side by side
// and share the weight tile through L2.
// OT: operand type (fp16 / bf16); WS: weights as hi + lo; AS: activations
// (down: the SwiGLU output) as hi + lo
template <int MODE, typename OT, typename TS, bool HAS_ZP, bool WS, bool AS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_b2,
                const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned start (128-byte swizzle), reached by pointer arithmetic
  // on the shared array so every access below compiles to a shared-memory
  // instruction rather than a generic one
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr bool GU = MODE == kModeGU;
  constexpr bool BLO = AS && !GU;  // second B tile (activation low part)
  const int K = GU ? p.H : p.I;       // reduction length
  const int NR = GU ? p.I : p.H;      // weight rows per expert matrix
  const int nb = K >> p.lbs;
  const int nst = p.nst, nsz = p.nsz, npk = p.npk;
  const GemmSmem L = gemm_smem(MODE, BLO, nb, HAS_ZP, nst, nsz, npk);
  constexpr uint32_t AW = WS ? 64 : 32;  // TMEM columns of one weight operand stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* b_full = bars;                  // [kMaxSt] token tile landed
  uint64_t* a_full = bars + kMaxSt;         // [kMaxSt] weights in TMEM (one arrival per dequant warp)
  uint64_t* empty = bars + 2 * kMaxSt;      // [kMaxSt] MMAs done with the stage
  uint64_t* pk_full = bars + 3 * kMaxSt;    // [kMaxPk] packed codes landed
  uint64_t* pk_empty = pk_full + kMaxPk;    // [kMaxPk] packed codes read
  uint64_t* tmem_full = pk_empty + kMaxPk;  // [2] accumulator complete
  uint64_t* tmem_empty = tmem_full + 2;     // [2] accumulator drained
  uint64_t* sz_full = tmem_empty + 2;       // [2] tile scales landed
  uint64_t* sz_empty = sz_full + 2;         // [2] tile scales no longer read
  uint64_t* gx_full = sz_empty + 2;         // [2] gate chunk in the exchange buffer
  uint64_t* gx_empty = gx_full + 2;         // [2] exchange buffer free
  uint64_t* fin = gx_empty + 2;             // drain on abort
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  uint8_t* szbuf = smem + L.sz_off;
  uint8_t* stages = smem + L.stage_off;
  uint8_t* pkbuf = smem + L.pk_off;
  float* gbuf = reinterpret_cast<float*>(smem + L.gbuf_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* status = p.ctl + kCtlStatus;
  const int KC = K / 64;
  const int MB = NR / (GU ? 64 : 128);

  if (tid == 0) {
    for (int s = 0; s < kMaxSt; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&a_full[s], kDeqWarps);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kMaxPk; ++s) {
      mbar_init(&pk_full[s], 1);
      mbar_init(&pk_empty[s], kDeqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 4);
      mbar_init(&sz_full[b], 1);
      mbar_init(&sz_empty[b], kDeqWarps);
      mbar_init(&gx_full[b], 2);
      mbar_init(&gx_empty[b], 2);
    }
    mbar_init(fin, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  pdl_wait();  // routing, token tiles and (down) the SwiGLU output come from earlier grids
  pdl_trigger();
  const int NT = (int)__ldcg(p.ctl + kCtlNtiles);
  const uint32_t wlim_k = __ldcg(p.ctl + kCtlWaitLimit);
  const uint32_t diag = __ldcg(p.ctl + kCtlDiag);
  const long long wlim = wlim_k ? (long long)wlim_k << 10 : kWaitLimitCycles;
  const int ntile_total = NT * MB;
  const int4* tiles = reinterpret_cast<const int4*>(p.tiles);

  if (warp == 9) {
    // ============================================================ token-tile producer
    if (lane == 0) {
      int it = 0;
      Ring rs;
      for (int t = blockIdx.x; t < ntile_total && !*s_abort; t += gridDim.x) {
        const int4 tl = __ldcg(tiles + t % NT);
        const int row0 = tl.y, npad = (tl.z + 15) & ~15;
        const int nbox = (npad + kBoxRows - 1) / kBoxRows;
        const uint32_t btx = nbox * kBoxRows * 128 * (BLO ? 2 : 1);
        for (int kc = 0; kc < KC; ++kc, ++it, rs.next(nst)) {
          if (it >= nst && !wait_or_abort(&empty[rs.i], rs.ph ^ 1u, status, s_abort, wlim, kNapNs)) break;
          uint8_t* st = stages + rs.i * L.stage;
          uint64_t* fb = &b_full[rs.i];
          mbar_arrive_expect_tx(fb, btx);
          for (int bx = 0; bx < nbox; ++bx) {
            tma_load_2d(st + bx * kBoxRows * 128, &tm_b, kc * 64, row0 + bx * kBoxRows, fb);
            if (BLO) tma_load_2d(st + L.b_lo + bx * kBoxRows * 128, &tm_b2, kc * 64, row0 + bx * kBoxRows, fb);
          }
        }
      }
      if (*s_abort) drain_ring(b_full, nst, it);
    }
  } else if (warp == 10) {
    // ============================================================ weight producer
    if (lane == 0) {
      int ip = 0, tc = 0;
      Ring rp, rz;
      const uint32_t sbytes = 128u * nb * 2, zbytes = HAS_ZP ? 128u * nb : 0u;
      for (int t = blockIdx.x; t < ntile_total && !*s_abort; t += gridDim.x, ++tc, rz.next(nsz)) {
        const int4 tl = __ldcg(tiles + t % NT);
        const int mb = t / NT, e = tl.x;
        if (tc >= nsz && !wait_or_abort(&sz_empty[rz.i], rz.ph ^ 1u, status, s_abort, wlim, kNapNs)) break;
        // block scales / zero points of the tile's 128 weight rows over the whole K
        uint8_t* sz = szbuf + rz.i * L.sz_bytes;
        uint64_t* zb = &sz_full[rz.i];
        mbar_arrive_expect_tx(zb, sbytes + zbytes);
        if (GU) {
          const size_t r = (size_t)e * NR + mb * 64;
          bulk_g2s(sz, static_cast<const uint8_t*>(p.s[0]) + r * nb * 2, sbytes / 2, zb);
          bulk_g2s(sz + sbytes / 2, static_cast<const uint8_t*>(p.s[1]) + r * nb * 2, sbytes / 2, zb);
          if (HAS_ZP) {
            bulk_g2s(sz + sbytes, p.z[0] + r * nb, zbytes / 2, zb);
            bulk_g2s(sz + sbytes + zbytes / 2, p.z[1] + r * nb, zbytes / 2, zb);
          }
        } else {
          const size_t r = (size_t)e * NR + mb * 128;
          bulk_g2s(sz, static_cast<const uint8_t*>(p.s[2]) + r * nb * 2, sbytes, zb);
          if (HAS_ZP) bulk_g2s(sz + sbytes, p.z[2] + r * nb, zbytes, zb);
        }
        for (int kc = 0; kc < KC; ++kc, ++ip, rp.next(npk)) {
          if (ip >= npk && !wait_or_abort(&pk_empty[rp.i], rp.ph ^ 1u, status, s_abort, wlim, kNapNs)) break;
          uint8_t* pk = pkbuf + rp.i * kPkBytes;
          uint64_t* fb = &pk_full[rp.i];
          mbar_arrive_expect_tx(fb, kPkBytes);
          if (GU) {
            tma_load_2d(pk, &tm_a0, kc * 32, e * NR + mb * 64, fb);
            tma_load_2d(pk + 64 * 32, &tm_a1, kc * 32, e * NR + mb * 64, fb);
          } else {
            tma_load_2d(pk, &tm_a0, kc * 32, e * NR + mb * 128, fb);
          }
        }
      }
      if (*s_abort) {  // let the copies already issued land before the CTA exits
        drain_ring(pk_full, npk, ip);
        drain_ring(sz_full, nsz, tc);
      }
    }
  } else if (warp == 8) {
    // ============================================================ MMA issuer
    // The whole warp runs the loop and one elected lane issues: a lone
    // active lane of a diverged warp issues tcgen05.mma at half the rate.
    int tc = 0;
    bool issued = false;
    Ring rs;
    constexpr bool bf = std::is_same<OT, __nv_bfloat16>::value;
    for (int t = blockIdx.x; t < ntile_total; t += gridDim.x, ++tc) {
      const int4 tl = __ldcg(tiles + t % NT);
      const uint32_t idesc = idesc_f16(128, (tl.z + 15) & ~15, bf);
      const int b = tc & 1;
      if (tc >= 2 && !wait_or_abort(&tmem_empty[b], ((tc >> 1) - 1) & 1, status, s_abort, wlim)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + b * kBN;
      bool ok = true;
      for (int kc = 0; kc < KC; ++kc, rs.next(nst)) {
        if (!wait_or_abort(&a_full[rs.i], rs.ph, status, s_abort, wlim, kMmaNapNs) ||
            !wait_or_abort(&b_full[rs.i], rs.ph, status, s_abort, wlim, kMmaNapNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_u32(stages + rs.i * L.stage);
        const uint64_t bh = sw128_desc(st), bl = sw128_desc(st + L.b_lo);
        const uint32_t ah = tmem_base + kAccCols + rs.i * AW, al = ah + 32;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // K = 16 per instruction: 8 TMEM columns, +32 bytes in the swizzled row
          mma_f16_ts_elect(d_tmem, ah + 8 * kk, bh + 2 * kk, idesc, (kc | kk) != 0);
          if (WS) mma_f16_ts_elect(d_tmem, al + 8 * kk, bh + 2 * kk, idesc, 1u);
          if (BLO) mma_f16_ts_elect(d_tmem, ah + 8 * kk, bl + 2 * kk, idesc, 1u);
        }
        issued = true;
        mma_commit_elect(&empty[rs.i]);
      }
      if (!ok) break;
      mma_commit_elect(&tmem_full[b]);
    }
    // every MMA must have finished before TMEM is freed: after an abort the
    // epilogue may not have waited for the last accumulator
    if (issued) {
      mma_commit_elect(fin);
      mbar_wait(fin, 0, nullptr);
    }
  } else if (warp < kDeqWarps) {
    // ============================================================ dequantisers
    const int qd = warp & 3;              // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;         // weight row of the tile
    const int hh = warp >> 2;             // which 32 codes of the 64-wide chunk
    const uint32_t a_row = tmem_base + ((uint32_t)(qd * 32) << 16) + kAccCols + hh * 16;
    const int nchunks = blockIdx.x < ntile_total ? ((ntile_total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * KC : 0;
    int it = 0;
    Ring rs, rp, rz;
    bool ok = true;
    // This chunk's codes are loaded one chunk ahead, so the shared-memory
    // latency overlaps the previous chunk's work.
    uint4 q = make_uint4(0, 0, 0, 0);
    if (nchunks > 0) {
      ok = wait_or_abort(&pk_full[0], 0, status, s_abort, wlim);
      // QMOE_DIAG_STALL_GEMM: then wait for the slot's second fill (phase
      // 1), which cannot come before this one is consumed, so the wait runs
      // out (timeout test).  A wait on parity 1 before phase 0 has completed
      // would return at once: it asks for the phase before the first.
      if (ok && (diag & QMOE_DIAG_STALL_GEMM)) ok = wait_or_abort(&pk_full[0], 1, status, s_abort, wlim);
      if (ok) q = *reinterpret_cast<const uint4*>(pkbuf + r * 32 + hh * 16);
    }
    // The rows of a tile's scales sit nb * 2 bytes apart: at 128 bytes the 32
    // rows of a warp fall into one bank.  When rows are 16-byte aligned a
    // lane reads 8 consecutive block scales (and 8 zero points) at once and
    // keeps them for the next chunks: one conflicted load per 8 blocks.
    const bool vec = (nb & 7) == 0;
    for (int t = blockIdx.x; t < ntile_total && ok; t += gridDim.x, rz.next(nsz)) {
      if (!wait_or_abort(&sz_full[rz.i], rz.ph, status, s_abort, wlim)) break;
      const uint8_t* sz = szbuf + rz.i * L.sz_bytes;
      const uint16_t* srow = reinterpret_cast<const uint16_t*>(sz) + (size_t)r * nb;
      const uint8_t* zrow = sz + 128u * nb * 2 + (size_t)r * nb;
      int cached = -8;
      uint4 sv = make_uint4(0, 0, 0, 0);
      uint2 zv = make_uint2(0, 0);
      for (int kc = 0; kc < KC; ++kc, ++it, rs.next(nst), rp.next(npk)) {
        // block_size >= 32: the 32 codes of this half share one block
        const int blk = (kc * 64 + hh * 32) >> p.lbs;
        uint32_t zpv;
        uint16_t scv;
        if (vec) {
          if ((blk & ~7) != cached) {
            cached = blk & ~7;
            sv = *reinterpret_cast<const uint4*>(srow + cached);
            if (HAS_ZP) zv = *reinterpret_cast<const uint2*>(zrow + cached);
          }
          const int j = blk & 7;
          const uint32_t sw = (j >> 1) == 0 ? sv.x : (j >> 1) == 1 ? sv.y : (j >> 1) == 2 ? sv.z : sv.w;
          scv = (uint16_t)(sw >> ((j & 1) * 16));
          zpv = HAS_ZP ? (((j >> 2) ? zv.y : zv.x) >> ((j & 3) * 8)) & 0xFFu : 8u;
        } else {
          scv = srow[blk];
          zpv = HAS_ZP ? (uint32_t)zrow[blk] : 8u;
        }
        Deq<OT, TS> d;
        d.set(zpv, scv);
        // column c of the row holds K elements 2c, 2c + 1 of the permuted
        // order: group g's pairs (0,4), (1,5), (2,6), (3,7) in columns 4g..4g+3
        uint32_t h[16], l[16];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int gg = 0; gg < 4; ++gg)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            if (WS)
              d.both(w[gg] >> (4 * jj), h[gg * 4 + jj], l[gg * 4 + jj]);
            else
              h[gg * 4 + jj] = d.hi(w[gg] >> (4 * jj));
          }
        if (it + 1 < nchunks) {  // the next chunk's codes (the next ring slot)
          Ring rn = rp;
          rn.next(npk);
          if (!wait_or_abort(&pk_full[rn.i], rn.ph, status, s_abort, wlim)) { ok = false; break; }
          q = *reinterpret_cast<const uint4*>(pkbuf + rn.i * kPkBytes + r * 32 + hh * 16);
        }
        if (it >= nst && !wait_or_abort(&empty[rs.i], rs.ph ^ 1u, status, s_abort, wlim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ta = a_row + rs.i * AW;
        tmem_st16(ta, h);
        if (WS) tmem_st16(ta + 32, l);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        // the packed slot is handed back only once the operand it produced
        // is stored: releasing it right after the load once let the next TMA
        // fill race with the chunk (wrong rows in a few tiles)
        if (lane == 0) {
          mbar_arrive(&a_full[rs.i]);
          mbar_arrive(&pk_empty[rp.i]);
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sz_empty[rz.i]);
    }
  } else if (warp >= 12) {
    // ============================================================ epilogue
    const int q = warp & 3;         // TMEM lane quadrant this warp may read
    const int row = q * 32 + lane;  // accumulator row = weight row of the tile
    int tc = 0, cc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntile_total; t += gridDim.x, ++tc) {
      const int4 tl = __ldcg(tiles + t % NT);
      const int mb = t / NT;
      const int row0 = tl.y, nrows = tl.z, npad = (nrows + 15) & ~15;
      const int b = tc & 1;
      if (!wait_or_abort(&tmem_full[b], (tc >> 1) & 1, status, s_abort, wlim, kNapNs)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * kBN;
      for (int c0 = 0; c0 < npad; c0 += 16, ++cc) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        if (GU) {
          // rows 0-63 gate, 64-127 up of the same 64 intermediate indices
          const int xb = cc & 1;
          float* gx = gbuf + xb * kGbufFloats;
          if (q < 2) {
            if (cc >= 2 && !wait_or_abort(&gx_empty[xb], ((cc >> 1) - 1) & 1, status, s_abort, wlim)) { ok = false; break; }
#pragma unroll
            for (int j = 0; j < 16; ++j) gx[row * 17 + j] = __uint_as_float(v[j]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&gx_full[xb]);
          } else {
            if (!wait_or_abort(&gx_full[xb], (cc >> 1) & 1, status, s_abort, wlim)) { ok = false; break; }
            const int i = row - 64;
            const int ig = mb * 64 + i;
            const size_t col = (ig & ~7) + kperm_pos(ig & 7);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c0 + j < nrows) {
                const float g = gx[i * 17 + j];
                const float a = g / (1.f + expf(-g)) * __uint_as_float(v[j]);
                const size_t o = (size_t)(row0 + c0 + j) * p.I + col;
                uint16_t h, l;
                split_act<OT>(a, h, l);
                if (std::is_same<OT, __half>::value && !(fabsf(a) <= 65504.f)) set_status(status, QMOE_ST_RANGE);
                p.act[o] = h;
                p.act_lo[o] = l;
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&gx_empty[xb]);
          }
        } else {
          // lanes 0-15 fetch the chunk's 16 assignments and routing weights
          int a_l = 0;
          float w_l = 0.f;
          if (lane < 16 && c0 + lane < nrows) {
            a_l = __ldg(p.perm + row0 + c0 + lane);
            w_l = __ldg(p.topk_w + a_l);
          }
          const int h = mb * 128 + row;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int a = __shfl_sync(0xffffffffu, a_l, j);
            const float w = __shfl_sync(0xffffffffu, w_l, j);
            if (c0 + j < nrows)
              atomicAdd(p.out_acc + (size_t)(a / p.k) * p.H + h, w * __uint_as_float(v[j]));
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host

// Operands of the grouped GEMM.  The operand type is fp16 when the block
// scales are bf16 or the activations fp16 (a bf16 token converts to fp16
// exactly inside fp16's normal range), else bf16.  One weight operand is
// exact when the scales are bf16 and there are no zero points: q - 8 lies in
// [-8, 7], whose magnitudes need at most 3 significant bits (8 needs one),
// so s (q - 8) has at most 8 + 3 = 11, fp16's significand.  With zero points
// q - zp reaches 15 (4 bits) and fp16 scales carry 11 bits, so those weights
// go hi + lo (the product's leading 11 bits, then the rest).
struct GemmOps {
  bool f16, ws;
};
static inline GemmOps gemm_ops(int act_dtype, int scale_dtype, bool has_zp) {
  return {scale_dtype == 1 || act_dtype == 0, scale_dtype == 0 || has_zp};
}

bool dense_fits(int N, int K, int bs, int act_dtype, int scale_dtype, bool has_zp) {
  if (N % 128 || K % 64 || bs < 32 || (bs & (bs - 1))) return false;
  int a, b, c;
  return gemm_plan(kModeDN, gemm_ops(act_dtype, scale_dtype, has_zp).ws, false, K / bs, has_zp, a, b, c);
}

bool prefill_fits(int H, int I, int bs, int act_dtype, int scale_dtype, bool has_zp_gu, bool has_zp_d) {
  if (H % 128 || I % 64 || bs < 32 || (bs & (bs - 1))) return false;
  int a, b, c;
  return gemm_plan(kModeGU, gemm_ops(act_dtype, scale_dtype, has_zp_gu).ws, false, H / bs, has_zp_gu, a, b, c) &&
         gemm_plan(kModeDN, gemm_ops(act_dtype, scale_dtype, has_zp_d).ws, true, I / bs, has_zp_d, a, b, c);
}

bool prefill_x_to_f16(int act_dtype, int scale_dtype) { return scale_dtype == 1 && act_dtype == 1; }

cudaError_t launch_prefill_permute(const PrefillParams& p, const void* x, int, cudaStream_t st, bool pdl) {
  const int A = p.T * p.k;
  const int blocks = A < 1024 ? A : 1024;
  return launch_kernel(permute_kernel, dim3(blocks), dim3(256), 0, st, pdl, static_cast<const uint16_t*>(x), p);
}

template <int MODE, typename OT, typename TS, bool Z, bool WS, bool AS>
static cudaError_t launch_gemm_t(PrefillParams p, const CUtensorMap* m, cudaStream_t st, bool pdl) {
  const int K = (MODE == kModeGU) ? p.H : p.I;
  constexpr bool BLO = AS && MODE == kModeDN;
  if (!gemm_plan(MODE, WS, BLO, K / p.bs, Z, p.nst, p.nsz, p.npk)) return cudaErrorInvalidValue;
  const GemmSmem L = gemm_smem(MODE, BLO, K / p.bs, Z, p.nst, p.nsz, p.npk);
  // the kernel takes all of the SM's TMEM: at least half the shared memory
  // keeps a second CTA off the SM
  const uint32_t smem = L.total > kSmemLimit / 2 + 1024 ? L.total : kSmemLimit / 2 + 1024;
  auto fn = gemm_kernel<MODE, OT, TS, Z, WS, AS>;
  cudaError_t err = ensure_smem(fn, smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(fn, dim3(device_sm_count()), dim3(kGemmThreads), (size_t)smem, st, pdl, m[0], m[1], m[2],
                       m[3], p);
}

// (operand type, weight split) follow from the dtypes and zero points
// (gemm_ops); AS: the down GEMM of the layer takes the SwiGLU output as
// hi + lo, the dense MatMulNBits takes x alone
template <int MODE, typename TS>
static cudaError_t dispatch_gemm_ts(const PrefillParams& p, bool f16, bool z, bool as, const CUtensorMap* m,
                                    cudaStream_t st, bool pdl) {
#define QMOE_G(OT, Z_, WS_) return as ? launch_gemm_t<MODE, OT, TS, Z_, WS_, true>(p, m, st, pdl) \
                                      : launch_gemm_t<MODE, OT, TS, Z_, WS_, false>(p, m, st, pdl)
  if (std::is_same<TS, __nv_bfloat16>::value) {  // fp16 operands; one weight operand without zero points
    if (z) QMOE_G(__half, true, true);
    QMOE_G(__half, false, false);
  }
  if (f16) {
    if (z) QMOE_G(__half, true, true);
    QMOE_G(__half, false, true);
  }
  if (z) QMOE_G(__nv_bfloat16, true, true);
  QMOE_G(__nv_bfloat16, false, true);
#undef QMOE_G
}

cudaError_t launch_prefill_gemm(const PrefillParams& p, int mode, int act_dtype, int scale_dtype, bool dense,
                                cudaStream_t st, bool pdl) {
  const int A = p.T * p.k;
  const GemmOps o = gemm_ops(act_dtype, scale_dtype, false);
  const CUtensorMapDataType odt = o.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap m[4];
  if (mode == kModeGU) {
    if (!make_map(&m[0], p.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.H / 2, (uint64_t)p.E * p.I, 32, 64,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&m[1], p.w[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.H / 2, (uint64_t)p.E * p.I, 32, 64,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&m[2], p.xp, odt, 2, p.H, A, 64, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;
    m[3] = m[2];
    return scale_dtype == 1
               ? dispatch_gemm_ts<kModeGU, __nv_bfloat16>(p, o.f16, p.z[0] != nullptr, false, m, st, pdl)
               : dispatch_gemm_ts<kModeGU, __half>(p, o.f16, p.z[0] != nullptr, false, m, st, pdl);
  }
  const bool as = !dense;
  if (!make_map(&m[0], p.w[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.I / 2, (uint64_t)p.E * p.H, 32, 128,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&m[2], p.act, odt, 2, p.I, A, 64, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m[3], as ? p.act_lo : p.act, odt, 2, p.I, A, 64, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  m[1] = m[0];
  return scale_dtype == 1 ? dispatch_gemm_ts<kModeDN, __nv_bfloat16>(p, o.f16, p.z[2] != nullptr, as, m, st, pdl)
                          : dispatch_gemm_ts<kModeDN, __half>(p, o.f16, p.z[2] != nullptr, as, m, st, pdl);
}

cudaError_t launch_dense_setup(const PrefillParams& p, const void* x, cudaStream_t st, bool pdl) {
  const size_t work = (size_t)p.T * (p.I / 8 > p.H / 4 ? p.I / 8 : p.H / 4);
  const int blocks = (int)((work + 255) / 256 < 1024 ? (work + 255) / 256 : 1024);
  return launch_kernel(dense_setup_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, st, pdl,
                       static_cast<const uint16_t*>(x), p);
}

cudaError_t launch_prefill_convert(const PrefillParams& p, void* out, int act_dtype, cudaStream_t st, bool pdl) {
  const size_t n4 = (size_t)p.T * p.H / 4;
  const int blocks = (int)((n4 + 255) / 256 < 2048 ? (n4 + 255) / 256 : 2048);
  if (act_dtype == 1)
    return launch_kernel(convert_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st, pdl, p,
                         static_cast<uint16_t*>(out));
  return launch_kernel(convert_kernel<__half>, dim3(blocks), dim3(256), 0, st, pdl, p, static_cast<uint16_t*>(out));
}

}  // namespace qmoe
