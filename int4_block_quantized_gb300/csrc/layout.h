// layout.h -- internal (non-ABI) definitions shared by host launchers and
// kernels: device status bits, the workspace map, the decode-path
// activation layout and the kernel parameter blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "qmoe.h"

#ifdef __CUDACC__
#define QMOE_HD __host__ __device__ __forceinline__
#else
#define QMOE_HD inline
#endif

namespace qmoe {

// ---- device status word bits (workspace control block, word 0)
// status bits: QMOE_ST_TIMEOUT, QMOE_ST_INDEX, QMOE_ST_RANGE (include/qmoe.h)

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;

// ---- control block (first kCtlBytes of the workspace, zeroed by init)
constexpr int kCtlStatus = 0;         // u32 sticky status bits
constexpr int kCtlGroupTicket = 1;    // u32 router: token tiles done with top-k
constexpr int kCtlNtiles = 2;         // u32 prefill: number of token tiles
constexpr int kCtlWaitLimit = 4;      // u32 grouped GEMM wait limit in units of 1024 SM cycles (0: ~2 s)
constexpr int kCtlDiag = 5;           // u32 diagnostic flags (QMOE_DIAG_*)
constexpr int kCtlSliceDone = 8;      // u32 x kMaxSplit, fused decode: clusters done with each output
                                      // slice (reset to 0 by the last arrival)
// fused decode: int64 fixed-point (2^-32) output accumulator [T][H], zero
// between calls (each call's last arrivals read and clear what it used)
constexpr size_t kCtlAccOffset = 1024;
constexpr size_t kCtlAccBytes = 128 * 1024;
constexpr int kCtlAccElems = (int)(kCtlAccBytes / 8);
constexpr size_t kCtlBytes = kCtlAccOffset + kCtlAccBytes;

// ---- router tiling
constexpr int kRouteThreads = 256;
constexpr int kMaxSplit = 8;          // H-splits (one cluster) for small T

// ---- decode path
constexpr int kDecodeMaxTokens = 16;  // T at or below: GEMV path
constexpr int kTokGroup = 4;          // tokens per decode stage

// Decode-path activation layout.  Lane l of a warp processes the two
// adjacent 16-byte weight chunks c = 64*s + 2*l + u (u = 0, 1; 32 codes
// each) of a row; the 32 activations of chunk c are 8 float4 at
// ((s*2 + u)*8 + f)*32 + l, f = 0..7, so consecutive lanes read consecutive
// float4 (no bank conflicts).  Element i is pre-multiplied by 16^-(i mod 4):
// the kernels turn nibble j of a 16-bit half-word into (q - zp) * 16^j
// exactly, and this power of two undoes it.
QMOE_HD int dec_row_floats(int K) { return ((K + 2047) / 2048) * 2048; }
QMOE_HD int dec_index(int i) {
  const int c = i >> 5;
  return (((((c >> 6) * 2 + (c & 1)) * 8 + ((i & 31) >> 2)) * 32 + ((c & 63) >> 1)) << 2) + (i & 3);
}
QMOE_HD float dec_prescale(int i) {
  const int j = i & 3;
  return j == 0 ? 1.0f : (j == 1 ? 0.0625f : (j == 2 ? 0.00390625f : 0.000244140625f));
}

// ---- workspace map (byte offsets, each region 256-byte aligned)
struct WsLayout {
  size_t ctl, ids, w, offsets, active, perm, act, xp, act16, act16lo, outacc, tiles, total;
};

QMOE_HD size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Router tiling: one cluster of kMaxSplit CTAs per tile of route_tokens()
// tokens; CTA s reduces rows [s*rps, (s+1)*rps) of H.  32-token tiles when
// there are many tokens and few experts (fewer re-reads of the router
// weight), else 8.  Every warp accumulates 8 tokens over a row subset.
QMOE_HD int route_split(int) { return kMaxSplit; }
QMOE_HD int route_tokens(int T, int E) { return (T > 4096 && E <= 64) ? 32 : 8; }
QMOE_HD int route_rows_per_split(int H) { return (((H + kMaxSplit - 1) / kMaxSplit) + 7) & ~7; }
// router weight rows staged in shared memory per pass (multiple of 8 rows,
// <= 32 KB for 8-token tiles, <= 16 KB for 32-token tiles)
QMOE_HD int route_chunk_rows(int H, int E, int tok) {
  const int rps = route_rows_per_split(H);
  int rc = ((tok == 32 ? 16384 : 32768) / (2 * E)) & ~7;
  if (rc < 8) rc = 8;
  return rc < rps ? rc : rps;
}
// chunks of the parallel counting sort (one thread each): E * chunks <= 8192
QMOE_HD int route_group_chunks(int E) {
  const int c = 8192 / E;
  return c < 128 ? c : 128;
}
// the grouping CTA stages up to this many assignment ids in shared memory
constexpr int kRouteStageIds = 16384;
// ints of shared memory the grouping CTA uses for A assignments
QMOE_HD size_t route_group_ints(int A, int E) {
  const size_t ch = route_group_chunks(E);
  const size_t L = (A + ch - 1) / ch;
  return (size_t)E * ch + 2 * kRouteThreads + (A <= kRouteStageIds ? L * (ch + 1) : 0);
}
QMOE_HD size_t route_align16(size_t v) { return (v + 15) & ~(size_t)15; }
// dynamic shared memory of a router CTA: x slice [rps][TOK] fp32, staged
// rows [rc][E] 16-bit, then one region used first for the raw x rows
// [TOK][rps+8] 16-bit and later for the partial logits [8/(TOK/8)][TOK][E]
// fp32; or, in the grouping CTA, the counting-sort arrays
QMOE_HD size_t route_smem_bytes(int T, int H, int E, int k) {
  const int tok = route_tokens(T, E);
  const size_t rps = route_rows_per_split(H);
  const size_t part = (size_t)4 * (64 / tok) * tok * E;
  const size_t xraw = (size_t)2 * tok * (rps + 8);
  const size_t compute = 4 * rps * tok + route_align16((size_t)2 * route_chunk_rows(H, E, tok) * E) +
                         (part > xraw ? part : xraw);
  const size_t A = (size_t)T * k;
  const size_t group = A > 256 ? 4 * route_group_ints((int)A, E) : 0;
  return compute > group ? compute : group;
}

QMOE_HD WsLayout ws_layout(int T, int H, int I, int E, int k) {
  WsLayout L;
  const size_t A = (size_t)T * k;
  size_t o = 0;
  L.ctl = o;      o = align256(o + kCtlBytes);
  L.ids = o;      o = align256(o + A * 4);
  L.w = o;        o = align256(o + A * 4);
  L.offsets = o;  o = align256(o + (size_t)(E + 1) * 4);
  L.active = o;   o = align256(o + (size_t)(E + 2) * 4);  // [0] = count, [1..] = ids
  L.perm = o;     o = align256(o + A * 4);
  L.act = o;  // decode path: act rows in decode layout
  if (T <= kDecodeMaxTokens) o = align256(o + A * dec_row_floats(I) * 4);
  L.xp = o;       o = align256(o + A * (size_t)H * 2);
  L.act16 = o;    o = align256(o + A * (size_t)I * 2);
  L.act16lo = o;  o = align256(o + A * (size_t)I * 2);
  L.outacc = o;   o = align256(o + (size_t)T * H * 4);
  L.tiles = o;    o = align256(o + ((size_t)E + A + 1) * 16);
  L.total = o;
  return L;
}

// ---- kernel parameter blocks
struct RouteParams {
  const void* x;          // [T, H] 16-bit
  const void* router_w;   // [H, E] 16-bit
  const float* bias;      // [E] or null
  int T, H, E, k, split, rows_per_split;
  float* topk_w;          // [T*k] workspace
  int32_t* topk_ids;      // [T*k] workspace
  float* user_w;          // optional user copies
  int32_t* user_ids;
  int32_t* offsets;       // [E+1] workspace
  int32_t* user_offsets;
  int32_t* active;        // [E+2] workspace: count, ids...
  int32_t* perm;          // [T*k] workspace
  int32_t* user_perm;
  uint32_t* ctl;          // control block
  int gate_sigmoid;       // 0: softmax over the E logits; 1: independent sigmoid per logit
};

// Decode kernel (weights streamed through shared memory by bulk copies).
enum DecodeMode { kModeGateUp = 0, kModeDown = 1, kModeDense = 2 };

struct DecodeParams {
  // matrices: mat 0 = gate / down / dense, mat 1 = up (gate-up only)
  const uint8_t* w[2];
  const void* s[2];
  const uint8_t* z[2];
  int N, K, bs, nb;        // rows per expert matrix, reduction length, block size
  int E, k, T;
  // routing (workspace); dense mode ignores these
  const int32_t* active;   // [0] = D, [1..D] = expert ids
  const int32_t* offsets;  // [E+1]
  const int32_t* perm;     // [T*k]
  const float* topk_w;     // [T*k]
  // down: act rows in decode layout (fp32)
  const float* src;
  int src_row_floats;
  // gate-up / dense: raw 16-bit x [T, K]
  const void* x16;
  // outputs
  float* act_out;          // gate-up: [T*k][dec_row_floats(N)]
  int act_row_floats;
  void* out;               // down / dense: [T, N] 16-bit
  int accumulate;
  // stage ring
  int rows_per_cta_max;
  uint32_t slot_base;  // byte offset of the stage ring in shared memory
  int nslots;
  uint32_t* ctl;
};

// Fused decode layer (router + gate-up + down in one launch, T <= kTokGroup):
// the gate-up and down views of the weights plus the router.
struct FusedParams {
  DecodeParams g, d;
  const void* x;          // [T, H] 16-bit
  const void* router_w;   // [H, E] 16-bit
  const float* bias;      // [E] or null
  int gate_sigmoid;
  int rps;                // router rows per split
  float* ws_w;            // workspace routing copies (written by CTA 0)
  int32_t* ws_ids;
  int32_t* ws_offsets;
  int32_t* ws_active;
  int32_t* ws_perm;
  float* user_w;          // optional user copies of the top-k
  int32_t* user_ids;
  long long* acc;         // [T][H] int64 fixed-point output accumulator (control block)
};

// Prefill path (grouped GEMM on the tensor cores).  The token tile table
// holds 4 ints per tile: expert, first sorted assignment, assignments.
struct PrefillParams {
  const uint8_t* w[3];      // gate, up, down packed codes [E, N, K/2]
  const void* s[3];         // block scales [E, N, K/bs]
  const uint8_t* z[3];      // zero points [E, N, K/bs] or null
  int T, H, I, E, k, bs, lbs;  // lbs = log2(bs)
  const int32_t* offsets;   // [E+1] workspace
  const int32_t* perm;      // [T*k] workspace: sorted -> assignment t*k+j
  const float* topk_w;      // [T*k] workspace
  uint16_t* xp;             // [T*k, H] gathered, K-permuted tokens
  uint16_t* act;            // [T*k, I] SwiGLU output (high part), K-permuted
  uint16_t* act_lo;         // [T*k, I] SwiGLU output minus its high part (split path)
  float* out_acc;           // [T, H] fp32 accumulator
  int32_t* tiles;           // [ntiles][4]
  uint32_t* ctl;            // control block (status, tile count)
  int accumulate;
  int x_to_f16;             // gather / dense setup convert bf16 x to the fp16 operands
  int nst, nsz, npk;        // operand stages, tile scale buffers, packed-code slots (per GEMM launch)
};

}  // namespace qmoe
