// layout.h -- internal (non-ABI) definitions shared by host launchers and
// kernels: device status bits, the workspace map, the decode-path
// activation layout and the kernel parameter blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define QMOE_HD __host__ __device__ __forceinline__
#else
#define QMOE_HD inline
#endif

namespace qmoe {

// ---- device status word bits (workspace control block, word 0)
constexpr uint32_t QMOE_ST_TIMEOUT = 1u;  // a bounded wait ran out
constexpr uint32_t QMOE_ST_INDEX = 2u;    // an index check failed

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;

// ---- control block (first kCtlBytes of the workspace, zeroed by init)
constexpr int kCtlStatus = 0;         // u32 sticky status bits
constexpr int kCtlGroupTicket = 1;    // u32 router: CTAs done with top-k
constexpr int kCtlTileTicket0 = 16;   // u32[kMaxRouteTiles] router split tickets
constexpr int kMaxRouteTiles = 64;
constexpr size_t kCtlBytes = 1024;

// ---- router tiling
constexpr int kRouteTokens = 8;       // tokens per router CTA (one warp each)
constexpr int kRouteThreads = 256;
constexpr int kMaxSplit = 16;         // H-splits for small T

// ---- decode path
constexpr int kDecodeMaxTokens = 16;  // T at or below: GEMV path
constexpr int kTokGroup = 4;          // tokens per decode stage

// Decode-path activation layout.  A K-long fp32 row is stored so that lane l
// of a warp, processing 16-byte weight chunk c = 32*s + l (32 elements), finds
// its 32 activations as 8 float4 at ((s*8 + f)*32 + l), f = 0..7: consecutive
// lanes read consecutive float4 (no bank conflicts).  Element i is
// pre-multiplied by 16^-(i mod 4): the kernels turn nibble j of a 16-bit
// half-word into (q - zp) * 16^j exactly, and this power of two undoes it.
QMOE_HD int dec_row_floats(int K) { return ((K + 1023) / 1024) * 1024; }
QMOE_HD int dec_index(int i) {
  return ((((i >> 10) * 8 + ((i & 31) >> 2)) * 32 + ((i >> 5) & 31)) << 2) + (i & 3);
}
QMOE_HD float dec_prescale(int i) {
  const int j = i & 3;
  return j == 0 ? 1.0f : (j == 1 ? 0.0625f : (j == 2 ? 0.00390625f : 0.000244140625f));
}

// ---- workspace map (byte offsets, each region 256-byte aligned)
struct WsLayout {
  size_t ctl, ids, w, offsets, active, perm, partial, act, xp, act16, outacc, tiles, total;
};

QMOE_HD size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

QMOE_HD int route_split(int T) {
  const int tiles = (T + kRouteTokens - 1) / kRouteTokens;
  if (tiles > 8) return 1;
  int s = kMaxSplit / tiles;
  return s < 1 ? 1 : s;
}

QMOE_HD WsLayout ws_layout(int T, int H, int I, int E, int k) {
  WsLayout L;
  const size_t A = (size_t)T * k;
  const int tiles = (T + kRouteTokens - 1) / kRouteTokens;
  size_t o = 0;
  L.ctl = o;      o = align256(o + kCtlBytes);
  L.ids = o;      o = align256(o + A * 4);
  L.w = o;        o = align256(o + A * 4);
  L.offsets = o;  o = align256(o + (size_t)(E + 1) * 4);
  L.active = o;   o = align256(o + (size_t)(E + 2) * 4);  // [0] = count, [1..] = ids
  L.perm = o;     o = align256(o + A * 4);
  L.partial = o;
  if (route_split(T) > 1) o = align256(o + (size_t)route_split(T) * tiles * kRouteTokens * E * 4);
  L.act = o;  // decode path: act rows in decode layout
  if (T <= kDecodeMaxTokens) o = align256(o + A * dec_row_floats(I) * 4);
  L.xp = o;       o = align256(o + A * (size_t)H * 2);
  L.act16 = o;    o = align256(o + A * (size_t)I * 2);
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
  float* partial;         // [split][tiles*8][E] when split > 1
  uint32_t* ctl;          // control block
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

}  // namespace qmoe
