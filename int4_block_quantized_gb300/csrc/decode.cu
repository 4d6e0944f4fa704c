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
#include "decode_core.cuh"

namespace qmoe {

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

}  // namespace qmoe
