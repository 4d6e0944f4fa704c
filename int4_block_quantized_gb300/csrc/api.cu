// api.cu -- the C ABI (include/qmoe.h): argument checks on the host, the
// workspace map, and the launch order of each entry point.  No allocation,
// no synchronisation (except qmoe_get_device_status, documented blocking).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "launch.h"
#include "qmoe.h"

using namespace qmoe;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// sm_103 (compute capability 10.3) only; cached per device
int check_device() {
  static int ok_cache[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return QMOE_ERR_UNSUPPORTED;
  if (!ok_cache[dev]) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QMOE_ERR_CUDA;
    ok_cache[dev] = (maj == 10 && min == 3) ? 1 : 2;
  }
  return ok_cache[dev] == 1 ? QMOE_OK : QMOE_ERR_UNSUPPORTED;
}

bool valid_dtype(int d) { return d == QMOE_F16 || d == QMOE_BF16; }
bool valid_bs(int bs) { return bs == 32 || bs == 64 || bs == 128; }

int check_qweight(const qmoe_qweight& q, int N, int K, int bs) {
  if (!q.w || !q.scales) return QMOE_ERR_INVALID_ARG;
  if (N < 1 || K < 32 || K % 32 || K % bs) return QMOE_ERR_INVALID_ARG;
  if (!aligned(q.w, 16) || !aligned(q.scales, 2)) return QMOE_ERR_INVALID_ARG;
  return QMOE_OK;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QMOE_OK;
  g_last_cuda_error = e;
  if (e == cudaErrorInvalidValue) return QMOE_ERR_UNSUPPORTED;  // shape outside the kernel plans
  return QMOE_ERR_CUDA;
}

struct Ws {
  WsLayout L;
  uint8_t* base;
  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

int check_route_args(const void* x, const void* router_w, int act_dtype, int T, int H, int E, int k) {
  if (!x || !router_w) return QMOE_ERR_INVALID_ARG;
  if (!valid_dtype(act_dtype)) return QMOE_ERR_INVALID_ARG;
  if (T < 1 || H < 1 || E < 1 || k < 1 || k > E) return QMOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || k > kMaxTopk) return QMOE_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(router_w, 2)) return QMOE_ERR_INVALID_ARG;
  if ((long long)T * k > (1LL << 30)) return QMOE_ERR_UNSUPPORTED;
  // router CTA shared memory: x slice, staged router rows, partial logits
  if (route_smem_bytes(T, H, E, k) > 200 * 1024) return QMOE_ERR_UNSUPPORTED;
  return QMOE_OK;
}

int enqueue_route(const Ws& ws, const void* x, const void* router_w, int act_dtype,
                  const float* bias, int T, int H, int E, int k, float* user_w,
                  int32_t* user_ids, int32_t* user_offsets, int32_t* user_perm, cudaStream_t st,
                  bool pdl = true, int gate_sigmoid = 0) {
  RouteParams p = {};
  p.gate_sigmoid = gate_sigmoid;
  p.x = x;
  p.router_w = router_w;
  p.bias = bias;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k = k;
  p.split = route_split(T);
  p.rows_per_split = route_rows_per_split(H);
  p.topk_w = ws.at<float>(ws.L.w);
  p.topk_ids = ws.at<int32_t>(ws.L.ids);
  p.user_w = user_w;
  p.user_ids = user_ids;
  p.offsets = ws.at<int32_t>(ws.L.offsets);
  p.user_offsets = user_offsets;
  p.active = ws.at<int32_t>(ws.L.active);
  p.perm = ws.at<int32_t>(ws.L.perm);
  p.user_perm = user_perm;
  p.ctl = ws.at<uint32_t>(ws.L.ctl);
  return cuda_status(launch_route(p, act_dtype, st, pdl));
}

}  // namespace

extern "C" {

const char* qmoe_status_string(int status) {
  switch (status) {
    case QMOE_OK: return "ok";
    case QMOE_ERR_INVALID_ARG: return "invalid argument";
    case QMOE_ERR_UNSUPPORTED: return "unsupported device or shape";
    case QMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case QMOE_ERR_CUDA: return "CUDA runtime error";
    case QMOE_ERR_TIMEOUT: return "device wait timed out";
    case QMOE_ERR_DEVICE_CHECK: return "device index check failed";
    default: return "unknown status";
  }
}

const char* qmoe_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

size_t qmoe_workspace_size(int T, int H, int I, int E, int k) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  return ws_layout(T, H, I, E, k).total;
}

int qmoe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kCtlBytes) return QMOE_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, kCtlBytes, (cudaStream_t)stream) == cudaSuccess ? QMOE_OK
                                                                                     : QMOE_ERR_CUDA;
}

int qmoe_workspace_set_diagnostics(void* workspace, size_t workspace_bytes, uint32_t wait_limit_kilocycles,
                                   uint32_t flags, void* stream) {
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < kCtlBytes) return QMOE_ERR_WORKSPACE;
  if (flags & ~(uint32_t)QMOE_DIAG_STALL_GEMM) return QMOE_ERR_INVALID_ARG;
  static_assert(kCtlDiag == kCtlWaitLimit + 1, "diagnostic words are adjacent");
  const uint32_t words[2] = {wait_limit_kilocycles, flags};
  return cudaMemcpyAsync(static_cast<uint32_t*>(workspace) + kCtlWaitLimit, words, sizeof(words),
                         cudaMemcpyHostToDevice, (cudaStream_t)stream) == cudaSuccess
             ? QMOE_OK
             : QMOE_ERR_CUDA;
}

int qmoe_route(const void* x, const void* router_w, int act_dtype, const float* router_bias, int T,
               int H, int E, int k, float* topk_w, int32_t* topk_ids, int32_t* expert_offsets,
               int32_t* perm, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_route_args(x, router_w, act_dtype, T, H, E, k);
  if (rc) return rc;
  if (!topk_w || !topk_ids) return QMOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, 32, E, k);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return QMOE_ERR_WORKSPACE;
  if ((rc = check_device())) return rc;
  Ws ws{L, static_cast<uint8_t*>(workspace)};
  return enqueue_route(ws, x, router_w, act_dtype, router_bias, T, H, E, k, topk_w, topk_ids,
                       expert_offsets, perm, (cudaStream_t)stream);
}

int matmul_nbits(const void* x, int act_dtype, const uint8_t* w, const void* scales,
                 int scale_dtype, const uint8_t* zp, int M, int N, int K, int block_size, void* y,
                 void* stream) {
  if (!x || !y || !valid_dtype(act_dtype) || !valid_dtype(scale_dtype)) return QMOE_ERR_INVALID_ARG;
  if (!valid_bs(block_size) || M < 1) return QMOE_ERR_INVALID_ARG;
  qmoe_qweight q{w, scales, zp};
  int rc = check_qweight(q, N, K, block_size);
  if (rc) return rc;
  if (!aligned(x, 16) || !aligned(y, 2)) return QMOE_ERR_INVALID_ARG;
  if ((rc = check_device())) return rc;
  // tokens per launch: as many (<= 16) as the kernel's shared-memory plan holds
  int chunk = M < kDecodeMaxTokens ? M : kDecodeMaxTokens;
  while (chunk > 0 && !decode_fits(kModeDense, chunk, N, K, block_size, zp != nullptr, 1)) --chunk;
  if (chunk == 0) return QMOE_ERR_UNSUPPORTED;
  for (int m0 = 0; m0 < M; m0 += chunk) {
    const int mt = (M - m0) < chunk ? (M - m0) : chunk;
    DecodeParams p = {};
    p.w[0] = w;
    p.s[0] = scales;
    p.z[0] = zp;
    p.N = N;
    p.K = K;
    p.bs = block_size;
    p.nb = K / block_size;
    p.E = 1;
    p.k = 1;
    p.T = mt;
    p.x16 = static_cast<const uint16_t*>(x) + (size_t)m0 * K;
    p.out = static_cast<uint16_t*>(y) + (size_t)m0 * N;
    p.src_row_floats = dec_row_floats(K);
    rc = cuda_status(launch_decode(p, kModeDense, act_dtype, scale_dtype, zp != nullptr,
                                   (cudaStream_t)stream, false));
    if (rc) return rc;
  }
  return QMOE_OK;
}

int matmul_nbits_ex(const void* x, int act_dtype, const uint8_t* w, const void* scales, int scale_dtype,
                    const uint8_t* zp, int M, int N, int K, int block_size, void* y, int path, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (path != QMOE_PATH_AUTO && path != QMOE_PATH_DECODE && path != QMOE_PATH_PREFILL) return QMOE_ERR_INVALID_ARG;
  if (path == QMOE_PATH_DECODE || (path == QMOE_PATH_AUTO && M <= kDecodeMaxTokens))
    return matmul_nbits(x, act_dtype, w, scales, scale_dtype, zp, M, N, K, block_size, y, stream);
  if (!x || !y || !valid_dtype(act_dtype) || !valid_dtype(scale_dtype)) return QMOE_ERR_INVALID_ARG;
  if (!valid_bs(block_size) || M < 1) return QMOE_ERR_INVALID_ARG;
  qmoe_qweight q{w, scales, zp};
  int rc = check_qweight(q, N, K, block_size);
  if (rc) return rc;
  if (!aligned(x, 16) || !aligned(y, 16)) return QMOE_ERR_INVALID_ARG;
  if ((long long)M * K > (1LL << 31)) return QMOE_ERR_UNSUPPORTED;
  // the GEMM's view: one expert with N rows and a K-long reduction, M tokens
  const WsLayout L = ws_layout(M, N, K, 1, 1);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return QMOE_ERR_WORKSPACE;
  if (!dense_fits(N, K, block_size, act_dtype, scale_dtype, zp != nullptr) || !aligned(scales, 16) ||
      !aligned(zp, 16))
    return QMOE_ERR_UNSUPPORTED;
  if ((rc = check_device())) return rc;
  Ws ws{L, static_cast<uint8_t*>(workspace)};
  PrefillParams p = {};
  p.w[2] = w;
  p.s[2] = scales;
  p.z[2] = zp;
  p.T = M; p.H = N; p.I = K; p.E = 1; p.k = 1; p.bs = block_size;
  p.lbs = block_size == 32 ? 5 : (block_size == 64 ? 6 : 7);
  p.offsets = ws.at<int32_t>(L.offsets);
  p.perm = ws.at<int32_t>(L.perm);
  p.topk_w = ws.at<float>(L.w);
  p.act = ws.at<uint16_t>(L.act16);
  p.act_lo = nullptr;  // x is exact in one operand
  p.x_to_f16 = prefill_x_to_f16(act_dtype, scale_dtype);
  p.out_acc = ws.at<float>(L.outacc);
  p.tiles = ws.at<int32_t>(L.tiles);
  p.ctl = ws.at<uint32_t>(L.ctl);
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = cuda_status(launch_dense_setup(p, x, st, true)))) return rc;
  if ((rc = cuda_status(launch_prefill_gemm(p, 1, act_dtype, scale_dtype, true, st, true)))) return rc;
  return cuda_status(launch_prefill_convert(p, y, act_dtype, st, true));
}

}  // extern "C"

namespace {

// The one-kernel decode layer: the default decode path at T = 1, where it
// is faster than three kernels; at T = 2..4 three kernels stream the larger
// weight volume faster (measured on GB300), so there it runs only when
// asked for (QMOE_PATH_DECODE_FUSED).
constexpr int kFusedAutoMaxTokens = 1;
// True if the decode layer at these sizes can run as the one cooperative kernel.
bool fused_fits(int T, int H, int I, int E, int k, int block_size, int act_dtype, int scale_dtype, bool zgu,
                bool zd) {
  if (T > kTokGroup || zgu != zd) return false;
  FusedParams f = {};
  f.g.T = T; f.g.K = H; f.g.N = I; f.g.E = E; f.g.k = k; f.g.bs = block_size;
  return launch_fused(f, act_dtype, scale_dtype, zgu, nullptr, false, true) == cudaSuccess;
}

int forward_impl(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                 qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                 int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                 int32_t* topk_ids_out, int accumulate, int path, void* workspace,
                 size_t workspace_bytes, void* stream, void* const* events, int n_events,
                 int gate_sigmoid = 0) {
  int rc = check_route_args(x, router_w, act_dtype, T, H, E, k);
  if (rc) return rc;
  if (!out || !aligned(out, 16) || !valid_dtype(scale_dtype) || !valid_bs(block_size))
    return QMOE_ERR_INVALID_ARG;
  if ((rc = check_qweight(gate, I, H, block_size)) || (rc = check_qweight(up, I, H, block_size)) ||
      (rc = check_qweight(down, H, I, block_size)))
    return rc;
  if ((gate.zp == nullptr) != (up.zp == nullptr)) return QMOE_ERR_INVALID_ARG;
  if (path < QMOE_PATH_AUTO || path > QMOE_PATH_DECODE_FUSED || path == 3) return QMOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, I, E, k);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return QMOE_ERR_WORKSPACE;
  if ((rc = check_device())) return rc;
  const bool zgu = gate.zp != nullptr, zd = down.zp != nullptr;
  const bool dec_ok = T <= kDecodeMaxTokens && decode_fits(kModeGateUp, T, I, H, block_size, zgu, k) &&
                      decode_fits(kModeDown, T, H, I, block_size, zd, k);
  // the grouped GEMM copies whole rows of scales / zero points in bulk: 16-byte aligned bases
  const bool pre_ok = prefill_fits(H, I, block_size, act_dtype, scale_dtype, zgu, zd) && aligned(gate.scales, 16) &&
                      aligned(up.scales, 16) && aligned(down.scales, 16) && aligned(gate.zp, 16) &&
                      aligned(up.zp, 16) && aligned(down.zp, 16);
  const bool split_decode = path == QMOE_PATH_DECODE_SPLIT;
  const bool force_fused = path == QMOE_PATH_DECODE_FUSED;
  if (split_decode || force_fused) path = QMOE_PATH_DECODE;
  if (path == QMOE_PATH_AUTO)
    path = dec_ok && (T <= QMOE_AUTO_DECODE_MAX_TOKENS || !pre_ok) ? QMOE_PATH_DECODE : QMOE_PATH_PREFILL;
  if (path == QMOE_PATH_DECODE && !dec_ok) return QMOE_ERR_UNSUPPORTED;
  if (path == QMOE_PATH_PREFILL && !pre_ok) return QMOE_ERR_UNSUPPORTED;

  Ws ws{L, static_cast<uint8_t*>(workspace)};
  cudaStream_t st = (cudaStream_t)stream;
  // profiling: an event before the first kernel and after each kernel; the
  // kernels then run back to back without programmatic overlap
  const bool pdl = events == nullptr;
  int ev_i = 0;
  auto mark = [&]() -> int {
    if (events && ev_i < n_events && events[ev_i]) {
      // under stream capture the record must be external to become a graph
      // node that timing can read (a plain record only orders the capture);
      // outside capture the flag is not accepted
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing(st, &cs);
      if (e == cudaSuccess)
        e = cs == cudaStreamCaptureStatusActive
                ? cudaEventRecordWithFlags((cudaEvent_t)events[ev_i], st, cudaEventRecordExternal)
                : cudaEventRecord((cudaEvent_t)events[ev_i], st);
      if (e != cudaSuccess) return cuda_status(e);
    }
    ++ev_i;
    return QMOE_OK;
  };
  DecodeParams g = {};
  g.w[0] = gate.w; g.s[0] = gate.scales; g.z[0] = gate.zp;
  g.w[1] = up.w;   g.s[1] = up.scales;   g.z[1] = up.zp;
  g.N = I; g.K = H; g.bs = block_size; g.nb = H / block_size;
  g.E = E; g.k = k; g.T = T;
  g.active = ws.at<int32_t>(L.active);
  g.offsets = ws.at<int32_t>(L.offsets);
  g.perm = ws.at<int32_t>(L.perm);
  g.topk_w = ws.at<float>(L.w);
  g.x16 = x;
  g.act_out = ws.at<float>(L.act);
  g.act_row_floats = dec_row_floats(I);
  g.src_row_floats = dec_row_floats(H);
  g.ctl = ws.at<uint32_t>(L.ctl);
  DecodeParams d = g;
  d.w[0] = down.w; d.s[0] = down.scales; d.z[0] = down.zp;
  d.w[1] = nullptr; d.s[1] = nullptr; d.z[1] = nullptr;
  d.N = H; d.K = I; d.nb = I / block_size;
  d.src = ws.at<float>(L.act);
  d.src_row_floats = dec_row_floats(I);
  d.x16 = nullptr;
  d.act_out = nullptr;
  d.out = out;
  d.accumulate = accumulate;

  const bool fused = path == QMOE_PATH_DECODE && !split_decode && (force_fused || T <= kFusedAutoMaxTokens) &&
                     fused_fits(T, H, I, E, k, block_size, act_dtype, scale_dtype, zgu, zd);
  if (force_fused && !fused) return QMOE_ERR_UNSUPPORTED;
  if (fused) {
    // the whole layer in one cooperative kernel, if its plan fits
    FusedParams f = {};
    f.g = g;
    f.d = d;
    f.x = x;
    f.router_w = router_w;
    f.bias = router_bias;
    f.gate_sigmoid = gate_sigmoid;
    f.rps = route_rows_per_split(H);
    f.ws_w = ws.at<float>(L.w);
    f.ws_ids = ws.at<int32_t>(L.ids);
    f.ws_offsets = ws.at<int32_t>(L.offsets);
    f.ws_active = ws.at<int32_t>(L.active);
    f.ws_perm = ws.at<int32_t>(L.perm);
    f.user_w = topk_w_out;
    f.user_ids = topk_ids_out;
    f.acc = ws.at<long long>(L.ctl + kCtlAccOffset);
    if ((rc = mark())) return rc;
    if ((rc = cuda_status(launch_fused(f, act_dtype, scale_dtype, zgu, st, pdl, false)))) return rc;
    return mark();
  }

  if ((rc = mark())) return rc;
  rc = enqueue_route(ws, x, router_w, act_dtype, router_bias, T, H, E, k, topk_w_out, topk_ids_out,
                     nullptr, nullptr, st, pdl, gate_sigmoid);
  if (rc || (rc = mark())) return rc;

  if (path == QMOE_PATH_PREFILL) {
    PrefillParams p = {};
    const qmoe_qweight* q[3] = {&gate, &up, &down};
    for (int m = 0; m < 3; ++m) {
      p.w[m] = q[m]->w;
      p.s[m] = q[m]->scales;
      p.z[m] = q[m]->zp;
    }
    p.T = T; p.H = H; p.I = I; p.E = E; p.k = k; p.bs = block_size;
    p.lbs = block_size == 32 ? 5 : (block_size == 64 ? 6 : 7);
    p.offsets = ws.at<int32_t>(L.offsets);
    p.perm = ws.at<int32_t>(L.perm);
    p.topk_w = ws.at<float>(L.w);
    p.xp = ws.at<uint16_t>(L.xp);
    p.act = ws.at<uint16_t>(L.act16);
    p.act_lo = ws.at<uint16_t>(L.act16lo);
    p.x_to_f16 = prefill_x_to_f16(act_dtype, scale_dtype);
    p.out_acc = ws.at<float>(L.outacc);
    p.tiles = ws.at<int32_t>(L.tiles);
    p.ctl = ws.at<uint32_t>(L.ctl);
    p.accumulate = accumulate;
    rc = cuda_status(launch_prefill_permute(p, x, act_dtype, st, pdl));
    if (rc || (rc = mark())) return rc;
    rc = cuda_status(launch_prefill_gemm(p, 0, act_dtype, scale_dtype, false, st, pdl));
    if (rc || (rc = mark())) return rc;
    rc = cuda_status(launch_prefill_gemm(p, 1, act_dtype, scale_dtype, false, st, pdl));
    if (rc || (rc = mark())) return rc;
    rc = cuda_status(launch_prefill_convert(p, out, act_dtype, st, pdl));
    if (rc) return rc;
    return mark();
  }

  rc = cuda_status(launch_decode(g, kModeGateUp, act_dtype, scale_dtype, zgu, st, pdl));
  if (rc || (rc = mark())) return rc;
  rc = cuda_status(launch_decode(d, kModeDown, act_dtype, scale_dtype, zd, st, pdl));
  if (rc) return rc;
  return mark();
}

}  // namespace

extern "C" {

int qmoe_forward_ex(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                    qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                    int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                    int32_t* topk_ids_out, int accumulate, int path, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return forward_impl(x, act_dtype, router_w, router_bias, gate, up, down, scale_dtype, T, H, I, E,
                      k, block_size, out, topk_w_out, topk_ids_out, accumulate, path, workspace,
                      workspace_bytes, stream, nullptr, 0);
}

int qmoe_forward_kernels(int T, int H, int I, int E, int k, int block_size, int act_dtype, int scale_dtype,
                         int gate_up_has_zp, int down_has_zp, int path) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1 || k > E || E > kMaxExperts || k > kMaxTopk || !valid_dtype(act_dtype) ||
      !valid_dtype(scale_dtype) || !valid_bs(block_size) || path < QMOE_PATH_AUTO || path > QMOE_PATH_DECODE_FUSED ||
      path == 3)
    return -QMOE_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc) return -rc;
  const bool zgu = gate_up_has_zp != 0, zd = down_has_zp != 0;
  const bool dec_ok = T <= kDecodeMaxTokens && decode_fits(kModeGateUp, T, I, H, block_size, zgu, k) &&
                      decode_fits(kModeDown, T, H, I, block_size, zd, k);
  const bool pre_ok = prefill_fits(H, I, block_size, act_dtype, scale_dtype, zgu, zd);
  if (path == QMOE_PATH_AUTO)
    path = dec_ok && (T <= QMOE_AUTO_DECODE_MAX_TOKENS || !pre_ok) ? QMOE_PATH_DECODE : QMOE_PATH_PREFILL;
  if (path == QMOE_PATH_DECODE || path == QMOE_PATH_DECODE_SPLIT || path == QMOE_PATH_DECODE_FUSED) {
    if (!dec_ok) return -QMOE_ERR_UNSUPPORTED;
    const bool fits = fused_fits(T, H, I, E, k, block_size, act_dtype, scale_dtype, zgu, zd);
    if (path == QMOE_PATH_DECODE_FUSED) return fits ? 1 : -QMOE_ERR_UNSUPPORTED;
    if (path == QMOE_PATH_DECODE && T <= kFusedAutoMaxTokens && fits) return 1;
    return 3;
  }
  return pre_ok ? 5 : -QMOE_ERR_UNSUPPORTED;
}

int qmoe_forward_profiled(const void* x, int act_dtype, const void* router_w,
                          const float* router_bias, qmoe_qweight gate, qmoe_qweight up,
                          qmoe_qweight down, int scale_dtype, int T, int H, int I, int E, int k,
                          int block_size, void* out, int path, void* workspace,
                          size_t workspace_bytes, void* stream, void* const* events,
                          int n_events) {
  if (!events || n_events < 1) return QMOE_ERR_INVALID_ARG;
  return forward_impl(x, act_dtype, router_w, router_bias, gate, up, down, scale_dtype, T, H, I, E,
                      k, block_size, out, nullptr, nullptr, 0, path, workspace, workspace_bytes,
                      stream, events, n_events);
}

int qmoe_forward(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                 qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                 int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                 int32_t* topk_ids_out, int accumulate, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return qmoe_forward_ex(x, act_dtype, router_w, router_bias, gate, up, down, scale_dtype, T, H, I,
                         E, k, block_size, out, topk_w_out, topk_ids_out, accumulate,
                         QMOE_PATH_AUTO, workspace, workspace_bytes, stream);
}

int qmoe_shared_expert(const void* x, int act_dtype, const void* shared_gate_w, qmoe_qweight gate,
                       qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T, int H, int I,
                       int block_size, void* out, int accumulate, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!shared_gate_w) return QMOE_ERR_INVALID_ARG;
  // the layer with one expert, top-1, the gate vector as its [H, 1] router
  // and a sigmoid in place of the softmax
  return forward_impl(x, act_dtype, shared_gate_w, nullptr, gate, up, down, scale_dtype, T, H, I, 1, 1,
                      block_size, out, nullptr, nullptr, accumulate, QMOE_PATH_AUTO, workspace,
                      workspace_bytes, stream, nullptr, 0, 1);
}

int qmoe_dequant(const uint8_t* w, const void* scales, int scale_dtype, const uint8_t* zp, int N,
                 int K, int block_size, float* out, void* stream) {
  if (!out || !valid_dtype(scale_dtype) || !valid_bs(block_size)) return QMOE_ERR_INVALID_ARG;
  qmoe_qweight q{w, scales, zp};
  int rc = check_qweight(q, N, K, block_size);
  if (rc) return rc;
  if (!aligned(out, 16)) return QMOE_ERR_INVALID_ARG;
  if ((rc = check_device())) return rc;
  return cuda_status(launch_dequant(w, scales, scale_dtype, zp, N, K, block_size, out,
                                    (cudaStream_t)stream));
}

int qmoe_rmsnorm(const void* x, void* out, int act_dtype, int T, int H, float eps, void* stream) {
  if (!x || !out || !valid_dtype(act_dtype) || T < 1 || H < 1 || !(eps >= 0.f))
    return QMOE_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(out, 2)) return QMOE_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc) return rc;
  return cuda_status(launch_rmsnorm(x, out, act_dtype, T, H, eps, (cudaStream_t)stream));
}

int qmoe_gptq_zero_offset(const int32_t* qzeros, size_t n_words, int32_t* offset_out, void* stream) {
  if (!qzeros || !offset_out || n_words < 1 || !aligned(qzeros, 4) || !aligned(offset_out, 4))
    return QMOE_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc) return rc;
  return cuda_status(launch_gptq_zero_offset(qzeros, n_words, offset_out, (cudaStream_t)stream));
}

int qmoe_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int E, int K, int N,
                     int block_size, int zero_offset, const int32_t* zero_offset_dev, uint8_t* w_out,
                     void* scales_out, uint8_t* zp_out, uint32_t* status_dev, void* stream) {
  if (!qweight || !scales || !w_out || !scales_out || (qzeros == nullptr) != (zp_out == nullptr))
    return QMOE_ERR_INVALID_ARG;
  if (E < 1 || E > 65535 || N < 8 || N % 8 || K < 32 || K % 32 || !valid_bs(block_size) || K % block_size)
    return QMOE_ERR_INVALID_ARG;
  if (zero_offset != 0 && zero_offset != 1) return QMOE_ERR_INVALID_ARG;
  if (!aligned(qweight, 4) || !aligned(qzeros, 4) || !aligned(w_out, 4) || !aligned(scales, 2) ||
      !aligned(scales_out, 2) || !aligned(zero_offset_dev, 4) || !aligned(status_dev, 4))
    return QMOE_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc) return rc;
  return cuda_status(launch_repack_gptq(qweight, qzeros, scales, E, K, N, block_size, zero_offset, zero_offset_dev,
                                        w_out, scales_out, zp_out, status_dev, (cudaStream_t)stream));
}

int qmoe_unpack_zero_points(const uint8_t* zp_packed, int rows, int nb, uint8_t* zp_out, void* stream) {
  if (!zp_packed || !zp_out || rows < 1 || nb < 1) return QMOE_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc) return rc;
  return cuda_status(launch_unpack_zp(zp_packed, zp_out, rows, nb, (cudaStream_t)stream));
}

int qmoe_get_device_status(void* workspace, uint32_t* bits_out, void* stream) {
  if (!workspace) return QMOE_ERR_WORKSPACE;
  uint32_t bits = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(bits), st) != cudaSuccess)
    return QMOE_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits & QMOE_ST_TIMEOUT) return QMOE_ERR_TIMEOUT;
  if (bits & (QMOE_ST_INDEX | QMOE_ST_RANGE)) return QMOE_ERR_DEVICE_CHECK;
  return QMOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// qmoe_forward_noalloc: qmoe_forward with the workspace in a static device
// array instead of caller memory.  For callers that cannot hand the library
// device memory: a plain C host program that links only this library and
// has no device allocator, or a plugin interface whose per-call hook gets
// no workspace argument and must not call cudaMalloc (which synchronises
// the device and so stalls every other stream in the process).

namespace {

// 2 MiB: the whole layout of qmoe_workspace_size for the Qwen1.5-MoE-A2.7B
// layer shape (H = 2048, I = 1408, E = 60, k = 4) at T <= 16 is ~1.3 MB.
// Zero-initialised at module load, which is what the control block (status
// word, counters, the fused decode layer's accumulator) must start as; every
// call leaves the counters and the accumulator back at zero.
constexpr size_t kNoAllocScratchBytes = QMOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// device address of the scratch array, looked up once per device
void* noalloc_scratch_ptr(int* rc) {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *rc = QMOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *rc = cuda_status(e);
      return nullptr;
    }
    ptrs[dev] = p;
  }
  *rc = QMOE_OK;
  return ptrs[dev];
}

}  // namespace

extern "C" {

int qmoe_forward_noalloc(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                         qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T, int H,
                         int I, int E, int k, int block_size, void* out, float* topk_w_out,
                         int32_t* topk_ids_out, int accumulate, void* stream) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1) return QMOE_ERR_INVALID_ARG;
  if (ws_layout(T, H, I, E, k).total > kNoAllocScratchBytes) return QMOE_ERR_UNSUPPORTED;
  int rc = QMOE_OK;
  void* scratch = noalloc_scratch_ptr(&rc);
  if (!scratch) return rc;
  return forward_impl(x, act_dtype, router_w, router_bias, gate, up, down, scale_dtype, T, H, I, E, k,
                      block_size, out, topk_w_out, topk_ids_out, accumulate, QMOE_PATH_AUTO, scratch,
                      kNoAllocScratchBytes, stream, nullptr, 0);
}

int qmoe_noalloc_status(uint32_t* bits_out, void* stream) {
  int rc = QMOE_OK;
  void* scratch = noalloc_scratch_ptr(&rc);
  if (!scratch) return rc;
  // the status word is the first word of the scratch's control block
  return qmoe_get_device_status(scratch, bits_out, stream);
}

}  // extern "C"
