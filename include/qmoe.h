/*
 * qmoe.h -- C ABI of the INT4 block-quantized mixture-of-experts FFN layer
 * library for NVIDIA GB300 (sm_103a).
 *
 * The layer (source: "Qwen MoE BringUp", IREE ONNX Runtime EP issue #34,
 * the Qwen1.5-MoE-A2.7B-Chat INT4 IR Guide, section 3 "MoE Block"):
 *   logits = x . router_w (+ router_bias)          (Router: gate linear)
 *   p      = softmax(logits) over all E experts     (Router, kernel step 1)
 *   top-k  = the k largest p, best first            (Router, kernel step 2)
 *   for each chosen expert e of token t:
 *     g = x . Wg_e^T, u = x . Wu_e^T                (Expert Computation, step 4)
 *     act = g * sigmoid(g) * u                      (step 5, SwiGLU)
 *     y = act . Wd_e^T                              (step 6)
 *   out[t] = sum_j p[t, j] * y_j                    (step 7, not renormalised)
 * with every expert weight dequantised per DequantizeLinear with block_size
 * along the input dimension: w = (q - zp) * scale ("Qwen MoE BringUp",
 * local fix A1: extui -> uitofp -> subf -> mulf).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor pointer is a DEVICE pointer owned by the caller
 *   (cudaMalloc, torch, ...), on the current CUDA device, contiguous
 *   row-major.  The library never allocates, frees or copies host memory
 *   and never synchronises; all work is enqueued on `stream` (a
 *   cudaStream_t passed as void*, NULL = the legacy default stream).
 * Packed weights.  A projection with N outputs and K inputs, for all E
 *   experts, is three tensors:
 *     w      uint8  [E, N, K/2]   two uint4 codes per byte; element k of a
 *                                 row is in byte k/2, LOW nibble for even k
 *     scales fp16 or bf16 [E, N, K/block_size]
 *     zp     uint8  [E, N, K/block_size], values 0..15, or NULL meaning
 *                                 zero point 8 (signed symmetric int4)
 *   This is the IR guide's pre-transposed layout ([out, in], Optimization
 *   Opportunities item 5); gate/up have N = I, K = H; down has N = H, K = I.
 * Alignment.  x, out, router_w and every w must be 16-byte aligned; K must
 *   be a multiple of 32 and of block_size; block_size is 32, 64 or 128.
 * Errors.  Arguments are checked on the host before anything is enqueued;
 *   a bad argument returns QMOE_ERR_INVALID_ARG / QMOE_ERR_UNSUPPORTED /
 *   QMOE_ERR_WORKSPACE and enqueues nothing.  A failed launch returns
 *   QMOE_ERR_CUDA.  Conditions found on the device (a bounded wait that ran
 *   out) set bits in a status word kept in the workspace; read and clear it
 *   with qmoe_get_device_status.  No C++ exception crosses this ABI.
 * Device.  Compute capability 10.3 (sm_103a) only; any other device
 *   returns QMOE_ERR_UNSUPPORTED.  There is no CPU fallback.
 * Concurrency.  Calls that share a workspace must be ordered on one stream.
 */
#ifndef QMOE_H_
#define QMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QMOE_OK = 0,
  QMOE_ERR_INVALID_ARG = 1,  /* NULL / out-of-range / misaligned argument   */
  QMOE_ERR_UNSUPPORTED = 2,  /* valid but not supported (device, shape)     */
  QMOE_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required     */
  QMOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed        */
  QMOE_ERR_TIMEOUT = 5,      /* device status: a bounded wait ran out       */
  QMOE_ERR_DEVICE_CHECK = 6  /* device status: an index or range check failed */
} qmoe_status;

/* Bits of a device status word (qmoe_get_device_status's *bits_out). */
typedef enum {
  QMOE_ST_TIMEOUT = 1, /* a bounded wait ran out                                 -> QMOE_ERR_TIMEOUT */
  QMOE_ST_INDEX = 2,   /* an index check failed                                  -> QMOE_ERR_DEVICE_CHECK */
  QMOE_ST_RANGE = 4    /* a value outside a format's or accumulator's range       -> QMOE_ERR_DEVICE_CHECK */
} qmoe_status_bit;

typedef enum { QMOE_F16 = 0, QMOE_BF16 = 1 } qmoe_dtype;

/* Path selection for qmoe_forward_ex.
 *   DECODE        per-token GEMV on CUDA cores, fp32 throughout (small T).
 *                 At T = 1 (gate/up and down either all with or all without
 *                 zero points, and a shared-memory plan that fits) the whole
 *                 layer runs as one kernel; otherwise as three kernels
 *                 (router; gate-up + SwiGLU; down + weighted sum).  The one
 *                 kernel splits the down projection along I over clusters of
 *                 4 CTAs and adds the partial outputs into an integer
 *                 fixed-point accumulator (2^-32), so the sum does not depend
 *                 on arrival order; it has no grid-wide wait, so it runs
 *                 with any number of SMs available, and its results are
 *                 bit-reproducible.
 *   PREFILL       tokens grouped by expert, grouped GEMM on the tensor cores
 *                 with fp32 accumulation and exact operands: with bf16 block
 *                 scales the operands are fp16 (bf16 activations convert
 *                 exactly within fp16's normal range) and, without zero
 *                 points, each dequantised weight is one fp16 operand
 *                 (s (q - 8) has at most 11 significant bits); with zero
 *                 points or fp16 scales each weight is the exact sum of two
 *                 operands (hi = RN(w), lo = w - hi) of fp16, or of bf16
 *                 for bf16 activations with fp16 scales.  The SwiGLU
 *                 output enters the down projection as hi + lo of the
 *                 operand type.  So the only roundings are fp32
 *                 accumulation, the hi + lo SwiGLU output and the final
 *                 output (on the fp16 operands, values below fp16's
 *                 normal range, 2^-14, round to its subnormals: an absolute
 *                 error of at most 2^-25).  A bf16 activation or SwiGLU value beyond fp16's
 *                 range (65504) on the fp16-operand form sets a device
 *                 status bit (QMOE_ERR_DEVICE_CHECK).  (Value 3 of this
 *                 enum is not used: a single-rounded-operand form that
 *                 missed the elementwise tolerance was withdrawn.)
 *   DECODE_SPLIT  DECODE as three kernels always.
 *   DECODE_FUSED  DECODE as the one kernel (for T <= 4 where a CTA's share
 *                 of the selected experts fits in shared memory: at the
 *                 Qwen1.5-MoE-A2.7B layer shape only T = 1);
 *                 QMOE_ERR_UNSUPPORTED where it does not fit.  Its routing
 *                 equals DECODE_SPLIT's bit for bit; its output differs from
 *                 DECODE_SPLIT's only by the order of fp32 sums in the down
 *                 projection.
 *   AUTO          DECODE for T <= QMOE_AUTO_DECODE_MAX_TOKENS, else PREFILL
 *                 (DECODE where PREFILL's shape rules do not hold). */
typedef enum {
  QMOE_PATH_AUTO = 0,
  QMOE_PATH_DECODE = 1,
  QMOE_PATH_PREFILL = 2,
  QMOE_PATH_DECODE_SPLIT = 4,
  QMOE_PATH_DECODE_FUSED = 5
} qmoe_path;

/* One projection for all E experts (see "Packed weights" above). */
typedef struct {
  const uint8_t* w;
  const void* scales;
  const uint8_t* zp; /* may be NULL: zero point 8 */
} qmoe_qweight;

/* Largest shapes accepted: E <= 256 experts, 1 <= k <= 8. */
#define QMOE_MAX_EXPERTS 256
#define QMOE_MAX_TOPK 8
/* Most tokens the decode (GEMV) path takes (QMOE_PATH_DECODE). */
#define QMOE_DECODE_MAX_TOKENS 16
/* Tokens at or below this count take the decode path under QMOE_PATH_AUTO,
 * more take the grouped GEMM (when its shape rules hold, else decode up to
 * QMOE_DECODE_MAX_TOKENS).  Measured on GB300 at the Qwen1.5-MoE-A2.7B layer
 * shape (H 2048, I 1408, E 60, k 4, block 32, fp16, zero points), per layer:
 * decode 80 / 132 / 182 / 234 us and grouped GEMM 88 / 122 / 150 / 172 us at
 * T = 4 / 8 / 12 / 16. */
#define QMOE_AUTO_DECODE_MAX_TOKENS 5

/* Human-readable name of a status code.  Never NULL. */
const char* qmoe_status_string(int status);

/* Text of the last CUDA runtime error an entry point on this thread turned
 * into QMOE_ERR_CUDA / QMOE_ERR_UNSUPPORTED ("no error" if none).  Never NULL. */
const char* qmoe_last_cuda_error(void);

/* Bytes of device workspace qmoe_route / qmoe_forward need for these
 * shapes (covers both paths).  The workspace is caller-owned, 256-byte
 * aligned device memory.  Before its FIRST use it must be prepared with
 * qmoe_workspace_init; every call leaves it ready for the next one. */
size_t qmoe_workspace_size(int T, int H, int I, int E, int k);

/* Zero the workspace's control block (device status, counters, and the
 * one-kernel decode layer's 128 KB output accumulator) on `stream`.  Every
 * call leaves the control block ready for the next one; after a call whose
 * device status reports QMOE_ERR_TIMEOUT or QMOE_ERR_DEVICE_CHECK, run this
 * again before the workspace's next use (a call that gave up part-way can
 * leave counters or the accumulator mid-update). */
int qmoe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Diagnostics of the failure path, kept in the workspace's control block
 * (qmoe_workspace_init clears both; callers otherwise leave them).
 *   wait_limit_kilocycles  the grouped GEMM's bounded waits (prefill path and
 *                          the tensor-core matmul_nbits_ex) give up after
 *                          this many x 1024 SM cycles; 0: the default,
 *                          about 2 s.
 *   flags                  QMOE_DIAG_STALL_GEMM: the GEMM's dequantiser warps
 *                          wait for a copy that cannot arrive, so that wait
 *                          runs out; 0: none.
 * A wait that gives up sets QMOE_ST_TIMEOUT; the kernel's roles then drain
 * their copies and MMAs in flight, free TMEM and return (no trap, no hang);
 * qmoe_get_device_status reports QMOE_ERR_TIMEOUT and that call's output is
 * undefined.  The workspace stays usable: with the diagnostics cleared the
 * next call computes normally.  Asynchronous on `stream` (an 8-byte copy
 * into the control block).  QMOE_ERR_INVALID_ARG for unknown flags. */
#define QMOE_DIAG_STALL_GEMM 1u
int qmoe_workspace_set_diagnostics(void* workspace, size_t workspace_bytes, uint32_t wait_limit_kilocycles,
                                   uint32_t flags, void* stream);

/* Router: logits = x[T,H] . router_w[H,E] (+ router_bias[E]) accumulated in
 * fp32 (on CUDA cores for T <= 16; on the tensor cores for T > 16 when H is
 * a multiple of 64, E <= 128 and x is 16-byte aligned: exact 16-bit products
 * summed in fp32, the sum of the K-split partials in a fixed order);
 * softmax over all E in fp32; the k largest probabilities, best first,
 * equal probabilities ordered by lower expert id; weights are the raw
 * probabilities (not renormalised).  Then the assignments a = t*k + j are
 * grouped by expert ("sort tokens by expert", IR guide Optimization
 * Opportunities item 9 step 1).
 *   x, router_w : act_dtype (fp16 or bf16), [T,H] and [H,E]
 *   router_bias : fp32 [E] or NULL
 *   topk_w      : fp32 [T,k] out;  topk_ids : int32 [T,k] out
 *   expert_offsets : int32 [E+1] out or NULL: offsets[e] = number of
 *                 assignments to experts < e, offsets[E] = T*k
 *   perm        : int32 [T*k] out or NULL: assignment ids grouped by
 *                 expert, increasing within an expert
 * Requires 1 <= T, 1 <= k <= min(E, 8), E <= 256. */
int qmoe_route(const void* x, const void* router_w, int act_dtype, const float* router_bias,
               int T, int H, int E, int k, float* topk_w, int32_t* topk_ids,
               int32_t* expert_offsets, int32_t* perm, void* workspace, size_t workspace_bytes,
               void* stream);

/* MatMulNBits: y[M,N] = x[M,K] . dequant(W)[N,K]^T with W one packed
 * [N, K/2] matrix (E = 1 in the layout above), fp32 accumulation, y rounded
 * to act_dtype.  Small M streams W through CUDA cores; no workspace. */
int matmul_nbits(const void* x, int act_dtype, const uint8_t* w, const void* scales,
                 int scale_dtype, const uint8_t* zp, int M, int N, int K, int block_size, void* y,
                 void* stream);

/* matmul_nbits with an explicit path and a workspace, for any M (MatMulNBits,
 * IR guide section 2 "Quantization Scheme" for the weight format and the
 * dequantize-then-matmul definition).  path:
 *   DECODE        the CUDA-core path above (workspace unused, may be NULL);
 *   PREFILL       tensor cores (tcgen05) with exact operands as in the
 *                 layer's prefill path (one fp16 weight operand for bf16
 *                 scales without zero points, else hi + lo) and x as one
 *                 operand;
 *   AUTO          DECODE for M <= QMOE_DECODE_MAX_TOKENS, else PREFILL.
 * The tensor-core path needs N % 128 == 0, K % 64 == 0, x, y, scales and
 * zero points 16-byte aligned and an initialised workspace (qmoe_workspace_init)
 * of at least qmoe_workspace_size(M, N, K, 1, 1) bytes (QMOE_ERR_WORKSPACE if
 * smaller); other shapes return QMOE_ERR_UNSUPPORTED.  y is fully written;
 * x, w, scales and zp are read only.  Stream-ordered. */
int matmul_nbits_ex(const void* x, int act_dtype, const uint8_t* w, const void* scales,
                    int scale_dtype, const uint8_t* zp, int M, int N, int K, int block_size,
                    void* y, int path, void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer: out[T,H] (act_dtype) = sum over the k chosen experts of
 * p * SwiGLU-FFN_e(x).  gate/up are [E, I, H/2] (N = I, K = H), down is
 * [E, H, I/2] (N = H, K = I); all three share scale_dtype and block_size.
 * topk_w_out / topk_ids_out ([T,k], may be NULL) return the routing used.
 * If accumulate is non-zero, out = out + layer(x) (residual add).
 * Requires H and I multiples of 32 and of block_size. */
int qmoe_forward(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                 qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                 int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                 int32_t* topk_ids_out, int accumulate, void* workspace, size_t workspace_bytes,
                 void* stream);

/* qmoe_forward with an explicit path (QMOE_PATH_*); AUTO picks decode for
 * T <= QMOE_AUTO_DECODE_MAX_TOKENS. */
int qmoe_forward_ex(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                    qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                    int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                    int32_t* topk_ids_out, int accumulate, int path, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Number of kernels one qmoe_forward_ex call with these sizes and this path
 * launches on the current device: 1 (decode layer fused into one
 * kernel), 3 (decode: router, gate-up, down) or 5 (prefill:
 * router, token permutation, two grouped GEMMs, output conversion).  Host
 * only, nothing launched.  Negative status (-QMOE_ERR_*) if the arguments
 * are invalid or the shape is unsupported.  Pointer alignment is not known
 * here and is assumed to meet the call's rules. */
int qmoe_forward_kernels(int T, int H, int I, int E, int k, int block_size, int act_dtype,
                         int scale_dtype, int gate_up_has_zp, int down_has_zp, int path);

/* qmoe_forward_ex for profiling: records events[0] before the first kernel
 * and events[i] after kernel i (router, gate-up, down on the decode path),
 * for i < n_events (cudaEvent_t passed as void*; NULL entries skipped).  The
 * kernels run back to back without programmatic overlap, so event pairs
 * bracket one kernel each.  Same arguments and results as qmoe_forward. */
int qmoe_forward_profiled(const void* x, int act_dtype, const void* router_w,
                          const float* router_bias, qmoe_qweight gate, qmoe_qweight up,
                          qmoe_qweight down, int scale_dtype, int T, int H, int I, int E, int k,
                          int block_size, void* out, int path, void* workspace,
                          size_t workspace_bytes, void* stream, void* const* events,
                          int n_events);

/* Shared expert of the MoE block ("Qwen MoE BringUp", IR guide section 3,
 * "Shared Expert"): every token goes through one more SwiGLU expert whose
 * output, scaled by a sigmoid gate, is added to the block's output:
 *   out[t] (+)= sigmoid(x[t] . shared_gate_w) * FFN(x[t])
 * shared_gate_w is a [H] vector in act_dtype.  The expert's weights use the
 * same INT4 block format as the routed experts with E = 1: gate/up
 * [1, I, H/2], down [1, H, I/2] (the pages' model keeps this expert in fp16;
 * here it is quantised like the others).  It runs as the layer with one
 * expert, top-1, the gate vector as its router and a sigmoid in place of the
 * softmax, so the whole MoE block is
 *   qmoe_forward(..., out, accumulate)  then
 *   qmoe_shared_expert(..., out, accumulate = 1).
 * Workspace: qmoe_workspace_size(T, H, I, 1, 1).  Same conventions and
 * errors as qmoe_forward; shared_gate_w NULL -> QMOE_ERR_INVALID_ARG. */
int qmoe_shared_expert(const void* x, int act_dtype, const void* shared_gate_w, qmoe_qweight gate,
                       qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T, int H, int I,
                       int block_size, void* out, int accumulate, void* workspace, size_t workspace_bytes,
                       void* stream);

/* qmoe_forward without a caller workspace.  An engineering addition with no
 * counterpart in the method's sources: it serves callers that cannot give
 * the library device memory, such as a plain C host program with no device
 * allocator, or a plugin hook that receives no workspace argument and must
 * not call cudaMalloc (which synchronises the whole device).
 *
 * The workspace is a library-owned static device array of
 * QMOE_NOALLOC_SCRATCH_BYTES (2 MiB) per device; the call allocates
 * nothing.  Its control block (device status word, counters, the one-kernel
 * decode layer's output accumulator) starts at zero when the library is
 * loaded and every call leaves the counters and the accumulator at zero
 * again.  The first call on a device
 * looks the array's address up (cudaGetSymbolAddress), so make that first
 * call, with the device current, before any stream capture.
 *
 * Same arguments and results as qmoe_forward (path chosen as by
 * QMOE_PATH_AUTO), minus the workspace.  Shapes whose workspace
 * (qmoe_workspace_size) exceeds QMOE_NOALLOC_SCRATCH_BYTES return
 * QMOE_ERR_UNSUPPORTED and enqueue nothing; the Qwen1.5-MoE-A2.7B layer
 * shape fits up to T = 16.  Overlapping calls on one device (two streams,
 * or two host threads without ordering) share the array and race: order
 * them on one stream.  Device-side conditions (a bounded wait that ran out)
 * are recorded in the scratch's status word: read it with
 * qmoe_noalloc_status. */
#define QMOE_NOALLOC_SCRATCH_BYTES (2u << 20)
int qmoe_forward_noalloc(const void* x, int act_dtype, const void* router_w, const float* router_bias,
                         qmoe_qweight gate, qmoe_qweight up, qmoe_qweight down, int scale_dtype, int T,
                         int H, int I, int E, int k, int block_size, void* out, float* topk_w_out,
                         int32_t* topk_ids_out, int accumulate, void* stream);

/* The device status word of qmoe_forward_noalloc's static scratch on the
 * current device, read and cleared like qmoe_get_device_status (blocking:
 * synchronises `stream`).  Returns QMOE_OK, or the first QMOE_ERR_* a kernel
 * recorded since the last read (a bounded wait that ran out, a failed index
 * or launch-shape check: the output of that call is not valid); *bits_out
 * (may be NULL) gets the raw bits.  After QMOE_ERR_TIMEOUT the scratch's
 * counters may be left mid-count: the library has no allocation-free way to
 * reset them, so such a process should stop using this entry point. */
int qmoe_noalloc_status(uint32_t* bits_out, void* stream);

/* DequantizeLinear of one [N, K] matrix (packed [N, K/2]) to fp32 out[N,K]:
 * (q - zp) * scale, which fp32 holds exactly. */
int qmoe_dequant(const uint8_t* w, const void* scales, int scale_dtype, const uint8_t* zp, int N,
                 int K, int block_size, float* out, void* stream);

/* RMSNorm of the layer stack ("IR guide", 1. RMSNorm) with unit weight:
 * out[t,h] = x[t,h] / sqrt(mean_h(x[t,h]^2) + eps), computed in fp32 and
 * rounded to act_dtype.  x and out may alias. */
int qmoe_rmsnorm(const void* x, void* out, int act_dtype, int T, int H, float eps, void* stream);

/* ---- Weight-format adapters (one-time conversion at model load).
 *
 * GPTQ checkpoints into the canonical layout above ("Qwen MoE BringUp",
 * "Bugs/Issues Found", item 1: GPTQ zero points are stored with an offset
 * of +1 or +0 depending on the exporter, told apart by the median stored
 * zero).  Source layout, per expert e (E experts stacked, input-major):
 *   qweight [E, K/8, N]    int32: bits 4j..4j+3 of word (i, n) = q[8i + j, n]
 *   qzeros  [E, K/bs, N/8] int32: bits 4j..4j+3 of word (g, i) = stored zero
 *                          of block g, column 8i + j; or NULL (symmetric
 *                          int4 without zero points)
 *   scales  [E, K/bs, N]   16-bit (fp16 or bf16, copied bit for bit)
 * Output: w_out [E, N, K/2], scales_out [E, N, K/bs], zp_out [E, N, K/bs]
 * (NULL exactly when qzeros is NULL; the canonical layout then implies
 * zero point 8).  zp = stored + offset: the offset is *zero_offset_dev
 * when that device pointer is given (for example the output of
 * qmoe_gptq_zero_offset, read by the kernel, so no host round trip), else
 * zero_offset (0 or 1).  A zero point of 16 (a stored 15 with offset 1)
 * does not fit the canonical 4-bit zero point: it is written as 15 and, if
 * status_dev (a 4-byte device word, may be NULL) is given, QMOE_ST_RANGE is
 * OR-ed into it; read it with qmoe_get_device_status(status_dev, ...),
 * which returns QMOE_ERR_DEVICE_CHECK when the bit is set.  The weights of
 * such blocks differ from the checkpoint's by one scale step, so a caller
 * should refuse the checkpoint.  Requires N a multiple of 8, K a
 * multiple of 32 and of block_size (32, 64, 128); 4-byte aligned int32
 * buffers and w_out, 2-byte aligned scales.  Asynchronous on `stream`;
 * input and output must not overlap.  Bound by HBM (every byte read and
 * written once). */
int qmoe_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int E, int K,
                     int N, int block_size, int zero_offset, const int32_t* zero_offset_dev,
                     uint8_t* w_out, void* scales_out, uint8_t* zp_out, uint32_t* status_dev, void* stream);

/* The GPTQ zero-point offset of a qzeros tensor (n_words int32 words, all
 * experts and projections the caller wants to judge together), written to
 * the device int *offset_out: 1 if the lower median of the stored zero
 * points is 7 (the exporter stored zero - 1), else 0.  Asynchronous; pass
 * offset_out to qmoe_repack_gptq as zero_offset_dev. */
int qmoe_gptq_zero_offset(const int32_t* qzeros, size_t n_words, int32_t* offset_out, void* stream);

/* Packed 4-bit zero points [rows, ceil(nb/2)] (two per byte, block 2b in
 * the low nibble, 2b + 1 in the high nibble, each row padded to a byte)
 * into the canonical one byte per block [rows, nb].  The pages' model
 * already stores one byte per block; this is the packing ONNX MatMulNBits
 * uses for 4-bit zero points.  rows = E * N for a stacked projection. */
int qmoe_unpack_zero_points(const uint8_t* zp_packed, int rows, int nb, uint8_t* zp_out, void* stream);

/* Read (blocking: synchronises `stream`) and clear the device status word
 * of `workspace` (its first 4 bytes; also any 4-byte status word such as
 * qmoe_repack_gptq's status_dev).  Returns QMOE_OK, or QMOE_ERR_TIMEOUT
 * if a wait ran out, else QMOE_ERR_DEVICE_CHECK if an index or range check
 * failed since the last read; *bits_out (may be NULL) gets the raw bits
 * (QMOE_ST_*). */
int qmoe_get_device_status(void* workspace, uint32_t* bits_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H_ */
