/*
 * qmoe_oracle.c -- plain, slow, single-threaded fp64 oracle for the INT4
 * block-quantized mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may
 * include, link, load or call this file; only the tests, the package's
 * smoke check and the bench's CPU-baseline / reference arm use it.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Sources (web pages describing the layer; cited by page title + section):
 *   [BringUp]  "Qwen MoE BringUp" (IREE ONNX Runtime EP issue #34)
 *     - local fix A1 "DequantizeLinear block_size decomposition":
 *       DequantizeLinear with block_size lowers to extui -> uitofp -> subf -> mulf.
 *     - "Qwen1.5-MoE-A2.7B-Chat INT4 -- IR Guide", 1. RMSNorm.
 *     - same guide, 3. MoE Block: "Router (TopK via extern GPU kernel)"
 *       (gate linear, softmax in f32 over all experts, top-k) and
 *       "Expert Computation (INT4 QDQ, gather-then-compute)" steps 1-7
 *       (gather, DequantizeLinear along axis 2 = input dim, MatMuls,
 *        SwiGLU = Mul(gate, Sigmoid(gate)) * up, down projection,
 *        routing-weighted sum of the k expert outputs).
 *
 * Everything is evaluated in double precision from the stored inputs,
 * which are converted to double exactly.  No blocking, fusion or
 * reordering beyond what the definitions state.
 *
 * Storage conventions (the pages print unpacked element counts and are
 * silent on nibble order; the reading adopted here):
 *   packed weights  [N, K/2] bytes per matrix; element k of a row sits in
 *                   byte k/2, low nibble for even k, high nibble for odd k;
 *   scales          [N, K/block_size], fp16 or bf16 bit patterns;
 *   zero points     [N, K/block_size], one byte per block holding 0..15;
 *                   a NULL zero-point tensor means zero point 8
 *                   (offset-binary storage of signed symmetric int4).
 *
 * Parity pins: every function here is pinned by tests that do not run
 * this file's arithmetic twice (hand-worked examples, closed forms,
 * library routines on special cases, brute force).  Nothing is marked
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F16 0
#define OR_BF16 1

/* ORACLE_PLANT selects a deliberately wrong variant, built only by the pin
 * tests to show that the pins catch it; every normal build has 0. */
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

/* ---- exact storage -> double conversions (IEEE binary16, bfloat16) ---- */

double oracle_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int mant = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(mant | 0x400), expo - 25); /* (1024+m) * 2^(e-15-10) */
  }
  return sign ? -v : v;
}

double oracle_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int expo = (b >> 7) & 0xff;
  int mant = b & 0x7f;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -133); /* subnormal: mant * 2^-126 * 2^-7 */
  } else if (expo == 255) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(mant | 0x80), expo - 134); /* (128+m) * 2^(e-127-7) */
  }
  return sign ? -v : v;
}

static double load16(const uint16_t* p, int64_t i, int dtype) {
  return dtype == OR_BF16 ? oracle_bf16_to_double(p[i]) : oracle_f16_to_double(p[i]);
}

/* Round a double to the nearest bfloat16 value (ties to even), returned as
 * a double.  Used only where the layer itself casts to the activation type
 * (the stack's RMSNorm output, per the IR guide's "Cast back" step). */
double oracle_round_to_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e);               /* |v| = m * 2^e, m in [0.5, 1) */
  int q = e - 8;              /* bf16 keeps 8 significant bits */
  if (q < -133) q = -133;     /* subnormal quantum 2^-133 */
  double scaled = ldexp(v, -q);
  double r = nearbyint(scaled); /* default rounding mode: ties to even */
  return ldexp(r, q);
}

/* ---- DequantizeLinear with block_size along the input (K) axis ----------
 * [BringUp] fix A1: extui (nibble -> integer) -> uitofp -> subf (zero
 * point) -> mulf (block scale).  One scale / zero point per block_size run
 * of consecutive K elements of a row.  Value = (q - zp) * scale, exact in
 * double. */
static int nibble(const uint8_t* w, int64_t row_bytes, int64_t n, int64_t kk) {
  uint8_t byte = w[n * row_bytes + kk / 2];
#if ORACLE_PLANT == 1 /* planted: nibble order swapped */
  return (kk % 2 == 1) ? (byte & 0x0f) : (byte >> 4);
#endif
  return (kk % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
}

double oracle_dequant_one(const uint8_t* w, const uint16_t* scales, int scale_dtype,
                          const uint8_t* zp, int N, int K, int block_size, int64_t n,
                          int64_t kk) {
  (void)N;
  int64_t nblk = K / block_size;
  int64_t b = kk / block_size;
#if ORACLE_PLANT == 2 /* planted: block index taken modulo instead of quotient */
  b = (kk % block_size) % nblk;
#endif
  double q = (double)nibble(w, K / 2, n, kk);            /* extui, uitofp */
  double z = zp ? (double)zp[n * nblk + b] : 8.0;         /* zero point    */
#if ORACLE_PLANT == 3 /* planted: zero point dropped */
  z = 0.0;
#endif
  double s = load16(scales, n * nblk + b, scale_dtype);   /* block scale   */
  return (q - z) * s;                                     /* subf, mulf    */
}

void oracle_dequant(const uint8_t* w, const uint16_t* scales, int scale_dtype,
                    const uint8_t* zp, int N, int K, int block_size, double* out) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t kk = 0; kk < K; ++kk)
      out[n * K + kk] = oracle_dequant_one(w, scales, scale_dtype, zp, N, K, block_size, n, kk);
}

/* ---- MatMulNBits: y[m, n] = sum_k x[m, k] * W[n, k], W dequantised -------
 * The expert weights are stored pre-transposed ([out, in], K contiguous),
 * IR guide "Optimization Opportunities" item 5. */
void oracle_matmul_nbits(const uint16_t* x, int x_dtype, const uint8_t* w,
                         const uint16_t* scales, int scale_dtype, const uint8_t* zp,
                         int M, int N, int K, int block_size, double* y) {
  double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t kk = 0; kk < K; ++kk)
      wrow[kk] = oracle_dequant_one(w, scales, scale_dtype, zp, N, K, block_size, n, kk);
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0;
      for (int64_t kk = 0; kk < K; ++kk) acc += load16(x, m * (int64_t)K + kk, x_dtype) * wrow[kk];
#if ORACLE_PLANT == 6 /* planted: last K element dropped */
      acc -= load16(x, m * (int64_t)K + K - 1, x_dtype) * wrow[K - 1];
#endif
      y[m * (int64_t)N + n] = acc;
    }
  }
  free(wrow);
}

/* ---- Router: gate linear, softmax over all E experts ---------------------
 * [BringUp] IR guide, 3. MoE Block, Router: logits = hidden[T,H] x
 * W_gate[H,E]; softmax over the E logits (max-subtracted), in higher
 * precision than the stored type; optional per-expert bias added to the
 * logits before the softmax. */
void oracle_router_probs(const uint16_t* x, int x_dtype, const uint16_t* router_w,
                         const float* bias, int T, int H, int E, double* probs) {
  double* logit = (double*)malloc(sizeof(double) * (size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h)
        acc += load16(x, t * (int64_t)H + h, x_dtype) * load16(router_w, h * (int64_t)E + e, x_dtype);
      logit[e] = acc + (bias ? (double)bias[e] : 0.0);
    }
    double mx = logit[0];
    for (int64_t e = 1; e < E; ++e)
      if (logit[e] > mx) mx = logit[e];
    double sum = 0.0;
    for (int64_t e = 0; e < E; ++e) sum += exp(logit[e] - mx);
    for (int64_t e = 0; e < E; ++e) probs[t * (int64_t)E + e] = exp(logit[e] - mx) / sum;
  }
  free(logit);
}

/* ---- Top-k over the probabilities ------------------------------------------
 * The pages select the k largest probabilities, best first (selection sort
 * in the extern kernel, "Kernel internals").  Ties are not addressed by the
 * pages; the reading adopted: equal probabilities order by lower expert id.
 * The oracle uses a full sort of (p descending, id ascending) and keeps the
 * first k.  The routing weights are the raw softmax probabilities of the
 * chosen experts (no renormalisation): they feed the weighted-sum MatMul
 * directly (Expert Computation, step 7). */
typedef struct {
  double p;
  int id;
} or_pid;

static int cmp_pid(const void* a, const void* b) {
  const or_pid* x = (const or_pid*)a;
  const or_pid* y = (const or_pid*)b;
  if (x->p > y->p) return -1;
  if (x->p < y->p) return 1;
#if ORACLE_PLANT == 5 /* planted: ties broken towards the higher id */
  return (x->id > y->id) ? -1 : (x->id < y->id);
#endif
  return (x->id < y->id) ? -1 : (x->id > y->id);
}

void oracle_topk(const double* probs, int T, int E, int k, int32_t* ids, double* weights) {
  or_pid* buf = (or_pid*)malloc(sizeof(or_pid) * (size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      buf[e].p = probs[t * (int64_t)E + e];
      buf[e].id = e;
    }
    qsort(buf, (size_t)E, sizeof(or_pid), cmp_pid);
    for (int j = 0; j < k; ++j) {
      ids[t * (int64_t)k + j] = buf[j].id;
      weights[t * (int64_t)k + j] = buf[j].p;
    }
  }
  free(buf);
}

/* ---- Assignment grouping ("sort tokens by expert") --------------------------
 * IR guide "Optimization Opportunities" item 9, step 1: flatten topk_ids
 * [T, k] to assignments a = t*k + j and group them contiguously by expert.
 * offsets[e] = number of assignments to experts < e (offsets[E] = T*k);
 * perm lists assignment ids grouped by expert, in increasing a within an
 * expert (stable). */
void oracle_group_by_expert(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                            int32_t* perm) {
  int64_t A = (int64_t)T * k;
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int64_t a = 0; a < A; ++a) offsets[ids[a] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int64_t a = 0; a < A; ++a) perm[fill[ids[a]]++] = (int32_t)a;
  free(fill);
}

/* ---- One expert's SwiGLU FFN on one token -----------------------------------
 * Expert Computation steps 4-6: g = x . Wg^T, u = x . Wu^T (per row of the
 * [I, H] pre-transposed weights), act = Mul(g, Sigmoid(g)) * u,
 * y = act . Wd^T with Wd stored [H, I].  All in double. */
typedef struct {
  const uint8_t* w;
  const uint16_t* scales;
  const uint8_t* zp;
} or_qw;

static void expert_ffn(const double* xrow, int64_t e, or_qw g, or_qw u, or_qw d, int scale_dtype,
                       int H, int I, int block_size, double* act, double* y) {
  int64_t nb_h = H / block_size, nb_i = I / block_size;
  /* expert e's slices of the stacked [E, N, ...] tensors */
  const uint8_t* gw = g.w + e * (int64_t)I * (H / 2);
  const uint8_t* uw = u.w + e * (int64_t)I * (H / 2);
  const uint8_t* dw = d.w + e * (int64_t)H * (I / 2);
  const uint16_t* gs = g.scales + e * (int64_t)I * nb_h;
  const uint16_t* us = u.scales + e * (int64_t)I * nb_h;
  const uint16_t* ds = d.scales + e * (int64_t)H * nb_i;
  const uint8_t* gz = g.zp ? g.zp + e * (int64_t)I * nb_h : NULL;
  const uint8_t* uz = u.zp ? u.zp + e * (int64_t)I * nb_h : NULL;
  const uint8_t* dz = d.zp ? d.zp + e * (int64_t)H * nb_i : NULL;
  for (int64_t i = 0; i < I; ++i) {
    double ga = 0.0, ua = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      ga += xrow[h] * oracle_dequant_one(gw, gs, scale_dtype, gz, I, H, block_size, i, h);
      ua += xrow[h] * oracle_dequant_one(uw, us, scale_dtype, uz, I, H, block_size, i, h);
    }
    double sig = 1.0 / (1.0 + exp(-ga));
    act[i] = ga * sig * ua;
#if ORACLE_PLANT == 4 /* planted: SiLU applied to the up projection */
    act[i] = ua / (1.0 + exp(-ua)) * ga;
#endif
  }
  for (int64_t h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i)
      acc += act[i] * oracle_dequant_one(dw, ds, scale_dtype, dz, H, I, block_size, h, i);
    y[h] = acc;
  }
}

/* ---- The whole layer -------------------------------------------------------------
 * out[t] = sum_j w[t, j] * FFN_{ids[t, j]}(x[t])   (Expert Computation step 7)
 * If forced_ids is non-NULL the routing is taken from forced_ids /
 * forced_w instead of being computed (used to re-evaluate near-tie tokens
 * with another implementation's choice of experts).
 * Outputs: out [T, H] double; ids_out [T, k], w_out [T, k], probs_out
 * [T, E] (each may be NULL).  Returns 0, or -1 on a bad argument. */
int oracle_qmoe_forward(const uint16_t* x, int x_dtype, const uint16_t* router_w,
                        const float* router_bias, const uint8_t* gate_w, const uint16_t* gate_s,
                        const uint8_t* gate_zp, const uint8_t* up_w, const uint16_t* up_s,
                        const uint8_t* up_zp, const uint8_t* down_w, const uint16_t* down_s,
                        const uint8_t* down_zp, int scale_dtype, int T, int H, int I, int E, int k,
                        int block_size, const int32_t* forced_ids, const double* forced_w,
                        double* out, int32_t* ids_out, double* w_out, double* probs_out) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E || block_size <= 0) return -1;
  if (H % block_size || I % block_size || H % 2 || I % 2) return -1;
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k + 1));
  double* wts = (double*)malloc(sizeof(double) * (size_t)(T * k + 1));
  double* probs = (double*)malloc(sizeof(double) * (size_t)(T * E + 1));
  if (forced_ids) {
    memcpy(ids, forced_ids, sizeof(int32_t) * (size_t)(T * k));
    memcpy(wts, forced_w, sizeof(double) * (size_t)(T * k));
    for (int64_t i = 0; i < (int64_t)T * E; ++i) probs[i] = NAN;
  } else {
    oracle_router_probs(x, x_dtype, router_w, router_bias, T, H, E, probs);
    oracle_topk(probs, T, E, k, ids, wts);
  }
  or_qw g = {gate_w, gate_s, gate_zp}, u = {up_w, up_s, up_zp}, d = {down_w, down_s, down_zp};
  double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
  double* act = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) xrow[h] = load16(x, t * (int64_t)H + h, x_dtype);
    for (int64_t h = 0; h < H; ++h) out[t * (int64_t)H + h] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = ids[t * (int64_t)k + j];
      if (e < 0 || e >= E) continue;
      expert_ffn(xrow, e, g, u, d, scale_dtype, H, I, block_size, act, y);
      double wj = wts[t * (int64_t)k + j];
#if ORACLE_PLANT == 7 /* planted: routing weights renormalised over the k chosen */
      { double sw = 0.0; for (int jj = 0; jj < k; ++jj) sw += wts[t * (int64_t)k + jj]; wj /= sw; }
#endif
      for (int64_t h = 0; h < H; ++h) out[t * (int64_t)H + h] += wj * y[h];
    }
  }
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)(T * k));
  if (w_out) memcpy(w_out, wts, sizeof(double) * (size_t)(T * k));
  if (probs_out) memcpy(probs_out, probs, sizeof(double) * (size_t)(T * E));
  free(ids);
  free(wts);
  free(probs);
  free(xrow);
  free(act);
  free(y);
  return 0;
}

/* Shared expert of the MoE block ("Qwen MoE BringUp", IR guide section 3,
 * "Shared Expert": every token goes through one gated SwiGLU expert whose
 * output, scaled by its gate, is added to the routed output).  Reading: the
 * gate is sigmoid(x . gate_w) with gate_w a [H] vector in x's dtype, and the
 * expert's weights use the same INT4 block format as the routed experts
 * ([1, I, H/2] gate/up, [1, H, I/2] down).
 *   out[t] = sigmoid(sum_h x[t,h] * gate_w[h]) * FFN(x[t])   (fp64) */
int oracle_shared_expert(const uint16_t* x, int x_dtype, const uint16_t* shared_gate_w,
                         const uint8_t* gate_w, const uint16_t* gate_s, const uint8_t* gate_zp,
                         const uint8_t* up_w, const uint16_t* up_s, const uint8_t* up_zp,
                         const uint8_t* down_w, const uint16_t* down_s, const uint8_t* down_zp,
                         int scale_dtype, int T, int H, int I, int block_size, double* out,
                         double* gate_out) {
  if (T < 0 || H <= 0 || I <= 0 || block_size <= 0 || !shared_gate_w) return -1;
  if (H % block_size || I % block_size || H % 2 || I % 2) return -1;
  or_qw g = {gate_w, gate_s, gate_zp}, u = {up_w, up_s, up_zp}, d = {down_w, down_s, down_zp};
  double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
  double* act = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int64_t t = 0; t < T; ++t) {
    double logit = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      xrow[h] = load16(x, t * (int64_t)H + h, x_dtype);
      logit += xrow[h] * load16(shared_gate_w, h, x_dtype);
    }
    const double gate = 1.0 / (1.0 + exp(-logit));
    if (gate_out) gate_out[t] = gate;
    expert_ffn(xrow, 0, g, u, d, scale_dtype, H, I, block_size, act, y);
    for (int64_t h = 0; h < H; ++h) out[t * (int64_t)H + h] = gate * y[h];
  }
  free(xrow);
  free(act);
  free(y);
  return 0;
}

/* ---- RMSNorm (the layer stack's pre-MoE norm) ---------------------------------
 * IR guide, 1. RMSNorm: y = x / sqrt(mean(x^2) + eps), computed in higher
 * precision; the learned per-channel weight is taken as 1 here (synthetic
 * stack, no trained weights).  If round_bf16 is set the result is rounded
 * to bfloat16 ("Cast back" to the activation type). */
void oracle_rmsnorm(const uint16_t* x, int x_dtype, int T, int H, double eps, int round_bf16,
                    double* out) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double v = load16(x, t * (int64_t)H + h, x_dtype);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t h = 0; h < H; ++h) {
      double v = load16(x, t * (int64_t)H + h, x_dtype) * inv;
      out[t * (int64_t)H + h] = round_bf16 ? oracle_round_to_bf16(v) : v;
    }
  }
}
