// common.cuh -- device helpers shared by the kernels: mbarrier / bulk-copy /
// tcgen05 PTX wrappers, bounded waits, packed fp32 math, 16-bit loads.
// Written for sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "layout.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a only"
#endif

namespace qmoe {

// ----------------------------------------------------------------- status
// Sticky device status word (first 4 bytes of the workspace control block).
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ----------------------------------------------------------- 16-bit values
template <typename T> struct Half;
template <> struct Half<__half> {
  static __device__ __forceinline__ float to_float(uint16_t b) {
    return __half2float(__ushort_as_half(b));
  }
  static __device__ __forceinline__ uint16_t from_float(float f) {
    return __half_as_ushort(__float2half_rn(f));
  }
};
template <> struct Half<__nv_bfloat16> {
  static __device__ __forceinline__ float to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
  }
  static __device__ __forceinline__ uint16_t from_float(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
};

// --------------------------------------------------------- smem addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// -------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the warp is descheduled until the
// phase completes or about `ns` nanoseconds pass, so waiting warps do not
// take issue slots from the warps doing the arithmetic.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~kWaitLimitCycles SM cycles, records
// QMOE_ST_TIMEOUT in the status word and returns false.  No trap, no hang.
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 100000u)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      set_status(status, QMOE_ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ bulk copies
// Non-tensor TMA copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Asynchronous 16-byte global -> shared copy (LDGSTS), no register round
// trip, so a thread can have many in flight; cp_async_wait_all() waits for
// this thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// --------------------------------------------------- packed fp32 (f32x2)
// Native paired fp32 operations of sm_100+ (one instruction for two lanes
// of work, round-to-nearest-even like the scalar ones).
using f2 = float2;
__device__ __forceinline__ f2 ffma2(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ f2 fadd2(f2 a, f2 b) { return __fadd2_rn(a, b); }

// ------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------- tensor TMA
// 2D tiled TMA load (cp.async.bulk.tensor) global -> shared, completion
// counted in bytes on `bar`.  c0 = innermost coordinate (elements; c0 times
// the element size must be a multiple of 16 bytes), c1 = row.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05
// Tensor memory (TMEM) allocation: the whole warp executes these.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] x B[smem desc]^T, bf16/f16 inputs, f32 accumulate,
// issued by one elected lane of a converged warp: every lane runs the MMA
// loop, so the operands stay warp-uniform.  Measured on GB300 an elected
// lane issues a tcgen05.mma about every 32 cycles, a lone active lane of a
// diverged warp about every 65.
__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem desc] x B[smem desc]^T by the elected lane of a converged warp.
__device__ __forceinline__ void mma_f16_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// tcgen05.commit by the elected lane (the lane that issued the MMAs).
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(smem_u32(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns (one row per thread of the
// warp), waited for in the same asm block so no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns stored from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05), K-major operand stored in the
// 128-byte-swizzled layout: rows of 128 bytes (64 16-bit elements), groups
// of 8 rows 1024 bytes apart, 16-byte chunks XOR-ed with (row mod 8).  The
// tile must start on a 1024-byte boundary; stepping K by 16 elements inside
// the 128-byte row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);       // start address
  d |= (uint64_t)1u << 16;                           // leading byte offset (unused: K fits a row)
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: 8-row group pitch
  d |= (uint64_t)1u << 46;                           // descriptor version
  d |= (uint64_t)2u << 61;                           // 128-byte swizzle
  return d;
}
// Instruction descriptor: kind::f16, D f32, A/B bf16 (or f16), both K-major.
__host__ __device__ __forceinline__ uint32_t idesc_f16(int M, int N, bool bf16) {
  uint32_t d = 0;
  d |= 1u << 4;                     // D format f32
  d |= (bf16 ? 1u : 0u) << 7;       // A format
  d |= (bf16 ? 1u : 0u) << 10;      // B format
  d |= (uint32_t)(N >> 3) << 17;    // N / 8
  d |= (uint32_t)(M >> 4) << 24;    // M / 16
  return d;
}

// ----------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 load from the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t addr = smem_u32(local), raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}

// ------------------------------------------------------ router top-k
// One warp, one token: lane holds the logits of experts lane + 32*m (m <
// ME; -inf beyond E).  Softmax over the E experts (or, for a gated shared
// expert, an independent sigmoid per logit), then k rounds of arg-max with
// ties to the lower expert id.  Every lane returns the k ids and raw
// probabilities.  Both router kernels call this, so they agree bit for bit.
template <int ME>
__device__ __forceinline__ void softmax_topk(const float (&lg)[ME], int E, int k, bool gate_sigmoid, int lane,
                                             int (&ids)[kMaxTopk], float (&wts)[kMaxTopk]) {
  float mx = -INFINITY;
#pragma unroll
  for (int m = 0; m < ME; ++m) mx = fmaxf(mx, lg[m]);
  {
    // warp max through the integer reduction unit: floats mapped to
    // unsigned keys with the same order
    uint32_t key = __float_as_uint(mx);
    key = (key & 0x80000000u) ? ~key : (key | 0x80000000u);
    key = __reduce_max_sync(0xffffffffu, key);
    mx = __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
  }
  float pr[ME];
  if (gate_sigmoid) {
#pragma unroll
    for (int m = 0; m < ME; ++m) pr[m] = (lane + 32 * m < E) ? 1.f / (1.f + expf(-lg[m])) : 0.f;
  } else {
    float ex[ME], sum = 0.f;
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      ex[m] = (lane + 32 * m < E) ? expf(lg[m] - mx) : 0.f;
      sum += ex[m];
    }
    sum = warp_sum(sum);
#pragma unroll
    for (int m = 0; m < ME; ++m) pr[m] = ex[m] / sum;
  }
  uint32_t chosen = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) {
    ids[j] = 0;
    wts[j] = 0.f;
  }
  for (int j = 0; j < k; ++j) {
    // the largest remaining probability (p >= 0: its bits order as
    // unsigned integers; + 1 keeps p = 0 above "no candidate"), then the
    // lowest expert id holding it, each by one warp reduction
    uint32_t bkey = 0u;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < ME; ++m) {
      const int e = lane + 32 * m;
      const uint32_t key = __float_as_uint(pr[m]) + 1u;
      if (e < E && !((chosen >> m) & 1u) && key > bkey) {
        bkey = key;
        bi = e;
      }
    }
    const uint32_t mkey = __reduce_max_sync(0xffffffffu, bkey);
    bi = (int)__reduce_min_sync(0xffffffffu, bkey == mkey ? (uint32_t)bi : 0xffffffffu);
    const float bp = __uint_as_float(mkey - 1u);
    if ((bi & 31) == lane) chosen |= 1u << (bi >> 5);
    // (select, not index: a runtime index would put the arrays in local memory)
#pragma unroll
    for (int q = 0; q < kMaxTopk; ++q)
      if (q == j) {
        ids[q] = bi;
        wts[q] = bp;
      }
  }
}


// ---------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace qmoe
