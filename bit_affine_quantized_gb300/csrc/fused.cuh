// Helpers of the persistent (one block per SM) layer kernels: consumer-only
// named barrier, grid barrier on a monotonic 64-bit counter, orderable keys
// for the top-k.  Both fused kernels use 16 consumer warps + 1 producer warp.
#pragma once

#include "common.cuh"

namespace moe {
namespace fused {

constexpr int kCons = 16;                     // consumer warps
constexpr int kConsThreads = kCons * 32;     // 512
constexpr int kThreads = kConsThreads + 32;  // + producer warp

__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsThreads) : "memory"); }
// Barrier of the consumer warps that also ANDs a predicate over them (so a
// bounded wait that ran out in some threads only is seen by all).
__device__ __forceinline__ bool cons_sync_and(bool v) {
  uint32_t res;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(res)
      : "r"((uint32_t)v), "n"(kConsThreads)
      : "memory");
  return res != 0;
}

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned long long *p) {
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

// Raise the transaction count of the current phase without arriving: the
// phase then needs both these bytes and the pending arrival.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// One arrival that counts as `count` (the phase needs the count the barrier
// was initialised with).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Orders this thread's generic-proxy global accesses with later (or, on the
// writer side, earlier) bulk copies, which run in the async proxy.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Grid barrier on one 64-bit arrival counter, run by the consumer threads of
// every block: each block adds 1 with a release reduction (no return value,
// so arrivals pipeline at L2 instead of serialising) and polls until the
// counter reaches `target`.  The counter only grows; a launch derives its
// targets from the value it reads after its dependency wait (every launch
// adds exactly nbarriers * gridDim.x).  Bounded: false after kWaitLimitNs.
__device__ __forceinline__ bool grid_sync(unsigned long long *count, unsigned long long target, unsigned *err,
                                          int *s_flag) {
  cons_sync();  // the block's writes happen-before thread 0's release below
  if (threadIdx.x == 0) {
    red_release_add(count);
    bool ok = true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire64(count) >= target) break;
      if ((it & 15u) == 15u && global_ns() - t0 > kWaitLimitNs) {
        ok = false;
        break;
      }
    }
    if (!ok) set_error(err, kErrTimeout);
    *s_flag = ok ? 1 : 0;
  }
  cons_sync();
  return *s_flag != 0;
}

// Orderable 32-bit key of a float (larger float -> larger key).
__device__ __forceinline__ unsigned ord_key(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of E <= 128 fp32 logits by one warp: ids by descending logit, ties to
// the lower id (two warp reductions per pick), softmax weights over the k.
// Non-finite logits count as -inf and set *nonfinite.  `logits` is read with
// plain loads: shared memory, or global memory this block wrote itself.
__device__ __forceinline__ void warp_topk(const float *logits, int E, int k, int32_t *ids_out, float *wts_out,
                                          const float *expert_scale, bool *nonfinite) {
  const int lane = threadIdx.x & 31;
  unsigned key[4];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;  // below every real key: never picked while k <= E
    if (e < E) {
      float x = logits[e];
      if (!isfinite(x)) {
        x = -INFINITY;
        bad = true;
      }
      key[i] = ord_key(x);
    }
  }
  *nonfinite = __any_sync(0xffffffffu, bad);
  float selv[kMaxTopK];
  int seli[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      unsigned bk = key[0];
      int bi = lane;
#pragma unroll
      for (int i = 1; i < 4; ++i)
        if (key[i] > bk) {
          bk = key[i];
          bi = lane + 32 * i;
        }
      const unsigned kmax = __reduce_max_sync(0xffffffffu, bk);
      const unsigned idmin = __reduce_min_sync(0xffffffffu, bk == kmax ? (unsigned)bi : 0xffffffffu);
      selv[j] = key_value(kmax);
      seli[j] = (int)idmin;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if ((int)idmin == lane + 32 * i) key[i] = 0u;  // taken (static indexing: no local memory)
    }
  }
  float ex[kMaxTopK], den = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) {
      ex[j] = expf(selv[j] - selv[0]);
      den += ex[j];
    }
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k && lane == j) {
      ids_out[j] = seli[j];
      wts_out[j] = ex[j] / den * (expert_scale ? expert_scale[seli[j]] : 1.0f);
    }
}

}  // namespace fused
}  // namespace moe
