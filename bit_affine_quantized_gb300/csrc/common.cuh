// Device helpers shared by the MoE kernels: PTX wrappers for mbarriers, bulk
// (TMA 1-D) copies, L2 prefetch, programmatic dependent launch and the
// legacy-path mma.sync used for the small-N (few tokens per expert) tiles;
// the packed-code -> tensor-core operand conversions; and the parameter
// blocks the host fills.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kGroup = 64;        // quantisation group along K
constexpr int kMaxTokens = 128;   // chunk bound of one call
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 128;
constexpr int kSharedSlot = -1;   // expert id used for the shared expert's slot

// device error bits (OR-ed into the handle's error word)
constexpr unsigned kErrBadId = 1u;
constexpr unsigned kErrTimeout = 2u;
constexpr unsigned kErrNonFinite = 4u;

// bounded waits give up after this many nanoseconds
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------------ params
struct Blob {
  size_t gate_q, gate_s, gate_b, up_q, up_s, up_b, down_q, down_s, down_b;
};

// Token/expert grouping produced by the router (or by the sort kernel).
// Positions [0, n_valid) hold routed pairs in (expert, pair index) order;
// positions [T*k, T*k + T) hold the shared expert's rows (row t = token t).
struct Routing {
  int32_t *ids;        // [T*k]
  float *wts;          // [T*k]
  int32_t *counts;     // [E]
  int32_t *offsets;    // [E+1]
  int32_t *perm;       // [T*k]  sorted position -> pair index
  int32_t *pos;        // [T*k]  pair index -> sorted position (-1: dropped)
  int32_t *act_e;      // [E+1]  expert of active slot a (kSharedSlot = shared)
  int32_t *act_beg;    // [E+1]  first position of slot a
  int32_t *act_cnt;    // [E+1]  rows of slot a
  int32_t *n_act;      // [1]
};

struct LayerPtrs {
  const uint8_t *router_q;      // [E, H] bytes
  const uint16_t *router_s;     // [E, H/64] bf16
  const uint16_t *router_b;     // [E, H/64] bf16
  const uint8_t *experts;       // E blobs
  size_t stride;
  const uint8_t *shared;        // shared blob
  Blob off;
  size_t blob_bytes;            // extent of one blob's sub-tensors (max end offset)
  const float *logit_bias;      // nullable [E]
  const uint16_t *router_scale; // nullable bf16 [H]: router input x * router_scale / sqrt(H)
  const float *expert_scale;    // nullable [E]: factor of a selected expert's routing weight
};

struct Dims {
  int H, I, E, k, T;
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with the given parity; false after limit_ns of
// global time (or 2^24 polls, whichever comes first).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 31u && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}
// The same for a warp that waits while other warps of its block compute (a
// producer): between polls it sleeps, so its polling does not take issue
// slots from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_wait_idle(uint64_t *bar, uint32_t parity, unsigned sleep_ns = 64,
                                               unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 7u && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// D(16x8, f32) += A(16x16) * B(16x8), f16 operands.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ codes
// Two 4-bit codes of word w as fp16 subnormals, one AND each: pair i holds
// codes (i, i+4).  Even i: (q_i, q_{i+4}) * 2^-24.  Odd i: the mask keeps the
// nibbles in place, i.e. 16 * (q_i, q_{i+4}) * 2^-24; the matching
// activations are stored divided by 16, so every product is q * x * 2^-24
// exactly (fp16 subnormal inputs are exact in the tensor cores).  The group
// correction multiplies the accumulator by scale * 2^24.
template <int i>
__device__ __forceinline__ uint32_t codes_sub(uint32_t w) {
  if (i == 0) return w & 0x000F000Fu;
  if (i == 1) return w & 0x00F000F0u;
  if (i == 2) return (w >> 8) & 0x000F000Fu;
  return (w >> 8) & 0x00F000F0u;
}
constexpr float kCodeScale = 16777216.0f;  // 2^24

// Gate/up weight tiles (16 rows of gate, then 16 of up) arrive as 4-row
// blocks of consecutive rows, one bulk copy each, at quad_pitch bytes: 8 mod
// 32 words, so the rows 4q + i of blocks q = 0..3 fall in disjoint banks.
// mma row m of a tile holds tile row quad_row(m): each half-warp's four rows
// come from four different blocks, so the fragment loads are conflict free.
__host__ __device__ inline int quad_pitch(int H) { return 2 * H + 32; }  // 4 rows of H/2 bytes + 32
__host__ __device__ inline int quad_row(int m) { return 4 * (m & 3) + (m >> 2); }
// bytes of a gate/up tile: 8 blocks, then gate scale/bias and up scale/bias [16][H/64] bf16
__host__ __device__ inline int quad_tile_bytes(int H) { return 8 * quad_pitch(H) + 4 * 16 * (H / 64) * 2; }

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// The tanh form of GELU (Hendrycks & Gimpel 2016), the gate activation of
// the GeGLU experts: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))).
__device__ __forceinline__ float gelu_tanh(float z) {
  const float c0 = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * z * (1.0f + tanhf(c0 * fmaf(0.044715f * z, z * z, z)));
}

// bf16 pair -> fp16 pair (exact in fp16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t *>(&h);
}
// fp16 pair * 1/16 (exact unless the result is subnormal).
__device__ __forceinline__ uint32_t f16x2_div16(uint32_t w) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x2C002C00u));
  return r;
}

// float -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Operand order inside one 64-wide group.  The tensor-core fragments take
// the 4-bit codes of a thread's two packed words in the order produced by
// codes_sub<i>: pair i of word w holds codes (i, i+4).  The activation vector
// is stored in shared memory permuted so that each B fragment (4 values) is
// one 8-byte load.  Slot j = 16c + 4s + m of a group holds element
// 16c + 8(s>>1) + 2(s&1) + {0,4,1,5}[m].
// Builds the 16 permuted values of quarter c from its 16 natural values
// (8 words, each two 16-bit elements).
__device__ __forceinline__ void permute_quarter(const uint32_t (&in)[8], uint32_t (&out)[8]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {     // s>>1
#pragma unroll
    for (int e = 0; e < 2; ++e) {   // s&1
      const uint32_t a = in[4 * h + e];      // elements 8h+2e, 8h+2e+1
      const uint32_t b = in[4 * h + e + 2];  // elements 8h+2e+4, 8h+2e+5
      out[4 * h + 2 * e + 0] = __byte_perm(a, b, 0x5410);  // (8h+2e,   8h+2e+4)
      out[4 * h + 2 * e + 1] = __byte_perm(a, b, 0x7632);  // (8h+2e+1, 8h+2e+5)
    }
  }
}

// The B-operand form of one 16-element quarter: permuted, converted to fp16
// (kBf16: the input is bf16), odd words (the slots facing the x16 codes)
// divided by 16.
template <bool kBf16>
__device__ __forceinline__ void operand_quarter(const uint32_t (&in)[8], uint32_t (&out)[8]) {
  uint32_t h[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) h[w] = kBf16 ? bf16x2_to_f16x2(in[w]) : in[w];
  permute_quarter(h, out);
#pragma unroll
  for (int w = 1; w < 8; w += 2) out[w] = f16x2_div16(out[w]);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void set_error(unsigned *err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Optional launch trace (null when tracing is off).  Each launch owns 4
// u64 slots, all combined with atomicMax so a zeroed buffer is the reset
// state: [0] ~first block entry, [1] ~first block past the dependency wait,
// [2] last block with its weights in shared memory, [3] last block exit.
enum TraceSlot { kTrEntry = 0, kTrWaited = 1, kTrLoaded = 2, kTrExit = 3 };
__device__ __forceinline__ void trace_min(unsigned long long *tr, int slot) {
  if (tr) atomicMax(tr + slot, ~global_ns());
}
__device__ __forceinline__ void trace_max(unsigned long long *tr, int slot) {
  if (tr) atomicMax(tr + slot, global_ns());
}

}  // namespace moe
