// Dense expert slots of the multi-token kernel on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory).
//
// Page "TurboFieldfare - System design", section "Metal execution": prefill
// projections with enough rows go to matrix operations, after one bounded
// weight tile is dequantised into FP16 on-chip memory.  Here a slot (an
// expert, or the shared expert) whose rows in the chunk reach a threshold is
// a dense contraction: per 64-wide K group the producer warp loads the
// 4-bit codes of 128 weight rows and the chunk's operand rows with tensor
// TMA copies, the consumer warps dequantise the codes into an fp16 A tile
// (w = q * s + b rounded once to fp16, the K order and the /16 of the odd
// words matching the operand rows), and one thread issues tcgen05.mma with
// M = 128 weight rows, N = the chunk's rows, the fp32 sums staying in tensor
// memory across all K groups.
//
// Shared-memory operands:
//   A  [128 rows x 64 k] fp16 per matrix, written by the consumer threads
//   B  [128 rows x 64 k] fp16 written by the TMA
// both K-major with the 128-byte swizzle: row r at 128 r bytes (8-row atoms
// of 1024 bytes), its 16-byte chunk j stored at chunk j ^ (r mod 8).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace dense {

constexpr int kRows = 128;   // weight rows per unit (the MMA M)
constexpr int kMaxN = 128;   // chunk rows per unit (the MMA N, a multiple of 16)
constexpr int kStages = 3;   // TMA stages (codes + operand rows of one K group)
constexpr int kAhead = 8;    // K groups whose codes are prefetched into L2 ahead of their TMA
// A slot with at least this many rows in the chunk is dense.  Measured on
// GB300: a dense gate/up unit (128 rows, K = 2816) costs about 40 light
// units of 16 rows x 8 tokens; for a slot of r rows the light path spends
// 8 ceil(r / 8) of them per 128 rows, so the dense path wins clearly from
// about 96 rows on (the shared expert and the heaviest experts of a chunk).
constexpr int kMinRows = 96;
// cost of one dense gate/up unit (128 rows of gate and up, all the chunk's
// rows) and of one dense down unit (128 rows of down) in light units (16
// gate/up rows or 128 down rows for 8 tokens): sizes the set of blocks that
// take the dense units (measured on GB300)
constexpr float kGuCost = 40.0f;
constexpr float kDnCost = 8.0f;

// Tensor maps of the dense path (encoded on the host for each call).
struct Maps {
  CUtensorMap x;      // operand rows of the chunk's tokens: fp16 [T][H], box {64, 128}, 128B swizzle
  CUtensorMap h;      // operand rows of h per sorted position: fp16 [T*k+T][I], box {64, 128}, 128B swizzle
  CUtensorMap gq[2];  // gate codes: [0] routed experts {H/2 bytes, I rows, E}, [1] the shared expert; box {32, 128, 1}
  CUtensorMap uq[2];  // up codes, the same
  CUtensorMap dq[2];  // down codes {I/2 bytes, H rows, E}; box {32, 128, 1}
};

// Shared-memory plan of a dense block (offsets from a 1024-aligned base).
struct Plan {
  int b[kStages];     // operand rows, 16 KB each
  int c[kStages];     // codes: gate [128][32 B] then up [128][32 B]
  int a[2];           // dequantised A: gate 16 KB then up 16 KB
  int s;              // scales and biases of the unit: [matrix][s, b][128 rows][groups] bf16
  int total;
};
__host__ __device__ inline Plan plan(int G) {
  Plan p;
  int o = 0;
  for (int i = 0; i < kStages; ++i) {
    p.b[i] = o;
    o += kRows * 128;
  }
  for (int i = 0; i < kStages; ++i) {
    p.c[i] = o;
    o += 2 * kRows * 32;
  }
  for (int i = 0; i < 2; ++i) {
    p.a[i] = o;
    o += 2 * kRows * 64 * 2;
  }
  p.s = o;
  o += 4 * kRows * G * 2;
  p.total = o;
  return p;
}

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// Prefetch of a 3-D tensor box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(c0), "r"(c1),
               "r"(c2)
               : "memory");
}

// Shared-memory matrix descriptor: start address, leading (K-direction) and
// stride (row-direction) byte offsets between core matrices, layout
// (0: no swizzle, 2: 128-byte swizzle); bits 46-47 = 1 for this architecture.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46) | ((uint64_t)layout << 61);
}
// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ dequantisation
// One code word (8 codes of a row, k positions 8j .. 8j+7 of its group) as the
// 16 bytes of A tile core column j: the four fp16 pairs in operand order
// (codes (0,4), 16*(1,5), (2,6), 16*(3,7), matching the operand rows'
// permutation and their odd words stored / 16), w = q * s + b with one fp16
// rounding (q, 16 q and s, b are exact in fp16; the fused multiply-add rounds
// once).  s2 = (s, s), b2 = (b, b), b16 = (16 b, 16 b) as fp16 pairs.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t b16) {
  const uint32_t magic = 0x64006400u;  // fp16 pair (1024, 1024): 1024 + c is exact for c < 1024
  const uint32_t p0 = codes_sub<0>(w) | magic, p1 = codes_sub<1>(w) | magic;
  const uint32_t p2 = codes_sub<2>(w) | magic, p3 = codes_sub<3>(w) | magic;
  uint4 o;
  asm("{\n .reg .b32 t;\n sub.rn.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %4;\n}\n"
      : "=r"(o.x) : "r"(p0), "r"(magic), "r"(s2), "r"(b2));
  asm("{\n .reg .b32 t;\n sub.rn.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %4;\n}\n"
      : "=r"(o.y) : "r"(p1), "r"(magic), "r"(s2), "r"(b16));
  asm("{\n .reg .b32 t;\n sub.rn.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %4;\n}\n"
      : "=r"(o.z) : "r"(p2), "r"(magic), "r"(s2), "r"(b2));
  asm("{\n .reg .b32 t;\n sub.rn.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %4;\n}\n"
      : "=r"(o.w) : "r"(p3), "r"(magic), "r"(s2), "r"(b16));
  return o;
}

__device__ __forceinline__ uint32_t f16x2_of(float v) {
  const __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Slot index inside a 64-group of the operand order for group element e
// (the inverse of the permutation the operand rows use), and whether that
// slot's word is an odd one (stored / 16).
__device__ __forceinline__ int operand_slot(int e, bool &odd) {
  const int c = e >> 4, hi = (e >> 3) & 1, f = e & 7;
  const int m = (f & 1) ? ((f & 4) ? 3 : 2) : ((f & 4) ? 1 : 0);
  odd = (f & 1) != 0;
  return 16 * c + 4 * (2 * hi + ((f >> 1) & 1)) + m;
}

}  // namespace dense
}  // namespace moe
