// The tied 4-bit head and embedding (page "TurboFieldfare - System design":
// section "Why the runtime has this shape" - the embedding and the
// language-model head share one 4-bit affine matrix and the model ends with a
// logit softcap of 30; section "Decode" - the head returns the argmax token in
// a pure-greedy configuration, else the full logits).
//
// head_kernel: logits[t, v] = cap * tanh(sum_k w[v, k] x[t, k] / cap) for up
// to 8 tokens, w = q * s + b per 64-wide group; with no cap and no argmax it
// is the plain dense 4-bit projection (the attention's Q/K/V and output
// projections use the same format).  An HBM-bound GEMV over the
// whole vocabulary: every warp streams 16-row units straight from global
// memory (per row pair and group each lane loads 8 bytes of codes, so the
// 4 lanes of a quad cover one 32-byte sector of a row), the products run on
// the tensor cores (mma m16n8k16 with the codes as fp16 subnormals and the
// tokens as the N dimension), and the per-group affine correction
// s * acc * 2^24 + b * sum(x) is applied in fp32.  Loads of the next groups
// are issued before the current ones are used.  Greedy tokens: every warp
// keeps its best (logit, id) per token, merges them with one 64-bit atomicMax
// per warp and token into a small state the handle owns, and the last block
// to finish writes the ids and clears the state.
//
// embed_kernel: one block per id; the dequantised row, q * s + b formed
// exactly in double and rounded once to bf16.
#include <math.h>

#include "kernels.h"

namespace moe {

namespace {
constexpr int kHeadWarps = 8;
constexpr int kHeadThreads = kHeadWarps * 32;
constexpr int kHeadRows = 16;   // rows of one unit (the mma M)
constexpr int kHeadAhead = 4;   // groups whose codes are in flight per warp

struct HeadLayout {
  int xperm, xsum, qsum, sb, total;
};

// Shared memory of a head block: the tokens' operand rows (fp16, permuted
// per group as the fragments read them, odd words / 16), their group sums,
// the quarter sums they come from, and per warp the scales and biases of its
// current unit ([16][G] bf16 each).
__host__ __device__ inline HeadLayout head_layout(int H, int T) {
  const int G = H / kGroup;
  HeadLayout L;
  int o = 0;
  L.xperm = o;
  o += T * H * 2;
  L.xsum = o;
  o += T * G * 4;
  L.qsum = o;
  o += T * (H / 16) * 4;
  L.sb = (o + 15) & ~15;
  o = L.sb + kHeadWarps * 2 * kHeadRows * G * 2;
  L.total = o;
  return L;
}

__device__ __forceinline__ uint2 ld_stream(const uint8_t *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Orders floats as unsigned integers (larger float, larger key).
__device__ __forceinline__ unsigned head_key(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (logit, id) packed so that the larger logit, then the lower id, compares larger.
__device__ __forceinline__ unsigned long long pack_best(float v, unsigned id) {
  return ((unsigned long long)head_key(v) << 32) | (0xFFFFFFFFu - id);
}

// One 64-wide group of a unit: rows r and r + 8, tokens 2cq and 2cq + 1.
__device__ __forceinline__ void head_group(uint2 w0, uint2 w1, int g, int r, int cq, int T, int H, int G,
                                           const uint8_t *xperm, const float *xsum, const uint16_t *ssb,
                                           float (&t)[4]) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint8_t *xb = xperm + (size_t)r * H * 2 + g * 128 + cq * 32;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint2 bx = r < T ? *reinterpret_cast<const uint2 *>(xb + s * 8) : make_uint2(0u, 0u);
    const uint32_t x0 = (s >> 1) ? w0.y : w0.x, x1 = (s >> 1) ? w1.y : w1.x;
    uint32_t A[4];
    if ((s & 1) == 0) {
      A[0] = codes_sub<0>(x0); A[1] = codes_sub<0>(x1); A[2] = codes_sub<1>(x0); A[3] = codes_sub<1>(x1);
    } else {
      A[0] = codes_sub<2>(x0); A[1] = codes_sub<2>(x1); A[2] = codes_sub<3>(x0); A[3] = codes_sub<3>(x1);
    }
    mma_f16(acc, A, bx.x, bx.y);
  }
  const int ta = 2 * cq, tb = 2 * cq + 1;
  const float xsa = ta < T ? xsum[ta * G + g] : 0.f, xsb = tb < T ? xsum[tb * G + g] : 0.f;
  const float s0 = bf16_bits_to_float(ssb[r * G + g]) * kCodeScale;
  const float s1 = bf16_bits_to_float(ssb[(r + 8) * G + g]) * kCodeScale;
  const float b0 = bf16_bits_to_float(ssb[kHeadRows * G + r * G + g]);
  const float b1 = bf16_bits_to_float(ssb[kHeadRows * G + (r + 8) * G + g]);
  t[0] = fmaf(b0, xsa, fmaf(s0, acc[0], t[0]));
  t[1] = fmaf(b0, xsb, fmaf(s0, acc[1], t[1]));
  t[2] = fmaf(b1, xsa, fmaf(s1, acc[2], t[2]));
  t[3] = fmaf(b1, xsb, fmaf(s1, acc[3], t[3]));
}

__global__ void __launch_bounds__(kHeadThreads) head_kernel(const HeadArgs a) {
  extern __shared__ __align__(16) uint8_t hsm[];
  __shared__ int s_last;
  const int T = a.T, H = a.H, G = H / kGroup, V = a.V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, cq = lane & 3;
  const HeadLayout L = head_layout(H, T);
  uint8_t *xperm = hsm + L.xperm;
  float *xsum = reinterpret_cast<float *>(hsm + L.xsum);
  float *qsum = reinterpret_cast<float *>(hsm + L.qsum);
  uint16_t *ssb = reinterpret_cast<uint16_t *>(hsm + L.sb) + warp * 2 * kHeadRows * G;
  const bool tracer = blockIdx.x == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);

  // operand rows of the tokens, 16 elements (one quarter of a group) per step
  const int nq = H / 16;
  for (int i = tid; i < T * nq; i += kHeadThreads) {
    const int t = i / nq, c = i - t * nq;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H + c * 16);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += bf16_bits_to_float(in[w] & 0xFFFFu) + bf16_bits_to_float(in[w] >> 16);
    uint32_t out[8];
    operand_quarter<true>(in, out);
    uint4 *dst = reinterpret_cast<uint4 *>(xperm + (size_t)t * H * 2 + c * 32);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    qsum[i] = sum;
  }
  __syncthreads();
  for (int i = tid; i < T * G; i += kHeadThreads) {
    const float *q = qsum + (size_t)(i / G) * nq + (i % G) * 4;
    xsum[i] = ((q[0] + q[1]) + q[2]) + q[3];
  }
  __syncthreads();

  const float cap = a.softcap;
  const bool want_tokens = a.tokens != nullptr;
  unsigned long long best[2] = {0ull, 0ull};
  bool bad = false;
  const int n_units = V / kHeadRows;
  const size_t row_bytes = (size_t)H / 2;
  for (int u = blockIdx.x * kHeadWarps + warp; u < n_units; u += gridDim.x * kHeadWarps) {
    const size_t row0 = (size_t)u * kHeadRows;
    // this unit's scales, then biases: 16 * G bf16 each, contiguous
    {
      const uint4 *s4 = reinterpret_cast<const uint4 *>(a.s + row0 * G);
      const uint4 *b4 = reinterpret_cast<const uint4 *>(a.b + row0 * G);
      uint4 *d4 = reinterpret_cast<uint4 *>(ssb);
      const int n4 = kHeadRows * G * 2 / 16;
      for (int i = lane; i < n4; i += 32) {
        d4[i] = __ldg(s4 + i);
        d4[n4 + i] = __ldg(b4 + i);
      }
    }
    __syncwarp();
    const uint8_t *q0 = reinterpret_cast<const uint8_t *>(a.q) + (row0 + r) * row_bytes + cq * 8;
    const uint8_t *q1 = q0 + 8 * row_bytes;
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    uint2 wa[kHeadAhead], wb[kHeadAhead];
#pragma unroll
    for (int j = 0; j < kHeadAhead; ++j) {
      wa[j] = j < G ? ld_stream(q0 + j * 32) : make_uint2(0u, 0u);
      wb[j] = j < G ? ld_stream(q1 + j * 32) : make_uint2(0u, 0u);
    }
    for (int g0 = 0; g0 < G; g0 += kHeadAhead) {
      uint2 na[kHeadAhead], nb[kHeadAhead];
#pragma unroll
      for (int j = 0; j < kHeadAhead; ++j) {
        const int g = g0 + kHeadAhead + j;
        na[j] = g < G ? ld_stream(q0 + g * 32) : make_uint2(0u, 0u);
        nb[j] = g < G ? ld_stream(q1 + g * 32) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kHeadAhead; ++j)
        if (g0 + j < G) head_group(wa[j], wb[j], g0 + j, r, cq, T, H, G, xperm, xsum, ssb, t);
#pragma unroll
      for (int j = 0; j < kHeadAhead; ++j) {
        wa[j] = na[j];
        wb[j] = nb[j];
      }
    }
    __syncwarp();  // every lane is done with ssb before the next unit overwrites it
    // softcap, logits out, best per token: t[0..3] = (row r, 2cq), (r, 2cq+1), (r+8, 2cq), (r+8, 2cq+1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * cq + (i & 1);
      const unsigned row = (unsigned)(row0 + r + 8 * (i >> 1));
      float v = cap > 0.f ? cap * tanhf(t[i] / cap) : t[i];
      if (tok < T) {
        if (a.logits) a.logits[(size_t)tok * V + row] = v;
        if (a.out_bf16) a.out_bf16[(size_t)tok * V + row] = float_to_bf16_bits(v);
        if (!isfinite(v)) {
          bad = true;
          v = -INFINITY;
        }
        const unsigned long long key = pack_best(v, row);
        if (key > best[i & 1]) best[i & 1] = key;
      }
    }
  }
  if (bad) set_error(a.err, kErrNonFinite);
  if (!want_tokens) {
    if (tracer) trace_max(a.trace, kTrExit);
    return;
  }
  // best over the 8 lanes of each token pair (lanes with equal cq), then one atomic per warp and token
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best[i], off);
      if (o > best[i]) best[i] = o;
    }
  }
  if (r == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (2 * cq + i < T && best[i] != 0ull) atomicMax(a.best + 2 * cq + i, best[i]);
    __threadfence();  // this thread's maxima are visible before the block takes its ticket
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  // the last block: ids out, and the state back to zero for the next launch
  if (s_last && tid < T) {
    __threadfence();
    const unsigned long long v = atomicExch(a.best + tid, 0ull);
    a.tokens[tid] = (int32_t)(0xFFFFFFFFu - (unsigned)(v & 0xFFFFFFFFull));
  }
  if (s_last && tid == 0) atomicExch(a.counter, 0u);
  if (tracer) trace_max(a.trace, kTrExit);
}

// Round a double to the nearest bf16 (ties to even), for values in bf16's
// normal range or zero; smaller magnitudes go through fp32 (they are far
// below any weight of interest and within one bf16 step of zero).
__device__ __forceinline__ uint16_t bf16_from_double(double v) {
  const unsigned long long u = (unsigned long long)__double_as_longlong(v);
  const unsigned long long mag = u & 0x7FFFFFFFFFFFFFFFull;
  const unsigned sign = (unsigned)(u >> 63);
  if (mag == 0ull) return (uint16_t)(sign << 15);
  const int e = (int)(mag >> 52) - 1023;
  if (e < -126 || e > 127) return float_to_bf16_bits((float)v);
  // keep the exponent and 7 fraction bits: drop 45 bits, round half to even
  unsigned long long keep = mag >> 45;
  const unsigned long long rem = mag & ((1ull << 45) - 1ull);
  const unsigned long long half = 1ull << 44;
  if (rem > half || (rem == half && (keep & 1ull))) ++keep;
  const unsigned long long e16 = (keep >> 7) - 1023ull + 127ull;  // a carry into the exponent is kept
  return (uint16_t)((sign << 15) | (unsigned)((e16 << 7) | (keep & 0x7Full)));
}

__global__ void __launch_bounds__(256) embed_kernel(const EmbedArgs a) {
  const int i = blockIdx.x, H = a.H, G = H / kGroup;
  pdl_wait();  // the ids may come from the launch before (the head's tokens)
  pdl_launch_dependents();
  const int id = a.ids[i];
  const bool ok = id >= 0 && id < a.V;
  if (!ok && threadIdx.x == 0) set_error(a.err, kErrBadId);
  uint4 *out = reinterpret_cast<uint4 *>(a.out + (size_t)i * H);
  for (int w = threadIdx.x; w < H / 8; w += blockDim.x) {
    uint32_t o[4] = {0u, 0u, 0u, 0u};
    if (ok) {
      const uint32_t word = __ldg(a.q + (size_t)id * (H / 8) + w);
      const int g = w / 8;
      const double s = (double)bf16_bits_to_float(__ldg(a.s + (size_t)id * G + g));
      const double b = (double)bf16_bits_to_float(__ldg(a.b + (size_t)id * G + g));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const double q = (double)((word >> (4 * j)) & 15u);
        const uint16_t bits = bf16_from_double(fma(q, s, b));
        o[j >> 1] |= (uint32_t)bits << (16 * (j & 1));
      }
    }
    out[w] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
}  // namespace

size_t head_smem(int H, int T) { return (size_t)head_layout(H, T).total; }

// The largest shared-memory request of any supported shape (H = 4096, 8
// tokens); the kernel also holds a few bytes of static shared memory, so the
// full 227 KB cannot be requested as dynamic memory.
cudaError_t head_set_attributes() {
  return cudaFuncSetAttribute(head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)head_smem(4096, kHeadMaxTokens));
}

cudaError_t launch_head(const HeadArgs &a, int n_blocks, cudaStream_t st, bool pdl) {
  if (a.T < 1 || a.T > kHeadMaxTokens || a.H % kGroup || a.V % kHeadRows || n_blocks < 1)
    return cudaErrorInvalidValue;
  return launch_k(head_kernel, dim3(n_blocks), dim3(kHeadThreads), head_smem(a.H, a.T), st, pdl, a);
}

int head_blocks_per_sm(int H, int T) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, head_kernel, kHeadThreads, head_smem(H, T)) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t st, bool pdl) {
  if (a.n < 1 || a.H % kGroup) return cudaErrorInvalidValue;
  return launch_k(embed_kernel, dim3(a.n), dim3(256), 0, st, pdl, a);
}

}  // namespace moe
