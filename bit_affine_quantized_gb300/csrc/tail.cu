// Layer tail (page "TurboFieldfare - System design", section "Decode", cb2
// phase: after the combine of the routed and shared branches, the post-FFN
// norm, the residual and the learned layer scalar), one block per token:
//
//   z = bf16(y / sqrt(mean(y^2) + 1e-6) * g)     (z = y without a norm weight)
//   s = bf16(h + z)
//   h <- bf16(lambda * s)                         (h <- s without a scalar)
//
// y is the block's bf16 output, h the residual stream (updated in place), g
// the norm weight (bf16 [H]) and lambda the layer scalar (fp32, on the
// device).  HBM-bound: per token it reads y, h and g and writes h once
// (y is read a second time from L1/L2 after the sum of squares).
#include "kernels.h"

namespace moe {

namespace {
constexpr int kTailThreads = 256;
constexpr float kTailEps = 1e-6f;

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kTailThreads) tail_kernel(const TailArgs a) {
  __shared__ float s_part[kTailThreads / 32];
  const int H = a.H, t = blockIdx.x, tid = threadIdx.x;
  const int n8 = H / 8;
  const bool tracer = t == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);
  const uint4 *y4 = reinterpret_cast<const uint4 *>(a.y + (size_t)t * H);
  uint4 *h4 = reinterpret_cast<uint4 *>(a.h + (size_t)t * H);
  const uint4 *g4 = reinterpret_cast<const uint4 *>(a.post_norm);
  float inv = 1.0f;
  if (a.post_norm) {
    float ss = 0.f;
    for (int i = tid; i < n8; i += kTailThreads) {
      const uint4 v = __ldcg(y4 + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) ss = fmaf(lo_f(w[q]), lo_f(w[q]), fmaf(hi_f(w[q]), hi_f(w[q]), ss));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kTailThreads / 32; ++w) tot += s_part[w];
    inv = 1.0f / sqrtf(tot / (float)H + kTailEps);
  }
  const float lambda = a.layer_scalar ? __ldg(a.layer_scalar) : 1.0f;
  for (int i = tid; i < n8; i += kTailThreads) {
    const uint4 yv = __ldcg(y4 + i), hv = h4[i];
    const uint4 gv = a.post_norm ? __ldg(g4 + i) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t ow[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float z0 = lo_f(yw[q]), z1 = hi_f(yw[q]);
      if (a.post_norm) {
        z0 = bf16_bits_to_float(float_to_bf16_bits(z0 * inv * lo_f(gw[q])));
        z1 = bf16_bits_to_float(float_to_bf16_bits(z1 * inv * hi_f(gw[q])));
      }
      float s0 = bf16_bits_to_float(float_to_bf16_bits(lo_f(hw[q]) + z0));
      float s1 = bf16_bits_to_float(float_to_bf16_bits(hi_f(hw[q]) + z1));
      if (a.layer_scalar) {
        s0 *= lambda;
        s1 *= lambda;
      }
      ow[q] = (uint32_t)float_to_bf16_bits(s0) | ((uint32_t)float_to_bf16_bits(s1) << 16);
    }
    h4[i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
  if (tracer) trace_max(a.trace, kTrExit);
}
}  // namespace

cudaError_t launch_tail(const TailArgs &a, cudaStream_t st, bool pdl) {
  return launch_k(tail_kernel, dim3(a.T), dim3(kTailThreads), 0, st, pdl, a);
}

}  // namespace moe
