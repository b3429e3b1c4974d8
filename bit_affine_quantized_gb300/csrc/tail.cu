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
// device).  Per token it reads y, h and g and writes h once, one 8-element
// vector per thread; h and g are loaded before the wait for the block's y.
#include "kernels.h"

namespace moe {

namespace {
constexpr int kTailThreads = 512;  // one 8-element vector per thread: H <= 4096
constexpr float kTailEps = 1e-6f;

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kTailThreads) tail_kernel(const TailArgs a) {
  __shared__ float s_part[kTailThreads / 32];
  const int H = a.H, t = blockIdx.x, tid = threadIdx.x;
  const bool mine = tid < H / 8;
  const bool tracer = t == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  // h, g and lambda do not come from the launch this one waits on: h was last
  // written by an earlier launch that every launch in between waited for
  // before letting its dependents start; g and lambda are weights
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 *h4 = reinterpret_cast<uint4 *>(a.h + (size_t)t * H);
  const uint4 hv = mine ? __ldcg(h4 + tid) : zero;
  const uint4 gv = mine && a.post_norm ? __ldg(reinterpret_cast<const uint4 *>(a.post_norm) + tid) : zero;
  const float lambda = a.layer_scalar ? __ldg(a.layer_scalar) : 1.0f;
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);
  const uint4 yv = mine ? __ldcg(reinterpret_cast<const uint4 *>(a.y + (size_t)t * H) + tid) : zero;
  const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  float inv = 1.0f;
  if (a.post_norm) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) ss = fmaf(lo_f(yw[q]), lo_f(yw[q]), fmaf(hi_f(yw[q]), hi_f(yw[q]), ss));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kTailThreads / 32; ++w) tot += s_part[w];
    inv = 1.0f / sqrtf(tot / (float)H + kTailEps);
  }
  if (!mine) return;
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
  h4[tid] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  if (tracer) trace_max(a.trace, kTrExit);
}
}  // namespace

cudaError_t launch_tail(const TailArgs &a, cudaStream_t st, bool pdl) {
  if (a.H % 8 || a.H > 8 * kTailThreads || a.T < 1) return cudaErrorInvalidValue;
  return launch_k(tail_kernel, dim3(a.T), dim3(kTailThreads), 0, st, pdl, a);
}

}  // namespace moe
