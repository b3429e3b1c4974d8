// Router projection (8-bit affine GEMV), top-k with softmax weights, and the
// token/expert grouping (stable counting sort), sm_103a.
//
// Page "TurboFieldfare - System design": section "Decode" (the router
// normalises and projects the hidden state to one score per expert, keeps
// the 8 highest and softmaxes over them), section "Why the runtime has this
// shape" (8-bit affine router, no router softcap), section "Prefill"
// (token/expert pairs of a chunk are grouped per expert).
//
// One launch does the whole router: every block computes the logits of 8
// experts for up to 8 tokens; the last block to finish (ticket on a device
// counter) selects the top-k of every token, writes the softmax weights and
// groups the pairs, so no second launch is needed.  Decode (T = 1) is bound
// by the 383 KB of router weights; the block count is kept small (16) so the
// last-block epilogue starts early.
#include <math.h>

#include "kernels.h"

namespace moe {

namespace {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kExpertsPerBlock = kWarps;  // one warp per expert row
}  // namespace

// -------------------------------------------------------------- grouping
// Stable counting sort of the pairs p = t*k + j by expert id, run by one
// whole block of 256 threads.  Pairs whose id is outside [0, E) are dropped
// (pos = -1) and flagged.  Writes counts, offsets (offsets[E] = kept pairs),
// perm, pos and, if r.act_e is set, the list of active slots (slot 0 = the
// shared expert when include_shared, then experts with rows by ascending id).
__device__ void group_pairs(const int32_t *ids, int T, int k, int E, const Routing &r, int include_shared,
                            unsigned *err) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_fill[kMaxExperts];
  __shared__ int s_wc[kWarps][kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = T * k;
  for (int e = tid; e < kMaxExperts; e += kThreads) {
    s_cnt[e] = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_wc[w][e] = 0;
  }
  __syncthreads();
  bool bad = false;
  for (int p = tid; p < n; p += kThreads) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&s_cnt[e], 1);
    else
      bad = true;
  }
  if (bad) set_error(err, kErrBadId);
  __syncthreads();
  if (warp == 0) {
    int c[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      c[i] = e < E ? s_cnt[e] : 0;
      sum += c[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int base = incl - sum;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      if (e < E) {
        s_fill[e] = base;
        r.offsets[e] = base;
        r.counts[e] = c[i];
      }
      base += c[i];
    }
    if (lane == 31) r.offsets[E] = incl;
    __syncwarp();
    if (r.act_e != nullptr) {
      int nact = include_shared ? 1 : 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 32 * j + lane;
        const bool f = e < E && s_cnt[e] > 0;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (f) {
          const int a = nact + __popc(m & lanemask_lt());
          r.act_e[a] = e;
          r.act_beg[a] = s_fill[e];
          r.act_cnt[a] = s_cnt[e];
        }
        nact += __popc(m);
      }
      if (lane == 0) {
        if (include_shared) {
          r.act_e[0] = kSharedSlot;
          r.act_beg[0] = T * k;
          r.act_cnt[0] = T;
        }
        r.n_act[0] = nact;
      }
    }
  }
  __syncthreads();
  for (int base = 0; base < n; base += kThreads) {
    const int p = base + tid;
    const int e = p < n ? ids[p] : -1;
    const bool valid = p < n && e >= 0 && e < E;
    const int key = valid ? e : (kMaxExperts + lane);  // invalid lanes never group
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lanemask_lt());
    if (valid && rank == 0) s_wc[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wc[w][e];
      const int q = s_fill[e] + before + rank;
      r.perm[q] = p;
      r.pos[p] = q;
    } else if (p < n) {
      r.pos[p] = -1;
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += kThreads) {
      int add = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        add += s_wc[w][e2];
        s_wc[w][e2] = 0;
      }
      s_fill[e2] += add;
    }
    __syncthreads();
  }
}

// Same result as group_pairs for n = T*k <= 32 pairs, computed by one warp
// with shuffles only (the decode path: no block-wide barriers).  Lane p owns
// pair p.
__device__ void group_pairs_warp(const int32_t *ids, int T, int k, int E, const Routing &r, int include_shared,
                                 unsigned *err) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  const int e = lane < n ? ids[lane] : -1;
  const bool valid = lane < n && e >= 0 && e < E;
  if (__any_sync(0xffffffffu, lane < n && !valid) && lane == 0) set_error(err, kErrBadId);
  const int key = valid ? e : 0x40000000 + lane;  // invalid pairs sort after every expert
  // stable rank: pairs with a smaller key, or the same key and a smaller index
  int rank = 0, nvalid = 0;
  for (int q = 0; q < n; ++q) {
    const int kq = __shfl_sync(0xffffffffu, key, q);
    rank += (kq < key) || (kq == key && q < lane);
    nvalid += kq < 0x40000000;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const bool leader = valid && (__popc(peers & lanemask_lt()) == 0);
  // distinct experts below mine (for the active-slot index)
  int below = 0;
  for (int q = 0; q < n; ++q) {
    const int kq = __shfl_sync(0xffffffffu, key, q);
    const bool lq = __shfl_sync(0xffffffffu, leader, q);
    below += lq && kq < key;
  }
  // every lane runs the same trip count: the shuffles need the whole warp
  for (int x0 = 0; x0 < E; x0 += 32) {
    const int x = x0 + lane;
    int c = 0, lt = 0;
    for (int q = 0; q < n; ++q) {
      const int kq = __shfl_sync(0xffffffffu, key, q);
      c += kq == x;
      lt += kq < x;
    }
    if (x < E) {
      r.counts[x] = c;
      r.offsets[x] = lt;
    }
  }
  if (lane == 0) r.offsets[E] = nvalid;
  if (lane < n) {
    if (valid) {
      r.perm[rank] = lane;
      r.pos[lane] = rank;
    } else {
      r.pos[lane] = -1;
    }
  }
  if (r.act_e != nullptr) {
    const int a0 = include_shared ? 1 : 0;
    if (leader) {
      r.act_e[a0 + below] = e;
      r.act_beg[a0 + below] = rank;
      r.act_cnt[a0 + below] = __popc(peers);
    }
    const int ndist = __popc(__ballot_sync(0xffffffffu, leader));
    if (lane == 0) {
      if (include_shared) {
        r.act_e[0] = kSharedSlot;
        r.act_beg[0] = T * k;
        r.act_cnt[0] = T;
      }
      r.n_act[0] = a0 + ndist;
    }
  }
}

// -------------------------------------------------------------- top-k
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Top-k of one token's logits by one warp (E <= 128: 4 candidates per lane).
// Ids come out by descending logit, ties to the lower id; weights are the
// softmax over the k selected logits.
__device__ void topk_token(const float *logits_row, int E, int k, int32_t *ids_out, float *wts_out,
                           int32_t *ids_user, float *wts_user, const float *expert_scale, unsigned *err) {
  const int lane = threadIdx.x & 31;
  float v[4];
  int id[4];
  bool nonfinite = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    id[i] = e;
    if (e < E) {
      const float x = __ldcg(logits_row + e);
      if (isfinite(x)) {
        v[i] = x;
      } else {
        v[i] = -INFINITY;
        nonfinite = true;
      }
    } else {
      v[i] = -INFINITY;
    }
  }
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) set_error(err, kErrNonFinite);
  unsigned taken = 0;
  float sel_v[kMaxTopK];
  int sel_i[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (!((taken >> i) & 1u) && beats(v[i], id[i], bv, bi)) {
          bv = v[i];
          bi = id[i];
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (beats(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      sel_v[j] = bv;
      sel_i[j] = bi;
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
  }
  const float m = sel_v[0];
  float ex[kMaxTopK];
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      ex[j] = expf(sel_v[j] - m);
      den += ex[j];
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k && lane == j) {
      const float wj = ex[j] / den * (expert_scale ? expert_scale[sel_i[j]] : 1.0f);
      ids_out[j] = sel_i[j];
      wts_out[j] = wj;
      if (ids_user) ids_user[j] = sel_i[j];
      if (wts_user) wts_user[j] = wj;
    }
  }
}

// -------------------------------------------------------------- router
// Up to kMaxRouterWords 32-bit code words per lane (H <= 4096).
constexpr int kMaxRouterWords = 32;
constexpr int kMaxVec = 2;  // 16-byte activation vectors per thread (H <= 4096)

template <int TB>
__global__ void __launch_bounds__(kThreads) router_kernel(const RouterArgs a) {
  extern __shared__ __align__(16) float sx[];  // [TB][H] fp32 copy of the inputs
  __shared__ float s_red[TB][kWarps];
  __shared__ float s_inv[TB];
  __shared__ int s_last;
  const int H = a.d.H, E = a.d.E, T = a.d.T, k = a.d.k, G = H / kGroup;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.y * TB;
  const int tb = min(TB, T - t0);
  const int nblocks = gridDim.x * gridDim.y;
  const int nwords = H / 4;  // code words per row

  // Router weights never change: pull this warp's expert row into registers
  // before waiting on the previous kernel.
  const bool tracer = blockIdx.x == 0 && blockIdx.y == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  const int e = blockIdx.x * kExpertsPerBlock + warp;
  uint32_t wq[kMaxRouterWords], wsb[kMaxRouterWords];
  if (e < E) {
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.w.router_q + (size_t)e * H);
    const uint16_t *srow = a.w.router_s + (size_t)e * G;
    const uint16_t *brow = a.w.router_b + (size_t)e * G;
#pragma unroll
    for (int m = 0; m < kMaxRouterWords; ++m) {
      const int c = lane + 32 * m;
      if (c < nwords) {
        wq[m] = __ldg(qrow + c);
        wsb[m] = (uint32_t)__ldg(srow + (c >> 4)) | ((uint32_t)__ldg(brow + (c >> 4)) << 16);
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);

  // stage the tile's inputs (fp32) -- all loads first, then the stores
  const int nvec = H / 8;
  uint4 u[TB][kMaxVec];
#pragma unroll
  for (int n = 0; n < TB; ++n)
#pragma unroll
    for (int v = 0; v < kMaxVec; ++v) {
      const int idx = tid + kThreads * v;
      if (n < tb && idx < nvec) {
        const uint16_t *src = (a.hres ? a.hres : a.x) + (size_t)(t0 + n) * H;
        u[n][v] = *reinterpret_cast<const uint4 *>(src + 8 * idx);
      }
    }
  if (a.normalize) {
    // rmsnorm without scale (fixed-order sums)
#pragma unroll
    for (int n = 0; n < TB; ++n) {
      float ss = 0.f;
#pragma unroll
      for (int v = 0; v < kMaxVec; ++v) {
        const int idx = tid + kThreads * v;
        if (n < tb && idx < nvec) {
          const uint32_t w4[4] = {u[n][v].x, u[n][v].y, u[n][v].z, u[n][v].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) s_red[n][warp] = ss;
    }
    __syncthreads();
    if (tid < tb) {
      float tot = 0.f;
      for (int w = 0; w < kWarps; ++w) tot += s_red[tid][w];
      s_inv[tid] = 1.0f / sqrtf(tot / (float)H + 1e-6f);
    }
    __syncthreads();
  }
#pragma unroll
  for (int n = 0; n < TB; ++n)
#pragma unroll
    for (int v = 0; v < kMaxVec; ++v) {
      const int idx = tid + kThreads * v;
      if (n < tb && idx < nvec) {
        const uint32_t w4[4] = {u[n][v].x, u[n][v].y, u[n][v].z, u[n][v].w};
        float f[8];
        uint32_t ob[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
          if (a.normalize) {
            const uint16_t lb = float_to_bf16_bits(lo * s_inv[n]), hb = float_to_bf16_bits(hi * s_inv[n]);
            ob[q] = (uint32_t)lb | ((uint32_t)hb << 16);
            lo = bf16_bits_to_float(lb);
            hi = bf16_bits_to_float(hb);
          }
          f[2 * q] = lo;
          f[2 * q + 1] = hi;
        }
        if (a.w.router_scale) {  // router input x * router_scale / sqrt(H)
          const uint4 rv = __ldg(reinterpret_cast<const uint4 *>(a.w.router_scale) + idx);
          const uint32_t r4[4] = {rv.x, rv.y, rv.z, rv.w};
          const float isq = rsqrtf((float)H);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] *= __uint_as_float(r4[q] << 16) * isq;
            f[2 * q + 1] *= __uint_as_float(r4[q] & 0xFFFF0000u) * isq;
          }
        }
        float4 *dst = reinterpret_cast<float4 *>(sx + n * H + 8 * idx);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        if (a.normalize && blockIdx.x == 0) {
          const size_t o = (size_t)(t0 + n) * H + 8 * idx;
          *reinterpret_cast<uint4 *>(a.xn + o) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
          if (a.xn_user) *reinterpret_cast<uint4 *>(a.xn_user + o) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        }
      }
    }
  __syncthreads();

  // logits of expert e (one warp) for the tile's tokens: w = q*s + b in
  // fp32, dotted with x; lane l covers codes 4c..4c+3, c = l + 32m.
  float acc[TB];
#pragma unroll
  for (int n = 0; n < TB; ++n) acc[n] = 0.f;
  if (e < E) {
#pragma unroll
    for (int m = 0; m < kMaxRouterWords; ++m) {
      const int c = lane + 32 * m;
      if (c < nwords) {
        const float s = bf16_bits_to_float(wsb[m] & 0xFFFFu);
        const float b = bf16_bits_to_float(wsb[m] >> 16);
        float w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float q = __uint_as_float(0x4B000000u | ((wq[m] >> (8 * i)) & 0xFFu)) - 8388608.0f;
          w4[i] = fmaf(q, s, b);
        }
#pragma unroll
        for (int n = 0; n < TB; ++n) {
          if (n < tb) {
            const float4 xv = *reinterpret_cast<const float4 *>(sx + n * H + 4 * c);
            float t = acc[n];
            t = fmaf(w4[0], xv.x, t);
            t = fmaf(w4[1], xv.y, t);
            t = fmaf(w4[2], xv.z, t);
            t = fmaf(w4[3], xv.w, t);
            acc[n] = t;
          }
        }
      }
    }
  }
#pragma unroll
  for (int n = 0; n < TB; ++n) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
  }
  if (e < E && lane == 0) {
    const float bias = a.w.logit_bias ? a.w.logit_bias[e] : 0.f;
#pragma unroll
    for (int n = 0; n < TB; ++n)
      if (n < tb) a.logits[(size_t)(t0 + n) * E + e] = acc[n] + bias;
  }

  // last block to finish selects, weights and groups
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(a.counter, 1u);
    s_last = ticket == (unsigned)(nblocks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) trace_max(a.trace, kTrLoaded);  // all logits written
  if (T * k <= 32) {
    // decode-sized: one warp does everything, no block barriers
    if (warp == 0) {
      for (int t = 0; t < T; ++t)
        topk_token(a.logits + (size_t)t * E, E, k, a.r.ids + t * k, a.r.wts + t * k,
                   a.ids_user ? a.ids_user + t * k : nullptr, a.wts_user ? a.wts_user + t * k : nullptr,
                   a.w.expert_scale, a.err);
      __syncwarp();
      group_pairs_warp(a.r.ids, T, k, E, a.r, 1, a.err);
      if (lane == 0) {
        *a.counter = 0u;
        trace_max(a.trace, kTrExit);
      }
    }
    return;
  }
  for (int t = warp; t < T; t += kWarps)
    topk_token(a.logits + (size_t)t * E, E, k, a.r.ids + t * k, a.r.wts + t * k,
               a.ids_user ? a.ids_user + t * k : nullptr, a.wts_user ? a.wts_user + t * k : nullptr,
                   a.w.expert_scale, a.err);
  __syncthreads();
  group_pairs(a.r.ids, T, k, E, a.r, 1, a.err);
  if (tid == 0) {
    *a.counter = 0u;
    trace_max(a.trace, kTrExit);
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// ever completes; after limit_ns it records kErrTimeout and returns.
__global__ void wait_timeout_kernel(unsigned *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) set_error(err, kErrTimeout);
  }
}

cudaError_t launch_wait_timeout(unsigned *err, unsigned long long limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

// One block: group caller-given ids (moe_route_sort, moe_expert_ffn).
__global__ void __launch_bounds__(kThreads) sort_kernel(const SortArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  if (a.T * a.k <= 32) {
    if (threadIdx.x < 32) group_pairs_warp(a.ids, a.T, a.k, a.E, a.r, a.include_shared, a.err);
    return;
  }
  group_pairs(a.ids, a.T, a.k, a.E, a.r, a.include_shared, a.err);
}

size_t router_smem(const Dims &d, int tb) { return (size_t)tb * d.H * sizeof(float); }

static int router_tb(const Dims &d) { return d.T == 1 ? 1 : 8; }

cudaError_t launch_router(const RouterArgs &a, cudaStream_t st, bool pdl) {
  const int tb = router_tb(a.d);
  const dim3 grid((a.d.E + kExpertsPerBlock - 1) / kExpertsPerBlock, (a.d.T + tb - 1) / tb);
  const size_t smem = router_smem(a.d, tb);
  if (tb == 1) return launch_k(router_kernel<1>, grid, dim3(kThreads), smem, st, pdl, a);
  return launch_k(router_kernel<8>, grid, dim3(kThreads), smem, st, pdl, a);
}

cudaError_t launch_sort(const SortArgs &a, cudaStream_t st, bool pdl) {
  return launch_k(sort_kernel, dim3(1), dim3(kThreads), 0, st, pdl, a);
}

cudaError_t router_set_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(router_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  if ((e = cudaFuncSetAttribute(router_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024))) return e;
  return cudaSuccess;
}

}  // namespace moe
