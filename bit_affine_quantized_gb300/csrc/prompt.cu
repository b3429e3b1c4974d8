// Whole-prompt MoE layer, sm_103a: the rows of a prompt (up to 4096) through
// one layer in six launches.
//
// Page "TurboFieldfare - System design", section "Prefill": execution is
// layer-major; the router scores every row, the token/expert pairs are
// grouped into bounded routed-MoE work, experts are streamed in tiles of at
// most eight and the next tile is fetched while the current tile's work is
// still queued, and the shared and routed branches are combined before the
// layer tail.  Section "Metal execution": prefill projections dequantise one
// bounded weight tile into FP16 on-chip memory and hand it to the matrix
// units.
//
// Here the weights stay resident in HBM and the "cache" the tiles stream
// through is the GPU's L2: every expert's weights come from HBM about once per
// layer for all of the prompt's rows instead of once per 128-row chunk.
//
//   prompt_router_kernel  16 rows per block, 16 warps: rmsnorm, the 8-bit
//                         router on the tensor cores (mma.m16n8k16, codes as
//                         exact fp16 integers, per-group affine correction in
//                         fp32), top-k and softmax per row.
//   prompt_sort_kernel    one block: stable counting sort of all pairs by
//                         expert, then the bounded chunks (at most 256 rows
//                         of one expert) in tile order: the shared expert,
//                         then experts 0-7, 8-15, ...
//   prompt_gather_kernel  the normalised rows at their sorted positions, in
//                         the operand order of the dense dequantisation.
//   prompt_gemm_kernel    persistent, one block per SM: a unit is one chunk
//                         against two 128-row weight matrices (gate and up
//                         rows of one 128-row tile of I, or two 128-row
//                         halves of a 256-row tile of W_down); per K group
//                         the producer warp loads the chunk's operand rows
//                         and the 4-bit codes with tensor TMA, 16 warps
//                         dequantise the codes into an fp16 A tile, one
//                         thread issues tcgen05.mma (M = 128 weight rows,
//                         N = the chunk's rows) into tensor memory, and 4
//                         epilogue warps apply GeGLU (gate/up) or the routing
//                         weight (down).  Each block prefetches its next
//                         unit's weights into L2 while the current unit runs.
//   combine_kernel        y[t] = sum of the token's weighted expert outputs
//                         in selection order + the shared expert's, added to
//                         the residual stream (ffn.cu).
#include <cuda.h>
#include <math.h>
#include <string.h>

#include "dense.cuh"
#include "fused.cuh"
#include "kernels.h"

namespace moe {
namespace {

// ------------------------------------------------------------------ router
constexpr int kRtTok = 16;        // rows per router block (one m16 tile)
constexpr int kRtThreads = 512;   // 16 warps, 8 experts (one n8 tile) each
constexpr int kRtNT = kMaxExperts / 8 / (kRtThreads / 32);  // n8 tiles per warp
constexpr int kRtGroups = 2;      // 64-wide K groups per code stage
constexpr int kRtCodePitch = 64 * kRtGroups + 16;  // bytes per expert row of a stage: rows 4 banks apart
constexpr int kRowVec = 16;       // 16-byte vectors of one row per lane (H <= 4096)

struct RtLayout {
  int xp, x, xs, sb, sbp, codes, total;  // sbp: byte offset of the biases after the scales (16-aligned)
};
__host__ __device__ inline RtLayout rt_layout(int H, int E, int kRtStages) {
  const int G = H / kGroup;
  RtLayout L;
  L.xp = 2 * H + 16;  // fp16 row pitch: consecutive rows 4 banks apart
  int o = 0;
  L.x = o;
  o += kRtTok * L.xp;
  L.xs = o;
  o += kRtTok * G * 4;
  L.sb = o;
  L.sbp = (E * G * 2 + 15) & ~15;
  o += 2 * L.sbp;
  L.codes = o;
  o += kRtStages * E * kRtCodePitch;
  L.total = o;
  return L;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Two 8-bit codes (little-endian pair) as an exact fp16 pair: the byte goes
// under the exponent of 1024, then 1024 is subtracted.
__device__ __forceinline__ uint32_t codes8_f16x2(uint32_t pair) {
  const uint32_t biased = __byte_perm(pair, 0x64646464u, 0x4140);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x64006400u));
  return r;
}

// kRtStages: code stages in flight (deeper when the row tile leaves room)
template <int kRtStages>
__global__ void __launch_bounds__(kRtThreads) prompt_router_kernel(const PromptArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = a.d.H, E = a.d.E, T = a.d.T, k = a.d.k, G = H / kGroup;
  const RtLayout L = rt_layout(H, E, kRtStages);
  uint8_t *sx = smem + L.x;
  float *sxs = reinterpret_cast<float *>(smem + L.xs);
  uint16_t *ssb = reinterpret_cast<uint16_t *>(smem + L.sb);            // scales [E][G]
  uint16_t *sbb = reinterpret_cast<uint16_t *>(smem + L.sb + L.sbp);    // biases [E][G]
  uint8_t *scodes = smem + L.codes;
  float *slogit = reinterpret_cast<float *>(scodes);  // [kRtTok][E], after the K loop
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTok, tb = min(kRtTok, T - t0);
  const int nst = (G + kRtGroups - 1) / kRtGroups;
  if (blockIdx.x == 0 && tid == 0) trace_min(a.trace, kTrEntry);

  // router weights never change: the first stages of codes and all scales
  // and biases are requested before the dependency wait
  auto load_stage = [&](int s) {
    if (s < nst) {
      const int g0 = s * kRtGroups, ng = min(kRtGroups, G - g0), per = 4 * ng;  // 16-byte pieces per row
      uint8_t *dst = scodes + (s % kRtStages) * E * kRtCodePitch;
      for (int i = tid; i < E * per; i += kRtThreads) {
        const int e = i / per, j = i - e * per;
        cp_async16(dst + e * kRtCodePitch + 16 * j, a.w.router_q + (size_t)e * H + 64 * g0 + 16 * j);
      }
    }
    cp_async_commit();
  };
  // scales and biases: 16-byte asynchronous copies (with the first code stage), the tail plainly
  {
    const int n16 = E * G * 2 / 16;
    for (int i = tid; i < 2 * n16; i += kRtThreads) {
      const int f = i >= n16, j = i - f * n16;
      cp_async16(reinterpret_cast<uint8_t *>(f ? sbb : ssb) + 16 * j,
                 reinterpret_cast<const uint8_t *>(f ? a.w.router_b : a.w.router_s) + 16 * j);
    }
    for (int i = 8 * n16 + tid; i < E * G; i += kRtThreads) {
      ssb[i] = __ldg(a.w.router_s + i);
      sbb[i] = __ldg(a.w.router_b + i);
    }
  }
  for (int s = 0; s < kRtStages - 1; ++s) load_stage(s);
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && tid == 0) trace_min(a.trace, kTrWaited);

  // rmsnorm of the block's rows (warp w: rows w, w + 8); normalised rows out
  // (bf16), router operand rows (fp16, natural order) and their 64-group sums
  const int nvec = H / 8;
  for (int rl = warp; rl < kRtTok; rl += kRtThreads / 32) {
    uint8_t *xrow = sx + rl * L.xp;
    if (rl >= tb) {  // rows past the prompt: zero operand
      for (int v = lane; v < nvec; v += 32) *reinterpret_cast<uint4 *>(xrow + 16 * v) = make_uint4(0u, 0u, 0u, 0u);
      for (int g = lane; g < G; g += 32) sxs[rl * G + g] = 0.f;
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(a.hres + (size_t)(t0 + rl) * H);
    uint4 u[kRowVec];  // the whole row, every load in flight at once
#pragma unroll
    for (int i = 0; i < kRowVec; ++i)
      if (lane + 32 * i < nvec) u[i] = __ldcg(src + lane + 32 * i);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
      if (lane + 32 * i < nvec) {
        const uint32_t w4[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
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
    const float inv = 1.0f / sqrtf(ss / (float)H + 1e-6f);
    const float isq = rsqrtf((float)H);
    // lanes 8q .. 8q+7 hold the eight vectors of one 64-group (nvec is a multiple of 8)
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
      const int v = lane + 32 * i;
      float gs = 0.f;
      if (v < nvec) {
        const uint32_t w4[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
        uint32_t ob[4], oh[4];
        uint4 rv = make_uint4(0u, 0u, 0u, 0u);
        if (a.w.router_scale) rv = __ldg(reinterpret_cast<const uint4 *>(a.w.router_scale) + v);
        const uint32_t r4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint16_t lb = float_to_bf16_bits(__uint_as_float(w4[q] << 16) * inv);
          const uint16_t hb = float_to_bf16_bits(__uint_as_float(w4[q] & 0xFFFF0000u) * inv);
          ob[q] = (uint32_t)lb | ((uint32_t)hb << 16);
          __half2 hv;
          if (a.w.router_scale)  // router input x * router_scale / sqrt(H), rounded once to fp16
            hv = __floats2half2_rn(bf16_bits_to_float(lb) * (__uint_as_float(r4[q] << 16) * isq),
                                   bf16_bits_to_float(hb) * (__uint_as_float(r4[q] & 0xFFFF0000u) * isq));
          else
            hv = __floats2half2_rn(bf16_bits_to_float(lb), bf16_bits_to_float(hb));
          oh[q] = *reinterpret_cast<const uint32_t *>(&hv);
          gs += __low2float(hv);
          gs += __high2float(hv);
        }
        *reinterpret_cast<uint4 *>(a.xn + (size_t)(t0 + rl) * H + 8 * v) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        if (a.xn_user)
          *reinterpret_cast<uint4 *>(a.xn_user + (size_t)(t0 + rl) * H + 8 * v) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        *reinterpret_cast<uint4 *>(xrow + 16 * v) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      }
      gs += __shfl_xor_sync(0xffffffffu, gs, 1);
      gs += __shfl_xor_sync(0xffffffffu, gs, 2);
      gs += __shfl_xor_sync(0xffffffffu, gs, 4);
      if ((lane & 7) == 0 && v < nvec) sxs[rl * G + v / 8] = gs;
    }
  }

  // logits: warp w owns experts 8 kRtNT w .. + 8 kRtNT - 1 for all 16 rows
  const int r = lane >> 2, c = lane & 3;
  const int n0 = 8 * kRtNT * warp;
  float tot[kRtNT][4];
#pragma unroll
  for (int nt = 0; nt < kRtNT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) tot[nt][i] = 0.f;
  for (int s = 0; s < nst; ++s) {
    cp_async_wait<kRtStages - 2>();
    __syncthreads();  // stage s landed for every thread; stage s - 1 fully consumed
    load_stage(s + kRtStages - 1);
    const uint8_t *cs = scodes + (s % kRtStages) * E * kRtCodePitch;
    const int g0 = s * kRtGroups, ng = min(kRtGroups, G - g0);
    if (n0 < E) {
      for (int gl = 0; gl < ng; ++gl) {
        const int g = g0 + gl;
        float acc[kRtNT][4];
#pragma unroll
        for (int nt = 0; nt < kRtNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const int kk = 64 * g + 16 * ks;
          uint32_t A[4];
          A[0] = *reinterpret_cast<const uint32_t *>(sx + r * L.xp + 2 * (kk + 2 * c));
          A[1] = *reinterpret_cast<const uint32_t *>(sx + (r + 8) * L.xp + 2 * (kk + 2 * c));
          A[2] = *reinterpret_cast<const uint32_t *>(sx + r * L.xp + 2 * (kk + 8 + 2 * c));
          A[3] = *reinterpret_cast<const uint32_t *>(sx + (r + 8) * L.xp + 2 * (kk + 8 + 2 * c));
#pragma unroll
          for (int nt = 0; nt < kRtNT; ++nt) {
            // experts past E (E not a multiple of 16) read expert E - 1: columns discarded below
            const uint8_t *crow = cs + min(n0 + 8 * nt + r, E - 1) * kRtCodePitch + 64 * gl + 16 * ks + 2 * c;
            const uint32_t b0 = codes8_f16x2(*reinterpret_cast<const uint16_t *>(crow));
            const uint32_t b1 = codes8_f16x2(*reinterpret_cast<const uint16_t *>(crow + 8));
            mma_f16(acc[nt], A, b0, b1);
          }
        }
        const float x0 = sxs[r * G + g], x1 = sxs[(r + 8) * G + g];
#pragma unroll
        for (int nt = 0; nt < kRtNT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = n0 + 8 * nt + 2 * c + (i & 1);
            const int ee = e < E ? e : E - 1;  // columns past E are discarded below
            const float sc = bf16_bits_to_float(ssb[ee * G + g]), bi = bf16_bits_to_float(sbb[ee * G + g]);
            tot[nt][i] = fmaf(bi, (i >> 1) ? x1 : x0, fmaf(sc, acc[nt][i], tot[nt][i]));
          }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the code stages become the logit table
#pragma unroll
  for (int nt = 0; nt < kRtNT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = n0 + 8 * nt + 2 * c + (i & 1), rl = r + 8 * (i >> 1);
      if (e < E) {
        const float v = tot[nt][i] + (a.w.logit_bias ? a.w.logit_bias[e] : 0.f);
        slogit[rl * E + e] = v;
        if (rl < tb) a.logits[(size_t)(t0 + rl) * E + e] = v;
      }
    }
  __syncthreads();
  for (int rl = warp; rl < tb; rl += kRtThreads / 32) {
    const int t = t0 + rl;
    bool bad = false;
    fused::warp_topk(slogit + rl * E, E, k, a.r.ids + (size_t)t * k, a.r.wts + (size_t)t * k, a.w.expert_scale, &bad);
    if (bad && lane == 0) set_error(a.err, kErrNonFinite);
    __syncwarp();
    if (lane < k) {
      if (a.ids_user) a.ids_user[(size_t)t * k + lane] = a.r.ids[(size_t)t * k + lane];
      if (a.wts_user) a.wts_user[(size_t)t * k + lane] = a.r.wts[(size_t)t * k + lane];
    }
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
}

// ------------------------------------------------------------------ grouping
constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortPer = kPromptMaxRows * kMaxTopK / (kSortWarps * 32);  // ids per lane
static_assert(kSortPer * kSortWarps * 32 >= kPromptMaxRows * kMaxTopK, "every pair has a lane");

// Exclusive scan of v over the 32 lanes of one warp; returns the lane's
// prefix and writes the total to *sum (every lane).
__device__ __forceinline__ int warp_excl_scan(int v, int *sum) {
  const int lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  *sum = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

// Lanes of the warp holding the same valid key e (E <= 128: seven key bits,
// one ballot each); a lane without a valid key is its own only peer.
__device__ __forceinline__ unsigned key_peers(int e, bool ok) {
  unsigned peers = __ballot_sync(0xffffffffu, ok);
#pragma unroll
  for (int b = 0; b < 7; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? bb : ~bb;
  }
  return ok ? peers : (1u << (threadIdx.x & 31));
}

__global__ void __launch_bounds__(kSortThreads) prompt_sort_kernel(const PromptArgs a) {
  __shared__ int s_hist[kSortWarps][kMaxExperts];  // pairs per (warp segment, expert), then segment bases
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_ch0[kMaxExperts + 1];           // first chunk of each expert
  const int T = a.d.T, k = a.d.k, E = a.d.E, n = T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) trace_min(a.trace, kTrWaited);
  for (int i = tid; i < kSortWarps * kMaxExperts; i += kSortThreads) (&s_hist[0][0])[i] = 0;
  __syncthreads();
  // each warp owns one contiguous segment of the pairs, 32 at a time in order
  const int seg = (n + kSortWarps - 1) / kSortWarps;  // <= kSortPer * 32
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  int ev[kSortPer];  // the segment's ids, every load in flight at once
#pragma unroll
  for (int q = 0; q < kSortPer; ++q) {
    const int p = s0 + 32 * q + lane;
    ev[q] = p < s1 ? __ldcg(a.r.ids + p) : -1;
  }
  bool bad = false;
#pragma unroll
  for (int q = 0; q < kSortPer; ++q) {
    if (s0 + 32 * q >= s1) break;  // warp-uniform
    const int p = s0 + 32 * q + lane, e = ev[q];
    const bool ok = p < s1 && e >= 0 && e < E;
    bad = bad || (p < s1 && !ok);
    const unsigned peers = key_peers(e, ok);
    if (ok && (peers & lanemask_lt()) == 0) s_hist[warp][e] += __popc(peers);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(a.err, kErrBadId);
  __syncthreads();
  // expert offsets (warp 0: four experts per lane)
  if (warp == 0) {
    int cnt[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      cnt[i] = 0;
      if (e < E)
        for (int w = 0; w < kSortWarps; ++w) cnt[i] += s_hist[w][e];
      sum += cnt[i];
    }
    int total;
    int base = warp_excl_scan(sum, &total);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      if (e < E) {
        s_off[e] = base;
        a.r.offsets[e] = base;
        a.r.counts[e] = cnt[i];
      }
      base += cnt[i];
    }
    if (lane == 0) {
      s_off[E] = total;
      a.r.offsets[E] = total;
    }
  }
  __syncthreads();
  if (tid < E) {  // segment bases of expert tid, in segment order (stable)
    int run = s_off[tid];
    for (int w = 0; w < kSortWarps; ++w) {
      const int c = s_hist[w][tid];
      s_hist[w][tid] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kSortPer; ++q) {
    if (s0 + 32 * q >= s1) break;  // warp-uniform
    const int p = s0 + 32 * q + lane, e = ev[q];
    const bool ok = p < s1 && e >= 0 && e < E;
    const unsigned peers = key_peers(e, ok);
    if (ok) {
      const int q = s_hist[warp][e] + __popc(peers & lanemask_lt());
      a.r.perm[q] = p;
      a.r.pos[p] = q;
    } else if (p < s1) {
      a.r.pos[p] = -1;
    }
    __syncwarp();
    if (ok && (peers & lanemask_lt()) == 0) s_hist[warp][e] += __popc(peers);
    __syncwarp();
  }
  // bounded chunks: the shared expert's rows first, then every expert's
  // sorted positions in runs of at most kPromptChunk, experts in ascending id
  // (tiles of eight consecutive experts follow one another)
  const int nsh = (T + kPromptChunk - 1) / kPromptChunk;
  if (warp == 0) {
    int nc[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      nc[i] = e < E ? (s_off[e + 1] - s_off[e] + kPromptChunk - 1) / kPromptChunk : 0;
      sum += nc[i];
    }
    int total;
    int base = nsh + warp_excl_scan(sum, &total);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * lane + i;
      if (e < E) s_ch0[e] = base;
      base += nc[i];
    }
    if (lane == 0) *a.n_ch = nsh + total;
  }
  __syncthreads();
  for (int j = tid; j < nsh; j += kSortThreads) {
    a.ch_e[j] = kSharedSlot;
    a.ch_beg[j] = n + j * kPromptChunk;
    a.ch_cnt[j] = min(kPromptChunk, T - j * kPromptChunk);
  }
  for (int e = warp; e < E; e += kSortWarps) {
    const int beg = s_off[e], cnt = s_off[e + 1] - beg;
    for (int j = lane; j * kPromptChunk < cnt; j += 32) {
      a.ch_e[s_ch0[e] + j] = e;
      a.ch_beg[s_ch0[e] + j] = beg + j * kPromptChunk;
      a.ch_cnt[s_ch0[e] + j] = min(kPromptChunk, cnt - j * kPromptChunk);
    }
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
}

// ------------------------------------------------------------------ gather
constexpr int kGatherThreads = 256;

// One warp per sorted position: the normalised row of its token in the
// operand order (fp16 pairs permuted within each 16-element quarter, odd
// words divided by 16), the B operand of the dense gate/up units.
__global__ void __launch_bounds__(kGatherThreads) prompt_gather_kernel(const PromptArgs a) {
  const int T = a.d.T, k = a.d.k, H = a.d.H, E = a.d.E;
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5);
  if (blockIdx.x == 0 && threadIdx.x == 0) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) trace_min(a.trace, kTrWaited);
  const int n = T * k;
  // positions of dropped pairs (bad ids) are never read: no row for them
  int tok = -1;
  if (pos >= n && pos < n + T)
    tok = pos - n;
  else if (pos < n && pos < __ldcg(a.r.offsets + E))
    tok = __ldcg(a.r.perm + pos) / k;
  const uint4 *src = reinterpret_cast<const uint4 *>(a.xn + (size_t)(tok < 0 ? 0 : tok) * H);
  uint4 *dst = reinterpret_cast<uint4 *>(a.xg + (size_t)pos * H);
  uint4 v[2 * kRowVec / 2];  // quarters lane, lane + 32, ... (H <= 4096: 8 per lane), loaded at once
  constexpr int kQ = kRowVec / 2;
#pragma unroll
  for (int i = 0; i < kQ; ++i) {
    const int q = lane + 32 * i;
    if (tok >= 0 && q < H / 16) {
      v[2 * i] = __ldcg(src + 2 * q);
      v[2 * i + 1] = __ldcg(src + 2 * q + 1);
    }
  }
#pragma unroll
  for (int i = 0; i < kQ; ++i) {
    const int q = lane + 32 * i;
    if (tok >= 0 && q < H / 16) {
      const uint32_t in[8] = {v[2 * i].x, v[2 * i].y, v[2 * i].z, v[2 * i].w,
                              v[2 * i + 1].x, v[2 * i + 1].y, v[2 * i + 1].z, v[2 * i + 1].w};
      uint32_t out[8];
      operand_quarter<true>(in, out);
      dst[2 * q] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[2 * q + 1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) trace_max(a.trace, kTrExit);
}

// ------------------------------------------------------------------ expert GEMM
constexpr int kGemmCons = fused::kCons;                 // 16 dequantisation warps
constexpr int kGemmProd = kGemmCons;                    // producer warp
constexpr int kGemmMma = kGemmCons + 1;                 // tcgen05 issue warp
constexpr int kGemmEpi0 = kGemmCons + 2;                // 4 epilogue warps (tensor-memory lane quarters 2, 3, 0, 1)
constexpr int kGemmEpiWarps = 4;
constexpr int kGemmThreads = (kGemmCons + 2 + kGemmEpiWarps) * 32;  // 704
constexpr int kTileRows = dense::kRows;                 // rows of one weight matrix (the MMA M)
// 128-row weight matrices per unit, all against one operand tile: gate and
// up for kMats / 2 row tiles of I (gate/up), or kMats row tiles of H (down).
// More matrices per operand tile means fewer operand bytes per flop.
constexpr int kMats = 2;
constexpr int kABuf = 2;                         // dequantised A tiles in flight
constexpr int gemm_smem(int n, int stages) {
  return stages * (n * 128 + kMats * kTileRows * 32) + kABuf * kMats * kTileRows * 128 + 320 + 1024;
}
constexpr int pick_stages(int n) {
  int st = 8;
  while (st > 2 && gemm_smem(n, st) > 227 * 1024) --st;
  return st;
}
// Per kernel: N = the chunk rows one unit takes (the MMA N and the
// tensor-memory columns per matrix), units per chunk and weight tile,
// accumulator sets, TMA stages, shared memory.  Measured on GB300: whole
// 256-row chunks with one accumulator set beat 128-row parts with two sets
// for both kernels (down: 267 against 272 us at 4096 rows).
template <bool kDown>
struct GemmShape {
  static constexpr int N = kPromptChunk;
  static constexpr int Sub = kPromptChunk / N;      // units per chunk and weight tile
  static constexpr int Sets = 512 / (N * kMats);
  static constexpr int Stages = pick_stages(N);
  static constexpr int Smem = gemm_smem(N, Stages);
  static_assert(Sets >= 1 && Smem <= 227 * 1024, "the unit's accumulators and stages fit");
};

// Shared-memory plan of a GEMM block (offsets from a 1024-aligned base).
struct GemmPlan {
  int stages, bstage, cstage, abuf;
  int b0, c0, a0, bar, total;
};
__host__ __device__ inline GemmPlan gemm_plan(int n, int stages) {
  GemmPlan P;
  P.stages = stages;
  P.bstage = n * 128;                   // the unit's operand rows x 64 fp16
  P.cstage = kMats * kTileRows * 32;    // 128 rows x 64 codes per matrix
  P.abuf = kMats * kTileRows * 128;     // dequantised A of every matrix
  int o = 0;
  P.b0 = o;
  o += stages * P.bstage;
  P.c0 = o;
  o += stages * P.cstage;
  P.a0 = o;
  o += kABuf * P.abuf;
  P.bar = o;
  o += 320;  // barriers [0, 8 (20 + 2 kABuf + 1)), tensor-memory address at 304
  P.total = o + 1024;  // slack for the 1024-byte alignment of the base
  return P;
}

struct GemmParams {
  dense::Maps m;  // 64-byte aligned: first
  PromptArgs a;
};

// Bounded wait for the phase with the given parity that suspends the thread
// in hardware (mbarrier.try_wait with a suspend-time hint) instead of
// polling, so waiting warps take no issue slots from the warps sharing their
// scheduler; false after limit_ns of global time.
__device__ __forceinline__ bool mbar_wait_susp(uint64_t *bar, uint32_t parity,
                                               unsigned long long limit_ns = kWaitLimitNs) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    if (ok) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Persistent GEMM over the units (chunk, weight tile), u = blockIdx.x,
// blockIdx.x + gridDim.x, ...  Roles: the producer warp streams each K
// group's operand rows and codes (TMA) through the stage buffers; 16 warps
// dequantise the codes of the unit's kMats weight matrices into a
// double-buffered fp16 A tile; the MMA warp issues the group's tcgen05.mma
// into the unit's accumulator set in tensor memory; 4 epilogue warps read a
// finished set (with two sets, while the next unit's MMAs run).
template <bool kDown>
__global__ void __launch_bounds__(kGemmThreads, 1) prompt_gemm_kernel(const __grid_constant__ GemmParams prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const PromptArgs &a = prm.a;
  const int H = a.d.H, I = a.d.I, T = a.d.T, k = a.d.k;
  const int K = kDown ? I : H, G = K / kGroup, M = kDown ? H : I;
  constexpr int kUnitRows = kDown ? kMats * kTileRows : kMats / 2 * kTileRows;  // rows of M one unit covers
  const int ntile = (M + kUnitRows - 1) / kUnitRows;
  constexpr int nm = kMats;                        // matrices per unit
  constexpr int kNmax = GemmShape<kDown>::N;        // rows of a unit (MMA N bound)
  constexpr int kSub = GemmShape<kDown>::Sub;       // units per (chunk, weight tile)
  constexpr int kSets = GemmShape<kDown>::Sets;
  constexpr uint32_t kAccCols = kNmax * nm;        // tensor-memory columns of one accumulator set
  constexpr uint32_t kTmemCols = kSets * kAccCols; // 512
  // matrix m of a unit: its first weight row past the unit's r0, and which
  // weights (gate/up: m even gate, m odd up, of row tile m / 2)
  auto moff = [](int m) { return kTileRows * (kDown ? m : (m >> 1)); };
  uint8_t *base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const GemmPlan P = gemm_plan(kNmax, GemmShape<kDown>::Stages);
  constexpr int S = GemmShape<kDown>::Stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + P.bar);  // [S] TMA landed
  uint64_t *empty = full + S;                                   // [S] MMAs done with a stage
  uint64_t *adone = empty + S;                                  // [kABuf] MMAs done with an A buffer
  uint64_t *afull = adone + kABuf;                              // [kABuf] A buffer written (every dequant warp)
  uint64_t *tfull = afull + kABuf;                              // [2] accumulator set complete
  uint64_t *tempty = tfull + 2;                                 // [2] accumulator set read out (every epilogue warp)
  uint64_t *tready = tempty + 2;                                // tensor memory allocated
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(base + P.bar + 304);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool tracer = blockIdx.x == 0 && tid == 0;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kABuf; ++i) {
      mbar_init(&adone[i], 1);
      mbar_init(&afull[i], kGemmCons / 2);  // the half of the dequant warps that owns the buffer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kGemmEpiWarps);
    }
    mbar_init(tready, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tracer) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);
  const int nunits = __ldcg(a.n_ch) * ntile * kSub;
  // unit u: chunk, weight tile, part of the chunk (consecutive units share the
  // weight tile, so its codes come from HBM once); rows beg .. beg + cnt - 1
  // of the sorted positions, none when the chunk is shorter than the part
  struct UnitPos {
    int ch, rt, beg, cnt;
  };
  auto unit_pos = [&](int u) {
    UnitPos q;
    q.ch = u / (ntile * kSub);
    const int rem = u - q.ch * ntile * kSub;
    q.rt = rem / kSub;
    const int sub = rem - q.rt * kSub;
    q.beg = __ldcg(a.ch_beg + q.ch) + sub * kNmax;
    q.cnt = min(kNmax, __ldcg(a.ch_cnt + q.ch) - sub * kNmax);
    return q;
  };
  const int npairs = T * k;

  // ============================================================ producer warp
  if (warp == kGemmProd) {
    fused::fence_proxy_async_global();  // operand rows written by the previous launch are read by the TMA
    bool ok = true;
    int gi = 0, st = 0, ph = 0;  // K groups issued; next stage and its use parity
    const CUtensorMap *bmap = kDown ? &prm.m.h : &prm.m.x;
    auto q_off = [&](int m) -> size_t { return kDown ? a.w.off.down_q : (m & 1) ? a.w.off.up_q : a.w.off.gate_q; };
    auto s_off = [&](int m) -> size_t { return kDown ? a.w.off.down_s : (m & 1) ? a.w.off.up_s : a.w.off.gate_s; };
    auto b_off = [&](int m) -> size_t { return kDown ? a.w.off.down_b : (m & 1) ? a.w.off.up_b : a.w.off.gate_b; };
    auto mrows = [&](int r0, int m) { return max(0, min(kTileRows, M - (r0 + moff(m)))); };
    // a unit's weights into L2: the codes, scales and biases of each
    // matrix's rows are contiguous ranges of the blob (a few bulk requests)
    auto prefetch_unit = [&](const uint8_t *bn, int r0n) {
      for (int mm = 0; mm < nm; ++mm) {
        const int rows = mrows(r0n, mm);
        if (rows == 0) continue;
        const size_t qrow = (size_t)K / 2;  // code bytes per row
        const uint8_t *q = bn + q_off(mm) + (size_t)(r0n + moff(mm)) * qrow;
        for (size_t o = 0; o < rows * qrow; o += 65536)
          prefetch_l2(q + o, (uint32_t)min((size_t)65536, rows * qrow - o));
        prefetch_l2(bn + s_off(mm) + (size_t)(r0n + moff(mm)) * G * 2, (uint32_t)(rows * G * 2));
        prefetch_l2(bn + b_off(mm) + (size_t)(r0n + moff(mm)) * G * 2, (uint32_t)(rows * G * 2));
      }
    };
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const UnitPos q = unit_pos(u);
      if (q.cnt <= 0) continue;
      const int ch = q.ch, rt = q.rt, beg = q.beg;
      const int e = __ldcg(a.ch_e + ch);
      const int sh = e < 0 ? 1 : 0;
      const uint8_t *blob = sh ? a.w.shared : a.w.experts + (size_t)e * a.w.stride;
      const int r0 = rt * kUnitRows;
      // the block's next unit (the next tile of the sweep): its weights
      // into L2 while this unit runs; the first unit's own
      if (lane == 0) {
        if (u == (int)blockIdx.x) prefetch_unit(blob, r0);
        const int un = u + gridDim.x;
        if (un < nunits) {
          const UnitPos qn = unit_pos(un);
          const int en = __ldcg(a.ch_e + qn.ch);
          prefetch_unit(en < 0 ? a.w.shared : a.w.experts + (size_t)en * a.w.stride, qn.rt * kUnitRows);
        }
      }
      for (int g = 0; g < G && ok; ++g, ++gi) {
        if (gi >= S) ok = __all_sync(0xffffffffu, mbar_wait_idle(&empty[st], ph ^ 1, 32));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], (uint32_t)(P.bstage + P.cstage));
          dense::tma_load_2d(base + P.b0 + st * P.bstage, bmap, 64 * g, beg, &full[st]);
          uint8_t *cd = base + P.c0 + st * P.cstage;
#pragma unroll
          for (int m = 0; m < nm; ++m) {  // every matrix (rows past M read as zero)
            const CUtensorMap *qm = kDown ? &prm.m.dq[sh] : (m & 1) ? &prm.m.uq[sh] : &prm.m.gq[sh];
            dense::tma_load_3d(cd + m * kTileRows * 32, qm, 32 * g, r0 + moff(m), sh ? 0 : e, &full[st]);
          }
        }
        __syncwarp();
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
      }
    }
    // copies in flight land before the block's shared memory is released
    if (lane == 0) {
      if (!ok) set_error(a.err, kErrTimeout);
      for (int j = gi - S > 0 ? gi - S : 0; j < gi; ++j) mbar_wait_idle(&full[j % S], (j / S) & 1);
    }
    return;
  }

  // ============================================================ MMA warp
  // Owns the tensor memory: accumulator set b at columns b * kAccCols (gate
  // first, then up).  Issues each K group's tcgen05.mma once the dequant
  // warps have written its A tile.
  if (warp == kGemmMma) {
    dense::tc_alloc(s_tmem, kTmemCols);
    dense::tc_fence_before();
    __syncwarp();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);
    if (lane == 0) mbar_arrive_expect_tx(tready, 0);
    bool ok = true;
    int gi = 0, du = 0, st = 0, ph = 0, ab = 0, aph = 0;
    // shared-memory descriptors of stage 0's operand rows and A buffer 0;
    // the others are these plus their byte offsets / 16
    const uint64_t bdesc0 = dense::sdesc(smem_addr(base + P.b0), 16, 1024, 2);
    const uint64_t adesc0 = dense::sdesc(smem_addr(base + P.a0), 16, 1024, 2);
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const UnitPos q = unit_pos(u);
      if (q.cnt <= 0) continue;
      const int N = (q.cnt + 15) & ~15;  // MMA N: the unit's rows, padded to 16
      const uint32_t idesc = dense::idesc_f16(kTileRows, N);
      const int tb = du % kSets;
      // the set's previous unit read out by the epilogue
      if (du >= kSets) ok = __all_sync(0xffffffffu, mbar_wait_idle(&tempty[tb], ((du / kSets) - 1) & 1, 32));
      ++du;
      dense::tc_fence_after();
      const uint32_t acc = tmem + tb * kAccCols;
      for (int g = 0; g < G && ok; ++g, ++gi) {
        ok = __all_sync(0xffffffffu, mbar_wait_susp(&full[st], ph) && mbar_wait_susp(&afull[ab], aph));
        if (!ok) break;
        dense::tc_fence_after();
        if (lane == 0) {
          const uint64_t bd0 = bdesc0 + (uint64_t)((st * P.bstage) >> 4);
          const uint64_t ad0 = adesc0 + (uint64_t)((ab * P.abuf) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // K = 16 per MMA: 32 bytes further along each row
#pragma unroll
            for (int m = 0; m < nm; ++m)
              dense::tc_mma(acc + m * kNmax, ad0 + (uint64_t)(((m * kTileRows * 128) >> 4) + 2 * ks), bd0 + 2 * ks, idesc,
                            (g > 0 || ks > 0) ? 1u : 0u);
          dense::tc_commit(&empty[st]);               // the TMA stage may be refilled
          dense::tc_commit(&adone[ab]);               // the A buffer may be rewritten
          if (g == G - 1) dense::tc_commit(&tfull[tb]);  // the unit's accumulators are complete
        }
        __syncwarp();
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
        if (++ab == kABuf) {
          ab = 0;
          aph ^= 1;
        }
      }
    }
    if (!ok && lane == 0) set_error(a.err, kErrTimeout);
    // tensor memory back once the last MMAs completed and the epilogue read them (bounded waits)
    if (gi > 0) mbar_wait(&adone[(gi - 1) % kABuf], ((gi - 1) / kABuf) & 1);
    if (du > 0) mbar_wait_idle(&tempty[(du - 1) % kSets], ((du - 1) / kSets) & 1, 64);
    dense::tc_fence_after();
    __syncwarp();
    dense::tc_dealloc(tmem, kTmemCols);
    return;
  }

  // ============================================================ epilogue warps
  // Warp w reads tensor-memory lanes 32 (w % 4) .. +31: weight rows r0 + rr.
  // Gate/up: h = gelu_tanh(gate) * up per (row, column), stored fp16 in the
  // operand order of the down units at the chunk's positions.  Down: the
  // routing weight of each column's pair times the output row, fp32.
  if (warp >= kGemmEpi0) {
    bool ok = mbar_wait(tready, 0);
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);
    const int rr = 32 * (warp & 3) + lane;
    int du = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++du) {
      const UnitPos q = unit_pos(u);
      if (q.cnt <= 0) {
        --du;  // no unit: the accumulator sets do not advance
        continue;
      }
      const int beg = q.beg, cnt = q.cnt;
      const int r0 = q.rt * kUnitRows;
      const int tb = du % kSets;
      // routing weights of columns lane, lane + 32, ... (down; shared rows: 1)
      float wq[kNmax / 32];
#pragma unroll
      for (int q = 0; q < kNmax / 32; ++q) wq[q] = 1.f;
      if (kDown)
#pragma unroll
        for (int q = 0; q < kNmax / 32; ++q) {
          const int n = 32 * q + lane;
          if (n < cnt && beg + n < npairs) wq[q] = __ldcg(a.r.wts + __ldcg(a.r.perm + beg + n));
        }
      ok = __all_sync(0xffffffffu, mbar_wait_susp(&tfull[tb], (du / kSets) & 1));
      if (!ok) break;
      dense::tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + tb * kAccCols;
      bool bad = false;
      for (int c0 = 0; c0 < cnt; c0 += 16) {  // 16 columns at a time (warp-uniform)
        if (!kDown) {
#pragma unroll 1
          for (int hr = 0; hr < nm / 2; ++hr) {  // row tile hr: gate in matrix 2 hr, up in 2 hr + 1
            float gv[16], uv[16];
            dense::tc_ld16(ta + 2 * kNmax * hr + c0, gv);
            dense::tc_ld16(ta + 2 * kNmax * hr + kNmax + c0, uv);
            const int i = r0 + kTileRows * hr + rr;
            if (i < M) {
              bool odd = false;
              const int slot = dense::operand_slot(i & 63, odd);
              __half *dst = a.hg + (size_t)(beg + c0) * I + (i & ~63) + slot;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (c0 + j < cnt) {
                  const float hv = gelu_tanh(gv[j]) * uv[j];
                  bad = bad || !(fabsf(hv) <= 65504.0f);
                  dst[(size_t)j * I] = __float2half_rn(odd ? hv * 0.0625f : hv);  // odd words / 16
                }
              }
            }
          }
        } else {
          const int q = c0 >> 5;  // the 16 columns share one group of 32 weights
          float wsel = wq[0];
#pragma unroll
          for (int i = 1; i < kNmax / 32; ++i)
            if (q == i) wsel = wq[i];
#pragma unroll 1
          for (int m = 0; m < nm; ++m) {  // output rows r0 + 128 m + rr
            float dv[16];
            dense::tc_ld16(ta + kNmax * m + c0, dv);
            const int row = r0 + kTileRows * m + rr;
            float *dst = a.obuf + (size_t)(beg + c0) * H + row;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = c0 + j;
              const float w = __shfl_sync(0xffffffffu, wsel, n & 31);
              if (n < cnt && row < M) dst[(size_t)j * H] = w * dv[j];
            }
          }
        }
      }
      if (bad) set_error(a.err, kErrNonFinite);
      dense::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&tempty[tb], 0);  // this warp is done with the set
    }
    if (!ok && lane == 0) set_error(a.err, kErrTimeout);
    if (tracer || (blockIdx.x == 0 && warp == kGemmEpi0 && lane == 0)) trace_max(a.trace, kTrExit);
    return;
  }

  // ============================================================ dequantisation warps
  // Two halves of 8 warps take alternate K groups (half h: the block's
  // groups gi with gi % 2 == h, into A buffer h), so each warp's wait,
  // fence and arrival cover a whole row per thread and the two halves
  // overlap on consecutive groups.  Thread: matrix m (gate / up, or the two
  // halves of W_down), weight row rr, all 64 codes of the group.  A row's
  // scale and bias come from global memory (the 32-byte sector of a row holds
  // 16 groups: after the first group of a sector the loads hit L1), one of
  // the half's groups ahead of their use.
  static_assert(nm == 2 && kABuf == 2, "one matrix per thread, one A buffer per half");
  const int half = tid >> 8, m = (tid >> 7) & 1, rr = tid & 127;
  bool okd = true;
  int gi = 0;  // the block's K groups before this unit
  for (int u = blockIdx.x; u < nunits && okd; u += gridDim.x) {
    const UnitPos q = unit_pos(u);
    if (q.cnt <= 0) continue;
    const int ch = q.ch, rt = q.rt;
    const int e = __ldcg(a.ch_e + ch);
    const uint8_t *blob = e < 0 ? a.w.shared : a.w.experts + (size_t)e * a.w.stride;
    const int wrow = rt * kUnitRows + moff(m) + rr;
    const bool rvalid = wrow < M;
    const size_t so = kDown ? a.w.off.down_s : ((m & 1) ? a.w.off.up_s : a.w.off.gate_s);
    const size_t bo = kDown ? a.w.off.down_b : ((m & 1) ? a.w.off.up_b : a.w.off.gate_b);
    const uint16_t *srow = reinterpret_cast<const uint16_t *>(blob + so) + (size_t)(rvalid ? wrow : 0) * G;
    const uint16_t *brow = reinterpret_cast<const uint16_t *>(blob + bo) + (size_t)(rvalid ? wrow : 0) * G;
    const int g0 = half ^ (gi & 1);  // this half's first group of the unit
    uint16_t sn = 0, bn = 0;
    if (g0 < G) {
      sn = __ldg(srow + g0);
      bn = __ldg(brow + g0);
    }
    for (int g = g0; g < G; g += 2) {
      const int gg = gi + g;  // the block's group index: stage, buffer and phases follow from it
      const int st = gg % S, ph = (gg / S) & 1, ab = half;
      const uint16_t sc = sn, bc = bn;
      if (g + 2 < G) {
        sn = __ldg(srow + g + 2);
        bn = __ldg(brow + g + 2);
      }
      okd = okd && mbar_wait_susp(&full[st], ph);
      if (gg >= kABuf) okd = okd && mbar_wait_susp(&adone[ab], ((gg >> 1) - 1) & 1);
      if (okd) {
        const uint8_t *cb = base + P.c0 + st * P.cstage + m * kTileRows * 32 + rr * 32;
        uint8_t *row = base + P.a0 + ab * P.abuf + m * kTileRows * 128 + rr * 128;
        const uint4 cw0 = *reinterpret_cast<const uint4 *>(cb), cw1 = *reinterpret_cast<const uint4 *>(cb + 16);
        const float sf = bf16_bits_to_float(sc);
        const float bf = bf16_bits_to_float(bc);
        const uint32_t s2 = dense::f16x2_of(sf), b2 = dense::f16x2_of(bf), b16 = dense::f16x2_of(16.0f * bf);
        // row rr of the 128-byte-swizzled tile: 16-byte chunk j at (j ^ (rr % 8))
        const int sw = rr & 7;
        *reinterpret_cast<uint4 *>(row + (0 ^ sw) * 16) = dense::dequant_word(cw0.x, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (1 ^ sw) * 16) = dense::dequant_word(cw0.y, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (2 ^ sw) * 16) = dense::dequant_word(cw0.z, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (3 ^ sw) * 16) = dense::dequant_word(cw0.w, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (4 ^ sw) * 16) = dense::dequant_word(cw1.x, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (5 ^ sw) * 16) = dense::dequant_word(cw1.y, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (6 ^ sw) * 16) = dense::dequant_word(cw1.z, s2, b2, b16);
        *reinterpret_cast<uint4 *>(row + (7 ^ sw) * 16) = dense::dequant_word(cw1.w, s2, b2, b16);
      }
      dense::fence_async_smem();  // the A tiles, written by threads, are read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&afull[ab], 0);  // this warp's part of the A tile is in place
    }
    gi += G;
    okd = __all_sync(0xffffffffu, okd);
  }
  if (!okd && lane == 0) set_error(a.err, kErrTimeout);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A tensor map over a row-major tensor (dims[0] innermost, byte strides of
// dims 1..); elements outside the tensor read as zero.
bool encode_map(EncodeTiledFn f, CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr,
                const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw) {
  const cuuint32_t estr[3] = {1, 1, 1};
  return f(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           sw, sw == CU_TENSOR_MAP_SWIZZLE_NONE ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand rows of x and h per sorted position (fp16, boxes of 64 elements x
// kNmax rows with the 128-byte swizzle), the codes of gate, up and down
// (boxes of 32 bytes x 128 rows of one expert) for the routed experts (3-D
// over the fixed-stride blobs) and the shared expert.
bool prompt_maps(const PromptArgs &a, dense::Maps &m) {
  const EncodeTiledFn f = encode_tiled();
  if (!f) return false;
  const cuuint64_t H = a.d.H, I = a.d.I, E = a.d.E, npos = (cuuint64_t)a.d.T * (a.d.k + 1);
  const cuuint32_t bxg[2] = {64, (cuuint32_t)GemmShape<false>::N}, bxd[2] = {64, (cuuint32_t)GemmShape<true>::N};
  bool ok = true;
  {
    const cuuint64_t dims[2] = {H, npos}, str[1] = {H * 2};
    ok = ok && encode_map(f, &m.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.xg, dims, str, bxg, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  {
    const cuuint64_t dims[2] = {I, npos}, str[1] = {I * 2};
    ok = ok && encode_map(f, &m.h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.hg, dims, str, bxd, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const cuuint32_t bq[3] = {32, (cuuint32_t)kTileRows, 1};
  auto codes = [&](CUtensorMap *mm, size_t off, cuuint64_t row_bytes, cuuint64_t rows) {
    const cuuint64_t dr[3] = {row_bytes, rows, E}, sr[2] = {row_bytes, a.w.stride};
    const cuuint64_t ds[3] = {row_bytes, rows, 1}, ss[2] = {row_bytes, row_bytes * rows};
    return encode_map(f, &mm[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w.experts + off, dr, sr, bq,
                      CU_TENSOR_MAP_SWIZZLE_NONE) &&
           encode_map(f, &mm[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w.shared + off, ds, ss, bq,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  };
  ok = ok && codes(m.gq, a.w.off.gate_q, H / 2, I) && codes(m.uq, a.w.off.up_q, H / 2, I) &&
       codes(m.dq, a.w.off.down_q, I / 2, H);
  return ok;
}
}  // namespace

int prompt_max_chunks(int T, int k, int E) {
  return (T * k + kPromptChunk - 1) / kPromptChunk + E + (T + kPromptChunk - 1) / kPromptChunk;
}

// code stages of the router: six when the row tile leaves room, else three
static int rt_stages(const Dims &d) { return rt_layout(d.H, d.E, 6).total <= 227 * 1024 ? 6 : 3; }

bool prompt_supported(const Dims &d) {
  if (rt_layout(d.H, d.E, 3).total > 227 * 1024) return false;
  return true;  // the GEMM plan does not depend on the shape (checked at compile time)
}

cudaError_t prompt_set_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prompt_router_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)))
    return e;
  if ((e = cudaFuncSetAttribute(prompt_router_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)))
    return e;
  if ((e = cudaFuncSetAttribute(prompt_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)))
    return e;
  return cudaFuncSetAttribute(prompt_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t launch_prompt(const PromptArgs &a, uint16_t *y, bool add_residual, int n_sm, cudaStream_t st, bool pdl) {
  const int T = a.d.T, k = a.d.k;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.a = a;
  if (!prompt_maps(a, prm.m)) return cudaErrorInvalidValue;
  auto with_trace = [&](int i) {
    PromptArgs b = a;
    if (b.trace) b.trace += 4 * i;
    return b;
  };
  const int rst = rt_stages(a.d);
  cudaError_t e = launch_k(rst == 6 ? prompt_router_kernel<6> : prompt_router_kernel<3>,
                           dim3((T + kRtTok - 1) / kRtTok), dim3(kRtThreads),
                           (size_t)rt_layout(a.d.H, a.d.E, rst).total, st, pdl, with_trace(0));
  if (e == cudaSuccess) e = launch_k(prompt_sort_kernel, dim3(1), dim3(kSortThreads), 0, st, pdl, with_trace(1));
  if (e == cudaSuccess) {
    const int npos = T * (k + 1);
    e = launch_k(prompt_gather_kernel, dim3((npos + kGatherThreads / 32 - 1) / (kGatherThreads / 32)),
                 dim3(kGatherThreads), 0, st, pdl, with_trace(2));
  }
  if (e == cudaSuccess) {
    prm.a = with_trace(3);
    e = launch_k(prompt_gemm_kernel<false>, dim3(n_sm), dim3(kGemmThreads), (size_t)GemmShape<false>::Smem, st, pdl,
                 prm);
  }
  if (e == cudaSuccess) {
    prm.a = with_trace(4);
    e = launch_k(prompt_gemm_kernel<true>, dim3(n_sm), dim3(kGemmThreads), (size_t)GemmShape<true>::Smem, st, pdl,
                 prm);
  }
  if (e == cudaSuccess) {
    FfnArgs c;
    memset(&c, 0, sizeof(c));
    c.w = a.w;
    c.d = a.d;
    c.r = a.r;
    c.obuf = a.obuf;
    c.y = y;
    c.hres = add_residual ? a.hres : nullptr;
    c.include_shared = 1;
    c.err = a.err;
    c.trace = a.trace ? a.trace + 4 * 5 : nullptr;
    e = launch_combine(c, st, pdl);
  }
  return e;
}

}  // namespace moe
