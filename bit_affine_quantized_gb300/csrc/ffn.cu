// Routed + shared expert FFN kernels, sm_103a.
//
// Page "TurboFieldfare - System design", section "Metal execution": the
// routed kernels fuse affine decode, GeGLU and the weighted reduction over
// the selected experts; section "Why the runtime has this shape": 4-bit
// affine experts (group 64, BF16 scale and bias), a shared expert added with
// no routing weight; section "Decode": the shared branch runs alongside the
// routed one.
//
// Work is organised around the active slots left by the grouping step
// (slot 0 = shared expert, then every expert with at least one row).
//
//  gateup_kernel<TT>   block = (16 rows of I, one slot).  The 16 gate rows,
//                      16 up rows and their scales/biases (~51 KB for
//                      H = 2816) arrive by 1-D bulk copies on one mbarrier;
//                      the slot's token rows are staged (TT at a time) while
//                      the copies fly.  4 warps split K; each 64-wide group
//                      is 4 mma.m16n8k16 (weights as A, tokens as N) on exact
//                      small-integer operands, followed by the affine
//                      correction s*acc + b*sum(x).  GeGLU in the epilogue,
//                      h stored as fp16 [position, I].
//  down_decode_kernel  T == 1: block = 16 output rows; all k + 1 rows of h
//                      and the matching 16-row tiles of every selected
//                      W_down; weighted sum in registers, bf16 out, optional
//                      residual add.  No scratch, one launch.
//  down_grouped_kernel T > 1: block = (64 output rows, one slot); writes the
//                      weighted expert outputs (fp32) per position.
//  combine_kernel      T > 1: y[t] = sum_j o[pos(t, j)] + o[shared row t],
//                      in selection order, bf16 out, optional residual add.
#include <math.h>

#include "kernels.h"

namespace moe {

namespace {
constexpr int kThreads = 256;  // gate/up and single-token down blocks
constexpr int kWarps = 8;
constexpr int kDgThreads = 128;  // grouped down: 4 warps x 16 rows
constexpr int kRows = 16;      // rows of one mma tile
constexpr int kDownRows = 64;  // output rows per grouped-down block
constexpr int kTokTile = 8;    // tokens per mma N

// Smallest row pitch (in 32-bit words) >= w with pitch % 16 == 8: eight
// consecutive rows then hit disjoint bank groups for the 8-byte fragment
// loads, so the 16 lanes of a half-warp never conflict.
__host__ __device__ inline int pitch_words(int w) { return w + ((8 - (w % 16)) + 16) % 16; }

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

struct GateUpLayout {
  int qp, xp, q, raw, sb, x, xs, bar, total;
};
__host__ __device__ inline GateUpLayout gateup_layout(int H, int tt) {
  const int G = H / kGroup;
  GateUpLayout L;
  L.qp = pitch_words(H / 8) * 4;
  L.xp = 2 * H + 8;
  int o = 0;
  L.q = o;
  o += 2 * kRows * L.qp;
  L.raw = o;
  o = align16(o + 4 * kRows * G * 2);
  L.sb = o;
  o = align16(o + 2 * kRows * G * 8);
  L.x = o;
  const int xbytes = tt * L.xp > kWarps * 32 * 8 * 4 ? tt * L.xp : kWarps * 32 * 8 * 4;
  o = align16(o + xbytes);
  L.xs = o;
  o = align16(o + tt * G * 4);
  L.bar = o;
  o += 16;
  L.total = o;
  return L;
}

struct DownLayout {
  int qp, hp, q, raw, sb, h, hs, wt, red, bar, total;
};
// nslot: weight tiles held (k + 1 for decode, 1 for grouped); rows: rows per
// tile (16 decode, 64 grouped); hrows: staged h rows (k + 1 or 8).
__host__ __device__ inline DownLayout down_layout(int I, int nslot, int rows, int hrows) {
  const int GI = I / kGroup;
  DownLayout L;
  L.qp = pitch_words(I / 8) * 4;
  L.hp = 2 * I + 8;
  int o = 0;
  L.q = o;
  o += nslot * rows * L.qp;
  L.raw = o;
  o = align16(o + nslot * 2 * rows * GI * 2);
  L.sb = o;
  o = align16(o + nslot * rows * GI * 8);
  L.h = o;
  o = align16(o + hrows * L.hp);
  L.hs = o;
  o = align16(o + hrows * GI * 4);
  L.wt = o;
  o = align16(o + hrows * 4);
  L.red = o;
  o = align16(o + kWarps * kRows * 4);
  L.bar = o;
  o += 16;
  L.total = o;
  return L;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float lo_f16(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float hi_f16(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Stages one 64-wide group of a 16-bit activation row into the permuted
// shared-memory order and returns the group's sum (fp32, element order).
template <bool kHalf>
__device__ __forceinline__ float stage_group(const uint16_t *__restrict__ src_row, int g, uint8_t *__restrict__ dst_row) {
  const uint4 *src = reinterpret_cast<const uint4 *>(src_row + g * kGroup);
  uint2 *dst = reinterpret_cast<uint2 *>(dst_row + g * 128);
  // all eight 16-byte loads in flight before any shared-memory store
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldcg(src + i);
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v0 = v[2 * c], v1 = v[2 * c + 1];
    const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t out[8];
    operand_quarter<!kHalf>(in, out);
#pragma unroll
    for (int w = 0; w < 4; ++w) dst[4 * c + w] = make_uint2(out[2 * w], out[2 * w + 1]);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      sum += kHalf ? lo_f16(in[w]) : lo_bf16(in[w]);
      sum += kHalf ? hi_f16(in[w]) : hi_bf16(in[w]);
    }
  }
  return sum;
}

__device__ __forceinline__ const uint8_t *slot_blob(const FfnArgs &a, int e) {
  return e == kSharedSlot ? a.w.shared : a.w.experts + (size_t)e * a.w.stride;
}

// Routing weight of sorted position `pos` (shared rows: 1).
__device__ __forceinline__ float pos_weight(const FfnArgs &a, int pos) {
  const int rows = a.d.T * a.d.k;
  return pos >= rows ? 1.0f : a.r.wts[a.r.perm[pos]];
}

// Bounded wait on a copy barrier by the whole block.  On timeout: record it,
// wait once more for the copies in flight, and tell the caller to return.
__device__ __forceinline__ bool block_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
  const bool ok = mbar_wait(bar, parity);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) set_error(err, kErrTimeout);
    if (!ok) mbar_wait(bar, parity);
    return false;
  }
  return true;
}
}  // namespace

// ------------------------------------------------------------------ gate/up
template <int TT>
__global__ void __launch_bounds__(kThreads) gateup_kernel(const FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.d.H, I = a.d.I, k = a.d.k;
  const int G = H / kGroup;
  const GateUpLayout L = gateup_layout(H, TT);
  uint8_t *sq = smem + L.q;
  uint16_t *sraw = reinterpret_cast<uint16_t *>(smem + L.raw);
  float2 *ssb = reinterpret_cast<float2 *>(smem + L.sb);
  uint8_t *sx = smem + L.x;
  float *sxs = reinterpret_cast<float *>(smem + L.xs);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar);
  float *sred = reinterpret_cast<float *>(sx);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.y;
  const int r0 = blockIdx.x * kRows;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Rows r0..r0+15 of gate and up (one bulk copy per row into a padded
  // pitch) plus the four 16-row scale/bias tiles.
  auto issue = [&](const uint8_t *blob) {
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(2 * kRows * (H / 2) + 4 * kRows * G * 2));
      __syncwarp();
      const int m = lane >> 4, row = lane & 15;
      const uint8_t *src = blob + (m == 0 ? a.w.off.gate_q : a.w.off.up_q) + (size_t)(r0 + row) * (H / 2);
      bulk_g2s(sq + (m * kRows + row) * L.qp, src, (uint32_t)(H / 2), bar);
      if (lane < 4) {
        const size_t off = lane == 0 ? a.w.off.gate_s : lane == 1 ? a.w.off.gate_b : lane == 2 ? a.w.off.up_s : a.w.off.up_b;
        bulk_g2s(sraw + lane * kRows * G, blob + off + (size_t)r0 * G * 2, (uint32_t)(kRows * G * 2), bar);
      }
    }
  };

  // Decode: this block also warms L2 with its share (1/gridDim.x of the
  // rows) of the same expert's W_down, so the down kernel reads from L2
  // while the HBM keeps streaming.  Ranges are rounded inwards to 16 bytes.
  auto prefetch_down = [&](const uint8_t *blob) {
    if (!a.prefetch_down || warp != 1 || lane != 0) return;
    const int GI = I / kGroup;
    const int per = (H + gridDim.x - 1) / gridDim.x;
    const int nb = blockIdx.x * per, ne = min(H, nb + per);
    if (nb >= ne) return;
    const size_t ranges[3][2] = {{a.w.off.down_q + (size_t)nb * (I / 2), (size_t)(ne - nb) * (I / 2)},
                                 {a.w.off.down_s + (size_t)nb * GI * 2, (size_t)(ne - nb) * GI * 2},
                                 {a.w.off.down_b + (size_t)nb * GI * 2, (size_t)(ne - nb) * GI * 2}};
    for (int i = 0; i < 3; ++i) {
      const uintptr_t s0 = ((uintptr_t)(blob + ranges[i][0]) + 15) & ~(uintptr_t)15;
      const uintptr_t s1 = ((uintptr_t)(blob + ranges[i][0] + ranges[i][1])) & ~(uintptr_t)15;
      for (uintptr_t p = s0; p < s1; p += 65536)
        prefetch_l2(reinterpret_cast<const void *>(p), (uint32_t)min((uintptr_t)65536, s1 - p));
    }
  };

  // The shared expert (slot 0) needs no routing: start its copies before
  // waiting on the previous kernel.
  const bool tracer = blockIdx.x == 0 && blockIdx.y == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  const bool early = a.include_shared && slot == 0;
  if (early) {
    issue(a.w.shared);
    prefetch_down(a.w.shared);
  }
  pdl_wait();
  if (tracer) trace_min(a.trace, kTrWaited);
  const int nact = a.r.n_act[0];
  if (slot >= nact) return;
  const int e = a.r.act_e[slot];
  const int beg = a.r.act_beg[slot];
  const int cnt = a.r.act_cnt[slot];
  if (!early) {
    issue(slot_blob(a, e));
    prefetch_down(slot_blob(a, e));
  }
  pdl_launch_dependents();

  const int r = lane >> 2, c = lane & 3;
  const bool bvalid = TT > 1 || r == 0;  // TT == 1 stages a single token row
  const uint8_t *qg0 = sq + r * L.qp + c * 8;
  const uint8_t *qg1 = sq + (r + 8) * L.qp + c * 8;
  const uint8_t *qu0 = sq + (kRows + r) * L.qp + c * 8;
  const uint8_t *qu1 = sq + (kRows + r + 8) * L.qp + c * 8;
  const uint8_t *xrow = sx + (bvalid ? r : 0) * L.xp + c * 32;
  bool ready = false;

  for (int j0 = 0; j0 < cnt; j0 += TT) {
    const int nt = min(TT, cnt - j0);
    for (int it = tid; it < nt * G; it += kThreads) {
      const int n = it / G, g = it - n * G;
      const int tok = e == kSharedSlot ? j0 + n : a.r.perm[beg + j0 + n] / k;
      sxs[n * G + g] = stage_group<false>(a.x + (size_t)tok * H, g, sx + n * L.xp);
    }
    __syncthreads();
    if (!ready) {
      if (!block_wait(bar, 0, a.err)) return;
      if (tid == 0) trace_max(a.trace, kTrLoaded);
      for (int it = tid; it < 2 * kRows * G; it += kThreads) {
        const int m = it / (kRows * G), rem = it - m * kRows * G;
        const float s = bf16_bits_to_float(sraw[(2 * m) * kRows * G + rem]);
        const float b = bf16_bits_to_float(sraw[(2 * m + 1) * kRows * G + rem]);
        ssb[it] = make_float2(s * kCodeScale, b);  // codes enter the mma as q * 2^-24
      }
      __syncthreads();
      ready = true;
    }

    float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = warp; g < G; g += kWarps) {
      const uint2 g0 = *reinterpret_cast<const uint2 *>(qg0 + g * 32);
      const uint2 g1 = *reinterpret_cast<const uint2 *>(qg1 + g * 32);
      const uint2 u0 = *reinterpret_cast<const uint2 *>(qu0 + g * 32);
      const uint2 u1 = *reinterpret_cast<const uint2 *>(qu1 + g * 32);
      float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint2 bx = bvalid ? *reinterpret_cast<const uint2 *>(xrow + g * 128 + s * 8) : make_uint2(0u, 0u);
        const uint32_t wg0 = (s >> 1) ? g0.y : g0.x, wg1 = (s >> 1) ? g1.y : g1.x;
        const uint32_t wu0 = (s >> 1) ? u0.y : u0.x, wu1 = (s >> 1) ? u1.y : u1.x;
        uint32_t A[4], B[4];
        if ((s & 1) == 0) {
          A[0] = codes_sub<0>(wg0); A[1] = codes_sub<0>(wg1); A[2] = codes_sub<1>(wg0); A[3] = codes_sub<1>(wg1);
          B[0] = codes_sub<0>(wu0); B[1] = codes_sub<0>(wu1); B[2] = codes_sub<1>(wu0); B[3] = codes_sub<1>(wu1);
        } else {
          A[0] = codes_sub<2>(wg0); A[1] = codes_sub<2>(wg1); A[2] = codes_sub<3>(wg0); A[3] = codes_sub<3>(wg1);
          B[0] = codes_sub<2>(wu0); B[1] = codes_sub<2>(wu1); B[2] = codes_sub<3>(wu0); B[3] = codes_sub<3>(wu1);
        }
        mma_f16(ag, A, bx.x, bx.y);
        mma_f16(au, B, bx.x, bx.y);
      }
      const float2 sg0 = ssb[r * G + g], sg1 = ssb[(r + 8) * G + g];
      const float2 su0 = ssb[(kRows + r) * G + g], su1 = ssb[(kRows + r + 8) * G + g];
      float xs0, xs1;
      if (TT > 1) {
        xs0 = sxs[(2 * c) * G + g];
        xs1 = sxs[(2 * c + 1) * G + g];
      } else {
        xs0 = c == 0 ? sxs[g] : 0.f;
        xs1 = 0.f;
      }
      tg[0] = fmaf(sg0.y, xs0, fmaf(sg0.x, ag[0], tg[0]));
      tg[1] = fmaf(sg0.y, xs1, fmaf(sg0.x, ag[1], tg[1]));
      tg[2] = fmaf(sg1.y, xs0, fmaf(sg1.x, ag[2], tg[2]));
      tg[3] = fmaf(sg1.y, xs1, fmaf(sg1.x, ag[3], tg[3]));
      tu[0] = fmaf(su0.y, xs0, fmaf(su0.x, au[0], tu[0]));
      tu[1] = fmaf(su0.y, xs1, fmaf(su0.x, au[1], tu[1]));
      tu[2] = fmaf(su1.y, xs0, fmaf(su1.x, au[2], tu[2]));
      tu[3] = fmaf(su1.y, xs1, fmaf(su1.x, au[3], tu[3]));
    }
    __syncthreads();  // sx is reused as the reduction buffer
    float4 *red = reinterpret_cast<float4 *>(sred + (warp * 32 + lane) * 8);
    red[0] = make_float4(tg[0], tg[1], tg[2], tg[3]);
    red[1] = make_float4(tu[0], tu[1], tu[2], tu[3]);
    __syncthreads();
    for (int o = tid; o < kRows * nt; o += kThreads) {
      const int row = o & 15, n = o >> 4;
      const int ln = (row & 7) * 4 + (n >> 1);
      const int idx = ((row >> 3) << 1) + (n & 1);
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        gs += sred[(w * 32 + ln) * 8 + idx];
        us += sred[(w * 32 + ln) * 8 + 4 + idx];
      }
      const float hv = gelu_tanh(gs) * us;
      if (!(fabsf(hv) <= 65504.0f)) set_error(a.err, kErrNonFinite);
      a.hbuf[(size_t)(beg + j0 + n) * I + r0 + row] = __float2half_rn(hv);
    }
    __syncthreads();
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
}

// ------------------------------------------------------------------ down, T == 1
// Block = 16 output rows.  Weight slots: s < n_valid routed positions (one
// per selected expert), slot k = shared expert.
__global__ void __launch_bounds__(kThreads) down_decode_kernel(const FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.d.H, I = a.d.I, k = a.d.k, E = a.d.E;
  const int GI = I / kGroup;
  const int nslot = k + 1;
  const DownLayout L = down_layout(I, nslot, kRows, nslot);
  uint8_t *sq = smem + L.q;
  uint16_t *sraw = reinterpret_cast<uint16_t *>(smem + L.raw);
  float2 *ssb = reinterpret_cast<float2 *>(smem + L.sb);
  uint8_t *sh = smem + L.h;
  float *shs = reinterpret_cast<float *>(smem + L.hs);
  float *swt = reinterpret_cast<float *>(smem + L.wt);
  float *sred = reinterpret_cast<float *>(smem + L.red);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar);  // [0] shared, [1] routed
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * kRows;
  const bool one_copy = L.qp == I / 2;  // rows contiguous in smem: one copy per tile
  const int nq = one_copy ? 1 : kRows;
  const uint32_t tile_tx = (uint32_t)(kRows * (I / 2) + 2 * kRows * GI * 2);

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // copy number `ci` of the tile for weight slot s taken from `blob`
  auto copy_one = [&](int s, const uint8_t *blob, int ci, uint64_t *b) {
    if (ci < nq) {
      const uint32_t bytes = one_copy ? (uint32_t)(kRows * (I / 2)) : (uint32_t)(I / 2);
      const size_t row = (size_t)n0 + (one_copy ? 0 : ci);
      bulk_g2s(sq + (s * kRows + (one_copy ? 0 : ci)) * L.qp, blob + a.w.off.down_q + row * (I / 2), bytes, b);
    } else {
      const int m = ci - nq;  // 0 scales, 1 biases
      bulk_g2s(sraw + (s * 2 + m) * kRows * GI, blob + (m == 0 ? a.w.off.down_s : a.w.off.down_b) + (size_t)n0 * GI * 2,
               (uint32_t)(kRows * GI * 2), b);
    }
  };

  const bool tracer = blockIdx.x == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  if (a.include_shared && warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(&bar[0], tile_tx);
    __syncwarp();
    for (int ci = lane; ci < nq + 2; ci += 32) copy_one(k, a.w.shared, ci, &bar[0]);
  }
  pdl_wait();
  if (tracer) trace_min(a.trace, kTrWaited);
  const int n_valid = a.r.offsets[E];
  const int a0 = a.include_shared ? 1 : 0;
  if (warp == 0 && n_valid > 0) {
    if (lane == 0) mbar_arrive_expect_tx(&bar[1], tile_tx * (uint32_t)n_valid);
    __syncwarp();
    const int nact = a.r.n_act[0];
    for (int ci = lane; ci < n_valid * (nq + 2); ci += 32) {
      const int s = ci / (nq + 2);
      int ex = 0;
      for (int sl = a0; sl < nact; ++sl)
        if (s >= a.r.act_beg[sl] && s < a.r.act_beg[sl] + a.r.act_cnt[sl]) ex = a.r.act_e[sl];
      copy_one(s, a.w.experts + (size_t)ex * a.w.stride, ci - s * (nq + 2), &bar[1]);
    }
  }
  pdl_launch_dependents();

  // stage h rows (permuted fp16) and group sums; slot weights
  const int nrows = n_valid + a0;
  for (int it = tid; it < nrows * GI; it += kThreads) {
    const int q = it / GI, g = it - q * GI;
    const int s = q < n_valid ? q : k;
    const int pos = q < n_valid ? q : k;  // T == 1: shared row at position k
    shs[s * GI + g] = stage_group<true>(reinterpret_cast<const uint16_t *>(a.hbuf) + (size_t)pos * I, g,
                                        sh + s * L.hp);
    if (g == 0) swt[s] = pos_weight(a, pos);
  }
  __syncthreads();
  if (a.include_shared && !block_wait(&bar[0], 0, a.err)) return;
  if (n_valid > 0 && !block_wait(&bar[1], 0, a.err)) return;
  if (tid == 0) trace_max(a.trace, kTrLoaded);
  for (int it = tid; it < nslot * kRows * GI; it += kThreads) {
    const int s = it / (kRows * GI), rem = it - s * kRows * GI;
    if (s < n_valid || (s == k && a.include_shared)) {
      const float sc = bf16_bits_to_float(sraw[(s * 2) * kRows * GI + rem]);
      const float bi = bf16_bits_to_float(sraw[(s * 2 + 1) * kRows * GI + rem]);
      ssb[it] = make_float2(sc * kCodeScale, bi);
    }
  }
  __syncthreads();

  // items (row q, group g); warp w takes a contiguous share
  const int nitems = nrows * GI;
  const int per = (nitems + kWarps - 1) / kWarps;
  const int ib = warp * per, ie = min(nitems, ib + per);
  const int r = lane >> 2, c = lane & 3;
  float t0 = 0.f, t2 = 0.f;
  for (int it = ib; it < ie; ++it) {
    const int q = it / GI, g = it - q * GI;
    const int s = q < n_valid ? q : k;
    const uint8_t *qb = sq + s * kRows * L.qp + g * 32 + c * 8;
    const uint2 w0 = *reinterpret_cast<const uint2 *>(qb + r * L.qp);
    const uint2 w1 = *reinterpret_cast<const uint2 *>(qb + (r + 8) * L.qp);
    const uint8_t *hrow = sh + s * L.hp + g * 128 + c * 32;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const uint2 bx = r == 0 ? *reinterpret_cast<const uint2 *>(hrow + st * 8) : make_uint2(0u, 0u);
      const uint32_t x0 = (st >> 1) ? w0.y : w0.x, x1 = (st >> 1) ? w1.y : w1.x;
      uint32_t A[4];
      if ((st & 1) == 0) {
        A[0] = codes_sub<0>(x0); A[1] = codes_sub<0>(x1); A[2] = codes_sub<1>(x0); A[3] = codes_sub<1>(x1);
      } else {
        A[0] = codes_sub<2>(x0); A[1] = codes_sub<2>(x1); A[2] = codes_sub<3>(x0); A[3] = codes_sub<3>(x1);
      }
      mma_f16(acc, A, bx.x, bx.y);
    }
    const float2 sb0 = ssb[(s * kRows + r) * GI + g], sb1 = ssb[(s * kRows + r + 8) * GI + g];
    const float hs = shs[s * GI + g], wt = swt[s];
    t0 = fmaf(wt, fmaf(sb0.x, acc[0], sb0.y * hs), t0);
    t2 = fmaf(wt, fmaf(sb1.x, acc[2], sb1.y * hs), t2);
  }
  if (c == 0) {
    sred[warp * kRows + r] = t0;
    sred[warp * kRows + r + 8] = t2;
  }
  __syncthreads();
  if (tid < kRows) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) y += sred[w * kRows + tid];
    const uint16_t yb = float_to_bf16_bits(y);
    if (a.y) a.y[n0 + tid] = yb;
    if (a.hres) a.hres[n0 + tid] = float_to_bf16_bits(bf16_bits_to_float(a.hres[n0 + tid]) + bf16_bits_to_float(yb));
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
  (void)H;
}

// ------------------------------------------------------------------ down, grouped
__global__ void __launch_bounds__(kDgThreads) down_grouped_kernel(const FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.d.H, I = a.d.I, k = a.d.k;
  const int GI = I / kGroup;
  const DownLayout L = down_layout(I, 1, kDownRows, kTokTile);
  uint8_t *sq = smem + L.q;
  uint16_t *sraw = reinterpret_cast<uint16_t *>(smem + L.raw);
  float2 *ssb = reinterpret_cast<float2 *>(smem + L.sb);
  uint8_t *sh = smem + L.h;
  float *shs = reinterpret_cast<float *>(smem + L.hs);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.y;
  const int n0 = blockIdx.x * kDownRows;
  const bool one_copy = L.qp == I / 2;
  const int nq = one_copy ? 1 : kDownRows;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](const uint8_t *blob) {
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(kDownRows * (I / 2) + 2 * kDownRows * GI * 2));
      __syncwarp();
      for (int ci = lane; ci < nq + 2; ci += 32) {
        if (ci < nq) {
          const uint32_t bytes = one_copy ? (uint32_t)(kDownRows * (I / 2)) : (uint32_t)(I / 2);
          const int row = one_copy ? 0 : ci;
          bulk_g2s(sq + row * L.qp, blob + a.w.off.down_q + (size_t)(n0 + row) * (I / 2), bytes, bar);
        } else {
          const int m = ci - nq;
          bulk_g2s(sraw + m * kDownRows * GI, blob + (m == 0 ? a.w.off.down_s : a.w.off.down_b) + (size_t)n0 * GI * 2,
                   (uint32_t)(kDownRows * GI * 2), bar);
        }
      }
    }
  };
  const bool tracer = blockIdx.x == 0 && blockIdx.y == 0 && tid == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  const bool early = a.include_shared && slot == 0;
  if (early) issue(a.w.shared);
  pdl_wait();
  if (tracer) trace_min(a.trace, kTrWaited);
  const int nact = a.r.n_act[0];
  if (slot >= nact) return;
  const int e = a.r.act_e[slot];
  const int beg = a.r.act_beg[slot];
  const int cnt = a.r.act_cnt[slot];
  if (!early) issue(slot_blob(a, e));
  pdl_launch_dependents();

  const int r = lane >> 2, c = lane & 3;
  const int wr = warp * kRows;  // this warp's first row in the tile
  bool ready = false;
  for (int j0 = 0; j0 < cnt; j0 += kTokTile) {
    const int nt = min(kTokTile, cnt - j0);
    for (int it = tid; it < nt * GI; it += kDgThreads) {
      const int n = it / GI, g = it - n * GI;
      shs[n * GI + g] = stage_group<true>(reinterpret_cast<const uint16_t *>(a.hbuf) + (size_t)(beg + j0 + n) * I,
                                          g, sh + n * L.hp);
    }
    __syncthreads();
    if (!ready) {
      if (!block_wait(bar, 0, a.err)) return;
      if (tid == 0) trace_max(a.trace, kTrLoaded);
      for (int it = tid; it < kDownRows * GI; it += kDgThreads) {
        ssb[it] = make_float2(bf16_bits_to_float(sraw[it]) * kCodeScale, bf16_bits_to_float(sraw[kDownRows * GI + it]));
      }
      __syncthreads();
      ready = true;
    }
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t *q0 = sq + (wr + r) * L.qp + c * 8;
    const uint8_t *q1 = sq + (wr + r + 8) * L.qp + c * 8;
    const uint8_t *hrow = sh + r * L.hp + c * 32;
    for (int g = 0; g < GI; ++g) {
      const uint2 w0 = *reinterpret_cast<const uint2 *>(q0 + g * 32);
      const uint2 w1 = *reinterpret_cast<const uint2 *>(q1 + g * 32);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint2 bx = *reinterpret_cast<const uint2 *>(hrow + g * 128 + st * 8);
        const uint32_t x0 = (st >> 1) ? w0.y : w0.x, x1 = (st >> 1) ? w1.y : w1.x;
        uint32_t A[4];
        if ((st & 1) == 0) {
          A[0] = codes_sub<0>(x0); A[1] = codes_sub<0>(x1); A[2] = codes_sub<1>(x0); A[3] = codes_sub<1>(x1);
        } else {
          A[0] = codes_sub<2>(x0); A[1] = codes_sub<2>(x1); A[2] = codes_sub<3>(x0); A[3] = codes_sub<3>(x1);
        }
        mma_f16(acc, A, bx.x, bx.y);
      }
      const float2 sb0 = ssb[(wr + r) * GI + g], sb1 = ssb[(wr + r + 8) * GI + g];
      const float hs0 = shs[(2 * c) * GI + g], hs1 = shs[(2 * c + 1) * GI + g];
      tot[0] = fmaf(sb0.y, hs0, fmaf(sb0.x, acc[0], tot[0]));
      tot[1] = fmaf(sb0.y, hs1, fmaf(sb0.x, acc[1], tot[1]));
      tot[2] = fmaf(sb1.y, hs0, fmaf(sb1.x, acc[2], tot[2]));
      tot[3] = fmaf(sb1.y, hs1, fmaf(sb1.x, acc[3], tot[3]));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = 2 * c + j;
      if (n < nt) {
        const int pos = beg + j0 + n;
        const float wt = pos_weight(a, pos);
        float *orow = a.obuf + (size_t)pos * H + n0 + wr;
        orow[r] = wt * tot[j];
        orow[r + 8] = wt * tot[2 + j];
      }
    }
    __syncthreads();
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
  (void)k;
}

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) combine_kernel(const FfnArgs a) {
  const int H = a.d.H, k = a.d.k, T = a.d.T;
  const int t = blockIdx.x;
  const bool tracer = t == 0 && threadIdx.x == 0;
  if (tracer) trace_min(a.trace, kTrEntry);
  pdl_wait();
  pdl_launch_dependents();
  if (tracer) trace_min(a.trace, kTrWaited);
  int pos[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) pos[j] = j < k ? a.r.pos[t * k + j] : -1;
  for (int i4 = threadIdx.x; i4 < H / 4; i4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (pos[j] >= 0) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.obuf + (size_t)pos[j] * H) + i4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    }
    if (a.include_shared) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.obuf + (size_t)(T * k + t) * H) + i4);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const uint16_t yb[4] = {float_to_bf16_bits(acc.x), float_to_bf16_bits(acc.y), float_to_bf16_bits(acc.z),
                            float_to_bf16_bits(acc.w)};
    const size_t o = (size_t)t * H + 4 * i4;
    if (a.y) {
      uint2 pk = make_uint2((uint32_t)yb[0] | ((uint32_t)yb[1] << 16), (uint32_t)yb[2] | ((uint32_t)yb[3] << 16));
      *reinterpret_cast<uint2 *>(a.y + o) = pk;
    }
    if (a.hres) {
      const uint2 hv = *reinterpret_cast<const uint2 *>(a.hres + o);
      const uint32_t hw[2] = {hv.x, hv.y};
      uint16_t nb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t hb = (hw[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
        nb[q] = float_to_bf16_bits(bf16_bits_to_float(hb) + bf16_bits_to_float(yb[q]));
      }
      *reinterpret_cast<uint2 *>(a.hres + o) =
          make_uint2((uint32_t)nb[0] | ((uint32_t)nb[1] << 16), (uint32_t)nb[2] | ((uint32_t)nb[3] << 16));
    }
  }
  if (threadIdx.x == 0) trace_max(a.trace, kTrExit);
}

// ------------------------------------------------------------------ host side
size_t gateup_smem(const Dims &d, int tt) { return (size_t)gateup_layout(d.H, tt).total; }
size_t down_decode_smem(const Dims &d) { return (size_t)down_layout(d.I, d.k + 1, kRows, d.k + 1).total; }
size_t down_grouped_smem(const Dims &d) { return (size_t)down_layout(d.I, 1, kDownRows, kTokTile).total; }

static constexpr size_t kSmemCap = 227 * 1024;

static int max_slots(const Dims &d, int include_shared) {
  const int routed = d.T * d.k < d.E ? d.T * d.k : d.E;
  return routed + (include_shared ? 1 : 0);
}

cudaError_t launch_gateup(const FfnArgs &a, cudaStream_t st, bool pdl) {
  const dim3 grid(a.d.I / kRows, max_slots(a.d, a.include_shared));
  if (a.d.T == 1) return launch_k(gateup_kernel<1>, grid, dim3(kThreads), gateup_smem(a.d, 1), st, pdl, a);
  return launch_k(gateup_kernel<kTokTile>, grid, dim3(kThreads), gateup_smem(a.d, kTokTile), st, pdl, a);
}

bool use_down_decode(const Dims &d) { return d.T == 1 && down_decode_smem(d) <= kSmemCap; }

cudaError_t launch_down(const FfnArgs &a, cudaStream_t st, bool pdl) {
  if (use_down_decode(a.d))
    return launch_k(down_decode_kernel, dim3(a.d.H / kRows), dim3(kThreads), down_decode_smem(a.d), st, pdl, a);
  cudaError_t e = launch_k(down_grouped_kernel, dim3(a.d.H / kDownRows, max_slots(a.d, a.include_shared)),
                           dim3(kDgThreads), down_grouped_smem(a.d), st, pdl, a);
  if (e != cudaSuccess) return e;
  FfnArgs c = a;
  if (c.trace) c.trace += 4;  // the combine launch traces into the next slot group
  return launch_combine(c, st, pdl);
}

cudaError_t launch_combine(const FfnArgs &a, cudaStream_t st, bool pdl) {
  return launch_k(combine_kernel, dim3(a.d.T), dim3(256), 0, st, pdl, a);
}

cudaError_t ffn_set_attributes() {
  cudaError_t e;
  const int cap = (int)kSmemCap;
  if ((e = cudaFuncSetAttribute(gateup_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap))) return e;
  if ((e = cudaFuncSetAttribute(gateup_kernel<kTokTile>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap))) return e;
  if ((e = cudaFuncSetAttribute(down_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap))) return e;
  if ((e = cudaFuncSetAttribute(down_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap))) return e;
  return cudaSuccess;
}

}  // namespace moe
