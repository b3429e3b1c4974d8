// Fused multi-token MoE layer (prefill chunks and batched decode, 2 <= T <= 128), sm_103a.
//
// Page "TurboFieldfare - System design", section "Prefill": a chunk of at
// most 128 rows goes through the layer at once; the router scores every row,
// token/expert pairs are grouped per expert, the routed experts run on their
// groups and the shared branch on every row, and the branches are combined.
//
// One persistent block per SM; 16 consumer warps and 1 producer warp.
//   A  tokens t = block, block + grid, ...: x = input (or rmsnorm of the
//      residual) -> bf16 copy, permuted fp16 operand rows and quarter sums
//      in the workspace;
//   B  router tasks (8 experts x 8 tokens): each task normalises its own 8
//      rows from the input, so no barrier separates it from A;
//   == barrier 1 ==  top-k of tokens t = block, ... (one warp each)
//   == barrier 2 ==  every block groups all pairs in shared memory (stable
//      counting sort) and derives the unit lists;
//   C  gate/up units (active slot, 8-token chunk, 16 rows of I): the
//      producer streams the 16-row gate/up tile and the chunk's operand rows
//      into a 2-slot ring; consumers compute GeGLU and write h as permuted
//      fp16 quarters with their sums;
//   == barrier 3 ==
//   D  down units (slot, chunk, 64 rows of H): weighted outputs w * o (fp32)
//      per sorted position; the weight tiles of the first units are already
//      in flight during the barrier;
//   == barrier 4 ==
//   E  combine of tokens t = block, ...: y = sum_j o[pos(t, j)] + o[shared t]
//      in selection order, bf16 out, optional residual add.
// The gate/up and down math is the tensor-core scheme of the other kernels:
// codes as exact fp16 subnormals, activations permuted and /16 on the odd
// slots, per-group correction (scale * 2^24) * acc + bias * sum.
#include <math.h>

#include "fused.cuh"
#include "kernels.h"

namespace moe {

namespace {
using fused::cons_sync;
using fused::kCons;
using fused::kConsThreads;
constexpr int kSlots = 2;
constexpr int kTC = 8;        // tokens per unit (one mma N tile)
constexpr int kGuRows = 16;   // gate/up rows per unit
constexpr int kDnRows = 64;   // down rows per unit (4 x m16)
constexpr int kNBar = 4;      // grid barriers per launch

__host__ __device__ inline int pw8(int w) { return w + ((8 - (w % 16)) + 16) % 16; }
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }

struct PL {
  int G, GI, nrt, nrt_dn;
  int gu_qp, gu_w, gu_x, gu_xq, gu_bytes;
  int dn_qp, dn_w, dn_h, dn_hq, dn_bytes;
  int slot, ring, grp, misc, total;
};

__host__ __device__ inline PL prefill_layout(int H, int I, int E, int k, int T) {
  PL L;
  L.G = H / kGroup;
  L.GI = I / kGroup;
  L.nrt = I / kGuRows;
  L.nrt_dn = H / kDnRows;
  L.gu_qp = pw8(H / 8) * 4;
  L.gu_w = 2 * kGuRows * L.gu_qp + 4 * kGuRows * L.G * 2;  // gate, up codes + 4 scale/bias tiles
  L.gu_x = al16(L.gu_w);                                   // kTC operand rows (fp16, H)
  L.gu_xq = L.gu_x + kTC * H * 2;                          // kTC rows of quarter sums (H/16 fp32)
  L.gu_bytes = al16(L.gu_xq + kTC * (H / 16) * 4);
  // the cross-warp reduction (8 floats per consumer lane) reuses the operand rows
  L.gu_bytes = max(L.gu_bytes, L.gu_x + kConsThreads * 8 * 4);
  L.dn_qp = pw8(I / 8) * 4;
  L.dn_w = kDnRows * L.dn_qp + 2 * kDnRows * L.GI * 2;
  L.dn_h = al16(L.dn_w);                                   // kTC h rows (fp16, I)
  L.dn_hq = L.dn_h + kTC * I * 2;
  L.dn_bytes = al16(L.dn_hq + kTC * (I / 16) * 4);
  L.dn_bytes = max(L.dn_bytes, L.dn_h + kConsThreads * 4 * 4);  // reduction: 4 floats per lane over the h rows
  L.slot = al16(L.gu_bytes > L.dn_bytes ? L.gu_bytes : L.dn_bytes);
  L.ring = 0;
  int o = kSlots * L.slot;
  L.grp = o;  // chunk0 int32 [E+2], perm int16 [T*k], pos int16 [T*k], act_e/beg/cnt int16 [E+1] each
  o = al16(o + (E + 2) * 4 + 2 * T * k * 2 + 3 * (E + 1) * 2);
  L.misc = o;  // flags, h staging [kTC][16] fp16, mbarriers
  o = al16(o + 1024);
  L.total = o;
  return L;
}

// Router scratch (8 rows of x as fp32) and the sort's temporaries alias the
// ring: neither is live once the producer starts.
__host__ __device__ inline bool prefill_fits(const PL &L, int H, int E) {
  return L.total <= 227 * 1024 && kSlots * L.slot >= kTC * H * 4 && kSlots * L.slot >= (1 + kCons) * E * 4;
}

// First index i in [0, n) with v[i + 1] > x (v ascending, v[0] == 0).
__device__ __forceinline__ int find_slot(const int *v, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (v[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One 64-wide group of a gate/up unit for an 8-token tile: rows r, r+8 of
// gate and up, token columns 2cq, 2cq+1.
__device__ __forceinline__ void gu_group8(const uint8_t *tile, const uint8_t *xrows, const float *xq, int H, int G,
                                          int qp, int g, int r, int cq, float (&tg)[4], float (&tu)[4]) {
  const uint16_t *raw = reinterpret_cast<const uint16_t *>(tile + 2 * 16 * qp);
  const uint2 g0 = *reinterpret_cast<const uint2 *>(tile + r * qp + g * 32 + cq * 8);
  const uint2 g1 = *reinterpret_cast<const uint2 *>(tile + (r + 8) * qp + g * 32 + cq * 8);
  const uint2 u0 = *reinterpret_cast<const uint2 *>(tile + (16 + r) * qp + g * 32 + cq * 8);
  const uint2 u1 = *reinterpret_cast<const uint2 *>(tile + (16 + r + 8) * qp + g * 32 + cq * 8);
  const uint8_t *xb = xrows + r * H * 2 + g * 128 + cq * 32;  // token row n = r
  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint2 bx = *reinterpret_cast<const uint2 *>(xb + s * 8);
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
  const int nq = H / 16;
  const float *q0 = xq + (2 * cq) * nq + 4 * g, *q1 = xq + (2 * cq + 1) * nq + 4 * g;
  const float xs0 = ((q0[0] + q0[1]) + q0[2]) + q0[3], xs1 = ((q1[0] + q1[1]) + q1[2]) + q1[3];
  const float sg0 = bf16_bits_to_float(raw[r * G + g]) * kCodeScale, bg0 = bf16_bits_to_float(raw[16 * G + r * G + g]);
  const float sg1 = bf16_bits_to_float(raw[(r + 8) * G + g]) * kCodeScale, bg1 = bf16_bits_to_float(raw[16 * G + (r + 8) * G + g]);
  const float su0 = bf16_bits_to_float(raw[32 * G + r * G + g]) * kCodeScale, bu0 = bf16_bits_to_float(raw[48 * G + r * G + g]);
  const float su1 = bf16_bits_to_float(raw[32 * G + (r + 8) * G + g]) * kCodeScale, bu1 = bf16_bits_to_float(raw[48 * G + (r + 8) * G + g]);
  tg[0] = fmaf(bg0, xs0, fmaf(sg0, ag[0], tg[0]));
  tg[1] = fmaf(bg0, xs1, fmaf(sg0, ag[1], tg[1]));
  tg[2] = fmaf(bg1, xs0, fmaf(sg1, ag[2], tg[2]));
  tg[3] = fmaf(bg1, xs1, fmaf(sg1, ag[3], tg[3]));
  tu[0] = fmaf(bu0, xs0, fmaf(su0, au[0], tu[0]));
  tu[1] = fmaf(bu0, xs1, fmaf(su0, au[1], tu[1]));
  tu[2] = fmaf(bu1, xs0, fmaf(su1, au[2], tu[2]));
  tu[3] = fmaf(bu1, xs1, fmaf(su1, au[3], tu[3]));
}

// One 64-wide group of a down unit: rows m16 + r, +8 of the 64-row tile,
// token columns 2cq, 2cq+1.
__device__ __forceinline__ void dn_group8(const uint8_t *tile, const uint8_t *hrows, const float *hq, int I, int GI,
                                          int qp, int row0, int g, int r, int cq, float (&t)[4]) {
  const uint16_t *sb = reinterpret_cast<const uint16_t *>(tile + kDnRows * qp);  // scales [64][GI], biases [64][GI]
  const uint2 w0 = *reinterpret_cast<const uint2 *>(tile + (row0 + r) * qp + g * 32 + cq * 8);
  const uint2 w1 = *reinterpret_cast<const uint2 *>(tile + (row0 + r + 8) * qp + g * 32 + cq * 8);
  const uint8_t *hb = hrows + r * I * 2 + g * 128 + cq * 32;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const uint2 bx = *reinterpret_cast<const uint2 *>(hb + st * 8);
    const uint32_t x0 = (st >> 1) ? w0.y : w0.x, x1 = (st >> 1) ? w1.y : w1.x;
    uint32_t A[4];
    if ((st & 1) == 0) {
      A[0] = codes_sub<0>(x0); A[1] = codes_sub<0>(x1); A[2] = codes_sub<1>(x0); A[3] = codes_sub<1>(x1);
    } else {
      A[0] = codes_sub<2>(x0); A[1] = codes_sub<2>(x1); A[2] = codes_sub<3>(x0); A[3] = codes_sub<3>(x1);
    }
    mma_f16(acc, A, bx.x, bx.y);
  }
  const int nq = I / 16;
  const float *q0 = hq + (2 * cq) * nq + 4 * g, *q1 = hq + (2 * cq + 1) * nq + 4 * g;
  const float hs0 = ((q0[0] + q0[1]) + q0[2]) + q0[3], hs1 = ((q1[0] + q1[1]) + q1[2]) + q1[3];
  const float s0 = bf16_bits_to_float(sb[(row0 + r) * GI + g]) * kCodeScale;
  const float b0 = bf16_bits_to_float(sb[kDnRows * GI + (row0 + r) * GI + g]);
  const float s1 = bf16_bits_to_float(sb[(row0 + r + 8) * GI + g]) * kCodeScale;
  const float b1 = bf16_bits_to_float(sb[kDnRows * GI + (row0 + r + 8) * GI + g]);
  t[0] = fmaf(b0, hs0, fmaf(s0, acc[0], t[0]));
  t[1] = fmaf(b0, hs1, fmaf(s0, acc[1], t[1]));
  t[2] = fmaf(b1, hs0, fmaf(s1, acc[2], t[2]));
  t[3] = fmaf(b1, hs1, fmaf(s1, acc[3], t[3]));
}
}  // namespace

size_t prefill_fused_smem(const Dims &d) {
  const PL L = prefill_layout(d.H, d.I, d.E, d.k, d.T);
  return prefill_fits(L, d.H, d.E) ? (size_t)L.total : 0;
}

__global__ void __launch_bounds__(fused::kThreads, 1) prefill_layer_kernel(const PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.d.H, I = a.d.I, E = a.d.E, k = a.d.k, T = a.d.T;
  const PL L = prefill_layout(H, I, E, k, T);
  const int G = L.G, GI = L.GI;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = gridDim.x, c = blockIdx.x;
  const int npairs = T * k;
  uint8_t *ring = smem + L.ring;
  int *chunk0 = reinterpret_cast<int *>(smem + L.grp);                  // [E+2]
  int16_t *g_perm = reinterpret_cast<int16_t *>(chunk0 + E + 2);        // [T*k]
  int16_t *g_pos = g_perm + npairs;                                     // [T*k]
  int16_t *g_act_e = g_pos + npairs;                                    // [E+1]
  int16_t *g_act_beg = g_act_e + (E + 1);                               // [E+1]
  int16_t *g_act_cnt = g_act_beg + (E + 1);                             // [E+1]
  int *s_flag = reinterpret_cast<int *>(smem + L.misc);                 // [16]
  __half *s_hst = reinterpret_cast<__half *>(smem + L.misc + 64);       // [kTC][16]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.misc + 64 + kTC * 16 * 2);
  uint64_t *empty = full + kSlots;
  uint64_t *route = empty + kSlots;   // grouping ready
  uint64_t *hready = route + 1;       // all h written (barrier 3 passed)

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(route, 1);
    mbar_init(hready, 1);
    fence_mbar_init();
    s_flag[8] = 0;  // abort
  }
  __syncthreads();
  if (c == 0 && tid == 0) trace_min(a.trace, kTrEntry);

  // ============================================================ producer warp
  if (warp == kCons) {
    bool ok = mbar_wait(route, 0) && *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
    fused::fence_proxy_async_global();  // operand rows written by other blocks before barrier 1
    int issued = 0;
    if (ok) {
      const int nact = s_flag[9];
      const int nchunks = chunk0[nact];
      const int n_gu = nchunks * L.nrt, n_dn = nchunks * L.nrt_dn;
      const int my_gu = c < n_gu ? (n_gu - 1 - c) / nb + 1 : 0;
      const int my_dn = c < n_dn ? (n_dn - 1 - c) / nb + 1 : 0;
      bool hr = false;
      for (int it = 0; it < my_gu + my_dn && ok; ++it) {
        const int slot = it % kSlots;
        if (it >= kSlots) ok = mbar_wait(&empty[slot], ((it / kSlots) - 1) & 1);
        if (!ok) break;
        uint8_t *dst = ring + slot * L.slot;
        const bool is_gu = it < my_gu;
        const int u = c + nb * (is_gu ? it : it - my_gu);
        const int per = is_gu ? L.nrt : L.nrt_dn;
        const int chg = u / per, tile = u - chg * per;
        const int sa = find_slot(chunk0, nact + 1, chg);
        const int ch = chg - chunk0[sa];
        const int e = g_act_e[sa], beg = g_act_beg[sa];
        const int nt = min(kTC, (int)g_act_cnt[sa] - kTC * ch);
        const uint8_t *blob = e < 0 ? a.w.shared : a.w.experts + (size_t)e * a.w.stride;
        if (is_gu) {
          const int r0 = tile * kGuRows;
          const uint32_t tx = (uint32_t)(2 * kGuRows * (H / 2) + 4 * kGuRows * G * 2 + nt * (H * 2 + (H / 16) * 4));
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], tx);
          __syncwarp();
          const int m = lane >> 4, row = lane & 15;
          bulk_g2s(dst + (m * kGuRows + row) * L.gu_qp,
                   blob + (m == 0 ? a.w.off.gate_q : a.w.off.up_q) + (size_t)(r0 + row) * (H / 2), (uint32_t)(H / 2),
                   &full[slot]);
          if (lane < 4) {
            const size_t off = lane == 0 ? a.w.off.gate_s : lane == 1 ? a.w.off.gate_b : lane == 2 ? a.w.off.up_s : a.w.off.up_b;
            bulk_g2s(dst + 2 * kGuRows * L.gu_qp + lane * kGuRows * G * 2, blob + off + (size_t)r0 * G * 2,
                     (uint32_t)(kGuRows * G * 2), &full[slot]);
          }
          if (lane < 2 * nt) {
            const int j = lane >> 1;
            const int tok = e < 0 ? kTC * ch + j : g_perm[beg + kTC * ch + j] / k;
            if ((lane & 1) == 0)
              bulk_g2s(dst + L.gu_x + j * H * 2, a.xperm + (size_t)tok * H, (uint32_t)(H * 2), &full[slot]);
            else
              bulk_g2s(dst + L.gu_xq + j * (H / 16) * 4, a.xq + (size_t)tok * (H / 16), (uint32_t)((H / 16) * 4),
                       &full[slot]);
          }
        } else {
          const int n0 = tile * kDnRows;
          // weights first (they do not depend on h): bytes expected without
          // the arrival, so the phase cannot complete before the h rows land
          if (lane == 0) fused::mbar_expect_tx(&full[slot], (uint32_t)(kDnRows * (I / 2) + 2 * kDnRows * GI * 2));
          __syncwarp();
          const bool one = L.dn_qp == I / 2;
          const int nq = one ? 1 : kDnRows;
          for (int ci = lane; ci < nq + 2; ci += 32) {
            if (ci < nq) {
              const int row = one ? 0 : ci;
              bulk_g2s(dst + row * L.dn_qp, blob + a.w.off.down_q + (size_t)(n0 + row) * (I / 2),
                       one ? (uint32_t)(kDnRows * (I / 2)) : (uint32_t)(I / 2), &full[slot]);
            } else {
              const int f = ci - nq;
              bulk_g2s(dst + kDnRows * L.dn_qp + f * kDnRows * GI * 2,
                       blob + (f == 0 ? a.w.off.down_s : a.w.off.down_b) + (size_t)n0 * GI * 2,
                       (uint32_t)(kDnRows * GI * 2), &full[slot]);
            }
          }
          // ... then the h rows, once every block has written them
          if (!hr) {
            ok = mbar_wait(hready, 0) && *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
            fused::fence_proxy_async_global();
            hr = true;
          }
          // on a failure the arrival alone ends the phase once the weights land
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], ok ? (uint32_t)(nt * (I * 2 + (I / 16) * 4)) : 0u);
          __syncwarp();
          if (ok && lane < 2 * nt) {
            const int j = lane >> 1;
            const int pos = beg + kTC * ch + j;
            if ((lane & 1) == 0)
              bulk_g2s(dst + L.dn_h + j * I * 2, a.hperm + (size_t)pos * I, (uint32_t)(I * 2), &full[slot]);
            else
              bulk_g2s(dst + L.dn_hq + j * (I / 16) * 4, a.hq + (size_t)pos * (I / 16), (uint32_t)((I / 16) * 4),
                       &full[slot]);
          }
        }
        issued = it + 1;
      }
    }
    // copies in flight must land before the block's shared memory is released
    if (lane == 0) {
      if (!ok) set_error(a.err, kErrTimeout);
      for (int it = issued - kSlots > 0 ? issued - kSlots : 0; it < issued; ++it)
        mbar_wait(&full[it % kSlots], (it / kSlots) & 1);
    }
    return;
  }

  // ============================================================ consumers
  pdl_wait();
  pdl_launch_dependents();
  if (c == 0 && tid == 0) trace_min(a.trace, kTrWaited);
  unsigned long long *bar_count = reinterpret_cast<unsigned long long *>(a.sync);
  const unsigned long long base =
      (fused::ld_acquire64(bar_count) / ((unsigned long long)kNBar * nb)) * ((unsigned long long)kNBar * nb);
  bool aborted = false;
  int nbar = 0;
  // every launch arrives at all kNBar barriers, even after a failure
  auto barrier = [&]() {
    ++nbar;
    if (!aborted) {
      aborted = !fused::grid_sync(bar_count, base + (unsigned long long)nbar * nb, a.err, &s_flag[nbar]);
    } else {
      cons_sync();
      if (tid == 0) fused::red_release_add(bar_count);
      cons_sync();
    }
  };
  const uint16_t *src = a.normalize ? a.hres : a.x;
  const int nquart = H / 16;

  // ---- A: operand rows of tokens t = c, c + nb, ...
  for (int t = c; t < T; t += nb) {
    uint32_t qin[8];
    float qss = 0.f;
    if (tid < nquart) {
      const uint4 v0 = __ldcg(reinterpret_cast<const uint4 *>(src + (size_t)t * H) + 2 * tid);
      const uint4 v1 = __ldcg(reinterpret_cast<const uint4 *>(src + (size_t)t * H) + 2 * tid + 1);
      qin[0] = v0.x; qin[1] = v0.y; qin[2] = v0.z; qin[3] = v0.w;
      qin[4] = v1.x; qin[5] = v1.y; qin[6] = v1.z; qin[7] = v1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float lo = __uint_as_float(qin[i] << 16), hi = __uint_as_float(qin[i] & 0xFFFF0000u);
        qss = fmaf(lo, lo, qss);
        qss = fmaf(hi, hi, qss);
      }
    }
    if (a.normalize) {
      float *s_part = reinterpret_cast<float *>(ring);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) qss += __shfl_xor_sync(0xffffffffu, qss, off);
      if (lane == 0) s_part[warp] = qss;
      cons_sync();
      float tot = 0.f;
      for (int w = 0; w < kCons; ++w) tot += s_part[w];
      const float inv = 1.0f / sqrtf(tot / (float)H + 1e-6f);
      if (tid < nquart) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint16_t lb = float_to_bf16_bits(__uint_as_float(qin[i] << 16) * inv);
          const uint16_t hb = float_to_bf16_bits(__uint_as_float(qin[i] & 0xFFFF0000u) * inv);
          qin[i] = (uint32_t)lb | ((uint32_t)hb << 16);
        }
      }
      cons_sync();
    }
    if (tid < nquart) {
      if (a.xn_user) {
        uint4 *xu = reinterpret_cast<uint4 *>(a.xn_user + (size_t)t * H) + 2 * tid;
        xu[0] = make_uint4(qin[0], qin[1], qin[2], qin[3]);
        xu[1] = make_uint4(qin[4], qin[5], qin[6], qin[7]);
      }
      uint32_t out[8];
      operand_quarter<true>(qin, out);
      uint4 *xp = reinterpret_cast<uint4 *>(a.xperm + (size_t)t * H) + 2 * tid;
      xp[0] = make_uint4(out[0], out[1], out[2], out[3]);
      xp[1] = make_uint4(out[4], out[5], out[6], out[7]);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        s += __uint_as_float(qin[i] << 16);
        s += __uint_as_float(qin[i] & 0xFFFF0000u);
      }
      a.xq[(size_t)t * nquart + tid] = s;
    }
  }

  // ---- B: router tasks (8 experts x 8 tokens), logits[t][e]
  {
    const int n_eb = (E + 7) / 8, n_tb = (T + 7) / 8;
    float *xs = reinterpret_cast<float *>(ring);  // [8][H] fp32
    for (int task = c; task < n_eb * n_tb; task += nb) {
      const int eb = task % n_eb, tb = task / n_eb;
      const int t0 = tb * 8, tn = min(8, T - t0);
      const int e = eb * 8 + (warp & 7);
      const int half = warp >> 3;  // tokens t0 + 4*half .. +3
      cons_sync();                 // xs free (previous task, phase A's s_part)
      // stage the 8 rows (normalised like phase A) as fp32
      for (int n = 0; n < tn; ++n) {
        uint32_t qin[8];
        float qss = 0.f;
        if (tid < nquart) {
          const uint4 v0 = __ldcg(reinterpret_cast<const uint4 *>(src + (size_t)(t0 + n) * H) + 2 * tid);
          const uint4 v1 = __ldcg(reinterpret_cast<const uint4 *>(src + (size_t)(t0 + n) * H) + 2 * tid + 1);
          qin[0] = v0.x; qin[1] = v0.y; qin[2] = v0.z; qin[3] = v0.w;
          qin[4] = v1.x; qin[5] = v1.y; qin[6] = v1.z; qin[7] = v1.w;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float lo = __uint_as_float(qin[i] << 16), hi = __uint_as_float(qin[i] & 0xFFFF0000u);
            qss = fmaf(lo, lo, qss);
            qss = fmaf(hi, hi, qss);
          }
        }
        float inv = 1.0f;
        if (a.normalize) {
          float *s_part = reinterpret_cast<float *>(smem + L.misc + 512);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) qss += __shfl_xor_sync(0xffffffffu, qss, off);
          if (lane == 0) s_part[warp] = qss;
          cons_sync();
          float tot = 0.f;
          for (int w = 0; w < kCons; ++w) tot += s_part[w];
          inv = 1.0f / sqrtf(tot / (float)H + 1e-6f);
          cons_sync();
        }
        if (tid < nquart) {
          float4 *dst = reinterpret_cast<float4 *>(xs + n * H + 16 * tid);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float f[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              float lo = __uint_as_float(qin[2 * i + j] << 16), hi = __uint_as_float(qin[2 * i + j] & 0xFFFF0000u);
              if (a.normalize) {
                lo = bf16_bits_to_float(float_to_bf16_bits(lo * inv));
                hi = bf16_bits_to_float(float_to_bf16_bits(hi * inv));
              }
              f[2 * j] = lo;
              f[2 * j + 1] = hi;
            }
            dst[i] = make_float4(f[0], f[1], f[2], f[3]);
          }
        }
      }
      cons_sync();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (e < E) {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.w.router_q + (size_t)e * H);
        const uint16_t *srow = a.w.router_s + (size_t)e * G, *brow = a.w.router_b + (size_t)e * G;
        for (int cw = lane; cw < H / 4; cw += 32) {
          const uint32_t wd = __ldg(qrow + cw);
          const float s = bf16_bits_to_float(__ldg(srow + (cw >> 4))), b = bf16_bits_to_float(__ldg(brow + (cw >> 4)));
          float w4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w4[i] = fmaf(__uint_as_float(0x4B000000u | ((wd >> (8 * i)) & 0xFFu)) - 8388608.0f, s, b);
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            const int tt = 4 * half + n;
            if (tt < tn) {
              const float4 xv = *reinterpret_cast<const float4 *>(xs + tt * H + 4 * cw);
              acc[n] = fmaf(w4[3], xv.w, fmaf(w4[2], xv.z, fmaf(w4[1], xv.y, fmaf(w4[0], xv.x, acc[n]))));
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
      if (e < E && lane == 0) {
        const float bias = a.w.logit_bias ? a.w.logit_bias[e] : 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n)
          if (4 * half + n < tn) a.logits[(size_t)(t0 + 4 * half + n) * E + e] = acc[n] + bias;
      }
    }
  }

  fused::fence_proxy_async_global();  // operand rows are read back by bulk copies
  barrier();  // 1: logits, operand rows, quarter sums
  // ---- top-k of tokens t = c, c + nb, ...
  if (!aborted && warp == 0) {
    for (int t = c; t < T; t += nb) {
      bool bad = false;
      fused::warp_topk(a.logits + (size_t)t * E, E, k, a.r.ids + t * k, a.r.wts + t * k, &bad);
      if (bad && lane == 0) set_error(a.err, kErrNonFinite);
      __syncwarp();
      if (lane < k) {
        if (a.ids_user) a.ids_user[t * k + lane] = a.r.ids[t * k + lane];
        if (a.wts_user) a.wts_user[t * k + lane] = a.r.wts[t * k + lane];
      }
    }
  }
  barrier();  // 2: ids, weights

  // ---- every block groups all pairs (stable counting sort by expert id)
  if (!aborted) {
    int *cnt = reinterpret_cast<int *>(ring);  // [E]
    int *wc = cnt + E;                         // [kCons][E]
    for (int i = tid; i < (1 + kCons) * E; i += kConsThreads) cnt[i] = 0;
    cons_sync();
    for (int p = tid; p < npairs; p += kConsThreads) atomicAdd(&cnt[__ldcg(a.r.ids + p)], 1);
    cons_sync();
    if (warp == 0) {
      // exclusive scan of counts -> offsets; active slots (shared first); chunk prefix
      int run = 0, nact = 1, chunks = (T + kTC - 1) / kTC;
      if (lane == 0) {
        g_act_e[0] = -1;
        g_act_beg[0] = (int16_t)npairs;
        g_act_cnt[0] = (int16_t)T;
        chunk0[0] = 0;
      }
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int ce = e < E ? cnt[e] : 0;
        int incl = ce;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        const int nch = (ce + kTC - 1) / kTC;
        int incl_ch = nch;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl_ch, off);
          if (lane >= off) incl_ch += v;
        }
        const unsigned act = __ballot_sync(0xffffffffu, ce > 0);
        if (ce > 0) {
          const int sa = nact + __popc(act & lanemask_lt());
          g_act_e[sa] = (int16_t)e;
          g_act_beg[sa] = (int16_t)(run + incl - ce);
          g_act_cnt[sa] = (int16_t)ce;
          chunk0[sa] = chunks + incl_ch - nch;
        }
        if (e < E) cnt[e] = run + incl - ce;  // from here on: next free position of expert e
        run +=__shfl_sync(0xffffffffu, incl, 31);
        chunks += __shfl_sync(0xffffffffu, incl_ch, 31);
        nact += __popc(act);
      }
      if (lane == 0) {
        chunk0[nact] = chunks;
        s_flag[9] = nact;
      }
    }
    cons_sync();
    for (int base0 = 0; base0 < npairs; base0 += kConsThreads) {
      const int p = base0 + tid;
      const int e = p < npairs ? __ldcg(a.r.ids + p) : -1;
      const int key = p < npairs ? e : kMaxExperts + lane;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int rank = __popc(peers & lanemask_lt());
      if (p < npairs && rank == 0) wc[warp * E + e] = __popc(peers);
      cons_sync();
      if (p < npairs) {
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wc[w * E + e];
        const int q = cnt[e] + before + rank;
        g_perm[q] = (int16_t)p;
        g_pos[p] = (int16_t)q;
      }
      cons_sync();
      for (int e2 = tid; e2 < E; e2 += kConsThreads) {
        int add = 0;
        for (int w = 0; w < kCons; ++w) {
          add += wc[w * E + e2];
          wc[w * E + e2] = 0;
        }
        cnt[e2] += add;
      }
      cons_sync();
    }
  }
  if (tid == 0) {
    if (aborted) s_flag[8] = 1;
    mbar_arrive_expect_tx(route, 0);  // the producer may stream (or, on abort, drain and exit)
  }
  if (c == 0 && tid == 0) trace_max(a.trace, kTrLoaded);

  // ---- C: gate/up units
  const int nact = s_flag[9];
  const int nchunks = aborted ? 0 : chunk0[nact];
  const int n_gu = nchunks * L.nrt, n_dn = nchunks * L.nrt_dn;
  const int my_gu = c < n_gu ? (n_gu - 1 - c) / nb + 1 : 0;
  const int my_dn = c < n_dn ? (n_dn - 1 - c) / nb + 1 : 0;
  const int r = lane >> 2, cq = lane & 3;
  int it = 0;
  for (; it < my_gu && !aborted; ++it) {
    const int slot = it % kSlots;
    if (!mbar_wait(&full[slot], (it / kSlots) & 1)) {
      aborted = true;
      set_error(a.err, kErrTimeout);
      break;
    }
    const uint8_t *tile = ring + slot * L.slot;
    const int u = c + nb * it;
    const int chg = u / L.nrt, rt = u - chg * L.nrt;
    const int sa = find_slot(chunk0, nact + 1, chg);
    const int ch = chg - chunk0[sa];
    const int beg = g_act_beg[sa];
    const int nt = min(kTC, (int)g_act_cnt[sa] - kTC * ch);
    float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
    float tg2[4] = {0.f, 0.f, 0.f, 0.f}, tu2[4] = {0.f, 0.f, 0.f, 0.f};
    int g = warp;
    for (; g + kCons < G; g += 2 * kCons) {
      gu_group8(tile, tile + L.gu_x, reinterpret_cast<const float *>(tile + L.gu_xq), H, G, L.gu_qp, g, r, cq, tg, tu);
      gu_group8(tile, tile + L.gu_x, reinterpret_cast<const float *>(tile + L.gu_xq), H, G, L.gu_qp, g + kCons, r, cq,
                tg2, tu2);
    }
    if (g < G)
      gu_group8(tile, tile + L.gu_x, reinterpret_cast<const float *>(tile + L.gu_xq), H, G, L.gu_qp, g, r, cq, tg, tu);
    cons_sync();  // the slot's operand rows become the reduction buffer
    float *red = reinterpret_cast<float *>(const_cast<uint8_t *>(tile) + L.gu_x);
    float4 *rw = reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 8);
    rw[0] = make_float4(tg[0] + tg2[0], tg[1] + tg2[1], tg[2] + tg2[2], tg[3] + tg2[3]);
    rw[1] = make_float4(tu[0] + tu2[0], tu[1] + tu2[1], tu[2] + tu2[2], tu[3] + tu2[3]);
    cons_sync();
    if (tid < kGuRows * kTC) {
      const int row = tid & 15, n = tid >> 4;
      const int ln = (row & 7) * 4 + (n >> 1), idx = ((row >> 3) << 1) + (n & 1);
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < kCons; ++w) {
        gs += red[(w * 32 + ln) * 8 + idx];
        us += red[(w * 32 + ln) * 8 + 4 + idx];
      }
      const float hv = fused::gelu_tanh(gs) * us;
      if (n < nt && !(fabsf(hv) <= 65504.0f)) set_error(a.err, kErrNonFinite);
      s_hst[n * 16 + row] = __float2half_rn(hv);
    }
    cons_sync();
    if (tid < nt) {  // one thread per token writes its 16-row quarter of h
      const int pos = beg + kTC * ch + tid;
      const uint4 *hv = reinterpret_cast<const uint4 *>(s_hst + tid * 16);
      const uint4 v0 = hv[0], v1 = hv[1];
      const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t out[8];
      operand_quarter<false>(in, out);
      uint4 *dst = reinterpret_cast<uint4 *>(a.hperm + (size_t)pos * I + rt * kGuRows);
      dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        s += __half2float(__ushort_as_half((unsigned short)(in[w] & 0xFFFFu)));
        s += __half2float(__ushort_as_half((unsigned short)(in[w] >> 16)));
      }
      a.hq[(size_t)pos * (I / 16) + rt] = s;
    }
    cons_sync();
    if (tid == 0) mbar_arrive_expect_tx(&empty[slot], 0);
  }

  fused::fence_proxy_async_global();  // h rows are read back by bulk copies
  barrier();  // 3: all of h
  if (tid == 0) {
    if (aborted) s_flag[8] = 1;
    mbar_arrive_expect_tx(hready, 0);
  }

  // ---- D: down units -> weighted outputs per sorted position
  for (int jd = 0; jd < my_dn && !aborted; ++jd, ++it) {
    const int slot = it % kSlots;
    if (!mbar_wait(&full[slot], (it / kSlots) & 1)) {
      aborted = true;
      set_error(a.err, kErrTimeout);
      break;
    }
    const uint8_t *tile = ring + slot * L.slot;
    const int u = c + nb * jd;
    const int chg = u / L.nrt_dn, nt64 = u - chg * L.nrt_dn;
    const int sa = find_slot(chunk0, nact + 1, chg);
    const int ch = chg - chunk0[sa];
    const int beg = g_act_beg[sa];
    const int nt = min(kTC, (int)g_act_cnt[sa] - kTC * ch);
    const int m = warp & 3, kq = warp >> 2;  // 16-row tile, K quarter
    float t4[4] = {0.f, 0.f, 0.f, 0.f}, t4b[4] = {0.f, 0.f, 0.f, 0.f};
    int g = kq;
    for (; g + 4 < GI; g += 8) {
      dn_group8(tile, tile + L.dn_h, reinterpret_cast<const float *>(tile + L.dn_hq), I, GI, L.dn_qp, 16 * m, g, r, cq, t4);
      dn_group8(tile, tile + L.dn_h, reinterpret_cast<const float *>(tile + L.dn_hq), I, GI, L.dn_qp, 16 * m, g + 4, r,
                cq, t4b);
    }
    if (g < GI)
      dn_group8(tile, tile + L.dn_h, reinterpret_cast<const float *>(tile + L.dn_hq), I, GI, L.dn_qp, 16 * m, g, r, cq, t4);
    cons_sync();  // the slot's h rows become the reduction buffer
    float *red = reinterpret_cast<float *>(const_cast<uint8_t *>(tile) + L.dn_h);
    *reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 4) =
        make_float4(t4[0] + t4b[0], t4[1] + t4b[1], t4[2] + t4b[2], t4[3] + t4b[3]);
    cons_sync();
    for (int o = tid; o < kDnRows * kTC; o += kConsThreads) {
      const int row = o & 63, n = o >> 6;
      if (n < nt) {
        const int mm = row >> 4, rr = row & 15;
        const int ln = (rr & 7) * 4 + (n >> 1), idx = ((rr >> 3) << 1) + (n & 1);
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) v += red[(((q << 2) | mm) * 32 + ln) * 4 + idx];
        const int pos = beg + kTC * ch + n;
        const float wt = pos >= npairs ? 1.0f : __ldcg(a.r.wts + g_perm[pos]);
        a.obuf[(size_t)pos * H + nt64 * kDnRows + row] = wt * v;
      }
    }
    cons_sync();
    if (tid == 0) mbar_arrive_expect_tx(&empty[slot], 0);
  }

  barrier();  // 4: all weighted outputs
  // ---- E: combine tokens t = c, c + nb, ...
  if (!aborted) {
    for (int t = c; t < T; t += nb) {
      int pos[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) pos[j] = j < k ? g_pos[t * k + j] : -1;
      for (int i4 = tid; i4 < H / 4; i4 += kConsThreads) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          if (pos[j] >= 0) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.obuf + (size_t)pos[j] * H) + i4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
        }
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.obuf + (size_t)(npairs + t) * H) + i4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        const uint16_t yb[4] = {float_to_bf16_bits(acc.x), float_to_bf16_bits(acc.y), float_to_bf16_bits(acc.z),
                                float_to_bf16_bits(acc.w)};
        const size_t o = (size_t)t * H + 4 * i4;
        if (a.y)
          *reinterpret_cast<uint2 *>(a.y + o) =
              make_uint2((uint32_t)yb[0] | ((uint32_t)yb[1] << 16), (uint32_t)yb[2] | ((uint32_t)yb[3] << 16));
        if (a.hres) {
          const uint2 hv = *reinterpret_cast<const uint2 *>(a.hres + o);
          const uint32_t hw[2] = {hv.x, hv.y};
          uint16_t nbits[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t hb = (hw[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
            nbits[q] = float_to_bf16_bits(bf16_bits_to_float(hb) + bf16_bits_to_float(yb[q]));
          }
          *reinterpret_cast<uint2 *>(a.hres + o) = make_uint2((uint32_t)nbits[0] | ((uint32_t)nbits[1] << 16),
                                                              (uint32_t)nbits[2] | ((uint32_t)nbits[3] << 16));
        }
      }
    }
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
}

cudaError_t launch_prefill_fused(const PrefillArgs &a, int n_blocks, cudaStream_t st, bool pdl) {
  return launch_k(prefill_layer_kernel, dim3(n_blocks), dim3(fused::kThreads), prefill_fused_smem(a.d), st, pdl, a);
}

cudaError_t prefill_set_attributes() {
  return cudaFuncSetAttribute(prefill_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

int prefill_blocks_per_sm(const Dims &d) {
  const size_t smem = prefill_fused_smem(d);
  if (smem == 0) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_layer_kernel, fused::kThreads, smem) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace moe
