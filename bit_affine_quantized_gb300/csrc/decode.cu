// Fused single-token MoE layer (decode, T == 1), sm_103a.
//
// Page "TurboFieldfare - System design", section "Decode": per layer the
// router picks 8 of 128 experts, the shared expert runs alongside, the routed
// outputs are reduced with the router weights and added to the shared one
// (section "Metal execution" fuses decode, GeGLU and the weighted reduction).
// There, the expert ids travel GPU -> CPU -> SSD reads -> GPU; here every
// expert is in HBM and the whole layer is one launch.
//
// One persistent block per SM (the grid is the SM count; shared memory use
// keeps it at one block per SM).  Phases:
//   0. before the dependency wait: this block's router row goes to
//      registers, and the producer warp starts the bulk copies of the
//      shared expert's gate/up tiles (they need no routing);
//   1. x = input (or rmsnorm of the residual), one logit per block row;
//   2. grid barrier; every block computes the top-k itself (no second
//      barrier), then the producer streams the routed gate/up tiles and the
//      down tiles through a 3-slot ring of shared memory;
//   3. gate/up + GeGLU per 16-row unit (mma.m16n8k16, exact integer
//      operands, per-group affine correction), h to global fp16;
//   4. grid barrier; down for 16 output rows over all k+1 experts, weighted
//      sum, bf16 out, optional residual add.
// All waits are bounded (2 s): a timeout records MOE_ERR_TIMEOUT, the block
// drains its copies in flight and exits.
#include <math.h>

#include "kernels.h"

namespace moe {

namespace {
constexpr int kCons = 16;                    // consumer warps
constexpr int kConsThreads = kCons * 32;     // 512
constexpr int kThreadsF = kConsThreads + 32; // + producer warp
constexpr int kSlots = 3;                    // ring slots
constexpr int kRowsU = 16;                   // rows per unit

__host__ __device__ inline int pw8(int w) { return w + ((8 - (w % 16)) + 16) % 16; }
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }

struct FusedLayout {
  int nrt;          // gate/up units per expert (I / 16)
  int n_gu, n_dn;   // gate/up units, down units
  int gu_qp;        // gate/up 4-row block pitch (bytes)
  int gu_bytes, dn_qp, dn_slot_bytes, dn_bytes, slot_bytes;
  int ring, xperm, xsum, qsum, hperm, hsum, red, misc, rsc, pes, total;
};

__host__ __device__ inline FusedLayout fused_layout(int H, int I, int k) {
  FusedLayout L;
  const int G = H / kGroup, GI = I / kGroup, S = k + 1;
  L.nrt = I / kRowsU;
  L.n_gu = S * L.nrt;
  L.n_dn = H / kRowsU;
  L.gu_qp = quad_pitch(H);
  L.gu_bytes = quad_tile_bytes(H);
  L.dn_qp = pw8(I / 8) * 4;
  L.dn_slot_bytes = kRowsU * L.dn_qp + 2 * kRowsU * GI * 2;
  L.dn_bytes = S * L.dn_slot_bytes;
  L.slot_bytes = al16(L.gu_bytes > L.dn_bytes ? L.gu_bytes : L.dn_bytes);
  int o = 0;
  L.ring = o;
  o += kSlots * L.slot_bytes;
  L.xperm = o;
  o = al16(o + H * 2);
  L.xsum = o;
  o = al16(o + G * 4);
  L.qsum = o;
  o = al16(o + (H / 16) * 4);
  L.hperm = o;
  o = al16(o + S * I * 2);
  L.hsum = o;
  o = al16(o + S * GI * 4);
  L.red = o;
  o = al16(o + kCons * 32 * 8 * 4);
  L.misc = o;  // partial sums, k ids, k weights, flags, 2*kSlots+1 mbarriers
  o = al16(o + 512);
  L.rsc = o;  // the router scale (when given), bf16 [H]
  o = al16(o + H * 2);
  L.pes = o;  // per-expert routing-weight scales (when given), fp32 [E]
  o = al16(o + kMaxExperts * 4);
  L.total = o;
  return L;
}

__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsThreads) : "memory"); }

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier on one 64-bit arrival counter, run by the consumer threads of
// every block: each block adds 1 with a release reduction (no return value,
// so arrivals pipeline at L2 instead of serialising) and polls until the
// counter reaches `target`.  The counter only grows; a launch's targets are
// derived from its value at launch start (see the caller).  Bounded.
// grid_arrive + grid_wait split the barrier so a block can work in between.
__device__ __forceinline__ void grid_arrive(unsigned long long *count) {
  cons_sync();  // the block's writes happen-before thread 0's release below
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(count) : "memory");
}
__device__ bool grid_wait(unsigned long long *count, unsigned long long target, unsigned *err, int *s_flag,
                          unsigned long long limit_ns) {
  if (threadIdx.x == 0) {
    bool ok = true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire64(count) >= target) break;
      if ((it & 15u) == 15u && global_ns() - t0 > limit_ns) {
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
// arrive = false withholds this block's arrival (the failure-detection hook)
__device__ bool grid_sync(unsigned long long *count, unsigned long long target, unsigned *err, int *s_flag,
                          unsigned long long limit_ns, bool arrive = true) {
  if (arrive) grid_arrive(count);
  return grid_wait(count, target, err, s_flag, limit_ns);
}

// Orderable 32-bit key of a float (larger float -> larger key).
__device__ __forceinline__ unsigned ord_key(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One 64-wide group of a gate/up unit: mma rows r, r+8 (tile rows quad_row(r),
// quad_row(r + 8)) of gate and up, token column 0 (valid in the lanes with
// cq == 0).  Accumulates the affine-corrected partials s*acc + b*sum(x).
__device__ __forceinline__ void gu_group(const uint8_t *tile, const uint8_t *xperm, const float *xsum, int g, int r,
                                         int cq, int G, int qp, float &tg0, float &tg2, float &tu0, float &tu2) {
  const int rowb = G * 32;                    // bytes of one row of codes (H / 2)
  const int sr0 = quad_row(r), sr1 = sr0 + 2;  // tile rows of mma rows r and r + 8
  const uint16_t *raw = reinterpret_cast<const uint16_t *>(tile + 8 * qp);  // gs, gb, us, ub [16][G]
  const uint8_t *ga = tile + (r & 3) * qp + (r >> 2) * rowb + g * 32 + cq * 8;
  const uint2 g0 = *reinterpret_cast<const uint2 *>(ga);
  const uint2 g1 = *reinterpret_cast<const uint2 *>(ga + 2 * rowb);
  const uint2 u0 = *reinterpret_cast<const uint2 *>(ga + 4 * qp);
  const uint2 u1 = *reinterpret_cast<const uint2 *>(ga + 4 * qp + 2 * rowb);
  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint2 bx = r == 0 ? *reinterpret_cast<const uint2 *>(xperm + g * 128 + cq * 32 + s * 8) : make_uint2(0u, 0u);
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
  const float xs = xsum[g];
  const float sg0 = bf16_bits_to_float(raw[sr0 * G + g]), bg0 = bf16_bits_to_float(raw[16 * G + sr0 * G + g]);
  const float sg1 = bf16_bits_to_float(raw[sr1 * G + g]), bg1 = bf16_bits_to_float(raw[16 * G + sr1 * G + g]);
  const float su0 = bf16_bits_to_float(raw[32 * G + sr0 * G + g]), bu0 = bf16_bits_to_float(raw[48 * G + sr0 * G + g]);
  const float su1 = bf16_bits_to_float(raw[32 * G + sr1 * G + g]), bu1 = bf16_bits_to_float(raw[48 * G + sr1 * G + g]);
  tg0 = fmaf(bg0, xs, fmaf(sg0 * kCodeScale, ag[0], tg0));
  tg2 = fmaf(bg1, xs, fmaf(sg1 * kCodeScale, ag[2], tg2));
  tu0 = fmaf(bu0, xs, fmaf(su0 * kCodeScale, au[0], tu0));
  tu2 = fmaf(bu1, xs, fmaf(su1 * kCodeScale, au[2], tu2));
}

// One (expert slot, 64-wide group) item of a down unit: rows r, r+8 of the
// 16-row tile, token column 0 (valid in the lanes with cq == 0).
//   tq   codes of the item in the tile, at this lane's 8 bytes (row 0)
//   sq   scale of row 0 of the item (bf16); biases follow 16 rows later
//   hq   the item's 64 operand values, at this lane's 32 bytes
//   hsw  router weight of the item's expert times the group sum of h
//   w24  router weight times 2^24 (undoes the code scale of the mma)
// Accumulates weight * (s * sum(q h) + b * sum(h)) into t0 (row r) and t2
// (row r + 8).
__device__ __forceinline__ void down_item(const uint8_t *tq, const uint16_t *sq, const uint8_t *hq, float hsw,
                                          float w24, int r, int qp_r0, int qp_r1, int GI, float &t0, float &t2) {
  const uint2 w0 = *reinterpret_cast<const uint2 *>(tq + qp_r0);
  const uint2 w1 = *reinterpret_cast<const uint2 *>(tq + qp_r1);
  uint4 b01 = make_uint4(0u, 0u, 0u, 0u), b23 = make_uint4(0u, 0u, 0u, 0u);
  if (r == 0) {
    b01 = *reinterpret_cast<const uint4 *>(hq);
    b23 = *reinterpret_cast<const uint4 *>(hq + 16);
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint32_t A[4] = {codes_sub<0>(w0.x), codes_sub<0>(w1.x), codes_sub<1>(w0.x), codes_sub<1>(w1.x)};
    mma_f16(acc, A, b01.x, b01.y);
  }
  {
    uint32_t A[4] = {codes_sub<2>(w0.x), codes_sub<2>(w1.x), codes_sub<3>(w0.x), codes_sub<3>(w1.x)};
    mma_f16(acc, A, b01.z, b01.w);
  }
  {
    uint32_t A[4] = {codes_sub<0>(w0.y), codes_sub<0>(w1.y), codes_sub<1>(w0.y), codes_sub<1>(w1.y)};
    mma_f16(acc, A, b23.x, b23.y);
  }
  {
    uint32_t A[4] = {codes_sub<2>(w0.y), codes_sub<2>(w1.y), codes_sub<3>(w0.y), codes_sub<3>(w1.y)};
    mma_f16(acc, A, b23.z, b23.w);
  }
  const float s0 = bf16_bits_to_float(sq[r * GI]), b0 = bf16_bits_to_float(sq[(16 + r) * GI]);
  const float s1 = bf16_bits_to_float(sq[(r + 8) * GI]), b1 = bf16_bits_to_float(sq[(24 + r) * GI]);
  t0 = fmaf(s0 * acc[0], w24, fmaf(b0, hsw, t0));
  t2 = fmaf(s1 * acc[2], w24, fmaf(b1, hsw, t2));
}
}  // namespace

size_t fused_decode_smem(const Dims &d) {
  if (d.H / 16 > kConsThreads) return 0;  // one 16-element quarter of x per consumer thread
  return (size_t)fused_layout(d.H, d.I, d.k).total;
}

// kScales: the layer has learned router scales (the router-scale code is
// compiled out of the plain instance).
template <bool kScales>
__global__ void __launch_bounds__(kThreadsF, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.d.H, I = a.d.I, E = a.d.E, k = a.d.k;
  const int G = H / kGroup, GI = I / kGroup, S = k + 1;
  const FusedLayout L = fused_layout(H, I, k);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = gridDim.x, c = blockIdx.x;
  uint8_t *ring = smem + L.ring;
  uint8_t *xperm = smem + L.xperm;
  float *xsum = reinterpret_cast<float *>(smem + L.xsum);
  float *qsum = reinterpret_cast<float *>(smem + L.qsum);
  uint8_t *hperm = smem + L.hperm;
  float *hsum = reinterpret_cast<float *>(smem + L.hsum);
  float *sred = reinterpret_cast<float *>(smem + L.red);
  float *s_part = reinterpret_cast<float *>(smem + L.misc);        // [2 * kCons]
  int *s_sel = reinterpret_cast<int *>(smem + L.misc + 128);       // [kMaxTopK]
  float *s_w = reinterpret_cast<float *>(smem + L.misc + 160);     // [kMaxTopK]
  int *s_flag = reinterpret_cast<int *>(smem + L.misc + 192);      // [4]
  float *s_w24 = reinterpret_cast<float *>(smem + L.misc + 320);   // [kMaxTopK + 1]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.misc + 256);  // [3]
  uint64_t *empty = full + kSlots;                                     // [3]
  uint64_t *route = empty + kSlots;                                    // [1]

  // This block's unit lists.  Shared gate/up units s = c + nb*i (computed
  // while the routing completes); routed gate/up units r = p + nb*i with
  // p = (c - nrt) mod nb, so the round-robin starts after the blocks that own
  // a shared unit and those get the fewer routed ones; down d = (nb-1-c) + nb*i.
  const int n_sh_mine = c < L.nrt ? (L.nrt - 1 - c) / nb + 1 : 0;
  const int n_rt_all = k * L.nrt;
  const int p_rt = ((c - L.nrt) % nb + nb) % nb;
  const int n_rt_mine = p_rt < n_rt_all ? (n_rt_all - 1 - p_rt) / nb + 1 : 0;
  const int n_gu_mine = n_sh_mine + n_rt_mine;
  const int c_dn = nb - 1 - c;
  const int n_dn_mine = c_dn < L.n_dn ? (L.n_dn - 1 - c_dn) / nb + 1 : 0;
  const int n_units = n_gu_mine + n_dn_mine;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(route, 1);
    fence_mbar_init();
    s_flag[2] = 0;  // abort: set by the consumers before releasing `route` on a failure
  }
  __syncthreads();
  if (c == 0 && tid == 0) trace_min(a.trace, kTrEntry);

  // ============================================================ producer warp
  if (warp == kCons) {
    bool routed = false, ok = true;
    int issued = 0;
    for (int it = 0; it < n_units && ok; ++it) {
      const int slot = it % kSlots;
      if (it >= kSlots) ok = mbar_wait_idle(&empty[slot], ((it / kSlots) - 1) & 1, 64, a.wait_ns);
      if (!ok) break;
      uint8_t *dst = ring + slot * L.slot_bytes;
      const bool is_gu = it < n_gu_mine;
      int u, gslot, rt = 0;
      if (it < n_sh_mine) {
        u = c + nb * it;
        gslot = 0;
        rt = u;
      } else if (is_gu) {
        const int r = p_rt + nb * (it - n_sh_mine);
        gslot = 1 + r / L.nrt;
        rt = r - (gslot - 1) * L.nrt;
        u = r;
      } else {
        u = c_dn + nb * (it - n_gu_mine);
        gslot = 0;
      }
      if ((!is_gu || gslot > 0) && !routed) {
        ok = mbar_wait_idle(route, 0, 32, a.wait_ns) && *reinterpret_cast<volatile int *>(&s_flag[2]) == 0;
        routed = true;
        if (!ok) break;
      }
      if (is_gu) {
        const int r0 = rt * kRowsU;
        const uint8_t *blob = gslot == 0 ? a.w.shared : a.w.experts + (size_t)s_sel[gslot - 1] * a.w.stride;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * kRowsU * (H / 2) + 4 * kRowsU * G * 2));
        __syncwarp();
        if (lane < 8) {  // 4-row blocks: lanes 0-3 gate, 4-7 up
          const int m = lane >> 2, q = lane & 3;
          bulk_g2s(dst + lane * L.gu_qp, blob + (m == 0 ? a.w.off.gate_q : a.w.off.up_q) + (size_t)(r0 + 4 * q) * (H / 2),
                   (uint32_t)(2 * H), &full[slot]);
        } else if (lane < 12) {
          const int f = lane - 8;
          const size_t off = f == 0 ? a.w.off.gate_s : f == 1 ? a.w.off.gate_b : f == 2 ? a.w.off.up_s : a.w.off.up_b;
          bulk_g2s(dst + 8 * L.gu_qp + f * kRowsU * G * 2, blob + off + (size_t)r0 * G * 2, (uint32_t)(kRowsU * G * 2),
                   &full[slot]);
        }
      } else {
        const int n0 = u * kRowsU;
        const bool one = L.dn_qp == I / 2;
        const int nq = one ? 1 : kRowsU;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(S * (kRowsU * (I / 2) + 2 * kRowsU * GI * 2)));
        __syncwarp();
        for (int ci = lane; ci < S * (nq + 2); ci += 32) {
          const int s = ci / (nq + 2), j = ci - s * (nq + 2);
          const uint8_t *blob = s == 0 ? a.w.shared : a.w.experts + (size_t)s_sel[s - 1] * a.w.stride;
          uint8_t *sd = dst + s * L.dn_slot_bytes;
          if (j < nq) {
            const int row = one ? 0 : j;
            bulk_g2s(sd + row * L.dn_qp, blob + a.w.off.down_q + (size_t)(n0 + row) * (I / 2),
                     one ? (uint32_t)(kRowsU * (I / 2)) : (uint32_t)(I / 2), &full[slot]);
          } else {
            const int f = j - nq;
            bulk_g2s(sd + kRowsU * L.dn_qp + f * kRowsU * GI * 2,
                     blob + (f == 0 ? a.w.off.down_s : a.w.off.down_b) + (size_t)n0 * GI * 2,
                     (uint32_t)(kRowsU * GI * 2), &full[slot]);
          }
        }
      }
      issued = it + 1;
    }
    // Copies still in flight must land before this block's shared memory is
    // released: wait (bounded) for every issued unit's full barrier phase.
    if (lane == 0) {
      if (!ok) set_error(a.err, kErrTimeout);
      for (int it = issued - kSlots > 0 ? issued - kSlots : 0; it < issued; ++it)
        mbar_wait_idle(&full[it % kSlots], (it / kSlots) & 1, 64, a.wait_ns);
    }
    return;
  }

  // ============================================================ consumers
  // router row of this block (expert e = c; E <= gridDim.x is checked on the
  // host), split like x below: thread t holds the 16 codes of elements
  // 16t .. 16t+15 and the scale and bias of their group
  const int nquart = H / 16;
  const bool has_row = c < E;
  uint4 rq = make_uint4(0u, 0u, 0u, 0u);
  float rs = 0.f, rb = 0.f;
  if (has_row && tid < nquart) {
    rq = __ldg(reinterpret_cast<const uint4 *>(a.w.router_q + (size_t)c * H) + tid);
    rs = bf16_bits_to_float(__ldg(a.w.router_s + (size_t)c * G + (tid >> 2)));
    rb = bf16_bits_to_float(__ldg(a.w.router_b + (size_t)c * G + (tid >> 2)));
  }
  const float lbias = has_row && a.w.logit_bias ? __ldg(a.w.logit_bias + c) : 0.f;
  // the router's learned scales, when given, staged in shared memory before
  // the dependency wait (weights: they do not depend on the previous launch)
  uint16_t *s_rsc = reinterpret_cast<uint16_t *>(smem + L.rsc);
  float *s_pes = reinterpret_cast<float *>(smem + L.pes);
  const bool rscale = kScales && a.w.router_scale != nullptr, escale = kScales && a.w.expert_scale != nullptr;
  if (rscale && tid < nquart) {
    const uint4 *src4 = reinterpret_cast<const uint4 *>(a.w.router_scale) + 2 * tid;
    reinterpret_cast<uint4 *>(s_rsc)[2 * tid] = __ldg(src4);
    reinterpret_cast<uint4 *>(s_rsc)[2 * tid + 1] = __ldg(src4 + 1);
  }
  if (escale && tid < E) s_pes[tid] = __ldg(a.w.expert_scale + tid);
  pdl_wait();
  pdl_launch_dependents();
  if (c == 0 && tid == 0) trace_min(a.trace, kTrWaited);
  // Epoch of this launch.  Every launch adds exactly nb to the counter (one
  // grid barrier); read after the dependency wait it is nb*epoch + (arrivals
  // of fast blocks of this launch, fewer than nb: this block has not
  // arrived), so the epoch follows by division.  It tags this launch's
  // logits in the mailboxes.
  unsigned long long *bar_count = reinterpret_cast<unsigned long long *>(a.sync);
  const unsigned long long epoch = ld_acquire64(bar_count) / (unsigned long long)nb;
  const unsigned long long base = epoch * (unsigned long long)nb;
  const unsigned long long tag = (unsigned long long)(uint32_t)(epoch + 1ull) << 32;

  // Residual values of this block's down rows, needed only at the very end:
  // load them now.  Only this block writes these rows, after it read them.
  uint32_t hres_pre0 = 0, hres_pre1 = 0;
  if (a.hres && warp == kCons - 1 && lane < kRowsU) {  // the warp that runs the down epilogue
    if (n_dn_mine > 0) hres_pre0 = a.hres[c_dn * kRowsU + lane];
    if (n_dn_mine > 1) hres_pre1 = a.hres[(c_dn + nb) * kRowsU + lane];
  }

  // ---- phase 1: x (one 16-element quarter per thread), its sum of squares
  // and the router row's dot product with the raw input, in one pass: a
  // single block reduction gives 1/rms and the dot product, so the logit
  // (dot * 1/rms) goes out before the operand rows are staged.
  uint32_t qin[8];
  float qss = 0.f, lg = 0.f;
  const uint16_t *src = a.hres ? a.hres : a.x;
  if (tid < nquart) {
    const uint4 v0 = __ldcg(reinterpret_cast<const uint4 *>(src) + 2 * tid);
    const uint4 v1 = __ldcg(reinterpret_cast<const uint4 *>(src) + 2 * tid + 1);
    qin[0] = v0.x; qin[1] = v0.y; qin[2] = v0.z; qin[3] = v0.w;
    qin[4] = v1.x; qin[5] = v1.y; qin[6] = v1.z; qin[7] = v1.w;
    const uint32_t rw[4] = {rq.x, rq.y, rq.z, rq.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float lo = __uint_as_float(qin[i] << 16), hi = __uint_as_float(qin[i] & 0xFFFF0000u);
      qss = fmaf(lo, lo, qss);
      qss = fmaf(hi, hi, qss);
      // codes of elements 2i, 2i+1: bytes 2i, 2i+1 of the quarter's 16 code bytes
      const uint32_t w = rw[i >> 1] >> (16 * (i & 1));
      const float qlo = __uint_as_float(0x4B000000u | (w & 0xFFu)) - 8388608.0f;
      const float qhi = __uint_as_float(0x4B000000u | ((w >> 8) & 0xFFu)) - 8388608.0f;
      if (rscale) {  // router input x * router_scale / sqrt(H)
        const uint32_t sc = reinterpret_cast<const uint32_t *>(s_rsc)[8 * tid + i];
        const float inv_sqrt_h = rsqrtf((float)H);
        lg = fmaf(fmaf(qlo, rs, rb), lo * (__uint_as_float(sc << 16) * inv_sqrt_h), lg);
        lg = fmaf(fmaf(qhi, rs, rb), hi * (__uint_as_float(sc & 0xFFFF0000u) * inv_sqrt_h), lg);
      } else {
        lg = fmaf(fmaf(qlo, rs, rb), lo, lg);
        lg = fmaf(fmaf(qhi, rs, rb), hi, lg);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    qss += __shfl_xor_sync(0xffffffffu, qss, off);
    lg += __shfl_xor_sync(0xffffffffu, lg, off);
  }
  if (lane == 0) {
    s_part[warp] = qss;
    s_part[kCons + warp] = lg;
  }
  cons_sync();
  // every thread forms 1/rms and the logit (same partials, same order)
  float inv = 1.0f;
  if (a.normalize) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kCons; ++w) tot += s_part[w];
    inv = 1.0f / sqrtf(tot / (float)H + 1e-6f);
  }
  if (has_row) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kCons; ++w) t += s_part[kCons + w];
    const float logit = t * inv + lbias;
    // this launch's logit of expert c, tagged with the epoch, into every
    // block's mailbox (one 8-byte store each: tag and value arrive together)
    const unsigned long long v = tag | __float_as_uint(logit);
    for (int b = tid; b < nb; b += kConsThreads)
      asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a.mbox + (size_t)b * kMaxExperts + c), "l"(v)
                   : "memory");
    if (tid == 0) a.logits[c] = logit;
  }
  // operand rows: normalised bf16 x -> permuted fp16, quarter and group sums
  if (tid < nquart) {
    if (a.normalize) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint16_t lb = float_to_bf16_bits(__uint_as_float(qin[i] << 16) * inv);
        const uint16_t hb = float_to_bf16_bits(__uint_as_float(qin[i] & 0xFFFF0000u) * inv);
        qin[i] = (uint32_t)lb | ((uint32_t)hb << 16);
      }
    }
    if (c == 0 && a.xn_user) {
      uint4 *xu = reinterpret_cast<uint4 *>(a.xn_user) + 2 * tid;
      xu[0] = make_uint4(qin[0], qin[1], qin[2], qin[3]);
      xu[1] = make_uint4(qin[4], qin[5], qin[6], qin[7]);
    }
    uint32_t out[8];
    operand_quarter<true>(qin, out);  // bf16 x -> fp16 B operand
    uint2 *dst = reinterpret_cast<uint2 *>(xperm + tid * 32);
#pragma unroll
    for (int w = 0; w < 4; ++w) dst[w] = make_uint2(out[2 * w], out[2 * w + 1]);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s += __uint_as_float(qin[i] << 16);
      s += __uint_as_float(qin[i] & 0xFFFF0000u);
    }
    qsum[tid] = s;
  }
  cons_sync();
  if (tid < G) xsum[tid] = ((qsum[4 * tid] + qsum[4 * tid + 1]) + qsum[4 * tid + 2]) + qsum[4 * tid + 3];
  cons_sync();

  // ---- phase 2: compute this block's shared gate/up units (their tiles and
  // x are here) while barrier 1 completes
  const int r = lane >> 2, cq = lane & 3;
  int it = 0;
  bool ok = true;
  // one gate/up unit: 16 rows of gate and up of one slot, GeGLU, h to global
  auto gu_unit = [&](int it) -> bool {
    const int slot = it % kSlots;
    int gslot, rt;
    if (it < n_sh_mine) {
      gslot = 0;
      rt = c + nb * it;
    } else {
      const int r = p_rt + nb * (it - n_sh_mine);
      gslot = 1 + r / L.nrt;
      rt = r - (gslot - 1) * L.nrt;
    }
    if (!mbar_wait(&full[slot], (it / kSlots) & 1, a.wait_ns)) return false;
    const uint8_t *tile = ring + slot * L.slot_bytes;
    // groups warp, warp + kCons, ...; two groups in flight per iteration
    float tg0a = 0.f, tg2a = 0.f, tu0a = 0.f, tu2a = 0.f, tg0b = 0.f, tg2b = 0.f, tu0b = 0.f, tu2b = 0.f;
    int g = warp;
    for (; g + kCons < G; g += 2 * kCons) {
      gu_group(tile, xperm, xsum, g, r, cq, G, L.gu_qp, tg0a, tg2a, tu0a, tu2a);
      gu_group(tile, xperm, xsum, g + kCons, r, cq, G, L.gu_qp, tg0b, tg2b, tu0b, tu2b);
    }
    if (g < G) gu_group(tile, xperm, xsum, g, r, cq, G, L.gu_qp, tg0a, tg2a, tu0a, tu2a);
    if (cq == 0) {
      float *red = sred + (it & 1) * (kCons * 64) + warp * 64;
      red[r] = tg0a + tg0b;
      red[r + 8] = tg2a + tg2b;
      red[16 + r] = tu0a + tu0b;
      red[16 + r + 8] = tu2a + tu2b;
    }
    cons_sync();
    if (tid == 0) mbar_arrive_expect_tx(&empty[slot], 0);  // every warp is done with the tile
    // epilogue in the last warp (the fewest groups), from this unit's half
    // of sred: the next unit writes the other half, the one after waits for
    // this warp at its own cons_sync
    if (warp == kCons - 1 && lane < kRowsU) {
      const float *rd = sred + (it & 1) * (kCons * 64);
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < kCons; ++w) {
        gs += rd[w * 64 + lane];
        us += rd[w * 64 + 16 + lane];
      }
      const float hv = gelu_tanh(gs) * us;
      if (!(fabsf(hv) <= 65504.0f)) set_error(a.err, kErrNonFinite);
      a.hbuf[(size_t)gslot * I + rt * kRowsU + quad_row(lane)] = __float2half_rn(hv);  // lane: mma row
    }
    return true;
  };

  for (; it < n_sh_mine && ok; ++it) ok = gu_unit(it);
  // ---- top-k, in warp 0 of every block, once this block's mailbox holds
  // every logit of this launch (lane l polls experts 4l .. 4l+3); lane l
  // holds the keys of experts 4l .. 4l+3 sorted (larger first, equal keys
  // lower id first); each round
  // takes the warp maximum of the lanes' heads, the lowest lane holding it
  // (= the lowest id among equal keys) pops its head.  The softmax terms
  // accumulate as the values come out, in selection order.
  unsigned long long mv[4] = {0ull, 0ull, 0ull, 0ull};  // warp 0: the polled logits
  if (warp == 0) {
    bool got = ok;
    if (got) {
      const unsigned long long *mb = a.mbox + (size_t)c * kMaxExperts + 4 * lane;
      const unsigned long long t0 = global_ns();
      for (uint32_t pi = 0;; ++pi) {
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(mv[0]), "=l"(mv[1]) : "l"(mb) : "memory");
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(mv[2]), "=l"(mv[3]) : "l"(mb + 2) : "memory");
        bool mine = true;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (4 * lane + i < E && (mv[i] & 0xFFFFFFFF00000000ull) != tag) mine = false;
        if (__all_sync(0xffffffffu, mine)) break;
        if ((pi & 7u) == 7u && __any_sync(0xffffffffu, global_ns() - t0 > a.wait_ns)) {
          got = false;
          break;
        }
      }
    }
    if (lane == 0) s_flag[0] = got ? 1 : 0;
  }
  cons_sync();
  if (s_flag[0] == 0) {
    if (tid == 0) {
      set_error(a.err, kErrTimeout);
      s_flag[2] = 1;                     // no routing: the producer must not stream routed tiles
      mbar_arrive_expect_tx(route, 0);   // release it; it drains its copies and exits
      // still count this block's arrival: every launch moves the counter by
      // exactly nb
      asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar_count) : "memory");
    }
    return;
  }
  if (warp == 0) {
    unsigned k0, k1, k2, k3;
    bool bad = false;
    {
      unsigned kq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = 4 * lane + i;
        kq[i] = 0u;  // below every real key: never picked while k <= E
        if (e < E) {
          float x = __uint_as_float((uint32_t)mv[i]);
          if (!isfinite(x)) {
            x = -INFINITY;
            bad = true;
          }
          kq[i] = ord_key(x);
        }
      }
      k0 = kq[0]; k1 = kq[1]; k2 = kq[2]; k3 = kq[3];
    }
    if (c == 0 && bad) set_error(a.err, kErrNonFinite);
    int i0 = 0, i1 = 1, i2 = 2, i3 = 3;
    // (key descending, index ascending): ordered pairs need no swap
    auto cswap = [](unsigned &ka, int &ia, unsigned &kb, int &ib) {
      if (kb > ka || (kb == ka && ib < ia)) {
        const unsigned tk = ka; ka = kb; kb = tk;
        const int ti = ia; ia = ib; ib = ti;
      }
    };
    cswap(k0, i0, k1, i1);
    cswap(k2, i2, k3, i3);
    cswap(k0, i0, k2, i2);
    cswap(k1, i1, k3, i3);
    cswap(k1, i1, k2, i2);
    // all kMaxTopK rounds run (k <= E; rounds past k pick unused entries);
    // the winner of a round is the lowest lane whose head equals the maximum
    unsigned mk[kMaxTopK];
    unsigned lt_mask;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt_mask));
    // local indices packed one per byte, popped with a shift; the pop is
    // branch-free (selects), only the winner's store is predicated
    unsigned idx = (unsigned)i0 | ((unsigned)i1 << 8) | ((unsigned)i2 << 16) | ((unsigned)i3 << 24);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      const unsigned m = __reduce_max_sync(0xffffffffu, k0);
      const bool eq = k0 == m;
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      const bool win = eq && (bal & lt_mask) == 0u;
      mk[j] = m;
      if (win) s_sel[j] = 4 * lane + (int)(idx & 0xFFu);
      k0 = win ? k1 : k0;
      k1 = win ? k2 : k1;
      k2 = win ? k3 : k2;
      k3 = win ? 0u : k3;
      idx = win ? idx >> 8 : idx;
    }
    // softmax over the k selected values, in selection order
    const float v0 = key_value(mk[0]);
    float den = 0.f, myex = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const float ex = __expf(key_value(mk[j]) - v0);
        den += ex;
        if (lane == j) myex = ex;
      }
    }
    __syncwarp();
    if (lane < k) {
      const float wj = myex / den * (escale ? s_pes[s_sel[lane]] : 1.0f);
      s_w[lane] = wj;
      if (c == 0) {
        if (a.ids_user) a.ids_user[lane] = s_sel[lane];
        if (a.wts_user) a.wts_user[lane] = wj;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(route, 0);  // routing known: producer may stream
  }
  cons_sync();
  if (c == 0 && tid == 0) trace_max(a.trace, kTrLoaded);

  // ---- phase 3: routed gate/up units
  for (; it < n_gu_mine && ok; ++it) ok = gu_unit(it);
  if (!ok) set_error(a.err, kErrTimeout);

  // ---- phase 4: grid barrier (all of h written), then the down units
  if (!grid_sync(bar_count, base + nb, a.err, &s_flag[1], a.wait_ns, c != a.skip_block) || !ok) return;
  // stage every expert's h row (permuted fp16) one 16-wide quarter per
  // thread (all loads in one round), then the group sums in quarter order
  {
    const int nq = S * (I / 16);
    float *hq = sred;  // quarter sums (sred is free until the first down unit)
    for (int q = tid; q < nq; q += kConsThreads) {
      const uint4 *srch = reinterpret_cast<const uint4 *>(a.hbuf) + 2 * q;
      const uint4 v0 = __ldcg(srch), v1 = __ldcg(srch + 1);
      const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t out[8];
      operand_quarter<false>(in, out);  // fp16 h -> B operand
      uint2 *dst = reinterpret_cast<uint2 *>(hperm + q * 32);
#pragma unroll
      for (int w = 0; w < 4; ++w) dst[w] = make_uint2(out[2 * w], out[2 * w + 1]);
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        sum += __half2float(__ushort_as_half((unsigned short)(in[w] & 0xFFFFu)));
        sum += __half2float(__ushort_as_half((unsigned short)(in[w] >> 16)));
      }
      hq[q] = sum;
    }
    cons_sync();
    // per item: router weight of its expert times the group sum of h; per
    // expert: the weight times 2^24 (the code scale the mma leaves in)
    for (int q = tid; q < S * GI; q += kConsThreads) {
      const int sl = q / GI;
      const float wt = sl == 0 ? 1.0f : s_w[sl - 1];
      hsum[q] = wt * (((hq[4 * q] + hq[4 * q + 1]) + hq[4 * q + 2]) + hq[4 * q + 3]);
    }
    if (tid < S) s_w24[tid] = (tid == 0 ? 1.0f : s_w[tid - 1]) * kCodeScale;
  }
  cons_sync();
  for (int jd = 0; jd < n_dn_mine; ++jd, ++it) {
    const int slot = it % kSlots;
    const int n0 = (c_dn + nb * jd) * kRowsU;
    if (!mbar_wait(&full[slot], (it / kSlots) & 1, a.wait_ns)) {
      set_error(a.err, kErrTimeout);
      return;
    }
    const uint8_t *tile = ring + slot * L.slot_bytes;
    const int nitems = S * GI;
    const int per = (nitems + kCons - 1) / kCons;
    const int ib = warp * per, ie = min(nitems, ib + per);
    // two independent accumulation chains per warp (items q and q+1); the
    // item pointers advance by one group, or to the next expert's slice of
    // the tile, without divisions
    float t0a = 0.f, t2a = 0.f, t0b = 0.f, t2b = 0.f;
    if (ib < ie) {
      int sl = ib / GI, g = ib - (ib / GI) * GI;
      const uint8_t *tq = tile + sl * L.dn_slot_bytes + g * 32 + cq * 8;
      const uint16_t *sq = reinterpret_cast<const uint16_t *>(tile + sl * L.dn_slot_bytes + kRowsU * L.dn_qp) + g;
      const int qp_r0 = r * L.dn_qp, qp_r1 = (r + 8) * L.dn_qp;
      auto adv = [&]() {
        ++g;
        tq += 32;
        ++sq;
        if (g == GI) {
          g = 0;
          ++sl;
          tq += L.dn_slot_bytes - GI * 32;
          sq = reinterpret_cast<const uint16_t *>(reinterpret_cast<const uint8_t *>(sq) + L.dn_slot_bytes) - GI;
        }
      };
      int q = ib;
      for (; q + 1 < ie; q += 2) {
        down_item(tq, sq, hperm + q * 128 + cq * 32, hsum[q], s_w24[sl], r, qp_r0, qp_r1, GI, t0a, t2a);
        adv();
        down_item(tq, sq, hperm + (q + 1) * 128 + cq * 32, hsum[q + 1], s_w24[sl], r, qp_r0, qp_r1, GI, t0b, t2b);
        adv();
      }
      if (q < ie) down_item(tq, sq, hperm + q * 128 + cq * 32, hsum[q], s_w24[sl], r, qp_r0, qp_r1, GI, t0a, t2a);
    }
    float *red = sred + (jd & 1) * (kCons * kRowsU);
    if (cq == 0) {
      red[warp * kRowsU + r] = t0a + t0b;
      red[warp * kRowsU + r + 8] = t2a + t2b;
    }
    cons_sync();
    if (tid == 0) mbar_arrive_expect_tx(&empty[slot], 0);  // every warp is done with the tile
    // epilogue in the last warp (the fewest items), from this unit's half of sred
    if (warp == kCons - 1 && lane < kRowsU) {
      float y = 0.f;
#pragma unroll
      for (int w = 0; w < kCons; ++w) y += red[w * kRowsU + lane];
      const uint16_t yb = float_to_bf16_bits(y);
      if (a.y) a.y[n0 + lane] = yb;
      if (a.hres) {
        const uint32_t hb = jd == 0 ? hres_pre0 : jd == 1 ? hres_pre1 : a.hres[n0 + lane];
        a.hres[n0 + lane] = float_to_bf16_bits(bf16_bits_to_float(hb) + bf16_bits_to_float(yb));
      }
    }
  }
  if (tid == 0) trace_max(a.trace, kTrExit);
}

cudaError_t launch_decode_fused(const DecodeArgs &a, int n_blocks, cudaStream_t st, bool pdl) {
  const bool scales = a.w.router_scale != nullptr || a.w.expert_scale != nullptr;
  return launch_k(scales ? decode_layer_kernel<true> : decode_layer_kernel<false>, dim3(n_blocks), dim3(kThreadsF),
                  fused_decode_smem(a.d), st, pdl, a);
}

cudaError_t decode_set_attributes() {
  const cudaError_t e =
      cudaFuncSetAttribute(decode_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

int decode_blocks_per_sm(const Dims &d) {
  int n = 0, n2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_layer_kernel<false>, kThreadsF, fused_decode_smem(d)) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n2, decode_layer_kernel<true>, kThreadsF, fused_decode_smem(d)) !=
          cudaSuccess)
    return 0;
  return n < n2 ? n : n2;
}

}  // namespace moe
