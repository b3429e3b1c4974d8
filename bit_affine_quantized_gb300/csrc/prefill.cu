// Fused multi-token MoE layer (prefill chunks and batched decode, 2 <= T <= 128), sm_103a.
//
// Page "TurboFieldfare - System design", section "Prefill": a chunk of at
// most 128 rows goes through the layer at once; the router scores every row,
// token/expert pairs are grouped per expert, the routed experts run on their
// groups and the shared branch on every row, and the branches are combined.
//
// One persistent block per SM; 16 consumer warps and 1 producer warp.  The
// producer streams weight tiles through a 3-slot ring (W) and operand rows
// into one buffer (X) that stays put while consecutive units share a chunk.
// In the unit phases the consumers work as two groups of 8 warps, each on
// every other unit with a named barrier of its own, so one group's
// reduction and epilogue overlap the other group's tensor-core loop.
//   R  tokens t = block, block + grid, ...: x = input (or rmsnorm of the
//      residual); permuted fp16 operand rows and quarter sums go to the
//      workspace for the experts; the block scores its own token against
//      the router streamed through W in 16-expert tiles (tensor cores, 8-bit
//      codes as exact fp16 subnormals), then selects the top-k;
//   == barrier 1 ==  every block groups all pairs in shared memory (stable
//      counting sort) and derives the unit lists;
//   G  gate/up units (slot, 8-token chunk, 16 rows of I), a contiguous
//      range per block: GeGLU, h written as permuted fp16 quarters + sums;
//   == barrier 2 ==
//   D  down units (slot, chunk, 128 rows of H): weighted outputs w * o in
//      fp32 per sorted position; their weight tiles stream during barrier 2;
//   == barrier 3 ==
//   C  combine of tokens t = block, ...: y = sum_j o[pos(t, j)] + o[shared t]
//      in selection order, bf16 out, optional residual add.
// Expert math: 4-bit codes as exact fp16 subnormals (code * 2^-24; odd
// nibbles come out * 16 and meet activations stored / 16), per-group
// correction (scale * 2^24) * acc + bias * sum(x).
#include <math.h>
#include <string.h>

#include "dense.cuh"
#include "fused.cuh"
#include "kernels.h"

namespace moe {

namespace {
using fused::cons_sync;
using fused::kCons;
using fused::kConsThreads;
constexpr int kWSlots = 3;   // weight ring
constexpr int kTC = 8;       // tokens per unit (one mma N tile)
constexpr int kGuRows = 16;  // gate/up rows per unit (each of gate and up)
constexpr int kDnRows = 128; // down rows per unit (8 x m16)
constexpr int kRtRows = 16;  // router experts per tile
constexpr int kNBar = 3;     // grid barriers per launch
constexpr int kRedBytes = kCons * 256 * 4;

// misc: s_flag int[16] | s_hst fp16[8][16] (group 0) | s_logit float[128] | s_part float[16] |
// mbarriers [10] | s_wt float[8] (group 0) | s_hst (group 1) | s_wt (group 1) | dense-path mbarriers [14] |
// tensor-memory address
constexpr int kMiscHst = 64, kMiscLogit = 320, kMiscPart = 832, kMiscBar = 896, kMiscWt = 976, kMiscHst1 = 1024,
              kMiscWt1 = 1280, kMiscDBar = 1320, kMiscTmem = 1432, kMiscBytes = 1536;
constexpr int kMiscLand = 1008;  // int [kWSlots]: last ring use seen landed per slot
constexpr int kMmaWarp = kCons + 1;             // issues the tcgen05.mma of dense blocks
constexpr int kThreadsP = fused::kThreads + 32;  // consumers + producer + MMA warp
constexpr int kMaxDense = 64;  // dense slots of a chunk (at most T*k / dense::kMinRows + 1)
static_assert(kMaxTokens * kMaxTopK / dense::kMinRows + 1 <= kMaxDense, "every dense slot has a list entry");

__host__ __device__ inline int pw8(int w) { return w + ((8 - (w % 16)) + 16) % 16; }
__host__ __device__ inline int al16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }
// Quarter-sum row pitch (floats): the lanes of a fragment read rows 0, 2, 4
// and 6 as float4s; a pitch of 4 mod 16 puts them in disjoint banks.
__host__ __device__ inline int qsum_pitch(int n) { return n + ((4 - n % 16) + 16) % 16; }

struct PL {
  int G, GI, nrt, nrt_dn, n_mt;
  int gu_qp, rt_qp, dn_qp, wslot;   // W slot: gate/up 4-row block pitch, code row pitches, slot bytes
  int xp, gp, x_xs;                 // X as gate/up operand: row pitch (B); group sums as bf16 hi/lo
                                    // [2][gp] per token (gp = G rounded up to 16, zero padded), offset
  int hp, hqp, x_hq;                // X as down operand
  int rx_q, rx_sb;                  // X as router operand: quarter sums after the fp16 row, then the
                                    // router's scales and biases (bf16 [16 n_mt][G] each)
  int rx_xq;                        // quarter sums of x itself when the router operand is scaled x
  int xbuf;
  int ring, xb, red, grp, misc, total;
};

// Pitches: gate/up and router tiles arrive as 4-row blocks (quad_row in
// common.cuh) whose pitch puts the four blocks in disjoint banks for the
// fragment loads (8 mod 32 words for the 8-byte gate/up loads, 64 mod 128
// bytes for the 16-byte router loads); down codes keep a row pitch of 8 mod
// 16 words; operand rows 4 mod 8 words; quarter sums: see qsum_pitch.
__host__ __device__ inline PL prefill_layout(int H, int I, int E, int k, int T, bool dense = false) {
  PL L;
  L.G = H / kGroup;
  L.GI = I / kGroup;
  L.nrt = I / kGuRows;
  L.nrt_dn = (H + kDnRows - 1) / kDnRows;
  L.n_mt = (E + kRtRows - 1) / kRtRows;
  L.gu_qp = quad_pitch(H);
  L.rt_qp = 4 * H + ((64 - (4 * H) % 128) + 128) % 128;  // 4-row block pitch
  L.dn_qp = pw8(I / 8) * 4;
  const int gu = quad_tile_bytes(H);
  const int rt = 4 * L.rt_qp;
  const int dn = kDnRows * L.dn_qp + 2 * kDnRows * L.GI * 2;
  L.wslot = al16(imax(gu, imax(rt, dn)));
  L.xp = 2 * H + 16;
  L.gp = (L.G + 15) & ~15;
  L.x_xs = kTC * L.xp;
  L.hp = 2 * I + 16;
  L.hqp = qsum_pitch(I / 16);
  L.x_hq = kTC * L.hp;
  L.rx_q = 2 * H;
  L.rx_sb = al16(L.rx_q + (H / 16) * 4);
  L.rx_xq = al16(L.rx_sb + 2 * kRtRows * L.n_mt * L.G * 2);
  L.xbuf = al16(imax(L.x_xs + kTC * 4 * L.gp, imax(L.x_hq + kTC * L.hqp * 4, L.rx_xq + (H / 16) * 4)));
  int o = 0;
  L.ring = o;
  o += kWSlots * L.wslot;
  L.xb = o;
  o += L.xbuf;
  L.red = o;  // cross-warp reductions, grouping temporaries
  o += imax(kRedBytes, (1 + kCons) * E * 4);
  // the dense instance reuses ring, X and red (from L.ring, aligned up to 1 KB) for its own plan
  if (dense) o = imax(o, L.ring + dense::plan(L.G).total + 1024);
  L.grp = o;  // chunk0 int32 [E+2], perm/pos int16 [T*k], act_e/beg/cnt int16 [E+1], dense slots int16
              // [kMaxDense], token -> position int16 [kMaxTokens], position weights float [kMaxTokens]
  o = al16(o + (E + 2) * 4 + 2 * T * k * 2 + 3 * (E + 1) * 2 + kMaxDense * 2 + kMaxTokens * 2);
  o = al16(o + kMaxTokens * 4);
  L.misc = o;
  o = al16(o + kMiscBytes);
  L.total = o;
  return L;
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

// Two 8-bit codes as exact fp16 subnormals: bytes 0 and 2, or 1 and 3.
__device__ __forceinline__ uint32_t bytes02(uint32_t w) { return __byte_perm(w, 0u, 0x4240); }
__device__ __forceinline__ uint32_t bytes13(uint32_t w) { return __byte_perm(w, 0u, 0x4341); }

// Router: one 64-wide group of a 16-expert tile against one token (column 0,
// supplied by the lanes with r == 0).  rx holds, per quarter, the pairs
// (x0,x2)(x1,x3)(x4,x6)... so that k-step s meets code word s of the lane.
// rs/rb: the tile's scales and biases ([row][G] bf16).
__device__ __forceinline__ void rt_group(const uint8_t *tile, const uint8_t *rx, const float *rq, const uint16_t *rs,
                                         const uint16_t *rb, int qp, int G, int g, int r, int cq, float &t0,
                                         float &t1) {
  // mma rows r, r + 8 hold tile rows quad_row(r), quad_row(r) + 2 (4-row blocks at pitch qp)
  const int rowb = G * 64, sr0 = quad_row(r), sr1 = sr0 + 2;
  const uint8_t *wa = tile + (r & 3) * qp + (r >> 2) * rowb + g * 64 + cq * 16;
  const uint4 w0 = *reinterpret_cast<const uint4 *>(wa);
  const uint4 w1 = *reinterpret_cast<const uint4 *>(wa + 2 * rowb);
  uint4 b0 = make_uint4(0u, 0u, 0u, 0u), b1 = b0;
  if (r == 0) {
    b0 = *reinterpret_cast<const uint4 *>(rx + g * 128 + cq * 32);
    b1 = *reinterpret_cast<const uint4 *>(rx + g * 128 + cq * 32 + 16);
  }
  const uint32_t a0[4] = {w0.x, w0.y, w0.z, w0.w}, a1[4] = {w1.x, w1.y, w1.z, w1.w};
  const uint32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t A[4] = {bytes02(a0[s]), bytes02(a1[s]), bytes13(a0[s]), bytes13(a1[s])};
    mma_f16(acc, A, bb[2 * s], bb[2 * s + 1]);
  }
  const float4 q = *reinterpret_cast<const float4 *>(rq + 4 * g);
  const float xs = ((q.x + q.y) + q.z) + q.w;
  t0 = fmaf(bf16_bits_to_float(rb[sr0 * G + g]), xs, fmaf(bf16_bits_to_float(rs[sr0 * G + g]) * kCodeScale, acc[0], t0));
  t1 = fmaf(bf16_bits_to_float(rb[sr1 * G + g]), xs,
            fmaf(bf16_bits_to_float(rs[sr1 * G + g]) * kCodeScale, acc[2], t1));
}

// One 64-wide group of a gate/up unit for the chunk's 8 tokens: mma rows r,
// r+8 (tile rows quad_row(r), quad_row(r) + 2), token columns 2cq, 2cq+1.
// Accumulates s*acc per row and token, which carries the 2^-24 of the code
// operands (the epilogue multiplies by 2^24 once); the bias terms
// b*sum(x)*2^-24 of all groups come from gu_bias once per unit.
__device__ __forceinline__ void gu_group(const uint8_t *tile, const uint8_t *xrows, int qp, int xp, int G, int g,
                                         int r, int cq, float (&tg)[4], float (&tu)[4]) {
  const int rowb = G * 32;                    // bytes of one row of codes (H / 2)
  const int sr0 = quad_row(r), sr1 = sr0 + 2;  // tile rows of mma rows r and r + 8
  const uint16_t *raw = reinterpret_cast<const uint16_t *>(tile + 8 * qp);  // gs, gb, us, ub [16][G]
  const uint8_t *ga = tile + (r & 3) * qp + (r >> 2) * rowb + g * 32 + cq * 8;
  const uint2 g0 = *reinterpret_cast<const uint2 *>(ga);
  const uint2 g1 = *reinterpret_cast<const uint2 *>(ga + 2 * rowb);
  const uint2 u0 = *reinterpret_cast<const uint2 *>(ga + 4 * qp);
  const uint2 u1 = *reinterpret_cast<const uint2 *>(ga + 4 * qp + 2 * rowb);
  const uint4 bA = *reinterpret_cast<const uint4 *>(xrows + r * xp + g * 128 + cq * 32);
  const uint4 bB = *reinterpret_cast<const uint4 *>(xrows + r * xp + g * 128 + cq * 32 + 16);
  const uint32_t bb[8] = {bA.x, bA.y, bA.z, bA.w, bB.x, bB.y, bB.z, bB.w};
  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
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
    mma_f16(ag, A, bb[2 * s], bb[2 * s + 1]);
    mma_f16(au, B, bb[2 * s], bb[2 * s + 1]);
  }
  const float sg0 = bf16_bits_to_float(raw[sr0 * G + g]), sg1 = bf16_bits_to_float(raw[sr1 * G + g]);
  const float su0 = bf16_bits_to_float(raw[32 * G + sr0 * G + g]), su1 = bf16_bits_to_float(raw[32 * G + sr1 * G + g]);
  tg[0] = fmaf(sg0, ag[0], tg[0]);
  tg[1] = fmaf(sg0, ag[1], tg[1]);
  tg[2] = fmaf(sg1, ag[2], tg[2]);
  tg[3] = fmaf(sg1, ag[3], tg[3]);
  tu[0] = fmaf(su0, au[0], tu[0]);
  tu[1] = fmaf(su0, au[1], tu[1]);
  tu[2] = fmaf(su1, au[2], tu[2]);
  tu[3] = fmaf(su1, au[3], tu[3]);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The bias terms of one matrix of a gate/up unit over all G groups, in the
// fragment layout of gu_group's accumulators: t[row][token] +=
// sum_g b[row][g] * sum(x[token], group g), as a bf16 tensor-core product of
// the tile's biases (A: rows, groups) with the chunk's group sums split in
// bf16 hi + lo parts (B: groups, tokens).  boff: offset of the bias rows in
// the tile's scale/bias area (16*G gate, 48*G up); xs: [kTC][2][gp].
__device__ __forceinline__ void gu_bias(const uint8_t *tile, const uint16_t *xs, int qp, int G, int gp, int boff,
                                        int r, int cq, float (&t)[4]) {
  const uint16_t *b = reinterpret_cast<const uint16_t *>(tile + 8 * qp) + boff;
  const int sr0 = quad_row(r), sr1 = sr0 + 2;
  auto pairv = [&](int row, int g) -> uint32_t {  // biases g, g+1 of a row (zero past G)
    const uint32_t lo = g < G ? b[row * G + g] : 0u, hi = g + 1 < G ? b[row * G + g + 1] : 0u;
    return lo | (hi << 16);
  };
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < gp; k0 += 16) {
    const int g0 = k0 + 2 * cq;
    const uint32_t A[4] = {pairv(sr0, g0), pairv(sr1, g0), pairv(sr0, g0 + 8), pairv(sr1, g0 + 8)};
    const uint32_t *xr = reinterpret_cast<const uint32_t *>(xs + r * 2 * gp);  // token r: hi then lo
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t *xp = xr + (part * gp + g0) / 2;
      mma_bf16(acc, A, xp[0], xp[4]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] += acc[i];
}

// Down: one 64-wide group; rows row0 + r, +8 of the 128-row tile, token
// columns 2cq, 2cq+1.
__device__ __forceinline__ void dn_group(const uint8_t *tile, const uint8_t *hrows, int qp, int hp, int GI, int row0,
                                         int g, int r, int cq, float (&t)[4]) {
  const uint16_t *sb = reinterpret_cast<const uint16_t *>(tile + kDnRows * qp);  // scales [128][GI], biases [128][GI]
  const uint2 w0 = *reinterpret_cast<const uint2 *>(tile + (row0 + r) * qp + g * 32 + cq * 8);
  const uint2 w1 = *reinterpret_cast<const uint2 *>(tile + (row0 + r + 8) * qp + g * 32 + cq * 8);
  const uint4 bA = *reinterpret_cast<const uint4 *>(hrows + r * hp + g * 128 + cq * 32);
  const uint4 bB = *reinterpret_cast<const uint4 *>(hrows + r * hp + g * 128 + cq * 32 + 16);
  const uint32_t bb[8] = {bA.x, bA.y, bA.z, bA.w, bB.x, bB.y, bB.z, bB.w};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const uint32_t x0 = (st >> 1) ? w0.y : w0.x, x1 = (st >> 1) ? w1.y : w1.x;
    uint32_t A[4];
    if ((st & 1) == 0) {
      A[0] = codes_sub<0>(x0); A[1] = codes_sub<0>(x1); A[2] = codes_sub<1>(x0); A[3] = codes_sub<1>(x1);
    } else {
      A[0] = codes_sub<2>(x0); A[1] = codes_sub<2>(x1); A[2] = codes_sub<3>(x0); A[3] = codes_sub<3>(x1);
    }
    mma_f16(acc, A, bb[2 * st], bb[2 * st + 1]);
  }
  const float s0 = bf16_bits_to_float(sb[(row0 + r) * GI + g]);
  const float s1 = bf16_bits_to_float(sb[(row0 + r + 8) * GI + g]);
  t[0] = fmaf(s0, acc[0], t[0]);
  t[1] = fmaf(s0, acc[1], t[1]);
  t[2] = fmaf(s1, acc[2], t[2]);
  t[3] = fmaf(s1, acc[3], t[3]);
}

// The bias terms of a warp's 16 rows of a down unit over all GI groups:
// t[row][token] += sum_g b[row][g] * sum(h[token], group g), a bf16
// tensor-core product of the tile's biases with the chunk's group sums of h
// (hi + lo parts, hs: [kTC][2][gip]).
__device__ __forceinline__ void dn_bias(const uint8_t *tile, const uint16_t *hs, int qp, int GI, int gip, int row0,
                                        int r, int cq, float (&t)[4]) {
  const uint16_t *b = reinterpret_cast<const uint16_t *>(tile + kDnRows * qp) + kDnRows * GI;
  auto pairv = [&](int row, int g) -> uint32_t {
    const uint32_t lo = g < GI ? b[row * GI + g] : 0u, hi = g + 1 < GI ? b[row * GI + g + 1] : 0u;
    return lo | (hi << 16);
  };
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < gip; k0 += 16) {
    const int g0 = k0 + 2 * cq;
    const uint32_t A[4] = {pairv(row0 + r, g0), pairv(row0 + r + 8, g0), pairv(row0 + r, g0 + 8),
                           pairv(row0 + r + 8, g0 + 8)};
    const uint32_t *hr = reinterpret_cast<const uint32_t *>(hs + r * 2 * gip);  // token r: hi then lo
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t *hp2 = hr + (part * gip + g0) / 2;
      mma_bf16(acc, A, hp2[0], hp2[4]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] += acc[i];
}

// Decoded work unit: active slot, chunk within it, tile within the chunk.
struct Unit {
  int sa, ch, tile, e, beg, nt;
};
__device__ __forceinline__ Unit decode_unit(int u, int per, const int *chunk0, int nact, const int16_t *act_e,
                                            const int16_t *act_beg, const int16_t *act_cnt) {
  Unit x;
  const int chg = u / per;
  x.tile = u - chg * per;
  x.sa = find_slot(chunk0, nact + 1, chg);
  x.ch = chg - chunk0[x.sa];
  x.e = act_e[x.sa];
  x.beg = act_beg[x.sa];
  x.nt = min(kTC, (int)act_cnt[x.sa] - kTC * x.ch);
  return x;
}
}  // namespace

size_t prefill_dense_smem(const Dims &d) {
  const PL L = prefill_layout(d.H, d.I, d.E, d.k, d.T, true);
  return L.total <= 227 * 1024 ? (size_t)L.total : 0;
}

size_t prefill_fused_smem(const Dims &d) {
  const PL L = prefill_layout(d.H, d.I, d.E, d.k, d.T);
  return L.total <= 227 * 1024 ? (size_t)L.total : 0;
}

namespace {
// Kernel parameters: the arguments and the shared-memory layout (computed on
// the host, so its fields are read from the parameter bank, not registers).
struct PrefillParams {
  dense::Maps dm;  // tensor maps of the dense path (64-byte aligned: first)
  PrefillArgs a;
  PL L;
  int dense_on;    // slots with at least dense::kMinRows rows take the tcgen05 path
};
}  // namespace

// kScales: the layer has learned router scales (the router-scale code is
// compiled out of the plain instance).
// kDense: the instance with the tcgen05 path for dense slots (one more warp,
// the MMA warp); the plain instance compiles the light path alone.
template <bool kScales, bool kDense>
__global__ void __launch_bounds__(kDense ? kThreadsP : fused::kThreads, 1)
    prefill_layer_kernel(const __grid_constant__ PrefillParams prm) {
  extern __shared__ __align__(128) uint8_t smem[];
  const PrefillArgs &a = prm.a;
  const PL &L = prm.L;
  const int H = a.d.H, I = a.d.I, E = a.d.E, k = a.d.k, T = a.d.T;
  const int G = L.G, GI = L.GI;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = gridDim.x, c = blockIdx.x;
  const int npairs = T * k;
  uint8_t *ring = smem + L.ring;
  uint8_t *xbuf = smem + L.xb;
  float *red = reinterpret_cast<float *>(smem + L.red);
  int *chunk0 = reinterpret_cast<int *>(smem + L.grp);                  // [E+2]
  int16_t *g_perm = reinterpret_cast<int16_t *>(chunk0 + E + 2);        // [T*k]
  int16_t *g_pos = g_perm + npairs;                                     // [T*k]
  int16_t *g_act_e = g_pos + npairs;                                    // [E+1]
  int16_t *g_act_beg = g_act_e + (E + 1);                               // [E+1]
  int16_t *g_act_cnt = g_act_beg + (E + 1);                             // [E+1]
  int16_t *g_dense = g_act_cnt + (E + 1);                               // [kMaxDense] dense active slots
  int16_t *g_tpos = g_dense + kMaxDense;                                // [kMaxTokens] token -> position (dense unit)
  float *g_wpos = reinterpret_cast<float *>(smem + L.grp + ((((E + 2) * 4 + 2 * npairs * 2 + 3 * (E + 1) * 2 +
                                                               kMaxDense * 2 + kMaxTokens * 2) + 15) & ~15));
  // the dense path: its plan on a 1 KB boundary inside ring + X + red, its barriers, tensor memory
  uint8_t *dbase = smem + L.ring + ((1024u - (smem_addr(smem + L.ring) & 1023u)) & 1023u);
  const dense::Plan DP = dense::plan(G);
  uint64_t *ddfull = reinterpret_cast<uint64_t *>(smem + L.misc + kMiscDBar);  // [kStages] TMA landed
  uint64_t *ddempty = ddfull + dense::kStages;                                  // [kStages] MMAs done with a stage
  uint64_t *dadone = ddempty + dense::kStages;                                  // [2] MMAs done with an A buffer
  uint64_t *dsfull = dadone + 2;                                                // scales of the unit landed
  uint64_t *dsempty = dsfull + 1;                                               // scales consumed (every warp)
  uint64_t *dafull = dsempty + 1;                                               // [2] A buffer written (every warp)
  uint64_t *dtfree = dafull + 2;                                                // epilogue done with tensor memory
  uint64_t *dtready = dtfree + 1;                                               // tensor memory allocated
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L.misc + kMiscTmem);
  int *s_flag = reinterpret_cast<int *>(smem + L.misc);
  float *s_logit = reinterpret_cast<float *>(smem + L.misc + kMiscLogit);
  float *s_part = reinterpret_cast<float *>(smem + L.misc + kMiscPart);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.misc + kMiscBar);  // [kWSlots]
  uint64_t *empty = full + kWSlots;                                         // [kWSlots], one arrival per warp
  uint64_t *xfull = empty + kWSlots;
  uint64_t *xempty = xfull + 1;
  uint64_t *route = xempty + 1;   // grouping ready
  // The two consumer groups share the ring but each consumes only its own
  // units, so a group can reach slot s for use j while use j - kWSlots (the
  // other group's, in the same slot) has not landed yet: a parity wait then
  // sees the older phase's parity and passes early.  Every consumer records
  // here the use it saw land in each slot, and waits for use j only once
  // use j - kWSlots is recorded.
  volatile int *s_land = reinterpret_cast<volatile int *>(smem + L.misc + kMiscLand);
  uint64_t *hready = route + 1;   // all h written (barrier 2 passed)
  // per consumer group: h staging of a gate/up unit, routing weights of the current down chunk
  const int gi = (warp >> 3) & 1, wl = warp & 7, gt = tid & 255;
  __half *s_hst_g = reinterpret_cast<__half *>(smem + L.misc + (gi ? kMiscHst1 : kMiscHst));
  float *s_wt_g = reinterpret_cast<float *>(smem + L.misc + (gi ? kMiscWt1 : kMiscWt));

  // this block's router tiles: every 16-expert tile once per own token
  const int n_tok = c < T ? (T - 1 - c) / nb + 1 : 0;
  const int n_ru = n_tok * L.n_mt;

  if (tid == 0) {
    for (int i = 0; i < kWSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCons);
    }
    mbar_init(xfull, 1);
    mbar_init(xempty, 2);  // one arrival per consumer group
    mbar_init(route, 1);
    mbar_init(hready, 1);
    for (int i = 0; i < kWSlots; ++i) s_land[i] = -1;
    for (int i = 0; i < dense::kStages; ++i) {
      mbar_init(&ddfull[i], 1);
      mbar_init(&ddempty[i], 1);
    }
    mbar_init(&dadone[0], 1);
    mbar_init(&dadone[1], 1);
    mbar_init(dsfull, 1);
    mbar_init(dsempty, kCons);
    mbar_init(&dafull[0], kCons);
    mbar_init(&dafull[1], kCons);
    mbar_init(dtfree, 1);
    mbar_init(dtready, 1);
    fence_mbar_init();
    s_flag[8] = 0;  // abort
  }
  __syncthreads();
  if (c == 0 && tid == 0) trace_min(a.trace, kTrEntry);

  // ============================================================ producer warp
  if (warp == kCons) {
    bool ok = true;
    int it = 0, xk = 0;
    // next W slot in ring order (waits for the consumers to release it)
    auto acquire = [&]() -> uint8_t * {
      const int slot = it % kWSlots;
      if (it >= kWSlots) ok = mbar_wait_idle(&empty[slot], ((it / kWSlots) - 1) & 1);
      return ring + slot * L.wslot;
    };
    // router tiles: weights only, so they are fetched before the dependency wait
    for (int i = 0; i < n_ru && ok; ++i) {
      uint8_t *dst = acquire();
      if (!ok) break;
      const int m = i % L.n_mt, e0 = m * kRtRows, rows = min(kRtRows, E - e0);
      uint64_t *bar = &full[it % kWSlots];
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(rows * H));
      __syncwarp();
      if (lane < (rows + 3) / 4)  // 4-row blocks (the last one may be short)
        bulk_g2s(dst + lane * L.rt_qp, a.w.router_q + (size_t)(e0 + 4 * lane) * H,
                 (uint32_t)(min(4, rows - 4 * lane) * H), bar);
      ++it;
    }
    if (ok) ok = mbar_wait_idle(route, 0, 32) && *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
    fused::fence_proxy_async_global();  // operand rows written by other blocks before barrier 1
    const int nbl = (kDense && ok) ? s_flag[11] : nb;  // light blocks; the rest take the dense slots
    int dgi = 0, du = 0;                   // dense path: K groups issued, units whose scales went out
    if (kDense && ok && c >= nbl) {
     if constexpr (kDense) {
      // ---- dense block: per unit the scales and biases (one bulk copy per
      // array), then per K group the operand rows (2-D TMA, 128-byte swizzle)
      // and the codes of 128 weight rows (3-D TMA) into a kStages ring
      const int nd = s_flag[10], nblk = nb - nbl, db = c - nbl;
      auto dense_loads = [&](bool down) {
        const int ntile = ((down ? H : I) + dense::kRows - 1) / dense::kRows;
        const int kg = down ? GI : G;
        for (int u = db; u < nd * ntile && ok; u += nblk) {
          const int ds = u / ntile, rt = u - ds * ntile, sa = g_dense[ds];
          const int e = g_act_e[sa];
          const int sh = e < 0 ? 1 : 0;
          const uint8_t *blob = sh ? a.w.shared : a.w.experts + (size_t)e * a.w.stride;
          const int r0 = rt * dense::kRows, nrows = min(dense::kRows, (down ? H : I) - r0);
          if (du >= 1) ok = __all_sync(0xffffffffu, mbar_wait_idle(dsempty, (du - 1) & 1, 32));
          if (!ok) break;
          const int nf = down ? 2 : 4;
          if (lane == 0) mbar_arrive_expect_tx(dsfull, (uint32_t)(nf * nrows * kg * 2));
          __syncwarp();
          if (lane < nf) {
            const size_t off = down ? (lane == 0 ? a.w.off.down_s : a.w.off.down_b)
                                    : (lane == 0 ? a.w.off.gate_s
                                                 : lane == 1 ? a.w.off.gate_b : lane == 2 ? a.w.off.up_s : a.w.off.up_b);
            bulk_g2s(dbase + DP.s + lane * dense::kRows * kg * 2, blob + off + (size_t)r0 * kg * 2,
                     (uint32_t)(nrows * kg * 2), dsfull);
          }
          ++du;
          const int by = down ? g_act_beg[sa] : 0;  // first operand row: the slot's positions, or token 0
          // the first groups' codes into L2 (later groups: kAhead ahead of their TMA below)
          if (lane == 0)
            for (int g = 0; g < kg && g < dense::kAhead; ++g) {
              if (down) {
                dense::tma_prefetch_3d(&prm.dm.dq[sh], 32 * g, r0, sh ? 0 : e);
              } else {
                dense::tma_prefetch_3d(&prm.dm.gq[sh], 32 * g, r0, sh ? 0 : e);
                dense::tma_prefetch_3d(&prm.dm.uq[sh], 32 * g, r0, sh ? 0 : e);
              }
            }
          for (int g = 0; g < kg && ok; ++g, ++dgi) {
            const int st = dgi % dense::kStages;
            if (dgi >= dense::kStages)
              ok = __all_sync(0xffffffffu, mbar_wait_idle(&ddempty[st], ((dgi / dense::kStages) - 1) & 1, 32));
            if (!ok) break;
            if (lane == 0) {
              const int gp = g + dense::kAhead;
              if (gp < kg) {
                if (down) {
                  dense::tma_prefetch_3d(&prm.dm.dq[sh], 32 * gp, r0, sh ? 0 : e);
                } else {
                  dense::tma_prefetch_3d(&prm.dm.gq[sh], 32 * gp, r0, sh ? 0 : e);
                  dense::tma_prefetch_3d(&prm.dm.uq[sh], 32 * gp, r0, sh ? 0 : e);
                }
              }
              mbar_arrive_expect_tx(&ddfull[st], (uint32_t)(dense::kRows * 128 + (down ? 1 : 2) * dense::kRows * 32));
              dense::tma_load_2d(dbase + DP.b[st], down ? &prm.dm.h : &prm.dm.x, 64 * g, by, &ddfull[st]);
              if (down) {
                dense::tma_load_3d(dbase + DP.c[st], &prm.dm.dq[sh], 32 * g, r0, sh ? 0 : e, &ddfull[st]);
              } else {
                dense::tma_load_3d(dbase + DP.c[st], &prm.dm.gq[sh], 32 * g, r0, sh ? 0 : e, &ddfull[st]);
                dense::tma_load_3d(dbase + DP.c[st] + dense::kRows * 32, &prm.dm.uq[sh], 32 * g, r0, sh ? 0 : e,
                                   &ddfull[st]);
              }
            }
            __syncwarp();
          }
        }
      };
      dense_loads(false);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_idle(hready, 0, 32)) &&
                   *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
      fused::fence_proxy_async_global();  // h rows written by other blocks before barrier 2
      if (ok) dense_loads(true);
     }
    } else if (ok) {
      const int nact = s_flag[9];
      const int nchunks = chunk0[nact];
      const int n_gu = nchunks * L.nrt, n_dn = nchunks * L.nrt_dn;
      int cur = -1;
      // gate/up: weight tile, then the chunk's operand rows when the chunk changes
      const uint8_t *blob = nullptr;  // weights of the current chunk's slot
      for (int u = c * n_gu / nbl; u < (c + 1) * n_gu / nbl && ok; ++u) {
        const int chg = u / L.nrt, tile = u - chg * L.nrt;
        Unit x;
        if (chg != cur) {
          x = decode_unit(u, L.nrt, chunk0, nact, g_act_e, g_act_beg, g_act_cnt);
          blob = x.e < 0 ? a.w.shared : a.w.experts + (size_t)x.e * a.w.stride;
        }
        uint8_t *dst = acquire();
        if (!ok) break;
        uint64_t *bar = &full[it % kWSlots];
        const int r0 = tile * kGuRows;
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(2 * kGuRows * (H / 2) + 4 * kGuRows * G * 2));
        __syncwarp();
        if (lane < 8) {  // 4-row blocks: lanes 0-3 gate, 4-7 up
          const int m = lane >> 2, q = lane & 3;
          bulk_g2s(dst + lane * L.gu_qp, blob + (m == 0 ? a.w.off.gate_q : a.w.off.up_q) + (size_t)(r0 + 4 * q) * (H / 2),
                   (uint32_t)(2 * H), bar);
        } else if (lane < 12) {
          const int f = lane - 8;
          const size_t off = f == 0 ? a.w.off.gate_s : f == 1 ? a.w.off.gate_b : f == 2 ? a.w.off.up_s : a.w.off.up_b;
          bulk_g2s(dst + 8 * L.gu_qp + f * kGuRows * G * 2, blob + off + (size_t)r0 * G * 2,
                   (uint32_t)(kGuRows * G * 2), bar);
        }
        ++it;
        if (chg != cur) {
          if (xk >= 1) ok = mbar_wait_idle(xempty, (xk - 1) & 1, 32);
          if (!ok) break;
          if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(x.nt * (H * 2 + 4 * L.gp)));
          __syncwarp();
          if (lane < 2 * x.nt) {
            const int j = lane >> 1;
            const int tok = x.e < 0 ? kTC * x.ch + j : g_perm[x.beg + kTC * x.ch + j] / k;
            if ((lane & 1) == 0)
              bulk_g2s(xbuf + j * L.xp, a.xperm + (size_t)tok * H, (uint32_t)(H * 2), xfull);
            else
              bulk_g2s(xbuf + L.x_xs + j * 4 * L.gp, a.xs + (size_t)tok * 2 * L.gp, (uint32_t)(4 * L.gp), xfull);
          }
          ++xk;
          cur = chg;
        }
      }
      // down: weight tiles go out at once (they stream during barrier 2); the
      // h rows of a chunk once every block has written them
      bool hr = false;
      cur = -1;
      for (int u = c * n_dn / nbl; u < (c + 1) * n_dn / nbl && ok; ++u) {
        const int chg = u / L.nrt_dn, tile = u - chg * L.nrt_dn;
        Unit x;
        if (chg != cur) {
          x = decode_unit(u, L.nrt_dn, chunk0, nact, g_act_e, g_act_beg, g_act_cnt);
          blob = x.e < 0 ? a.w.shared : a.w.experts + (size_t)x.e * a.w.stride;
        }
        uint8_t *dst = acquire();
        if (!ok) break;
        uint64_t *bar = &full[it % kWSlots];
        const int n0 = tile * kDnRows, rows = min(kDnRows, H - n0);
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(rows * (I / 2) + 2 * rows * GI * 2));
        __syncwarp();
        const bool one = L.dn_qp == I / 2;
        const int nq = one ? 1 : rows;
        for (int ci = lane; ci < nq + 2; ci += 32) {
          if (ci < nq) {
            const int row = one ? 0 : ci;
            bulk_g2s(dst + row * L.dn_qp, blob + a.w.off.down_q + (size_t)(n0 + row) * (I / 2),
                     one ? (uint32_t)(rows * (I / 2)) : (uint32_t)(I / 2), bar);
          } else {
            const int f = ci - nq;
            bulk_g2s(dst + kDnRows * L.dn_qp + f * kDnRows * GI * 2,
                     blob + (f == 0 ? a.w.off.down_s : a.w.off.down_b) + (size_t)n0 * GI * 2,
                     (uint32_t)(rows * GI * 2), bar);
          }
        }
        ++it;
        if (chg != cur) {
          if (!hr) {
            ok = mbar_wait_idle(hready, 0, 32) && *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
            fused::fence_proxy_async_global();
            hr = true;
          }
          if (ok && xk >= 1) ok = mbar_wait_idle(xempty, (xk - 1) & 1, 32);
          if (!ok) break;
          if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(x.nt * (I * 2 + (I / 16) * 4)));
          __syncwarp();
          if (lane < 2 * x.nt) {
            const int j = lane >> 1;
            const int pos = x.beg + kTC * x.ch + j;
            if ((lane & 1) == 0)
              bulk_g2s(xbuf + j * L.hp, a.hperm + (size_t)pos * I, (uint32_t)(I * 2), xfull);
            else
              bulk_g2s(xbuf + L.x_hq + j * L.hqp * 4, a.hq + (size_t)pos * (I / 16), (uint32_t)((I / 16) * 4), xfull);
          }
          ++xk;
          cur = chg;
        }
      }
    }
    // copies in flight must land before the block's shared memory is released
    if (lane == 0) {
      if (!ok) set_error(a.err, kErrTimeout);
      for (int j = it - kWSlots > 0 ? it - kWSlots : 0; j < it; ++j) mbar_wait_idle(&full[j % kWSlots], (j / kWSlots) & 1);
      if (xk >= 1) mbar_wait_idle(xfull, (xk - 1) & 1);
      for (int j = dgi - dense::kStages > 0 ? dgi - dense::kStages : 0; j < dgi; ++j)
        mbar_wait_idle(&ddfull[j % dense::kStages], (j / dense::kStages) & 1);
      if (du >= 1) mbar_wait_idle(dsfull, (du - 1) & 1);
    }
    return;
  }

  // ============================================================ MMA warp
  // Dense blocks only: owns the tensor memory (256 columns: gate, up) and
  // issues each K group's tcgen05.mma once the consumers have written its A
  // tile, so the dequantisation of the next group overlaps the MMAs.
  if constexpr (kDense) if (warp == kMmaWarp) {
    const bool okr = __all_sync(0xffffffffu, mbar_wait_idle(route, 0, 64)) &&
                     *reinterpret_cast<volatile int *>(&s_flag[8]) == 0;
    const int nbl = okr ? s_flag[11] : nb;
    if (!okr || c < nbl) return;
    dense::tc_alloc(s_tmem, 256);
    dense::tc_fence_before();
    __syncwarp();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);
    if (lane == 0) mbar_arrive_expect_tx(dtready, 0);
    const int nd = s_flag[10], nblk = nb - nbl;
    int dgi = 0, du = 0;
    bool ok = true;
    auto mma_units = [&](bool down) {
      const int ntile = ((down ? H : I) + dense::kRows - 1) / dense::kRows;
      const int kg = down ? GI : G;
      const int nm = down ? 1 : 2;
      for (int u = c - nbl; u < nd * ntile && ok; u += nblk) {
        const int sa = g_dense[u / ntile];
        const int N = ((down ? (int)g_act_cnt[sa] : T) + 15) & ~15;
        const uint32_t idesc = dense::idesc_f16(dense::kRows, N);
        if (du >= 1) ok = __all_sync(0xffffffffu, mbar_wait_idle(dtfree, (du - 1) & 1, 32));  // TMEM read out
        ++du;
        dense::tc_fence_after();
        for (int g = 0; g < kg && ok; ++g) {
          const int st = dgi % dense::kStages, ab = dgi & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&ddfull[st], (dgi / dense::kStages) & 1) &&
                                           mbar_wait(&dafull[ab], (dgi >> 1) & 1));
          if (!ok) break;
          dense::tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = dense::sdesc(smem_addr(dbase + DP.b[st]) + ks * 32, 16, 1024, 2);
              for (int m = 0; m < nm; ++m) {
                const uint64_t ad =
                    dense::sdesc(smem_addr(dbase + DP.a[ab] + m * dense::kRows * 128) + ks * 32, 16, 1024, 2);
                dense::tc_mma(tmem + m * 128, ad, bd, idesc, (g > 0 || ks > 0) ? 1u : 0u);
              }
            }
            dense::tc_commit(&ddempty[st]);  // the TMA stage may be refilled
            dense::tc_commit(&dadone[ab]);   // the A buffer may be rewritten; after the last group: unit done
          }
          __syncwarp();
          ++dgi;
        }
      }
    };
    mma_units(false);
    if (ok) mma_units(true);
    // tensor memory back once the last MMAs completed and the last epilogue read them (bounded waits)
    if (dgi > 0) mbar_wait(&dadone[(dgi - 1) & 1], ((dgi - 1) >> 1) & 1);
    if (du > 0) mbar_wait_idle(dtfree, (du - 1) & 1, 64);
    dense::tc_fence_after();
    __syncwarp();
    dense::tc_dealloc(tmem, 256);
    return;
  }

  // ============================================================ consumers
  // the router's scales and biases (weights: read before the dependency wait)
  uint16_t *rsb = reinterpret_cast<uint16_t *>(xbuf + L.rx_sb);  // scales [16 n_mt][G], then biases
  const int rsb_n = kRtRows * L.n_mt * G;
  if (n_tok > 0) {
    for (int i = tid; i < E * G; i += kConsThreads) {
      rsb[i] = __ldg(a.w.router_s + i);
      rsb[rsb_n + i] = __ldg(a.w.router_b + i);
    }
  }
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
    if (aborted) s_flag[8] = 1;  // make a failure of either group the block's
    cons_sync();
    aborted = s_flag[8] != 0;
    if (!aborted) {
      aborted = !fused::grid_sync(bar_count, base + (unsigned long long)nbar * nb, a.err, &s_flag[nbar]);
    } else {
      cons_sync();
      if (tid == 0) fused::red_release_add(bar_count);
      cons_sync();
    }
  };
  // a W slot is released by 16 arrivals: one per consumer warp (router
  // tiles, used by all warps) or two per warp of the group that used it
  auto release = [&](int slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&empty[slot], 0);
  };
  auto release_g = [&](int slot) {
    __syncwarp();
    if (lane == 0) fused::mbar_arrive_cnt(&empty[slot], 2);
  };
  auto gsync = [&]() { asm volatile("bar.sync %0, 256;" ::"r"(2 + gi) : "memory"); };
  // ring use j of a group: wait until use j - kWSlots of its slot has landed
  // (bounded), then for use j's own phase; record it
  auto wait_use = [&](int j) -> bool {
    const int slot = j % kWSlots;
    if (j >= kWSlots && s_land[slot] < j - kWSlots) {
      const unsigned long long t0 = global_ns();
      while (s_land[slot] < j - kWSlots)
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    if (!mbar_wait(&full[slot], (j / kWSlots) & 1)) return false;
    if (gt == 0) s_land[slot] = j;
    return true;
  };
  const uint16_t *src = a.hres ? a.hres : a.x;
  const int nquart = H / 16;
  const int r = lane >> 2, cq = lane & 3;
  int it = 0, xk = 0;

  // ---- R: operand rows, router scores and top-k of tokens t = c, c + nb, ...
  for (int t = c; t < T && !aborted; t += nb) {
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
      // router operand: fp16 pairs (x0,x2)(x1,x3)(x4,x6)(x5,x7)... of this
      // quarter, of x or (router scale given) of x * router_scale / sqrt(H);
      // its sum over the quarter feeds the router's bias terms
      uint32_t h[8];
      float rsum = s;
      if (kScales && a.w.router_scale) {
        const uint4 *rs4 = reinterpret_cast<const uint4 *>(a.w.router_scale) + 2 * tid;
        const uint4 r0 = __ldg(rs4), r1 = __ldg(rs4 + 1);
        const uint32_t rw8[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const float isq = rsqrtf((float)H);
        rsum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const __half2 hv = __floats2half2_rn(
              __uint_as_float(qin[i] << 16) * (__uint_as_float(rw8[i] << 16) * isq),
              __uint_as_float(qin[i] & 0xFFFF0000u) * (__uint_as_float(rw8[i] & 0xFFFF0000u) * isq));
          h[i] = *reinterpret_cast<const uint32_t *>(&hv);
          rsum += __low2float(hv);
          rsum += __high2float(hv);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = bf16x2_to_f16x2(qin[i]);
      }
      uint32_t rp[8];
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) {
        rp[2 * s2] = __byte_perm(h[2 * s2], h[2 * s2 + 1], 0x5410);      // x[4s], x[4s+2]
        rp[2 * s2 + 1] = __byte_perm(h[2 * s2], h[2 * s2 + 1], 0x7632);  // x[4s+1], x[4s+3]
      }
      uint4 *rx = reinterpret_cast<uint4 *>(xbuf + tid * 32);
      rx[0] = make_uint4(rp[0], rp[1], rp[2], rp[3]);
      rx[1] = make_uint4(rp[4], rp[5], rp[6], rp[7]);
      reinterpret_cast<float *>(xbuf + L.rx_q)[tid] = rsum;
      if (kScales && a.w.router_scale) reinterpret_cast<float *>(xbuf + L.rx_xq)[tid] = s;
    }
    cons_sync();  // rx complete
    // group sums of x for the gate/up bias terms, as bf16 hi + lo (zero padded to gp)
    if (tid < L.gp) {
      uint16_t hi = 0, lo = 0;
      if (tid < G) {
        const float *q = reinterpret_cast<const float *>(xbuf + (kScales && a.w.router_scale ? L.rx_xq : L.rx_q)) + 4 * tid;
        const float gs = (((q[0] + q[1]) + q[2]) + q[3]) * (1.0f / kCodeScale);  // 2^-24, as the code products
        hi = float_to_bf16_bits(gs);
        lo = float_to_bf16_bits(gs - bf16_bits_to_float(hi));
      }
      a.xs[(size_t)t * 2 * L.gp + tid] = hi;
      a.xs[(size_t)t * 2 * L.gp + L.gp + tid] = lo;
    }
    float rt0[8], rt1[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      rt0[m] = 0.f;
      rt1[m] = 0.f;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (m < L.n_mt && !aborted) {
        const int slot = it % kWSlots;
        if (!mbar_wait(&full[slot], (it / kWSlots) & 1)) {
          aborted = true;
          set_error(a.err, kErrTimeout);
        } else {
          if (tid == 0) s_land[slot] = it;  // every warp consumes router tiles, in order
          const uint8_t *tile = ring + slot * L.wslot;
          const uint16_t *rs = rsb + m * kRtRows * G, *rb = rsb + rsb_n + m * kRtRows * G;
          for (int g = warp; g < G; g += kCons)
            rt_group(tile, xbuf, reinterpret_cast<const float *>(xbuf + L.rx_q), rs, rb, L.rt_qp, G, g, r, cq, rt0[m],
                     rt1[m]);
          release(slot);
          ++it;
        }
      }
    }
    if (cq == 0) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < L.n_mt) {
          red[warp * 128 + m * 16 + quad_row(r)] = rt0[m];
          red[warp * 128 + m * 16 + quad_row(r) + 2] = rt1[m];
        }
    }
    cons_sync();
    if (tid < E) {
      float v = a.w.logit_bias ? a.w.logit_bias[tid] : 0.f;
      float sum = 0.f;
      for (int w = 0; w < kCons; ++w) sum += red[w * 128 + tid];
      v += sum;
      s_logit[tid] = v;
      a.logits[(size_t)t * E + tid] = v;
    }
    cons_sync();
    if (warp == 0) {
      bool bad = false;
      fused::warp_topk(s_logit, E, k, a.r.ids + t * k, a.r.wts + t * k, kScales ? a.w.expert_scale : nullptr, &bad);
      if (bad && lane == 0) set_error(a.err, kErrNonFinite);
      __syncwarp();
      if (lane < k) {
        if (a.ids_user) a.ids_user[t * k + lane] = a.r.ids[t * k + lane];
        if (a.wts_user) a.wts_user[t * k + lane] = a.r.wts[t * k + lane];
      }
    }
    cons_sync();  // rx, red and s_logit are reused by the next token
  }

  fused::fence_proxy_async_global();  // operand rows are read back by bulk copies
  barrier();  // 1: operand rows, quarter sums, routing

  // ---- every block groups all pairs (stable counting sort by expert id)
  if (!aborted) {
    int *cnt = reinterpret_cast<int *>(red);  // [E]
    int *wc = cnt + E;                        // [kCons][E]
    for (int i = tid; i < (1 + kCons) * E; i += kConsThreads) cnt[i] = 0;
    cons_sync();
    for (int p = tid; p < npairs; p += kConsThreads) atomicAdd(&cnt[__ldcg(a.r.ids + p)], 1);
    cons_sync();
    if (warp == 0) {
      // exclusive scan of counts -> fill positions; active slots (shared first); chunk prefix
      const bool don = kDense && prm.dense_on != 0;
      int run = 0, nact = 1, chunks = (don && T >= dense::kMinRows) ? 0 : (T + kTC - 1) / kTC;
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
        const int nch = (don && ce >= dense::kMinRows) ? 0 : (ce + kTC - 1) / kTC;
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
        run += __shfl_sync(0xffffffffu, incl, 31);
        chunks += __shfl_sync(0xffffffffu, incl_ch, 31);
        nact += __popc(act);
      }
      if (lane == 0) {
        chunk0[nact] = chunks;
        s_flag[9] = nact;
      }
      __syncwarp();
      // dense slots in active-slot order; the blocks that take them: the
      // last n_db blocks, as many as the cost of their gate/up units asks
      // for against the light ones (a dense unit ~ dense::kGuCost light units)
      int nd = 0;
      for (int a0 = 0; a0 < nact; a0 += 32) {
        const int sa = a0 + lane;
        const bool dn = don && sa < nact && g_act_cnt[sa] >= dense::kMinRows;
        const unsigned bal = __ballot_sync(0xffffffffu, dn);
        if (dn && nd + __popc(bal & lanemask_lt()) < kMaxDense) g_dense[nd + __popc(bal & lanemask_lt())] = (int16_t)sa;
        nd += __popc(bal);
      }
      if (lane == 0) {
        nd = nd < kMaxDense ? nd : kMaxDense;
        const int n_dg = nd * ((I + dense::kRows - 1) / dense::kRows);
        const int n_dd = nd * ((H + dense::kRows - 1) / dense::kRows);
        const float dc = (float)n_dg * dense::kGuCost + (float)n_dd * dense::kDnCost;
        const float lc = (float)chunks * ((float)L.nrt + (float)L.nrt_dn);
        // at least one dense block per gate/up unit while they are few: a
        // second unit on one block would hold every block at barrier 2
        int ndb = 0;
        if (n_dg > 0) {
          ndb = lc > 0.f ? (int)rintf((float)nb * dc / (dc + lc)) : nb;
          if (n_dg <= nb / 4 && ndb < n_dg) ndb = n_dg;
          ndb = ndb < 1 ? 1 : ndb;
          ndb = ndb > n_dg ? n_dg : ndb;
          if (lc > 0.f && ndb > nb - 1) ndb = nb - 1;
        }
        s_flag[10] = nd;
        s_flag[11] = nb - ndb;  // light blocks [0, nbl), dense blocks [nbl, nb)
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

  const int nact = aborted ? 0 : s_flag[9];
  const int nchunks = aborted ? 0 : chunk0[nact];
  const int nbl = (kDense && !aborted) ? s_flag[11] : nb;  // light blocks [0, nbl); dense blocks [nbl, nb)
  const bool dense_blk = kDense && !aborted && c >= nbl;

  // ---- dense blocks: the MMA warp owns the tensor memory of the
  // accumulators (gate in columns 0..127, up in 128..255; down uses the
  // first 128); its address once the allocation is done
  uint32_t tmem = 0;
  bool have_tmem = false;
  int dgi = 0, du = 0;  // K groups consumed, units whose scales were consumed
  // The dense units of this block: (dense slot, 128 weight rows) for u = c -
  // nbl, c - nbl + (nb - nbl), ...  Gate/up: A = 128 rows of gate and of up,
  // B = the chunk's operand rows (every token; the epilogue keeps those
  // routed to the slot).  Down: A = 128 rows of W_down, B = h of the slot's
  // sorted positions.  Per K group every consumer thread dequantises one
  // quarter (down: one eighth) of the A tiles and each warp signals the MMA
  // warp, which issues the K = 64 step as four tcgen05.mma per matrix.
  auto dense_units = [&](bool down) {
    const int nd = s_flag[10], nblk = nb - nbl;
    const int ntile = ((down ? H : I) + dense::kRows - 1) / dense::kRows;
    const int kg = down ? GI : G;
    const uint16_t *sb = reinterpret_cast<const uint16_t *>(dbase + DP.s);
    for (int u = c - nbl; u < nd * ntile && !aborted; u += nblk) {
      const int ds = u / ntile, rt = u - ds * ntile, sa = g_dense[ds];
      const int e = g_act_e[sa], beg = g_act_beg[sa], cnt = g_act_cnt[sa];
      const int r0 = rt * dense::kRows, nrows = min(dense::kRows, (down ? H : I) - r0);
      const int N = ((down ? cnt : T) + 15) & ~15;  // MMA N: operand rows, padded to 16
      if (!down) {
        for (int t = tid; t < T; t += kConsThreads) {  // token -> its position in this slot, or -1
          int pos = -1;
          if (e < 0) {
            pos = npairs + t;
          } else {
            for (int j = 0; j < k; ++j)
              if (__ldcg(a.r.ids + t * k + j) == e) pos = g_pos[t * k + j];
          }
          g_tpos[t] = (int16_t)pos;
        }
      } else {
        for (int n = tid; n < cnt; n += kConsThreads) g_wpos[n] = e < 0 ? 1.0f : __ldcg(a.r.wts + g_perm[beg + n]);
      }
      cons_sync();  // the tables are complete before any warp's epilogue reads them
      bool okd = mbar_wait(dsfull, du & 1);
      ++du;
      for (int g = 0; g < kg; ++g, ++dgi) {
        const int st = dgi % dense::kStages, ab = dgi & 1;
        okd = okd && mbar_wait(&ddfull[st], (dgi / dense::kStages) & 1);
        if (dgi >= 2) okd = okd && mbar_wait(&dadone[ab], ((dgi >> 1) - 1) & 1);
        if (okd) {
          const uint8_t *cb = dbase + DP.c[st];
          uint8_t *ab_ = dbase + DP.a[ab];
          const int rr = tid & 127;
          if (!down) {
            const int m = tid >> 8, hh = (tid >> 7) & 1;  // matrix (gate, up), half of the group
            const uint4 cw = *reinterpret_cast<const uint4 *>(cb + m * dense::kRows * 32 + rr * 32 + hh * 16);
            const float sf = bf16_bits_to_float(sb[(2 * m) * dense::kRows * kg + rr * kg + g]);
            const float bf = bf16_bits_to_float(sb[(2 * m + 1) * dense::kRows * kg + rr * kg + g]);
            const uint32_t s2 = dense::f16x2_of(sf), b2 = dense::f16x2_of(bf), b16 = dense::f16x2_of(16.0f * bf);
            // row rr of the 128-byte-swizzled tile: 16-byte chunk j at (j ^ (rr % 8))
            uint8_t *row = ab_ + m * dense::kRows * 128 + rr * 128;
            const int sw = rr & 7, j0 = 4 * hh;
            *reinterpret_cast<uint4 *>(row + ((j0 + 0) ^ sw) * 16) = dense::dequant_word(cw.x, s2, b2, b16);
            *reinterpret_cast<uint4 *>(row + ((j0 + 1) ^ sw) * 16) = dense::dequant_word(cw.y, s2, b2, b16);
            *reinterpret_cast<uint4 *>(row + ((j0 + 2) ^ sw) * 16) = dense::dequant_word(cw.z, s2, b2, b16);
            *reinterpret_cast<uint4 *>(row + ((j0 + 3) ^ sw) * 16) = dense::dequant_word(cw.w, s2, b2, b16);
          } else {
            const int qq = tid >> 7;  // quarter of the group
            const uint2 cw = *reinterpret_cast<const uint2 *>(cb + rr * 32 + qq * 8);
            const float sf = bf16_bits_to_float(sb[rr * kg + g]);
            const float bf = bf16_bits_to_float(sb[dense::kRows * kg + rr * kg + g]);
            const uint32_t s2 = dense::f16x2_of(sf), b2 = dense::f16x2_of(bf), b16 = dense::f16x2_of(16.0f * bf);
            uint8_t *row = ab_ + rr * 128;
            const int sw = rr & 7, j0 = 2 * qq;
            *reinterpret_cast<uint4 *>(row + ((j0 + 0) ^ sw) * 16) = dense::dequant_word(cw.x, s2, b2, b16);
            *reinterpret_cast<uint4 *>(row + ((j0 + 1) ^ sw) * 16) = dense::dequant_word(cw.y, s2, b2, b16);
          }
        }
        dense::fence_async_smem();  // the A tiles, written by threads, are read by the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&dafull[ab], 0);  // this warp's part of the A tile is in place
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(dsempty, 0);  // this warp is done with the unit's scales
      okd = okd && mbar_wait(&dadone[(dgi - 1) & 1], ((dgi - 1) >> 1) & 1);  // every MMA of the unit done
      if (!have_tmem) {
        okd = okd && mbar_wait(dtready, 0);
        tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);
        have_tmem = true;
      }
      okd = __all_sync(0xffffffffu, okd);  // tcgen05.ld below is warp-collective
      dense::tc_fence_after();
      // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (weight
      // rows) and columns 32 (w / 4) .. +31 (operand rows)
      const int w4 = warp & 3, cbk = warp >> 2, rr = 32 * w4 + lane;
      if (okd && 32 * cbk < N) {
        const uint32_t ta = tmem + ((uint32_t)(32 * w4) << 16) + 32 * cbk;
        bool odd = false;
        const int i = r0 + rr;
        const int slot = dense::operand_slot(i & 63, odd);
        for (int hf = 0; hf < 2; ++hf) {  // 16 columns at a time
          if (!down) {
            float gv[16], uv[16];
            dense::tc_ld16(ta + 16 * hf, gv);
            dense::tc_ld16(ta + 128 + 16 * hf, uv);
            if (rr < nrows) {
              __half *dst = a.hperm + (i & ~63) + slot;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int t = 32 * cbk + 16 * hf + j;
                const int pos = t < T ? g_tpos[t] : -1;
                if (pos >= 0) {
                  const float hv = gelu_tanh(gv[j]) * uv[j];
                  if (!(fabsf(hv) <= 65504.0f)) set_error(a.err, kErrNonFinite);
                  dst[(size_t)pos * I] = __float2half_rn(odd ? hv * 0.0625f : hv);  // odd words / 16
                }
              }
            }
          } else {
            float dv[16];
            dense::tc_ld16(ta + 16 * hf, dv);
            if (rr < nrows) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = 32 * cbk + 16 * hf + j;
                if (n < cnt) a.obuf[(size_t)(beg + n) * H + r0 + rr] = g_wpos[n] * dv[j];
              }
            }
          }
        }
      }
      dense::tc_fence_before();
      if (!fused::cons_sync_and(okd)) {
        aborted = true;
        set_error(a.err, kErrTimeout);
        break;
      }
      if (tid == 0) mbar_arrive_expect_tx(dtfree, 0);  // the MMA warp may overwrite the accumulators
    }
  };

  // ---- G: gate/up units [c * n_gu / nb, (c + 1) * n_gu / nb).  Steps of two
  // consecutive units of one chunk (group 0 takes the first, group 1 the
  // second) or one unit at a chunk's end; both groups walk every step so they
  // leave each X phase (chunk) together.
  if (dense_blk) {
    if constexpr (kDense) dense_units(false);
  } else {
    const int n_gu = nchunks * L.nrt;
    const int lo = c * n_gu / nbl, hi = (c + 1) * n_gu / nbl;
    int u = lo, itu = it, ph = -1, xp = xk - 1, p0 = 0, nt = 0;
    while (u < hi && !aborted) {
      const int chg = u / L.nrt;
      const bool pair = u + 1 < hi && (u + 1) / L.nrt == chg;
      if (chg != ph) {
        // leave the old chunk, then wait for the new one's rows even without a
        // unit in it: a group never runs a phase ahead, so the release barrier
        // (two arrivals, one per group) completes phase by phase
        if (ph >= 0 && gt == 0) fused::mbar_arrive_cnt(xempty, 1);
        ph = chg;
        ++xp;
        const Unit x = decode_unit(u, L.nrt, chunk0, nact, g_act_e, g_act_beg, g_act_cnt);
        p0 = x.beg + kTC * x.ch;
        nt = x.nt;
        if (!mbar_wait(xfull, xp & 1)) {
          aborted = true;
          set_error(a.err, kErrTimeout);
          break;
        }
      }
      const int mine = gi == 0 ? u : (pair ? u + 1 : -1);
      if (mine >= 0) {
        const int myit = itu + gi, slot = myit % kWSlots, tile = mine - chg * L.nrt;
        if (!wait_use(myit)) {
          aborted = true;
          set_error(a.err, kErrTimeout);
          break;
        }
        const uint8_t *wt = ring + slot * L.wslot;
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(xbuf + L.x_xs);
        float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
        float tg2[4] = {0.f, 0.f, 0.f, 0.f}, tu2[4] = {0.f, 0.f, 0.f, 0.f};
        int g = wl;
        for (; g + 8 < G; g += 16) {
          gu_group(wt, xbuf, L.gu_qp, L.xp, G, g, r, cq, tg, tu);
          gu_group(wt, xbuf, L.gu_qp, L.xp, G, g + 8, r, cq, tg2, tu2);
        }
        if (g < G) gu_group(wt, xbuf, L.gu_qp, L.xp, G, g, r, cq, tg, tu);
        // bias terms: gate in the group's last warp, up in the one before
        // (the warps with the fewest groups)
        if (wl == 7) gu_bias(wt, xs, L.gu_qp, G, L.gp, 16 * G, r, cq, tg2);
        if (wl == 6) gu_bias(wt, xs, L.gu_qp, G, L.gp, 48 * G, r, cq, tu2);
        release_g(slot);
        // reduction over the group's 8 warps, transposed (conflict-free): red[w][i][lane]
        float *red_g = red + gi * 8 * 256;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          red_g[wl * 256 + i * 32 + lane] = tg[i] + tg2[i];
          red_g[wl * 256 + (i + 4) * 32 + lane] = tu[i] + tu2[i];
        }
        gsync();
        if (gt < kGuRows * kTC) {
          const int idx = gt >> 5, ln = gt & 31;
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            gs += red_g[w * 256 + idx * 32 + ln];
            us += red_g[w * 256 + (idx + 4) * 32 + ln];
          }
          const int m = (ln >> 2) + 8 * (idx >> 1), n = 2 * (ln & 3) + (idx & 1);  // mma row, token
          const float hv = gelu_tanh(gs * kCodeScale) * (us * kCodeScale);
          if (n < nt && !(fabsf(hv) <= 65504.0f)) set_error(a.err, kErrNonFinite);
          s_hst_g[n * 16 + quad_row(m)] = __float2half_rn(hv);
        }
        gsync();
        if (gt < nt) {  // one thread per token writes its 16-row quarter of h
          const int pos = p0 + gt;
          const uint4 *hv = reinterpret_cast<const uint4 *>(s_hst_g + gt * 16);
          const uint4 v0 = hv[0], v1 = hv[1];
          const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          uint32_t out[8];
          operand_quarter<false>(in, out);
          uint4 *dst = reinterpret_cast<uint4 *>(a.hperm + (size_t)pos * I + tile * kGuRows);
          dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
          dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
          float sm = 0.f;
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            sm += __half2float(__ushort_as_half((unsigned short)(in[w] & 0xFFFFu)));
            sm += __half2float(__ushort_as_half((unsigned short)(in[w] >> 16)));
          }
          a.hq[(size_t)pos * (I / 16) + tile] = sm;
        }
        // red_g is rewritten after the group's next tensor-core loop, s_hst_g
        // after its next barrier: both after every thread's reads here
      }
      u += pair ? 2 : 1;
      itu += pair ? 2 : 1;
    }
    if (ph >= 0 && gt == 0) fused::mbar_arrive_cnt(xempty, 1);
    it += hi - lo;
    xk = xp + 1;
  }

  fused::fence_proxy_async_global();  // h rows are read back by bulk copies
  barrier();  // 2: all of h
  if (tid == 0) {
    if (aborted) s_flag[8] = 1;
    mbar_arrive_expect_tx(hready, 0);
  }

  const int gip = (GI + 15) & ~15;  // padded group count of the h group-sum tables
  uint16_t *hs_g = reinterpret_cast<uint16_t *>(red + gi * 8 * 256);
  // ---- D: down units [c * n_dn / nb, (c + 1) * n_dn / nb) -> weighted outputs,
  // in the same two-group steps.  A group's warp w owns rows 16w..16w+15 of its
  // 128-row unit over the whole K, so its results leave straight from registers.
  if (dense_blk) {
    if constexpr (kDense) dense_units(true);
  } else {
    const int n_dn = nchunks * L.nrt_dn;
    const int lo = c * n_dn / nbl, hi = (c + 1) * n_dn / nbl;
    int u = lo, itu = it, ph = -1, xp = xk - 1, p0 = 0, nt = 0;
    while (u < hi && !aborted) {
      const int chg = u / L.nrt_dn;
      const bool pair = u + 1 < hi && (u + 1) / L.nrt_dn == chg;
      if (chg != ph) {
        // a down unit ends without a group barrier: only after this one has
        // every warp of the group left the old chunk's h rows (and its
        // routing weights), so only then may the producer refill them
        gsync();
        if (ph >= 0 && gt == 0) fused::mbar_arrive_cnt(xempty, 1);
        ph = chg;
        ++xp;
        const Unit x = decode_unit(u, L.nrt_dn, chunk0, nact, g_act_e, g_act_beg, g_act_cnt);
        p0 = x.beg + kTC * x.ch;
        nt = x.nt;
        if (gt < nt) {
          const int pos = p0 + gt;
          s_wt_g[gt] = pos >= npairs ? 1.0f : __ldcg(a.r.wts + g_perm[pos]);
        }
        gsync();
        if (!mbar_wait(xfull, xp & 1)) {  // as for gate/up: never a phase ahead
          aborted = true;
          set_error(a.err, kErrTimeout);
          break;
        }
        // the chunk's group sums of h, bf16 hi + lo, in this group's table
        // (its reduction area, unused by the down units)
        if (gt < kTC * gip) {
          const int tok = gt / gip, gg = gt - tok * gip;
          uint16_t hi = 0, lo = 0;
          if (gg < GI) {
            const float *q = reinterpret_cast<const float *>(xbuf + L.x_hq) + tok * L.hqp + 4 * gg;
            const float v = (((q[0] + q[1]) + q[2]) + q[3]) * (1.0f / kCodeScale);
            hi = float_to_bf16_bits(v);
            lo = float_to_bf16_bits(v - bf16_bits_to_float(hi));
          }
          hs_g[tok * 2 * gip + gg] = hi;
          hs_g[tok * 2 * gip + gip + gg] = lo;
        }
        gsync();
      }
      const int mine = gi == 0 ? u : (pair ? u + 1 : -1);
      if (mine >= 0) {
        const int myit = itu + gi, slot = myit % kWSlots, tile = mine - chg * L.nrt_dn;
        if (!wait_use(myit)) {
          aborted = true;
          set_error(a.err, kErrTimeout);
          break;
        }
        const uint8_t *wt = ring + slot * L.wslot;
        float t4[4] = {0.f, 0.f, 0.f, 0.f}, t4b[4] = {0.f, 0.f, 0.f, 0.f};
        int g = 0;
        for (; g + 1 < GI; g += 2) {
          dn_group(wt, xbuf, L.dn_qp, L.hp, GI, 16 * wl, g, r, cq, t4);
          dn_group(wt, xbuf, L.dn_qp, L.hp, GI, 16 * wl, g + 1, r, cq, t4b);
        }
        if (g < GI) dn_group(wt, xbuf, L.dn_qp, L.hp, GI, 16 * wl, g, r, cq, t4);
        dn_bias(wt, hs_g, L.dn_qp, GI, gip, 16 * wl, r, cq, t4b);
        release_g(slot);
        const int n0 = tile * kDnRows, rows = min(kDnRows, H - n0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 16 * wl + r + 8 * (i >> 1), n = 2 * cq + (i & 1);
          if (n < nt && row < rows)
            a.obuf[(size_t)(p0 + n) * H + n0 + row] = s_wt_g[n] * ((t4[i] + t4b[i]) * kCodeScale);
        }
      }
      u += pair ? 2 : 1;
      itu += pair ? 2 : 1;
    }
    if (ph >= 0 && gt == 0) fused::mbar_arrive_cnt(xempty, 1);
    it += hi - lo;
    xk = xp + 1;
  }

  barrier();  // 3: all weighted outputs
  // ---- C: combine tokens t = c, c + nb, ...
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

namespace {
// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point (no link against the driver library)
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
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

// A tensor map over a row-major tensor of `rank` dims (dims[0] innermost),
// byte strides of dims 1.. in `strides`; out-of-range elements read as zero.
bool encode(EncodeTiledFn f, CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
            const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw,
            CUtensorMapL2promotion l2) {
  const cuuint32_t estr[3] = {1, 1, 1};
  return f(m, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The dense path's maps: operand rows of x and of h (fp16, boxes of 64
// elements x 128 rows with the 128-byte swizzle the tensor cores read), and
// the 4-bit codes of gate, up and down (boxes of 32 bytes x 128 rows of one
// expert), for the routed experts (3-D over the fixed-stride blobs) and the
// shared expert.
bool dense_maps(const PrefillArgs &a, dense::Maps &dm) {
  const EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t H = a.d.H, I = a.d.I, E = a.d.E, T = a.d.T, npos = (cuuint64_t)a.d.T * (a.d.k + 1);
  const cuuint32_t bx[2] = {64, dense::kRows};
  bool ok = true;
  {
    const cuuint64_t dims[2] = {H, T}, str[1] = {H * 2};
    ok = ok && encode(f, &dm.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.xperm, dims, str, bx, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  }
  {
    const cuuint64_t dims[2] = {I, npos}, str[1] = {I * 2};
    ok = ok && encode(f, &dm.h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.hperm, dims, str, bx, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  }
  const cuuint32_t bq[3] = {32, dense::kRows, 1};
  auto codes = [&](CUtensorMap *m, size_t off, cuuint64_t row_bytes, cuuint64_t rows) {
    const cuuint64_t dr[3] = {row_bytes, rows, E}, sr[2] = {row_bytes, a.w.stride};
    const cuuint64_t ds[3] = {row_bytes, rows, 1}, ss[2] = {row_bytes, row_bytes * rows};
    return encode(f, &m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w.experts + off, dr, sr, bq, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B) &&
           encode(f, &m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w.shared + off, ds, ss, bq, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  };
  ok = ok && codes(dm.gq, a.w.off.gate_q, H / 2, I) && codes(dm.uq, a.w.off.up_q, H / 2, I) &&
       codes(dm.dq, a.w.off.down_q, I / 2, H);
  return ok;
}
}  // namespace

cudaError_t launch_prefill_fused(const PrefillArgs &a, int n_blocks, cudaStream_t st, bool pdl, bool allow_dense) {
  PrefillParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.a = a;
  const bool scales = a.w.router_scale != nullptr || a.w.expert_scale != nullptr;
  // the tcgen05 instance: only when asked for, the chunk can hold a dense
  // slot, its shared memory fits one block per SM, and the maps encode
  const size_t dsmem = allow_dense && a.d.T >= dense::kMinRows ? prefill_dense_smem(a.d) : 0;
  bool dense_on = dsmem != 0;
  if (dense_on) {
    int n = 0;
    dense_on = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                   &n, scales ? prefill_layer_kernel<true, true> : prefill_layer_kernel<false, true>, kThreadsP,
                   dsmem) == cudaSuccess &&
               n >= 1 && dense_maps(a, prm.dm);
  }
  prm.dense_on = dense_on ? 1 : 0;
  prm.L = prefill_layout(a.d.H, a.d.I, a.d.E, a.d.k, a.d.T, dense_on);
  if (dense_on)
    return launch_k(scales ? prefill_layer_kernel<true, true> : prefill_layer_kernel<false, true>, dim3(n_blocks),
                    dim3(kThreadsP), dsmem, st, pdl, prm);
  return launch_k(scales ? prefill_layer_kernel<true, false> : prefill_layer_kernel<false, false>, dim3(n_blocks),
                  dim3(fused::kThreads), prefill_fused_smem(a.d), st, pdl, prm);
}

cudaError_t prefill_set_attributes() {
  const void *ks[4] = {(const void *)prefill_layer_kernel<false, false>, (const void *)prefill_layer_kernel<true, false>,
                       (const void *)prefill_layer_kernel<false, true>, (const void *)prefill_layer_kernel<true, true>};
  for (const void *kf : ks) {
    const cudaError_t e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int prefill_blocks_per_sm(const Dims &d) {
  const size_t smem = prefill_fused_smem(d);
  if (smem == 0) return 0;
  int n = 0, n2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_layer_kernel<false, false>, fused::kThreads, smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n2, prefill_layer_kernel<true, false>, fused::kThreads, smem) !=
          cudaSuccess)
    return 0;
  return n < n2 ? n : n2;
}

}  // namespace moe
