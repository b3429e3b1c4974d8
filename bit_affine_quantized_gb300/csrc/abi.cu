// C ABI of the MoE block: argument checks, workspace carving, launches.
// Declarations and the contract of every call: include/moe.h.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "abi_internal.h"
#include "kernels.h"
#include "moe.h"

struct moe_handle {
  int device;
  unsigned *dwords;  // [0] device error bits, [1] router ticket counter
  bool pdl;
  int prefetch_max;  // bytes; 0 disables the L2 prefetch of selected experts
  unsigned long long *trace;  // caller's trace buffer (nullable)
  int trace_groups;           // 4-slot groups in it
  int trace_next;             // next group handed to a launch
  int n_sm;                   // multiprocessors: grid of the fused decode kernel
  bool fused;                 // single-token calls use the fused layer kernel
  int fused_key[3], fused_ok; // cached shape check (hidden, inter, top_k) -> usable
  bool prefill;               // multi-token layer calls use the fused prefill kernel
  int prefill_key[4], prefill_ok;  // cached check (hidden, inter, n_experts, top_k) -> usable
  bool head_ready;            // the head kernel's attributes are set (first head call)
  bool prefill_dense;         // multi-token calls may run dense slots on the tensor cores (tcgen05)
  // failure-detection hook, consumed by the next fused single-token launch
  int skip_block_next;                  // -1: none
  unsigned long long wait_ns_next;      // 0: the default limit
  // expert offload: streams that fill missing slots in parallel (created on
  // the first offload call), an event per stream the layer's stream waits on
  static constexpr int kCopyStreams = 4;
  cudaStream_t copy_st[kCopyStreams];
  cudaEvent_t copy_ev[kCopyStreams];
  bool copy_ready;
};

namespace {
// Trace slots of the next `n` launches (null when tracing is off).
unsigned long long *take_trace(moe_handle *h, int n) {
  if (!h->trace || h->trace_groups < n) return nullptr;
  if (h->trace_next + n > h->trace_groups) h->trace_next = 0;
  unsigned long long *p = h->trace + 4 * (size_t)h->trace_next;
  h->trace_next += n;
  return p;
}
}  // namespace

namespace {

constexpr size_t kSmemCap = 227 * 1024;
// handle-owned device words: [0] error bits, [1] router ticket; at
// kSyncOffset the single-token kernel's 64-bit grid barrier counter, at
// kPrefillSyncOffset the prefill kernel's (each launch of a kernel adds a
// fixed multiple of its grid size to its own counter, so they stay apart)
constexpr size_t kSyncOffset = 256;
// kHeadStateOffset: the head's greedy state, [kHeadMaxTokens] 64-bit maxima
// then its finished-block ticket (zero between launches)
constexpr size_t kHeadStateOffset = 64;
static_assert(kHeadStateOffset + 2 * moe::kHeadMaxTokens + 1 <= kSyncOffset, "head state overlaps");
constexpr size_t kPrefillSyncOffset = kSyncOffset + 16;
constexpr size_t kDeviceWords = kSyncOffset + 64 + 1024;
// kMboxOffset: the single-token kernel's logit mailboxes, [SM count][128]
// 64-bit words (each launch tags its logits with its epoch; zero at start)
constexpr size_t kMboxOffset = 1536;
static_assert(kDeviceWords <= kMboxOffset, "mailboxes overlap the device words");
size_t device_words(int n_sm) { return kMboxOffset + (size_t)n_sm * moe::kMaxExperts * 2; }

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

moe::Dims to_dims(const moe_dims &d, int T) { return moe::Dims{d.hidden, d.inter, d.n_experts, d.top_k, T}; }

int check_dims(const moe_dims *d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->group != 64) return MOE_ERR_UNSUPPORTED;
  if (d->hidden < 64 || d->hidden > 4096 || d->hidden % 64) return MOE_ERR_UNSUPPORTED;
  if (d->inter < 64 || d->inter > 2048 || d->inter % 64) return MOE_ERR_UNSUPPORTED;
  if (d->top_k < 1 || d->top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (d->n_experts < d->top_k || d->n_experts > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
  const moe::Dims dd = to_dims(*d, moe::kMaxTokens);
  if (moe::gateup_smem(dd, 8) > kSmemCap || moe::down_grouped_smem(dd) > kSmemCap ||
      moe::router_smem(dd, 8) > 200 * 1024)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_tokens(int T) { return (T >= 1 && T <= moe::kMaxTokens) ? MOE_OK : MOE_ERR_INVALID_ARG; }

struct WsLayout {
  size_t logits, ids, wts, counts, offsets, perm, pos, act_e, act_beg, act_cnt, n_act, xn, h, o, xq, hq, y, total;
};

WsLayout ws_layout(const moe_dims &d, int T) {
  const size_t H = d.hidden, I = d.inter, E = d.n_experts, k = d.top_k;
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.logits = take((size_t)T * E * 4);
  L.ids = take((size_t)T * k * 4);
  L.wts = take((size_t)T * k * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take((size_t)T * k * 4);
  L.pos = take((size_t)T * k * 4);
  L.act_e = take((E + 1) * 4);
  L.act_beg = take((E + 1) * 4);
  L.act_cnt = take((E + 1) * 4);
  L.n_act = take(4);
  L.xn = take((size_t)T * H * 2);
  L.h = take(((size_t)T * k + T) * I * 2);
  L.o = moe::use_down_decode(to_dims(d, T)) ? off : take(((size_t)T * k + T) * H * 4);
  // quarter sums of the fused prefill kernel (its operand rows reuse xn and h)
  L.xq = T > 1 ? take((size_t)T * 4 * ((H / 64 + 15) & ~(size_t)15)) : off;  // x group sums, bf16 hi/lo
  L.hq = T > 1 ? take(((size_t)T * k + T) * (I / 16) * 4) : off;
  L.y = take((size_t)T * H * 2);  // block output ahead of a layer tail
  L.total = off;
  return L;
}

// Workspace of the whole-prompt layer (T rows, T*k + T sorted positions).
struct PromptWs {
  size_t logits, ids, wts, counts, offsets, perm, pos, ch_e, ch_beg, ch_cnt, n_ch, xn, xg, hg, o, y, total;
};

PromptWs prompt_ws(const moe_dims &d, int T) {
  const size_t H = d.hidden, I = d.inter, E = d.n_experts, k = d.top_k;
  const size_t npos = (size_t)T * (k + 1);
  const size_t nch = (size_t)moe::prompt_max_chunks(T, (int)k, (int)E);
  PromptWs L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.logits = take((size_t)T * E * 4);
  L.ids = take((size_t)T * k * 4);
  L.wts = take((size_t)T * k * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take((size_t)T * k * 4);
  L.pos = take((size_t)T * k * 4);
  L.ch_e = take(nch * 4);
  L.ch_beg = take(nch * 4);
  L.ch_cnt = take(nch * 4);
  L.n_ch = take(4);
  L.xn = take((size_t)T * H * 2);
  L.xg = take(npos * H * 2);
  L.hg = take(npos * I * 2);
  L.o = take(npos * H * 4);
  L.y = take((size_t)T * H * 2);  // block output ahead of a layer tail
  L.total = off;
  return L;
}

moe::Routing routing_in(uint8_t *ws, const WsLayout &L) {
  moe::Routing r;
  r.ids = (int32_t *)(ws + L.ids);
  r.wts = (float *)(ws + L.wts);
  r.counts = (int32_t *)(ws + L.counts);
  r.offsets = (int32_t *)(ws + L.offsets);
  r.perm = (int32_t *)(ws + L.perm);
  r.pos = (int32_t *)(ws + L.pos);
  r.act_e = (int32_t *)(ws + L.act_e);
  r.act_beg = (int32_t *)(ws + L.act_beg);
  r.act_cnt = (int32_t *)(ws + L.act_cnt);
  r.n_act = (int32_t *)(ws + L.n_act);
  return r;
}

}  // namespace

namespace moe_abi {

size_t blob_extent(const moe_layer_weights &w) {
  const size_t H = w.dims.hidden, I = w.dims.inter;
  const size_t q = I * H / 2, sb = I * (H / 64) * 2;
  const size_t ends[9] = {w.layout.gate_q + q, w.layout.gate_s + sb, w.layout.gate_b + sb,
                          w.layout.up_q + q,   w.layout.up_s + sb,   w.layout.up_b + sb,
                          w.layout.down_q + q, w.layout.down_s + sb, w.layout.down_b + sb};
  return *std::max_element(ends, ends + 9);
}

moe::LayerPtrs layer_ptrs(const moe_layer_weights &w) {
  moe::LayerPtrs p;
  p.router_q = (const uint8_t *)w.router.q;
  p.router_s = (const uint16_t *)w.router.scales;
  p.router_b = (const uint16_t *)w.router.biases;
  p.experts = (const uint8_t *)w.experts;
  p.stride = w.expert_stride;
  p.shared = (const uint8_t *)w.shared;
  p.off = moe::Blob{w.layout.gate_q, w.layout.gate_s, w.layout.gate_b, w.layout.up_q,  w.layout.up_s,
                    w.layout.up_b,   w.layout.down_q, w.layout.down_s, w.layout.down_b};
  p.blob_bytes = blob_extent(w);
  p.logit_bias = w.logit_bias;
  p.router_scale = (const uint16_t *)w.router_scale;
  p.expert_scale = w.per_expert_scale;
  return p;
}

int check_weights(const moe_layer_weights *w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  int st = check_dims(&w->dims);
  if (st) return st;
  const void *ptrs[5] = {w->router.q, w->router.scales, w->router.biases, w->experts, w->shared};
  for (const void *p : ptrs)
    if (!p || !aligned(p, 16)) return MOE_ERR_INVALID_ARG;
  if (w->logit_bias && !aligned(w->logit_bias, 4)) return MOE_ERR_INVALID_ARG;
  if (w->router_scale && !aligned(w->router_scale, 16)) return MOE_ERR_INVALID_ARG;
  if (w->per_expert_scale && !aligned(w->per_expert_scale, 4)) return MOE_ERR_INVALID_ARG;
  if (w->post_norm && !aligned(w->post_norm, 16)) return MOE_ERR_INVALID_ARG;
  if (w->layer_scalar && !aligned(w->layer_scalar, 4)) return MOE_ERR_INVALID_ARG;
  const size_t offs[9] = {w->layout.gate_q, w->layout.gate_s, w->layout.gate_b, w->layout.up_q, w->layout.up_s,
                          w->layout.up_b,   w->layout.down_q, w->layout.down_s, w->layout.down_b};
  for (size_t o : offs)
    if (o % 256) return MOE_ERR_INVALID_ARG;
  if (w->expert_stride % 256 || w->expert_stride < blob_extent(*w)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool decode_fused_supported(const moe_dims &d, int n_sm) {
  if (d.n_experts > n_sm || n_sm > 1024) return false;
  const moe::Dims dd = to_dims(d, 1);
  return moe::fused_decode_smem(dd) <= kSmemCap && moe::decode_blocks_per_sm(dd) >= 1;
}

}  // namespace moe_abi

namespace {
using moe_abi::blob_extent;
using moe_abi::layer_ptrs;
int check_weights_impl(const moe_layer_weights *w) { return moe_abi::check_weights(w); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int check_head(const moe_head_weights *w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (w->hidden < 64 || w->hidden > 4096 || w->hidden % 64) return MOE_ERR_UNSUPPORTED;
  if (w->vocab < 16 || w->vocab % 16 || w->vocab > (1 << 28)) return MOE_ERR_UNSUPPORTED;
  const void *p[3] = {w->w.q, w->w.scales, w->w.biases};
  for (const void *q : p)
    if (!q || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int check_ws(const moe_dims &d, int T, const void *ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(d, T).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int run_router(moe_handle *h, const moe_layer_weights *w, int T, const void *x, void *hres, void *x_out,
               float *logits, int32_t *ids, float *wts, uint8_t *ws, cudaStream_t st, bool normalize) {
  const WsLayout L = ws_layout(w->dims, T);
  moe::RouterArgs a;
  a.w = layer_ptrs(*w);
  a.d = to_dims(w->dims, T);
  a.x = (const uint16_t *)x;
  a.hres = (uint16_t *)hres;
  a.xn = (uint16_t *)(ws + L.xn);
  a.xn_user = (uint16_t *)x_out;
  a.logits = logits ? logits : (float *)(ws + L.logits);
  a.ids_user = ids;
  a.wts_user = wts;
  a.r = routing_in(ws, L);
  a.counter = h->dwords + 1;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  a.normalize = normalize;
  a.prefetch_bytes_max = h->prefetch_max;
  return cuda_status(moe::launch_router(a, st, h->pdl));
}

// The fused single-token kernel needs one resident block per SM (grid
// barriers) and one router row per block.
bool use_fused(moe_handle *h, const moe_layer_weights *w, int T) {
  if (!h->fused || T != 1) return false;
  const int key[3] = {w->dims.hidden, w->dims.inter, w->dims.top_k};
  if (key[0] != h->fused_key[0] || key[1] != h->fused_key[1] || key[2] != h->fused_key[2]) {
    h->fused_ok = moe_abi::decode_fused_supported(w->dims, h->n_sm);
    memcpy(h->fused_key, key, sizeof(key));
  }
  return h->fused_ok != 0;
}

int run_fused(moe_handle *h, const moe_layer_weights *w, const void *x, void *hres, void *y, void *x_out,
              float *logits, int32_t *ids, float *wts, uint8_t *ws, cudaStream_t st, bool normalize) {
  const WsLayout L = ws_layout(w->dims, 1);
  moe::DecodeArgs a;
  a.w = layer_ptrs(*w);
  a.d = to_dims(w->dims, 1);
  a.x = (const uint16_t *)x;
  a.hres = (uint16_t *)hres;
  a.xn_user = (uint16_t *)x_out;
  a.logits = logits ? logits : (float *)(ws + L.logits);
  a.ids_user = ids;
  a.wts_user = wts;
  a.hbuf = (__half *)(ws + L.h);
  a.y = (uint16_t *)y;
  a.sync = h->dwords + kSyncOffset;
  a.mbox = reinterpret_cast<unsigned long long *>(h->dwords + kMboxOffset);
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  a.normalize = normalize;
  a.skip_block = h->skip_block_next;
  a.wait_ns = h->wait_ns_next ? h->wait_ns_next : moe::kWaitLimitNs;
  h->skip_block_next = -1;
  h->wait_ns_next = 0;
  return cuda_status(moe::launch_decode_fused(a, h->n_sm, st, h->pdl));
}

// The fused prefill kernel: one resident block per SM (grid barriers).
bool use_prefill(moe_handle *h, const moe_layer_weights *w, int T) {
  if (!h->prefill || T < 2 || h->n_sm > 1024) return false;
  const int key[4] = {w->dims.hidden, w->dims.inter, w->dims.n_experts, w->dims.top_k};
  if (memcmp(key, h->prefill_key, sizeof(key)) != 0) {
    const moe::Dims d = to_dims(w->dims, moe::kMaxTokens);
    h->prefill_ok = moe::prefill_fused_smem(d) != 0 && moe::prefill_blocks_per_sm(d) >= 1;
    memcpy(h->prefill_key, key, sizeof(key));
  }
  return h->prefill_ok != 0;
}

int run_prefill(moe_handle *h, const moe_layer_weights *w, int T, const void *x, void *hres, void *y, void *x_out,
                float *logits, int32_t *ids, float *wts, uint8_t *ws, cudaStream_t st, bool normalize) {
  const WsLayout L = ws_layout(w->dims, T);
  moe::PrefillArgs a;
  a.w = layer_ptrs(*w);
  a.d = to_dims(w->dims, T);
  a.x = (const uint16_t *)x;
  a.hres = (uint16_t *)hres;
  a.xn_user = (uint16_t *)x_out;
  a.logits = logits ? logits : (float *)(ws + L.logits);
  a.ids_user = ids;
  a.wts_user = wts;
  a.r = routing_in(ws, L);
  a.xperm = (__half *)(ws + L.xn);
  a.xs = (uint16_t *)(ws + L.xq);
  a.hperm = (__half *)(ws + L.h);
  a.hq = (float *)(ws + L.hq);
  a.obuf = (float *)(ws + L.o);
  a.y = (uint16_t *)y;
  a.sync = h->dwords + kPrefillSyncOffset;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  a.normalize = normalize;
  return cuda_status(moe::launch_prefill_fused(a, h->n_sm, st, h->pdl, h->prefill_dense));
}

int run_ffn(moe_handle *h, const moe_layer_weights *w, int T, const void *x, const moe::Routing &r, int include_shared,
            void *y, void *hres, uint8_t *ws, cudaStream_t st) {
  const WsLayout L = ws_layout(w->dims, T);
  moe::FfnArgs a;
  a.w = layer_ptrs(*w);
  a.d = to_dims(w->dims, T);
  a.x = (const uint16_t *)x;
  a.r = r;
  a.hbuf = (__half *)(ws + L.h);
  a.obuf = (float *)(ws + L.o);
  a.y = (uint16_t *)y;
  a.hres = (uint16_t *)hres;
  a.include_shared = include_shared;
  // W_down of the selected experts fits L2 comfortably only for small T
  a.prefetch_down = h->prefetch_max > 0 && (size_t)(w->dims.top_k * T + 1) * blob_extent(*w) <= (size_t)h->prefetch_max;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  cudaError_t e = moe::launch_gateup(a, st, h->pdl);
  a.trace = take_trace(h, 2);  // down (+ combine)
  if (e == cudaSuccess) e = moe::launch_down(a, st, h->pdl);
  return cuda_status(e);
}

}  // namespace

extern "C" {

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id out of range (skipped on the device)";
    case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite router logit or activation";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int moe_create(moe_handle **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  if (moe::router_set_attributes() != cudaSuccess || moe::ffn_set_attributes() != cudaSuccess ||
      moe::decode_set_attributes() != cudaSuccess || moe::prefill_set_attributes() != cudaSuccess ||
      moe::prompt_set_attributes() != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_handle *h = (moe_handle *)calloc(1, sizeof(moe_handle));
  if (!h) return MOE_ERR_CUDA;
  h->device = dev;
  h->n_sm = prop.multiProcessorCount;
  h->skip_block_next = -1;
  const char *fz = getenv("MOE_DECODE_FUSED");
  h->fused = !(fz && fz[0] == '0');
  const char *pz = getenv("MOE_PREFILL_FUSED");
  h->prefill = !(pz && pz[0] == '0');
  // the tcgen05 instance of the multi-token kernel for dense slots: opt-in
  // (MOE_PREFILL_DENSE=1); on the target workloads it is not yet faster than
  // the default instance
  const char *dz = getenv("MOE_PREFILL_DENSE");
  h->prefill_dense = dz && dz[0] == '1';
  if (cudaMalloc(&h->dwords, device_words(h->n_sm) * sizeof(unsigned)) != cudaSuccess) {
    free(h);
    return MOE_ERR_CUDA;
  }
  if (cudaMemset(h->dwords, 0, device_words(h->n_sm) * sizeof(unsigned)) != cudaSuccess) {
    cudaFree(h->dwords);
    free(h);
    return MOE_ERR_CUDA;
  }
  const char *pdl = getenv("MOE_PDL");
  h->pdl = !(pdl && pdl[0] == '0');
  const char *pf = getenv("MOE_L2_PREFETCH_MB");
  h->prefetch_max = pf ? atoi(pf) * (1 << 20) : 64 * (1 << 20);
  *out = h;
  return MOE_OK;
}

int moe_destroy(moe_handle *h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->copy_ready)
    for (int i = 0; i < moe_handle::kCopyStreams; ++i) {
      cudaStreamDestroy(h->copy_st[i]);
      cudaEventDestroy(h->copy_ev[i]);
    }
  const cudaError_t e = cudaFree(h->dwords);
  free(h);
  return cuda_status(e);
}

int moe_check_weights(const moe_layer_weights *w) { return check_weights_impl(w); }

size_t moe_workspace_bytes(const moe_dims *dims, int n_tokens) {
  if (check_dims(dims) != MOE_OK || check_tokens(n_tokens) != MOE_OK) return 0;
  return ws_layout(*dims, n_tokens).total;
}

int moe_router_topk(moe_handle *h, const void *x, int n_tokens, const moe_layer_weights *w, float *logits,
                    int32_t *ids, float *weights, void *ws, size_t ws_bytes, moe_stream_t stream) {
  if (!h || !x || !ids || !weights) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if ((st = check_tokens(n_tokens))) return st;
  if (!aligned(x, 16) || (logits && !aligned(logits, 16))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(w->dims, n_tokens, ws, ws_bytes))) return st;
  return run_router(h, w, n_tokens, x, nullptr, nullptr, logits, ids, weights, (uint8_t *)ws, (cudaStream_t)stream,
                    false);
}

int moe_route_sort(moe_handle *h, const int32_t *ids, int n_tokens, const moe_dims *dims, int32_t *counts,
                   int32_t *offsets, int32_t *perm, int32_t *pos, moe_stream_t stream) {
  if (!h || !ids || !counts || !offsets || !perm || !pos) return MOE_ERR_INVALID_ARG;
  int st = check_dims(dims);
  if (st) return st;
  if ((st = check_tokens(n_tokens))) return st;
  moe::SortArgs a;
  a.ids = ids;
  a.T = n_tokens;
  a.k = dims->top_k;
  a.E = dims->n_experts;
  memset(&a.r, 0, sizeof(a.r));
  a.r.counts = counts;
  a.r.offsets = offsets;
  a.r.perm = perm;
  a.r.pos = pos;
  a.include_shared = 0;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  return cuda_status(moe::launch_sort(a, (cudaStream_t)stream, h->pdl));
}

int moe_expert_ffn(moe_handle *h, const void *x, int n_tokens, const int32_t *ids, const float *weights,
                   const moe_layer_weights *w, int include_shared, void *y, void *ws, size_t ws_bytes,
                   moe_stream_t stream) {
  if (!h || !x || !ids || !weights || !y) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if ((st = check_tokens(n_tokens))) return st;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(w->dims, n_tokens, ws, ws_bytes))) return st;
  uint8_t *wsb = (uint8_t *)ws;
  const WsLayout L = ws_layout(w->dims, n_tokens);
  moe::Routing r = routing_in(wsb, L);
  r.ids = const_cast<int32_t *>(ids);
  r.wts = const_cast<float *>(weights);
  moe::SortArgs sa;
  sa.ids = ids;
  sa.T = n_tokens;
  sa.k = w->dims.top_k;
  sa.E = w->dims.n_experts;
  sa.r = r;
  sa.include_shared = include_shared ? 1 : 0;
  sa.err = h->dwords;
  sa.trace = take_trace(h, 1);
  cudaError_t e = moe::launch_sort(sa, (cudaStream_t)stream, h->pdl);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return run_ffn(h, w, n_tokens, x, r, include_shared ? 1 : 0, y, nullptr, wsb, (cudaStream_t)stream);
}

int moe_layer_forward(moe_handle *h, const void *x, int n_tokens, const moe_layer_weights *w, void *y,
                      int32_t *ids_out, float *logits_out, float *weights_out, void *ws, size_t ws_bytes,
                      moe_stream_t stream) {
  if (!h || !x || !y) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if ((st = check_tokens(n_tokens))) return st;
  if (!aligned(x, 16) || !aligned(y, 16) || (logits_out && !aligned(logits_out, 16))) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(w->dims, n_tokens, ws, ws_bytes))) return st;
  uint8_t *wsb = (uint8_t *)ws;
  if (use_fused(h, w, n_tokens))
    return run_fused(h, w, x, nullptr, y, nullptr, logits_out, ids_out, weights_out, wsb, (cudaStream_t)stream,
                     false);
  if (use_prefill(h, w, n_tokens))
    return run_prefill(h, w, n_tokens, x, nullptr, y, nullptr, logits_out, ids_out, weights_out, wsb,
                       (cudaStream_t)stream, false);
  if ((st = run_router(h, w, n_tokens, x, nullptr, nullptr, logits_out, ids_out, weights_out, wsb,
                       (cudaStream_t)stream, false)))
    return st;
  return run_ffn(h, w, n_tokens, x, routing_in(wsb, ws_layout(w->dims, n_tokens)), 1, y, nullptr, wsb,
                 (cudaStream_t)stream);
}

int moe_layer_forward_residual(moe_handle *h, void *hidden, int n_tokens, const moe_layer_weights *w, void *y_out,
                               void *x_out, int32_t *ids_out, float *logits_out, void *ws, size_t ws_bytes,
                               moe_stream_t stream) {
  if (!h || !hidden) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if ((st = check_tokens(n_tokens))) return st;
  if (!aligned(hidden, 16) || (y_out && !aligned(y_out, 16)) || (x_out && !aligned(x_out, 16)) ||
      (logits_out && !aligned(logits_out, 16)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(w->dims, n_tokens, ws, ws_bytes))) return st;
  uint8_t *wsb = (uint8_t *)ws;
  const WsLayout L = ws_layout(w->dims, n_tokens);
  const cudaStream_t s = (cudaStream_t)stream;
  // With a layer tail the block reads the residual stream as its input only
  // (x = hidden, normalised), writes y, and the tail launch updates hidden.
  const bool tail = w->post_norm != nullptr || w->layer_scalar != nullptr;
  void *res = tail ? nullptr : hidden;
  const void *xin = tail ? hidden : nullptr;
  void *yb = tail && !y_out ? (void *)(wsb + L.y) : y_out;
  if (use_fused(h, w, n_tokens))
    st = run_fused(h, w, xin, res, yb, x_out, logits_out, ids_out, nullptr, wsb, s, true);
  else if (use_prefill(h, w, n_tokens))
    st = run_prefill(h, w, n_tokens, xin, res, yb, x_out, logits_out, ids_out, nullptr, wsb, s, true);
  else if (!(st = run_router(h, w, n_tokens, xin, res, x_out, logits_out, ids_out, nullptr, wsb, s, true)))
    st = run_ffn(h, w, n_tokens, wsb + L.xn, routing_in(wsb, L), 1, yb, res, wsb, s);
  if (st || !tail) return st;
  moe::TailArgs ta;
  ta.y = (const uint16_t *)yb;
  ta.h = (uint16_t *)hidden;
  ta.post_norm = (const uint16_t *)w->post_norm;
  ta.layer_scalar = w->layer_scalar;
  ta.T = n_tokens;
  ta.H = w->dims.hidden;
  ta.trace = take_trace(h, 1);
  return cuda_status(moe::launch_tail(ta, s, h->pdl));
}

size_t moe_prompt_workspace_bytes(const moe_dims *dims, int n_rows) {
  if (check_dims(dims) != MOE_OK || n_rows < 1 || n_rows > moe::kPromptMaxRows) return 0;
  if (!moe::prompt_supported(to_dims(*dims, n_rows))) return 0;
  return prompt_ws(*dims, n_rows).total;
}

int moe_layer_forward_prompt(moe_handle *h, void *hidden, int n_rows, const moe_layer_weights *w, void *y_out,
                             void *x_out, int32_t *ids_out, float *logits_out, void *ws, size_t ws_bytes,
                             moe_stream_t stream) {
  if (!h || !hidden) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if (n_rows < 1 || n_rows > moe::kPromptMaxRows) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || (y_out && !aligned(y_out, 16)) || (x_out && !aligned(x_out, 16)) ||
      (logits_out && !aligned(logits_out, 16)))
    return MOE_ERR_INVALID_ARG;
  const moe::Dims d = to_dims(w->dims, n_rows);
  if (!moe::prompt_supported(d)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  const PromptWs L = prompt_ws(w->dims, n_rows);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  uint8_t *wsb = (uint8_t *)ws;
  const cudaStream_t s = (cudaStream_t)stream;
  // With a layer tail the combine writes y and the tail launch updates hidden.
  const bool tail = w->post_norm != nullptr || w->layer_scalar != nullptr;
  moe::PromptArgs a;
  memset(&a, 0, sizeof(a));
  a.w = layer_ptrs(*w);
  a.d = d;
  a.hres = (uint16_t *)hidden;
  a.xn = (uint16_t *)(wsb + L.xn);
  a.xn_user = (uint16_t *)x_out;
  a.logits = logits_out ? logits_out : (float *)(wsb + L.logits);
  a.ids_user = ids_out;
  a.r.ids = (int32_t *)(wsb + L.ids);
  a.r.wts = (float *)(wsb + L.wts);
  a.r.counts = (int32_t *)(wsb + L.counts);
  a.r.offsets = (int32_t *)(wsb + L.offsets);
  a.r.perm = (int32_t *)(wsb + L.perm);
  a.r.pos = (int32_t *)(wsb + L.pos);
  a.ch_e = (int32_t *)(wsb + L.ch_e);
  a.ch_beg = (int32_t *)(wsb + L.ch_beg);
  a.ch_cnt = (int32_t *)(wsb + L.ch_cnt);
  a.n_ch = (int32_t *)(wsb + L.n_ch);
  a.xg = (__half *)(wsb + L.xg);
  a.hg = (__half *)(wsb + L.hg);
  a.obuf = (float *)(wsb + L.o);
  a.err = h->dwords;
  a.trace = take_trace(h, 6);
  void *yb = tail && !y_out ? (void *)(wsb + L.y) : y_out;
  st = cuda_status(moe::launch_prompt(a, (uint16_t *)yb, !tail, h->n_sm, s, h->pdl));
  if (st || !tail) return st;
  moe::TailArgs ta;
  ta.y = (const uint16_t *)yb;
  ta.h = (uint16_t *)hidden;
  ta.post_norm = (const uint16_t *)w->post_norm;
  ta.layer_scalar = w->layer_scalar;
  ta.T = n_rows;
  ta.H = w->dims.hidden;
  ta.trace = take_trace(h, 1);
  return cuda_status(moe::launch_tail(ta, s, h->pdl));
}

int moe_layer_forward_stack(moe_handle *h, void *hidden, int n_layers, const moe_layer_weights *layers, void *ws,
                            size_t ws_bytes, moe_stream_t stream) {
  if (!h || !hidden || !layers || n_layers < 1) return MOE_ERR_INVALID_ARG;
  int st;
  for (int l = 0; l < n_layers; ++l) {
    if ((st = check_weights_impl(&layers[l]))) return st;
    if (memcmp(&layers[l].dims, &layers[0].dims, sizeof(moe_dims)) != 0) return MOE_ERR_INVALID_ARG;
  }
  for (int l = 0; l < n_layers; ++l)
    if ((st = moe_layer_forward_residual(h, hidden, 1, &layers[l], nullptr, nullptr, nullptr, nullptr, ws, ws_bytes,
                                         stream)))
      return st;
  return MOE_OK;
}

int moe_layer_forward_offload(moe_handle *h, moe_expert_cache *c, int layer, void *hidden,
                              const moe_layer_weights *w, void *slots, void *ws, size_t ws_bytes,
                              moe_stream_t stream) {
  if (!h || !c || !hidden || !w || !slots || !ws) return MOE_ERR_INVALID_ARG;
  int st = check_weights_impl(w);
  if (st) return st;
  if (w->post_norm || w->layer_scalar) return MOE_ERR_UNSUPPORTED;
  if (!aligned(hidden, 16) || !aligned(slots, 256)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(w->dims, 1, ws, ws_bytes))) return st;
  if (moe_cache_slot_expert(c, layer, 0) < -1) return MOE_ERR_INVALID_ARG;  // no such layer in the cache
  const int k = w->dims.top_k;
  if (k > moe::kMaxTopK || moe_cache_slots(c) < k || moe_cache_slots(c) > w->dims.n_experts) return MOE_ERR_UNSUPPORTED;
  uint8_t *wsb = (uint8_t *)ws;
  const WsLayout L = ws_layout(w->dims, 1);
  const cudaStream_t s = (cudaStream_t)stream;
  // cb1: rmsnorm + router + top-k (ids and weights into the workspace)
  if ((st = run_router(h, w, 1, nullptr, hidden, nullptr, nullptr, nullptr, nullptr, wsb, s, true))) return st;
  // the handoff: the ids to the host
  int32_t ids[moe::kMaxTopK], sl[moe::kMaxTopK], load_slots[moe::kMaxTopK], load_ids[moe::kMaxTopK];
  if (cudaMemcpyAsync(ids, wsb + L.ids, k * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  int n_loads = 0;
  if ((st = moe_cache_lookup(c, layer, ids, k, sl, load_slots, load_ids, &n_loads))) return st;
  // io: one copy per missing expert into its slot, spread over the copy
  // streams so distinct misses move in parallel ("no two reads write the
  // same slot": each slot appears once per step).  The layer's stream is idle
  // here (synchronised above), so no earlier work still reads these slots.
  if (!h->copy_ready) {
    for (int i = 0; i < moe_handle::kCopyStreams; ++i)
      if (cudaStreamCreateWithFlags(&h->copy_st[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&h->copy_ev[i], cudaEventDisableTiming) != cudaSuccess)
        return MOE_ERR_CUDA;
    h->copy_ready = true;
  }
  const size_t blob = blob_extent(*w);
  for (int i = 0; i < n_loads; ++i)
    if (load_ids[i] >= w->dims.n_experts) return MOE_ERR_BAD_EXPERT_ID;
  // Host memory the device can read (pinned and mapped): the GPU copies the
  // blobs itself (one launch, every blob in parallel); otherwise the copy
  // engines do, one copy per blob over the copy streams.
  cudaPointerAttributes pa;
  const bool mapped = (blob % 16) == 0 && cudaPointerGetAttributes(&pa, w->experts) == cudaSuccess &&
                      pa.type == cudaMemoryTypeHost && pa.devicePointer != nullptr &&
                      ((uintptr_t)pa.devicePointer % 16) == 0 && (w->expert_stride % 16) == 0;
  if (n_loads > 0 && mapped) {
    moe::FillArgs fa;
    fa.n = n_loads;
    fa.bytes = blob;
    for (int i = 0; i < n_loads; ++i) {
      fa.src[i] = (const uint8_t *)pa.devicePointer + (size_t)load_ids[i] * w->expert_stride;
      fa.dst[i] = (uint8_t *)slots + (size_t)load_slots[i] * w->expert_stride;
    }
    if (moe::launch_fill_slots(fa, s) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    for (int i = 0; i < n_loads; ++i)
      if (cudaMemcpyAsync((uint8_t *)slots + (size_t)load_slots[i] * w->expert_stride,
                          (const uint8_t *)w->experts + (size_t)load_ids[i] * w->expert_stride, blob,
                          cudaMemcpyHostToDevice, h->copy_st[i % moe_handle::kCopyStreams]) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (int i = 0; i < n_loads && i < moe_handle::kCopyStreams; ++i)
      if (cudaEventRecord(h->copy_ev[i], h->copy_st[i]) != cudaSuccess ||
          cudaStreamWaitEvent(s, h->copy_ev[i], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
  }
  // cb2: the ids relabelled by slot (the copy reads host memory that stays
  // valid: cudaMemcpyAsync from pageable memory returns once the data is staged)
  if (cudaMemcpyAsync(wsb + L.ids, sl, k * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_layer_weights wl = *w;
  wl.experts = slots;  // expert id = slot index from here on
  moe::Routing r = routing_in(wsb, L);
  moe::SortArgs sa;
  sa.ids = r.ids;
  sa.T = 1;
  sa.k = k;
  sa.E = w->dims.n_experts;
  sa.r = r;
  sa.include_shared = 1;
  sa.err = h->dwords;
  sa.trace = take_trace(h, 1);
  if (moe::launch_sort(sa, s, h->pdl) != cudaSuccess) return MOE_ERR_CUDA;
  return run_ffn(h, &wl, 1, wsb + L.xn, r, 1, nullptr, hidden, wsb, s);
}

int moe_head_forward(moe_handle *h, const void *x, int n_tokens, const moe_head_weights *w, float softcap,
                     float *logits, int32_t *tokens, moe_stream_t stream) {
  if (!h || !x || (!logits && !tokens)) return MOE_ERR_INVALID_ARG;
  int st = check_head(w);
  if (st) return st;
  if (n_tokens < 1 || n_tokens > moe::kHeadMaxTokens) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (logits && !aligned(logits, 4)) || (tokens && !aligned(tokens, 4)))
    return MOE_ERR_INVALID_ARG;
  if (!(softcap == softcap)) return MOE_ERR_INVALID_ARG;
  if (!h->head_ready) {
    if (moe::head_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    h->head_ready = true;
  }
  const int per_sm = moe::head_blocks_per_sm(w->hidden, n_tokens);
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  // the fewest warps that still give every warp the same number of 16-row units
  const long long n_units = w->vocab / 16, max_warps = (long long)h->n_sm * per_sm * 8;
  const long long per_warp = (n_units + max_warps - 1) / max_warps;
  const long long warps = (n_units + per_warp - 1) / per_warp;
  moe::HeadArgs a;
  a.x = (const uint16_t *)x;
  a.q = (const uint32_t *)w->w.q;
  a.s = (const uint16_t *)w->w.scales;
  a.b = (const uint16_t *)w->w.biases;
  a.logits = logits;
  a.out_bf16 = nullptr;
  a.tokens = tokens;
  a.best = reinterpret_cast<unsigned long long *>(h->dwords + kHeadStateOffset);
  a.counter = h->dwords + kHeadStateOffset + 2 * moe::kHeadMaxTokens;
  a.softcap = softcap;
  a.T = n_tokens;
  a.V = w->vocab;
  a.H = w->hidden;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  return cuda_status(moe::launch_head(a, (int)((warps + 7) / 8), (cudaStream_t)stream, h->pdl));
}

int moe_dense_forward(moe_handle *h, const void *x, int n_tokens, const moe_head_weights *w, void *y, float *y32,
                      moe_stream_t stream) {
  if (!h || !x || (!y && !y32)) return MOE_ERR_INVALID_ARG;
  int st = check_head(w);
  if (st) return st;
  if (n_tokens < 1 || n_tokens > moe::kHeadMaxTokens) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (y && !aligned(y, 2)) || (y32 && !aligned(y32, 4))) return MOE_ERR_INVALID_ARG;
  if (!h->head_ready) {
    if (moe::head_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    h->head_ready = true;
  }
  const int per_sm = moe::head_blocks_per_sm(w->hidden, n_tokens);
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  const long long n_units = w->vocab / 16, max_warps = (long long)h->n_sm * per_sm * 8;
  const long long per_warp = (n_units + max_warps - 1) / max_warps;
  const long long warps = (n_units + per_warp - 1) / per_warp;
  moe::HeadArgs a;
  a.x = (const uint16_t *)x;
  a.q = (const uint32_t *)w->w.q;
  a.s = (const uint16_t *)w->w.scales;
  a.b = (const uint16_t *)w->w.biases;
  a.logits = y32;
  a.out_bf16 = (uint16_t *)y;
  a.tokens = nullptr;  // no argmax: the greedy state is neither read nor written
  a.best = reinterpret_cast<unsigned long long *>(h->dwords + kHeadStateOffset);
  a.counter = h->dwords + kHeadStateOffset + 2 * moe::kHeadMaxTokens;
  a.softcap = 0.0f;
  a.T = n_tokens;
  a.V = w->vocab;
  a.H = w->hidden;
  a.err = h->dwords;
  a.trace = take_trace(h, 1);
  return cuda_status(moe::launch_head(a, (int)((warps + 7) / 8), (cudaStream_t)stream, h->pdl));
}

int moe_embed(moe_handle *h, const int32_t *ids, int n, const moe_head_weights *w, void *out, moe_stream_t stream) {
  if (!h || !ids || !out || n < 1) return MOE_ERR_INVALID_ARG;
  int st = check_head(w);
  if (st) return st;
  if (!aligned(ids, 4) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  moe::EmbedArgs a;
  a.ids = ids;
  a.q = (const uint32_t *)w->w.q;
  a.s = (const uint16_t *)w->w.scales;
  a.b = (const uint16_t *)w->w.biases;
  a.out = (uint16_t *)out;
  a.n = n;
  a.V = w->vocab;
  a.H = w->hidden;
  a.err = h->dwords;
  return cuda_status(moe::launch_embed(a, (cudaStream_t)stream, h->pdl));
}

int moe_set_trace(moe_handle *h, unsigned long long *buffer, int n_launches) {
  if (!h || (buffer && n_launches < 1) || (buffer && !aligned(buffer, 8))) return MOE_ERR_INVALID_ARG;
  h->trace = buffer;
  h->trace_groups = buffer ? n_launches : 0;
  h->trace_next = 0;
  return MOE_OK;
}

int moe_selftest_wait_timeout(moe_handle *h, unsigned long long limit_ns, moe_stream_t stream) {
  if (!h || limit_ns == 0 || limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_wait_timeout(h->dwords, limit_ns, (cudaStream_t)stream));
}

int moe_selftest_skip_arrival(moe_handle *h, int block, unsigned long long limit_ns) {
  if (!h || block < 0 || block >= h->n_sm || limit_ns == 0 || limit_ns > moe::kWaitLimitNs)
    return MOE_ERR_INVALID_ARG;
  h->skip_block_next = block;
  h->wait_ns_next = limit_ns;
  return MOE_OK;
}

int moe_get_error(moe_handle *h, int *status) {
  if (!h || !status) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpy(&bits, h->dwords, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  // After a timeout a launch may have left its grid-barrier counter short of
  // a whole number of grids (a block that never arrived), which would give
  // the next launch a stale epoch: with the device idle, every counter,
  // ticket and mailbox goes back to its initial zero state.
  const size_t clear = (bits & moe::kErrTimeout) ? device_words(h->n_sm) * sizeof(unsigned) : sizeof(unsigned);
  if (cudaMemset(h->dwords, 0, clear) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits & moe::kErrTimeout)
    *status = MOE_ERR_TIMEOUT;
  else if (bits & moe::kErrBadId)
    *status = MOE_ERR_BAD_EXPERT_ID;
  else if (bits & moe::kErrNonFinite)
    *status = MOE_ERR_NONFINITE;
  else
    *status = MOE_OK;
  return MOE_OK;
}

}  // extern "C"
