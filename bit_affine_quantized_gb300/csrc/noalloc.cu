// moe_layer_forward_static: the single-token layer call for callers that
// cannot allocate device memory.
//
// Some host programs hand the whole device memory to their own pool, or run
// the per-token loop where an allocation would stall the device (cudaMalloc
// can synchronise) and is not capturable.  They still pass inputs, weights
// and outputs, but cannot give this library a workspace or create a handle.
// This entry point keeps the scratch of the fused single-token kernel (the
// expert activations h, the logits when the caller passes none, the grid
// barrier counter, the logit mailboxes and the device error word) in
// file-scope device arrays and calls no cudaMalloc, cudaFree or allocating
// library routine.
#include <mutex>

#include "kernels.h"
#include "moe.h"

namespace {

// Scratch shared by every call on a device (it lives until the process exits):
//   [0, 256)      device error word (cleared by every call, not reported)
//   [256, 512)    grid-barrier arrival counter (zero at load; it only grows:
//                 its value gives each launch the epoch that tags its logits)
//   [512, 1024)   logits when the caller passes none: fp32 [E], E <= 128
//   [1024, 16 KiB) expert activations h: fp16 [(top_k + 1) * inter]
//                  (the target model, top-8 of inter 704, needs 12,672 B)
constexpr size_t kScratchBytes = 16 * 1024;
constexpr size_t kErrOff = 0, kBarOff = 256, kLogitsOff = 512, kHOff = 1024;
__device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];
// logit mailboxes of the fused kernel: [grid][128] epoch-tagged 64-bit words
constexpr int kMaxStaticSm = 160;
__device__ __align__(256) unsigned long long g_static_mbox[kMaxStaticSm * moe::kMaxExperts];

// The array's name is a host-side stand-in in host code: its device address
// is looked up once per device, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char *g_scratch_ptr[kMaxDevices];
unsigned long long *g_mbox_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

int setup_device(int dev, unsigned char **ptr, int *n_sm) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    void *mb = nullptr;
    if (cudaGetSymbolAddress(&mb, g_static_mbox) != cudaSuccess || !mb) return MOE_ERR_CUDA;
    g_mbox_ptr[dev] = static_cast<unsigned long long *>(mb);
    if (moe::decode_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    g_sm_count[dev] = sms;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *ptr = g_scratch_ptr[dev];
  *n_sm = g_sm_count[dev];
  return MOE_OK;
}

size_t extent(const moe_layer_weights &w) {
  const size_t H = w.dims.hidden, I = w.dims.inter;
  const size_t q = I * H / 2, sb = I * (H / 64) * 2;
  const size_t e[9] = {w.layout.gate_q + q, w.layout.gate_s + sb, w.layout.gate_b + sb,
                       w.layout.up_q + q,   w.layout.up_s + sb,   w.layout.up_b + sb,
                       w.layout.down_q + q, w.layout.down_s + sb, w.layout.down_b + sb};
  size_t m = 0;
  for (size_t v : e) m = v > m ? v : m;
  return m;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int moe_layer_forward_static(const void *x, const moe_layer_weights *w, void *y, int32_t *ids_out,
                                        float *logits_out, float *weights_out, moe_stream_t stream) {
  if (!x || !y || !w) return MOE_ERR_INVALID_ARG;
  int st = moe_check_weights(w);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(y) || (logits_out && !aligned16(logits_out))) return MOE_ERR_INVALID_ARG;
  // sizes beyond the static scratch are rejected
  const size_t h_bytes = (size_t)(w->dims.top_k + 1) * w->dims.inter * 2;
  if (h_bytes > kScratchBytes - kHOff || (size_t)w->dims.n_experts * 4 > kHOff - kLogitsOff)
    return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned char *scratch = nullptr;
  int n_sm = 0;
  if ((st = setup_device(dev, &scratch, &n_sm)) != MOE_OK) return st;
  const moe::Dims d{w->dims.hidden, w->dims.inter, w->dims.n_experts, w->dims.top_k, 1};
  // the fused kernel's own limits: one router row per block, one block per SM
  if (w->dims.n_experts > n_sm || n_sm > kMaxStaticSm || moe::fused_decode_smem(d) > 227 * 1024 ||
      moe::decode_blocks_per_sm(d) < 1)
    return MOE_ERR_UNSUPPORTED;

  // the error word starts at zero for every call
  if (cudaMemsetAsync(scratch + kErrOff, 0, kBarOff - kErrOff, (cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;

  moe::DecodeArgs a;
  a.w.router_q = (const uint8_t *)w->router.q;
  a.w.router_s = (const uint16_t *)w->router.scales;
  a.w.router_b = (const uint16_t *)w->router.biases;
  a.w.experts = (const uint8_t *)w->experts;
  a.w.stride = w->expert_stride;
  a.w.shared = (const uint8_t *)w->shared;
  a.w.off = moe::Blob{w->layout.gate_q, w->layout.gate_s, w->layout.gate_b, w->layout.up_q,  w->layout.up_s,
                      w->layout.up_b,   w->layout.down_q, w->layout.down_s, w->layout.down_b};
  a.w.blob_bytes = extent(*w);
  a.w.logit_bias = w->logit_bias;
  a.w.router_scale = (const uint16_t *)w->router_scale;
  a.w.expert_scale = w->per_expert_scale;
  a.d = d;
  a.x = (const uint16_t *)x;
  a.hres = nullptr;
  a.xn_user = nullptr;
  a.logits = logits_out ? logits_out : reinterpret_cast<float *>(scratch + kLogitsOff);
  a.ids_user = ids_out;
  a.wts_user = weights_out;
  a.hbuf = reinterpret_cast<__half *>(scratch + kHOff);
  a.y = (uint16_t *)y;
  a.sync = reinterpret_cast<unsigned *>(scratch + kBarOff);
  a.mbox = g_mbox_ptr[dev];
  a.err = reinterpret_cast<unsigned *>(scratch + kErrOff);
  a.trace = nullptr;
  a.normalize = 0;
  return moe::launch_decode_fused(a, n_sm, (cudaStream_t)stream, true) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
