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
// library routine.  moe_static_get_error reads (and clears) its error word.
#include <mutex>

#include "abi_internal.h"
#include "kernels.h"
#include "moe.h"

namespace {

// Scratch shared by every call on a device (it lives until the process exits):
//   [0, 256)      device error word (accumulates until moe_static_get_error)
//   [256, 512)    grid-barrier arrival counter (zero at load; it only grows:
//                 its value gives each launch the epoch that tags its logits)
//   [512, 1024)   logits when the caller passes none: fp32 [E], E <= 128
//   [1024, 16 KiB) expert activations h: fp16 [(top_k + 1) * inter]
//                  (the target model, top-8 of inter 704, needs 12,672 B)
constexpr size_t kScratchBytes = 16 * 1024;
constexpr size_t kErrOff = 0, kBarOff = 256, kLogitsOff = 512, kHOff = 1024;
__device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];
// logit mailboxes of the fused kernel: [grid][128] epoch-tagged 64-bit words
// (160 KiB: devices with up to 160 multiprocessors)
constexpr int kMaxStaticSm = 160;
__device__ __align__(256) unsigned long long g_static_mbox[kMaxStaticSm * moe::kMaxExperts];

// The arrays' names are host-side stand-ins in host code: their device
// addresses are looked up once per device, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char *g_scratch_ptr[kMaxDevices];
unsigned long long *g_mbox_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

int setup_device(int dev) {
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
    if (moe::decode_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    g_mbox_ptr[dev] = static_cast<unsigned long long *>(mb);
    g_sm_count[dev] = sms;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
  }
  return MOE_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int moe_layer_forward_static(const void *x, const moe_layer_weights *w, void *y, int32_t *ids_out,
                                        float *logits_out, float *weights_out, moe_stream_t stream) {
  if (!x || !y || !w) return MOE_ERR_INVALID_ARG;
  int st = moe_abi::check_weights(w);
  if (st != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(y) || (logits_out && !aligned16(logits_out))) return MOE_ERR_INVALID_ARG;
  // sizes beyond the static scratch are rejected
  const size_t h_bytes = (size_t)(w->dims.top_k + 1) * w->dims.inter * 2;
  if (h_bytes > kScratchBytes - kHOff || (size_t)w->dims.n_experts * 4 > kHOff - kLogitsOff)
    return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = setup_device(dev)) != MOE_OK) return st;
  const int n_sm = g_sm_count[dev];
  unsigned char *scratch = g_scratch_ptr[dev];
  // the fused kernel's own limits (one router row per block, one block per
  // SM) and the size of the mailbox array
  if (n_sm > kMaxStaticSm || !moe_abi::decode_fused_supported(w->dims, n_sm)) return MOE_ERR_UNSUPPORTED;

  moe::DecodeArgs a;
  a.w = moe_abi::layer_ptrs(*w);
  a.d = moe::Dims{w->dims.hidden, w->dims.inter, w->dims.n_experts, w->dims.top_k, 1};
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
  a.skip_block = -1;
  a.wait_ns = moe::kWaitLimitNs;
  return moe::launch_decode_fused(a, n_sm, (cudaStream_t)stream, true) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_static_get_error(int *status) {
  if (!status) return MOE_ERR_INVALID_ARG;
  *status = MOE_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  unsigned char *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    scratch = g_scratch_ptr[dev];
  }
  if (!scratch) return MOE_OK;  // no static call has run on this device
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpy(&bits, scratch + kErrOff, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(scratch + kErrOff, 0, sizeof(unsigned)) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits & moe::kErrTimeout) {
    // a launch that timed out may have left the barrier counter short of a
    // whole grid: with the device idle, counter and mailboxes go back to zero
    if (cudaMemset(scratch + kBarOff, 0, kLogitsOff - kBarOff) != cudaSuccess ||
        cudaMemset(g_mbox_ptr[dev], 0, sizeof(g_static_mbox)) != cudaSuccess)
      return MOE_ERR_CUDA;
    *status = MOE_ERR_TIMEOUT;
  } else if (bits & moe::kErrBadId) {
    *status = MOE_ERR_BAD_EXPERT_ID;
  } else if (bits & moe::kErrNonFinite) {
    *status = MOE_ERR_NONFINITE;
  }
  return MOE_OK;
}
