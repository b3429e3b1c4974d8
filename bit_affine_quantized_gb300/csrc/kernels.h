// Host-side launchers of the MoE kernels (defined next to each kernel).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

struct RouterArgs {
  LayerPtrs w;
  Dims d;
  const uint16_t *x;       // bf16 [T, H] block input (normalised first when normalize == 1 and hres is null)
  uint16_t *hres;          // nullable bf16 [T, H] residual stream (normalize == 1)
  uint16_t *xn;            // bf16 [T, H] normalised input out (normalize == 1)
  uint16_t *xn_user;       // nullable copy of xn
  float *logits;           // fp32 [T, E]
  int32_t *ids_user;       // nullable copies of the routing
  float *wts_user;
  Routing r;
  unsigned *counter;       // last-block ticket, zero between launches
  unsigned *err;
  unsigned long long *trace;  // nullable: 4 trace slots of this launch (common.cuh)
  int normalize;
  int prefetch_bytes_max;  // L2-prefetch the selected experts if their total fits
};

struct FfnArgs {
  LayerPtrs w;
  Dims d;
  const uint16_t *x;       // bf16 [T, H] block input
  Routing r;
  __half *hbuf;            // fp16 [T*k + T, I]
  float *obuf;             // fp32 [T*k + T, H] (grouped down path)
  uint16_t *y;             // nullable bf16 [T, H]
  uint16_t *hres;          // nullable bf16 [T, H]: hres <- bf16(hres + y)
  int include_shared;
  int prefetch_down;       // gate/up blocks warm L2 with the selected W_down
  unsigned *err;
  unsigned long long *trace;  // nullable: 4 trace slots of this launch (common.cuh)
};

struct SortArgs {
  const int32_t *ids;
  int T, k, E;
  Routing r;               // counts/offsets/perm/pos required; act_* nullable
  int include_shared;
  unsigned *err;
  unsigned long long *trace;  // nullable: 4 trace slots of this launch (common.cuh)
};

// Fused single-token layer (decode.cu): one persistent block per SM.
struct DecodeArgs {
  LayerPtrs w;
  Dims d;                   // T == 1
  const uint16_t *x;        // bf16 [H] block input (normalised first when normalize == 1 and hres is null)
  uint16_t *hres;           // nullable bf16 [H] residual stream (normalize == 1), updated in place
  uint16_t *xn_user;        // nullable: normalised input out
  float *logits;            // fp32 [E] (user buffer or workspace)
  int32_t *ids_user;        // nullable [k]
  float *wts_user;          // nullable [k]
  __half *hbuf;             // fp16 [k+1, I]: slot 0 shared, slot j+1 = j-th selected
  uint16_t *y;              // nullable bf16 [H]
  unsigned *sync;           // 64-bit grid barrier counter (this kernel's own)
  unsigned long long *mbox; // [grid][kMaxExperts] epoch-tagged logits, zero-initialised, this kernel's own
  unsigned *err;
  unsigned long long *trace;
  int normalize;
  // failure-detection hook: every bounded wait of the launch gives up after
  // wait_ns; block skip_block (-1: none) withholds its barrier-2 arrival
  int skip_block;
  unsigned long long wait_ns;
};

// Fused multi-token layer (prefill.cu): one persistent block per SM, 2 <= T <= 128.
struct PrefillArgs {
  LayerPtrs w;
  Dims d;
  const uint16_t *x;        // bf16 [T, H] block input (normalised first when normalize == 1 and hres is null)
  uint16_t *hres;           // nullable bf16 [T, H] residual stream (normalize == 1), updated in place
  uint16_t *xn_user;        // nullable: normalised input out
  float *logits;            // fp32 [T, E] (user buffer or workspace)
  int32_t *ids_user;        // nullable [T, k]
  float *wts_user;          // nullable [T, k]
  Routing r;                // ids, wts used
  __half *xperm;            // fp16 [T, H] permuted operand rows
  uint16_t *xs;             // bf16 [T][2][G rounded up to 16]: group sums of x, hi and lo parts
  __half *hperm;            // fp16 [T*k + T, I] permuted h rows per sorted position
  float *hq;                // fp32 [T*k + T, I/16] quarter sums of h
  float *obuf;              // fp32 [T*k + T, H] weighted expert outputs
  uint16_t *y;              // nullable bf16 [T, H]
  unsigned *sync;           // 64-bit grid barrier counter (this kernel's own)
  unsigned *err;
  unsigned long long *trace;
  int normalize;
};

// Layer tail (tail.cu): post-FFN norm, residual, layer scalar; one block per token.
struct TailArgs {
  const uint16_t *y;          // bf16 [T, H] block output
  uint16_t *h;                // bf16 [T, H] residual stream, updated in place
  const uint16_t *post_norm;  // nullable bf16 [H]: norm weight (null: no norm)
  const float *layer_scalar;  // nullable fp32 [1] (null: 1)
  int T, H;
  unsigned long long *trace;
};
cudaError_t launch_tail(const TailArgs &a, cudaStream_t st, bool pdl);

// Tied head and embedding (head.cu).
constexpr int kHeadMaxTokens = 8;
struct HeadArgs {
  const uint16_t *x;          // bf16 [T, H]
  const uint32_t *q;          // [V, H/8] packed 4-bit codes
  const uint16_t *s, *b;      // bf16 [V, H/64]
  float *logits;              // nullable fp32 [T, V]
  uint16_t *out_bf16;         // nullable bf16 [T, V]: the same values rounded to bf16
  int32_t *tokens;            // nullable [T]: greedy token ids
  unsigned long long *best;   // [8] packed (logit, id) maxima: zero between launches
  unsigned *counter;          // finished-block ticket: zero between launches
  float softcap;              // <= 0: none
  int T, V, H;
  unsigned *err;
  unsigned long long *trace;
};
struct EmbedArgs {
  const int32_t *ids;         // [n]
  const uint32_t *q;
  const uint16_t *s, *b;
  uint16_t *out;              // bf16 [n, H]
  int n, V, H;
  unsigned *err;
};
size_t head_smem(int H, int T);
cudaError_t head_set_attributes();
int head_blocks_per_sm(int H, int T);
cudaError_t launch_head(const HeadArgs &a, int n_blocks, cudaStream_t st, bool pdl);
cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t st, bool pdl);

size_t prefill_fused_smem(const Dims &d);  // 0: shape not supported
int prefill_blocks_per_sm(const Dims &d);
cudaError_t prefill_set_attributes();
// allow_dense: slots with many rows in the chunk may take the tcgen05 path
cudaError_t launch_prefill_fused(const PrefillArgs &a, int n_blocks, cudaStream_t st, bool pdl, bool allow_dense);

size_t fused_decode_smem(const Dims &d);
int decode_blocks_per_sm(const Dims &d);
cudaError_t decode_set_attributes();
cudaError_t launch_decode_fused(const DecodeArgs &a, int n_blocks, cudaStream_t st, bool pdl);

// Expert offload: copy whole blobs from device-mapped host memory into slots.
constexpr int kMaxFill = 16;
struct FillArgs {
  const void *src[kMaxFill];  // device-side addresses of the host blobs (16-byte aligned)
  void *dst[kMaxFill];        // slots
  size_t bytes;               // per blob, a multiple of 16
  int n;
};
cudaError_t launch_fill_slots(const FillArgs &a, cudaStream_t st);

// Whole-prompt layer (prompt.cu): up to kPromptMaxRows rows through one
// layer; the expert work in chunks of at most kPromptChunk rows of one expert
// (the N of one tcgen05.mma).
constexpr int kPromptMaxRows = 4096;
constexpr int kPromptChunk = 256;
struct PromptArgs {
  LayerPtrs w;
  Dims d;                   // T = the prompt's rows
  uint16_t *hres;           // bf16 [T, H] residual stream, updated in place
  uint16_t *xn;             // bf16 [T, H] normalised rows
  uint16_t *xn_user;        // nullable copy of xn
  float *logits;            // fp32 [T, E] (user buffer or workspace)
  int32_t *ids_user;        // nullable [T, k]
  float *wts_user;          // nullable [T, k]
  Routing r;                // ids, wts, counts, offsets, perm, pos
  int32_t *ch_e;            // [prompt_max_chunks] expert of each chunk (kSharedSlot: shared)
  int32_t *ch_beg;          // first sorted position of the chunk
  int32_t *ch_cnt;          // rows of the chunk (1 .. kPromptChunk)
  int32_t *n_ch;            // [1] chunks
  __half *xg;               // fp16 [T*k + T, H] operand rows per sorted position
  __half *hg;               // fp16 [T*k + T, I] h rows per sorted position (operand order)
  float *obuf;              // fp32 [T*k + T, H] weighted expert outputs
  unsigned *err;
  unsigned long long *trace;  // nullable: 6 launches x 4 slots
};
int prompt_max_chunks(int T, int k, int E);
bool prompt_supported(const Dims &d);
cudaError_t prompt_set_attributes();
// router, grouping, gather, gate/up GEMM, down GEMM, combine (6 launches);
// the combine writes y (nullable) and, if add_residual, hres <- bf16(hres + y)
cudaError_t launch_prompt(const PromptArgs &a, uint16_t *y, bool add_residual, int n_sm, cudaStream_t st, bool pdl);

// smem budgets (bytes) for a given shape; 0 = shape not supported by that kernel
size_t router_smem(const Dims &d, int tb);
size_t gateup_smem(const Dims &d, int tt);
size_t down_decode_smem(const Dims &d);
size_t down_grouped_smem(const Dims &d);

cudaError_t router_set_attributes();
cudaError_t ffn_set_attributes();
cudaError_t launch_router(const RouterArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_sort(const SortArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_gateup(const FfnArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_down(const FfnArgs &a, cudaStream_t st, bool pdl);
// y[t] = sum of the token's weighted expert outputs (obuf) + the shared row; T blocks
cudaError_t launch_combine(const FfnArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_wait_timeout(unsigned *err, unsigned long long limit_ns, cudaStream_t st);
bool use_down_decode(const Dims &d);

// generic launch with optional programmatic dependent launch
template <typename Kern, typename Arg>
cudaError_t launch_k(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, const Arg &arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

}  // namespace moe
