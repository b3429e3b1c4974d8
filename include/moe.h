/*
 * moe.h - C ABI of the GB300 (sm_103a) mixture-of-experts FFN block with
 * MLX-style group-64 affine quantised weights.
 *
 * The block (page "TurboFieldfare - System design"):
 *   1. router: logits[t, e] = sum_k W_r[e, k] x[t, k], W_r 8-bit affine,
 *      no softcap (section "Why the runtime has this shape"; section
 *      "Decode", router description);
 *   2. top-k (k = 8 of E = 128) with ties to the lower expert id, softmax
 *      over the k selected logits (section "Decode");
 *   3. per selected expert a 4-bit affine GeGLU FFN
 *      o = W_down (gelu_tanh(W_gate x) * (W_up x)) (section "Metal
 *      execution": fused affine decode + GeGLU + weighted reduction);
 *   4. y = sum_j w_j o_j + o_shared, the dense shared expert added with no
 *      routing weight (section "Why the runtime has this shape").
 * Prefill handles chunks of at most 128 rows (section "Prefill"), so every
 * call takes 1 <= n_tokens <= 128.
 *
 * Quantised matrix format (section "Why the runtime has this shape"): a
 * matrix W[N, K] is three arrays
 *   q      : packed codes, row-major, little-endian uint32 words; code i of a
 *            row at bits 4*(i%8) of word i/8 (4-bit) or 8*(i%4) of word i/4
 *            (8-bit, i.e. plain byte order);
 *   scales : bf16 [N, K/64], row-major;
 *   biases : bf16 [N, K/64], row-major;
 * and W[n, k] = q[n, k] * scales[n, k/64] + biases[n, k/64].
 *
 * Expert storage (section ".gturbo directory": fixed-stride, page-aligned
 * expert blobs whose sub-tensors sit at their own offsets): routed expert e
 * is the blob at experts + e * expert_stride; inside a blob the nine
 * sub-tensors (gate/up [I, H], down [H, I]; q, scales, biases each) sit at
 * the byte offsets of moe_blob_layout.  The shared expert is one more blob
 * with the same layout.
 *
 * Conventions for every call
 *   - Returns MOE_OK (0) or a MOE_ERR_* code; nothing throws across the ABI.
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never frees them.  The workspace `ws` is caller-owned device
 *     memory of at least moe_workspace_bytes() bytes, 256-byte aligned, and
 *     must not be shared by calls that may run concurrently.
 *   - Launches are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream); no call synchronises the host except
 *     moe_get_error.  Inputs must stay valid until the stream reaches the
 *     call.
 *   - Arguments are checked on the host before anything is launched:
 *     null pointers, n_tokens outside [1, 128], dims the kernels do not
 *     support, pointers not 16-byte aligned (tensor data) or offsets not
 *     256-byte aligned -> MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED and no
 *     launch.  Faults found on the device (an expert id out of range in
 *     moe_expert_ffn / moe_route_sort, non-finite router logits) never trap:
 *     the offending item is skipped and a device error word is set, read
 *     back by moe_get_error.
 *   - A handle may be used from one stream at a time (it owns the device
 *     error word and the router's completion counter).
 *   - The layer calls run one persistent launch per layer (one block per
 *     SM, blocks that wait for one another at grid barriers).  Their blocks
 *     must all be resident at once: while such a call runs, no other work
 *     may hold SMs of the device (a kernel on another stream, another
 *     process under MPS, a green context).  Otherwise blocks wait at a
 *     barrier until the bounded wait (2 s) gives up, the call records
 *     MOE_ERR_TIMEOUT and its outputs are not valid; moe_get_error then
 *     reports the timeout and restores the barrier state for the next call.
 *     Handles created with MOE_DECODE_FUSED=0 / MOE_PREFILL_FUSED=0 in the
 *     environment run separate launches that never wait for one another.
 */
#ifndef MOE_AFFINE_H
#define MOE_AFFINE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* == cudaStream_t */

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size or alignment          */
  MOE_ERR_UNSUPPORTED = 2,   /* dims outside what the kernels implement       */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed                    */
  MOE_ERR_BAD_EXPERT_ID = 4, /* device: expert id outside [0, E) was skipped  */
  MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up                */
  MOE_ERR_NONFINITE = 6,     /* device: a router logit was NaN or infinite    */
  MOE_ERR_WORKSPACE = 7      /* workspace smaller than moe_workspace_bytes    */
};

/* Shapes.  Supported: group == 64; hidden, inter multiples of 64 with
 * 64 <= hidden <= 4096 and 64 <= inter <= 2048; 1 <= top_k <= 8;
 * top_k <= n_experts <= 128.  The target workload is hidden 2816,
 * inter 704, 128 experts, top-8. */
typedef struct {
  int hidden;    /* H: model width, input/output features of the block      */
  int inter;     /* I: expert intermediate width                            */
  int n_experts; /* E: routed experts                                       */
  int top_k;     /* k: experts selected per token                           */
  int group;     /* quantisation group along K; must be 64                  */
} moe_dims;

/* One quantised matrix: device pointers to codes, scales, biases. */
typedef struct {
  const void *q;
  const void *scales;
  const void *biases;
} moe_qmat;

/* Byte offsets of the nine sub-tensors inside one expert blob; each must be
 * a multiple of 256. */
typedef struct {
  size_t gate_q, gate_s, gate_b;
  size_t up_q, up_s, up_b;
  size_t down_q, down_s, down_b;
} moe_blob_layout;

/* Weights of one MoE layer (all device pointers). */
typedef struct {
  moe_dims dims;
  moe_qmat router;          /* 8-bit [E, H]                                   */
  const void *experts;      /* E routed blobs, fixed stride                   */
  size_t expert_stride;     /* bytes between blobs; multiple of 256           */
  moe_blob_layout layout;   /* sub-tensor offsets (routed and shared blobs)   */
  const void *shared;       /* the shared expert's blob                       */
  const float *logit_bias;  /* nullable [E]: added to the logits before top-k */
  /* The router's learned scales (section "Decode", router description),
   * both nullable (null: identity):
   *   router_scale      bf16 [H], 16-byte aligned: the router projects
   *                     x * router_scale / sqrt(H) instead of x (the experts
   *                     still take x);
   *   per_expert_scale  fp32 [E]: the routing weight of a selected expert e
   *                     is softmax(...) * per_expert_scale[e]. */
  const void *router_scale;
  const float *per_expert_scale;
  /* The layer tail (section "Decode", cb2 phase: post-FFN norm, residual,
   * learned layer scalar), both nullable; read only by the residual calls
   * (moe_layer_forward_residual, moe_layer_forward_stack):
   *   post_norm     bf16 [H], 16-byte aligned: norm weight g of
   *                 z = bf16(y / sqrt(mean(y^2) + 1e-6) * g) (null: z = y);
   *   layer_scalar  fp32 [1] on the device: h <- bf16(layer_scalar * bf16(h + z))
   *                 (null: h <- bf16(h + z)). */
  const void *post_norm;
  const float *layer_scalar;
} moe_layer_weights;

typedef struct moe_handle moe_handle;

/* Human-readable name of a status code (static string). */
const char *moe_status_string(int status);

/* Create / destroy a handle on the current CUDA device.  moe_create
 * allocates a few bytes of device memory (error word, counters) and sets
 * kernel attributes; it is the only call that allocates. */
int moe_create(moe_handle **out);
int moe_destroy(moe_handle *h);

/* Host-side validation of a layer description (no device access). */
int moe_check_weights(const moe_layer_weights *w);

/* Workspace bytes needed by moe_router_topk / moe_expert_ffn /
 * moe_layer_forward / moe_layer_forward_residual for n_tokens rows;
 * 0 if dims are unsupported or n_tokens is outside [1, 128]. */
size_t moe_workspace_bytes(const moe_dims *dims, int n_tokens);

/* Steps 1-2 (router projection, top-k, softmax weights).
 *   x        bf16 [T, H] row-major, the block input (already normalised)
 *   logits   nullable fp32 [T, E]: raw logits + logit_bias
 *   ids      int32 [T, k]: selected experts, by descending logit, ties to
 *            the lower id
 *   weights  fp32 [T, k]: softmax over the selected logits
 * Also leaves the token->expert grouping of step 3 in the workspace. */
int moe_router_topk(moe_handle *h, const void *x, int n_tokens, const moe_layer_weights *w,
                    float *logits, int32_t *ids, float *weights, void *ws, size_t ws_bytes,
                    moe_stream_t stream);

/* Step 3 on its own: stable counting sort of the pairs p = t*k + j by
 * expert id (section "Prefill": token/expert pairs grouped per expert).
 *   ids      int32 [T, k] device
 *   counts   int32 [E]       pairs per expert
 *   offsets  int32 [E + 1]   exclusive prefix sums of counts
 *   perm     int32 [T*k]     pair index at each sorted position
 *   pos      int32 [T*k]     sorted position of each pair (-1 if its id was
 *                            out of range; such pairs are dropped and
 *                            MOE_ERR_BAD_EXPERT_ID is recorded)
 * Runs one thread block; needs no workspace. */
int moe_route_sort(moe_handle *h, const int32_t *ids, int n_tokens, const moe_dims *dims,
                   int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *pos,
                   moe_stream_t stream);

/* Steps 3-4 with caller-given routing (e.g. forced ids).
 *   x        bf16 [T, H];  ids int32 [T, k];  weights fp32 [T, k]
 *   include_shared  1: add the shared expert; 0: routed sum only
 *   y        bf16 [T, H] output
 * Out-of-range ids are skipped on the device (MOE_ERR_BAD_EXPERT_ID). */
int moe_expert_ffn(moe_handle *h, const void *x, int n_tokens, const int32_t *ids,
                   const float *weights, const moe_layer_weights *w, int include_shared, void *y,
                   void *ws, size_t ws_bytes, moe_stream_t stream);

/* The whole block, steps 1-4: y = MoE(x).
 *   x bf16 [T, H] in;  y bf16 [T, H] out;
 *   ids_out (int32 [T, k]), logits_out (fp32 [T, E]), weights_out
 *   (fp32 [T, k]) are nullable copies of the routing. */
int moe_layer_forward(moe_handle *h, const void *x, int n_tokens, const moe_layer_weights *w,
                      void *y, int32_t *ids_out, float *logits_out, float *weights_out, void *ws,
                      size_t ws_bytes, moe_stream_t stream);

/* One layer of a residual stack (the decode/prefill harness around the
 * block): x = bf16(h / sqrt(mean(h^2) + 1e-6)) (rmsnorm without scale, as
 * the router's input normalisation in section "Decode"); y = MoE(x);
 * h <- bf16(h + y) in place.  With a layer tail in w (post_norm and/or
 * layer_scalar set), h <- bf16(lambda * bf16(h + bf16(g * y / rms(y))))
 * instead, by one more launch after the block.
 *   hidden   bf16 [T, H] in/out
 *   y_out    nullable bf16 [T, H]: the block output before the add (and
 *            before the tail)
 *   x_out    nullable bf16 [T, H]: the normalised block input */
int moe_layer_forward_residual(moe_handle *h, void *hidden, int n_tokens,
                               const moe_layer_weights *w, void *y_out, void *x_out,
                               int32_t *ids_out, float *logits_out, void *ws, size_t ws_bytes,
                               moe_stream_t stream);

/* ---- whole-prompt layer (section "Prefill": layer-major execution; the
 * token/expert pairs grouped into bounded routed-MoE work; experts streamed
 * in tiles of at most eight, the next tile fetched while the current tile's
 * work is queued; shared and routed branches combined before the tail).
 *
 * The same function as moe_layer_forward_residual, for a prompt of up to
 * MOE_PROMPT_MAX_ROWS rows in one call:
 *   hidden <- bf16(hidden + MoE(rmsnorm(hidden)))   (or the layer's tail)
 * row by row.  Rows are routed independently; all rows' token/expert pairs
 * are grouped per expert and cut into chunks of at most 256 rows of one
 * expert, and every (chunk, 128 weight rows) is one unit of a persistent
 * tensor-core GEMM (tcgen05.mma, weights dequantised once per unit into fp16
 * on chip: w = q * s + b rounded once to fp16).  Units run the shared
 * expert first, then experts in ascending id, i.e. tile after tile of eight
 * experts, so an expert's weights come from HBM about once per layer and
 * its later chunks read them from L2; each SM prefetches its next unit's
 * weights into L2 while the current one runs.
 *   hidden    bf16 [n_rows, H] in/out
 *   n_rows    1 <= n_rows <= MOE_PROMPT_MAX_ROWS
 *   y_out, x_out, ids_out, logits_out: nullable, as in
 *             moe_layer_forward_residual ([n_rows, ...])
 *   ws        moe_prompt_workspace_bytes(dims, n_rows) bytes, 256-aligned
 *             (about 0.7 GB at 4096 rows of the target shape: the operand,
 *             h and fp32 expert-output rows of every sorted position)
 * Six launches (router, grouping, operand gather, gate/up GEMM, down GEMM,
 * combine; a seventh for a layer tail), none of which waits for another
 * block, so the call may share the device.  Errors as for the other layer
 * calls; MOE_ERR_UNSUPPORTED when the shape's tiles do not fit on chip.
 * Capturable in a CUDA graph (the tensor maps are kernel parameters). */
#define MOE_PROMPT_MAX_ROWS 4096
size_t moe_prompt_workspace_bytes(const moe_dims *dims, int n_rows);
int moe_layer_forward_prompt(moe_handle *h, void *hidden, int n_rows, const moe_layer_weights *w,
                             void *y_out, void *x_out, int32_t *ids_out, float *logits_out,
                             void *ws, size_t ws_bytes, moe_stream_t stream);

/* n_layers single-token layers of a residual stack in one call (the decode
 * step of the section "Decode": every layer's router input is the residual
 * stream normalised, its block output is added back):
 *   for l in 0 .. n_layers-1:  hidden <- bf16(hidden + MoE_l(rmsnorm(hidden)))
 * (or layer l's tail around it, as in moe_layer_forward_residual)
 * with MoE_l the block of layers[l] (all with the same dims); the same
 * launches as n_layers calls of moe_layer_forward_residual with n_tokens = 1.
 *   hidden   bf16 [H] in/out;  layers: host array of n_layers weight sets;
 *   ws       workspace of moe_workspace_bytes(dims, 1)
 * Validates every layer before the first launch; capturable. */
int moe_layer_forward_stack(moe_handle *h, void *hidden, int n_layers, const moe_layer_weights *layers,
                            void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---- Expert offload (sections "Resource split", "Load and ownership" and
 * "Decode": every opened layer owns 16 routed-expert slots; after the router
 * (cb1) the host looks the selected experts up in the layer's cache, fills
 * only the missing slots (io), then the routed branch runs on the slots
 * (cb2); eviction is least frequently used, recency breaking ties).  Here
 * the routed experts stay in pinned host memory and the slots are device
 * memory, filled over the host link.
 *
 * moe_expert_cache is the host-side policy state of n_layers layers of
 * n_slots slots each (n_slots <= MOE_CACHE_MAX_SLOTS); it owns no device
 * memory.  Readings of the policy: an expert's use count starts at 1 when it
 * enters a slot and grows by 1 at each step that selects it; recency is the
 * step of its last selection; empty slots are taken first (lowest index);
 * a step's own experts are never evicted by its misses; remaining ties go to
 * the lower slot. */
#define MOE_CACHE_MAX_SLOTS 64
typedef struct moe_expert_cache moe_expert_cache;
int moe_cache_create(int n_layers, int n_slots, moe_expert_cache **out);
void moe_cache_destroy(moe_expert_cache *c);
/* One step of the policy for `n` selected experts `ids` (host int32) of
 * `layer`: slots[j] (host int32 [n]) = the slot holding ids[j] afterwards;
 * load_slots / load_ids (nullable host int32 [n]) = the slots to fill and
 * their experts, *n_loads of them.  MOE_ERR_UNSUPPORTED if the step has more
 * distinct experts than slots, MOE_ERR_BAD_EXPERT_ID for a negative id. */
int moe_cache_lookup(moe_expert_cache *c, int layer, const int32_t *ids, int n, int32_t *slots,
                     int32_t *load_slots, int32_t *load_ids, int *n_loads);
/* Hits and misses of a layer so far (a hit: a selected expert already in a slot). */
int moe_cache_stats(const moe_expert_cache *c, int layer, long long *hits, long long *misses);
/* The expert in a slot (-1: empty; -2: bad arguments). */
int moe_cache_slot_expert(const moe_expert_cache *c, int layer, int slot);
int moe_cache_slots(const moe_expert_cache *c);

/* One single-token layer of a residual stack with its routed experts in host
 * memory: the router on the device (rmsnorm of hidden, logits, top-k), the
 * ids copied to the host (one stream synchronisation: the CPU handoff of the
 * pages), moe_cache_lookup, one host-to-device copy per missing expert into
 * its slot, then the block (shared expert + the routed experts on their
 * slots) with hidden <- bf16(hidden + y) in place.  Results equal those of
 * moe_layer_forward_residual on resident experts with the chained launches
 * (the same kernels, the experts relabelled by slot).
 *   w        the layer: router and shared expert in device memory; w->experts
 *            pinned host memory of the E expert blobs (w->expert_stride apart)
 *   slots    device memory of this layer's slots: moe_cache_slots(c) blobs at
 *            w->expert_stride bytes each, 256-byte aligned, owned by the caller
 *   ws       workspace of moe_workspace_bytes(dims, 1)
 * No layer tail (MOE_ERR_UNSUPPORTED); not capturable in a CUDA graph (it
 * waits on the stream). */
int moe_layer_forward_offload(moe_handle *h, moe_expert_cache *c, int layer, void *hidden,
                              const moe_layer_weights *w, void *slots, void *ws, size_t ws_bytes,
                              moe_stream_t stream);

/* Single-token layer call that allocates nothing (the pages have no
 * counterpart: it exists for hosts that cannot allocate device memory,
 * e.g. a program whose own pool owns the whole device, or a per-token loop
 * where an allocation would stall the device and cannot be captured).
 * Same computation as moe_layer_forward with n_tokens = 1 on the fused
 * single-token kernel, but with no handle and no workspace.  Its scratch
 * lives in two static device arrays that every GPU loading this library
 * holds until the process exits:
 *   - 16 KiB: h, the logits when logits_out is NULL, the grid-barrier
 *     counter and the device error word;
 *   - 160 KiB: the logit mailboxes, 128 64-bit words per block of the grid
 *     (one block per SM, so devices with at most 160 SMs).
 *   x    bf16 [H] in;  y bf16 [H] out;  ids_out int32 [k], logits_out
 *        fp32 [E], weights_out fp32 [k] nullable.
 * Limits: (top_k + 1) * inter * 2 <= 15 KiB (top-8 of inter 704 uses
 * 12,672 B), at most 160 SMs, and the fused kernel's conditions
 * (n_experts <= SM count, its shared memory fits); otherwise
 * MOE_ERR_UNSUPPORTED and nothing is launched.  The first call on a device
 * looks up the arrays' device addresses and sets kernel attributes, so make
 * it before any stream capture.  The grid-barrier counter only grows (its
 * value gives each launch the epoch that tags its logits); the arrays keep
 * the last call's contents.  Calls that overlap on the GPU (different
 * streams, or the same arrays from two threads) race on the shared scratch.
 * Device-side errors (bounded-wait timeouts, non-finite values) accumulate
 * in the static error word until moe_static_get_error reads them. */
int moe_layer_forward_static(const void *x, const moe_layer_weights *w, void *y, int32_t *ids_out,
                             float *logits_out, float *weights_out, moe_stream_t stream);

/* The error word of moe_layer_forward_static on the current device: waits
 * for all work on the device, returns (in *status) the first device-side
 * error recorded since the last read (MOE_OK if none, or if no static call
 * ran on this device) and clears it.  After a timeout it also puts the
 * static grid-barrier counter and mailboxes back to zero, so the next static
 * call starts from a consistent state.  Allocates nothing. */
int moe_static_get_error(int *status);

/* ---- The tied 4-bit head and embedding (section "Why the runtime has this
 * shape": the embedding and the language-model head share one 4-bit affine
 * matrix, and the model ends with a logit softcap of 30; section "Decode":
 * the head returns the argmax token in a pure-greedy configuration, else the
 * full logits vector). */
typedef struct {
  int vocab;   /* V rows: a multiple of 16, at most 2^28                       */
  int hidden;  /* H columns: 64 .. 4096, a multiple of 64                      */
  moe_qmat w;  /* q uint32 [V, H/8] (code i at bits 4*(i%8) of word i/8),
                  scales and biases bf16 [V, H/64]; all 16-byte aligned        */
} moe_head_weights;

/* The head on up to 8 rows:
 *   logits[t, v] = cap * tanh((W x_t)[v] / cap)   (cap <= 0: no softcap)
 *   tokens[t]    = argmax_v logits[t, v], ties to the lower id
 *   x        bf16 [T, H], 16-byte aligned, T in [1, 8]
 *   logits   nullable fp32 [T, V];  tokens nullable int32 [T]; not both null
 * One kernel launch, graph-capturable.  The argmax state lives in the
 * handle (cleared by the launch that used it), so head calls on one handle
 * must not overlap on the GPU.  A non-finite logit is skipped by the argmax
 * and records MOE_ERR_NONFINITE. */
int moe_head_forward(moe_handle *h, const void *x, int n_tokens, const moe_head_weights *w, float softcap,
                     float *logits, int32_t *tokens, moe_stream_t stream);

/* A dense 4-bit affine projection in the same matrix format (section ".gturbo
 * directory": the production manifest stores the attention weights 4-bit
 * affine, group 64, like the embedding; section "Metal execution": single-
 * token decode runs projections as custom GEMV kernels), e.g. the
 * attention's Q/K/V and output projections:
 *   y[t, n] = sum_k W[n, k] x[t, k]
 *   w        W [N, K] as moe_head_weights (vocab = N rows, a multiple of 16;
 *            hidden = K columns, 64 .. 4096, a multiple of 64)
 *   x        bf16 [T, K], 16-byte aligned, T in [1, 8]
 *   y        nullable bf16 [T, N] (the fp32 sum rounded to nearest even)
 *   y32      nullable fp32 [T, N]; not both null
 * One launch of the head kernel with no softcap and no argmax, graph-
 * capturable; it does not touch the head's greedy state. */
int moe_dense_forward(moe_handle *h, const void *x, int n_tokens, const moe_head_weights *w, void *y, float *y32,
                      moe_stream_t stream);

/* The tied embedding: out[i] = bf16(q[ids[i], :] * scale + bias), the
 * dequantised row rounded once to bf16 (no scale factor).
 *   ids int32 [n] on the device, n >= 1;  out bf16 [n, H], 16-byte aligned.
 * An id outside [0, V) gives a zero row and records MOE_ERR_BAD_EXPERT_ID. */
int moe_embed(moe_handle *h, const int32_t *ids, int n, const moe_head_weights *w, void *out,
              moe_stream_t stream);

/* Launch tracing (diagnostics).  With a non-null device buffer of
 * 4 * n_launches u64, each subsequent kernel launch by this handle takes the
 * next 4 slots (wrapping) and records %globaltimer values, combined with
 * atomicMax so a zeroed buffer is the reset state:
 *   [0] bitwise NOT of the first block's entry time
 *   [1] bitwise NOT of the time that block passed its dependency wait
 *   [2] latest time a block had its weights in shared memory (0: n/a)
 *   [3] latest block exit time (the router: its last block's exit).
 * A call launches 3 (T == 1) or 4 kernels; slot groups are reserved as
 * router 1, gate/up 1, down (+ combine) 2, sort 1.  Buffer owned by the
 * caller; NULL turns tracing off.  Tracing adds a few atomics per block. */
int moe_set_trace(moe_handle *h, unsigned long long *buffer, int n_launches);

/* Self-test of the device-side bounded waits (failure detection without a
 * GPU fault): launches one thread that waits on a barrier nothing ever
 * completes; after limit_ns (1 .. 2e9 ns) of device time it gives up and
 * records MOE_ERR_TIMEOUT in the error word, which moe_get_error then
 * reports.  Every wait in the kernels above uses the same bounded wait. */
int moe_selftest_wait_timeout(moe_handle *h, unsigned long long limit_ns, moe_stream_t stream);

/* Self-test of a grid barrier that never completes (failure detection
 * without a GPU fault): arms the handle's next fused single-token launch so
 * that block `block` (0 <= block < SM count) withholds its arrival at the
 * barrier between the gate/up and down phases, and every bounded wait of
 * that launch gives up after limit_ns (1 .. 2e9 ns) of device time.  The
 * blocks then record MOE_ERR_TIMEOUT and leave (the launch's outputs are not
 * valid); moe_get_error reports it and restores the barrier state, so the
 * next call is correct again.  Host-side only: launches nothing itself. */
int moe_selftest_skip_arrival(moe_handle *h, int block, unsigned long long limit_ns);

/* Waits for all work on the device, then returns (in *status) the first
 * device-side error recorded since the last call (MOE_OK if none) and
 * clears it.  After a timeout it also resets the handle's grid-barrier
 * counters, tickets and logit mailboxes (a launch whose blocks did not all
 * arrive leaves its counter out of step).  The return value reports
 * failures of the call itself. */
int moe_get_error(moe_handle *h, int *status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_AFFINE_H */
