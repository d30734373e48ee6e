/*
 * e0.h — C ABI of libe0: the MoE decode layer-step with a cross-token prerouter,
 * int4 group-64 experts and an unmerged recovery LoRA, for NVIDIA GB300 (sm_103a).
 *
 * What the calls compute comes from "The Other Half of the Memory Wall: Serving 35B
 * MoEs from SSD with Trained Routing Prediction" (Edge0):
 *   §3.1 "Problem", "Executor paths", "Math contract" — int4 affine group-64 expert
 *        weights with per-group scale and bias; an expert is down(silu(gate x) * up x);
 *        staged experts addressed through a slot table that never leaves the GPU.
 *   §3.2 "Head", "Prediction-as-routing" — the head of layer N reads layer N's norm
 *        output plus the one-hots of this layer's routing at this token and at the
 *        previous token; fc1 -> erf-GELU -> fc2 plus a linear residual gives the
 *        logits that ARE the routing of layer N+1 at the next token.
 *   §3.3 — the recovery LoRA is served unmerged: y = W_int4 x + (alpha/r) B A x.
 *   Appendix A "Softmax-topk" — w = softmax(l)[ids] / sum over ids.
 *
 * Conventions (every call):
 *   - All tensor pointers are DEVICE pointers unless a comment says "host".  The
 *     caller owns all memory; the library never frees a caller pointer.  Device
 *     pointers must be 16-byte aligned.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Matrices are row-major.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Argument and shape errors return a negative e0_status before anything is
 *     launched; e0_last_error() then describes the problem (thread-local text).
 *   - Errors found on the device (bad expert id, expert not resident in its slot
 *     pool, a wait that ran out of time) never trap: they set bits in the status
 *     word of the workspace, the kernel finishes early, and the caller reads the
 *     word with e0_get_device_status() after synchronising.  After a non-zero
 *     status the workspace must be cleared with e0_workspace_reset().
 *   - A workspace is caller-allocated device memory of e0_*_workspace_size()
 *     bytes, ZERO-FILLED before its first use (cudaMemset or e0_workspace_reset).
 *     Calls that share a workspace must be ordered on one stream.  Holding it
 *     between calls carries the engine's counters; nothing else persists.
 *
 * int4 format ("affine group-64"): a group is 64 consecutive input columns of one
 * output row; scale s = bf16((max-min)/15), bias b = bf16(min), code
 * q = clamp(rint((w-b)/s), 0, 15) in fp32 (q = 0 when s == 0); weight = s*q + b.
 *   E0_LAYOUT_ROWS:    q uint32 [rows][cols/8] (column j at bits 4*(j%8) of word j/8),
 *                      scale, bias bf16 [rows][cols/64].
 *   E0_LAYOUT_COLSLAB: the same codes stored 32 columns at a time:
 *                      q uint32 [cols/32][rows][4], scale, bias bf16 [cols/64][rows].
 *   Both layouts are batched over a leading index (experts).
 */
#ifndef E0_H
#define E0_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* e0_stream;   /* == cudaStream_t */
typedef struct CUevent_st*  e0_event;    /* == cudaEvent_t  */
typedef int32_t e0_status;

enum {
  E0_OK = 0,
  E0_ERR_INVALID = -1,      /* bad pointer, alignment or argument */
  E0_ERR_SHAPE = -2,        /* unsupported or inconsistent dimensions */
  E0_ERR_CUDA = -3,         /* a CUDA runtime call failed (text in e0_last_error) */
  E0_ERR_TIMEOUT = -4,      /* host-side wait ran out of time */
  E0_ERR_NOMEM = -5,        /* workspace too small / allocation failed */
  E0_ERR_UNSUPPORTED = -6,  /* valid request this build does not implement */
  E0_ERR_DEVICE = -7        /* e0_get_device_status() reported device-side errors */
};

/* Bits of the device status word. */
enum {
  E0_DEV_TIMEOUT = 1,       /* a bounded spin-wait gave up */
  E0_DEV_BAD_ID = 2,        /* an expert id outside [0, E) or repeated; expert skipped */
  E0_DEV_NOT_RESIDENT = 4,  /* slot_of[id] < 0: expert absent from its slot pool; skipped */
  E0_DEV_ABORTED = 8        /* another CTA aborted; this one stopped early */
};

enum { E0_LAYOUT_ROWS = 0, E0_LAYOUT_COLSLAB = 1 };

/* Thread-local description of the last error returned on this thread. */
const char* e0_last_error(void);
const char* e0_version(void);

/* --------------------------------------------------------------------------------
 * e0_pack_int4 — quantise fp32 weights to int4 affine group-64 (§3.1, §2
 * "Quantization").  w: fp32 [batch][rows][cols] (device).  cols % 64 == 0 and
 * group == 64.  For E0_LAYOUT_COLSLAB cols % 32 == 0 (implied).  Outputs per the
 * layout comments above.  Bit-exact: IEEE fp32 arithmetic, no fast-math.
 * ------------------------------------------------------------------------------ */
e0_status e0_pack_int4(const float* w, int64_t batch, int64_t rows, int64_t cols,
                       int32_t group, int32_t layout,
                       uint32_t* q, uint16_t* scale, uint16_t* bias, e0_stream stream);

/* One packed int4 matrix (layout given by where it is used). */
typedef struct {
  const uint32_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} e0_q4;

/* A stack of SwiGLU experts (§3.1 "nine stacked tensors per layer").
 *   gate_up: E0_LAYOUT_ROWS, [n][2F][d]; row 2j is gate row j, row 2j+1 is up row j.
 *   down:    E0_LAYOUT_COLSLAB, [n][d][F] (i.e. q [n][F/32][d][4], s/b [n][F/64][d]).
 *   n:       experts stored (E for a full stack, 1 for a shared expert, S slots).
 *   slot_of: int16 [E] expert id -> stored index, < 0 = not resident; NULL = identity.
 *   stride:  bytes between consecutive stored experts in all six tensors (a slot pool
 *            keeps each expert's six tensors together in one bundle); 0 = each tensor
 *            packed densely, [n][...].  A multiple of 16.
 */
typedef struct {
  e0_q4 gate_up;
  e0_q4 down;
  int32_t n;
  const int16_t* slot_of;
  int64_t stride;
  const uint32_t* ready;  /* nullable; decode stack only: a word (a slot pool's, see
                             e0_slot_pool_view) that reaches the token index once this
                             token's experts and slot_of table are in place; the stack
                             step waits for it (bounded) before reading either.  With
                             ready set, slot_of holds two tables [2][E], used by tokens
                             of even and odd index */
} e0_experts;

/* Unmerged recovery LoRA linear (§3.3): y = W x + (alpha/r) * B (A x).
 *   w: E0_LAYOUT_ROWS [out][in];  a: bf16 [r][in];  bt: bf16 [r][out] (B transposed).
 *   r == 0 or a/bt NULL -> base only. */
typedef struct {
  e0_q4 w;
  const uint16_t* a;
  const uint16_t* bt;
  int32_t out;
  int32_t r;
  float alpha;
} e0_qlora;

/* Cross-token prerouter head (§3.2 "Head").  The feature is [x ; onehot(ids_cur) ;
 * onehot(ids_prev)] with x the RMS-normed hidden state; fc1 is stored split:
 *   w1h [H][d] (hidden block), w1c_t [E][H] and w1p_t [E][H] (the two one-hot
 *   blocks, transposed so a committed id selects one contiguous row).
 *   b1 [H] (nullable), w2t [H][E] (fc2 transposed), b2 [E] (nullable),
 *   lres [E][d] (linear residual path).  H == 0 leaves only lres (+ b2): a plain
 *   linear router. */
typedef struct {
  int32_t H;
  const uint16_t* w1h;
  const uint16_t* w1c_t;
  const uint16_t* w1p_t;
  const uint16_t* b1;
  const uint16_t* w2t;
  const uint16_t* b2;
  const uint16_t* lres;
} e0_prerouter;

/* Routing families (Appendix A "Routing Math"). */
enum {
  E0_ROUTE_SOFTMAX_TOPK = 0,  /* ids = top-K of the logits; w = softmax over all E, picked,
                                 renormalised (equal to the softmax of the picked logits) */
  E0_ROUTE_SIGMOID_GROUP = 1  /* sigma = sigmoid(logits); a group's score is the sum of its
                                 two largest sigma; the top topk_group of n_group groups
                                 (contiguous blocks of E / n_group experts) survive; ids =
                                 top-K of sigma within them; w = route_scale * sigma[ids] /
                                 (sum sigma[ids] + 1e-20).  The page selects on "the biased
                                 score" without printing the bias: an optional per-expert
                                 score_bias is added to sigma for the group scores and the
                                 top-K only. */
};

typedef struct {
  int32_t d;    /* hidden width: 256, 512, 1024 or 2048 */
  int32_t E;    /* routed experts, multiple of 8, <= 1024 */
  int32_t F;    /* expert width, multiple of 64 */
  int32_t K;    /* experts per token, 1..16 */
  int32_t route;        /* routing family, E0_ROUTE_*; 0 (softmax-top-K) when zero-filled */
  int32_t n_group;      /* sigmoid-group: groups (2 <= E / n_group, n_group <= 32) */
  int32_t topk_group;   /* sigmoid-group: groups kept (topk_group * E / n_group >= K) */
  float route_scale;    /* sigmoid-group: s */
  const float* score_bias;  /* sigmoid-group: nullable device fp32 [E], the selection bias of
                               the routing being chosen (single-layer calls; the decode
                               stack takes it per layer from e0_layer.score_bias) */
} e0_dims;

/* Workspace for every engine call below; layers = 1 for single-layer calls. */
size_t e0_workspace_size(const e0_dims* dims, int32_t layers);
/* Zero a workspace on `stream` (use after allocation and after a device error). */
e0_status e0_workspace_reset(void* workspace, size_t bytes, e0_stream stream);
/* Read the device status word (blocks until `stream` is idle). */
e0_status e0_get_device_status(const void* workspace, uint32_t* status_out, e0_stream stream);

/* --------------------------------------------------------------------------------
 * e0_prerouter_forward — one head evaluation per token (§3.2 "Head"; Appendix A).
 *   h: bf16 [T][d], the layer's hidden state; the head reads x = RMSNorm(h)
 *      (unit gain, eps 1e-6) — the "post-attention norm output".
 *   ids_cur, ids_prev: int32 [T][K] distinct ids in [0, E); ids_prev nullable
 *      (previous one-hot all zero).
 *   logit_bias: fp32 [E] added to the logits before top-K (nullable).
 *   logits_out fp32 [T][E]; ids_out int32 [T][K] (descending, ties -> lower id);
 *   weights_out fp32 [T][K] renormalised softmax over ids_out (nullable).
 *   T > 1 (at most 16) reads each head weight row once for all tokens; h must then be
 *   16-byte aligned and the workspace 256-byte aligned, holding
 *   e0_decode_workspace_size(dims, T, 0, H).
 * ------------------------------------------------------------------------------ */
e0_status e0_prerouter_forward(const e0_prerouter* head, int32_t d, int32_t E,
                               const uint16_t* h, const int32_t* ids_cur,
                               const int32_t* ids_prev, int32_t T, int32_t K,
                               const float* logit_bias, float* logits_out,
                               int32_t* ids_out, float* weights_out,
                               void* workspace, size_t workspace_bytes, e0_stream stream);

/* --------------------------------------------------------------------------------
 * e0_qlinear_lora — y[T][out] = (accumulate ? y : 0) + W x + (alpha/r) B A x (§3.3).
 *   x: bf16 [T][in] used as given (no norm); in in {256, 512, 1024, 2048}.
 *   y: bf16 [T][out] (written, and read when accumulate != 0); y_f32 fp32 [T][out]
 *   (nullable) receives the same sum before bf16 rounding.
 * ------------------------------------------------------------------------------ */
e0_status e0_qlinear_lora(const e0_qlora* lora, int32_t in, const uint16_t* x, int32_t T,
                          int32_t accumulate, uint16_t* y, float* y_f32,
                          void* workspace, size_t workspace_bytes, e0_stream stream);

/* --------------------------------------------------------------------------------
 * e0_moe_decode_layer — one MoE layer-step for T tokens (north star parts 1-4).
 *   x = RMSNorm(h_in);  delta = sum_k w_k E_{ids_k}(x) + E_shared(x) + LoRA(x);
 *   h_out = bf16(h_in + delta).  w = softmax(logits)[ids] renormalised (App. A).
 *   routed: the layer's expert stack (slot_of for slot pools); shared, lora, head
 *   nullable.  ids: int32 [T][K] this layer's committed routing, logits fp32 [T][E]
 *   the logits it was committed from.  ids_prev int32 [T][K] nullable (the ids
 *   this layer used at the previous token; only read by the head).
 *   delta_f32 fp32 [T][d] nullable.  If head != NULL the call also commits the next
 *   layer's routing for the next token: next_logits fp32 [T][E], next_ids int32
 *   [T][K], next_weights fp32 [T][K] (nullable).  The weights follow dims->route.
 *   T == 1 runs the streaming GEMV engine (workspace: e0_workspace_size(dims, 1)).
 *   2 <= T <= 16 (several tokens of a batch) reads every weight once for all tokens:
 *   the experts on the grouped tensor-core path of e0_moe_prefill_layer (each expert
 *   any token picked, once; fp16 products, fp32 accumulation), the head with each
 *   weight row dotted with every token's hidden state; the routed stack must hold all
 *   E experts (no slot pool), d and 2F multiples of 256; workspace:
 *   e0_decode_workspace_size(dims, T, lora_out, H) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------------ */
/* Workspace bytes of e0_moe_decode_layer for T tokens (lora_out: the LoRA output width,
 * 0 without LoRA; H: the head's fc1 width, 0 without a head).  T == 1 gives
 * e0_workspace_size(dims, 1). */
size_t e0_decode_workspace_size(const e0_dims* dims, int32_t T, int32_t lora_out, int32_t H);
e0_status e0_moe_decode_layer(const e0_dims* dims, const e0_experts* routed,
                              const e0_experts* shared, const e0_qlora* lora,
                              const e0_prerouter* head, const uint16_t* h_in,
                              const int32_t* ids, const float* logits,
                              const int32_t* ids_prev, int32_t T, uint16_t* h_out,
                              float* delta_f32, float* next_logits, int32_t* next_ids,
                              float* next_weights, void* workspace,
                              size_t workspace_bytes, e0_stream stream);

/* --------------------------------------------------------------------------------
 * e0_moe_prefill_layer — a chunk of T tokens through one MoE layer (prefill), on the
 * tcgen05 tensor cores.  "The Other Half of the Memory Wall", §3.1 "Executor paths"
 * (same expert math as decode), Appendix A "Softmax-topk" (routing), §3.3 (LoRA); the
 * pages run no prerouter in prefill, so there is no head here.
 *   Per token t: x = RMSNorm(h_in[t]); ids = top-K of logits[t] (descending, ties to
 *   the lower id), w = softmax over the selected logits; delta = sum_k w_k E_{ids_k}(x)
 *   + E_shared(x) + LoRA(x); h_out[t] = bf16(h_in[t] + delta).
 *   h_in, h_out: bf16 bits [T][d] (16-byte aligned); logits fp32 [T][E].
 *   delta_f32 fp32 [T][d] (16-byte aligned), ids_out int32 [T][K], weights_out fp32
 *   [T][K]: nullable.  routed: all E experts resident (slot_of must be NULL); shared,
 *   lora nullable; the LoRA linear must be d x d, its B^T 8-byte aligned; every int4
 *   code, scale and bias array 16-byte aligned.  Shapes: d and 2F multiples of 256, F of 64, E <= 1024,
 *   K <= 16, T*K <= 65536.
 *   workspace: caller-owned device memory of e0_prefill_workspace_size(dims, T,
 *   lora_out) bytes (lora_out = the LoRA output width, 0 without LoRA); its first 256
 *   bytes carry a device status word readable with e0_get_device_status.
 *   The products run in fp16 (x and the dequantised weights each rounded once) with
 *   fp32 accumulation; the routing and the combine run in fp32.
 * ------------------------------------------------------------------------------ */
size_t e0_prefill_workspace_size(const e0_dims* dims, int32_t T, int32_t lora_out);
e0_status e0_moe_prefill_layer(const e0_dims* dims, const e0_experts* routed,
                               const e0_experts* shared, const e0_qlora* lora,
                               const uint16_t* h_in, const float* logits, int32_t T,
                               uint16_t* h_out, float* delta_f32, int32_t* ids_out,
                               float* weights_out, void* workspace, size_t workspace_bytes,
                               e0_stream stream);

/* --------------------------------------------------------------------------------
 * e0_moe_decode_layer_noalloc — the same single-token layer-step (T = 1) as
 * e0_moe_decode_layer, for callers that cannot allocate device memory (a host
 * callback or real-time loop that must not enter the allocator, a plugin whose host
 * framework owns every allocation).  No counterpart in the paper: it is a packaging
 * of this library.  The workspace lives in a fixed 128 KiB array inside the library's
 * device memory, reserved on every GPU that loads it until the process exits; dims
 * whose workspace (e0_workspace_size(dims, 1)) exceeds it return E0_ERR_NOMEM.  The
 * first call on a device looks the array up (make it before any stream capture).
 * Each call clears the part it uses on `stream` first; calls that overlap on the GPU
 * (different streams) share the array and race.  Arguments as e0_moe_decode_layer.
 * ------------------------------------------------------------------------------ */
e0_status e0_moe_decode_layer_noalloc(const e0_dims* dims, const e0_experts* routed,
                                      const e0_experts* shared, const e0_qlora* lora,
                                      const e0_prerouter* head, const uint16_t* h_in,
                                      const int32_t* ids, const float* logits,
                                      const int32_t* ids_prev, uint16_t* h_out,
                                      float* delta_f32, float* next_logits, int32_t* next_ids,
                                      float* next_weights, e0_stream stream);

/* --------------------------------------------------------------------------------
 * Decode stack: L layer-steps for one token in ONE launch.  Where a layer's routing
 * comes from (route_src[l]):
 *    1  the prediction head l-1 made at the previous token ("The Other Half of the
 *       Memory Wall" §3.2 "Two consumption profiles", "Prediction-as-routing"); at the
 *       first token such a layer routes with its own gate;
 *    0  its own gate R_l x_l;
 *   -N  route-ahead by N layers (the route-ahead notes of BigMoeOnEdge, "The idea"):
 *       its own gate applied to the input of layer l - N at the same token, with the
 *       combine weights taken from those logits (the prediction's own, as for a head);
 *       needs l >= N.
 * Every layer's gate logits get logit_bias[0][l] (e0_stack_step).
 * The stack object is library-owned (layer descriptors and the CTA work plan in
 * device memory); the weights it points to stay caller-owned and must outlive it.
 * ------------------------------------------------------------------------------ */
typedef struct {
  e0_experts routed;
  e0_experts shared;            /* n == 0 -> none */
  e0_qlora lora;                /* w.q == NULL -> none */
  e0_prerouter head;            /* lres == NULL -> no head on this layer */
  const uint16_t* router;       /* bf16 [E][d]; required on layers that may self-route */
  const float* score_bias;      /* sigmoid-group routing: this layer's selection bias fp32
                                   [E] (device), nullable */
} e0_layer;

typedef struct e0_stack e0_stack;

/* layers: HOST array of L descriptors (copied).  route_src: HOST int8 [L] as above
 * (NULL: every layer routes with its own gate). */
e0_status e0_stack_create(e0_stack** out, const e0_dims* dims, const e0_layer* layers,
                          int32_t L, const int8_t* route_src);
void e0_stack_destroy(e0_stack* stack);
size_t e0_stack_workspace_size(const e0_stack* stack);

/* Optional per-token outputs of e0_stack_step; every pointer is nullable device memory.
 *   ids       int32 [L][K]: the routing each layer used at this token;
 *   weights   fp32 [L][K]: its combine weights;
 *   h_trace   bf16 [L][d]: each layer's input hidden state;
 *   delta     fp32 [L][d]: each layer's delta (expert, shared and LoRA sum) before the
 *             bf16 rounding of h_out;
 *   logits    fp32 [2][L][E]: [0][l] the gate logits layer l routed by at this token
 *             (own-gate and route-ahead layers), [1][l] the logits committed for layer
 *             l at the next token (layers routed by the previous layer's head); both
 *             include logit_bias; rows that do not apply are left untouched;
 *   next_ids  int32 [L][K]: the routing committed for the next token (-1 on layers not
 *             routed by a head), the device ids e0_stage_slots consumes;
 *   commit_box  e0_commit_box_device() of a commit box: each head-routed layer's committed
 *             ids are also written there, as soon as its head is done, for
 *             e0_stage_slots_committed to stage while the launch goes on. */
typedef struct {
  int32_t* ids;
  float* weights;
  uint16_t* h_trace;
  float* delta;
  float* logits;
  int32_t* next_ids;
  void* commit_box;
} e0_stack_outputs;

/* One decode token through all L layers.
 *   step: token index (0 = first token: every layer routed by a head routes with its
 *   own gate instead).  Pooled layers (e0_experts.ready set) wait for their ready word
 *   to equal `step` (as uint32).
 *   h0: bf16 [d]; incr: bf16 [L][d] per-layer residual increments standing in for
 *   attention (h_l = bf16(h_out_{l-1} + incr_l), h_out_{-1} = h0);
 *   h_out: bf16 [d] output of the last layer.  outs: nullable (see e0_stack_outputs).
 *   logit_bias fp32 [2][L][E], nullable: [0][l] is added to layer l's gate logits at
 *   this token, [1][l] to the head logits that commit layer l's routing for the next
 *   token, before the top-K (a synthetic routing trace is injected this way: a large
 *   bias on the trace's ids makes the routing pick them). */
e0_status e0_stack_step(e0_stack* stack, int32_t step, const uint16_t* h0,
                        const uint16_t* incr, uint16_t* h_out, const e0_stack_outputs* outs,
                        const float* logit_bias, void* workspace, size_t workspace_bytes,
                        e0_stream stream);

/* --------------------------------------------------------------------------------
 * Bounded HBM expert-slot pool (§3.1 "Executor paths", the staged path; §3.2
 * "Motivation": experts stay off the GPU and a bounded set of slots holds the ones the
 * routing needs; the prerouter's one-token lead is the time to stage them).  Experts
 * live in pinned host memory as one bundle per (layer, expert): gate/up codes, scales,
 * biases, down codes, scales, biases, at the offsets e0_expert_bundle_bytes reports
 * (layouts as in e0_experts).  Each layer owns `slots` bundle slots in HBM, replaced
 * least-recently-used; the experts of the previous staging of a layer and the ones
 * being staged are never evicted, so 2K <= slots.  Each layer also has a ready word
 * (e0_experts.ready of its view): a staging call writes its `tag` there after the
 * layer's bundle copies and id -> slot table, all on the copy stream, so a decode-stack
 * launch for token t (tag t) can start before the copies end and waits, layer by layer,
 * only where it needs them.
 * ------------------------------------------------------------------------------ */
typedef struct e0_slot_pool e0_slot_pool;
typedef struct {
  int32_t hits;        /* staged ids already resident */
  int32_t misses;      /* staged ids copied in */
  int32_t evictions;   /* misses that replaced a resident expert */
  int64_t h2d_bytes;   /* bytes copied host -> device */
} e0_stage_stats;

/* Bytes of one expert bundle for these dims; offsets6 (nullable) receives the byte
 * offsets of the six tensors inside a bundle. */
size_t e0_expert_bundle_bytes(const e0_dims* dims, size_t* offsets6);
/* host_bundles: pinned host memory [layers][E][bundle_bytes], caller-owned, outliving
 * the pool.  The pool (slots, id -> slot tables, ready words) is library-owned. */
e0_status e0_slot_pool_create(e0_slot_pool** out, const e0_dims* dims, int32_t layers,
                              int32_t slots, const void* host_bundles, size_t bundle_bytes);
void e0_slot_pool_destroy(e0_slot_pool* pool);
/* The device view of a layer's slots, to pass as e0_layer.routed (n = slots, slot_of
 * the layer's two id -> slot tables, int16 [2][E], for tokens of even and odd index,
 * stride = bundle bytes, ready = its ready word). */
e0_status e0_slot_pool_view(const e0_slot_pool* pool, int32_t layer, e0_experts* out);

/* Stage the routing a decode-stack launch committed: next_ids is DEVICE int32 [*][K]
 * (e0_stack_outputs.next_ids), rows HOST int32 [n_layers] gives the row of next_ids
 * for each pool layer in layers (HOST int32 [n_layers]).  On copy_stream: wait for
 * `after` (the launch that wrote next_ids; nullable only if the ids are already
 * complete), copy the ids to the host, and block this thread until they arrive; then
 * for each layer, in order: one copy per missing bundle, the id -> slot table, and
 * `tag` into the layer's ready word.  Because the copies wait for `after`, no slot that
 * launch (or an earlier one) reads is overwritten while it runs.  stats (nullable) is
 * accumulated into.  On an error nothing of the failing layer is marked resident that
 * was not copied, its ready word keeps its old value, and later calls stay valid. */
e0_status e0_stage_slots(e0_slot_pool* pool, const int32_t* layers, int32_t n_layers,
                         const int32_t* next_ids, const int32_t* rows, int32_t K, uint32_t tag,
                         e0_stream copy_stream, e0_event after, e0_stage_stats* stats);
/* The same with HOST ids [n_layers][K]: priming a pool before the first token (whose
 * routing no head committed) or a routing the host already knows.  The slots a staging
 * may overwrite are those of neither this staging nor the previous one of the layer:
 * pass as `after` the last launch that may read such a slot (NULL only when none is
 * still queued or running). */
e0_status e0_stage_slots_host(e0_slot_pool* pool, const int32_t* layers, int32_t n_layers,
                              const int32_t* ids, int32_t K, uint32_t tag, e0_stream copy_stream,
                              e0_event after, e0_stage_stats* stats);
/* Staging from the routing while it is being committed.  A commit box is pinned,
 * host-mapped memory (library-owned) that a decode-stack launch for token t writes,
 * layer by layer, as each head finishes: the ids committed for token t + 1 and then the
 * tag t + 1 (two halves, by the tag's parity).  e0_stage_slots_committed waits on the
 * host (polling, bounded by timeout_ns; E0_ERR_TIMEOUT after) for each pool layer's row
 * (rows HOST int32 [n_layers]: the stack layer of each pool layer) to carry `tag`, then
 * stages it exactly as e0_stage_slots does.  Call it right after queueing launch `tag`
 * behind launch `tag` - 1: the copies of token `tag` then overlap launch `tag` - 1, and
 * launch `tag` waits only for the layers whose copies are still in flight.  Safe while
 * launch `tag` - 1 runs: its experts are pinned in the pool and each layer keeps two
 * id -> slot tables, for even and odd tokens. */
typedef struct e0_commit_box e0_commit_box;
e0_status e0_commit_box_create(e0_commit_box** out, int32_t layers);
void e0_commit_box_destroy(e0_commit_box* box);
void* e0_commit_box_device(const e0_commit_box* box);
e0_status e0_stage_slots_committed(e0_slot_pool* pool, const e0_commit_box* box, const int32_t* layers,
                                   const int32_t* rows, int32_t n_layers, int32_t K, uint32_t tag,
                                   e0_stream copy_stream, uint64_t timeout_ns, e0_stage_stats* stats);
/* The pool's own record of a layer's id -> slot table (HOST int16 [E], -1 = absent), as
 * it will be on the device once the queued copies have run. */
e0_status e0_slot_pool_resident(const e0_slot_pool* pool, int32_t layer, int16_t* slot_of_out);
/* Tests: make the staging calls fail (as a failed cudaMemcpyAsync would, E0_ERR_CUDA)
 * when they are about to queue their (n+1)-th bundle copy from now; n < 0 disarms. */
e0_status e0_debug_fail_copies(e0_slot_pool* pool, int32_t n);

/* --------------------------------------------------------------------------------
 * Input generation (not part of the method): the seeded counter-based generator
 * "e0synth" (SplitMix64 draws, Irwin-Hall-12 normal) writing n values of tensor
 * (seed, stream) starting at element `offset`; out is fp32 (bf16 != 0: bf16 bits).
 * ------------------------------------------------------------------------------ */
e0_status e0_synth_normal(void* out, int64_t n, uint64_t seed, uint32_t stream_id,
                          int64_t offset, double sigma, int32_t bf16, e0_stream stream);

/* Debug / tests: make the next engine launch on this workspace wait on a flag that
 * nothing sets, with the given time limit (ns), so the timeout path can be tested.
 * limit_ns == 0 restores normal operation. */
e0_status e0_debug_inject_stall(void* workspace, uint64_t limit_ns, e0_stream stream);

/* Debug / profiling: when buf != NULL, later engine launches from this thread write
 * %globaltimer stamps to buf[cta][layer][16] (u64, zero-filled device memory of at
 * least ncta * layers * 128 bytes; ncta <= 160).  Slots: 0 consumer layer start,
 * 1 layer dependency satisfied, 2 layer input built, 3 layer's units done,
 * 4 routing warp published the layer's routing, 5 copy warp issued the layer's last
 * copy, 6 ns consumer warp 0 waited for stages, 7 stages it took, 8 own-gate routing
 * started, 8 + unit type: ns spent in units of that type (accumulated; for U_ROUTER = 6
 * the time this CTA's gate rows were published).  buf == NULL switches tracing off. */
e0_status e0_debug_trace(uint64_t* buf, size_t bytes);

/* Debug / tests: the CTA work plan a stack of 35B-class-shaped layers would use, built
 * on the host (no device needed), for one layer kind: 0 a layer with a prerouter head
 * (routed and shared experts, d x d LoRA linear of rank lr, head of H fc1 rows), 1 the
 * same without a head, 2 the own-gate router rows (over the CTAs that kind 0 leaves on
 * the critical path), 3 a layer without a head after one with a head (kind 1's work
 * over the CTAs that kind 0 leaves on the critical path: the CTAs with prerouter work
 * run behind the layers).  units_out: ncta * 8 units of 8 bytes, {type u8, k u8, r0 u16,
 * r1 u16, flags u16}, unit types as in the engine (1 expert slab, 2 LoRA base rows,
 * 3 LoRA A ranks, 4 head fc1 rows, 5 head residual rows, 6 gate rows, 7 LoRA B rows);
 * counts_out[ncta] units per CTA; defer_out[ncta] = 1 where a CTA holds only
 * prerouter work.  ncta <= 160. */
e0_status e0_debug_plan(int32_t d, int32_t E, int32_t F, int32_t K, int32_t H, int32_t lr, int32_t ncta,
                        int32_t kind, void* units_out, uint8_t* counts_out, uint8_t* defer_out);

#ifdef __cplusplus
}
#endif
#endif /* E0_H */
