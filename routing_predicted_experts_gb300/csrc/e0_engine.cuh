// Streaming layer-step engine: definitions shared by the kernel (e0_engine.cu) and
// the host-side planner / C ABI (e0_api.cu).
//
// One persistent cooperative launch runs one layer-step (or a stack of layer-steps
// for one token).  Every CTA owns a list of work units per layer.  A producer warp
// streams the weight bytes of those units, in consumption order, into a ring of
// shared-memory stages with bulk asynchronous copies (cp.async.bulk, mbarrier
// completion); fourteen consumer warps dequantise and reduce them against the
// layer input held in shared memory.  Because weight addresses do not depend on
// activations, the producer runs ahead across layer boundaries: the next layer's
// weights stream in while the grid waits for the current layer to finish.
//
// The layer-step is split so that every unit depends only on the layer input x:
//   U_EXPERT  one expert (routed slot k < K, or the shared expert k == K) restricted
//             to 32 columns of its SwiGLU width: 32 gate rows + 32 up rows give 32
//             activations a = silu(g) * u, which the matching 32-column slab of the
//             down projection turns into a contribution to all d outputs;
//   U_QROWS   rows of the LoRA base W;  U_LORA_A  ranks of the LoRA down projection,
//             v = A x: all of them kept in shared memory for the CTA's own B rows, or a
//             slice published to the other CTAs;  U_LORA_B  (alpha/r) B v for LoRA rows
//             once v is there (last on its CTA, so v is rarely waited for);
//   U_HEAD    rows of prerouter fc1 (plus the one-hot
//             columns picked by the committed ids), erf-GELU, then the matching rows
//             of fc2^T;  U_LRES  rows of the head's linear residual;  U_ROUTER  rows
//             of a layer's own gate.
// Contributions are summed in fp32 with vector reductions into a per-layer
// accumulator, so a layer has exactly one grid-wide dependency point (two when it
// routes with its own gate).
#pragma once

#include "e0_common.cuh"

namespace e0eng {

constexpr int NCW = 14;                       // consumer warps (16 warps in all: 4 per SM sub-partition)
constexpr int NTHREADS = (NCW + 2) * 32;      // + producer warp + routing warp
constexpr int NCT = NCW * 32;                 // consumer threads
constexpr int STAGE_BYTES = 20480;
constexpr int NSTAGES = 9;
static_assert(NSTAGES <= 32, "the copy warp issues up to a ring's worth of stages with one lane each");
constexpr int KMAX = 16;
constexpr int EMAX = 1024;
constexpr int DMAX = 2048;
constexpr int OUTMAX = 4096;                  // accumulator length per layer
constexpr int MAXU = 8;                       // units per CTA per plan kind
constexpr int MAX_CTAS = 160;
constexpr int HEAD_ROWS = 64;                 // max fc1 rows per U_HEAD unit
constexpr int RANKS_MAX = 64;                 // max LoRA rank
constexpr int KINDS_MAX = 4;
constexpr int LMAX = 48;                      // layers per launch
constexpr float RMS_EPS = 1e-6f;

constexpr uint16_t UF_LOCAL_V = 1;

enum UnitType : uint8_t { U_NONE = 0, U_EXPERT, U_QROWS, U_LORA_A, U_HEAD, U_LRES, U_ROUTER, U_LORA_B };

struct Unit {
  uint8_t type;
  uint8_t k;       // U_EXPERT: expert slot (k == K: shared expert)
  uint16_t r0;     // first row / slab / rank
  uint16_t r1;     // end row / rank (exclusive)
  uint16_t flags;   // U_LORA_A: UF_LOCAL_V = v stays in this CTA's shared memory (its own B rows)
};
static_assert(sizeof(Unit) == 8, "Unit must stay 8 bytes");

enum Mode : int32_t { MODE_LAYER = 0, MODE_HEAD = 1, MODE_QLINEAR = 2, MODE_STACK = 3 };

// Plan kinds (stack mode): main phase with head / without head, router phase.
// KIND_TAIL: the layers without a head that follow a layer with one; their work stays
// off the CTAs that hold the prerouter's (deferred) work, which run behind the layers.
enum Kind : int32_t { KIND_MAIN = 0, KIND_MAIN_NOHEAD = 1, KIND_ROUTER = 2, KIND_TAIL = 3 };

struct LayerDesc {
  // routed experts
  const uint32_t* gu_q;
  const uint16_t* gu_s;
  const uint16_t* gu_b;
  const uint32_t* dn_q;
  const uint16_t* dn_s;
  const uint16_t* dn_b;
  const int16_t* slot_of;
  int64_t ex_stride;  // bytes between stored routed experts (0: dense per tensor)
  int32_t n_routed;
  int32_t has_shared;
  // shared expert (same layouts, one expert)
  const uint32_t* sgu_q;
  const uint16_t* sgu_s;
  const uint16_t* sgu_b;
  const uint32_t* sdn_q;
  const uint16_t* sdn_s;
  const uint16_t* sdn_b;
  // LoRA linear
  const uint32_t* lw_q;
  const uint16_t* lw_s;
  const uint16_t* lw_b;
  const uint16_t* la;
  const uint16_t* lbt;
  int32_t lr;
  float lscale;      // alpha / r
  int32_t lout;
  int32_t has_lora;
  // prerouter head
  int32_t has_head;
  int32_t H;
  const uint16_t* w1h;
  const uint16_t* w1c_t;
  const uint16_t* w1p_t;
  const uint16_t* b1;
  const uint16_t* w2t;
  const uint16_t* b2;
  const uint16_t* lres;
  // own gate
  const uint16_t* router;
  const float* score_bias;  // sigmoid-group routing: selection bias of this layer's routing (nullable)
  const uint32_t* ready;    // stack, slot pools: word equal to the token index once this layer's
                            // experts and slot_of table are in place (nullable)
  int32_t plan_kind;  // KIND_MAIN, KIND_MAIN_NOHEAD or KIND_TAIL
  int32_t prerouted;  // 1: routing comes from the previous layer's head (after step 0)
  int32_t ahead;      // N > 0: route-ahead, this layer's gate runs on layer (l - N)'s input
  int32_t gate_for;   // stack: the layer whose route-ahead gate rows run on this layer's input, or -1
};

// Workspace: header, then parity-duplicated buffers so that one launch uses one half
// while it clears the other half for the next launch.
struct WsHeader {
  uint32_t epoch;      // launches completed on this workspace
  uint32_t status;     // E0_DEV_* bits
  uint32_t abort;      // set by a CTA that gave up; others stop early
  uint32_t never;      // always 0: the flag the stall-injection wait polls
  uint64_t stall_ns;   // != 0: next launch waits on `never` for this long (tests)
  uint64_t pad[5];
};
static_assert(sizeof(WsHeader) == 64, "header size");

struct WsLayout {
  size_t counters;   // u32 [2][L][4]: layer done, prerouter work done (deferred CTAs), spare
  size_t acc;        // f32 [2][L][OUTMAX]
  size_t zhat;       // f32 [3][L][E]
  size_t zr;         // u64 [2][L][E]  own-gate logits, tagged with the launch (see st_tagged)
  size_t ids;        // i32 [2][L][KMAX]
  size_t wts;        // f32 [2][L][KMAX]
  size_t rg_ids;     // i32 [2][L][KMAX] routes committed for the next launch
  size_t rg_w;       // f32 [2][L][KMAX]
  size_t rg_tag;     // u32 [2][L]  epoch the route is for
  size_t lv;         // u64 [2][L][RANKS_MAX]  LoRA v = A x, tagged with the launch
  size_t total;
};

__host__ __device__ constexpr size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ constexpr WsLayout ws_layout(int E, int L) {
  WsLayout w{};
  size_t o = 256;
  w.counters = o; o = ws_align(o + sizeof(uint32_t) * 2 * L * 4);
  w.acc = o;      o = ws_align(o + sizeof(float) * 2 * (size_t)L * OUTMAX);
  w.zhat = o;     o = ws_align(o + sizeof(float) * 3 * (size_t)L * E);
  w.zr = o;       o = ws_align(o + sizeof(uint64_t) * 2 * (size_t)L * E);
  w.ids = o;      o = ws_align(o + sizeof(int32_t) * 2 * (size_t)L * KMAX);
  w.wts = o;      o = ws_align(o + sizeof(float) * 2 * (size_t)L * KMAX);
  w.rg_ids = o;   o = ws_align(o + sizeof(int32_t) * 2 * (size_t)L * KMAX);
  w.rg_w = o;     o = ws_align(o + sizeof(float) * 2 * (size_t)L * KMAX);
  w.rg_tag = o;   o = ws_align(o + sizeof(uint32_t) * 2 * (size_t)L);
  w.lv = o;       o = ws_align(o + sizeof(uint64_t) * 2 * (size_t)L * RANKS_MAX);
  w.total = o;
  return w;
}

enum RouteFamily : int32_t { ROUTE_SOFTMAX = 0, ROUTE_SIGMOID_GROUP = 1 };

struct EngineParams {
  int32_t d, E, F, K, L, ncta, mode, norm, out_dim, kinds, step;
  int32_t route;               // RouteFamily
  int32_t n_group, topk_group; // sigmoid-group routing
  float route_scale;
  uint32_t pad0;
  const float* score_bias;     // single-layer calls: selection bias of the routing being chosen
  uint64_t router_mask;        // stack: bit l set = the routing warp routes layer l from its gate
                               // logits (own gate, or route-ahead gate rows run N layers earlier)
  uint64_t gate_mask;          // stack: bit l set = layer l's own gate rows run on its own input
  uint64_t timeout_ns;
  const LayerDesc* layers;     // stack: device array [L]; else nullptr (inline_layer)
  const Unit* plan;            // stack: device [kinds][ncta][MAXU]; else nullptr (inline)
  const uint8_t* plan_n;       // stack: device [kinds][ncta]
  const uint8_t* defer;        // stack: device [kinds][ncta], 1 = the CTA holds only prerouter work
                               // of that kind: it arrives on the head counter, not the layer's
  int32_t n_arrive[KINDS_MAX]; // CTAs arriving on a layer's counter, per plan kind
  int32_t n_defer[KINDS_MAX];  // CTAs arriving on its head counter instead
  // inputs
  const uint16_t* h_in;
  const uint16_t* incr;
  const int32_t* ids_in;
  const float* logits_in;
  const int32_t* ids_prev_in;
  const float* logit_bias;
  // outputs
  uint16_t* h_out;
  float* delta_out;
  float* next_logits;
  int32_t* next_ids;
  float* next_w;
  int32_t* ids_trace;
  float* w_trace;
  uint16_t* h_trace;
  float* delta_trace;          // stack, nullable: [L][d] each layer's delta (fp32)
  float* z_trace;              // stack, nullable: [2][L][E] gate logits used / logits committed
  int32_t* next_ids_out;       // stack, nullable: [L][K] routing committed for the next token
  uint32_t* commit_box;        // stack, nullable: host-mapped [2][L][KMAX + 1]: per layer the token
                               // index the committed ids are for (word 0), then the ids
  int32_t accumulate;
  int32_t pad1;
  uint64_t* trace;             // nullable: [ncta][L][16] %globaltimer diagnostics: 0 layer start,
                               // 1 input dependency met, 2 input built, 3 units done, 4 route
                               // published, 5 copies issued, 6/7 stage-wait time/count, 8 own-gate
                               // routing started, 8 + type: time in units of that type (for
                               // U_ROUTER: when this CTA's gate rows were published)
  uint8_t* ws;
  WsLayout wl;
  LayerDesc inline_layer;
  uint8_t inline_n[MAX_CTAS];
  Unit inline_plan[MAX_CTAS * MAXU];
};

// ---- stage geometry, shared by the producer, the consumers and the planner ----
__host__ __device__ inline int q4_row_bytes(int in) { return in / 2 + in / 16; }
__host__ __device__ inline int q4_rows_per_stage(int in) {
  int n = (STAGE_BYTES / q4_row_bytes(in)) / 16 * 16;
  return n < 16 ? 16 : (n > 64 ? 64 : n);
}
__host__ __device__ inline int bf_rows_per_stage(int in) {
  int n = STAGE_BYTES / (2 * in);
  return n < 1 ? 1 : n;
}
__host__ __device__ inline int dn_rows_per_stage(int d) { return d < 1024 ? d : 1024; }

size_t smem_bytes();

}  // namespace e0eng
