// Streaming layer-step engine kernel (see e0_engine.cuh for the decomposition).
//
// Per CTA: warp NCW is the producer (route resolution + bulk-copy issue), warps
// 0..NCW-1 are consumers.  Every wait is bounded by %globaltimer; a wait that runs
// out sets E0_DEV_TIMEOUT and the abort flag, after which every thread still walks
// the same control flow (so all named barriers are reached) but skips work, and
// the producer waits for its outstanding copies before the CTA exits.
#include "e0_engine.cuh"

using namespace e0dev;

namespace e0eng {

struct Ctl {
  uint64_t full[NSTAGES];
  uint64_t empty[NSTAGES];
  uint64_t rt_bar[LMAX];      // per layer: completes (phase 0) when its route is published
  float res[DMAX];            // residual h of the layer, fp32 (exact bf16 values); x = res * xscale
  uint4 xq[4][DMAX / 32];     // x as int16: xq[t][c] = group t (of 4) of chunk c, stored [0,2,4,6,1,3,5,7]
                              // (group-major, so that lanes reading consecutive chunks hit distinct banks)
  float xinv[DMAX / 32];      // per 32-element chunk: dequant step of xq (max |x| of the chunk / 32767)
  float xsum[DMAX / 32];      // per 32-element chunk: sum of the dequantised chunk
  float abuf[2][64];          // gate/up row values of the last two expert slabs (rows 2j, 2j + 1 = gate, up of j)
  uint4 aqw[NCW][4];          // per warp: the activations quantised to int16 in the dot32 order
  float b2buf[HEAD_ROWS];     // head fc2 bias slice of the current LRES unit
  float ubuf[HEAD_ROWS];      // head fc1 pre-activation, then erf-GELU output
  float vbuf[RANKS_MAX];      // LoRA A x for the current rank slice
  float lvs[RANKS_MAX];       // LoRA v = A x of the layer (all ranks), for the B rows
  float zbuf[EMAX];           // logits staged for top-K
  // routing of every layer of this launch
  int16_t rt_ids[LMAX][KMAX];   // committed expert ids
  int16_t rt_idx[LMAX][KMAX];   // stored index (slot) of each id
  int16_t rt_prev[LMAX][KMAX];  // ids the layer used at the previous token
  float rt_w[LMAX][KMAX];       // renormalised combine weights
  uint32_t rt_valid[LMAX];
  uint32_t rt_pvalid[LMAX];
  volatile int32_t rt_ready[LMAX];
  float red[NCW];
  float xscale;               // RMSNorm factor of the current layer input
  volatile int32_t abort_flag;
  int32_t is_last;
  uint32_t epoch;
  Unit su[KINDS_MAX][MAXU];   // this CTA's work units per plan kind
  uint8_t defer[KINDS_MAX];   // per plan kind: this CTA holds only prerouter work
  int32_t sn[KINDS_MAX];
  uint32_t rt_tag[LMAX];      // staged: epoch each committed route is for
  uint64_t ttype[8];          // diagnostics (tid 0): time per unit type in the current layer
  int32_t lv_layer;           // layer whose LoRA v (all ranks) this CTA computed into lvs, else -1
};

// Dynamic shared memory: the stage ring, the control block, then a copy of the
// layer descriptors (read on every layer by every warp, so kept on chip).
constexpr size_t CTL_OFFSET = (size_t)NSTAGES * STAGE_BYTES;
constexpr size_t LD_OFFSET = (CTL_OFFSET + sizeof(Ctl) + 15) & ~size_t(15);
size_t smem_bytes() { return LD_OFFSET + sizeof(LayerDesc) * LMAX; }
static_assert(LD_OFFSET + sizeof(LayerDesc) * LMAX <= 227 * 1024, "shared memory per CTA is 227 KB at most");

extern __shared__ __align__(1024) uint8_t e0_smem[];

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ const LayerDesc& layer_at(const EngineParams& P, int l) {
  (void)P;
  return reinterpret_cast<const LayerDesc*>(e0_smem + LD_OFFSET)[l];
}

__device__ __forceinline__ const Unit* units_of(const EngineParams& P, int kind, int cta, int& n) {
  (void)P;
  (void)cta;
  const Ctl& C = *reinterpret_cast<const Ctl*>(e0_smem + CTL_OFFSET);
  n = C.sn[kind];
  return C.su[kind];
}

__device__ __forceinline__ WsHeader* hdr(const EngineParams& P) { return reinterpret_cast<WsHeader*>(P.ws); }
__device__ __forceinline__ uint32_t* ctr(const EngineParams& P, uint32_t par, int l, int which) {
  return reinterpret_cast<uint32_t*>(P.ws + P.wl.counters) + ((size_t)par * P.L + l) * 4 + which;
}
__device__ __forceinline__ uint64_t* lv_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<uint64_t*>(P.ws + P.wl.lv) + ((size_t)par * P.L + l) * RANKS_MAX;
}
__device__ __forceinline__ float* acc_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.acc) + ((size_t)par * P.L + l) * OUTMAX;
}
__device__ __forceinline__ float* zhat_ptr(const EngineParams& P, uint32_t p3, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.zhat) + ((size_t)p3 * P.L + l) * P.E;
}
__device__ __forceinline__ uint64_t* zr_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<uint64_t*>(P.ws + P.wl.zr) + ((size_t)par * P.L + l) * P.E;
}
__device__ __forceinline__ int32_t* idsu_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<int32_t*>(P.ws + P.wl.ids) + ((size_t)par * P.L + l) * KMAX;
}
__device__ __forceinline__ float* wu_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.wts) + ((size_t)par * P.L + l) * KMAX;
}
// routes committed for the next launch: ids [2][L][KMAX], weights, tag [2][L]
__device__ __forceinline__ int32_t* rg_ids_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<int32_t*>(P.ws + P.wl.rg_ids) + ((size_t)par * P.L + l) * KMAX;
}
__device__ __forceinline__ float* rg_w_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.rg_w) + ((size_t)par * P.L + l) * KMAX;
}
__device__ __forceinline__ uint32_t* rg_tag_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<uint32_t*>(P.ws + P.wl.rg_tag) + (size_t)par * P.L + l;
}

__device__ __noinline__ void raise_error(const EngineParams& P, Ctl& C, uint32_t bits) {
  atomicOr(&hdr(P)->status, bits);
  if (bits & E0_DEV_TIMEOUT) {
    atomicExch(&hdr(P)->abort, 1u);
    C.abort_flag = 1;
  }
}

__device__ __forceinline__ bool aborted(const EngineParams& P, Ctl& C) {
  if (C.abort_flag) return true;
  if (*reinterpret_cast<volatile uint32_t*>(&hdr(P)->abort)) {
    C.abort_flag = 1;
    return true;
  }
  return false;
}

template <class Pred>
__device__ __forceinline__ bool spin_until(const EngineParams& P, Ctl& C, Pred pred, uint64_t limit_ns) {
  if (C.abort_flag) return false;
  if (pred()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (pred()) return true;
    if ((it & 15u) == 0) {
      if (aborted(P, C)) return false;
      if (globaltimer() - t0 > limit_ns) {
        raise_error(P, C, E0_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Polling loops (inlined: an out-of-line call needs a stack frame, and local memory
// is slow here because nearly all of L1 is given to shared memory).
__device__ __forceinline__ bool wait_mbar(const EngineParams& P, Ctl& C, uint64_t* bar, uint32_t par) {
  return spin_until(P, C, [&] { return mbar_try_wait(bar, par); }, P.timeout_ns);
}
__device__ __forceinline__ bool wait_flag(const EngineParams& P, Ctl& C, volatile int32_t* f) {
  return spin_until(P, C, [&] { return *f != 0; }, P.timeout_ns);
}
__device__ __forceinline__ bool wait_count(const EngineParams& P, Ctl& C, const uint32_t* c, uint32_t target) {
  return spin_until(P, C, [&] { return ld_acquire_u32(c) >= target; }, P.timeout_ns);
}

__device__ __forceinline__ void cbar() { named_bar_sync(1, NCT); }

// Mark layer l's route published (lane 0 of the routing warp, its only writer): the flag
// for pollers that test it once, and one arrival on the layer's mbarrier, which the
// consumers wait on suspended in try_wait (a flag spun on by every consumer thread
// takes the shared-memory pipe from the routing warp while it computes the route).
__device__ __forceinline__ void mark_route(Ctl& C, int l) {
  if (C.rt_ready[l]) return;
  __threadfence_block();
  C.rt_ready[l] = 1;
  mbar_arrive(&C.rt_bar[l]);
}

// Diagnostics: stamp %globaltimer into trace[cta][l][slot] when a trace buffer is set.
// Slots: 0 consumer layer start, 1 dependency satisfied, 2 layer input built,
// 3 units done, 4 producer route published, 5 producer issued the layer's last stage,
// 6 ns warp 0 waited for stages, 7 stages it took, 8 routing warp began the layer's own-
// gate routing, 8 + unit type (types >= 1): ns in that unit type.
__device__ __forceinline__ void stamp(const EngineParams& P, int l, int slot) {
  if (P.trace) P.trace[((size_t)blockIdx.x * P.L + l) * 16 + slot] = globaltimer();
}

__device__ __forceinline__ float bflo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bfhi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Exact integer dot product of 32 int4 codes (one uint4 in the row layout) with 32
// int16 activations held as 16 registers (pairs ordered [0,2],[4,6],[1,3],[5,7] per
// 8-element group, matching the even/odd nibble split below).
__device__ __forceinline__ int dot32(const uint4 q, const uint32_t* xp) {
  int a0 = 0, a1 = 0;
  uint32_t lo, hi;
  lo = q.x & 0x0F0F0F0Fu; hi = (q.x >> 4) & 0x0F0F0F0Fu;
  a0 = dp2a_lo(xp[0], lo, a0); a0 = dp2a_hi(xp[1], lo, a0); a0 = dp2a_lo(xp[2], hi, a0); a0 = dp2a_hi(xp[3], hi, a0);
  lo = q.y & 0x0F0F0F0Fu; hi = (q.y >> 4) & 0x0F0F0F0Fu;
  a1 = dp2a_lo(xp[4], lo, a1); a1 = dp2a_hi(xp[5], lo, a1); a1 = dp2a_lo(xp[6], hi, a1); a1 = dp2a_hi(xp[7], hi, a1);
  lo = q.z & 0x0F0F0F0Fu; hi = (q.z >> 4) & 0x0F0F0F0Fu;
  a0 = dp2a_lo(xp[8], lo, a0); a0 = dp2a_hi(xp[9], lo, a0); a0 = dp2a_lo(xp[10], hi, a0); a0 = dp2a_hi(xp[11], hi, a0);
  lo = q.w & 0x0F0F0F0Fu; hi = (q.w >> 4) & 0x0F0F0F0Fu;
  a1 = dp2a_lo(xp[12], lo, a1); a1 = dp2a_hi(xp[13], lo, a1); a1 = dp2a_lo(xp[14], hi, a1); a1 = dp2a_hi(xp[15], hi, a1);
  return a0 + a1;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_f(float u) { return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f)); }

// ------------------------------------------------------------------ routing (one warp)
// Sigmoid-group routing (sigmoid_group_route in e0_common.cuh) with the family's
// parameters; kept out of line: it is off the hot path.
__device__ __noinline__ void route_sigmoid_group(const EngineParams& P, const float* z, const float* sbias, int lane,
                                                 int& id_out, float& w_out) {
  sigmoid_group_route(z, sbias, P.E, P.K, P.n_group, P.topk_group, P.route_scale, lane, id_out, w_out);
}

// Softmax-top-K of logits held in registers (lane holds z[lane + 32 j], j < NPL):
// lane k < K receives id k (-1 if none) and its weight, the softmax over the picked.
template <int NPL>
__device__ __forceinline__ void softmax_topk_regs(const float (&z)[NPL], int E, int K, int lane, int& id, float& w) {
  float val;
  warp_topk_regs<NPL>(z, E, K, lane, id, val);
  const float v0 = __shfl_sync(0xffffffffu, val, 0);
  const float ex = (lane < K && id >= 0) ? expf(val - v0) : 0.f;
  const float tot = warp_sum(ex);
  w = tot > 0.f ? ex / tot : 0.f;
}
template <int NPL>
__device__ __forceinline__ void softmax_topk_smem_n(const EngineParams& P, const float* z, int lane, int& id,
                                                    float& w) {
  float zv[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    zv[j] = e < P.E ? z[e] : 0.f;
  }
  softmax_topk_regs<NPL>(zv, P.E, P.K, lane, id, w);
}

// The routing of one token from its logits in shared memory z[0..E) by the family in P;
// every lane of the warp calls.  Lane k < K receives id k (-1 if none) in descending
// score order and its FINAL combine weight.
__device__ __noinline__ void route_smem(const EngineParams& P, const float* z, const float* sbias, int lane, int& id,
                                        float& w) {
  if (P.route == ROUTE_SIGMOID_GROUP)
    route_sigmoid_group(P, z, sbias, lane, id, w);
  else if (P.E <= 256)
    softmax_topk_smem_n<8>(P, z, lane, id, w);
  else if (P.E <= 512)
    softmax_topk_smem_n<16>(P, z, lane, id, w);
  else
    softmax_topk_smem_n<32>(P, z, lane, id, w);
}

// ------------------------------------------------------------------ producer
// The whole producer warp runs this code in lock step; lane 0 issues the copies and
// all lanes take part in routing (loads of logits and ids, warp top-K).
struct Prod {
  const EngineParams& P;
  Ctl& C;
  uint8_t* ring;
  uint32_t n;      // stages issued
  bool ok;
  int lane;
  uint32_t par, p3, epoch;
};

// Stack: the routing warp routes layer l from gate logits (its own gate, or route-ahead
// gate rows computed on an earlier layer's input) rather than from a committed route.
__device__ __forceinline__ bool self_routes(const EngineParams& P, int l) {
  return P.mode == MODE_STACK && ((P.router_mask >> l) & 1ull);
}
// Stack: layer l's own gate rows run on its own input.
__device__ __forceinline__ bool gate_here(const EngineParams& P, int l) {
  return P.mode == MODE_STACK && ((P.gate_mask >> l) & 1ull);
}

__device__ __forceinline__ bool prod_keep_waiting(Prod& pr, uint64_t t0, uint32_t it);

// Slot pools (stack): wait (bounded) until the layer's ready word says that this
// token's experts and id -> slot table are in place.  The word is written by a copy on
// the pool's copy stream after the bundles and the table, so seeing it makes them
// visible too.  A pool keeps two tables per layer, for even and odd tokens, so that the
// next token's can be written while this token runs.  False after a timeout or an abort.
__device__ __forceinline__ bool wait_slots_ready(Prod& pr, const LayerDesc& Ld) {
  if (pr.P.mode != MODE_STACK || !Ld.ready) return true;
  const uint32_t want = (uint32_t)pr.P.step;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    bool r = false;
    // staged for this token or a later one (the next token's staging may already have
    // finished: it leaves this token's table half and slots alone)
    if (pr.lane == 0) r = (int32_t)(ld_acquire_sys_u32(Ld.ready) - want) >= 0;
    if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0)) return true;
    if (!prod_keep_waiting(pr, t0, it)) return false;
  }
}

// Publish the routing of layer l in the route table.  Lane k (< K) brings id k
// (-1 = none) and its combine weight; ids are checked (range, duplicates, slot table).
// Softmax-top-K weights arrive unnormalised and are renormalised over the ids that
// survive; sigmoid-group weights arrive final (their scale is not a normalisation).
__device__ __forceinline__ void publish_route(Prod& pr, int l, int id, float w) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const LayerDesc& Ld = layer_at(P, l);
  const int lane = pr.lane, K = P.K;
  const bool ready = wait_slots_ready(pr, Ld);
  if (!ready) pr.ok = false;
  if (lane < K) C.rt_ids[l][lane] = (int16_t)id;
  __syncwarp();
  bool v = ready && lane < K && id >= 0 && id < P.E;
  if (lane < K)
    for (int j = 0; j < lane; ++j)
      if (C.rt_ids[l][j] == id) v = false;
  if (ready && lane < K && id != -1 && !v) raise_error(P, C, E0_DEV_BAD_ID);
  int idx = v ? id : 0;
  if (v && Ld.slot_of) {
    const int half = (P.mode == MODE_STACK && Ld.ready) ? (P.step & 1) * P.E : 0;
    idx = __ldcg(Ld.slot_of + half + id);
    if (idx < 0) {
      v = false;
      raise_error(P, C, E0_DEV_NOT_RESIDENT);
    }
  }
  if (v && Ld.gu_q && idx >= Ld.n_routed) {
    v = false;
    raise_error(P, C, E0_DEV_BAD_ID);
  }
  const uint32_t valid = __ballot_sync(0xffffffffu, v);
  const float wv = v ? w : 0.f;
  float tot = wv;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane < K) {
    C.rt_idx[l][lane] = (int16_t)idx;
    C.rt_w[l][lane] = P.route == ROUTE_SIGMOID_GROUP ? wv : ((v && tot > 0.f) ? wv / tot : 0.f);
  }
  if (lane == 0) C.rt_valid[l] = valid;
  if (P.mode == MODE_STACK && Ld.has_head) {
    // the previous-token ids this layer's head one-hots (staged at launch): valid ones
    bool pv = false;
    if (lane < K) {
      const int pid = C.rt_prev[l][lane];
      pv = pid >= 0 && pid < P.E;
      for (int j = 0; j < lane; ++j)
        if (C.rt_prev[l][j] == pid) pv = false;
    }
    const uint32_t pvalid = __ballot_sync(0xffffffffu, pv);
    if (lane == 0) C.rt_pvalid[l] = pvalid;
  }
  __syncwarp();
  if (lane == 0) {
    mark_route(C, l);
    stamp(P, l, 4);
  }
  __syncwarp();
}

// Kernel start: routing known at launch time (given ids, or the routes the previous
// launch committed for this token) and the previous-token ids the heads one-hot.
__device__ __forceinline__ void load_routes(Prod& pr) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const int lane = pr.lane, K = P.K;
  if (P.mode == MODE_LAYER || P.mode == MODE_HEAD) {
    int id = -1, pid = -1;
    float z = 0.f;
    if (P.ids_in && lane < K) id = P.ids_in[lane];
    if (P.ids_prev_in && lane < K) pid = P.ids_prev_in[lane];
    const bool inr = id >= 0 && id < P.E;
    if (P.logits_in && inr) z = P.logits_in[id];
    float w;
    if (P.route == ROUTE_SIGMOID_GROUP) {
      const float sig = (P.logits_in && inr) ? 1.0f / (1.0f + expf(-z)) : 0.f;
      w = P.route_scale * sig / (warp_sum(sig) + 1e-20f);
    } else {
      float mx = inr ? z : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      w = (P.logits_in && inr) ? expf(z - mx) : 0.f;
    }
    if (lane < K) C.rt_prev[0][lane] = (int16_t)pid;
    __syncwarp();
    bool pv = lane < K && pid >= 0 && pid < P.E;
    if (lane < K)
      for (int j = 0; j < lane; ++j)
        if (C.rt_prev[0][j] == pid) pv = false;
    if (lane < K && pid != -1 && !pv) raise_error(P, C, E0_DEV_BAD_ID);
    const uint32_t pvalid = __ballot_sync(0xffffffffu, pv);
    if (lane == 0) C.rt_pvalid[0] = pvalid;
    __syncwarp();
    if (P.ids_in) {
      publish_route(pr, 0, id, w);
    } else if (lane == 0) {
      C.rt_valid[0] = 0u;
      mark_route(C, 0);
    }
    __syncwarp();
    return;
  }
  if (P.mode != MODE_STACK) return;
  // Stage, with independent loads issued back to back: the previous-token ids of every
  // layer (recorded by the previous launch) and the routes it committed for this token.
  const int L = P.L;
  for (int j0 = 0; j0 < L * K; j0 += 32 * 8) {
    int pid[8], id[8];
    float w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // loads first, all in flight together
      const int j = j0 + 32 * u + lane, l = j / K, k = j % K;
      pid[u] = -1;
      id[u] = -1;
      w[u] = 0.f;
      if (j < L * K) {
        if (P.step > 0) pid[u] = __ldcg(idsu_ptr(P, pr.par ^ 1u, l) + k);
        if (!self_routes(P, l)) {
          id[u] = __ldcg(rg_ids_ptr(P, pr.par, l) + k);
          w[u] = __ldcg(rg_w_ptr(P, pr.par, l) + k);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + 32 * u + lane, l = j / K, k = j % K;
      if (j < L * K) {
        C.rt_prev[l][k] = (int16_t)pid[u];
        if (!self_routes(P, l)) {  // a self-routed layer may already have its route published
          C.rt_ids[l][k] = (int16_t)id[u];
          C.rt_w[l][k] = w[u];
        }
      }
    }
  }
  {
    const uint32_t t0 = lane < L ? __ldcg(rg_tag_ptr(P, pr.par, lane)) : 0u;
    const uint32_t t1 = lane + 32 < L ? __ldcg(rg_tag_ptr(P, pr.par, lane + 32)) : 0u;
    if (lane < L) C.rt_tag[lane] = t0;
    if (lane + 32 < L) C.rt_tag[lane + 32] = t1;
  }
  __syncwarp();
  // (the previous-token validity of each head's layer is settled when its route is
  // published: publish_route)
}

// Publish the staged route of a prerouted layer (committed by the previous launch).
__device__ __forceinline__ void publish_staged_route(Prod& pr, int l) {
  Ctl& C = pr.C;
  const bool fresh = C.rt_tag[l] == pr.epoch;
  int id = -1;
  float w = 0.f;
  if (pr.lane < pr.P.K && fresh) {
    id = C.rt_ids[l][pr.lane];
    w = C.rt_w[l][pr.lane];
  }
  __syncwarp();
  if (!fresh && pr.lane == 0) raise_error(pr.P, C, E0_DEV_BAD_ID);  // not the step after the last one
  publish_route(pr, l, id, w);
}

// Bounded wait helper for the producer warp: true while we may keep waiting.
__device__ __forceinline__ bool prod_keep_waiting(Prod& pr, uint64_t t0, uint32_t it) {
  if ((it & 15u) != 0) return true;
  bool go = true;
  if (pr.lane == 0) {
    if (aborted(pr.P, pr.C)) {
      go = false;
    } else if (globaltimer() - t0 > pr.P.timeout_ns) {
      raise_error(pr.P, pr.C, E0_DEV_TIMEOUT);
      go = false;
    }
  }
  return __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
}

// Wait (bounded) until counter `which` of layer l has every CTA's arrival.
__device__ __forceinline__ bool prod_wait_counter(Prod& pr, int l, int which, uint32_t target) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    bool r = false;
    if (pr.lane == 0) r = ld_acquire_u32(ctr(pr.P, pr.par, l, which)) >= target;
    if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0)) return true;
    if (!prod_keep_waiting(pr, t0, it)) return false;
  }
}

// A layer that routes with its own gate: wait until every CTA wrote its gate rows,
// then publish the top-K of the gate logits (routing warp).
template <int NPL>
__device__ __forceinline__ void self_route_regs(Prod& pr, int l) {
  const EngineParams& P = pr.P;
  const uint64_t* z = zr_ptr(P, pr.par, l);
  const uint32_t tag = pr.epoch + 1u;
  float zv[NPL];
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    bool have = true;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = pr.lane + 32 * j;
      zv[j] = 0.f;
      if (e < P.E) {
        const uint64_t w = ld_relaxed_u64(z + e);
        have = have && (uint32_t)(w >> 32) == tag;
        zv[j] = __uint_as_float((uint32_t)w);
        if (P.mode == MODE_STACK && P.logit_bias) zv[j] += P.logit_bias[(size_t)l * P.E + e];
      }
    }
    if (__all_sync(0xffffffffu, have)) break;
    if (!prod_keep_waiting(pr, t0, it)) {
      pr.ok = false;
      return;
    }
  }
  if (P.z_trace && blockIdx.x == 0) {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = pr.lane + 32 * j;
      if (e < P.E) P.z_trace[(size_t)l * P.E + e] = zv[j];
    }
  }
  int id;
  float w;
  if (P.route == ROUTE_SIGMOID_GROUP) {
    // (the routing warp owns zbuf in the stack)
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = pr.lane + 32 * j;
      if (e < P.E) pr.C.zbuf[e] = zv[j];
    }
    __syncwarp();
    route_sigmoid_group(P, pr.C.zbuf, layer_at(P, l).score_bias, pr.lane, id, w);
    __syncwarp();
  } else {
    float val;
    warp_topk_regs<NPL>(zv, P.E, P.K, pr.lane, id, val);
    const float v0 = __shfl_sync(0xffffffffu, val, 0);
    w = pr.lane < P.K && id >= 0 ? expf(val - v0) : 0.f;  // unnormalised: publish_route normalises
  }
  publish_route(pr, l, pr.lane < P.K ? id : -1, pr.lane < P.K && id >= 0 ? w : 0.f);
}

// A layer that routes with its own gate: wait until every gate logit of this launch
// is published (tagged words, see st_tagged), then publish their top-K (routing warp).
__device__ __forceinline__ void compute_self_route(Prod& pr, int l) {
  if (!pr.ok || pr.C.rt_ready[l]) return;
  if (pr.lane == 0) stamp(pr.P, l, 8);
  if (pr.P.E <= 256)
    self_route_regs<8>(pr, l);
  else if (pr.P.E <= 512)
    self_route_regs<16>(pr, l);
  else
    self_route_regs<32>(pr, l);
}

// Producer: wait (bounded) until the routing warp has published layer l's route.
__device__ __forceinline__ void need_route(Prod& pr, int l) {
  if (!pr.ok || pr.C.rt_ready[l]) return;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; !mbar_try_wait(&pr.C.rt_bar[l], 0u); ++it) {
    if (!prod_keep_waiting(pr, t0, it)) {
      pr.ok = false;
      return;
    }
  }
}

// Wait until stage n's slot is free; returns its base (nullptr after an abort).
__device__ __forceinline__ uint8_t* prod_begin(Prod& pr, uint32_t& slot) {
  slot = pr.n % NSTAGES;
  const uint32_t round = pr.n / NSTAGES;
  if (round > 0) {
    uint64_t* bar = &pr.C.empty[slot];
    const uint32_t par = (round - 1) & 1u;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      bool fr = false;
      if (pr.lane == 0) fr = mbar_try_wait(bar, par);
      if (__shfl_sync(0xffffffffu, fr ? 1 : 0, 0)) break;
      if (!prod_keep_waiting(pr, t0, it)) {
        pr.ok = false;
        return nullptr;
      }
    }
  }
  return pr.ring + (size_t)slot * STAGE_BYTES;
}

// Per-lane bounded wait until stage m's slot is free (lanes of the copy warp wait on
// different slots at once).  False after an abort or a timeout.
__device__ __forceinline__ bool lane_wait_slot(Prod& pr, uint32_t m) {
  const uint32_t round = m / NSTAGES;
  if (round == 0) return true;
  uint64_t* bar = &pr.C.empty[m % NSTAGES];
  const uint32_t par = (round - 1) & 1u;
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, par)) return true;
    if ((it & 15u) == 0) {
      if (aborted(pr.P, pr.C)) return false;
      if (globaltimer() - t0 > pr.P.timeout_ns) {
        raise_error(pr.P, pr.C, E0_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Issue stages pr.n .. pr.n + nst - 1 (nst <= NSTAGES: distinct slots) at once, lane i
// taking stage pr.n + i:
// stage i < nq holds int4 rows [row0 + i * per, ...) of a row-layout matrix (in columns);
// the rest come from `extra` (a callable issuing stage i's copies into its slot).
template <class Extra>
__device__ __forceinline__ void issue_parallel(Prod& pr, int nst, int nq, const uint32_t* q, const uint16_t* s,
                                               const uint16_t* b, int in, int row0, int row1, Extra extra) {
  if (!pr.ok) return;
  bool ok = true;
  if (pr.lane < nst) {
    const uint32_t m = pr.n + (uint32_t)pr.lane, slot = m % NSTAGES;
    ok = lane_wait_slot(pr, m);
    if (ok) {
      uint8_t* st = pr.ring + (size_t)slot * STAGE_BYTES;
      if (pr.lane < nq) {
        const int per = q4_rows_per_stage(in);
        const int r = row0 + pr.lane * per, nr = min(per, row1 - r);
        const uint32_t qb = (uint32_t)nr * in / 2, sb = (uint32_t)nr * in / 32;
        mbar_arrive_expect_tx(&pr.C.full[slot], qb + 2 * sb);
        tma_bulk_g2s(st, q + (size_t)r * (in / 8), qb, &pr.C.full[slot]);
        tma_bulk_g2s(st + qb, s + (size_t)r * (in / 64), sb, &pr.C.full[slot]);
        tma_bulk_g2s(st + qb + sb, b + (size_t)r * (in / 64), sb, &pr.C.full[slot]);
      } else {
        extra(pr.lane, st, &pr.C.full[slot]);
      }
    }
  }
  if (!__all_sync(0xffffffffu, ok)) pr.ok = false;
  pr.n += (uint32_t)nst;
}

__device__ __forceinline__ void issue_bytes(Prod& pr, const void* src, uint32_t bytes) {
  if (!pr.ok) return;
  uint32_t slot;
  uint8_t* st = prod_begin(pr, slot);
  if (!st) return;
  if (pr.lane == 0) {
    mbar_arrive_expect_tx(&pr.C.full[slot], bytes);
    tma_bulk_g2s(st, src, bytes, &pr.C.full[slot]);
  }
  ++pr.n;
}

// Issue bf16 rows [row0, row1) of a [rows][in] matrix, in stage-sized chunks.
__device__ __forceinline__ void issue_bf_rows(Prod& pr, const uint16_t* m, int in, int row0, int row1) {
  const int per = bf_rows_per_stage(in);
  for (int r = row0; r < row1; r += per) issue_bytes(pr, m + (size_t)r * in, (uint32_t)min(per, row1 - r) * in * 2);
}

__device__ __forceinline__ void issue_unit(Prod& pr, const LayerDesc& Ld, const Unit& u, int l) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const int d = P.d;
  switch (u.type) {
    case U_EXPERT: {
      const bool shared = u.k >= P.K;
      if (!shared) need_route(pr, l);
      if (!pr.ok) return;
      if (shared ? !Ld.has_shared : !((C.rt_valid[l] >> u.k) & 1u)) return;
      const int idx = shared ? 0 : C.rt_idx[l][u.k];
      // a stored expert: dense per-tensor arrays, or one bundle per slot (slot pools)
      const int64_t xs = shared ? 0 : Ld.ex_stride;
      auto at = [&](const auto* base, size_t dense_elems) {
        return xs ? reinterpret_cast<decltype(base)>(reinterpret_cast<const uint8_t*>(base) + (size_t)idx * xs)
                  : base + (size_t)idx * dense_elems;
      };
      const uint32_t* guq = at(shared ? Ld.sgu_q : Ld.gu_q, (size_t)(2 * P.F) * (d / 8));
      const uint16_t* gus = at(shared ? Ld.sgu_s : Ld.gu_s, (size_t)(2 * P.F) * (d / 64));
      const uint16_t* gub = at(shared ? Ld.sgu_b : Ld.gu_b, (size_t)(2 * P.F) * (d / 64));
      const int per = q4_rows_per_stage(d);
      const uint32_t* dq = at(shared ? Ld.sdn_q : Ld.dn_q, (size_t)(P.F / 32) * d * 4) + (size_t)u.r0 * d * 4;
      const uint16_t* ds = at(shared ? Ld.sdn_s : Ld.dn_s, (size_t)(P.F / 64) * d) + (size_t)(u.r0 >> 1) * d;
      const uint16_t* db = at(shared ? Ld.sdn_b : Ld.dn_b, (size_t)(P.F / 64) * d) + (size_t)(u.r0 >> 1) * d;
      const int pd = dn_rows_per_stage(d);
      const int ngu = (64 + per - 1) / per, ndn = (d + pd - 1) / pd;
      // the gate/up stages and the down-projection stages of the slab, one lane each
      issue_parallel(pr, ngu + ndn, ngu, guq, gus, gub, d, 64 * u.r0, 64 * u.r0 + 64,
                     [&](int i, uint8_t* st, uint64_t* full) {
                       const int i0 = (i - ngu) * pd, nr = min(pd, d - i0);
                       mbar_arrive_expect_tx(full, (uint32_t)nr * 20);
                       tma_bulk_g2s(st, dq + (size_t)i0 * 4, nr * 16, full);
                       tma_bulk_g2s(st + nr * 16, ds + i0, nr * 2, full);
                       tma_bulk_g2s(st + nr * 18, db + i0, nr * 2, full);
                     });
      break;
    }
    case U_QROWS: {
      const int per = q4_rows_per_stage(d);
      for (int r0 = u.r0; r0 < u.r1; r0 += NSTAGES * per) {  // up to a ring's worth of stages at once
        const int r1 = min((int)u.r1, r0 + NSTAGES * per), nst = (r1 - r0 + per - 1) / per;
        issue_parallel(pr, nst, nst, Ld.lw_q, Ld.lw_s, Ld.lw_b, d, r0, r1, [](int, uint8_t*, uint64_t*) {});
      }
      break;
    }
    case U_LORA_B: {
      // one stage: Bt[q][r0, r1) for every rank q, stored [q][row]
      const int nr = u.r1 - u.r0;
      uint32_t slot;
      uint8_t* st = prod_begin(pr, slot);
      if (!st) return;
      if (pr.lane == 0) {
        mbar_arrive_expect_tx(&C.full[slot], (uint32_t)(Ld.lr * nr * 2));
        for (int q = 0; q < Ld.lr; ++q)
          tma_bulk_g2s(st + (size_t)q * nr * 2, Ld.lbt + (size_t)q * Ld.lout + u.r0, (uint32_t)nr * 2,
                       &C.full[slot]);
      }
      ++pr.n;
      break;
    }
    case U_LORA_A: {
      issue_bf_rows(pr, Ld.la, d, u.r0, u.r1);
      break;
    }
    case U_HEAD: {
      issue_bf_rows(pr, Ld.w1h, d, u.r0, u.r1);
      need_route(pr, l);
      if (!pr.ok) return;
      const int nr = u.r1 - u.r0;
      const uint32_t slotb = (uint32_t)nr * 2;
      uint32_t slot;
      uint8_t* st = prod_begin(pr, slot);
      if (!st) return;
      if (pr.lane == 0) {
        const uint32_t cv = C.rt_valid[l], pv = C.rt_pvalid[l];
        uint32_t bytes = 0;
        if (Ld.b1) bytes += slotb;
        for (int k = 0; k < P.K; ++k) {
          if ((cv >> k) & 1u) bytes += slotb;
          if ((pv >> k) & 1u) bytes += slotb;
        }
        mbar_arrive_expect_tx(&C.full[slot], bytes);
        if (Ld.b1) tma_bulk_g2s(st, Ld.b1 + u.r0, slotb, &C.full[slot]);
        for (int k = 0; k < P.K; ++k) {
          if ((cv >> k) & 1u)
            tma_bulk_g2s(st + (1 + k) * slotb, Ld.w1c_t + (size_t)C.rt_ids[l][k] * Ld.H + u.r0, slotb,
                         &C.full[slot]);
          if ((pv >> k) & 1u)
            tma_bulk_g2s(st + (1 + P.K + k) * slotb, Ld.w1p_t + (size_t)C.rt_prev[l][k] * Ld.H + u.r0, slotb,
                         &C.full[slot]);
        }
      }
      ++pr.n;
      const int per = max(1, STAGE_BYTES / (2 * P.E));
      for (int i = u.r0; i < u.r1; i += per)
        issue_bytes(pr, Ld.w2t + (size_t)i * P.E, (uint32_t)min(per, u.r1 - i) * P.E * 2);
      break;
    }
    case U_LRES:
      issue_bf_rows(pr, Ld.lres, d, u.r0, u.r1);
      break;
    case U_ROUTER:
      issue_bf_rows(pr, Ld.router, d, u.r0, u.r1);
      break;
    default:
      break;
  }
}

// L2 prefetch of the weight rows of one of this CTA's units (addresses as issue_unit
// computes them); the routed expert slabs only once their layer's route is published.
// Lanes take the contiguous ranges round robin.
__device__ __forceinline__ void prefetch_unit(Prod& pr, const LayerDesc& Ld, const Unit& u, int l) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const int d = P.d;
  int n = 0;  // ranges seen so far: lane n issues range n
  auto add = [&](const void* p, size_t b) {
    if (p && b >= 16) {
      if (pr.lane == n) l2_prefetch(p, (uint32_t)(b & ~size_t(15)));
      ++n;
    }
  };
  switch (u.type) {
    case U_EXPERT: {
      const bool shared = u.k >= P.K;
      if (shared ? !Ld.has_shared : (!C.rt_ready[l] || !((C.rt_valid[l] >> u.k) & 1u))) return;
      const int idx = shared ? 0 : C.rt_idx[l][u.k];
      const int64_t xs = shared ? 0 : Ld.ex_stride;
      auto at = [&](const auto* base, size_t dense_elems) {
        return xs ? reinterpret_cast<decltype(base)>(reinterpret_cast<const uint8_t*>(base) + (size_t)idx * xs)
                  : base + (size_t)idx * dense_elems;
      };
      const uint32_t* guq = at(shared ? Ld.sgu_q : Ld.gu_q, (size_t)(2 * P.F) * (d / 8));
      const uint16_t* gus = at(shared ? Ld.sgu_s : Ld.gu_s, (size_t)(2 * P.F) * (d / 64));
      const uint16_t* gub = at(shared ? Ld.sgu_b : Ld.gu_b, (size_t)(2 * P.F) * (d / 64));
      const size_t r0 = 64 * (size_t)u.r0;
      add(guq + r0 * (d / 8), (size_t)64 * d / 2);
      add(gus + r0 * (d / 64), (size_t)64 * (d / 64) * 2);
      add(gub + r0 * (d / 64), (size_t)64 * (d / 64) * 2);
      add(at(shared ? Ld.sdn_q : Ld.dn_q, (size_t)(P.F / 32) * d * 4) + (size_t)u.r0 * d * 4, (size_t)d * 16);
      add(at(shared ? Ld.sdn_s : Ld.dn_s, (size_t)(P.F / 64) * d) + (size_t)(u.r0 >> 1) * d, (size_t)d * 2);
      add(at(shared ? Ld.sdn_b : Ld.dn_b, (size_t)(P.F / 64) * d) + (size_t)(u.r0 >> 1) * d, (size_t)d * 2);
      break;
    }
    case U_QROWS:
      add(Ld.lw_q + (size_t)u.r0 * (d / 8), (size_t)(u.r1 - u.r0) * d / 2);
      add(Ld.lw_s + (size_t)u.r0 * (d / 64), (size_t)(u.r1 - u.r0) * (d / 64) * 2);
      add(Ld.lw_b + (size_t)u.r0 * (d / 64), (size_t)(u.r1 - u.r0) * (d / 64) * 2);
      break;
    case U_LORA_A:
      add(Ld.la + (size_t)u.r0 * d, (size_t)(u.r1 - u.r0) * d * 2);
      break;
    case U_HEAD:
      add(Ld.w1h + (size_t)u.r0 * d, (size_t)(u.r1 - u.r0) * d * 2);
      add(Ld.w2t + (size_t)u.r0 * P.E, (size_t)(u.r1 - u.r0) * P.E * 2);
      break;
    case U_LRES:
      add(Ld.lres + (size_t)u.r0 * d, (size_t)(u.r1 - u.r0) * d * 2);
      break;
    default:
      break;
  }
}

// L2 prefetch of layer l's units of this CTA (issued one layer ahead of the stage ring,
// so that DRAM keeps streaming through the grid-wide waits between layers).
__device__ __forceinline__ void prefetch_layer(Prod& pr, int l) {
  const EngineParams& P = pr.P;
  if (l >= P.L || !pr.ok) return;
  const LayerDesc& Ld = layer_at(P, l);
  int nu;
  const Unit* us = units_of(P, P.plan ? Ld.plan_kind : 0, blockIdx.x, nu);
  for (int i = 0; i < nu; ++i) prefetch_unit(pr, Ld, us[i], l);
}

__device__ void producer(const EngineParams& P, Ctl& C, uint8_t* ring) {
  Prod pr{P, C, ring, 0u, true, (int)(threadIdx.x & 31), C.epoch & 1u, C.epoch % 3u, C.epoch};
  for (int l = 0; l < P.L && pr.ok; ++l) {
    const LayerDesc& Ld = layer_at(P, l);
    prefetch_layer(pr, l + 1);
    // gate rows on this layer's input: its own gate, then the gate of the layer that
    // routes ahead from here
    const uint16_t* gates[2] = {gate_here(P, l) ? Ld.router : nullptr,
                                P.mode == MODE_STACK && Ld.gate_for >= 0 ? layer_at(P, Ld.gate_for).router : nullptr};
    for (int g = 0; g < 2; ++g) {
      if (!gates[g]) continue;
      int nu;
      const Unit* us = units_of(P, KIND_ROUTER, blockIdx.x, nu);
      for (int i = 0; i < nu; ++i) issue_bf_rows(pr, gates[g], P.d, us[i].r0, us[i].r1);
    }
    int nu;
    const Unit* us = units_of(P, P.plan ? Ld.plan_kind : 0, blockIdx.x, nu);
    for (int i = 0; i < nu; ++i) issue_unit(pr, Ld, us[i], l);
    if (pr.lane == 0) stamp(P, l, 5);
  }
  // Wait for every issued copy to land before the CTA may exit.
  if (pr.lane == 0) {
    const uint32_t n = pr.n;
    for (uint32_t s = 0; s < NSTAGES && s < n; ++s) {
      const uint32_t last_round = (n - 1 - s) / NSTAGES;
      uint64_t* bar = &C.full[s];
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar, last_round & 1u)) {
        if (globaltimer() - t0 > P.timeout_ns) {
          atomicOr(&hdr(P)->status, (uint32_t)E0_DEV_TIMEOUT);
          break;
        }
      }
    }
  }
}

// The CTA that keeps the books of layer l: one of the CTAs that hold the prerouter's
// deferred work when there are any (they hold no work of the layers after the last
// head, so their routing warps may wait for the heads without holding up a route that
// their consumers need), else CTA l.
__device__ __forceinline__ int bookkeeper(const EngineParams& P, int l) {
  const int nd = P.plan ? P.n_defer[KIND_MAIN] : 0;
  return nd > 0 ? P.ncta - 1 - l % nd : l % P.ncta;
}

// Stack bookkeeping of layer l on CTA bookkeeper(l), once its route is published:
// record the ids the layer used (the heads' previous-token one-hot at the next step)
// and commit the next token's routing of a head-routed layer: the top-K of the logits
// the previous layer's head produced.
__device__ __forceinline__ void bookkeep_layer(Prod& pr, int l) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  if (bookkeeper(P, l) != (int)blockIdx.x) return;
  {
    const uint32_t pnext3 = (pr.epoch + 1) % 3u;
    {
      need_route(pr, l);
      if (!pr.ok) return;
      if (pr.lane < P.K) {
        const bool v = (C.rt_valid[l] >> pr.lane) & 1u;
        const int id = v ? C.rt_ids[l][pr.lane] : -1;
        idsu_ptr(P, pr.par, l)[pr.lane] = id;
        wu_ptr(P, pr.par, l)[pr.lane] = C.rt_w[l][pr.lane];
        if (P.ids_trace) P.ids_trace[l * P.K + pr.lane] = id;
        if (P.w_trace) P.w_trace[l * P.K + pr.lane] = C.rt_w[l][pr.lane];
      }
      if (layer_at(P, l).prerouted && l > 0) {
        // head l-1 done: on its own counter when that work runs on deferred CTAs
        const int hk = layer_at(P, l - 1).plan_kind;
        const bool on_head = P.plan && P.n_defer[hk] > 0;
        if (!prod_wait_counter(pr, l - 1, on_head ? 1 : 0,
                               (uint32_t)(on_head ? P.n_defer[hk] : (P.plan ? P.n_arrive[hk] : P.ncta)))) {
          pr.ok = false;
          return;
        }
        const float* z = zhat_ptr(P, pnext3, l - 1);
#pragma unroll 8
        for (int e = pr.lane; e < P.E; e += 32) {
          const float v = __ldcg(z + e) + (P.logit_bias ? P.logit_bias[((size_t)P.L + l) * P.E + e] : 0.f);
          C.zbuf[e] = v;
          if (P.z_trace) P.z_trace[((size_t)P.L + l) * P.E + e] = v;
        }
        __syncwarp();
        int id;
        float w;
        route_smem(P, C.zbuf, layer_at(P, l).score_bias, pr.lane, id, w);
        if (pr.lane < P.K) {
          rg_ids_ptr(P, pr.par ^ 1u, l)[pr.lane] = id;
          rg_w_ptr(P, pr.par ^ 1u, l)[pr.lane] = w;
          if (P.next_ids_out) P.next_ids_out[l * P.K + pr.lane] = id;
        }
        if (P.commit_box) {
          // the committed ids, then the token they are for, into host-mapped memory: the
          // host can stage this layer's experts while the launch goes on
          uint32_t* box = P.commit_box + ((size_t)((P.step + 1) & 1) * P.L + l) * (KMAX + 1);
          if (pr.lane < P.K) box[1 + pr.lane] = (uint32_t)id;
          __syncwarp();
          if (pr.lane == 0) {
            __threadfence_system();
            *reinterpret_cast<volatile uint32_t*>(box) = (uint32_t)(P.step + 1);
          }
        }
        __syncwarp();
        if (pr.lane == 0) *rg_tag_ptr(P, pr.par ^ 1u, l) = pr.epoch + 1u;
      } else if (P.next_ids_out && pr.lane < P.K) {
        P.next_ids_out[l * P.K + pr.lane] = -1;  // no head commits this layer's routing
      }
    }
  }
}

// Routing warp: publishes every layer's route in the route table (routes known at
// launch, then the layers that route with their own gate as their gate logits
// complete) and, in the stack, the bookkeeping for the next token.
__device__ void router_warp(const EngineParams& P, Ctl& C) {
  Prod pr{P, C, nullptr, 0u, true, (int)(threadIdx.x & 31), C.epoch & 1u, C.epoch % 3u, C.epoch};
  // The steps in order, each kind from a single call site (so that its code is still in
  // the instruction cache when the next layer needs it):
  //   A  the own-gate routes of the leading layers without a head: they need nothing
  //      staged (the staging takes several microseconds; a head's layer needs its
  //      previous-token ids)
  //   S  the staged routes and previous-token ids (load_routes)
  //   B  the routes up to the last layer not routed from gate logits
  //   C  this CTA's bookkeeping of those layers (a committed route leaves as soon as its
  //      head is done, while the launch goes on)
  //   D  the trailing gate-routed layers, E  their bookkeeping
  const bool stack = P.mode == MODE_STACK;
  int lead = 0, lc = 0;
  if (stack) {
    while (lead < P.L && self_routes(P, lead) && !layer_at(P, lead).has_head) ++lead;
    for (int l = 0; l < P.L; ++l)
      if (!self_routes(P, l)) lc = l + 1;
    lc = max(lc, lead);
  }
  const int eA = lead, eS = eA + 1, eB = eS + (lc - lead), eC = eB + lc, eD = eC + (P.L - lc);
  const int total = stack ? eD + (P.L - lc) : 1;
  for (int st = 0; st < total && pr.ok; ++st) {
    int act = 3, l = 0;  // 0 own-gate route, 1 staged route, 2 bookkeeping, 3 load_routes
    if (stack) {
      if (st < eA) {
        act = 0;
        l = st;
      } else if (st < eS) {
        act = 3;
      } else if (st < eB) {
        l = lead + st - eS;
        act = self_routes(P, l) ? 0 : 1;
      } else if (st < eC) {
        act = 2;
        l = st - eB;
      } else if (st < eD) {
        act = 0;
        l = lc + st - eC;
      } else {
        act = 2;
        l = lc + st - eD;
      }
    }
    if (act == 0)
      compute_self_route(pr, l);
    else if (act == 1)
      publish_staged_route(pr, l);
    else if (act == 2)
      bookkeep_layer(pr, l);
    else
      load_routes(pr);
  }
  // After an abort, mark every route published so that no consumer waits on one.
  if (pr.lane == 0 && !pr.ok)
    for (int l = 0; l < P.L; ++l) mark_route(C, l);
}

// ------------------------------------------------------------------ consumers
constexpr int GMAX = 4;  // stages a consumer holds at once (the ring has NSTAGES)

struct Cons {
  const EngineParams& P;
  Ctl& C;
  uint8_t* ring;
  uint32_t n;  // stages consumed
  int cw, lane, tid;
  uint64_t t_acq = 0;   // diagnostics (warp 0, lane 0): time waiting for stages
  uint64_t n_acq = 0;   // stages acquired in the current layer
  uint32_t nx = 0;      // expert slabs consumed (selects the activation buffer)

  __device__ __forceinline__ const uint8_t* stage(int i) const {
    return ring + (size_t)((n + i) % NSTAGES) * STAGE_BYTES;
  }
  // Wait until the next cnt stages (cnt <= GMAX) have landed.  False on abort.
  __device__ __forceinline__ bool acquire(int cnt) {
    const bool timed = P.trace && tid == 0;
    const uint64_t t0 = timed ? globaltimer() : 0;
    bool ok = true;
    // fast path: all the stages have landed (the usual case: the copy warp runs ahead)
    {
      const uint64_t* bar[4];
      uint32_t par[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t m = n + (uint32_t)min(i, cnt - 1);
        bar[i] = &C.full[m % NSTAGES];
        par[i] = (m / NSTAGES) & 1u;
      }
      if (!mbar_try_wait4(bar[0], par[0], bar[1], par[1], bar[2], par[2], bar[3], par[3]))
        for (int i = 0; i < cnt && ok; ++i) {
          const uint32_t m = n + i;
          ok = wait_mbar(P, C, &C.full[m % NSTAGES], (m / NSTAGES) & 1u);
        }
    }
    if (timed) {
      t_acq += globaltimer() - t0;
      n_acq += cnt;
    }
    // warp-uniform, so that the shuffles that follow a successful acquire see every lane
    return __all_sync(0xffffffffu, ok);
  }
  // Wait until the routing warp has published layer l's route (every lane waits on the
  // layer's mbarrier: a single waiting lane followed by a warp barrier measured several
  // times slower in the code that follows).
  __device__ __forceinline__ void wait_route(int l) { wait_mbar(P, C, &C.rt_bar[l], 0u); }
  // This warp is done reading the next cnt stages.
  __device__ void release(int cnt) {
    __syncwarp();
    if (lane == 0)
      for (int i = 0; i < cnt; ++i) mbar_arrive(&C.empty[(n + i) % NSTAGES]);
    n += cnt;
  }
};

template <int D>
struct Q4Frag {
  static constexpr int LPR = (D / 32) < 32 ? (D / 32) : 32;   // lanes per row
  static constexpr int RPW = 32 / LPR;                         // rows per warp pass
  static constexpr int CPL = (D / 32) / LPR;                   // 32-element chunks per lane
  uint32_t xp[CPL][16];
  float inv[CPL], sum[CPL];
  __device__ __forceinline__ void load(const Ctl& C, int lane) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane % LPR + LPR * j;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint4 v = C.xq[t][c];
        xp[j][4 * t] = v.x; xp[j][4 * t + 1] = v.y; xp[j][4 * t + 2] = v.z; xp[j][4 * t + 3] = v.w;
      }
      inv[j] = C.xinv[c];
      sum[j] = C.xsum[c];
    }
  }
};

// Lane partial of row `lr` of an int4 stage holding `nr` rows (row layout, in = D).
template <int D>
__device__ __forceinline__ float q4_partial(const uint8_t* st, int nr, int lr, int lane, const Q4Frag<D>& f) {
  constexpr int LPR = Q4Frag<D>::LPR, CPL = Q4Frag<D>::CPL;
  const uint4* q = reinterpret_cast<const uint4*>(st);
  const uint16_t* s = reinterpret_cast<const uint16_t*>(st + (size_t)nr * D / 2);
  const uint16_t* b = s + nr * (D / 64);
  float v = 0.f;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane % LPR + LPR * j;
    const int a = dot32(q[lr * (D / 32) + c], f.xp[j]);
    const float sf = bf(s[lr * (D / 64) + (c >> 1)]);
    const float bb = bf(b[lr * (D / 64) + (c >> 1)]);
    v += sf * ((float)a * f.inv[j]) + bb * f.sum[j];
  }
  return v;
}

template <int LPR>
__device__ __forceinline__ float reduce_lpr(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// A group of int4 stages holding rows [g0, g0 + R) of a part cut into stages of `per`
// rows (part_rows rows in total).  When a row takes a whole warp (D >= 1024) the rows go
// to warps round robin, up to NI1 rows per warp and pass (64 rows: 4 or 5 per warp);
// otherwise items of IR rows go to warps round robin, up to NI items per warp and pass.
// GU: each row value goes to abuf[row] (rows 2j / 2j + 1 are gate / up of activation j,
// combined by the caller).  Otherwise each row value is added to out[row0 + row].
template <int D, bool GU>
__device__ __forceinline__ void q4_group(const Cons& cs, int g0, int R, int per, int part_rows,
                                         const Q4Frag<D>& f, float* abuf, float* out, int row0) {
  constexpr int LPR = Q4Frag<D>::LPR, RPW = Q4Frag<D>::RPW;
  const int lane = cs.lane;
  if constexpr (RPW == 1) {
    constexpr int NI1 = 5;
    for (int it = cs.cw; it < R; it += NI1 * NCW) {
      float v[NI1];
#pragma unroll
      for (int u = 0; u < NI1; ++u) {
        v[u] = 0.f;
        if (it + u * NCW < R) {
          const int rho = g0 + it + u * NCW;  // row within the part
          const int si = rho / per - g0 / per;
          const int nr = min(per, part_rows - (rho / per) * per);
          v[u] = q4_partial<D>(cs.stage(si), nr, rho % per, lane, f);
        }
      }
#pragma unroll
      for (int u = 0; u < NI1; ++u) v[u] = reduce_lpr<LPR>(v[u]);
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < NI1; ++u) {
          if (it + u * NCW >= R) break;
          const int row = g0 + it + u * NCW;
          if (GU)
            abuf[row] = v[u];
          else
            red_add_f32(out + row0 + row, v[u]);
        }
      }
    }
    return;
  }
  constexpr int IR = RPW > 2 ? RPW : 2;
  constexpr int NP = IR / RPW;
  constexpr int NI = 3;
  const int items = R / IR;
  for (int it = cs.cw; it < items; it += NI * NCW) {
    float v[NI][NP];
#pragma unroll
    for (int u = 0; u < NI; ++u) {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        v[u][p] = 0.f;
        if (it + u * NCW < items) {
          const int rho = g0 + (it + u * NCW) * IR + p * RPW + lane / LPR;  // row within the part
          const int si = rho / per - g0 / per;
          const int nr = min(per, part_rows - (rho / per) * per);
          v[u][p] = q4_partial<D>(cs.stage(si), nr, rho % per, lane, f);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < NI; ++u)
#pragma unroll
      for (int p = 0; p < NP; ++p) v[u][p] = reduce_lpr<LPR>(v[u][p]);
#pragma unroll
    for (int u = 0; u < NI; ++u) {
      if (it + u * NCW >= items) break;
      const int rbase = g0 + (it + u * NCW) * IR;
      if (lane % LPR == 0) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          if (GU)
            abuf[rbase + p * RPW + lane / LPR] = v[u][p];
          else
            red_add_f32(out + row0 + rbase + p * RPW + lane / LPR, v[u][p]);
        }
      }
    }
  }
}

// Consume the int4 rows [0, rows) of a part in groups of at most GMAX stages.
template <int D, bool GU>
__device__ __forceinline__ void consume_q4_part(Cons& cs, int rows, float* abuf, float* out, int row0) {
  Q4Frag<D> f;
  f.load(cs.C, cs.lane);
  const int per = q4_rows_per_stage(D);
  const int nst = (rows + per - 1) / per;
  for (int s0 = 0; s0 < nst; s0 += GMAX) {
    const int cnt = min(GMAX, nst - s0);
    const int g0 = s0 * per, R = min(rows, (s0 + cnt) * per) - g0;
    if (cs.acquire(cnt)) q4_group<D, GU>(cs, g0, R, per, rows, f, abuf, out, row0);
    cs.release(cnt);
  }
}

template <int D>
struct BfFrag {
  static constexpr int NV = D / 128;  // float4 groups per lane: lane owns elements 4 (lane + 32 j) .. + 3
  float x[NV][4];                     // residual h; the row dot is scaled by sc afterwards
  float sc;                           // RMSNorm factor: x = h * sc
  __device__ __forceinline__ void load(const Ctl& C, int lane) {
    sc = C.xscale;
    const float4* p = reinterpret_cast<const float4*>(C.res);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float4 a = p[lane + 32 * j];  // consecutive lanes, consecutive 16 bytes
      x[j][0] = a.x; x[j][1] = a.y; x[j][2] = a.z; x[j][3] = a.w;
    }
  }
};

// Lane partial of w . x for one bf16 row (x = h * sc); the lane reads 4 bf16 (8 bytes)
// per group, so a warp reads 256 contiguous bytes per load.
template <int D>
__device__ __forceinline__ float bf_partial(const uint8_t* row, int lane, const BfFrag<D>& f) {
  const uint2* w = reinterpret_cast<const uint2*>(row);
  float v0 = 0.f, v1 = 0.f;
#pragma unroll
  for (int j = 0; j < BfFrag<D>::NV; ++j) {
    const uint2 u = w[lane + 32 * j];
    v0 = fmaf(bflo(u.x), f.x[j][0], v0); v1 = fmaf(bfhi(u.x), f.x[j][1], v1);
    v0 = fmaf(bflo(u.y), f.x[j][2], v0); v1 = fmaf(bfhi(u.y), f.x[j][3], v1);
  }
  return (v0 + v1) * f.sc;
}

// Where consume_bf_rows puts a row value: a shared buffer (dst[row] = v), the head
// logits accumulator (dst[row] += v + bias[row]), or a layer's gate logits (dst[row] = v).
enum BfOut : int { BF_SMEM = 0, BF_ADD_BIAS = 1, BF_TAGGED = 2 };

// bf16 rows [0, rows) of a part (in = D), stages of bf_rows_per_stage(D) rows, in
// groups of at most GMAX stages; one warp per row, two rows per pass.
template <int D>
__device__ __forceinline__ void consume_bf_rows(Cons& cs, int rows, int mode, float* dst, const float* bias) {
  BfFrag<D> f;
  f.load(cs.C, cs.lane);
  const int per = bf_rows_per_stage(D);
  const int nst = (rows + per - 1) / per;
  for (int s0 = 0; s0 < nst; s0 += GMAX) {
    const int cnt = min(GMAX, nst - s0);
    const int g0 = s0 * per, R = min(rows, (s0 + cnt) * per) - g0;
    if (cs.acquire(cnt)) {
      for (int r = cs.cw; r < R; r += 2 * NCW) {
        const bool two = r + NCW < R;
        const int ra = g0 + r, rb = g0 + r + NCW;
        float va = bf_partial<D>(cs.stage(ra / per - s0) + (size_t)(ra % per) * 2 * D, cs.lane, f);
        float vb = two ? bf_partial<D>(cs.stage(rb / per - s0) + (size_t)(rb % per) * 2 * D, cs.lane, f) : 0.f;
        va = warp_sum(va);
        vb = warp_sum(vb);
        if (cs.lane == 0) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u == 1 && !two) break;
            const int row = u ? rb : ra;
            const float v = u ? vb : va;
            if (mode == BF_ADD_BIAS)
              red_add_f32(dst + row, v + (bias ? bias[row] : 0.f));
            else if (mode == BF_TAGGED)
              st_tagged(reinterpret_cast<uint64_t*>(dst) + row, cs.C.epoch + 1u, v);
            else
              dst[row] = v;
          }
        }
      }
    }
    cs.release(cnt);
  }
}

// dst[0, n) += scale * sum_r v[r] * W[r][0, n) over the nr bf16 rows W of one stage
// (n a multiple of 4, dst 16-byte aligned).  A thread owns 4 adjacent outputs; when
// there are fewer 4-output groups than threads, the rows are split between
// NCT / (n / 4) thread groups, each adding its partial sums with vector reductions.
__device__ __forceinline__ void bf_axpy_rows(const uint8_t* st, int nr, int n, const float* v, float scale,
                                             float* dst, int tid) {
  const int n4 = n >> 2;
  const int G = n4 >= NCT ? 1 : NCT / n4;
  const int rg = tid / n4;
  if (rg >= G) return;
  for (int c = tid % n4; c < n4; c += NCT) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int r = rg; r < nr; r += G) {
      const uint2 w = reinterpret_cast<const uint2*>(st + (size_t)r * 2 * n)[c];
      const float x = v[r];
      s0 = fmaf(bflo(w.x), x, s0);
      s1 = fmaf(bfhi(w.x), x, s1);
      s2 = fmaf(bflo(w.y), x, s2);
      s3 = fmaf(bfhi(w.y), x, s3);
    }
    red_add_v4_f32(dst + 4 * c, scale * s0, scale * s1, scale * s2, scale * s3);
  }
}

template <int D>
__device__ __forceinline__ void consume_unit(Cons& cs, const LayerDesc& Ld, const Unit& u, int l, float* acc, float* zhat,
                             float* zr) {
  const EngineParams& P = cs.P;
  Ctl& C = cs.C;
  const int tid = cs.tid;
  switch (u.type) {
    case U_EXPERT: {
      const bool shared = u.k >= P.K;
      if (!shared) cs.wait_route(l);
      // The named barrier below is executed unconditionally so that every warp
      // reaches it even if the route table were read inconsistently.
      const bool valid = shared ? Ld.has_shared != 0 : ((C.rt_valid[l] >> u.k) & 1u) != 0;
      // Two gate/up value buffers: a warp writes buffer (n & 1) of unit n only after the
      // barrier of unit n - 1, which every warp passes after reading buffer (n & 1) of
      // unit n - 2.
      float* ab = C.abuf[cs.nx & 1u];
      ++cs.nx;
      if (valid) consume_q4_part<D, true>(cs, 64, ab, nullptr, 0);
      cbar();  // all 64 gate/up values ready
      if (valid) {
        // Every warp forms and quantises the 32 activations itself (lane j holds
        // a_j = silu(gate_j) * up_j): one step
        // m / 32767 for the slab, m = max |a_j| (the bit patterns of non-negative
        // floats order like their values, so an unsigned max reduction finds it).
        const float a = silu_f(ab[2 * cs.lane]) * ab[2 * cs.lane + 1];
        const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(a))));
        const float r = m > 0.f ? __fdividef(32767.0f, m) : 0.f;
        const float ainv = m * (1.0f / 32767.0f);
        int q = __float2int_rn(a * r);
        q = q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
        const float asum = (float)__reduce_add_sync(0xffffffffu, q) * ainv;
        const int j = cs.lane, idx = j & 7;
        __syncwarp();  // the previous slab's reads of aqw are done
        reinterpret_cast<int16_t*>(C.aqw[cs.cw])[8 * (j >> 3) + ((idx & 1) ? 4 + (idx >> 1) : (idx >> 1))] =
            (int16_t)q;
        __syncwarp();
        uint32_t ap[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 v = C.aqw[cs.cw][t];
          ap[4 * t] = v.x; ap[4 * t + 1] = v.y; ap[4 * t + 2] = v.z; ap[4 * t + 3] = v.w;
        }
        const float wk = shared ? 1.0f : C.rt_w[l][u.k];
        const int pd = dn_rows_per_stage(D);
        constexpr int NDS = (D + 1023) / 1024;   // down-projection stages (<= 2)
        constexpr int RPT = (D + NCT - 1) / NCT;  // rows per thread (<= 5)
        static_assert(D % 32 == 0 && NCT % 32 == 0, "a warp owns whole 32-row blocks");
        if (cs.acquire(NDS)) {
#pragma unroll
          for (int m = 0; m < RPT; ++m) {
            const int base = 32 * cs.cw + NCT * m;  // this warp's 32 rows
            if (base < D) {                          // warp-uniform
              const int rho = base + cs.lane;
              const int si = rho / pd, lr = rho % pd, nr = min(pd, D - si * pd);
              const uint8_t* st = cs.stage(si);
              const uint4 qq = reinterpret_cast<const uint4*>(st)[lr];
              const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + nr * 16);
              const int a = dot32(qq, ap);
              const float v = wk * (bf(sc[lr]) * ((float)a * ainv) + bf(sc[nr + lr]) * asum);
              // lanes 0..7 add 4 consecutive rows each with one vector reduction
              const int src = 4 * (cs.lane & 7);
              const float t0 = __shfl_sync(0xffffffffu, v, src);
              const float t1 = __shfl_sync(0xffffffffu, v, src + 1);
              const float t2 = __shfl_sync(0xffffffffu, v, src + 2);
              const float t3 = __shfl_sync(0xffffffffu, v, src + 3);
              if (cs.lane < 8) red_add_v4_f32(acc + base + src, t0, t1, t2, t3);
            }
          }
        }
        cs.release(NDS);
      }
      break;
    }
    case U_QROWS:
      consume_q4_part<D, false>(cs, u.r1 - u.r0, nullptr, acc, u.r0);
      break;
    case U_LORA_B: {
      // (alpha/r) B v for rows [r0, r1), once every rank of v is published: warp 0
      // polls the launch-tagged words of v (one round trip when they are there)
      const uint32_t par = C.epoch & 1u;
      if (cs.cw == 0 && C.lv_layer != l) {  // (v computed on this CTA is already in lvs)
        const uint64_t* lvp = lv_ptr(P, par, l);
        const uint32_t tag = C.epoch + 1u;
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 1;; ++it) {
          bool have = true;
          float v0 = 0.f, v1 = 0.f;
          if (cs.lane < Ld.lr) {
            const uint64_t w = ld_relaxed_u64(lvp + cs.lane);
            have = (uint32_t)(w >> 32) == tag;
            v0 = __uint_as_float((uint32_t)w);
          }
          if (cs.lane + 32 < Ld.lr) {
            const uint64_t w = ld_relaxed_u64(lvp + cs.lane + 32);
            have = have && (uint32_t)(w >> 32) == tag;
            v1 = __uint_as_float((uint32_t)w);
          }
          if (__all_sync(0xffffffffu, have)) {
            if (cs.lane < Ld.lr) C.lvs[cs.lane] = v0;
            if (cs.lane + 32 < Ld.lr) C.lvs[cs.lane + 32] = v1;
            break;
          }
          if ((it & 15u) == 0) {
            int stop = 0;
            if (cs.lane == 0) {
              if (aborted(P, C)) {
                stop = 1;
              } else if (globaltimer() - t0 > P.timeout_ns) {
                raise_error(P, C, E0_DEV_TIMEOUT);
                stop = 1;
              }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
          }
        }
      }
      cbar();
      const int nr = u.r1 - u.r0;
      if (cs.acquire(1)) {
        const uint16_t* bt = reinterpret_cast<const uint16_t*>(cs.stage(0));
        for (int rho = tid; rho < nr; rho += NCT) {
          float s0 = 0.f, s1 = 0.f;
          int q = 0;
          for (; q + 1 < Ld.lr; q += 2) {
            s0 = fmaf(bf(bt[q * nr + rho]), C.lvs[q], s0);
            s1 = fmaf(bf(bt[(q + 1) * nr + rho]), C.lvs[q + 1], s1);
          }
          if (q < Ld.lr) s0 = fmaf(bf(bt[q * nr + rho]), C.lvs[q], s0);
          red_add_f32(acc + u.r0 + rho, Ld.lscale * (s0 + s1));
        }
      }
      cs.release(1);
      break;
    }
    case U_LORA_A: {
      // v = A x for ranks [r0, r1), published for the CTAs that own the B rows
      // (each rank's value goes out as a launch-tagged word: no counter, no fence)
      const uint32_t par = C.epoch & 1u;
      const int n = u.r1 - u.r0;
      if (u.flags & UF_LOCAL_V) {
        // every rank, for this CTA's own B rows only (no other CTA holds B rows): v stays
        // in shared memory
        consume_bf_rows<D>(cs, n, BF_SMEM, C.lvs, nullptr);
        if (tid == 0) C.lv_layer = l;
      } else {
        consume_bf_rows<D>(cs, n, BF_TAGGED, reinterpret_cast<float*>(lv_ptr(P, par, l) + u.r0), nullptr);
      }
      break;
    }
    case U_HEAD: {
      cbar();  // ubuf reuse
      float* ub = C.ubuf;
      consume_bf_rows<D>(cs, u.r1 - u.r0, BF_SMEM, ub, nullptr);
      cs.wait_route(l);
      cbar();
      const int nr = u.r1 - u.r0;
      if (cs.acquire(1) && tid < nr) {
        const uint16_t* g = reinterpret_cast<const uint16_t*>(cs.stage(0));
        float v = ub[tid];
        if (Ld.b1) v += bf(g[tid]);
        const uint32_t cv = C.rt_valid[l], pv = C.rt_pvalid[l];
        for (int k = 0; k < P.K; ++k) {
          if ((cv >> k) & 1u) v += bf(g[(1 + k) * nr + tid]);
          if ((pv >> k) & 1u) v += bf(g[(1 + P.K + k) * nr + tid]);
        }
        ub[tid] = gelu_f(v);
      }
      cs.release(1);
      cbar();
      const int E = P.E;
      const int per = max(1, STAGE_BYTES / (2 * E));
      for (int i0 = 0; i0 < nr; i0 += per) {
        const int ni = min(per, nr - i0);
        if (cs.acquire(1)) bf_axpy_rows(cs.stage(0), ni, E, ub + i0, 1.0f, zhat, tid);
        cs.release(1);
      }
      break;
    }
    case U_LRES: {
      const uint16_t* b2 = Ld.b2;
      const int e0 = u.r0;
      float* bb = C.b2buf;
      cbar();  // b2buf reuse
      if (b2)  // stage the bias slice in shared memory (read-only input)
        for (int e = tid; e < u.r1 - u.r0; e += NCT) bb[e] = bf(b2[e0 + e]);
      cbar();
      consume_bf_rows<D>(cs, u.r1 - u.r0, BF_ADD_BIAS, zhat + e0, b2 ? bb : nullptr);
      break;
    }
    case U_ROUTER: {
      const int e0 = u.r0;
      consume_bf_rows<D>(cs, u.r1 - u.r0, BF_TAGGED, reinterpret_cast<float*>(reinterpret_cast<uint64_t*>(zr) + e0),
                         nullptr);
      break;
    }
    default:
      break;
  }
}

// Build the layer input: residual h (fp32 of bf16 values), the RMSNorm factor, and
// the int16 copy of x = h * factor used by the int4 rows, with one quantisation step
// per 32-element chunk (max |x| of the chunk / 32767), so the only block-wide
// reduction is the one that the norm needs anyway (the sum of squares).  Thread t
// owns elements t + NCT*k: warp w owns the whole 32-element chunks w + NCW*k, whose
// maxima and sums come from warp reductions.  inc[] holds this thread's residual
// increments, loaded before the dependency wait.
template <int D>
__device__ __forceinline__ void layer_input(Cons& cs, int l, uint32_t par, const float* inc) {
  const EngineParams& P = cs.P;
  Ctl& C = cs.C;
  const int tid = cs.tid;
  constexpr int PER = (D + NCT - 1) / NCT;
  float h[PER];
  float ss = 0.f;
  const float* accp = (P.mode == MODE_STACK && l > 0) ? acc_ptr(P, par, l - 1) : nullptr;
  float a[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + NCT * k;
    a[k] = (accp && i < D) ? __ldcg(accp + i) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + NCT * k;
    h[k] = 0.f;
    if (i < D) {
      float v;
      if (P.mode == MODE_STACK) {
        const uint16_t hb = l == 0 ? P.h_in[i] : f32_to_bf16_bits(C.res[i] + a[k]);
        v = P.incr ? bf(f32_to_bf16_bits(bf(hb) + inc[k])) : bf(hb);
      } else {
        v = bf(P.h_in[i]);
      }
      h[k] = v;
      C.res[i] = v;
      ss += v * v;
    }
  }
  ss = warp_sum(ss);
  if (cs.lane == 0) C.red[cs.cw] = ss;
  // the largest |h| of each 32-element chunk (a warp owns whole chunks)
  uint32_t cm[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k)
    cm[k] = (tid - cs.lane) + NCT * k < D ? __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h[k]))) : 0u;
  cbar();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) tot += C.red[w];
  const float scale = P.norm ? rsqrtf(tot * (1.0f / (float)D) + RMS_EPS) : 1.0f;
  int16_t* xq16 = reinterpret_cast<int16_t*>(C.xq);
  // one quantisation step per 32-element chunk, max|x of the chunk| / 32767, so that an
  // outlier costs resolution only within its own chunk.  (The step needs no correctly
  // rounded division: the codes are clamped and scaled back by the same inv.)
  // Independent chunks: codes first, then their stores and sums, so the steps overlap.
  int q[PER], sq[PER];
  float inv[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const float xmax = __uint_as_float(cm[k]) * scale;
    const float r = xmax > 0.f ? __fdividef(32767.0f, xmax) : 0.f;
    inv[k] = xmax * (1.0f / 32767.0f);
    const int v = __float2int_rn(h[k] * scale * r);
    q[k] = v > 32767 ? 32767 : (v < -32767 ? -32767 : v);
  }
  const int j = cs.lane, idx = j & 7;
  const int pos = (j >> 3) * (DMAX / 32) * 8 + ((idx & 1) ? 4 + (idx >> 1) : (idx >> 1));
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + NCT * k;
    sq[k] = 0;
    if (i < D) {  // warp-uniform: chunks are warp-aligned
      xq16[(i >> 5) * 8 + pos] = (int16_t)q[k];
      sq[k] = __reduce_add_sync(0xffffffffu, q[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + NCT * k;
    if (i < D) {
      if (cs.lane == 0) {
        C.xinv[i >> 5] = inv[k];
        C.xsum[i >> 5] = (float)sq[k] * inv[k];
      }
      if (P.mode == MODE_STACK && P.h_trace && blockIdx.x == 0)
        P.h_trace[(size_t)l * D + i] = f32_to_bf16_bits(h[k]);
      if (P.mode == MODE_STACK && P.delta_trace && blockIdx.x == 0 && l > 0)
        P.delta_trace[(size_t)(l - 1) * D + i] = a[k];
    }
  }
  if (tid == 0) C.xscale = scale;
  cbar();
}

template <int D>
__device__ void consumer(const EngineParams& P, Ctl& C, uint8_t* ring) {
  Cons cs{P, C, ring, 0u, (int)(threadIdx.x >> 5), (int)(threadIdx.x & 31), (int)threadIdx.x};
  const int tid = cs.tid;
  const uint32_t par = C.epoch & 1u;
  const uint32_t pnext3 = (C.epoch + 1) % 3u, pclr3 = (C.epoch + 2) % 3u;
  const int ncta = P.ncta, cta = blockIdx.x;

  if (tid == 0) {
    const uint64_t stall = *reinterpret_cast<volatile uint64_t*>(&hdr(P)->stall_ns);
    if (stall) {
      volatile uint32_t* never = &hdr(P)->never;
      spin_until(P, C, [&] { return *never != 0u; }, stall);
    }
  }
  cbar();

  for (int l = 0; l < P.L; ++l) {
    const LayerDesc& Ld = layer_at(P, l);
    if (tid == 0) stamp(P, l, 0);
    // residual increments of this layer are inputs: load them before the dependency wait
    float inc[(D + NCT - 1) / NCT];
#pragma unroll
    for (int k = 0; k < (D + NCT - 1) / NCT; ++k) {
      const int i = tid + NCT * k;
      inc[k] = (P.mode == MODE_STACK && P.incr && i < D) ? bf(P.incr[(size_t)l * D + i]) : 0.f;
    }
    if (l > 0 && P.mode == MODE_STACK) {
      if (tid == 0)
        wait_count(P, C, ctr(P, par, l - 1, 0),
                   (uint32_t)(P.plan ? P.n_arrive[layer_at(P, l - 1).plan_kind] : ncta));
      cbar();
    }
    if (tid == 0) stamp(P, l, 1);
    layer_input<D>(cs, l, par, inc);
    if (tid == 0) stamp(P, l, 2);
    float* acc = acc_ptr(P, par, l);
    float* zh = zhat_ptr(P, pnext3, l);
    float* zr = reinterpret_cast<float*>(zr_ptr(P, par, l));  // tagged u64 words
    if (gate_here(P, l)) {
      // gate rows first: the routing warps pick this layer's experts from them
      int nu;
      const Unit* us = units_of(P, KIND_ROUTER, cta, nu);
      for (int i = 0; i < nu; ++i) consume_unit<D>(cs, Ld, us[i], l, acc, zh, zr);
      if (tid == 0) stamp(P, l, 8 + U_ROUTER);  // gate rows of this CTA published
    }
    if (P.mode == MODE_STACK && Ld.gate_for >= 0) {
      // route-ahead: the gate rows of layer gate_for on this layer's input
      float* zra = reinterpret_cast<float*>(zr_ptr(P, par, Ld.gate_for));
      int nu;
      const Unit* us = units_of(P, KIND_ROUTER, cta, nu);
      for (int i = 0; i < nu; ++i) consume_unit<D>(cs, Ld, us[i], l, acc, zh, zra);
    }
    int nu;
    const Unit* us = units_of(P, P.plan ? Ld.plan_kind : 0, cta, nu);
    if (P.trace && tid == 0)
      for (int t = 0; t < 8; ++t) C.ttype[t] = 0;
    for (int i = 0; i < nu; ++i) {
      const uint64_t tu = (P.trace && tid == 0) ? globaltimer() : 0;
      consume_unit<D>(cs, Ld, us[i], l, acc, zh, zr);
      if (P.trace && tid == 0) C.ttype[us[i].type & 7] += globaltimer() - tu;
    }
    if (tid == 0) {
      stamp(P, l, 3);
      if (P.trace) {
        // plain stores only (a read-modify-write here would stall the CTA's arrival)
        uint64_t* tr = P.trace + ((size_t)cta * P.L + l) * 16;
        tr[6] = cs.t_acq;
        tr[7] = cs.n_acq;
        for (int t = 1; t < 8; ++t)
          if (t != U_ROUTER) tr[8 + t] = C.ttype[t];
      }
      cs.t_acq = 0;
      cs.n_acq = 0;
    }

    if (l == P.L - 1) {
      // Clear the other half of the parity-duplicated buffers for the next launch.
      const size_t n_ctr = (size_t)P.L * 4, n_acc = (size_t)P.L * P.out_dim, n_z = (size_t)P.L * P.E;
      const size_t total = n_ctr + n_acc + n_z;
      const size_t per = (total + ncta - 1) / ncta;
      const size_t b0 = (size_t)cta * per, b1 = min(total, b0 + per);
      uint32_t* c1 = ctr(P, par ^ 1u, 0, 0);
      for (size_t i = b0 + tid; i < b1; i += NCT) {
        if (i < n_ctr) {
          c1[i] = 0u;
        } else if (i < n_ctr + n_acc) {
          const size_t j = i - n_ctr;
          acc_ptr(P, par ^ 1u, (int)(j / P.out_dim))[j % P.out_dim] = 0.f;
        } else {
          const size_t j = i - n_ctr - n_acc;
          zhat_ptr(P, pclr3, (int)(j / P.E))[j % P.E] = 0.f;
        }
      }
    }
    cbar();
    if (tid == 0) {
      // the bar.sync above orders every consumer thread's reductions before this release
      const int kind = P.plan ? Ld.plan_kind : 0;
      if (P.plan && C.defer[kind]) {
        // prerouter work only: the next layer does not wait for it, the commit does
        red_release_add_u32(ctr(P, par, l, 1), 1u);
        if (l == P.L - 1) C.is_last = 0;
      } else if (l == P.L - 1) {
        const uint32_t old = atom_acq_rel_add_u32(ctr(P, par, l, 0), 1u);
        C.is_last = (old == (uint32_t)(P.plan ? P.n_arrive[kind] : ncta) - 1u);
      } else {
        red_release_add_u32(ctr(P, par, l, 0), 1u);
      }
    }
  }
  cbar();
  if (!C.is_last) return;

  // ---------------- finisher: the last CTA to arrive writes the outputs
  __threadfence();
  const int L1 = P.L - 1;
  const float* acc = acc_ptr(P, par, L1);
  const bool ok = !C.abort_flag;  // all consumer waits are over: stable from here on
  if (ok && (P.mode == MODE_LAYER || P.mode == MODE_STACK)) {
    for (int i = tid; i < P.d; i += NCT) {
      const float a = ld_cg_f32(acc + i);
      P.h_out[i] = f32_to_bf16_bits(C.res[i] + a);
      if (P.delta_out) P.delta_out[i] = a;
    }
  } else if (ok && P.mode == MODE_QLINEAR) {
    for (int i = tid; i < P.out_dim; i += NCT) {
      float a = ld_cg_f32(acc + i);
      if (P.accumulate) a += bf(P.h_out[i]);
      if (P.delta_out) P.delta_out[i] = a;
      P.h_out[i] = f32_to_bf16_bits(a);
    }
  }
  const LayerDesc& L0 = layer_at(P, 0);
  const bool want_next = ok && (P.mode == MODE_HEAD || (P.mode == MODE_LAYER && L0.has_head));
  if (want_next) {
    const float* zh = zhat_ptr(P, pnext3, 0);
    for (int e = tid; e < P.E; e += NCT) {
      const float z = ld_cg_f32(zh + e) + (P.logit_bias ? P.logit_bias[e] : 0.f);
      C.zbuf[e] = z;
      if (P.next_logits) P.next_logits[e] = z;
    }
  }
  cbar();
  if (want_next && cs.cw == 0) {
    int id;
    float w;
    route_smem(P, C.zbuf, P.score_bias, cs.lane, id, w);
    if (cs.lane < P.K) {
      if (P.next_ids) P.next_ids[cs.lane] = id;
      if (P.next_w) P.next_w[cs.lane] = w;
    }
  }
  cbar();
  if (tid == 0) {
    __threadfence();
    if (C.abort_flag) atomicOr(&hdr(P)->status, (uint32_t)E0_DEV_ABORTED);
    hdr(P)->epoch = C.epoch + 1u;
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) engine_kernel(const __grid_constant__ EngineParams P) {
  uint8_t* ring = e0_smem;
  Ctl& C = *reinterpret_cast<Ctl*>(e0_smem + CTL_OFFSET);
  {
    // layer descriptors and this CTA's work units, copied on chip once
    const int nl = P.layers ? P.L : 1;
    const uint64_t* src = reinterpret_cast<const uint64_t*>(P.layers ? P.layers : &P.inline_layer);
    uint64_t* dst = reinterpret_cast<uint64_t*>(e0_smem + LD_OFFSET);
    const int nw = nl * (int)(sizeof(LayerDesc) / 8);
    for (int i = threadIdx.x; i < nw; i += NTHREADS) dst[i] = src[i];
    for (int i = threadIdx.x; i < KINDS_MAX * MAXU; i += NTHREADS) {
      const int kind = i / MAXU, u = i % MAXU;
      if (P.plan) {
        if (kind < P.kinds) {
          C.su[kind][u] = P.plan[((size_t)kind * P.ncta + blockIdx.x) * MAXU + u];
          if (u == 0) {
            C.sn[kind] = P.plan_n[kind * P.ncta + blockIdx.x];
            C.defer[kind] = P.defer ? P.defer[kind * P.ncta + blockIdx.x] : 0;
          }
        }
      } else if (kind == 0) {
        C.su[0][u] = P.inline_plan[(size_t)blockIdx.x * MAXU + u];
        if (u == 0) C.sn[0] = P.inline_n[blockIdx.x];
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGES; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], NCW);
    }
    for (int l = 0; l < LMAX; ++l) mbar_init(&C.rt_bar[l], 1);
    fence_mbar_init();
    for (int l = 0; l < LMAX; ++l) C.rt_ready[l] = 0;
    C.abort_flag = 0;
    C.is_last = 0;
    C.lv_layer = -1;
    C.epoch = *reinterpret_cast<volatile uint32_t*>(&hdr(P)->epoch);
  }
  __syncthreads();
  if (threadIdx.x >= NCT + 32)
    router_warp(P, C);
  else if (threadIdx.x >= NCT)
    producer(P, C, ring);
  else
    consumer<D>(P, C, ring);
}

// ------------------------------------------------------------------ host launch
template <int D>
static cudaError_t launch_d(const EngineParams& P, cudaStream_t stream) {
  static bool attr_done = false;
  const size_t smem = smem_bytes();
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(engine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.ncta);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, engine_kernel<D>, P);
}

cudaError_t launch_engine(const EngineParams& P, cudaStream_t stream) {
  switch (P.d) {
    case 256: return launch_d<256>(P, stream);
    case 512: return launch_d<512>(P, stream);
    case 1024: return launch_d<1024>(P, stream);
    case 2048: return launch_d<2048>(P, stream);
    default: return cudaErrorInvalidValue;
  }
}

int max_ctas_per_sm(int d) {
  int n = 0;
  const size_t smem = smem_bytes();
  switch (d) {
    case 256: cudaFuncSetAttribute(engine_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_kernel<256>, NTHREADS, smem); break;
    case 512: cudaFuncSetAttribute(engine_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_kernel<512>, NTHREADS, smem); break;
    case 1024: cudaFuncSetAttribute(engine_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_kernel<1024>, NTHREADS, smem); break;
    case 2048: cudaFuncSetAttribute(engine_kernel<2048>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_kernel<2048>, NTHREADS, smem); break;
    default: break;
  }
  return n;
}

}  // namespace e0eng
