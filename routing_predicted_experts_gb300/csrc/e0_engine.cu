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
  float x[DMAX];              // layer input x (normed), fp32
  float res[DMAX];            // residual h of the layer, fp32 (exact bf16 values)
  uint4 xq[DMAX / 8];         // x as int16, 8-element groups stored [0,2,4,6,1,3,5,7]
  float xinv[DMAX / 32];      // per 32-element chunk: dequant step of xq
  float xsum[DMAX / 32];      // per 32-element chunk: sum of x
  float abuf[32];             // SwiGLU activations of the current expert slab
  float ubuf[HEAD_ROWS];      // head fc1 pre-activation, then erf-GELU output
  float vbuf[RANKS_MAX];      // LoRA A x for the current rank slice
  float zbuf[EMAX];           // logits staged for top-K
  int32_t r_ids[4][KMAX];     // committed expert ids per layer (ring of 4 layers)
  int32_t r_idx[4][KMAX];     // stored index (slot) of each id
  float r_w[4][KMAX];         // renormalised combine weights
  int32_t r_prev[4][KMAX];    // ids this layer used at the previous token
  uint32_t r_valid[4];
  uint32_t r_prev_valid[4];
  float red[NCW];
  int32_t f_ids[KMAX];        // finisher top-K
  float f_vals[KMAX];
  volatile int32_t route_seq;
  volatile int32_t cons_done;
  volatile int32_t abort_flag;
  int32_t is_last;
  uint32_t epoch;
};

size_t smem_bytes() { return (size_t)NSTAGES * STAGE_BYTES + sizeof(Ctl); }

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ const LayerDesc& layer_at(const EngineParams& P, int l) {
  return P.layers ? P.layers[l] : P.inline_layer;
}

__device__ __forceinline__ const Unit* units_of(const EngineParams& P, int kind, int cta, int& n) {
  if (P.plan) {
    n = P.plan_n[kind * P.ncta + cta];
    return P.plan + ((size_t)kind * P.ncta + cta) * MAXU;
  }
  n = P.inline_n[cta];
  return P.inline_plan + (size_t)cta * MAXU;
}

__device__ __forceinline__ WsHeader* hdr(const EngineParams& P) { return reinterpret_cast<WsHeader*>(P.ws); }
__device__ __forceinline__ uint32_t* ctr(const EngineParams& P, uint32_t par, int l, int which) {
  return reinterpret_cast<uint32_t*>(P.ws + P.wl.counters) + ((size_t)par * P.L + l) * 2 + which;
}
__device__ __forceinline__ float* acc_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.acc) + ((size_t)par * P.L + l) * OUTMAX;
}
__device__ __forceinline__ float* zhat_ptr(const EngineParams& P, uint32_t p3, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.zhat) + ((size_t)p3 * P.L + l) * P.E;
}
__device__ __forceinline__ float* zr_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.zr) + ((size_t)par * P.L + l) * P.E;
}
__device__ __forceinline__ int32_t* idsu_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<int32_t*>(P.ws + P.wl.ids) + ((size_t)par * P.L + l) * KMAX;
}
__device__ __forceinline__ float* wu_ptr(const EngineParams& P, uint32_t par, int l) {
  return reinterpret_cast<float*>(P.ws + P.wl.wts) + ((size_t)par * P.L + l) * KMAX;
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

__device__ __forceinline__ void cbar() { named_bar_sync(1, NCT); }

// Diagnostics: stamp %globaltimer into trace[cta][l][slot] when a trace buffer is set.
// Slots: 0 consumer layer start, 1 dependency satisfied, 2 layer input built,
// 3 units done, 4 producer route published, 5 producer issued the layer's last stage.
__device__ __forceinline__ void stamp(const EngineParams& P, int l, int slot) {
  if (P.trace) P.trace[((size_t)blockIdx.x * P.L + l) * 8 + slot] = globaltimer();
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

// Quantise 32 fp32 values (one chunk) to int16 with step m/32767 (m = max |v|) and
// pack them in the dot32 order.  Returns the step; *sum receives the fp32 sum.
__device__ __forceinline__ float quant_chunk32(const float* v, uint32_t* xp, float* sum) {
  float m = 0.f, s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    m = fmaxf(m, fabsf(v[i]));
    s += v[i];
  }
  *sum = s;
  const float r = m > 0.f ? 32767.0f / m : 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    int q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int t = __float2int_rn(v[8 * g + j] * r);
      q[j] = t > 32767 ? 32767 : (t < -32767 ? -32767 : t);
    }
    xp[4 * g + 0] = (uint32_t)(q[0] & 0xFFFF) | ((uint32_t)q[2] << 16);
    xp[4 * g + 1] = (uint32_t)(q[4] & 0xFFFF) | ((uint32_t)q[6] << 16);
    xp[4 * g + 2] = (uint32_t)(q[1] & 0xFFFF) | ((uint32_t)q[3] << 16);
    xp[4 * g + 3] = (uint32_t)(q[5] & 0xFFFF) | ((uint32_t)q[7] << 16);
  }
  return m > 0.f ? m / 32767.0f : 0.f;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_f(float u) { return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f)); }

// ------------------------------------------------------------------ top-K (one warp)
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  if (v != v) u = 0u;
  return ((uint64_t)u << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

// Top-K of z[0..E) (shared memory), descending, ties to the lower index.  Writes
// ids/vals (lane 0).  All 32 lanes must call.
__device__ void warp_topk(const float* z, int E, int K, int lane, int32_t* ids, float* vals) {
  uint32_t taken = 0;
  uint64_t best = 0;
  for (int e = lane, m = 0; e < E; e += 32, ++m) best = max(best, topk_key(z[e], e));
  for (int k = 0; k < K; ++k) {
    uint64_t m = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = (int)(0xFFFFFFFFu - (uint32_t)m);
    if (lane == 0) {
      ids[k] = e;
      vals[k] = z[e];
    }
    if ((e & 31) == lane) {
      taken |= 1u << (e >> 5);
      best = 0;
      for (int e2 = lane, mm = 0; e2 < E; e2 += 32, ++mm)
        if (!((taken >> mm) & 1u)) best = max(best, topk_key(z[e2], e2));
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ producer
struct Prod {
  const EngineParams& P;
  Ctl& C;
  uint8_t* ring;
  uint32_t n;      // stages issued
  bool ok;
  int lane;

  // lane 0: wait until stage n's slot is free, return its base (nullptr on failure)
  __device__ uint8_t* begin(uint32_t& slot) {
    slot = n % NSTAGES;
    const uint32_t round = n / NSTAGES;
    if (round > 0) {
      uint64_t* bar = &C.empty[slot];
      const uint32_t par = (round - 1) & 1u;
      if (!spin_until(P, C, [&] { return mbar_try_wait(bar, par); }, P.timeout_ns)) return nullptr;
    }
    return ring + (size_t)slot * STAGE_BYTES;
  }
  __device__ void commit() { ++n; }
};

// Issue one stage worth of int4 rows [row0, row0+nr) of a row-layout matrix (in = D).
__device__ __forceinline__ bool issue_q4_rows(Prod& pr, const uint32_t* q, const uint16_t* s, const uint16_t* b,
                                              int in, int row0, int nr) {
  if (pr.lane == 0 && pr.ok) {
    uint32_t slot;
    uint8_t* st = pr.begin(slot);
    if (!st) {
      pr.ok = false;
    } else {
      const uint32_t qb = (uint32_t)nr * in / 2, sb = (uint32_t)nr * in / 32;
      mbar_arrive_expect_tx(&pr.C.full[slot], qb + 2 * sb);
      tma_bulk_g2s(st, q + (size_t)row0 * (in / 8), qb, &pr.C.full[slot]);
      tma_bulk_g2s(st + qb, s + (size_t)row0 * (in / 64), sb, &pr.C.full[slot]);
      tma_bulk_g2s(st + qb + sb, b + (size_t)row0 * (in / 64), sb, &pr.C.full[slot]);
      pr.commit();
    }
  }
  return true;
}

__device__ __forceinline__ void issue_bytes(Prod& pr, const void* src, uint32_t bytes) {
  if (pr.lane == 0 && pr.ok) {
    uint32_t slot;
    uint8_t* st = pr.begin(slot);
    if (!st) {
      pr.ok = false;
    } else {
      mbar_arrive_expect_tx(&pr.C.full[slot], bytes);
      tma_bulk_g2s(st, src, bytes, &pr.C.full[slot]);
      pr.commit();
    }
  }
}

// Issue bf16 rows [row0, row1) of a [rows][in] matrix, in stage-sized chunks.
__device__ void issue_bf_rows(Prod& pr, const uint16_t* m, int in, int row0, int row1) {
  const int per = bf_rows_per_stage(in);
  for (int r = row0; r < row1; r += per) {
    const int nr = min(per, row1 - r);
    issue_bytes(pr, m + (size_t)r * in, (uint32_t)nr * in * 2);
  }
}

__device__ void issue_unit(Prod& pr, const LayerDesc& Ld, const Unit& u, int l) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const int d = P.d;
  const int slot4 = l & 3;
  switch (u.type) {
    case U_EXPERT: {
      const bool shared = u.k >= P.K;
      if (shared ? !Ld.has_shared : !((C.r_valid[slot4] >> u.k) & 1u)) return;
      const int idx = shared ? 0 : C.r_idx[slot4][u.k];
      const uint32_t* guq = (shared ? Ld.sgu_q : Ld.gu_q) + (size_t)idx * (2 * P.F) * (d / 8);
      const uint16_t* gus = (shared ? Ld.sgu_s : Ld.gu_s) + (size_t)idx * (2 * P.F) * (d / 64);
      const uint16_t* gub = (shared ? Ld.sgu_b : Ld.gu_b) + (size_t)idx * (2 * P.F) * (d / 64);
      const int per = q4_rows_per_stage(d);
      for (int r = 64 * u.r0; r < 64 * u.r0 + 64; r += per) issue_q4_rows(pr, guq, gus, gub, d, r, min(per, 64 * u.r0 + 64 - r));
      const uint32_t* dq = (shared ? Ld.sdn_q : Ld.dn_q) + (size_t)idx * (P.F / 32) * d * 4 + (size_t)u.r0 * d * 4;
      const uint16_t* ds = (shared ? Ld.sdn_s : Ld.dn_s) + (size_t)idx * (P.F / 64) * d + (size_t)(u.r0 >> 1) * d;
      const uint16_t* db = (shared ? Ld.sdn_b : Ld.dn_b) + (size_t)idx * (P.F / 64) * d + (size_t)(u.r0 >> 1) * d;
      const int pd = dn_rows_per_stage(d);
      for (int i0 = 0; i0 < d; i0 += pd) {
        const int nr = min(pd, d - i0);
        if (pr.lane == 0 && pr.ok) {
          uint32_t slot;
          uint8_t* st = pr.begin(slot);
          if (!st) {
            pr.ok = false;
          } else {
            mbar_arrive_expect_tx(&C.full[slot], (uint32_t)nr * 20);
            tma_bulk_g2s(st, dq + (size_t)i0 * 4, nr * 16, &C.full[slot]);
            tma_bulk_g2s(st + nr * 16, ds + i0, nr * 2, &C.full[slot]);
            tma_bulk_g2s(st + nr * 18, db + i0, nr * 2, &C.full[slot]);
            pr.commit();
          }
        }
      }
      break;
    }
    case U_QROWS: {
      const int per = q4_rows_per_stage(d);
      for (int r = u.r0; r < u.r1; r += per) issue_q4_rows(pr, Ld.lw_q, Ld.lw_s, Ld.lw_b, d, r, min(per, u.r1 - r));
      break;
    }
    case U_LORA_AB: {
      issue_bf_rows(pr, Ld.la, d, u.r0, u.r1);
      const int per = max(1, STAGE_BYTES / (2 * Ld.lout));
      for (int q = u.r0; q < u.r1; q += per)
        issue_bytes(pr, Ld.lbt + (size_t)q * Ld.lout, (uint32_t)min(per, u.r1 - q) * Ld.lout * 2);
      break;
    }
    case U_HEAD: {
      issue_bf_rows(pr, Ld.w1h, d, u.r0, u.r1);
      const int nr = u.r1 - u.r0;
      const uint32_t slotb = (uint32_t)nr * 2;
      if (pr.lane == 0 && pr.ok) {
        uint32_t slot;
        uint8_t* st = pr.begin(slot);
        if (!st) {
          pr.ok = false;
        } else {
          uint32_t bytes = 0;
          if (Ld.b1) bytes += slotb;
          for (int k = 0; k < P.K; ++k) {
            if ((C.r_valid[slot4] >> k) & 1u) bytes += slotb;
            if ((C.r_prev_valid[slot4] >> k) & 1u) bytes += slotb;
          }
          mbar_arrive_expect_tx(&C.full[slot], bytes);
          if (Ld.b1) tma_bulk_g2s(st, Ld.b1 + u.r0, slotb, &C.full[slot]);
          for (int k = 0; k < P.K; ++k) {
            if ((C.r_valid[slot4] >> k) & 1u)
              tma_bulk_g2s(st + (1 + k) * slotb, Ld.w1c_t + (size_t)C.r_ids[slot4][k] * Ld.H + u.r0, slotb,
                           &C.full[slot]);
            if ((C.r_prev_valid[slot4] >> k) & 1u)
              tma_bulk_g2s(st + (1 + P.K + k) * slotb, Ld.w1p_t + (size_t)C.r_prev[slot4][k] * Ld.H + u.r0, slotb,
                           &C.full[slot]);
          }
          pr.commit();
        }
      }
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

// Resolve the routing of layer l and publish it in route slot l & 3.
__device__ void resolve_route(Prod& pr, const LayerDesc& Ld, int l, bool self_route, uint32_t par, uint32_t p3) {
  const EngineParams& P = pr.P;
  Ctl& C = pr.C;
  const int lane = pr.lane;
  const int slot = l & 3;
  const int K = P.K, E = P.E;
  bool ok = pr.ok;
  if (ok && lane == 0) ok = spin_until(P, C, [&] { return C.cons_done >= l - 3; }, P.timeout_ns);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  pr.ok = ok;
  if (ok && P.mode != MODE_QLINEAR) {
    const int32_t* given = nullptr;
    const float* z = nullptr;
    const int32_t* prev = nullptr;
    bool z_remote = false;
    if (P.mode == MODE_LAYER) {
      given = P.ids_in; z = P.logits_in; prev = P.ids_prev_in;
    } else if (P.mode == MODE_HEAD) {
      given = P.ids_in; prev = P.ids_prev_in;
    } else {  // stack
      if (self_route) {
        bool w = true;
        if (lane == 0)
          w = spin_until(P, C, [&] { return ld_acquire_u32(ctr(P, par, l, 1)) >= (uint32_t)P.ncta; }, P.timeout_ns);
        w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
        pr.ok = w;
        z = zr_ptr(P, par, l);
      } else {
        z = zhat_ptr(P, p3, l - 1);
      }
      z_remote = true;
      if (P.step > 0) prev = idsu_ptr(P, par ^ 1u, l);
    }
    if (pr.ok) {
      if (z) {
        for (int e = lane; e < E; e += 32) C.zbuf[e] = z_remote ? ld_cg_f32(z + e) : z[e];
        __syncwarp();
      }
      uint32_t valid = 0;
      if (given) {
        int id = -1;
        if (lane < K) {
          id = given[lane];
          C.r_ids[slot][lane] = id;
        }
        __syncwarp();
        bool v = lane < K && id >= 0 && id < E;
        if (lane < K)
          for (int j = 0; j < lane; ++j)
            if (C.r_ids[slot][j] == id) v = false;
        if (lane < K && !v) raise_error(P, C, E0_DEV_BAD_ID);
        valid = __ballot_sync(0xffffffffu, v);
      } else if (z) {
        warp_topk(C.zbuf, E, K, lane, C.r_ids[slot], C.r_w[slot]);  // r_w holds the logits for now
        valid = (K >= 32) ? 0xffffffffu : ((1u << K) - 1u);
      } else {
        valid = 0u;  // no current routing (head without one-hot input)
      }
      __syncwarp();
      // stored index through the slot table
      bool vk = lane < K && ((valid >> lane) & 1u);
      if (lane < K) {
        int idx = C.r_ids[slot][lane];
        if (vk && Ld.slot_of) {
          idx = Ld.slot_of[idx];
          if (idx < 0) { vk = false; raise_error(P, C, E0_DEV_NOT_RESIDENT); }
        }
        if (vk && Ld.gu_q && idx >= Ld.n_routed) { vk = false; raise_error(P, C, E0_DEV_BAD_ID); }
        C.r_idx[slot][lane] = vk ? idx : 0;
      }
      valid = __ballot_sync(0xffffffffu, vk);
      // combine weights: softmax over the selected logits
      if (z && lane == 0) {
        float mx = -INFINITY;
        for (int k = 0; k < K; ++k)
          if ((valid >> k) & 1u) mx = fmaxf(mx, C.zbuf[C.r_ids[slot][k]]);
        float s = 0.f;
        for (int k = 0; k < K; ++k)
          if ((valid >> k) & 1u) s += expf(C.zbuf[C.r_ids[slot][k]] - mx);
        for (int k = 0; k < K; ++k)
          C.r_w[slot][k] = ((valid >> k) & 1u) ? expf(C.zbuf[C.r_ids[slot][k]] - mx) / s : 0.f;
      } else if (!z && lane < K) {
        C.r_w[slot][lane] = 0.f;
      }
      // previous-token ids (one-hot of the previous step)
      uint32_t pvalid = 0;
      if (prev) {
        int pid = -1;
        if (lane < K) {
          pid = P.mode == MODE_STACK ? ld_cg_s32(prev + lane) : prev[lane];
          C.r_prev[slot][lane] = pid;
        }
        __syncwarp();
        bool v = lane < K && pid >= 0 && pid < E;
        if (lane < K)
          for (int j = 0; j < lane; ++j)
            if (C.r_prev[slot][j] == pid) v = false;
        if (lane < K && pid != -1 && !v && P.mode != MODE_STACK) raise_error(P, C, E0_DEV_BAD_ID);
        pvalid = __ballot_sync(0xffffffffu, v);
      }
      if (lane == 0) {
        C.r_valid[slot] = valid;
        C.r_prev_valid[slot] = pvalid;
      }
      __syncwarp();
      if (P.mode == MODE_STACK && blockIdx.x == 0 && lane < K) {
        const int id = ((valid >> lane) & 1u) ? C.r_ids[slot][lane] : -1;
        idsu_ptr(P, par, l)[lane] = id;
        wu_ptr(P, par, l)[lane] = C.r_w[slot][lane];
        if (P.ids_trace) P.ids_trace[l * K + lane] = id;
        if (P.w_trace) P.w_trace[l * K + lane] = C.r_w[slot][lane];
      }
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    C.route_seq = l + 1;
  }
  __syncwarp();
}

__device__ void producer(const EngineParams& P, Ctl& C, uint8_t* ring) {
  Prod pr{P, C, ring, 0u, true, (int)(threadIdx.x & 31)};
  const uint32_t par = C.epoch & 1u, p3 = C.epoch % 3u;
  for (int l = 0; l < P.L; ++l) {
    const LayerDesc& Ld = layer_at(P, l);
    const bool self_route = P.mode == MODE_STACK && ((P.router_mask >> l) & 1ull);
    if (self_route) {
      int nu;
      const Unit* us = units_of(P, KIND_ROUTER, blockIdx.x, nu);
      for (int i = 0; i < nu; ++i) issue_bf_rows(pr, Ld.router, P.d, us[i].r0, us[i].r1);
    }
    pr.ok = __shfl_sync(0xffffffffu, pr.ok ? 1 : 0, 0) != 0;
    resolve_route(pr, Ld, l, self_route, par, p3);
    if (pr.lane == 0) stamp(P, l, 4);
    int nu;
    const Unit* us = units_of(P, P.plan ? Ld.plan_kind : 0, blockIdx.x, nu);
    for (int i = 0; i < nu; ++i) issue_unit(pr, Ld, us[i], l);
    if (pr.lane == 0) stamp(P, l, 5);
    pr.ok = __shfl_sync(0xffffffffu, pr.ok ? 1 : 0, 0) != 0;
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

// ------------------------------------------------------------------ consumers
struct Cons {
  const EngineParams& P;
  Ctl& C;
  uint8_t* ring;
  uint32_t n;  // stages consumed
  int cw, lane, tid;

  // wait for the next stage; returns its base or nullptr (abort)
  __device__ const uint8_t* acquire(uint32_t& slot) {
    slot = n % NSTAGES;
    const uint32_t par = (n / NSTAGES) & 1u;
    uint64_t* bar = &C.full[slot];
    bool ok = spin_until(P, C, [&] { return mbar_try_wait(bar, par); }, P.timeout_ns);
    return ok ? ring + (size_t)slot * STAGE_BYTES : nullptr;
  }
  __device__ void release(uint32_t slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.empty[slot]);
    ++n;
  }
};

template <int D>
struct Q4Frag {
  static constexpr int LPR = (D / 32) < 32 ? (D / 32) : 32;
  static constexpr int CPL = (D / 32) / LPR;
  uint32_t xp[CPL][16];
  float inv[CPL], sum[CPL];
  __device__ __forceinline__ void load(const Ctl& C, int lane) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane % LPR + LPR * j;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint4 v = C.xq[4 * c + t];
        xp[j][4 * t] = v.x; xp[j][4 * t + 1] = v.y; xp[j][4 * t + 2] = v.z; xp[j][4 * t + 3] = v.w;
      }
      inv[j] = C.xinv[c];
      sum[j] = C.xsum[c];
    }
  }
};

// int4 rows of one stage: GU = gate/up pairs -> abuf; else rows -> red.add(out + row)
template <int D, bool GU>
__device__ __forceinline__ void q4_stage(const uint8_t* st, int nr, int rho0, const Q4Frag<D>& f, int cw, int lane,
                                         float* abuf, float* out) {
  constexpr int LPR = Q4Frag<D>::LPR, RPW = 32 / LPR, CPL = Q4Frag<D>::CPL;
  constexpr int IR = RPW > 2 ? RPW : 2;
  constexpr int NP = IR / RPW;
  const uint4* q = reinterpret_cast<const uint4*>(st);
  const uint16_t* s = reinterpret_cast<const uint16_t*>(st + (size_t)nr * D / 2);
  const uint16_t* b = s + nr * (D / 64);
  for (int it = 0; it < nr / IR; ++it) {
    if (((rho0 / IR) + it) % NCW != cw) continue;
    float vals[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int r = it * IR + p * RPW + lane / LPR;
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane % LPR + LPR * j;
        const uint4 qq = q[r * (D / 32) + c];
        const int a = dot32(qq, f.xp[j]);
        const float sf = bf(s[r * (D / 64) + (c >> 1)]);
        const float bb = bf(b[r * (D / 64) + (c >> 1)]);
        v += sf * ((float)a * f.inv[j]) + bb * f.sum[j];
      }
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      vals[p] = v;
    }
    if (GU) {
      if (RPW == 1) {
        if (lane == 0) abuf[(rho0 + it * IR) / 2] = silu_f(vals[0]) * vals[NP - 1];
      } else {
        const float up = __shfl_down_sync(0xffffffffu, vals[0], LPR);
        if (lane % (2 * LPR) == 0) abuf[(rho0 + it * IR + lane / LPR) / 2] = silu_f(vals[0]) * up;
      }
    } else {
      if (lane % LPR == 0) {
#pragma unroll
        for (int p = 0; p < NP; ++p) red_add_f32(out + rho0 + it * IR + p * RPW + lane / LPR, vals[p]);
      }
    }
  }
}

template <int D>
struct BfFrag {
  static constexpr int CPL = D / 256;  // chunks of 8 per lane
  float x[CPL][8];
  __device__ __forceinline__ void load(const Ctl& C, int lane) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const float4* p = reinterpret_cast<const float4*>(C.x + 8 * (lane + 32 * j));
      const float4 a = p[0], c = p[1];
      x[j][0] = a.x; x[j][1] = a.y; x[j][2] = a.z; x[j][3] = a.w;
      x[j][4] = c.x; x[j][5] = c.y; x[j][6] = c.z; x[j][7] = c.w;
    }
  }
};

// bf16 rows (in = D) of one stage, one warp per row; out(row_in_part, value) on lane 0.
template <int D, class Out>
__device__ __forceinline__ void bf_stage(const uint8_t* st, int nr, int rho0, const BfFrag<D>& f, int cw, int lane,
                                         Out out) {
  const uint4* w = reinterpret_cast<const uint4*>(st);
  for (int r = 0; r < nr; ++r) {
    if ((rho0 + r) % NCW != cw) continue;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int j = 0; j < BfFrag<D>::CPL; ++j) {
      const uint4 u = w[r * (D / 8) + lane + 32 * j];
      v0 = fmaf(bflo(u.x), f.x[j][0], v0); v1 = fmaf(bfhi(u.x), f.x[j][1], v1);
      v0 = fmaf(bflo(u.y), f.x[j][2], v0); v1 = fmaf(bfhi(u.y), f.x[j][3], v1);
      v0 = fmaf(bflo(u.z), f.x[j][4], v0); v1 = fmaf(bfhi(u.z), f.x[j][5], v1);
      v0 = fmaf(bflo(u.w), f.x[j][6], v0); v1 = fmaf(bfhi(u.w), f.x[j][7], v1);
    }
    const float v = warp_sum(v0 + v1);
    if (lane == 0) out(rho0 + r, v);
  }
}

template <int D, class Out>
__device__ void consume_bf_rows(Cons& cs, int rows, Out out) {
  BfFrag<D> f;
  f.load(cs.C, cs.lane);
  const int per = bf_rows_per_stage(D);
  for (int r = 0; r < rows; r += per) {
    uint32_t slot;
    const uint8_t* st = cs.acquire(slot);
    if (st) bf_stage<D>(st, min(per, rows - r), r, f, cs.cw, cs.lane, out);
    cs.release(slot);
  }
}

template <int D>
__device__ void consume_unit(Cons& cs, const LayerDesc& Ld, const Unit& u, int l, float* acc, float* zhat,
                             float* zr) {
  const EngineParams& P = cs.P;
  Ctl& C = cs.C;
  const int slot4 = l & 3;
  const int cw = cs.cw, lane = cs.lane, tid = cs.tid;
  switch (u.type) {
    case U_EXPERT: {
      const bool shared = u.k >= P.K;
      cbar();  // abuf reuse
      if (!shared) spin_until(P, C, [&] { return C.route_seq > l; }, P.timeout_ns);
      // The named barriers below are executed unconditionally so that every warp
      // reaches the same barriers even if the route table were read inconsistently.
      const bool valid = shared ? Ld.has_shared != 0 : ((C.r_valid[slot4] >> u.k) & 1u) != 0;
      if (valid) {
        Q4Frag<D> f;
        f.load(C, lane);
        const int per = q4_rows_per_stage(D);
        for (int r = 0; r < 64; r += per) {
          uint32_t slot;
          const uint8_t* st = cs.acquire(slot);
          if (st) q4_stage<D, true>(st, min(per, 64 - r), r, f, cw, lane, C.abuf, nullptr);
          cs.release(slot);
        }
      }
      cbar();  // all 32 activations ready
      if (valid) {
        float av[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) av[i] = C.abuf[i];
        uint32_t ap[16];
        float asum;
        const float ainv = quant_chunk32(av, ap, &asum);
        const float wk = shared ? 1.0f : C.r_w[slot4][u.k];
        const int pd = dn_rows_per_stage(P.d);
        for (int i0 = 0; i0 < P.d; i0 += pd) {
          const int nr = min(pd, P.d - i0);
          uint32_t slot;
          const uint8_t* st = cs.acquire(slot);
          if (st) {
            const uint4* q = reinterpret_cast<const uint4*>(st);
            const uint16_t* s = reinterpret_cast<const uint16_t*>(st + nr * 16);
            const uint16_t* b = s + nr;
            for (int r = cw * 32 + lane; r < nr; r += NCT) {
              const int a = dot32(q[r], ap);
              const float v = bf(s[r]) * ((float)a * ainv) + bf(b[r]) * asum;
              red_add_f32(acc + i0 + r, wk * v);
            }
          }
          cs.release(slot);
        }
      }
      break;
    }
    case U_QROWS: {
      Q4Frag<D> f;
      f.load(C, lane);
      const int per = q4_rows_per_stage(D);
      for (int r = u.r0; r < u.r1; r += per) {
        uint32_t slot;
        const uint8_t* st = cs.acquire(slot);
        if (st) q4_stage<D, false>(st, min(per, u.r1 - r), r, f, cw, lane, nullptr, acc);
        cs.release(slot);
      }
      break;
    }
    case U_LORA_AB: {
      cbar();  // vbuf reuse
      float* vb = C.vbuf;
      consume_bf_rows<D>(cs, u.r1 - u.r0, [&](int r, float v) { vb[r] = v; });
      cbar();
      const int out = Ld.lout;
      const int per = max(1, STAGE_BYTES / (2 * out));
      for (int q0 = 0; q0 < u.r1 - u.r0; q0 += per) {
        const int nr = min(per, u.r1 - u.r0 - q0);
        uint32_t slot;
        const uint8_t* st = cs.acquire(slot);
        if (st) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(st);
          for (int i2 = tid; i2 < out / 2; i2 += NCT) {
            float s0 = 0.f, s1 = 0.f;
            for (int r = 0; r < nr; ++r) {
              const uint32_t ww = w[r * (out / 2) + i2];
              const float v = vb[q0 + r];
              s0 = fmaf(bflo(ww), v, s0);
              s1 = fmaf(bfhi(ww), v, s1);
            }
            red_add_f32(acc + 2 * i2, Ld.lscale * s0);
            red_add_f32(acc + 2 * i2 + 1, Ld.lscale * s1);
          }
        }
        cs.release(slot);
      }
      break;
    }
    case U_HEAD: {
      cbar();  // ubuf reuse
      float* ub = C.ubuf;
      consume_bf_rows<D>(cs, u.r1 - u.r0, [&](int r, float v) { ub[r] = v; });
      spin_until(P, C, [&] { return C.route_seq > l; }, P.timeout_ns);
      cbar();
      const int nr = u.r1 - u.r0;
      {
        uint32_t slot;
        const uint8_t* st = cs.acquire(slot);
        if (st && tid < nr) {
          const uint16_t* g = reinterpret_cast<const uint16_t*>(st);
          float v = ub[tid];
          if (Ld.b1) v += bf(g[tid]);
          const uint32_t cv = C.r_valid[slot4], pv = C.r_prev_valid[slot4];
          for (int k = 0; k < P.K; ++k) {
            if ((cv >> k) & 1u) v += bf(g[(1 + k) * nr + tid]);
            if ((pv >> k) & 1u) v += bf(g[(1 + P.K + k) * nr + tid]);
          }
          ub[tid] = gelu_f(v);
        }
        cs.release(slot);
      }
      cbar();
      const int E = P.E;
      const int per = max(1, STAGE_BYTES / (2 * E));
      for (int i0 = 0; i0 < nr; i0 += per) {
        const int ni = min(per, nr - i0);
        uint32_t slot;
        const uint8_t* st = cs.acquire(slot);
        if (st) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(st);
          for (int e2 = tid; e2 < E / 2; e2 += NCT) {
            float s0 = 0.f, s1 = 0.f;
            for (int r = 0; r < ni; ++r) {
              const uint32_t ww = w[r * (E / 2) + e2];
              const float p = ub[i0 + r];
              s0 = fmaf(bflo(ww), p, s0);
              s1 = fmaf(bfhi(ww), p, s1);
            }
            red_add_f32(zhat + 2 * e2, s0);
            red_add_f32(zhat + 2 * e2 + 1, s1);
          }
        }
        cs.release(slot);
      }
      break;
    }
    case U_LRES: {
      const uint16_t* b2 = Ld.b2;
      const int e0 = u.r0;
      consume_bf_rows<D>(cs, u.r1 - u.r0, [&](int r, float v) {
        red_add_f32(zhat + e0 + r, v + (b2 ? bf(b2[e0 + r]) : 0.f));
      });
      break;
    }
    case U_ROUTER: {
      const int e0 = u.r0;
      consume_bf_rows<D>(cs, u.r1 - u.r0, [&](int r, float v) { zr[e0 + r] = v; });
      break;
    }
    default:
      break;
  }
}

// Build the layer input: residual h (fp32 of bf16 values) and normed x, plus the
// int16 copy of x used by the int4 rows.  All consumer threads.
__device__ void layer_input(Cons& cs, int l, uint32_t par) {
  const EngineParams& P = cs.P;
  Ctl& C = cs.C;
  const int d = P.d, tid = cs.tid;
  float ss = 0.f;
  for (int i = tid; i < d; i += NCT) {
    float h;
    if (P.mode == MODE_STACK) {
      uint16_t hb;
      if (l == 0) {
        hb = P.h_in[i];
      } else {
        hb = f32_to_bf16_bits(C.res[i] + ld_cg_f32(acc_ptr(P, par, l - 1) + i));
      }
      h = P.incr ? bf(f32_to_bf16_bits(bf(hb) + bf(P.incr[(size_t)l * d + i]))) : bf(hb);
    } else {
      h = bf(P.h_in[i]);
    }
    C.res[i] = h;
    ss += h * h;
  }
  ss = warp_sum(ss);
  if (cs.lane == 0) C.red[cs.cw] = ss;
  cbar();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) tot += C.red[w];
  const float scale = P.norm ? rsqrtf(tot / (float)d + RMS_EPS) : 1.0f;
  for (int i = tid; i < d; i += NCT) C.x[i] = C.res[i] * scale;
  cbar();
  for (int c = tid; c < d / 32; c += NCT) {
    uint32_t xp[16];
    float s;
    const float inv = quant_chunk32(C.x + 32 * c, xp, &s);
    uint4* dst = C.xq + 4 * c;
    dst[0] = make_uint4(xp[0], xp[1], xp[2], xp[3]);
    dst[1] = make_uint4(xp[4], xp[5], xp[6], xp[7]);
    dst[2] = make_uint4(xp[8], xp[9], xp[10], xp[11]);
    dst[3] = make_uint4(xp[12], xp[13], xp[14], xp[15]);
    C.xinv[c] = inv;
    C.xsum[c] = s;
  }
  if (P.mode == MODE_STACK && P.h_trace && blockIdx.x == 0)
    for (int i = tid; i < d; i += NCT) P.h_trace[(size_t)l * d + i] = f32_to_bf16_bits(C.res[i]);
  cbar();
}

template <int D>
__device__ void consumer(const EngineParams& P, Ctl& C, uint8_t* ring) {
  Cons cs{P, C, ring, 0u, (int)(threadIdx.x >> 5), (int)(threadIdx.x & 31), (int)threadIdx.x};
  const int tid = cs.tid;
  const uint32_t par = C.epoch & 1u, p3 = C.epoch % 3u;
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
    if (l > 0 && P.mode == MODE_STACK) {
      if (tid == 0)
        spin_until(P, C, [&] { return ld_acquire_u32(ctr(P, par, l - 1, 0)) >= (uint32_t)ncta; }, P.timeout_ns);
      cbar();
    }
    if (tid == 0) stamp(P, l, 1);
    layer_input(cs, l, par);
    if (tid == 0) stamp(P, l, 2);
    float* acc = acc_ptr(P, par, l);
    float* zh = zhat_ptr(P, pnext3, l);
    float* zr = zr_ptr(P, par, l);
    const bool self_route = P.mode == MODE_STACK && ((P.router_mask >> l) & 1ull);
    if (self_route) {
      int nu;
      const Unit* us = units_of(P, KIND_ROUTER, cta, nu);
      for (int i = 0; i < nu; ++i) consume_unit<D>(cs, Ld, us[i], l, acc, zh, zr);
      cbar();
      if (tid == 0) {
        __threadfence();
        red_release_add_u32(ctr(P, par, l, 1), 1u);
      }
    }
    int nu;
    const Unit* us = units_of(P, P.plan ? Ld.plan_kind : 0, cta, nu);
    for (int i = 0; i < nu; ++i) consume_unit<D>(cs, Ld, us[i], l, acc, zh, zr);
    if (tid == 0) stamp(P, l, 3);

    if (l == P.L - 1) {
      // Clear the other half of the parity-duplicated buffers for the next launch.
      const size_t n_ctr = (size_t)P.L * 2, n_acc = (size_t)P.L * P.out_dim, n_z = (size_t)P.L * P.E;
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
      __threadfence();
      if (l == P.L - 1) {
        const uint32_t old = atom_acq_rel_add_u32(ctr(P, par, l, 0), 1u);
        C.is_last = (old == (uint32_t)ncta - 1u);
      } else {
        red_release_add_u32(ctr(P, par, l, 0), 1u);
      }
      C.cons_done = l + 1;
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
    warp_topk(C.zbuf, P.E, P.K, cs.lane, C.f_ids, C.f_vals);
    if (cs.lane == 0) {
      const float mx = C.f_vals[0];
      float s = 0.f;
      for (int k = 0; k < P.K; ++k) s += expf(C.f_vals[k] - mx);
      for (int k = 0; k < P.K; ++k) {
        if (P.next_ids) P.next_ids[k] = C.f_ids[k];
        if (P.next_w) P.next_w[k] = expf(C.f_vals[k] - mx) / s;
      }
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
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  Ctl& C = *reinterpret_cast<Ctl*>(smem + (size_t)NSTAGES * STAGE_BYTES);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGES; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], NCW);
    }
    fence_mbar_init();
    C.route_seq = 0;
    C.cons_done = 0;
    C.abort_flag = 0;
    C.is_last = 0;
    C.epoch = *reinterpret_cast<volatile uint32_t*>(&hdr(P)->epoch);
  }
  __syncthreads();
  if (threadIdx.x >= NCT)
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
