// Shared device/host helpers for libe0 (sm_103a).  Inline PTX for the Blackwell
// async-copy machinery: mbarriers, cp.async.bulk (TMA bulk copies into shared
// memory), proxy fences, %globaltimer, scoped atomics.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string>

#include "../../include/e0.h"

// ------------------------------------------------------------------ host errors
namespace e0 {
void set_error(const std::string& msg);
e0_status fail(e0_status code, const std::string& msg);
e0_status cuda_fail(cudaError_t err, const char* what);
// Dimension and routing-family checks shared by every entry point.
e0_status check_dims(const e0_dims* dm);
e0_status check_route(const e0_dims* dm);  // the routing family's parameters only
}  // namespace e0

#define E0_CHECK_CUDA(call)                                        \
  do {                                                             \
    cudaError_t e0_err__ = (call);                                 \
    if (e0_err__ != cudaSuccess) return e0::cuda_fail(e0_err__, #call); \
  } while (0)

#define E0_REQUIRE(cond, code, msg)                                \
  do {                                                             \
    if (!(cond)) return e0::fail((code), (msg));                   \
  } while (0)

// ------------------------------------------------------------------ device helpers
namespace e0dev {

// Routing family of a call ("The Other Half of the Memory Wall", Appendix A).
struct RouteArgs {
  int32_t family;              // E0_ROUTE_*
  int32_t n_group, topk_group;
  float scale;
  const float* sbias;          // sigmoid-group selection bias [E] (nullable)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Phase test that lets the hardware suspend the thread until the phase completes or
// about `hint_ns` pass (no busy issue slots while a warp waits).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Four phase tests issued back to back (independent, so their latencies overlap); true
// when all four phases have completed.  Unused slots repeat a barrier already tested.
__device__ __forceinline__ bool mbar_try_wait4(const uint64_t* b0, uint32_t p0, const uint64_t* b1, uint32_t p1,
                                               const uint64_t* b2, uint32_t p2, const uint64_t* b3, uint32_t p3) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred q0, q1, q2, q3;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
      "and.pred q0, q0, q1;\n\tand.pred q2, q2, q3;\n\tand.pred q0, q0, q2;\n\t"
      "selp.u32 %0, 1, 0, q0; }"
      : "=r"(ok)
      : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2), "r"(smem_u32(b3)),
        "r"(p3)
      : "memory");
  return ok != 0;
}

// Bulk async copy global -> shared, completion signalled on `bar` (complete_tx).
// dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void tma_bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (no completion to wait for); src 16-byte
// aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order this thread's earlier generic-proxy accesses to shared memory before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// System-scope acquire: for words written by a host-to-device copy on another stream.
__device__ __forceinline__ uint32_t ld_acquire_sys_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_acq_rel_add_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void red_add_v4_f32(float* p, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// A value published with its tag in one 64-bit word: a reader that sees the tag it
// expects also sees the value written with it (single-copy atomic 64-bit access), so
// no counter or fence is needed between writer and reader.
__device__ __forceinline__ void st_tagged(uint64_t* p, uint32_t tag, float v) {
  const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// L2-coherent loads for data written by other CTAs during the same launch.
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cg_s32(const int* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ top-K keys
// Order key of (logit, id): larger logit first, equal logits to the lower id.
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  if (v != v) u = 0u;
  return ((uint64_t)u << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

// Top-K of logits held in registers (lane holds z[lane + 32 j], j < NPL), descending,
// ties to the lower index, with the same key order as warp_topk.  Each round takes the
// warp maximum of the keys below the previous pick with two integer reductions (high
// then low word).  Lane k < K receives the k-th id (-1 if none) and its logit.
__device__ __forceinline__ float topk_key_value(uint32_t hi) {
  return __uint_as_float((hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi);
}
template <int NPL>
__device__ __forceinline__ void warp_topk_regs(const float (&z)[NPL], int E, int K, int lane, int& id, float& val) {
  uint64_t key[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? topk_key(z[j], e) : 0ull;
  }
  uint64_t prev = ~0ull;
  id = -1;
  val = 0.f;
  for (int k = 0; k < K; ++k) {
    uint64_t m = 0ull;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
      if (key[j] < prev && key[j] > m) m = key[j];
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(m >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(m >> 32) == hi ? (uint32_t)m : 0u);
    prev = ((uint64_t)hi << 32) | lo;
    if (lane == k && prev != 0ull) {
      id = (int)(0xFFFFFFFFu - lo);
      val = topk_key_value(hi);
    }
  }
}

// Warp maximum of a 64-bit key (two integer reductions: high word, then low word).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32) == hi ? (uint32_t)k : 0u);
  return ((uint64_t)hi << 32) | lo;
}

// Sigmoid-group routing of one token ("The Other Half of the Memory Wall", Appendix A
// "Sigmoid-group") from its logits z[0..E) (shared or global memory); every lane of the
// warp calls.  sigma = 1/(1+e^-z); score = sigma + sbias (selection only); a group (a
// contiguous block of E/n_group experts) scores the sum of its two best scores; the
// topk_group best groups survive (ties to the lower group); ids = top-K of the scores
// within them (descending, ties to the lower id); w = scale * sigma / (sum of the picked
// sigma + 1e-20).  Lane k < K receives id k (-1 if none) and its final weight.
__device__ __forceinline__ void sigmoid_group_route(const float* z, const float* sbias, int E, int K, int n_group,
                                                    int topk_group, float scale, int lane, int& id_out,
                                                    float& w_out) {
  const int gs = E / n_group;
  auto score = [&](int e) { return 1.0f / (1.0f + expf(-z[e])) + (sbias ? sbias[e] : 0.f); };
  float gscore = -INFINITY;  // lane g < n_group: group g's score
  for (int g = 0; g < n_group; ++g) {
    uint64_t k1 = 0ull, k2 = 0ull;
    for (int e = g * gs + lane; e < (g + 1) * gs; e += 32) k1 = max(k1, topk_key(score(e), e));
    k1 = warp_max_key(k1);
    for (int e = g * gs + lane; e < (g + 1) * gs; e += 32) {
      const uint64_t k = topk_key(score(e), e);
      if (k < k1) k2 = max(k2, k);
    }
    k2 = warp_max_key(k2);
    if (lane == g) gscore = topk_key_value((uint32_t)(k1 >> 32)) + topk_key_value((uint32_t)(k2 >> 32));
  }
  int rank = 0;
  for (int o = 0; o < 32; ++o) {
    const float og = __shfl_sync(0xffffffffu, gscore, o);
    if (o < n_group && (og > gscore || (og == gscore && o < lane))) ++rank;
  }
  const uint32_t keep = __ballot_sync(0xffffffffu, lane < n_group && rank < topk_group);
  int id = -1;
  uint64_t prev = ~0ull;
  for (int k = 0; k < K; ++k) {
    uint64_t m = 0ull;
    for (int e = lane; e < E; e += 32)
      if ((keep >> (e / gs)) & 1u) {
        const uint64_t key = topk_key(score(e), e);
        if (key < prev && key > m) m = key;
      }
    prev = warp_max_key(m);
    if (lane == k && prev != 0ull) id = (int)(0xFFFFFFFFu - (uint32_t)prev);
  }
  const float sig = (lane < K && id >= 0) ? 1.0f / (1.0f + expf(-z[id])) : 0.f;
  const float tot = warp_sum(sig);
  id_out = id;
  w_out = scale * sig / (tot + 1e-20f);
}

}  // namespace e0dev

// Host launchers shared between translation units.
cudaError_t e0pf_route_topk(const float* logits, int T, int E, int K, const e0dev::RouteArgs& ra, int32_t* ids,
                            float* w, cudaStream_t st);
e0_status e0pf_grouped_layer(const e0_dims* dims, const e0_experts* routed, const e0_experts* shared,
                             const e0_qlora* lora, const uint16_t* h_in, const float* logits,
                             const int32_t* given_ids, int32_t T, uint16_t* h_out, float* delta_f32,
                             int32_t* ids_out, float* weights_out, void* workspace, size_t workspace_bytes,
                             e0_stream stream);
e0_status e0mt_head(const e0_prerouter* head, const e0_dims* dims, const uint16_t* h, const int32_t* ids_cur,
                    const int32_t* ids_prev, int32_t T, const float* logit_bias, float* logits_out,
                    int32_t* ids_out, float* weights_out, void* scratch, size_t scratch_bytes, uint32_t* status,
                    e0_stream stream);
size_t e0mt_head_scratch(const e0_dims* dims, int32_t T, int32_t H);
