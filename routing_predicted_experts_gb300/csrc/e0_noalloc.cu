// e0_moe_decode_layer_noalloc: the single-token MoE layer-step for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not allowed —
// for example inside a host callback or a real-time loop that must not block on the
// allocator, a plugin whose host framework owns every device allocation, or a process
// that has pinned its memory budget up front.  Such callers cannot provide the
// workspace that e0_moe_decode_layer needs for its grid-wide counters and fp32
// accumulators.  This entry point keeps that workspace in a fixed array in the
// library's own device memory instead, so the caller passes only inputs and outputs.
//
// The array below is reserved on every GPU that loads the library, for the life of
// the process.  Its address is looked up once per device, the first time this entry
// point runs on that device (make that first call before any stream capture).  Each
// call clears the part of the array it uses on `stream` before launching, so no state
// carries over from earlier calls; calls on different streams that overlap on the
// GPU share the array and race, so order them on one stream.
#include <mutex>

#include "e0_engine.cuh"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 128 * 1024;  // upper bound on the workspace used
constexpr int NOALLOC_MAX_DEVICES = 64;
// every valid dims fits: the single-layer workspace grows only with E (<= EMAX)
static_assert(e0eng::ws_layout(e0eng::EMAX, 1).total <= NOALLOC_SCRATCH_BYTES,
              "the scratch array must hold the largest single-layer workspace");

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device (set-up once per device).
e0_status noalloc_scratch(void** out) {
  int dev = 0;
  E0_CHECK_CUDA(cudaGetDevice(&dev));
  E0_REQUIRE(dev >= 0 && dev < NOALLOC_MAX_DEVICES, E0_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    E0_CHECK_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return E0_OK;
}

}  // namespace

extern "C" e0_status e0_moe_decode_layer_noalloc(const e0_dims* dims, const e0_experts* routed,
                                                 const e0_experts* shared, const e0_qlora* lora,
                                                 const e0_prerouter* head, const uint16_t* h_in,
                                                 const int32_t* ids, const float* logits,
                                                 const int32_t* ids_prev, uint16_t* h_out, float* delta_f32,
                                                 float* next_logits, int32_t* next_ids, float* next_weights,
                                                 e0_stream stream) {
  E0_REQUIRE(dims, E0_ERR_INVALID, "e0_moe_decode_layer_noalloc: dims is NULL");
  // every argument check comes before anything is queued on the stream
  e0_status st = e0::check_dims(dims);
  if (st != E0_OK) return st;
  E0_REQUIRE(routed && h_in && ids && logits && h_out, E0_ERR_INVALID,
             "e0_moe_decode_layer_noalloc: NULL required argument");
  const size_t need = e0_workspace_size(dims, 1);
  E0_REQUIRE(need > 0, E0_ERR_SHAPE, "e0_moe_decode_layer_noalloc: unsupported dims");
  E0_REQUIRE(need <= NOALLOC_SCRATCH_BYTES, E0_ERR_NOMEM,
             "e0_moe_decode_layer_noalloc: these dims need a workspace larger than the built-in 128 KiB scratch");
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != E0_OK) return st;
  E0_CHECK_CUDA(cudaMemsetAsync(ws, 0, need, (cudaStream_t)stream));
  return e0_moe_decode_layer(dims, routed, shared, lora, head, h_in, ids, logits, ids_prev, 1, h_out, delta_f32,
                             next_logits, next_ids, next_weights, ws, need, stream);
}
