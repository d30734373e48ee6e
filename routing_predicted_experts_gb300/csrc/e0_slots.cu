// Bounded HBM expert-slot pool for decode with host-resident experts.
//
// "The Other Half of the Memory Wall" (Edge0), §3.1 and §3.2: experts live off the GPU
// and a bounded set of slots holds the ones the routing needs; the prerouter commits
// the next layer's routing one token ahead, which is the lead time for staging its
// experts.  Here the experts live in pinned host memory, one bundle per (layer,
// expert) holding its six tensors; each layer owns S slots in HBM with the same bundle
// layout, replaced least-recently-used.  The experts the running token uses and the
// ones being staged are never evicted.  A miss is one asynchronous host-to-device copy
// of the bundle on the caller's copy stream, followed by the layer's id -> slot table.
#include <cstring>
#include <vector>

#include "e0_engine.cuh"

using namespace e0eng;

struct e0_slot_pool {
  e0_dims dims{};
  int L = 0, E = 0, S = 0;
  size_t bundle = 0;
  size_t off[6] = {};
  const uint8_t* host = nullptr;  // [L][E][bundle], pinned, caller-owned
  uint8_t* dev = nullptr;         // [L][S][bundle]
  int16_t* d_slot_of = nullptr;   // [L][E]
  int16_t* h_snap = nullptr;      // pinned [L][2][E]: table snapshots for the copies
  std::vector<cudaEvent_t> snap_done;  // [L][2]
  std::vector<int> slot_id;       // [L][S] expert held by a slot, -1 = free
  std::vector<int> id_slot;       // [L][E]
  std::vector<uint64_t> stamp;    // [L][S] last use
  std::vector<int> cur;           // [L][KMAX] experts of the previous staging (in use by the running token)
  std::vector<int> ncur;          // [L]
  std::vector<int> flip;          // [L]
  uint64_t clock = 0;
};

namespace {

// Bundle layout of one expert: gate/up codes, scales, biases, then down codes, scales,
// biases, each 256-byte aligned.
void bundle_layout(const e0_dims* dm, size_t off[6], size_t* total) {
  const size_t d = dm->d, F = dm->F;
  const size_t sz[6] = {2 * F * d / 2, 2 * F * (d / 64) * 2, 2 * F * (d / 64) * 2,
                        d * F / 2,     (F / 64) * d * 2,     (F / 64) * d * 2};
  size_t o = 0;
  for (int i = 0; i < 6; ++i) {
    off[i] = o;
    o = (o + sz[i] + 255) & ~size_t(255);
  }
  *total = o;
}

}  // namespace

extern "C" size_t e0_expert_bundle_bytes(const e0_dims* dims, size_t* offsets6) {
  if (!dims || dims->d <= 0 || dims->F <= 0) return 0;
  size_t off[6], total;
  bundle_layout(dims, off, &total);
  if (offsets6) std::memcpy(offsets6, off, sizeof(off));
  return total;
}

extern "C" void e0_slot_pool_destroy(e0_slot_pool* p) {
  if (!p) return;
  for (cudaEvent_t e : p->snap_done)
    if (e) cudaEventDestroy(e);
  if (p->dev) cudaFree(p->dev);
  if (p->d_slot_of) cudaFree(p->d_slot_of);
  if (p->h_snap) cudaFreeHost(p->h_snap);
  delete p;
}

extern "C" e0_status e0_slot_pool_create(e0_slot_pool** out, const e0_dims* dims, int32_t layers, int32_t slots,
                                         const void* host_bundles, size_t bundle_bytes) {
  E0_REQUIRE(out && dims && host_bundles, E0_ERR_INVALID, "e0_slot_pool_create: NULL argument");
  *out = nullptr;
  E0_REQUIRE(layers >= 1 && dims->E >= 1 && dims->K >= 1, E0_ERR_SHAPE, "e0_slot_pool_create: layers, E, K");
  E0_REQUIRE(slots >= 2 * dims->K && slots <= dims->E, E0_ERR_SHAPE,
             "e0_slot_pool_create: need 2K <= slots <= E (the running and the staged experts are pinned)");
  E0_REQUIRE(slots <= 32767, E0_ERR_SHAPE, "e0_slot_pool_create: slot index must fit int16");
  size_t off[6], total;
  bundle_layout(dims, off, &total);
  E0_REQUIRE(bundle_bytes == total, E0_ERR_SHAPE,
             "e0_slot_pool_create: bundle_bytes must equal e0_expert_bundle_bytes(dims)");
  e0_slot_pool* p = new e0_slot_pool;
  p->dims = *dims;
  p->L = layers;
  p->E = dims->E;
  p->S = slots;
  p->bundle = total;
  std::memcpy(p->off, off, sizeof(off));
  p->host = static_cast<const uint8_t*>(host_bundles);
  auto fail = [&](cudaError_t e, const char* what) {
    e0_slot_pool_destroy(p);
    return e0::cuda_fail(e, what);
  };
  cudaError_t e = cudaMalloc(&p->dev, (size_t)layers * slots * total);
  if (e != cudaSuccess) return fail(e, "cudaMalloc(slots)");
  e = cudaMalloc(&p->d_slot_of, sizeof(int16_t) * (size_t)layers * p->E);
  if (e != cudaSuccess) return fail(e, "cudaMalloc(slot_of)");
  e = cudaMemset(p->d_slot_of, 0xFF, sizeof(int16_t) * (size_t)layers * p->E);  // -1: nothing resident
  if (e != cudaSuccess) return fail(e, "cudaMemset(slot_of)");
  e = cudaHostAlloc(&p->h_snap, sizeof(int16_t) * (size_t)layers * 2 * p->E, cudaHostAllocDefault);
  if (e != cudaSuccess) return fail(e, "cudaHostAlloc(snapshots)");
  p->snap_done.assign((size_t)layers * 2, nullptr);
  for (auto& ev : p->snap_done) {
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(e, "cudaEventCreate");
  }
  p->slot_id.assign((size_t)layers * slots, -1);
  p->id_slot.assign((size_t)layers * p->E, -1);
  p->stamp.assign((size_t)layers * slots, 0);
  p->cur.assign((size_t)layers * KMAX, -1);
  p->ncur.assign(layers, 0);
  p->flip.assign(layers, 0);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(e, "cudaDeviceSynchronize");
  *out = p;
  return E0_OK;
}

extern "C" e0_status e0_slot_pool_view(const e0_slot_pool* p, int32_t layer, e0_experts* out) {
  E0_REQUIRE(p && out, E0_ERR_INVALID, "e0_slot_pool_view: NULL argument");
  E0_REQUIRE(layer >= 0 && layer < p->L, E0_ERR_INVALID, "e0_slot_pool_view: layer out of range");
  uint8_t* base = p->dev + (size_t)layer * p->S * p->bundle;
  out->gate_up.q = reinterpret_cast<const uint32_t*>(base + p->off[0]);
  out->gate_up.scale = reinterpret_cast<const uint16_t*>(base + p->off[1]);
  out->gate_up.bias = reinterpret_cast<const uint16_t*>(base + p->off[2]);
  out->down.q = reinterpret_cast<const uint32_t*>(base + p->off[3]);
  out->down.scale = reinterpret_cast<const uint16_t*>(base + p->off[4]);
  out->down.bias = reinterpret_cast<const uint16_t*>(base + p->off[5]);
  out->n = p->S;
  out->slot_of = p->d_slot_of + (size_t)layer * p->E;
  out->stride = (int64_t)p->bundle;
  return E0_OK;
}

namespace {
e0_status stage_one(e0_slot_pool* p, int32_t layer, const int32_t* next_ids, int32_t K, cudaStream_t st,
                    e0_stage_stats* stats);
}  // namespace

extern "C" e0_status e0_stage_slots(e0_slot_pool* p, int32_t layer, const int32_t* next_ids, int32_t K,
                                    e0_stream copy_stream, e0_event ready, e0_stage_stats* stats) {
  E0_REQUIRE(p && next_ids, E0_ERR_INVALID, "e0_stage_slots: NULL argument");
  e0_status s = stage_one(p, layer, next_ids, K, (cudaStream_t)copy_stream, stats);
  if (s != E0_OK) return s;
  if (ready) E0_CHECK_CUDA(cudaEventRecord((cudaEvent_t)ready, (cudaStream_t)copy_stream));
  return E0_OK;
}

extern "C" e0_status e0_stage_slots_layers(e0_slot_pool* p, const int32_t* layers, int32_t n_layers,
                                           const int32_t* next_ids, int32_t K, e0_stream copy_stream, e0_event ready,
                                           e0_stage_stats* stats) {
  E0_REQUIRE(p && layers && next_ids && n_layers >= 0, E0_ERR_INVALID, "e0_stage_slots_layers: NULL argument");
  for (int i = 0; i < n_layers; ++i) {
    e0_status s = stage_one(p, layers[i], next_ids + (size_t)i * K, K, (cudaStream_t)copy_stream, stats);
    if (s != E0_OK) return s;
  }
  if (ready) E0_CHECK_CUDA(cudaEventRecord((cudaEvent_t)ready, (cudaStream_t)copy_stream));
  return E0_OK;
}

namespace {
e0_status stage_one(e0_slot_pool* p, int32_t layer, const int32_t* next_ids, int32_t K, cudaStream_t st,
                    e0_stage_stats* stats) {
  E0_REQUIRE(layer >= 0 && layer < p->L, E0_ERR_INVALID, "e0_stage_slots: layer out of range");
  E0_REQUIRE(K >= 1 && K <= KMAX && 2 * K <= p->S, E0_ERR_SHAPE, "e0_stage_slots: K out of range");
  const int E = p->E, S = p->S;
  int* slot_id = &p->slot_id[(size_t)layer * S];
  int* id_slot = &p->id_slot[(size_t)layer * E];
  uint64_t* stamp = &p->stamp[(size_t)layer * S];
  const int* cur = &p->cur[(size_t)layer * KMAX];
  const int ncur = p->ncur[layer];
  for (int k = 0; k < K; ++k)
    E0_REQUIRE(next_ids[k] >= 0 && next_ids[k] < E, E0_ERR_INVALID, "e0_stage_slots: expert id out of range");
  auto pinned = [&](int id) {
    for (int k = 0; k < K; ++k)
      if (next_ids[k] == id) return true;
    for (int k = 0; k < ncur; ++k)
      if (cur[k] == id) return true;
    return false;
  };
  e0_stage_stats s{};
  bool changed = false;
  for (int k = 0; k < K; ++k) {
    const int id = next_ids[k];
    bool dup = false;
    for (int j = 0; j < k; ++j) dup = dup || next_ids[j] == id;
    if (dup) continue;
    int slot = id_slot[id];
    if (slot >= 0) {
      ++s.hits;
    } else {
      // victim: a free slot, else the least recently used slot not pinned
      int victim = -1;
      for (int i = 0; i < S && victim < 0; ++i)
        if (slot_id[i] < 0) victim = i;
      if (victim < 0) {
        uint64_t best = ~0ull;
        for (int i = 0; i < S; ++i)
          if (!pinned(slot_id[i]) && stamp[i] < best) {
            best = stamp[i];
            victim = i;
          }
      }
      E0_REQUIRE(victim >= 0, E0_ERR_UNSUPPORTED, "e0_stage_slots: every slot is pinned");
      if (slot_id[victim] >= 0) {
        id_slot[slot_id[victim]] = -1;
        ++s.evictions;
      }
      slot_id[victim] = id;
      id_slot[id] = victim;
      slot = victim;
      ++s.misses;
      s.h2d_bytes += (int64_t)p->bundle;
      E0_CHECK_CUDA(cudaMemcpyAsync(p->dev + ((size_t)layer * S + victim) * p->bundle,
                                    p->host + ((size_t)layer * E + id) * p->bundle, p->bundle,
                                    cudaMemcpyHostToDevice, st));
      changed = true;
    }
    stamp[slot] = ++p->clock;
  }
  if (changed) {
    // the id -> slot table, from one of two pinned snapshots per layer (the one whose
    // previous copy has finished)
    const int f = p->flip[layer];
    cudaEvent_t ev = p->snap_done[(size_t)layer * 2 + f];
    E0_CHECK_CUDA(cudaEventSynchronize(ev));
    int16_t* snap = p->h_snap + ((size_t)layer * 2 + f) * E;
    for (int e = 0; e < E; ++e) snap[e] = (int16_t)id_slot[e];
    E0_CHECK_CUDA(cudaMemcpyAsync(p->d_slot_of + (size_t)layer * E, snap, sizeof(int16_t) * E,
                                  cudaMemcpyHostToDevice, st));
    E0_CHECK_CUDA(cudaEventRecord(ev, st));
    p->flip[layer] = f ^ 1;
  }
  int* cw = &p->cur[(size_t)layer * KMAX];
  for (int k = 0; k < K; ++k) cw[k] = next_ids[k];
  p->ncur[layer] = K;
  if (stats) {
    stats->hits += s.hits;
    stats->misses += s.misses;
    stats->evictions += s.evictions;
    stats->h2d_bytes += s.h2d_bytes;
  }
  return E0_OK;
}
}  // namespace
