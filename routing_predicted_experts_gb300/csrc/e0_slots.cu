// Bounded HBM expert-slot pool for decode with host-resident experts.
//
// "The Other Half of the Memory Wall" (Edge0), §3.1 and §3.2: experts live off the GPU
// and a bounded set of slots holds the ones the routing needs; the prerouter commits
// the next layer's routing one token ahead, which is the lead time for staging its
// experts.  Here the experts live in pinned host memory, one bundle per (layer,
// expert) holding its six tensors; each layer owns S slots in HBM with the same bundle
// layout, replaced least-recently-used.  The experts the running token uses and the
// ones being staged are never evicted.  A miss is one asynchronous host-to-device copy
// of the bundle on the caller's copy stream, followed by the layer's id -> slot table
// and then the layer's ready word (the token the staging is for), which the decode
// stack polls before it reads the layer's slots.  The routing that drives the copies
// is the one a stack launch committed on the device; it comes to the host once, as a
// small copy after that launch, and the bundle copies run while the next launch
// (already queued) works through the layers before the pooled ones.
//
// Consistency: the pool's host record of which expert each slot holds changes only
// for copies that were queued, and a layer's table is rewritten while it differs from
// what the device last received; a ready word moves only after its layer's copies and
// table are queued.  Each layer has two tables, for tokens of even and odd index, so
// that the next token's staging never rewrites the table the running token reads, and
// the LRU never evicts the running token's experts (the previous staging's).  A failed call therefore leaves the record matching the device
// once the queued copies have run, and a launch waiting for that layer times out (it
// never reads a half-staged layer).
#include <algorithm>
#include <atomic>
#include <chrono>
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
  int16_t* d_slot_of = nullptr;   // [L][2][E]: tables for tokens of even and odd index
  uint32_t* d_ready = nullptr;    // [L] tag of the last completed staging of each layer
  int16_t* h_tab = nullptr;       // pinned [2][L][E]: table snapshots, by the tag's parity
  uint32_t* h_tag = nullptr;      // pinned [2][L]: ready-word snapshots, by the tag's parity
  cudaEvent_t snap_done[2] = {};  // the copies that last read each half of the snapshots
  int32_t* h_ids = nullptr;       // pinned landing buffer for committed device ids
  size_t ids_cap = 0;             // its capacity in ids
  cudaEvent_t ids_done = nullptr;
  std::vector<int> slot_id;       // [L][S] expert held by a slot, -1 = free
  std::vector<int> id_slot;       // [L][E]
  std::vector<uint64_t> stamp;    // [L][S] last use
  std::vector<int> cur;           // [L][KMAX] experts of the previous staging (in use by the running token)
  std::vector<int> ncur;          // [L]
  std::vector<uint8_t> dirty;     // [L][2] the device table of that parity differs from id_slot
  uint64_t clock = 0;
  int fail_after = -1;            // tests: bundle copies left before an injected failure
};

// Layers whose tables and ready words go out together, in one 2-D table copy and one
// ready-word copy: each copy operation has a fixed cost of several microseconds, which
// per layer would exceed the bundle copies themselves.
constexpr int GROUP_LAYERS = 8;

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
    if (e) cudaEventSynchronize(e), cudaEventDestroy(e);
  if (p->ids_done) cudaEventDestroy(p->ids_done);
  if (p->dev) cudaFree(p->dev);
  if (p->d_slot_of) cudaFree(p->d_slot_of);
  if (p->d_ready) cudaFree(p->d_ready);
  if (p->h_tab) cudaFreeHost(p->h_tab);
  if (p->h_tag) cudaFreeHost(p->h_tag);
  if (p->h_ids) cudaFreeHost(p->h_ids);
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
  e = cudaMalloc(&p->d_slot_of, sizeof(int16_t) * (size_t)layers * 2 * p->E);
  if (e != cudaSuccess) return fail(e, "cudaMalloc(slot_of)");
  e = cudaMemset(p->d_slot_of, 0xFF, sizeof(int16_t) * (size_t)layers * 2 * p->E);  // -1: nothing resident
  if (e != cudaSuccess) return fail(e, "cudaMemset(slot_of)");
  e = cudaMalloc(&p->d_ready, sizeof(uint32_t) * (size_t)layers);
  if (e != cudaSuccess) return fail(e, "cudaMalloc(ready)");
  e = cudaMemset(p->d_ready, 0xFF, sizeof(uint32_t) * (size_t)layers);  // no token staged yet
  if (e != cudaSuccess) return fail(e, "cudaMemset(ready)");
  e = cudaHostAlloc(&p->h_tab, sizeof(int16_t) * 2 * (size_t)layers * p->E, cudaHostAllocDefault);
  if (e != cudaSuccess) return fail(e, "cudaHostAlloc(table snapshots)");
  e = cudaHostAlloc(&p->h_tag, sizeof(uint32_t) * 2 * (size_t)layers, cudaHostAllocDefault);
  if (e != cudaSuccess) return fail(e, "cudaHostAlloc(ready snapshots)");
  for (auto& ev : p->snap_done) {
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(e, "cudaEventCreate");
  }
  e = cudaEventCreateWithFlags(&p->ids_done, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(e, "cudaEventCreate");
  p->slot_id.assign((size_t)layers * slots, -1);
  p->id_slot.assign((size_t)layers * p->E, -1);
  p->stamp.assign((size_t)layers * slots, 0);
  p->cur.assign((size_t)layers * KMAX, -1);
  p->ncur.assign(layers, 0);
  p->dirty.assign((size_t)layers * 2, 0);
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
  out->slot_of = p->d_slot_of + (size_t)layer * 2 * p->E;
  out->stride = (int64_t)p->bundle;
  out->ready = p->d_ready + layer;
  return E0_OK;
}

extern "C" e0_status e0_slot_pool_resident(const e0_slot_pool* p, int32_t layer, int16_t* slot_of_out) {
  E0_REQUIRE(p && slot_of_out, E0_ERR_INVALID, "e0_slot_pool_resident: NULL argument");
  E0_REQUIRE(layer >= 0 && layer < p->L, E0_ERR_INVALID, "e0_slot_pool_resident: layer out of range");
  for (int e = 0; e < p->E; ++e) slot_of_out[e] = (int16_t)p->id_slot[(size_t)layer * p->E + e];
  return E0_OK;
}

extern "C" e0_status e0_debug_fail_copies(e0_slot_pool* p, int32_t n) {
  E0_REQUIRE(p, E0_ERR_INVALID, "e0_debug_fail_copies: NULL pool");
  p->fail_after = n < 0 ? -1 : n;
  return E0_OK;
}

namespace {

// Make ids[0..K) resident in pool layer `layer`: the LRU picks the slots, one copy per
// missing bundle is queued on st.  The bookkeeping changes only for copies that were
// queued; the layer's tables are marked as differing from the record.
e0_status stage_bundles(e0_slot_pool* p, int32_t layer, const int32_t* ids, int32_t K, cudaStream_t st,
                        e0_stage_stats* stats) {
  E0_REQUIRE(layer >= 0 && layer < p->L, E0_ERR_INVALID, "e0_stage_slots: layer out of range");
  const int E = p->E, S = p->S;
  for (int k = 0; k < K; ++k)
    E0_REQUIRE(ids[k] >= 0 && ids[k] < E, E0_ERR_INVALID,
               "e0_stage_slots: expert id out of range (a layer without committed routing?)");
  int* slot_id = &p->slot_id[(size_t)layer * S];
  int* id_slot = &p->id_slot[(size_t)layer * E];
  uint64_t* stamp = &p->stamp[(size_t)layer * S];
  const int* cur = &p->cur[(size_t)layer * KMAX];
  const int ncur = p->ncur[layer];
  auto pinned = [&](int id) {
    for (int k = 0; k < K; ++k)
      if (ids[k] == id) return true;
    for (int k = 0; k < ncur; ++k)
      if (cur[k] == id) return true;
    return false;
  };
  e0_stage_stats s{};
  e0_status result = E0_OK;
  for (int k = 0; k < K && result == E0_OK; ++k) {
    const int id = ids[k];
    bool dup = false;
    for (int j = 0; j < k; ++j) dup = dup || ids[j] == id;
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
      if (victim < 0) {
        result = e0::fail(E0_ERR_UNSUPPORTED, "e0_stage_slots: every slot is pinned");
        break;
      }
      cudaError_t err = cudaSuccess;
      if (p->fail_after == 0) {
        p->fail_after = -1;
        err = cudaErrorInvalidValue;  // injected: as if the copy call had failed
      } else {
        if (p->fail_after > 0) --p->fail_after;
        err = cudaMemcpyAsync(p->dev + ((size_t)layer * S + victim) * p->bundle,
                              p->host + ((size_t)layer * E + id) * p->bundle, p->bundle, cudaMemcpyHostToDevice, st);
      }
      if (err != cudaSuccess) {
        result = e0::cuda_fail(err, "cudaMemcpyAsync(expert bundle)");
        break;
      }
      // the copy is queued: from here on the slot holds `id` for every later copy and launch
      if (slot_id[victim] >= 0) {
        id_slot[slot_id[victim]] = -1;
        ++s.evictions;
      }
      slot_id[victim] = id;
      id_slot[id] = victim;
      slot = victim;
      p->dirty[(size_t)layer * 2] = p->dirty[(size_t)layer * 2 + 1] = 1;
      ++s.misses;
      s.h2d_bytes += (int64_t)p->bundle;
    }
    stamp[slot] = ++p->clock;
  }
  if (stats) {
    stats->hits += s.hits;
    stats->misses += s.misses;
    stats->evictions += s.evictions;
    stats->h2d_bytes += s.h2d_bytes;
  }
  if (result != E0_OK) return result;
  int* cw = &p->cur[(size_t)layer * KMAX];
  for (int k = 0; k < K; ++k) cw[k] = ids[k];
  p->ncur[layer] = K;
  return E0_OK;
}

// Queue, after the bundles of pool layers [l0, l1), their tables of the tag's parity
// (one 2-D copy, when any differs from the record) and then `tag` into their ready words
// (one copy), from the tag's half of the pinned snapshots.
e0_status flush_group(e0_slot_pool* p, int l0, int l1, uint32_t tag, cudaStream_t st) {
  if (l1 <= l0) return E0_OK;
  const int E = p->E, half = (int)(tag & 1u);
  bool any = false;
  for (int l = l0; l < l1; ++l) any = any || p->dirty[(size_t)l * 2 + half];
  if (any) {
    int16_t* snap = p->h_tab + ((size_t)half * p->L + l0) * E;
    for (int l = l0; l < l1; ++l)
      for (int e = 0; e < E; ++e) snap[(size_t)(l - l0) * E + e] = (int16_t)p->id_slot[(size_t)l * E + e];
    E0_CHECK_CUDA(cudaMemcpy2DAsync(p->d_slot_of + ((size_t)l0 * 2 + half) * E, sizeof(int16_t) * 2 * E, snap,
                                    sizeof(int16_t) * E, sizeof(int16_t) * E, l1 - l0, cudaMemcpyHostToDevice, st));
    for (int l = l0; l < l1; ++l) p->dirty[(size_t)l * 2 + half] = 0;
  }
  uint32_t* tg = p->h_tag + (size_t)half * p->L;
  for (int l = l0; l < l1; ++l) tg[l] = tag;
  E0_CHECK_CUDA(cudaMemcpyAsync(p->d_ready + l0, tg + l0, sizeof(uint32_t) * (l1 - l0), cudaMemcpyHostToDevice, st));
  return E0_OK;
}

// One staging call: the layers in order, their small copies grouped over runs of
// consecutive pool layers (at most GROUP_LAYERS).  ids_of(i) returns pool layer
// layers[i]'s ids (or nullptr with an error status set); the tag's snapshot half is
// free once the call two tags back has been copied out.
template <class IdsOf>
e0_status stage_call(e0_slot_pool* p, const int32_t* layers, int32_t n, int32_t K, uint32_t tag, cudaStream_t st,
                     e0_stage_stats* stats, IdsOf ids_of) {
  for (int i = 0; i < n; ++i)
    E0_REQUIRE(layers[i] >= 0 && layers[i] < p->L, E0_ERR_INVALID, "e0_stage_slots: layer out of range");
  E0_CHECK_CUDA(cudaEventSynchronize(p->snap_done[tag & 1u]));
  int g0 = 0;  // first index of the current group
  for (int i = 0; i < n; ++i) {
    e0_status err = E0_OK;
    const int32_t* ids = ids_of(i, err);
    if (err != E0_OK) return err;
    e0_status s = stage_bundles(p, layers[i], ids, K, st, stats);
    if (s != E0_OK) return s;
    const bool last = i + 1 == n || layers[i + 1] != layers[i] + 1 || i + 1 - g0 == GROUP_LAYERS;
    if (last) {
      s = flush_group(p, layers[g0], layers[i] + 1, tag, st);
      if (s != E0_OK) return s;
      g0 = i + 1;
    }
  }
  E0_CHECK_CUDA(cudaEventRecord(p->snap_done[tag & 1u], st));
  return E0_OK;
}

}  // namespace

extern "C" e0_status e0_stage_slots_host(e0_slot_pool* p, const int32_t* layers, int32_t n_layers,
                                         const int32_t* ids, int32_t K, uint32_t tag, e0_stream copy_stream,
                                         e0_event after, e0_stage_stats* stats) {
  E0_REQUIRE(p && layers && ids && n_layers >= 0, E0_ERR_INVALID, "e0_stage_slots_host: NULL argument");
  E0_REQUIRE(K >= 1 && K <= KMAX && 2 * K <= p->S, E0_ERR_SHAPE, "e0_stage_slots_host: K out of range");
  const cudaStream_t st = (cudaStream_t)copy_stream;
  if (after) E0_CHECK_CUDA(cudaStreamWaitEvent(st, (cudaEvent_t)after, 0));
  return stage_call(p, layers, n_layers, K, tag, st, stats,
                    [&](int i, e0_status&) { return ids + (size_t)i * K; });
}

extern "C" e0_status e0_stage_slots(e0_slot_pool* p, const int32_t* layers, int32_t n_layers, const int32_t* next_ids,
                                    const int32_t* rows, int32_t K, uint32_t tag, e0_stream copy_stream,
                                    e0_event after, e0_stage_stats* stats) {
  E0_REQUIRE(p && layers && rows && next_ids && n_layers >= 0, E0_ERR_INVALID, "e0_stage_slots: NULL argument");
  E0_REQUIRE(K >= 1 && K <= KMAX && 2 * K <= p->S, E0_ERR_SHAPE, "e0_stage_slots: K out of range");
  int nrows = 0;
  for (int i = 0; i < n_layers; ++i) {
    E0_REQUIRE(rows[i] >= 0 && rows[i] < 65536, E0_ERR_INVALID, "e0_stage_slots: row out of range");
    nrows = std::max(nrows, rows[i] + 1);
  }
  if (n_layers == 0) return E0_OK;
  const size_t need = (size_t)nrows * K;
  if (need > p->ids_cap) {
    // (every earlier call waited for its own landing copy, so the old buffer is idle)
    if (p->h_ids) cudaFreeHost(p->h_ids);
    p->h_ids = nullptr;
    p->ids_cap = 0;
    E0_CHECK_CUDA(cudaHostAlloc(&p->h_ids, need * sizeof(int32_t), cudaHostAllocDefault));
    p->ids_cap = need;
  }
  const cudaStream_t st = (cudaStream_t)copy_stream;
  if (after) E0_CHECK_CUDA(cudaStreamWaitEvent(st, (cudaEvent_t)after, 0));
  E0_CHECK_CUDA(cudaMemcpyAsync(p->h_ids, next_ids, need * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  E0_CHECK_CUDA(cudaEventRecord(p->ids_done, st));
  E0_CHECK_CUDA(cudaEventSynchronize(p->ids_done));
  return stage_call(p, layers, n_layers, K, tag, st, stats,
                    [&](int i, e0_status&) { return p->h_ids + (size_t)rows[i] * K; });
}

// ------------------------------------------------------------------ commit box
struct e0_commit_box {
  int L = 0;
  uint32_t* host = nullptr;  // pinned, mapped: [2][L][KMAX + 1]
  uint32_t* dev = nullptr;   // the same memory as the device addresses it
};

extern "C" void e0_commit_box_destroy(e0_commit_box* b) {
  if (!b) return;
  if (b->host) cudaFreeHost(b->host);
  delete b;
}

extern "C" e0_status e0_commit_box_create(e0_commit_box** out, int32_t layers) {
  E0_REQUIRE(out && layers >= 1 && layers <= LMAX, E0_ERR_INVALID, "e0_commit_box_create: need 1..48 layers");
  *out = nullptr;
  e0_commit_box* b = new e0_commit_box;
  b->L = layers;
  const size_t words = (size_t)2 * layers * (KMAX + 1);
  cudaError_t e = cudaHostAlloc(&b->host, words * sizeof(uint32_t), cudaHostAllocMapped);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&b->dev), b->host, 0);
  if (e != cudaSuccess) {
    e0_commit_box_destroy(b);
    return e0::cuda_fail(e, "e0_commit_box_create");
  }
  for (size_t i = 0; i < words; ++i) b->host[i] = 0xFFFFFFFFu;  // no token committed yet
  *out = b;
  return E0_OK;
}

extern "C" void* e0_commit_box_device(const e0_commit_box* b) { return b ? b->dev : nullptr; }

extern "C" e0_status e0_stage_slots_committed(e0_slot_pool* p, const e0_commit_box* box, const int32_t* layers,
                                              const int32_t* rows, int32_t n_layers, int32_t K, uint32_t tag,
                                              e0_stream copy_stream, uint64_t timeout_ns, e0_stage_stats* stats) {
  E0_REQUIRE(p && box && layers && rows && n_layers >= 0, E0_ERR_INVALID, "e0_stage_slots_committed: NULL argument");
  E0_REQUIRE(K >= 1 && K <= KMAX && 2 * K <= p->S, E0_ERR_SHAPE, "e0_stage_slots_committed: K out of range");
  for (int i = 0; i < n_layers; ++i)
    E0_REQUIRE(rows[i] >= 0 && rows[i] < box->L, E0_ERR_INVALID, "e0_stage_slots_committed: row out of range");
  const cudaStream_t st = (cudaStream_t)copy_stream;
  const auto t0 = std::chrono::steady_clock::now();
  int32_t ids[KMAX];
  return stage_call(p, layers, n_layers, K, tag, st, stats, [&](int i, e0_status& err) -> const int32_t* {
    const volatile uint32_t* row = box->host + ((size_t)(tag & 1u) * box->L + rows[i]) * (KMAX + 1);
    // the launch writes the ids, then (after a system-scope fence) the tag
    for (uint32_t it = 0; row[0] != tag; ++it) {
      if ((it & 255u) == 0 &&
          (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now() - t0)
                  .count() > timeout_ns) {
        err = e0::fail(E0_ERR_TIMEOUT, "e0_stage_slots_committed: the launch did not commit this layer in time");
        return nullptr;
      }
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    for (int k = 0; k < K; ++k) ids[k] = (int32_t)row[1 + k];
    return ids;
  });
}
