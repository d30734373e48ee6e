// Host side of libe0: argument checks, the per-CTA work planner and the C ABI
// entry points that launch the streaming engine (e0_engine.cu).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "e0_engine.cuh"

namespace e0 {
static thread_local std::string g_err;
void set_error(const std::string& msg) { g_err = msg; }
e0_status fail(e0_status code, const std::string& msg) {
  g_err = msg;
  return code;
}
e0_status cuda_fail(cudaError_t err, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(err);
  return E0_ERR_CUDA;
}
}  // namespace e0

namespace e0eng {
cudaError_t launch_engine(const EngineParams& P, cudaStream_t stream);
int max_ctas_per_sm(int d);
}  // namespace e0eng

using namespace e0eng;

extern "C" const char* e0_last_error(void) { return e0::g_err.c_str(); }
extern "C" const char* e0_version(void) { return "libe0 0.1 (sm_103a)"; }

namespace {

constexpr uint64_t DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s per bounded wait
thread_local uint64_t* g_trace = nullptr;                // diagnostics buffer for the next launches

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

e0_status device_ctas(int d, int* ncta) {
  int dev = 0;
  E0_CHECK_CUDA(cudaGetDevice(&dev));
  int sms = 0;
  E0_CHECK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  int coop = 0;
  E0_CHECK_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
  E0_REQUIRE(coop, E0_ERR_UNSUPPORTED, "device does not support cooperative launches");
  const int per = max_ctas_per_sm(d);
  E0_REQUIRE(per >= 1, E0_ERR_UNSUPPORTED, "engine kernel cannot be resident (shared memory)");
  *ncta = std::min(sms, MAX_CTAS);
  return E0_OK;
}

}  // namespace

// Shared with the other translation units (declared in e0_common.cuh).
e0_status e0::check_dims(const e0_dims* dm) {
  E0_REQUIRE(dm, E0_ERR_INVALID, "dims is NULL");
  E0_REQUIRE(dm->d == 256 || dm->d == 512 || dm->d == 1024 || dm->d == 2048, E0_ERR_SHAPE,
             "d must be 256, 512, 1024 or 2048");
  E0_REQUIRE(dm->E >= 8 && dm->E <= EMAX && dm->E % 8 == 0, E0_ERR_SHAPE, "E must be a multiple of 8 in [8, 1024]");
  E0_REQUIRE(dm->F >= 64 && dm->F % 64 == 0 && dm->F <= 8192, E0_ERR_SHAPE, "F must be a multiple of 64");
  E0_REQUIRE(dm->K >= 1 && dm->K <= KMAX && dm->K <= dm->E, E0_ERR_SHAPE, "K must be in [1, min(16, E)]");
  return e0::check_route(dm);
}

e0_status e0::check_route(const e0_dims* dm) {
  if (dm->route == E0_ROUTE_SIGMOID_GROUP) {
    E0_REQUIRE(dm->n_group >= 1 && dm->n_group <= 32 && dm->E % dm->n_group == 0 && dm->E / dm->n_group >= 2,
               E0_ERR_SHAPE, "sigmoid-group routing: n_group must divide E into groups of >= 2, n_group <= 32");
    E0_REQUIRE(dm->topk_group >= 1 && dm->topk_group <= dm->n_group &&
                   dm->topk_group * (dm->E / dm->n_group) >= dm->K,
               E0_ERR_SHAPE, "sigmoid-group routing: topk_group in [1, n_group] with topk_group * E/n_group >= K");
    E0_REQUIRE(std::isfinite(dm->route_scale), E0_ERR_INVALID, "sigmoid-group routing: route_scale must be finite");
  } else {
    E0_REQUIRE(dm->route == E0_ROUTE_SOFTMAX_TOPK, E0_ERR_UNSUPPORTED, "unknown routing family");
  }
  return E0_OK;
}

namespace {
using e0::check_dims;

// ------------------------------------------------------------------ planner
struct PlanSpec {
  int d = 0, E = 0, F = 0, K = 0;
  bool routed = false, shared = false, lora = false, lora_ab = false, head = false, lres = false, router = false;
  int lout = 0, lr = 0, H = 0;
  bool operator<(const PlanSpec& o) const {
    return std::memcmp(this, &o, sizeof(PlanSpec)) < 0;
  }
};

struct Granule {
  uint8_t type;
  int row;
  int rows;
  double cost;
};

// Relative cost of a streamed byte: int4 rows need about twice the ALU work per
// byte of bf16 rows.
constexpr double W_INT4 = 1.25;
constexpr double W_BF16 = 1.0;
// LoRA base rows measure slower per byte than expert slabs (each CTA also runs their B
// rows after waiting for v)
constexpr double W_QROWS = 1.25;
// Fixed cost of one unit on a CTA, in the same units (bf16 bytes): the fragment load
// of x, the first stage's wait and the barriers between phases take about as long as
// streaming 32 KB.  It steers the planner away from giving one CTA several small units.
constexpr double UNIT_COST = 32768.0;

// Water-fill granules over CTAs [c0, c1): the level T at which the CTAs below it take
// exactly the granules and one unit cost each, sum_c max(0, T - load[c]) = total +
// UNIT_COST * n_below (CTAs already above T, e.g. ones with an expert slab heavier than
// the mean, get nothing more); granules are assigned in order with cumulative
// capacity, so rounding spreads evenly, and contiguous granules of one type merge.
void waterfill(const PlanSpec& s, const std::vector<Granule>& gs, int c0, int c1, std::vector<double>& load,
               std::vector<std::vector<Unit>>& lists) {
  if (gs.empty() || c1 <= c0) return;
  double gtotal = 0.0;
  bool rows_with_b = false;  // LoRA rows bring a second unit (their B rows) to every CTA
  for (auto& g : gs) {
    gtotal += g.cost;
    rows_with_b = rows_with_b || (g.type == U_QROWS && s.lr > 0);
  }
  const double per_cta = UNIT_COST * (rows_with_b ? 2.0 : 1.0);
  double level = 0.0;
  {
    std::vector<double> sorted(load.begin() + c0, load.begin() + c1);
    std::sort(sorted.begin(), sorted.end());
    const int n = (int)sorted.size();
    double below = 0.0;  // sum of the loads of the CTAs under the level
    for (int c = 0; c < n; ++c) {
      below += sorted[c];
      const double t = (gtotal + below) / (c + 1) + per_cta;  // level if CTAs 0..c take everything
      if (c + 1 == n || t <= sorted[c + 1]) {
        level = t;
        break;
      }
    }
  }
  // place granule gr on CTA c (merging with a contiguous unit of its type); its cost
  auto place = [&](int c, const Granule& gr, bool dry) -> double {
    auto& L = lists[c];
    Unit* into = nullptr;
    for (auto& u : L) {
      if (u.type == gr.type && u.r1 == gr.row) {
        // unit size limits: head buffers; the B slice of a LoRA row unit fits one stage
        const int limit = (gr.type == U_HEAD || gr.type == U_LRES) ? HEAD_ROWS
                          : gr.type == U_QROWS && s.lr > 0 ? (STAGE_BYTES / (2 * s.lr)) / 16 * 16
                          : gr.type == U_LORA_A            ? 4
                                                           : 65535;
        if ((int)u.r1 - (int)u.r0 + gr.rows <= limit) into = &u;
        break;
      }
    }
    double cost = gr.cost + (into ? 0.0 : UNIT_COST);
    bool new_b = false;
    if (gr.type == U_QROWS && s.lr > 0) {
      new_b = true;
      for (auto& u : L)
        if (u.type == U_LORA_B && u.r1 == gr.row &&
            (int)u.r1 - (int)u.r0 + gr.rows <= (STAGE_BYTES / (2 * s.lr)) / 16 * 16) {
          if (!dry) u.r1 = (uint16_t)(gr.row + gr.rows);
          new_b = false;
          break;
        }
      if (new_b) cost += UNIT_COST;  // waits for v: one more unit's worth of latency
    }
    if (dry) return cost;
    if (into)
      into->r1 = (uint16_t)(gr.row + gr.rows);
    else
      L.push_back(Unit{gr.type, 0, (uint16_t)gr.row, (uint16_t)(gr.row + gr.rows), 0});
    if (new_b) L.push_back(Unit{U_LORA_B, 0, (uint16_t)gr.row, (uint16_t)(gr.row + gr.rows), 0});
    load[c] += cost;
    return cost;
  };
  double cum_cap = 0.0, cum_assigned = 0.0;
  size_t g = 0;
  for (int c = c0; c < c1 && g < gs.size(); ++c) {
    cum_cap += std::max(0.0, level - load[c]);
    while (g < gs.size()) {
      const double cost = place(c, gs[g], true);
      if (cum_assigned + 0.5 * cost > cum_cap) break;
      cum_assigned += place(c, gs[g], false);
      ++g;
    }
  }
  // what rounding left over goes, one granule at a time, to the least loaded CTA
  for (; g < gs.size(); ++g) {
    int best = c0;
    for (int c = c0 + 1; c < c1; ++c)
      if (load[c] < load[best]) best = c;
    place(best, gs[g], false);
  }
}

// The work plan of one layer kind: expert slabs round robin, then the divisible work.
// With `defer` (stack layers with a head) and room beside the expert CTAs, the layer's
// LoRA work goes one unit per CTA to the next CTAs and the prerouter's work (HEAD, LRES:
// needed only by the next token) in contiguous runs to CTAs of its own, [n_crit, ncta),
// which do not hold up the layer: defer[c] = 1 there, *n_crit_out = n_crit.  Otherwise
// the divisible work is water-filled by cost.  With crit_limit > 0 every unit goes to
// CTAs [0, crit_limit) (the router rows of an own-gate layer; the layers after a head
// layer, whose CTAs [crit_limit, ncta) hold the deferred prerouter work).
e0_status build_plan(const PlanSpec& s, int ncta, Unit* units, uint8_t* counts, uint8_t* defer = nullptr,
                     int* n_crit_out = nullptr, int crit_limit = 0) {
  std::vector<std::vector<Unit>> lists(ncta);
  std::vector<double> load(ncta, 0.0);
  const int d = s.d;
  const double c_exp = W_INT4 * (64.0 * q4_row_bytes(d) + 20.0 * d) + UNIT_COST;
  const int limit = crit_limit > 0 ? std::min(crit_limit, ncta) : ncta;
  int n_slabs = 0;
  // 1. expert slabs, round robin
  if (s.routed || s.shared) {
    int idx = 0;
    const int kmax = s.routed ? s.K : 0;
    for (int k = 0; k <= kmax; ++k) {
      if (k < kmax || s.shared) {
        if (k == kmax && !s.shared) break;
        for (int sl = 0; sl < s.F / 32; ++sl) {
          const int c = idx++ % limit;
          lists[c].push_back(Unit{U_EXPERT, (uint8_t)(k < kmax ? k : s.K), (uint16_t)sl, (uint16_t)(sl + 1), 0});
          load[c] += c_exp;
        }
      }
    }
    n_slabs = idx;
  }
  // 2. split (layers with a head, when there is room): the layer's own LoRA work on CTAs
  //    beside the expert ones: 64 LoRA base rows (one consumer stage group) per CTA, and
  //    a few CTAs that each compute all of v = A x and the B v of a slice of the rows (no
  //    CTA waits for another's v); the prerouter's work (HEAD, LRES: needed only by the
  //    next token) on the rest
  const int qstage = q4_rows_per_stage(d);
  const bool has_def = s.lres || s.head;
  // LoRA base rows per CTA in the split plan: whole stages, about as many bytes as an
  // expert slab, so that those CTAs finish with the expert CTAs and as many CTAs as
  // possible are left to the prerouter (whose CTAs must keep pace with the layers: the
  // launch ends only when the last head is done)
  const int slab_bytes = 64 * q4_row_bytes(d) + 20 * d;
  const int q_rows = std::max(4 * qstage, slab_bytes / q4_row_bytes(d) / qstage * qstage);
  const int n_q = s.lora ? (s.lout + q_rows - 1) / q_rows : 0;
  // B slices of one stage each: rows in multiples of 16 with lr * rows * 2 <= STAGE_BYTES
  const int b_rows = s.lora_ab && s.lr > 0 ? std::max(16, (STAGE_BYTES / (2 * s.lr)) / 16 * 16) : 0;
  const int n_ab = s.lora_ab && s.lr > 0 ? std::max(1, (s.lout + b_rows - 1) / b_rows) : 0;
  const int n_own = n_q + n_ab;
  const bool split = defer && has_def && !s.router && n_slabs > 0 && n_slabs + n_own <= ncta - 8;
  const int n_crit = split ? n_slabs + n_own : ncta;
  // 3. divisible work as granules: the layer's own (crit) and the prerouter's (def)
  std::vector<Granule> crit, def;
  // the LoRA down projection first: the CTAs that own LoRA base rows wait for its v
  // (its cost adds the latency of publishing v), in slices of 4 ranks so that v is
  // published early
  if (s.lora_ab)
    for (int q = 0; q < s.lr; q += 4)
      crit.push_back({U_LORA_A, q, std::min(4, s.lr - q), W_BF16 * 2.0 * d * std::min(4, s.lr - q) + 4.0 * UNIT_COST});
  const int qg = split ? 4 * qstage : qstage;
  if (s.lora)
    for (int r = 0; r < s.lout; r += qg) {
      const int nr = std::min(qg, s.lout - r);
      crit.push_back({U_QROWS, r, nr, W_QROWS * nr * (double)q4_row_bytes(d) + W_BF16 * nr * 2.0 * s.lr});
    }
  if (s.router)
    for (int e = 0; e < s.E; e += 4) crit.push_back({U_ROUTER, e, std::min(4, s.E - e), W_BF16 * 4.0 * 2.0 * d});
  if (s.lres)
    for (int e = 0; e < s.E; e += 8) def.push_back({U_LRES, e, 8, W_BF16 * 8.0 * 2.0 * d});
  if (s.head)
    for (int i = 0; i < s.H; i += 8)
      def.push_back({U_HEAD, i, 8, W_BF16 * 8.0 * (2.0 * d + 2.0 * s.E + 2.0 * (1 + 2 * s.K))});
  if (split) {
    for (int i = 0; i < n_ab; ++i) {  // all ranks of v, then the B rows of an even slice
      auto& L = lists[n_slabs + i];
      const int r0 = (int)((long long)s.lout * i / n_ab) / 16 * 16;
      const int r1 = i + 1 == n_ab ? s.lout : (int)((long long)s.lout * (i + 1) / n_ab) / 16 * 16;
      L.push_back(Unit{U_LORA_A, 0, 0, (uint16_t)s.lr, UF_LOCAL_V});
      L.push_back(Unit{U_LORA_B, 0, (uint16_t)r0, (uint16_t)r1, 0});
    }
    const int q_st = (s.lout + qstage - 1) / qstage;  // stages of LoRA base rows, spread evenly
    for (int i = 0; i < n_q; ++i) {
      const int r0 = (int)((long long)q_st * i / n_q) * qstage;
      const int r1 = std::min(s.lout, (int)((long long)q_st * (i + 1) / n_q) * qstage);
      lists[n_slabs + n_ab + i].push_back(Unit{U_QROWS, 0, (uint16_t)r0, (uint16_t)r1, 0});
    }
    // the prerouter's rows in contiguous runs, LRES on the first CTAs of the pool and
    // HEAD on the rest, the CTA counts in proportion to the bytes (a head unit has three
    // dependent phases and a high fixed cost: one run per CTA, split only at HEAD_ROWS)
    const int n_def = ncta - n_crit;
    double c_l = 0.0, c_h = 0.0;
    for (auto& g : def) (g.type == U_LRES ? c_l : c_h) += g.cost;
    int n_l = c_l > 0.0 ? (int)std::lround(n_def * c_l / (c_l + c_h)) : 0;
    if (c_l > 0.0) n_l = std::max(1, std::min(n_l, n_def - (c_h > 0.0 ? 1 : 0)));
    const int n_h = n_def - n_l;
    auto spread = [&](uint8_t type, int rows, int c0, int nc) {
      if (rows <= 0 || nc <= 0) return;
      const int gran = 8, ng = (rows + gran - 1) / gran;
      for (int i = 0; i < nc; ++i) {
        const int g0 = (int)((long long)ng * i / nc), g1 = (int)((long long)ng * (i + 1) / nc);
        for (int r = g0 * gran; r < std::min(rows, g1 * gran); r += HEAD_ROWS)
          lists[c0 + i].push_back(Unit{type, 0, (uint16_t)r, (uint16_t)std::min({rows, g1 * gran, r + HEAD_ROWS}), 0});
      }
    };
    spread(U_LRES, s.lres ? s.E : 0, n_crit, n_l);
    spread(U_HEAD, s.head ? s.H : 0, n_crit + n_l, n_h);
  } else {
    std::vector<Granule> all(crit);
    all.insert(all.end(), def.begin(), def.end());
    waterfill(s, all, 0, limit, load, lists);
  }
  if (defer)
    for (int c = 0; c < ncta; ++c) defer[c] = c >= n_crit ? 1 : 0;
  if (n_crit_out) *n_crit_out = n_crit;
  // 4. order: id-independent work first, experts last.  U_LORA_A must precede U_LORA_B
  //    on a CTA that has both (B waits for the v that A publishes); B goes late so that
  //    v is normally there by the time it is needed.
  auto rank = [](uint8_t t) {
    switch (t) {
      case U_ROUTER: return 0;
      case U_LORA_A: return 1;
      case U_QROWS: return 2;
      case U_LRES: return 3;
      case U_HEAD: return 4;
      case U_LORA_B: return 5;
      default: return 6;
    }
  };
  for (int c = 0; c < ncta; ++c) {
    auto& L = lists[c];
    std::stable_sort(L.begin(), L.end(), [&](const Unit& a, const Unit& b) { return rank(a.type) < rank(b.type); });
    E0_REQUIRE((int)L.size() <= MAXU, E0_ERR_UNSUPPORTED, "work plan needs more units per CTA than supported");
    counts[c] = (uint8_t)L.size();
    for (size_t i = 0; i < L.size(); ++i) units[(size_t)c * MAXU + i] = L[i];
    for (size_t i = L.size(); i < (size_t)MAXU; ++i) units[(size_t)c * MAXU + i] = Unit{U_NONE, 0, 0, 0, 0};
  }
  return E0_OK;
}

struct CachedPlan {
  std::vector<Unit> units;
  std::vector<uint8_t> counts;
};
std::mutex g_plan_mu;
std::map<std::pair<PlanSpec, int>, CachedPlan> g_plans;

e0_status get_plan(const PlanSpec& s, int ncta, const CachedPlan** out) {
  std::lock_guard<std::mutex> lk(g_plan_mu);
  auto key = std::make_pair(s, ncta);
  auto it = g_plans.find(key);
  if (it == g_plans.end()) {
    CachedPlan cp;
    cp.units.assign((size_t)ncta * MAXU, Unit{});
    cp.counts.assign(ncta, 0);
    e0_status st = build_plan(s, ncta, cp.units.data(), cp.counts.data());
    if (st != E0_OK) return st;
    it = g_plans.emplace(key, std::move(cp)).first;
  }
  *out = &it->second;
  return E0_OK;
}

// ------------------------------------------------------------------ descriptors
e0_status fill_experts(const e0_experts* ex, const e0_dims* dm, bool routed, LayerDesc* L) {
  E0_REQUIRE(ex->gate_up.q && ex->gate_up.scale && ex->gate_up.bias && ex->down.q && ex->down.scale && ex->down.bias,
             E0_ERR_INVALID, "expert stack has a NULL tensor");
  E0_REQUIRE(al16(ex->gate_up.q) && al16(ex->gate_up.scale) && al16(ex->gate_up.bias) && al16(ex->down.q) &&
                 al16(ex->down.scale) && al16(ex->down.bias),
             E0_ERR_INVALID, "expert tensors must be 16-byte aligned");
  E0_REQUIRE(ex->n >= 1, E0_ERR_INVALID, "expert stack needs n >= 1");
  if (routed) {
    L->gu_q = ex->gate_up.q; L->gu_s = ex->gate_up.scale; L->gu_b = ex->gate_up.bias;
    L->dn_q = ex->down.q; L->dn_s = ex->down.scale; L->dn_b = ex->down.bias;
    L->slot_of = ex->slot_of;
    L->ready = ex->ready;
    L->n_routed = ex->n;
    E0_REQUIRE(ex->stride >= 0 && ex->stride % 16 == 0, E0_ERR_INVALID, "expert stride must be a multiple of 16");
    L->ex_stride = ex->stride;
    E0_REQUIRE(ex->slot_of || ex->n >= dm->E, E0_ERR_INVALID, "routed stack without slot_of must hold all E experts");
  } else {
    L->sgu_q = ex->gate_up.q; L->sgu_s = ex->gate_up.scale; L->sgu_b = ex->gate_up.bias;
    L->sdn_q = ex->down.q; L->sdn_s = ex->down.scale; L->sdn_b = ex->down.bias;
    L->has_shared = 1;
  }
  return E0_OK;
}

e0_status fill_lora(const e0_qlora* lo, int in, LayerDesc* L, bool* has_ab) {
  E0_REQUIRE(lo->w.q && lo->w.scale && lo->w.bias, E0_ERR_INVALID, "LoRA base W has a NULL tensor");
  E0_REQUIRE(al16(lo->w.q) && al16(lo->w.scale) && al16(lo->w.bias), E0_ERR_INVALID, "LoRA W must be 16-byte aligned");
  E0_REQUIRE(lo->out >= 16 && lo->out % 16 == 0 && lo->out <= OUTMAX, E0_ERR_SHAPE,
             "LoRA out must be a multiple of 16 in [16, 4096]");
  E0_REQUIRE(lo->r >= 0 && lo->r <= RANKS_MAX, E0_ERR_SHAPE, "LoRA rank must be in [0, 64]");
  L->lw_q = lo->w.q; L->lw_s = lo->w.scale; L->lw_b = lo->w.bias;
  L->lout = lo->out;
  L->has_lora = 1;
  *has_ab = lo->r > 0 && lo->a && lo->bt;
  if (*has_ab) {
    E0_REQUIRE(al16(lo->a) && al16(lo->bt), E0_ERR_INVALID, "LoRA A/Bt must be 16-byte aligned");
    L->la = lo->a; L->lbt = lo->bt; L->lr = lo->r;
    L->lscale = lo->alpha / (float)lo->r;
  }
  (void)in;
  return E0_OK;
}

e0_status fill_head(const e0_prerouter* hd, const e0_dims* dm, LayerDesc* L) {
  E0_REQUIRE(hd->lres && al16(hd->lres), E0_ERR_INVALID, "prerouter lres must be non-NULL and 16-byte aligned");
  E0_REQUIRE(hd->H >= 0 && hd->H % 8 == 0 && hd->H <= 8192, E0_ERR_SHAPE, "prerouter H must be a multiple of 8");
  L->has_head = 1;
  L->H = hd->H;
  L->lres = hd->lres;
  L->b2 = hd->b2;
  if (hd->H > 0) {
    E0_REQUIRE(hd->w1h && hd->w1c_t && hd->w1p_t && hd->w2t, E0_ERR_INVALID, "prerouter fc1/fc2 tensor is NULL");
    E0_REQUIRE(al16(hd->w1h) && al16(hd->w1c_t) && al16(hd->w1p_t) && al16(hd->w2t) && (!hd->b1 || al16(hd->b1)),
               E0_ERR_INVALID, "prerouter tensors must be 16-byte aligned");
    L->w1h = hd->w1h; L->w1c_t = hd->w1c_t; L->w1p_t = hd->w1p_t; L->b1 = hd->b1; L->w2t = hd->w2t;
  }
  (void)dm;
  return E0_OK;
}

void base_params(EngineParams& P, int d, int E, int F, int K, int L, int ncta, int mode) {
  std::memset(&P, 0, sizeof(P));
  P.d = d; P.E = E; P.F = F; P.K = K; P.L = L; P.ncta = ncta; P.mode = mode;
  P.norm = 1; P.out_dim = d; P.kinds = 1;
  for (int k = 0; k < KINDS_MAX; ++k) P.n_arrive[k] = ncta;
  P.timeout_ns = DEFAULT_TIMEOUT_NS;
  P.wl = ws_layout(E, L);
  P.trace = g_trace;
}

// The routing family of the call (dims are checked already).
void set_route(EngineParams& P, const e0_dims* dm) {
  P.route = dm->route;
  P.n_group = dm->n_group;
  P.topk_group = dm->topk_group;
  P.route_scale = dm->route_scale;
  P.score_bias = dm->score_bias;
}

void set_inline_plan(EngineParams& P, const CachedPlan& cp) {
  std::memcpy(P.inline_plan, cp.units.data(), sizeof(Unit) * cp.units.size());
  std::memcpy(P.inline_n, cp.counts.data(), cp.counts.size());
}

}  // namespace

// ====================================================================== C ABI
extern "C" size_t e0_workspace_size(const e0_dims* dims, int32_t layers) {
  if (!dims || layers < 1) return 0;
  return ws_layout(std::max(dims->E, 8), layers).total;
}

extern "C" e0_status e0_workspace_reset(void* ws, size_t bytes, e0_stream stream) {
  E0_REQUIRE(ws && bytes >= sizeof(WsHeader), E0_ERR_INVALID, "e0_workspace_reset: bad workspace");
  E0_CHECK_CUDA(cudaMemsetAsync(ws, 0, bytes, (cudaStream_t)stream));
  return E0_OK;
}

extern "C" e0_status e0_get_device_status(const void* ws, uint32_t* status_out, e0_stream stream) {
  E0_REQUIRE(ws && status_out, E0_ERR_INVALID, "e0_get_device_status: NULL argument");
  E0_CHECK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  WsHeader h;
  E0_CHECK_CUDA(cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  *status_out = h.status;
  return E0_OK;
}

extern "C" e0_status e0_debug_plan(int32_t d, int32_t E, int32_t F, int32_t K, int32_t H, int32_t lr, int32_t ncta,
                                   int32_t kind, void* units_out, uint8_t* counts_out, uint8_t* defer_out) {
  E0_REQUIRE(units_out && counts_out && defer_out, E0_ERR_INVALID, "e0_debug_plan: NULL argument");
  E0_REQUIRE(ncta >= 1 && ncta <= MAX_CTAS && kind >= 0 && kind <= 3, E0_ERR_INVALID, "e0_debug_plan: ncta or kind");
  E0_REQUIRE(d > 0 && d % 256 == 0 && E >= 1 && F % 32 == 0 && K >= 1 && K <= E && lr >= 0 && lr <= RANKS_MAX &&
                 H >= 0 && H % 8 == 0,
             E0_ERR_SHAPE, "e0_debug_plan: shape");
  PlanSpec ps;
  ps.d = d; ps.E = E; ps.F = F; ps.K = K;
  ps.routed = ps.shared = ps.lora = true;
  ps.lora_ab = lr > 0; ps.lr = lr; ps.lout = d;
  if (kind == 0) { ps.head = H > 0; ps.lres = true; ps.H = H; }
  std::memset(units_out, 0, sizeof(Unit) * (size_t)ncta * MAXU);
  std::memset(defer_out, 0, (size_t)ncta);
  Unit* u = static_cast<Unit*>(units_out);
  if (kind < 2) return build_plan(ps, ncta, u, counts_out, kind == 0 ? defer_out : nullptr);
  std::vector<Unit> tmp((size_t)ncta * MAXU);
  std::vector<uint8_t> tc(ncta), td(ncta);
  int n_crit = ncta;
  PlanSpec hs = ps;
  hs.head = H > 0; hs.lres = true; hs.H = H;
  e0_status st = build_plan(hs, ncta, tmp.data(), tc.data(), td.data(), &n_crit);
  if (st) return st;
  if (kind == 3) return build_plan(ps, ncta, u, counts_out, nullptr, nullptr, n_crit);
  PlanSpec rs;
  rs.d = d; rs.E = E; rs.F = F; rs.K = K; rs.router = true;
  return build_plan(rs, ncta, u, counts_out, nullptr, nullptr, n_crit);
}

extern "C" e0_status e0_debug_trace(uint64_t* buf, size_t bytes) {
  E0_REQUIRE(!buf || bytes >= 8, E0_ERR_INVALID, "e0_debug_trace: buffer too small");
  g_trace = buf;
  return E0_OK;
}

extern "C" e0_status e0_debug_inject_stall(void* ws, uint64_t limit_ns, e0_stream stream) {
  E0_REQUIRE(ws, E0_ERR_INVALID, "e0_debug_inject_stall: NULL workspace");
  E0_CHECK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  E0_CHECK_CUDA(cudaMemcpy(reinterpret_cast<uint8_t*>(ws) + offsetof(WsHeader, stall_ns), &limit_ns,
                           sizeof(limit_ns), cudaMemcpyHostToDevice));
  return E0_OK;
}

static e0_status check_ws(const e0_dims* dm, int L, void* ws, size_t bytes) {
  E0_REQUIRE(ws && al16(ws), E0_ERR_INVALID, "workspace must be non-NULL and 16-byte aligned");
  E0_REQUIRE(bytes >= ws_layout(dm->E, L).total, E0_ERR_NOMEM, "workspace smaller than e0_workspace_size()");
  return E0_OK;
}

extern "C" e0_status e0_moe_decode_layer(const e0_dims* dims, const e0_experts* routed, const e0_experts* shared,
                                         const e0_qlora* lora, const e0_prerouter* head, const uint16_t* h_in,
                                         const int32_t* ids, const float* logits, const int32_t* ids_prev,
                                         int32_t T, uint16_t* h_out, float* delta_f32, float* next_logits,
                                         int32_t* next_ids, float* next_weights, void* workspace,
                                         size_t workspace_bytes, e0_stream stream) {
  e0_status st = check_dims(dims);
  if (st) return st;
  E0_REQUIRE(routed && h_in && ids && logits && h_out, E0_ERR_INVALID, "e0_moe_decode_layer: NULL required argument");
  E0_REQUIRE(T >= 0, E0_ERR_INVALID, "T must be >= 0");
  if (T == 0) return E0_OK;
  if (T > 1) {
    // several tokens: each weight read once for all of them (grouped tensor-core experts,
    // multi-token head)
    E0_REQUIRE(T <= 16, E0_ERR_SHAPE, "e0_moe_decode_layer: T must be <= 16");
    const bool has_head = head && head->lres;
    E0_REQUIRE(!has_head || next_logits || next_ids, E0_ERR_INVALID, "a head needs next_logits or next_ids");
    const int lora_out = lora && lora->w.q ? lora->out : 0;
    const int H = has_head ? head->H : 0;
    E0_REQUIRE(workspace && al16(workspace) && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
               E0_ERR_INVALID, "workspace must be 256-byte aligned");
    E0_REQUIRE(workspace_bytes >= e0_decode_workspace_size(dims, T, lora_out, H), E0_ERR_NOMEM,
               "workspace smaller than e0_decode_workspace_size(dims, T, lora_out, H)");
    const size_t pf = (e0_prefill_workspace_size(dims, T, lora_out) + 255) & ~size_t(255);
    st = e0pf_grouped_layer(dims, routed, shared, lora, h_in, logits, ids, T, h_out, delta_f32, nullptr, nullptr,
                            workspace, pf, stream);
    if (st) return st;
    if (!has_head) return E0_OK;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return e0mt_head(head, dims, h_in, ids, ids_prev, T, nullptr, next_logits, next_ids, next_weights, ws + pf,
                     workspace_bytes - pf, reinterpret_cast<uint32_t*>(ws + 4), stream);
  }
  st = check_ws(dims, 1, workspace, workspace_bytes);
  if (st) return st;
  E0_REQUIRE(al16(h_in) && al16(h_out) && (!delta_f32 || al16(delta_f32)), E0_ERR_INVALID,
             "activation buffers must be 16-byte aligned");
  int ncta;
  st = device_ctas(dims->d, &ncta);
  if (st) return st;

  static thread_local EngineParams P;
  base_params(P, dims->d, dims->E, dims->F, dims->K, 1, ncta, MODE_LAYER);
  set_route(P, dims);
  LayerDesc& L = P.inline_layer;
  PlanSpec ps;
  ps.d = dims->d; ps.E = dims->E; ps.F = dims->F; ps.K = dims->K;
  st = fill_experts(routed, dims, true, &L);
  if (st) return st;
  ps.routed = true;
  if (shared && shared->n > 0) {
    st = fill_experts(shared, dims, false, &L);
    if (st) return st;
    ps.shared = true;
  }
  if (lora && lora->w.q) {
    bool ab = false;
    st = fill_lora(lora, dims->d, &L, &ab);
    if (st) return st;
    E0_REQUIRE(lora->out == dims->d, E0_ERR_SHAPE, "in a layer-step the LoRA linear must be d x d");
    ps.lora = true; ps.lora_ab = ab; ps.lout = lora->out; ps.lr = ab ? lora->r : 0;
  }
  if (head && head->lres) {
    st = fill_head(head, dims, &L);
    if (st) return st;
    ps.head = head->H > 0; ps.lres = true; ps.H = head->H;
    E0_REQUIRE(next_logits || next_ids, E0_ERR_INVALID, "a head needs next_logits or next_ids");
  }
  const CachedPlan* cp;
  st = get_plan(ps, ncta, &cp);
  if (st) return st;
  set_inline_plan(P, *cp);
  P.kinds = 1;
  const int d = dims->d, E = dims->E, K = dims->K;
  for (int t = 0; t < T; ++t) {
    P.h_in = h_in + (size_t)t * d;
    P.ids_in = ids + (size_t)t * K;
    P.logits_in = logits + (size_t)t * E;
    P.ids_prev_in = ids_prev ? ids_prev + (size_t)t * K : nullptr;
    P.h_out = h_out + (size_t)t * d;
    P.delta_out = delta_f32 ? delta_f32 + (size_t)t * d : nullptr;
    P.next_logits = next_logits ? next_logits + (size_t)t * E : nullptr;
    P.next_ids = next_ids ? next_ids + (size_t)t * K : nullptr;
    P.next_w = next_weights ? next_weights + (size_t)t * K : nullptr;
    P.ws = reinterpret_cast<uint8_t*>(workspace);
    E0_CHECK_CUDA(launch_engine(P, (cudaStream_t)stream));
  }
  return E0_OK;
}

extern "C" e0_status e0_prerouter_forward(const e0_prerouter* head, int32_t d, int32_t E, const uint16_t* h,
                                          const int32_t* ids_cur, const int32_t* ids_prev, int32_t T, int32_t K,
                                          const float* logit_bias, float* logits_out, int32_t* ids_out,
                                          float* weights_out, void* workspace, size_t workspace_bytes,
                                          e0_stream stream) {
  e0_dims dm{d, E, 64, K};
  e0_status st = check_dims(&dm);
  if (st) return st;
  E0_REQUIRE(head && h && (logits_out || ids_out), E0_ERR_INVALID, "e0_prerouter_forward: NULL required argument");
  E0_REQUIRE(T >= 0, E0_ERR_INVALID, "T must be >= 0");
  if (T == 0) return E0_OK;
  st = check_ws(&dm, 1, workspace, workspace_bytes);
  if (st) return st;
  if (T > 1) {
    // several tokens: each head weight row read once for all of them
    E0_REQUIRE(T <= 16, E0_ERR_SHAPE, "e0_prerouter_forward: T must be <= 16");
    E0_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, E0_ERR_INVALID,
               "workspace must be 256-byte aligned");
    E0_REQUIRE(al16(h), E0_ERR_INVALID, "e0_prerouter_forward: h must be 16-byte aligned for T > 1");
    E0_REQUIRE(workspace_bytes >= 256 + e0mt_head_scratch(&dm, T, head->H), E0_ERR_NOMEM,
               "workspace smaller than e0_decode_workspace_size(dims, T, 0, H)");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return e0mt_head(head, &dm, h, ids_cur, ids_prev, T, logit_bias, logits_out, ids_out, weights_out, ws + 256,
                     workspace_bytes - 256, reinterpret_cast<uint32_t*>(ws + 4), stream);
  }
  int ncta;
  st = device_ctas(d, &ncta);
  if (st) return st;
  static thread_local EngineParams P;
  base_params(P, d, E, 64, K, 1, ncta, MODE_HEAD);
  st = fill_head(head, &dm, &P.inline_layer);
  if (st) return st;
  E0_REQUIRE(head->H == 0 || ids_cur, E0_ERR_INVALID, "a head with an MLP needs ids_cur");
  PlanSpec ps;
  ps.d = d; ps.E = E; ps.F = 64; ps.K = K;
  ps.head = head->H > 0; ps.lres = true; ps.H = head->H;
  const CachedPlan* cp;
  st = get_plan(ps, ncta, &cp);
  if (st) return st;
  set_inline_plan(P, *cp);
  P.logit_bias = logit_bias;
  for (int t = 0; t < T; ++t) {
    P.h_in = h + (size_t)t * d;
    P.ids_in = ids_cur ? ids_cur + (size_t)t * K : nullptr;
    P.ids_prev_in = ids_prev ? ids_prev + (size_t)t * K : nullptr;
    P.next_logits = logits_out ? logits_out + (size_t)t * E : nullptr;
    P.next_ids = ids_out ? ids_out + (size_t)t * K : nullptr;
    P.next_w = weights_out ? weights_out + (size_t)t * K : nullptr;
    P.ws = reinterpret_cast<uint8_t*>(workspace);
    E0_CHECK_CUDA(launch_engine(P, (cudaStream_t)stream));
  }
  return E0_OK;
}

extern "C" e0_status e0_qlinear_lora(const e0_qlora* lora, int32_t in, const uint16_t* x, int32_t T,
                                     int32_t accumulate, uint16_t* y, float* y_f32, void* workspace,
                                     size_t workspace_bytes, e0_stream stream) {
  E0_REQUIRE(lora && x && y, E0_ERR_INVALID, "e0_qlinear_lora: NULL required argument");
  E0_REQUIRE(in == 256 || in == 512 || in == 1024 || in == 2048, E0_ERR_SHAPE, "in must be 256, 512, 1024 or 2048");
  E0_REQUIRE(T >= 0, E0_ERR_INVALID, "T must be >= 0");
  if (T == 0) return E0_OK;
  e0_dims dm{in, 8, 64, 1};
  e0_status st = check_ws(&dm, 1, workspace, workspace_bytes);
  if (st) return st;
  E0_REQUIRE(al16(x) && al16(y) && (!y_f32 || al16(y_f32)), E0_ERR_INVALID, "x, y must be 16-byte aligned");
  int ncta;
  st = device_ctas(in, &ncta);
  if (st) return st;
  static thread_local EngineParams P;
  base_params(P, in, 8, 64, 1, 1, ncta, MODE_QLINEAR);
  bool ab = false;
  st = fill_lora(lora, in, &P.inline_layer, &ab);
  if (st) return st;
  P.norm = 0;
  P.out_dim = lora->out;
  P.accumulate = accumulate;
  PlanSpec ps;
  ps.d = in; ps.E = 8; ps.F = 64; ps.K = 1;
  ps.lora = true; ps.lora_ab = ab; ps.lout = lora->out; ps.lr = ab ? lora->r : 0;
  const CachedPlan* cp;
  st = get_plan(ps, ncta, &cp);
  if (st) return st;
  set_inline_plan(P, *cp);
  for (int t = 0; t < T; ++t) {
    P.h_in = x + (size_t)t * in;
    P.h_out = y + (size_t)t * lora->out;
    P.delta_out = y_f32 ? y_f32 + (size_t)t * lora->out : nullptr;
    P.ws = reinterpret_cast<uint8_t*>(workspace);
    E0_CHECK_CUDA(launch_engine(P, (cudaStream_t)stream));
  }
  return E0_OK;
}

// ------------------------------------------------------------------ stack
struct e0_stack {
  e0_dims dims;
  int L;
  int ncta;
  std::vector<int8_t> prerouted;   // 1: routed by head l-1 after the first token
  uint64_t ahead_mask = 0;         // route-ahead layers
  LayerDesc* d_layers = nullptr;
  Unit* d_plan = nullptr;
  uint8_t* d_counts = nullptr;
  uint8_t* d_defer = nullptr;   // [KINDS_MAX][ncta]: CTAs that only hold prerouter work
  int n_defer[KINDS_MAX] = {};
};

extern "C" e0_status e0_stack_create(e0_stack** out, const e0_dims* dims, const e0_layer* layers, int32_t L,
                                     const int8_t* route_src) {
  E0_REQUIRE(out && layers && L >= 1 && L <= LMAX, E0_ERR_INVALID, "e0_stack_create: need 1..48 layers");
  *out = nullptr;
  e0_status st = check_dims(dims);
  if (st) return st;
  int ncta;
  st = device_ctas(dims->d, &ncta);
  if (st) return st;
  std::vector<LayerDesc> descs(L);
  PlanSpec spec[KINDS_MAX];
  bool have_spec[KINDS_MAX] = {};
  bool head_before = false;  // a layer before this one has a head
  for (int l = 0; l < L; ++l) {
    LayerDesc& D = descs[l];
    std::memset(&D, 0, sizeof(D));
    const e0_layer& ly = layers[l];
    PlanSpec ps;
    ps.d = dims->d; ps.E = dims->E; ps.F = dims->F; ps.K = dims->K;
    st = fill_experts(&ly.routed, dims, true, &D);
    if (st) return st;
    ps.routed = true;
    if (ly.shared.n > 0) {
      st = fill_experts(&ly.shared, dims, false, &D);
      if (st) return st;
      ps.shared = true;
    }
    if (ly.lora.w.q) {
      bool ab = false;
      st = fill_lora(&ly.lora, dims->d, &D, &ab);
      if (st) return st;
      E0_REQUIRE(ly.lora.out == dims->d, E0_ERR_SHAPE, "stack LoRA linears must be d x d");
      ps.lora = true; ps.lora_ab = ab; ps.lout = ly.lora.out; ps.lr = ab ? ly.lora.r : 0;
    }
    if (ly.head.lres) {
      st = fill_head(&ly.head, dims, &D);
      if (st) return st;
      ps.head = ly.head.H > 0; ps.lres = true; ps.H = ly.head.H;
    }
    E0_REQUIRE(ly.router && al16(ly.router), E0_ERR_INVALID,
               "every stack layer needs its own gate (used at the first token)");
    D.router = ly.router;
    D.score_bias = ly.score_bias;
    D.gate_for = -1;
    const int src = route_src ? route_src[l] : 0;
    E0_REQUIRE(src <= 1, E0_ERR_INVALID, "route_src must be 1 (head), 0 (own gate) or -N (route-ahead by N)");
    D.prerouted = src == 1 ? 1 : 0;
    if (D.prerouted) {
      E0_REQUIRE(l > 0 && layers[l - 1].head.lres, E0_ERR_INVALID,
                 "a prerouted layer needs a head on the previous layer");
    }
    if (src < 0) {
      E0_REQUIRE(l + src >= 0, E0_ERR_INVALID, "route-ahead by N needs N layers before the layer");
      D.ahead = -src;
    }
    const int kind = D.has_head ? KIND_MAIN : (head_before ? KIND_TAIL : KIND_MAIN_NOHEAD);
    head_before = head_before || D.has_head;
    if (have_spec[kind]) {
      E0_REQUIRE(std::memcmp(&spec[kind], &ps, sizeof(ps)) == 0, E0_ERR_UNSUPPORTED,
                 "stack layers of one kind must share one shape");
    } else {
      spec[kind] = ps;
      have_spec[kind] = true;
    }
    D.plan_kind = kind;
  }
  PlanSpec rs;
  rs.d = dims->d; rs.E = dims->E; rs.F = dims->F; rs.K = dims->K; rs.router = true;
  std::vector<Unit> units((size_t)KINDS_MAX * ncta * MAXU);
  std::vector<uint8_t> counts((size_t)KINDS_MAX * ncta, 0);
  std::vector<uint8_t> defer((size_t)KINDS_MAX * ncta, 0);
  // layers with a head: the prerouter's work on CTAs of its own (deferred, see build_plan)
  int n_crit = ncta;
  for (int k = 0; k < 2; ++k)
    if (have_spec[k]) {
      int nc = ncta;
      st = build_plan(spec[k], ncta, units.data() + (size_t)k * ncta * MAXU, counts.data() + (size_t)k * ncta,
                      k == KIND_MAIN ? defer.data() + (size_t)k * ncta : nullptr, &nc);
      if (st) return st;
      n_crit = std::min(n_crit, nc);
    }
  if (have_spec[KIND_TAIL]) {
    st = build_plan(spec[KIND_TAIL], ncta, units.data() + (size_t)KIND_TAIL * ncta * MAXU,
                    counts.data() + (size_t)KIND_TAIL * ncta, nullptr, nullptr, n_crit);
    if (st) return st;
  }
  // route-ahead: the gate rows of layer l run on layer l - N's input (one target per layer)
  for (int l = 0; l < L; ++l)
    if (descs[l].ahead > 0) {
      LayerDesc& src = descs[l - descs[l].ahead];
      E0_REQUIRE(src.gate_for < 0, E0_ERR_INVALID, "two route-ahead layers read the same earlier layer");
      src.gate_for = l;
    }
  // the router rows of own-gate layers stay off the deferred CTAs
  st = build_plan(rs, ncta, units.data() + (size_t)KIND_ROUTER * ncta * MAXU,
                  counts.data() + (size_t)KIND_ROUTER * ncta, nullptr, nullptr, n_crit);
  if (st) return st;

  e0_stack* s = new e0_stack();
  s->dims = *dims;
  s->L = L;
  s->ncta = ncta;
  s->prerouted.assign(L, 0);
  for (int l = 0; l < L; ++l) {
    s->prerouted[l] = descs[l].prerouted ? 1 : 0;
    if (descs[l].ahead > 0) s->ahead_mask |= 1ull << l;
  }
  for (int k = 0; k < KINDS_MAX; ++k) {
    int nd = 0;
    for (int c = 0; c < ncta; ++c) nd += defer[(size_t)k * ncta + c];
    s->n_defer[k] = nd;
  }
  cudaError_t e = cudaMalloc(&s->d_layers, sizeof(LayerDesc) * L);
  if (e == cudaSuccess) e = cudaMalloc(&s->d_plan, sizeof(Unit) * units.size());
  if (e == cudaSuccess) e = cudaMalloc(&s->d_counts, counts.size());
  if (e == cudaSuccess) e = cudaMalloc(&s->d_defer, defer.size());
  if (e == cudaSuccess) e = cudaMemcpy(s->d_defer, defer.data(), defer.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(s->d_layers, descs.data(), sizeof(LayerDesc) * L, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(s->d_plan, units.data(), sizeof(Unit) * units.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(s->d_counts, counts.data(), counts.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    e0_stack_destroy(s);
    return e0::cuda_fail(e, "e0_stack_create");
  }
  *out = s;
  return E0_OK;
}

extern "C" void e0_stack_destroy(e0_stack* s) {
  if (!s) return;
  if (s->d_layers) cudaFree(s->d_layers);
  if (s->d_plan) cudaFree(s->d_plan);
  if (s->d_counts) cudaFree(s->d_counts);
  if (s->d_defer) cudaFree(s->d_defer);
  delete s;
}

extern "C" size_t e0_stack_workspace_size(const e0_stack* s) {
  if (!s) return 0;
  return ws_layout(s->dims.E, s->L).total;
}

extern "C" e0_status e0_stack_step(e0_stack* s, int32_t step, const uint16_t* h0, const uint16_t* incr,
                                   uint16_t* h_out, const e0_stack_outputs* outs, const float* logit_bias,
                                   void* workspace, size_t workspace_bytes, e0_stream stream) {
  E0_REQUIRE(s && h0 && h_out, E0_ERR_INVALID, "e0_stack_step: NULL required argument");
  E0_REQUIRE(step >= 0, E0_ERR_INVALID, "step must be >= 0");
  e0_status st = check_ws(&s->dims, s->L, workspace, workspace_bytes);
  if (st) return st;
  E0_REQUIRE(al16(h0) && al16(h_out) && (!incr || al16(incr)), E0_ERR_INVALID, "hidden buffers must be 16-byte aligned");
  static thread_local EngineParams P;
  base_params(P, s->dims.d, s->dims.E, s->dims.F, s->dims.K, s->L, s->ncta, MODE_STACK);
  set_route(P, &s->dims);
  P.score_bias = nullptr;  // per layer in the stack
  P.layers = s->d_layers;
  P.plan = s->d_plan;
  P.plan_n = s->d_counts;
  P.defer = s->d_defer;
  for (int k = 0; k < KINDS_MAX; ++k) {
    P.n_defer[k] = s->n_defer[k];
    P.n_arrive[k] = s->ncta - s->n_defer[k];
  }
  P.kinds = KINDS_MAX;
  P.step = step;
  // routed from gate logits: own-gate layers (and head-routed ones at the first token),
  // whose gate rows run on their own input, and route-ahead layers, whose gate rows run
  // N layers earlier
  uint64_t own = 0;
  for (int l = 0; l < s->L; ++l)
    if (!((s->ahead_mask >> l) & 1ull) && (step == 0 || !s->prerouted[l])) own |= 1ull << l;
  P.gate_mask = own;
  P.router_mask = own | s->ahead_mask;
  P.h_in = h0;
  P.incr = incr;
  P.h_out = h_out;
  if (outs) {
    P.ids_trace = outs->ids;
    P.w_trace = outs->weights;
    P.h_trace = outs->h_trace;
    P.delta_trace = outs->delta;
    P.delta_out = outs->delta ? outs->delta + (size_t)(s->L - 1) * s->dims.d : nullptr;
    P.z_trace = outs->logits;
    P.next_ids_out = outs->next_ids;
    P.commit_box = static_cast<uint32_t*>(outs->commit_box);
  }
  P.logit_bias = logit_bias;
  P.ws = reinterpret_cast<uint8_t*>(workspace);
  E0_CHECK_CUDA(launch_engine(P, (cudaStream_t)stream));
  return E0_OK;
}
