// Prefill: T tokens through one MoE layer on the fifth-generation tensor cores.
//
// "The Other Half of the Memory Wall" (Edge0), §3.1 "Executor paths": the same expert
// math as decode, down(silu(gate(x)) * up(x)) over int4 affine group-64 weights,
// combined with the renormalised softmax of the selected logits (Appendix A), plus the
// shared expert and the unmerged LoRA linear (§3.3); no prerouter in prefill.
//
// Path (one stream, in order):
//   route      top-K of each token's logits, combine weights        (one warp per token)
//   sort       counting sort of the T*K (token, k) pairs by expert   (one CTA)
//   gather     x = RMSNorm(h) in fp16, once per token and once per pair, grouped by expert
//   gemm_q4    grouped GEMM, int4 weights dequantised to fp16 in tensor memory, tcgen05.mma
//              with the fp32 accumulator in tensor memory:
//                gate/up  [rows_e x d] x [d x 2F]  -> SwiGLU epilogue -> fp16 a [rows_e x F]
//                down     [rows_e x F] x [F x d]   -> x w_(t,k)        -> fp32 y per pair
//              the shared expert rides in the gate/up and down launches as one more
//              group (its own token rows, weights and outputs); the LoRA base runs
//              through the same kernel as one group
//   lora_a     v = A x on the CUDA cores (r = 16: too thin for a tile)
//   combine    h_out = bf16(h + sum_k y_(t,k) + y_shared + y_lora), sum over k in k order,
//              with y_lora = W_int4 x + (alpha/r) B v formed here
//
// fp16 (not bf16) operands: the dequantised weight s*q + b and x are each rounded once
// to fp16 (11-bit significand), which keeps the rounding error of the products well
// inside the parity bar; bf16 would leave it at the bar.  Within every group of 8
// reduction indices the operands are stored in the order [0,4,1,5,2,6,3,7] on both
// sides (the order in which the nibble-to-fp16 conversion produces pairs), which leaves
// every dot product unchanged.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "e0_engine.cuh"
#include "e0_tc.cuh"

using namespace e0dev;
using namespace e0tc;

namespace e0pf {

constexpr int WM = 128;                      // weight rows per tile: the MMA's M
constexpr int TT = 64;                       // token rows per tile, at most: the MMA's N
constexpr int BK = 64;                       // reduction block
constexpr int NWD = 2;                       // dequantise -> MMA hand-over buffers
constexpr int X_BYTES = TT * BK * 2;         // 8 KB of fp16 token rows
constexpr int Q_BYTES = WM * BK / 2;         // 4 KB of int4 codes
constexpr int RAW_BYTES = X_BYTES + Q_BYTES;
constexpr int EMAXP = 1024;
constexpr int MAXT = 256;  // tiles of a CTA whose placement is tabulated in shared memory
// A hand-over carries the MMA's operands for HK k-blocks (HK = 4 when the reduction
// length allows it, else 2): the dequantised weights (A) in tensor memory, 32 columns per
// k-block (lane = weight row, two fp16 per column), and a copy of the token rows (B) in
// shared memory, so that a copy stage is free as soon as it has been converted and only
// the hand-over buffers wait for the tensor core.  Four k-blocks per hand-over halve the
// waits, fences and index work per converted weight.
template <int HK>
struct Cfg {
  static constexpr int STAGES = HK == 4 ? 12 : 14;       // copy stages in flight
  static constexpr int A_COLS = HK * BK / 2;             // tensor-memory columns of one hand-over
  static constexpr int HB_BYTES = HK * X_BYTES;          // token rows of one hand-over buffer
  static constexpr int TMEM_COLS = 2 * TT + NWD * A_COLS <= 256 ? 256 : 512;
  static constexpr size_t SMEM =
      1024 + (size_t)STAGES * RAW_BYTES + NWD * HB_BYTES + 2 * (EMAXP + 2) * sizeof(int) + MAXT * sizeof(uint2);
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(STAGES % HK == 0, "a hand-over's stages sit in one ring pass");
  static_assert(2 * TT + NWD * A_COLS <= TMEM_COLS, "tensor memory columns");
};
// roles: warps 0..3 copy (job j by warp j % 4), warps 4..19 dequantise, warp 20 issues the
// MMAs, warps 21..24 run the epilogue (tensor-memory lane quadrants 1, 2, 3, 0)
constexpr int W_COPY = 0, N_COPY = 4, W_DQ0 = 4, N_DQ = 16, W_MMA = 20, W_EPI0 = 21, N_EPI = 4;
// the dequantising warps form two groups that take alternate hand-overs (buffer g for
// group g), so that one group's proxy fence and hand-over overlap the other's work
constexpr int DQ_GROUPS = 2, N_DQG = N_DQ / DQ_GROUPS;
// warp i of a group writes tensor-memory lanes 32 (warp % 4) .. + 31 (the lane quadrant a
// warp may access) and half i / 4 of each 64-wide k-block: 4 code words, 16 columns
constexpr int GT = 32 * (W_EPI0 + N_EPI);
static_assert(X_BYTES % 1024 == 0 && RAW_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
static_assert(N_DQG == 8 && WM == 128 && W_DQ0 % 4 == 0, "two warps per lane quadrant in a group, one per half block");
static_assert(NWD == DQ_GROUPS && NWD == 2, "one hand-over buffer per dequantising group; p & 1 picks it");

enum Epi : int { EPI_SWIGLU = 0, EPI_F32 = 1 };

struct GemmArgs {
  const __half* A;        // token rows [rows][K] fp16, reduction index permuted within groups of 8
  int lda;
  int K, N;               // reduction length (multiple of 128), outputs per group (multiple of 128)
  int ngroups;
  const int* row_off;     // [ngroups + 1] rows of group g: [row_off[g], row_off[g + 1])
  const int* tile_off;    // [ngroups + 1] prefix sums of ceil(rows_g / TT)
  const uint32_t* q;      // int4 codes of all groups (group g = weight slot g)
  const uint16_t* s;      // bf16 scales
  const uint16_t* b;      // bf16 biases
  __half* out16;          // EPI_SWIGLU: [rows][N / 2] fp16, permuted within groups of 8
  float* out32;           // EPI_F32: [rows][N]
  int ldo;
  const float* rowscale;  // EPI_F32: factor per row (nullable)
  // one extra group after the ngroups (the shared expert), xrows > 0: its own token rows
  // A2 [xrows][K] (same lda), weights q2/s2/b2 (one expert) and outputs out16b/out32b
  // [xrows][...] (same ldo, no row factor), so that its tiles share the launch
  int xrows;
  const __half* A2;
  const uint32_t* q2;
  const uint16_t* s2;
  const uint16_t* b2;
  __half* out16b;
  float* out32b;
  uint32_t* status;
  uint64_t timeout_ns;
};

// A tile: rows [m0, m0 + rows) of its group's token rows (of A, or of A2 for the extra
// group, counted from 0 there), weight rows [n0, n0 + WM) of weight slot `slot`
// (slot == ngroups: the extra group).
struct Tile {
  int m0, rows, n0, slot;
};

// Dequantise 32 codes (one uint4: half of a 64-code weight row segment) to 16 fp16 pairs:
// codes j and j + 4 of each 8-code word become one pair, which is the element order
// [0,4,1,5,2,6,3,7] within every group of 8 that the token rows use as well.  A pair is
// formed by the exponent trick without a shift for j = 0, 1 (and one shift of the word
// by 8 for j = 2, 3): masked into the mantissa of 1024 (0x6400), a code c in the low
// nibble of each half gives 1024 + c, in the high nibble 1024 + 16 c; c is recovered
// exactly as t - 1024 or t / 16 - 64, then s * c + b.
__device__ __forceinline__ void dequant32(const uint8_t* codes, __half2 s2, __half2 b2, uint32_t (&out)[16]) {
  const uint4 w0 = *reinterpret_cast<const uint4*>(codes);
  const uint32_t words[4] = {w0.x, w0.y, w0.z, w0.w};
  const __half2 k1024 = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
  const __half2 k16th = __halves2half2(__ushort_as_half((unsigned short)0x2C00), __ushort_as_half((unsigned short)0x2C00));
  const __half2 km64 = __halves2half2(__ushort_as_half((unsigned short)0xD400), __ushort_as_half((unsigned short)0xD400));
#pragma unroll
  for (int mm = 0; mm < 4; ++mm) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const uint32_t v = words[mm] >> (8 * hb);
      const uint32_t tl = (v & 0x000F000Fu) | 0x64006400u;  // codes 2hb, 2hb + 4: 1024 + c
      const uint32_t th = (v & 0x00F000F0u) | 0x64006400u;  // codes 2hb + 1, 2hb + 5: 1024 + 16 c
      const __half2 cl = __hsub2(*reinterpret_cast<const __half2*>(&tl), k1024);
      const __half2 ch = __hfma2(*reinterpret_cast<const __half2*>(&th), k16th, km64);
      const __half2 wl = __hfma2(cl, s2, b2);
      const __half2 wh = __hfma2(ch, s2, b2);
      out[4 * mm + 2 * hb] = *reinterpret_cast<const uint32_t*>(&wl);
      out[4 * mm + 2 * hb + 1] = *reinterpret_cast<const uint32_t*>(&wh);
    }
  }
}

// Position of a job (tile i, k-block kb) tracked as the job index advances, so that the
// loops divide by the runtime k-block count only once.
struct JobPos {
  int i, kb;
  __device__ __forceinline__ JobPos(int j, int KB) : i(j / KB), kb(j % KB) {}
  __device__ __forceinline__ void advance(int n, int KB) {
    kb += n;
    while (kb >= KB) {
      kb -= KB;
      ++i;
    }
  }
};

__device__ __forceinline__ void cp_async_bar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Grouped GEMM out[rows][n] = sum_k x[row][k] W_g[n][k] with the operands swapped for
// the tensor core: the weight tile (128 rows, dequantised to fp16 in tensor memory) is
// the MMA's A and the group's token rows (up to 64, rounded up to 16, in shared memory)
// its B, so a group of few tokens costs few MMA columns.  The accumulator [weight row]
// [token] lives in tensor memory, double-buffered so the epilogue of one tile overlaps
// the next tile's MMAs.  Copy, dequantisation, MMA and epilogue run in their own warps,
// handing stages over through mbarriers; every wait is bounded.
template <int LAYOUT, int EPI, int HK>
__global__ void __launch_bounds__(GT, 1) gemm_q4_kernel(const __grid_constant__ GemmArgs g) {
  using C = Cfg<HK>;
  constexpr int STAGES = C::STAGES, A_COLS = C::A_COLS, HB_BYTES = C::HB_BYTES, TMEM_COLS = C::TMEM_COLS;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  uint8_t* raw = sm;                                // STAGES x [token rows | codes]
  uint8_t* hbuf = sm + (size_t)STAGES * RAW_BYTES;  // NWD x token rows of a hand-over
  int* s_row = reinterpret_cast<int*>(hbuf + NWD * HB_BYTES);
  int* s_tile = s_row + (EMAXP + 2);
  uint2* s_tt = reinterpret_cast<uint2*>(s_tile + (EMAXP + 2));  // [MAXT] this CTA's tiles
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], wd_full[NWD], wd_empty[NWD], acc_full[2], acc_empty[2], fin;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int WT = g.N / WM, KB = g.K / BK;

  for (int i = tid; i <= g.ngroups; i += GT) {
    s_row[i] = g.row_off[i];
    s_tile[i] = g.tile_off[i];
  }
  const int ng = g.ngroups + (g.xrows > 0 ? 1 : 0);  // groups with the extra one
  if (tid == 0 && g.xrows > 0) {
    s_row[g.ngroups + 1] = g.row_off[g.ngroups] + g.xrows;
    s_tile[g.ngroups + 1] = g.tile_off[g.ngroups] + (g.xrows + TT - 1) / TT;
  }
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 32);
      mbar_init(&empty[i], N_DQG);  // freed by the dequantising group that converts it
    }
    for (int i = 0; i < NWD; ++i) {
      mbar_init(&wd_full[i], N_DQG);
      mbar_init(&wd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], N_EPI);
    }
    mbar_init(&fin, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == W_MMA) tmem_alloc(&tmem_slot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const int total = s_tile[ng] * WT;
  const int my_tiles = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int jobs = my_tiles * KB;

  // tile i of this CTA: token rows, weight rows and weight slot (group search in shared memory)
  auto find_tile = [&](int i) -> Tile {
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    int lo = 0, hi = ng;  // s_tile[lo] * WT <= t < s_tile[hi] * WT
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile[mid] * WT <= t) lo = mid; else hi = mid;
    }
    const int tt_g = s_tile[lo + 1] - s_tile[lo];  // token tiles of the group
    const int local = t - s_tile[lo] * WT;
    Tile T;
    T.m0 = s_row[lo] + (local % tt_g) * TT;
    T.rows = min(TT, s_row[lo + 1] - T.m0);
    T.n0 = (local / tt_g) * WM;
    T.slot = lo;
    if (lo == g.ngroups) T.m0 -= s_row[g.ngroups];  // the extra group's own rows
    return T;
  };
  // the first MAXT tiles tabulated once (every role looks tiles up, several times each):
  // {m0, rows | n0 / WM << 8 | slot << 20}
  for (int i = tid; i < my_tiles && i < MAXT; i += GT) {
    const Tile T = find_tile(i);
    s_tt[i] = make_uint2((uint32_t)T.m0, (uint32_t)T.rows | ((uint32_t)(T.n0 / WM) << 8) | ((uint32_t)T.slot << 20));
  }
  __syncthreads();
  auto tile_of = [&](int i) -> Tile {
    if (i >= MAXT) return find_tile(i);
    const uint2 e = s_tt[i];
    Tile T;
    T.m0 = (int)e.x;
    T.rows = (int)(e.y & 0xFFu);
    T.n0 = (int)((e.y >> 8) & 0xFFFu) * WM;
    T.slot = (int)(e.y >> 20);
    return T;
  };
  // bounded wait: false after an abort or once the time limit passes (sets the status)
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait_hint(bar, parity, 10000u)) return true;  // suspended, not spinning
      if ((it & 3u) == 0) {
        if (s_abort) return false;
        if (globaltimer() - t0 > g.timeout_ns) {
          atomicOr(g.status, (uint32_t)E0_DEV_TIMEOUT);
          s_abort = 1;
          return false;
        }
      }
    }
  };

  if (warp >= W_COPY && warp < W_COPY + N_COPY) {
    // ---------------- copies: token rows and codes of job j into stage j % STAGES
    int cur_i = -1;
    Tile T{};
    JobPos jp(warp - W_COPY, KB);
    int st = (warp - W_COPY) % STAGES, round = (warp - W_COPY) / STAGES;
    // lane roles: 16-byte chunk ch of token rows r0, r0 + 4, ... (chunk stored at ch ^ (r % 8));
    // code row (lane >> 1) + 16 m, half lane & 1
    const int ch = lane & 7, r0 = lane >> 3, qn = lane >> 1, qh = lane & 1;
    const uint32_t xsw0 = (uint32_t)((ch ^ r0) << 4), xsw1 = (uint32_t)((ch ^ (r0 + 4)) << 4);
    for (int j = warp - W_COPY; j < jobs; j += N_COPY, jp.advance(N_COPY, KB)) {
      if (round > 0 && !wait(&empty[st], (round - 1) & 1)) break;
      if (jp.i != cur_i) {
        cur_i = jp.i;
        T = tile_of(cur_i);
      }
      const int kb = jp.kb;
      uint8_t* sx = raw + (size_t)st * RAW_BYTES;
      uint8_t* sq = sx + X_BYTES;
      const bool xt = T.slot == g.ngroups;  // the extra group: its own rows and weights
      const int wslot = xt ? 0 : T.slot;
      const __half* xsrc = (xt ? g.A2 : g.A) + (size_t)(T.m0 + r0) * g.lda + kb * BK + ch * 8;
      const size_t xstep = (size_t)4 * g.lda;
      uint8_t* xdst = sx + r0 * 128;
      for (int r = r0, k = 0; r < T.rows; r += 4, ++k, xsrc += xstep, xdst += 4 * 128)
        cp_async16(xdst + ((k & 1) ? xsw1 : xsw0), xsrc, 16u);
      const uint32_t* qsrc;
      size_t qstep;
      if (LAYOUT == E0_LAYOUT_ROWS) {
        qsrc = (xt ? g.q2 : g.q) + ((size_t)wslot * g.N + T.n0 + qn) * (g.K / 8) + kb * 8 + qh * 4;
        qstep = (size_t)16 * (g.K / 8);
      } else {
        qsrc = (xt ? g.q2 : g.q) + (((size_t)wslot * (g.K / 32) + 2 * kb + qh) * g.N + T.n0 + qn) * 4;
        qstep = 16 * 4;
      }
#pragma unroll
      for (int m = 0; m < WM * 2 / 32; ++m) cp_async16(sq + (qn + 16 * m) * 32 + qh * 16, qsrc + m * qstep, 16u);
      cp_async_bar_arrive(&full[st]);  // completes when this lane's copies have landed
      st += N_COPY;
      if (st >= STAGES) {
        st -= STAGES;
        ++round;
      }
    }
    cp_async_wait<0>();
  } else if (warp >= W_DQ0 && warp < W_DQ0 + N_DQ) {
    // ---------------- dequantisation: group grp takes hand-overs p = grp, grp + 2, ...;
    // a thread owns weight row n (its tensor-memory lane) and half h of each 64-wide block
    const int dt = tid - 32 * W_DQ0, grp = dt / (32 * N_DQG), gtid = dt % (32 * N_DQG);
    const int n = 32 * (warp & 3) + lane, h = (gtid >> 5) >> 2;
    const uint32_t a_lane = (uint32_t)(32 * (warp & 3)) << 16;
    // scales and biases of this row for the HK k-blocks of hand-over p, as HK / 2 words
    // of two bf16 each (prefetched two hand-overs of the group ahead; in the rows layout
    // they are HK contiguous bf16: one vector load); the tile of the last fetch is cached
    int t_i = -1;
    Tile tt{};
    using SW = uint32_t[HK / 2];
    // the fetches come in order, p = grp, grp + 2, ...: their job position advances
    JobPos fp(HK * grp, KB);
    auto fetch = [&](int p, SW& sv, SW& bv) {
#pragma unroll
      for (int u = 0; u < HK / 2; ++u) sv[u] = bv[u] = 0u;
      if (HK * p >= jobs) return;
      const int i = fp.i, kb = fp.kb;
      fp.advance(HK * DQ_GROUPS, KB);
      if (i != t_i) {
        t_i = i;
        tt = tile_of(i);
      }
      const bool xt = tt.slot == g.ngroups;  // the extra group's weights
      const int wslot = xt ? 0 : tt.slot;
      const uint16_t* gs = xt ? g.s2 : g.s;
      const uint16_t* gb = xt ? g.b2 : g.b;
      if (LAYOUT == E0_LAYOUT_ROWS) {
        // K / 64 is a multiple of HK and kb of HK: HK * 2 bytes, aligned
        const size_t idx = ((size_t)wslot * g.N + tt.n0 + n) * (g.K / 64) + kb;
        if (HK == 4) {
          const uint2 a = __ldg(reinterpret_cast<const uint2*>(gs + idx));
          const uint2 b = __ldg(reinterpret_cast<const uint2*>(gb + idx));
          sv[0] = a.x; sv[HK / 2 - 1] = a.y;
          bv[0] = b.x; bv[HK / 2 - 1] = b.y;
        } else {
          sv[0] = __ldg(reinterpret_cast<const uint32_t*>(gs + idx));
          bv[0] = __ldg(reinterpret_cast<const uint32_t*>(gb + idx));
        }
      } else {
#pragma unroll
        for (int u = 0; u < HK; ++u) {
          const size_t idx = ((size_t)wslot * (g.K / 64) + kb + u) * g.N + tt.n0 + n;
          const uint32_t sh = (uint32_t)__ldg(gs + idx), bh = (uint32_t)__ldg(gb + idx);
          sv[u / 2] |= sh << (16 * (u & 1));
          bv[u / 2] |= bh << (16 * (u & 1));
        }
      }
    };
    // three hand-overs of scales in flight: current, next and the one after
    SW cs, cb, ns, nb, ms, mb;
    fetch(grp, cs, cb);
    fetch(grp + DQ_GROUPS, ns, nb);
    fetch(grp + 2 * DQ_GROUPS, ms, mb);
    int x_i = -1, x_bytes = X_BYTES;  // token-row bytes to hand over: the tile's rows rounded to 16
    int st0 = (HK * grp) % STAGES;      // first stage of hand-over p, and its ring pass
    uint32_t ph0 = (uint32_t)((HK * grp) / STAGES) & 1u;
    JobPos hp(HK * grp, KB);  // this hand-over's first job
    for (int p = grp; HK * p < jobs; p += DQ_GROUPS, hp.advance(HK * DQ_GROUPS, KB)) {
      const int buf = p & (NWD - 1);  // this group's buffer: p % NWD == grp
      if (hp.i != x_i) {
        x_i = hp.i;
        x_bytes = ((tile_of(x_i).rows + 15) & ~15) * 128;
      }
      bool ok = true;
#pragma unroll
      for (int h2 = 0; h2 < HK; ++h2) ok = ok && wait(&full[st0 + h2], ph0);
      if (!ok) break;
      if (p >= NWD && !wait(&wd_empty[buf], ((p >> 1) - 1) & 1)) break;
      fence_after_sync();  // the MMAs that read this buffer's tensor memory are complete
      // the scales and biases of two k-blocks at a time to fp16 (one packing conversion)
      __half2 sp[HK / 2], bp[HK / 2];
#pragma unroll
      for (int u = 0; u < HK / 2; ++u) {
        sp[u] = __floats2half2_rn(__uint_as_float(cs[u] << 16), __uint_as_float(cs[u] & 0xFFFF0000u));
        bp[u] = __floats2half2_rn(__uint_as_float(cb[u] << 16), __uint_as_float(cb[u] & 0xFFFF0000u));
      }
#pragma unroll
      for (int h2 = 0; h2 < HK; ++h2) {
        uint32_t w[16];
        const __half2 s2 = (h2 & 1) ? __high2half2(sp[h2 / 2]) : __low2half2(sp[h2 / 2]);
        const __half2 b2 = (h2 & 1) ? __high2half2(bp[h2 / 2]) : __low2half2(bp[h2 / 2]);
        dequant32(raw + (size_t)(st0 + h2) * RAW_BYTES + X_BYTES + n * 32 + h * 16, s2, b2, w);
        tmem_st16(tmem + a_lane + (uint32_t)(2 * TT + buf * A_COLS + h2 * (BK / 2) + h * 16), w);
      }
      // token rows of the k-blocks into the hand-over buffer (16-byte chunks keep their
      // swizzled places; the MMA reads the tile's rows rounded up to 16)
#pragma unroll
      for (int h2 = 0; h2 < HK; ++h2) {
        const uint4* src = reinterpret_cast<const uint4*>(raw + (size_t)(st0 + h2) * RAW_BYTES);
        uint4* dst = reinterpret_cast<uint4*>(hbuf + (size_t)buf * HB_BYTES + (size_t)h2 * X_BYTES);
        for (int c = gtid; c < x_bytes / 16; c += 32 * N_DQG) dst[c] = src[c];
      }
      // the weights (tensor memory) and token rows (async proxy) are read by the tensor core
      tmem_st_wait();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wd_full[buf]);
#pragma unroll
        for (int h2 = 0; h2 < HK; ++h2) mbar_arrive(&empty[st0 + h2]);  // this warp is done with the stages
      }
#pragma unroll
      for (int u = 0; u < HK / 2; ++u) {
        cs[u] = ns[u];
        cb[u] = nb[u];
        ns[u] = ms[u];
        nb[u] = mb[u];
      }
      fetch(p + 3 * DQ_GROUPS, ms, mb);
      st0 += HK * DQ_GROUPS;  // the group's next hand-over
      while (st0 >= STAGES) {
        st0 -= STAGES;
        ph0 ^= 1u;
      }
    }
  } else if (warp == W_MMA) {
    // ---------------- the MMA warp: every lane walks the hand-overs (operand addresses
    // stay warp-uniform), one elected lane issues the MMAs and commits them
    int cur_i = -1;
    Tile T{};
    uint32_t idesc = 0;
    JobPos mp(0, KB);
    for (int p = 0; HK * p < jobs; ++p, mp.advance(HK, KB)) {
      const int kb = mp.kb, buf = p & (NWD - 1);
      const int i = mp.i, ab = i & 1;
      if (i != cur_i) {
        cur_i = i;
        T = tile_of(i);
        idesc = idesc_f16_f32(WM, (T.rows + 15) & ~15);
        // the epilogue is done with this accumulator
        if (!__all_sync(0xffffffffu, i < 2 || wait(&acc_empty[ab], ((i >> 1) - 1) & 1))) break;
      }
      if (!__all_sync(0xffffffffu, wait(&wd_full[buf], (p >> 1) & 1))) break;
      fence_after_sync();
      if (elect_one()) {
#pragma unroll
        for (int h2 = 0; h2 < HK; ++h2) {
          const uint32_t a_col = tmem + (uint32_t)(2 * TT + buf * A_COLS + h2 * (BK / 2));
          const uint64_t xd = sdesc_k128(smem_u32(hbuf + (size_t)buf * HB_BYTES + (size_t)h2 * X_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // a 16-wide k step: 8 columns of A, 32 bytes of B
            mma_f16_ta(tmem + (uint32_t)(ab * TT), a_col + (uint32_t)(8 * kk), xd + (uint64_t)(2 * kk), idesc,
                       kb > 0 || h2 > 0 || kk > 0);
        }
        commit(&wd_empty[buf]);
        if (kb + HK == KB) commit(&acc_full[ab]);
      }
      __syncwarp();
    }
    if (elect_one()) {
      commit(&fin);  // every MMA issued so far has completed when this arrives
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&fin, 0) && globaltimer() - t0 < g.timeout_ns) {
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: accumulator [weight row][token] from tensor memory
    const int quad = warp & 3, r = quad * 32 + lane;  // this thread's weight row
    for (int i = 0; i < my_tiles; ++i) {
      const int ab = i & 1;
      const bool ok = wait(&acc_full[ab], (i >> 1) & 1);
      fence_after_sync();
      if (!ok) break;
      const Tile T = tile_of(i);
      const int nout = T.n0 + r;
      const bool xt = T.slot == g.ngroups;  // the extra group writes its own outputs
      __half* out16 = xt ? g.out16b : g.out16;
      float* out32 = xt ? g.out32b : g.out32;
      const float* rowscale = xt ? nullptr : g.rowscale;
#pragma unroll 1
      for (int c0 = 0; c0 < T.rows; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(ab * TT + c0), v);
        const int nc = min(32, T.rows - c0);
        if (EPI == EPI_SWIGLU) {
          // rows 2j / 2j + 1 of the weight tile (lanes 2j / 2j + 1) are gate / up of output j
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float gt = __uint_as_float(v[c]);
            const float up = __shfl_down_sync(0xffffffffu, gt, 1);
            if ((lane & 1) == 0 && c < nc) {
              const int o = nout >> 1;  // output index
              const int pos = (o & ~7) + ((o & 7) < 4 ? 2 * (o & 7) : 2 * ((o & 7) - 4) + 1);
              out16[(size_t)(T.m0 + c0 + c) * g.ldo + pos] = __float2half_rn(__fdividef(gt, 1.0f + __expf(-gt)) * up);
            }
          }
        } else {
          // lane c brings the factor of token row c of the chunk
          const float fl = rowscale && lane < nc ? rowscale[T.m0 + c0 + lane] : 1.0f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float f = __shfl_sync(0xffffffffu, fl, c);
            if (c < nc) out32[(size_t)(T.m0 + c0 + c) * g.ldo + nout] = f * __uint_as_float(v[c]);
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == W_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ small kernels
// Routing: one warp per token.  Softmax-top-K: top-K of the logits and their
// renormalised softmax; sigmoid-group: sigmoid_group_route.
template <int NPL>
__global__ void route_kernel(const float* logits, int T, int E, int K, RouteArgs ra, int32_t* ids, float* w,
                             int32_t* ids_out, float* w_out) {
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  if (ra.family == E0_ROUTE_SIGMOID_GROUP) {
    int id;
    float wk;
    sigmoid_group_route(logits + (size_t)t * E, ra.sbias, E, K, ra.n_group, ra.topk_group, ra.scale, lane, id, wk);
    if (lane < K && id < 0) {  // NaN logits leave no id: contribute nothing through expert 0
      id = 0;
      wk = 0.f;
    }
    if (lane < K) {
      ids[t * K + lane] = id;
      w[t * K + lane] = wk;
      if (ids_out) ids_out[t * K + lane] = id;
      if (w_out) w_out[t * K + lane] = wk;
    }
    return;
  }
  float z[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    z[j] = e < E ? logits[(size_t)t * E + e] : 0.f;
  }
  int id;
  float val;
  warp_topk_regs<NPL>(z, E, K, lane, id, val);
  const float v0 = __shfl_sync(0xffffffffu, val, 0);
  float ex = lane < K ? expf(val - v0) : 0.f;
  if (lane < K && id < 0) {  // NaN logits leave no id: contribute nothing through expert 0
    id = 0;
    ex = 0.f;
  }
  const float tot = warp_sum(ex);
  if (lane < K) {
    ids[t * K + lane] = id;
    w[t * K + lane] = ex / tot;
    if (ids_out) ids_out[t * K + lane] = id;
    if (w_out) w_out[t * K + lane] = ex / tot;
  }
}

// Committed routing (decode of several tokens): one warp per token takes the given ids
// and the family's combine weights of the token's logits over them: the softmax over
// the picked logits, or scale * sigmoid / (sum + 1e-20).  An id outside [0, E) or
// repeated is reported (E0_DEV_BAD_ID) and contributes nothing through expert 0.
__global__ void route_given_kernel(const float* logits, const int32_t* given, int T, int E, int K, RouteArgs ra,
                                   int32_t* ids, float* w, int32_t* ids_out, float* w_out, uint32_t* status) {
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  int id = lane < K ? given[(size_t)t * K + lane] : -1;
  bool v = lane < K && id >= 0 && id < E;
  for (int j = 0; j < K; ++j) {
    const int o = __shfl_sync(0xffffffffu, id, j);
    if (j < lane && o == id) v = false;
  }
  if (lane < K && !v) atomicOr(status, (uint32_t)E0_DEV_BAD_ID);
  const float z = v ? logits[(size_t)t * E + id] : 0.f;
  float wk;
  if (ra.family == E0_ROUTE_SIGMOID_GROUP) {
    const float sig = v ? 1.0f / (1.0f + expf(-z)) : 0.f;
    wk = ra.scale * sig / (warp_sum(sig) + 1e-20f);
  } else {
    float mx = v ? z : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = v ? expf(z - mx) : 0.f;
    const float tot = warp_sum(ex);
    wk = tot > 0.f ? ex / tot : 0.f;
  }
  if (lane < K) {
    ids[t * K + lane] = v ? id : 0;
    w[t * K + lane] = v ? wk : 0.f;
    if (ids_out) ids_out[t * K + lane] = v ? id : -1;
    if (w_out) w_out[t * K + lane] = v ? wk : 0.f;
  }
}

// Block-wide exclusive scan of one value per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int x = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    s_warp[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  total = s_warp[31];
  const int before = warp > 0 ? s_warp[warp - 1] : 0;
  __syncthreads();
  return before + inc - v;
}

// Counting sort of the (token, k) pairs by expert; tile offsets for the grouped GEMM;
// the one-group tables (all T rows) for the shared expert and the LoRA linear.
__global__ void __launch_bounds__(1024) sort_kernel(const int32_t* ids, const float* w, int T, int K, int E,
                                                    int* row_off, int* tile_off, int* inv, int* perm, float* wrow,
                                                    int* one_row, int* one_tile) {
  __shared__ int cnt[EMAXP], cur[EMAXP];
  __shared__ int s_warp[32];
  const int P = T * K, e = threadIdx.x;
  cnt[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&cnt[ids[p]], 1);
  __syncthreads();
  const int n = e < E ? cnt[e] : 0;
  int tot_rows, tot_tiles;
  const int ro = block_excl_scan(n, s_warp, tot_rows);
  const int to = block_excl_scan((n + TT - 1) / TT, s_warp, tot_tiles);
  if (e < E) {
    row_off[e] = ro;
    tile_off[e] = to;
    cur[e] = ro;
  }
  if (e == 0) {
    row_off[E] = tot_rows;
    tile_off[E] = tot_tiles;
    one_row[0] = 0;
    one_row[1] = T;
    one_tile[0] = 0;
    one_tile[1] = (T + TT - 1) / TT;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int pos = atomicAdd(&cur[ids[p]], 1);
    inv[p] = pos;
    perm[pos] = p / K;
    wrow[pos] = w[p];
  }
}

// x = RMSNorm(h) in fp16 (reduction order permuted within groups of 8), once per
// token and once per (token, k) pair at its sorted row.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* h, int d, int K, const int* inv, __half* x16,
                                                     __half* x16s, float* xscale) {
  __shared__ float red[8];
  const int t = blockIdx.x;
  const uint16_t* ht = h + (size_t)t * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = bf16_bits_to_f32(ht[i]);
    ss += v * v;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  const float scale = rsqrtf(tot / (float)d + e0eng::RMS_EPS);
  if (threadIdx.x == 0) xscale[t] = scale;
  for (int gi = threadIdx.x; gi < d / 8; gi += blockDim.x) {
    const uint4 raw = reinterpret_cast<const uint4*>(ht)[gi];
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(u[i] << 16) * scale;
      x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u) * scale;
    }
    uint32_t o[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const __half2 h2 = __floats2half2_rn(x[jj], x[jj + 4]);
      o[jj] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<uint4*>(x16 + (size_t)t * d)[gi] = ov;
    for (int k = 0; k < K; ++k) reinterpret_cast<uint4*>(x16s + (size_t)inv[t * K + k] * d)[gi] = ov;
  }
}

// LoRA down projection v[t][q] = xscale_t * (A_q . h_t) (= A x_t, fp32): one CTA per
// token and group of four ranks, its eight warps splitting the row (one 16-byte chunk
// per lane and pass), partial sums combined in shared memory.
constexpr int LA_RANKS = 4;
__global__ void __launch_bounds__(256) lora_a_kernel(const uint16_t* h, const float* xscale, int T, int d,
                                                     const uint16_t* a, int r, float* v) {
  __shared__ float part[8][LA_RANKS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int groups = (r + LA_RANKS - 1) / LA_RANKS;
  const int t = blockIdx.x / groups, q0 = (blockIdx.x % groups) * LA_RANKS;
  float s[LA_RANKS] = {};
  const uint4* hp = reinterpret_cast<const uint4*>(h + (size_t)t * d);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    const uint4 hv = __ldg(hp + c);
    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
    for (int u = 0; u < LA_RANKS; ++u)
      if (q0 + u < r) {
        const uint4 av = __ldg(reinterpret_cast<const uint4*>(a + (size_t)(q0 + u) * d) + c);
        const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          s[u] = fmaf(__uint_as_float(aw[m] << 16), __uint_as_float(hw[m] << 16), s[u]);
          s[u] = fmaf(__uint_as_float(aw[m] & 0xFFFF0000u), __uint_as_float(hw[m] & 0xFFFF0000u), s[u]);
        }
      }
  }
#pragma unroll
  for (int u = 0; u < LA_RANKS; ++u) {
    const float w = warp_sum(s[u]);
    if (lane == 0) part[warp][u] = w;
  }
  __syncthreads();
  if (threadIdx.x < LA_RANKS && q0 + (int)threadIdx.x < r) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += part[w][threadIdx.x];
    v[(size_t)t * r + q0 + threadIdx.x] = tot * xscale[t];
  }
}

// h_out = bf16(h + sum_k y_(t,k) + y_shared + y_lora), the pairs summed in k order, with
// y_lora = W_int4 x + (alpha/r) B v (the LoRA up projection formed here from v).  A thread
// owns 4 adjacent outputs of one token (16-byte loads); the pair rows' indices are read
// first so that all K row loads are in flight together.
constexpr int CK = 16;  // K at most
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* h, int T, int d, int K, const int* inv,
                                                      const float* yslot, const float* ys, const float* yl,
                                                      const float* v, const uint16_t* bt, int r, float lscale,
                                                      uint16_t* h_out, float* delta) {
  __shared__ float vs[e0eng::RANKS_MAX];
  __shared__ int rows[CK];
  const int t = blockIdx.x;
  const int nv = v ? r : 0;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) vs[i] = v[(size_t)t * nv + i];
  if (threadIdx.x < K) rows[threadIdx.x] = inv[t * K + threadIdx.x];
  __syncthreads();
  const int i0 = 4 * (blockIdx.y * blockDim.x + threadIdx.x);
  if (i0 >= d) return;
  float4 y[CK];
#pragma unroll
  for (int k = 0; k < CK; ++k)
    if (k < K) y[k] = __ldg(reinterpret_cast<const float4*>(yslot + (size_t)rows[k] * d + i0));
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < CK; ++k)
    if (k < K) {
      s.x += y[k].x; s.y += y[k].y; s.z += y[k].z; s.w += y[k].w;
    }
  if (ys) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(ys + (size_t)t * d + i0));
    s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
  }
  if (yl) {
    float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int q = 0; q < nv; ++q) {
      const uint2 bw = __ldg(reinterpret_cast<const uint2*>(bt + (size_t)q * d + i0));
      const float vq = vs[q];
      b.x = fmaf(__uint_as_float(bw.x << 16), vq, b.x);
      b.y = fmaf(__uint_as_float(bw.x & 0xFFFF0000u), vq, b.y);
      b.z = fmaf(__uint_as_float(bw.y << 16), vq, b.z);
      b.w = fmaf(__uint_as_float(bw.y & 0xFFFF0000u), vq, b.w);
    }
    const float4 a = __ldg(reinterpret_cast<const float4*>(yl + (size_t)t * d + i0));
    s.x += a.x + lscale * b.x; s.y += a.y + lscale * b.y; s.z += a.z + lscale * b.z; s.w += a.w + lscale * b.w;
  }
  if (delta) *reinterpret_cast<float4*>(delta + (size_t)t * d + i0) = s;
  const uint2 hw = *reinterpret_cast<const uint2*>(h + (size_t)t * d + i0);
  uint2 o;
  o.x = (uint32_t)f32_to_bf16_bits(__uint_as_float(hw.x << 16) + s.x) |
        ((uint32_t)f32_to_bf16_bits(__uint_as_float(hw.x & 0xFFFF0000u) + s.y) << 16);
  o.y = (uint32_t)f32_to_bf16_bits(__uint_as_float(hw.y << 16) + s.z) |
        ((uint32_t)f32_to_bf16_bits(__uint_as_float(hw.y & 0xFFFF0000u) + s.w) << 16);
  *reinterpret_cast<uint2*>(h_out + (size_t)t * d + i0) = o;
}

// ------------------------------------------------------------------ workspace
struct PfLayout {
  size_t ids, w, row_off, tile_off, one_row, one_tile, inv, perm, wrow, xscale, x16, x16s, a16s, yslot, as16, ys, yl,
      lv, total;
};

inline size_t al(size_t x) { return (x + 255) & ~size_t(255); }

PfLayout pf_layout(int d, int E, int F, int K, int T, int out, bool shared, bool lora) {
  PfLayout L;
  const size_t P = (size_t)T * K;
  size_t o = 256;  // header (device status word at the same offset as the decode workspace)
  L.ids = o;      o = al(o + 4 * P);
  L.w = o;        o = al(o + 4 * P);
  L.row_off = o;  o = al(o + 4 * (size_t)(E + 1));
  L.tile_off = o; o = al(o + 4 * (size_t)(E + 1));
  L.one_row = o;  o = al(o + 8);
  L.one_tile = o; o = al(o + 8);
  L.inv = o;      o = al(o + 4 * P);
  L.perm = o;     o = al(o + 4 * P);
  L.wrow = o;     o = al(o + 4 * P);
  L.xscale = o;   o = al(o + 4 * (size_t)T);
  L.x16 = o;      o = al(o + 2 * (size_t)T * d);
  L.x16s = o;     o = al(o + 2 * P * d);
  L.a16s = o;     o = al(o + 2 * P * F);
  L.yslot = o;    o = al(o + 4 * P * d);
  L.as16 = o;     o = al(o + (shared ? 2 * (size_t)T * F : 0));
  L.ys = o;       o = al(o + (shared ? 4 * (size_t)T * d : 0));
  L.yl = o;       o = al(o + (lora ? 4 * (size_t)T * out : 0));
  L.lv = o;       o = al(o + (lora ? 4 * (size_t)T * e0eng::RANKS_MAX : 0));
  L.total = o;
  return L;
}

int g_num_sms = 0;
std::once_flag g_sm_once;

template <int LAYOUT, int EPI, int HK>
cudaError_t launch_gemm_hk(const GemmArgs& a, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_q4_kernel<LAYOUT, EPI, HK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)Cfg<HK>::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  gemm_q4_kernel<LAYOUT, EPI, HK><<<g_num_sms, GT, Cfg<HK>::SMEM, st>>>(a);
  return cudaGetLastError();
}

// Four k-blocks per hand-over when the reduction length allows it.  The rows layout
// always reduces over d (a multiple of 256: 4 k-blocks divide it); the column-slab layout
// reduces over F (a multiple of 128).
template <int LAYOUT, int EPI>
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  const int KB = a.K / BK;
  if constexpr (LAYOUT == E0_LAYOUT_ROWS) {
    if (KB % 4 != 0) return cudaErrorInvalidValue;
    return launch_gemm_hk<LAYOUT, EPI, 4>(a, st);
  } else {
    if (KB % 4 == 0) return launch_gemm_hk<LAYOUT, EPI, 4>(a, st);
    return launch_gemm_hk<LAYOUT, EPI, 2>(a, st);
  }
}

}  // namespace e0pf

using namespace e0pf;

namespace {
bool al16p(const void* p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

extern "C" size_t e0_prefill_workspace_size(const e0_dims* dims, int32_t T, int32_t lora_out) {
  if (!dims || T < 1) return 0;
  return pf_layout(dims->d, dims->E, dims->F, dims->K, T, lora_out > 0 ? lora_out : dims->d, true, lora_out > 0)
      .total;
}

// The grouped (tensor-core) MoE layer for T tokens: routed by the top-K of `logits`, or,
// when given_ids is set, by those committed ids with the combine weights of `logits`.
// Also the multi-token decode path of e0_moe_decode_layer.
e0_status e0pf_grouped_layer(const e0_dims* dims, const e0_experts* routed, const e0_experts* shared,
                             const e0_qlora* lora, const uint16_t* h_in, const float* logits,
                             const int32_t* given_ids, int32_t T, uint16_t* h_out, float* delta_f32,
                             int32_t* ids_out, float* weights_out, void* workspace, size_t workspace_bytes,
                             e0_stream stream) {
  E0_REQUIRE(dims && routed && h_in && logits && h_out && workspace, E0_ERR_INVALID,
             "e0_moe_prefill_layer: NULL argument");
  {
    const e0_status cs = e0::check_route(dims);
    if (cs != E0_OK) return cs;
  }
  const int d = dims->d, E = dims->E, F = dims->F, K = dims->K;
  E0_REQUIRE(T >= 1 && T <= 65536 / (K > 0 ? K : 1), E0_ERR_SHAPE, "e0_moe_prefill_layer: T * K must be <= 65536");
  E0_REQUIRE(d % 256 == 0 && d >= 256 && (2 * F) % 256 == 0 && F % 64 == 0, E0_ERR_SHAPE,
             "e0_moe_prefill_layer: d and 2F must be multiples of 256, F of 64");
  E0_REQUIRE(E >= 8 && E <= EMAXP && K >= 1 && K <= 16 && K <= E, E0_ERR_SHAPE, "e0_moe_prefill_layer: E or K");
  E0_REQUIRE(routed->gate_up.q && routed->down.q && routed->n == E, E0_ERR_INVALID,
             "e0_moe_prefill_layer: the routed stack must hold all E experts");
  E0_REQUIRE(routed->slot_of == nullptr, E0_ERR_UNSUPPORTED,
             "e0_moe_prefill_layer: slot pools are a decode feature; prefill needs every expert resident");
  const bool has_shared = shared && shared->gate_up.q;
  const bool has_lora = lora && lora->w.q;
  const int out = has_lora ? lora->out : d;
  if (has_lora) {
    E0_REQUIRE(lora->out == d, E0_ERR_SHAPE, "e0_moe_prefill_layer: the LoRA linear must be d x d");
    E0_REQUIRE(lora->r >= 0 && lora->r <= e0eng::RANKS_MAX, E0_ERR_SHAPE, "e0_moe_prefill_layer: LoRA rank must be in [0, 64]");
  }
  E0_REQUIRE(al16p(h_in) && al16p(h_out) && (!delta_f32 || al16p(delta_f32)), E0_ERR_INVALID,
             "e0_moe_prefill_layer: h_in/h_out/delta_f32 must be 16-byte aligned");
  E0_REQUIRE(!has_lora || !lora->bt || ((uintptr_t)lora->bt & 7u) == 0, E0_ERR_INVALID,
             "e0_moe_prefill_layer: the LoRA B^T matrix must be 8-byte aligned");
  E0_REQUIRE(!has_lora || !lora->a || al16p(lora->a), E0_ERR_INVALID,
             "e0_moe_prefill_layer: the LoRA A matrix must be 16-byte aligned");
  {
    // the codes are copied and the scales read with vector accesses
    auto al_q4 = [](const e0_q4& m) { return al16p(m.q) && al16p(m.scale) && al16p(m.bias); };
    E0_REQUIRE(al_q4(routed->gate_up) && al_q4(routed->down) &&
                   (!has_shared || (al_q4(shared->gate_up) && al_q4(shared->down))) && (!has_lora || al_q4(lora->w)),
               E0_ERR_INVALID, "e0_moe_prefill_layer: int4 codes, scales and biases must be 16-byte aligned");
  }
  const PfLayout L = pf_layout(d, E, F, K, T, out, true, has_lora);
  E0_REQUIRE(workspace_bytes >= L.total, E0_ERR_NOMEM, "e0_moe_prefill_layer: workspace too small");
  std::call_once(g_sm_once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  });
  E0_REQUIRE(g_num_sms > 0, E0_ERR_CUDA, "e0_moe_prefill_layer: no device");
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto P = [&](size_t off) { return ws + off; };
  int32_t* ids = (int32_t*)P(L.ids);
  float* w = (float*)P(L.w);
  int* row_off = (int*)P(L.row_off);
  int* tile_off = (int*)P(L.tile_off);
  int* one_row = (int*)P(L.one_row);
  int* one_tile = (int*)P(L.one_tile);
  int* inv = (int*)P(L.inv);
  float* xscale = (float*)P(L.xscale);
  __half* x16 = (__half*)P(L.x16);
  __half* x16s = (__half*)P(L.x16s);
  __half* a16s = (__half*)P(L.a16s);
  float* yslot = (float*)P(L.yslot);
  uint32_t* status = (uint32_t*)(ws + 4);
  E0_CHECK_CUDA(cudaMemsetAsync(ws, 0, 256, st));

  const int warps = 8;
  const int rb = (T + warps - 1) / warps;
  const RouteArgs ra{dims->route, dims->n_group, dims->topk_group, dims->route_scale, dims->score_bias};
  if (given_ids)
    route_given_kernel<<<rb, 32 * warps, 0, st>>>(logits, given_ids, T, E, K, ra, ids, w, ids_out, weights_out,
                                                  status);
  else if (E <= 256)
    route_kernel<8><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, ids_out, weights_out);
  else if (E <= 512)
    route_kernel<16><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, ids_out, weights_out);
  else
    route_kernel<32><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, ids_out, weights_out);
  E0_CHECK_CUDA(cudaGetLastError());
  sort_kernel<<<1, 1024, 0, st>>>(ids, w, T, K, E, row_off, tile_off, inv, (int*)P(L.perm), (float*)P(L.wrow), one_row,
                                  one_tile);
  E0_CHECK_CUDA(cudaGetLastError());
  gather_kernel<<<T, 256, 0, st>>>(h_in, d, K, inv, x16, x16s, xscale);
  E0_CHECK_CUDA(cudaGetLastError());

  const uint64_t timeout = 2000000000ull;
  GemmArgs g{};
  g.status = status;
  g.timeout_ns = timeout;
  // routed gate/up -> a, with the shared expert as one more group (its tiles share the
  // launch): its rows are the T token rows x16, its output as16
  float* ys = has_shared ? (float*)P(L.ys) : nullptr;
  __half* as16 = has_shared ? (__half*)P(L.as16) : nullptr;
  g.A = x16s; g.lda = d; g.K = d; g.N = 2 * F; g.ngroups = E; g.row_off = row_off; g.tile_off = tile_off;
  g.q = routed->gate_up.q; g.s = routed->gate_up.scale; g.b = routed->gate_up.bias;
  g.out16 = a16s; g.ldo = F; g.out32 = nullptr; g.rowscale = nullptr;
  g.xrows = has_shared ? T : 0;
  if (has_shared) {
    g.A2 = x16; g.q2 = shared->gate_up.q; g.s2 = shared->gate_up.scale; g.b2 = shared->gate_up.bias;
    g.out16b = as16; g.out32b = nullptr;
  }
  E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_ROWS, EPI_SWIGLU>(g, st)));
  // routed down x w -> y per pair; the shared expert's down projection -> ys
  g.A = a16s; g.lda = F; g.K = F; g.N = d;
  g.q = routed->down.q; g.s = routed->down.scale; g.b = routed->down.bias;
  g.out16 = nullptr; g.out32 = yslot; g.ldo = d; g.rowscale = (const float*)P(L.wrow);
  if (has_shared) {
    g.A2 = as16; g.q2 = shared->down.q; g.s2 = shared->down.scale; g.b2 = shared->down.bias;
    g.out16b = nullptr; g.out32b = ys;
  }
  E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_COLSLAB, EPI_F32>(g, st)));
  g.xrows = 0;
  float* yl = nullptr;
  float* lv = nullptr;
  if (has_lora) {
    yl = (float*)P(L.yl);
    g.A = x16; g.lda = d; g.K = d; g.N = out; g.ngroups = 1; g.row_off = one_row; g.tile_off = one_tile;
    g.q = lora->w.q; g.s = lora->w.scale; g.b = lora->w.bias;
    g.out16 = nullptr; g.out32 = yl; g.ldo = out; g.rowscale = nullptr;
    E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_ROWS, EPI_F32>(g, st)));
    if (lora->r > 0 && lora->a && lora->bt) {
      lv = (float*)P(L.lv);
      lora_a_kernel<<<T * ((lora->r + LA_RANKS - 1) / LA_RANKS), 256, 0, st>>>(h_in, xscale, T, d, lora->a, lora->r,
                                                                                 lv);
      E0_CHECK_CUDA(cudaGetLastError());
    }
  }
  const dim3 cgrid(T, (d / 4 + 255) / 256);
  combine_kernel<<<cgrid, 256, 0, st>>>(h_in, T, d, K, inv, yslot, ys, yl, lv, lv ? lora->bt : nullptr,
                                        lv ? lora->r : 0, lv ? lora->alpha / lora->r : 0.f, h_out, delta_f32);
  E0_CHECK_CUDA(cudaGetLastError());
  return E0_OK;
}

extern "C" e0_status e0_moe_prefill_layer(const e0_dims* dims, const e0_experts* routed, const e0_experts* shared,
                                          const e0_qlora* lora, const uint16_t* h_in, const float* logits,
                                          int32_t T, uint16_t* h_out, float* delta_f32, int32_t* ids_out,
                                          float* weights_out, void* workspace, size_t workspace_bytes,
                                          e0_stream stream) {
  return e0pf_grouped_layer(dims, routed, shared, lora, h_in, logits, nullptr, T, h_out, delta_f32, ids_out,
                            weights_out, workspace, workspace_bytes, stream);
}

// Top-K routing of T tokens' logits by the family (one warp per token), for the other
// translation units.
cudaError_t e0pf_route_topk(const float* logits, int T, int E, int K, const RouteArgs& ra, int32_t* ids, float* w,
                            cudaStream_t st) {
  const int warps = 8, rb = (T + warps - 1) / warps;
  if (E <= 256)
    route_kernel<8><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, nullptr, nullptr);
  else if (E <= 512)
    route_kernel<16><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, nullptr, nullptr);
  else
    route_kernel<32><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ra, ids, w, nullptr, nullptr);
  return cudaGetLastError();
}
