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
//   gemm_q4    grouped GEMM, int4 weights dequantised to fp16 in shared memory, tcgen05.mma
//              with the fp32 accumulator in tensor memory:
//                gate/up  [rows_e x d] x [d x 2F]  -> SwiGLU epilogue -> fp16 a [rows_e x F]
//                down     [rows_e x F] x [F x d]   -> x w_(t,k)        -> fp32 y per pair
//              the shared expert and the LoRA base run through the same kernel as one group
//   lora_ab    (alpha/r) B (A x) per token on the CUDA cores (r = 16: too thin for a tile)
//   combine    h_out = bf16(h + sum_k y_(t,k) + y_shared + y_lora), sum over k in k order
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

constexpr int BM = 128, BN = 256, BK = 64;  // tile: rows x output columns x reduction block
constexpr int GT = 512;                      // threads per GEMM CTA: two per B row
constexpr int STAGES = 5;                    // raw (A tile + packed B) stages in flight
constexpr int LOOK = STAGES - 2;             // k-blocks loaded ahead
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int BQ_BYTES = BN * BK / 2;        // 8 KB of int4 codes
constexpr int RAW_BYTES = A_BYTES + BQ_BYTES;
constexpr int BD_BYTES = BN * BK * 2;        // 32 KB of dequantised fp16 B
constexpr int EMAXP = 1024;
constexpr size_t GEMM_SMEM = 1024 + (size_t)STAGES * RAW_BYTES + 2 * BD_BYTES + 2 * (EMAXP + 1) * sizeof(int);
static_assert(RAW_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
static_assert(GEMM_SMEM <= 227 * 1024, "shared memory");

enum Epi : int { EPI_SWIGLU = 0, EPI_F32 = 1 };

struct GemmArgs {
  const __half* A;        // [rows][K] fp16, reduction index permuted within groups of 8
  int lda;
  int K, N;               // reduction length (multiple of 64), outputs per group (multiple of 256)
  int ngroups;
  const int* row_off;     // [ngroups + 1] rows of group g: [row_off[g], row_off[g + 1])
  const int* tile_off;    // [ngroups + 1] prefix sums of ceil(rows_g / BM)
  const uint32_t* q;      // int4 codes of all groups (group g = weight slot g)
  const uint16_t* s;      // bf16 scales
  const uint16_t* b;      // bf16 biases
  __half* out16;          // EPI_SWIGLU: [rows][N / 2] fp16, permuted within groups of 8
  float* out32;           // EPI_F32: [rows][N]
  int ldo;
  const float* rowscale;  // EPI_F32: factor per row (nullable)
  uint32_t* status;
  uint64_t timeout_ns;
};

// Bounded wait on an mbarrier phase; false (and a device status bit) if it runs out.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const GemmArgs& g) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && globaltimer() - t0 > g.timeout_ns) {
      atomicOr(g.status, (uint32_t)E0_DEV_TIMEOUT);
      return false;
    }
  }
}

struct Tile {
  int m0, rows, n0, slot;
};

// Dequantise half of a 64-code row segment (one uint4 = 32 codes, chunks 4h .. 4h + 3
// of the row) into the swizzled fp16 row.
__device__ __forceinline__ void dequant_half_row(const uint8_t* codes, uint8_t* dst_row, int n, int h, __half2 s2,
                                                 __half2 b2) {
  const uint4 w0 = *reinterpret_cast<const uint4*>(codes);
  const uint32_t words[4] = {w0.x, w0.y, w0.z, w0.w};
  const __half2 magic = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
#pragma unroll
  for (int mm = 0; mm < 4; ++mm) {
    const int m = 4 * h + mm;
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // codes j and j + 4 of this word as fp16 (1024 + c), then exactly c, then s*c + b
      const uint32_t t = ((words[mm] >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
      __half2 c = *reinterpret_cast<const __half2*>(&t);
      c = __hsub2(c, magic);
      const __half2 w = __hfma2(c, s2, b2);
      out[j] = *reinterpret_cast<const uint32_t*>(&w);
    }
    *reinterpret_cast<uint4*>(dst_row + ((m ^ (n & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__device__ __forceinline__ __half2 bf16pair_to_h2(uint16_t v) {
  const __half h = __float2half_rn(__uint_as_float((uint32_t)v << 16));
  return __halves2half2(h, h);
}

template <int LAYOUT, int EPI>
__global__ void __launch_bounds__(GT, 1) gemm_q4_kernel(const __grid_constant__ GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  uint8_t* raw = sm;                               // STAGES x [A tile | packed B]
  uint8_t* bdq = sm + (size_t)STAGES * RAW_BYTES;  // 2 x dequantised B
  int* s_row = reinterpret_cast<int*>(bdq + 2 * BD_BYTES);
  int* s_tile = s_row + (EMAXP + 1);
  __shared__ __align__(8) uint64_t mma_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NT = g.N / BN, KB = g.K / BK;

  for (int i = tid; i <= g.ngroups; i += GT) {
    s_row[i] = g.row_off[i];
    s_tile[i] = g.tile_off[i];
  }
  if (tid == 0) {
    mbar_init(&mma_bar[0], 1);
    mbar_init(&mma_bar[1], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_slot, BN);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const int total = s_tile[g.ngroups] * NT;
  const int my_tiles = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int jobs = my_tiles * KB;

  // tile i of this CTA -> rows, output columns and weight slot (group search in shared memory)
  auto tile_of = [&](int i) -> Tile {
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    int lo = 0, hi = g.ngroups;  // s_tile[lo] * NT <= t < s_tile[hi] * NT
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile[mid] * NT <= t) lo = mid; else hi = mid;
    }
    const int mt_g = s_tile[lo + 1] - s_tile[lo];
    const int local = t - s_tile[lo] * NT;
    Tile T;
    T.m0 = s_row[lo] + (local % mt_g) * BM;
    T.rows = min(BM, s_row[lo + 1] - T.m0);
    T.n0 = (local / mt_g) * BN;
    T.slot = lo;
    return T;
  };

  // all threads: issue the copies of job j (tile j / KB, k-block j % KB) into its stage
  int ld_i = -1;  // tile the loader decoded last
  Tile ld_T{};
  auto load_job = [&](int j) {
    if (j < jobs) {
      if (j / KB != ld_i) {
        ld_i = j / KB;
        ld_T = tile_of(ld_i);
      }
      const Tile T = ld_T;
      const int kb = j % KB;
      uint8_t* sA = raw + (size_t)(j % STAGES) * RAW_BYTES;
      uint8_t* sBq = sA + A_BYTES;
      // rows past the group's end are not loaded: they only feed accumulator rows that
      // the epilogue discards
      for (int c = tid; c < T.rows * 8; c += GT) {
        const int r = c >> 3, ch = c & 7;
        const __half* src = g.A + (size_t)(T.m0 + r) * g.lda + kb * BK + ch * 8;
        cp_async16(sA + r * 128 + ((ch ^ (r & 7)) << 4), src, 16u);
      }
#pragma unroll
      for (int c = tid; c < BN * 2; c += GT) {
        const int n = c >> 1, h = c & 1;
        const uint32_t* src;
        if (LAYOUT == E0_LAYOUT_ROWS)
          src = g.q + ((size_t)T.slot * g.N + T.n0 + n) * (g.K / 8) + kb * 8 + h * 4;
        else
          src = g.q + ((size_t)T.slot * (g.K / 32) + 2 * kb + h) * (size_t)g.N * 4 + (size_t)(T.n0 + n) * 4;
        cp_async16(sBq + n * 32 + h * 16, src, 16u);
      }
    }
    cp_async_commit();
  };

  // scale and bias of row (tid) of the B tile, loaded 8 k-blocks ahead
  uint16_t cs[8], cb[8], ns[8], nb[8];
  auto load_sb = [&](int j, uint16_t (&ds)[8], uint16_t (&db)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) ds[u] = db[u] = 0;
    if (j >= jobs) return;
    const Tile T = tile_of(j / KB);
    const int kb0 = j % KB;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int kb = kb0 + u;
      if (kb < KB) {
        size_t idx;
        if (LAYOUT == E0_LAYOUT_ROWS)
          idx = ((size_t)T.slot * g.N + T.n0 + (tid >> 1)) * (g.K / 64) + kb;
        else
          idx = ((size_t)T.slot * (g.K / 64) + kb) * g.N + T.n0 + (tid >> 1);
        ds[u] = __ldg(g.s + idx);
        db[u] = __ldg(g.b + idx);
      }
    }
  };

  const uint32_t idesc = idesc_f16_f32(BM, BN);
  for (int j = 0; j < LOOK; ++j) load_job(j);
  // Scales and biases come in chunks of up to 8 k-blocks of one tile; the next chunk
  // is loaded while the current one is in use.
  load_sb(0, ns, nb);

  for (int j = 0; j < jobs; ++j) {
    const int kb = j % KB;
    // 1. the tensor core is done with job j - 2: its dequantised B buffer and raw stage are free
    if (j >= 2 && !wait_bar(&mma_bar[j & 1], ((j >> 1) - 1) & 1, g)) s_abort = 1;
    // 2. copies of job j + LOOK into the stage job j - 2 used
    load_job(j + LOOK);
    // 3. job j's copies have landed (this thread's), and are visible to the tensor core
    cp_async_wait<LOOK>();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (s_abort) break;
    // 4. scales of this k-block
    if ((kb & 7) == 0) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        cs[u] = ns[u];
        cb[u] = nb[u];
      }
      load_sb(kb + 8 < KB ? j + 8 : (j / KB + 1) * KB, ns, nb);
    }
    // 5. dequantise this thread's B row into the swizzled fp16 buffer
    {
      const int u = kb & 7;
      uint16_t sv = 0, bv = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q == u) {
          sv = cs[q];
          bv = cb[q];
        }
      const int n = tid >> 1, h = tid & 1;
      const uint8_t* codes = raw + (size_t)(j % STAGES) * RAW_BYTES + A_BYTES + n * 32 + h * 16;
      dequant_half_row(codes, bdq + (size_t)(j & 1) * BD_BYTES + n * 128, n, h, bf16pair_to_h2(sv), bf16pair_to_h2(bv));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    fence_before_sync();
    __syncthreads();
    // 6. one thread issues the four K=16 steps of this k-block and commits them
    if (tid == 0) {
      fence_after_sync();
      const uint32_t a_addr = smem_u32(raw + (size_t)(j % STAGES) * RAW_BYTES);
      const uint32_t b_addr = smem_u32(bdq + (size_t)(j & 1) * BD_BYTES);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_f16(tmem, sdesc_k128(a_addr + 32 * kk), sdesc_k128(b_addr + 32 * kk), idesc, kb > 0 || kk > 0);
      commit(&mma_bar[j & 1]);
    }
    // 7. last k-block of a tile: epilogue from tensor memory
    if (kb == KB - 1) {
      const bool done = wait_bar(&mma_bar[j & 1], (j >> 1) & 1, g);
      fence_after_sync();
      const Tile T = tile_of(j / KB);
      const int quad = warp & 3, cblk = warp >> 2;  // lanes 32 quad.., columns 64 cblk..
      const int r = quad * 32 + lane;
      const bool row_ok = done && r < T.rows;
#pragma unroll 1
      for (int c0 = 0; c0 < BN / 4; c0 += 32) {
        const int col = cblk * (BN / 4) + c0;
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)col, v);
        if (!row_ok) continue;
        if (EPI == EPI_SWIGLU) {
          // columns 2i / 2i + 1 are gate / up of output (n0 + col) / 2 + i
          float a[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gt = __uint_as_float(v[2 * i]), up = __uint_as_float(v[2 * i + 1]);
            a[i] = __fdividef(gt, 1.0f + __expf(-gt)) * up;
          }
          __half* dst = g.out16 + (size_t)(T.m0 + r) * g.ldo + (T.n0 + col) / 2;
#pragma unroll
          for (int grp = 0; grp < 2; ++grp) {
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const __half2 h2 = __floats2half2_rn(a[8 * grp + jj], a[8 * grp + jj + 4]);
              w[jj] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + 8 * grp) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          const float f = g.rowscale ? g.rowscale[T.m0 + r] : 1.0f;
          float* dst = g.out32 + (size_t)(T.m0 + r) * g.ldo + T.n0 + col;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                make_float4(f * __uint_as_float(v[i]), f * __uint_as_float(v[i + 1]), f * __uint_as_float(v[i + 2]),
                            f * __uint_as_float(v[i + 3]));
        }
      }
      if (!done) s_abort = 1;
      fence_before_sync();
      __syncthreads();
      if (s_abort) break;
    }
  }
  cp_async_wait<0>();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BN);
}

// ------------------------------------------------------------------ small kernels
// Routing: one warp per token, top-K of the logits and their renormalised softmax.
template <int NPL>
__global__ void route_kernel(const float* logits, int T, int E, int K, int32_t* ids, float* w, int32_t* ids_out,
                             float* w_out) {
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
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
  const int to = block_excl_scan((n + BM - 1) / BM, s_warp, tot_tiles);
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
    one_tile[1] = (T + BM - 1) / BM;
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

// (alpha/r) B (A x) added to the LoRA base output of each token (fp32 x).
__global__ void __launch_bounds__(256) lora_ab_kernel(const uint16_t* h, const float* xscale, int d, int out,
                                                      const uint16_t* a, const uint16_t* bt, int r, float lscale,
                                                      float* yl) {
  __shared__ float v[e0eng::RANKS_MAX];
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* ht = h + (size_t)t * d;
  const float sc = xscale[t];
  for (int q = warp; q < r; q += blockDim.x >> 5) {
    float s = 0.f;
    for (int i = lane; i < d; i += 32) s += bf16_bits_to_f32(a[(size_t)q * d + i]) * bf16_bits_to_f32(ht[i]);
    s = warp_sum(s);
    if (lane == 0) v[q] = s * sc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < out; i += blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < r; ++q) s += bf16_bits_to_f32(bt[(size_t)q * out + i]) * v[q];
    yl[(size_t)t * out + i] += lscale * s;
  }
}

// h_out = bf16(h + sum_k y_(t,k) + y_shared + y_lora), the pairs summed in k order.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* h, int d, int K, const int* inv,
                                                      const float* yslot, const float* ys, const float* yl,
                                                      uint16_t* h_out, float* delta) {
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < K; ++k) s += yslot[(size_t)inv[t * K + k] * d + i];
    if (ys) s += ys[(size_t)t * d + i];
    if (yl) s += yl[(size_t)t * d + i];
    if (delta) delta[(size_t)t * d + i] = s;
    h_out[(size_t)t * d + i] = f32_to_bf16_bits(bf16_bits_to_f32(h[(size_t)t * d + i]) + s);
  }
}

// ------------------------------------------------------------------ workspace
struct PfLayout {
  size_t ids, w, row_off, tile_off, one_row, one_tile, inv, perm, wrow, xscale, x16, x16s, a16s, yslot, as16, ys, yl,
      total;
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
  L.total = o;
  return L;
}

int g_num_sms = 0;
std::once_flag g_sm_once;

template <int LAYOUT, int EPI>
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_q4_kernel<LAYOUT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)GEMM_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  gemm_q4_kernel<LAYOUT, EPI><<<g_num_sms, GT, GEMM_SMEM, st>>>(a);
  return cudaGetLastError();
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

extern "C" e0_status e0_moe_prefill_layer(const e0_dims* dims, const e0_experts* routed, const e0_experts* shared,
                                          const e0_qlora* lora, const uint16_t* h_in, const float* logits,
                                          int32_t T, uint16_t* h_out, float* delta_f32, int32_t* ids_out,
                                          float* weights_out, void* workspace, size_t workspace_bytes,
                                          e0_stream stream) {
  E0_REQUIRE(dims && routed && h_in && logits && h_out && workspace, E0_ERR_INVALID,
             "e0_moe_prefill_layer: NULL argument");
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
  E0_REQUIRE(al16p(h_in) && al16p(h_out), E0_ERR_INVALID, "e0_moe_prefill_layer: h_in/h_out must be 16-byte aligned");
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
  if (E <= 256)
    route_kernel<8><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ids, w, ids_out, weights_out);
  else if (E <= 512)
    route_kernel<16><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ids, w, ids_out, weights_out);
  else
    route_kernel<32><<<rb, 32 * warps, 0, st>>>(logits, T, E, K, ids, w, ids_out, weights_out);
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
  // routed gate/up -> a
  g.A = x16s; g.lda = d; g.K = d; g.N = 2 * F; g.ngroups = E; g.row_off = row_off; g.tile_off = tile_off;
  g.q = routed->gate_up.q; g.s = routed->gate_up.scale; g.b = routed->gate_up.bias;
  g.out16 = a16s; g.ldo = F; g.out32 = nullptr; g.rowscale = nullptr;
  E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_ROWS, EPI_SWIGLU>(g, st)));
  // routed down x w -> y per pair
  g.A = a16s; g.lda = F; g.K = F; g.N = d;
  g.q = routed->down.q; g.s = routed->down.scale; g.b = routed->down.bias;
  g.out16 = nullptr; g.out32 = yslot; g.ldo = d; g.rowscale = (const float*)P(L.wrow);
  E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_COLSLAB, EPI_F32>(g, st)));
  float* ys = nullptr;
  if (has_shared) {
    __half* as16 = (__half*)P(L.as16);
    ys = (float*)P(L.ys);
    g.A = x16; g.lda = d; g.K = d; g.N = 2 * F; g.ngroups = 1; g.row_off = one_row; g.tile_off = one_tile;
    g.q = shared->gate_up.q; g.s = shared->gate_up.scale; g.b = shared->gate_up.bias;
    g.out16 = as16; g.ldo = F; g.out32 = nullptr; g.rowscale = nullptr;
    E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_ROWS, EPI_SWIGLU>(g, st)));
    g.A = as16; g.lda = F; g.K = F; g.N = d;
    g.q = shared->down.q; g.s = shared->down.scale; g.b = shared->down.bias;
    g.out16 = nullptr; g.out32 = ys; g.ldo = d;
    E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_COLSLAB, EPI_F32>(g, st)));
  }
  float* yl = nullptr;
  if (has_lora) {
    yl = (float*)P(L.yl);
    g.A = x16; g.lda = d; g.K = d; g.N = out; g.ngroups = 1; g.row_off = one_row; g.tile_off = one_tile;
    g.q = lora->w.q; g.s = lora->w.scale; g.b = lora->w.bias;
    g.out16 = nullptr; g.out32 = yl; g.ldo = out; g.rowscale = nullptr;
    E0_CHECK_CUDA((launch_gemm<E0_LAYOUT_ROWS, EPI_F32>(g, st)));
    if (lora->r > 0 && lora->a && lora->bt) {
      lora_ab_kernel<<<T, 256, 0, st>>>(h_in, xscale, d, out, lora->a, lora->bt, lora->r, lora->alpha / lora->r, yl);
      E0_CHECK_CUDA(cudaGetLastError());
    }
  }
  combine_kernel<<<T, 256, 0, st>>>(h_in, d, K, inv, yslot, ys, yl, h_out, delta_f32);
  E0_CHECK_CUDA(cudaGetLastError());
  return E0_OK;
}
