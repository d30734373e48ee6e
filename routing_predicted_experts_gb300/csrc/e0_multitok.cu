// Several decode tokens through one layer-step (T = 2..16): every weight is read once
// for all the tokens.
//
// "The Other Half of the Memory Wall" (Edge0): the layer-step of §3.1 and the head of
// §3.2 are per token; §6 "Limitations" leaves batching to the serving layer.  Batching
// T tokens changes only how often each weight byte is read: the routed experts run on
// the grouped tensor-core path (e0pf_grouped_layer: each expert picked by any of the
// tokens is read once, for all of them), and the prerouter head runs here:
//   norm      x_t = h_t / rms(h_t): the per-token factor                (one warp per token)
//   rows      fc1 hidden rows and the linear-residual rows, each row read once and dotted
//             with all T tokens' hidden states held in shared memory
//   fc2       per 32 fc1 rows: erf-GELU of (fc1 + b1 + the one-hot columns picked by each
//             token's current and previous ids), then their fc2 rows into the logits
//   route     the family's top-K of each token's logits (the next layer's routing)
// fp32 accumulation throughout, bf16 weights, as in the single-token engine.
#include <algorithm>

#include "e0_engine.cuh"

using namespace e0dev;

namespace e0mt {

constexpr int TMAX = 16;        // tokens per call
constexpr int ROWS_WARPS = 8;   // warps per CTA of rows_kernel
constexpr int FC2_ROWS = 16;    // fc1 rows per CTA of fc2_kernel

__device__ __forceinline__ float bflo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bfhi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
__device__ __forceinline__ float gelu_erf(float u) { return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f)); }

// RMSNorm factor of each token's hidden state (unit gain, eps 1e-6).
__global__ void norm_kernel(const uint16_t* h, int d, int T, float* sc) {
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  float ss = 0.f;
  const uint4* hp = reinterpret_cast<const uint4*>(h + (size_t)t * d);  // d is a multiple of 256
  for (int c = lane; c < d / 8; c += 32) {
    const uint4 v = hp[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float a = bflo(w[m]), b = bfhi(w[m]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) sc[t] = rsqrtf(ss / (float)d + e0eng::RMS_EPS);
}

__device__ __forceinline__ float dot8(const uint4 w, const uint4 x) {
  float a = bflo(w.x) * bflo(x.x);
  a = fmaf(bfhi(w.x), bfhi(x.x), a);
  a = fmaf(bflo(w.y), bflo(x.y), a);
  a = fmaf(bfhi(w.y), bfhi(x.y), a);
  a = fmaf(bflo(w.z), bflo(x.z), a);
  a = fmaf(bfhi(w.z), bfhi(x.z), a);
  a = fmaf(bflo(w.w), bflo(x.w), a);
  return fmaf(bfhi(w.w), bfhi(x.w), a);
}

// Rows r < H of fc1's hidden block and rows H + e of the linear residual, against TP
// token slots (tokens T..TP-1 are zero).  A warp takes one row at a time; lane L owns
// the 8 columns 8 L + 256 j, so a row is read with 16-byte loads, once.
//   u[t][r] = x_t . W1h[r];   z[t][e] = x_t . Lres[e] + b2[e] + bias[e]
template <int TP>
__global__ void __launch_bounds__(32 * ROWS_WARPS) rows_kernel(const uint16_t* h, int d, int T, const float* sc,
                                                               const uint16_t* w1h, int H, const uint16_t* lres,
                                                               int E, const uint16_t* b2, const float* bias,
                                                               float* u, float* z) {
  extern __shared__ __align__(16) uint16_t hs[];  // [TP][d]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n16 = d / 8;  // 16-byte chunks of a row
  for (int i = threadIdx.x; i < TP * n16; i += blockDim.x) {
    const int t = i / n16, c = i % n16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t < T) v = reinterpret_cast<const uint4*>(h + (size_t)t * d)[c];
    reinterpret_cast<uint4*>(hs + (size_t)t * d)[c] = v;
  }
  __syncthreads();
  const int R = H + E;
  const int nchunks = d / 256;
  for (int r = blockIdx.x * ROWS_WARPS + warp; r < R; r += gridDim.x * ROWS_WARPS) {
    const uint16_t* w0 = r < H ? w1h + (size_t)r * d : lres + (size_t)(r - H) * d;
    float a0[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) a0[t] = 0.f;
    for (int j = 0; j < nchunks; ++j) {
      const int c = lane + 32 * j;  // 16-byte chunk index
      const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(w0) + c);
#pragma unroll
      for (int t = 0; t < TP; ++t) a0[t] += dot8(q0, reinterpret_cast<const uint4*>(hs + (size_t)t * d)[c]);
    }
#pragma unroll
    for (int t = 0; t < TP; ++t) a0[t] = warp_sum(a0[t]);
    if (lane == 0) {
      for (int t = 0; t < T; ++t) {
        const float v = a0[t] * sc[t];
        if (r < H) {
          u[(size_t)t * H + r] = v;
        } else {
          const int e = r - H;
          z[(size_t)t * E + e] = v + (b2 ? bf(b2[e]) : 0.f) + (bias ? bias[e] : 0.f);
        }
      }
    }
  }
}

// Whether ids[k] is a valid one-hot entry: in range and not repeated earlier in the row.
__device__ __forceinline__ bool onehot_valid(const int32_t* ids, int k, int E) {
  const int id = ids[k];
  if (id < 0 || id >= E) return false;
  for (int j = 0; j < k; ++j)
    if (ids[j] == id) return false;
  return true;
}

// fc1 rows [i0, i0 + 32) of every token: erf-GELU of the hidden-block dot + b1 + the
// one-hot columns of the token's current and previous ids; then those rows of fc2
// (stored transposed, [H][E]) added into every token's logits.
template <int TP>
__global__ void __launch_bounds__(256) fc2_kernel(const float* u, int T, int H, int E, int K, const uint16_t* b1,
                                                  const uint16_t* w1c_t, const uint16_t* w1p_t, const int32_t* ids,
                                                  const int32_t* prev, const uint16_t* w2t, float* z,
                                                  uint32_t* status) {
  __shared__ float p[TP][FC2_ROWS];
  const int i0 = blockIdx.x * FC2_ROWS;
  for (int idx = threadIdx.x; idx < TP * FC2_ROWS; idx += blockDim.x) {
    const int t = idx / FC2_ROWS, i = idx % FC2_ROWS, r = i0 + i;
    float v = 0.f;
    if (t < T && r < H) {
      v = u[(size_t)t * H + r] + (b1 ? bf(b1[r]) : 0.f);
      const int32_t* ct = ids + (size_t)t * K;
      for (int k = 0; k < K; ++k) {
        if (onehot_valid(ct, k, E))
          v += bf(w1c_t[(size_t)ct[k] * H + r]);
        else if (status && i == 0 && ct[k] != -1)
          atomicOr(status, (uint32_t)E0_DEV_BAD_ID);
      }
      if (prev) {
        const int32_t* pt = prev + (size_t)t * K;
        for (int k = 0; k < K; ++k) {
          if (onehot_valid(pt, k, E))
            v += bf(w1p_t[(size_t)pt[k] * H + r]);
          else if (status && i == 0 && pt[k] != -1)
            atomicOr(status, (uint32_t)E0_DEV_BAD_ID);
        }
      }
      v = gelu_erf(v);
    }
    p[t][i] = v;
  }
  __syncthreads();
  const int nr = min(FC2_ROWS, H - i0);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) acc[t] = 0.f;
    for (int i = 0; i < nr; ++i) {
      const float w = bf(w2t[(size_t)(i0 + i) * E + e]);
#pragma unroll
      for (int t = 0; t < TP; ++t) acc[t] = fmaf(w, p[t][i], acc[t]);
    }
    for (int t = 0; t < T; ++t) atomicAdd(z + (size_t)t * E + e, acc[t]);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Scratch {
  float* sc;
  float* u;
  float* z;
  int32_t* ids;
  float* w;
  size_t total;
};

Scratch scratch_layout(uint8_t* base, int T, int H, int E, int K) {
  Scratch s{};
  size_t o = 0;
  s.sc = reinterpret_cast<float*>(base + o);   o = align256(o + sizeof(float) * T);
  s.u = reinterpret_cast<float*>(base + o);    o = align256(o + sizeof(float) * (size_t)T * std::max(H, 1));
  s.z = reinterpret_cast<float*>(base + o);    o = align256(o + sizeof(float) * (size_t)T * E);
  s.ids = reinterpret_cast<int32_t*>(base + o); o = align256(o + sizeof(int32_t) * (size_t)T * K);
  s.w = reinterpret_cast<float*>(base + o);    o = align256(o + sizeof(float) * (size_t)T * K);
  s.total = o;
  return s;
}

template <int TP>
cudaError_t launch_rows(const uint16_t* h, int d, int T, const float* sc, const e0_prerouter* hd, int E,
                        const float* bias, float* u, float* z, cudaStream_t st) {
  const size_t smem = (size_t)TP * d * sizeof(uint16_t);
  cudaError_t e = cudaFuncSetAttribute(rows_kernel<TP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (hd->H + E + ROWS_WARPS - 1) / ROWS_WARPS;
  rows_kernel<TP><<<grid, 32 * ROWS_WARPS, smem, st>>>(h, d, T, sc, hd->w1h, hd->H, hd->lres, E, hd->b2, bias, u,
                                                       z);
  return cudaGetLastError();
}

template <int TP>
cudaError_t launch_fc2(const float* u, int T, int H, int E, int K, const e0_prerouter* hd, const int32_t* ids,
                       const int32_t* prev, float* z, uint32_t* status, cudaStream_t st) {
  fc2_kernel<TP><<<(H + FC2_ROWS - 1) / FC2_ROWS, 256, 0, st>>>(u, T, H, E, K, hd->b1, hd->w1c_t, hd->w1p_t, ids, prev,
                                                               hd->w2t, z, status);
  return cudaGetLastError();
}

}  // namespace e0mt

using namespace e0mt;

size_t e0mt_head_scratch(const e0_dims* dims, int32_t T, int32_t H) {
  return scratch_layout(nullptr, T, H, dims->E, dims->K).total;
}

// The prerouter head for T tokens (2 <= T <= 16): next-layer logits and routing.
// scratch: device memory of e0mt_head_scratch bytes (256-byte aligned); status: the
// device status word that invalid one-hot ids are reported in.
e0_status e0mt_head(const e0_prerouter* hd, const e0_dims* dims, const uint16_t* h, const int32_t* ids_cur,
                    const int32_t* ids_prev, int32_t T, const float* logit_bias, float* logits_out,
                    int32_t* ids_out, float* weights_out, void* scratch, size_t scratch_bytes, uint32_t* status,
                    e0_stream stream) {
  E0_REQUIRE(hd && hd->lres && h, E0_ERR_INVALID, "multi-token head: NULL argument");
  E0_REQUIRE(T >= 1 && T <= TMAX, E0_ERR_SHAPE, "multi-token head: T must be in [1, 16]");
  E0_REQUIRE(hd->H == 0 || ids_cur, E0_ERR_INVALID, "a head with an MLP needs the current ids");
  const int d = dims->d, E = dims->E, K = dims->K, H = hd->H;
  E0_REQUIRE(d % 256 == 0, E0_ERR_SHAPE, "multi-token head: d must be a multiple of 256");
  E0_REQUIRE(((uintptr_t)h & 15u) == 0 && ((uintptr_t)hd->lres & 15u) == 0 && (H == 0 || ((uintptr_t)hd->w1h & 15u) == 0),
             E0_ERR_INVALID, "multi-token head: hidden states and weight rows must be 16-byte aligned");
  Scratch s = scratch_layout(static_cast<uint8_t*>(scratch), T, H, E, K);
  E0_REQUIRE(scratch && ((uintptr_t)scratch & 255u) == 0 && scratch_bytes >= s.total, E0_ERR_NOMEM,
             "multi-token head: scratch too small (e0_decode_workspace_size)");
  cudaStream_t st = (cudaStream_t)stream;
  float* z = logits_out ? logits_out : s.z;
  int32_t* ids = ids_out ? ids_out : s.ids;
  float* w = weights_out ? weights_out : s.w;
  norm_kernel<<<(T + 7) / 8, 256, 0, st>>>(h, d, T, s.sc);
  E0_CHECK_CUDA(cudaGetLastError());
  const int TP = T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
  switch (TP) {
    case 2: E0_CHECK_CUDA(launch_rows<2>(h, d, T, s.sc, hd, E, logit_bias, s.u, z, st)); break;
    case 4: E0_CHECK_CUDA(launch_rows<4>(h, d, T, s.sc, hd, E, logit_bias, s.u, z, st)); break;
    case 8: E0_CHECK_CUDA(launch_rows<8>(h, d, T, s.sc, hd, E, logit_bias, s.u, z, st)); break;
    default: E0_CHECK_CUDA(launch_rows<16>(h, d, T, s.sc, hd, E, logit_bias, s.u, z, st)); break;
  }
  if (H > 0) {
    switch (TP) {
      case 2: E0_CHECK_CUDA(launch_fc2<2>(s.u, T, H, E, K, hd, ids_cur, ids_prev, z, status, st)); break;
      case 4: E0_CHECK_CUDA(launch_fc2<4>(s.u, T, H, E, K, hd, ids_cur, ids_prev, z, status, st)); break;
      case 8: E0_CHECK_CUDA(launch_fc2<8>(s.u, T, H, E, K, hd, ids_cur, ids_prev, z, status, st)); break;
      default: E0_CHECK_CUDA(launch_fc2<16>(s.u, T, H, E, K, hd, ids_cur, ids_prev, z, status, st)); break;
    }
  }
  const RouteArgs ra{dims->route, dims->n_group, dims->topk_group, dims->route_scale, dims->score_bias};
  E0_CHECK_CUDA(e0pf_route_topk(z, T, E, K, ra, ids, w, st));
  return E0_OK;
}

extern "C" size_t e0_decode_workspace_size(const e0_dims* dims, int32_t T, int32_t lora_out, int32_t H) {
  if (!dims || T < 1) return 0;
  const size_t one = e0_workspace_size(dims, 1);
  if (T == 1) return one;
  const size_t pf = align256(e0_prefill_workspace_size(dims, T, lora_out));
  return std::max(one, pf + e0mt_head_scratch(dims, T, H));
}
