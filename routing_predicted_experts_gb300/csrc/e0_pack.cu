// int4 affine group-64 packing (e0_pack_int4) and the seeded input generator
// (e0_synth_normal).
//
// Packing follows "The Other Half of the Memory Wall" §3.1 / §2 "Quantization"
// (int4 affine, group 64, per-group scale and bias).  The rounding contract is
// stated in include/e0.h; every step uses explicitly rounded IEEE fp32 intrinsics
// so the result does not depend on contraction or fast-math settings.
#include "e0_common.cuh"

namespace {

__global__ void pack_int4_kernel(const float* __restrict__ w, int64_t batch, int64_t rows, int64_t cols,
                                 int layout, uint32_t* __restrict__ q, uint16_t* __restrict__ scale,
                                 uint16_t* __restrict__ bias) {
  const int64_t groups_per_row = cols / 64;
  const int64_t total = batch * rows * groups_per_row;
  for (int64_t gid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; gid < total;
       gid += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = gid % groups_per_row;
    const int64_t rr = gid / groups_per_row;  // batch*rows + row
    const int64_t r = rr % rows;
    const int64_t bt = rr / rows;
    const float4* src = reinterpret_cast<const float4*>(w + rr * cols + g * 64);
    float v[64];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float4 f = src[i];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int i = 1; i < 64; ++i) {
      lo = fminf(lo, v[i]);
      hi = fmaxf(hi, v[i]);
    }
    const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    const uint16_t sb = e0dev::f32_to_bf16_bits(s32);
    const uint16_t bb = e0dev::f32_to_bf16_bits(lo);
    const float sf = e0dev::bf16_bits_to_f32(sb);
    const float bf = e0dev::bf16_bits_to_f32(bb);
    uint32_t words[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t code = 0;
        if (sf != 0.0f) {
          float t = rintf(__fdiv_rn(__fsub_rn(v[8 * m + j], bf), sf));
          t = fminf(fmaxf(t, 0.0f), 15.0f);
          code = (uint32_t)t;
        }
        word |= code << (4 * j);
      }
      words[m] = word;
    }
    if (layout == E0_LAYOUT_ROWS) {
      uint4* dst = reinterpret_cast<uint4*>(q + rr * (cols / 8) + g * 8);
      dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
      dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
      scale[rr * groups_per_row + g] = sb;
      bias[rr * groups_per_row + g] = bb;
    } else {
      const int64_t slabs = cols / 32;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t c = 2 * g + h;
        uint4* dst = reinterpret_cast<uint4*>(q + ((bt * slabs + c) * rows + r) * 4);
        dst[0] = make_uint4(words[4 * h], words[4 * h + 1], words[4 * h + 2], words[4 * h + 3]);
      }
      scale[(bt * groups_per_row + g) * rows + r] = sb;
      bias[(bt * groups_per_row + g) * rows + r] = bb;
    }
  }
}

// ---------------------------------------------------------------- e0synth
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__global__ void synth_normal_kernel(void* out, int64_t n, uint64_t base, int64_t offset, double sigma,
                                    int bf16) {
  const uint64_t G = 0x9E3779B97F4A7C15ull;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t idx = (uint64_t)(offset + i) * 12ull;
    int64_t s = 0;
#pragma unroll
    for (int k = 0; k < 12; ++k) s += (int64_t)(mix64(base + (idx + k + 1) * G) >> 40);
    const double v = __dmul_rn(__dmul_rn((double)(s - 6ll * (1ll << 24)), sigma), 5.9604644775390625e-08);
    const float f = __double2float_rn(v);
    if (bf16)
      reinterpret_cast<uint16_t*>(out)[i] = e0dev::f32_to_bf16_bits(f);
    else
      reinterpret_cast<float*>(out)[i] = f;
  }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" e0_status e0_pack_int4(const float* w, int64_t batch, int64_t rows, int64_t cols, int32_t group,
                                  int32_t layout, uint32_t* q, uint16_t* scale, uint16_t* bias,
                                  e0_stream stream) {
  E0_REQUIRE(w && q && scale && bias, E0_ERR_INVALID, "e0_pack_int4: null pointer");
  E0_REQUIRE(aligned16(w) && aligned16(q), E0_ERR_INVALID, "e0_pack_int4: w and q must be 16-byte aligned");
  E0_REQUIRE(group == 64, E0_ERR_UNSUPPORTED, "e0_pack_int4: only group == 64 is supported");
  E0_REQUIRE(batch > 0 && rows > 0 && cols > 0 && cols % 64 == 0, E0_ERR_SHAPE,
             "e0_pack_int4: need batch, rows > 0 and cols a positive multiple of 64");
  E0_REQUIRE(layout == E0_LAYOUT_ROWS || layout == E0_LAYOUT_COLSLAB, E0_ERR_INVALID,
             "e0_pack_int4: unknown layout");
  const int64_t total = batch * rows * (cols / 64);
  const int threads = 128;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  pack_int4_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(w, batch, rows, cols, layout, q,
                                                                           scale, bias);
  E0_CHECK_CUDA(cudaGetLastError());
  return E0_OK;
}

extern "C" e0_status e0_synth_normal(void* out, int64_t n, uint64_t seed, uint32_t stream_id, int64_t offset,
                                     double sigma, int32_t bf16, e0_stream stream) {
  E0_REQUIRE(out != nullptr && n >= 0 && offset >= 0, E0_ERR_INVALID, "e0_synth_normal: bad arguments");
  if (n == 0) return E0_OK;
  // base = mix(seed*G + stream*H + 1), computed on the host with wrapping arithmetic
  uint64_t z = seed * 0x9E3779B97F4A7C15ull + (uint64_t)stream_id * 0xD1B54A32D192ED03ull + 1ull;
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  synth_normal_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(out, n, z, offset, sigma,
                                                                              bf16);
  E0_CHECK_CUDA(cudaGetLastError());
  return E0_OK;
}
