// Low-bit expert weights: the quantizer that turns bf16 expert matrices into
// 4-bit codes with one bf16 scale per row and group of 64 K elements.
//
// The pages name INT4 for one deployment of the model ("Clover-35B-A3B: how a
// diffusion model gets to 680 tokens a second, read from its files", section
// "What 680 tokens a second has to be") but give no format; this one is
// this library's own. Per group: s = bf16(float32(max |w|) / 7) (IEEE fp32 division,
// round to nearest even); per element u = clamp(rint(w / s), -8, 7) + 8
// (u = 8 where s = 0); the weight a product uses is bf16((u - 8) s). Eight
// codes fill a 32-bit word in the nibble order e0 e2 e4 e6 e1 e3 e5 e7, so
// that (word >> 4i) & 0x000F000F holds the adjacent pair (e_2i, e_2i+1).
// Scales are stored group-major: [K/64][R] per matrix.
#include <math.h>

#include "kernels.cuh"
#include "launch.cuh"

namespace clover {

// One thread per (matrix, row, group of 64): reads 128 B of bf16, writes 32 B
// of codes and one scale.
__global__ void __launch_bounds__(256) k_quantize_q4(QuantArgs a) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int groups = a.cols / 64;
  const int64_t total = static_cast<int64_t>(a.n_mats) * a.rows * groups;
  if (gid >= total) return;
  const int g = static_cast<int>(gid % groups);
  const int64_t mr = gid / groups;  // matrix * rows + row
  const int r = static_cast<int>(mr % a.rows);
  const int64_t mat = mr / a.rows;
  const uint4* src = reinterpret_cast<const uint4*>(a.w + mr * a.cols + g * 64);
  float v[64];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = src[i];
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(wd[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(amax, 7.0f));
  const float s = __bfloat162float(sb);
  uint32_t words[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // nibble i holds element (0, 2, 4, 6, 1, 3, 5, 7)[i] of the eight
      const int e = (i < 4) ? 2 * i : 2 * (i - 4) + 1;
      float q = 0.f;
      if (s > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(v[8 * w + e], s)), -8.f), 7.f);
      word |= static_cast<uint32_t>(static_cast<int>(q) + 8) << (4 * i);
    }
    words[w] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(a.q + mr * (a.cols / 2) + g * 32);
  dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
  dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
  a.s[(mat * groups + g) * a.rows + r] = __bfloat16_as_ushort(sb);
}

cudaError_t launch_quantize_q4(const QuantArgs& a, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(a.n_mats) * a.rows * (a.cols / 64);
  const int64_t blocks = (total + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  return launch_kernel(k_quantize_q4, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, false, a);
}

}  // namespace clover
