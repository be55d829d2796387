// Per-warp routing arithmetic shared by the standalone routing kernel and
// the fused layer kernel, so both take identical decisions bit for bit.
//
// Follows "Clover-35B-A3B: how a diffusion model gets to 680 tokens a second,
// read from its files", sections "What Clover is" (256 experts, 8 per token)
// and "The expert selection" (top-8 routing probabilities).
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "sm100.cuh"

namespace clover {

// Reciprocal RMS of one row, computed by one warp: 1 / sqrt(mean(x^2) + eps).
// Loads are unrolled so that several are in flight per lane.
__device__ __forceinline__ float row_rstd(const float* xr, int H, float eps, int lane) {
  float ss = 0.f;
#pragma unroll 8
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum_f(ss);
  return 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
}

// As row_rstd + warp_router_dots for H <= 128 * kChunks, with the row held
// in registers between the two (one load of the row, all loads in flight at
// once). Same arithmetic order, so the results are identical.
template <int kMaxE, int kChunks>
__device__ __forceinline__ float warp_router_row_reg(const float* xr, float eps, const __nv_bfloat16* w_rows, int ne,
                                                     int H, int lane, __nv_bfloat16* xn_out) {
  float4 xv[kChunks];
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = lane * 4 + 128 * j;
    xv[j] = (c < H) ? *reinterpret_cast<const float4*>(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) ss += xv[j].x * xv[j].x + xv[j].y * xv[j].y + xv[j].z * xv[j].z + xv[j].w * xv[j].w;
  ss = warp_sum_f(ss);
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  float acc[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) acc[e] = 0.f;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = lane * 4 + 128 * j;
    if (c < H) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(xv[j].x * rstd, xv[j].y * rstd);
      __nv_bfloat162 hi = __floats2bfloat162_rn(xv[j].z * rstd, xv[j].w * rstd);
      if (xn_out != nullptr) {
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(xn_out + c) = pk;
      }
      const float x0 = __low2float(lo), x1 = __high2float(lo), x2 = __low2float(hi), x3 = __high2float(hi);
#pragma unroll
      for (int e = 0; e < kMaxE; ++e) {
        if (e < ne) {
          const uint2 wb = *reinterpret_cast<const uint2*>(w_rows + static_cast<size_t>(e) * H + c);
          const __nv_bfloat162 w01 = *reinterpret_cast<const __nv_bfloat162*>(&wb.x);
          const __nv_bfloat162 w23 = *reinterpret_cast<const __nv_bfloat162*>(&wb.y);
          acc[e] = fmaf(x0, __low2float(w01), acc[e]);
          acc[e] = fmaf(x1, __high2float(w01), acc[e]);
          acc[e] = fmaf(x2, __low2float(w23), acc[e]);
          acc[e] = fmaf(x3, __high2float(w23), acc[e]);
        }
      }
    }
  }
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) {
    const float sm = warp_sum_f(acc[e]);
    if (lane == e) mine = sm;
  }
  return mine;
}

// One warp, one token row xr: xn = bf16(xr * rstd) (stored to xn_out when
// non-null) and the router logits of experts w_rows[0..ne) (ne <= 8), each a
// bf16 row of H. Lane e (< ne) receives logit e (without bias).
template <int kMaxE>
__device__ __forceinline__ float warp_router_dots(const float* xr, float rstd, const __nv_bfloat16* w_rows, int ne,
                                                  int H, int lane, __nv_bfloat16* xn_out) {
  float acc[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * rstd, v.y * rstd);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * rstd, v.w * rstd);
    if (xn_out != nullptr) {
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(xn_out + c) = pk;
    }
    const float x0 = __low2float(lo), x1 = __high2float(lo), x2 = __low2float(hi), x3 = __high2float(hi);
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) {
      if (e < ne) {
        const uint2 wb = *reinterpret_cast<const uint2*>(w_rows + static_cast<size_t>(e) * H + c);
        const __nv_bfloat162 w01 = *reinterpret_cast<const __nv_bfloat162*>(&wb.x);
        const __nv_bfloat162 w23 = *reinterpret_cast<const __nv_bfloat162*>(&wb.y);
        acc[e] = fmaf(x0, __low2float(w01), acc[e]);
        acc[e] = fmaf(x1, __high2float(w01), acc[e]);
        acc[e] = fmaf(x2, __low2float(w23), acc[e]);
        acc[e] = fmaf(x3, __high2float(w23), acc[e]);
      }
    }
  }
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) {
    const float s = warp_sum_f(acc[e]);
    if (lane == e) mine = s;
  }
  return mine;
}

struct TopkSel {
  int e;    // selected expert
  float w;  // weight: softmax over the selected logits
  float p;  // softmax probability over all E logits (coreset mass)
};

// One warp, one token: top-k of E (<= 256) logits by descending value, the
// lower expert id first on ties, restricted to the experts whose bit is set in
// `allowed` (8 words; null = all). Weights = softmax over the selected
// logits (= the top-k probabilities renormalised). Lane k (< K) receives
// selection k, its weight and its probability under the softmax over all E.
__device__ __forceinline__ TopkSel warp_topk(const float* logits_row, int E, int K, int lane,
                                             const uint32_t* allowed = nullptr) {
  float v[8];
  float all_max = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(logits_row + e) : -INFINITY;
    all_max = fmaxf(all_max, v[i]);
  }
  all_max = warp_max_f(all_max);
  float all_sum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) all_sum += (lane + 32 * i < E) ? expf(v[i] - all_max) : 0.f;
  all_sum = warp_sum_f(all_sum);
  if (allowed != nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((allowed[e >> 5] >> (e & 31)) & 1u)) v[i] = -INFINITY;
    }
  }
  float my_v = -INFINITY;
  int my_e = 0;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i == (be >> 5)) v[i] = -INFINITY;
    }
    if (lane == k) {
      my_v = bv;
      my_e = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < K) ? expf(my_v - top) : 0.f;
  const float sum = warp_sum_f(ex);
  TopkSel r;
  r.e = my_e;
  r.w = ex / sum;
  r.p = (lane < K) ? expf(my_v - all_max) / all_sum : 0.f;
  return r;
}

}  // namespace clover
