// Per-warp routing arithmetic: the fused layer kernel's CUDA-core router
// dot products, the top-k selection that both routing paths share, and the
// warp tensor-core contraction of the standalone routing kernel. The two
// paths sum the router dot products in different orders, so their logits
// can differ in the last bits; the selection rule itself is the same code.
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
// (l2: the row is global memory that other CTAs of this launch wrote, read
// through L2 rather than the SM's L1.)
__device__ __forceinline__ float4 row_load4(const float* p, bool l2) {
  return l2 ? __ldcg(reinterpret_cast<const float4*>(p)) : *reinterpret_cast<const float4*>(p);
}

__device__ __forceinline__ float row_rstd(const float* xr, int H, float eps, int lane, bool l2 = false) {
  float ss = 0.f;
#pragma unroll 8
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = row_load4(xr + c, l2);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum_f(ss);
  return 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
}

// Reciprocal RMS of a row of H <= 2,048 values that a warp holds as 16
// float4 per lane (lane l: columns 4l + 128c, zeros past H): the lane's sum
// of squares in column order, then the warp butterfly. Every rounding is
// explicit, so the standalone routing kernel and the combine that normalises
// the next layer's input compute the same bits.
__device__ __forceinline__ float rstd_row16(const float4 (&xv)[16], int H, float eps) {
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const float4 v = xv[c];
    const float p = __fadd_rn(__fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)),
                              __fadd_rn(__fmul_rn(v.z, v.z), __fmul_rn(v.w, v.w)));
    ss = __fadd_rn(ss, p);
  }
  ss = warp_sum_f(ss);
  return 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
}

// As row_rstd + warp_router_dots for H <= 128 * kChunks, with the row held
// in registers between the two (one load of the row, all loads in flight at
// once). Same arithmetic order, so the results are identical.
template <int kMaxE, int kChunks>
__device__ __forceinline__ float warp_router_row_reg(const float* xr, float eps, const __nv_bfloat16* w_rows, int ne,
                                                     int H, int lane, __nv_bfloat16* xn_out, bool l2 = false) {
  float4 xv[kChunks];
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = lane * 4 + 128 * j;
    xv[j] = (c < H) ? row_load4(xr + c, l2) : make_float4(0.f, 0.f, 0.f, 0.f);
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

// warp_router_row_reg for the common shape, with both operands staged in
// shared memory (32-bit shared addresses) and the hidden size and expert
// count fixed at compile time: explicit shared loads, no per-element guards
// and constant offsets let every load of a chunk issue ahead of its FMAs.
// The same expressions in the same order, so the results are identical.
template <int kE, int kH>
__device__ __forceinline__ float warp_router_row_smem(uint32_t xr, float eps, uint32_t w_rows, int lane,
                                                      __nv_bfloat16* xn_out) {
  constexpr int kChunks = kH / 128;
  static_assert(kH % 128 == 0, "hidden size must be a multiple of 128");
  float4 xv[kChunks];
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const uint32_t a = xr + static_cast<uint32_t>(lane * 4 + 128 * j) * 4u;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(xv[j].x), "=f"(xv[j].y), "=f"(xv[j].z), "=f"(xv[j].w)
                 : "r"(a));
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) ss += xv[j].x * xv[j].x + xv[j].y * xv[j].y + xv[j].z * xv[j].z + xv[j].w * xv[j].w;
  ss = warp_sum_f(ss);
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(kH) + eps);
  float acc[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) acc[e] = 0.f;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = lane * 4 + 128 * j;
    __nv_bfloat162 lo = __floats2bfloat162_rn(xv[j].x * rstd, xv[j].y * rstd);
    __nv_bfloat162 hi = __floats2bfloat162_rn(xv[j].z * rstd, xv[j].w * rstd);
    if (xn_out != nullptr) {
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(xn_out + c) = pk;
    }
    const float x0 = __low2float(lo), x1 = __high2float(lo), x2 = __low2float(hi), x3 = __high2float(hi);
    uint2 wb[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const uint32_t a = w_rows + static_cast<uint32_t>(e * kH + c) * 2u;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(wb[e].x), "=r"(wb[e].y) : "r"(a));
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const __nv_bfloat162 w01 = *reinterpret_cast<const __nv_bfloat162*>(&wb[e].x);
      const __nv_bfloat162 w23 = *reinterpret_cast<const __nv_bfloat162*>(&wb[e].y);
      acc[e] = fmaf(x0, __low2float(w01), acc[e]);
      acc[e] = fmaf(x1, __high2float(w01), acc[e]);
      acc[e] = fmaf(x2, __low2float(w23), acc[e]);
      acc[e] = fmaf(x3, __high2float(w23), acc[e]);
    }
  }
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const float sm = warp_sum_f(acc[e]);
    if (lane == e) mine = sm;
  }
  return mine;
}

// D (16x8, fp32) += A (16x16, bf16, row-major) * B (16x8, bf16, column-major)
// on the warp's tensor cores. Fragment ownership (g = lane / 4, q = lane % 4):
// a0 = A[g][2q..2q+1], a1 = A[g+8][2q..], a2 = A[g][2q+8..], a3 = A[g+8][2q+8..];
// b0 = B[2q..2q+1][g], b1 = B[2q+8..2q+9][g]; d = D[g][2q..2q+1], D[g+8][2q..2q+1].
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Router logits of one routing item on the warp tensor cores, at the Clover
// shape: up to 8 tokens (fp32 rows of kH, staged in shared memory at x_rows)
// against 8 experts (bf16 router rows at w_rows, row stride kH + 8
// elements). Called by warps 0..7 together (named barrier `bar` of 256
// threads). Warp w normalises token w (xn = bf16(x * rstd), stored into
// shared memory at xn_rows with the same padded stride, and to
// xn_out + w * kH when xn_out is non-null; rows past n_tok are zero), then
// every warp contracts one eighth of the hidden size with mma.sync m16n8k16
// (tokens x experts; the eight missing token rows of the 16-row tile are
// zero registers), and the eight partial tiles (part: 8 x 8 x 8 floats) are
// summed in warp order. The padding puts the eight rows a fragment load
// touches in different banks. Lane e (< 8) of warp w receives the logit of
// token w and expert e (without bias).
template <int kH>
__device__ __forceinline__ float cta_router_item_mma(uint32_t x_rows, int n_tok, float eps, uint32_t w_rows,
                                                     uint32_t xn_rows, float* part, __nv_bfloat16* xn_out, int warp,
                                                     int lane, uint32_t bar) {
  constexpr int kLd = kH + 8;
  constexpr int kChunks = kH / 128;
  static_assert(kH % 128 == 0, "hidden size must be a multiple of 128");
  const uint32_t my_row = xn_rows + static_cast<uint32_t>(warp * kLd) * 2u;
  if (warp < n_tok) {
    float4 xv[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      const uint32_t a = x_rows + static_cast<uint32_t>(warp * kH + lane * 4 + 128 * j) * 4u;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(xv[j].x), "=f"(xv[j].y), "=f"(xv[j].z), "=f"(xv[j].w)
                   : "r"(a));
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kChunks; ++j)
      ss += xv[j].x * xv[j].x + xv[j].y * xv[j].y + xv[j].z * xv[j].z + xv[j].w * xv[j].w;
    ss = warp_sum_f(ss);
    const float rstd = 1.0f / sqrtf(ss / static_cast<float>(kH) + eps);
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      const int c = lane * 4 + 128 * j;
      __nv_bfloat162 lo = __floats2bfloat162_rn(xv[j].x * rstd, xv[j].y * rstd);
      __nv_bfloat162 hi = __floats2bfloat162_rn(xv[j].z * rstd, xv[j].w * rstd);
      const uint32_t ulo = *reinterpret_cast<uint32_t*>(&lo), uhi = *reinterpret_cast<uint32_t*>(&hi);
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(my_row + static_cast<uint32_t>(c) * 2u), "r"(ulo), "r"(uhi)
                   : "memory");
      if (xn_out != nullptr) {
        uint2 pk;
        pk.x = ulo;
        pk.y = uhi;
        *reinterpret_cast<uint2*>(xn_out + static_cast<size_t>(warp) * kH + c) = pk;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kChunks; ++j)
      asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(my_row + static_cast<uint32_t>(lane * 4 + 128 * j) * 2u),
                   "r"(0u)
                   : "memory");
  }
  named_bar_sync(bar, 256);
  const int g = lane >> 2, q = lane & 3;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t xa = xn_rows + static_cast<uint32_t>(g * kLd + 2 * q) * 2u;
  const uint32_t wa = w_rows + static_cast<uint32_t>(g * kLd + 2 * q) * 2u;
#pragma unroll 4
  for (int kb = warp * (kH / 8); kb < (warp + 1) * (kH / 8); kb += 16) {
    uint32_t a0, a2, b0, b1;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a0) : "r"(xa + kb * 2u));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a2) : "r"(xa + (kb + 8) * 2u));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(b0) : "r"(wa + kb * 2u));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(b1) : "r"(wa + (kb + 8) * 2u));
    mma_bf16_16816(acc, a0, 0u, a2, 0u, b0, b1);
  }
  // acc[0], acc[1]: token g, experts 2q and 2q + 1 (acc[2], acc[3]: the zero rows)
  part[(warp * 8 + g) * 8 + 2 * q] = acc[0];
  part[(warp * 8 + g) * 8 + 2 * q + 1] = acc[1];
  named_bar_sync(bar, 256);
  float lg = 0.f;
  if (lane < 8) {
#pragma unroll
    for (int w = 0; w < 8; ++w) lg += part[(w * 8 + warp) * 8 + lane];
  }
  return lg;
}

// One warp, one token row xr: xn = bf16(xr * rstd) (stored to xn_out when
// non-null) and the router logits of experts w_rows[0..ne) (ne <= 8), each a
// bf16 row of H. Lane e (< ne) receives logit e (without bias).
template <int kMaxE>
__device__ __forceinline__ float warp_router_dots(const float* xr, float rstd, const __nv_bfloat16* w_rows, int ne,
                                                  int H, int lane, __nv_bfloat16* xn_out, bool l2 = false) {
  float acc[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = row_load4(xr + c, l2);
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

// Unsigned key with the order of the float values (-0 and +0, equal as
// floats, share one key), and back.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp, NT tokens at once (independent chains, interleaved for latency):
// top-k of E (<= 256) logits by descending value, the lower expert id first
// on ties, restricted to the experts whose bit is set in `allowed` (8 words;
// null = all). v[n * 8 + i] holds the logit of expert lane + 32 i of token n
// (-inf past E). Weights = softmax over the selected logits (= the top-k
// probabilities renormalised). Lane k (< K) receives selection k of token n
// in out[n], with its weight and, when want_p, its probability under the
// softmax over all E. Tokens with valid[n] false give meaningless out[n].
// Each round takes the warp-wide largest key with one reduction and the
// lowest expert id holding it with a second one; the per-token arithmetic
// does not depend on NT.
template <int NT>
__device__ __forceinline__ void warp_topk_regs(const float (&v)[NT * 8], int E, int K, int lane,
                                               const uint32_t* allowed, bool want_p, TopkSel (&out)[NT]) {
  float all_max[NT], all_sum[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    all_max[n] = -INFINITY;
    all_sum[n] = 1.f;
  }
  if (want_p) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int i = 0; i < 8; ++i) all_max[n] = fmaxf(all_max[n], v[n * 8 + i]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) all_max[n] = warp_max_f(all_max[n]);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      all_sum[n] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) all_sum[n] += (lane + 32 * i < E) ? expf(v[n * 8 + i] - all_max[n]) : 0.f;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) all_sum[n] = warp_sum_f(all_sum[n]);
  }
  // Removed and disallowed experts compete as -inf (as a -inf logit would);
  // slots past E have key 0, below every value.
  const uint32_t kNegInf = order_key(-INFINITY);
  uint32_t key[NT * 8];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      const bool ok = allowed == nullptr || ((allowed[e >> 5] >> (e & 31)) & 1u);
      key[n * 8 + i] = (e < E) ? (ok ? order_key(v[n * 8 + i]) : kNegInf) : 0u;
    }
  }
  float my_v[NT];
  int my_e[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    my_v[n] = -INFINITY;
    my_e[n] = 0;
  }
  for (int k = 0; k < K; ++k) {
    uint32_t lmax[NT], gmax[NT], esel[NT];
    int li[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      // pairwise tree over the 8 slots; on equal keys the lower slot (= the
      // lower expert id) wins; key 0 never wins (li stays 8)
      uint32_t k4[4];
      int i4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a = key[n * 8 + 2 * q], b = key[n * 8 + 2 * q + 1];
        k4[q] = (b > a) ? b : a;
        i4[q] = (b > a) ? 2 * q + 1 : 2 * q;
      }
      const uint32_t k01 = (k4[1] > k4[0]) ? k4[1] : k4[0];
      const int i01 = (k4[1] > k4[0]) ? i4[1] : i4[0];
      const uint32_t k23 = (k4[3] > k4[2]) ? k4[3] : k4[2];
      const int i23 = (k4[3] > k4[2]) ? i4[3] : i4[2];
      lmax[n] = (k23 > k01) ? k23 : k01;
      li[n] = (k23 > k01) ? i23 : i01;
      if (lmax[n] == 0u) li[n] = 8;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) gmax[n] = __reduce_max_sync(0xffffffffu, lmax[n]);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint32_t cand = (li[n] < 8 && lmax[n] == gmax[n]) ? static_cast<uint32_t>(lane + 32 * li[n]) : 0xffffffffu;
      esel[n] = __reduce_min_sync(0xffffffffu, cand);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const bool mine = static_cast<int>(esel[n] & 31u) == lane;
      const int slot = static_cast<int>(esel[n] >> 5);
#pragma unroll
      for (int i = 0; i < 8; ++i) key[n * 8 + i] = (mine && i == slot) ? kNegInf : key[n * 8 + i];
      if (lane == k) {
        my_v[n] = key_value(gmax[n]);
        my_e[n] = static_cast<int>(esel[n]);
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const float top = __shfl_sync(0xffffffffu, my_v[n], 0);
    const float ex = (lane < K) ? expf(my_v[n] - top) : 0.f;
    const float sum = warp_sum_f(ex);
    out[n].e = my_e[n];
    out[n].w = ex / sum;
    out[n].p = (want_p && lane < K) ? expf(my_v[n] - all_max[n]) / all_sum[n] : 0.f;
  }
}

// As warp_topk_regs (without the full-softmax probabilities), reading token
// n's logits from the global row rows[n] (written by other CTAs of this
// launch: loads bypass L1). Tokens with valid[n] false read nothing.
template <int NT>
__device__ __forceinline__ void warp_topk_n(const float* const (&rows)[NT], const bool (&valid)[NT], int E, int K,
                                            int lane, const uint32_t* allowed, TopkSel (&out)[NT]) {
  float v[NT * 8];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[n * 8 + i] = (valid[n] && e < E) ? __ldcg(rows[n] + e) : -INFINITY;
    }
  }
  warp_topk_regs<NT>(v, E, K, lane, allowed, false, out);
}



// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of
// 32, at most 512). Returns the exclusive prefix; *total receives the sum.
// s_tmp holds 17 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* s_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = static_cast<int>(blockDim.x >> 5);
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wv = lane < nw ? s_tmp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) s_tmp[lane] = wi - wv;  // exclusive warp offsets
    if (lane == nw - 1) s_tmp[16] = wi;    // total
  }
  __syncthreads();
  const int res = s_tmp[warp] + incl - v;
  *total = s_tmp[16];
  __syncthreads();
  return res;
}

// Shared-memory tables of one CTA's token -> expert permutation.
struct PermTables {
  uint8_t* idx;       // [M*K] selections (clamped expert ids; E <= 256)
  uint16_t* row_tok;  // [M*K] token of each gathered row (tokens < 65536)
  uint32_t* bm;       // [E][perm_stride(M)] token bitmask per expert
  uint16_t* pre;      // [E][perm_stride(M)] tokens of the expert in the words before each word
  int* off;           // [E] first row of each expert
  int* cnt;           // [E] tokens per expert
  int* tmp;           // [32] scan scratch
};

// Words per expert in the bitmask and prefix tables: one per 32 tokens,
// rounded up to an odd count so that the rows of different experts start in
// different shared-memory banks (warps read one word of many experts at once).
__host__ __device__ constexpr int perm_stride(int M) { return ((M + 31) >> 5) | 1; }

// Builds, with every thread of the CTA (blockDim.x >= E), the permutation of
// the M*K top-k selections: per-expert token bitmasks, per-expert counts and a prefix count per
// word, a scan over experts for the row offsets, and each selection's row =
// its expert's offset + the number of lower tokens routed to that expert, so
// rows of one expert are in token order. Returns the number of active
// experts; `slot_out` (nullable) receives each selection's row.
__device__ __forceinline__ int cta_permutation(const int32_t* topk_idx, int M, int K, int E, const PermTables& t,
                                               int32_t* slot_out) {
  const int tid = threadIdx.x;
  const int MK = M * K, nw = (M + 31) >> 5, ws = perm_stride(M);
  // Eight loads in flight per thread before any store: the loads read global
  // memory and the stores shared memory through generic pointers, so the
  // compiler would otherwise keep every load behind the previous store.
  for (int i0 = tid; i0 < MK; i0 += 8 * blockDim.x) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * blockDim.x;
      v[j] = i < MK ? __ldcg(topk_idx + i) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * blockDim.x;
      const int e = v[j];
      if (i < MK) t.idx[i] = static_cast<uint8_t>(e < 0 ? 0 : (e >= E ? E - 1 : e));  // ids come from another kernel; clamping keeps indexing safe
    }
  }
  for (int i = tid; i < E * ws; i += blockDim.x) t.bm[i] = 0u;
  __syncthreads();
  // one shared-memory OR per selection (order-independent, so every CTA gets
  // the same bits)
  for (int i = tid; i < MK; i += blockDim.x) {
    const int tk = i / K;
    atomicOr(&t.bm[t.idx[i] * ws + (tk >> 5)], 1u << (tk & 31));
  }
  __syncthreads();
  int c = 0;
  if (tid < E)
    for (int wd = 0; wd < nw; ++wd) {
      t.pre[tid * ws + wd] = static_cast<uint16_t>(c);
      c += __popc(t.bm[tid * ws + wd]);
    }
  int total = 0;
  const int off = block_excl_scan(c, t.tmp, &total);
  const int n_act = __syncthreads_count(tid < E && c > 0);
  if (tid < E) {
    t.off[tid] = off;
    t.cnt[tid] = c;
  }
  __syncthreads();
  for (int i = tid; i < MK; i += blockDim.x) {
    const int e = t.idx[i], tk = i / K;
    const int wd = tk >> 5, bit = tk & 31;
    const int row = t.off[e] + t.pre[e * ws + wd] + __popc(t.bm[e * ws + wd] & ((1u << bit) - 1u));
    t.row_tok[row] = static_cast<uint16_t>(tk);
    if (slot_out != nullptr) slot_out[i] = row;
  }
  __syncthreads();
  return n_act;
}

}  // namespace clover
