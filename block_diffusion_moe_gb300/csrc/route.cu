// Input assembly, RMSNorm, router with softmax top-k, and the parallel
// combine of the standalone path.
//
// Follows "Clover-35B-A3B: how a diffusion model gets to 680 tokens a second,
// read from its files": section "What Clover is" (256 routed experts, each
// token routed to 8, block of mask tokens), section "The expert selection"
// (per-token top-8 routing probabilities) and section "How it writes",
// step 1 (the block re-enters with mask-token embeddings until committed).
#include <math.h>

#include <algorithm>

#include "kernels.cuh"
#include "launch.cuh"
#include "routing.cuh"
#include "sm100.cuh"

namespace clover {

// ------------------------------------------------------------------ embed
// x_p = E[t_p] + c_p. One CTA per position.
__global__ void __launch_bounds__(256) k_embed(EmbedArgs a) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x;
  int t = a.tokens[p];
  if (t < 0 || t >= a.V) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrBadToken);
    t = t < 0 ? 0 : a.V - 1;
  }
  const bf16* er = a.embed + static_cast<size_t>(t) * a.H;
  const float* cr = a.ctx + static_cast<size_t>(p) * a.H;
  float* xr = a.x + static_cast<size_t>(p) * a.H;
  for (int c = threadIdx.x * 4; c < a.H; c += blockDim.x * 4) {
    const uint2 eb = *reinterpret_cast<const uint2*>(er + c);
    const float4 cv = *reinterpret_cast<const float4*>(cr + c);
    const __nv_bfloat162 e01 = *reinterpret_cast<const __nv_bfloat162*>(&eb.x);
    const __nv_bfloat162 e23 = *reinterpret_cast<const __nv_bfloat162*>(&eb.y);
    float4 o;
    o.x = __low2float(e01) + cv.x;
    o.y = __high2float(e01) + cv.y;
    o.z = __low2float(e23) + cv.z;
    o.w = __high2float(e23) + cv.w;
    *reinterpret_cast<float4*>(xr + c) = o;
  }
}

// ---------------------------------------------------------------- rmsnorm
// xn = bf16(x * rstd). One warp per row.
__global__ void __launch_bounds__(256) k_rmsnorm(NormArgs a) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t < a.M) {
    const float* xr = a.x + static_cast<size_t>(t) * a.H;
    const float rstd = row_rstd(xr, a.H, a.eps, lane);
    bf16* out = a.xn + static_cast<size_t>(t) * a.H;
    for (int c = lane * 4; c < a.H; c += 128) {
      const float4 v = *reinterpret_cast<const float4*>(xr + c);
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * rstd, v.y * rstd);
      __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * rstd, v.w * rstd);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + c) = pk;
    }
  }
}

// ------------------------------------------------------------------ route
// Routing for more than 32 tokens. Grid (ceil(E/32), ceil(M/16)): each CTA
// owns a tile of 16 tokens x 32 experts.
//  1. Its 32 router rows are bulk-copied into shared memory before the
//     dependency wait (they do not depend on earlier kernels).
//  2. Each warp normalises two token rows (row kept in registers for
//     H <= 2048): xn = bf16(x * rstd), rstd = 1 / sqrt(mean(x^2) + eps),
//     into shared memory, and expert tile 0 also writes them to xn_rows.
//  3. The tile's logits are one bf16 contraction with fp32 accumulation on
//     the warp tensor cores (mma m16n8k16: tokens x experts, the hidden size
//     split eight ways across the warps, the partials summed in warp order).
//  4. The last CTA to finish a token tile takes softmax top-k for its tokens:
//     selection by descending logit with the lower expert id first on ties,
//     weights = softmax over the selected logits (= top-k probabilities
//     renormalised to sum to one).
// H above 2048 is contracted in chunks of 2048 columns.
__global__ void __launch_bounds__(256, 1) k_route(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = a.H, E = a.E, M = a.M;
  const int Hc = min(H, kRouteChunk);
  const int ld = Hc + 8;  // padded row stride (elements): fragment loads hit 32 distinct banks
  bf16* s_w = reinterpret_cast<bf16*>(smem);                                      // [32][ld]
  bf16* s_x = s_w + kRouteTileExperts * ld;                                        // [16][ld]
  float* s_part = reinterpret_cast<float*>(s_x + kRouteTileTokens * ld);          // [8][16][32]
  uint64_t* wbar = reinterpret_cast<uint64_t*>(s_part + 8 * kRouteTileTokens * kRouteTileExperts + 16);
  uint64_t* xbar = wbar + 1;  // the normed rows, when the previous combine wrote them
  __shared__ int s_last;
  __shared__ int s_bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * kRouteTileExperts;
  const int ne = min(kRouteTileExperts, E - e0);
  const int t0 = blockIdx.y * kRouteTileTokens;
  const int nt = min(kRouteTileTokens, M - t0);
  const int n_chunks = (H + kRouteChunk - 1) / kRouteChunk;

  // Rows past the tile's experts / tokens stay zero (their outputs are dropped).
  for (int i = tid; i < (kRouteTileExperts - ne) * ld; i += blockDim.x) s_w[ne * ld + i] = __float2bfloat16_rn(0.f);
  for (int i = tid; i < (kRouteTileTokens - nt) * ld; i += blockDim.x) s_x[nt * ld + i] = __float2bfloat16_rn(0.f);
  if (tid == 0) {
    s_bad = 0;
    mbar_init(wbar, 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
    const int len = min(H, kRouteChunk);
    mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(ne * len * 2));
    for (int r = 0; r < ne; ++r)
      bulk_load(smem_u32(s_w + r * ld), a.wr + static_cast<size_t>(e0 + r) * H, len * 2, wbar);
  }
  pdl_wait();
  pdl_trigger();

  // This warp's two token rows: tile rows warp and warp + 8.
  float rs[2];
  if (a.xn_ready) {
    // The previous layer's combine wrote the normed rows: copy them in.
    if (tid == 0) {
      mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(nt * H * 2));
      for (int r = 0; r < nt; ++r)
        bulk_load(smem_u32(s_x + r * ld), a.xn_rows + static_cast<size_t>(t0 + r) * H, static_cast<uint32_t>(H * 2), xbar);
    }
    if (!mbar_wait_for(xbar, 0, kWaitLimitNs) && lane == 0) {
      atomicOr(a.err, kErrMbarTimeout);
      s_bad = 1;
    }
  } else if (H <= kRouteChunk) {
    float4 xv[2][16];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = warp + 8 * j;
      const float* xr = a.x + static_cast<size_t>(t0 + r) * H;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int col = lane * 4 + 128 * c;
        xv[j][c] = (r < nt && col < H) ? *reinterpret_cast<const float4*>(xr + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) rs[j] = rstd_row16(xv[j], H, a.eps);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = warp + 8 * j;
      if (r >= nt) continue;
      bf16* gx = blockIdx.x == 0 ? a.xn_rows + static_cast<size_t>(t0 + r) * H : nullptr;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int col = lane * 4 + 128 * c;
        if (col < H) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(xv[j][c].x * rs[j], xv[j][c].y * rs[j]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(xv[j][c].z * rs[j], xv[j][c].w * rs[j]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(s_x + r * ld + col) = pk;
          if (gx != nullptr) *reinterpret_cast<uint2*>(gx + col) = pk;
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = warp + 8 * j;
      rs[j] = r < nt ? row_rstd(a.x + static_cast<size_t>(t0 + r) * H, H, a.eps, lane) : 0.f;
    }
  }

  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  for (int ch = 0; ch < n_chunks; ++ch) {
    const int c0 = ch * kRouteChunk;
    const int len = min(kRouteChunk, H - c0);
    if (ch > 0) {
      // Refill: every warp is done with the previous chunk's rows.
      __syncthreads();
      if (tid == 0) {
        fence_proxy_async_shared();
        mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(ne * len * 2));
        for (int r = 0; r < ne; ++r)
          bulk_load(smem_u32(s_w + r * ld), a.wr + static_cast<size_t>(e0 + r) * H + c0, len * 2, wbar);
      }
    }
    if (n_chunks > 1) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = warp + 8 * j;
        if (r >= nt) continue;
        const float* xr = a.x + static_cast<size_t>(t0 + r) * H + c0;
        bf16* gx = blockIdx.x == 0 ? a.xn_rows + static_cast<size_t>(t0 + r) * H + c0 : nullptr;
        for (int col = lane * 4; col < len; col += 128) {
          const float4 v = *reinterpret_cast<const float4*>(xr + col);
          __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * rs[j], v.y * rs[j]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * rs[j], v.w * rs[j]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(s_x + r * ld + col) = pk;
          if (gx != nullptr) *reinterpret_cast<uint2*>(gx + col) = pk;
        }
      }
    }
    __syncthreads();
    if (!mbar_wait_for(wbar, static_cast<uint32_t>(ch & 1), kWaitLimitNs) && lane == 0) {
      atomicOr(a.err, kErrMbarTimeout);
      s_bad = 1;
    }
    // This warp's eighth of the chunk (len / 8 is a multiple of 16).
    const int kw = len >> 3;
    const bf16* xa = s_x + g * ld + 2 * q + warp * kw;
    const bf16* wa = s_w + g * ld + 2 * q + warp * kw;
    for (int kb = 0; kb < kw; kb += 16) {
      const uint32_t a0 = *reinterpret_cast<const uint32_t*>(xa + kb);
      const uint32_t a1 = *reinterpret_cast<const uint32_t*>(xa + 8 * ld + kb);
      const uint32_t a2 = *reinterpret_cast<const uint32_t*>(xa + kb + 8);
      const uint32_t a3 = *reinterpret_cast<const uint32_t*>(xa + 8 * ld + kb + 8);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bf16* wb = wa + 8 * j * ld + kb;
        mma_bf16_16816(acc[j], a0, a1, a2, a3, *reinterpret_cast<const uint32_t*>(wb),
                       *reinterpret_cast<const uint32_t*>(wb + 8));
      }
    }
  }

  // Partials [warp][token][expert], then fixed-order sums over the warps.
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float* pw = s_part + (warp * kRouteTileTokens + g) * kRouteTileExperts + 8 * j + 2 * q;
    *reinterpret_cast<float2*>(pw) = make_float2(acc[j][0], acc[j][1]);
    *reinterpret_cast<float2*>(pw + 8 * kRouteTileExperts) = make_float2(acc[j][2], acc[j][3]);
  }
  __syncthreads();
  // A router copy that did not land has been flagged; wait once more
  // (bounded) so that no copy is still writing shared memory when this CTA
  // exits, and carry on so that the arrival counters stay consistent.
  if (s_bad) mbar_wait_for(wbar, static_cast<uint32_t>((n_chunks - 1) & 1), kWaitLimitNs);
  if (s_bad && a.xn_ready) mbar_wait_for(xbar, 0, kWaitLimitNs);
  for (int o = tid; o < kRouteTileTokens * kRouteTileExperts; o += blockDim.x) {
    const int r = o / kRouteTileExperts, c = o % kRouteTileExperts;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += s_part[(w * kRouteTileTokens + r) * kRouteTileExperts + c];
    if (r < nt && c < ne) {
      const int e = e0 + c;
      a.logits[static_cast<size_t>(t0 + r) * E + e] = sum + (a.bias ? a.bias[e] : 0.f);
    }
  }
  // One fence on each side by the arriving thread: the CTA barrier orders the
  // other threads' logit stores before it, and their later loads after it.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&a.tg_ctr[blockIdx.y], 1);
    __threadfence();
    s_last = (old == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // Top-k for this token tile: warp w takes tile rows w and w + 8 together.
  const float* rows[2];
  bool valid[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = warp + 8 * j;
    valid[j] = r < nt;
    rows[j] = a.logits + static_cast<size_t>(t0 + (valid[j] ? r : 0)) * E;
  }
  TopkSel sel[2];
  warp_topk_n<2>(rows, valid, E, a.K, lane, nullptr, sel);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int t = t0 + warp + 8 * j;
    if (valid[j] && lane < a.K) {
      a.topk_idx[static_cast<size_t>(t) * a.K + lane] = sel[j].e;
      a.topk_w[static_cast<size_t>(t) * a.K + lane] = sel[j].w;
    }
  }
  if (tid == 0) a.tg_ctr[blockIdx.y] = 0;
}

// ---------------------------------------------------------------- combine
// x_out = x_in + (sum_k w_tk y_{slot(t,k)}) + y_shared(t), one float4 of
// outputs per thread; the sum runs in selection order, then the shared row,
// then the residual (the same order as the expert kernel's own combine).
__global__ void __launch_bounds__(256) k_combine(CombineArgs a) {
  pdl_wait();
  pdl_trigger();
  const int q = a.H >> 2;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.M * q) return;
  const int t = i / q;
  const size_t col = static_cast<size_t>(i - t * q) * 4;
  const size_t H = a.H;
  const int K = a.K, MK = a.M * a.K;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < K; k0 += 8) {
    int r[8];
    float wk[8];
    float4 y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool v = k0 + j < K;
      r[j] = v ? a.tok_slot[t * K + k0 + j] : MK + t;
      wk[j] = v ? a.topk_w[t * K + k0 + j] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __ldcg(reinterpret_cast<const float4*>(a.yslot + static_cast<size_t>(r[j]) * H + col));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (k0 + j < K) {
        acc.x = fmaf(wk[j], y[j].x, acc.x);
        acc.y = fmaf(wk[j], y[j].y, acc.y);
        acc.z = fmaf(wk[j], y[j].z, acc.z);
        acc.w = fmaf(wk[j], y[j].w, acc.w);
      }
    }
  }
  const float4 ys = __ldcg(reinterpret_cast<const float4*>(a.yslot + static_cast<size_t>(MK + t) * H + col));
  const float4 xi = *reinterpret_cast<const float4*>(a.x_in + static_cast<size_t>(t) * H + col);
  acc.x += ys.x;
  acc.y += ys.y;
  acc.z += ys.z;
  acc.w += ys.w;
  float4 o;
  o.x = xi.x + acc.x;
  o.y = xi.y + acc.y;
  o.z = xi.z + acc.z;
  o.w = xi.w + acc.w;
  *reinterpret_cast<float4*>(a.x_out + static_cast<size_t>(t) * H + col) = o;
}

// Combine + the next layer's input normalisation, one token per CTA of 512
// threads: every thread combines one float4 of the row (the same arithmetic
// as k_combine; H <= 2,048) and stages it in shared memory; warp 0 then takes the row in
// the router's layout (16 float4 per lane) for rstd_row16, so the normed
// row is bit-identical to the one the routing kernel would compute, and all
// threads write it as bf16.
__global__ void __launch_bounds__(512) k_combine_norm(CombineArgs a) {
  __shared__ __align__(16) float s_row[kRouteChunk];
  __shared__ float s_rs;
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int H = a.H, K = a.K, MK = a.M * a.K;
  const int q = H >> 2;
  for (int f = threadIdx.x; f < q; f += blockDim.x) {
    const size_t col = static_cast<size_t>(f) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < K; k0 += 8) {
      int r[8];
      float wk[8];
      float4 y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool v = k0 + j < K;
        r[j] = v ? a.tok_slot[t * K + k0 + j] : MK + t;
        wk[j] = v ? a.topk_w[t * K + k0 + j] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        y[j] = __ldcg(reinterpret_cast<const float4*>(a.yslot + static_cast<size_t>(r[j]) * H + col));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j < K) {
          acc.x = fmaf(wk[j], y[j].x, acc.x);
          acc.y = fmaf(wk[j], y[j].y, acc.y);
          acc.z = fmaf(wk[j], y[j].z, acc.z);
          acc.w = fmaf(wk[j], y[j].w, acc.w);
        }
      }
    }
    const float4 ys = __ldcg(reinterpret_cast<const float4*>(a.yslot + static_cast<size_t>(MK + t) * H + col));
    const float4 xi = *reinterpret_cast<const float4*>(a.x_in + static_cast<size_t>(t) * H + col);
    acc.x += ys.x;
    acc.y += ys.y;
    acc.z += ys.z;
    acc.w += ys.w;
    float4 o;
    o.x = xi.x + acc.x;
    o.y = xi.y + acc.y;
    o.z = xi.z + acc.z;
    o.w = xi.w + acc.w;
    *reinterpret_cast<float4*>(a.x_out + static_cast<size_t>(t) * H + col) = o;
    *reinterpret_cast<float4*>(s_row + col) = o;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float4 xv[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int col = lane * 4 + 128 * c;
      xv[c] = col < H ? *reinterpret_cast<const float4*>(s_row + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float rs = rstd_row16(xv, H, a.eps);
    if (lane == 0) s_rs = rs;
  }
  __syncthreads();
  const float rs = s_rs;
  for (int f = threadIdx.x; f < q; f += blockDim.x) {
    const float4 o = *reinterpret_cast<const float4*>(s_row + static_cast<size_t>(f) * 4);
    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * rs, o.y * rs);
    __nv_bfloat162 hi = __floats2bfloat162_rn(o.z * rs, o.w * rs);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(a.xn_out + static_cast<size_t>(t) * H + static_cast<size_t>(f) * 4) = pk;
  }
}

// ---------------------------------------------------------------- launches

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  const int n = a.M * (a.H >> 2);
  return launch_kernel(k_combine, dim3((n + 255) / 256), dim3(256), 0, s, pdl, a);
}


cudaError_t launch_combine_norm(const CombineArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(k_combine_norm, dim3(a.M), dim3(512), 0, s, pdl, a);
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(k_embed, dim3(a.M), dim3(256), 0, s, pdl, a);
}

cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(k_rmsnorm, dim3((a.M + 7) / 8), dim3(256), 0, s, pdl, a);
}

size_t route_smem_bytes(int H) {
  const size_t ld = static_cast<size_t>(std::min(H, kRouteChunk)) + 8;
  return (kRouteTileExperts + kRouteTileTokens) * ld * sizeof(bf16) +
         (8 * kRouteTileTokens * kRouteTileExperts + 16) * sizeof(float) + 2 * sizeof(uint64_t);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = route_smem_bytes(a.H);
  cudaError_t e = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.E + kRouteTileExperts - 1) / kRouteTileExperts, (a.M + kRouteTileTokens - 1) / kRouteTileTokens);
  return launch_kernel(k_route, grid, dim3(256), smem, s, pdl, a);
}


}  // namespace clover
