// Input assembly, RMSNorm, router with softmax top-k, and the token->expert
// permutation with the gather of normed inputs.
//
// Follows "Clover-35B-A3B: how a diffusion model gets to 680 tokens a second,
// read from its files": section "What Clover is" (256 routed experts, each
// token routed to 8, block of mask tokens), section "The expert selection"
// (per-token top-8 routing probabilities) and section "How it writes",
// step 1 (the block re-enters with mask-token embeddings until committed).
#include <math.h>

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
// Grid (ceil(E/8), ceil(M/8)). Each CTA normalises its 8 tokens (one warp
// per token), writes the bf16 normed rows (expert group 0 only) and the
// router logits of its 8 experts. The last CTA to finish a token group then
// takes softmax top-k for those tokens: selection by descending logit with
// the lower expert id first on ties, weights = softmax over the selected
// logits (= top-k probabilities renormalised to sum to one).
__global__ void __launch_bounds__(256) k_route(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* w = reinterpret_cast<bf16*>(smem);  // [8][H]
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kRouteExperts;
  const int ne = min(kRouteExperts, a.E - e0);
  const int t0 = blockIdx.y * kRouteTokens;
  const int t1 = min(a.M, t0 + kRouteTokens);  // one token per warp
  const int H = a.H;

  // Router rows do not depend on earlier kernels: stage them before waiting.
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.wr + static_cast<size_t>(e0) * H);
    uint4* dst = reinterpret_cast<uint4*>(w);
    const int n16 = ne * H / 8;
    for (int i = tid; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  for (int t = t0 + warp; t < t1; t += 8) {
    const float* xr = a.x + static_cast<size_t>(t) * H;
    const float rstd = row_rstd(xr, H, a.eps, lane);
    const float mine = warp_router_dots<kRouteExperts>(
        xr, rstd, w, ne, H, lane, blockIdx.x == 0 ? a.xn_rows + static_cast<size_t>(t) * H : nullptr);
    if (lane < ne) {
      const int e = e0 + lane;
      a.logits[static_cast<size_t>(t) * a.E + e] = mine + (a.bias ? a.bias[e] : 0.f);
    }
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&a.tg_ctr[blockIdx.y], 1);
    s_last = (old == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Top-k for this token group (one warp per token; lane l holds experts
  // l, l+32, ..., up to 256).
  for (int t = t0 + warp; t < t1; t += 8) {
    const TopkSel sel = warp_topk(a.logits + static_cast<size_t>(t) * a.E, a.E, a.K, lane);
    if (lane < a.K) {
      a.topk_idx[static_cast<size_t>(t) * a.K + lane] = sel.e;
      a.topk_w[static_cast<size_t>(t) * a.K + lane] = sel.w;
    }
  }
  if (tid == 0) a.tg_ctr[blockIdx.y] = 0;
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 256).
__device__ __forceinline__ int block_excl_scan_256(int v, int* s_tmp /*[8]*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < 8 ? s_tmp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < 8) s_tmp[lane] = wi - wv;  // exclusive warp offsets
    if (lane == 7) s_tmp[8] = wi;         // total
  }
  __syncthreads();
  const int res = s_tmp[warp] + incl - v;
  *total = s_tmp[8];
  __syncthreads();
  return res;
}

// ------------------------------------------------------------------- perm
// Every CTA rebuilds the same token->expert permutation from the top-k ids
// (cheap, and it avoids a grid-wide barrier): per-expert token bitmasks, a
// scan over experts for the row offsets, and each (token, slot)'s row =
// offset of its expert + number of lower tokens routed to that expert. Rows
// of one expert are therefore in token order. CTA 0 publishes the metadata
// and resets the expert kernel's counters; all CTAs gather rows of the
// normed input into expert-grouped order.
__global__ void __launch_bounds__(256) k_perm(PermArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  int* s_idx = reinterpret_cast<int*>(smem);  // [M*K]
  int* s_row_tok = s_idx + a.M * a.K;         // [M*K]
  __shared__ uint32_t s_bm[kMaxExperts][kMaxTokens / 32];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_tmp[9];
  const int tid = threadIdx.x;
  const int MK = a.M * a.K;
  const int nw = (a.M + 31) >> 5;

  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < MK; i += blockDim.x) {
    const int e = a.topk_idx[i];
    s_idx[i] = e < 0 ? 0 : (e >= a.E ? a.E - 1 : e);  // ids come from k_route; clamp keeps smem indexing safe
  }
  for (int i = tid; i < kMaxExperts * (kMaxTokens / 32); i += blockDim.x) (&s_bm[0][0])[i] = 0u;
  __syncthreads();
  for (int i = tid; i < MK; i += blockDim.x) {
    const int e = s_idx[i], t = i / a.K;
    atomicOr(&s_bm[e][t >> 5], 1u << (t & 31));
  }
  __syncthreads();
  int c = 0;
  if (tid < a.E)
    for (int wd = 0; wd < nw; ++wd) c += __popc(s_bm[tid][wd]);
  int total = 0;
  const int off = block_excl_scan_256(c, s_tmp, &total);
  const int apos = block_excl_scan_256(c > 0 ? 1 : 0, s_tmp, &total);
  if (tid < a.E) s_off[tid] = off;
  __syncthreads();
  for (int i = tid; i < MK; i += blockDim.x) {
    const int e = s_idx[i], t = i / a.K;
    const int wd = t >> 5, bit = t & 31;
    int pre = __popc(s_bm[e][wd] & ((1u << bit) - 1u));
    for (int j = 0; j < wd; ++j) pre += __popc(s_bm[e][j]);
    const int row = s_off[e] + pre;
    s_row_tok[row] = t;
    if (blockIdx.x == 0) a.tok_slot[i] = row;
  }
  if (blockIdx.x == 0) {
    if (tid < a.E) {
      a.cnt[tid] = c;
      a.off[tid] = off;
      if (c > 0) a.act[apos] = tid;
    }
    if (tid == 0) {
      *a.n_active = total;
      *a.unit_ctr = 0;
    }
    for (int i = tid; i <= a.E; i += blockDim.x) a.gu_done[i] = 0;
    for (int i = tid; i < a.H / 128; i += blockDim.x) a.dn_done[i] = 0;
    if (a.out_idx)
      for (int i = tid; i < MK; i += blockDim.x) a.out_idx[i] = s_idx[i];
    if (a.out_w)
      for (int i = tid; i < MK; i += blockDim.x) a.out_w[i] = a.topk_w[i];
  }
  __syncthreads();
  const size_t H = a.H;
  for (int r = blockIdx.x; r < MK; r += gridDim.x) {
    const int t = s_row_tok[r];
    const uint4* src = reinterpret_cast<const uint4*>(a.xg + static_cast<size_t>(MK + t) * H);
    uint4* dst = reinterpret_cast<uint4*>(a.xg + static_cast<size_t>(r) * H);
    for (int i = tid; i < static_cast<int>(H / 8); i += blockDim.x) dst[i] = src[i];
  }
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

// ---------------------------------------------------------------- launches

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  const int n = a.M * (a.H >> 2);
  return launch_kernel(k_combine, dim3((n + 255) / 256), dim3(256), 0, s, pdl, a);
}


cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(k_embed, dim3(a.M), dim3(256), 0, s, pdl, a);
}

cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(k_rmsnorm, dim3((a.M + 7) / 8), dim3(256), 0, s, pdl, a);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = static_cast<size_t>(kRouteExperts) * a.H * sizeof(bf16);
  cudaError_t e = cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.E + kRouteExperts - 1) / kRouteExperts, (a.M + kRouteTokens - 1) / kRouteTokens);
  return launch_kernel(k_route, grid, dim3(256), smem, s, pdl, a);
}

cudaError_t launch_perm(const PermArgs& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = static_cast<size_t>(2) * a.M * a.K * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(k_perm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(k_perm, dim3(grid), dim3(256), smem, s, pdl, a);
}

}  // namespace clover
