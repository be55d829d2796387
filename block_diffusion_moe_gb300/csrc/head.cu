// Untied output head fused with the per-position statistics and the
// low-confidence unmask rule.
//
// Follows "Clover-35B-A3B: how a diffusion model gets to 680 tokens a second,
// read from its files": section "What Clover is" (the 248,320 x 2,048 head is
// untied and read in full at every step; mask token 151669; low-confidence
// threshold 0.95) and section "How it writes", steps 2-3 (the mask token's
// logit is minus infinity; every still-masked slot above the threshold is
// committed, else the single most confident one).
//
// Each CTA owns vocabulary tiles blockIdx.x, blockIdx.x + G, ...; a tile is
// 128 head rows (the M = 128 side of tcgen05.mma) against all positions (the
// N side). The epilogue turns each 128 x N accumulator into per-position
// (max, sum of exp relative to the max, argmax) and folds it into a running
// per-CTA state, so the logits never leave the SM. A second, small launch
// (k_head_merge) merges the G partial states, one warp per position
// (maximum first, then the sums rescaled to it, combined in a fixed order),
// derives log-sum-exp and the maximum probability, and its last CTA applies
// the unmask rule to every block of positions. Ties in the argmax go to the
// lowest vocabulary id at every level.
//
// The accept form (section "Two ways to run it": self-speculative decoding
// keeps the longest prefix of drafts that the causal pass accepts, plus one
// token at the boundary; exact keeps a draft equal to the argmax, threshold
// one whose probability is at least min(ratio, delta e^-H)) carries two more
// per-position quantities through the same pipeline: t = sum of
// e^(z - m) (z - m), from which the entropy is H = ln s - t / s, and the
// draft token's logit. The merge launch's last CTA then takes the accept
// test per block of rows instead of the unmask rule.
#include <math.h>

#include "kernels.cuh"
#include "launch.cuh"
#include "sm100.cuh"

namespace clover {

namespace {

struct HeadSmem {
  uint8_t* ring;  // stages x (A tile 16 KB + B tile nb x 128 B)
  float* wp_m;    // [4][nb]
  float* wp_s;    // [4][nb]
  int* wp_a;      // [4][nb]
  float* run_m;   // [nb]
  float* run_s;   // [nb]
  int* run_a;     // [nb]
  float* alpha;   // [nb]
  float* wp_t;    // [4][nb] accept form only
  float* wp_zd;   // [4][nb]
  float* run_t;   // [nb]
  float* run_zd;  // [nb]
  float* tr;      // [4][32][33] per-warp transpose tiles
  uint64_t *full, *empty, *tfull, *tempty, *drain;
  uint32_t* tmem_slot;
  volatile uint32_t* abort;
  volatile int* s_ok;
  uint32_t half_bytes;   // one K group: A tile 16 KiB + B tile nb x 128 B
  uint32_t stage_bytes;  // kg K groups
};

__device__ __forceinline__ HeadSmem carve(uint8_t* raw, const HeadArgs& p, int nb, bool accept) {
  HeadSmem s;
  const uint32_t r = smem_u32(raw);
  uint8_t* base = raw + ((1024u - (r & 1023u)) & 1023u);
  s.half_bytes = kATileBytes + static_cast<uint32_t>(nb) * 128u;
  s.stage_bytes = s.half_bytes * static_cast<uint32_t>(p.kg);
  s.ring = base;
  float* f = reinterpret_cast<float*>(base + static_cast<size_t>(p.stages) * s.stage_bytes);
  s.wp_m = f;
  s.wp_s = s.wp_m + 4 * nb;
  s.wp_a = reinterpret_cast<int*>(s.wp_s + 4 * nb);
  s.run_m = reinterpret_cast<float*>(s.wp_a + 4 * nb);
  s.run_s = s.run_m + nb;
  s.run_a = reinterpret_cast<int*>(s.run_s + nb);
  s.alpha = reinterpret_cast<float*>(s.run_a + nb);
  s.wp_t = s.alpha + nb;
  s.wp_zd = s.wp_t + (accept ? 4 * nb : 0);
  s.run_t = s.wp_zd + (accept ? 4 * nb : 0);
  s.run_zd = s.run_t + (accept ? nb : 0);
  s.tr = s.run_zd + (accept ? nb : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.tr + 4 * 32 * 33);  // nb % 16 == 0 keeps 8-byte alignment
  s.full = bars;
  s.empty = s.full + p.stages;
  s.tfull = s.empty + p.stages;
  s.tempty = s.tfull + 2;
  s.drain = s.tempty + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
  s.abort = s.tmem_slot + 1;
  s.s_ok = reinterpret_cast<volatile int*>(s.tmem_slot + 2);
  return s;
}

// Folds the partial (m2, s2, a2) into (m, s, a): m = max, s rescaled to the
// new max, a = lowest id attaining the max.
__device__ __forceinline__ void lse_merge(float& m, float& s, int& a, float m2, float s2, int a2) {
  if (m2 > m) {
    s = s * expf(m - m2) + s2;  // expf(-inf) = 0 covers an empty (m = -inf) state
    m = m2;
    a = a2;
  } else if (m2 == m) {
    s += s2;
    a = min(a, a2);
  } else {
    s += s2 * expf(m2 - m);
  }
}

// lse_merge that also carries t = sum e^(z - m) (z - m), re-expressed at
// the merged maximum: t' = e^(m - m') (t + (m - m') s). Empty states (m =
// -inf, s = t = 0) are skipped, so no -inf x 0 product arises.
__device__ __forceinline__ void lse_merge_t(float& m, float& s, float& t, int& a, float m2, float s2, float t2,
                                            int a2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    t = t2;
    a = a2;
  } else if (m2 > m) {
    const float f = expf(m - m2);
    t = f * (t + (m - m2) * s) + t2;
    s = s * f + s2;
    m = m2;
    a = a2;
  } else if (m2 == m) {
    s += s2;
    t += t2;
    a = min(a, a2);
  } else {
    const float f = expf(m2 - m);
    t += f * (t2 + (m2 - m) * s2);
    s += s2 * f;
  }
}

// Weight (A) and position (B) tiles for the MMA. The head's weights are
// written by no kernel, so the A tiles of the first ring's worth of stages
// are requested before the dependency wait (overlapping the normalisation
// kernel that writes the positions); their B tiles follow after it.
__device__ void head_producer(const HeadArgs& p, const HeadSmem& s, int nb) {
  const uint64_t pol_w = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  const int nk = p.H >> 6;
  // Each CTA walks the K chunks from its own starting point, so that the
  // CTAs' simultaneous requests do not all share the same offset within the
  // head rows (which would concentrate them on few DRAM channels). The MMA
  // consumes stages in issue order; only the accumulation order changes.
  const int kg = p.kg;
  const int rot = kg * static_cast<int>((blockIdx.x * 7u) % static_cast<unsigned>(nk / kg));
  const int steps_per_tile = nk / kg;
  const int my_tiles = (p.n_tiles > static_cast<int>(blockIdx.x)) ? (p.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int n_steps = my_tiles * steps_per_tile;
  // (tile, first K group) of pipeline step i
  auto coords = [&](int i, int& tile, int& kc) {
    const int t = i / steps_per_tile, k0 = (i - t * steps_per_tile) * kg;
    tile = blockIdx.x + t * gridDim.x;
    kc = (k0 + rot < nk) ? k0 + rot : k0 + rot - nk;
  };
  auto load_a = [&](int st, int tile, int kc) {
    const uint32_t dst0 = smem_u32(s.ring + static_cast<size_t>(st) * s.stage_bytes);
    for (int h = 0; h < kg; ++h)
      tma_load_2d(dst0 + h * s.half_bytes, &p.tm_w, &s.full[st], (kc + h) * 64, tile * 128, pol_w);
  };
  auto load_b = [&](int st, int kc) {
    const uint32_t dst0 = smem_u32(s.ring + static_cast<size_t>(st) * s.stage_bytes);
    for (int h = 0; h < kg; ++h)
      for (int i = 0; i < nb; i += p.x_box)
        tma_load_2d(dst0 + h * s.half_bytes + kATileBytes + i * 128, &p.tm_x, &s.full[st], (kc + h) * 64, i, pol_x);
  };
  // first pass over the ring: the stages are free, nothing to wait for
  const int pre = min(p.stages, n_steps);
  for (int i = 0; i < pre; ++i) {
    int tile, kc;
    coords(i, tile, kc);
    mbar_arrive_expect_tx(&s.full[i], s.stage_bytes);
    load_a(i, tile, kc);
  }
  pdl_wait();
  for (int i = 0; i < pre; ++i) {
    int tile, kc;
    coords(i, tile, kc);
    load_b(i, kc);
  }
  int st = pre == p.stages ? 0 : pre;
  uint32_t ph = pre == p.stages ? 1u : 0u;
  uint32_t issued = (pre >= 32) ? 0xffffffffu : ((1u << pre) - 1u), parity_bits = 0;
  for (int i = pre; i < n_steps; ++i) {
    int tile, kc;
    coords(i, tile, kc);
    if (!mbar_wait(&s.empty[st], ph ^ 1u, s.abort)) {
      atomicOr(p.err, kErrMbarTimeout);
      *s.abort = 1u;
      break;
    }
    mbar_arrive_expect_tx(&s.full[st], s.stage_bytes);
    load_a(st, tile, kc);
    load_b(st, kc);
    issued |= 1u << st;
    parity_bits = (parity_bits & ~(1u << st)) | (ph << st);
    if (++st == p.stages) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (*s.abort) {
    for (int i = 0; i < p.stages; ++i)
      if (issued & (1u << i)) mbar_wait_for(&s.full[i], (parity_bits >> i) & 1u, 200000000ull);
  }
}

__device__ void head_mma(const HeadArgs& p, const HeadSmem& s, int nb, uint32_t tmem_base) {
  const int nk = p.H >> 6;
  const uint32_t idesc = umma_idesc_bf16(128, nb);
  int st = 0;
  uint32_t ph = 0;
  int it = 0;
  bool ok = true;
  for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++it) {
    const int acc = it & 1;
    const uint32_t apar = (it >> 1) & 1;
    if (!mbar_wait(&s.tempty[acc], apar ^ 1u, s.abort)) {
      atomicOr(p.err, kErrMbarTimeout);
      *s.abort = 1u;
      break;
    }
    tc_fence_after();
    const uint32_t d = tmem_base + static_cast<uint32_t>(acc) * 256u;
    for (int kc = 0; kc < nk; kc += p.kg) {
      if (!mbar_wait(&s.full[st], ph, s.abort)) {
        atomicOr(p.err, kErrMbarTimeout);
        *s.abort = 1u;
        ok = false;
        break;
      }
      tc_fence_after();
      for (int h = 0; h < p.kg; ++h) {
        const uint32_t a_addr = smem_u32(s.ring + static_cast<size_t>(st) * s.stage_bytes + h * s.half_bytes);
        const uint64_t ad = umma_desc_sw128(a_addr);
        const uint64_t bd = umma_desc_sw128(a_addr + kATileBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16(d, ad + static_cast<uint64_t>(2 * k), bd + static_cast<uint64_t>(2 * k), idesc,
                    (kc | h | k) != 0 ? 1u : 0u);
      }
      umma_commit(&s.empty[st]);
      if (++st == p.stages) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (ok) umma_commit(&s.tfull[acc]);
  }
  umma_commit(s.drain);
  mbar_wait_for(s.drain, 0, 200000000ull);
}

// Per tile, each epilogue warp owns 32 vocabulary rows (its TMEM lane
// quarter) of the 128 x nb accumulator. It moves them 32 token columns at a
// time through a padded shared-memory tile so that lane j then walks column j
// serially: tile max, first row reaching it, and the sum of exp(z - max).
// That folds into a running (max, sum, argmax) per column held in the lane's
// registers across all of the CTA's tiles; warps never wait on each other
// until the end. The accept form also folds t and picks the draft's logit
// out of the transposed tile.
template <bool kAccept>
__device__ void head_epilogue(const HeadArgs& p, const HeadSmem& s, int nb, uint32_t tmem_base) {
  constexpr int kMaxChunks = kTileTokens / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const int etid = threadIdx.x - 64;  // 0..127
  const int nch = (nb + 31) >> 5;
  float* tr = s.tr + q * (32 * 33);
  float rm[kMaxChunks], rs[kMaxChunks], al[kMaxChunks], rt[kMaxChunks], rzd[kMaxChunks];
  int ra[kMaxChunks], dr[kMaxChunks];
#pragma unroll
  for (int ch = 0; ch < kMaxChunks; ++ch) {
    const int c = ch * 32 + lane;
    rm[ch] = -INFINITY;
    rs[ch] = 0.f;
    ra[ch] = 0x7fffffff;
    al[ch] = (c < p.M && p.alpha != nullptr) ? p.alpha[c] : 1.0f;
    rt[ch] = 0.f;
    rzd[ch] = -INFINITY;
    dr[ch] = (kAccept && c < p.M) ? p.draft[c] : -1;
  }
  bool ok = true;
  int it = 0;
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++it) {
    const int acc = it & 1;
    const uint32_t apar = (it >> 1) & 1;
    int good = 1;
    if (lane == 0) {
      good = mbar_wait(&s.tfull[acc], apar, s.abort) ? 1 : 0;
      if (!good) {
        atomicOr(p.err, kErrMbarTimeout);
        *s.abort = 1u;
      }
    }
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc) * 256u;
    const int vid = tile * 128 + row;
    const bool valid_row = (vid < p.V) && (vid != p.mask_id);
    const int row0 = tile * 128 + q * 32;
#pragma unroll
    for (int ch = 0; ch < kMaxChunks; ++ch) {
      if (ch < nch) {
        float v[16];
        __syncwarp();
        tmem_ld16(tb + ch * 32, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) tr[lane * 33 + j] = valid_row ? v[j] : -INFINITY;
        if (ch * 32 + 16 < nb) {
          tmem_ld16(tb + ch * 32 + 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) tr[lane * 33 + 16 + j] = valid_row ? v[j] : -INFINITY;
        }
        __syncwarp();
        if (ch * 32 + lane < nb) {
          float z[32];
          float m = -INFINITY;
          int a = 0x7fffffff;
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            const float raw = tr[r * 33 + lane];
            z[r] = (raw == -INFINITY) ? -INFINITY : raw * al[ch];
            if (z[r] > m) {
              m = z[r];
              a = row0 + r;
            }
          }
          float sum = 0.f, t = 0.f;
          if (m != -INFINITY) {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              const float d = z[r] - m;
              const float e = expf(d);
              sum += e;
              // a row at -inf has e = 0; the clamp keeps 0 x -inf out
              if (kAccept) t = fmaf(e, fmaxf(d, -1e30f), t);
            }
          }
          if (kAccept) {
            lse_merge_t(rm[ch], rs[ch], rt[ch], ra[ch], m, sum, t, a);
            const int dj = dr[ch] - row0;
            if (dj >= 0 && dj < 32) {
              const float raw = tr[dj * 33 + lane];  // -inf for the mask token
              rzd[ch] = (raw == -INFINITY) ? -INFINITY : raw * al[ch];
            }
          } else {
            lse_merge(rm[ch], rs[ch], ra[ch], m, sum, a);
          }
        }
      }
    }
    // this warp is done reading the accumulator
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.tempty[acc]);
  }
  // Merge the four warps (rows 0-31, 32-63, 64-95, 96-127 of every tile).
#pragma unroll
  for (int ch = 0; ch < kMaxChunks; ++ch) {
    const int c = ch * 32 + lane;
    if (ch < nch && c < nb) {
      s.wp_m[q * nb + c] = rm[ch];
      s.wp_s[q * nb + c] = rs[ch];
      s.wp_a[q * nb + c] = ra[ch];
      if (kAccept) {
        s.wp_t[q * nb + c] = rt[ch];
        s.wp_zd[q * nb + c] = rzd[ch];
      }
    }
  }
  named_bar_sync(1, 128);
  for (int c = etid; c < nb; c += 128) {
    float m = -INFINITY, sm = 0.f, t = 0.f, zd = -INFINITY;
    int a = 0x7fffffff;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (kAccept) {
        lse_merge_t(m, sm, t, a, s.wp_m[w * nb + c], s.wp_s[w * nb + c], s.wp_t[w * nb + c], s.wp_a[w * nb + c]);
        zd = fmaxf(zd, s.wp_zd[w * nb + c]);
      } else {
        lse_merge(m, sm, a, s.wp_m[w * nb + c], s.wp_s[w * nb + c], s.wp_a[w * nb + c]);
      }
    }
    s.run_m[c] = m;
    s.run_s[c] = sm;
    s.run_a[c] = a;
    if (kAccept) {
      s.run_t[c] = t;
      s.run_zd[c] = zd;
    }
  }
  (void)ok;
  // Leave together if any role gave up (the decision is broadcast so that no
  // epilogue thread is left waiting on the named barrier).
  named_bar_sync(1, 128);
  if (etid == 0) *s.s_ok = (*s.abort == 0u) ? 1 : 0;
  named_bar_sync(1, 128);
  if (!*s.s_ok) return;

  // Publish this CTA's partial state; k_head_merge combines them.
  for (int n = etid; n < p.M; n += 128) {
    const size_t g = static_cast<size_t>(blockIdx.x) * p.M + n;
    p.part_m[g] = s.run_m[n];
    p.part_s[g] = s.run_s[n];
    p.part_a[g] = s.run_a[n];
    if (kAccept) {
      p.part_t[g] = s.run_t[n];
      p.part_zd[g] = s.run_zd[n];
    }
  }
}

}  // namespace

template <bool kAccept>
__global__ void __launch_bounds__(kHeadThreads, 1) k_head(const __grid_constant__ HeadArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const int nb = (p.M + 15) & ~15;
  const HeadSmem s = carve(smem_raw, p, nb, kAccept);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(s.drain, 1);
    *s.abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_w);
    tma_prefetch_desc(&p.tm_x);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s.tmem_slot;
  // (the producer thread waits for the previous kernel itself, after it has
  // requested the weight tiles that do not depend on it)
  if (!(warp == 0 && lane == 0)) pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) head_producer(p, s, nb);
  } else if (warp == 1) {
    if (lane == 0) head_mma(p, s, nb, tmem_base);
  } else {
    head_epilogue<kAccept>(p, s, nb, tmem_base);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Merge of the G per-CTA partial states of one k_head launch, one warp per
// position: each lane takes CTAs lane, lane + 32, ..., first the maximum and
// its token (ties to the lower id), then the sums rescaled to that maximum;
// the lanes' results combine in a fixed butterfly, so the outcome does not
// depend on timing. The last CTA to finish then applies the unmask rule (or
// the accept test) to every block of positions, reading the per-position
// decision inputs back from the workspace.
template <bool kAccept>
__global__ void __launch_bounds__(256) k_head_merge(const __grid_constant__ HeadArgs p) {
  constexpr int kPer = kHeadMaxCtas / 32;  // partials per lane at most
  __shared__ int s_last;
  __shared__ int s_counts[2];
  __shared__ float s_dm[kTileTokens];
  __shared__ float s_ds[kTileTokens];
  __shared__ int s_da[kTileTokens];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.n_parts;
  const int n = blockIdx.x * 8 + warp;
  if (n < p.M) {
    // every partial of this lane in registers, all loads in flight at once
    float vm[kPer], vs[kPer], vt[kPer], vz[kPer];
    int va[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int b = lane + 32 * i;
      vm[i] = -INFINITY;
      vs[i] = vt[i] = 0.f;
      vz[i] = -INFINITY;
      va[i] = 0x7fffffff;
      if (b < G) {
        const size_t g = static_cast<size_t>(b) * p.M + n;
        vm[i] = __ldcg(p.part_m + g);
        vs[i] = __ldcg(p.part_s + g);
        va[i] = __ldcg(p.part_a + g);
        if (kAccept) {
          vt[i] = __ldcg(p.part_t + g);
          vz[i] = __ldcg(p.part_zd + g);
        }
      }
    }
    float m = -INFINITY;
    int a = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (vm[i] > m || (vm[i] == m && va[i] < a)) {
        m = vm[i];
        a = va[i];
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
      if (m2 > m || (m2 == m && a2 < a)) {
        m = m2;
        a = a2;
      }
    }
    float sm = 0.f, t = 0.f, zd = -INFINITY;
    if (m != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        if (vm[i] == -INFINITY) continue;  // an empty partial (s = t = 0), or none
        const float f = expf(vm[i] - m);
        sm += vs[i] * f;
        if (kAccept) {
          t += f * (vt[i] + (vm[i] - m) * vs[i]);
          zd = fmaxf(zd, vz[i]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (kAccept) {
        t += __shfl_xor_sync(0xffffffffu, t, o);
        zd = fmaxf(zd, __shfl_xor_sync(0xffffffffu, zd, o));
      }
    }
    if (lane == 0) {
      const float lse = m + logf(sm);
      const float pmax = 1.0f / sm;  // = exp(m - lse)
      if (p.argmax) p.argmax[n] = a;
      if (p.max_logit) p.max_logit[n] = m;
      if (p.lse) p.lse[n] = lse;
      if (p.max_prob) p.max_prob[n] = pmax;
      if (kAccept) {
        const float ent = fmaxf(logf(sm) - t / sm, 0.f);  // t <= 0
        const float pd = expf(zd - lse);                   // 0 for a draft never seen
        if (p.entropy) p.entropy[n] = ent;
        if (p.p_draft) p.p_draft[n] = pd;
        p.dec_m[n] = pd;
        p.dec_s[n] = ent;
      } else {
        p.dec_m[n] = pmax;
      }
      p.dec_a[n] = a;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // (cumulative over the CTA's stores ordered by the barrier)
    const int old = atomicAdd(p.done_ctr, 1);
    __threadfence();
    s_last = (old == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
    s_counts[0] = 0;
    s_counts[1] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  // The last CTA: every position's decision inputs into shared memory at
  // once (M <= kTileTokens per launch), then one thread per block.
  for (int i = threadIdx.x; i < p.M; i += blockDim.x) {
    const float dm = __ldcg(p.dec_m + i);
    const int da = __ldcg(p.dec_a + i);
    const float ds = kAccept ? __ldcg(p.dec_s + i) : 0.f;
    s_dm[i] = dm;
    s_da[i] = da;
    s_ds[i] = ds;
  }
  __syncthreads();
  if (kAccept) {
    // Accept test, one thread per block of rows: the longest prefix of
    // accepted drafts, then the boundary row's argmax.
    const int nblk = p.M / p.block;
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
      const int p0 = b * p.block;
      int r = 0;
      while (r < p.block - 1) {
        const int i = p0 + r;
        const bool acc = (p.rule == 0) ? (p.draft[i] == s_da[i])
                                       : (s_dm[i] >= fminf(p.ratio, p.delta * expf(-s_ds[i])));
        if (!acc) break;
        ++r;
      }
      p.accept_len[b] = r;
      for (int j = 0; j < p.block; ++j)
        p.out_tokens[p0 + j] = (j < r) ? p.draft[p0 + j] : (j == r ? s_da[p0 + j] : -1);
    }
    __syncthreads();
    if (threadIdx.x == 0) *p.done_ctr = 0;
    return;
  }
  // Unmask rule, one thread per block of positions.
  const int nblk = (p.M + p.block - 1) / p.block;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    const int p0 = b * p.block, p1 = min(p.M, p0 + p.block);
    int n_commit = 0, best = -1;
    float best_p = 0.f;
    bool bad = false;
    for (int i = p0; i < p1; ++i) {
      if (!p.masked[i]) {
        // a committed slot must hold a vocabulary id; report one that does not
        const int tk = p.tokens[i];
        bad |= (tk < 0 || tk >= p.V);
        continue;
      }
      const float pm = s_dm[i];
      if (pm > p.threshold) ++n_commit;
      if (best < 0 || pm > best_p) {
        best = i;
        best_p = pm;
      }
    }
    int still = 0, done = 0;
    for (int i = p0; i < p1; ++i) {
      if (!p.masked[i]) continue;
      const bool c = (n_commit > 0) ? (s_dm[i] > p.threshold) : (i == best);
      if (c) {
        p.tokens[i] = s_da[i];
        p.masked[i] = 0;
        ++done;
      } else {
        ++still;
      }
    }
    atomicAdd(&s_counts[0], done);
    atomicAdd(&s_counts[1], still);
    if (bad) atomicOr(p.err, kErrBadToken);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (p.n_committed) *p.n_committed = (p.accumulate ? *p.n_committed : 0) + s_counts[0];
    if (p.n_masked_left) *p.n_masked_left = (p.accumulate ? *p.n_masked_left : 0) + s_counts[1];
    *p.done_ctr = 0;
  }
}

size_t head_smem_bytes(int stages, int nb, bool accept, int kg) {
  return 1024 + static_cast<size_t>(stages) * kg * (kATileBytes + static_cast<size_t>(nb) * 128) +
         static_cast<size_t>(nb) * (4 * 12 + 12 + 4 + (accept ? 4 * 8 + 8 : 0)) + 4 * 32 * 33 * sizeof(float) +
         static_cast<size_t>(2 * stages + 5) * 8 + 64;
}

cudaError_t launch_head(const HeadArgs& a, bool accept, int grid, size_t smem, cudaStream_t s, bool pdl) {
  auto* k = accept ? k_head<true> : k_head<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(kHeadThreads), smem, s, pdl, a);
}

cudaError_t launch_head_merge(const HeadArgs& a, bool accept, cudaStream_t s, bool pdl) {
  auto* k = accept ? k_head_merge<true> : k_head_merge<false>;
  return launch_kernel(k, dim3((a.M + 7) / 8), dim3(256), 0, s, pdl, a);
}

}  // namespace clover
