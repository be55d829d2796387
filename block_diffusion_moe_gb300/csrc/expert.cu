// Grouped SwiGLU experts (routed + shared) with the weighted combine, as one
// persistent tcgen05 kernel per MoE sublayer.
//
// Follows "Clover-35B-A3B: how a diffusion model gets to 680 tokens a second,
// read from its files", section "What Clover is" (one expert = gate and up at
// 2,048 x 512, down at 512 x 2,048; one always-on shared expert) and section
// "The expert selection" (a block reads the union of its tokens' experts).
//
// Work is cut into equal-sized units that every CTA pulls from a global
// counter:
//   gate/up unit (expert a, slice s): A = 64 gate rows + the matching 64 up
//     rows (128 x H, 512 KB at H = 2048), B = the expert's gathered bf16
//     inputs; the epilogue forms h = silu(gate) * up, rounds it to bf16 and
//     stores its 64 columns of h.
//   down unit (expert a, slice j): A = rows j*128..j*128+127 of W_down
//     (128 x F, 128 KB), B = the expert's h rows; the epilogue stores the
//     unweighted expert output rows for those 128 hidden dims.
// Weights play the M = 128 side of tcgen05.mma and tokens the N side (N = the
// expert's token count rounded up to 16), so each selected expert's weights
// stream from HBM exactly once per call while the MMA shape stays legal for
// one or two tokens. All gate/up units come before all down units in the
// counter order; a down unit's activation loads wait (bounded) until the 8
// gate/up slices of its expert have published h, which cannot deadlock
// because those units were claimed earlier by running CTAs.
// The last down unit to finish a 128-wide hidden slice sums, for every token,
// its K weighted expert rows in selection order plus the shared expert row
// and adds them to the residual stream: a fixed summation order, so results
// do not depend on scheduling.
//
// Warp roles (224 threads): warp 0 lane 0 streams weights (A) with TMA,
// warp 1 owns TMEM and lane 0 issues the MMAs, warp 2 lane 0 streams
// activations (B) with TMA, warps 3..6 are the epilogue (each reads the TMEM
// lane quarter warp % 4). Two TMEM accumulators of 256 columns let the
// epilogue of one unit overlap the MMAs of the next.
//
// k_layer (at most 32 tokens) also does the layer's routing itself, so a
// whole MoE sublayer is one launch: every CTA normalises the tokens and
// computes the router logits of its share of the experts, one grid barrier
// publishes the logits, then every CTA takes the same top-k and permutation
// into shared memory. Its gate/up units use all the tokens' normed rows as
// the B operand (N = 32 at most) and keep only the routed columns, so no
// gather is needed.
#include <math.h>

#include "kernels.cuh"
#include "launch.cuh"
#include "routing.cuh"
#include "sm100.cuh"

namespace clover {

namespace {

constexpr int kUnitEnd = -1;
constexpr int kUnitAbort = -2;

struct Unit {
  int kind;   // 0 gate/up, 1 down
  int a;      // index of the active expert (fused kernel; 0 is the shared expert) or chunk (standalone)
  int e;      // expert id (E for the shared expert)
  int slice;  // F/64 slice (gate/up) or H/128 slice (down)
  int cnt;    // tokens of the expert (chunk)
  int off;    // first row of the expert (chunk) in the gathered buffers
  int pair;   // 1: slices slice and slice + 1 together (two accumulators sharing each B tile)
};

// Where a launch finds its routing: global tables written in the prologue
// of k_expert, or shared-memory tables built by k_layer itself.
struct Rt {
  const int* act;           // fused: active routed expert ids; standalone: expert id of each chunk
  const int* cnt;           // fused: [E] tokens per expert; standalone: rows of each chunk
  const int* off;           // fused: [E] first row per expert; standalone: first row of each chunk
  const uint32_t* mask;     // [E] token bitmask (dense mode)
  const int32_t* tok_slot;  // [M][K] row of each selection
  const float* topk_w;      // [M][K] weight of each selection
  int n_exp;                // fused: active routed experts + the shared expert; standalone: chunks
  int n_pair;               // standalone: the leading chunks whose units are paired (0: none)
  int dense;                // gate/up B operand = all M normed rows
  int chunked;              // standalone: units index chunks of at most kExpertTileTokens rows
  // standalone: warps 3-7 gather this CTA's share of the token rows
  const uint16_t* row_tok;  // token of every routed row
  uint16_t* list;           // [n_list] the rows this CTA gathers
  int n_list;
  int gather;
};

// Unit numbering: the gate/up units of the paired chunks (two slices each),
// then those of the other chunks, then the down units in the same pattern.
__device__ __forceinline__ int n_units(const Rt& rt, const ExpertArgs& p) {
  const int SF = p.F >> 6, SH = p.H >> 7;
  return rt.n_pair * ((SF + SH) >> 1) + (rt.n_exp - rt.n_pair) * (SF + SH);
}

__device__ __forceinline__ Unit decode_unit(int u, const Rt& rt, const ExpertArgs& p) {
  const int SF = p.F >> 6, SH = p.H >> 7;
  const int P = rt.n_pair;
  Unit w;
  const int g_pair = P * (SF >> 1);
  const int n_gu = g_pair + (rt.n_exp - P) * SF;
  w.pair = 0;
  if (u < g_pair) {
    w.kind = 0;
    w.a = u / (SF >> 1);
    w.slice = 2 * (u - w.a * (SF >> 1));
    w.pair = 1;
  } else if (u < n_gu) {
    const int v = u - g_pair;
    w.kind = 0;
    w.a = P + v / SF;
    w.slice = v - (w.a - P) * SF;
  } else {
    const int v = u - n_gu;
    const int d_pair = P * (SH >> 1);
    w.kind = 1;
    if (v < d_pair) {
      w.a = v / (SH >> 1);
      w.slice = 2 * (v - w.a * (SH >> 1));
      w.pair = 1;
    } else {
      const int v2 = v - d_pair;
      w.a = P + v2 / SH;
      w.slice = v2 - (w.a - P) * SH;
    }
  }
  if (rt.chunked) {
    w.e = rt.act[w.a];
    w.cnt = rt.cnt[w.a];
    w.off = rt.off[w.a];
  } else if (w.a == 0) {
    w.e = p.E;
    w.cnt = p.M;
    w.off = p.M * p.K;
  } else {
    w.e = rt.act[w.a - 1];
    w.cnt = rt.cnt[w.e];
    w.off = rt.off[w.e];
  }
  return w;
}

// B rows (the MMA N) of a unit: dense gate/up units take all M token rows.
// Start of a unit's K walk (in K steps), fixed by (expert, slice) so that
// concurrent units request different offsets within the weight rows and
// independent of scheduling, so results stay reproducible. A multiple of kq
// (the K groups of one low-bit staging slot; 1 for bf16 weights).
__device__ __forceinline__ int unit_rot(const Unit& w, int nk, int kq) {
  const int ns = nk / kq;
  return kq * static_cast<int>((static_cast<unsigned>(w.e) * 5u + static_cast<unsigned>(w.slice) * 3u) %
                               static_cast<unsigned>(ns));
}

__device__ __forceinline__ int unit_kq(const Unit& w, const ExpertArgs& p) {
  return p.q4 ? (w.kind == 0 ? p.kq_gu : p.kq_dn) : 1;
}

// K groups per A/B stage of a unit (1, 2 or 4).
__device__ __forceinline__ int unit_kg(const Unit& w, const ExpertArgs& p) {
  if (w.pair) return 1;                     // two weight slices of one K group fill an A stage
  return w.kind == 0 ? p.kg_gu : p.kg_dn;
}

// Granularity of a unit's K walk: a low-bit slot (kq groups, a multiple of
// kg) or one A/B stage (kg groups).
__device__ __forceinline__ int unit_kstep(const Unit& w, const ExpertArgs& p) {
  return p.q4 ? unit_kq(w, p) : unit_kg(w, p);
}

__device__ __forceinline__ int unit_rows(const Unit& w, const Rt& rt, const ExpertArgs& p) {
  return ((w.kind == 0 && rt.dense) ? p.M + 15 : w.cnt + 15) & ~15;
}

struct Smem {
  uint8_t* a_ring;
  uint8_t* b_ring;
  uint8_t* q_ring;  // low-bit staging slots (stages_q x kQSlotBytes)
  float* xch;  // [2][64][20] gate/up half exchange for SwiGLU
  uint64_t *full_a, *empty_a, *full_b, *empty_b, *tfull, *tempty, *ufull, *uempty, *drain, *full_q, *empty_q;
  int* unit_ids;  // [4]
  uint32_t* tmem_slot;
  volatile uint32_t* abort;
  volatile int* s_last;
  volatile int* s_unit;
  volatile int* s_ok;
  volatile int* cvt_unit;  // converter teams' unit ids, double-buffered by iteration
  uint8_t* rt_region;  // k_layer's routing tables
  uint32_t a_stage_bytes;  // kg_stage A tiles of 16 KiB
  uint32_t b_stage_bytes;  // kg_stage B tiles of nb_max x 128 bytes
  uint32_t b_half_bytes;   // one B tile
};

__device__ __forceinline__ Smem carve(uint8_t* raw, const ExpertArgs& p) {
  Smem s;
  const uint32_t r = smem_u32(raw);
  uint8_t* base = raw + ((1024u - (r & 1023u)) & 1023u);
  s.b_half_bytes = static_cast<uint32_t>(p.nb_max) * 128u;
  s.b_stage_bytes = s.b_half_bytes * static_cast<uint32_t>(p.kg_stage);
  s.a_stage_bytes = static_cast<uint32_t>(kATileBytes) * static_cast<uint32_t>(p.kg_stage);
  s.a_ring = base;
  s.b_ring = s.a_ring + static_cast<size_t>(p.smem_a) * s.a_stage_bytes;
  uint8_t* after_b = s.b_ring + static_cast<size_t>(p.stages_b) * s.b_stage_bytes;  // 1 KiB aligned
  s.q_ring = p.q_in_a ? s.a_ring : after_b;
  s.xch = reinterpret_cast<float*>(p.q_in_a ? after_b : after_b + static_cast<size_t>(p.stages_q) * kQSlotBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.xch + 2 * 64 * 20);
  s.full_a = bars;
  s.empty_a = s.full_a + p.stages_a;
  s.full_b = s.empty_a + p.stages_a;
  s.empty_b = s.full_b + p.stages_b;
  s.tfull = s.empty_b + p.stages_b;
  s.tempty = s.tfull + 2;
  s.ufull = s.tempty + 2;
  s.uempty = s.ufull + kExpertUnitRing;
  s.drain = s.uempty + kExpertUnitRing;
  s.full_q = s.drain + 1;
  s.empty_q = s.full_q + p.stages_q;
  s.unit_ids = reinterpret_cast<int*>(s.empty_q + p.stages_q);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.unit_ids + kExpertUnitRing);
  s.abort = s.tmem_slot + 1;
  s.s_last = reinterpret_cast<volatile int*>(s.tmem_slot + 2);
  s.s_unit = s.s_last + 1;
  s.s_ok = s.s_last + 2;
  s.cvt_unit = reinterpret_cast<volatile int*>(s.tmem_slot + 8);  // [2 teams][2] (bytes 32-47)
  s.rt_region = reinterpret_cast<uint8_t*>(s.tmem_slot) + 128;
  return s;
}

__device__ __forceinline__ void raise_abort(const Smem& s, int* err, int code) {
  atomicOr(err, code);
  *s.abort = 1u;
}

// Waits (bounded) for the TMA copies still in flight on a ring after an
// abort, so that the CTA never exits with copies landing in its memory.
__device__ void drain_ring(uint64_t* full, int stages, uint32_t issued_mask, uint32_t parity_bits) {
  for (int i = 0; i < stages; ++i)
    if (issued_mask & (1u << i)) mbar_wait_for(&full[i], (parity_bits >> i) & 1u, 200000000ull);
}

// Weight producer. bf16 weights go straight into the A ring by TMA; low-bit
// weights (kQ4) go into the staging ring, codes by TMA and scales by bulk
// copy, for the converter warps to expand.
template <bool kQ4>
__device__ void producer_a(const ExpertArgs& p, const Smem& s, const Rt& rt, int n_total) {
  const uint64_t pol = l2_policy_evict_first();
  const int SA = kQ4 ? p.stages_q : p.stages_a;
  uint64_t* const full = kQ4 ? s.full_q : s.full_a;
  uint64_t* const empty = kQ4 ? s.empty_q : s.empty_a;
  int sa = 0;
  uint32_t pha = 0, issued = 0, parity_bits = 0;
  for (int it = 0;; ++it) {
    // A CTA that gave up (n_total == 0) draws no unit, so it never takes
    // work away from the others.
    int u = n_total > 0 ? atomicAdd(p.unit_ctr, 1) : n_total;
    if (u < 0) {  // a counter left negative: take no unit, report it
      atomicOr(p.err, kErrState);
      u = n_total;
    }
    if (u >= n_total) {
      u = kUnitEnd;
      // No unit left: while the last units drain, ask L2 for the router rows
      // this CTA will stage in the next layer (same item mapping) and for
      // this CTA's share of the next layer's shared expert, which the next
      // layer always streams (it then comes from L2 while HBM would otherwise
      // idle through the routing prelude; same box: 5.631 -> 5.620 ms per
      // step).
      if (p.wr_next != nullptr) {
        const int n_eg = (p.E + kRouteExperts - 1) / kRouteExperts;
        const int n_items = n_eg * ((p.M + kRouteTokens - 1) / kRouteTokens);
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
          const int eg = item % n_eg;
          const int ne = min(kRouteExperts, p.E - eg * kRouteExperts);
          bulk_prefetch_l2(p.wr_next + static_cast<size_t>(eg) * kRouteExperts * p.H,
                           static_cast<uint32_t>(ne * p.H * 2));
        }
      }
      if (p.sgu_next != nullptr && p.sdn_next != nullptr) {
        const size_t b_gu = static_cast<size_t>(2) * p.F * p.H * 2, b_dn = static_cast<size_t>(p.H) * p.F * 2;
        const size_t tot = b_gu + b_dn;
        const size_t per = ((tot + gridDim.x - 1) / gridDim.x + 4095) & ~static_cast<size_t>(4095);
        const size_t o0 = static_cast<size_t>(blockIdx.x) * per, o1 = o0 + per < tot ? o0 + per : tot;
        for (size_t o = o0; o < o1;) {
          const bool gu = o < b_gu;  // gate/up bytes first, then down
          const size_t lim = gu ? (o1 < b_gu ? o1 : b_gu) : o1;
          const uint8_t* base = gu ? reinterpret_cast<const uint8_t*>(p.sgu_next) + o
                                   : reinterpret_cast<const uint8_t*>(p.sdn_next) + (o - b_gu);
          bulk_prefetch_l2(base, static_cast<uint32_t>(lim - o));
          o = lim;
        }
      }
    }
    const int us = it & (kExpertUnitRing - 1);
    const uint32_t upar = (it / kExpertUnitRing) & 1;
    if (!mbar_wait(&s.uempty[us], upar ^ 1u, s.abort)) {
      raise_abort(s, p.err, kErrMbarTimeout);
      break;
    }
    s.unit_ids[us] = u;
    mbar_arrive(&s.ufull[us]);
    if (u < 0) break;
    const Unit w = decode_unit(u, rt, p);
    const CUtensorMap* m;
    int row, nk;
    if (w.kind == 0) {
      m = (w.e == p.E) ? &p.tm_sgu : &p.tm_gu;
      row = (w.e == p.E ? 0 : w.e * 2 * p.F) + w.slice * 64;
      nk = p.H >> 6;
    } else {
      m = (w.e == p.E) ? &p.tm_sdn : &p.tm_dn;
      row = (w.e == p.E ? 0 : w.e * p.H) + w.slice * 128;
      nk = p.F >> 6;
    }
    const int kq = kQ4 ? unit_kq(w, p) : 1;
    const int kg = unit_kg(w, p);
    const int kstep = unit_kstep(w, p);
    const int rot = unit_rot(w, nk, kstep);
    bool ok = true;
    // one stage per kg K groups (bf16) or one slot per kq K groups (low-bit)
    for (int kc0 = 0; kc0 < nk; kc0 += kstep) {
      const int kc = (kc0 + rot < nk) ? kc0 + rot : kc0 + rot - nk;
      if (!mbar_wait(&empty[sa], pha ^ 1u, s.abort)) {
        raise_abort(s, p.err, kErrMbarTimeout);
        ok = false;
        break;
      }
      if (kQ4) {
        // codes: rows of kq x 32 bytes (gate/up: 64 gate rows then 64 up
        // rows; down: 128 rows), then the kq groups' 128 row scales each
        const uint32_t dst = smem_u32(s.q_ring + static_cast<size_t>(sa) * kQSlotBytes);
        mbar_arrive_expect_tx(&full[sa], static_cast<uint32_t>(kq * kQGroupBytes));
        const uint32_t sdst = dst + kq * 4096;
        const bool sh = w.e == p.E;
        if (p.q4_views && w.kind == 0) {  // gate and up codes in one box, the kq groups' scales in another
          tma_load_3d(dst, sh ? &p.tm_sgu_q3 : &p.tm_gu_q3, &full[sa], kc * 32, row, 0, pol);
          tma_load_3d(sdst, sh ? &p.tm_sgu_sv : &p.tm_gu_sv, &full[sa], w.slice * 64, 0,
                      (sh ? 0 : w.e * (p.H >> 6)) + kc, pol);
        } else if (p.q4_views) {
          tma_load_2d(dst, sh ? &p.tm_sdn_q : &p.tm_dn_q, &full[sa], kc * 32, row, pol);
          tma_load_2d(sdst, sh ? &p.tm_sdn_sv : &p.tm_dn_sv, &full[sa], w.slice * 128,
                      (sh ? 0 : w.e * (p.F >> 6)) + kc, pol);
        } else if (w.kind == 0) {
          const CUtensorMap* mq = (w.e == p.E) ? &p.tm_sgu_q : &p.tm_gu_q;
          tma_load_2d(dst, mq, &full[sa], kc * 32, row, pol);
          tma_load_2d(dst + kq * 2048, mq, &full[sa], kc * 32, row + p.F, pol);
          const uint16_t* sc = (w.e == p.E ? p.sgu_s : p.gu_s + static_cast<size_t>(w.e) * (p.H >> 6) * 2 * p.F) +
                               static_cast<size_t>(kc) * 2 * p.F + w.slice * 64;
          for (int g = 0; g < kq; ++g) {
            bulk_load(sdst + g * 256, sc + static_cast<size_t>(g) * 2 * p.F, 128, &full[sa]);
            bulk_load(sdst + g * 256 + 128, sc + static_cast<size_t>(g) * 2 * p.F + p.F, 128, &full[sa]);
          }
        } else {
          const CUtensorMap* mq = (w.e == p.E) ? &p.tm_sdn_q : &p.tm_dn_q;
          tma_load_2d(dst, mq, &full[sa], kc * 32, row, pol);
          const uint16_t* sc = (w.e == p.E ? p.sdn_s : p.dn_s + static_cast<size_t>(w.e) * (p.F >> 6) * p.H) +
                               static_cast<size_t>(kc) * p.H + w.slice * 128;
          for (int g = 0; g < kq; ++g) bulk_load(sdst + g * 256, sc + static_cast<size_t>(g) * p.H, 256, &full[sa]);
        }
      } else {
        const uint32_t dst0 = smem_u32(s.a_ring + static_cast<size_t>(sa) * s.a_stage_bytes);
        // kg K groups of one slice, or one K group of a pair's two slices
        const int nt = w.pair ? 2 : kg;
        mbar_arrive_expect_tx(&full[sa], static_cast<uint32_t>(nt * kATileBytes));
        // Two K groups of one slice in one box (same layout). (One box for a
        // pair's two slices measured 0.4% slower on the batched step.)
        const bool one_box = p.stage_maps && !w.pair && kg == 2;
        if (one_box) {
          const bool sh = w.e == p.E;
          if (w.kind == 0)
            tma_load_4d(dst0, sh ? &p.tm_sgu_k2 : &p.tm_gu_k2, &full[sa], 0, row, 0, kc, pol);
          else
            tma_load_3d(dst0, sh ? &p.tm_sdn_k2 : &p.tm_dn_k2, &full[sa], 0, row, kc, pol);
        }
        for (int h = 0; h < nt && !one_box; ++h) {
          const uint32_t dst = dst0 + h * kATileBytes;
          const int kx = w.pair ? kc : kc + h;
          const int rx = w.pair ? row + h * (w.kind == 0 ? 64 : 128) : row;
          if (w.kind == 0) {
            tma_load_2d(dst, m, &full[sa], kx * 64, rx, pol);            // 64 gate rows
            tma_load_2d(dst + 8192, m, &full[sa], kx * 64, rx + p.F, pol);  // 64 up rows
          } else {
            tma_load_2d(dst, m, &full[sa], kx * 64, rx, pol);  // 128 down rows
          }
        }
      }
      issued |= 1u << sa;
      parity_bits = (parity_bits & ~(1u << sa)) | (pha << sa);
      if (++sa == SA) {
        sa = 0;
        pha ^= 1u;
      }
    }
    if (!ok) break;
  }
  if (*s.abort) drain_ring(full, SA, issued, parity_bits);
}

// Low-bit tiles -> bf16 A tiles (warps 8-11, one tile row per thread). In a
// slot of kq K groups, row r's codes of group g and its scale sit at
// slot + r kq 32 + 32 g (16-byte chunks swizzled when the row is 128 bytes)
// and slot + kq 4096 + 256 g + 2 r, for both unit kinds.
// Each pair of codes becomes a bf16x2 by the exponent trick
// (0x4300 | u = 128 + u), then (128 + u) - 136 = u - 8 exactly and one bf16
// multiply by the scale gives bf16((u - 8) s). The row is written in the
// 128-byte swizzle the TMA would have used, so the MMA is unchanged; or, with
// p.a_tmem, into tensor memory (the thread's own lane, 32 columns per group),
// where the MMA reads A directly: no shared-memory stores, no proxy fence,
// and the MMA reads only B from shared memory.
__device__ void converter(const ExpertArgs& p, const Smem& s, const Rt& rt, uint32_t tmem_base) {
  // With p.q_teams == 2 two teams of four warps take the staging slots in
  // turn (team t: slots t, t + 2, ...). The host enables this only when the
  // slot count is even and the bf16 stage count a multiple of twice the
  // stages per slot, so each team owns its own slots and stages and never
  // runs more than one ring round ahead of their consumer (a parity wait
  // cannot tell two rounds apart). With one team, team 1 only takes part in
  // the unit handshake. Both teams walk every unit and slot to keep the ring
  // counters. Control flow stays uniform across a team: the unit id comes
  // from the team leader through shared memory, and a failed wait only
  // skips work, so no thread is left at a team barrier.
  const int team = (threadIdx.x - 8 * 32) >> 7;  // 0 or 1
  const int r = (threadIdx.x - 8 * 32) & 127;    // tile row
  const int lane = threadIdx.x & 31;
  const int SA = p.stages_a, SQ = p.stages_q;
  int sa = 0, sq = 0;
  uint32_t pha = 0, phq = 0;
  uint32_t gslot = 0;  // slots of all units so far
  const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.f, 136.f);
  for (int it = 0;; ++it) {
    const int us = it & (kExpertUnitRing - 1);
    const uint32_t upar = (it / kExpertUnitRing) & 1;
    volatile int* bcast = s.cvt_unit + team * 2 + (it & 1);
    if (r == 0) {
      const bool got = mbar_wait(&s.ufull[us], upar, s.abort);
      *bcast = got ? s.unit_ids[us] : kUnitAbort;
      if (got) mbar_arrive(&s.uempty[us]);
      else raise_abort(s, p.err, kErrMbarTimeout);
    }
    named_bar_sync(2 + team, 128);  // the unit id is published to the team
    const int u = *bcast;
    if (u < 0) break;
    const Unit w = decode_unit(u, rt, p);
    const int nk = (w.kind == 0) ? (p.H >> 6) : (p.F >> 6);
    const int kq = unit_kq(w, p);
    const int kg = unit_kg(w, p);  // kq is a multiple of kg
    for (int kc0 = 0; kc0 < nk; kc0 += kq, ++gslot) {
      const bool mine = (p.q_teams == 2) ? ((gslot & 1u) == static_cast<uint32_t>(team)) : (team == 0);
      if (!mine) {  // another team's slot: step the counters
        for (int st = 0; st < kq / kg; ++st) {
          if (++sa == SA) {
            sa = 0;
            pha ^= 1u;
          }
        }
        if (++sq == SQ) {
          sq = 0;
          phq ^= 1u;
        }
        continue;
      }
      bool ok = mbar_wait(&s.full_q[sq], phq, s.abort);
      if (!ok) raise_abort(s, p.err, kErrMbarTimeout);
      const uint8_t* slot = s.q_ring + static_cast<size_t>(sq) * kQSlotBytes;
      for (int g = 0; g < kq; ++g) {
        const int h = g % kg;  // half of the A stage this group fills
        if (h == 0 && ok && !mbar_wait(&s.empty_a[sa], pha ^ 1u, s.abort)) {
          raise_abort(s, p.err, kErrMbarTimeout);
          ok = false;
        }
        if (h == 0 && p.a_tmem) tc_fence_after();  // the MMAs that read this stage are complete
        if (ok) {
          // 128-byte code rows (kq = 4) arrive in the 128-byte swizzle
          const uint8_t* src = slot + r * kq * 32;
          const int ch0 = (kq == 4) ? ((2 * g) ^ (r & 7)) : 2 * g;
          const int ch1 = (kq == 4) ? ((2 * g + 1) ^ (r & 7)) : 2 * g + 1;
          const uint4 c0 = *reinterpret_cast<const uint4*>(src + ch0 * 16);
          const uint4 c1 = *reinterpret_cast<const uint4*>(src + ch1 * 16);
          const unsigned short sb = *reinterpret_cast<const unsigned short*>(slot + kq * 4096 + g * 256 + 2 * r);
          const __nv_bfloat162 sc = __halves2bfloat162(__ushort_as_bfloat16(sb), __ushort_as_bfloat16(sb));
          const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t o[32];  // word 4j + i holds elements 8j + 2i (low half) and 8j + 2i + 1
#pragma unroll
          for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t x = ((words[j] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
              const __nv_bfloat162 v = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&x), k136), sc);
              o[4 * j + i] = *reinterpret_cast<const uint32_t*>(&v);
            }
          }
          if (p.a_tmem) {
            // lane r of the stage's columns (the warp's lane quarter is r / 32)
            tmem_st32(tmem_base + (static_cast<uint32_t>(r & ~31) << 16) + static_cast<uint32_t>(kTmemAStage0) +
                          static_cast<uint32_t>(sa) * 128u + static_cast<uint32_t>(h) * 32u,
                      o);
          } else {
            uint8_t* row = s.a_ring + static_cast<size_t>(sa) * s.a_stage_bytes + h * kATileBytes + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) =
                  make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
        if (h == kg - 1) {
          if (p.a_tmem) {
            tmem_wait_st();     // this thread's columns are written
            tc_fence_before();  // ordered before the arrival the MMA waits on
          } else {
            fence_proxy_async_shared();  // the MMA reads the tile through the async proxy
          }
          __syncwarp();
          if (lane == 0 && ok) mbar_arrive(&s.full_a[sa]);
          if (++sa == SA) {
            sa = 0;
            pha ^= 1u;
          }
        }
      }
      // this thread's reads of the slot are done (the fence above ordered
      // them before any later copy into it)
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&s.empty_q[sq]);
      if (++sq == SQ) {
        sq = 0;
        phq ^= 1u;
      }
    }
  }
}

__device__ void producer_b(const ExpertArgs& p, const Smem& s, const Rt& rt) {
  const uint64_t pol = l2_policy_evict_last();
  const int SB = p.stages_b;
  const int SF = p.F >> 6;
  int sb = 0;
  uint32_t phb = 0, issued = 0, parity_bits = 0;
  for (int it = 0;; ++it) {
    const int us = it & (kExpertUnitRing - 1);
    const uint32_t upar = (it / kExpertUnitRing) & 1;
    if (!mbar_wait(&s.ufull[us], upar, s.abort)) {
      raise_abort(s, p.err, kErrMbarTimeout);
      break;
    }
    const int u = s.unit_ids[us];
    mbar_arrive(&s.uempty[us]);
    if (u < 0) break;
    const Unit w = decode_unit(u, rt, p);
    const int nrows = unit_rows(w, rt, p);
    const int row0 = (w.kind == 0 && rt.dense) ? 0 : w.off;
    const CUtensorMap* m;
    const CUtensorMap* mb;
    int nk, box;
    if (w.kind == 0) {
      m = &p.tm_xg;
      mb = &p.tm_xg_big;
      box = p.xg_box;
      nk = p.H >> 6;
      if (rt.chunked && w.e != p.E) {
        // The chunk's token rows are gathered by warps 3-7 of every CTA at
        // the start of the launch: wait (bounded) until all of them are in.
        const unsigned long long t0 = global_ns();
        bool ok = true;
        while (ld_acquire_gpu(&p.gathered[w.a]) < w.cnt) {
          if (*s.abort) {
            ok = false;
            break;
          }
          if (global_ns() - t0 > kWaitLimitNs) {
            raise_abort(s, p.err, kErrDepTimeout);
            ok = false;
            break;
          }
          __nanosleep(32);
        }
        if (!ok) break;
        fence_proxy_async_global();
      }
    } else {
      m = &p.tm_h;
      mb = &p.tm_h_big;
      box = p.h_box;
      nk = p.F >> 6;
      // The expert's SwiGLU rows must be complete before they are loaded.
      const unsigned long long t0 = global_ns();
      bool ok = true;
      while (ld_acquire_gpu(&p.gu_done[w.a]) < SF) {
        if (*s.abort) {
          ok = false;
          break;
        }
        if (global_ns() - t0 > kWaitLimitNs) {
          raise_abort(s, p.err, kErrDepTimeout);
          ok = false;
          break;
        }
        __nanosleep(64);
      }
      if (!ok) break;
      fence_proxy_async_global();
    }
    const int kg = unit_kg(w, p);
    const int rot = unit_rot(w, nk, unit_kstep(w, p));
    bool ok = true;
    for (int kc0 = 0; kc0 < nk; kc0 += kg) {
      const int kc = (kc0 + rot < nk) ? kc0 + rot : kc0 + rot - nk;
      if (!mbar_wait(&s.empty_b[sb], phb ^ 1u, s.abort)) {
        raise_abort(s, p.err, kErrMbarTimeout);
        ok = false;
        break;
      }
      const uint32_t dst0 = smem_u32(s.b_ring + static_cast<size_t>(sb) * s.b_stage_bytes);
      mbar_arrive_expect_tx(&s.full_b[sb], static_cast<uint32_t>(kg * nrows) * 128u);
      // the dense normed rows of all kg groups in one box (same layout)
      const bool one_box = p.xg_k && w.kind == 0 && rt.dense && kg == p.kg_gu && nrows == box &&
                           static_cast<uint32_t>(nrows) * 128u == s.b_half_bytes;
      if (one_box) tma_load_3d(dst0, &p.tm_xg_k, &s.full_b[sb], 0, 0, kc, pol);
      for (int h = 0; h < kg && !one_box; ++h) {
        const uint32_t dst = dst0 + h * s.b_half_bytes;
        for (int i = 0; i < nrows;) {
          const bool big = nrows - i >= box;
          tma_load_2d(dst + i * 128, big ? mb : m, &s.full_b[sb], (kc + h) * 64, row0 + i, pol);
          i += big ? box : 16;
        }
      }
      issued |= 1u << sb;
      parity_bits = (parity_bits & ~(1u << sb)) | (phb << sb);
      if (++sb == SB) {
        sb = 0;
        phb ^= 1u;
      }
    }
    if (!ok) break;
  }
  if (*s.abort) drain_ring(s.full_b, SB, issued, parity_bits);
}

__device__ void mma_issuer(const ExpertArgs& p, const Smem& s, const Rt& rt, uint32_t tmem_base) {
  const int SA = p.stages_a, SB = p.stages_b;
  int sa = 0, sb = 0;
  uint32_t pha = 0, phb = 0;
  for (int it = 0;; ++it) {
    const int us = it & (kExpertUnitRing - 1);
    const uint32_t upar = (it / kExpertUnitRing) & 1;
    if (!mbar_wait(&s.ufull[us], upar, s.abort)) {
      raise_abort(s, p.err, kErrMbarTimeout);
      break;
    }
    const int u = s.unit_ids[us];
    mbar_arrive(&s.uempty[us]);
    if (u < 0) break;
    const Unit w = decode_unit(u, rt, p);
    const int n = unit_rows(w, rt, p);
    const int nk = (w.kind == 0) ? (p.H >> 6) : (p.F >> 6);
    const uint32_t idesc = umma_idesc_bf16(128, n);
    const int acc = it & 1;
    const uint32_t apar = (it >> 1) & 1;
    if (!mbar_wait(&s.tempty[acc], apar ^ 1u, s.abort)) {
      raise_abort(s, p.err, kErrMbarTimeout);
      break;
    }
    tc_fence_after();
    const uint32_t d = tmem_base + static_cast<uint32_t>(acc) * static_cast<uint32_t>(p.acc_cols);
    bool ok = true;
    const int kg = unit_kg(w, p);
    for (int kc = 0; kc < nk; kc += kg) {
      if (!mbar_wait(&s.full_a[sa], pha, s.abort) || !mbar_wait(&s.full_b[sb], phb, s.abort)) {
        raise_abort(s, p.err, kErrMbarTimeout);
        ok = false;
        break;
      }
      tc_fence_after();
      for (int h = 0; h < kg; ++h) {
        const uint64_t bd =
            umma_desc_sw128(smem_u32(s.b_ring + static_cast<size_t>(sb) * s.b_stage_bytes + h * s.b_half_bytes));
        if (w.pair) {
          // the pair's two slices, each into its own accumulator (128 columns apart)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint64_t ad = umma_desc_sw128(
                smem_u32(s.a_ring + static_cast<size_t>(sa) * s.a_stage_bytes + t * kATileBytes));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(d + 128u * t, ad + static_cast<uint64_t>(2 * k), bd + static_cast<uint64_t>(2 * k), idesc,
                        (kc | k) != 0 ? 1u : 0u);
          }
        } else if (p.a_tmem) {
          const uint32_t at = tmem_base + static_cast<uint32_t>(kTmemAStage0) + static_cast<uint32_t>(sa) * 128u +
                              static_cast<uint32_t>(h) * 32u;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16_ta(d, at + 8u * k, bd + static_cast<uint64_t>(2 * k), idesc, (kc | h | k) != 0 ? 1u : 0u);
        } else {
          const uint64_t ad =
              umma_desc_sw128(smem_u32(s.a_ring + static_cast<size_t>(sa) * s.a_stage_bytes + h * kATileBytes));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(d, ad + static_cast<uint64_t>(2 * k), bd + static_cast<uint64_t>(2 * k), idesc,
                      (kc | h | k) != 0 ? 1u : 0u);
        }
      }
      umma_commit(&s.empty_a[sa]);
      umma_commit(&s.empty_b[sb]);
      if (++sa == SA) {
        sa = 0;
        pha ^= 1u;
      }
      if (++sb == SB) {
        sb = 0;
        phb ^= 1u;
      }
    }
    if (!ok) break;
    umma_commit(&s.tfull[acc]);
  }
  // Every MMA this thread issued must be complete before TMEM is released.
  umma_commit(s.drain);
  mbar_wait_for(s.drain, 0, 200000000ull);
}

// Sums the weighted expert rows of one 128-wide hidden slice into the
// residual stream: x_out = x_in + (sum_k w_tk y_{slot(t,k)}) + y_shared(t).
// One token's combined output column block (see combine_slice); the loads of
// up to 8 selections are issued before any is used.
struct CombineAcc {
  float4 acc, ys, xi;
};

__device__ __forceinline__ void combine_loads(const ExpertArgs& p, const Rt& rt, int t, size_t col, int k0,
                                              int r[8], float wk[8], float4 y[8]) {
  const int K = p.K, MK = p.M * p.K;
  const size_t H = p.H;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool v = k0 + i < K;
    r[i] = v ? rt.tok_slot[t * K + k0 + i] : MK + t;
    wk[i] = v ? rt.topk_w[t * K + k0 + i] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    y[i] = __ldcg(reinterpret_cast<const float4*>(p.yslot + static_cast<size_t>(r[i]) * H + col));
}

__device__ __forceinline__ void combine_accumulate(float4& acc, const float wk[8], const float4 y[8], int k0,
                                                   int K) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (k0 + i < K) {
      acc.x = fmaf(wk[i], y[i].x, acc.x);
      acc.y = fmaf(wk[i], y[i].y, acc.y);
      acc.z = fmaf(wk[i], y[i].z, acc.z);
      acc.w = fmaf(wk[i], y[i].w, acc.w);
    }
  }
}

__device__ __forceinline__ void combine_store(const ExpertArgs& p, int t, size_t col, float4 acc, float4 ys,
                                              float4 xi) {
  acc.x += ys.x;
  acc.y += ys.y;
  acc.z += ys.z;
  acc.w += ys.w;
  float4 o;
  o.x = xi.x + acc.x;
  o.y = xi.y + acc.y;
  o.z = xi.z + acc.z;
  o.w = xi.w + acc.w;
  *reinterpret_cast<float4*>(p.x_out + static_cast<size_t>(t) * p.H + col) = o;
}

// Sums the weighted expert rows of tokens t0..t1-1 in one 128-wide hidden
// slice into the residual stream: x_out = x_in + (sum_k w_tk y_{slot(t,k)})
// + y_shared(t), selections in order, then the shared row, then the
// residual. Two tokens are in flight per thread.
__device__ void combine_slice(const ExpertArgs& p, const Rt& rt, int j, int t0, int t1, int etid) {
  const int c4 = (etid & 31) * 4;
  const int g = etid >> 5;
  const size_t H = p.H;
  const size_t col = static_cast<size_t>(j) * 128 + c4;
  const int MK = p.M * p.K;
  const int K = p.K;
  for (int t = t0 + g; t < t1; t += 8) {
    const int t2 = t + 4;
    const bool two = t2 < t1;
    const float4 ys = __ldcg(reinterpret_cast<const float4*>(p.yslot + static_cast<size_t>(MK + t) * H + col));
    const float4 xi = *reinterpret_cast<const float4*>(p.x_in + static_cast<size_t>(t) * H + col);
    float4 ys2 = make_float4(0.f, 0.f, 0.f, 0.f), xi2 = ys2;
    if (two) {
      ys2 = __ldcg(reinterpret_cast<const float4*>(p.yslot + static_cast<size_t>(MK + t2) * H + col));
      xi2 = *reinterpret_cast<const float4*>(p.x_in + static_cast<size_t>(t2) * H + col);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), acc2 = acc;
    for (int k0 = 0; k0 < K; k0 += 8) {
      int r[8], r2[8];
      float wk[8], wk2[8];
      float4 y[8], y2[8];
      combine_loads(p, rt, t, col, k0, r, wk, y);
      if (two) combine_loads(p, rt, t2, col, k0, r2, wk2, y2);
      combine_accumulate(acc, wk, y, k0, K);
      if (two) combine_accumulate(acc2, wk2, y2, k0, K);
    }
    combine_store(p, t, col, acc, ys, xi);
    if (two) combine_store(p, t2, col, acc2, ys2, xi2);
  }
}

// Combines token t's 128-wide hidden slice j with one warp (lane l takes
// columns 4l..4l+3), in the same order as combine_slice.
__device__ void combine_token(const ExpertArgs& p, const Rt& rt, int j, int t, int lane) {
  const size_t col = static_cast<size_t>(j) * 128 + lane * 4;
  const int MK = p.M * p.K;
  const float4 ys = __ldcg(reinterpret_cast<const float4*>(p.yslot + static_cast<size_t>(MK + t) * p.H + col));
  const float4 xi = *reinterpret_cast<const float4*>(p.x_in + static_cast<size_t>(t) * p.H + col);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < p.K; k0 += 8) {
    int r[8];
    float wk[8];
    float4 y[8];
    combine_loads(p, rt, t, col, k0, r, wk, y);
    combine_accumulate(acc, wk, y, k0, p.K);
  }
  combine_store(p, t, col, acc, ys, xi);
}

__device__ void epilogue(const ExpertArgs& p, const Smem& s, const Rt& rt, uint32_t tmem_base) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;             // TMEM lane quarter this warp may read
  const int row = q * 32 + lane;      // accumulator row
  const int etid = threadIdx.x - 96;  // 0..127
  const int SF = p.F >> 6;
  for (int it = 0;; ++it) {
    const int us = it & (kExpertUnitRing - 1);
    const uint32_t upar = (it / kExpertUnitRing) & 1;
    if (etid == 0) {
      int u = kUnitAbort;
      if (mbar_wait(&s.ufull[us], upar, s.abort)) {
        u = s.unit_ids[us];
        mbar_arrive(&s.uempty[us]);
      } else {
        raise_abort(s, p.err, kErrMbarTimeout);
      }
      *s.s_unit = u;
    }
    named_bar_sync(1, 128);
    const int u = *s.s_unit;
    if (u < 0) break;
    const Unit w = decode_unit(u, rt, p);
    const int n = unit_rows(w, rt, p);
    const int acc = it & 1;
    const uint32_t apar = (it >> 1) & 1;
    if (etid == 0) {
      const bool ok = mbar_wait(&s.tfull[acc], apar, s.abort);
      if (!ok) raise_abort(s, p.err, kErrMbarTimeout);
      *s.s_ok = ok ? 1 : 0;
    }
    named_bar_sync(1, 128);
    if (!*s.s_ok) break;
    tc_fence_after();
    const uint32_t tb0 =
        tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc) * static_cast<uint32_t>(p.acc_cols);
    if (w.kind == 0) {
     for (int t = 0; t <= w.pair; ++t) {  // a pair's second slice is 128 columns on
      const uint32_t tb = tb0 + 128u * static_cast<uint32_t>(t);
      const int slice = w.slice + t;
      // Rows 0..63 of the tile are gate rows f, rows 64..127 the up rows of
      // the same f. Per 32 columns the gate warps take columns 0..15 and the
      // up warps 16..31, each handing the other half of its values over.
      const bool gate_half = q < 2;
      const int r64 = gate_half ? row : row - 64;
      bf16* hrow = p.hbuf + static_cast<size_t>(w.off) * p.F + slice * 64 + r64;
      float* x_up = s.xch;              // [64][20] up values of columns 0..15
      float* x_gate = s.xch + 64 * 20;  // [64][20] gate values of columns 16..31
      const uint32_t tm = (rt.dense && w.e != p.E) ? rt.mask[w.e] : 0xffffffffu;
      for (int c0 = 0; c0 < n; c0 += 32) {
        float v[32];
        __syncwarp();
        tmem_ld32(tb + c0, v);  // columns past n are read but never kept
        float4* mine = reinterpret_cast<float4*>((gate_half ? x_gate : x_up) + r64 * 20);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = 4 * j;
          mine[j] = gate_half ? make_float4(v[16 + k], v[17 + k], v[18 + k], v[19 + k])
                              : make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
        named_bar_sync(1, 128);
        float o[16];
        const float4* other = reinterpret_cast<const float4*>((gate_half ? x_up : x_gate) + r64 * 20);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 t4 = other[j];
          o[4 * j] = t4.x;
          o[4 * j + 1] = t4.y;
          o[4 * j + 2] = t4.z;
          o[4 * j + 3] = t4.w;
        }
        named_bar_sync(1, 128);  // the exchange rows are free again
        // silu(g) = g / (1 + e^-g); the exponent is capped so that the fast
        // divide stays in its range (the capped terms are below 1e-33)
        float hv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float g = gate_half ? v[j] : o[j];
          const float up = gate_half ? o[j] : v[16 + j];
          hv[j] = __fdividef(g, 1.0f + __expf(fminf(-g, 80.f))) * up;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + (gate_half ? j : 16 + j);
          // dense mode: column c is token c; a routed expert keeps the
          // columns of its tokens, stored at their rank among them
          int slot = c;
          bool keep = c < w.cnt;
          if (rt.dense) {
            keep = c < p.M && ((tm >> c) & 1u);
            slot = (w.e == p.E) ? c : __popc(tm & ((1u << c) - 1u));
          }
          if (keep) hrow[static_cast<size_t>(slot) * p.F] = __float2bfloat16_rn(hv[j]);
        }
      }
     }
      // The h rows are published by one release after the epilogue barrier
      // (which orders every epilogue thread's stores before it); each thread
      // orders its stores for the TMA loads that read them.
      tc_fence_before();
      fence_proxy_async_global();
      named_bar_sync(1, 128);
      if (etid == 0) {
        mbar_arrive(&s.tempty[acc]);
        red_release_gpu_add(&p.gu_done[w.a], 1 + w.pair);
      }
    } else {
      for (int t = 0; t <= w.pair; ++t) {
        const uint32_t tb = tb0 + 128u * static_cast<uint32_t>(t);
        float* ycol = p.yslot + static_cast<size_t>(w.off) * p.H + static_cast<size_t>(w.slice + t) * 128 + row;
        for (int c0 = 0; c0 < n; c0 += 32) {
          float v[32];
          __syncwarp();
          tmem_ld32(tb + c0, v);  // columns past n are read but never stored
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j;
            if (c < w.cnt) ycol[static_cast<size_t>(c) * p.H] = v[j];
          }
        }
      }
      tc_fence_before();
      if (p.combine == 1) __threadfence();  // otherwise the rows are read by a later kernel
      named_bar_sync(1, 128);
      if (kPhaseStamps && etid == 0 && p.stamps != nullptr) atomicMax(p.stamps + 6, global_ns());
      if (etid == 0) {
        mbar_arrive(&s.tempty[acc]);
        int last = 0;
        if (p.combine == 1) last = (atomicAdd(&p.dn_done[w.slice], 1) == rt.n_exp - 1) ? 1 : 0;
        *s.s_last = last;
      }
      named_bar_sync(1, 128);
      if (*s.s_last) {  // this unit completed the slice: combine it for all tokens
        __threadfence();
        combine_slice(p, rt, w.slice, 0, p.M, etid);
      }
    }
  }
  (void)SF;
}


// Barrier setup, TMEM allocation and descriptor prefetch (before the
// dependency wait, so they overlap the previous kernel).
template <bool kQ4>
__device__ __forceinline__ uint32_t expert_prologue(const ExpertArgs& p, const Smem& s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages_a; ++i) {
      mbar_init(&s.full_a[i], kQ4 ? 4 : 1);  // low-bit: one arrival per converter warp
      mbar_init(&s.empty_a[i], 1);
    }
    for (int i = 0; kQ4 && i < p.stages_q; ++i) {
      mbar_init(&s.full_q[i], 1);
      mbar_init(&s.empty_q[i], 4);
    }
    for (int i = 0; i < p.stages_b; ++i) {
      mbar_init(&s.full_b[i], 1);
      mbar_init(&s.empty_b[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 1);
    }
    for (int i = 0; i < kExpertUnitRing; ++i) {
      mbar_init(&s.ufull[i], 1);
      mbar_init(&s.uempty[i], kQ4 ? 5 : 3);  // B loader, MMA issuer, epilogue leader (+ two converter team leaders)
    }
    mbar_init(s.drain, 1);
    *s.abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(kQ4 ? &p.tm_gu_q : &p.tm_gu);
    tma_prefetch_desc(kQ4 ? &p.tm_sgu_q : &p.tm_sgu);
    tma_prefetch_desc(kQ4 ? &p.tm_dn_q : &p.tm_dn);
    tma_prefetch_desc(kQ4 ? &p.tm_sdn_q : &p.tm_sdn);
    if (p.xg_k) tma_prefetch_desc(&p.tm_xg_k);
    if (kQ4 && p.q4_views) {
      tma_prefetch_desc(&p.tm_gu_q3);
      tma_prefetch_desc(&p.tm_sgu_q3);
      tma_prefetch_desc(&p.tm_gu_sv);
      tma_prefetch_desc(&p.tm_sgu_sv);
      tma_prefetch_desc(&p.tm_dn_sv);
      tma_prefetch_desc(&p.tm_sdn_sv);
    }
    if (!kQ4 && p.stage_maps) {
      tma_prefetch_desc(&p.tm_gu_k2);
      tma_prefetch_desc(&p.tm_sgu_k2);
      tma_prefetch_desc(&p.tm_dn_k2);
      tma_prefetch_desc(&p.tm_sdn_k2);
    }
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&p.tm_xg);
    tma_prefetch_desc(&p.tm_xg_big);
    tma_prefetch_desc(&p.tm_h);
    tma_prefetch_desc(&p.tm_h_big);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *s.tmem_slot;
}

// Rows of chunk a that this CTA gathers. Pieces of four rows: piece q of
// chunk a belongs to CTA (7 a + q) mod G, so a CTA owns pieces q0, q0 + G,
// ... of each chunk (usually at most one: a chunk has at most 32 pieces).
__device__ __forceinline__ int first_piece(int a, int G) {
  return static_cast<int>((static_cast<unsigned>(blockIdx.x) + static_cast<unsigned>(G) -
                           (7u * static_cast<unsigned>(a)) % static_cast<unsigned>(G)) %
                          static_cast<unsigned>(G));
}

__device__ __forceinline__ int owned_rows(const Rt& rt, int a, int G) {
  const int cnt = rt.cnt[a], n_q = (cnt + 3) >> 2;
  int nr = 0;
  for (int q = first_piece(a, G); q < n_q; q += G) nr += min(4, cnt - 4 * q);
  return nr;
}

// The standalone kernel's gather, by warps 3-7 while the other roles start
// (the epilogue warps have no accumulator to drain yet): copies the normed
// rows of the routed chunks' tokens into expert order (row r of the
// gathered buffer = normed row of token row_tok[r]), this CTA's share of the
// pieces. Warp 7 lists the rows (hottest chunks first); then each of the
// five warps copies every fifth row with 16-byte loads and stores, two rows
// in flight (one lane moving the rows with bulk copies, one per row each
// way, was slower: the rate of an SM's copies follows their number more
// than their size, and the first units waited ~4 µs for their rows);
// finally warp 7 publishes, per chunk, how many rows this CTA gathered
// (release). A
// gate/up unit of the chunk loads them once the chunk's counter reaches its
// row count; no CTA waits for all others.
__device__ void gather_rows(const ExpertArgs& p, const Rt& rt) {
  constexpr int kW = 5;
  const int G = gridDim.x, lane = threadIdx.x & 31, gw = (threadIdx.x >> 5) - 3;
  __shared__ int s_nrows;
  if (gw == kW - 1) {
    int base = 0;
    for (int a0 = 0; a0 < rt.n_exp; a0 += 32) {
      const int a = a0 + lane;
      const bool mine = a < rt.n_exp && rt.act[a] != p.E;
      const int nr = mine ? owned_rows(rt, a, G) : 0;
      int incl = nr;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (mine) {
        int at = base + incl - nr;
        const int cnt = rt.cnt[a], n_q = (cnt + 3) >> 2;
        for (int q = first_piece(a, G); q < n_q; q += G)
          for (int j = 4 * q; j < min(4 * q + 4, cnt); ++j, ++at)
            if (at < rt.n_list) rt.list[at] = static_cast<uint16_t>(rt.off[a] + j);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_nrows = min(base, rt.n_list);
  }
  named_bar_sync(5, 32 * kW);
  const int n_rows = s_nrows;
  const int nv = p.H >> 3;  // 16-byte pieces per row
  for (int r = gw; r < n_rows; r += 2 * kW) {
    const bool two = r + kW < n_rows;
    const int ra = rt.list[r], rb = two ? rt.list[r + kW] : ra;
    const uint4* a_src = reinterpret_cast<const uint4*>(p.xn + static_cast<size_t>(rt.row_tok[ra]) * p.H);
    const uint4* b_src = reinterpret_cast<const uint4*>(p.xn + static_cast<size_t>(rt.row_tok[rb]) * p.H);
    uint4* a_dst = reinterpret_cast<uint4*>(p.xg + static_cast<size_t>(ra) * p.H);
    uint4* b_dst = reinterpret_cast<uint4*>(p.xg + static_cast<size_t>(rb) * p.H);
    for (int v0 = 0; v0 < nv; v0 += 256) {
      uint4 va[8], vb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < nv) {
          va[j] = __ldcg(a_src + v);
          if (two) vb[j] = __ldcg(b_src + v);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < nv) {
          a_dst[v] = va[j];
          if (two) b_dst[v] = vb[j];
        }
      }
    }
  }
  // each thread orders its stores for the TMA loads that read them; the
  // barrier orders all of them before warp 7's releases
  fence_proxy_async_global();
  named_bar_sync(5, 32 * kW);
  if (gw == kW - 1) {
    for (int a = lane; a < rt.n_exp; a += 32) {
      if (rt.act[a] == p.E) continue;
      const int nr = owned_rows(rt, a, G);
      if (nr > 0) red_release_gpu_add(&p.gathered[a], nr);
    }
  }
}

template <bool kQ4>
__device__ __forceinline__ void expert_roles(const ExpertArgs& p, const Smem& s, const Rt& rt, uint32_t tmem_base) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_total = n_units(rt, p);
  if (warp == 0) {
    if (lane == 0) producer_a<kQ4>(p, s, rt, n_total);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(p, s, rt, tmem_base);
  } else if (warp == 2) {
    if (lane == 0) producer_b(p, s, rt);
  } else if (warp < 7) {
    if (rt.gather) gather_rows(p, rt);
    epilogue(p, s, rt, tmem_base);
  } else if (warp == 7) {
    if (rt.gather) gather_rows(p, rt);  // otherwise warp 7 has no role here
  } else if (kQ4) {
    converter(p, s, rt, tmem_base);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

namespace {

// Grid-wide barrier for a persistent launch (every CTA is resident: one per
// SM). The arrival count only grows: the arrival number a CTA draws tells it
// which multiple of the grid size ends its barrier, so nothing is reset and
// the last CTA to arrive leaves at once. Waits are bounded; returns false on
// timeout.
__device__ bool grid_barrier(unsigned long long* count, int* err) {
  __shared__ int s_pass;
  // Ordering: the CTA barrier orders every thread's earlier stores before
  // thread 0's release (its acq_rel arrival), and thread 0's acquire before
  // every thread's later loads (which read other CTAs' data through L2 or
  // TMA), so no thread needs a fence of its own (same box: a fence in every
  // thread on both sides cost 5.690 vs 5.630 ms per step).
  fence_proxy_async_global();  // rows stored before the barrier are read by TMA after it
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long g = gridDim.x;
    const unsigned long long old = atom_add_acq_rel_gpu_u64(count, 1ull);
    const unsigned long long target = (old / g + 1ull) * g;
    int pass = 1;
    if (old + 1ull != target) {
      const unsigned long long t0 = global_ns();
      while (ld_acquire_gpu_u64(count) < target) {
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, kErrDepTimeout);
          pass = 0;
          break;
        }
        __nanosleep(20);
      }
    }
    s_pass = pass;
  }
  __syncthreads();
  fence_proxy_async_global();
  return s_pass != 0;
}

}  // namespace

// Every CTA calls this last. The CTA that finishes last resets the unit
// counter and the per-unit-table counters the launch used, so that the next
// launch on the workspace finds them at zero without a barrier of its own
// (the next kernel reads them only after its dependency wait, which sees
// this grid complete). A clean launch leaves the unit counter at n_total
// plus one failed draw per CTA; anything else (units skipped or never
// drawn) is reported.
__device__ void exit_reset(const ExpertArgs& p, int n_entries, int n_total, bool gathered) {
  __shared__ int s_lastx;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // (cumulative over the CTA's accesses ordered by the barrier)
    const int old = atomicAdd(p.exit_ctr, 1);
    __threadfence();
    s_lastx = (old == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_lastx) {
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) {
      p.gu_done[i] = 0;
      if (gathered) p.gathered[i] = 0;
    }
    if (threadIdx.x == 0) {
      if (n_total > 0 && *reinterpret_cast<volatile int*>(p.unit_ctr) != n_total + static_cast<int>(gridDim.x))
        atomicOr(p.err, kErrState);
      *p.unit_ctr = 0;
      *p.exit_ctr = 0;
    }
  }
}

template <bool kQ4>
__global__ void __launch_bounds__(kQ4 ? kExpertThreadsQ4 : kExpertThreads, 1)
    k_expert(const __grid_constant__ ExpertArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve(smem_raw, p);
  const uint32_t tmem_base = expert_prologue<kQ4>(p, s);
  pdl_wait();
  pdl_trigger();
  const int M = p.M, K = p.K, E = p.E, MK = M * K;
  // Every CTA builds the same permutation of the routing kernel's top-k (its
  // scratch in the still idle weight ring) and keeps the token of every row
  // and the unit tables in its own shared memory, so no CTA waits for
  // another before its units: the weight stream starts right after the
  // permutation, while warps 3-7 gather the token rows chunk by chunk
  // and each gate/up unit waits only for its own chunk's rows.
  uint16_t* row_tok = reinterpret_cast<uint16_t*>(s.rt_region);
  const int NC = p.max_chunks;
  int* c_act = reinterpret_cast<int*>(s.rt_region + ((2 * MK + 15) & ~15));
  int* c_off = c_act + NC;
  int* c_cnt = c_off + NC;
  uint16_t* list = reinterpret_cast<uint16_t*>(c_cnt + NC);  // [M*K] rows this CTA gathers
  PermTables pt;
  const int ws = perm_stride(M);
  // (every table starts on a 16-byte boundary of the 1 KiB-aligned ring)
  const int E4 = (E + 3) & ~3;
  pt.bm = reinterpret_cast<uint32_t*>(s.a_ring);
  pt.off = reinterpret_cast<int*>(pt.bm + ((E * ws + 3) & ~3));
  pt.cnt = pt.off + E4;
  pt.tmp = pt.cnt + E4;
  int* by_rank = pt.tmp + 32;  // [E] active expert ids, heaviest first
  pt.pre = reinterpret_cast<uint16_t*>(by_rank + E4);
  pt.idx = reinterpret_cast<uint8_t*>(pt.pre + ((E * ws + 7) & ~7));
  pt.row_tok = row_tok;
  const int n_act = cta_permutation(p.topk_idx, M, K, E, pt, blockIdx.x == 0 ? p.tok_slot : nullptr);
  const int tid = threadIdx.x;
  // Unit tables: the expert's tokens in chunks of at most kExpertTileTokens rows
  // (one accumulator's width): the shared expert's chunks first, then the
  // routed experts heaviest first (ties: lower id first), so that the
  // longest units are handed out first and do not end the launch; an
  // expert's chunks are adjacent, so its weight tiles are asked for at
  // nearly the same time by the CTAs that take them.
  constexpr int TR = kExpertTileTokens;
  const int n_sh = (M + TR - 1) / TR;
  if (tid < E) {
    const int c = pt.cnt[tid];
    if (c > 0) {
      int rank = 0;
      const int4* c4 = reinterpret_cast<const int4*>(pt.cnt);  // 16-byte aligned; the tail past E / 4 is read below
      const int e4 = E >> 2;
      for (int j = 0; j < e4; ++j) {
        const int4 v = c4[j];
        const int b = 4 * j;
        rank += (v.x > c || (v.x == c && b < tid)) + (v.y > c || (v.y == c && b + 1 < tid)) +
                (v.z > c || (v.z == c && b + 2 < tid)) + (v.w > c || (v.w == c && b + 3 < tid));
      }
      for (int j = e4 * 4; j < E; ++j) {
        const int cj = pt.cnt[j];
        rank += (cj > c || (cj == c && j < tid)) ? 1 : 0;
      }
      by_rank[rank] = tid;
    }
  }
  if (tid < n_sh) {
    c_act[tid] = E;
    c_off[tid] = MK + tid * TR;
    c_cnt[tid] = min(TR, M - tid * TR);
  }
  __syncthreads();
  const int e = tid < n_act ? by_rank[tid] : 0;
  const int ce = tid < n_act ? pt.cnt[e] : 0;
  const int nch = (ce + TR - 1) / TR;
  int n_chunks = 0;
  const int first = n_sh + block_excl_scan(nch, pt.tmp, &n_chunks);
  const bool fits = n_sh + n_chunks <= NC;  // the host sized the tables for the worst case
  for (int c = 0; c < nch && first + c < NC; ++c) {
    c_act[first + c] = e;
    c_off[first + c] = pt.off[e] + c * TR;
    c_cnt[first + c] = min(TR, ce - c * TR);
  }
  if (blockIdx.x == 0) {
    if (!fits && tid == 0) atomicOr(p.err, kErrBadRoute);
    if (p.out_idx)
      for (int i = tid; i < MK; i += blockDim.x) p.out_idx[i] = pt.idx[i];
    if (p.out_w)
      for (int i = tid; i < MK; i += blockDim.x) p.out_w[i] = p.topk_w[i];
  }
  // Paired chunks: those of the experts with more than p.pair_rows tokens, a
  // prefix of the chunk list (the shared expert's chunks first, then the
  // routed experts heaviest first).
  __shared__ int s_npair;
  if (tid == 0) s_npair = 0;
  __syncthreads();
  if (p.pair_rows >= 0 && tid < n_act && ce > p.pair_rows) atomicAdd(&s_npair, nch);
  fence_proxy_async_shared();  // the ring was used generically; TMA refills it
  __syncthreads();
  Rt rt;
  rt.act = c_act;
  rt.cnt = c_cnt;
  rt.off = c_off;
  rt.mask = nullptr;
  rt.tok_slot = p.tok_slot;
  rt.topk_w = p.topk_w;
  rt.n_exp = fits ? n_sh + n_chunks : 0;
  rt.n_pair = (p.pair_rows >= 0 && M > p.pair_rows && fits) ? n_sh + s_npair : 0;
  rt.dense = 0;
  rt.chunked = 1;
  rt.row_tok = row_tok;
  rt.list = list;
  rt.n_list = MK;
  rt.gather = 1;
  expert_roles<kQ4>(p, s, rt, tmem_base);
  exit_reset(p, rt.n_exp, n_units(rt, p), true);
}


// One MoE sublayer for M <= 32 tokens in one launch: routing, experts and
// combine (see the file comment).
template <bool kQ4>
__global__ void __launch_bounds__(kQ4 ? kExpertThreadsQ4 : kExpertThreads, 1)
    k_layer(const __grid_constant__ ExpertArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve(smem_raw, p);
  // bulk-copy barriers: router slices, token rows
  uint64_t* wbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.tmem_slot) + 96);
  uint64_t* xbar = wbar + 1;
  if (threadIdx.x == 0) {  // made visible by the prologue's fence
    mbar_init(wbar, 1);
    mbar_init(xbar, 1);
  }
  const uint32_t tmem_base = expert_prologue<kQ4>(p, s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int M = p.M, K = p.K, E = p.E, H = p.H;
  const int MK = M * K;

  // shared routing tables
  int32_t* s_idx = reinterpret_cast<int32_t*>(s.rt_region);  // [M*K]
  float* s_w = reinterpret_cast<float*>(s_idx + MK);         // [M*K]
  int32_t* s_slot = reinterpret_cast<int32_t*>(s_w + MK);    // [M*K]
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_slot + MK);  // [E]
  int* s_cnt = reinterpret_cast<int*>(s_mask + E);             // [E]
  int* s_off = s_cnt + E;                                       // [E]
  int* s_act = s_off + E;                                       // [E]
  int* s_nact = s_act + E;                                      // [1]

  // Phase 1 work items: (8 experts, 8 tokens); one token per warp.
  const int n_eg = (E + kRouteExperts - 1) / kRouteExperts;
  const int n_tg = (M + kRouteTokens - 1) / kRouteTokens;
  const int n_items = n_eg * n_tg;
  // Router rows do not depend on earlier kernels: copy this CTA's slices
  // into the (still idle) weight ring before waiting.
  const int my_items = (n_items > static_cast<int>(blockIdx.x)) ? (n_items - 1 - blockIdx.x) / G + 1 : 0;
  const uint32_t ring_bytes = static_cast<uint32_t>(p.smem_a) * s.a_stage_bytes;
  // At the Clover shape a CTA with one item of 8 experts contracts it on the
  // warp tensor cores: router rows, token rows, normed rows and partials in
  // the idle ring, the bf16 rows padded by 8 elements (bank-conflict-free
  // fragment loads).
  constexpr int kMmaH = 2048;
  constexpr uint32_t kMmaRow = (kMmaH + 8) * 2;
  const int my_ne = my_items == 1 ? min(kRouteExperts, E - (static_cast<int>(blockIdx.x) % n_eg) * kRouteExperts) : 0;
  const bool mma_route = my_items == 1 && H == kMmaH && my_ne == kRouteExperts &&
                         kRouteExperts * kMmaRow + kRouteTokens * kMmaH * 4 + kRouteTokens * kMmaRow +
                                 kRouteTokens * kRouteTokens * 8 * 4 <= ring_bytes;
  const uint32_t wslice = mma_route ? kRouteExperts * kMmaRow : kRouteExperts * H * 2;
  const bool wr_staged = my_items * wslice <= ring_bytes;
  // A CTA with one item also stages that item's token rows (contiguous in
  // x_in) behind its router slices, when they fit.
  const int xt0 = (blockIdx.x / n_eg) * kRouteTokens;
  const uint32_t x_off = my_items * wslice;
  const uint32_t x_bytes = my_items == 1 ? static_cast<uint32_t>(min(kRouteTokens, M - xt0)) * H * 4 : 0u;
  const bool x_staged = wr_staged && my_items == 1 && x_off + x_bytes <= ring_bytes;
  const uint32_t xn_off = x_off + kRouteTokens * kMmaH * 4;            // mma_route: normed rows
  const uint32_t part_off = xn_off + kRouteTokens * kMmaRow;           // mma_route: partial tiles
  if (threadIdx.x == 0 && wr_staged && my_items > 0) {
    uint32_t bytes = 0;
    for (int j = 0; j < my_items; ++j) {
      const int eg = (blockIdx.x + j * G) % n_eg;
      bytes += min(kRouteExperts, E - eg * kRouteExperts) * H * 2;
    }
    mbar_arrive_expect_tx(wbar, bytes);
    for (int j = 0; j < my_items; ++j) {
      const int eg = (blockIdx.x + j * G) % n_eg;
      const int ne = min(kRouteExperts, E - eg * kRouteExperts);
      const bf16* src = p.wr + static_cast<size_t>(eg) * kRouteExperts * H;
      if (mma_route) {
        for (int r = 0; r < ne; ++r) bulk_load(smem_u32(s.a_ring) + r * kMmaRow, src + static_cast<size_t>(r) * H, H * 2, wbar);
      } else {
        bulk_load(smem_u32(s.a_ring) + j * wslice, src, ne * H * 2, wbar);
      }
    }
  }
  unsigned long long* st = (kPhaseStamps && blockIdx.x == 0 && threadIdx.x == 0) ? p.stamps : nullptr;
  if (st) st[0] = global_ns();
  pdl_wait();
  pdl_trigger();
  if (st) st[1] = global_ns();
  if (p.pend) {
    // The previous layer left its combine to this launch: every CTA combines
    // its share of (token, 128-wide slice) pieces from the previous layer's
    // expert rows and published tables, one warp per piece, then a grid
    // barrier before any CTA reads the combined rows.
    Rt prev;
    prev.tok_slot = p.tok_slot;
    prev.topk_w = p.fin_w;
    const int SH = H >> 7, n_pieces = M * SH, nw = blockDim.x >> 5;
    for (int pc = blockIdx.x + G * warp; pc < n_pieces; pc += G * nw)
      combine_token(p, prev, pc % SH, pc / SH, lane);
    if (!grid_barrier(p.bar_count, p.err)) *s.abort = 1u;
  }
  if (threadIdx.x == 0 && x_staged) {  // written by the previous kernel (or just combined)
    mbar_arrive_expect_tx(xbar, x_bytes);
    bulk_load(smem_u32(s.a_ring) + x_off, p.x_in + static_cast<size_t>(xt0) * H, x_bytes, xbar);
  }

  // Phase 1: norms, normed rows (written once) and router logits.
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) p.gu_done[i] = 0;
    for (int i = threadIdx.x; i < (H >> 7); i += blockDim.x) p.dn_done[i] = 0;
    if (threadIdx.x == 0) {
      *p.unit_ctr = 0;
    }
  }
  if (wr_staged && my_items > 0 && !mbar_wait(wbar, 0, s.abort)) {
    atomicOr(p.err, kErrMbarTimeout);
    *s.abort = 1u;
  }
  if (mma_route && warp < kRouteTokens) {
    const int item = blockIdx.x;
    const int eg = item % n_eg, tg = item / n_eg;
    const int e0 = eg * kRouteExperts;
    const int t = tg * kRouteTokens + warp;
    if (x_staged && !mbar_wait(xbar, 0, s.abort)) {
      atomicOr(p.err, kErrMbarTimeout);
      *s.abort = 1u;
    }
    const float lg = cta_router_item_mma<kMmaH>(smem_u32(s.a_ring + x_off), min(kRouteTokens, M - tg * kRouteTokens),
                                                p.eps, smem_u32(s.a_ring), smem_u32(s.a_ring + xn_off),
                                                reinterpret_cast<float*>(s.a_ring + part_off),
                                                eg == 0 ? p.xn + static_cast<size_t>(tg) * kRouteTokens * H : nullptr,
                                                warp, lane, 6);
    if (t < M && lane < kRouteExperts) {
      const float v = lg + (p.bias ? p.bias[e0 + lane] : 0.f);
      p.logits[static_cast<size_t>(t) * E + e0 + lane] = v;
    }
  }
  for (int item = blockIdx.x, j = 0; item < n_items && !mma_route; item += G, ++j) {
    const int eg = item % n_eg, tg = item / n_eg;
    const int e0 = eg * kRouteExperts;
    const int ne = min(kRouteExperts, E - e0);
    const int t = tg * kRouteTokens + warp;
    if (warp < kRouteTokens && t < M) {
      if (x_staged && !mbar_wait(xbar, 0, s.abort)) {
        atomicOr(p.err, kErrMbarTimeout);
        *s.abort = 1u;
      }
      const float* xr = x_staged ? reinterpret_cast<const float*>(s.a_ring + x_off) + static_cast<size_t>(warp) * H
                                 : p.x_in + static_cast<size_t>(t) * H;
      const __nv_bfloat16* w_rows = wr_staged ? reinterpret_cast<const __nv_bfloat16*>(s.a_ring + j * wslice)
                                              : p.wr + static_cast<size_t>(e0) * H;
      __nv_bfloat16* xn_out = eg == 0 ? p.xn + static_cast<size_t>(t) * H : nullptr;
      float lg;
      if (x_staged && wr_staged && H == 2048 && ne == kRouteExperts) {
        lg = warp_router_row_smem<kRouteExperts, 2048>(smem_u32(xr), p.eps, smem_u32(w_rows), lane, xn_out);
      } else if (H <= 128 * 16) {
        lg = warp_router_row_reg<kRouteExperts, 16>(xr, p.eps, w_rows, ne, H, lane, xn_out, !x_staged);
      } else {
        const float rstd = row_rstd(xr, H, p.eps, lane, !x_staged);
        lg = warp_router_dots<kRouteExperts>(xr, rstd, w_rows, ne, H, lane, xn_out, !x_staged);
      }
      if (lane < ne) {
        const float v = lg + (p.bias ? p.bias[e0 + lane] : 0.f);
        p.logits[static_cast<size_t>(t) * E + e0 + lane] = v;
      }
    }
  }
  fence_proxy_async_shared();  // the ring was read generically; TMA refills it later
  if (kPhaseStamps && p.stamps != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(p.stamps + 2, global_ns());
  }
  if (!grid_barrier(p.bar_count, p.err)) *s.abort = 1u;
  if (st) st[3] = global_ns();

  // Top-k: CTA t (< M) takes token t with one warp and publishes its
  // selections; a second barrier, then every CTA copies all of them into
  // its routing tables. (The same selection in every CTA for all M tokens
  // costs several µs of cross-lane reductions per CTA; spread over M CTAs it
  // is one token's worth.)
  const bool coreset = p.coreset_top_p > 0.f;
  float* s_p = reinterpret_cast<float*>(s_nact + 1);  // [M*K] full-softmax probability of each selection
  auto route_token = [&](int t, const uint32_t* allowed, bool want_p, int32_t* out_idx, float* out_w, float* out_p) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? __ldcg(p.logits + static_cast<size_t>(t) * E + e) : -INFINITY;
    }
    TopkSel sel[1];
    warp_topk_regs<1>(v, E, K, lane, allowed, want_p, sel);
    if (lane < K) {
      out_idx[t * K + lane] = sel[0].e;
      out_w[t * K + lane] = sel[0].w;
      if (want_p) out_p[t * K + lane] = sel[0].p;
    }
  };
  if (static_cast<int>(blockIdx.x) < M && warp == 0) route_token(blockIdx.x, nullptr, coreset, p.pub_idx, p.pub_w, p.pub_p);
  if (!grid_barrier(p.bar_count, p.err)) *s.abort = 1u;
  for (int i = threadIdx.x; i < MK; i += blockDim.x) {
    // all loads before the stores (shared and global through generic
    // pointers would otherwise keep each load behind the previous store)
    const int e = __ldcg(p.pub_idx + i);
    const float wv = __ldcg(p.pub_w + i);
    const float pv = coreset ? __ldcg(p.pub_p + i) : 0.f;
    s_idx[i] = e < 0 ? 0 : (e >= E ? E - 1 : e);
    s_w[i] = wv;
    if (coreset) s_p[i] = pv;
  }
  if (coreset) {
    // Block coreset (the M tokens are one block): every CTA computes the
    // same kept set from the first-pass selections, CTA t re-routes token t
    // within it, and a third barrier publishes the result.
    float* s_mass = s_p + MK;                                // [E]
    float* s_smass = s_mass + E;                             // [E] masses in kept order
    int* s_sid = reinterpret_cast<int*>(s_smass + E);        // [E] expert ids in kept order
    uint32_t* s_allow = reinterpret_cast<uint32_t*>(s_sid + E);  // [8]
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0u;
    if (threadIdx.x < 8) s_allow[threadIdx.x] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < MK; i += blockDim.x) atomicOr(&s_mask[s_idx[i]], 1u << (i / K));
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {  // mass: probabilities in token order
      float m = 0.f;
      for (uint32_t bm = s_mask[e]; bm != 0u; bm &= bm - 1u) {
        const int t = __ffs(bm) - 1;
        for (int k = 0; k < K; ++k)
          if (s_idx[t * K + k] == e) m += s_p[t * K + k];
      }
      s_mass[e] = m;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {  // rank by (mass desc, id asc)
      const float me = s_mass[e];
      int r = 0;
      for (int e2 = 0; e2 < E; ++e2) {
        const float m2 = s_mass[e2];
        r += (m2 > me || (m2 == me && e2 < e)) ? 1 : 0;
      }
      s_smass[r] = me;
      s_sid[r] = e;
    }
    __syncthreads();
    if (warp == 0) {
      // total in kept order, then the shortest prefix reaching top_p x total
      // that holds at least K experts
      float total = 0.f;
      for (int c0 = 0; c0 < E; c0 += 32) total += warp_sum_f(c0 + lane < E ? s_smass[c0 + lane] : 0.f);
      const float target = p.coreset_top_p * total;
      float carry = 0.f;
      int cut = E - 1;
      for (int c0 = 0; c0 < E; c0 += 32) {
        float cv = c0 + lane < E ? s_smass[c0 + lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float nb = __shfl_up_sync(0xffffffffu, cv, o);
          if (lane >= o) cv += nb;
        }
        const float cum = carry + cv;
        const unsigned hit = __ballot_sync(0xffffffffu, c0 + lane < E && cum >= target && c0 + lane >= K - 1);
        if (hit) {
          cut = c0 + __ffs(hit) - 1;
          break;
        }
        carry += __shfl_sync(0xffffffffu, cv, 31);
      }
      for (int r = lane; r <= cut; r += 32) atomicOr(&s_allow[s_sid[r] >> 5], 1u << (s_sid[r] & 31));
    }
    __syncthreads();
    if (static_cast<int>(blockIdx.x) < M && warp == 0)
      route_token(blockIdx.x, s_allow, false, p.pub2_idx, p.pub2_w, nullptr);
    if (!grid_barrier(p.bar_count, p.err)) *s.abort = 1u;
    for (int i = threadIdx.x; i < MK; i += blockDim.x) {
      const int e = __ldcg(p.pub2_idx + i);
      const float wv = __ldcg(p.pub2_w + i);
      s_idx[i] = e < 0 ? 0 : (e >= E ? E - 1 : e);
      s_w[i] = wv;
    }
  }

  // Phase 2: every CTA builds the same permutation from its top-k tables.
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < MK; i += blockDim.x) atomicOr(&s_mask[s_idx[i]], 1u << (i / K));
  __syncthreads();
  {  // counts, offsets and the active list: warp w scans experts 32w..32w+31
    __shared__ int s_wsum[2][kMaxExperts / 32];
    const int e = threadIdx.x;
    const bool in = warp < kMaxExperts / 32;
    const int c = (in && e < E) ? __popc(s_mask[e]) : 0;
    int incl = c, acti = c > 0 ? 1 : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n1 = __shfl_up_sync(0xffffffffu, incl, o);
      const int n2 = __shfl_up_sync(0xffffffffu, acti, o);
      if (lane >= o) {
        incl += n1;
        acti += n2;
      }
    }
    if (in && lane == 31) {
      s_wsum[0][warp] = incl;
      s_wsum[1][warp] = acti;
    }
    __syncthreads();
    if (in && e < E) {
      int base_off = 0, base_act = 0;
      for (int w2 = 0; w2 < warp; ++w2) {
        base_off += s_wsum[0][w2];
        base_act += s_wsum[1][w2];
      }
      s_cnt[e] = c;
      s_off[e] = base_off + incl - c;
      if (c > 0) s_act[base_act + acti - 1] = e;
    }
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w2 = 0; w2 < kMaxExperts / 32; ++w2) tot += s_wsum[1][w2];
      *s_nact = tot;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < MK; i += blockDim.x) {
    const int e = s_idx[i], t = i / K;
    s_slot[i] = s_off[e] + __popc(s_mask[e] & ((1u << t) - 1u));
  }
  if (blockIdx.x == 0) {
    if (p.out_idx)
      for (int i = threadIdx.x; i < MK; i += blockDim.x) p.out_idx[i] = s_idx[i];
    if (p.out_w)
      for (int i = threadIdx.x; i < MK; i += blockDim.x) p.out_w[i] = s_w[i];
    if (p.combine == 2) {  // the next launch (or the combine kernel) combines from these
      for (int i = threadIdx.x; i < MK; i += blockDim.x) {
        p.tok_slot[i] = s_slot[i];
        p.fin_w[i] = s_w[i];
      }
    }
  }
  __syncthreads();

  Rt rt;
  rt.act = s_act;
  rt.cnt = s_cnt;
  rt.off = s_off;
  rt.mask = s_mask;
  rt.tok_slot = s_slot;
  rt.topk_w = s_w;
  rt.n_exp = (*s.abort) ? 0 : *s_nact + 1;  // after a failed barrier no unit runs
  rt.n_pair = 0;
  rt.dense = 1;
  rt.chunked = 0;
  rt.row_tok = nullptr;
  rt.list = nullptr;
  rt.n_list = 0;
  rt.gather = 0;
  if (st) st[4] = global_ns();
  expert_roles<kQ4>(p, s, rt, tmem_base);
  if (kPhaseStamps && p.stamps != nullptr && threadIdx.x == 0) atomicMax(p.stamps + 5, global_ns());
  exit_reset(p, E + 1, n_units(rt, p), false);
}

// smem_a: A stages in shared memory; stages_a: A barriers; kg: K groups of
// room per A/B stage.
size_t expert_smem_bytes(int smem_a, int stages_a, int stages_b, int nb_max, int stages_q, int kg) {
  return 1024 + static_cast<size_t>(smem_a) * kg * kATileBytes + static_cast<size_t>(stages_b) * kg * nb_max * 128 +
         static_cast<size_t>(stages_q) * kQSlotBytes + 2 * 64 * 20 * sizeof(float) +
         static_cast<size_t>(2 * stages_a + 2 * stages_b + 2 * stages_q + 5 + 2 * kExpertUnitRing) * 8 + 256;
}

// (k_layer) idx, w, slot, coreset probability [M*K] each; mask, count, offset, active,
// coreset mass, sorted mass, sorted id [E] each; the active count and the
// coreset's allowed-set words.
size_t perm_smem_bytes(int M, int K, int E) {
  const size_t ws = static_cast<size_t>(perm_stride(M)), e4 = (static_cast<size_t>(E) + 3) & ~static_cast<size_t>(3);
  return (((E * ws + 3) & ~static_cast<size_t>(3)) + 3 * e4 + 32) * 4 + ((E * ws + 7) & ~static_cast<size_t>(7)) * 2 +
         static_cast<size_t>(M) * K;
}

size_t expert_tables_bytes(int M, int K, int max_chunks) {
  // row tokens [M*K] u16, chunk tables 3 x [max_chunks] i32, gather list [M*K] u16
  return ((static_cast<size_t>(2) * M * K + 15) & ~static_cast<size_t>(15)) + static_cast<size_t>(3) * max_chunks * 4 +
         ((static_cast<size_t>(2) * M * K + 15) & ~static_cast<size_t>(15));
}

size_t layer_rt_bytes(int M, int K, int E) { return static_cast<size_t>(4 * M * K + 7 * E + 16) * 4; }

cudaError_t expert_resident_per_sm(bool fused, bool q4, size_t smem, int* n) {
  auto* k = fused ? (q4 ? k_layer<true> : k_layer<false>) : (q4 ? k_expert<true> : k_expert<false>);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k, q4 ? kExpertThreadsQ4 : kExpertThreads, smem);
}

cudaError_t launch_layer(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  auto* k = a.q4 ? k_layer<true> : k_layer<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(a.q4 ? kExpertThreadsQ4 : kExpertThreads), smem, s, pdl, a);
}

cudaError_t launch_expert(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  auto* k = a.q4 ? k_expert<true> : k_expert<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(a.q4 ? kExpertThreadsQ4 : kExpertThreads), smem, s, pdl, a);
}

}  // namespace clover
