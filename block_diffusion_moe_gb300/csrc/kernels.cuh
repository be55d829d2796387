// Kernel argument blocks and launch wrappers shared by the host API and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace clover {

using bf16 = __nv_bfloat16;

// Routing kernel tiling: 8 experts x 8 tokens (one per warp) per CTA.
constexpr int kRouteExperts = 8;
constexpr int kRouteTokens = 8;
// The standalone routing kernel (more than 32 tokens): one CTA per tile of 16
// tokens x 32 experts, contracted over the hidden size in chunks of 2048.
constexpr int kRouteTileTokens = 16;
constexpr int kRouteTileExperts = 32;
constexpr int kRouteChunk = 2048;
// Tokens per call, and per token tile: an expert's tokens and the head's
// positions are processed in tiles of at most kTileTokens (the N side of a
// tcgen05.mma and of one TMEM accumulator).
constexpr int kMaxTokens = 1024;
constexpr int kTileTokens = 256;
// The standalone expert kernel's token tile: an expert's tokens run in
// chunks of at most this many rows. 128 rather than 256 halves the B stages
// (16 KiB per K group), which leaves room for a deeper weight ring (the
// weight stream's rate follows the bytes in flight); an expert with more
// tokens streams its weights once per chunk, the chunks' requests for the
// same tile arriving together (the repeat is served by L2).
constexpr int kExpertTileTokens = 128;
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;

// Expert kernel: 8 warps (A loads, MMA, B loads, 4 epilogue warps, and one
// more that only takes part in the fused kernel's routing phase).
constexpr int kExpertThreads = 256;
// With low-bit expert weights eight more warps (two teams of four) expand
// the 4-bit codes.
constexpr int kExpertThreadsQ4 = 512;
constexpr int kExpertUnitRing = 4;
// Head kernel: 6 warps (loads, MMA, 4 epilogue warps).
constexpr int kHeadThreads = 192;
constexpr int kHeadMaxCtas = 512;

constexpr int kATileBytes = 128 * 64 * 2;  // 128 rows x 64 bf16
// Low-bit staging: per K group of 64, a tile is 128 rows x 32 bytes of codes
// (4 KiB) + 128 bf16 scales; a slot holds up to 4 consecutive groups, so each
// row arrives as one contiguous piece of up to 128 bytes.
constexpr int kQGroupBytes = 128 * 32 + 128 * 2;
constexpr int kQSlotGroups = 4;
constexpr int kQSlotBytes = kQSlotGroups * kQGroupBytes;
// First TMEM column of the A stages when A lives in tensor memory (after the
// two 64-column accumulators); each stage of four K groups takes 128 columns.
constexpr int kTmemAStage0 = 128;
constexpr int kSmemBudget = 227 * 1024;

// Phase timestamps of the fused layer kernel (a diagnostic: a barrier and
// global atomics per launch). Off unless built with -DCLOVER_PHASE_STAMPS=1.
#ifndef CLOVER_PHASE_STAMPS
#define CLOVER_PHASE_STAMPS 0
#endif
constexpr bool kPhaseStamps = CLOVER_PHASE_STAMPS != 0;

struct EmbedArgs {
  const int32_t* tokens;
  const bf16* embed;  // [V][H]
  const float* ctx;   // [M][H]
  float* x;           // [M][H]
  int* err;
  int M, H, V;
};

struct NormArgs {
  const float* x;  // [M][H]
  bf16* xn;        // [M][H]
  int M, H;
  float eps;
};

struct RouteArgs {
  const float* x;       // [M][H] residual stream
  const bf16* wr;       // [E][H]
  const float* bias;    // [E] or null
  float* logits;        // [M][E]
  bf16* xn_rows;        // [M][H] normed input (the shared expert's rows of the gathered buffer)
  int* tg_ctr;          // [ceil(M/16)] arrival counters, zero between launches
  int* err;             // error bits (kErr*)
  int32_t* topk_idx;    // [M][K]
  float* topk_w;        // [M][K]
  int M, H, E, K;
  float eps;
  int xn_ready;  // 1: xn_rows already hold the normed rows (the previous layer's combine wrote them; H <= kRouteChunk)
};


struct CombineArgs {
  const float* x_in;        // [M][H]
  float* x_out;             // [M][H] (may equal x_in)
  const float* yslot;       // [M*K + M][H] unweighted expert outputs
  const int32_t* tok_slot;  // [M][K]
  const float* topk_w;      // [M][K]
  int M, H, K;
  bf16* xn_out;  // non-null: also write the next layer's normed rows [M][H] (H <= kRouteChunk)
  float eps;
};

struct ExpertArgs {
  CUtensorMap tm_gu;   // routed gate/up  [E*2F][H]
  CUtensorMap tm_sgu;  // shared gate/up  [2F][H]
  CUtensorMap tm_dn;   // routed down     [E*H][F]
  CUtensorMap tm_sdn;  // shared down     [H][F]
  // Whole-stage views of the same bf16 weights (stage_maps != 0): an A
  // stage of two K groups of one slice in one TMA instruction instead of
  // two (down) or four (gate/up): gate/up (64 c, rows, gate|up, K group),
  // box 64 x 64 x 2 x 2; down (64 c, rows, K group), box 64 x 128 x 2. Each
  // view aliases dimensions of the 2-D matrix, its row extent cut so that
  // no in-range coordinate reaches past the tensor.
  CUtensorMap tm_gu_k2, tm_sgu_k2, tm_dn_k2, tm_sdn_k2;
  int stage_maps;
  CUtensorMap tm_xg;   // gathered inputs [M*K+M][H], boxes of 16 rows
  CUtensorMap tm_h;    // SwiGLU outputs  [M*K+M][F], boxes of 16 rows
  CUtensorMap tm_xg_big;  // the same, boxes of xg_box rows
  CUtensorMap tm_h_big;   // the same, boxes of h_box rows
  int xg_box, h_box;      // rows per big box (multiples of 16)
  // Fused kernel (xg_k != 0): the normed rows of a gate/up stage's kg_gu K
  // groups in one box (64 c, rows, K group at a stride of 128 bytes; box 64 x
  // xg_box x kg_gu), the same layout as kg_gu 2-D boxes.
  CUtensorMap tm_xg_k;
  int xg_k;
  // Low-bit expert weights (q4 != 0): codes by TMA (uint8, box 32 B x rows),
  // scales by bulk copy; stages_q staging slots of kQSlotBytes.
  CUtensorMap tm_gu_q;   // [E*2F][H/2]
  CUtensorMap tm_sgu_q;  // [2F][H/2]
  CUtensorMap tm_dn_q;   // [E*H][F/2]
  CUtensorMap tm_sdn_q;  // [H][F/2]
  // Whole-slot views (q4_views != 0): a gate/up slot's codes in one box
  // (kq*32 bytes, 64 rows, gate|up at a stride of F rows) and every slot's
  // scales in one box (gate/up: 64 scales, gate|up, kq K groups; down: 128
  // scales, kq K groups) instead of two code boxes and 2 kq (gate/up) or kq
  // (down) scale copies (fewer copies per slot measured faster).
  CUtensorMap tm_gu_q3, tm_sgu_q3, tm_gu_sv, tm_sgu_sv, tm_dn_sv, tm_sdn_sv;
  int q4_views;
  const uint16_t* gu_s;   // [E][H/64][2F]
  const uint16_t* sgu_s;  // [H/64][2F]
  const uint16_t* dn_s;   // [E][F/64][H]
  const uint16_t* sdn_s;  // [F/64][H]
  int q4, stages_q;
  int q_teams;  // converter teams (1 or 2; 2 only when every team owns its stages and slots)
  int kq_gu, kq_dn;  // K groups per staging slot for gate/up and down units (1, 2 or 4)
  // Low-bit, fused kernel, four K groups per stage: the converters write the
  // bf16 A tiles into tensor memory (columns kTmemAStage0 + 128 s for stage
  // s) and the MMA reads A from there; the staging slots then take the A
  // ring's shared memory, which only the prelude uses.
  int a_tmem;
  int q_in_a;
  int acc_cols;  // TMEM columns per accumulator: 256, or 64 with a_tmem
  // Standalone bf16 kernel: the chunks of experts with more than pair_rows
  // tokens run as paired units (two weight slices of one K group per stage,
  // two accumulators of at most 128 columns sharing each B tile); negative:
  // none.
  int pair_rows;
  int smem_a;  // A stages in shared memory (= stages_a)
  // K groups of 64 per A/B stage (1, 2, or 4 on the low-bit path) for
  // gate/up and down units; a stage holds kg_stage groups of room (part h
  // of a stage: group h).
  int kg_gu, kg_dn, kg_stage;
  const float* x_in;
  float* x_out;
  bf16* hbuf;          // [M*K+M][F]
  float* yslot;        // [M*K+M][H]
  int* n_active;
  int* act;
  int* cnt;
  int* off;
  int32_t* tok_slot;
  const float* topk_w;
  const int32_t* topk_idx;  // standalone kernel: [M][K] selections to permute
  bf16* xg;                 // standalone kernel: gathered rows [M*K][H] (normed rows follow at xn)
  int* unit_ctr;
  int* gu_done;
  int* dn_done;
  int* gathered;   // standalone kernel: [max_chunks] rows of each chunk gathered so far
  int* exit_ctr;   // CTAs that finished this launch; the last one resets the unit counters
  int max_chunks;  // standalone kernel: room of the chunk tables
  int* err;
  int M, H, F, E, K;
  int stages_a, stages_b, nb_max;  // ring depths and B-tile rows per stage
  int combine;  // 1: the down unit that completes a hidden slice combines it; 0: k_combine does;
                // 2 (fused kernel): no combine here, the final tables are published for a later one
  int pend;     // fused kernel: first combine the previous launch's deferred output (same workspace)
  float* fin_w; // [M][K] final selection weights published for a deferred combine
  // fused-layer launches only (k_layer)
  const bf16* wr;      // [E][H] router
  const bf16* sgu_next;  // the next layer's shared expert (nullable): prefetched into L2 at the end
  const bf16* sdn_next;
  const bf16* wr_next; // [E][H] the next layer's router (nullable): its slices are prefetched into L2
  const float* bias;   // [E] or null
  float* logits;       // [M][E]
  bf16* xn;            // [M][H] normed rows = the gate/up B operand
  unsigned long long* bar_count;  // grid barrier arrivals (only grows; 8-byte aligned)
  int32_t* pub_idx;    // [M][K] top-k ids published by CTA t for token t
  float* pub_w;        // [M][K] top-k weights, likewise
  float* pub_p;        // [M][K] full-softmax probability of each selection (coreset mass)
  int32_t* pub2_idx;   // [M][K] selections after the coreset re-routing
  float* pub2_w;       // [M][K] their weights
  float coreset_top_p; // 0: no coreset
  int32_t* out_idx;    // optional [M][K] copies for the caller
  float* out_w;
  float eps;
  unsigned long long* stamps;  // optional phase timestamps (diagnostics): [0] start, [1] after the
                               // dependency wait, [2] last CTA done with the router logits, [3]
                               // after the barrier, [4] routing done, [5] last CTA done, [6] last
                               // down unit's outputs stored
};

struct HeadArgs {
  CUtensorMap tm_w;  // head [V][H]
  CUtensorMap tm_x;  // normed positions [M][H]
  const float* alpha;  // [M] or null
  float* part_m;       // [G][M]
  float* part_s;       // [G][M]
  int* part_a;         // [G][M]
  int* done_ctr;       // scalar, zero between launches (the merge kernel's arrivals)
  float* dec_m;        // [M] per-position decision input: max probability (accept: p(draft))
  float* dec_s;        // [M] accept: entropy
  int* dec_a;          // [M] argmax
  int n_parts;         // G: CTAs of the head launch (partial states to merge)
  int32_t* tokens;     // [M] in/out
  uint8_t* masked;     // [M] in/out
  int32_t* argmax;     // [M] out (nullable)
  float* max_logit;    // [M] out (nullable)
  float* lse;          // [M] out (nullable)
  float* max_prob;     // [M] out (nullable)
  int* n_committed;    // scalar out (nullable)
  int* n_masked_left;  // scalar out (nullable)
  int* err;
  int M, H, V, mask_id, block, n_tiles, stages;
  int accumulate;  // 1: add this call's counts to *n_committed / *n_masked_left (a later sub-call of a split call)
  int kg;     // K groups of 64 per pipeline stage (1 or 2)
  int x_box;  // rows per TMA box of the normed positions (a multiple of 16)
  float threshold;
  // Accept mode (self-speculative verify): blocks of `block` rows, row j
  // testing draft[j]; the unmask fields above are unused then.
  const int32_t* draft;  // [M]
  float* part_t;         // [G][M] sum of e^(z - m) (z - m)
  float* part_zd;        // [G][M] the draft's logit (-inf where not seen)
  float* entropy;        // [M] out (nullable)
  float* p_draft;        // [M] out (nullable)
  int32_t* accept_len;   // [M / block] out
  int32_t* out_tokens;   // [M] out
  int rule;              // 0 exact, 1 threshold
  float ratio, delta;
};

struct QuantArgs {
  const bf16* w;  // [n_mats][rows][cols]
  uint8_t* q;     // [n_mats][rows][cols / 2] codes
  uint16_t* s;    // [n_mats][cols / 64][rows] bf16 scales
  int n_mats, rows, cols;
};

// Launch wrappers (return the cudaError_t of the launch).
cudaError_t launch_quantize_q4(const QuantArgs& a, cudaStream_t s);
cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_rmsnorm(const NormArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl);
// k_combine_norm: the combine, then rmsnorm of each output row into a.xn_out.
cudaError_t launch_combine_norm(const CombineArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_expert(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_layer(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl);
// (both launch the low-bit form when a.q4 != 0)
// CTAs of the fused (k_layer) or standalone (k_expert) expert kernel that
// can be resident on one SM at the given dynamic shared memory size.
cudaError_t expert_resident_per_sm(bool fused, bool q4, size_t smem, int* n);
size_t layer_rt_bytes(int M, int K, int E);
// Shared memory the standalone expert kernel's permutation needs (in its weight ring).
size_t perm_smem_bytes(int M, int K, int E);
// Shared memory the standalone expert kernel keeps for its whole run: the
// token of every gathered row and the chunk tables.
size_t expert_tables_bytes(int M, int K, int max_chunks);
// Largest token count the fused layer kernel takes (one 32-bit mask per expert).
constexpr int kLayerMaxTokens = 32;
// Launches the unmask or the accept form of the head kernel.
cudaError_t launch_head(const HeadArgs& a, bool accept, int grid, size_t smem, cudaStream_t s, bool pdl);
// k_head_merge: merges the partial states of a k_head launch (one warp per
// position) and applies the unmask rule / accept test per block.
cudaError_t launch_head_merge(const HeadArgs& a, bool accept, cudaStream_t s, bool pdl);

size_t expert_smem_bytes(int smem_a, int stages_a, int stages_b, int nb_max, int stages_q, int kg);
size_t head_smem_bytes(int stages, int nb, bool accept, int kg);

}  // namespace clover
