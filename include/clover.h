/*
 * clover.h - C ABI of the GB300 (sm_103a) block-diffusion MoE denoising step.
 *
 * The operations follow "Clover-35B-A3B: how a diffusion model gets to 680
 * tokens a second, read from its files" (cited below as "Files"):
 *   - "What Clover is": per layer 256 routed experts, top-8 routing, one
 *     always-on shared expert; hidden 2,048; expert = gate and up 2,048 x 512,
 *     down 512 x 2,048; untied output head 248,320 x 2,048 read in full each
 *     step; block_size 32, mask_token_id 151669, low-confidence threshold 0.95.
 *   - "The expert selection": per-token top-8 routing probabilities.
 *   - "How it writes", steps 1-4: the block denoising loop and its unmask rule.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller. The library allocates no device memory; every
 *     scratch buffer lives in a caller-provided workspace whose size the
 *     matching *_workspace_bytes() call returns. A workspace must be
 *     zero-filled before its first use; afterwards the library keeps its
 *     control words consistent between calls. One workspace must not be used
 *     by two calls that may run at the same time.
 *   - bf16 tensors are passed as `const uint16_t*` (their bit patterns),
 *     row-major, densely packed, 16-byte aligned.
 *   - Every call is asynchronous on `stream` unless stated otherwise, and
 *     returns CLOVER_OK or a negative status. Argument errors are detected on
 *     the host before anything is enqueued. clover_last_error() returns the
 *     message of the last failing call on the calling thread.
 *   - Kernels never trap. A wait inside a kernel that exceeds its time limit
 *     records a flag in the workspace and the kernel returns;
 *     clover_workspace_status() reports it as CLOVER_ERR_DEVICE_TIMEOUT.
 *   - Shapes: hidden % 128 == 0, d_ff % 64 == 0, 1 <= top_k <= 32,
 *     top_k <= n_experts <= 256, hidden <= 8192, 1 <= tokens <= 1024,
 *     vocab >= 2, 0 <= mask_id < vocab. Other shapes return
 *     CLOVER_ERR_UNSUPPORTED_SHAPE; there is no fallback path. Above 32
 *     tokens an expert's tokens are processed in tiles of at most 128: an
 *     expert that more tokens select is streamed once per tile of its tokens
 *     (the tiles run side by side, so the repeat reads mostly come from L2);
 *     above 256 positions the head streams once per 256 positions.
 */
#ifndef CLOVER_H_
#define CLOVER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CLOVER_OK 0
#define CLOVER_ERR_INVALID_ARG (-1)
#define CLOVER_ERR_WORKSPACE_TOO_SMALL (-2)
#define CLOVER_ERR_CUDA (-3)
#define CLOVER_ERR_NOT_CONVERGED (-4)
#define CLOVER_ERR_UNSUPPORTED_SHAPE (-5)
#define CLOVER_ERR_DEVICE_TIMEOUT (-6)

/* cudaStream_t and cudaEvent_t are pointers to these opaque structs. */
typedef struct CUstream_st* clover_stream_t;
typedef struct CUevent_st* clover_event_t;

/* Model dimensions. Files, "What Clover is": hidden 2048, n_experts 256,
 * top_k 8, d_ff 512, vocab 248320, mask_id 151669; moe_block_coreset_enabled
 * with top_p 0.9. rms_eps is the epsilon of the unit-weight RMSNorm placed
 * before each MoE sublayer and before the head (a reading; the pages give no
 * norm).
 * coreset_top_p: 0 disables the block coreset; a value in (0, 1] enables it
 * (Files, "The expert selection"): per block, each expert's mass is the sum of
 * the softmax probabilities of the slots that select it; the kept set is the
 * shortest prefix of experts by mass (descending, lower id first) whose
 * cumulative mass reaches coreset_top_p x total and that holds at least
 * top_k experts; every token then takes its top_k within the kept set. The
 * coreset is available for calls of at most 32 positions forming one block. */
typedef struct {
    int32_t hidden;    /* H */
    int32_t n_experts; /* E, routed experts per layer */
    int32_t top_k;     /* K */
    int32_t d_ff;      /* F, expert intermediate width */
    int32_t vocab;     /* V */
    int32_t mask_id;   /* mask token id; never predicted */
    float rms_eps;
    float coreset_top_p; /* 0 = off */
} clover_dims;

/* One MoE layer's weights (device pointers). Files, "What Clover is". */
typedef struct {
    const uint16_t* router_w;   /* bf16 [E][H]                                   */
    const float* router_bias;   /* fp32 [E] added to the router logits, or NULL  */
    const uint16_t* gate_up;    /* bf16 [E][2F][H]: rows 0..F-1 gate, F..2F-1 up */
    const uint16_t* down;       /* bf16 [E][H][F]                                */
    const uint16_t* sh_gate_up; /* bf16 [2F][H], shared expert                   */
    const uint16_t* sh_down;    /* bf16 [H][F],  shared expert                   */
    /* Low-bit expert weights (format of clover_quantize_q4). When gate_up_q is
     * non-NULL all eight fields below must be set and the four bf16 expert
     * pointers above are ignored (may be NULL); the router stays bf16. */
    const uint8_t* gate_up_q;    /* codes [E][2F][H/2]   */
    const uint16_t* gate_up_s;   /* scales [E][H/64][2F] */
    const uint8_t* down_q;       /* codes [E][H][F/2]    */
    const uint16_t* down_s;      /* scales [E][F/64][H]  */
    const uint8_t* sh_gate_up_q; /* codes [2F][H/2]      */
    const uint16_t* sh_gate_up_s;/* scales [H/64][2F]    */
    const uint8_t* sh_down_q;    /* codes [H][F/2]       */
    const uint16_t* sh_down_s;   /* scales [F/64][H]     */
} clover_moe_layer;

/* Bytes of workspace clover_moe_block_step needs for up to max_tokens tokens.
 * Returns 0 for an unsupported shape. Host-only. */
size_t clover_moe_workspace_bytes(const clover_dims* dims, int32_t max_tokens);

/* One pre-norm MoE sublayer on M tokens (Files, "What Clover is" and "The
 * expert selection"):
 *   xn  = bf16(RMSNorm(x_in))
 *   p   = softmax(xn W_r^T + b), top-k by p (ties to the lower expert id),
 *         w = p_sel / sum(p_sel)
 *   y_t = sum_k w_tk * E_{i_tk}(xn_t) + S(xn_t),  E(x) = bf16(silu(x W_g^T) *
 *         (x W_u^T)) W_d^T, S the shared expert with weight 1
 *   x_out = x_in + y
 * x_in, x_out: fp32 [M][H]; x_out may equal x_in (in place), other overlap is
 * not allowed. topk_idx (int32 [M][K]) and topk_w (fp32 [M][K]) receive the
 * selection in descending probability order; either may be NULL.
 * Each selected expert's weights are read from HBM once per call (up to 32
 * tokens; above, once per tile of 128 of its tokens, the repeats of one
 * expert's tiles requested together so that L2 serves them). */
int clover_moe_block_step(const clover_dims* dims, const clover_moe_layer* layer,
                          const float* x_in, float* x_out,
                          int32_t* topk_idx, float* topk_w, int32_t M,
                          void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Low-bit expert weights. The pages name INT4 for one deployment (Files,
 * "What 680 tokens a second has to be") but give no format; this format is
 * the library's own. Quantizes n_mats bf16 matrices w [n_mats][rows][cols]
 * (cols % 64 == 0) into 4-bit codes q [n_mats][rows][cols/2] and bf16 scales
 * s [n_mats][cols/64][rows]: per row and group of 64 columns,
 *   s = bf16(float32(max |w|) / 7)          (IEEE fp32 division, nearest even)
 *   u = clamp(rint(float32(w) / s), -8, 7) + 8   (u = 8 where s = 0)
 * and the weight a product then uses is bf16((u - 8) s). Codes are packed
 * eight to a little-endian 32-bit word, nibble i (bits 4i..4i+3) holding
 * element (0, 2, 4, 6, 1, 3, 5, 7)[i] of the eight. All pointers are device
 * pointers, 16-byte aligned; asynchronous on `stream`. */
int clover_quantize_q4(const uint16_t* w, int32_t n_mats, int32_t rows, int32_t cols, uint8_t* q,
                       uint16_t* s, clover_stream_t stream);

/* Bytes of workspace clover_lmhead_unmask needs. Host-only. */
size_t clover_head_workspace_bytes(const clover_dims* dims, int32_t max_tokens);

/* Output head, statistics and the low-confidence unmask rule on M positions
 * (Files, "What Clover is": untied head read in full; "How it writes", steps
 * 2-3).
 *   z_p,v = alpha_p * (bf16(RMSNorm(x_p)) . W_h[v]),  z_p,mask_id = -inf
 *   argmax_p = lowest v with the largest z, max_logit_p = max z,
 *   lse_p = log sum_v exp(z_p,v), max_prob_p = exp(max_logit_p - lse_p)
 * The full logits are never written. Then, for each group of `block`
 * consecutive positions: every position with masked_p != 0 and
 * max_prob_p > threshold is committed; if none is, the masked position with
 * the largest max_prob (lowest index on ties) is committed. Committing sets
 * tokens_p = argmax_p and masked_p = 0.
 * head_w: bf16 [V][H]. x: fp32 [M][H] (pre-norm). logit_scale: fp32 [M] or
 * NULL (= 1). tokens int32 [M], masked uint8 [M]: in/out. argmax int32 [M],
 * max_logit, lse, max_prob fp32 [M]: out. n_committed: device int32 scalar,
 * out (number committed by this call). M % block == 0 is not required; the
 * last group may be shorter. Above 256 positions, block must be at most 256
 * (the head then runs on whole blocks, at most 256 positions at a time). A committed slot (masked_p == 0) whose token id
 * lies outside [0, V) is left as it is and reported through the workspace
 * status word (clover_workspace_status). */
int clover_lmhead_unmask(const clover_dims* dims, const uint16_t* head_w, const float* x,
                         const float* logit_scale, float threshold, int32_t block,
                         int32_t* tokens, uint8_t* masked,
                         int32_t* argmax, float* max_logit, float* lse, float* max_prob,
                         int32_t* n_committed, int32_t M,
                         void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Accept rules of clover_lmhead_accept. */
#define CLOVER_ACCEPT_EXACT 0
#define CLOVER_ACCEPT_THRESHOLD 1

/* Bytes of workspace clover_lmhead_accept needs for up to max_rows rows.
 * Host-only. */
size_t clover_accept_workspace_bytes(const clover_dims* dims, int32_t max_rows);

/* Output head of a verify pass fused with the self-speculative accept test
 * (Files, "Two ways to run it": a round keeps the longest prefix of drafts
 * the causal pass accepts, plus one token at the boundary; the exact rule
 * keeps a draft only if it is the causal pass's argmax, the threshold rule
 * if its probability is at least min(ratio, delta e^-H), H the entropy of the
 * causal distribution, defaults ratio 0.9 and delta 0.6).
 * The M rows form M / block blocks; in each, row j < block - 1 is the
 * distribution draft[j] is tested against and the last row gives the token
 * after the final draft. Per row, as clover_lmhead_unmask (mask token at
 * -inf): argmax, max_logit, lse, max_prob, plus
 *   entropy_p = -sum_v p_v ln p_v  (p = softmax of z_p),
 *   p_draft_p = p at draft[p]      (0 for the mask token or an id outside
 *                                   [0, V); the last row of a block: ignored)
 * Per block b: accept_len[b] = r, the number of leading rows whose draft is
 * accepted (exact: draft == argmax; threshold: p_draft >= min(ratio,
 * delta e^-entropy), fp32), and out_tokens[b*block + j] = draft for j < r,
 * argmax of row r at j = r, -1 after (r + 1 tokens).
 * head_w: bf16 [V][H]. x: fp32 [M][H] (pre-norm). logit_scale: fp32 [M] or
 * NULL. draft: int32 [M], in. rule: CLOVER_ACCEPT_EXACT or
 * CLOVER_ACCEPT_THRESHOLD (then 0 < ratio <= 1 and a finite delta > 0).
 * argmax, max_logit, lse, max_prob, entropy, p_draft: [M] out, each may be
 * NULL. accept_len int32 [M / block], out_tokens int32 [M]: out. Requires
 * block >= 2 and M % block == 0. */
int clover_lmhead_accept(const clover_dims* dims, const uint16_t* head_w, const float* x,
                         const float* logit_scale, const int32_t* draft, int32_t rule, float ratio,
                         float delta, int32_t block,
                         int32_t* argmax, float* max_logit, float* lse, float* max_prob,
                         float* entropy, float* p_draft, int32_t* accept_len, int32_t* out_tokens,
                         int32_t M, void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Bytes of workspace the denoise entry points need. Host-only. */
size_t clover_denoise_workspace_bytes(const clover_dims* dims, int32_t max_tokens);

/* Byte offset, within a denoise workspace sized for max_tokens, of the
 * residual stream that the last clover_denoise_step left there: fp32 [M][H],
 * the output of the last MoE sublayer (the input of the final RMSNorm and
 * the head). Host-only. Returns 0 for invalid dims or max_tokens (the offset
 * itself is never 0). */
size_t clover_denoise_hidden_offset(const clover_dims* dims, int32_t max_tokens);

/* One block-diffusion denoising step over M positions (Files, "How it
 * writes", steps 1-3): x_p = E[tokens_p] + ctx_p (the mask token's embedding
 * while masked), n_layers MoE sublayers as in clover_moe_block_step, a final
 * RMSNorm, then clover_lmhead_unmask's statistics and unmask rule.
 * layers: HOST array of n_layers structs (the pointers inside are device
 * pointers). embed: bf16 [V][H]. ctx: fp32 [M][H], fixed per block.
 * head_w: bf16 [V][H]. logit_scale: fp32 [M] or NULL. tokens, masked: in/out.
 * The positions form M / block independent blocks (M % block == 0). */
int clover_denoise_step(const clover_dims* dims, const clover_moe_layer* layers, int32_t n_layers,
                        const uint16_t* embed, const float* ctx, const uint16_t* head_w,
                        const float* logit_scale, float threshold, int32_t block,
                        int32_t* tokens, uint8_t* masked, int32_t M,
                        void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Repeats clover_denoise_step until no position is masked or max_steps steps
 * ran (Files, "How it writes", step 4). Synchronises `stream` once per step to
 * read the number of masked positions left. *steps_taken (host) receives the
 * number of steps. Returns CLOVER_ERR_NOT_CONVERGED if positions are still
 * masked after max_steps steps. */
int clover_denoise_block(const clover_dims* dims, const clover_moe_layer* layers, int32_t n_layers,
                         const uint16_t* embed, const float* ctx, const uint16_t* head_w,
                         const float* logit_scale, float threshold, int32_t block,
                         int32_t* tokens, uint8_t* masked, int32_t M, int32_t max_steps,
                         int32_t* steps_taken,
                         void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Synchronises `stream`, then reads and clears the device status word of a
 * workspace used by any call above. Returns CLOVER_OK, or
 * CLOVER_ERR_DEVICE_TIMEOUT if a kernel gave up on a wait (the message names
 * which), or CLOVER_ERR_CUDA. */
int clover_workspace_status(void* workspace, size_t workspace_bytes, clover_stream_t stream);

/* Timing hook: when `begin`/`end` are non-NULL, every later launch of the
 * expert kernel (one per MoE sublayer) records begin[i % capacity] before and
 * end[i % capacity] after launch i on the launching stream; i restarts at 0
 * at each call of this function. Pass NULL to stop. Process-wide, not
 * thread-safe. Returns the number of launches recorded since the last call. */
int32_t clover_profile_expert_events(clover_event_t* begin, clover_event_t* end, int32_t capacity);

/* Copies the last error message of the calling thread into buf (at most n
 * bytes, NUL-terminated). Returns its full length. */
int32_t clover_last_error(char* buf, size_t n);

/* Same operation and arguments as clover_lmhead_unmask, without the
 * workspace. (The pages have no counterpart: this is a library convenience.)
 * For callers that cannot allocate device memory -- a plug-in inside an
 * application that owns all GPU memory and hands out no allocator, or a
 * latency-critical loop that must not synchronise on an allocation. The
 * scratch lives in a 1 MiB array inside the library that
 * every GPU loading the library keeps until the process exits; it fits up to
 * 102 positions at hidden 2048 (the rule: clover_head_workspace_bytes(dims, M)
 * <= 1 MiB). Larger sizes return CLOVER_ERR_WORKSPACE_TOO_SMALL and nothing
 * runs. Every call looks up the array's device address in the current
 * context; the first call on a device also loads the library's kernels
 * there, so make that first call before any stream capture. The call
 * allocates nothing. It checks every argument before it enqueues anything,
 * then clears the array's control words on the stream, so the status of a
 * call must be read (clover_lmhead_unmask_static_status) before the next
 * call. All calls share the one array: calls that may overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller. */
int clover_lmhead_unmask_static(const clover_dims* dims, const uint16_t* head_w, const float* x,
                                const float* logit_scale, float threshold, int32_t block,
                                int32_t* tokens, uint8_t* masked,
                                int32_t* argmax, float* max_logit, float* lse, float* max_prob,
                                int32_t* n_committed, int32_t M, clover_stream_t stream);

/* The device status of the last clover_lmhead_unmask_static call, which has
 * no workspace to pass to clover_workspace_status: synchronises `stream`,
 * reads the status word of the library's static scratch array, and if it is
 * set clears the array's control words and returns
 * CLOVER_ERR_DEVICE_TIMEOUT (a wait that gave up, or a committed slot whose
 * token id lies outside [0, V); the message names which); else CLOVER_OK.
 * (The pages have no counterpart.) */
int clover_lmhead_unmask_static_status(clover_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int32_t clover_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CLOVER_H_ */
