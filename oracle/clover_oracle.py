"""CPU oracle for the block-diffusion MoE denoising step.

TEST INFRASTRUCTURE. Only the test suite, the smoke check in
__graft_entry__.py and the CPU-baseline leg of bench.py may import this
module. The product path (the CUDA library and its Python binding) never
calls it and shares no code with it.

What it follows (page titles and sections; "Files" is "Clover-35B-A3B: how a
diffusion model gets to 680 tokens a second, read from its files"):

* Files, "What Clover is": every layer has 256 routed experts, each token is
  routed to 8 of them, one shared expert is always on; hidden 2,048,
  vocabulary 248,320; block_size 32, mask_token_id 151669, a low-confidence
  denoiser with threshold 0.95. One expert is gate and up at 2,048 x 512 and
  down at 512 x 2,048. The output head is untied from the embedding and read
  in full at every step.
* Files, "The expert selection": the router yields per-token top-8 routing
  probabilities.
* Files, "How it writes", steps 1-4: fill the block with the mask token, run
  the model, take every slot's most likely token and its probability with the
  mask token's logit set to minus infinity, commit every still-masked slot
  whose probability is above the threshold, and if none clears it commit the
  single most confident one; repeat until no slot is masked.
* "Deep Dive - Clover 35B: a diffusion LLM at Qwen parity, 680 tok/s",
  "What DiffuSpace actually shipped": block of 32 masked positions resolved
  by a 0.95 confidence threshold.

Readings where the pages are silent:

* Top-k routing is softmax over all routed experts, then the top-k
  probabilities renormalised to sum to one. Ties go to the lower expert id.
* The shared expert is ungated (weight 1). The routed experts and the shared
  expert are SwiGLU: h = silu(x W_g^T) * (x W_u^T), out = h W_d^T, with
  silu(z) = z / (1 + e^-z).
* The layers outside this path (attention, recurrent) are left out. Each MoE
  sublayer is pre-norm residual, x <- x + MoE(RMSNorm(x)), with a unit-weight
  RMSNorm (eps 1e-6); a final RMSNorm precedes the head.
* Input assembly: x_p = E[t_p] + c_p, with c_p a fixed per-position context
  term standing in for the omitted layers.
* The model is BF16: every matrix product takes bf16 operands (the stored
  weights, and the activation rounded to bf16 where it enters a product:
  the normed input of the router, the experts and the head, and the SwiGLU
  output entering the down projection). Products accumulate exactly here
  (float64); everything else (residual stream, norms, softmax, log-sum-exp)
  is float64.
* Integer decisions are taken on float32 values, as the kernels take them:
  top-k on the float32-rounded router logits, argmax on the float32-rounded
  head logits, the threshold test on the float32-rounded probability.
* Coreset selection (optional): the mass of an expert is the sum of the
  softmax probabilities (not renormalised) of the slots that select it; the
  kept set is the shortest prefix of experts sorted by mass (descending, ties
  to the lower id) whose cumulative mass reaches top_p x total and that holds
  at least k experts (the page says at least the top expert; k keeps every
  token's k-way routing defined).
* "Above 0.95" is a strict comparison. Fallback ties go to the lowest
  position, argmax ties to the lowest vocabulary id. The fallback considers
  only still-masked slots. Each block of `block` positions applies the rule
  on its own.
* Self-speculative accept test (Files, "Two ways to run it"): a verify pass
  over B drafts gives B + 1 rows, row j being the distribution against which
  draft j is tested and row B the one after the last draft. Exact keeps a
  draft that equals its row's argmax; threshold keeps it when its probability
  is at least min(ratio, delta e^-H), H the entropy of the row (the page's
  printed formula is lost; this is the form its text describes: defaults 0.9
  and 0.6, "the ratio never binds", 0.6 when certain and 0.22 at one nat).
  The round keeps the longest accepted prefix of r drafts plus the boundary
  token, taken greedily as the argmax of row r. The mask token has
  probability zero, so it is never accepted; a draft id outside the
  vocabulary is never accepted either.

* Low-bit expert weights (the pages name INT4 for one deployment but give
  no format, so this format is this implementation's own): each
  expert matrix [R][K] keeps one bf16 scale per row and group of 64
  consecutive K elements, s = bf16(float32(max |w|) / 7) (fp32 IEEE division,
  then round to nearest even), and per element the 4-bit code
  u = clamp(rint(float32(w) / float32(s)), -8, 7) + 8 (u = 8 where s = 0).
  The weight the product uses is bf16((u - 8) s). Codes are packed eight to a
  32-bit little-endian word in the nibble order e0 e2 e4 e6 e1 e3 e5 e7
  (nibble i at bits 4i); scales are stored group-major, [K/64][R].

All float arithmetic is numpy float64 unless stated; bf16 tensors arrive as
uint16 arrays holding their bit patterns.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bf16 helpers


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    The value is first rounded to float32 (ties to even), then the float32
    bit pattern is rounded to its upper 16 bits (ties to even)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# building blocks


def rms_norm(x, eps: float) -> np.ndarray:
    """Unit-weight RMSNorm over the last axis: x / sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def softmax(r) -> np.ndarray:
    r = np.asarray(r, dtype=np.float64)
    m = np.max(r, axis=-1, keepdims=True)
    e = np.exp(r - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def route(xb, router_w_bits, top_k: int, router_bias=None):
    """Router, softmax and top-k with renormalisation (Files, "What Clover is"
    and "The expert selection").

    xb: bf16-valued float64 [M][H]. Returns (logits float64 [M][E],
    p float64 [M][E], idx int32 [M][K] in selection order, w float64 [M][K])."""
    wr = bf16_to_f64(router_w_bits)
    logits = xb @ wr.T
    if router_bias is not None:
        logits = logits + np.asarray(router_bias, dtype=np.float64)[None, :]
    p = softmax(logits)
    r32 = logits.astype(np.float32)
    M, E = logits.shape
    idx = np.empty((M, top_k), dtype=np.int32)
    for t in range(M):
        # descending float32 logit, then ascending expert id
        order = np.lexsort((np.arange(E), -r32[t].astype(np.float64)))
        idx[t] = order[:top_k]
    psel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    w = psel / np.sum(psel, axis=1, keepdims=True)
    return logits, p, idx, w


def coreset(p, idx, top_p: float) -> np.ndarray:
    """Block coreset expert selection (Files, "The expert selection"): add up
    each token's top-k routing probabilities per expert, sort the experts by
    that total (ties to the lower id), keep the smallest prefix whose share of
    the total reaches top_p, and always at least the top expert -- read here
    as at least k experts, so that every token can still select k. Returns
    the kept expert ids in that order.

    p: float64 [M][E] softmax probabilities; idx: [M][K] each token's top-k."""
    p = np.asarray(p, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    E = p.shape[1]
    mass = np.zeros(E)
    for t in range(idx.shape[0]):
        for e in idx[t]:
            mass[e] += p[t, e]
    order = sorted(range(E), key=lambda e: (-mass[e], e))
    total = float(np.sum(mass))
    k = idx.shape[1]
    kept, acc = [], 0.0
    for e in order:
        kept.append(e)
        acc += mass[e]
        if acc >= top_p * total and len(kept) >= k:
            break
    return np.asarray(kept, dtype=np.int32)


def route_within(logits, allowed, top_k: int):
    """Top-k restricted to the allowed experts (descending float32 logit, lower
    id on ties); weights = softmax over the selected logits. A token selects
    min(top_k, len(allowed)) experts."""
    logits = np.asarray(logits, dtype=np.float64)
    M, E = logits.shape
    mask = np.zeros(E, dtype=bool)
    mask[np.asarray(allowed, dtype=np.int64)] = True
    k = min(top_k, int(mask.sum()))
    r32 = logits.astype(np.float32).astype(np.float64)
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k))
    for t in range(M):
        cand = [e for e in range(E) if mask[e]]
        cand.sort(key=lambda e: (-r32[t, e], e))
        sel = cand[:k]
        idx[t] = sel
        z = logits[t, sel]
        ez = np.exp(z - np.max(z))
        w[t] = ez / np.sum(ez)
    return idx, w


def swiglu_expert(xb, gate_up_bits, down_bits) -> np.ndarray:
    """One SwiGLU expert on bf16 inputs xb [m][H].

    gate_up_bits: [2F][H] (rows 0..F-1 gate, F..2F-1 up); down_bits: [H][F].
    The SwiGLU output is rounded to bf16 before the down projection."""
    gu = bf16_to_f64(gate_up_bits)
    F = gu.shape[0] // 2
    g = xb @ gu[:F].T
    u = xb @ gu[F:].T
    h = round_to_bf16(silu(g) * u)
    return h @ bf16_to_f64(down_bits).T


def moe_layer(x, layer: dict, top_k: int, eps: float, force_idx=None, coreset_top_p=None,
              block: int | None = None) -> dict:
    """One pre-norm MoE sublayer: x_out = x + sum_k w_k E_{i_k}(xb) + S(xb).

    layer: dict with router_w, gate_up, down, sh_gate_up, sh_down (uint16 bit
    arrays; gate_up and down may be any object indexable by expert id) and
    optional router_bias (float32 [E]).
    force_idx: optional [M][K] expert ids to use instead of the oracle's own
    selection (teacher forcing); the weights are then the oracle's
    renormalised probabilities of those experts."""
    x = np.asarray(x, dtype=np.float64)
    xb = round_to_bf16(rms_norm(x, eps))
    logits, p, idx, w = route(xb, layer["router_w"], top_k, layer.get("router_bias"))
    kept = []
    if coreset_top_p is not None:
        # Files, "The expert selection": the block's coreset, then every token
        # routes within it (denoising passes only).
        M = x.shape[0]
        blk = block or M
        new_idx = np.empty_like(idx)
        new_w = np.empty_like(w)
        for b0 in range(0, M, blk):
            sl = slice(b0, min(M, b0 + blk))
            keep = coreset(p[sl], idx[sl], coreset_top_p)
            kept.append(keep)
            new_idx[sl], new_w[sl] = route_within(logits[sl], keep, top_k)
        idx, w = new_idx, new_w
    if force_idx is not None:
        idx = np.asarray(force_idx, dtype=np.int32)
        psel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        w = psel / np.sum(psel, axis=1, keepdims=True)
    y = np.zeros_like(x)
    for e in np.unique(idx):
        toks, ks = np.nonzero(idx == e)
        o = swiglu_expert(xb[toks], layer["gate_up"][int(e)], layer["down"][int(e)])
        y[toks] += w[toks, ks][:, None] * o
    y += swiglu_expert(xb, layer["sh_gate_up"], layer["sh_down"])
    return {"x_out": x + y, "idx": idx, "w": w, "logits": logits, "p": p, "xb": xb, "coreset": kept}


def head_logits(x, head_bits, eps: float, alpha=None, chunk: int = 16384) -> np.ndarray:
    """z = alpha_p * (bf16(RMSNorm(x)) W_h^T), float64 [M][V]."""
    xb = round_to_bf16(rms_norm(x, eps))
    V = head_bits.shape[0]
    z = np.empty((xb.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, chunk):
        z[:, v0:v0 + chunk] = xb @ bf16_to_f64(head_bits[v0:v0 + chunk]).T
    if alpha is not None:
        z *= np.asarray(alpha, dtype=np.float64)[:, None]
    return z


def head_stats(z, mask_id: int) -> dict:
    """Per-position argmax, max logit, log-sum-exp and max probability with the
    mask token excluded (Files, "How it writes", step 2)."""
    z = np.array(z, dtype=np.float64, copy=True)
    z[:, mask_id] = -np.inf
    m = np.max(z, axis=1)
    lse = m + np.log(np.sum(np.exp(z - m[:, None]), axis=1))
    pmax = np.exp(m - lse)
    z32 = z.astype(np.float32)
    argmax = np.argmax(z32, axis=1).astype(np.int32)   # first (lowest) id on ties
    return {"argmax": argmax, "max_logit": m, "lse": lse, "max_prob": pmax}


def unmask(tokens, masked, argmax, max_prob, threshold: float, block: int):
    """Low-confidence unmask rule (Files, "How it writes", step 3), applied to
    each block of `block` consecutive positions. Returns new (tokens, masked,
    committed bool mask)."""
    tokens = np.array(tokens, dtype=np.int32, copy=True)
    masked = np.array(masked, dtype=np.uint8, copy=True)
    p32 = np.asarray(max_prob, dtype=np.float64).astype(np.float32)
    tau = np.float32(threshold)
    n = tokens.shape[0]
    commit = np.zeros(n, dtype=bool)
    for b0 in range(0, n, block):
        sl = range(b0, min(n, b0 + block))
        still = [p for p in sl if masked[p]]
        chosen = [p for p in still if p32[p] > tau]
        if not chosen and still:
            best = still[0]
            for p in still[1:]:
                if p32[p] > p32[best]:
                    best = p
            chosen = [best]
        for p in chosen:
            commit[p] = True
    tokens[commit] = np.asarray(argmax, dtype=np.int32)[commit]
    masked[commit] = 0
    return tokens, masked, commit


ACCEPT_EXACT = 0
ACCEPT_THRESHOLD = 1


def verify_stats(z, mask_id: int, draft) -> dict:
    """head_stats plus, per row, the entropy H = -sum_v p_v ln p_v of the
    softmax with the mask token excluded and the probability of the row's
    draft token (Files, "Two ways to run it"). A draft outside [0, V) has
    probability 0."""
    st = head_stats(z, mask_id)
    z = np.array(z, dtype=np.float64, copy=True)
    z[:, mask_id] = -np.inf
    logp = z - st["lse"][:, None]
    p = np.exp(logp)
    ent = np.empty(z.shape[0])
    pd = np.zeros(z.shape[0])
    draft = np.asarray(draft, dtype=np.int64)
    for n in range(z.shape[0]):
        live = p[n] > 0
        ent[n] = -np.sum(p[n, live] * logp[n, live])
        if 0 <= draft[n] < z.shape[1]:
            pd[n] = p[n, draft[n]]
    st["entropy"] = ent
    st["p_draft"] = pd
    return st


def accept_threshold(entropy, ratio: float, delta: float) -> np.ndarray:
    """Probability a draft needs under the threshold rule: min(ratio,
    delta * e^-H), float64."""
    return np.minimum(ratio, delta * np.exp(-np.asarray(entropy, dtype=np.float64)))


def accept(draft, argmax, p_draft, entropy, rule: int, ratio: float, delta: float, block: int) -> dict:
    """The accept test over blocks of `block` rows (block - 1 drafts + the
    boundary row). Per row j < block - 1 the decision is taken in float32:
    exact, draft_j == argmax_j; threshold, float32(p_draft_j) >=
    float32(min(ratio, delta e^-H_j)). r = the number of leading accepted
    drafts; the round's tokens are drafts 0..r-1 then argmax of row r, the
    remaining entries -1."""
    draft = np.asarray(draft, dtype=np.int64)
    argmax = np.asarray(argmax, dtype=np.int64)
    n = draft.shape[0]
    assert block >= 2 and n % block == 0
    p32 = np.asarray(p_draft, dtype=np.float64).astype(np.float32)
    t32 = accept_threshold(entropy, ratio, delta).astype(np.float32)
    ok = np.zeros(n, dtype=bool)
    acc_len = np.zeros(n // block, dtype=np.int32)
    out = np.full(n, -1, dtype=np.int32)
    for b in range(n // block):
        r = 0
        for j in range(block - 1):
            i = b * block + j
            if rule == ACCEPT_EXACT:
                ok[i] = draft[i] == argmax[i]
            else:
                ok[i] = bool(p32[i] >= t32[i])
        while r < block - 1 and ok[b * block + r]:
            r += 1
        acc_len[b] = r
        out[b * block:b * block + r] = draft[b * block:b * block + r]
        out[b * block + r] = argmax[b * block + r]
    return {"accepted": ok, "accept_len": acc_len, "tokens": out}


Q4_GROUP = 64
_Q4_NIBBLE_OF = np.array([0, 2, 4, 6, 1, 3, 5, 7])   # element held by nibble i of a word


def quantize_q4(w_bits):
    """bf16 matrix [R][K] (K % 64 == 0) -> (packed codes uint8 [R][K/2],
    scale bits uint16 [K/64][R]) in the low-bit format above."""
    w = bf16_to_f64(w_bits).astype(np.float32)
    R, K = w.shape
    g = w.reshape(R, K // Q4_GROUP, Q4_GROUP)
    amax = np.abs(g).max(axis=2)                                   # exact
    s32 = (amax / np.float32(7.0)).astype(np.float32)              # fp32 IEEE division
    s_bits = bf16_bits_of(s32)
    s = bf16_to_f64(s_bits).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / s[:, :, None]).astype(np.float32)          # fp32 division, half to even
    q = np.where(s[:, :, None] > 0, q, 0.0)
    u = (np.clip(q, -8, 7) + 8).astype(np.uint32).reshape(R, K // 8, 8)
    words = np.zeros((R, K // 8), dtype=np.uint32)
    for i in range(8):
        words |= u[:, :, _Q4_NIBBLE_OF[i]] << np.uint32(4 * i)
    packed = words.astype("<u4").view(np.uint8).reshape(R, K // 2)
    return packed, np.ascontiguousarray(s_bits.T)


def dequantize_q4(packed, scale_bits) -> np.ndarray:
    """Packed codes [R][K/2] + scale bits [K/64][R] -> the bf16 bit patterns
    [R][K] of bf16((u - 8) s)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    R = packed.shape[0]
    K = packed.shape[1] * 2
    words = packed.view("<u4").reshape(R, K // 8)
    u = np.empty((R, K // 8, 8), dtype=np.int64)
    for i in range(8):
        u[:, :, _Q4_NIBBLE_OF[i]] = (words >> np.uint32(4 * i)) & 0xF
    s = bf16_to_f64(np.asarray(scale_bits).T)                      # [R][K/64]
    w = (u.reshape(R, K) - 8) * np.repeat(s, Q4_GROUP, axis=1)     # exact in float64
    return bf16_bits_of(w)


def bf16_bits_of(x) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even)."""
    y = np.ascontiguousarray(round_to_bf16(np.asarray(x, dtype=np.float64)), dtype=np.float32)
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def embed(tokens, embed_bits, ctx) -> np.ndarray:
    """Input assembly x_p = E[t_p] + c_p (mask-token embedding while masked)."""
    e = bf16_to_f64(np.asarray(embed_bits)[np.asarray(tokens, dtype=np.int64)])
    return e + np.asarray(ctx, dtype=np.float64)


def denoise_step(tokens, masked, model: dict, threshold: float, block: int,
                 alpha=None) -> dict:
    """One block-diffusion denoising step: assemble the block, run every MoE
    sublayer, the head statistics and the unmask rule."""
    d = model["dims"]
    x = embed(tokens, model["embed"], model["ctx"])
    routes = []
    for layer in model["layers"]:
        out = moe_layer(x, layer, d["top_k"], d["rms_eps"])
        routes.append(out["idx"])
        x = out["x_out"]
    z = head_logits(x, model["head"], d["rms_eps"], alpha)
    st = head_stats(z, d["mask_id"])
    nt, nm, commit = unmask(tokens, masked, st["argmax"], st["max_prob"], threshold, block)
    return {"tokens": nt, "masked": nm, "committed": commit, "x": x, "routes": routes, **st}


def denoise_block(tokens, masked, model: dict, threshold: float, block: int,
                  max_steps: int, alpha=None) -> dict:
    """Repeat denoise_step until no slot is masked or max_steps steps ran
    (Files, "How it writes", step 4)."""
    tokens = np.array(tokens, dtype=np.int32, copy=True)
    masked = np.array(masked, dtype=np.uint8, copy=True)
    history = []
    steps = 0
    while steps < max_steps and masked.any():
        st = denoise_step(tokens, masked, model, threshold, block, alpha)
        tokens, masked = st["tokens"], st["masked"]
        history.append(st)
        steps += 1
    return {"tokens": tokens, "masked": masked, "steps": steps, "history": history}


# ---------------------------------------------------------------------------
# dense brute force used to pin the sparse path


def moe_layer_dense(x, layer: dict, top_k: int, eps: float) -> np.ndarray:
    """Every expert evaluated on every token, then combined through a dense
    [M][E] gate matrix built from a full stable sort of the logits."""
    x = np.asarray(x, dtype=np.float64)
    xb = round_to_bf16(rms_norm(x, eps))
    wr = bf16_to_f64(layer["router_w"])
    logits = xb @ wr.T
    if layer.get("router_bias") is not None:
        logits = logits + np.asarray(layer["router_bias"], dtype=np.float64)[None, :]
    p = softmax(logits)
    M, E = p.shape
    G = np.zeros((M, E))
    r32 = logits.astype(np.float32).astype(np.float64)
    for t in range(M):
        ranked = sorted(range(E), key=lambda e: (-r32[t, e], e))
        keep = ranked[:top_k]
        tot = sum(p[t, e] for e in keep)
        for e in keep:
            G[t, e] = p[t, e] / tot
    y = np.zeros_like(x)
    for e in range(E):
        o = swiglu_expert(xb, layer["gate_up"][e], layer["down"][e])
        y += G[:, e:e + 1] * o
    y += swiglu_expert(xb, layer["sh_gate_up"], layer["sh_down"])
    return x + y
