"""GPU vs oracle at Clover-35B-A3B shapes (hidden 2,048, 256 experts top-8 +
shared, SwiGLU 2048->512->2048, vocabulary 248,320, blocks of 32), in the
launch configuration the benchmark uses:

* one MoE layer on a 32-position block (all outputs against the oracle), and
  on 1, 33 and 100 tokens (both routing paths, ragged tiles);
* head + unmask on 32 positions with logit scales calibrated so ~40% of the
  positions clear 0.95;
* head + unmask on 256 positions (8 blocks of 32; the widest token tile);
* the full 40-layer denoising step: the fused entry point equals the
  layer-by-layer composition bit for bit (hidden state and decisions), every
  one of the 40 layers matches the oracle under teacher forcing, and the
  block-level invariants hold over a whole block (never re-masks, progresses
  every step, every slot ends with the token it predicted while masked,
  commits in descending confidence), both step by step and through the
  clover_denoise_block loop itself;
* 8 blocks x 32 positions with Zipf(1.2)-biased routing, all 40 layers
  teacher-forced against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import (bits, calibrate_alpha, compare_head, compare_routing, decisions_clear, hidden_close,
                           layer_to_oracle)

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = synth.CLOVER


@pytest.fixture(scope="module")
def model():
    torch.cuda.synchronize()
    layers = [synth.make_layer(D, 0, l, DEV) for l in range(D.n_layers)]
    embed = synth.make_embed(D, 0, DEV)
    head = synth.make_head(D, 0, DEV)
    torch.cuda.synchronize()
    return {"layers": layers, "embed": embed, "head": head}


def _check_layer(layer, x, M):
    x_out, idx, w = clover.moe_block_step(D, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer, lazy=True)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, D.top_k, D.rms_eps)
    ties = compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, D.top_k)
    forced = O.moe_layer(xh, L, D.top_k, D.rms_eps, force_idx=idx.cpu().numpy())
    g = x_out.cpu().numpy()
    ok, worst = hidden_close(g, forced["x_out"])
    assert ok, worst
    ok, worst = hidden_close(g - xh, forced["x_out"] - xh)
    assert ok, worst
    return idx.cpu().numpy(), ties


def test_one_layer_block_of_32(model):
    x = synth.make_x(D, 32, 1, DEV)
    idx, ties = _check_layer(model["layers"][0], x, 32)
    assert ties <= 2
    u = len(np.unique(idx))
    assert 140 <= u <= 185          # ~163 experts touched under uniform routing


@pytest.mark.parametrize("M", [1, 33, 100])
def test_one_layer_ragged_token_counts(model, M):
    """One token (the fused kernel's smallest block), 33 (the first count that
    takes the standalone routing and expert kernels) and 100 (a ragged tile of
    the standalone path) at full Clover size."""
    x = synth.make_x(D, M, 40 + M, DEV)
    idx, ties = _check_layer(model["layers"][2], x, M)
    assert ties <= max(1, M // 16)


def test_one_layer_256_tokens_zipf(model):
    base = model["layers"][1]
    layer = synth.Layer(base.router_w, base.gate_up, base.down, base.sh_gate_up, base.sh_down,
                        synth.zipf_router_bias(D, 0, 1, 1.2, DEV))
    x = synth.make_x(D, 256, 2, DEV)
    idx, ties = _check_layer(layer, x, 256)
    counts = np.bincount(idx.ravel(), minlength=D.n_experts)
    assert counts.max() >= 100        # the hot experts carry ~half the block


def test_head_unmask_32_positions(model):
    M = 32
    x = synth.make_x(D, M, 3, DEV)
    xh = x.cpu().numpy()
    hb = bits(model["head"])
    z_raw = O.head_logits(xh, hb, D.rms_eps)
    alpha = calibrate_alpha(z_raw, D.mask_id, synth.confidence_targets(M, 4).numpy(), O)
    tokens, masked = synth.masked_block(D, M, DEV)
    t0, m0 = tokens.cpu().numpy(), masked.cpu().numpy()
    out = clover.lmhead_unmask(D, model["head"], x, tokens, masked, logit_scale=torch.from_numpy(alpha).to(DEV),
                               threshold=0.95, block=32)
    torch.cuda.synchronize()
    z = z_raw * alpha.astype(np.float64)[:, None]
    ref = O.head_stats(z, D.mask_id)
    z[:, D.mask_id] = -np.inf
    ref["z"] = z
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_head(got, ref)
    frac = float(np.mean(ref["max_prob"] >= 0.95))
    assert 0.2 <= frac <= 0.6
    assert decisions_clear(ref["max_prob"], m0, 0.95, 32)
    rt, rm, rc = O.unmask(t0, m0, ref["argmax"], ref["max_prob"], 0.95, 32)
    assert np.array_equal(tokens.cpu().numpy(), rt)
    assert np.array_equal(masked.cpu().numpy(), rm)


def test_head_unmask_256_positions(model):
    """Eight blocks of 32 in one head call: the 256-column token tile, with
    logit scales calibrated so that about 40% of the positions clear 0.95
    (the unmask rule then runs per block of 32)."""
    M = 256
    x = synth.make_x(D, M, 8, DEV)
    xh = x.cpu().numpy()
    hb = bits(model["head"])
    z_raw = O.head_logits(xh, hb, D.rms_eps)
    alpha = calibrate_alpha(z_raw, D.mask_id, synth.confidence_targets(M, 9).numpy(), O, iters=40)
    tokens, masked = synth.masked_block(D, M, DEV)
    masked[5::7] = 0                       # some slots committed earlier
    tokens[5::7] = 11
    t0, m0 = tokens.cpu().numpy(), masked.cpu().numpy()
    out = clover.lmhead_unmask(D, model["head"], x, tokens, masked, logit_scale=torch.from_numpy(alpha).to(DEV),
                               threshold=0.95, block=32)
    torch.cuda.synchronize()
    z = z_raw * alpha.astype(np.float64)[:, None]
    ref = O.head_stats(z, D.mask_id)
    z[:, D.mask_id] = -np.inf
    ref["z"] = z
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_head(got, ref)
    assert decisions_clear(ref["max_prob"], m0, 0.95, 32)
    rt, rm, rc = O.unmask(t0, m0, ref["argmax"], ref["max_prob"], 0.95, 32)
    assert np.array_equal(tokens.cpu().numpy(), rt)
    assert np.array_equal(masked.cpu().numpy(), rm)
    assert int(out["n_committed"][0]) == int(np.sum(rc))


def _teacher_forced(layers, xs, idxs, xf, ties_allowed):
    """Every layer l: the oracle on the GPU's own input x_l and (where the
    routing is a near-tie) the GPU's selection, against the GPU's output
    x_(l+1). Returns the number of tokens whose routing was a near-tie."""
    ties = 0
    for l, layer in enumerate(layers):
        L = layer_to_oracle(layer, lazy=True)
        xh = xs[l].cpu().numpy()
        ig = idxs[l].cpu().numpy()
        free = O.moe_layer(xh, L, D.top_k, D.rms_eps)
        ref = O.moe_layer(xh, L, D.top_k, D.rms_eps, force_idx=ig)
        ties += compare_routing(ig, ref["w"], free, D.top_k)
        g = (xs[l + 1] if l + 1 < len(xs) else xf).cpu().numpy()
        ok, worst = hidden_close(g - xh, ref["x_out"] - xh)
        assert ok, (l, worst)
        ok, worst = hidden_close(g, ref["x_out"])
        assert ok, (l, worst)
    assert ties <= ties_allowed, ties
    return ties


def _compose_step(model, layers, ctx, tokens, masked, alpha=None, block=32):
    """The denoising step as separate entry-point calls; returns the inputs of
    every layer and its routing."""
    emb = model["embed"]
    x = emb[tokens.long()].float() + ctx
    xs, idxs = [], []
    for layer in layers:
        xs.append(x)
        x, idx, _ = clover.moe_block_step(D, layer, x)
        idxs.append(idx)
    out = clover.lmhead_unmask(D, model["head"], x, tokens, masked, logit_scale=alpha, block=block)
    return xs, idxs, x, out


def test_full_step_composition_and_every_layer(model):
    M = 32
    ctx = synth.make_ctx(D, M, 5, DEV)
    cmodel = clover.Model(D, model["layers"], model["embed"], model["head"])
    t1, m1 = synth.masked_block(D, M, DEV)
    ws = clover.denoise_step(cmodel, ctx, t1, m1, block=32)
    t2, m2 = synth.masked_block(D, M, DEV)
    xs, idxs, xf, out = _compose_step(model, model["layers"], ctx, t2, m2)
    torch.cuda.synchronize()
    assert torch.equal(t1, t2) and torch.equal(m1, m2)
    assert int(m1.sum()) == M - 1
    # the step's own residual stream (each layer's combine deferred into the
    # next launch) equals the composition's, bit for bit
    assert torch.equal(clover.denoise_hidden(D, ws, M), xf)
    # every layer against the oracle under teacher forcing (40 x 32 tokens)
    _teacher_forced(model["layers"], xs, idxs, xf, ties_allowed=40)
    # head statistics on the final residual stream
    z = O.head_logits(xf.cpu().numpy(), bits(model["head"]), D.rms_eps)
    ref = O.head_stats(z, D.mask_id)
    z[:, D.mask_id] = -np.inf
    ref["z"] = z
    compare_head({k: v.cpu().numpy() for k, v in out.items()}, ref)


def test_full_block_invariants(model):
    """A whole block at logit scale 1: one commit per step, 32 steps. Since
    positions do not mix on this path, a masked slot's prediction is the same
    at every step, so every slot must end with its step-1 argmax, committed in
    descending step-1 confidence."""
    M = 32
    ctx = synth.make_ctx(D, M, 6, DEV)
    cmodel = clover.Model(D, model["layers"], model["embed"], model["head"])
    tokens, masked = synth.masked_block(D, M, DEV)
    ws = clover.workspace(clover.denoise_workspace_bytes(D, M))
    t2, m2 = synth.masked_block(D, M, DEV)
    _, _, _, first = _compose_step(model, model["layers"], ctx, t2, m2)
    torch.cuda.synchronize()
    arg1 = first["argmax"].cpu().numpy()
    p1 = first["max_prob"].cpu().numpy()
    order = []
    prev = masked.cpu().numpy()
    for step in range(M):
        clover.denoise_step(cmodel, ctx, tokens, masked, block=32, ws=ws)
        now = masked.cpu().numpy()
        assert not np.any((prev == 0) & (now == 1))
        newly = np.nonzero((prev == 1) & (now == 0))[0]
        assert len(newly) == 1
        order.append(int(newly[0]))
        prev = now
    clover.workspace_status(ws)
    assert int(masked.sum()) == 0
    assert np.array_equal(tokens.cpu().numpy(), arg1)
    want = sorted(range(M), key=lambda p: (-float(p1[p]), p))
    assert order == want


def test_denoise_block_loop_entry_point(model):
    """clover_denoise_block itself on one Clover block at logit scale 1: it
    must run exactly 32 steps (one commit per step), leave no slot masked,
    and leave every slot with the token it predicted at step 1. With a step
    cap of 5 it stops early and reports NOT_CONVERGED with 27 slots left."""
    M = 32
    ctx = synth.make_ctx(D, M, 10, DEV)
    cmodel = clover.Model(D, model["layers"], model["embed"], model["head"])
    t2, m2 = synth.masked_block(D, M, DEV)
    _, _, _, first = _compose_step(model, model["layers"], ctx, t2, m2)
    torch.cuda.synchronize()
    arg1 = first["argmax"].cpu().numpy()
    ws = clover.workspace(clover.denoise_workspace_bytes(D, M))
    tokens, masked = synth.masked_block(D, M, DEV)
    steps = clover.denoise_block(cmodel, ctx, tokens, masked, block=32, max_steps=32, ws=ws)
    clover.workspace_status(ws)
    assert steps == 32
    assert int(masked.sum()) == 0
    assert np.array_equal(tokens.cpu().numpy(), arg1)
    tokens, masked = synth.masked_block(D, M, DEV)
    with pytest.raises(clover.CloverError) as ei:
        clover.denoise_block(cmodel, ctx, tokens, masked, block=32, max_steps=5, ws=ws)
    assert ei.value.code == clover.ERR_NOT_CONVERGED
    assert int(masked.sum()) == 27
    m = masked.cpu().numpy()
    assert np.array_equal(tokens.cpu().numpy()[m == 0], arg1[m == 0])


def test_batched_zipf_8_blocks(model):
    B, M = 8, 256
    layers = [synth.Layer(L.router_w, L.gate_up, L.down, L.sh_gate_up, L.sh_down,
                          synth.zipf_router_bias(D, 0, l, 1.2, DEV)) for l, L in enumerate(model["layers"])]
    ctx = synth.make_ctx(D, M, 7, DEV)
    cmodel = clover.Model(D, layers, model["embed"], model["head"])
    t1, m1 = synth.masked_block(D, M, DEV)
    clover.denoise_step(cmodel, ctx, t1, m1, block=32)
    t2, m2 = synth.masked_block(D, M, DEV)
    xs, idxs, xf, out = _compose_step(model, layers, ctx, t2, m2)
    torch.cuda.synchronize()
    assert torch.equal(t1, t2) and torch.equal(m1, m2)
    m = m1.cpu().numpy().reshape(B, 32)
    assert np.all(m.sum(axis=1) == 31)             # one commit per block
    # every layer against the oracle under teacher forcing (40 x 256 tokens)
    _teacher_forced(layers, xs, idxs, xf, ties_allowed=320)
    counts = np.bincount(idxs[20].cpu().numpy().ravel(), minlength=D.n_experts)
    assert counts.max() >= 100                     # hot experts carry a large share of the batch
