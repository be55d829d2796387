"""GPU vs oracle on the tiny configuration (1 MoE layer, hidden 256, 16
experts top-2 + shared, SwiGLU 256->64->256, vocabulary 1,024, blocks of 8),
plus ragged shapes and edge cases. Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import (bits, calibrate_alpha, compare_head, compare_routing, decisions_clear, hidden_close,
                           layer_to_oracle)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dims(**kw):
    import dataclasses
    return dataclasses.replace(synth.TINY, **kw)


@pytest.mark.parametrize("M", [8, 1, 5, 16, 37, 256])
def test_moe_layer_matches_oracle(M):
    d = synth.TINY
    layer = synth.make_layer(d, 0, 0, DEV)
    x = synth.make_x(d, M, 3, DEV)
    x_out, idx, w = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    g = x_out.cpu().numpy()
    ok, worst = hidden_close(g, forced["x_out"])
    assert ok, worst
    ok, worst = hidden_close(g - xh, forced["x_out"] - xh)   # the MoE update alone
    assert ok, worst


@pytest.mark.parametrize("M", [8, 40])
def test_wide_hidden_matches_oracle(M):
    """Hidden 4,096 (above the 2,048-column chunk of the standalone router
    contraction, and above the fused kernel's register-resident rows), 32
    experts top-4: the chunked routing path (M = 40) and the fused path
    (M = 8) against the oracle."""
    d = _dims(hidden=4096, n_experts=32, top_k=4)
    layer = synth.make_layer(d, 14, 0, DEV, zipf_s=0.5)
    x = synth.make_x(d, M, 15, DEV)
    x_out, idx, w = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    ok, worst = hidden_close(x_out.cpu().numpy() - xh, forced["x_out"] - xh)
    assert ok, worst


@pytest.mark.parametrize("M", [40, 100, 256])
def test_hot_experts_match_oracle(M):
    """Experts that carry more than 32 tokens: with 4 of 16 experts per
    token, d_ff 128 and a skewed router, several routed experts and the
    shared one take more token columns than one 32-column step of the
    epilogue (M = 40 and 100), and at M = 256 the heaviest experts and the
    shared one fill more than 128 of the accumulator's 256 columns. Their
    units stream each weight tile once against all of the expert's token
    rows."""
    d = _dims(n_experts=16, top_k=4, d_ff=128)
    layer = synth.make_layer(d, 16, 0, DEV, zipf_s=1.0)
    x = synth.make_x(d, M, 17, DEV)
    x_out, idx, w = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    ok, worst = hidden_close(x_out.cpu().numpy() - xh, forced["x_out"] - xh)
    assert ok, worst
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=d.n_experts)
    assert (counts > 32).sum() >= 3             # routed experts over 32 tokens
    if M == 256:
        assert (counts > 128).sum() >= 1        # over half of the accumulator's columns


def test_moe_layer_in_place_and_deterministic():
    d = synth.TINY
    layer = synth.make_layer(d, 1, 0, DEV, zipf_s=1.2)
    x = synth.make_x(d, 64, 4, DEV)
    a, ia, wa = clover.moe_block_step(d, layer, x)
    b, ib, wb = clover.moe_block_step(d, layer, x)
    xi = x.clone()
    c, _, _ = clover.moe_block_step(d, layer, xi, x_out=xi)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ia, ib) and torch.equal(wa, wb)
    assert torch.equal(a, c)


def test_zipf_bias_routes_like_oracle():
    d = synth.TINY
    layer = synth.make_layer(d, 2, 0, DEV, zipf_s=1.2)
    x = synth.make_x(d, 128, 5, DEV)
    x_out, idx, w = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer)
    ref = O.moe_layer(x.cpu().numpy(), L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    # the bias makes the popular experts popular
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=d.n_experts)
    top = int(np.argmax(layer.router_bias.cpu().numpy()))
    assert counts[top] == counts.max()


def _head_ref(d, head, x, alpha):
    z = O.head_logits(x, bits(head), d.rms_eps, alpha)
    st = O.head_stats(z, d.mask_id)
    z = z.copy()
    z[:, d.mask_id] = -np.inf
    st["z"] = z
    return st


@pytest.mark.parametrize("V,M", [(1024, 8), (1000, 37), (1024, 256), (1100, 200)])
def test_head_unmask_matches_oracle(V, M):
    d = _dims(vocab=V, mask_id=V - 1)
    head = synth.make_head(d, 7, DEV)
    x = synth.make_x(d, M, 8, DEV)
    xh = x.cpu().numpy()
    z_raw = O.head_logits(xh, bits(head), d.rms_eps)
    alpha = calibrate_alpha(z_raw, d.mask_id, synth.confidence_targets(M, 9).numpy(), O)
    tokens, masked = synth.masked_block(d, M, DEV)
    masked[::3] = 0                       # some slots already committed
    tokens[::3] = 5
    t0, m0 = tokens.cpu().numpy(), masked.cpu().numpy()
    a = torch.from_numpy(alpha).to(DEV)
    out = clover.lmhead_unmask(d, head, x, tokens, masked, logit_scale=a, threshold=0.95, block=d.block)
    torch.cuda.synchronize()
    ref = _head_ref(d, head, xh, alpha)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_head(got, ref)
    assert not np.any(got["argmax"] == d.mask_id)
    if decisions_clear(ref["max_prob"], m0, 0.95, d.block):
        rt, rm, rc = O.unmask(t0, m0, ref["argmax"], ref["max_prob"], 0.95, d.block)
        assert np.array_equal(tokens.cpu().numpy(), rt)
        assert np.array_equal(masked.cpu().numpy(), rm)
        assert int(got["n_committed"][0]) == int(rc.sum())


def test_head_mask_token_never_predicted():
    d = synth.TINY
    M = 16
    x = synth.make_x(d, M, 10, DEV)
    xh = x.cpu().numpy()
    xb = O.round_to_bf16(O.rms_norm(xh, d.rms_eps))
    head = synth.make_head(d, 11, DEV)
    hh = head.float().cpu().numpy()
    hh[d.mask_id] = xb[0] * 0.2          # the mask row would win position 0 by far
    head = torch.from_numpy(hh).to(torch.bfloat16).to(DEV)
    tokens, masked = synth.masked_block(d, M, DEV)
    out = clover.lmhead_unmask(d, head, x, tokens, masked, block=M)
    torch.cuda.synchronize()
    assert int(out["argmax"][0]) != d.mask_id
    ref = _head_ref(d, head, xh, None)
    compare_head({k: v.cpu().numpy() for k, v in out.items()}, ref)


def test_tiny_denoise_four_steps():
    """Tiny configuration: 4 denoising steps with the 0.95 rule, against the
    oracle's loop, step by step."""
    d = synth.TINY
    n = 8
    layer = synth.make_layer(d, 0, 0, DEV)
    embed = synth.make_embed(d, 0, DEV)
    head = synth.make_head(d, 0, DEV)
    ctx = synth.make_ctx(d, n, 0, DEV)
    model = clover.Model(d, [layer], embed, head)
    ref_model = {"dims": {"top_k": d.top_k, "rms_eps": d.rms_eps, "mask_id": d.mask_id},
                 "layers": [layer_to_oracle(layer)], "embed": bits(embed), "head": bits(head),
                 "ctx": ctx.cpu().numpy()}
    # logit scales so that a few slots clear the threshold at step 1
    t0, m0 = synth.masked_block(d, n)
    x1 = O.embed(t0.numpy(), ref_model["embed"], ref_model["ctx"])
    x1 = O.moe_layer(x1, ref_model["layers"][0], d.top_k, d.rms_eps)["x_out"]
    alpha = calibrate_alpha(O.head_logits(x1, ref_model["head"], d.rms_eps), d.mask_id,
                            synth.confidence_targets(n, 1).numpy(), O)
    tokens, masked = synth.masked_block(d, n, DEV)
    a = torch.from_numpy(alpha).to(DEV)
    rt, rm = t0.numpy(), m0.numpy()
    ws = clover.workspace(clover.denoise_workspace_bytes(d, n))
    for step in range(4):
        ref = O.denoise_step(rt, rm, ref_model, 0.95, d.block, alpha)
        clover.denoise_step(model, ctx, tokens, masked, logit_scale=a, block=d.block, ws=ws)
        torch.cuda.synchronize()
        assert decisions_clear(ref["max_prob"], rm, 0.95, d.block), step
        rt, rm = ref["tokens"], ref["masked"]
        assert np.array_equal(tokens.cpu().numpy(), rt), step
        assert np.array_equal(masked.cpu().numpy(), rm), step
    clover.workspace_status(ws)


@pytest.mark.parametrize("M", [8, 32, 40])
def test_multi_layer_step_hidden_equals_composition(M):
    """Three layers: the denoise step's residual stream (up to 32 positions
    each layer's combine runs at the start of the next layer's launch, the
    last in a combine kernel) equals per-layer calls bit for bit, and every
    layer of the composition matches the oracle under its own routing."""
    d = synth.TINY
    layers = [synth.make_layer(d, 5, l, DEV) for l in range(3)]
    embed = synth.make_embed(d, 5, DEV)
    head = synth.make_head(d, 5, DEV)
    ctx = synth.make_ctx(d, M, 5, DEV)
    model = clover.Model(d, layers, embed, head)
    tokens, masked = synth.masked_block(d, M, DEV)
    t0 = tokens.clone()
    ws = clover.denoise_step(model, ctx, tokens, masked, block=d.block)
    x = embed[t0.long()].float() + ctx
    for layer in layers:
        xi = x
        x, idx, _ = clover.moe_block_step(d, layer, xi)
        torch.cuda.synchronize()
        L = layer_to_oracle(layer)
        ref = O.moe_layer(xi.cpu().numpy(), L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
        ok, worst = hidden_close(x.cpu().numpy(), ref["x_out"])
        assert ok, worst
    assert torch.equal(clover.denoise_hidden(d, ws, M), x)
    clover.workspace_status(ws)


def test_denoise_block_runs_to_completion_and_reports():
    d = synth.TINY
    n = 16
    layer = synth.make_layer(d, 3, 0, DEV)
    model = clover.Model(d, [layer], synth.make_embed(d, 3, DEV), synth.make_head(d, 3, DEV))
    ctx = synth.make_ctx(d, n, 3, DEV)
    tokens, masked = synth.masked_block(d, n, DEV)
    steps = clover.denoise_block(model, ctx, tokens, masked, block=d.block, max_steps=n)
    torch.cuda.synchronize()
    assert 1 <= steps <= d.block
    assert int(masked.sum()) == 0
    assert not bool((tokens == d.mask_id).any())
    # too few steps -> not converged, with the steps taken reported
    tokens, masked = synth.masked_block(d, n, DEV)
    with pytest.raises(clover.CloverError) as ei:
        clover.denoise_block(model, ctx, tokens, masked, block=d.block, max_steps=2)
    assert ei.value.code == clover.ERR_NOT_CONVERGED
    assert int(masked.sum()) == n - 4            # one commit per step per block of 8
    # nothing masked -> zero steps
    steps = clover.denoise_block(model, ctx, tokens, torch.zeros_like(masked), block=d.block, max_steps=4)
    assert steps == 0


def test_bad_token_id_is_clamped_and_reported():
    d = synth.TINY
    n = 8
    layer = synth.make_layer(d, 4, 0, DEV)
    model = clover.Model(d, [layer], synth.make_embed(d, 4, DEV), synth.make_head(d, 4, DEV))
    ctx = synth.make_ctx(d, n, 4, DEV)
    tokens, masked = synth.masked_block(d, n, DEV)
    tokens[2] = d.vocab + 5
    masked[2] = 0
    ws = clover.denoise_step(model, ctx, tokens, masked, block=d.block)
    with pytest.raises(clover.CloverError) as ei:
        clover.workspace_status(ws)
    assert ei.value.code == clover.ERR_DEVICE_TIMEOUT and "token id" in str(ei.value)
    clover.workspace_status(ws)    # the status word was cleared


@pytest.mark.parametrize("M", [8, 40])
def test_router_exact_ties_take_the_lower_expert_id(M):
    """Experts 2 and 5 (and 9 and 12) get identical router rows, scaled up so
    that the pair wins wherever its dot product is positive: their logits tie
    exactly and the rule takes the lower expert id first, with equal weights.
    Both routing paths: the fused kernel (8 tokens) and the standalone router
    (40 tokens)."""
    d = synth.TINY
    layer = synth.make_layer(d, 21, 0, DEV)
    w = layer.router_w
    w[2] = w[2] * 8.0
    w[5] = w[2]
    w[9] = w[9] * 8.0
    w[12] = w[9]
    x = synth.make_x(d, M, 22, DEV)
    x_out, idx, wt = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    ref = O.moe_layer(x.cpu().numpy(), layer_to_oracle(layer), d.top_k, d.rms_eps)
    idx_g, w_g = idx.cpu().numpy(), wt.cpu().numpy()
    pairs = [(2, 5), (9, 12)]
    hits = 0
    for t in range(M):
        sel = tuple(int(e) for e in ref["idx"][t])
        if sel in pairs:  # the oracle picked a tied pair: order and weights are fixed
            assert tuple(int(e) for e in idx_g[t]) == sel, (t, idx_g[t], sel)
            assert np.allclose(w_g[t], [0.5, 0.5], atol=1e-6), (t, w_g[t])
            hits += 1
        ps = np.sort(ref["p"][t])[::-1]
        if ps[d.top_k - 1] == ps[d.top_k]:  # a planted tie at the cut: the lower id is kept
            assert set(idx_g[t].tolist()) == set(sel), (t, idx_g[t], sel)
    assert hits >= M // 4, hits  # the planted ties decide a good share of the tokens
    compare_routing(idx_g, w_g, ref, d.top_k)


@pytest.mark.parametrize("M", [8, 40])
def test_dependency_timeout_is_reported_and_cleared(M):
    """Failure detection without a fault. Fused kernel (8 tokens): the grid
    barrier's arrival count in the workspace control block (bytes 24-31, a
    64-bit count that only grows) is set one past a multiple of the grid
    size, so the last CTA to arrive waits for a count that no CTA will reach.
    Standalone expert kernel (40 tokens, no grid barrier): the unit counter
    (bytes 4-7) is set to 1, so unit 0 (the first gate/up slice of the
    shared expert) is never drawn and the shared expert's down units wait
    for a slice that never comes. Either bounded wait gives up after about
    two seconds and sets the status word; the status call reports the
    timeout and clears the control block, and the same workspace then gives
    the oracle's result."""
    d = synth.TINY
    layer = synth.make_layer(d, 31, 0, DEV)
    x = synth.make_x(d, M, 32, DEV)
    ws = clover.workspace(clover.moe_workspace_bytes(d, M), x.device)
    if M <= 32:
        ws[24:32].view(torch.int64).fill_(1)
    else:
        ws[4:8].view(torch.int32).fill_(1)
    clover.moe_block_step(d, layer, x, ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(clover.CloverError) as ei:
        clover.workspace_status(ws)
    assert ei.value.code == clover.ERR_DEVICE_TIMEOUT and "dependency wait timed out" in str(ei.value)
    clover.workspace_status(ws)  # cleared
    x_out, idx, w = clover.moe_block_step(d, layer, x, ws=ws)
    torch.cuda.synchronize()
    clover.workspace_status(ws)
    L = layer_to_oracle(layer)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    ok, worst = hidden_close(x_out.cpu().numpy() - xh, forced["x_out"] - xh)
    assert ok, worst
