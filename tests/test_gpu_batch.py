"""Calls of more than 256 tokens (several 32-position blocks batched), against
the oracle.

The standalone expert kernel processes an expert's tokens in chunks of at
most 128 rows, and the head takes the positions in sub-calls of whole blocks
of at most 256 positions. Zipf-biased routers make the hot experts carry far
more than 256 tokens here, so multi-chunk experts, the routing counters for
more than 16 token tiles and the split head all run. Every call goes through
the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import (bits, calibrate_alpha, compare_head, compare_routing, decisions_clear, hidden_close,
                           layer_to_oracle)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layer_vs_oracle(d, layer, M, seed):
    x = synth.make_x(d, M, seed, DEV)
    x_out, idx, w = clover.moe_block_step(d, layer, x)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer, lazy=True)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    ties = compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    g = x_out.cpu().numpy()
    ok, worst = hidden_close(g, forced["x_out"])
    assert ok, worst
    ok, worst = hidden_close(g - xh, forced["x_out"] - xh)
    assert ok, worst
    return idx.cpu().numpy(), ties


@pytest.mark.parametrize("M", [300, 600, 1024])
def test_tiny_layer_beyond_256_tokens(M):
    """16 experts top-2 with a Zipf(1.2) router: the hottest experts take
    several hundred tokens each (two to four chunks), the shared expert all M
    (two to four chunks)."""
    d = synth.TINY
    layer = synth.make_layer(d, 31, 0, DEV, zipf_s=1.2)
    idx, ties = _layer_vs_oracle(d, layer, M, 32 + M)
    counts = np.bincount(idx.ravel(), minlength=d.n_experts)
    if M >= 600:
        assert counts.max() > 256
    assert ties <= max(2, M // 64)


def test_tiny_layer_deterministic_and_in_place_at_1024():
    d = synth.TINY
    layer = synth.make_layer(d, 33, 0, DEV, zipf_s=1.2)
    x = synth.make_x(d, 1024, 34, DEV)
    a, ia, wa = clover.moe_block_step(d, layer, x)
    b, ib, wb = clover.moe_block_step(d, layer, x)
    xi = x.clone()
    c, _, _ = clover.moe_block_step(d, layer, xi, x_out=xi)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ia, ib) and torch.equal(wa, wb)
    assert torch.equal(a, c)


def test_clover_layer_512_tokens_zipf():
    """16 blocks of 32 through one Clover-shaped layer with a Zipf(1.2)
    router: the hot experts carry more than 256 of the 512 tokens."""
    d = synth.CLOVER
    layer = synth.make_layer(d, 35, 3, DEV, zipf_s=1.2)
    idx, ties = _layer_vs_oracle(d, layer, 512, 36)
    counts = np.bincount(idx.ravel(), minlength=d.n_experts)
    assert counts.max() > 256
    assert ties <= 8


@pytest.mark.parametrize("V,M,block", [(1024, 300, 8), (1100, 600, 32), (1024, 1024, 32)])
def test_head_unmask_beyond_256_positions(V, M, block):
    """The head in sub-calls of whole blocks (256 positions at most): every
    position's statistics and every block's unmask decision against the
    oracle, and the committed count summed over the sub-calls."""
    d = dataclasses.replace(synth.TINY, vocab=V, mask_id=V - 1)
    head = synth.make_head(d, 37, DEV)
    x = synth.make_x(d, M, 38, DEV)
    xh = x.cpu().numpy()
    z_raw = O.head_logits(xh, bits(head), d.rms_eps)
    alpha = calibrate_alpha(z_raw, d.mask_id, synth.confidence_targets(M, 39).numpy(), O, iters=40)
    tokens, masked = synth.masked_block(d, M, DEV)
    masked[::5] = 0
    tokens[::5] = 3
    t0, m0 = tokens.cpu().numpy(), masked.cpu().numpy()
    out = clover.lmhead_unmask(d, head, x, tokens, masked, logit_scale=torch.from_numpy(alpha).to(DEV),
                               threshold=0.95, block=block)
    torch.cuda.synchronize()
    z = z_raw * alpha.astype(np.float64)[:, None]
    ref = O.head_stats(z, d.mask_id)
    z[:, d.mask_id] = -np.inf
    ref["z"] = z
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_head(got, ref)
    assert decisions_clear(ref["max_prob"], m0, 0.95, block)
    rt, rm, rc = O.unmask(t0, m0, ref["argmax"], ref["max_prob"], 0.95, block)
    assert np.array_equal(tokens.cpu().numpy(), rt)
    assert np.array_equal(masked.cpu().numpy(), rm)
    assert int(got["n_committed"][0]) == int(rc.sum())


def test_head_rejects_wide_blocks_beyond_256_positions():
    d = dataclasses.replace(synth.TINY, vocab=1024, mask_id=1023)
    head = synth.make_head(d, 40, DEV)
    x = synth.make_x(d, 600, 41, DEV)
    tokens, masked = synth.masked_block(d, 600, DEV)
    with pytest.raises(clover.CloverError) as ei:
        clover.lmhead_unmask(d, head, x, tokens, masked, block=300)
    assert ei.value.code == clover.ERR_UNSUPPORTED_SHAPE


def test_accept_beyond_256_rows():
    """Ten verify blocks of 32 drafts + 1 (330 rows): sub-calls of 7 and 3
    blocks; each block's accepted length and tokens against the oracle."""
    d = dataclasses.replace(synth.TINY, vocab=1024, mask_id=1023)
    B, blk = 10, 33
    M = B * blk
    head = synth.make_head(d, 42, DEV)
    x = synth.make_x(d, M, 43, DEV)
    xh = x.cpu().numpy()
    z = O.head_logits(xh, bits(head), d.rms_eps)
    st0 = O.head_stats(z, d.mask_id)
    rng = np.random.default_rng(44)
    draft = st0["argmax"].copy()
    flip = rng.random(M) > 0.8
    draft[flip] = rng.integers(0, d.vocab - 1, flip.sum())
    dr = torch.from_numpy(draft.astype(np.int32)).to(DEV)
    out = clover.lmhead_accept(d, head, x, dr, blk, rule=clover.ACCEPT_EXACT)
    torch.cuda.synchronize()
    vs = O.verify_stats(z, d.mask_id, draft)
    ref = O.accept(draft, vs["argmax"], vs["p_draft"], vs["entropy"], 0, 0.9, 0.6, blk)
    top2 = np.sort(np.where(np.arange(d.vocab) == d.mask_id, -np.inf, z), axis=1)[:, -2:]
    gap = np.exp(top2[:, 1] - vs["lse"]) - np.exp(top2[:, 0] - vs["lse"])
    got_len = out["accept_len"].cpu().numpy()
    for b in range(B):
        rows = range(b * blk, (b + 1) * blk)
        if any(gap[r] < 1e-3 for r in rows):
            continue                     # a near-tie may flip the exact rule
        assert got_len[b] == ref["accept_len"][b], b
        assert np.array_equal(out["tokens"].cpu().numpy()[b * blk:(b + 1) * blk], ref["tokens"][b * blk:(b + 1) * blk])
    assert np.array_equal(out["argmax"].cpu().numpy()[gap >= 1e-3], vs["argmax"][gap >= 1e-3])


def test_clover_denoise_step_512_positions_zipf():
    """16 blocks x 32 positions through 40 Clover-shaped layers with
    Zipf(1.2) routers: the fused step equals the layer-by-layer composition
    bit for bit, one commit per block, and every layer matches the oracle
    under teacher forcing."""
    D = synth.CLOVER
    B, M = 16, 512
    base = [synth.make_layer(D, 0, l, DEV) for l in range(D.n_layers)]
    layers = [synth.Layer(L.router_w, L.gate_up, L.down, L.sh_gate_up, L.sh_down,
                          synth.zipf_router_bias(D, 0, l, 1.2, DEV)) for l, L in enumerate(base)]
    embed = synth.make_embed(D, 0, DEV)
    head = synth.make_head(D, 0, DEV)
    ctx = synth.make_ctx(D, M, 45, DEV)
    cmodel = clover.Model(D, layers, embed, head)
    t1, m1 = synth.masked_block(D, M, DEV)
    ws = clover.denoise_step(cmodel, ctx, t1, m1, block=32)
    t2, m2 = synth.masked_block(D, M, DEV)
    x = embed[t2.long()].float() + ctx
    xs, idxs = [], []
    for layer in layers:
        xs.append(x)
        x, idx, _ = clover.moe_block_step(D, layer, x)
        idxs.append(idx)
    out = clover.lmhead_unmask(D, head, x, t2, m2, block=32)
    torch.cuda.synchronize()
    clover.workspace_status(ws)
    assert torch.equal(t1, t2) and torch.equal(m1, m2)
    assert torch.equal(clover.denoise_hidden(D, ws, M), x)
    assert np.all(m1.cpu().numpy().reshape(B, 32).sum(axis=1) == 31)
    assert int(out["n_committed"][0]) == B
    hot = 0
    ties = 0
    for l, layer in enumerate(layers):
        L = layer_to_oracle(layer, lazy=True)
        xh = xs[l].cpu().numpy()
        ig = idxs[l].cpu().numpy()
        hot = max(hot, int(np.bincount(ig.ravel(), minlength=D.n_experts).max()))
        free = O.moe_layer(xh, L, D.top_k, D.rms_eps)
        ref = O.moe_layer(xh, L, D.top_k, D.rms_eps, force_idx=ig)
        ties += compare_routing(ig, ref["w"], free, D.top_k)
        g = (xs[l + 1] if l + 1 < len(xs) else x).cpu().numpy()
        ok, worst = hidden_close(g - xh, ref["x_out"] - xh)
        assert ok, (l, worst)
    assert hot > 256
    assert ties <= 640
