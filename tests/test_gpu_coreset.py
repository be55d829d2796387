"""Block coreset expert selection on the GPU against the oracle (Files, "The
expert selection"): the kept set, the re-routed selections and the layer
output, on the tiny and the Clover shapes, plus its identities."""
import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import compare_routing, hidden_close, layer_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _masses(ref_p, first_idx):
    E = ref_p.shape[1]
    mass = np.zeros(E)
    for t in range(first_idx.shape[0]):
        for e in first_idx[t]:
            mass[e] += ref_p[t, e]
    return mass


def _check(d, layer, x, top_p, lazy=False):
    x_out, idx, w = clover.moe_block_step(d, layer, x, coreset_top_p=top_p)
    torch.cuda.synchronize()
    L = layer_to_oracle(layer, lazy=lazy)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps, coreset_top_p=top_p, block=xh.shape[0])
    gi = idx.cpu().numpy()
    gw = w.cpu().numpy()
    # kept set: the GPU's routed union equals the oracle's kept experts that
    # some token selected in the first pass, unless the cut is within the
    # tie band (cumulative mass within 1e-4 of the target)
    kept = ref["coreset"][0]
    first = O.route(ref["xb"], L["router_w"], d.top_k, L.get("router_bias"))
    mass = _masses(first[1], first[2])
    total = mass.sum()
    cum = np.cumsum(mass[kept])
    union = set(np.unique(gi).tolist())
    want = {int(e) for e in kept if mass[e] > 0}
    if union != want:
        near = np.abs(cum - top_p * total) < 1e-4 * total
        assert near.any(), (sorted(union ^ want))
        ref = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=gi)
    else:
        assert set(gi.ravel().tolist()) <= set(kept.tolist())
        compare_routing(gi, gw, ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=gi)
    ok, worst = hidden_close(x_out.cpu().numpy() - xh, forced["x_out"] - xh)
    assert ok, worst
    return gi, len(want)


@pytest.mark.parametrize("M", [8, 5])
def test_coreset_tiny(M):
    d = synth.TINY
    layer = synth.make_layer(d, 7, 0, DEV)
    x = synth.make_x(d, M, 8, DEV)
    _check(d, layer, x, 0.9)
    _check(d, layer, x, 0.5)


def test_coreset_clover_block_of_32():
    d = synth.CLOVER
    layer = synth.make_layer(d, 9, 0, DEV)
    x = synth.make_x(d, 32, 10, DEV)
    gi, kept = _check(d, layer, x, 0.9, lazy=True)
    plain = clover.moe_block_step(d, layer, x)[1]
    torch.cuda.synchronize()
    assert kept < len(np.unique(plain.cpu().numpy()))          # fewer experts streamed


def test_coreset_top_p_one_equals_no_coreset():
    d = synth.CLOVER
    layer = synth.make_layer(d, 11, 0, DEV)
    x = synth.make_x(d, 32, 12, DEV)
    a = clover.moe_block_step(d, layer, x)
    b = clover.moe_block_step(d, layer, x, coreset_top_p=1.0)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]) and torch.equal(a[0], b[0])


def test_coreset_rejected_beyond_one_block():
    d = synth.TINY
    layer = synth.make_layer(d, 7, 0, DEV)
    x = synth.make_x(d, 64, 8, DEV)
    with pytest.raises(clover.CloverError) as ei:
        clover.moe_block_step(d, layer, x, coreset_top_p=0.9)
    assert ei.value.code == clover.ERR_UNSUPPORTED_SHAPE


def test_denoise_step_with_coreset():
    d = synth.TINY
    n = 8
    layer = synth.make_layer(d, 13, 0, DEV)
    embed = synth.make_embed(d, 13, DEV)
    head = synth.make_head(d, 13, DEV)
    ctx = synth.make_ctx(d, n, 13, DEV)
    model = clover.Model(d, [layer], embed, head, coreset_top_p=0.9)
    tokens, masked = synth.masked_block(d, n, DEV)
    steps = clover.denoise_block(model, ctx, tokens, masked, block=n, max_steps=n)
    torch.cuda.synchronize()
    assert steps == n and int(masked.sum()) == 0
    assert not bool((tokens == d.mask_id).any())
