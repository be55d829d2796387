"""Low-bit expert weights on the GPU against the oracle: the quantizer bit for
bit, then MoE layers and a denoising step whose experts stream 4-bit codes.
The oracle quantizes the same bf16 weights itself and runs its bf16 path on
the weights the codes stand for. Every call goes through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import bits, calibrate_alpha, compare_routing, decisions_clear, hidden_close, layer_to_oracle_q4

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_quantizer(w):
    q, s = clover.quantize_q4(w)
    torch.cuda.synchronize()
    w3 = w.view(1, *w.shape) if w.dim() == 2 else w
    q3 = q.view(1, *q.shape) if w.dim() == 2 else q
    s3 = s.view(1, *s.shape) if w.dim() == 2 else s
    for m in range(w3.shape[0]):
        rq, rs = O.quantize_q4(bits(w3[m]))
        assert np.array_equal(q3[m].cpu().numpy(), rq), m
        assert np.array_equal(s3[m].cpu().numpy().view(np.uint16), rs), m


def test_quantizer_bit_exact_planted_cases():
    # ties at exactly half a step (rint goes to even), an all-zero group, a
    # negative maximum, large and tiny magnitudes
    k = np.zeros((4, 192))
    k[0, :64] = np.array([7, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 1.5] * 8)
    k[1, 64:128] = 0.0
    k[1, :64] = -7.0 * np.linspace(1, 0, 64)
    k[2] = np.linspace(-1000, 1000, 192)
    k[3] = np.linspace(-1e-30, 1e-30, 192)
    w = torch.from_numpy(O.bf16_to_f64(O.bf16_bits_of(k * 2.0 ** -6)).astype(np.float32)).to(torch.bfloat16)
    w = w.to(DEV).contiguous()
    _check_quantizer(w)


def test_quantizer_bit_exact_expert_tensors():
    d = synth.TINY
    L = synth.make_layer(d, 3, 0, DEV)
    _check_quantizer(L.gate_up)
    _check_quantizer(L.down)
    _check_quantizer(L.sh_down)
    C = synth.CLOVER
    w = synth.normal((3, 2 * C.d_ff, C.hidden), synth.WEIGHT_STD, 77, DEV)
    _check_quantizer(w)
    _check_quantizer(synth.normal((2, C.hidden, C.d_ff), synth.WEIGHT_STD, 78, DEV))


def _layer_check(d, layer, x, lazy=False):
    q4 = clover.quantize_layer_q4(layer)
    x_out, idx, w = clover.moe_block_step(d, q4, x)
    torch.cuda.synchronize()
    L = layer_to_oracle_q4(layer, lazy=lazy)
    xh = x.cpu().numpy()
    ref = O.moe_layer(xh, L, d.top_k, d.rms_eps)
    compare_routing(idx.cpu().numpy(), w.cpu().numpy(), ref, d.top_k)
    forced = O.moe_layer(xh, L, d.top_k, d.rms_eps, force_idx=idx.cpu().numpy())
    ok, worst = hidden_close(x_out.cpu().numpy() - xh, forced["x_out"] - xh)
    assert ok, worst
    return q4, x_out


@pytest.mark.parametrize("M", [8, 5, 40])
def test_q4_layer_tiny(M):
    """The fused path (M <= 32) and the standalone path (M = 40)."""
    d = synth.TINY
    _layer_check(d, synth.make_layer(d, 4, 0, DEV, zipf_s=0.5), synth.make_x(d, M, 5, DEV))


def test_q4_layer_wider_ffn():
    d = dataclasses.replace(synth.TINY, n_experts=16, top_k=4, d_ff=128)
    _layer_check(d, synth.make_layer(d, 6, 0, DEV, zipf_s=1.0), synth.make_x(d, 100, 7, DEV))


@pytest.mark.parametrize("M,zipf", [(32, None), (256, 1.2)])
def test_q4_clover_layer(M, zipf):
    d = synth.CLOVER
    layer = synth.make_layer(d, 8, 0, DEV, zipf_s=zipf)
    q4, x_out = _layer_check(d, layer, synth.make_x(d, M, 9, DEV), lazy=True)
    # the same layer in bf16 differs by the quantization only
    ref, _, _ = clover.moe_block_step(d, layer, synth.make_x(d, M, 9, DEV))
    torch.cuda.synchronize()
    rel = float(torch.linalg.norm(x_out - ref) / torch.linalg.norm(ref))
    assert rel < 0.05


def test_q4_denoise_steps_tiny():
    """Four denoising steps of the tiny configuration with low-bit experts,
    step by step against the oracle's loop on the same weights."""
    d = synth.TINY
    n = 8
    layer = synth.make_layer(d, 10, 0, DEV)
    embed = synth.make_embed(d, 10, DEV)
    head = synth.make_head(d, 10, DEV)
    ctx = synth.make_ctx(d, n, 10, DEV)
    model = clover.Model(d, [clover.quantize_layer_q4(layer)], embed, head)
    ref_model = {"dims": {"top_k": d.top_k, "rms_eps": d.rms_eps, "mask_id": d.mask_id},
                 "layers": [layer_to_oracle_q4(layer)], "embed": bits(embed), "head": bits(head),
                 "ctx": ctx.cpu().numpy()}
    t0, m0 = synth.masked_block(d, n)
    x1 = O.embed(t0.numpy(), ref_model["embed"], ref_model["ctx"])
    x1 = O.moe_layer(x1, ref_model["layers"][0], d.top_k, d.rms_eps)["x_out"]
    alpha = calibrate_alpha(O.head_logits(x1, ref_model["head"], d.rms_eps), d.mask_id,
                            synth.confidence_targets(n, 11).numpy(), O)
    a = torch.from_numpy(alpha).to(DEV)
    tokens, masked = synth.masked_block(d, n, DEV)
    rt, rm = t0.numpy(), m0.numpy()
    for step in range(4):
        ref = O.denoise_step(rt, rm, ref_model, 0.95, d.block, alpha)
        clover.denoise_step(model, ctx, tokens, masked, logit_scale=a, block=d.block)
        torch.cuda.synchronize()
        assert decisions_clear(ref["max_prob"], rm, 0.95, d.block), step
        rt, rm = ref["tokens"], ref["masked"]
        assert np.array_equal(tokens.cpu().numpy(), rt), step
        assert np.array_equal(masked.cpu().numpy(), rm), step
