"""Seeded synthetic inputs for the block-diffusion MoE denoising step.

This module only draws numbers: weights, embeddings, per-position context
terms, router biases and token states. It contains none of the method's
arithmetic (no normalisation, routing, expert, head or unmask computation), so
both the CUDA path and the CPU oracle may consume what it produces.

Shapes follow the Clover-35B-A3B description in "Clover-35B-A3B: how a
diffusion model gets to 680 tokens a second, read from its files"
(section "What Clover is"): hidden 2,048, 256 routed experts with top-8 plus
one always-on shared expert per layer, 40 layers, vocabulary 248,320, block 32,
mask token 151669; one expert is gate and up at 2,048 x 512 and down at
512 x 2,048.

Every tensor comes from its own torch.Generator, seeded from
(seed, layer, tensor tag, expert), so any expert or layer can be regenerated
alone and the draw does not depend on chunking. Values drawn on a CUDA device
differ from values drawn on the CPU for the same seed; a comparison therefore
always feeds both sides the same bytes (copied to the host when needed).
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    hidden: int
    n_experts: int
    top_k: int
    d_ff: int
    vocab: int
    mask_id: int
    rms_eps: float = 1e-6
    n_layers: int = 1
    block: int = 32

    @property
    def expert_params(self) -> int:
        return 3 * self.hidden * self.d_ff

    @property
    def expert_bytes(self) -> int:
        return 2 * self.expert_params

    @property
    def router_bytes(self) -> int:
        return 2 * self.n_experts * self.hidden

    @property
    def head_bytes(self) -> int:
        return 2 * self.vocab * self.hidden


# Tiny oracle-check shape: 1 layer, hidden 256, 16 routed experts top-2 plus a
# shared expert, SwiGLU 256->64->256, vocabulary 1,024, blocks of 8 positions.
# The Clover mask id (151669) lies outside a 1,024-row vocabulary, so the last
# row (1023) plays the mask token here.
TINY = Dims(hidden=256, n_experts=16, top_k=2, d_ff=64, vocab=1024,
            mask_id=1023, n_layers=1, block=8)

# Clover-35B-A3B shape.
CLOVER = Dims(hidden=2048, n_experts=256, top_k=8, d_ff=512, vocab=248320,
              mask_id=151669, n_layers=40, block=32)

WEIGHT_STD = 0.02

_TAG = {"router": 1, "gate_up": 2, "down": 3, "sh_gate_up": 4, "sh_down": 5,
        "head": 6, "embed": 7, "ctx": 8, "x": 9, "bias_perm": 10, "targets": 11}


def _seed(seed: int, layer: int, tag: str, index: int = 0) -> int:
    return (seed * 1_000_003 + layer * 10_007 + _TAG[tag] * 101 + index * 7_919) % (2**62)


def _gen(device, s: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def normal(shape, std: float, s: int, device, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std^2) draw in fp32, stored as `dtype`."""
    g = _gen(device, s)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(dtype)


@dataclasses.dataclass
class Layer:
    router_w: torch.Tensor      # bf16 [E][H]
    gate_up: torch.Tensor       # bf16 [E][2F][H]   rows 0..F-1 gate, F..2F-1 up
    down: torch.Tensor          # bf16 [E][H][F]
    sh_gate_up: torch.Tensor    # bf16 [2F][H]
    sh_down: torch.Tensor       # bf16 [H][F]
    router_bias: torch.Tensor | None = None  # fp32 [E]


def make_router(d: Dims, seed: int, layer: int, device="cpu") -> torch.Tensor:
    return normal((d.n_experts, d.hidden), WEIGHT_STD, _seed(seed, layer, "router"), device)


def make_expert(d: Dims, seed: int, layer: int, e: int, device="cpu"):
    """Routed expert e of a layer: (gate_up bf16 [2F][H], down bf16 [H][F]),
    the same values make_layer draws for it on the same device."""
    return (normal((2 * d.d_ff, d.hidden), WEIGHT_STD, _seed(seed, layer, "gate_up", e), device),
            normal((d.hidden, d.d_ff), WEIGHT_STD, _seed(seed, layer, "down", e), device))


def make_layer(d: Dims, seed: int, layer: int, device="cpu", zipf_s: float | None = None) -> Layer:
    E, H, F = d.n_experts, d.hidden, d.d_ff
    router_w = make_router(d, seed, layer, device)
    gate_up = torch.empty((E, 2 * F, H), dtype=torch.bfloat16, device=device)
    down = torch.empty((E, H, F), dtype=torch.bfloat16, device=device)
    for e in range(E):
        gate_up[e], down[e] = make_expert(d, seed, layer, e, device)
    sh_gate_up = normal((2 * F, H), WEIGHT_STD, _seed(seed, layer, "sh_gate_up"), device)
    sh_down = normal((H, F), WEIGHT_STD, _seed(seed, layer, "sh_down"), device)
    bias = zipf_router_bias(d, seed, layer, zipf_s, device) if zipf_s else None
    return Layer(router_w, gate_up, down, sh_gate_up, sh_down, bias)


def zipf_router_bias(d: Dims, seed: int, layer: int, s: float, device="cpu") -> torch.Tensor:
    """Per-expert router bias b_e = -s * ln(rank_e), ranks a seeded permutation
    of 1..E per layer, so that expert popularity falls off like rank^-s."""
    g = _gen("cpu", _seed(seed, layer, "bias_perm"))
    rank = torch.randperm(d.n_experts, generator=g).to(torch.float64) + 1.0
    return (-s * torch.log(rank)).to(torch.float32).to(device)


def make_head(d: Dims, seed: int, device="cpu") -> torch.Tensor:
    """Untied output head, bf16 [V][H]."""
    return normal((d.vocab, d.hidden), WEIGHT_STD, _seed(seed, 0, "head"), device)


def make_embed(d: Dims, seed: int, device="cpu") -> torch.Tensor:
    """Token embedding table, bf16 [V][H], N(0, 1)."""
    return normal((d.vocab, d.hidden), 1.0, _seed(seed, 0, "embed"), device)


def make_ctx(d: Dims, n_pos: int, seed: int, device="cpu") -> torch.Tensor:
    """Per-position context term c_p ~ N(0, 1), fp32 [n_pos][H], fixed for the
    block. It stands in for what the attention / recurrent layers (outside this
    path) contribute to each position."""
    return normal((n_pos, d.hidden), 1.0, _seed(seed, 0, "ctx"), device, dtype=torch.float32)


def make_x(d: Dims, n_tok: int, seed: int, device="cpu") -> torch.Tensor:
    """Residual-stream activations for a single-layer call: N(0, 1) values that
    are exactly representable in bf16, stored as fp32 [n_tok][H]."""
    return normal((n_tok, d.hidden), 1.0, _seed(seed, 0, "x"), device).to(torch.float32)


def masked_block(d: Dims, n_pos: int, device="cpu"):
    """A freshly opened block: every slot holds the mask token."""
    tokens = torch.full((n_pos,), d.mask_id, dtype=torch.int32, device=device)
    masked = torch.ones((n_pos,), dtype=torch.uint8, device=device)
    return tokens, masked


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def confidence_targets(n_pos: int, seed: int, frac_confident: float = 0.4):
    """Target max-probabilities for a head test: about `frac_confident` of the
    positions drawn from U(0.97, 0.995), the rest from U(0.30, 0.90), so that
    every target stays clear of the 0.95 threshold."""
    g = _gen("cpu", _seed(seed, 0, "targets"))
    u = torch.rand(n_pos, generator=g, dtype=torch.float64)
    sel = torch.rand(n_pos, generator=g, dtype=torch.float64) < frac_confident
    hi = 0.97 + 0.025 * u
    lo = 0.30 + 0.60 * u
    return torch.where(sel, hi, lo)
