"""Shared test helpers: conversions from synthetic torch tensors to the
oracle's numpy inputs, tolerance checks, and logit-scale calibration."""
from __future__ import annotations

import numpy as np
import torch

from block_diffusion_moe_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


class LazyExperts:
    """Index by expert id -> uint16 bit array of that expert, copied from the
    (possibly device-resident) tensor only when the oracle asks for it."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = bits(self.t[e])
        return self.cache[e]


def layer_to_oracle(layer: synth.Layer, lazy: bool = False) -> dict:
    d = {
        "router_w": bits(layer.router_w),
        "sh_gate_up": bits(layer.sh_gate_up),
        "sh_down": bits(layer.sh_down),
        "router_bias": None if layer.router_bias is None
        else layer.router_bias.detach().cpu().numpy().astype(np.float32),
    }
    if lazy:
        d["gate_up"] = LazyExperts(layer.gate_up)
        d["down"] = LazyExperts(layer.down)
    else:
        d["gate_up"] = bits(layer.gate_up)
        d["down"] = bits(layer.down)
    return d


def hidden_close(g, r, rtol=2e-2):
    """Hidden-state tolerance: |g - r| <= rtol * (|r| + rms(row of r))
    elementwise and ||g - r|| / ||r|| <= rtol per row. Returns (ok, worst)."""
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    el = np.abs(g - r) / (np.abs(r) + rms)
    row = np.linalg.norm(g - r, axis=-1) / np.maximum(np.linalg.norm(r, axis=-1), 1e-300)
    worst = max(float(el.max(initial=0.0)), float(row.max(initial=0.0)))
    return worst <= rtol, worst


def calibrate_alpha(z_raw: np.ndarray, mask_id: int, targets, oracle_mod,
                    iters: int = 60) -> np.ndarray:
    """Per-position logit scale alpha_p such that the oracle's max probability
    at scale alpha_p equals targets[p] (bisection; p_max grows with alpha)."""
    z_raw = np.asarray(z_raw, dtype=np.float64)
    targets = np.asarray(targets, dtype=np.float64)
    out = np.empty(z_raw.shape[0])
    for p in range(z_raw.shape[0]):
        lo, hi = 0.0, 1.0
        zp = z_raw[p:p + 1]

        def pm(a):
            return float(oracle_mod.head_stats(zp * a, mask_id)["max_prob"][0])

        while pm(hi) < targets[p] and hi < 1e6:
            hi *= 2.0
        for _ in range(iters):
            mid = 0.5 * (lo + hi)
            if pm(mid) < targets[p]:
                lo = mid
            else:
                hi = mid
        out[p] = 0.5 * (lo + hi)
    return out.astype(np.float32)
