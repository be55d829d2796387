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


# ----------------------------------------------------------- GPU comparisons
# Decision bands. The stated tolerance is 1e-3 in probability; on top of it a
# decision is allowed to differ only when the oracle's own margin is below the
# relative error the fp32 kernels can introduce (REL_BAND), so near-miss
# decisions with a clear margin must agree exactly.
PROB_BAND = 1e-3
REL_BAND = 1e-4


def compare_routing(idx_g, w_g, ref, K):
    """Expert sets must be identical per token except where the oracle's K-th
    and (K+1)-th routing probabilities lie within the tie band; the weights of
    matching tokens agree within 2e-2 relative. Returns the number of tokens
    excused by the band."""
    idx_g = np.asarray(idx_g)
    w_g = np.asarray(w_g, dtype=np.float64)
    p = ref["p"]
    ties = 0
    for t in range(idx_g.shape[0]):
        sg, so = set(idx_g[t].tolist()), set(ref["idx"][t].tolist())
        assert len(sg) == K, (t, idx_g[t])
        if sg != so:
            ps = np.sort(p[t])[::-1]
            gap = ps[K - 1] - ps[K]
            # the kernels' bf16 normed input can differ from the oracle's by one
            # ulp in a few elements, moving a logit by ~1e-4: allow a swap only
            # when the probability margin is below 1e-3 relative (and 1e-3 absolute)
            assert gap < PROB_BAND and gap < 1e-3 * ps[K - 1], (t, sorted(sg), sorted(so), gap)
            ties += 1
            continue
        wo = dict(zip(ref["idx"][t].tolist(), ref["w"][t].tolist()))
        for e, w in zip(idx_g[t].tolist(), w_g[t].tolist()):
            assert abs(w - wo[e]) <= 2e-2 * wo[e] + 1e-7, (t, e, w, wo[e])
        assert abs(w_g[t].sum() - 1.0) < 1e-5
    return ties


def compare_head(out, ref, tau=0.95):
    """argmax exact unless the top-2 probabilities are within the band;
    max logit and log-sum-exp within 2e-2 relative (against max(|r|, 1));
    max probability within 2e-2 relative."""
    am = np.asarray(out["argmax"])
    ml = np.asarray(out["max_logit"], dtype=np.float64)
    ls = np.asarray(out["lse"], dtype=np.float64)
    pm = np.asarray(out["max_prob"], dtype=np.float64)
    excused = 0
    for p in range(am.shape[0]):
        if am[p] != ref["argmax"][p]:
            z = ref["z"][p]
            top2 = np.sort(z)[-2:]
            dp = np.exp(top2[1] - ref["lse"][p]) - np.exp(top2[0] - ref["lse"][p])
            assert dp < PROB_BAND, (p, am[p], ref["argmax"][p], dp)
            excused += 1
        assert abs(ml[p] - ref["max_logit"][p]) <= 2e-2 * max(abs(ref["max_logit"][p]), 1.0)
        assert abs(ls[p] - ref["lse"][p]) <= 2e-2 * max(abs(ref["lse"][p]), 1.0)
        assert abs(pm[p] - ref["max_prob"][p]) <= 2e-2 * ref["max_prob"][p]
    return excused


def decisions_clear(max_prob, masked, tau, block):
    """True when every unmask decision of this step has a margin above the
    band: no masked probability within the band of tau, and the fallback
    choice (when no slot clears tau) is separated from the runner-up."""
    pm = np.asarray(max_prob, dtype=np.float64)
    masked = np.asarray(masked)
    for b0 in range(0, pm.shape[0], block):
        idx = [i for i in range(b0, min(pm.shape[0], b0 + block)) if masked[i]]
        if not idx:
            continue
        vals = pm[idx]
        if np.any(np.abs(vals - tau) < REL_BAND * tau):
            return False
        if not np.any(vals > tau) and len(vals) > 1:
            s = np.sort(vals)[::-1]
            if s[0] - s[1] < REL_BAND * s[0]:
                return False
    return True


def q4_bits(b: np.ndarray) -> np.ndarray:
    """The oracle's own low-bit round trip of a bf16 matrix: the bf16 bits of
    the weights a product uses after quantization."""
    import oracle as O
    return O.dequantize_q4(*O.quantize_q4(b))


class LazyQ4Experts(LazyExperts):
    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = q4_bits(bits(self.t[e]))
        return self.cache[e]


def layer_to_oracle_q4(layer: synth.Layer, lazy: bool = False) -> dict:
    """layer_to_oracle with every expert matrix replaced by the oracle's own
    low-bit round trip of it (the router stays bf16)."""
    d = layer_to_oracle(layer, lazy=True)
    d["sh_gate_up"] = q4_bits(d["sh_gate_up"])
    d["sh_down"] = q4_bits(d["sh_down"])
    if lazy:
        d["gate_up"] = LazyQ4Experts(layer.gate_up)
        d["down"] = LazyQ4Experts(layer.down)
    else:
        d["gate_up"] = np.stack([q4_bits(bits(layer.gate_up[e])) for e in range(layer.gate_up.shape[0])])
        d["down"] = np.stack([q4_bits(bits(layer.down[e])) for e in range(layer.down.shape[0])])
    return d
