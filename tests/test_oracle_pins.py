"""Pins for the CPU oracle: each check ties a part of the oracle to something
other than itself (a library routine, a closed form, brute force on tiny
inputs, an invariant of the method, a number printed on the pages)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import synth
from tests.helpers import bits, layer_to_oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits_of(vals):
    return bits(torch.tensor(np.asarray(vals), dtype=torch.float32).to(torch.bfloat16))


# --------------------------------------------------------------------- bf16


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(200_000, generator=g, dtype=torch.float64) * 3.0
    # exact float32 halfway cases between two bf16 neighbours
    base = torch.randn(1000, generator=g).to(torch.bfloat16).to(torch.float32)
    half = (base.view(torch.int32) | 0x8000).view(torch.float32).to(torch.float64)
    x = torch.cat([x, half, torch.tensor([0.0, -0.0, 1.0, -2.5, 1e-30, 3e38], dtype=torch.float64)])
    want = x.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(x.numpy())
    assert np.array_equal(got, want)


def test_bf16_rounding_goes_through_float32():
    """The oracle rounds a float64 value to bf16 in two steps, first to the
    float32 the kernels hold and then to bf16, each to nearest even. The two
    steps differ from one direct rounding only where the float32 step lands
    exactly on a bf16 tie: 1 + 2^-8 + 2^-30 is above the tie between 1 and
    1 + 2^-7, but its float32 rounding is the tie itself, which then goes to
    the even neighbour 1. With 2^-20 instead of 2^-30 the excess survives in
    float32 and the value rounds up."""
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -8 + 2.0 ** -20, -(1.0 + 2.0 ** -8 + 2.0 ** -30),
                  1.0 + 3 * 2.0 ** -8 - 2.0 ** -31])
    got = O.round_to_bf16(x)
    assert got[0] == 1.0
    assert got[1] == 1.0 + 2.0 ** -7
    assert got[2] == -1.0
    # 1 + 3 * 2^-8 is the tie between 1 + 2^-7 and 1 + 2^-6 (odd and even
    # last bits); just below it float32 rounds onto the tie, which goes up
    assert got[3] == 1.0 + 2.0 ** -6


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(2)
    t = torch.randn(10_000, generator=g).to(torch.bfloat16)
    assert np.array_equal(O.bf16_to_f64(bits(t)), t.to(torch.float64).numpy())


# ------------------------------------------------------------------ rmsnorm


@pytest.mark.parametrize("H", [8, 256, 2048])
def test_rms_norm_closed_forms(H):
    eps = 1e-6
    c = -3.25
    xn = O.rms_norm(np.full((1, H), c), eps)
    assert np.allclose(xn, c / math.sqrt(c * c + eps), rtol=1e-15, atol=0)
    s = 7.0
    x = np.zeros((1, H))
    x[0, 3] = s
    xn = O.rms_norm(x, eps)
    assert xn[0, 3] == pytest.approx(s / math.sqrt(s * s / H + eps), rel=1e-14)
    assert np.count_nonzero(xn) == 1


def test_silu_identities():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=0, atol=1e-12)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert O.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


# ------------------------------------------------------------------- router


def _planted_router(logit_vals, H=8):
    """Router rows with one nonzero (bf16-exact) entry each, so that an
    all-ones input (RMSNorm -> bf16 1.0) yields exactly these logits."""
    E = len(logit_vals)
    w = np.zeros((E, H), dtype=np.float32)
    for e, v in enumerate(logit_vals):
        w[e, (3 * e + 1) % H] = v
    return bits(torch.from_numpy(w).to(torch.bfloat16))


def test_route_planted_logits_and_tie_break():
    vals = [0.5, 2.0, -1.0, 2.0, 0.25, -4.0]
    wr = _planted_router(vals, H=8)
    xb = O.round_to_bf16(O.rms_norm(np.ones((1, 8)), 1e-6))
    assert np.all(xb == 1.0)
    logits, p, idx, w = O.route(xb, wr, 3)
    assert np.array_equal(logits[0], np.array(vals))
    assert list(idx[0]) == [1, 3, 0]  # tie at 2.0 -> lower id first
    denom = 2 * math.exp(2.0) + math.exp(0.5)
    assert w[0, 0] == pytest.approx(math.exp(2.0) / denom, rel=1e-14)
    assert w[0, 2] == pytest.approx(math.exp(0.5) / denom, rel=1e-14)
    # a bias reorders the selection
    bias = np.array([3.0, 0, 0, 0, 0, 0], dtype=np.float32)
    _, _, idx_b, _ = O.route(xb, wr, 2, bias)
    assert list(idx_b[0]) == [0, 1]


def test_route_topk_is_max_sum_subset_bruteforce():
    rng = np.random.default_rng(3)
    E, H, K = 9, 16, 3
    wr = _bf16_bits_of(rng.normal(0, 0.3, (E, H)))
    xb = O.round_to_bf16(O.rms_norm(rng.normal(size=(20, H)), 1e-6))
    logits, p, idx, w = O.route(xb, wr, K)
    for t in range(20):
        best = max(itertools.combinations(range(E), K), key=lambda s: sum(logits[t, list(s)]))
        assert set(idx[t]) == set(best)
        assert len(set(idx[t])) == K
        assert math.fsum(p[t]) == pytest.approx(1.0, abs=1e-12)
        assert math.fsum(w[t]) == pytest.approx(1.0, abs=1e-12)
        # renormalised probabilities = softmax restricted to the chosen logits
        sel = logits[t, idx[t]]
        ref = [math.exp(v - max(sel)) for v in sel]
        ref = [v / math.fsum(ref) for v in ref]
        assert np.allclose(w[t], ref, rtol=1e-12, atol=0)


# ------------------------------------------------------------------ experts


def test_swiglu_expert_closed_form_nonsquare():
    # H = 3, F = 2: gate picks x0 and x2, up = 2 * gate, down maps
    # h0 -> out2 and h1 -> out0 (out1 stays 0).
    gate = np.array([[1, 0, 0], [0, 0, 1]], dtype=np.float32)
    up = 2.0 * gate
    gu = _bf16_bits_of(np.concatenate([gate, up]))
    down = _bf16_bits_of(np.array([[0, 1], [0, 0], [1, 0]], dtype=np.float32))
    xb = np.array([[0.5, -7.0, -1.25]])
    out = O.swiglu_expert(xb, gu, down)

    def h(v):
        s = v / (1.0 + math.exp(-v))
        return float(O.round_to_bf16(np.array([s * 2.0 * v]))[0])

    assert out[0, 0] == pytest.approx(h(-1.25), rel=1e-15)
    assert out[0, 1] == 0.0
    assert out[0, 2] == pytest.approx(h(0.5), rel=1e-15)


def _tiny_layer(seed=0, zipf=None):
    return synth.make_layer(synth.TINY, seed, 0, "cpu", zipf_s=zipf)


@pytest.mark.parametrize("zipf", [None, 1.2])
def test_sparse_moe_equals_dense_bruteforce(zipf):
    d = synth.TINY
    L = layer_to_oracle(_tiny_layer(0, zipf))
    x = synth.make_x(d, 8, 0).numpy()
    sparse = O.moe_layer(x, L, d.top_k, d.rms_eps)["x_out"]
    dense = O.moe_layer_dense(x, L, d.top_k, d.rms_eps)
    assert np.allclose(sparse, dense, rtol=1e-12, atol=1e-12)


def test_moe_identical_experts_ignore_routing():
    """With every routed expert equal, the combine weights sum to one, so the
    output equals that expert plus the shared expert whatever the routing."""
    d = synth.TINY
    L = layer_to_oracle(_tiny_layer(1))
    L["gate_up"] = np.repeat(L["gate_up"][:1], d.n_experts, axis=0)
    L["down"] = np.repeat(L["down"][:1], d.n_experts, axis=0)
    x = synth.make_x(d, 8, 1).numpy()
    out = O.moe_layer(x, L, d.top_k, d.rms_eps)
    xb = out["xb"]
    want = x + O.swiglu_expert(xb, L["gate_up"][0], L["down"][0]) \
        + O.swiglu_expert(xb, L["sh_gate_up"], L["sh_down"])
    assert np.allclose(out["x_out"], want, rtol=1e-12, atol=1e-12)
    # zero routed experts -> only the shared expert remains
    L["gate_up"] = np.zeros_like(L["gate_up"])
    out = O.moe_layer(x, L, d.top_k, d.rms_eps)
    assert np.allclose(out["x_out"], x + O.swiglu_expert(xb, L["sh_gate_up"], L["sh_down"]),
                       rtol=1e-13, atol=1e-13)


def test_teacher_forced_routing_uses_given_experts():
    d = synth.TINY
    L = layer_to_oracle(_tiny_layer(2))
    x = synth.make_x(d, 8, 2).numpy()
    free = O.moe_layer(x, L, d.top_k, d.rms_eps)
    forced = O.moe_layer(x, L, d.top_k, d.rms_eps, force_idx=free["idx"])
    assert np.array_equal(free["x_out"], forced["x_out"])
    other = (free["idx"] + 1) % d.n_experts
    forced2 = O.moe_layer(x, L, d.top_k, d.rms_eps, force_idx=other)
    assert not np.allclose(forced2["x_out"], free["x_out"])


# --------------------------------------------------------------------- head


def test_head_stats_bruteforce_fsum():
    rng = np.random.default_rng(4)
    V, M, mask = 50, 3, 17
    z = rng.normal(0, 3, (M, V))
    st = O.head_stats(z, mask)
    for p in range(M):
        vals = [(z[p, v], v) for v in range(V) if v != mask]
        m = max(v for v, _ in vals)
        a = min(i for v, i in vals if v == m)
        lse = m + math.log(math.fsum(math.exp(v - m) for v, _ in vals))
        assert st["argmax"][p] == a
        assert st["max_logit"][p] == m
        assert st["lse"][p] == pytest.approx(lse, rel=1e-14)
        assert st["max_prob"][p] == pytest.approx(math.exp(m - lse), rel=1e-13)


def test_head_stats_closed_forms():
    V = 1024
    z = np.full((2, V), 1.5)
    st = O.head_stats(z, 0)
    # all logits equal, mask id 0 excluded -> lowest non-mask id, p = 1/(V-1)
    assert list(st["argmax"]) == [1, 1]
    assert st["max_prob"][0] == pytest.approx(1.0 / (V - 1), rel=1e-13)
    assert st["lse"][0] == pytest.approx(1.5 + math.log(V - 1), rel=1e-14)
    # the mask token never wins, even with the largest logit
    z = np.zeros((1, V))
    z[0, 5] = 50.0
    z[0, 9] = 10.0
    st = O.head_stats(z, 5)
    assert st["argmax"][0] == 9
    assert st["max_logit"][0] == 10.0


def test_head_logits_planted_row_and_scale():
    d = synth.TINY
    rng = np.random.default_rng(5)
    x = rng.normal(size=(2, d.hidden))
    head = rng.normal(0, 0.02, (d.vocab, d.hidden))
    xb = O.round_to_bf16(O.rms_norm(x, d.rms_eps))
    head[700] = xb[0] * 0.05      # aligned with position 0
    head[33] = xb[1] * 0.05       # aligned with position 1
    hb = _bf16_bits_of(head)
    z = O.head_logits(x, hb, d.rms_eps, alpha=np.array([1.0, 2.0]))
    st = O.head_stats(z, d.mask_id)
    assert list(st["argmax"]) == [700, 33]
    z1 = O.head_logits(x, hb, d.rms_eps)
    assert np.allclose(z[1], 2.0 * z1[1], rtol=1e-15)


# ------------------------------------------------------------------- unmask


def test_unmask_golden_cases():
    with open(os.path.join(HERE, "golden", "unmask_rule_cases.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        t, m, com = O.unmask(c["tokens"], c["masked"], c["argmax"], c["max_prob"],
                             c["threshold"], c["block"])
        assert list(t) == c["want_tokens"], c["name"]
        assert list(m) == c["want_masked"], c["name"]
        assert [int(v) for v in com] == c["want_committed"], c["name"]


# ---------------------------------------------------------- denoise loop


def _tiny_model(seed=0, n_pos=8):
    d = synth.TINY
    return {
        "dims": {"top_k": d.top_k, "rms_eps": d.rms_eps, "mask_id": d.mask_id},
        "layers": [layer_to_oracle(_tiny_layer(seed))],
        "embed": bits(synth.make_embed(d, seed)),
        "head": bits(synth.make_head(d, seed)),
        "ctx": synth.make_ctx(d, n_pos, seed).numpy(),
    }


@pytest.mark.parametrize("alpha_val", [1.0, 60.0])
def test_denoise_loop_invariants(alpha_val):
    d = synth.TINY
    n = 8
    model = _tiny_model(0, n)
    tok, msk = synth.masked_block(d, n)
    alpha = np.full(n, alpha_val)
    res = O.denoise_block(tok.numpy(), msk.numpy(), model, 0.95, d.block, max_steps=n, alpha=alpha)
    hist = res["history"]
    assert not res["masked"].any()
    assert 1 <= res["steps"] <= n
    first = hist[0]
    # every slot ends with the token it predicted while still masked at step 1
    assert np.array_equal(res["tokens"], first["argmax"])
    assert not np.any(res["tokens"] == d.mask_id)
    prev_masked = msk.numpy()
    for st in hist:
        # never re-masks, always progresses
        assert not np.any((prev_masked == 0) & (st["masked"] == 1))
        assert st["committed"].sum() >= 1
        prev_masked = st["masked"]
    # commit order: all slots above the threshold at step 1, then one per step
    # in descending probability
    p1 = first["max_prob"].astype(np.float32)
    above = p1 > np.float32(0.95)
    if above.any():
        assert np.array_equal(first["committed"], above)
        assert res["steps"] == 1 + int((~above).sum())
    else:
        assert res["steps"] == n
    rest = [p for p in np.argsort(-p1, kind="stable") if not above[p]]
    later = [int(np.nonzero(st["committed"])[0][0]) for st in hist[1 if above.any() else 0:]]
    assert later == rest[:len(later)]


def test_denoise_four_steps_tiny_config():
    d = synth.TINY
    model = _tiny_model(0, 8)
    tok, msk = synth.masked_block(d, 8)
    res = O.denoise_block(tok.numpy(), msk.numpy(), model, 0.95, d.block, max_steps=4)
    assert res["steps"] == 4
    assert int(res["masked"].sum()) == 8 - 4   # random head: one commit per step


# ------------------------------------------------------- byte model / shapes


def test_clover_shape_sums_match_pages():
    """Files, 'What Clover is': one expert is 3,145,728 parameters; routed
    experts are 32,212,254,720; the head is 508,559,360."""
    c = synth.CLOVER
    assert c.expert_params == 3_145_728
    assert c.n_layers * c.n_experts * c.expert_params == 32_212_254_720
    assert c.vocab * c.hidden == 508_559_360
    assert c.expert_bytes == 6_291_456


def test_uniform_routing_union_matches_closed_form():
    """Files, 'The expert selection': a 32-token block under independent
    routing touches 256(1-(1-8/256)^32) ~ 163.3 experts (their simulation:
    163.4). The oracle's router on the synthetic Clover-shaped inputs must
    land there."""
    c = synth.CLOVER
    closed = c.n_experts * (1 - (1 - c.top_k / c.n_experts) ** 32)
    assert closed == pytest.approx(163.31, abs=0.01)
    wr = bits(synth.make_router(c, 12345, 0))
    unions = []
    for b in range(40):
        x = synth.make_x(c, 32, 1000 + b).numpy()
        xb = O.round_to_bf16(O.rms_norm(x, c.rms_eps))
        _, _, idx, _ = O.route(xb, wr, c.top_k)
        unions.append(len(np.unique(idx)))
    mean = float(np.mean(unions))
    assert abs(mean - closed) < 2.5, mean
    assert abs(mean - 163.4) < 2.5


def test_embed_closed_form():
    """Input assembly x_p = E[t_p] + c_p: with a planted table (row v holds the
    constant v/4) and context c_p = p/8, x_p is (t_p/4 + p/8) everywhere."""
    V, H = 12, 6
    table = np.repeat((np.arange(V, dtype=np.float32) / 4.0)[:, None], H, axis=1)
    tb = _bf16_bits_of(table)
    tokens = np.array([11, 3, 3, 0])
    ctx = np.repeat((np.arange(4) / 8.0)[:, None], H, axis=1)
    x = O.embed(tokens, tb, ctx)
    want = (tokens / 4.0 + np.arange(4) / 8.0)[:, None] * np.ones((1, H))
    assert np.array_equal(x, want)


# ------------------------------------------------------------------ coreset


def test_coreset_hand_example():
    """Three tokens, k = 2. Masses (summed top-k probabilities): e0 0.5,
    e1 0.3, e2 0.1, e3 0.1. top_p 0.9 keeps {0, 1, 2} (0.5, 0.8, 0.9);
    0.95 keeps all four; 0.5 keeps {0, 1} (at least k = 2). e2 and e3 tie at
    0.1 and e2 (lower id) comes first."""
    p = np.zeros((3, 6))
    p[0, [0, 1]] = [0.3, 0.2]
    p[1, [0, 2]] = [0.2, 0.1]
    p[2, [1, 3]] = [0.1, 0.1]
    idx = np.array([[0, 1], [0, 2], [1, 3]])
    assert list(O.coreset(p, idx, 0.9)) == [0, 1, 2]
    assert list(O.coreset(p, idx, 0.95)) == [0, 1, 2, 3]
    assert list(O.coreset(p, idx, 0.5)) == [0, 1]
    assert list(O.coreset(p, idx, 0.0)) == [0, 1]


def test_coreset_top_p_one_is_identity():
    """top_p = 1 keeps every expert any token selected, so no token re-routes."""
    d = synth.TINY
    L = layer_to_oracle(_tiny_layer(4))
    x = synth.make_x(d, 8, 4).numpy()
    a = O.moe_layer(x, L, d.top_k, d.rms_eps)
    b = O.moe_layer(x, L, d.top_k, d.rms_eps, coreset_top_p=1.0, block=8)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.allclose(a["x_out"], b["x_out"], rtol=1e-12, atol=1e-12)


def test_coreset_invariants_clover_shape():
    c = synth.CLOVER
    wr = bits(synth.make_router(c, 5, 0))
    for blk in range(4):
        x = synth.make_x(c, 32, 50 + blk).numpy()
        xb = O.round_to_bf16(O.rms_norm(x, c.rms_eps))
        logits, p, idx, w = O.route(xb, wr, c.top_k)
        keep = O.coreset(p, idx, 0.9)
        union = set(np.unique(idx).tolist())
        assert set(keep.tolist()) <= union
        assert len(keep) >= c.top_k
        mass = np.zeros(c.n_experts)
        for t in range(32):
            for e in idx[t]:
                mass[e] += p[t, e]
        cum = mass[keep].sum()
        assert cum >= 0.9 * mass.sum()
        assert cum - mass[keep[-1]] < 0.9 * mass.sum()          # minimal
        assert np.all(np.diff(mass[keep]) <= 0)                 # kept by mass
        ki, kw = O.route_within(logits, keep, c.top_k)
        assert set(np.unique(ki).tolist()) <= set(keep.tolist())
        assert np.allclose(kw.sum(axis=1), 1.0)
        for t in range(32):                                     # untouched tokens keep their routing
            if set(idx[t].tolist()) <= set(keep.tolist()):
                assert set(ki[t].tolist()) == set(idx[t].tolist())
                assert np.allclose(np.sort(kw[t]), np.sort(w[t]))


def test_coreset_shrinks_the_union_like_the_pages():
    """Files, 'The expert selection': under independent routing a 32-token
    block touches 163.4 experts and the selector at 0.9 keeps 126.7,
    re-routing about 1.1 of a token's 8 slots (their synthetic logits; the
    noise model is not given, so the check is a band; these inputs give
    127.3 kept and 1.11 re-routed)."""
    c = synth.CLOVER
    wr = bits(synth.make_router(c, 6, 0))
    kept, rerouted = [], []
    for b in range(12):
        x = synth.make_x(c, 32, 200 + b).numpy()
        xb = O.round_to_bf16(O.rms_norm(x, c.rms_eps))
        logits, p, idx, w = O.route(xb, wr, c.top_k)
        keep = O.coreset(p, idx, 0.9)
        ki, _ = O.route_within(logits, keep, c.top_k)
        kept.append(len(keep))
        rerouted.append(np.mean([len(set(idx[t]) - set(ki[t])) for t in range(32)]))
    assert abs(np.mean(kept) - 126.7) < 6, np.mean(kept)
    assert abs(np.mean(rerouted) - 1.1) < 0.3, np.mean(rerouted)


def test_route_within_planted_ties_and_weights():
    logits = np.array([[1.0, 2.0, 2.0, 0.5, 3.0]])
    idx, w = O.route_within(logits, [1, 2, 3], 2)      # 4 is not allowed
    assert list(idx[0]) == [1, 2]                        # tie at 2.0 -> lower id first
    assert np.allclose(w[0], [0.5, 0.5])
    idx, w = O.route_within(logits, [0, 3, 2], 2)
    assert list(idx[0]) == [2, 0]
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-14)


# ---------------------------------------------------------------------------
# Self-speculative accept test (Files, "Two ways to run it")


def _verify_rows(z):
    return O.verify_stats(np.asarray(z, dtype=np.float64), z.shape[1] - 1, np.full(z.shape[0], -1))


def test_entropy_closed_forms():
    V = 1024
    # uniform over the V - 1 tokens left once the mask token (id V - 1) is out
    st = _verify_rows(np.full((2, V), 0.37))
    assert np.allclose(st["entropy"], math.log(V - 1), rtol=0, atol=1e-12)
    # two live tokens with probabilities 1/4 and 3/4
    z = np.full((1, V), -1e4)
    z[0, 5] = 0.0
    z[0, 9] = math.log(3.0)
    st = O.verify_stats(z, V - 1, np.array([9]))
    want = -(0.25 * math.log(0.25) + 0.75 * math.log(0.75))
    assert abs(st["entropy"][0] - want) < 1e-12
    assert abs(st["p_draft"][0] - 0.75) < 1e-12
    # a certain row: entropy 0, the argmax has probability 1
    z = np.zeros((1, V))
    z[0, 17] = 5000.0
    st = O.verify_stats(z, V - 1, np.array([17]))
    assert st["entropy"][0] == 0.0 and st["p_draft"][0] == 1.0 and st["argmax"][0] == 17


def test_entropy_matches_scipy_and_bounds():
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(3)
    V = 257
    z = rng.normal(0.0, 2.0, size=(6, V))
    st = _verify_rows(z)
    for n in range(6):
        p = np.exp(z[n, :V - 1] - z[n, :V - 1].max())
        assert abs(st["entropy"][n] - scipy_stats.entropy(p)) < 1e-10
    assert np.all(st["entropy"] >= 0) and np.all(st["entropy"] <= math.log(V - 1) + 1e-12)


def test_verify_stats_bruteforce_loops():
    # pure-Python softmax, entropy and draft probability on a 3 x 7 matrix,
    # mask id 3 excluded
    rng = np.random.default_rng(4)
    z = rng.normal(0.0, 1.5, size=(3, 7))
    z[1, 3] = 40.0               # the mask token's logit must not count
    draft = np.array([2, 3, 6])  # row 1 drafts the mask token
    st = O.verify_stats(z, 3, draft)
    for n in range(3):
        ex = [math.exp(z[n, v]) if v != 3 else 0.0 for v in range(7)]
        tot = math.fsum(ex)
        p = [e / tot for e in ex]
        h = -math.fsum(q * math.log(q) for q in p if q > 0)
        assert abs(st["entropy"][n] - h) < 1e-12
        assert abs(st["p_draft"][n] - p[draft[n]]) < 1e-12
    assert st["p_draft"][1] == 0.0


def test_accept_threshold_matches_the_pages():
    # defaults 0.9 / 0.6: probability 0.6 when certain, 0.22 at one nat
    assert O.accept_threshold([0.0], 0.9, 0.6)[0] == 0.6
    assert round(float(O.accept_threshold([1.0], 0.9, 0.6)[0]), 2) == 0.22
    # with the defaults the ratio never binds
    H = np.linspace(0.0, 12.0, 97)
    assert np.allclose(O.accept_threshold(H, 0.9, 0.6), 0.6 * np.exp(-H), rtol=0, atol=0)
    # a larger delta lets the ratio bind while the entropy is low
    assert O.accept_threshold([0.0], 0.9, 3.0)[0] == 0.9
    assert O.accept_threshold([3.0], 0.9, 3.0)[0] == pytest.approx(3.0 * math.exp(-3.0))


def test_accept_golden_cases():
    path = os.path.join(os.path.dirname(__file__), "golden", "accept_rule_cases.json")
    cases = json.load(open(path))["cases"]
    assert len(cases) >= 7
    for c in cases:
        got = O.accept(c["draft"], c["argmax"], c["p_draft"], c["entropy"], c["rule"], c["ratio"], c["delta"],
                       c["block"])
        assert got["accept_len"].tolist() == c["want_len"], c["name"]
        assert got["tokens"].tolist() == c["want_tokens"], c["name"]


def test_accept_invariants():
    rng = np.random.default_rng(5)
    V, block, nb = 64, 9, 40                  # rounds of 8 drafts: at most 9 tokens
    z = rng.normal(0.0, 2.5, size=(nb * block, V))
    st0 = _verify_rows(z)
    draft = np.where(rng.random(nb * block) < 0.7, st0["argmax"], rng.integers(0, V - 1, nb * block))
    st = O.verify_stats(z, V - 1, draft)
    ex = O.accept(draft, st["argmax"], st["p_draft"], st["entropy"], O.ACCEPT_EXACT, 0.9, 0.6, block)
    prev = None
    for delta in (10.0, 3.0, 0.6, 0.1):
        th = O.accept(draft, st["argmax"], st["p_draft"], st["entropy"], O.ACCEPT_THRESHOLD, 0.9, delta, block)
        if prev is not None:                  # a more lenient rule never keeps fewer drafts
            assert np.all(th["accept_len"] >= prev)
        prev = th["accept_len"]
    for b in range(nb):
        r = ex["accept_len"][b]
        toks = ex["tokens"][b * block:(b + 1) * block]
        assert 0 <= r <= block - 1 and np.sum(toks >= 0) == r + 1
        # exact matching reproduces the verifier's own greedy tokens
        assert toks[:r + 1].tolist() == st["argmax"][b * block:b * block + r + 1].tolist()
        assert np.all(toks[r + 1:] == -1)


# ---------------------------------------------------------------------------
# Low-bit expert weight format (this implementation's own; the pages give none)


def _bf16_bits(x):
    return O.bf16_bits_of(np.asarray(x, dtype=np.float64))


def test_q4_round_trip_is_exact_on_the_grid():
    # each group holds multiples of 2^-6 from -7 to 7 with its maximum at 7:
    # the scale is exactly 2^-6, the codes are the multiples, dequant is exact
    rng = np.random.default_rng(6)
    k = rng.integers(-7, 8, size=(3, 128)).astype(np.float64)
    k[:, 0] = 7
    k[:, 64] = -7
    w = _bf16_bits(k * 2.0 ** -6)
    packed, s = O.quantize_q4(w)
    assert s.shape == (2, 3) and np.all(O.bf16_to_f64(s) == 2.0 ** -6)
    assert np.array_equal(O.dequantize_q4(packed, s), w)


def test_q4_packing_order_hand_example():
    # codes u = 1..8 for elements 0..7 of row 0: nibble i holds element
    # (0, 2, 4, 6, 1, 3, 5, 7)[i], so the word is 0x86427531
    k = np.zeros((1, 64))
    k[0, :8] = np.arange(1, 9) - 8          # q = u - 8
    k[0, 8] = 7                             # sets the group maximum: s = 2^-6 below
    w = _bf16_bits(k * 2.0 ** -6)
    packed, s = O.quantize_q4(w)
    assert O.bf16_to_f64(s)[0, 0] == 2.0 ** -6
    assert packed[0, :4].tolist() == [0x31, 0x75, 0x42, 0x86]
    assert packed[0, 4] & 0xF == 7 + 8      # element 8 is nibble 0 of the next word


def test_q4_error_bound_and_extremes():
    rng = np.random.default_rng(7)
    w = _bf16_bits(rng.normal(0.0, 0.02, size=(5, 256)))
    w[2, 64:128] = 0                        # an all-zero group
    packed, s = O.quantize_q4(w)
    sv = O.bf16_to_f64(s).T                 # [R][K/64]
    wd = O.bf16_to_f64(O.dequantize_q4(packed, s))
    wf = O.bf16_to_f64(w)
    step = np.repeat(sv, 64, axis=1)
    assert np.all(np.abs(wd - wf) <= step / 2 + np.abs(wd) * 2.0 ** -8 + 1e-30)
    assert sv[2, 1] == 0 and np.all(wd[2, 64:128] == 0)
    words = packed.view("<u4")
    codes = np.stack([(words >> (4 * i)) & 0xF for i in range(8)], axis=-1)
    assert codes.min() >= 1 and codes.max() <= 15   # |q| <= 7 with the /7 scale
    # the element of largest magnitude in every live group gets code +-7
    el = np.empty((5, 256), dtype=np.int64)           # codes in element order
    nib = (0, 2, 4, 6, 1, 3, 5, 7)
    for i in range(8):
        el.reshape(5, 32, 8)[:, :, nib[i]] = codes[:, :, i]
    g = wf.reshape(5, 4, 64)
    at_max = el.reshape(5, 4, 64)[np.arange(5)[:, None], np.arange(4)[None, :], np.abs(g).argmax(axis=2)]
    live = np.abs(g).max(axis=2) > 0
    assert np.all(np.abs(at_max[live] - 8) == 7)


def test_q4_scales_are_group_major():
    k = np.zeros((2, 128))
    k[0, 3] = 7 * 2.0 ** -4                 # row 0 group 0: s = 2^-4
    k[1, 70] = 7 * 2.0 ** -2                # row 1 group 1: s = 2^-2
    packed, s = O.quantize_q4(_bf16_bits(k))
    sv = O.bf16_to_f64(s)
    assert s.shape == (2, 2)
    assert sv[0, 0] == 2.0 ** -4 and sv[1, 1] == 2.0 ** -2 and sv[0, 1] == 0 and sv[1, 0] == 0
