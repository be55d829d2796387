"""GPU verify-pass head fused with the self-speculative accept test, against
the oracle (Files, "Two ways to run it"): per-row entropy and draft
probability, the exact and threshold rules, the accepted prefix and the
round's tokens, on the tiny head and the Clover head; and agreement with the
unmask form of the same head. Every call goes through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from block_diffusion_moe_gb300 import clover, synth
from tests.helpers import PROB_BAND, bits, calibrate_alpha, compare_head

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ref(d, head_bits, xh, alpha, draft):
    z = O.head_logits(xh, head_bits, d.rms_eps, alpha)
    st = O.verify_stats(z, d.mask_id, draft)
    z[:, d.mask_id] = -np.inf
    st["z"] = z
    return st


def _drafts(argmax, V, block, seed, keep=0.75):
    """Mostly the row's argmax, else a random id; boundary rows carry none."""
    rng = np.random.default_rng(seed)
    n = argmax.shape[0]
    dr = np.where(rng.random(n) < keep, argmax, rng.integers(0, V, n)).astype(np.int32)
    dr[block - 1::block] = -1
    return dr


def _top2_gap(ref, n):
    top2 = np.sort(ref["z"][n])[-2:]
    return np.exp(top2[1] - ref["lse"][n]) - np.exp(top2[0] - ref["lse"][n])


def _check(got, ref, draft, rule, ratio, delta, block):
    compare_head(got, ref)
    n_rows = draft.shape[0]
    live = np.arange(n_rows) % block != block - 1
    assert np.all(np.abs(got["entropy"] - ref["entropy"]) <= 1e-3 + 1e-3 * ref["entropy"])
    assert np.all(np.abs(got["p_draft"][live] - ref["p_draft"][live]) <= 1e-3)
    # the GPU's own decisions, from its own per-row values
    thr_g = np.minimum(np.float32(ratio), np.float32(delta) * np.exp(-got["entropy"].astype(np.float32)))
    dec_g = (draft == got["argmax"]) if rule == O.ACCEPT_EXACT else (got["p_draft"] >= thr_g)
    # the oracle's decisions; inside the band the GPU's stand
    dec_r = O.accept(draft, ref["argmax"], ref["p_draft"], ref["entropy"], rule, ratio, delta, block)["accepted"]
    merged = dec_r.copy()
    thr_r = O.accept_threshold(ref["entropy"], ratio, delta)
    for i in np.where(live)[0]:
        if dec_g[i] == dec_r[i]:
            continue
        if rule == O.ACCEPT_EXACT:
            assert _top2_gap(ref, i) < PROB_BAND, (i, draft[i], got["argmax"][i], ref["argmax"][i])
        else:
            assert abs(ref["p_draft"][i] - thr_r[i]) < PROB_BAND, (i, ref["p_draft"][i], thr_r[i])
        merged[i] = dec_g[i]
    n_blk = n_rows // block
    assert got["accept_len"].shape[0] >= n_blk
    for b in range(n_blk):
        r = 0
        while r < block - 1 and merged[b * block + r]:
            r += 1
        assert got["accept_len"][b] == r, (b, got["accept_len"][b], r)
        toks = got["tokens"][b * block:(b + 1) * block]
        assert toks[:r].tolist() == draft[b * block:b * block + r].tolist()
        assert toks[r] == got["argmax"][b * block + r]
        assert np.all(toks[r + 1:] == -1)
    return got["accept_len"][:n_blk]


def _run(d, head, x, alpha, draft, block, rule, ratio, delta):
    out = clover.lmhead_accept(d, head, x, torch.from_numpy(draft).to(DEV), block, rule, ratio, delta,
                               logit_scale=None if alpha is None else torch.from_numpy(alpha).to(DEV))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("rule,delta", [(O.ACCEPT_EXACT, 0.6), (O.ACCEPT_THRESHOLD, 0.6),
                                        (O.ACCEPT_THRESHOLD, 3.0), (O.ACCEPT_THRESHOLD, 10.0)])
def test_accept_tiny_rounds_of_eight(rule, delta):
    """Rounds of 8 drafts (9 rows, at most 9 tokens), 6 rounds, confidence
    spread by per-row logit scales."""
    d = dataclasses.replace(synth.TINY, vocab=1000, mask_id=999)
    block, M = 9, 54
    head = synth.make_head(d, 21, DEV)
    x = synth.make_x(d, M, 22, DEV)
    xh = x.cpu().numpy()
    hb = bits(head)
    z_raw = O.head_logits(xh, hb, d.rms_eps)
    alpha = calibrate_alpha(z_raw, d.mask_id, synth.confidence_targets(M, 23).numpy(), O)
    am = O.head_stats(z_raw * alpha[:, None], d.mask_id)["argmax"]
    draft = _drafts(am, d.vocab, block, 24)
    draft[3] = d.mask_id                     # the mask token is never accepted
    draft[12] = d.vocab + 5                  # nor an id outside the vocabulary
    ref = _ref(d, hb, xh, alpha, draft)
    got = _run(d, head, x, alpha, draft, block, rule, 0.9, delta)
    lens = _check(got, ref, draft, rule, 0.9, delta, block)
    assert got["p_draft"][3] == 0.0 and got["p_draft"][12] == 0.0
    assert lens[0] <= 3 and lens[1] <= 3
    assert lens.max() > 0                   # some drafts do pass


@pytest.mark.parametrize("M,block,rule", [(33, 33, O.ACCEPT_EXACT), (72, 9, O.ACCEPT_THRESHOLD)])
def test_accept_clover_head(M, block, rule):
    """The 248,320-row head: one Clover block of 32 drafts (33 rows), and 8
    rounds of 8 drafts under the default threshold rule."""
    d = synth.CLOVER
    head = synth.make_head(d, 31, DEV)
    x = synth.make_x(d, M, 32, DEV)
    xh = x.cpu().numpy()
    hb = bits(head)
    z_raw = O.head_logits(xh, hb, d.rms_eps)
    alpha = calibrate_alpha(z_raw, d.mask_id, synth.confidence_targets(M, 33).numpy(), O)
    am = O.head_stats(z_raw * alpha[:, None], d.mask_id)["argmax"]
    draft = _drafts(am, d.vocab, block, 34, keep=0.85)
    ref = _ref(d, hb, xh, alpha, draft)
    got = _run(d, head, x, alpha, draft, block, rule, 0.9, 0.6)
    _check(got, ref, draft, rule, 0.9, 0.6, block)


def test_accept_form_agrees_with_unmask_form():
    """Both forms of the head produce bit-identical per-row statistics."""
    d = synth.TINY
    M = 40
    head = synth.make_head(d, 41, DEV)
    x = synth.make_x(d, M, 42, DEV)
    alpha = torch.linspace(0.5, 3.0, M, device=DEV)
    tokens, masked = synth.masked_block(d, M, DEV)
    u = clover.lmhead_unmask(d, head, x, tokens, masked, logit_scale=alpha, block=8)
    draft = torch.zeros(M, dtype=torch.int32, device=DEV)
    a = clover.lmhead_accept(d, head, x, draft, 8, clover.ACCEPT_EXACT, logit_scale=alpha)
    torch.cuda.synchronize()
    for k in ("argmax", "max_logit", "lse", "max_prob"):
        assert torch.equal(u[k], a[k]), k


def test_accept_drafts_equal_to_argmax_pass_every_rule():
    """Drafts copied from the head's own argmax pass the exact rule in full
    (r = block - 1 and the round is the argmax sequence), and the threshold
    rule with a small delta; boundary rows give the last token."""
    d = synth.TINY
    M, block = 32, 8
    head = synth.make_head(d, 51, DEV)
    x = synth.make_x(d, M, 52, DEV)
    first = clover.lmhead_accept(d, head, x, torch.zeros(M, dtype=torch.int32, device=DEV), block)
    draft = first["argmax"].clone()
    for rule, delta in ((clover.ACCEPT_EXACT, 0.6), (clover.ACCEPT_THRESHOLD, 1e-6)):
        out = clover.lmhead_accept(d, head, x, draft, block, rule, 0.9, delta)
        torch.cuda.synchronize()
        assert out["accept_len"].cpu().tolist() == [block - 1] * (M // block)
        assert torch.equal(out["tokens"], first["argmax"])


def test_accept_rejects_bad_arguments():
    d = synth.TINY
    head = synth.make_head(d, 61, DEV)
    x = synth.make_x(d, 18, 62, DEV)
    draft = torch.zeros(18, dtype=torch.int32, device=DEV)
    for kw in (dict(block=1), dict(block=4), dict(block=9, rule=2), dict(block=9, rule=1, delta=0.0),
               dict(block=9, rule=1, ratio=1.5)):
        block = kw.pop("block")
        with pytest.raises(clover.CloverError) as ei:
            clover.lmhead_accept(d, head, x, draft, block, **kw)
        assert ei.value.code == clover.ERR_INVALID_ARG
