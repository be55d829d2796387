"""The allocation-free head + unmask entry point.

clover_lmhead_unmask_static exists for callers that cannot allocate device
memory (a plug-in inside an application that owns all GPU memory,
latency-critical loops that must not wait on an allocation): its scratch is a
fixed 1 MiB array inside the library. These checks call it through the C ABI,
twice in a row, and compare each result with the regular workspace-based
clover_lmhead_unmask on the same inputs: the two run the same kernels in the
same order, so every output must be bit-identical. The status of a static
call, which has no workspace, is read back through
clover_lmhead_unmask_static_status. This file is collected last on purpose."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from block_diffusion_moe_gb300 import clover, synth

DEV = "cuda"


def _call_static(d, head, x, tokens, masked, alpha, block):
    M = x.shape[0]
    out = {"argmax": torch.empty(M, dtype=torch.int32, device=DEV),
           "max_logit": torch.empty(M, dtype=torch.float32, device=DEV),
           "lse": torch.empty(M, dtype=torch.float32, device=DEV),
           "max_prob": torch.empty(M, dtype=torch.float32, device=DEV),
           "n_committed": torch.zeros(1, dtype=torch.int32, device=DEV)}
    dims = clover.make_dims(d)
    p = clover._ptr
    rc = clover.lib().clover_lmhead_unmask_static(
        ctypes.byref(dims), p(head), p(x), p(alpha), 0.95, block, p(tokens), p(masked), p(out["argmax"]),
        p(out["max_logit"]), p(out["lse"]), p(out["max_prob"]), p(out["n_committed"]), M, clover._stream())
    assert rc == clover.OK, clover.last_error()
    return out


def _same(a, b, tokens_a, tokens_b, masked_a, masked_b):
    for k in ("argmax", "n_committed", "max_logit", "lse", "max_prob"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(tokens_a, tokens_b)
    assert torch.equal(masked_a, masked_b)


def _static_status():
    return clover.lib().clover_lmhead_unmask_static_status(clover._stream())


@pytest.mark.gpu
@pytest.mark.parametrize("hidden,vocab,M", [(256, 1024, 37), (2048, 4096, 32), (2048, 1000, 102)])
def test_static_scratch_matches_workspace_call_twice(hidden, vocab, M):
    d = dataclasses.replace(synth.TINY, hidden=hidden, vocab=vocab, mask_id=vocab - 1)
    head = synth.make_head(d, 21, DEV)
    alpha_np = np.linspace(1.0, 40.0, M).astype(np.float32)
    alpha = torch.from_numpy(alpha_np).to(DEV)
    for call in range(2):
        x = synth.make_x(d, M, 30 + call, DEV)
        t_ref, m_ref = synth.masked_block(d, M, DEV)
        m_ref[::4] = 0
        t_ref[::4] = 7            # committed slots hold a vocabulary id
        t_static, m_static = t_ref.clone(), m_ref.clone()
        ref = clover.lmhead_unmask(d, head, x, t_ref, m_ref, logit_scale=alpha, block=d.block)
        got = _call_static(d, head, x, t_static, m_static, alpha, d.block)
        assert _static_status() == clover.OK, clover.last_error()
        _same(got, ref, t_static, t_ref, m_static, m_ref)
        assert int(got["n_committed"][0]) >= 1


@pytest.mark.gpu
def test_static_status_reports_and_clears():
    """A committed slot holding a token id outside the vocabulary is input
    the head reports through the status word. The static call has no
    workspace, so the status comes back through the static status query,
    which clears it; the next static call then runs clean and matches the
    workspace call bit for bit."""
    d = dataclasses.replace(synth.TINY, hidden=256, vocab=1024, mask_id=1023)
    M = 16
    head = synth.make_head(d, 22, DEV)
    x = synth.make_x(d, M, 40, DEV)
    tokens, masked = synth.masked_block(d, M, DEV)
    masked[3] = 0
    tokens[3] = d.vocab + 5
    _call_static(d, head, x, tokens, masked, None, d.block)
    rc = _static_status()
    assert rc == clover.ERR_DEVICE_TIMEOUT
    assert "token id out of range" in clover.last_error()
    assert _static_status() == clover.OK           # cleared by the query
    t_ref, m_ref = synth.masked_block(d, M, DEV)
    t_static, m_static = t_ref.clone(), m_ref.clone()
    ref = clover.lmhead_unmask(d, head, x, t_ref, m_ref, block=d.block)
    got = _call_static(d, head, x, t_static, m_static, None, d.block)
    assert _static_status() == clover.OK, clover.last_error()
    _same(got, ref, t_static, t_ref, m_static, m_ref)


@pytest.mark.gpu
def test_static_scratch_rejects_sizes_beyond_its_capacity():
    d = synth.CLOVER
    dims = clover.make_dims(d)
    # 103 positions at hidden 2,048 need more than the 1 MiB array holds
    assert clover.head_workspace_bytes(d, 103) > (1 << 20) >= clover.head_workspace_bytes(d, 102)
    rc = clover.lib().clover_lmhead_unmask_static(ctypes.byref(dims), 0x10000, 0x20000, None, 0.95, 32, 0x30000,
                                                  0x40000, None, None, None, None, None, 103, None)
    assert rc == clover.ERR_WORKSPACE_TOO_SMALL
    assert "static scratch" in clover.last_error()


def test_static_call_checks_arguments_before_any_cuda_call():
    """Argument errors come back from the host checks alone (this runs
    without a GPU): nothing is looked up or enqueued for a rejected call."""
    from block_diffusion_moe_gb300 import build as B
    B.build()
    d = synth.CLOVER
    dims = clover.make_dims(d)
    f = clover.lib().clover_lmhead_unmask_static
    assert f(ctypes.byref(dims), None, 0x20000, None, 0.95, 32, 0x30000, 0x40000, None, None, None, None, None,
             32, None) == clover.ERR_INVALID_ARG
    assert f(ctypes.byref(dims), 0x10000, 0x20000, None, float("nan"), 32, 0x30000, 0x40000, None, None, None,
             None, None, 32, None) == clover.ERR_INVALID_ARG
    assert f(ctypes.byref(dims), 0x10000, 0x20000, None, 0.95, 0, 0x30000, 0x40000, None, None, None, None, None,
             32, None) == clover.ERR_INVALID_ARG
    assert f(ctypes.byref(dims), 0x10000, 0x20000, None, 0.95, 32, 0x30000, 0x40000, None, None, None, None, None,
             1100, None) == clover.ERR_UNSUPPORTED_SHAPE
    assert f(ctypes.byref(dims), 0x10000, 0x20000, None, 0.95, 32, 0x30000, 0x40000, None, None, None, None, None,
             103, None) == clover.ERR_WORKSPACE_TOO_SMALL
