"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/clover.h declares, and rejects bad arguments on the host (no compute
calls are made here)."""
import ctypes
import os
import re
import subprocess

import pytest

from block_diffusion_moe_gb300 import build as B
from block_diffusion_moe_gb300 import clover as C
from block_diffusion_moe_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clover.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(clover_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", C.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (clover_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(C.EXPORTS) == set(names)


def test_version(lib):
    assert lib.clover_version() == 100


def _dims(**kw):
    d = synth.CLOVER
    base = dict(hidden=d.hidden, n_experts=d.n_experts, top_k=d.top_k, d_ff=d.d_ff, vocab=d.vocab,
                mask_id=d.mask_id, rms_eps=d.rms_eps, coreset_top_p=0.0)
    base.update(kw)
    return C.Dims(**base)


def test_workspace_sizes(lib):
    d = _dims()
    m32 = lib.clover_moe_workspace_bytes(ctypes.byref(d), 32)
    m256 = lib.clover_moe_workspace_bytes(ctypes.byref(d), 256)
    assert 0 < m32 < m256
    # the gathered inputs, SwiGLU rows and expert outputs dominate:
    # (M*K + M) rows of H bf16 + F bf16 + H fp32
    R = 32 * 8 + 32
    assert m32 >= R * (2048 * 2 + 512 * 2 + 2048 * 4)
    h = lib.clover_head_workspace_bytes(ctypes.byref(d), 32)
    dn = lib.clover_denoise_workspace_bytes(ctypes.byref(d), 32)
    assert dn >= m32 + h - 2 * 256
    assert lib.clover_moe_workspace_bytes(ctypes.byref(d), 0) == 0
    assert lib.clover_moe_workspace_bytes(ctypes.byref(d), 1025) == 0
    assert lib.clover_moe_workspace_bytes(ctypes.byref(d), 1024) > m256
    assert lib.clover_moe_workspace_bytes(None, 32) == 0
    # the residual stream the denoise step leaves: an fp32 [M][H] block that
    # lies inside the workspace for every M up to the size it was built for
    for m in (1, 32):
        o = lib.clover_denoise_hidden_offset(ctypes.byref(d), m)
        assert o > 0 and o % 16 == 0
        assert o + m * 2048 * 4 <= lib.clover_denoise_workspace_bytes(ctypes.byref(d), m)
    assert lib.clover_denoise_hidden_offset(ctypes.byref(d), 0) == 0
    assert lib.clover_denoise_hidden_offset(None, 32) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=2000), C.ERR_UNSUPPORTED_SHAPE),
    (dict(d_ff=500), C.ERR_UNSUPPORTED_SHAPE),
    (dict(n_experts=300), C.ERR_UNSUPPORTED_SHAPE),
    (dict(top_k=33), C.ERR_UNSUPPORTED_SHAPE),
    (dict(mask_id=248320), C.ERR_INVALID_ARG),
    (dict(hidden=0), C.ERR_INVALID_ARG),
    (dict(coreset_top_p=1.5), C.ERR_INVALID_ARG),
])
def test_bad_dims_rejected_on_host(lib, kw, code):
    d = _dims(**kw)
    lay = C.MoeLayer(0x10000, None, 0x20000, 0x30000, 0x40000, 0x50000)
    rc = lib.clover_moe_block_step(ctypes.byref(d), ctypes.byref(lay), 0x60000, 0x60000, None, None, 32,
                                   0x100000, 1 << 30, None)
    assert rc == code
    assert C.last_error()


def test_bad_args_rejected_on_host(lib):
    d = _dims()
    lay = C.MoeLayer(0x10000, None, 0x20000, 0x30000, 0x40000, 0x50000)
    f = lib.clover_moe_block_step
    assert f(ctypes.byref(d), ctypes.byref(lay), 0x60000, 0x60000, None, None, 0, 0x100000, 1 << 30, None) \
        == C.ERR_UNSUPPORTED_SHAPE
    assert f(ctypes.byref(d), ctypes.byref(lay), None, 0x60000, None, None, 32, 0x100000, 1 << 30, None) \
        == C.ERR_INVALID_ARG
    assert f(ctypes.byref(d), ctypes.byref(lay), 0x60004, 0x60004, None, None, 32, 0x100000, 1 << 30, None) \
        == C.ERR_INVALID_ARG
    # partial overlap of x_in and x_out
    assert f(ctypes.byref(d), ctypes.byref(lay), 0x60000, 0x60010, None, None, 32, 0x100000, 1 << 30, None) \
        == C.ERR_INVALID_ARG
    need = lib.clover_moe_workspace_bytes(ctypes.byref(d), 32)
    assert f(ctypes.byref(d), ctypes.byref(lay), 0x60000, 0x60000, None, None, 32, 0x100000, need - 1, None) \
        == C.ERR_WORKSPACE_TOO_SMALL
    assert "needs" in C.last_error()
    assert f(ctypes.byref(d), ctypes.byref(lay), 0x60000, 0x60000, None, None, 32, 0x100010, need, None) \
        == C.ERR_INVALID_ARG
    bad = C.MoeLayer(0x10000, None, None, 0x30000, 0x40000, 0x50000)
    assert f(ctypes.byref(d), ctypes.byref(bad), 0x60000, 0x60000, None, None, 32, 0x100000, need, None) \
        == C.ERR_INVALID_ARG


def test_head_and_denoise_arg_checks(lib):
    d = _dims()
    need = lib.clover_head_workspace_bytes(ctypes.byref(d), 32)
    f = lib.clover_lmhead_unmask
    args = [ctypes.byref(d), 0x10000, 0x20000, None, 0.95, 32, 0x30000, 0x40000, None, None, None, None, None, 32,
            0x100000, need, None]
    a = list(args)
    a[5] = 0
    assert f(*a) == C.ERR_INVALID_ARG          # block < 1
    a = list(args)
    a[4] = float("nan")
    assert f(*a) == C.ERR_INVALID_ARG          # NaN threshold
    a = list(args)
    a[15] = need - 1
    assert f(*a) == C.ERR_WORKSPACE_TOO_SMALL
    lay = (C.MoeLayer * 1)(C.MoeLayer(0x10000, None, 0x20000, 0x30000, 0x40000, 0x50000))
    dn = lib.clover_denoise_workspace_bytes(ctypes.byref(d), 32)
    g = lib.clover_denoise_step
    # block must divide the number of positions
    assert g(ctypes.byref(d), lay, 1, 0x1000, 0x2000, 0x3000, None, 0.95, 5, 0x4000, 0x5000, 32, 0x100000, dn,
             None) == C.ERR_INVALID_ARG
    steps = ctypes.c_int32(7)
    assert lib.clover_denoise_block(ctypes.byref(d), lay, 1, 0x1000, 0x2000, 0x3000, None, 0.95, 32, 0x4000,
                                    0x5000, 32, -1, ctypes.byref(steps), 0x100000, dn, None) == C.ERR_INVALID_ARG
    assert steps.value == 0


def test_last_error_truncates(lib):
    d = _dims(hidden=2000)
    lib.clover_moe_workspace_bytes(ctypes.byref(d), 32)
    n = lib.clover_last_error(None, 0)
    assert n > 10
    buf = ctypes.create_string_buffer(8)
    lib.clover_last_error(buf, 8)
    assert len(buf.value) == 7


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(C, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(C, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        C.lib()


def test_accept_arg_checks(lib):
    d = _dims()
    need = lib.clover_accept_workspace_bytes(ctypes.byref(d), 33)
    assert need > lib.clover_head_workspace_bytes(ctypes.byref(d), 33)
    assert lib.clover_accept_workspace_bytes(ctypes.byref(d), 0) == 0
    assert lib.clover_accept_workspace_bytes(ctypes.byref(d), 1025) == 0
    f = lib.clover_lmhead_accept
    #      dims          head_w   x        scale draft   rule ratio delta block
    base = [ctypes.byref(d), 0x10000, 0x20000, None, 0x30000, 1, 0.9, 0.6, 33,
            None, None, None, None, None, None, 0x40000, 0x50000, 33, 0x100000, need, None]

    def call(**kw):
        a = list(base)
        pos = {"draft": 4, "rule": 5, "ratio": 6, "delta": 7, "block": 8, "accept_len": 15, "M": 17, "ws_bytes": 19}
        for k, v in kw.items():
            a[pos[k]] = v
        return f(*a)

    assert call(block=1) == C.ERR_INVALID_ARG                  # no draft row
    assert call(block=10) == C.ERR_INVALID_ARG                 # does not divide M
    assert call(rule=3) == C.ERR_INVALID_ARG
    assert call(delta=0.0) == C.ERR_INVALID_ARG
    assert call(ratio=1.5) == C.ERR_INVALID_ARG
    assert call(delta=float("inf")) == C.ERR_INVALID_ARG
    assert call(draft=None) == C.ERR_INVALID_ARG
    assert call(accept_len=None) == C.ERR_INVALID_ARG
    assert call(M=1100, block=50) == C.ERR_UNSUPPORTED_SHAPE
    assert call(ws_bytes=need - 1) == C.ERR_WORKSPACE_TOO_SMALL
