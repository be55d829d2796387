"""ctypes binding of libclover (include/clover.h).

Argument marshalling only: every step of the denoising path runs in the CUDA
library. PyTorch supplies device memory and the current stream. There is no
CPU or PyTorch fallback: if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import synth

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libclover.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_WORKSPACE_TOO_SMALL = -2
ERR_CUDA = -3
ERR_NOT_CONVERGED = -4
ERR_UNSUPPORTED_SHAPE = -5
ERR_DEVICE_TIMEOUT = -6


class CloverError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"clover error {code}: {msg}")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("vocab", ctypes.c_int32), ("mask_id", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("coreset_top_p", ctypes.c_float)]


class MoeLayer(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("gate_up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("sh_gate_up", ctypes.c_void_p), ("sh_down", ctypes.c_void_p),
                ("gate_up_q", ctypes.c_void_p), ("gate_up_s", ctypes.c_void_p), ("down_q", ctypes.c_void_p),
                ("down_s", ctypes.c_void_p), ("sh_gate_up_q", ctypes.c_void_p), ("sh_gate_up_s", ctypes.c_void_p),
                ("sh_down_q", ctypes.c_void_p), ("sh_down_s", ctypes.c_void_p)]


EXPORTS = {
    "clover_moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int32]),
    "clover_moe_block_step": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(MoeLayer), ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clover_head_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int32]),
    "clover_lmhead_unmask": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_float, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.c_void_p]),
    "clover_lmhead_unmask_static": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_float, ctypes.c_int32, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int32, ctypes.c_void_p]),
    "clover_lmhead_unmask_static_status": (ctypes.c_int, [ctypes.c_void_p]),
    "clover_quantize_q4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "clover_accept_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int32]),
    "clover_lmhead_accept": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.c_void_p]),
    "clover_denoise_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int32]),
    "clover_denoise_hidden_offset": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int32]),
    "clover_denoise_step": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(MoeLayer), ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_float, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clover_denoise_block": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(MoeLayer), ctypes.c_int32,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_float, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clover_workspace_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clover_profile_expert_events": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]),
    "clover_last_error": (ctypes.c_int32, [ctypes.c_char_p, ctypes.c_size_t]),
    "clover_version": (ctypes.c_int32, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libclover.so (built by __graft_entry__.build()). Raises if it is
    missing: there is no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libclover.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().clover_last_error(buf, 512)
    return buf.value.decode()


def _check(rc: int):
    if rc != OK:
        raise CloverError(rc, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_dims(d: synth.Dims, coreset_top_p: float = 0.0) -> Dims:
    return Dims(d.hidden, d.n_experts, d.top_k, d.d_ff, d.vocab, d.mask_id, d.rms_eps, coreset_top_p)


class Q4Layer:
    """A layer whose expert weights are in the low-bit format
    (clover_quantize_q4): codes uint8 and scales int16 (bf16 bits), device
    tensors; the router stays bf16."""

    def __init__(self, router_w, router_bias, gate_up_q, gate_up_s, down_q, down_s, sh_gate_up_q, sh_gate_up_s,
                 sh_down_q, sh_down_s):
        self.router_w, self.router_bias = router_w, router_bias
        self.gate_up_q, self.gate_up_s, self.down_q, self.down_s = gate_up_q, gate_up_s, down_q, down_s
        self.sh_gate_up_q, self.sh_gate_up_s, self.sh_down_q, self.sh_down_s = (sh_gate_up_q, sh_gate_up_s,
                                                                                sh_down_q, sh_down_s)


def quantize_q4(w, stream=None):
    """bf16 [n_mats][rows][cols] (or [rows][cols]) -> (codes uint8
    [..][rows][cols/2], scales int16 [..][cols/64][rows]) on the device."""
    assert w.is_cuda and w.dtype == torch.bfloat16 and w.is_contiguous()
    shape = tuple(w.shape)
    w3 = w.view(1, *shape) if w.dim() == 2 else w
    n, rows, cols = w3.shape
    q = torch.empty((n, rows, cols // 2), dtype=torch.uint8, device=w.device)
    sc = torch.empty((n, cols // 64, rows), dtype=torch.int16, device=w.device)
    _check(lib().clover_quantize_q4(_ptr(w3), n, rows, cols, _ptr(q), _ptr(sc), _stream(stream)))
    if w.dim() == 2:
        return q[0], sc[0]
    return q, sc


def quantize_layer_q4(L: synth.Layer, stream=None) -> Q4Layer:
    gq, gs = quantize_q4(L.gate_up, stream)
    dq, ds = quantize_q4(L.down, stream)
    sgq, sgs = quantize_q4(L.sh_gate_up, stream)
    sdq, sds = quantize_q4(L.sh_down, stream)
    return Q4Layer(L.router_w, L.router_bias, gq, gs, dq, ds, sgq, sgs, sdq, sds)


def make_layer(L) -> MoeLayer:
    if L.router_bias is not None:
        assert L.router_bias.is_cuda and L.router_bias.dtype == torch.float32
    bias = None if L.router_bias is None else L.router_bias.data_ptr()
    if isinstance(L, Q4Layer):
        ts = (L.gate_up_q, L.gate_up_s, L.down_q, L.down_s, L.sh_gate_up_q, L.sh_gate_up_s, L.sh_down_q, L.sh_down_s)
        for t in ts:
            assert t.is_cuda and t.is_contiguous()
        return MoeLayer(L.router_w.data_ptr(), bias, None, None, None, None, *[t.data_ptr() for t in ts])
    for t in (L.router_w, L.gate_up, L.down, L.sh_gate_up, L.sh_down):
        assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    return MoeLayer(L.router_w.data_ptr(), bias, L.gate_up.data_ptr(), L.down.data_ptr(), L.sh_gate_up.data_ptr(),
                    L.sh_down.data_ptr())


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled, 256-byte aligned device workspace (torch allocations are)."""
    if nbytes <= 0:
        raise CloverError(ERR_UNSUPPORTED_SHAPE, last_error())
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def moe_workspace_bytes(d: synth.Dims, max_tokens: int) -> int:
    return lib().clover_moe_workspace_bytes(ctypes.byref(make_dims(d)), max_tokens)


def head_workspace_bytes(d: synth.Dims, max_tokens: int) -> int:
    return lib().clover_head_workspace_bytes(ctypes.byref(make_dims(d)), max_tokens)


def denoise_workspace_bytes(d: synth.Dims, max_tokens: int) -> int:
    return lib().clover_denoise_workspace_bytes(ctypes.byref(make_dims(d)), max_tokens)


def denoise_hidden(d: synth.Dims, ws: torch.Tensor, M: int) -> torch.Tensor:
    """The fp32 [M][H] residual stream the last denoise step left in `ws`
    (a view into the workspace)."""
    o = lib().clover_denoise_hidden_offset(ctypes.byref(make_dims(d)), M)
    if o == 0:
        raise CloverError(ERR_INVALID_ARG, last_error())
    return ws[o:o + M * d.hidden * 4].view(torch.float32).view(M, d.hidden)


def moe_block_step(d: synth.Dims, layer: synth.Layer, x_in: torch.Tensor, x_out: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None, with_topk: bool = True, stream=None, coreset_top_p: float = 0.0):
    M = x_in.shape[0]
    if x_out is None:
        x_out = torch.empty_like(x_in)
    if ws is None:
        ws = workspace(moe_workspace_bytes(d, M), x_in.device)
    idx = torch.empty((M, d.top_k), dtype=torch.int32, device=x_in.device) if with_topk else None
    w = torch.empty((M, d.top_k), dtype=torch.float32, device=x_in.device) if with_topk else None
    dims = make_dims(d, coreset_top_p)
    lay = make_layer(layer)
    _check(lib().clover_moe_block_step(ctypes.byref(dims), ctypes.byref(lay), _ptr(x_in), _ptr(x_out), _ptr(idx),
                                       _ptr(w), M, _ptr(ws), ws.numel(), _stream(stream)))
    return x_out, idx, w


def lmhead_unmask(d: synth.Dims, head_w, x, tokens, masked, logit_scale=None, threshold: float = 0.95,
                  block: int = 32, ws=None, stream=None, out=None) -> dict:
    """Head statistics + unmask over M = x.shape[0] positions. `out` (a dict
    this function returned before, for the same M) is reused; the library
    writes every entry, including the committed count."""
    M = x.shape[0]
    dev = x.device
    if ws is None:
        ws = workspace(head_workspace_bytes(d, M), dev)
    if out is None:
        out = {"argmax": torch.empty(M, dtype=torch.int32, device=dev),
               "max_logit": torch.empty(M, dtype=torch.float32, device=dev),
               "lse": torch.empty(M, dtype=torch.float32, device=dev),
               "max_prob": torch.empty(M, dtype=torch.float32, device=dev),
               "n_committed": (torch.empty if M > 0 else torch.zeros)(1, dtype=torch.int32, device=dev)}
    dims = make_dims(d)
    _check(lib().clover_lmhead_unmask(ctypes.byref(dims), _ptr(head_w), _ptr(x), _ptr(logit_scale), threshold, block,
                                      _ptr(tokens), _ptr(masked), _ptr(out["argmax"]), _ptr(out["max_logit"]),
                                      _ptr(out["lse"]), _ptr(out["max_prob"]), _ptr(out["n_committed"]), M,
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return out


ACCEPT_EXACT = 0
ACCEPT_THRESHOLD = 1


def accept_workspace_bytes(d: synth.Dims, max_rows: int) -> int:
    return lib().clover_accept_workspace_bytes(ctypes.byref(make_dims(d)), max_rows)


def lmhead_accept(d: synth.Dims, head_w, x, draft, block: int, rule: int = ACCEPT_EXACT, ratio: float = 0.9,
                  delta: float = 0.6, logit_scale=None, ws=None, stream=None, out=None) -> dict:
    """Verify-pass head + accept test over M = x.shape[0] rows in blocks of
    `block` rows (block - 1 drafts + the boundary row). `out` (a dict this
    function returned before, for the same M and block) is reused."""
    M = x.shape[0]
    dev = x.device
    if ws is None:
        ws = workspace(accept_workspace_bytes(d, M), dev)
    if out is None:
        f32 = lambda: torch.empty(M, dtype=torch.float32, device=dev)
        out = {"argmax": torch.empty(M, dtype=torch.int32, device=dev), "max_logit": f32(), "lse": f32(),
               "max_prob": f32(), "entropy": f32(), "p_draft": f32(),
               "accept_len": torch.empty(max(1, M // max(block, 1)), dtype=torch.int32, device=dev),
               "tokens": torch.empty(M, dtype=torch.int32, device=dev)}
    dims = make_dims(d)
    _check(lib().clover_lmhead_accept(ctypes.byref(dims), _ptr(head_w), _ptr(x), _ptr(logit_scale), _ptr(draft),
                                      rule, ratio, delta, block, _ptr(out["argmax"]), _ptr(out["max_logit"]),
                                      _ptr(out["lse"]), _ptr(out["max_prob"]), _ptr(out["entropy"]),
                                      _ptr(out["p_draft"]), _ptr(out["accept_len"]), _ptr(out["tokens"]), M,
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return out


class Model:
    """Device-resident weights of a stack of MoE sublayers plus embedding and
    head, with the ctypes layer array the denoise entry points take."""

    def __init__(self, d: synth.Dims, layers, embed, head_w, coreset_top_p: float = 0.0):
        self.d = d
        self.layers = list(layers)
        self.embed = embed
        self.head_w = head_w
        self.c_layers = (MoeLayer * max(1, len(self.layers)))(*[make_layer(L) for L in self.layers])
        self.c_dims = make_dims(d, coreset_top_p)


def denoise_step(m: Model, ctx, tokens, masked, logit_scale=None, threshold: float = 0.95, block: int = 32,
                 ws=None, stream=None):
    M = tokens.shape[0]
    if ws is None:
        ws = workspace(denoise_workspace_bytes(m.d, M), tokens.device)
    _check(lib().clover_denoise_step(ctypes.byref(m.c_dims), m.c_layers, len(m.layers), _ptr(m.embed), _ptr(ctx),
                                     _ptr(m.head_w), _ptr(logit_scale), threshold, block, _ptr(tokens),
                                     _ptr(masked), M, _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def denoise_block(m: Model, ctx, tokens, masked, logit_scale=None, threshold: float = 0.95, block: int = 32,
                  max_steps: int = 32, ws=None, stream=None) -> int:
    M = tokens.shape[0]
    if ws is None:
        ws = workspace(denoise_workspace_bytes(m.d, M), tokens.device)
    steps = ctypes.c_int32(0)
    _check(lib().clover_denoise_block(ctypes.byref(m.c_dims), m.c_layers, len(m.layers), _ptr(m.embed), _ptr(ctx),
                                      _ptr(m.head_w), _ptr(logit_scale), threshold, block, _ptr(tokens),
                                      _ptr(masked), M, max_steps, ctypes.byref(steps), _ptr(ws), ws.numel(),
                                      _stream(stream)))
    return steps.value


def workspace_status(ws: torch.Tensor, stream=None):
    _check(lib().clover_workspace_status(_ptr(ws), ws.numel(), _stream(stream)))
