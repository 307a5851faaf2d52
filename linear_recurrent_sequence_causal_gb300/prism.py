"""Thin Python binding of libprism.so (the C ABI in include/prism.h).

Argument marshalling only: every step of the mixer forward pass runs in the
library's CUDA kernels.  PyTorch supplies device memory and the stream.  If the
library has not been built (``__graft_entry__.build()`` or
``python -m linear_recurrent_sequence_causal_gb300.build``) every call raises;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PRISM_F32, PRISM_BF16 = 0, 1
PRISM_FLAG_NO_GELU = 1
PRISM_FLAG_VHIST_TOKEN_MAJOR = 2
PRISM_FLAG_NO_SEQ_SPLIT = 4
PRISM_FLAG_CHECK_WAIT_TIMEOUT = 8
ERRORS = {0: "PRISM_OK", 1: "PRISM_ERR_INVALID_ARG", 2: "PRISM_ERR_UNSUPPORTED",
          3: "PRISM_ERR_MISALIGNED", 4: "PRISM_ERR_WORKSPACE", 5: "PRISM_ERR_LAUNCH",
          6: "PRISM_ERR_CUDA", 7: "PRISM_ERR_SCRATCH_LIMIT"}
STATIC_SCRATCH_BYTES = 32 << 20
PRISM_HOST_MAX_PIECES = 16
EXPORTS = ("prism_workspace_bytes", "prism_workspace_layout", "prism_forward", "prism_prepare",
           "prism_scan", "prism_forward_static", "prism_strerror", "prism_forward_from",
           "prism_decode_step", "prism_backward_workspace_bytes", "prism_backward",
           "prism_device_status", "prism_host_plan", "prism_host_arena_bytes",
           "prism_forward_host", "prism_scan_segments", "prism_debug_bounds",
           "prism_debug_activation", "prism_static_status")
WS_REGIONS = ("status", "Kl", "Dl", "wblocks", "WQ", "QK", "U", "Oi", "N", "gC", "seg")


class PrismError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("conv_width", ctypes.c_int),
                ("L", ctypes.c_int), ("chunk", ctypes.c_int), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint)]


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def library_path() -> str:
    return _build.LIB


def load():
    """Load libprism.so (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            # PRISM_LIBRARY selects another build of the same library (the bounds-checked
            # debug build, build.build_debug())
            path = os.environ.get("PRISM_LIBRARY") or _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libprism.so not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            lib.prism_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
            lib.prism_workspace_bytes.restype = ctypes.c_size_t
            lib.prism_workspace_layout.argtypes = [ctypes.POINTER(Dims),
                                                   ctypes.POINTER(ctypes.c_size_t), ctypes.c_int]
            lib.prism_workspace_layout.restype = ctypes.c_int
            lib.prism_forward.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 13 + [ctypes.c_size_t, _vp]
            lib.prism_forward.restype = ctypes.c_int
            lib.prism_prepare.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 11 + [ctypes.c_size_t, _vp]
            lib.prism_prepare.restype = ctypes.c_int
            lib.prism_scan.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 7 + [ctypes.c_size_t] + [_vp] * 3
            lib.prism_scan.restype = ctypes.c_int
            lib.prism_forward_static.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 13
            lib.prism_forward_from.restype = ctypes.c_int
            lib.prism_forward_from.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 15 + [ctypes.c_size_t, _vp]
            lib.prism_decode_step.restype = ctypes.c_int
            lib.prism_decode_step.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 13
            lib.prism_forward_static.restype = ctypes.c_int
            lib.prism_backward_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
            lib.prism_backward_workspace_bytes.restype = ctypes.c_size_t
            lib.prism_backward.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 21 + [ctypes.c_size_t, _vp]
            lib.prism_backward.restype = ctypes.c_int
            lib.prism_device_status.argtypes = [ctypes.POINTER(Dims), _vp, ctypes.c_size_t,
                                                 ctypes.POINTER(ctypes.c_int), _vp]
            lib.prism_device_status.restype = ctypes.c_int
            lib.prism_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
            lib.prism_debug_bounds.restype = ctypes.c_int
            lib.prism_debug_activation.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong,
                                                    ctypes.c_void_p]
            lib.prism_debug_activation.restype = ctypes.c_int
            lib.prism_static_status.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
            lib.prism_static_status.restype = ctypes.c_int
            lib.prism_host_plan.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_size_t,
                                            ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
            lib.prism_host_plan.restype = ctypes.c_int
            lib.prism_host_arena_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_size_t]
            lib.prism_host_arena_bytes.restype = ctypes.c_size_t
            lib.prism_forward_host.argtypes = ([ctypes.POINTER(Dims)] + [_vp] * 12
                                               + [ctypes.c_int, ctypes.c_size_t, _vp, ctypes.c_size_t,
                                                  ctypes.POINTER(ctypes.c_void_p)])
            lib.prism_forward_host.restype = ctypes.c_int
            lib.prism_scan_segments.argtypes = [ctypes.POINTER(Dims)]
            lib.prism_scan_segments.restype = ctypes.c_int
            lib.prism_strerror.argtypes = [ctypes.c_int]
            lib.prism_strerror.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load().prism_strerror(code).decode()


def _check(code: int):
    if code != 0:
        raise PrismError(code, strerror(code))


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return PRISM_BF16
    if t == torch.float32:
        return PRISM_F32
    raise PrismError(1, f"unsupported I/O dtype {t}")


def make_dims(B, T, H, d_k, d_v, conv_width, L, chunk, dtype, no_gelu=False, flags=0) -> Dims:
    return Dims(B=B, T=T, H=H, d_k=d_k, d_v=d_v, conv_width=conv_width, L=L, chunk=chunk,
                dtype=_dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype),
                flags=(PRISM_FLAG_NO_GELU if no_gelu else 0) | flags)


def workspace_bytes(dims: Dims) -> int:
    return int(load().prism_workspace_bytes(ctypes.byref(dims)))


def scan_segments(dims: Dims) -> int:
    """Segments the scan cuts each sequence of these dims into (1: one serial chain)."""
    return int(load().prism_scan_segments(ctypes.byref(dims)))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise PrismError(1, "tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def workspace_layout(dims: Dims) -> dict:
    """Byte offsets of the workspace regions (None where absent)."""
    offs = (ctypes.c_size_t * len(WS_REGIONS))()
    _check(load().prism_workspace_layout(ctypes.byref(dims), offs, len(WS_REGIONS)))
    absent = (1 << (8 * ctypes.sizeof(ctypes.c_size_t))) - 1
    return {n: (None if offs[i] == absent else int(offs[i])) for i, n in enumerate(WS_REGIONS)}


def _dims_for(q, v, conv_w, L, chunk, no_gelu=False, flags=0) -> Dims:
    B, T, H, dk = q.shape
    return make_dims(B, T, H, dk, v.shape[-1], conv_w.shape[1], L, chunk, q.dtype, no_gelu, flags)


def alloc_workspace(dims: Dims, device) -> torch.Tensor:
    return torch.empty(max(workspace_bytes(dims), 1), dtype=torch.uint8, device=device)


def debug_bounds(clear: bool = True):
    """The debug build's word of out-of-bounds accesses (0: none; synchronises the
    device), or None when the loaded library is the normal build."""
    word = ctypes.c_int(-1)
    rc = load().prism_debug_bounds(ctypes.byref(word), 1 if clear else 0)
    if ERRORS.get(rc) == "PRISM_ERR_UNSUPPORTED":   # not the debug build
        return None
    _check(rc)
    return word.value


def debug_activation(x: torch.Tensor, stream=None) -> torch.Tensor:
    """GELU of the fp32 device tensor ``x`` as the bf16 prepare kernel evaluates it."""
    if x.dtype != torch.float32:
        raise PrismError(1, "x must be fp32")
    y = torch.empty_like(x)
    _check(load().prism_debug_activation(_ptr(x), _ptr(y), x.numel(), _stream_ptr(stream)))
    return y


def static_status(dims: Dims, stream=None) -> int:
    """The device status word of the last prism_forward_static call (0: every bounded
    wait completed).  Synchronises ``stream``."""
    word = ctypes.c_int(-1)
    _check(load().prism_static_status(ctypes.byref(dims), ctypes.byref(word), _stream_ptr(stream)))
    return word.value


def device_status(dims: Dims, workspace, stream=None) -> int:
    """The device status word a forward call left in ``workspace`` (0: every bounded wait
    completed).  Synchronises ``stream``."""
    word = ctypes.c_int(-1)
    _check(load().prism_device_status(ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                                      ctypes.byref(word), _stream_ptr(stream)))
    return word.value


def prism_forward(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, chunk, *, out=None,
                  final_state=None, seq_lens=None, workspace=None, stream=None,
                  no_gelu=False, want_state=True, flags=0):
    """The mixer forward pass on CUDA tensors laid out as in include/prism.h.

    Returns ``(out, final_state)`` (out is fp32); ``final_state`` is None when
    ``want_state`` is False and none was passed.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = _dims_for(q, v, conv_w, L, chunk, no_gelu, flags)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
    rc = load().prism_forward(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                              _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp), _ptr(wbeta),
                              _ptr(out), _ptr(final_state), _ptr(seq_lens), _ptr(workspace),
                              workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return out, final_state


def prism_forward_from(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, chunk, *,
                       initial_state=None, v_hist=None, out=None, final_state=None,
                       seq_lens=None, workspace=None, stream=None, no_gelu=False, want_state=True,
                       v_hist_token_major=False, flags=0):
    """prism_forward resuming from ``initial_state`` [B,H,dv,dk] fp32 and ``v_hist``
    [B,H,w,dv] (I/O dtype; the v rows of the w tokens before t = 0, oldest first), or
    [B,w,H,dv] (the layout of v) with ``v_hist_token_major``."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = _dims_for(q, v, conv_w, L, chunk, no_gelu,
                     (PRISM_FLAG_VHIST_TOKEN_MAJOR if v_hist_token_major else 0) | flags)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
    rc = load().prism_forward_from(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                   _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp), _ptr(wbeta),
                                   _ptr(initial_state), _ptr(v_hist), _ptr(out), _ptr(final_state),
                                   _ptr(seq_lens), _ptr(workspace), workspace.numel(),
                                   _stream_ptr(stream))
    _check(rc)
    return out, final_state


def prism_backward(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, d_out, *,
                   d_final_state=None, seq_lens=None, workspace=None, grads=None, stream=None,
                   no_gelu=False):
    """Gradients through prism_forward given ``d_out`` [B,T,H,dv] fp32 (and optionally
    ``d_final_state`` [B,H,dv,dk] fp32).  Returns a dict of fp32 CUDA tensors keyed q, k,
    v, log_alpha, beta, conv_w, Wk, Wp, wbeta (shapes of the inputs; Wk, Wp, wbeta are
    None when L = 0).  ``grads`` may pass preallocated outputs with the same keys."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = _dims_for(q, v, conv_w, L, 64, no_gelu)
    dev = q.device
    g = dict(grads) if grads else {}
    shapes = {"q": (B, T, H, dk), "k": (B, T, H, dk), "v": (B, T, H, dv), "log_alpha": (B, T, H),
              "beta": (B, T, H), "conv_w": tuple(conv_w.shape)}
    if L > 0:
        shapes.update(Wk=(H, L, dk, dv), Wp=(H, L, dv, dv), wbeta=(H, L, dv))
    for n, shp in shapes.items():
        if g.get(n) is None:
            g[n] = torch.empty(shp, dtype=torch.float32, device=dev)
    for n in ("Wk", "Wp", "wbeta"):
        g.setdefault(n, None)
    if workspace is None:
        nbytes = load().prism_backward_workspace_bytes(ctypes.byref(dims))
        if nbytes == 0:
            raise PrismError(2, "prism_backward_workspace_bytes rejected the dims")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rc = load().prism_backward(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                               _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp), _ptr(wbeta),
                               _ptr(d_out), _ptr(d_final_state), _ptr(g["q"]), _ptr(g["k"]),
                               _ptr(g["v"]), _ptr(g["log_alpha"]), _ptr(g["beta"]), _ptr(g["conv_w"]),
                               _ptr(g["Wk"]), _ptr(g["Wp"]), _ptr(g["wbeta"]), _ptr(seq_lens),
                               _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return g


def prism_decode_step(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, state, v_hist, *,
                      out=None, stream=None, no_gelu=False):
    """One token for every (b, h): q, k, v [B,H,d]; log_alpha, beta [B,H]; ``state``
    [B,H,dv,dk] fp32 and ``v_hist`` [B,H,w,dv] are updated in place.  Returns out
    [B,H,dv] fp32."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    dims = make_dims(B, 1, H, dk, dv, conv_w.shape[1], L, 16, q.dtype, no_gelu)
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    rc = load().prism_decode_step(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                  _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp), _ptr(wbeta),
                                  _ptr(state), _ptr(v_hist), _ptr(out), _stream_ptr(stream))
    _check(rc)
    return out


def v_history(v, w, end=None):
    """The v rows of the w tokens before ``end`` (default: the end), oldest first, as a
    contiguous [B,H,w,dv] tensor; rows before token 0 are zero."""
    B, T, H, dv = v.shape
    end = T if end is None else end
    hist = torch.zeros((B, H, w, dv), dtype=v.dtype, device=v.device)
    n = min(w, end)
    if n > 0:
        hist[:, :, w - n:] = v[:, end - n:end].permute(0, 2, 1, 3)
    return hist.contiguous()


def prism_forward_static(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, chunk, *, out=None,
                         final_state=None, seq_lens=None, stream=None, no_gelu=False,
                         want_state=True, flags=0):
    """prism_forward using the library's static device scratch (no workspace).

    For callers that cannot allocate device memory on their hot path; see
    include/prism.h for the size limit and the sharing rules.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = _dims_for(q, v, conv_w, L, chunk, no_gelu, flags)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    rc = load().prism_forward_static(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_alpha), _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp),
                                     _ptr(wbeta), _ptr(out), _ptr(final_state), _ptr(seq_lens),
                                     _stream_ptr(stream))
    _check(rc)
    return out, final_state


def prism_prepare(q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, L, chunk, workspace, *,
                  seq_lens=None, stream=None, no_gelu=False, flags=0):
    """State-independent stage into ``workspace`` (see include/prism.h)."""
    dims = _dims_for(q, v, conv_w, L, chunk, no_gelu, flags)
    rc = load().prism_prepare(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                              _ptr(beta), _ptr(conv_w), _ptr(Wk), _ptr(Wp), _ptr(wbeta),
                              _ptr(seq_lens), _ptr(workspace), workspace.numel(),
                              _stream_ptr(stream))
    _check(rc)
    return workspace


def prism_scan(q, k, v, log_alpha, beta, L, chunk, conv_width, workspace, *, out=None,
               final_state=None, seq_lens=None, stream=None, want_state=True, no_gelu=False,
               flags=0):
    """Serial stage from a prepared workspace; returns (out, final_state)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = make_dims(B, T, H, dk, dv, conv_width, L, chunk, q.dtype, no_gelu, flags)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    rc = load().prism_scan(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                           _ptr(beta), _ptr(seq_lens), _ptr(workspace), workspace.numel(),
                           _ptr(out), _ptr(final_state), _stream_ptr(stream))
    _check(rc)
    return out, final_state


def inputs_to_device(inp: dict, device="cuda") -> dict:
    """Copy an input dict (see ``inputs.generate``) to the device, contiguous."""
    return {k: (v.to(device).contiguous() if v is not None else None) for k, v in inp.items()}


def forward_inputs(inp: dict, L: int, chunk: int, **kw):
    """prism_forward on an input dict already on the device."""
    return prism_forward(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"],
                         inp["conv_w"], inp["Wk"], inp["Wp"], inp["wbeta"], L, chunk,
                         seq_lens=inp.get("seq_lens"), **kw)


def plan_pieces(dims: Dims, pieces=12, min_piece_bytes=8 << 20):
    """How prism_forward_host cuts the work for these dims: a list of (start, end) ranges of
    sequences when B > 1, or of chunk-aligned token ranges when B = 1 (each at least
    max(chunk, w) tokens so the next segment's history lies inside its predecessor), at
    most ``pieces`` of them and, when ``min_piece_bytes`` > 0, none moving fewer bytes
    than that."""
    n = ctypes.c_int(0)
    bounds = (ctypes.c_int * (pieces + 1))()
    _check(load().prism_host_plan(ctypes.byref(dims), pieces, min_piece_bytes, ctypes.byref(n), bounds))
    return [(bounds[i], bounds[i + 1]) for i in range(n.value)]


def host_arena_bytes(dims: Dims, pieces=12, min_piece_bytes=8 << 20) -> int:
    return int(load().prism_host_arena_bytes(ctypes.byref(dims), pieces, min_piece_bytes))


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise PrismError(1, "host buffers must be contiguous CPU tensors")
    return t.data_ptr()


class HostPipeline:
    """The forward pass from host (pinned) inputs to host outputs through prism_forward_host:
    the library cuts the work into pieces (groups of sequences when B > 1; token segments
    when B = 1, each resumed from the previous segment's final state and its last w v rows)
    and overlaps the copies in, the kernels and the copies out on three streams.  The device
    arena and the streams are kept across calls.
    """

    def __init__(self, shapes: dict, dtype, L, chunk, *, pieces=12, device="cuda", no_gelu=False,
                 min_piece_bytes=8 << 20):
        B, T, H, D = shapes["q"]
        self.dev = torch.device(device)
        self.dims = make_dims(B, T, H, D, D, shapes["conv_w"][1], L, chunk, dtype, no_gelu)
        self.max_pieces, self.min_piece_bytes = pieces, min_piece_bytes
        self.pieces = plan_pieces(self.dims, pieces, min_piece_bytes)
        nbytes = host_arena_bytes(self.dims, pieces, min_piece_bytes)
        if nbytes == 0:
            raise PrismError(2, "HostPipeline: unsupported dims")
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        self.streams = [torch.cuda.Stream(self.dev) for _ in range(3)]

    def h2d_bytes(self, host: dict) -> int:
        return sum(t.numel() * t.element_size() for n, t in host.items() if t is not None)

    def run(self, host: dict, host_out, host_fs, stream=None):
        """host: pinned CPU tensors keyed like ``inputs.generate``; host_out [B,T,H,D] fp32 and
        host_fs [B,H,D,D] fp32 pinned.  Ordered after ``stream`` (default: current) and
        finished before later work on it."""
        caller = stream or torch.cuda.current_stream(self.dev)
        if len(self.pieces) == 1:                  # one piece: everything on the caller's stream
            handles = (ctypes.c_void_p * 3)(*([caller.cuda_stream] * 3))
        else:
            for s in self.streams:
                s.wait_stream(caller)
            handles = (ctypes.c_void_p * 3)(*[s.cuda_stream for s in self.streams])
        with torch.cuda.device(self.dev):         # the library's events live on this device
            rc = load().prism_forward_host(
                ctypes.byref(self.dims), _host_ptr(host["q"]), _host_ptr(host["k"]), _host_ptr(host["v"]),
                _host_ptr(host["log_alpha"]), _host_ptr(host["beta"]), _host_ptr(host.get("conv_w")),
                _host_ptr(host.get("Wk")), _host_ptr(host.get("Wp")), _host_ptr(host.get("wbeta")),
                _host_ptr(host_out), _host_ptr(host_fs), _host_ptr(host.get("seq_lens")),
                self.max_pieces, self.min_piece_bytes, self.arena.data_ptr(), self.arena.numel(),
                handles)
        _check(rc)
        if len(self.pieces) > 1:
            caller.wait_stream(self.streams[2])
