"""CPU oracle for the PRISM mixer forward pass (fp64, token by token).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA path never
imports, links or runs anything here, and this module imports nothing from
the CUDA package.

The arithmetic lives in ``prism_oracle.c`` (plain C, fp64); this module builds
it with gcc and marshals numpy arrays into it.  See that file's header for the
passages of "Technical Summary: PRISM (Parallel Residual Iterative Sequence
Model)" each step follows.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(L = 0 against an independent Gated DeltaNet loop, the rank of the write,
the telescoping residual, brute-force products of explicit A_t for short
sequences, closed-form special cases and library routines for the ShortConv,
GELU and sigmoid).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "prism_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


class _Trace(ctypes.Structure):
    _fields_ = [(n, _dp) for n in ("u", "r1", "r_final", "kl", "pl", "delta", "betal", "dl", "Bt")]


class _Problem(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int) for n in ("B", "T", "H", "dk", "dv", "w", "L", "identity_act")]
                + [(n, _dp) for n in ("q", "k", "v", "log_alpha", "beta", "conv_w", "Wk", "Wp",
                                      "wbeta")]
                + [("seq_lens", _ip), ("out", _dp), ("final_state", _dp),
                   ("trace", ctypes.POINTER(_Trace)), ("initial_state", _dp), ("v_hist", _dp)])


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no target-specific flags)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(os.path.join(_HERE, f)) > os.path.getmtime(_LIB)
        for f in ("prism_oracle.c", "prism_oracle.h"))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC,
                        "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _open(path):
    lib = ctypes.CDLL(path)
    lib.prism_oracle_forward.argtypes = [ctypes.POINTER(_Problem), _ip, ctypes.c_int,
                                         ctypes.c_int]
    lib.prism_oracle_forward.restype = ctypes.c_int
    return lib


def _load(lib_path=None):
    """The built oracle, or (for tests that plant mistakes) another build of it."""
    global _lib
    if lib_path is not None:
        return _open(lib_path)
    with _lock:
        if _lib is None:
            build()
            _lib = _open(_LIB)
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(_dp) if a is not None else None


def forward(inp: dict, *, L: int | None = None, trace: bool = False, bh_items=None,
            threads: int | None = None, identity_act: bool = False, lib_path=None,
            initial_state=None, v_hist=None):
    """Run the oracle on one input dict (see ``inputs.generate``).

    Returns ``(out [B,T,H,dv], final_state [B,H,dv,dk], trace_dict_or_None)``
    as fp64 numpy arrays.  ``bh_items`` restricts the work to a list of (b, h)
    pairs; rows of the other pairs are left as NaN.  ``initial_state``
    [B,H,dv,dk] and ``v_hist`` [B,H,w,dv] (the v rows of the w tokens before
    t = 0, oldest first) resume a sequence; None means zeros.
    """
    lib = _load(lib_path)
    q, k, v = _f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"])
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    la, be = _f64(inp["log_alpha"]), _f64(inp["beta"])
    conv_w = _f64(inp["conv_w"])
    Wk, Wp, wb = _f64(inp["Wk"]), _f64(inp["Wp"]), _f64(inp["wbeta"])
    if L is None:
        L = Wk.shape[1]
    Wk, Wp, wb = (np.ascontiguousarray(a[:, :L]) for a in (Wk, Wp, wb))
    w = conv_w.shape[1]
    sl = inp.get("seq_lens")
    sl = None if sl is None else np.ascontiguousarray(np.asarray(sl, dtype=np.int32))
    assert k.shape == q.shape and v.shape[:3] == (B, T, H) and la.shape == (B, T, H)
    assert conv_w.shape == (H, w, dv) and Wk.shape == (H, L, dk, dv) and Wp.shape == (H, L, dv, dv)
    s0 = _f64(initial_state)
    vh = _f64(v_hist)
    assert s0 is None or s0.shape == (B, H, dv, dk)
    assert vh is None or vh.shape == (B, H, w, dv)
    out = np.full((B, T, H, dv), np.nan)
    fs = np.full((B, H, dv, dk), np.nan)
    tr_arrays = None
    tr = None
    if trace:
        tr_arrays = dict(
            u=np.full((B, T, H, dv), np.nan), r1=np.full((B, T, H, dv), np.nan),
            r_final=np.full((B, T, H, dv), np.nan), kl=np.full((B, T, H, L, dk), np.nan),
            pl=np.full((B, T, H, L, dv), np.nan), delta=np.full((B, T, H, L, dv), np.nan),
            betal=np.full((B, T, H, L), np.nan), dl=np.full((B, T, H, L, dv), np.nan),
            Bt=np.full((B, T, H, dv, dk), np.nan) if B * T * H * dv * dk <= 1 << 24 else None)
        tr = _Trace(**{n: _ptr(a) for n, a in tr_arrays.items()})
    P = _Problem(B=B, T=T, H=H, dk=dk, dv=dv, w=w, L=L, identity_act=int(identity_act),
                 q=_ptr(q), k=_ptr(k), v=_ptr(v), log_alpha=_ptr(la), beta=_ptr(be),
                 conv_w=_ptr(conv_w), Wk=_ptr(Wk), Wp=_ptr(Wp), wbeta=_ptr(wb),
                 seq_lens=sl.ctypes.data_as(_ip) if sl is not None else None,
                 out=_ptr(out), final_state=_ptr(fs),
                 trace=ctypes.pointer(tr) if tr is not None else None,
                 initial_state=_ptr(s0), v_hist=_ptr(vh))
    items = None
    n_items = 0
    if bh_items is not None:
        items = np.ascontiguousarray(np.asarray([b * H + h for b, h in bh_items], dtype=np.int32))
        n_items = len(items)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.prism_oracle_forward(ctypes.byref(P), items.ctypes.data_as(_ip) if items is not None
                                  else None, n_items, int(threads))
    if rc != 0:
        raise RuntimeError(f"prism_oracle_forward failed with code {rc}")
    return out, fs, tr_arrays
