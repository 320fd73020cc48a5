"""CPU oracle for the Mamba2 SSD scan and its gradient -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it: the two share no code.

Three independent statements of the same mathematics live here:

* ``ssd_oracle.c`` (driven by :func:`fwd` / :func:`bwd`): the token-serial
  fp64 recurrence and its hand-derived reverse sweep.  This is *the* oracle.
* :mod:`oracle.chunked`: the chunked (state-space-duality) form in fp64 numpy,
  exposing every intermediate of the chunked algorithm.
* :mod:`oracle.quadratic`: the materialised quadratic form, differentiated by
  torch autograd in fp64 on the CPU.

The subject is the Mamba2 SSD forward/backward pair that "Deterministic bwd
kernel for mamba2" (Mamba PR #827) makes deterministic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_ssd_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle in-tree with gcc (plain IEEE fp64, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.ssd_oracle_fwd.argtypes = [i64] * 7 + [vp] * 8 + [i64, vp, vp, ci]
            lib.ssd_oracle_fwd.restype = ci
            lib.ssd_oracle_bwd.argtypes = [i64] * 7 + [vp] * 9 + [vp] * 7 + [ci]
            lib.ssd_oracle_bwd.restype = ci
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):          # torch tensor -> exact widening to fp64
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _prep(x, dt, A, B, C, D, seq_idx, init):
    x, dt, A, B, C, D, init = (_f64(v) for v in (x, dt, A, B, C, D, init))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (b, T, H) and A.shape == (H,) and D.shape == (H,)
    assert B.shape == (b, T, G, N) and C.shape == (b, T, G, N)
    if seq_idx is not None:
        if hasattr(seq_idx, "detach"):
            seq_idx = seq_idx.detach().cpu().numpy()
        seq_idx = np.ascontiguousarray(np.asarray(seq_idx, dtype=np.int32))
        assert seq_idx.shape == (b, T)
        nseq = int(seq_idx.max()) + 1
    else:
        nseq = b
    if init is not None:
        nseq = init.shape[0]
        assert init.shape == (nseq, H, P, N)
    return x, dt, A, B, C, D, seq_idx, init, (b, T, H, P, G, N, nseq)


def fwd(x, dt, A, B, C, D, seq_idx=None, init=None, chunk: int = 0, nthreads: int | None = None):
    """y (b,T,H,P) and, when ``chunk`` > 0, the state entering each chunk
    (b, ceil(T/chunk), H, P, N); all fp64 numpy."""
    x, dt, A, B, C, D, seq_idx, init, dims = _prep(x, dt, A, B, C, D, seq_idx, init)
    b, T, H, P, G, N, nseq = dims
    y = np.zeros((b, T, H, P))
    states = None
    if chunk > 0:
        states = np.zeros((b, (T + chunk - 1) // chunk, H, P, N))
    rc = _load().ssd_oracle_fwd(b, T, H, P, G, N, nseq, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(seq_idx), _ptr(init), chunk, _ptr(y), _ptr(states),
                                nthreads or default_threads())
    if rc:
        raise ValueError("ssd_oracle_fwd rejected its arguments (code %d)" % rc)
    return (y, states) if chunk > 0 else y


def bwd(x, dt, A, B, C, D, dout, seq_idx=None, init=None, nthreads: int | None = None):
    """Gradients of sum(y * dout): dict with dx, ddt, dA, dB, dC, dD and
    (when ``init`` is given) dinit; all fp64 numpy."""
    x, dt, A, B, C, D, seq_idx, init, dims = _prep(x, dt, A, B, C, D, seq_idx, init)
    b, T, H, P, G, N, nseq = dims
    g = _f64(dout)
    assert g.shape == x.shape
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(H), dB=np.zeros_like(B),
               dC=np.zeros_like(C), dD=np.zeros(H))
    dinit = np.zeros_like(init) if init is not None else None
    rc = _load().ssd_oracle_bwd(b, T, H, P, G, N, nseq, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(seq_idx), _ptr(init), _ptr(g), _ptr(out["dx"]),
                                _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                                _ptr(out["dD"]), _ptr(dinit), nthreads or default_threads())
    if rc:
        raise ValueError("ssd_oracle_bwd rejected its arguments (code %d)" % rc)
    if init is not None:
        out["dinit"] = dinit
    return out
