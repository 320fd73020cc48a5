"""CPU oracle of the two steps either side of the SSD scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the CUDA library shares no code with it.

"Deterministic bwd kernel for mamba2" (Mamba PR #827) lists ``chunk_cumsum_bwd``
among the backward kernels it makes deterministic; in Mamba2 that step also
carries the gradient of the step-size preprocessing, and the model gates the
scan's output with z.  The pages print neither formula, so the plainest
reading is taken (the one Mamba2 itself uses):

* step size:  dt = clamp(sp(dt_raw + dt_bias), dt_min, dt_max), sp = softplus
  (log(1 + e^v)) or the identity; the gradient passes the clamp where
  dt_min <= sp(v) <= dt_max (the usual clamp rule) and is zero elsewhere;
  ddt_bias[h] = sum over all rows of ddt_raw[., h];
* gate:  out = y * silu(z), silu(z) = z * sigmoid(z).

Plain fp64 numpy, written straight from these definitions.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def softplus(v):
    """log(1 + e^v), evaluated without overflow."""
    v = _f64(v)
    return np.logaddexp(0.0, v)


def sigmoid(v):
    v = _f64(v)
    out = np.empty_like(v)
    pos = v >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-v[pos]))
    e = np.exp(v[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def dt_fwd(dt_raw, dt_bias=None, use_softplus=True, dt_min=0.0, dt_max=np.inf):
    """dt (rows, H) from dt_raw (rows, H) and dt_bias (H) or None."""
    v = _f64(dt_raw)
    if dt_bias is not None:
        v = v + _f64(dt_bias)[None, :]
    s = softplus(v) if use_softplus else v
    return np.minimum(np.maximum(s, dt_min), dt_max)


def dt_bwd(dt_raw, ddt, dt_bias=None, use_softplus=True, dt_min=0.0, dt_max=np.inf):
    """(ddt_raw (rows, H), ddt_bias (H)) from the gradient ddt w.r.t. dt."""
    v = _f64(dt_raw)
    if dt_bias is not None:
        v = v + _f64(dt_bias)[None, :]
    s = softplus(v) if use_softplus else v
    pass_clamp = (s >= dt_min) & (s <= dt_max)
    dsdv = sigmoid(v) if use_softplus else np.ones_like(v)
    ddt_raw = np.where(pass_clamp, _f64(ddt) * dsdv, 0.0)
    return ddt_raw, ddt_raw.sum(axis=0)


def gate_fwd(y, z):
    z = _f64(z)
    return _f64(y) * z * sigmoid(z)


def gate_bwd(y, z, dout):
    """(dy, dz) of out = y * silu(z)."""
    y, z, g = _f64(y), _f64(z), _f64(dout)
    s = sigmoid(z)
    silu = z * s
    dsilu = s * (1.0 + z * (1.0 - s))
    return g * silu, g * y * dsilu
