"""CPU oracle of the causal depthwise convolution before the SSD scan -- TEST
INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the CUDA library shares no code with it.

"Deterministic bwd kernel for mamba2" (Mamba PR #827), section "Atomic add
non-determinism", names the atomics of causal-conv1d, next to those of the
SSD backward, as a source of run-to-run differences in a Mamba2 training
step.  The page prints no formula, so the plainest reading of a causal
depthwise convolution of width K is taken, per batch row b, token t and
channel c (x laid out (batch, seqlen, channels)):

    pre[b,t,c] = bias[c] + sum_{k<K} w[c,k] * x[b, t-K+1+k, c]
    y[b,t,c]   = act(pre[b,t,c]),   act = identity or silu(v) = v * sigmoid(v)

where a tap reads zero before the start of the row and, in a packed batch
(seq_idx, batch 1), zero for a token of another sequence than t (a window
never reaches across a sequence start).  The backward of L = sum(y * dy):

    dpre[b,t,c] = dy[b,t,c] * act'(pre[b,t,c])
    dx[b,s,c]   = sum_k w[c,k] * dpre[b, s+K-1-k, c]   (same sequence, in range)
    dw[c,k]     = sum_{b,t} dpre[b,t,c] * x[b, t-K+1+k, c]   (same masks)
    dbias[c]    = sum_{b,t} dpre[b,t,c]

Plain fp64 numpy loops over the taps, written from these definitions.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def _sigmoid(v):
    out = np.empty_like(v)
    pos = v >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-v[pos]))
    e = np.exp(v[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def _tap_mask(T, K, seq_idx):
    """mask[t, k] = 1 where tap k of token t reads a token of t's own sequence
    (t - K + 1 + k >= 0 and, with seq_idx, the same id)."""
    t = np.arange(T)[:, None]
    src = t - (K - 1) + np.arange(K)[None, :]
    ok = src >= 0
    if seq_idx is not None:
        sid = np.asarray(seq_idx).reshape(-1)
        ok &= sid[np.clip(src, 0, T - 1)] == sid[t]
    return ok


def _pre(x, w, bias, seq_idx):
    b, T, C = x.shape
    K = w.shape[1]
    mask = _tap_mask(T, K, seq_idx)
    pre = np.zeros_like(x) + (0.0 if bias is None else bias[None, None, :])
    for k in range(K):
        src = np.arange(T) - (K - 1) + k
        xs = x[:, np.clip(src, 0, T - 1), :] * mask[:, k][None, :, None]
        pre += w[None, None, :, k] * xs
    return pre, mask


def fwd(x, w, bias=None, seq_idx=None, activation="silu"):
    """y (b, T, C) from x (b, T, C), w (C, K), bias (C) or None."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    pre, _ = _pre(x, w, bias, seq_idx)
    return pre * _sigmoid(pre) if activation == "silu" else pre


def bwd(x, w, dy, bias=None, seq_idx=None, activation="silu"):
    """(dx (b, T, C), dw (C, K), dbias (C)) of L = sum(y * dy)."""
    x, w, bias, dy = _f64(x), _f64(w), _f64(bias), _f64(dy)
    b, T, C = x.shape
    K = w.shape[1]
    pre, mask = _pre(x, w, bias, seq_idx)
    if activation == "silu":
        s = _sigmoid(pre)
        dpre = dy * s * (1.0 + pre * (1.0 - s))
    else:
        dpre = dy
    dx = np.zeros_like(x)
    dw = np.zeros((C, K))
    for k in range(K):
        src = np.arange(T) - (K - 1) + k          # token read by tap k of token t
        m = mask[:, k]
        contrib = dpre * m[None, :, None]          # dpre of the tokens whose tap k is live
        dw[:, k] = np.einsum("btc,btc->c", contrib, x[:, np.clip(src, 0, T - 1), :])
        for t in range(T):
            if m[t]:
                dx[:, src[t], :] += w[None, :, k] * dpre[:, t, :]
    return dx, dw, dpre.sum(axis=(0, 1))
