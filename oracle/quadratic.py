"""Materialised quadratic form of the Mamba2 SSD, differentiated by torch
autograd in fp64 on the CPU -- TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Third, independent statement of the same map (the state-space-duality view
of the recurrence behind "Deterministic bwd kernel for mamba2", Mamba PR #827):
unrolling state_t = exp(dt_t A) state_{t-1} + dt_t x_t B_t^T gives, per batch
row and head,

    y = (Lmat o (C B^T)) (dt o x) + (decay o (C . init)) + D x

with Lmat[t, s] = exp(sum_{s<k<=t} dt_k A) when s <= t and no sequence starts
in (s, t], else 0, and decay[t] = exp(sum_{t0<=k<=t} dt_k A) for the start t0
of t's sequence.  Gradients come from torch.autograd -- a route that shares
nothing with the hand-derived reverse sweep of the C oracle.  Sizes are kept
small (T x T matrices).
"""
from __future__ import annotations

import numpy as np
import torch


def _segment_ids(seq_idx, b, T):
    """seg[b, t]: index of the sequence start at or before t."""
    starts = np.zeros((b, T), dtype=bool)
    starts[:, 0] = True
    if seq_idx is not None:
        starts[:, 1:] = seq_idx[:, 1:] != seq_idx[:, :-1]
    return np.cumsum(starts, axis=1) - 1, starts


def forward_torch(x, dt, A, B, C, D, seq_idx=None, init=None):
    """All tensor arguments are fp64 torch tensors (may require grad)."""
    b, T, H, P = x.shape
    G = B.shape[2]
    hpg = H // G
    seg, starts = _segment_ids(seq_idx, b, T)
    ys = []
    for bi in range(b):
        same = torch.from_numpy(seg[bi][:, None] == seg[bi][None, :])
        causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
        mask = same & causal
        # first token of each token's sequence
        first = np.zeros(T, dtype=np.int64)
        cur = 0
        for t in range(T):
            if starts[bi, t]:
                cur = t
            first[t] = cur
        yh = []
        for h in range(H):
            g = h // hpg
            a = dt[bi, :, h] * A[h]                       # (T,)
            cs = torch.cumsum(a, 0)
            seg_sum = cs[:, None] - cs[None, :]            # sum_{s<k<=t} a_k
            Lmat = torch.where(mask, torch.exp(torch.where(mask, seg_sum, torch.zeros_like(seg_sum))),
                               torch.zeros_like(seg_sum))
            CB = C[bi, :, g] @ B[bi, :, g].T
            y = (Lmat * CB) @ (dt[bi, :, h][:, None] * x[bi, :, h])
            y = y + D[h] * x[bi, :, h]
            if init is not None:
                # decay from the sequence start t0 through t: sum_{t0<=k<=t} a_k
                cs0 = torch.cat([torch.zeros(1, dtype=cs.dtype), cs])
                dec = torch.exp(cs - cs0[torch.from_numpy(first)])
                sid = (seq_idx[bi] if seq_idx is not None else np.full(T, bi)).astype(np.int64)
                st0 = init[torch.from_numpy(sid), h]          # (T, P, N)
                y = y + dec[:, None] * torch.einsum("tpn,tn->tp", st0, C[bi, :, g])
            yh.append(y)
        ys.append(torch.stack(yh, dim=1))
    return torch.stack(ys, dim=0)


def fwd_bwd(x, dt, A, B, C, D, dout, seq_idx=None, init=None):
    """Returns (y, grads dict) as fp64 numpy arrays."""
    def t(a):
        return torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float64, requires_grad=True)
    xs = dict(x=t(x), dt=t(dt), A=t(A), B=t(B), C=t(C), D=t(D))
    if init is not None:
        xs["init"] = t(init)
    sidx = None if seq_idx is None else np.asarray(seq_idx)
    y = forward_torch(xs["x"], xs["dt"], xs["A"], xs["B"], xs["C"], xs["D"], sidx, xs.get("init"))
    loss = (y * torch.tensor(np.asarray(dout, dtype=np.float64))).sum()
    loss.backward()
    grads = {"d" + k: v.grad.numpy().copy() for k, v in xs.items()}
    return y.detach().numpy(), grads
