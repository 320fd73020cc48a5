"""Chunked (state-space-duality) form of the Mamba2 SSD in fp64 numpy --
TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

This is the second statement of the method: the sequence is cut into chunks
of ``chunk`` tokens; inside a chunk the scan is the quadratic (attention-like)
form, across chunks a state is carried.  It is written chunk by chunk, head by
head, straight from the per-kernel formulas of the chunked backward that
"Deterministic bwd kernel for mamba2" (Mamba PR #827, per-kernel breakdown
table) lists: chunk_cumsum, chunk_state (dx / db / ddAcs), state passing and
chunk_scan (dC / dx), followed by the head-to-group and chunk-to-total sums.

Its purpose is twofold: (1) it is pinned to the token-serial oracle for many
chunk sizes (equivalence of the two forms), and (2) it exposes the chunked
intermediates (in-chunk cumulative decay, chunk states, state gradients) so a
GPU kernel can be checked step by step.

Notation per (batch b, chunk c, head h): local token t; a_t = dt_t A_h;
Acs_t = sum_{k<=t} a_k (in-chunk inclusive prefix sum); E = Acs of the last
token; g_t = dout_t.  States are stored (P, N).  Sequence starts must fall on
chunk boundaries here.
"""
from __future__ import annotations

import numpy as np


def _starts(seq_idx, b, T):
    st = np.zeros((b, T), dtype=bool)
    st[:, 0] = True
    if seq_idx is not None:
        st[:, 1:] = seq_idx[:, 1:] != seq_idx[:, :-1]
    return st


def _seq_of(seq_idx, bi, t):
    return int(seq_idx[bi, t]) if seq_idx is not None else bi


def _check_aligned(starts, chunk):
    pos = np.nonzero(starts)[1]
    if np.any(pos % chunk != 0):
        raise ValueError("chunked form: every sequence start must be a multiple of the chunk size")


def _as(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def forward(x, dt, A, B, C, D, chunk, seq_idx=None, init=None):
    """Returns dict: y (b,T,H,P), Acs (b,H,nc,chunk) (padded with the last
    value), E (b,H,nc), S (b,nc,H,P,N) chunk contributions, states
    (b,nc,H,P,N) the state entering each chunk, final (b,H,P,N)."""
    x, dt, A, B, C, D, init = (_as(v) for v in (x, dt, A, B, C, D, init))
    if seq_idx is not None and hasattr(seq_idx, "detach"):
        seq_idx = seq_idx.detach().cpu().numpy()
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    Q = int(chunk)
    nc = (T + Q - 1) // Q
    starts = _starts(seq_idx, b, T)
    _check_aligned(starts, Q)

    Acs = np.zeros((b, H, nc, Q))
    E = np.zeros((b, H, nc))
    S = np.zeros((b, nc, H, P, N))
    states = np.zeros((b, nc, H, P, N))
    final = np.zeros((b, H, P, N))
    y = np.zeros_like(x)
    for bi in range(b):
        # chunk_cumsum: in-chunk inclusive prefix sum of dt*A
        for c in range(nc):
            t0, t1 = c * Q, min(T, (c + 1) * Q)
            a = dt[bi, t0:t1, :] * A[None, :]                  # (L, H)
            cs = np.cumsum(a, axis=0)
            Acs[bi, :, c, : t1 - t0] = cs.T
            Acs[bi, :, c, t1 - t0:] = cs[-1][:, None]
            E[bi, :, c] = cs[-1]
        # chunk_state: S_c = sum_t exp(E - Acs_t) dt_t x_t (outer) B_t
        for c in range(nc):
            t0, t1 = c * Q, min(T, (c + 1) * Q)
            L = t1 - t0
            for h in range(H):
                g = h // hpg
                w = np.exp(E[bi, h, c] - Acs[bi, h, c, :L]) * dt[bi, t0:t1, h]
                S[bi, c, h] = np.einsum("t,tp,tn->pn", w, x[bi, t0:t1, h], B[bi, t0:t1, g])
        # state passing: H_c (state entering chunk c)
        run = np.zeros((H, P, N))
        for c in range(nc):
            t0 = c * Q
            if starts[bi, t0]:
                run = init[_seq_of(seq_idx, bi, t0)].copy() if init is not None else np.zeros((H, P, N))
            states[bi, c] = run
            run = np.exp(E[bi, :, c])[:, None, None] * run + S[bi, c]
        final[bi] = run
        # chunk_scan: y = intra (L o C B^T)(dt x) + exp(Acs) C . H_c + D x
        for c in range(nc):
            t0, t1 = c * Q, min(T, (c + 1) * Q)
            L = t1 - t0
            for h in range(H):
                g = h // hpg
                acs = Acs[bi, h, c, :L]
                Lm = np.tril(np.exp(acs[:, None] - acs[None, :]))
                CB = C[bi, t0:t1, g] @ B[bi, t0:t1, g].T
                M = CB * Lm
                yi = M @ (dt[bi, t0:t1, h][:, None] * x[bi, t0:t1, h])
                yo = np.exp(acs)[:, None] * (C[bi, t0:t1, g] @ states[bi, c, h].T)
                y[bi, t0:t1, h] = yi + yo + D[h] * x[bi, t0:t1, h]
    return dict(y=y, Acs=Acs, E=E, S=S, states=states, final=final)


def backward(x, dt, A, B, C, D, dout, chunk, seq_idx=None, init=None):
    """Gradients of sum(y * dout) by the chunked backward.  Returns dict with
    dx, ddt, dA, dB, dC, dD, (dinit), and intermediates: dHscan and dS
    (b,nc,H,P,N) -- the per-chunk state gradient from the chunk's own outputs
    and the gradient reaching the chunk's end state -- dEpass (b,H,nc), dAcs
    (b,H,nc,chunk) before the reverse cumsum, and the forward dict 'fwd'."""
    x, dt, A, B, C, D, init, g_all = (_as(v) for v in (x, dt, A, B, C, D, init, dout))
    if seq_idx is not None and hasattr(seq_idx, "detach"):
        seq_idx = seq_idx.detach().cpu().numpy()
    f = forward(x, dt, A, B, C, D, chunk, seq_idx, init)
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    Q = int(chunk)
    nc = (T + Q - 1) // Q
    starts = _starts(seq_idx, b, T)
    Acs, E, states = f["Acs"], f["E"], f["states"]

    dx = np.zeros_like(x)
    ddt = np.zeros_like(dt)
    dA = np.zeros(H)
    dB = np.zeros_like(B)
    dC = np.zeros_like(C)
    dD = np.zeros(H)
    dinit = np.zeros_like(init) if init is not None else None
    dHscan = np.zeros((b, nc, H, P, N))
    dS = np.zeros((b, nc, H, P, N))
    dEpass = np.zeros((b, H, nc))
    dAcs_all = np.zeros((b, H, nc, Q))

    for bi in range(b):
        # per-chunk state gradient from the chunk's own outputs
        for c in range(nc):
            t0, t1 = c * Q, min(T, (c + 1) * Q)
            L = t1 - t0
            for h in range(H):
                g = h // hpg
                sc = np.exp(Acs[bi, h, c, :L])
                dHscan[bi, c, h] = (sc[:, None] * g_all[bi, t0:t1, h]).T @ C[bi, t0:t1, g]
        # state passing backward (reverse over chunks)
        for c in range(nc - 1, -1, -1):
            nxt_is_start = (c + 1 >= nc) or starts[bi, (c + 1) * Q]
            carry = np.zeros((H, P, N)) if nxt_is_start else dH_next
            dS[bi, c] = carry
            dEpass[bi, :, c] = np.exp(E[bi, :, c]) * np.einsum("hpn,hpn->h", states[bi, c], carry)
            dH_c = dHscan[bi, c] + np.exp(E[bi, :, c])[:, None, None] * carry
            if starts[bi, c * Q] and init is not None:
                dinit[_seq_of(seq_idx, bi, c * Q)] += dH_c
            dH_next = dH_c
        for c in range(nc):
            t0, t1 = c * Q, min(T, (c + 1) * Q)
            L = t1 - t0
            for h in range(H):
                g = h // hpg
                acs = Acs[bi, h, c, :L]
                e = E[bi, h, c]
                dtc = dt[bi, t0:t1, h]
                xc = x[bi, t0:t1, h]
                gc = g_all[bi, t0:t1, h]
                Bc = B[bi, t0:t1, g]
                Cc = C[bi, t0:t1, g]
                Hc = states[bi, c, h]
                dSc = dS[bi, c, h]
                dAcs = np.zeros(L)
                # chunk_state_bwd: dx / db / ddAcs through S_c
                w = np.exp(e - acs) * dtc
                Y = Bc @ dSc.T                                   # (L, P): dS B_t
                xY = np.sum(xc * Y, axis=1)
                dx[bi, t0:t1, h] += w[:, None] * Y
                dB[bi, t0:t1, g] += w[:, None] * (xc @ dSc)
                ddt[bi, t0:t1, h] += np.exp(e - acs) * xY
                u = w * xY
                dAcs -= u
                dAcs[L - 1] += u.sum()
                # chunk_scan_bwd: intra-chunk quadratic term and carried-in state
                Lm = np.tril(np.exp(acs[:, None] - acs[None, :]))
                CB = Cc @ Bc.T
                Gx = gc @ xc.T                                   # Gx[t,s] = g_t . x_s
                M = CB * Lm
                dx[bi, t0:t1, h] += dtc[:, None] * (M.T @ gc) + D[h] * gc
                ddt[bi, t0:t1, h] += np.sum(M * Gx, axis=0)
                W = Lm * Gx * dtc[None, :]
                dC[bi, t0:t1, g] += W @ Bc + np.exp(acs)[:, None] * (gc @ Hc)
                dB[bi, t0:t1, g] += W.T @ Cc
                Pm = Gx * M * dtc[None, :]
                dAcs += np.tril(Pm, -1).sum(axis=1) - np.tril(Pm, -1).sum(axis=0)
                dAcs += np.exp(acs) * np.sum(gc * (Cc @ Hc.T), axis=1)
                dAcs[L - 1] += dEpass[bi, h, c]
                dD[h] += np.sum(gc * xc)
                dAcs_all[bi, h, c, :L] = dAcs
                # chunk_cumsum_bwd: reverse prefix sum, then through a = dt*A
                da = np.cumsum(dAcs[::-1])[::-1]
                ddt[bi, t0:t1, h] += A[h] * da
                dA[h] += np.sum(dtc * da)
    out = dict(dx=dx, ddt=ddt, dA=dA, dB=dB, dC=dC, dD=dD, dHscan=dHscan, dS=dS,
               dEpass=dEpass, dAcs=dAcs_all, fwd=f)
    if init is not None:
        out["dinit"] = dinit
    return out
