"""The chunked-form formulas for sequences that start inside a chunk, written
out in fp64 numpy, against the token-serial oracle (which simply resets the
state where the sequence id changes).  These are the formulas the general
CUDA path evaluates for SSD_DIMS_SEQ_ANY_START, derived from the recurrence:

  f_i        local start of token i's sequence in its chunk (0: entered from before)
  din_i      exp(Acs_i) if f_i = 0, else exp(Acs_i - Acs_{f_i - 1})
  Hin_i      the state entering the chunk if f_i = 0, else init[seq(i)] (or 0)
  L[i, j]    exp(Acs_i - Acs_j) for f_i <= j <= i, else 0
  y_i        = sum_j (C_i . B_j) L[i, j] dt_j x_j + din_i Hin_i C_i + D x_i
  S_c        = sum_{j >= fe} exp(E - Acs_j) dt_j x_j B_j^T      (fe = f of the last token)
  carry      = exp(E) H_c if fe = 0, else exp(E - Acs_{fe-1}) init[seq(last)]

and their reverse-mode derivatives (the gradient of exp(Acs_i - Acs_{f-1})
terms lands on Acs_{f-1}).  Nothing here is shared with the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from deterministic_mamba2_ssd_gb300.inputs import make_inputs


def chunked_with_starts(x, dt, A, B, C, D, g, sid, init, Q):
    """fp64 forward (y, chunk states) and backward of the chunked form, batch row 0."""
    T, H, P = x.shape[1], x.shape[2], x.shape[3]
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    nseq = int(sid.max()) + 1
    first = {}
    for t in range(T):
        if t == 0 or sid[t] != sid[t - 1]:
            first[sid[t]] = t
    nc = -(-T // Q)
    x, dt, B, C, g = x[0], dt[0], B[0], C[0], g[0]
    Z = np.zeros((P, N))

    def ls(t, t0):
        return max(first[sid[t]] - t0, 0)

    Acs = np.zeros((H, nc, Q))
    for c in range(nc):
        t0, L = c * Q, min(Q, T - c * Q)
        for h in range(H):
            cs = np.cumsum(dt[t0:t0 + L, h] * A[h])
            Acs[h, c, :L], Acs[h, c, L:] = cs, cs[-1]

    def init_of(s, h):
        return init[s, h] if init is not None else Z

    # forward: chunk contributions, state passing, outputs
    S = np.zeros((nc, H, P, N))
    states = np.zeros((nc, H, P, N))
    y = np.zeros((T, H, P))
    for h in range(H):
        gg = h // hpg
        run = Z
        for c in range(nc):
            t0, L = c * Q, min(Q, T - c * Q)
            e = Acs[h, c, L - 1]
            fe = ls(t0 + L - 1, t0)
            for j in range(fe, L):
                S[c, h] += np.exp(e - Acs[h, c, j]) * dt[t0 + j, h] * np.outer(x[t0 + j, h], B[t0 + j, gg])
            if t0 == 0 or sid[t0] != sid[t0 - 1]:
                run = init_of(sid[t0], h)
            states[c, h] = run
            carried = np.exp(e) * run if fe == 0 else np.exp(e - Acs[h, c, fe - 1]) * init_of(sid[t0 + L - 1], h)
            run = carried + S[c, h]

    def hin(t, c, h):
        t0 = c * Q
        f, i = ls(t, t0), t - t0
        if f == 0:
            return states[c, h], np.exp(Acs[h, c, i])
        return init_of(sid[t], h), np.exp(Acs[h, c, i] - Acs[h, c, f - 1])

    for t in range(T):
        c = t // Q
        t0, i = c * Q, t - c * Q
        for h in range(H):
            gg = h // hpg
            acc = np.zeros(P)
            for j in range(ls(t, t0), i + 1):
                acc += (C[t, gg] @ B[t0 + j, gg]) * np.exp(Acs[h, c, i] - Acs[h, c, j]) * dt[t0 + j, h] * x[t0 + j, h]
            hn, dn = hin(t, c, h)
            y[t, h] = acc + dn * (hn @ C[t, gg]) + D[h] * x[t, h]

    # backward
    dx = np.zeros((T, H, P)); ddt = np.zeros((T, H)); dA = np.zeros(H); dD = np.zeros(H)
    dB = np.zeros((T, G, N)); dC = np.zeros((T, G, N)); dinit = np.zeros((nseq, H, P, N))
    dS = np.zeros((nc, H, P, N)); dEp = np.zeros((H, nc))
    for h in range(H):
        gg = h // hpg
        carry = Z
        for c in range(nc - 1, -1, -1):
            t0, L = c * Q, min(Q, T - c * Q)
            nxt_start = c + 1 >= nc or sid[(c + 1) * Q] != sid[(c + 1) * Q - 1]
            cur = Z if nxt_start else carry
            fe = ls(t0 + L - 1, t0)
            e = Acs[h, c, L - 1]
            dhscan = sum((np.exp(Acs[h, c, i]) * np.outer(g[t0 + i, h], C[t0 + i, gg])
                          for i in range(L) if ls(t0 + i, t0) == 0), Z)
            dS[c, h] = cur
            if fe == 0:
                dEp[h, c] = np.exp(e) * np.sum(states[c, h] * cur)
                carry = dhscan + np.exp(e) * cur
            else:
                dEp[h, c] = np.exp(e - Acs[h, c, fe - 1]) * np.sum(init_of(sid[t0 + L - 1], h) * cur)
                carry = dhscan
            if t0 == 0 or sid[t0] != sid[t0 - 1]:
                dinit[sid[t0], h] += carry
    for s, ts in first.items():       # sequences that start inside a chunk
        if ts % Q == 0:
            continue
        c, f = ts // Q, ts % Q
        t0, L = c * Q, min(Q, T - c * Q)
        for h in range(H):
            gg = h // hpg
            i, acc = f, np.zeros((P, N))
            while i < L and sid[t0 + i] == s:
                acc += np.exp(Acs[h, c, i] - Acs[h, c, f - 1]) * np.outer(g[t0 + i, h], C[t0 + i, gg])
                i += 1
            if sid[t0 + L - 1] == s:
                acc += np.exp(Acs[h, c, L - 1] - Acs[h, c, f - 1]) * dS[c, h]
            dinit[s, h] = acc
    for c in range(nc):
        t0, L = c * Q, min(Q, T - c * Q)
        fe = ls(t0 + L - 1, t0)
        for h in range(H):
            gg = h // hpg
            M, W, MG = np.zeros((L, L)), np.zeros((L, L)), np.zeros((L, L))
            for i in range(L):
                for j in range(ls(t0 + i, t0), i + 1):
                    Lij = np.exp(Acs[h, c, i] - Acs[h, c, j])
                    gx = g[t0 + i, h] @ x[t0 + j, h]
                    M[i, j] = (C[t0 + i, gg] @ B[t0 + j, gg]) * Lij
                    W[i, j] = Lij * gx * dt[t0 + j, h]
                    MG[i, j] = M[i, j] * gx
            e = Acs[h, c, L - 1]
            dacs, u, vin, part = np.zeros(L), np.zeros(L), np.zeros(L), np.zeros(L)
            for i in range(L):
                t = t0 + i
                dti = dt[t, h]
                eEi = 0.0 if i < fe else np.exp(e - Acs[h, c, i])
                wi = eEi * dti
                hn, dn = hin(t, c, h)
                dx[t, h] = dti * (M[:, i] @ g[t0:t0 + L, h]) + wi * (dS[c, h] @ B[t, gg]) + D[h] * g[t, h]
                dC[t, gg] += W[i] @ B[t0:t0 + L, gg] + dn * (hn.T @ g[t, h])
                dB[t, gg] += W[:, i] @ C[t0:t0 + L, gg] + wi * (dS[c, h].T @ x[t, h])
                sx = x[t, h] @ (dS[c, h] @ B[t, gg])
                v = dn * (g[t, h] @ (hn @ C[t, gg]))
                part[i] = MG[i + 1:, i].sum() + MG[i, i] + eEi * sx
                dacs[i] = MG[i, :i] @ dt[t0:t0 + i, h] - dti * MG[i + 1:, i].sum() + v - wi * sx
                u[i] = wi * sx
                vin[i] = v if ls(t, t0) > 0 else 0.0
                dD[h] += g[t, h] @ x[t, h]
            da = u.sum() + dEp[h, c]
            pend = dEp[h, c] if fe > 0 else 0.0
            for i in range(L - 1, -1, -1):
                d = dacs[i]
                if i + 1 < L and sid[t0 + i] != sid[t0 + i + 1]:
                    d -= pend       # token i + 1 starts a sequence: its decays are measured from Acs_i
                    pend = 0.0
                da += d
                pend += vin[i]
                ddt[t0 + i, h] = part[i] + A[h] * da
                dA[h] += dt[t0 + i, h] * da
    grads = dict(dx=dx[None], ddt=ddt[None], dA=dA, dB=dB[None], dC=dC[None], dD=dD)
    if init is not None:
        grads["dinit"] = dinit
    return y[None], states[None], grads


@pytest.mark.parametrize("lens,Q,with_init", [
    ((1, 15, 16), 16, True),            # a start at the second token of a chunk
    ((15, 1, 16, 2), 16, True),         # a start at the last token; a one-token sequence
    ((5, 3, 7, 1, 9, 2, 13), 8, True),  # several starts per chunk, ragged tail
    ((5, 3, 7, 1, 9, 2, 13), 8, False),
    ((20, 6, 11), 8, True),             # a sequence wholly inside one chunk
    ((40,), 8, True),                   # one sequence: no boundaries
])
def test_chunked_formulas_with_starts_inside_chunks(lens, Q, with_init):
    d = make_inputs(1, sum(lens), 2, 3, 1, 4, dtype=torch.float64, seed=len(lens) + Q, dt_shift=1.0,
                    d_mode="normal", seq_lens=lens, with_init=with_init)
    f = {k: (None if v is None else (v.numpy() if v.dtype == torch.int32 else v.double().numpy()))
         for k, v in d.items()}
    y, states, grads = chunked_with_starts(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["dout"],
                                           f["seq_idx"][0], f["init"], Q)
    y_ref, states_ref = oracle.fwd(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], seq_idx=f["seq_idx"],
                                   init=f["init"], chunk=Q)
    ref = oracle.bwd(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["dout"], seq_idx=f["seq_idx"],
                     init=f["init"])
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(states, states_ref, rtol=1e-11, atol=1e-12)
    for k, v in grads.items():
        np.testing.assert_allclose(v, ref[k], rtol=1e-10, atol=1e-11, err_msg=k)
