"""The padded form of packed batches whose sequences start inside a chunk,
checked on the host.

The library cuts the token stream at every sequence start and every 128
tokens and pads each piece to a 128-token chunk of its own with tokens that
have dt = 0 and x = B = C = dout = 0.  Here (1) its piece table is compared
with a segmentation written out independently, including the case where the
padded chunk count reaches its bound ceil(T / 128) + nseq - 1, and (2) the
identity the form rests on -- such padding tokens leave y, every gradient of
the real tokens, dA, dD, dinit and the state entering each of the caller's
chunks unchanged (the recurrence of "Mamba2 / state space duality": exp(0 A)
= 1 keeps the state, dt B x = 0 adds nothing, C = 0 and x = 0 give y = 0) --
is checked on the fp64 oracle for padded problems built from that table."""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
import oracle
from deterministic_mamba2_ssd_gb300.inputs import make_inputs


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return ssd.lib()


def fused_dims(T, nseq, Q=128, N=128, H=4, G=1):
    return ssd.make_dims(1, T, H, 64, G, N, Q, nseq=nseq, seq_idx=True, any_start=True)


def piece_table(L, dims, seq):
    npc = L.mamba2_ssd_padded_chunks(ctypes.byref(dims))
    nc = ssd.lib().mamba2_ssd_num_chunks(ctypes.byref(dims))
    assert npc > 0
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    tab = np.full(3 * npc + nc, -7, dtype=np.int32)
    rc = L.mamba2_ssd_padded_piece_table(ctypes.byref(dims), seq.ctypes.data, tab.ctypes.data)
    assert rc == 0
    return npc, tab[:npc], tab[npc:2 * npc], tab[2 * npc:3 * npc], tab[3 * npc:]


def pieces_by_hand(seq):
    """Maximal runs of one sequence id that stay inside one 128-token chunk."""
    out, t, T = [], 0, len(seq)
    while t < T:
        end = min(T, (t // 128 + 1) * 128)
        u = t + 1
        while u < end and seq[u] == seq[t]:
            u += 1
        out.append((t, u - t, int(seq[t])))
        t = u
    return out


def seq_of(lens):
    return np.repeat(np.arange(len(lens)), lens).astype(np.int32)


CASES = [
    ((100, 300, 1, 111), 128),
    ((1, 127, 128, 2, 1, 253, 400), 128),
    ((5, 3, 7, 1, 9, 2, 13, 1000), 128),
    ((200,), 128),
    ((50, 17, 100, 133), 128),            # ragged length 300
    ((1, 128, 128, 128, 127), 128),       # every start inside a chunk: the bound is reached
    ((100, 300, 1, 111), 256),
    ((300, 212, 600), 256),
    ((100, 300, 1, 111), (256, 128)),     # chunk 256 with dstate 128
    ((5, 600, 3, 700), (512, 128)),       # chunk 512 with dstate 128
]


def q_and_n(Q):
    """(chunk, dstate) of a case: chunk 128 with dstate 128, chunk 256 with dstate 256, or as given."""
    return Q if isinstance(Q, tuple) else (Q, 128 if Q == 128 else 256)


@pytest.mark.parametrize("lens,Q", CASES)
def test_piece_table_matches_the_segmentation(L, lens, Q):
    T = sum(lens)
    seq = seq_of(lens)
    Q, N = q_and_n(Q)
    dims = fused_dims(T, len(lens), Q=Q, N=N)
    assert ssd.config_name(dims, 0).startswith("fused-padded" if N == 128 else "fused-split-padded")
    npc, start, ln, ids, cmap = piece_table(L, dims, seq)
    assert npc == (T + 127) // 128 + len(lens) - 1
    ref = pieces_by_hand(seq)
    assert len(ref) <= npc
    for k, (s0, n, i) in enumerate(ref):
        assert (start[k], ln[k], ids[k]) == (s0, n, i), k
    # trailing chunks: padding only, inside the last sequence
    assert np.all(ln[len(ref):] == 0) and np.all(start[len(ref):] == T) and np.all(ids[len(ref):] == seq[-1])
    # every caller chunk begins a piece, and the map names it
    nc = (T + Q - 1) // Q
    assert len(cmap) == nc
    for c in range(nc):
        assert start[cmap[c]] == c * Q
    # the pieces tile the tokens exactly once
    cover = np.zeros(T, np.int32)
    for k in range(npc):
        cover[start[k]:start[k] + ln[k]] += 1
    assert np.all(cover == 1)


def test_bound_is_reached_when_every_start_falls_inside_a_chunk(L):
    lens = (1, 128, 128, 128, 127)
    npc, _, ln, _, _ = piece_table(L, fused_dims(sum(lens), len(lens)), seq_of(lens))
    assert npc == 8 and np.all(ln > 0)


def test_path_selection_and_launches(L):
    dims = fused_dims(512, 4)
    assert ssd.config_name(dims, 0) == "fused-padded/0" and ssd.config_name(dims, 1) == "fused-padded/1"
    assert ssd.bwd_launch_names(dims, 0, 0) == ["pad_gather", "fused_bwd", "fold_scalars", "pad_scatter"]
    assert ssd.bwd_launch_names(dims, 0, 1) == ["pad_gather", "fused_bwd_atomic", "pad_scatter"]
    split = fused_dims(512, 4, Q=256, N=256)
    assert ssd.config_name(split, 0) == "fused-split-padded/0"
    assert ssd.bwd_launch_names(split, 1, 0) == ["pad_gather", "fused_bwd", "fused_bwd", "split_fold",
                                                 "split_scalars", "pad_scatter"]
    assert ssd.bwd_launch_names(split, 0, 1) == ["pad_gather", "fused_bwd_atomic", "fused_bwd_atomic", "split_fold",
                                                 "pad_scatter"]
    # a ragged length is fine in the padded form
    assert ssd.config_name(fused_dims(300, 4), 0) == "fused-padded/0"
    # too many sequences for the padding bound, fp32, batch 2, other shapes: the general path
    for d in (fused_dims(512, 6), ssd.make_dims(1, 512, 4, 64, 1, 128, 128, nseq=4, dtype=torch.float32,
                                                seq_idx=True, any_start=True),
              ssd.make_dims(2, 512, 4, 64, 1, 128, 128, nseq=4, seq_idx=True, any_start=True),
              fused_dims(512, 4, Q=64), fused_dims(512, 4, Q=256, N=256, H=3)):
        assert ssd.config_name(d, 0).startswith("simt"), d
        assert L.mamba2_ssd_padded_chunks(ctypes.byref(d)) == 0
    assert ssd.bwd_workspace_size(dims, 0, 2) == 0   # no ordered variant on the fused kernels


def test_piece_table_rejects_bad_ids(L):
    dims = fused_dims(256, 2)
    tab = np.zeros(3 * 3 + 2, np.int32)
    for seq in (np.r_[np.zeros(100), np.ones(156) * 2], np.r_[np.ones(100), np.zeros(156)],
                np.r_[np.zeros(100), -np.ones(156)]):
        s = np.ascontiguousarray(seq, dtype=np.int32)
        assert L.mamba2_ssd_padded_piece_table(ctypes.byref(dims), s.ctypes.data, tab.ctypes.data) == 1
    plain = ssd.make_dims(1, 256, 4, 64, 1, 128, 128, nseq=2, seq_idx=True)
    s = np.ascontiguousarray(seq_of((128, 128)))
    assert L.mamba2_ssd_padded_piece_table(ctypes.byref(plain), s.ctypes.data, tab.ctypes.data) == 1


def pad(a, start, ln, npc):
    """Rows of the caller's (1, T, ...) array placed at the padded rows, zero elsewhere."""
    out = np.zeros((1, npc * 128) + a.shape[2:], dtype=a.dtype)
    for k in range(npc):
        out[0, k * 128:k * 128 + ln[k]] = a[0, start[k]:start[k] + ln[k]]
    return out


def unpad(a, start, ln, T):
    out = np.zeros((1, T) + a.shape[2:], dtype=a.dtype)
    for k in range(len(start)):
        out[0, start[k]:start[k] + ln[k]] = a[0, k * 128:k * 128 + ln[k]]
    return out


@pytest.mark.parametrize("lens,Q,init", [
    ((100, 300, 1, 111), 128, True),
    ((5, 3, 7, 1, 9, 2, 13, 1000), 128, False),
    ((50, 17, 100, 133), 128, True),
    ((1, 128, 128, 128, 127), 128, True),
    ((100, 300, 1, 111), 256, True),
])
def test_padding_leaves_the_oracle_results_unchanged(L, lens, Q, init):
    T, nseq = sum(lens), len(lens)
    seq = seq_of(lens)
    npc, start, ln, ids, cmap = piece_table(L, fused_dims(T, nseq, Q=Q, N=128 if Q == 128 else 256), seq)
    d = make_inputs(1, T, 2, 8, 1, 16, dtype=torch.float32, seed=T + nseq, dt_shift=1.0, d_mode="normal",
                    seq_lens=lens, with_init=init)
    a = {k: (v.double().numpy() if v is not None else None) for k, v in d.items()}
    p = {k: pad(a[k], start, ln, npc) for k in ("x", "dt", "B", "C", "dout")}
    seq_p = np.repeat(ids, 128)[None, :].astype(np.int32)
    y, st = oracle.fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], seq_idx=seq[None, :], init=a["init"], chunk=Q)
    yp, stp = oracle.fwd(p["x"], p["dt"], a["A"], p["B"], p["C"], a["D"], seq_idx=seq_p, init=a["init"], chunk=128)
    np.testing.assert_allclose(unpad(yp, start, ln, T), y, rtol=1e-12, atol=1e-12)
    assert np.all(yp[0, [k * 128 + j for k in range(npc) for j in range(ln[k], 128)]] == 0)
    np.testing.assert_allclose(stp[0, cmap], st[0], rtol=1e-12, atol=1e-12)
    g = oracle.bwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["dout"], seq_idx=seq[None, :], init=a["init"])
    gp = oracle.bwd(p["x"], p["dt"], a["A"], p["B"], p["C"], a["D"], p["dout"], seq_idx=seq_p, init=a["init"])
    for k in ("dx", "ddt", "dB", "dC"):
        np.testing.assert_allclose(unpad(gp[k], start, ln, T), g[k], rtol=1e-10, atol=1e-11, err_msg=k)
    for k in ("dA", "dD") + (("dinit",) if init else ()):
        np.testing.assert_allclose(gp[k], g[k], rtol=1e-10, atol=1e-11, err_msg=k)
