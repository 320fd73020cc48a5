"""Pins of the CPU oracle against things other than itself (no GPU needed).

* central finite differences of the oracle's own forward (the gradient is the
  derivative of sum(y * dout), whatever the code says);
* the materialised quadratic form differentiated by torch autograd;
* the chunked form for many chunk sizes (equivalence of the SSD's two forms);
* closed forms (one token, zero step, zero decay = causal linear attention,
  a hand-worked two-token example stored under tests/golden/);
* invariants (packed variable-length = separate runs, group sharing =
  repeated heads, linearity, thread-count independence).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.chunked as chunked
import oracle.quadratic as quadratic
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRADS = ["dx", "ddt", "dA", "dB", "dC", "dD"]


def f64(d):
    return {k: (None if v is None else (v.numpy() if v.dtype == torch.int32 else v.double().numpy()))
            for k, v in d.items()}


def small(seed=0, b=1, T=12, H=2, P=3, G=1, N=3, seq_lens=(), with_init=False, dt_shift=1.0):
    d = make_inputs(b, T, H, P, G, N, dtype=torch.float64, seed=seed, dt_shift=dt_shift,
                    d_mode="normal", seq_lens=seq_lens, with_init=with_init)
    return f64(d)


def relerr(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def loss(d, **over):
    dd = dict(d)
    dd.update(over)
    y = oracle.fwd(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], seq_idx=dd["seq_idx"],
                   init=dd["init"], nthreads=1)
    return float(np.sum(y * dd["dout"]))


@pytest.mark.parametrize("case", [
    dict(G=1), dict(G=2, H=4), dict(b=2, G=1, with_init=True),
    dict(T=12, seq_lens=(5, 7), with_init=True), dict(T=11, seq_lens=(4, 3, 4), with_init=False),
])
def test_finite_differences(case):
    d = small(seed=7, **case)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], seq_idx=d["seq_idx"],
                   init=d["init"], nthreads=1)
    names = ["x", "dt", "A", "B", "C", "D"] + (["init"] if d["init"] is not None else [])
    for name in names:
        arr = d[name]
        fd = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for i in range(flat.size):
            v = flat[i]
            h = 1e-5 * max(1.0, abs(v))
            p, m = arr.copy(), arr.copy()
            p.reshape(-1)[i] = v + h
            m.reshape(-1)[i] = v - h
            fd.reshape(-1)[i] = (loss(d, **{name: p}) - loss(d, **{name: m})) / (2 * h)
        got = g["d" + name]
        assert relerr(got, fd) < 1e-7, (name, relerr(got, fd))


@pytest.mark.parametrize("case", [
    dict(T=40, H=4, G=2, P=4, N=5),
    dict(T=37, H=4, G=1, P=2, N=3, b=2, with_init=True),
    dict(T=40, H=2, G=2, P=3, N=4, seq_lens=(10, 20, 10), with_init=True),
    dict(T=33, H=2, G=1, P=3, N=4, seq_lens=(1, 31, 1)),
])
def test_quadratic_form_autograd(case):
    d = small(seed=3, **case)
    y = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], seq_idx=d["seq_idx"], init=d["init"])
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], seq_idx=d["seq_idx"],
                   init=d["init"])
    yq, gq = quadratic.fwd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"],
                               seq_idx=d["seq_idx"], init=d["init"])
    assert relerr(y, yq) < 1e-12
    for k in GRADS + (["dinit"] if d["init"] is not None else []):
        assert relerr(g[k], gq[k]) < 1e-11, (k, relerr(g[k], gq[k]))


@pytest.mark.parametrize("T", [64, 50])
@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 8, 16, 64, "T"])
def test_chunked_equivalence(T, chunk):
    Q = T if chunk == "T" else chunk
    d = small(seed=11, T=T, H=4, G=2, P=4, N=5, with_init=True)
    y, states = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], init=d["init"], chunk=Q)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], init=d["init"])
    cb = chunked.backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], Q, init=d["init"])
    assert relerr(cb["fwd"]["y"], y) < 1e-12
    assert relerr(cb["fwd"]["states"], states) < 1e-12
    for k in GRADS + ["dinit"]:
        assert relerr(cb[k], g[k]) < 1e-11, (k, relerr(cb[k], g[k]))


def test_chunked_equivalence_varlen_aligned():
    d = small(seed=5, T=48, H=2, G=1, P=3, N=4, seq_lens=(16, 8, 24), with_init=True)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], seq_idx=d["seq_idx"],
                   init=d["init"])
    for Q in (4, 8):
        cb = chunked.backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], Q,
                              seq_idx=d["seq_idx"], init=d["init"])
        for k in GRADS + ["dinit"]:
            assert relerr(cb[k], g[k]) < 1e-11, (Q, k)


def test_golden_scalar_worked_example():
    with open(os.path.join(GOLDEN, "scalar_T2.json")) as fh:
        gold = json.load(fh)
    inp = gold["inputs"]
    x = np.array(inp["x"]).reshape(1, 2, 1, 1)
    dt = np.array(inp["dt"]).reshape(1, 2, 1)
    A = np.array([-math.log(2.0)])
    B = np.array(inp["B"]).reshape(1, 2, 1, 1)
    C = np.array(inp["C"]).reshape(1, 2, 1, 1)
    D = np.array([inp["D"]])
    dout = np.array(inp["dout"]).reshape(1, 2, 1, 1)
    y = oracle.fwd(x, dt, A, B, C, D)
    g = oracle.bwd(x, dt, A, B, C, D, dout)
    e = gold["expected"]
    np.testing.assert_allclose(y.reshape(-1), e["y"], rtol=1e-14)
    np.testing.assert_allclose(g["dx"].reshape(-1), e["dx"], rtol=1e-14)
    np.testing.assert_allclose(g["dB"].reshape(-1), e["dB"], rtol=1e-14)
    np.testing.assert_allclose(g["dC"].reshape(-1), e["dC"], rtol=1e-14)
    np.testing.assert_allclose(g["dD"], [e["dD"]], rtol=1e-14)
    np.testing.assert_allclose(g["ddt"].reshape(-1), [2.5, 6.0 - 0.5 * math.log(2.0)], rtol=1e-14)
    np.testing.assert_allclose(g["dA"], [e["dA"]], rtol=1e-14)


def test_closed_form_single_token():
    d = small(seed=2, T=1, H=2, G=1, P=3, N=4)
    y = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"])
    cb = float(d["C"][0, 0, 0] @ d["B"][0, 0, 0])
    for h in range(2):
        dt, x, go = d["dt"][0, 0, h], d["x"][0, 0, h], d["dout"][0, 0, h]
        np.testing.assert_allclose(y[0, 0, h], dt * cb * x + d["D"][h] * x, rtol=1e-13)
        np.testing.assert_allclose(g["dx"][0, 0, h], dt * cb * go + d["D"][h] * go, rtol=1e-13)
        np.testing.assert_allclose(g["ddt"][0, 0, h], cb * (go @ x), rtol=1e-13)
    gx = [float(d["dout"][0, 0, h] @ d["x"][0, 0, h]) * d["dt"][0, 0, h] for h in range(2)]
    np.testing.assert_allclose(g["dB"][0, 0, 0], sum(gx) * d["C"][0, 0, 0], rtol=1e-13)
    np.testing.assert_allclose(g["dC"][0, 0, 0], sum(gx) * d["B"][0, 0, 0], rtol=1e-13)
    np.testing.assert_allclose(g["dA"], 0.0, atol=0)


def test_closed_form_zero_step():
    d = small(seed=4, T=9, H=2, G=1, P=3, N=4)
    d["dt"][:] = 0.0
    y = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"])
    np.testing.assert_allclose(y, d["D"][None, None, :, None] * d["x"], rtol=1e-15)
    np.testing.assert_allclose(g["dx"], d["D"][None, None, :, None] * d["dout"], rtol=1e-15)
    assert np.all(g["dB"] == 0) and np.all(g["dC"] == 0) and np.all(g["dA"] == 0)


def test_closed_form_no_decay_is_causal_linear_attention():
    d = small(seed=6, T=10, H=2, G=1, P=3, N=4)
    d["A"][:] = 0.0
    y = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    for h in range(2):
        v = d["dt"][0, :, h, None] * d["x"][0, :, h]                 # (T, P)
        kv = np.cumsum(v[:, :, None] * d["B"][0, :, 0, None, :], axis=0)   # (T, P, N)
        want = np.einsum("tpn,tn->tp", kv, d["C"][0, :, 0]) + d["D"][h] * d["x"][0, :, h]
        np.testing.assert_allclose(y[0, :, h], want, rtol=1e-12)


def test_varlen_equals_separate_runs():
    lens = (5, 9, 6)
    d = small(seed=8, T=sum(lens), H=2, G=1, P=3, N=4, seq_lens=lens, with_init=True)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], seq_idx=d["seq_idx"],
                   init=d["init"])
    y = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], seq_idx=d["seq_idx"], init=d["init"])
    off = 0
    dA = np.zeros(2)
    dD = np.zeros(2)
    for s, L in enumerate(lens):
        sl = slice(off, off + L)
        part = {k: d[k][:, sl] for k in ("x", "dt", "B", "C", "dout")}
        ys = oracle.fwd(part["x"], part["dt"], d["A"], part["B"], part["C"], d["D"], init=d["init"][s:s + 1])
        gs = oracle.bwd(part["x"], part["dt"], d["A"], part["B"], part["C"], d["D"], part["dout"],
                        init=d["init"][s:s + 1])
        np.testing.assert_allclose(y[:, sl], ys, rtol=1e-13, atol=1e-14)
        for k in ("dx", "ddt", "dB", "dC"):
            np.testing.assert_allclose(g[k][:, sl], gs[k], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dinit"][s:s + 1], gs["dinit"], rtol=1e-12, atol=1e-13)
        dA += gs["dA"]
        dD += gs["dD"]
        off += L
    np.testing.assert_allclose(g["dA"], dA, rtol=1e-12)
    np.testing.assert_allclose(g["dD"], dD, rtol=1e-12)


def test_group_sharing_equals_repeated_heads():
    d = small(seed=9, T=14, H=4, G=2, P=3, N=4)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"])
    Br = np.repeat(d["B"], 2, axis=2)
    Cr = np.repeat(d["C"], 2, axis=2)
    gr = oracle.bwd(d["x"], d["dt"], d["A"], Br, Cr, d["D"], d["dout"])
    for k in ("dx", "ddt", "dA", "dD"):
        np.testing.assert_allclose(g[k], gr[k], rtol=1e-13)
    np.testing.assert_allclose(g["dB"], gr["dB"].reshape(1, 14, 2, 2, 4).sum(3), rtol=1e-12)
    np.testing.assert_allclose(g["dC"], gr["dC"].reshape(1, 14, 2, 2, 4).sum(3), rtol=1e-12)


def test_linearity_in_x_C_init():
    d = small(seed=10, T=13, H=2, G=1, P=3, N=4, with_init=True)
    e = small(seed=12, T=13, H=2, G=1, P=3, N=4, with_init=True)

    def y(x, C, init):
        return oracle.fwd(x, d["dt"], d["A"], d["B"], C, d["D"], init=init)
    zero_init = np.zeros_like(d["init"])
    # y is linear in x when C and init are held, and linear in (C) and in (init)
    np.testing.assert_allclose(y(2 * d["x"] - e["x"], d["C"], zero_init),
                               2 * y(d["x"], d["C"], zero_init) - y(e["x"], d["C"], zero_init),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y(d["x"], 3 * d["C"] + e["C"], d["init"]) - y(d["x"], 0 * d["C"], d["init"]),
                               3 * (y(d["x"], d["C"], d["init"]) - y(d["x"], 0 * d["C"], d["init"]))
                               + (y(d["x"], e["C"], d["init"]) - y(d["x"], 0 * d["C"], d["init"])),
                               rtol=1e-11, atol=1e-11)


def test_thread_count_does_not_change_bits():
    d = small(seed=13, T=70, H=6, G=2, P=3, N=4)
    a = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], nthreads=1)
    b = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], nthreads=4)
    for k in GRADS:
        assert np.array_equal(a[k], b[k]), k


def test_checkpoint_spacing_crossed():
    # a sequence longer than the oracle's checkpoint spacing (256 tokens)
    d = small(seed=14, T=600, H=1, G=1, P=2, N=2, dt_shift=3.0)
    g = oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"])
    cb = chunked.backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], 100)
    for k in GRADS:
        assert relerr(g[k], cb[k]) < 1e-11, k
