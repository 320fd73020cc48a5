"""Parity of the CUDA path with the fp64 CPU oracle, element by element.

Tolerances (relative L2 error per output tensor, oracle run on the very
inputs the GPU saw, bf16 values widened exactly): 1e-5 for fp32 inputs and
2e-3 for bf16 inputs with fp32 accumulation.  A bf16 forward output y is
compared with the oracle's y rounded to bf16 (its own output rounding is
not an error of the computation).
"""
import numpy as np
import pytest
import torch

from _helpers import GRADS, head_slice, relerr, run_gpu, run_oracle, to_dev, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


def check_all(d, chunk, tol, config=0, sample=None):
    y, saved, g = run_gpu(d, chunk, config=config)
    ref = run_oracle(d, chunk=chunk)
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    for k in GRADS:
        errs[k] = relerr(g[k], ref[k])
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    bad = {k: v for k, v in errs.items() if not v < tol}
    assert not bad, (bad, errs)
    return errs


def test_tiny_fp32_workload():
    w = WORKLOADS["tiny_fp32"]
    check_all(workload_inputs("tiny_fp32"), w.chunk, 1e-5)


@pytest.mark.parametrize("T,Q", [(63, 64), (64, 64), (65, 64), (129, 64), (200, 64), (50, 64), (1, 16), (97, 32)])
def test_fp32_ragged_lengths(T, Q):
    d = make_inputs(1, T, 4, 16, 2, 16, dtype=torch.float32, seed=T * 7 + Q, dt_shift=2.0, d_mode="normal")
    check_all(d, Q, 1e-5)


@pytest.mark.parametrize("case", [
    dict(b=2, H=4, G=1, P=16, N=16, with_init=True),
    dict(b=1, H=8, G=2, P=32, N=64),
    dict(b=1, H=2, G=2, P=8, N=8),          # one head per group
    dict(b=3, H=6, G=3, P=16, N=32, with_init=True),
])
def test_fp32_shapes(case):
    d = make_inputs(case["b"], 160, case["H"], case["P"], case["G"], case["N"], dtype=torch.float32, seed=21,
                    dt_shift=2.0, d_mode="normal", with_init=case.get("with_init", False))
    check_all(d, 64, 1e-5)


def test_fp32_varlen_chunk_aligned_with_init():
    d = make_inputs(1, 256, 4, 16, 1, 16, dtype=torch.float32, seed=5, dt_shift=2.0, d_mode="normal",
                    seq_lens=(64, 32, 128, 32), with_init=True)
    check_all(d, 32, 1e-5)


@pytest.mark.parametrize("config", [0, 1])
def test_bf16_small(config):
    d = make_inputs(1, 400, 8, 64, 2, 128, dtype=torch.bfloat16, seed=3, dt_shift=4.0, d_mode="normal")
    check_all(d, 128, 2e-3, config=config)


def test_bf16_T2048_full():
    w = WORKLOADS["bf16_T2048"]
    errs = check_all(workload_inputs("bf16_T2048"), w.chunk, 2e-3)
    print("bf16_T2048 relL2:", {k: "%.2e" % v for k, v in errs.items()})


def test_bf16_T16384_sampled_group():
    """The benchmarked workload at full size, in the benchmarked launch
    configuration; the oracle checks one whole group (its 32 heads and the
    group's dB/dC), which it can compute alone."""
    w = WORKLOADS["bf16_T16384"]
    d = workload_inputs("bf16_T16384")
    y, saved, g = run_gpu(d, w.chunk, config=0)
    hpg = w.nheads // w.ngroups
    for g0 in (0, w.ngroups - 1):
        sub = head_slice(d, g0, hpg)
        ref = run_oracle(sub, chunk=w.chunk)
        hs = slice(g0 * hpg, (g0 + 1) * hpg)
        errs = {"y": y_relerr(y[:, :, hs], ref["y"]), "states": relerr(saved.states_fp32()[:, :, hs], ref["states"]),
                "dx": relerr(g["dx"][:, :, hs], ref["dx"]), "ddt": relerr(g["ddt"][:, :, hs], ref["ddt"]),
                "dA": relerr(g["dA"][hs], ref["dA"]), "dD": relerr(g["dD"][hs], ref["dD"]),
                "dB": relerr(g["dB"][:, :, g0:g0 + 1], ref["dB"]), "dC": relerr(g["dC"][:, :, g0:g0 + 1], ref["dC"])}
        bad = {k: v for k, v in errs.items() if not v < 2e-3}
        assert not bad, (g0, bad)


def test_bf16_T16384_with_initial_states_sampled_group():
    """The benchmarked shape at full size with initial states, in the other
    launch configuration: one whole group against the oracle, its initial-state
    gradient included."""
    w = WORKLOADS["bf16_T16384"]
    d = make_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, dtype=w.dtype, seed=4242,
                    dt_shift=w.dt_shift, d_mode=w.d_mode, with_init=True)
    y, saved, g = run_gpu(d, w.chunk, config=1)
    hpg = w.nheads // w.ngroups
    g0 = 3
    sub = head_slice(d, g0, hpg)
    ref = run_oracle(sub, chunk=w.chunk)
    hs = slice(g0 * hpg, (g0 + 1) * hpg)
    errs = {"y": y_relerr(y[:, :, hs], ref["y"]), "states": relerr(saved.states_fp32()[:, :, hs], ref["states"]),
            "dx": relerr(g["dx"][:, :, hs], ref["dx"]), "ddt": relerr(g["ddt"][:, :, hs], ref["ddt"]),
            "dA": relerr(g["dA"][hs], ref["dA"]), "dD": relerr(g["dD"][hs], ref["dD"]),
            "dB": relerr(g["dB"][:, :, g0:g0 + 1], ref["dB"]), "dC": relerr(g["dC"][:, :, g0:g0 + 1], ref["dC"]),
            "dinit": relerr(g["dinit"][:, hs], ref["dinit"])}
    bad = {k: v for k, v in errs.items() if not v < 2e-3}
    assert not bad, (bad, errs)


def test_bf16_varlen_T32768_sampled_sequence():
    """Packed variable-length workload: sequence 0 checked against the oracle
    (sequences never interact); dA/dD, which sum over sequences, checked as
    the sum of per-sequence GPU runs."""
    w = WORKLOADS["bf16_varlen_T32768"]
    d = workload_inputs("bf16_varlen_T32768")
    y, saved, g = run_gpu(d, w.chunk)
    lens = w.seq_lens
    off = 0
    dA = torch.zeros_like(g["dA"], dtype=torch.float64)
    dD = torch.zeros_like(g["dD"], dtype=torch.float64)
    for s, L in enumerate(lens):
        sl = slice(off, off + L)
        part = dict(x=d["x"][:, sl].contiguous(), dt=d["dt"][:, sl].contiguous(), A=d["A"],
                    B=d["B"][:, sl].contiguous(), C=d["C"][:, sl].contiguous(), D=d["D"],
                    dout=d["dout"][:, sl].contiguous(), seq_idx=None, init=d["init"][s:s + 1].contiguous())
        ys, ss, gs = run_gpu(part, w.chunk)
        # chunks are identical in both runs: per-token outputs agree bit for bit
        for k in ("dx", "ddt", "dB", "dC"):
            assert torch.equal(g[k][:, sl], gs[k]), (s, k)
        assert torch.equal(y[:, sl], ys)
        assert torch.equal(g["dinit"][s:s + 1], gs["dinit"])
        dA += gs["dA"].double()
        dD += gs["dD"].double()
        if s == 0:
            ref = run_oracle(part, chunk=w.chunk)
            errs = {k: relerr(gs[k], ref[k]) for k in GRADS + ("dinit",)}
            errs["y"] = y_relerr(ys, ref["y"])
            bad = {k: v for k, v in errs.items() if not v < 2e-3}
            assert not bad, bad
        off += L
    assert relerr(g["dA"], dA.cpu().numpy()) < 1e-5
    assert relerr(g["dD"], dD.cpu().numpy()) < 1e-5


def test_zero_step_gives_skip_only():
    d = make_inputs(1, 100, 4, 16, 2, 16, dtype=torch.float32, seed=9, dt_shift=2.0, d_mode="normal")
    d["dt"].zero_()
    y, saved, g = run_gpu(d, 32)
    D = d["D"].view(1, 1, -1, 1)
    assert torch.allclose(y.cpu(), D * d["x"], rtol=1e-6, atol=1e-6)
    assert torch.allclose(g["dx"].cpu(), D * d["dout"], rtol=1e-6, atol=1e-6)
    assert torch.count_nonzero(g["dB"]) == 0 and torch.count_nonzero(g["dC"]) == 0


@pytest.mark.parametrize("case", [
    # several 64-wide tiles of tokens, state columns and head dims, each with a ragged edge
    dict(T=500, H=6, G=3, P=72, N=160, Q=192, init=True),
    dict(T=333, H=4, G=1, P=130, N=66, Q=80, init=False),
    dict(T=257, H=2, G=2, P=64, N=128, Q=128, init=True, lens=(40, 100, 1, 116)),
])
def test_fp32_multi_tile_shapes(case):
    """The general path's tiled products with more than one tile along every
    dimension and ragged tile edges, against the oracle; both launch
    configurations and the ordered dB/dC fold give the same bits."""
    lens = case.get("lens", ())
    d = make_inputs(1, case["T"], case["H"], case["P"], case["G"], case["N"], dtype=torch.float32,
                    seed=case["T"] + case["P"], dt_shift=2.0, d_mode="normal", seq_lens=lens,
                    with_init=case["init"])
    y, saved, g = run_gpu(d, case["Q"], any_start=bool(lens))
    ref = run_oracle(d, chunk=case["Q"])
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    for k in GRADS:
        errs[k] = relerr(g[k], ref[k])
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    bad = {k: v for k, v in errs.items() if not v < 1e-5}
    assert not bad, (bad, errs)
    dev = to_dev(d)
    for config, variant in ((1, 0), (0, 2)):
        o = run_gpu(d, case["Q"], config=config, variant=variant, g=dev, any_start=bool(lens))[2]
        for k in g:
            assert torch.equal(g[k].view(torch.int32), o[k].view(torch.int32)), (config, variant, k)
