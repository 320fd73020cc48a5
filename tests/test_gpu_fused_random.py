"""Seeded random shapes of the fused tensor-core family (bf16, headdim 64,
dstate 128, and dstate 256 with one group on the split form) against the
fp64 oracle: the number of heads and groups, the
sequence length (a multiple of 128), the batch, initial states, packed
sequences with chunk-aligned starts and the chunk length (128, 256 or 512,
the last two run in 128-token chunks) are drawn from a fixed seed, so that
the cases cover combinations no hand-written case names.  Every gradient,
dinit, y (against the oracle's y rounded to bf16) and the saved states are
held to relL2 2e-3, the bar for bf16 inputs with fp32 accumulation."""
import random

import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, relerr, run_gpu, run_oracle, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def draw(seed):
    rng = random.Random(seed)
    G = rng.choice([1, 1, 2, 4])
    H = G * rng.choice([1, 2, 3, 4, 8])
    Q = rng.choice([128, 128, 256, 512])
    b = rng.choice([1, 1, 2])
    T = 128 * rng.randint(max(1, Q // 128), 8)
    init = rng.random() < 0.5
    lens = ()
    if b == 1 and rng.random() < 0.7:   # packed sequences, starts on multiples of the chunk
        cuts = sorted(rng.sample(range(1, T // Q), min(3, T // Q - 1))) if T // Q > 1 else []
        edges = [0] + [Q * c for c in cuts] + [T]
        lens = tuple(e1 - e0 for e0, e1 in zip(edges, edges[1:]))
    return dict(b=b, T=T, H=H, G=G, Q=Q, init=init, lens=lens, dt_shift=rng.choice([2.0, 4.0]))


@pytest.mark.parametrize("seed", range(16))
def test_random_fused_shapes_match_oracle(seed):
    c = draw(1000 + seed)
    d = make_inputs(c["b"], c["T"], c["H"], 64, c["G"], 128, dtype=torch.bfloat16, seed=2000 + seed,
                    dt_shift=c["dt_shift"], d_mode="normal", seq_lens=c["lens"], with_init=c["init"])
    y, saved, g = run_gpu(d, c["Q"])
    name = ssd.config_name(saved.dims, 0)
    assert name.startswith("fused/" if c["Q"] == 128 else "fused-chunk128/"), (c, name)
    ref = run_oracle(d, chunk=c["Q"])
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print(c, name, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (c, bad, errs)


def draw_split(seed):
    rng = random.Random(seed)
    H = 2 * rng.choice([1, 2, 3, 4, 8])   # an even head count: two or four head slices per state half
    Q = rng.choice([128, 256])
    b = rng.choice([1, 1, 2])
    T = Q * rng.randint(1, 1024 // Q)
    init = rng.random() < 0.6
    lens = ()
    if b == 1 and T // Q > 1 and rng.random() < 0.7:
        cuts = sorted(rng.sample(range(1, T // Q), min(2, T // Q - 1)))
        edges = [0] + [Q * c for c in cuts] + [T]
        lens = tuple(e1 - e0 for e0, e1 in zip(edges, edges[1:]))
    return dict(b=b, T=T, H=H, Q=Q, init=init, lens=lens, dt_shift=rng.choice([2.0, 4.0]))


@pytest.mark.parametrize("seed", range(8))
def test_random_split_shapes_match_oracle(seed):
    c = draw_split(3000 + seed)
    d = make_inputs(c["b"], c["T"], c["H"], 64, 1, 256, dtype=torch.bfloat16, seed=4000 + seed,
                    dt_shift=c["dt_shift"], d_mode="normal", seq_lens=c["lens"], with_init=c["init"])
    y, saved, g = run_gpu(d, c["Q"])
    name = ssd.config_name(saved.dims, 0)
    assert name.startswith("fused-split/"), (c, name)
    ref = run_oracle(d, chunk=c["Q"])
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print(c, name, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (c, bad, errs)
