"""Degenerate inputs on the fused tensor-core path (bf16, headdim 64,
dstate 128, chunk 128), against the fp64 oracle and the closed forms of the
recurrence ("Mamba2 / state space duality": h_t = exp(dt_t A) h_{t-1} +
dt_t B_t x_t^T, y_t = C_t h_t + D x_t):

- dt = 0 everywhere: the state never leaves zero, so y = D x, dx = D dout,
  and dA, dB, dC are exactly zero (every term carries a factor dt);
- A = 0: no decay at all (causal linear attention);
- decay so strong that exp(dt A) underflows within a few tokens;
- one chunk with one head and one group;
- on the padded form, sequences of a single token between longer ones."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, relerr, run_gpu, run_oracle, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def check(d, Q=128, any_start=False, prefix="fused"):
    y, saved, g = run_gpu(d, Q, any_start=any_start)
    assert ssd.config_name(saved.dims, 0).startswith(prefix), ssd.config_name(saved.dims, 0)
    ref = run_oracle(d, chunk=Q)
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print({k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)
    return y, saved, g


def test_zero_step_everywhere():
    d = make_inputs(1, 384, 4, 64, 2, 128, dtype=torch.bfloat16, seed=31, dt_shift=4.0, d_mode="normal")
    d["dt"].zero_()
    y, saved, g = run_gpu(d, 128)
    assert ssd.config_name(saved.dims, 0).startswith("fused/")
    D = d["D"].view(1, 1, -1, 1)
    # (D reaches the forward's product as a bf16 hi + lo pair: y within the bf16 rounding of D x)
    assert y_relerr(y, (D.double() * d["x"].double()).numpy()) < TOL
    assert torch.allclose(g["dx"].cpu(), D * d["dout"].float(), rtol=1e-6, atol=0)
    for k in ("dA", "dB", "dC"):
        assert torch.count_nonzero(g[k]) == 0, k
    # ddt is not zero (the derivative at dt = 0): against the oracle
    ref = run_oracle(d, chunk=128)
    assert relerr(g["ddt"], ref["ddt"]) < TOL
    assert relerr(g["dD"], ref["dD"]) < TOL


def test_no_decay():
    d = make_inputs(1, 512, 4, 64, 1, 128, dtype=torch.bfloat16, seed=32, dt_shift=4.0, d_mode="normal",
                    with_init=True)
    d["A"].zero_()
    check(d)


def test_decay_underflowing_within_a_few_tokens():
    d = make_inputs(1, 512, 4, 64, 1, 128, dtype=torch.bfloat16, seed=33, dt_shift=-3.0, d_mode="normal",
                    with_init=True)
    # dt around 3 and A in [-16, -1]: exp(dt A) at most about e^-3 per token
    assert float((d["dt"] * d["A"].view(1, 1, -1)).max()) < -1.0
    check(d)


def test_one_chunk_one_head():
    d = make_inputs(1, 128, 1, 64, 1, 128, dtype=torch.bfloat16, seed=34, dt_shift=4.0, d_mode="normal",
                    with_init=True)
    check(d)


def test_single_token_sequences_on_the_padded_form():
    lens = (1, 300, 1, 1, 336, 1)   # six sequences in five 128-token chunks: the padding bound
    d = make_inputs(1, sum(lens), 4, 64, 1, 128, dtype=torch.bfloat16, seed=35, dt_shift=4.0, d_mode="normal",
                    seq_lens=lens, with_init=True)
    check(d, any_start=True, prefix="fused-padded")
