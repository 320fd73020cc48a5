"""The tensor-core forward (bf16, chunk 128, dstate 128, headdim 64) against
the fp64 oracle: y (compared with the oracle's y rounded to bf16) and the
saved state entering every chunk (the fp32 view of the packed pair), on
shapes that span several chunks, heads per group (including one and an odd
number, and enough heads in few units that each unit's heads run as several
slices), batch rows, initial states, packed sequences and strong decay, and
on the 2K workload in full.  Parity bar: relL2 2e-3 per tensor (bf16 inputs,
fp32 accumulation)."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import relerr, run_oracle, to_dev, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def run_fwd(d, chunk=128):
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=chunk, seq_idx=g["seq_idx"],
                       init_states=g["init"])
    torch.cuda.synchronize()
    return y, saved


@pytest.mark.parametrize("case", [
    dict(b=1, T=128, H=2, G=1),
    dict(b=1, T=384, H=8, G=2),
    dict(b=2, T=256, H=4, G=2, with_init=True),
    dict(b=1, T=256, H=3, G=3),              # one head per group
    dict(b=1, T=512, H=6, G=2),              # odd heads per group
    dict(b=1, T=512, H=4, G=1, seq_lens=(128, 256, 128), with_init=True),
    dict(b=1, T=1024, H=32, G=1, dt_shift=2.0),   # strong decay; the units' heads in two slices
    dict(b=1, T=256, H=64, G=1, with_init=True),  # two units of 64 heads: four slices of 16
])
def test_forward_matches_oracle(case):
    d = make_inputs(case["b"], case["T"], case["H"], 64, case["G"], 128, dtype=torch.bfloat16,
                    seed=case["T"] + 3 * case["H"], dt_shift=case.get("dt_shift", 4.0), d_mode="normal",
                    seq_lens=case.get("seq_lens", ()), with_init=case.get("with_init", False))
    y, saved = run_fwd(d)
    assert ssd.config_name(saved.dims, 0).startswith("fused")
    ref = run_oracle(d, chunk=128, with_y=True)
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    print(case, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)


def test_forward_T2048_full_and_repeatable():
    w = WORKLOADS["bf16_T2048"]
    d = workload_inputs("bf16_T2048")
    y, saved = run_fwd(d, w.chunk)
    ref = run_oracle(d, chunk=w.chunk, with_y=True)
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    print("bf16_T2048 forward relL2:", {k: "%.2e" % v for k, v in errs.items()})
    assert all(v < TOL for v in errs.values()), errs
    y2, saved2 = run_fwd(d, w.chunk)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(saved.states.view(torch.int32), saved2.states.view(torch.int32))
