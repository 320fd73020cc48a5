"""bf16 problems with dstate 128 and a chunk that is a larger multiple of 128
(256 as in Mamba2's defaults, and 512) on the fused tensor-core kernels run
in 128-token chunks ("fused-chunk128"), against the fp64 oracle at the
caller's chunk length: y (against the oracle's y rounded to bf16), the state
entering each of the caller's chunks, every gradient and dinit.  Also, since
y, the gradients and the chunk-entry states of the recurrence do not depend
on the chunk length ("Mamba2 / state space duality": the chunked form is the
recurrence regrouped), the run is compared bit for bit with the same inputs
at chunk 128; and with sequence starts inside a chunk the padded form takes
the caller's chunk 256 as well.  Parity bar: relL2 2e-3 per tensor."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, bits, relerr, run_gpu, run_oracle, same_bits, to_dev, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3

CASES = [
    dict(b=1, T=512, H=4, G=1, Q=256),
    dict(b=2, T=640, H=8, G=2, Q=256, with_init=True),                 # a short last chunk
    dict(b=1, T=1024, H=4, G=1, Q=256, seq_lens=(256, 512, 256), with_init=True),
    dict(b=1, T=1024, H=6, G=2, Q=512),
]


def inputs(case):
    return make_inputs(case["b"], case["T"], case["H"], 64, case["G"], 128, dtype=torch.bfloat16,
                       seed=case["T"] + 7 * case["H"] + case["Q"], dt_shift=4.0, d_mode="normal",
                       seq_lens=case.get("seq_lens", ()), with_init=case.get("with_init", False))


@pytest.mark.parametrize("case", CASES)
def test_chunk128_form_matches_oracle(case):
    d = inputs(case)
    y, saved, g = run_gpu(d, case["Q"])
    assert ssd.config_name(saved.dims, 0) == "fused-chunk128/ring4", ssd.config_name(saved.dims, 0)
    ref = run_oracle(d, chunk=case["Q"])
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print(case, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)


@pytest.mark.parametrize("case", CASES[:3])
def test_chunk128_form_equals_the_chunk_128_run_bit_for_bit(case):
    d = inputs(case)
    g_dev = to_dev(d)
    y, saved, g = run_gpu(d, case["Q"], g=g_dev)
    y1, saved1, g1 = run_gpu(d, 128, g=g_dev)
    assert ssd.config_name(saved1.dims, 0) == "fused/ring4"
    assert torch.equal(bits(y), bits(y1))
    assert same_bits(g, g1)
    ratio = case["Q"] // 128
    st, st1 = saved.states_fp32(), saved1.states_fp32()
    assert torch.equal(bits(st), bits(st1[:, ::ratio].contiguous()))


def test_chunk128_form_bitwise_across_runs_and_configs_with_clean_status():
    d = inputs(CASES[2])
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=256, seq_idx=g["seq_idx"],
                       init_states=g["init"])
    assert ssd.fwd_check(saved) == 0
    first = ssd.bwd(saved, g["dout"])
    for config in range(ssd.num_configs(saved.dims)):
        ws = torch.empty(ssd.bwd_workspace_size(saved.dims, config, 0), dtype=torch.uint8, device="cuda")
        for _ in range(3):
            assert same_bits(first, ssd.bwd(saved, g["dout"], config=config, workspace=ws)), config
            assert ssd.bwd_check(saved, ws, config) == 0


def test_padded_form_takes_the_callers_chunk_256():
    lens = (100, 300, 1, 111)
    d = make_inputs(1, sum(lens), 4, 64, 1, 128, dtype=torch.bfloat16, seed=4242, dt_shift=4.0, d_mode="normal",
                    seq_lens=lens, with_init=True)
    y, saved, g = run_gpu(d, 256, any_start=True)
    assert ssd.config_name(saved.dims, 0) == "fused-padded/0"
    ref = run_oracle(d, chunk=256)
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"]),
            "dinit": relerr(g["dinit"], ref["dinit"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    print({k: "%.2e" % v for k, v in errs.items()})
    assert all(v < TOL for v in errs.values()), errs
