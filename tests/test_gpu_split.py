"""The fused tensor-core path on dstate 256 with one group ("fused-split":
the fused kernels run once per 128-wide state half, in 128-token chunks, and
the halves' contributions are summed in a fixed order) against the fp64
oracle: y (against the oracle's y rounded to bf16), the saved states, every
gradient and dinit, on shapes with chunk 128 and 256, several batch rows,
odd head counts, initial states and packed sequences; and its determinism.
Parity bar: relL2 2e-3 per tensor (bf16 inputs, fp32 accumulation)."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, digest, relerr, run_gpu, run_oracle, same_bits, to_dev, y_relerr
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.mark.parametrize("case", [
    dict(b=1, T=512, H=4, Q=256),
    dict(b=2, T=256, H=4, Q=128, with_init=True),
    dict(b=1, T=1024, H=6, Q=256, seq_lens=(256, 512, 256), with_init=True),
    dict(b=1, T=768, H=2, Q=256, dt_shift=2.0),      # strong decay
    dict(b=1, T=512, H=64, Q=256, with_init=True),   # 64 heads: the forward's head slices, 16 per backward slice
])
def test_split_matches_oracle(case):
    d = make_inputs(case["b"], case["T"], case["H"], 64, 1, 256, dtype=torch.bfloat16, seed=case["T"] + case["H"],
                    dt_shift=case.get("dt_shift", 4.0), d_mode="normal", seq_lens=case.get("seq_lens", ()),
                    with_init=case.get("with_init", False))
    y, saved, g = run_gpu(d, case["Q"])
    assert ssd.config_name(saved.dims, 0).startswith("fused-split"), ssd.config_name(saved.dims, 0)
    ref = run_oracle(d, chunk=case["Q"])
    errs = {"y": y_relerr(y, ref["y"]), "states": relerr(saved.states_fp32(), ref["states"])}
    errs.update({k: relerr(g[k], ref[k]) for k in GRADS})
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print(case, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)


def test_split_bitwise_across_runs_and_configs():
    d = make_inputs(1, 1024, 8, 64, 1, 256, dtype=torch.bfloat16, seed=5, dt_shift=4.0, d_mode="normal",
                    seq_lens=(512, 256, 256), with_init=True)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=256, seq_idx=g["seq_idx"],
                       init_states=g["init"])
    first = ssd.bwd(saved, g["dout"])
    for config in range(ssd.num_configs(saved.dims)):
        for _ in range(5):
            assert same_bits(first, ssd.bwd(saved, g["dout"], config=config)), config


def test_split_status_word_is_clean():
    d = make_inputs(1, 512, 4, 64, 1, 256, dtype=torch.bfloat16, seed=2, dt_shift=4.0)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=256)
    ws = torch.empty(ssd.bwd_workspace_size(saved.dims, 0, 0), dtype=torch.uint8, device="cuda")
    ssd.bwd(saved, g["dout"], workspace=ws)
    assert ssd.bwd_check(saved, ws) == 0
    assert ssd.fwd_check(saved) == 0
