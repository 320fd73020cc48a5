"""The fused tensor-core backward (bf16, chunk 128, dstate 128, headdim 64)
against the fp64 oracle on small shapes that still span several chunks,
several heads per group, batch rows, initial states and packed sequences;
plus its status word and its bounded-wait fault injection."""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, relerr, run_gpu, run_oracle, to_dev
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def dims_of(d, Q=128):
    return ssd.make_dims(d["x"].shape[0], d["x"].shape[1], d["x"].shape[2], d["x"].shape[3], d["B"].shape[2],
                         d["B"].shape[3], Q, nseq=d["init"].shape[0] if d["init"] is not None else None,
                         dtype=d["x"].dtype, seq_idx=d["seq_idx"] is not None)


@pytest.mark.parametrize("case", [
    dict(b=1, T=128, H=2, G=1),
    dict(b=1, T=384, H=8, G=2),
    dict(b=2, T=256, H=4, G=2, with_init=True),
    dict(b=1, T=256, H=3, G=3),              # one head per group
    dict(b=1, T=512, H=6, G=2),              # odd heads per group
    dict(b=1, T=512, H=4, G=1, seq_lens=(128, 256, 128), with_init=True),
    dict(b=1, T=1024, H=32, G=1, dt_shift=2.0),   # strong decay: large |cumulative decay|
])
def test_fused_matches_oracle(case):
    d = make_inputs(case["b"], case["T"], case["H"], 64, case["G"], 128, dtype=torch.bfloat16, seed=case["T"] + case["H"],
                    dt_shift=case.get("dt_shift", 4.0), d_mode="normal", seq_lens=case.get("seq_lens", ()),
                    with_init=case.get("with_init", False))
    dims = dims_of(d)
    assert ssd.config_name(dims, 0).startswith("fused"), ssd.config_name(dims, 0)
    y, saved, g = run_gpu(d, 128)
    ref = run_oracle(d, chunk=128)
    errs = {k: relerr(g[k], ref[k]) for k in GRADS}
    if d["init"] is not None:
        errs["dinit"] = relerr(g["dinit"], ref["dinit"])
    print(case, {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, (bad, errs)


def test_fused_status_word_is_clean():
    d = make_inputs(1, 256, 4, 64, 1, 128, dtype=torch.bfloat16, seed=2, dt_shift=4.0)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    ws = torch.empty(ssd.bwd_workspace_size(saved.dims, 0, 0), dtype=torch.uint8, device="cuda")
    ssd.bwd(saved, g["dout"], workspace=ws)
    assert ssd.bwd_check(saved, ws) == 0
    assert ssd.fwd_check(saved) == 0


def test_fused_chain_wait_gives_up_and_reports():
    """A chunk whose units never publish their state gradient: the unit of
    the chunk before it must give up after a short bounded wait, report
    SSD_ERR_TIMEOUT, and leave the context usable."""
    d = make_inputs(1, 512, 4, 64, 1, 128, dtype=torch.bfloat16, seed=3, dt_shift=4.0)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    need = ssd.bwd_workspace_size(saved.dims, 0, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = {k: torch.empty_like(v, dtype=torch.float32) for k, v in
           dict(dx=g["x"], ddt=g["dt"], dA=g["A"], dB=g["B"], dC=g["C"], dD=g["D"]).items()}
    L = ssd.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.mamba2_ssd_bwd_fault_test(ctypes.byref(saved.struct), g["dout"].data_ptr(),
                                     *[out[k].data_ptr() for k in ("dx", "ddt", "dA", "dB", "dC", "dD")], None,
                                     ws.data_ptr(), need, 3, 2000, stream)
    assert rc == 0
    assert ssd.bwd_check(saved, ws) == 5        # SSD_ERR_TIMEOUT
    # the context is still usable and a normal call is correct again
    good = ssd.bwd(saved, g["dout"], workspace=ws)
    assert ssd.bwd_check(saved, ws) == 0
    ref = run_oracle(d, chunk=128, with_y=False)
    assert relerr(good["dx"], ref["dx"]) < TOL
