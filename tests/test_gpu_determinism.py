"""Bitwise reproducibility of the CUDA path.

Pattern from the pages: run the same backward repeatedly and require the
bytes to match exactly (a tolerance check cannot detect reordering noise of
about an ulp); use shapes where several writers meet in each reduced element
(heads per group > 1, chunks > 1), otherwise equality holds by construction;
and show that the test has teeth with the atomic variant.
"""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import bits, grads_digest, run_gpu, same_bits, to_dev
from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

REPEATS = 20


def repeat_digests(d, chunk, n, config=0, variant=0):
    """sha256 of the first run's outputs, then, for each further run, that
    digest again if its bits equal the first run's (compared on the GPU) or
    a fresh digest if not."""
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=chunk,
                       seq_idx=g["seq_idx"], init_states=g["init"])
    first = ssd.bwd(saved, g["dout"], config=config, variant=variant)
    torch.cuda.synchronize()
    h0 = grads_digest(first)
    out = [h0]
    for _ in range(n - 1):
        grads = ssd.bwd(saved, g["dout"], config=config, variant=variant)
        torch.cuda.synchronize()
        out.append(h0 if same_bits(first, grads) else grads_digest(grads))
    return out


@pytest.mark.parametrize("name", ["bf16_T2048", "bf16_T16384", "bf16_varlen_T32768"])
def test_bitwise_repeat_20(name):
    w = WORKLOADS[name]
    assert w.nheads // w.ngroups > 1 and w.seqlen // w.chunk > 1   # several writers per reduced element
    hs = repeat_digests(workload_inputs(name), w.chunk, REPEATS)
    assert len(set(hs)) == 1


def test_bitwise_across_every_config():
    cases = [(workload_inputs("bf16_T2048"), 128), (workload_inputs("tiny_fp32"), 64),
             (make_inputs(1, 256, 4, 16, 1, 16, dtype=torch.float32, seed=2, seq_lens=(64, 192),
                          with_init=True), 64),
             (make_inputs(2, 333, 6, 32, 3, 32, dtype=torch.bfloat16, seed=4, dt_shift=4.0), 64)]
    for d, Q in cases:
        dims = ssd.make_dims(d["x"].shape[0], d["x"].shape[1], d["x"].shape[2], d["x"].shape[3],
                             d["B"].shape[2], d["B"].shape[3], Q,
                             nseq=d["init"].shape[0] if d["init"] is not None else None, dtype=d["x"].dtype)
        n = ssd.num_configs(dims)
        assert n >= 2
        digests = {ssd.config_name(dims, c): repeat_digests(d, Q, 2, config=c) for c in range(n)}
        flat = {h for v in digests.values() for h in v}
        assert len(flat) == 1, digests


@pytest.mark.parametrize("name", ["bf16_T16384", "bf16_varlen_T32768", "simt_bf16"])
def test_atomic_variant_shows_the_test_has_teeth(name):
    """The same kernels with atomic accumulation: expected to differ between
    runs at these shapes (fused paths: per-warp dA/dD shares; general path:
    dB/dC/dA/dD).  If they happen not to, the repeat test above is not proof
    of anything and this test says so."""
    if name == "simt_bf16":
        d, Q = make_inputs(1, 2000, 64, 64, 2, 128, dtype=torch.bfloat16, seed=8, dt_shift=4.0), 128
    else:
        d, Q = workload_inputs(name), WORKLOADS[name].chunk
    hs = repeat_digests(d, Q, REPEATS, variant=1)
    if len(set(hs)) == 1:
        pytest.skip("atomic variant was reproducible in %d runs: repeat test non-probative here" % REPEATS)
    assert len(set(hs)) > 1


@pytest.mark.parametrize("case", [
    dict(T=300, H=8, P=32, G=2, N=64, Q=64, path="simt"),
    dict(T=512, H=8, P=64, G=2, N=128, Q=128, path="fused/"),
    dict(T=640, H=8, P=64, G=2, N=128, Q=256, path="fused-chunk128/"),
    dict(T=512, H=8, P=64, G=1, N=256, Q=256, path="fused-split/"),
    dict(T=500, H=4, P=64, G=1, N=128, Q=128, path="fused-padded/", lens=(100, 300, 100)),
    dict(T=700, H=8, P=64, G=1, N=256, Q=256, path="fused-split-padded/", lens=(99, 1, 600)),
])
def test_outputs_fully_written_and_guards_untouched(case):
    """Every output element is written (outputs pre-filled with NaN) and no
    byte outside the outputs or past the workspace size is touched, on each
    kind of path (stores, TMA stores and reduce-adds, folds, scatters)."""
    lens = case.get("lens", ())
    d = make_inputs(1, case["T"], case["H"], case["P"], case["G"], case["N"], dtype=torch.bfloat16, seed=6,
                    dt_shift=4.0, with_init=True, seq_lens=lens)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=case["Q"], seq_idx=g["seq_idx"],
                       init_states=g["init"], any_start=bool(lens))
    assert ssd.config_name(saved.dims, 0).startswith(case["path"]), ssd.config_name(saved.dims, 0)
    pad = 4096
    out, guards = {}, []
    shapes = dict(dx=g["x"].shape, ddt=g["dt"].shape, dA=g["A"].shape, dB=g["B"].shape, dC=g["C"].shape,
                  dD=g["D"].shape, dinit=g["init"].shape)
    for k, shp in shapes.items():
        n = 1
        for s in shp:
            n *= s
        buf = torch.full((n + 2 * pad,), float("nan"), device="cuda")
        buf[:pad] = 7.0
        buf[pad + n:] = 7.0
        out[k] = buf[pad:pad + n].view(shp)
        guards.append((k, buf, n))
    need = ssd.bwd_workspace_size(saved.dims, 0, 0)
    ws = torch.full((need + 65536,), 0xA5, dtype=torch.uint8, device="cuda")
    ssd.bwd(saved, g["dout"], out=out, workspace=ws)
    torch.cuda.synchronize()
    for k, buf, n in guards:
        assert not torch.isnan(out[k]).any(), k
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0), k
    assert torch.all(ws[need:] == 0xA5)
