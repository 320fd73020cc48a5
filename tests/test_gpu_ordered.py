"""The ordered-semaphore dB/dC fold (SSD_VARIANT_ORDERED, general path):
the CTA of head k of a group adds its tile after head k-1 has published, so
every element is summed over heads in the slot fold's order -- the result
must be bit-identical to the default variant, and within tolerance of the
oracle.  Also: not offered on the fused shapes, status word clean."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import GRADS, relerr, run_gpu, run_oracle, same_bits, to_dev
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    dict(T=256, Q=64, H=8, G=2, P=16, N=32),
    dict(T=200, Q=64, H=6, G=3, P=16, N=16),            # ragged last chunk, a tile past its end
    dict(T=130, Q=128, H=4, G=4, P=16, N=16),           # one head per group: no waiting
    dict(T=300, Q=48, H=12, G=1, P=16, N=64, seq=(50, 17, 100, 133)),   # starts inside chunks
    dict(T=160, Q=32, H=4, G=2, P=16, N=256),           # 64 KB tile in shared memory
])
@pytest.mark.parametrize("config", [0, 1])
def test_ordered_equals_slots_bitwise(case, config):
    seq = case.get("seq", ())
    d = make_inputs(1, case["T"], case["H"], case["P"], case["G"], case["N"], dtype=torch.float32,
                    seed=case["T"] + case["N"], dt_shift=2.0, d_mode="normal", seq_lens=seq, with_init=bool(seq))
    g = to_dev(d)
    any_start = bool(seq)
    _, saved, ref_bits = run_gpu(d, case["Q"], config=config, g=g, any_start=any_start)
    out = ssd.bwd(saved, g["dout"], config=config, variant=2)
    torch.cuda.synchronize()
    assert same_bits(out, ref_bits)
    ws = torch.empty(max(16, ssd.bwd_workspace_size(saved.dims, config, 2)), dtype=torch.uint8, device="cuda")
    ssd.bwd(saved, g["dout"], config=config, variant=2, workspace=ws)
    assert ssd.bwd_check(saved, ws, config) == 0
    ref = run_oracle(d, chunk=case["Q"], with_y=False)
    for k in GRADS:
        assert relerr(out[k], ref[k]) < 1e-5, k


def test_ordered_repeats_bitwise():
    d = make_inputs(1, 512, 16, 32, 2, 64, dtype=torch.float32, seed=3, dt_shift=2.0, d_mode="normal")
    g = to_dev(d)
    _, saved, _ = run_gpu(d, 64, g=g)
    runs = [ssd.bwd(saved, g["dout"], variant=2) for _ in range(5)]
    for r in runs[1:]:
        assert same_bits(r, runs[0])


def test_ordered_not_offered_on_fused_shapes():
    d = make_inputs(1, 256, 4, 64, 1, 128, dtype=torch.bfloat16, seed=1, dt_shift=4.0, d_mode="normal")
    g = to_dev(d)
    _, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    assert ssd.bwd_workspace_size(saved.dims, 0, 2) == 0
    with pytest.raises(ssd.SsdError) as e:
        ssd.bwd(saved, g["dout"], variant=2, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 2
