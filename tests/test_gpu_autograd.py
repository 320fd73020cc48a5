"""The autograd wrapper hands tensors to the library and back: its gradients
are the library's backward, bit for bit (cast to each input's dtype)."""
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import same_bits, to_dev
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,T,P,N,Q", [(torch.float32, 200, 16, 16, 64), (torch.bfloat16, 256, 64, 128, 128)])
def test_autograd_matches_direct_backward(dtype, T, P, N, Q):
    d = to_dev(make_inputs(1, T, 4, P, 1, N, dtype=dtype, seed=4, dt_shift=2.0, d_mode="normal", with_init=True))
    leaves = {k: d[k].clone().requires_grad_(True) for k in ("x", "dt", "A", "B", "C", "D", "init")}
    y = ssd.ssd(leaves["x"], leaves["dt"], leaves["A"], leaves["B"], leaves["C"], leaves["D"], Q,
                init_states=leaves["init"])
    y.backward(d["dout"])
    y2, saved = ssd.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], Q, init_states=d["init"])
    ref = ssd.bwd(saved, d["dout"])
    torch.cuda.synchronize()
    assert torch.equal(y.detach().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       y2.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init": "dinit"}
    got = {names[k]: v.grad for k, v in leaves.items()}
    want = {k: ref[k].to(got[k].dtype) for k in got}
    assert same_bits(got, want)
