"""The allocation-free backward entry point, called through the C ABI.

Callers that cannot allocate device memory use mamba2_ssd_bwd_static_scratch,
whose scratch is a fixed array inside the library.  Its results must match
the regular entry point (given a caller-allocated workspace) within the
tolerance the parity tests use -- here they are expected to be identical --
on two calls in a row (the second call reuses the array the first one
dirtied).  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
from _helpers import relerr, to_dev
from deterministic_mamba2_ssd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

GRADS = ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit")


def _fn():
    L = ssd.lib()
    return L.mamba2_ssd_bwd_static_scratch, L.mamba2_ssd_static_scratch_bytes()


def _empty_like_grads(ref):
    return {k: torch.full_like(v, float("nan")) for k, v in ref.items()}


@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-5), (torch.bfloat16, 2e-3)])
def test_static_scratch_matches_regular_entry_point(dtype, tol):
    f, cap = _fn()
    d = make_inputs(1, 300, 8, 32, 2, 32, dtype=dtype, seed=17, dt_shift=2.0 if dtype == torch.float32 else 4.0,
                    d_mode="normal", with_init=True)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=64, init_states=g["init"])
    assert ssd.bwd_workspace_size(saved.dims, 0, 0) <= cap
    ref = ssd.bwd(saved, g["dout"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = _empty_like_grads(ref)
        rc = f(ctypes.byref(saved.struct), g["dout"].data_ptr(),
               *[ctypes.c_void_p(out[k].data_ptr()) for k in GRADS], 0, stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        for k in GRADS:
            assert relerr(out[k], ref[k].cpu().double().numpy()) <= tol, (call, k)
            assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), (call, k)


def test_static_scratch_rejects_oversized_shapes():
    f, cap = _fn()
    d = make_inputs(1, 4096, 64, 64, 8, 128, dtype=torch.float32, seed=1, dt_shift=4.0)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    assert ssd.bwd_workspace_size(saved.dims, 0, 0) > cap
    outs = [torch.empty(1, device="cuda") for _ in range(6)]
    rc = f(ctypes.byref(saved.struct), g["dout"].data_ptr(), *[o.data_ptr() for o in outs], None, 0, None)
    assert rc == 3   # SSD_ERR_WORKSPACE, nothing launched
