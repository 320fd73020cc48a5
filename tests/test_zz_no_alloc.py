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


def _check_fn():
    return ssd.lib().mamba2_ssd_static_scratch_check


def _call_static(f, saved, dout, out, config):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.byref(saved.struct), dout.data_ptr(),
             *[ctypes.c_void_p(out[k].data_ptr()) if k in out else None for k in GRADS], config, stream)


@pytest.mark.parametrize("config", [0, 1])
def test_static_scratch_runs_the_fused_tensor_core_path(config):
    """The fused kernel keeps its ticket, chain flags and state-gradient ring in
    the scratch; the second call finds them dirty from the first."""
    f, cap = _fn()
    d = make_inputs(1, 512, 4, 64, 1, 128, dtype=torch.bfloat16, seed=23, dt_shift=4.0, d_mode="normal",
                    with_init=True)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128, init_states=g["init"])
    assert ssd.config_name(saved.dims, config).startswith("fused")
    assert ssd.bwd_workspace_size(saved.dims, config, 0) <= cap
    ref = ssd.bwd(saved, g["dout"], config=config)
    for call in range(2):
        out = _empty_like_grads(ref)
        assert _call_static(f, saved, g["dout"], out, config) == 0
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert _check_fn()(ctypes.byref(saved.dims), config, stream) == 0
        torch.cuda.synchronize()
        for k in ref:
            assert relerr(out[k], ref[k].cpu().double().numpy()) <= 2e-3, (call, k)
            assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), (call, k)


def test_static_scratch_headline_shape_fits_with_the_shallow_ring_only():
    """bf16, seqlen 16384, 256 heads of 64, 8 groups, dstate 128, chunk 128: the
    ring of depth 4 needs 32 MiB on its own, so config 0 does not fit the array
    and is refused; config 1 (ring depth 2) fits and runs the fused kernel."""
    from deterministic_mamba2_ssd_gb300.inputs import workload_inputs
    f, cap = _fn()
    g = to_dev(workload_inputs("bf16_T16384"))
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    assert ssd.bwd_workspace_size(saved.dims, 0, 0) > cap >= ssd.bwd_workspace_size(saved.dims, 1, 0)
    ref = ssd.bwd(saved, g["dout"], config=1)
    out = _empty_like_grads(ref)
    assert _call_static(f, saved, g["dout"], out, 0) == 3   # SSD_ERR_WORKSPACE, nothing launched
    assert _call_static(f, saved, g["dout"], out, 1) == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _check_fn()(ctypes.byref(saved.dims), 1, stream) == 0
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), k


def test_static_scratch_rejects_oversized_shapes():
    f, cap = _fn()
    d = make_inputs(1, 4096, 64, 64, 8, 128, dtype=torch.float32, seed=1, dt_shift=4.0)
    g = to_dev(d)
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=128)
    assert ssd.bwd_workspace_size(saved.dims, 0, 0) > cap
    outs = [torch.empty(1, device="cuda") for _ in range(6)]
    rc = f(ctypes.byref(saved.struct), g["dout"].data_ptr(), *[o.data_ptr() for o in outs], None, 0, None)
    assert rc == 3   # SSD_ERR_WORKSPACE, nothing launched
