"""Parity of the adjacent-step kernels (step-size preprocessing, z-gate)
with the fp64 oracle in oracle/adjacent.py, element by element.

fp32 arithmetic on both inputs dtypes: relL2 <= 1e-6 for fp32 outputs (a few
ulp from expf/log1pf), and for bf16 outputs the oracle's value rounded to
bf16 must match within one bf16 ulp elementwise.  The dt_bias gradient is a
fixed-order reduction: bitwise equal across repeated runs.
"""
import numpy as np
import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd
import oracle.adjacent as adj
from _helpers import relerr

pytestmark = pytest.mark.gpu

INF = float("inf")


def inputs(rows, H, seed):
    g = torch.Generator().manual_seed(seed)
    raw = torch.randn((rows, H), generator=g) * 3 - 2
    bias = torch.randn((H,), generator=g)
    ddt = torch.randn((rows, H), generator=g)
    return raw, bias, ddt


@pytest.mark.parametrize("rows,H,softplus,lo,hi,bias", [
    (16384, 256, True, 0.0, INF, True),        # the 16K workload's step-size tensor
    (1000, 8, True, 0.001, 0.1, True),         # ragged tile, clamp on both sides
    (77, 6, False, -1.0, 1.0, False),          # heads not a multiple of 4 (scalar path)
    (1, 3, True, 0.0, INF, False),
    (130, 300, True, 0.01, 5.0, True),         # more heads than threads per CTA
])
def test_dt_parity(rows, H, softplus, lo, hi, bias):
    raw, b, ddt = inputs(rows, H, rows + H)
    b = b if bias else None
    dev = lambda t: None if t is None else t.cuda()
    dt = ssd.dt_fwd(dev(raw), dev(b), softplus, lo, hi)
    ddt_raw, ddt_bias = ssd.dt_bwd(dev(raw), dev(ddt), dev(b), softplus, lo, hi)
    ref = adj.dt_fwd(raw, b, softplus, lo, hi)
    rraw, rbias = adj.dt_bwd(raw, ddt, b, softplus, lo, hi)
    assert relerr(dt, ref) < 1e-6
    assert relerr(ddt_raw, rraw) < 1e-6
    assert relerr(ddt_bias, rbias) < 1e-5
    # the clamp decides which gradients are zero: both sides agree on the mask
    # except where fp32 and fp64 straddle a bound (none expected at these sizes)
    assert torch.equal(ddt_raw.cpu() == 0, torch.from_numpy(rraw == 0))


def test_dt_bias_grad_bitwise_repeat():
    raw, b, ddt = (t.cuda() for t in inputs(16384, 256, 9))
    first = ssd.dt_bwd(raw, ddt, b)[1]
    for _ in range(5):
        assert torch.equal(ssd.dt_bwd(raw, ddt, b)[1].view(torch.int32), first.view(torch.int32))


def test_dt_empty_rows():
    raw = torch.empty((0, 4), device="cuda")
    ddt_raw, ddt_bias = ssd.dt_bwd(raw, raw.clone(), None)
    assert ddt_raw.numel() == 0 and torch.count_nonzero(ddt_bias) == 0


@pytest.mark.parametrize("dtype,n", [(torch.float32, 4096 * 64 + 3), (torch.bfloat16, 16384 * 64 * 4 + 5),
                                     (torch.bfloat16, 7), (torch.float32, 1)])
def test_gate_parity(dtype, n):
    g = torch.Generator().manual_seed(n)
    y = torch.randn(n, generator=g).to(dtype)
    z = (torch.randn(n, generator=g) * 4).to(dtype)
    dout = torch.randn(n, generator=g).to(dtype)
    out = ssd.gate_fwd(y.cuda(), z.cuda())
    dy, dz = ssd.gate_bwd(y.cuda(), z.cuda(), dout.cuda())
    rout = adj.gate_fwd(y, z)
    rdy, rdz = adj.gate_bwd(y, z, dout)
    assert relerr(dz, rdz) < 1e-6
    if dtype == torch.float32:
        assert relerr(out, rout) < 1e-6 and relerr(dy, rdy) < 1e-6
    else:
        # one rounding to bf16 of an fp32 value within a few ulp of the exact one
        for got, want in ((out, rout), (dy, rdy)):
            w = torch.from_numpy(want)
            ulp = torch.where(w == 0, torch.full_like(w, 2.0 ** -133), w.abs() * 2.0 ** -7)
            assert torch.all((got.cpu().double() - w).abs() <= ulp)
