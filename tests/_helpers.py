"""Shared helpers of the GPU tests: run the CUDA path and the oracle on the
same seeded inputs and compare them."""
from __future__ import annotations

import hashlib

import numpy as np
import torch

import deterministic_mamba2_ssd_gb300 as ssd
import oracle

GRADS = ("dx", "ddt", "dA", "dB", "dC", "dD")


def relerr(gpu, ref):
    """relL2 = ||gpu - ref|| / ||ref|| in fp64 after exact widening."""
    a = gpu.detach().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    b = np.asarray(ref, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def y_relerr(y, y_ref):
    """relL2 of a forward output y against the oracle's fp64 y.  For a bf16 y
    the oracle value is rounded to bf16 first: the GPU must round its own y,
    and that output rounding alone is ~1.7e-3 relL2 on N(0,1) data, which is
    not an error of the computation."""
    if y.dtype == torch.bfloat16:
        y_ref = torch.from_numpy(np.asarray(y_ref, np.float64)).to(torch.bfloat16).double().numpy()
    return relerr(y, y_ref)


def to_dev(d, dev="cuda"):
    return {k: (v.to(dev) if v is not None else None) for k, v in d.items()}


def run_gpu(d, chunk, config=0, variant=0, g=None, any_start=False):
    g = to_dev(d) if g is None else g
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=chunk,
                       seq_idx=g["seq_idx"], init_states=g["init"], any_start=any_start)
    grads = ssd.bwd(saved, g["dout"], config=config, variant=variant)
    torch.cuda.synchronize()
    return y, saved, grads


def run_oracle(d, chunk=0, with_y=True):
    kw = dict(seq_idx=d["seq_idx"], init=d["init"])
    out = {}
    if with_y:
        r = oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk=chunk, **kw)
        out["y"], out["states"] = (r if chunk else (r, None))
    out.update(oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], **kw))
    return out


def digest(tensors):
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def grads_digest(grads):
    return digest([grads[k] for k in sorted(grads)])


def bits(t):
    """Integer view of a float tensor: equality of bits, not of values."""
    return t.detach().contiguous().view(torch.int32 if t.element_size() == 4 else torch.int16)


def same_bits(a, b):
    return all(torch.equal(bits(a[k]), bits(b[k])) for k in a)


def head_slice(d, g0, hpg):
    """Sub-problem of one group: heads [g0*hpg, (g0+1)*hpg) with that group's
    B and C (groups never interact, so the oracle can run it alone)."""
    h0, h1 = g0 * hpg, (g0 + 1) * hpg
    out = dict(d)
    for k in ("x", "dout"):
        out[k] = d[k][:, :, h0:h1].contiguous()
    out["dt"] = d["dt"][:, :, h0:h1].contiguous()
    out["A"] = d["A"][h0:h1].contiguous()
    out["D"] = d["D"][h0:h1].contiguous()
    out["B"] = d["B"][:, :, g0:g0 + 1].contiguous()
    out["C"] = d["C"][:, :, g0:g0 + 1].contiguous()
    if d["init"] is not None:
        out["init"] = d["init"][:, h0:h1].contiguous()
    return out
