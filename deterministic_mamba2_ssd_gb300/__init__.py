"""Deterministic Mamba2 SSD chunked scan for GB300 -- thin Python binding.

The compute lives in ``libmamba2_ssd.so`` (hand-written CUDA for sm_103a,
C ABI declared in ``include/mamba2_ssd.h``).  This module only marshals
arguments: it checks shapes, allocates outputs and workspace with PyTorch's
device allocator and passes raw pointers and the current CUDA stream to the
library.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["lib", "fwd", "bwd", "Saved", "SsdError", "make_dims", "num_configs", "config_name",
           "bwd_workspace_size", "fwd_workspace_size", "bwd_num_launches", "bwd_launch_names", "LIB_PATH",
           "dt_fwd", "dt_bwd", "gate_fwd", "gate_bwd", "conv1d_fwd", "conv1d_bwd", "SSDFunction", "ssd"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmamba2_ssd.so")

SSD_F32, SSD_BF16 = 0, 1
VARIANT_DETERMINISTIC, VARIANT_ATOMIC = 0, 1
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_WORKSPACE",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_HANDLE"}


class SsdError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (what, STATUS.get(status, status),
                                                   lib().mamba2_ssd_status_string(status).decode()))


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("nseq", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class SavedStruct(ctypes.Structure):
    _fields_ = [("dims", Dims)] + [(n, ctypes.c_void_p) for n in
                                   ("x", "dt", "A", "B", "C", "D", "seq_idx", "init_states", "states", "aux")] + \
               [("magic", ctypes.c_uint32), ("flags", ctypes.c_uint32)]


_lib = None


def lib():
    """The loaded CUDA library (raises if it is absent: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmamba2_ssd.so is not built (run __graft_entry__.build()); "
                               "this package has no CPU or PyTorch fallback")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, ci, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
        pd = ctypes.POINTER(Dims)
        L.mamba2_ssd_status_string.argtypes = [ci]
        L.mamba2_ssd_status_string.restype = ctypes.c_char_p
        L.mamba2_ssd_num_chunks.argtypes = [pd]
        L.mamba2_ssd_num_chunks.restype = i64
        L.mamba2_ssd_fwd_workspace_size.argtypes = [pd]
        L.mamba2_ssd_fwd_workspace_size.restype = sz
        L.mamba2_ssd_bwd_workspace_size.argtypes = [pd, ci, ci]
        L.mamba2_ssd_bwd_workspace_size.restype = sz
        L.mamba2_ssd_num_configs.argtypes = [pd]
        L.mamba2_ssd_num_configs.restype = ci
        L.mamba2_ssd_config_name.argtypes = [pd, ci]
        L.mamba2_ssd_config_name.restype = ctypes.c_char_p
        L.mamba2_ssd_bwd_num_launches.argtypes = [pd, ci, ci]
        L.mamba2_ssd_bwd_num_launches.restype = ci
        L.mamba2_ssd_fwd.argtypes = [pd] + [vp] * 10 + [vp, sz, vp, ctypes.POINTER(SavedStruct)]
        L.mamba2_ssd_fwd.restype = ci
        L.mamba2_ssd_bwd.argtypes = [ctypes.POINTER(SavedStruct)] + [vp] * 9 + [sz, ci, ci, vp]
        L.mamba2_ssd_bwd.restype = ci
        L.mamba2_ssd_bwd_traced.argtypes = [ctypes.POINTER(SavedStruct)] + [vp] * 9 + [sz, ci, ci, vp, vp, ci]
        L.mamba2_ssd_bwd_traced.restype = ci
        L.mamba2_ssd_bwd_launch_name.argtypes = [pd, ci, ci, ci]
        L.mamba2_ssd_bwd_launch_name.restype = ctypes.c_char_p
        L.mamba2_ssd_bwd_check.argtypes = [pd, ci, vp, vp]
        L.mamba2_ssd_bwd_check.restype = ci
        L.mamba2_ssd_fwd_check.argtypes = [pd, vp, vp]
        L.mamba2_ssd_fwd_check.restype = ci
        L.mamba2_ssd_bwd_fault_test.argtypes = [ctypes.POINTER(SavedStruct)] + [vp] * 9 + [sz, i64, ctypes.c_uint32,
                                                                                           vp]
        L.mamba2_ssd_bwd_fault_test.restype = ci
        L.mamba2_ssd_states_unpack.argtypes = [ctypes.POINTER(SavedStruct), vp, vp]
        L.mamba2_ssd_states_unpack.restype = ci
        L.mamba2_ssd_padded_chunks.argtypes = [pd]
        L.mamba2_ssd_padded_chunks.restype = i64
        L.mamba2_ssd_padded_piece_table.argtypes = [pd, vp, vp]
        L.mamba2_ssd_padded_piece_table.restype = ci
        L.mamba2_ssd_selftest_umma.argtypes = [vp] * 3 + [ci] * 6 + [vp]
        L.mamba2_ssd_selftest_umma.restype = ci
        L.mamba2_ssd_static_scratch_bytes.argtypes = []
        L.mamba2_ssd_static_scratch_bytes.restype = sz
        L.mamba2_ssd_bwd_static_scratch.argtypes = [ctypes.POINTER(SavedStruct)] + [vp] * 8 + [ci, vp]
        L.mamba2_ssd_bwd_static_scratch.restype = ci
        L.mamba2_ssd_static_scratch_check.argtypes = [pd, ci, vp]
        L.mamba2_ssd_static_scratch_check.restype = ci
        f32 = ctypes.c_float
        L.mamba2_ssd_dt_fwd.argtypes = [i64, i64, vp, vp, ci, f32, f32, vp, vp]
        L.mamba2_ssd_dt_fwd.restype = ci
        L.mamba2_ssd_dt_bwd_workspace_size.argtypes = [i64, i64]
        L.mamba2_ssd_dt_bwd_workspace_size.restype = sz
        L.mamba2_ssd_dt_bwd.argtypes = [i64, i64, vp, vp, ci, f32, f32, vp, vp, vp, vp, sz, vp]
        L.mamba2_ssd_dt_bwd.restype = ci
        L.mamba2_ssd_gate_fwd.argtypes = [i64, ctypes.c_int32, vp, vp, vp, vp]
        L.mamba2_ssd_gate_fwd.restype = ci
        L.mamba2_ssd_gate_bwd.argtypes = [i64, ctypes.c_int32, vp, vp, vp, vp, vp, vp]
        L.mamba2_ssd_gate_bwd.restype = ci
        i32 = ctypes.c_int32
        L.mamba2_ssd_conv1d_num_configs.argtypes = []
        L.mamba2_ssd_conv1d_num_configs.restype = ci
        L.mamba2_ssd_conv1d_fwd.argtypes = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, ci, vp]
        L.mamba2_ssd_conv1d_fwd.restype = ci
        L.mamba2_ssd_conv1d_bwd_workspace_size.argtypes = [i64, i64, i64, i32]
        L.mamba2_ssd_conv1d_bwd_workspace_size.restype = sz
        L.mamba2_ssd_conv1d_bwd.argtypes = [i64, i64, i64, i32, i32, i32] + [vp] * 9 + [sz, ci, ci, vp]
        L.mamba2_ssd_conv1d_bwd.restype = ci
        _lib = L
    return _lib


DIMS_SEQ_IDX = 1
DIMS_SEQ_ANY_START = 2


def make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, nseq=None, dtype=torch.bfloat16,
              seq_idx=False, any_start=False):
    return Dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size,
                batch if nseq is None else nseq, SSD_BF16 if dtype == torch.bfloat16 else SSD_F32,
                (DIMS_SEQ_IDX if seq_idx else 0) | (DIMS_SEQ_ANY_START if any_start else 0))


def num_configs(dims: Dims) -> int:
    return lib().mamba2_ssd_num_configs(ctypes.byref(dims))


def config_name(dims: Dims, config: int) -> str:
    return lib().mamba2_ssd_config_name(ctypes.byref(dims), config).decode()


def fwd_workspace_size(dims: Dims) -> int:
    return lib().mamba2_ssd_fwd_workspace_size(ctypes.byref(dims))


def bwd_workspace_size(dims: Dims, config: int = 0, variant: int = 0) -> int:
    return lib().mamba2_ssd_bwd_workspace_size(ctypes.byref(dims), config, variant)


def bwd_num_launches(dims: Dims, config: int = 0, variant: int = 0) -> int:
    return lib().mamba2_ssd_bwd_num_launches(ctypes.byref(dims), config, variant)


def bwd_launch_names(dims: Dims, config: int = 0, variant: int = 0):
    n = bwd_num_launches(dims, config, variant)
    return [lib().mamba2_ssd_bwd_launch_name(ctypes.byref(dims), config, variant, k).decode() for k in range(n)]


def bwd_check(saved: "Saved", workspace, config: int = 0, stream=None) -> int:
    """Status word the device left in ``workspace`` after a backward."""
    return lib().mamba2_ssd_bwd_check(ctypes.byref(saved.dims), config, _ptr(workspace), _stream(stream))


def fwd_check(saved: "Saved", stream=None) -> int:
    """Status word the device left in the forward's workspace (kept with ``saved``)."""
    return lib().mamba2_ssd_fwd_check(ctypes.byref(saved.dims), _ptr(saved.tensors["ws"]), _stream(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, shape, dtype, device):
    if t is None:
        raise ValueError("%s is required" % name)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise ValueError("%s: expected contiguous %s %s on %s, got %s %s %s" %
                         (name, tuple(shape), dtype, device, tuple(t.shape), t.dtype, t.device))


class Saved:
    """What the backward needs: the filled C struct plus references that keep
    the borrowed tensors (inputs and chunk states) alive."""

    def __init__(self, struct, tensors, dims):
        self.struct = struct
        self.tensors = tensors
        self.dims = dims

    @property
    def states(self):
        """The saved-state buffer as the backward takes it (packed on the fused shapes)."""
        return self.tensors["states"]

    def states_fp32(self, stream=None):
        """fp32 (b, nc, H, P, N) view of the saved chunk states (a new tensor)."""
        out = torch.empty_like(self.tensors["states"])
        rc = lib().mamba2_ssd_states_unpack(ctypes.byref(self.struct), _ptr(out), _stream(stream))
        if rc:
            raise SsdError(rc, "mamba2_ssd_states_unpack")
        return out


def fwd(x, dt, A, B, C, D, chunk_size, seq_idx=None, init_states=None, stream=None, any_start=False):
    """Forward.  Returns (y, saved).  x (b,T,H,P) and B, C (b,T,G,N) in
    bf16 or fp32; dt (b,T,H), A (H), D (H), init_states (nseq,H,P,N) fp32;
    seq_idx (1,T) int32, non-decreasing, with sequence starts at multiples of
    chunk_size unless ``any_start`` (starts anywhere: the padded fused form on
    the bf16 fused shapes, the general kernels otherwise)."""
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    nseq = init_states.shape[0] if init_states is not None else (
        int(seq_idx.max().item()) + 1 if seq_idx is not None else b)
    _check(x, "x", (b, T, H, P), x.dtype, dev)
    _check(dt, "dt", (b, T, H), torch.float32, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(B, "B", (b, T, G, N), x.dtype, dev)
    _check(C, "C", (b, T, G, N), x.dtype, dev)
    _check(D, "D", (H,), torch.float32, dev)
    if seq_idx is not None:
        _check(seq_idx, "seq_idx", (b, T), torch.int32, dev)
    if init_states is not None:
        _check(init_states, "init_states", (nseq, H, P, N), torch.float32, dev)
    if any_start and seq_idx is None:
        raise ValueError("any_start needs seq_idx")
    dims = make_dims(b, T, H, P, G, N, chunk_size, nseq, x.dtype, seq_idx=seq_idx is not None,
                     any_start=any_start)
    nc = lib().mamba2_ssd_num_chunks(ctypes.byref(dims))
    if nc < 0:
        raise ValueError("invalid dims")
    y = torch.empty_like(x)
    states = torch.empty((b, nc, H, P, N), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, fwd_workspace_size(dims)), dtype=torch.uint8, device=dev)
    sv = SavedStruct()
    rc = lib().mamba2_ssd_fwd(ctypes.byref(dims), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                              _ptr(seq_idx), _ptr(init_states), _ptr(y), _ptr(states), _ptr(ws), ws.numel(),
                              _stream(stream), ctypes.byref(sv))
    if rc:
        raise SsdError(rc, "mamba2_ssd_fwd")
    keep = dict(x=x, dt=dt, A=A, B=B, C=C, D=D, seq_idx=seq_idx, init=init_states, states=states, ws=ws)
    return y, Saved(sv, keep, dims)


def bwd(saved: Saved, dout, config: int = 0, variant: int = VARIANT_DETERMINISTIC, stream=None, out=None,
        workspace=None, events=None):
    """Backward of sum(y * dout).  Returns dict of fp32 tensors dx, ddt, dA,
    dB, dC, dD (and dinit when the forward had initial states).  ``out`` may
    supply preallocated outputs and ``workspace`` a uint8 buffer."""
    t = saved.tensors
    x = t["x"]
    dev = x.device
    _check(dout, "dout", tuple(x.shape), x.dtype, dev)
    if out is None:
        out = dict(dx=torch.empty(x.shape, dtype=torch.float32, device=dev),
                   ddt=torch.empty(t["dt"].shape, dtype=torch.float32, device=dev),
                   dA=torch.empty(t["A"].shape, dtype=torch.float32, device=dev),
                   dB=torch.empty(t["B"].shape, dtype=torch.float32, device=dev),
                   dC=torch.empty(t["C"].shape, dtype=torch.float32, device=dev),
                   dD=torch.empty(t["D"].shape, dtype=torch.float32, device=dev))
        if t["init"] is not None:
            out["dinit"] = torch.empty(t["init"].shape, dtype=torch.float32, device=dev)
    need = bwd_workspace_size(saved.dims, config, variant)
    if workspace is None:
        workspace = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
    args = (ctypes.byref(saved.struct), _ptr(dout), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
            _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out.get("dinit")), _ptr(workspace),
            workspace.numel(), config, variant, _stream(stream))
    if events is None:
        rc = lib().mamba2_ssd_bwd(*args)
    else:
        # events: recorded torch.cuda.Event objects (enable_timing=True)
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        rc = lib().mamba2_ssd_bwd_traced(*args, arr, len(events))
    if rc:
        raise SsdError(rc, "mamba2_ssd_bwd")
    return out


# ---- steps either side of the scan ------------------------------------------

def _dt_check(dt_raw, dt_bias):
    if dt_raw.dim() < 2:
        raise ValueError("dt_raw must be (..., nheads)")
    H = dt_raw.shape[-1]
    _check(dt_raw, "dt_raw", tuple(dt_raw.shape), torch.float32, dt_raw.device)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", (H,), torch.float32, dt_raw.device)
    return dt_raw.numel() // H, H


def dt_fwd(dt_raw, dt_bias=None, softplus=True, dt_min=0.0, dt_max=float("inf"), stream=None):
    """dt = clamp(softplus(dt_raw + dt_bias), dt_min, dt_max) (softplus optional);
    dt_raw (..., nheads) fp32, dt_bias (nheads,) fp32 or None."""
    rows, H = _dt_check(dt_raw, dt_bias)
    dt = torch.empty_like(dt_raw)
    rc = lib().mamba2_ssd_dt_fwd(rows, H, _ptr(dt_raw), _ptr(dt_bias), int(bool(softplus)), dt_min, dt_max,
                                 _ptr(dt), _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_dt_fwd")
    return dt


def dt_bwd(dt_raw, ddt, dt_bias=None, softplus=True, dt_min=0.0, dt_max=float("inf"), stream=None,
           want_bias_grad=True):
    """(ddt_raw, ddt_bias or None) from ddt, the gradient w.r.t. dt_fwd's output."""
    rows, H = _dt_check(dt_raw, dt_bias)
    _check(ddt, "ddt", tuple(dt_raw.shape), torch.float32, dt_raw.device)
    ddt_raw = torch.empty_like(dt_raw)
    ddt_bias = torch.empty((H,), dtype=torch.float32, device=dt_raw.device) if want_bias_grad else None
    need = lib().mamba2_ssd_dt_bwd_workspace_size(rows, H)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=dt_raw.device)
    rc = lib().mamba2_ssd_dt_bwd(rows, H, _ptr(dt_raw), _ptr(dt_bias), int(bool(softplus)), dt_min, dt_max,
                                 _ptr(ddt), _ptr(ddt_raw), _ptr(ddt_bias), _ptr(ws), ws.numel(), _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_dt_bwd")
    return ddt_raw, ddt_bias


def _gate_dtype(y, z):
    if y.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("y must be bf16 or fp32")
    _check(y, "y", tuple(y.shape), y.dtype, y.device)
    _check(z, "z", tuple(y.shape), y.dtype, y.device)
    return SSD_BF16 if y.dtype == torch.bfloat16 else SSD_F32


def gate_fwd(y, z, stream=None):
    """out = y * silu(z), same shape and dtype as y."""
    dt = _gate_dtype(y, z)
    out = torch.empty_like(y)
    rc = lib().mamba2_ssd_gate_fwd(y.numel(), dt, _ptr(y), _ptr(z), _ptr(out), _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_gate_fwd")
    return out


def gate_bwd(y, z, dout, stream=None):
    """(dy in y's dtype, dz fp32) of out = y * silu(z)."""
    dt = _gate_dtype(y, z)
    _check(dout, "dout", tuple(y.shape), y.dtype, y.device)
    dy = torch.empty_like(y)
    dz = torch.empty(y.shape, dtype=torch.float32, device=y.device)
    rc = lib().mamba2_ssd_gate_bwd(y.numel(), dt, _ptr(y), _ptr(z), _ptr(dout), _ptr(dy), _ptr(dz),
                                   _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_gate_bwd")
    return dy, dz


# ---- causal conv1d before the scan -------------------------------------------

def _conv_check(x, weight, bias, seq_idx):
    if x.dim() != 3 or x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be (batch, seqlen, channels) bf16 or fp32")
    b, T, C = x.shape
    _check(x, "x", (b, T, C), x.dtype, x.device)
    if weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("weight must be (channels, width)")
    _check(weight, "weight", (C, weight.shape[1]), torch.float32, x.device)
    if bias is not None:
        _check(bias, "bias", (C,), torch.float32, x.device)
    if seq_idx is not None:
        _check(seq_idx, "seq_idx", (b, T), torch.int32, x.device)
    return b, T, C, int(weight.shape[1]), SSD_BF16 if x.dtype == torch.bfloat16 else SSD_F32


def conv1d_fwd(x, weight, bias=None, seq_idx=None, activation="silu", config=0, stream=None):
    """y = act(bias + causal depthwise conv of x with weight (channels, width)), same dtype as x."""
    b, T, C, K, dt = _conv_check(x, weight, bias, seq_idx)
    y = torch.empty_like(x)
    rc = lib().mamba2_ssd_conv1d_fwd(b, T, C, K, dt, 1 if activation == "silu" else 0, _ptr(x), _ptr(weight),
                                     _ptr(bias), _ptr(seq_idx), _ptr(y), config, _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_conv1d_fwd")
    return y


def conv1d_bwd(x, weight, dy, bias=None, seq_idx=None, activation="silu", config=0, variant=VARIANT_DETERMINISTIC,
               stream=None, want_bias_grad=True):
    """(dx fp32, dweight fp32, dbias fp32 or None) of sum(conv1d_fwd(...) * dy)."""
    b, T, C, K, dt = _conv_check(x, weight, bias, seq_idx)
    _check(dy, "dy", tuple(x.shape), x.dtype, x.device)
    dx = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    dw = torch.empty_like(weight)
    db = torch.empty((C,), dtype=torch.float32, device=x.device) if want_bias_grad else None
    need = lib().mamba2_ssd_conv1d_bwd_workspace_size(b, T, C, K)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=x.device)
    rc = lib().mamba2_ssd_conv1d_bwd(b, T, C, K, dt, 1 if activation == "silu" else 0, _ptr(x), _ptr(weight),
                                     _ptr(bias), _ptr(seq_idx), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(db), _ptr(ws),
                                     ws.numel(), config, variant, _stream(stream))
    if rc:
        raise SsdError(rc, "mamba2_ssd_conv1d_bwd")
    return dx, dw, db


# ---- autograd -------------------------------------------------------------

class SSDFunction(torch.autograd.Function):
    """y = SSD(x, dt, A, B, C, D) as a differentiable op: the forward and the
    deterministic backward are the library's (mamba2_ssd_fwd / mamba2_ssd_bwd);
    this class only hands tensors across.  The library's gradients are fp32;
    autograd casts each to its input's dtype."""

    @staticmethod
    def forward(ctx, x, dt, A, B, C, D, chunk_size, seq_idx=None, init_states=None, any_start=False):
        y, saved = fwd(x, dt, A, B, C, D, chunk_size, seq_idx=seq_idx, init_states=init_states,
                       any_start=any_start)
        ctx.ssd_saved = saved
        ctx.has_init = init_states is not None
        return y

    @staticmethod
    def backward(ctx, dy):
        saved = ctx.ssd_saved
        g = bwd(saved, dy.contiguous())
        dinit = g.get("dinit") if ctx.has_init else None
        return g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"], g["dD"], None, None, dinit, None


def ssd(x, dt, A, B, C, D, chunk_size, seq_idx=None, init_states=None, any_start=False):
    """Differentiable Mamba2 SSD chunked scan (see SSDFunction)."""
    return SSDFunction.apply(x, dt, A, B, C, D, chunk_size, seq_idx, init_states, any_start)
