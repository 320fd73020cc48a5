"""Seeded synthetic inputs for the SSD forward/backward.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic.  It is the one module that both the CUDA path (tests,
benchmark) and the CPU oracle's callers use, so that both see the very same
values.  Everything is drawn on the CPU from one ``torch.Generator`` seeded
with ``seed``, in the fixed order x, dt, A, B, C, D, dout, init, then cast to
the stated dtypes.

Workload presets (``WORKLOADS``) mirror the shapes and value distributions of
the per-kernel breakdown in "Deterministic bwd kernel for mamba2" (Mamba PR
#827: seqlen 2048 / 4096 / 16384), with the model dimensions this library is
specified for; the page gives no model dimensions of its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    chunk: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    dtype: torch.dtype          # dtype of x, B, C, dout (and y)
    dt_shift: float             # dt = softplus(N(0,1) - dt_shift)
    d_mode: str                 # "one" or "normal"
    seq_lens: tuple = field(default=())   # packed variable-length batch (batch must be 1)
    with_init: bool = False
    any_start: bool = False     # sequence starts may fall inside a chunk


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 256, 64, 4, 16, 1, 16, torch.float32, 2.0, "one"),
    "bf16_T2048": Workload("bf16_T2048", 1, 2048, 128, 256, 64, 8, 128, torch.bfloat16, 4.0, "normal"),
    "bf16_T4096": Workload("bf16_T4096", 1, 4096, 128, 256, 64, 8, 128, torch.bfloat16, 4.0, "normal"),
    "bf16_T16384": Workload("bf16_T16384", 1, 16384, 128, 256, 64, 8, 128, torch.bfloat16, 4.0, "normal"),
    "bf16_varlen_T32768": Workload("bf16_varlen_T32768", 1, 32768, 256, 128, 64, 1, 256, torch.bfloat16,
                                   4.0, "normal", seq_lens=(4096, 8192, 8192, 12288), with_init=True),
    # the packed batch with every sequence start inside a 128-token chunk
    "bf16_varlen_T32768_midchunk": Workload("bf16_varlen_T32768_midchunk", 1, 32768, 256, 128, 64, 1, 256,
                                            torch.bfloat16, 4.0, "normal", seq_lens=(9001, 7000, 333, 16434),
                                            with_init=True, any_start=True),
    # fp32 inputs on the 2K shape: runs the general CUDA-core path (fp32 tolerance rules out
    # tensor-core operands); used to compare its two deterministic dB/dC folds
    "fp32_T2048": Workload("fp32_T2048", 1, 2048, 128, 256, 64, 8, 128, torch.float32, 4.0, "normal"),
}

#: seed offset per preset, in the order the presets are listed above
SEED_BASE = 1234
WORKLOAD_ORDER = ["tiny_fp32", "bf16_T2048", "bf16_T4096", "bf16_T16384", "bf16_varlen_T32768", "fp32_T2048",
                  "bf16_varlen_T32768_midchunk"]


def seed_of(name: str) -> int:
    return SEED_BASE + WORKLOAD_ORDER.index(name)


def make_inputs(batch, seqlen, nheads, headdim, ngroups, dstate, *, dtype=torch.float32, seed=0,
                dt_shift=2.0, d_mode="one", seq_lens=(), with_init=False):
    """Returns a dict of CPU tensors: x, dout (b,T,H,P) and B, C (b,T,G,N) in
    ``dtype``; dt (b,T,H), A (H), D (H) fp32; seq_idx (b,T) int32 or None;
    init (nseq,H,P,N) fp32 or None."""
    g = torch.Generator().manual_seed(int(seed))
    b, T, H, P, G, N = batch, seqlen, nheads, headdim, ngroups, dstate
    x = torch.randn((b, T, H, P), generator=g)
    dt = torch.nn.functional.softplus(torch.randn((b, T, H), generator=g) - dt_shift)
    A = -torch.exp(torch.rand((H,), generator=g) * (math.log(16.0) - math.log(1.0)) + math.log(1.0))
    Bm = torch.randn((b, T, G, N), generator=g)
    Cm = torch.randn((b, T, G, N), generator=g)
    D = torch.ones(H) if d_mode == "one" else torch.randn((H,), generator=g)
    dout = torch.randn((b, T, H, P), generator=g)
    seq_idx = None
    nseq = b
    if seq_lens:
        assert b == 1 and sum(seq_lens) == T
        seq_idx = torch.repeat_interleave(torch.arange(len(seq_lens), dtype=torch.int32),
                                          torch.tensor(seq_lens)).reshape(1, T).contiguous()
        nseq = len(seq_lens)
    init = torch.randn((nseq, H, P, N), generator=g) if with_init else None
    return dict(x=x.to(dtype).contiguous(), dt=dt.float().contiguous(), A=A.float().contiguous(),
                B=Bm.to(dtype).contiguous(), C=Cm.to(dtype).contiguous(), D=D.float().contiguous(),
                dout=dout.to(dtype).contiguous(), seq_idx=seq_idx, init=init)


def workload_inputs(name: str, seqlen: int | None = None, seed: int | None = None):
    """Inputs of a named preset (seed SEED_BASE + its index unless given).
    ``seqlen`` may shorten the sequence (the shapes otherwise stay)."""
    w = WORKLOADS[name]
    T = w.seqlen if seqlen is None else int(seqlen)
    seq_lens = w.seq_lens if seqlen is None else ()
    return make_inputs(w.batch, T, w.nheads, w.headdim, w.ngroups, w.dstate, dtype=w.dtype,
                       seed=seed_of(name) if seed is None else seed, dt_shift=w.dt_shift,
                       d_mode=w.d_mode, seq_lens=seq_lens, with_init=w.with_init)


def make_conv_inputs(batch, seqlen, channels, width, *, dtype=torch.bfloat16, seed=0, seq_lens=()):
    """Inputs of the causal depthwise conv before the scan, drawn in the order
    x, weight, bias, dy: x, dy ~ N(0,1) in ``dtype`` (batch, seqlen,
    channels); weight (channels, width) and bias (channels) ~ U(-1/sqrt(width),
    1/sqrt(width)) fp32 (the usual initialisation of a depthwise conv with
    `width` inputs per output); seq_idx (1, seqlen) int32 for a packed batch."""
    g = torch.Generator().manual_seed(int(seed))
    bound = 1.0 / math.sqrt(width)
    x = torch.randn((batch, seqlen, channels), generator=g)
    w = (torch.rand((channels, width), generator=g) * 2 - 1) * bound
    bias = (torch.rand((channels,), generator=g) * 2 - 1) * bound
    dy = torch.randn((batch, seqlen, channels), generator=g)
    seq_idx = None
    if seq_lens:
        assert batch == 1 and sum(seq_lens) == seqlen
        seq_idx = torch.repeat_interleave(torch.arange(len(seq_lens), dtype=torch.int32),
                                          torch.tensor(seq_lens)).reshape(1, seqlen).contiguous()
    return dict(x=x.to(dtype).contiguous(), w=w.float().contiguous(), bias=bias.float().contiguous(),
                dy=dy.to(dtype).contiguous(), seq_idx=seq_idx)


#: the conv before the scan on the two workloads of this library: its channels are the
#: concatenated x, B, C inputs of the scan (nheads * headdim + 2 * ngroups * dstate), width 4
CONV_WORKLOADS = {
    "conv_T16384": dict(batch=1, seqlen=16384, channels=256 * 64 + 2 * 8 * 128, width=4, seq_lens=()),
    "conv_varlen_T32768": dict(batch=1, seqlen=32768, channels=128 * 64 + 2 * 1 * 256, width=4,
                               seq_lens=(4096, 8192, 8192, 12288)),
}
