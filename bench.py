#!/usr/bin/env python
"""Benchmark of the deterministic Mamba2 SSD backward on GB300.

One step = one backward pass (mamba2_ssd_bwd: every kernel of the backward)
over the workload's synthetic batch; the forward that produces the saved
chunk states runs once, untimed.  Default workload: bf16, batch 1, seqlen
16384, 256 heads of headdim 64, 8 groups, dstate 128, chunk 128 -- the
long-sequence row of the per-kernel breakdown in "Deterministic bwd kernel
for mamba2" (Mamba PR #827), with the model dimensions of this library's
specification.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead (on the host cores, bounded samples of the same workload).
``--op dt_bwd`` / ``--op gate_bwd`` time the steps either side of the scan
(step-size preprocessing, z-gate) on the same workload's tensors instead.
Under torchrun each rank runs an independent replica (the backward does not
shard across GPUs here): value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "SSD bwd tokens/s @ seqlen 16K; % of roofline; bitwise repeat over 20 runs"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_T16384")
    ap.add_argument("--config", type=int, default=0)
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-atomic", action="store_true", help="skip the atomic-variant overhead run")
    ap.add_argument("--cpu-sample-tokens", type=int, default=8192)
    ap.add_argument("--no-others", action="store_true", help="skip the other workload presets")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="shorten the workload to this many tokens (one sequence; for small profiling cases)")
    ap.add_argument("--op", default="ssd_bwd", choices=["ssd_bwd", "dt_bwd", "gate_bwd", "conv1d_bwd"],
                    help="what one step runs: the scan's backward (default) or an adjacent step's backward")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput of independent replicas: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------ clocks ----
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------ byte models ----
def api_bytes(w, es):
    """Algorithmic bytes of one backward: its API inputs read once and its
    outputs written once (x, dout, B, C in the input dtype; dt and the saved
    chunk states fp32; dx, ddt, dB, dC fp32; init/dinit when present)."""
    b, T, H, P, G, N, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk
    nc = -(-T // Q)
    rd = 2 * b * T * H * P * es + 2 * b * T * G * N * es + b * T * H * 4 + b * nc * H * P * N * 4 + 3 * H * 4
    wr = b * T * H * P * 4 + 2 * b * T * G * N * 4 + b * T * H * 4 + 2 * H * 4
    if w.with_init:
        nseq = len(w.seq_lens) if w.seq_lens else b
        rd += nseq * H * P * N * 4
        wr += nseq * H * P * N * 4
    return rd + wr


def algorithmic_flops(w):
    """Tensor-core FLOPs of one backward (elementwise work excluded): per
    (batch, chunk, head) the two Q x Q x P products (g x^T and the intra-chunk
    dx) and the four Q x N x P products (state dx, dHscan, inter-chunk dC,
    state dB); per (batch, chunk, group) the three Q x Q x N products (C B^T
    and the head-summed intra-chunk dC and dB)."""
    b, T, H, P, G, N, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk
    nc = -(-T // Q)
    per_head = 2 * Q * Q * P * 2 + 2 * Q * N * P * 4
    per_group = 2 * Q * Q * N * 3
    return b * nc * (H * per_head + G * per_group)


def nominal_roofline(w, es, ms, tensor_peak_tflops):
    """The slower of HBM bytes at 8 TB/s and tensor FLOPs at the tensor peak,
    as a fraction of the measured backward time."""
    t_hbm = api_bytes(w, es) / 8e12
    t_tc = algorithmic_flops(w) / (tensor_peak_tflops * 1e12)
    bound = max(t_hbm, t_tc)
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor", "t_hbm_us": t_hbm * 1e6, "t_tensor_us": t_tc * 1e6,
            "roofline_us": bound * 1e6, "frac": bound / (ms / 1e3), "algorithmic_bytes": api_bytes(w, es),
            "algorithmic_flops": algorithmic_flops(w), "hbm_tbps": 8.0, "tensor_peak_tflops": tensor_peak_tflops}


def kernel_bytes(name, w, es):
    """Algorithmic bytes of one launch of a kernel of the general path: the
    arrays it must read and write, each once."""
    b, T, H, P, G, N, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk
    nc = -(-T // Q)
    f4 = 4
    x = b * T * H * P * es
    bc = b * T * G * N * es
    dt = b * T * H * f4
    acs = 2 * b * H * nc * Q * f4
    qq = b * nc * H * Q * Q * f4
    cbq = b * nc * G * Q * Q * f4
    st = b * nc * H * P * N * f4
    slots = b * T * H * N * f4
    # mwg leaves the sums of M o Gx per 64-wide tile (rows and columns) and its diagonal
    parts = 2 * b * nc * H * (-(-Q // 64)) * Q * f4 + b * nc * H * Q * f4
    tab = {
        "cumsum_fwd": dt + acs,
        "cb": 2 * bc + cbq,
        "mwg": 2 * x + cbq + acs + dt + 2 * qq + parts,
        "dhscan": x + bc + acs + st,
        "state_passing_bwd": 3 * st + acs,
        "dx": x + bc + dt + qq + st + acs + b * T * H * P * f4,
        "dbdc": 2 * x + 2 * bc + dt + qq + 2 * st + acs + 2 * slots,
        "dbdc_atomic": 2 * x + 2 * bc + dt + qq + 2 * st + acs + 2 * b * T * G * N * f4,
        "dbdc_ordered": 2 * x + 2 * bc + dt + qq + 2 * st + acs + 2 * b * T * G * N * f4,
        "ddt_dacs": 2 * x + 2 * bc + dt + parts + 2 * st + acs + dt + 4 * b * H * nc * Q * f4,
        "cumsum_bwd": 2 * dt + 4 * b * H * nc * Q * f4,
        "cumsum_bwd_atomic": 2 * dt + 4 * b * H * nc * Q * f4,
        "reduce_heads": 2 * slots + 2 * b * T * G * N * f4,
        "reduce_heads_scalars": 2 * b * nc * H * f4,
    }
    return tab.get(name)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the fused
# backward kernel per token, measured with ncu on the revision of its source
# whose SHA-256 is the key (see the profiles/ summaries).  A changed kernel has
# no entry, and the bench then reports traffic as null until it is measured.
FUSED_TRAFFIC_PER_TOKEN = {
    "f14fc64d3878896514b8dcb059c560d377437f5724f802b8126fe02dd7d1c162": {
        "bytes_per_token": (2283115776 + 1239713024) / 16384,
        "capture": "bf16_T16384, one launch, dram__bytes_read.sum + dram__bytes_write.sum (1-pass ncu)",
    },
}


def fused_traffic(tokens):
    import hashlib
    path = os.path.join(ROOT, "deterministic_mamba2_ssd_gb300", "csrc", "ssd_fused_bwd.cu")
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    rec = FUSED_TRAFFIC_PER_TOKEN.get(digest)
    return None if rec is None else rec["bytes_per_token"] * tokens


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: the backward is one short kernel)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def cpu_model():
    """Model name of the host CPU (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


# ------------------------------------------------------- CPU oracle ----
def oracle_tokens_per_s(w, sample_tokens, nthreads=None):
    """Times the fp64 CPU oracle (forward + backward: its backward recomputes
    the forward) on the first ``sample_tokens`` tokens of the workload, all
    heads.  Returns (tokens/s, seconds, threads)."""
    import oracle
    from deterministic_mamba2_ssd_gb300.inputs import workload_inputs
    T = min(sample_tokens, w.seqlen)
    d = workload_inputs(w.name, seqlen=T)
    if w.with_init:
        d["init"] = d["init"][:1].contiguous()
    nt = nthreads or oracle.default_threads()
    oracle.build()
    t0 = time.perf_counter()
    oracle.fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], init=d["init"], nthreads=nt)
    oracle.bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dout"], init=d["init"], nthreads=nt)
    dt = time.perf_counter() - t0
    return w.batch * T / dt, dt, nt


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    sample = 256
    for _ in range(args.warmup):
        oracle_tokens_per_s(w, sample)
    times = []
    nt = None
    for _ in range(args.steps):
        _, dt, nt = oracle_tokens_per_s(w, sample)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = w.batch * min(sample, w.seqlen) / (ms / 1e3)
    desc = "first %d tokens of the workload, all %d heads, fwd+bwd in fp64 per step" % (min(sample, w.seqlen),
                                                                                         w.nheads)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "seq_len": w.seqlen, "global_batch": w.batch,
                       "sample_tokens_per_step": min(sample, w.seqlen)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# -------------------------------------------------- adjacent steps ----
def run_adjacent(args):
    """Times the backward of a step either side of the scan on the workload's
    tensors: dt_bwd (step-size preprocessing; (b*T, H) fp32) or gate_bwd
    (z-gate; (b, T, H, P) in the workload dtype).  Inputs seeded, synthetic,
    resident in HBM; L2 flushed between steps."""
    import __graft_entry__
    __graft_entry__.build()
    import deterministic_mamba2_ssd_gb300 as ssd
    from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    es = 2 if w.dtype == torch.bfloat16 else 4
    rows = w.batch * w.seqlen
    gen = torch.Generator().manual_seed(4321)
    atomic_step = None
    if args.op == "conv1d_bwd":
        # the conv before the scan on the same workload: its channels are the scan's x, B and C
        # concatenated (nheads * headdim + 2 * ngroups * dstate), width 4, silu
        from deterministic_mamba2_ssd_gb300.inputs import make_conv_inputs
        C = w.nheads * w.headdim + 2 * w.ngroups * w.dstate
        cd = make_conv_inputs(w.batch, w.seqlen, C, 4, dtype=w.dtype, seed=4321, seq_lens=w.seq_lens)
        cg = {k: (v.to(dev) if v is not None else None) for k, v in cd.items()}
        n = w.batch * w.seqlen * C
        dxc = torch.empty((w.batch, w.seqlen, C), dtype=torch.float32, device=dev)
        dwc = torch.empty_like(cg["w"])
        dbc = torch.empty_like(cg["bias"])
        need = ssd.lib().mamba2_ssd_conv1d_bwd_workspace_size(w.batch, w.seqlen, C, 4)
        wsc = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
        import ctypes
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        dtc = 1 if w.dtype == torch.bfloat16 else 0

        def conv_step(variant):
            rc = ssd.lib().mamba2_ssd_conv1d_bwd(w.batch, w.seqlen, C, 4, dtc, 1, ptr(cg["x"]), ptr(cg["w"]),
                                                 ptr(cg["bias"]), ptr(cg["seq_idx"]), ptr(cg["dy"]), ptr(dxc),
                                                 ptr(dwc), ptr(dbc), ptr(wsc), wsc.numel(), 0, variant, st)
            if rc:
                raise ssd.SsdError(rc, "mamba2_ssd_conv1d_bwd")

        def step():
            conv_step(0)

        def atomic_step():
            conv_step(1)
        alg = 2 * n * es + n * 4 + 2 * C * 4 * 4 + 2 * C * 4
        launches = 2
        kernel = "conv1d_bwd"
        dtype = "bf16" if es == 2 else "f32"
    elif args.op == "dt_bwd":
        raw = (torch.randn((rows, w.nheads), generator=gen) - 4.0).to(dev)
        bias = torch.randn((w.nheads,), generator=gen).to(dev)
        ddt = torch.randn((rows, w.nheads), generator=gen).to(dev)
        ddt_raw = torch.empty_like(raw)
        ddt_bias = torch.empty_like(bias)
        wsb = ssd.lib().mamba2_ssd_dt_bwd_workspace_size(rows, w.nheads)
        ws = torch.empty(max(16, wsb), dtype=torch.uint8, device=dev)
        import ctypes
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())

        def step():
            rc = ssd.lib().mamba2_ssd_dt_bwd(rows, w.nheads, ptr(raw), ptr(bias), 1, 0.0, float("inf"), ptr(ddt),
                                             ptr(ddt_raw), ptr(ddt_bias), ptr(ws), ws.numel(), st)
            if rc:
                raise ssd.SsdError(rc, "mamba2_ssd_dt_bwd")
        alg = 3 * rows * w.nheads * 4 + 2 * w.nheads * 4
        launches = 2
        kernel = "dt_bwd"
        dtype = "f32"
    else:
        shape = (w.batch, w.seqlen, w.nheads, w.headdim)
        y = torch.randn(shape, generator=gen).to(w.dtype).to(dev)
        z = torch.randn(shape, generator=gen).to(w.dtype).to(dev)
        gout = torch.randn(shape, generator=gen).to(w.dtype).to(dev)
        n = y.numel()

        def step():
            ssd.gate_bwd(y, z, gout)
        alg = 4 * n * es + n * 4
        launches = 1
        kernel = "gate_bwd"
        dtype = "bf16" if es == 2 else "f32"
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier(world, dev)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.fill_(1.0)
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    clocks = clk.stop()
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), world, dev)
    peak, peak_kind = load_peaks()
    achieved = alg / (ms / 1e3) / 1e9
    det_vs_atomic = None
    if atomic_step is not None:
        ta = []
        for _ in range(max(3, args.steps // 2)):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            atomic_step()
            b.record(stream)
            torch.cuda.synchronize()
            ta.append(a.elapsed_time(b))
        det_vs_atomic = {"det_ms": ms, "atomic_ms": statistics.mean(ta), "overhead": ms / statistics.mean(ta) - 1.0}
    if rank == 0:
        print(json.dumps({
            "metric": "%s tokens/s @ seqlen %d" % (kernel, w.seqlen), "value": world * rows / (ms / 1e3),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": w.name, "op": kernel, "seq_len": w.seqlen, "nheads": w.nheads,
                       "headdim": w.headdim, "l2": "flushed between steps (256 MB write)"},
            "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": alg},
            "gpu_launches": launches * args.steps, "clocks": clocks, "e2e": None, "cpu_baseline": None,
            "deterministic_vs_atomic": det_vs_atomic}))
    return 0


# ------------------------------------------------- other workloads ----
def time_workload(ssd, name, dev, steps, warmup=3, repeats=5):
    """Backward (and forward) time of another workload preset, inputs resident
    in HBM, L2 flushed between steps; bitwise repeat over `repeats` runs."""
    from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[name]
    es = 2 if w.dtype == torch.bfloat16 else 4
    d = workload_inputs(name)
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def fwd():
        return ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=w.chunk, seq_idx=g["seq_idx"],
                       init_states=g["init"], any_start=w.any_start)
    y, saved = fwd()
    out = ssd.bwd(saved, g["dout"])
    ws = torch.empty(max(16, ssd.bwd_workspace_size(saved.dims, 0, 0)), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        flush.fill_(1.0)
        ssd.bwd(saved, g["dout"], out=out, workspace=ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush.fill_(1.0)
        a.record()
        ssd.bwd(saved, g["dout"], out=out, workspace=ws)
        b.record()
    fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(max(2, steps // 2))]
    for a, b in fe:
        flush.fill_(1.0)
        a.record()
        fwd()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fe)
    ref = {k: v.view(torch.int32).clone() for k, v in out.items()}
    same = 0
    for _ in range(repeats):
        o = ssd.bwd(saved, g["dout"], workspace=ws)
        same += all(torch.equal(ref[k], v.view(torch.int32)) for k, v in o.items())
    peak, peak_kind = load_peaks()
    tpeak, _ = load_tensor_peak()
    tokens = w.batch * w.seqlen
    return {"workload": name, "launch_config": ssd.config_name(saved.dims, 0), "bwd_ms": ms,
            "tokens_per_s": tokens / (ms / 1e3), "fwd_ms": fwd_ms, "steps": steps,
            "bwd_hbm_frac": api_bytes(w, es) / (ms / 1e3) / 1e9 / peak, "peak_kind": peak_kind,
            "nominal_roofline": nominal_roofline(w, es, ms, tpeak),
            "bitwise_equal_repeats": "%d/%d" % (same, repeats)}


# ------------------------------------------------------------- ours ----
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.op != "ssd_bwd":
        return run_adjacent(args)
    import __graft_entry__
    __graft_entry__.build()
    import deterministic_mamba2_ssd_gb300 as ssd
    from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS, workload_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = WORKLOADS[args.workload]
    if args.seqlen:
        import dataclasses
        w = dataclasses.replace(w, seqlen=args.seqlen, seq_lens=())
    es = 2 if w.dtype == torch.bfloat16 else 4
    d = workload_inputs(w.name, seqlen=args.seqlen)
    g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
    y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=w.chunk,
                       seq_idx=g["seq_idx"], init_states=g["init"], any_start=w.any_start)
    # the forward that produces the saved states (untimed by the metric), timed on its own
    fwd_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for a, b in fwd_ev:
        a.record()
        y, saved = ssd.fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=w.chunk,
                           seq_idx=g["seq_idx"], init_states=g["init"], any_start=w.any_start)
        b.record()
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev[1:])
    out = ssd.bwd(saved, g["dout"], config=args.config, variant=args.variant)
    ws = torch.empty(max(16, ssd.bwd_workspace_size(saved.dims, args.config, args.variant)), dtype=torch.uint8,
                     device=dev)
    names = ssd.bwd_launch_names(saved.dims, args.config, args.variant)
    nl = len(names)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)     # materialise the event objects
        return evs

    for _ in range(args.warmup):
        flush.fill_(1.0)
        ssd.bwd(saved, g["dout"], config=args.config, variant=args.variant, out=out, workspace=ws)
    traces = [new_events(2 * nl) for _ in range(args.steps)]
    torch.cuda.synchronize()

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier(world, dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(1.0)   # evict L2 between steps (outside the traced region)
        ssd.bwd(saved, g["dout"], config=args.config, variant=args.variant, out=out, workspace=ws,
                events=traces[k])
    torch.cuda.synchronize()
    barrier(world, dev)
    wall = time.perf_counter() - t0
    clocks = clk.stop()

    step_ms = [traces[k][0].elapsed_time(traces[k][-1]) for k in range(args.steps)]
    per_kernel = {}
    for k in range(args.steps):
        for j, n in enumerate(names):
            per_kernel.setdefault((j, n), []).append(traces[k][2 * j].elapsed_time(traces[k][2 * j + 1]))
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    tokens = w.batch * w.seqlen
    value = job_throughput(tokens, world, ms_max)

    # dominant kernel and its roofline
    tot = {key: sum(v) for key, v in per_kernel.items()}
    (jdom, ndom), tdom = max(tot.items(), key=lambda kv: kv[1])
    dom_ms = tdom / args.steps
    peak, peak_kind = load_peaks()
    if ndom.startswith("fused_bwd"):
        alg = api_bytes(w, es)      # the fused kernel moves the whole backward's API I/O
    else:
        alg = kernel_bytes(ndom, w, es)
    achieved = alg / (dom_ms / 1e3) / 1e9 if alg else None
    shares = {}
    for (j, n), t in tot.items():   # launches of the same kernel summed (two state halves on dstate 256)
        shares[n] = shares.get(n, 0.0) + t / sum(tot.values())
    shares = {n: round(v, 4) for n, v in shares.items()}
    tpeak, tpeak_kind = load_tensor_peak()
    roofline = {"bound": "hbm", "kernel": ndom, "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "traffic": fused_traffic(w.batch * w.seqlen) if ndom == "fused_bwd" else None,
                "algorithmic_bytes_per_launch": alg, "launch_ms": dom_ms}
    if nominal_roofline(w, es, 1.0, tpeak)["bound"] == "tensor" and ndom.startswith("fused_bwd"):
        # tensor-bound shape (dstate 256): the fused kernel runs once per state half, both halves
        # at once, so it is timed over the whole backward and held against the tensor peak
        flops = algorithmic_flops(w)
        ach = flops / (ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": "fused_bwd (both state halves, concurrent; whole backward)",
                    "achieved": ach, "peak": tpeak, "peak_kind": tpeak_kind, "unit": "TFLOP/s",
                    "frac": ach / tpeak, "traffic": None, "algorithmic_flops_per_launch": flops, "launch_ms": ms}

    # bitwise repeat (after the timed region): 20 more backward passes, each compared bit for bit
    # with the first, and one pass under every other launch configuration
    def bits_of(o):
        return {k: v.view(torch.int32).clone() for k, v in o.items()}
    ref_bits = bits_of(out)
    repeats_equal = 0
    for _ in range(20):
        ssd.bwd(saved, g["dout"], config=args.config, variant=args.variant, out=out, workspace=ws)
        repeats_equal += all(torch.equal(ref_bits[k], v.view(torch.int32)) for k, v in out.items())
    configs_equal = []
    for cfg in range(ssd.num_configs(saved.dims)):
        o = ssd.bwd(saved, g["dout"], config=cfg, variant=args.variant)
        configs_equal.append(all(torch.equal(ref_bits[k], v.view(torch.int32)) for k, v in o.items()))
    determinism = {"repeats": 20, "bitwise_equal_repeats": int(repeats_equal),
                   "configs": [ssd.config_name(saved.dims, c) for c in range(len(configs_equal))],
                   "bitwise_equal_across_configs": all(configs_equal)}
    del ref_bits

    # determinism overhead: the same kernels with atomic accumulation
    atomic_ms = None
    if not args.no_atomic and args.variant == 0:
        ws_a = torch.empty(max(16, ssd.bwd_workspace_size(saved.dims, args.config, 1)), dtype=torch.uint8,
                           device=dev)
        out_a = {k: torch.empty_like(v) for k, v in out.items()}
        for _ in range(2):
            ssd.bwd(saved, g["dout"], config=args.config, variant=1, out=out_a, workspace=ws_a)
        na = len(ssd.bwd_launch_names(saved.dims, args.config, 1))
        ta = []
        for _ in range(max(3, args.steps // 2)):
            flush.fill_(1.0)
            ev = new_events(2 * na)
            ssd.bwd(saved, g["dout"], config=args.config, variant=1, out=out_a, workspace=ws_a, events=ev)
            torch.cuda.synchronize()
            ta.append(ev[0].elapsed_time(ev[-1]))
        atomic_ms = statistics.mean(ta)
        del ws_a, out_a

    # End to end through the public API with host buffers.  The headline mode is the call
    # sequence of a caller whose data sits in host memory: every step copies the forward's inputs
    # and dout from pinned host memory, calls mamba2_ssd_fwd (which leaves the chunk states the
    # backward reads in device memory; a saved handle comes only from the forward) and
    # mamba2_ssd_bwd, and copies every gradient back.  The second mode copies the saved chunk
    # states from the host instead of running the forward (1.07 GB more per step at T=16384) and
    # runs the backward alone.  Steps are pipelined over two buffer sets and three streams
    # (inputs of step k+1 travel while step k computes and its gradients travel back), as a
    # training loop's data path would run them; the serial step time (copies, compute and copies
    # back on one stream) is reported beside.
    e2e = None
    if not args.no_e2e:
        host = {k: v.pin_memory() for k, v in d.items() if v is not None}
        # (the states-from-host mode runs only where the backward reads the caller's state buffer)
        host_states = None if saved.struct.aux else saved.states.cpu().pin_memory()
        d2h = sum(v.numel() * v.element_size() for v in out.values())
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

        def fwd_on(dev_in, stream):
            return ssd.fwd(dev_in["x"], dev_in["dt"], dev_in["A"], dev_in["B"], dev_in["C"], dev_in["D"],
                           chunk_size=w.chunk, seq_idx=dev_in.get("seq_idx"), init_states=dev_in.get("init"),
                           stream=stream, any_start=w.any_start)[1]

        def make_sets(states_from_host):
            src = dict(host, states=host_states) if states_from_host else host
            sets = []
            for _ in range(2):
                dev_in = {k: v.to(dev) for k, v in src.items()}
                sv = None
                if states_from_host:
                    # a saved handle whose chunk states are this set's copy of the host's
                    sv = fwd_on(dev_in, None)
                    sv.struct.states = dev_in["states"].data_ptr()
                    sv.tensors["states"] = dev_in["states"]
                sets.append({"in": dev_in, "saved": sv, "out": {k: torch.empty_like(v) for k, v in out.items()},
                             "ws": torch.empty_like(ws),
                             "host_out": {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                                          for k, v in out.items()}})
            torch.cuda.synchronize()
            return src, sets

        def run_steps(src, sets, n, serial, with_fwd):
            """Mean ms per step over n steps, and the median interval between step completions."""
            ev_cmp = [None, None]   # compute of the step that last used each set (inputs read)
            ev_out = [None, None]   # copy-back of the step that last used each set (outputs read)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            done = []
            start.record(s_in)
            for k in range(n):
                i = k % 2
                bs = sets[i]
                si, sc, so = (s_in, s_in, s_in) if serial else (s_in, s_cmp, s_out)
                if ev_cmp[i] is not None:
                    si.wait_event(ev_cmp[i])
                with torch.cuda.stream(si):
                    for key, v in src.items():
                        bs["in"][key].copy_(v, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(si)
                sc.wait_event(e_in)
                if ev_out[i] is not None:
                    sc.wait_event(ev_out[i])
                with torch.cuda.stream(sc):   # the forward's buffers are allocated on this stream
                    if with_fwd:
                        bs["saved"] = fwd_on(bs["in"], sc)
                    ssd.bwd(bs["saved"], bs["in"]["dout"], config=args.config, out=bs["out"], workspace=bs["ws"],
                            stream=sc)
                ev_cmp[i] = torch.cuda.Event()
                ev_cmp[i].record(sc)
                so.wait_event(ev_cmp[i])
                with torch.cuda.stream(so):
                    for key, v in bs["out"].items():
                        bs["host_out"][key].copy_(v, non_blocking=True)
                ev_out[i] = torch.cuda.Event(enable_timing=True)
                ev_out[i].record(so)
                done.append(ev_out[i])
            for e in ev_out:
                if e is not None:
                    s_in.wait_event(e)
            end.record(s_in)
            end.synchronize()
            t = [start.elapsed_time(e) for e in done]
            gaps = [b - a for a, b in zip([0.0] + t[:-1], t)]
            return start.elapsed_time(end) / n, statistics.median(gaps)

        def measure(states_from_host):
            src, sets = make_sets(states_from_host)
            with_fwd = not states_from_host
            run_steps(src, sets, args.warmup, False, with_fwd)
            pipe_ms, pipe_med = run_steps(src, sets, args.steps, False, with_fwd)
            pipe_ms = max_over_ranks(pipe_ms, world, dev)
            run_steps(src, sets, 2, True, with_fwd)
            serial_ms, serial_med = run_steps(src, sets, args.steps, True, with_fwd)
            serial_ms = max_over_ranks(serial_ms, world, dev)
            h2d = sum(v.numel() * v.element_size() for v in src.values())
            # the gradients the last steps copied back to the host equal the device-timed run's,
            # bit for bit (both buffer sets)
            same = None if ref_host is None else all(
                torch.equal(bs["host_out"][k].view(torch.int32), ref_host[k].view(torch.int32))
                for bs in sets for k in ref_host)
            del sets
            # value from the mean over all steps; the medians show how much of it comes from
            # occasional stalls of the host copies (steps of 80-200 ms seen on a shared machine)
            return {"value": world * tokens / (pipe_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": pipe_ms, "pipelined": True,
                    "ms_per_step_median": pipe_med, "serial_ms_per_step": serial_ms,
                    "serial_ms_per_step_median": serial_med, "bitwise_equal_to_device_run": same}

        # (the end-to-end steps run the deterministic variant)
        ref_host = {k: v.detach().cpu() for k, v in out.items()} if args.variant == 0 else None
        e2e = measure(False)
        e2e["calls_per_step"] = "mamba2_ssd_fwd + mamba2_ssd_bwd"
        if not saved.struct.aux:
            e2e["states_from_host"] = measure(True)
            e2e["states_from_host"]["calls_per_step"] = "mamba2_ssd_bwd (saved chunk states copied from the host)"
        else:   # the backward reads the packed states kept in the forward's workspace, not `states`
            e2e["states_from_host"] = {"value": None, "reason": "this shape's backward reads the packed states "
                                       "kept in the forward workspace, not the caller's state buffer"}
        del host, host_states, ref_host

    # the other workload presets (the 2K and 4K rows of the pages' tables, the packed
    # variable-length batch, and fp32 inputs on the general path), timed after the headline
    # run, single GPU only
    others = None
    if world == 1 and not args.no_others and args.workload == "bf16_T16384":
        others = [time_workload(ssd, n, dev, steps=st) for n, st in
                  (("bf16_T2048", 20), ("bf16_T4096", 20), ("bf16_varlen_T32768", 2),
                   ("bf16_varlen_T32768_midchunk", 2), ("fp32_T2048", 10))]

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v, secs, nt = oracle_tokens_per_s(w, args.cpu_sample_tokens)
            cpu = {"value": v, "unit": UNIT, "cores": nt, "kind": "oracle", "cpu_model": cpu_model(),
                   "sample": "first %d tokens of the workload, all %d heads, fp64 forward+backward, %.1f s" %
                             (min(args.cpu_sample_tokens, w.seqlen), w.nheads, secs)}
            # one thread on the 2K workload (a 512-token sample of it)
            from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS
            w1 = WORKLOADS["bf16_T2048"]
            v1, secs1, _ = oracle_tokens_per_s(w1, 512, nthreads=1)
            cpu["one_thread"] = {"value": v1, "unit": UNIT, "threads": 1,
                                 "sample": "first 512 tokens of bf16_T2048, all %d heads, fp64 forward+backward, "
                                           "%.1f s" % (w1.nheads, secs1)}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if es == 2 else "f32", "data": "synthetic",
            "config": {"workload": w.name, "global_batch": w.batch * world, "seq_len": w.seqlen,
                       "nheads": w.nheads, "headdim": w.headdim, "ngroups": w.ngroups, "dstate": w.dstate,
                       "chunk_size": w.chunk, "parallelism": "replicas" if world > 1 else "single",
                       "launch_config": ssd.config_name(saved.dims, args.config),
                       "l2": "flushed between steps (256 MB write) and inputs larger than L2"},
            "roofline": roofline,
            "nominal_roofline": nominal_roofline(w, es, ms_max, tpeak),
            "fwd_ms": fwd_ms,
            "other_workloads": others,
            "kernel_share": shares,
            "gpu_launches": nl * args.steps,
            "bitwise_repeat": determinism,
            "deterministic_vs_atomic": {"det_ms": ms_max, "atomic_ms": atomic_ms,
                                        "overhead": (ms_max / atomic_ms - 1.0) if atomic_ms else None},
            "wall_s_timed_region": wall,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
