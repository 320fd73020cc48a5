"""The C ABI without a GPU: the library loads, exports every function the
header declares, answers its queries, and rejects bad arguments on the host
before launching anything (all pointers below are fake and never touched)."""
import ctypes
import os
import re

import pytest
import torch

import deterministic_mamba2_ssd_gb300 as ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba2_ssd.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba2_ssd_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return ssd.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(7):
        assert L.mamba2_ssd_status_string(code).decode() not in ("", "unknown status")
    assert L.mamba2_ssd_status_string(99).decode() == "unknown status"


def test_queries(L):
    d = ssd.make_dims(1, 16384, 256, 64, 8, 128, 128)
    assert L.mamba2_ssd_num_chunks(ctypes.byref(d)) == 128
    n = ssd.num_configs(d)
    assert n >= 2
    names = [ssd.config_name(d, c) for c in range(n)]
    assert len(set(names)) == n and "invalid" not in names
    assert ssd.config_name(d, n) == "invalid"
    for c in range(n):
        assert ssd.bwd_workspace_size(d, c, 0) > 0
        assert ssd.bwd_num_launches(d, c, 0) > 0
    assert ssd.fwd_workspace_size(d) > 0
    ragged = ssd.make_dims(2, 1000, 4, 16, 2, 16, 64)
    assert L.mamba2_ssd_num_chunks(ctypes.byref(ragged)) == 16


@pytest.mark.parametrize("field,value", [("batch", 0), ("seqlen", 0), ("seqlen", -1), ("nheads", 0), ("ngroups", 4),
                                         ("chunk_size", 0), ("chunk_size", 4096), ("dtype", 7),
                                         ("flags", 2), ("flags", 4), ("nseq", 0)])
def test_invalid_dims_rejected(L, field, value):
    d = ssd.make_dims(1, 256, 4, 16, 1, 16, 64)
    if field == "ngroups":
        d.nheads = 6
    setattr(d, field, value)
    assert L.mamba2_ssd_num_chunks(ctypes.byref(d)) == -1
    assert L.mamba2_ssd_num_configs(ctypes.byref(d)) == 0
    assert L.mamba2_ssd_fwd_workspace_size(ctypes.byref(d)) == 0
    assert L.mamba2_ssd_bwd_workspace_size(ctypes.byref(d), 0, 0) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails on the host first


def call_fwd(L, d, ptrs=None, ws_bytes=0, saved=True):
    p = [ctypes.c_void_p(FAKE + 256 * i) for i in range(10)] if ptrs is None else ptrs
    sv = ssd.SavedStruct()
    return L.mamba2_ssd_fwd(ctypes.byref(d), *p, ctypes.c_void_p(FAKE), ws_bytes, None,
                            ctypes.byref(sv) if saved else None)


def test_fwd_argument_checks(L):
    d = ssd.make_dims(1, 256, 4, 16, 1, 16, 64, dtype=torch.float32)
    need = ssd.fwd_workspace_size(d)
    no_seq = [ctypes.c_void_p(FAKE + 256 * i) for i in range(10)]
    no_seq[6] = None      # seq_idx
    no_seq[7] = None      # init
    # workspace too small -> SSD_ERR_WORKSPACE, before any launch
    assert call_fwd(L, d, no_seq, need - 1) == 3
    # a required pointer missing -> SSD_ERR_INVALID_ARG
    for k in (0, 1, 2, 3, 4, 5, 8, 9):
        p = list(no_seq)
        p[k] = None
        assert call_fwd(L, d, p, need) == 1, k
    # misaligned pointer -> SSD_ERR_INVALID_ARG
    p = list(no_seq)
    p[0] = ctypes.c_void_p(FAKE + 4)
    assert call_fwd(L, d, p, need) == 1
    # missing saved_out
    assert call_fwd(L, d, no_seq, need, saved=False) == 1
    # nseq must equal batch without seq_idx
    d2 = ssd.make_dims(1, 256, 4, 16, 1, 16, 64, nseq=3, dtype=torch.float32)
    assert call_fwd(L, d2, no_seq, need) == 1


def test_bwd_argument_checks(L):
    d = ssd.make_dims(1, 256, 4, 16, 1, 16, 64, dtype=torch.float32)
    sv = ssd.SavedStruct()
    sv.dims = d
    outs = [ctypes.c_void_p(FAKE + 256 * i) for i in range(7)] + [None]  # dout, dx..dD, dinit
    args = lambda sv, o, ws, cfg=0, var=0: (ctypes.byref(sv), *o, ctypes.c_void_p(FAKE), ws, cfg, var, None)
    # not produced by the forward -> SSD_ERR_HANDLE
    assert L.mamba2_ssd_bwd(*args(sv, outs, 1 << 40)) == 6
    assert L.mamba2_ssd_bwd(None, *outs, ctypes.c_void_p(FAKE), 0, 0, 0, None) == 6
    # forge a structurally valid saved struct with fake pointers
    for n in ("x", "dt", "A", "B", "C", "D", "states"):
        setattr(sv, n, FAKE + 4096)
    sv.magic = 0x53534432
    need = ssd.bwd_workspace_size(d, 0, 0)
    assert L.mamba2_ssd_bwd(*args(sv, outs, need - 1)) == 3
    assert L.mamba2_ssd_bwd(*args(sv, outs, need, cfg=99)) == 1
    assert L.mamba2_ssd_bwd(*args(sv, outs, need, var=5)) == 1
    o = list(outs)
    o[1] = None     # dx
    assert L.mamba2_ssd_bwd(*args(sv, o, need)) == 1
    o = list(outs)
    o[7] = ctypes.c_void_p(FAKE)   # dinit without initial states
    assert L.mamba2_ssd_bwd(*args(sv, o, need)) == 1


def test_any_start_dims_take_the_padded_fused_path_or_the_general_one(L):
    fused = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128, nseq=3, seq_idx=True)
    padded = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128, nseq=3, seq_idx=True, any_start=True)
    assert ssd.config_name(fused, 0) == "fused/ring4"
    assert ssd.config_name(padded, 0) == "fused-padded/0"
    # fp32: the general path, with its sequence-start kernels
    anyst = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128, nseq=3, dtype=torch.float32, seq_idx=True, any_start=True)
    assert ssd.config_name(anyst, 0).startswith("simt")
    for var in (0, 1):
        names = ssd.bwd_launch_names(anyst, 0, var)
        assert names[0] == "seq_first" and names[6] == "dinit_mid" and names[5] == "state_passing_bwd"
        assert "invalid" not in names and len(names) == ssd.bwd_num_launches(anyst, 0, var)
    plain = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128, dtype=torch.float32)
    assert ssd.bwd_launch_names(plain, 0, 0)[0] == "cumsum_fwd"
    assert ssd.bwd_num_launches(anyst, 0, 0) == ssd.bwd_num_launches(plain, 0, 0) + 2


def test_ordered_variant_only_on_the_general_path(L):
    fused = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128)
    simt = ssd.make_dims(1, 1024, 8, 64, 2, 128, 128, dtype=torch.float32)
    assert ssd.bwd_workspace_size(fused, 0, 2) == 0 and ssd.bwd_num_launches(fused, 0, 2) == 0
    assert ssd.bwd_workspace_size(simt, 0, 2) > 0
    names = ssd.bwd_launch_names(simt, 0, 2)
    assert "dbdc_ordered" in names and "reduce_heads" not in names and "dbdc" not in names
    assert "invalid" not in names and names[-1] == "reduce_heads_scalars"
    # no per-head slots: smaller workspace than the slot fold
    assert ssd.bwd_workspace_size(simt, 0, 2) < ssd.bwd_workspace_size(simt, 0, 0)
    big_n = ssd.make_dims(1, 256, 4, 16, 1, 1024, 64, dtype=torch.float32)
    assert ssd.bwd_workspace_size(big_n, 0, 2) == 0 and ssd.bwd_workspace_size(big_n, 0, 0) > 0
    assert ssd.bwd_workspace_size(simt, 0, 3) == 0


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ssd, "_lib", None)
    monkeypatch.setattr(ssd, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU or PyTorch fallback"):
        ssd.lib()


def test_selftest_and_static_entry_reject_bad_arguments_on_host(L):
    # exercises the ctypes signatures without touching a GPU
    assert L.mamba2_ssd_selftest_umma(None, None, None, 128, 64, 64, 0, 0, 0, None) == 1
    assert L.mamba2_ssd_selftest_umma(FAKE, FAKE, FAKE, 64, 64, 64, 0, 0, 0, None) == 1
    assert L.mamba2_ssd_static_scratch_bytes() == 32 << 20
    assert L.mamba2_ssd_bwd_static_scratch(None, None, None, None, None, None, None, None, None, 0, None) == 6
    # its status check validates dims and config before looking the array up
    assert L.mamba2_ssd_static_scratch_check(None, 0, None) == 1
    fused = ssd.make_dims(1, 256, 4, 64, 1, 128, 128)
    assert L.mamba2_ssd_static_scratch_check(ctypes.byref(fused), 2, None) == 1


def test_adjacent_steps_reject_bad_arguments_on_host(L):
    f32 = ctypes.c_float
    p = lambda k: ctypes.c_void_p(FAKE + 256 * k)
    inf = float("inf")
    # clamp bounds out of order or NaN; zero heads
    assert L.mamba2_ssd_dt_fwd(4, 8, p(0), None, 1, f32(1.0), f32(0.5), p(1), None) == 1
    assert L.mamba2_ssd_dt_fwd(4, 8, p(0), None, 1, f32(float("nan")), f32(inf), p(1), None) == 1
    assert L.mamba2_ssd_dt_fwd(4, 0, p(0), None, 1, f32(0.0), f32(inf), p(1), None) == 1
    # misaligned or missing pointers
    assert L.mamba2_ssd_dt_fwd(4, 8, ctypes.c_void_p(FAKE + 4), None, 1, f32(0.0), f32(inf), p(1), None) == 1
    assert L.mamba2_ssd_dt_fwd(4, 8, None, None, 1, f32(0.0), f32(inf), p(1), None) == 1
    # empty input: nothing to do, nothing launched
    assert L.mamba2_ssd_dt_fwd(0, 8, None, None, 1, f32(0.0), f32(inf), None, None) == 0
    need = L.mamba2_ssd_dt_bwd_workspace_size(1000, 8)
    assert need == 32 * 8 * 4      # 32 row slabs, one partial per head each
    assert L.mamba2_ssd_dt_bwd_workspace_size(-1, 8) == 0
    assert L.mamba2_ssd_dt_bwd(1000, 8, p(0), None, 1, f32(0.0), f32(inf), p(1), p(2), p(3), p(4), need - 1,
                               None) == 3
    assert L.mamba2_ssd_dt_bwd(1000, 8, p(0), None, 1, f32(0.0), f32(inf), None, p(2), p(3), p(4), need,
                               None) == 1
    # gate: bad dtype, misaligned, missing output; empty is a no-op
    assert L.mamba2_ssd_gate_fwd(16, 7, p(0), p(1), p(2), None) == 1
    assert L.mamba2_ssd_gate_fwd(16, 1, p(0), ctypes.c_void_p(FAKE + 2), p(2), None) == 1
    assert L.mamba2_ssd_gate_bwd(16, 0, p(0), p(1), p(2), p(3), None, None) == 1
    assert L.mamba2_ssd_gate_fwd(0, 1, None, None, None, None) == 0
    assert L.mamba2_ssd_gate_bwd(-1, 1, p(0), p(1), p(2), p(3), p(4), None) == 1


def test_states_unpack_rejects_bad_arguments_on_host(L):
    sv = ssd.SavedStruct()
    assert L.mamba2_ssd_states_unpack(None, ctypes.c_void_p(FAKE), None) == 6
    assert L.mamba2_ssd_states_unpack(ctypes.byref(sv), ctypes.c_void_p(FAKE), None) == 6   # not from fwd
    sv.dims = ssd.make_dims(1, 256, 4, 64, 1, 128, 128)
    sv.magic = 0x53534432
    sv.states = FAKE
    assert L.mamba2_ssd_states_unpack(ctypes.byref(sv), None, None) == 1
    assert L.mamba2_ssd_states_unpack(ctypes.byref(sv), ctypes.c_void_p(FAKE + 4), None) == 1


def test_binding_checks_shapes_before_calling_the_library():
    x = torch.zeros(1, 8, 2, 4)
    dt = torch.zeros(1, 8, 2)
    A = torch.zeros(2)
    Bm = torch.zeros(1, 8, 1, 4)
    D = torch.zeros(2)
    with pytest.raises(ValueError, match="bf16 or fp32"):
        ssd.fwd(x.half(), dt, A, Bm.half(), Bm.half(), D, 4)
    with pytest.raises(ValueError, match="B"):
        ssd.fwd(x, dt, A, torch.zeros(1, 7, 1, 4), Bm, D, 4)
    with pytest.raises(ValueError, match="dt"):
        ssd.fwd(x, dt[:, :, :1].contiguous(), A, Bm, Bm, D, 4)
    with pytest.raises(ValueError, match="any_start"):
        ssd.fwd(x, dt, A, Bm, Bm, D, 4, any_start=True)
    with pytest.raises(ValueError, match="z"):
        ssd.gate_fwd(x, torch.zeros(1, 8, 2, 5))
    with pytest.raises(ValueError, match="dt_raw"):
        ssd.dt_fwd(torch.zeros(5))


def test_binding_declares_argument_types_of_every_entry_point(L):
    # ctypes would otherwise pass Python ints as C int and floats as double
    missing = [n for n in declared_functions() if getattr(L, n).argtypes is None]
    assert not missing, missing


def test_conv1d_rejects_bad_arguments_on_host(L):
    p = lambda k: ctypes.c_void_p(FAKE + 256 * k)
    assert L.mamba2_ssd_conv1d_num_configs() == 2
    need = L.mamba2_ssd_conv1d_bwd_workspace_size(1, 300, 64, 4)
    assert need == 3 * 5 * 64 * 4          # 3 tiles of 128 tokens, (width + 1) x channels each
    assert L.mamba2_ssd_conv1d_bwd_workspace_size(1, 300, 62, 4) == 0    # channels not a multiple of 4
    assert L.mamba2_ssd_conv1d_bwd_workspace_size(1, 300, 64, 5) == 0    # width above 4
    # bad width, dtype, activation, config, misaligned pointer, seq_idx with batch > 1
    assert L.mamba2_ssd_conv1d_fwd(1, 300, 64, 0, 1, 1, p(0), p(1), None, None, p(2), 0, None) == 1
    assert L.mamba2_ssd_conv1d_fwd(1, 300, 64, 4, 7, 1, p(0), p(1), None, None, p(2), 0, None) == 1
    assert L.mamba2_ssd_conv1d_fwd(1, 300, 64, 4, 1, 2, p(0), p(1), None, None, p(2), 0, None) == 1
    assert L.mamba2_ssd_conv1d_fwd(1, 300, 64, 4, 1, 1, p(0), p(1), None, None, p(2), 2, None) == 1
    assert L.mamba2_ssd_conv1d_fwd(1, 300, 64, 4, 1, 1, ctypes.c_void_p(FAKE + 8), p(1), None, None, p(2), 0,
                                   None) == 1
    assert L.mamba2_ssd_conv1d_fwd(2, 300, 64, 4, 1, 1, p(0), p(1), None, p(3), p(2), 0, None) == 1
    # workspace too small (deterministic variant); bad variant
    assert L.mamba2_ssd_conv1d_bwd(1, 300, 64, 4, 1, 1, p(0), p(1), None, None, p(2), p(3), p(4), p(5), p(6),
                                   need - 1, 0, 0, None) == 3
    assert L.mamba2_ssd_conv1d_bwd(1, 300, 64, 4, 1, 1, p(0), p(1), None, None, p(2), p(3), p(4), p(5), p(6),
                                   need, 0, 2, None) == 1


def test_dstate_256_shapes_pick_the_split_fused_path_or_the_general_one(L):
    # one group, even head count, chunk 128 or 256: the fused kernels once per state half
    assert ssd.config_name(ssd.make_dims(1, 512, 4, 64, 1, 256, 256), 0) == "fused-split/ring4"
    assert ssd.config_name(ssd.make_dims(1, 512, 4, 64, 1, 256, 128), 1) == "fused-split/ring2"
    assert ssd.bwd_launch_names(ssd.make_dims(1, 512, 4, 64, 1, 256, 256)) == [
        "fused_bwd", "fused_bwd", "split_fold", "split_scalars"]
    # odd head count, two groups, fp32, or a ragged length: the general path
    for dims in (ssd.make_dims(1, 512, 3, 64, 1, 256, 256), ssd.make_dims(1, 512, 4, 64, 2, 256, 256),
                 ssd.make_dims(1, 512, 4, 64, 1, 256, 256, dtype=torch.float32),
                 ssd.make_dims(1, 500, 4, 64, 1, 256, 256)):
        assert ssd.config_name(dims, 0).startswith("simt"), dims


def test_fwd_check_on_host(L):
    FAKE = 0x7f0000000000
    simt = ssd.make_dims(1, 256, 4, 16, 1, 16, 64, dtype=torch.float32)
    assert L.mamba2_ssd_fwd_check(ctypes.byref(simt), ctypes.c_void_p(FAKE), None) == 0   # no device waits: nothing read
    assert L.mamba2_ssd_fwd_check(ctypes.byref(simt), None, None) == 1
    bad = ssd.make_dims(1, 256, 3, 16, 2, 16, 64)   # heads not a multiple of groups
    assert L.mamba2_ssd_fwd_check(ctypes.byref(bad), ctypes.c_void_p(FAKE), None) == 1


def test_longer_chunks_with_dstate_128_run_the_fused_kernels_in_128_token_chunks(L):
    base = ssd.make_dims(1, 2048, 8, 64, 2, 128, 128)
    for Q in (256, 512, 1024):
        d = ssd.make_dims(1, 2048, 8, 64, 2, 128, Q)
        assert ssd.config_name(d, 0) == "fused-chunk128/ring4" and ssd.config_name(d, 1) == "fused-chunk128/ring2"
        assert ssd.bwd_launch_names(d) == ["fused_bwd", "fold_scalars"]
        assert ssd.bwd_launch_names(d, 0, 1) == ["fused_bwd_atomic"]
        # the backward is that of the same problem in 128-token chunks
        assert ssd.bwd_workspace_size(d, 0, 0) == ssd.bwd_workspace_size(base, 0, 0)
        # the forward keeps the packed state of every 128 tokens besides the 128-token forward's workspace
        assert ssd.fwd_workspace_size(d) >= ssd.fwd_workspace_size(base) + 16 * 8 * 64 * 128 * 4
        assert ssd.bwd_workspace_size(d, 0, 2) == 0   # no ordered variant on the fused kernels
    # seqlen not a multiple of 128, a chunk that is not a multiple of 128, fp32: the general path
    for d in (ssd.make_dims(1, 2000, 8, 64, 2, 128, 256), ssd.make_dims(1, 2048, 8, 64, 2, 128, 192),
              ssd.make_dims(1, 2048, 8, 64, 2, 128, 256, dtype=torch.float32)):
        assert ssd.config_name(d, 0).startswith("simt"), d
    # sequence starts inside a chunk of 256: the padded form, whose chunks are 128 tokens anyway
    d = ssd.make_dims(1, 2048, 8, 64, 2, 128, 256, nseq=3, seq_idx=True, any_start=True)
    assert ssd.config_name(d, 0) == "fused-padded/0"
    assert L.mamba2_ssd_padded_chunks(ctypes.byref(d)) == 16 + 2
