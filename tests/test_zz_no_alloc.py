"""ssd_chunk_scan_static_ws: the scan entry point that allocates nothing (its split-scan
workspace is a 16 MiB device array inside the library).

Collected last on purpose: it must pass after the rest of the suite has run on the same
device, as well as alone.  The GPU test calls the new entry through the C ABI twice in a
row on two split workloads and holds each result to the bf16 bar against the existing
entry point run with a caller-owned workspace.
"""
import ctypes

import numpy as np
import pytest
import torch

from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import scan_args_struct as _args
from tolerance import check_bf16

SCRATCH_BYTES = 16 << 20


def test_static_ws_rejects_oversize_plans_and_caller_workspace():
    """Host-side checks, before any launch: a plan wanting more than 16 MiB, and a
    caller workspace passed to the entry that uses its own."""
    lib = ssd.load_library()
    a = ssd.ScanArgs()
    a.struct_size = ctypes.sizeof(ssd.ScanArgs)
    a.x = a.dt = a.A = a.B = a.C = a.cu_seqlens = a.y = 0x1000
    a.act_dtype = ssd.SSD_BF16
    a.nseq, a.T, a.H, a.P, a.G, a.N, a.chunk_size = 1, 65536, 128, 64, 8, 128, 256
    a.seg_chunks = 8          # 64 segments of 4 MiB states
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(a)) > SCRATCH_BYTES
    assert lib.ssd_chunk_scan_static_ws(ctypes.byref(a), None) == 2      # UNSUPPORTED
    a.seg_chunks = -1
    a.workspace, a.workspace_bytes = 0x1000, 256
    assert lib.ssd_chunk_scan_static_ws(ctypes.byref(a), None) == 1      # INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="host-only: the accepted call goes on to launch on a GPU")
def test_static_ws_automatic_plan_keeps_to_the_array():
    """With seg_chunks = 0 the entry plans within its 16 MiB array instead of refusing: a
    long single sequence whose unconstrained plan wants more is
    accepted (without a GPU the call then fails at the launch, SSD_ERR_CUDA, not before
    it with SSD_ERR_UNSUPPORTED); an explicit split that needs more is still refused.
    The shape: one 131072-token sequence on 16 heads of one group."""
    lib = ssd.load_library()
    a = ssd.ScanArgs()
    a.struct_size = ctypes.sizeof(ssd.ScanArgs)
    a.x = a.dt = a.A = a.B = a.C = a.cu_seqlens = a.y = 0x1000
    a.act_dtype = ssd.SSD_BF16
    a.nseq, a.T, a.H, a.P, a.G, a.N, a.chunk_size = 1, 131072, 16, 64, 1, 128, 256
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(a)) > SCRATCH_BYTES
    assert lib.ssd_chunk_scan_static_ws(ctypes.byref(a), None) == 6      # reached the launch
    a.seg_chunks = 2
    assert lib.ssd_chunk_scan_static_ws(ctypes.byref(a), None) == 2      # UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["single_16384_planned", "varlen_seg2", "single_131072_capped"])
def test_static_ws_matches_caller_workspace_twice(case):
    lib = ssd.load_library()
    capped = case == "single_131072_capped"
    if case == "single_16384_planned":
        s = I.scan_workload("mamba2_130m", seqlens=[16384])
        seg = 0
    elif capped:   # 16 heads of one group: the unconstrained plan wants about 17 MiB
        s = I.make_scan_inputs([131072], H=16, P=64, G=1, N=128, chunk_size=256, act="bf16",
                               seed=157, init="all")
        seg = 0
    else:
        s = I.make_scan_inputs([700, 129, 1, 0, 300, 1000, 257, 128, 385], H=4, P=64, G=2,
                               N=128, chunk_size=256, act="bf16", seed=151, init="all")
        seg = 2
    dev = torch.device("cuda")
    T_ = lambda t: torch.from_numpy(np.ascontiguousarray(t.values)).to(
        dev, torch.bfloat16 if t.dtype == "bf16" else torch.float32)
    x, dt, A, B, C, D, bias, init = (T_(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias,
                                                     s.initial_states))
    cu = torch.from_numpy(s.cu_seqlens).to(dev)
    need = ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu, chunk_size=s.chunk_size,
                                         seg_chunks=seg)
    if capped:   # the unconstrained plan wants more than the array: the entry plans within it
        assert need > SCRATCH_BYTES
    else:
        assert 0 < need <= SCRATCH_BYTES      # the case does use the scratch
    y_ref, f_ref = ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=s.chunk_size, D=D,
                                  dt_bias=bias, initial_states=init, seg_chunks=seg)
    torch.cuda.synchronize()
    y_ref, f_ref = y_ref.float().cpu().numpy(), f_ref.cpu().numpy()
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        fs = torch.full((s.nseq, s.H, s.P, s.N), float("nan"), device=dev)
        status = ssd.new_status(dev)
        a = _args(x, dt, A, B, C, cu, s.chunk_size, D=D, dt_bias=bias, init=init, y=y, fs=fs,
                  status=status, seg_chunks=seg)
        rc = lib.ssd_chunk_scan_static_ws(ctypes.byref(a),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, ssd_status(lib, rc)
        rc, bits = ssd.read_status(status)
        assert bits == 0
        check_bf16(f"{case} call {call} y", y.float().cpu().numpy(), y_ref)
        check_bf16(f"{case} call {call} final", fs.cpu().numpy(), f_ref)


@pytest.mark.gpu
def test_static_ws_back_to_back_on_one_stream():
    """Two calls on one stream with different inputs and no synchronisation between them:
    the second call's scan kernel runs after the first call's fix-up kernel (which reads
    the shared array and is launched as a programmatic dependent) on the same stream, so
    reusing the array is safe.  Each result is held to the bf16 bar against the
    caller-workspace entry point."""
    lib = ssd.load_library()
    dev = torch.device("cuda")
    T_ = lambda t: torch.from_numpy(np.ascontiguousarray(t.values)).to(
        dev, torch.bfloat16 if t.dtype == "bf16" else torch.float32)
    cases = []
    for seed in (161, 163):
        s = I.make_scan_inputs([900, 257, 640, 1], H=4, P=64, G=2, N=128, chunk_size=128,
                               act="bf16", seed=seed, init="all")
        t = {k: T_(getattr(s, k)) for k in ("x", "dt", "A", "B", "C", "D", "dt_bias",
                                            "initial_states")}
        t["cu"] = torch.from_numpy(s.cu_seqlens).to(dev)
        y_ref, f_ref = ssd.chunk_scan(t["x"], t["dt"], t["A"], t["B"], t["C"], cu_seqlens=t["cu"],
                                      chunk_size=128, D=t["D"], dt_bias=t["dt_bias"],
                                      initial_states=t["initial_states"], seg_chunks=2)
        cases.append((s, t, y_ref, f_ref))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    outs = []
    for s, t, _, _ in cases:   # launched back to back: no synchronisation in between
        y = torch.full_like(t["x"], float("nan"))
        fs = torch.full((s.nseq, s.H, s.P, s.N), float("nan"), device=dev)
        status = ssd.new_status(dev)
        a = _args(t["x"], t["dt"], t["A"], t["B"], t["C"], t["cu"], 128, D=t["D"],
                  dt_bias=t["dt_bias"], init=t["initial_states"], y=y, fs=fs, status=status,
                  seg_chunks=2)
        assert lib.ssd_chunk_scan_static_ws(ctypes.byref(a),
                                            ctypes.c_void_p(stream.cuda_stream)) == 0
        outs.append((y, fs, status))
    torch.cuda.synchronize()
    for k, ((y, fs, status), (_, _, y_ref, f_ref)) in enumerate(zip(outs, cases)):
        assert ssd.read_status(status)[1] == 0
        check_bf16(f"back-to-back call {k} y", y.float().cpu().numpy(),
                   y_ref.float().cpu().numpy())
        check_bf16(f"back-to-back call {k} final", fs.cpu().numpy(), f_ref.cpu().numpy())


def ssd_status(lib, rc):
    return lib.ssd_status_string(rc).decode()
