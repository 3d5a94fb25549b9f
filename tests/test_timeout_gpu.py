"""Failure detection of the tensor-core scan, exercised without a GPU fault.

Every pipeline wait of the scan kernels is bounded: a wait that runs out raises a CTA-wide
abort flag, each role drains the copies and MMAs it has in flight, TMEM is freed, and the
kernel returns with SSD_DEV_TIMEOUT in the caller's status word.  To make a wait run out
on purpose, the test builds a separate variant of the library (``-DSSD_FAULT_INJECT``,
wait limit 2e8 SM cycles, about 0.1 s) whose decay warp can be told to withhold the
"prologue ready" arrival of one chunk.  Nothing is left waiting without a limit, no
address is bad and nothing traps: the kernel gives up, reports, and returns.

The test then runs a normal scan through the regular library on the same CUDA context and
holds it to the bf16 bar against the oracle, so the context is shown to be still usable.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from mamba2_ssd_state_gb300 import build as B
from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev, scan_args_struct, scan_gpu, scan_oracle
from tolerance import check_bf16

pytestmark = pytest.mark.gpu

VARIANT_DIR = os.path.join(B.HERE, "_build_fault")
VARIANT_LIB = os.path.join(VARIANT_DIR, "libssd_fault.so")
FLAGS = ["-DSSD_FAULT_INJECT", "-DSSD_WAIT_LIMIT_CYCLES=200000000LL"]


@pytest.fixture(scope="module")
def fault_lib():
    path = B.build(lib=VARIANT_LIB, build_dir=VARIANT_DIR, extra_flags=FLAGS)
    lib = ctypes.CDLL(path)
    lib.ssd_chunk_scan.argtypes = [ctypes.POINTER(ssd.ScanArgs), ctypes.c_void_p]
    lib.ssd_chunk_scan.restype = ctypes.c_int
    lib.ssd_chunk_scan_gated_norm.argtypes = [ctypes.POINTER(ssd.ScanArgs), ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int32,
                                              ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    lib.ssd_chunk_scan_gated_norm.restype = ctypes.c_int
    lib.ssd_chunk_scan_gated_norm_workspace_size.argtypes = [
        ctypes.POINTER(ssd.ScanArgs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p]
    lib.ssd_chunk_scan_gated_norm_workspace_size.restype = ctypes.c_size_t
    lib.ssd_test_withhold_chunk.argtypes = [ctypes.c_int]
    lib.ssd_test_withhold_chunk.restype = ctypes.c_int
    yield lib
    lib.ssd_test_withhold_chunk(-1)


def _case():
    # one 600-token sequence (5 chunks of 128) on 2 heads: a handful of CTAs, every one of
    # which reaches the withheld chunk
    return I.make_scan_inputs([600], H=2, P=64, G=1, N=128, chunk_size=256, act="bf16",
                              seed=907, init="none")


def test_no_withheld_chunk_runs_clean(fault_lib):
    """The variant with nothing withheld is the regular kernel: no timeout, right answer."""
    s = _case()
    x, dt, A, Bm, C, D, bias = (dev(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias))
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    y = torch.zeros_like(x)
    fs = torch.zeros((s.nseq, s.H, s.P, s.N), device="cuda")
    status = ssd.new_status()
    a = scan_args_struct(x, dt, A, Bm, C, cu, s.chunk_size, D=D, dt_bias=bias, y=y, fs=fs,
                         status=status, seg_chunks=-1)
    a.impl = 2
    assert fault_lib.ssd_test_withhold_chunk(-1) == 0
    rc = fault_lib.ssd_chunk_scan(ctypes.byref(a),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    rc, bits = ssd.read_status(status)
    assert (rc, bits) == (0, 0)
    y_ref, f_ref = scan_oracle(s)
    check_bf16("variant y", y.float().cpu().numpy(), y_ref)
    check_bf16("variant final", fs.cpu().numpy(), f_ref)


def test_withheld_chunk_times_out_and_context_survives(fault_lib):
    s = _case()
    x, dt, A, Bm, C, D, bias = (dev(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias))
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    y = torch.zeros_like(x)
    fs = torch.zeros((s.nseq, s.H, s.P, s.N), device="cuda")
    status = ssd.new_status()
    a = scan_args_struct(x, dt, A, Bm, C, cu, s.chunk_size, D=D, dt_bias=bias, y=y, fs=fs,
                         status=status, seg_chunks=-1)
    a.impl = 2  # SSD_IMPL_TC: the path with the pipelined waits
    assert fault_lib.ssd_test_withhold_chunk(1) == 0
    try:
        rc = fault_lib.ssd_chunk_scan(ctypes.byref(a),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0                       # the launch itself is fine
        rc, bits = ssd.read_status(status)   # synchronises: the kernel has returned
    finally:
        fault_lib.ssd_test_withhold_chunk(-1)
    assert bits & 0x8, f"SSD_DEV_TIMEOUT not raised (bits={bits:#x})"
    assert rc == 7                           # SSD_ERR_TIMEOUT
    assert torch.cuda.synchronize() is None  # no sticky error on the context

    # the same context still runs the regular library correctly
    y_gpu, f_gpu, bits = scan_gpu(s, impl="tc")
    assert bits == 0
    y_ref, f_ref = scan_oracle(s)
    check_bf16("after timeout y", y_gpu, y_ref)
    check_bf16("after timeout final", f_gpu, f_ref)


@pytest.mark.parametrize("hb,seg", [(1, -1), (2, -1), (2, 8)])
def test_overlapped_norm_stops_waiting_when_the_scan_aborts(fault_lib, hb, seg):
    """The scan + norm call in its overlapped form (the norm drains a queue the scan fills
    as it runs): when the scan gives up on a withheld chunk, it raises the queue's abort
    flag, the norm's blocks stop waiting for the chunks that will not come, and the call
    ends with SSD_DEV_TIMEOUT on a context that still runs the regular library.  With
    seg = 8 the scan is a two-head split (state pass, fold, then every segment from its
    entering state: each segment's chunk 1 is withheld)."""
    # 4 heads (two head pairs), one norm group over their 256 channels; 4200 tokens (the
    # overlapped form needs at least 3072)
    s = I.make_scan_inputs([4200], H=4, P=64, G=2, N=128, chunk_size=256, act="bf16",
                           seed=911, init="none")
    x, dt, A, Bm, C, D, bias = (dev(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias))
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    T, d = s.T, s.H * s.P
    nrm = I.make_norm_inputs(T, d, d, act="bf16", seed=909)
    z, w = dev(nrm.z), dev(nrm.weight)
    out = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    fs = torch.zeros((s.nseq, s.H, s.P, s.N), device="cuda")
    status = ssd.new_status()
    a = scan_args_struct(x, dt, A, Bm, C, cu, s.chunk_size, D=D, dt_bias=bias, fs=fs,
                         status=status, seg_chunks=seg, head_block=hb)
    a.impl, a.p_block = 2, 64
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    nws = fault_lib.ssd_chunk_scan_gated_norm_workspace_size(ctypes.byref(a), ptr(z), ptr(w),
                                                            d, ptr(out))
    assert nws > 0, "the case must take the overlapped form"
    if seg > 0:  # the split's part comes first, then the ready counters
        split = ssd.chunk_scan_workspace_size(x, Bm, C, cu_seqlens=cu, chunk_size=s.chunk_size,
                                              seg_chunks=seg, head_block=hb, p_block=64)
        assert 0 < split < nws
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), nws
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert fault_lib.ssd_test_withhold_chunk(1) == 0
    try:
        rc = fault_lib.ssd_chunk_scan_gated_norm(ctypes.byref(a), ptr(z), ptr(w), ssd.SSD_BF16,
                                                 d, ctypes.c_float(1e-5), ptr(out), stream)
        assert rc == 0
        rc, bits = ssd.read_status(status)
    finally:
        fault_lib.ssd_test_withhold_chunk(-1)
    assert bits & 0x8, f"SSD_DEV_TIMEOUT not raised (bits={bits:#x})"
    assert rc == 7
    assert torch.cuda.synchronize() is None

    # the same context: the regular library's overlapped call equals its plain calls
    out2, _ = ssd.chunk_scan_gated_norm(x, dt, A, Bm, C, z, w, cu_seqlens=cu,
                                        chunk_size=s.chunk_size, group_size=d, D=D,
                                        dt_bias=bias, seg_chunks=seg, head_block=hb, p_block=64)
    y_sep, _ = ssd.chunk_scan(x, dt, A, Bm, C, cu_seqlens=cu, chunk_size=s.chunk_size, D=D,
                              dt_bias=bias, seg_chunks=seg, head_block=hb, p_block=64)
    out_sep = ssd.gated_rmsnorm(y_sep.view(T, d), z, w, group_size=d)
    torch.cuda.synchronize()
    assert torch.equal(out2, out_sep)
