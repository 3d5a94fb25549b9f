"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the
library through its binding, and run the oracle on the same values."""
import ctypes

import numpy as np
import torch

import oracle
from mamba2_ssd_state_gb300 import ssd


def dev(t, device="cuda"):
    """inputs.Tensor -> torch tensor in its storage dtype (exact: values are representable)."""
    if t is None:
        return None
    dtype = torch.bfloat16 if t.dtype == "bf16" else torch.float32
    return torch.from_numpy(np.ascontiguousarray(t.values)).to(device=device, dtype=dtype)


def scan_gpu(s, impl="auto", p_block=0, final=True, chunk_size=None, D=True, seg_chunks=0,
             head_block=0):
    status = ssd.new_status()
    hi = None if s.has_initial_state is None else torch.from_numpy(s.has_initial_state).cuda()
    y, fs = ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C),
                           cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda(),
                           chunk_size=chunk_size or s.chunk_size,
                           D=dev(s.D) if D else None, dt_bias=dev(s.dt_bias),
                           initial_states=dev(s.initial_states), has_initial_state=hi,
                           return_final_states=final, status=status, impl=impl,
                           p_block=p_block, seg_chunks=seg_chunks, head_block=head_block)
    rc, bits = ssd.read_status(status)
    torch.cuda.synchronize()
    yf = y.float().cpu().numpy()
    ff = fs.cpu().numpy() if fs is not None else None
    return yf, ff, bits


def scan_oracle(s, heads=None, with_abs=False, D=True):
    """Oracle over all heads, or over a subset of heads (each head's recurrence is
    independent: the subset is run as its own layer with one group per head)."""
    x, dt, A, B, C = s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values
    Dv, bias = s.D.values, s.dt_bias.values
    init = None if s.initial_states is None else s.initial_states.values
    if heads is not None:
        heads = np.asarray(heads)
        g = heads // (s.H // s.G)
        x, dt, A, Dv, bias = x[:, heads], dt[:, heads], A[heads], Dv[heads], bias[heads]
        B, C = B[:, g], C[:, g]
        if init is not None:
            init = init[:, heads]
    return oracle.scan_seq(x, dt, A, B, C, D=Dv if D else None, dt_bias=bias,
                           initial_states=init, has_initial_state=s.has_initial_state,
                           cu_seqlens=s.cu_seqlens, with_abs=with_abs)


def scan_args_struct(x, dt, A, B, C, cu, chunk_size, *, D=None, dt_bias=None, init=None, y=None,
          fs=None, status=None, seg_chunks=0, head_block=0):
    """ssd_scan_args for the given tensors (the marshalling of ssd.chunk_scan), for tests
    that call an entry point of the C ABI directly."""
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    a = ssd.ScanArgs()
    a.struct_size = ctypes.sizeof(ssd.ScanArgs)
    a.x, a.x_stride_t = ssd._ptr(x), H * P
    a.dt, a.dt_bias, a.dt_softplus = ssd._ptr(dt), ssd._ptr(dt_bias), 1
    a.A, a.D = ssd._ptr(A), ssd._ptr(D)
    a.B, a.B_stride_t = ssd._ptr(B), G * N
    a.C, a.C_stride_t = ssd._ptr(C), G * N
    a.initial_states = ssd._ptr(init)
    a.cu_seqlens = ssd._ptr(cu)
    a.nseq, a.T, a.H, a.P, a.G, a.N = cu.shape[0] - 1, T, H, P, G, N
    a.chunk_size = chunk_size
    a.act_dtype = ssd._act(x)
    a.y, a.final_states, a.d_status = ssd._ptr(y), ssd._ptr(fs), ssd._ptr(status)
    a.seg_chunks, a.head_block = seg_chunks, head_block
    return a
