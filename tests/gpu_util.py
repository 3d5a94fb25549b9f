"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the
library through its binding, and run the oracle on the same values."""
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


def scan_gpu(s, impl="auto", p_block=0, final=True, chunk_size=None, D=True, seg_chunks=0):
    status = ssd.new_status()
    hi = None if s.has_initial_state is None else torch.from_numpy(s.has_initial_state).cuda()
    y, fs = ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C),
                           cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda(),
                           chunk_size=chunk_size or s.chunk_size,
                           D=dev(s.D) if D else None, dt_bias=dev(s.dt_bias),
                           initial_states=dev(s.initial_states), has_initial_state=hi,
                           return_final_states=final, status=status, impl=impl,
                           p_block=p_block, seg_chunks=seg_chunks)
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
