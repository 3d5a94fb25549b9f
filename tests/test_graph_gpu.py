"""The library's calls are asynchronous on the caller's stream and capturable: a CUDA graph
of one layer step (a split scan, whose fix-up kernel is launched with programmatic
dependent launch, then the gated norm, with a decode update on a second stream forked
and joined inside the capture) replays to the same results as the calls made eagerly."""
import numpy as np
import pytest
import torch

from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev

pytestmark = pytest.mark.gpu


def test_layer_step_in_a_cuda_graph_matches_eager():
    s = I.scan_workload("mamba2_130m", seqlens=[3000, 1000])
    H, P, G, N, T = s.H, s.P, s.G, s.N, s.T
    d = H * P
    x, dt, A, B, C, D, bias = (dev(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias))
    init = dev(s.initial_states)
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    nrm = I.make_norm_inputs(T, d, 1536, act="bf16", seed=601)
    z, w = dev(nrm.z), dev(nrm.weight)
    u = I.make_update_inputs(4, [2, 0], H, P, G, N, act="bf16", seed=603)
    ws = torch.empty(ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu, chunk_size=256,
                                                   seg_chunks=4), dtype=torch.uint8,
                     device="cuda")
    assert ws.numel() > 0

    side = torch.cuda.Stream()

    def run(y, fs, out, pool, uy):
        # the decode token forks onto a second stream and joins at the end
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            ssd.state_update(pool, idx, ux, udt, uA, uB, uC, D=uD, dt_bias=ubias, y=uy)
        ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=256, D=D, dt_bias=bias,
                       initial_states=init, y=y, final_states=fs, seg_chunks=4, workspace=ws)
        ssd.gated_rmsnorm(y.view(T, d), z, w, group_size=1536, out=out)
        main.wait_stream(side)

    idx = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    ux, udt, uA, uB, uC, uD, ubias = (dev(t) for t in (u.x, u.dt, u.A, u.B, u.C, u.D,
                                                       u.dt_bias))
    bufs = [dict(y=torch.empty_like(x), fs=torch.empty((2, H, P, N), device="cuda"),
                 out=torch.empty((T, d), dtype=torch.bfloat16, device="cuda"),
                 pool=dev(u.pool), uy=torch.empty((2, H, P), dtype=torch.bfloat16,
                                                  device="cuda")) for _ in range(2)]
    run(**bufs[0])                              # eager
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(**bufs[1])
    g.replay()
    torch.cuda.synchronize()
    for k in ("y", "fs", "out", "pool", "uy"):
        assert torch.equal(bufs[0][k], bufs[1][k]), k
