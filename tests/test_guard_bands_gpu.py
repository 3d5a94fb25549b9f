"""Memory safety of every entry point, checked with guard bands (compute-sanitizer is
closed on this pool).

Every buffer a call writes (y, out, final states, per-token states, the decode pools,
the slot-copy destination, the scan's workspace, the status word) is cut from the middle
of a larger allocation whose head and tail are filled with a sentinel byte.  After the
call the bands must still hold the sentinel, bit for bit: a write one element past an
output (the kind of out-of-bounds bug the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)"
reports fixing with clamps in its #675 message) lands in a band and fails the test.
The shapes hit the kernels' edges: a sequence's partial last 128-token tile, empty and
one-token sequences, P = 128 (two channel blocks per head), 1-, 2- and 3-chunk segments
of the split scan, -1 rows and a 4-token decode step.  Each guarded call's outputs are
also checked against the same call on plain buffers.
"""
import numpy as np
import pytest
import torch

from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev

pytestmark = pytest.mark.gpu

PAD = 4096         # bytes of band on each side (keeps every view 4 KiB-aligned)
SENTINEL = 0xA5


class Guarded:
    """A tensor of the given shape and dtype inside [band | tensor | band]."""

    def __init__(self, shape, dtype, fill=None):
        esz = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * esz
        self.buf = torch.full((PAD + self.nbytes + PAD,), SENTINEL, dtype=torch.uint8,
                              device="cuda")
        self.t = self.buf[PAD:PAD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, name):
        torch.cuda.synchronize()
        head = self.buf[:PAD].cpu().numpy()
        tail = self.buf[PAD + self.nbytes:].cpu().numpy()
        bad_h = np.flatnonzero(head != SENTINEL)
        bad_t = np.flatnonzero(tail != SENTINEL)
        assert bad_h.size == 0, f"{name}: {bad_h.size} bytes written before the buffer"
        assert bad_t.size == 0, f"{name}: {bad_t.size} bytes written past the buffer " \
                                f"(first at +{bad_t[0]})"


SEQS = [300, 129, 1, 0, 128, 127, 700, 255]     # partial tiles, empty, one token


def _scan_case(P, H=4, G=2, seqs=SEQS, seed=601):
    return I.make_scan_inputs(seqs, H=H, P=P, G=G, N=128, chunk_size=128, act="bf16",
                              seed=seed, init=[1, 0] * (len(seqs) // 2) + [1] * (len(seqs) % 2))


def _scan_inputs(s):
    return dict(x=dev(s.x), dt=dev(s.dt), A=dev(s.A), B=dev(s.B), C=dev(s.C), D=dev(s.D),
                bias=dev(s.dt_bias), init=dev(s.initial_states),
                hi=torch.from_numpy(s.has_initial_state).cuda(),
                cu=torch.from_numpy(s.cu_seqlens).cuda())


@pytest.mark.parametrize("impl,head_block,seg,P", [
    ("tc", 2, -1, 64), ("tc", 2, 1, 64), ("tc", 2, 2, 128), ("tc", 1, -1, 64),
    ("tc", 1, 3, 64), ("tc", 1, 2, 128), ("simt", 0, -1, 64)])
def test_scan_outputs_stay_in_bounds(impl, head_block, seg, P):
    s = _scan_case(P)
    i = _scan_inputs(s)
    T, H, N, nseq = s.T, s.H, s.N, s.nseq
    kw = dict(cu_seqlens=i["cu"], chunk_size=128, D=i["D"], dt_bias=i["bias"],
              initial_states=i["init"], has_initial_state=i["hi"], impl=impl,
              head_block=head_block, seg_chunks=seg)
    args = (i["x"], i["dt"], i["A"], i["B"], i["C"])
    y_ref, f_ref = ssd.chunk_scan(*args, **kw)
    nws = ssd.chunk_scan_workspace_size(i["x"], i["B"], i["C"], cu_seqlens=i["cu"],
                                        chunk_size=128, impl=impl, seg_chunks=seg,
                                        head_block=head_block)
    y = Guarded((T, H, P), torch.bfloat16)
    fs = Guarded((nseq, H, P, N), torch.float32)
    st = Guarded((1,), torch.int32, fill=torch.zeros(1, dtype=torch.int32, device="cuda"))
    ws = Guarded((max(nws, 256),), torch.uint8) if seg > 0 else None
    ssd.chunk_scan(*args, y=y.t, final_states=fs.t, status=st.t,
                   workspace=None if ws is None else ws.t, **kw)
    for g, nm in ((y, "y"), (fs, "final_states"), (st, "status")):
        g.check(nm)
    if ws is not None:
        ws.check("workspace")
    assert int(st.t.item()) == 0
    torch.testing.assert_close(y.t, y_ref, rtol=0, atol=0)
    torch.testing.assert_close(fs.t, f_ref, rtol=0, atol=0)


@pytest.mark.parametrize("with_y", [True, False])
def test_scan_gated_norm_outputs_stay_in_bounds(with_y):
    s = _scan_case(64, H=16, G=1, seed=607)
    i = _scan_inputs(s)
    T, H, P, N, nseq = s.T, s.H, s.P, s.N, s.nseq
    nrm = I.make_norm_inputs(T, H * P, 256, act="bf16", seed=609)
    z, w = dev(nrm.z), dev(nrm.weight)
    kw = dict(cu_seqlens=i["cu"], chunk_size=128, group_size=256, eps=1e-5, D=i["D"],
              dt_bias=i["bias"], initial_states=i["init"], has_initial_state=i["hi"])
    args = (i["x"], i["dt"], i["A"], i["B"], i["C"], z, w)
    out_ref, f_ref = ssd.chunk_scan_gated_norm(*args, **kw)
    out = Guarded((T, H * P), torch.bfloat16)
    fs = Guarded((nseq, H, P, N), torch.float32)
    y = Guarded((T, H, P), torch.bfloat16) if with_y else None
    ssd.chunk_scan_gated_norm(*args, out=out.t, final_states=fs.t,
                              y=None if y is None else y.t, **kw)
    out.check("out")
    fs.check("final_states")
    if y is not None:
        y.check("y")
    torch.testing.assert_close(out.t, out_ref, rtol=0, atol=0)
    torch.testing.assert_close(fs.t, f_ref, rtol=0, atol=0)


@pytest.mark.parametrize("with_y,hb", [(True, 2), (False, 2), (True, 1)])
def test_overlapped_scan_gated_norm_stays_in_bounds(with_y, hb):
    """The overlapped form (head pairs, unsplit): its outputs and its ready queue (the
    workspace) stay inside their buffers, and the outputs equal the chained form's."""
    s = _scan_case(64, H=16, G=1, seqs=SEQS + [2600], seed=611)   # >= 3072 tokens
    i = _scan_inputs(s)
    T, H, P, N, nseq = s.T, s.H, s.P, s.N, s.nseq
    nrm = I.make_norm_inputs(T, H * P, 256, act="bf16", seed=613)
    z, w = dev(nrm.z), dev(nrm.weight)
    kw = dict(cu_seqlens=i["cu"], chunk_size=128, group_size=256, eps=1e-5, D=i["D"],
              dt_bias=i["bias"], initial_states=i["init"], has_initial_state=i["hi"],
              seg_chunks=-1, head_block=hb, p_block=64)
    args = (i["x"], i["dt"], i["A"], i["B"], i["C"], z, w)
    chained = torch.empty(0, dtype=torch.uint8, device="cuda")
    out_ref, f_ref = ssd.chunk_scan_gated_norm(*args, workspace=chained, **kw)
    out = Guarded((T, H * P), torch.bfloat16)
    fs = Guarded((nseq, H, P, N), torch.float32)
    y = Guarded((T, H, P), torch.bfloat16) if with_y else None
    nws = ssd.chunk_scan_gated_norm_workspace_size(
        i["x"], i["B"], i["C"], z, w, out.t, y=None if y is None else y.t, cu_seqlens=i["cu"],
        chunk_size=128, group_size=256, seg_chunks=-1, head_block=hb, p_block=64)
    assert nws > 0
    ws = Guarded((nws,), torch.uint8)
    st = Guarded((1,), torch.int32, fill=torch.zeros(1, dtype=torch.int32, device="cuda"))
    ssd.chunk_scan_gated_norm(*args, out=out.t, final_states=fs.t, status=st.t, workspace=ws.t,
                              y=None if y is None else y.t, **kw)
    for g, nm in ((out, "out"), (fs, "final_states"), (ws, "workspace"), (st, "status")):
        g.check(nm)
    if y is not None:
        y.check("y")
    assert int(st.t.item()) == 0
    torch.testing.assert_close(out.t, out_ref, rtol=0, atol=0)
    torch.testing.assert_close(fs.t, f_ref, rtol=0, atol=0)


def test_static_ws_scan_outputs_stay_in_bounds():
    import ctypes

    from gpu_util import scan_args_struct

    s = _scan_case(64, seqs=[900, 1, 0, 385], seed=611)
    i = _scan_inputs(s)
    T, H, P, N, nseq = s.T, s.H, s.P, s.N, s.nseq
    y_ref, f_ref = ssd.chunk_scan(i["x"], i["dt"], i["A"], i["B"], i["C"], cu_seqlens=i["cu"],
                                  chunk_size=128, D=i["D"], dt_bias=i["bias"],
                                  initial_states=i["init"], seg_chunks=2)
    y = Guarded((T, H, P), torch.bfloat16)
    fs = Guarded((nseq, H, P, N), torch.float32)
    a = scan_args_struct(i["x"], i["dt"], i["A"], i["B"], i["C"], i["cu"], 128, D=i["D"],
                         dt_bias=i["bias"], init=i["init"], y=y.t, fs=fs.t, seg_chunks=2)
    lib = ssd.load_library()
    assert lib.ssd_chunk_scan_static_ws(
        ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    y.check("y")
    fs.check("final_states")
    torch.testing.assert_close(y.t, y_ref, rtol=0, atol=0)
    torch.testing.assert_close(fs.t, f_ref, rtol=0, atol=0)


def _decode_case(ntok=None, seed=613):
    S, H, P, G, N, batch = 6, 4, 64, 2, 128, 5
    idx = np.array([4, -1, 0, 5, 2], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=seed, ntok=ntok)
    return u, S, H, P, G, N, batch, idx


def test_state_update_outputs_stay_in_bounds():
    u, S, H, P, G, N, batch, idx = _decode_case()
    args = lambda pool: (pool, torch.from_numpy(idx).cuda(), dev(u.x), dev(u.dt), dev(u.A),  # noqa
                         dev(u.B), dev(u.C))
    kw = dict(D=dev(u.D), dt_bias=dev(u.dt_bias))
    pool_ref = dev(u.pool).clone()
    y_ref = ssd.state_update(*args(pool_ref), **kw)
    pool = Guarded((S, H, P, N), torch.float32, fill=dev(u.pool))
    y = Guarded((batch, H, P), torch.bfloat16)
    ssd.state_update(*args(pool.t), y=y.t, **kw)
    pool.check("state_pool")
    y.check("y")
    torch.testing.assert_close(pool.t, pool_ref, rtol=0, atol=0)
    torch.testing.assert_close(y.t, y_ref, rtol=0, atol=0)


def test_state_update_multi_outputs_stay_in_bounds():
    ntok = 4
    u, S, H, P, G, N, batch, idx = _decode_case(ntok=ntok, seed=617)
    args = lambda pool: (pool, torch.from_numpy(idx).cuda(), dev(u.x), dev(u.dt), dev(u.A),  # noqa
                         dev(u.B), dev(u.C))
    kw = dict(D=dev(u.D), dt_bias=dev(u.dt_bias))
    pool_ref = dev(u.pool).clone()
    y_ref, inter_ref = ssd.state_update_multi(*args(pool_ref), inter_states=True, **kw)
    pool = Guarded((S, H, P, N), torch.float32, fill=dev(u.pool))
    y = Guarded((batch, ntok, H, P), torch.bfloat16)
    inter = Guarded((batch, ntok, H, P, N), torch.float32,
                    fill=torch.zeros((batch, ntok, H, P, N), device="cuda"))
    ssd.state_update_multi(*args(pool.t), y=y.t, inter_states=inter.t, **kw)
    for g, nm in ((pool, "state_pool"), (y, "y"), (inter, "inter_states")):
        g.check(nm)
    torch.testing.assert_close(pool.t, pool_ref, rtol=0, atol=0)
    torch.testing.assert_close(y.t, y_ref, rtol=0, atol=0)
    active = idx >= 0
    torch.testing.assert_close(inter.t[torch.from_numpy(active)],
                               inter_ref[torch.from_numpy(active)], rtol=0, atol=0)


def test_decode_layer_step_outputs_stay_in_bounds():
    u, S, H, P, G, N, batch, idx = _decode_case(seed=619)
    d = H * P
    z = torch.randn((batch, d), device="cuda").to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(d, device="cuda")).to(torch.bfloat16)
    args = lambda pool: (pool, torch.from_numpy(idx).cuda(), dev(u.x), dev(u.dt), dev(u.A),  # noqa
                         dev(u.B), dev(u.C), z, w)
    kw = dict(group_size=128, D=dev(u.D), dt_bias=dev(u.dt_bias))
    pool_ref = dev(u.pool).clone()
    out_ref = ssd.decode_layer_step(*args(pool_ref), **kw)
    pool = Guarded((S, H, P, N), torch.float32, fill=dev(u.pool))
    y = Guarded((batch, H, P), torch.bfloat16)
    out = Guarded((batch, d), torch.bfloat16)
    ssd.decode_layer_step(*args(pool.t), y=y.t, out=out.t, **kw)
    for g, nm in ((pool, "state_pool"), (y, "y"), (out, "out")):
        g.check(nm)
    torch.testing.assert_close(out.t, out_ref, rtol=0, atol=0)


def test_state_copy_destination_stays_in_bounds():
    H, P, N = 2, 64, 128
    src = torch.randn((5, H, P, N), device="cuda")
    dst = Guarded((4, H, P, N), torch.float32, fill=torch.zeros((4, H, P, N), device="cuda"))
    si = torch.tensor([4, -1, 0, 2], dtype=torch.int32, device="cuda")
    di = torch.tensor([3, 1, 0, -1], dtype=torch.int32, device="cuda")
    ssd.state_copy(src, si, dst.t, di)
    dst.check("dst_pool")
    torch.testing.assert_close(dst.t[3], src[4], rtol=0, atol=0)
    torch.testing.assert_close(dst.t[0], src[0], rtol=0, atol=0)
    assert torch.count_nonzero(dst.t[1]) == 0 and torch.count_nonzero(dst.t[2]) == 0


@pytest.mark.parametrize("rows,d,gs", [(37, 1536, 1536), (129, 8192, 1024), (5, 64, 16)])
def test_gated_rmsnorm_output_stays_in_bounds(rows, d, gs):
    nrm = I.make_norm_inputs(rows, d, gs, act="bf16", seed=621)
    x, z, w = dev(nrm.x), dev(nrm.z), dev(nrm.weight)
    out_ref = ssd.gated_rmsnorm(x, z, w, group_size=gs)
    out = Guarded((rows, d), torch.bfloat16)
    ssd.gated_rmsnorm(x, z, w, group_size=gs, out=out.t)
    out.check("out")
    torch.testing.assert_close(out.t, out_ref, rtol=0, atol=0)
