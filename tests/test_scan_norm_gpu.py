"""ssd_chunk_scan_gated_norm: the scan, then the gated RMSNorm over its output, in one
call, with the norm launched as a programmatic dependent of the scan (its blocks load z
while the scan runs and wait for it before reading y).

Each case is held to the bar against the oracle's composition (scan, then gated norm)
and, bit for bit, to ssd_chunk_scan followed by gated_rmsnorm as two plain calls.  The
outputs start as NaN, so a norm that read y before the scan had written it would show.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev
from tolerance import TINY, check_bf16, check_fp32, norm_carried_rounding, rtol_K, scan_K

pytestmark = pytest.mark.gpu


def _dev_inputs(s):
    hi = None if s.has_initial_state is None else torch.from_numpy(s.has_initial_state).cuda()
    return dict(x=dev(s.x), dt=dev(s.dt), A=dev(s.A), B=dev(s.B), C=dev(s.C), D=dev(s.D),
                dt_bias=dev(s.dt_bias), initial_states=dev(s.initial_states),
                has_initial_state=hi, cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda())


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def _fused(s, n, gs, *, want_y, seg_chunks=0, z=True, graph=False):
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    zt, wt = (dev(n.z) if z else None), dev(n.weight)
    y = _nan((T, H, P), d["x"].dtype) if want_y else None
    out = _nan((T, H * P), d["x"].dtype)
    fs = _nan((s.nseq, H, P, s.N), torch.float32)
    status = ssd.new_status()

    def call():
        ssd.chunk_scan_gated_norm(d["x"], d["dt"], d["A"], d["B"], d["C"], zt, wt,
                                  cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size,
                                  group_size=gs, eps=n.eps, D=d["D"], dt_bias=d["dt_bias"],
                                  initial_states=d["initial_states"],
                                  has_initial_state=d["has_initial_state"], y=y, out=out,
                                  final_states=fs, status=status, seg_chunks=seg_chunks)

    if graph:
        call()                       # warm-up outside capture (any workspace, module load)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream()
        with torch.cuda.stream(s2):
            with torch.cuda.graph(g, stream=s2):
                call()
        torch.cuda.synchronize()
        for _ in range(2):           # every replay starts from NaN outputs
            out.fill_(float("nan"))
            fs.fill_(float("nan"))
            if y is not None:
                y.fill_(float("nan"))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
    else:
        call()
    _, bits = ssd.read_status(status)
    return out, y, fs, bits


def _separate(s, n, gs, *, seg_chunks=0, z=True, head_block=0, p_block=0):
    d = _dev_inputs(s)
    y, fs = ssd.chunk_scan(d["x"], d["dt"], d["A"], d["B"], d["C"], cu_seqlens=d["cu_seqlens"],
                           chunk_size=s.chunk_size, D=d["D"], dt_bias=d["dt_bias"],
                           initial_states=d["initial_states"],
                           has_initial_state=d["has_initial_state"], seg_chunks=seg_chunks,
                           head_block=head_block, p_block=p_block)
    T, H, P = y.shape
    out = ssd.gated_rmsnorm(y.view(T, H * P), dev(n.z) if z else None, dev(n.weight),
                            group_size=gs, eps=n.eps)
    torch.cuda.synchronize()
    return out, y, fs


def _oracle(s, n, gs, z=True):
    return oracle.scan_gated_norm(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                                  n.z.values if z else None, n.weight.values, group_size=gs,
                                  eps=n.eps, D=s.D.values, dt_bias=s.dt_bias.values,
                                  initial_states=None if s.initial_states is None
                                  else s.initial_states.values,
                                  has_initial_state=s.has_initial_state,
                                  cu_seqlens=s.cu_seqlens)


CASES = {
    # Mamba2-130M-shaped layer: 2 x 2048 tokens, one norm group over d_inner = 1536
    "mamba2_130m": (lambda: I.scan_workload("mamba2_130m"), 1536, 0),
    # ragged varlen with empty and one-token sequences, split into 2-chunk segments
    # (scan kernel, fix-up kernel, then the norm), norm groups of two heads
    "varlen_split": (lambda: I.make_scan_inputs([700, 129, 1, 0, 300, 1000, 257, 128, 385],
                                                H=4, P=64, G=2, N=128, chunk_size=256,
                                                act="bf16", seed=171, init="all"), 128, 2),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("want_y", [True, False])
def test_scan_gated_norm_bf16(case, want_y):
    make, gs, seg = CASES[case]
    s = make()
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=173)
    out, y, fs, bits = _fused(s, n, gs, want_y=want_y, seg_chunks=seg)
    assert bits == 0
    out_sep, y_sep, fs_sep = _separate(s, n, gs, seg_chunks=seg)
    assert torch.equal(out, out_sep), "differs from the two plain calls"
    assert torch.equal(fs, fs_sep)
    if want_y:
        assert torch.equal(y, y_sep)
    yr, fr, outr = _oracle(s, n, gs)
    # y is held in bf16 between the scan and the norm (the layer's activation type), and
    # the norm's gain carries that rounding to out: the max-abs bar counts the error
    # beyond it and beyond out's own rounding
    T = yr.shape[0]
    carried = norm_carried_rounding(yr.reshape(T, -1), n.z.values, n.weight.values, gs, n.eps)
    check_bf16(f"{case} out", out.float().cpu().numpy(), outr, stored_bf16=True,
               carried=carried)
    check_bf16(f"{case} final", fs.cpu().numpy(), fr)
    if want_y:
        check_bf16(f"{case} y", y.float().cpu().numpy(), yr)


def test_scan_gated_norm_in_a_cuda_graph():
    """Captured once and replayed twice from NaN outputs: the dependent launch survives
    capture, and each replay matches the plain calls bit for bit."""
    make, gs, seg = CASES["mamba2_130m"]
    s = make()
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=177)
    out, y, fs, bits = _fused(s, n, gs, want_y=True, seg_chunks=seg, graph=True)
    assert bits == 0
    out_sep, y_sep, fs_sep = _separate(s, n, gs, seg_chunks=seg)
    assert torch.equal(out, out_sep)
    assert torch.equal(y, y_sep)
    assert torch.equal(fs, fs_sep)


def test_scan_gated_norm_fp32_no_gate():
    """fp32 activations (the SIMT scan), no gate, bit for bit to the plain calls.  y is
    held to rtol(K) against the oracle; out to the oracle's composition within rtol(K)
    of y carried through the norm's gain, plus rtol(group_size) of the norm's own
    arithmetic."""
    s = I.scan_workload("tiny_fp32")
    gs = s.H * s.P
    n = I.make_norm_inputs(s.x.values.shape[0], gs, gs, act="f32", seed=179)
    out, y, fs, bits = _fused(s, n, gs, want_y=True, z=False)
    assert bits == 0
    out_sep, _, _ = _separate(s, n, gs, z=False)
    assert torch.equal(out, out_sep)
    yr, fr, ya, fa = oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values,
                                     s.C.values, D=s.D.values, dt_bias=s.dt_bias.values,
                                     cu_seqlens=s.cu_seqlens, with_abs=True)
    Ky, Kf = scan_K(s.cu_seqlens, s.H, s.P, s.N, None)
    check_fp32("fp32 y", y.cpu().numpy(), yr, ya, Ky)
    check_fp32("fp32 final", fs.cpu().numpy(), fr, fa, Kf)
    T = yr.shape[0]
    outr = oracle.gated_rmsnorm(yr.reshape(T, gs), None, n.weight.values, group_size=gs,
                                eps=n.eps)
    dy = (rtol_K(Ky) * ya + TINY).reshape(T, gs)
    bar = (norm_carried_rounding(yr.reshape(T, gs), None, n.weight.values, gs, n.eps, dy=dy)
           + rtol_K(gs) * np.abs(outr) + TINY)
    err = np.abs(out.cpu().numpy().astype(np.float64) - outr)
    frac = float(np.max(err / bar))
    print(f"[bar] fp32 out: worst element used {100 * frac:.3f}% of its bar")
    assert frac <= 1.0


def test_scan_gated_norm_no_tokens():
    """T = 0: nothing to normalise; the final states are the initial states."""
    s = I.make_scan_inputs([0, 0], H=2, P=64, G=1, N=128, chunk_size=256, act="bf16",
                           seed=181, init="all")
    n = I.make_norm_inputs(0, s.H * s.P, s.P, act="bf16", seed=183)
    out, _, fs, bits = _fused(s, n, s.P, want_y=False)
    assert bits == 0 and out.numel() == 0
    assert torch.equal(fs.cpu(), torch.from_numpy(s.initial_states.values).float())


def test_layer_mixed_nemotron_h_shapes_with_concurrent_decode():
    """The mixed layer workload at reduced size, Nemotron-H head shapes (H=128, P=64, G=8,
    norm groups of 16 heads): six ragged packed prefills through the scan + norm call
    while the decode update of 16 pooled slots runs on a second stream.  Both results
    equal the same calls made one after the other, bit for bit; two norm groups and the
    pool are held to the oracle."""
    from gpu_util import scan_oracle
    s = I.make_scan_inputs([300, 129, 1000, 1, 700, 257], H=128, P=64, G=8, N=128,
                           chunk_size=128, act="bf16", seed=191, init=[1, 0, 1, 0, 0, 1])
    T, gs = s.T, 1024
    n = I.make_norm_inputs(T, 128 * 64, gs, act="bf16", seed=193)
    S = 16
    idx = np.random.default_rng(195).permutation(S).astype(np.int32)  # every slot active
    u = I.make_update_inputs(S, idx, 128, 64, 8, 128, act="bf16", seed=197)
    d = _dev_inputs(s)
    zt, wt = dev(n.z), dev(n.weight)
    didx = torch.from_numpy(idx).cuda()

    def run(concurrent):
        pool = dev(u.pool)
        out = _nan((T, 128 * 64), torch.bfloat16)
        fs = _nan((s.nseq, 128, 64, 128), torch.float32)
        uy = _nan((S, 128, 64), torch.bfloat16)
        status = ssd.new_status()
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream() if concurrent else main
        side.wait_stream(main)
        ssd.state_update(pool, didx, dev(u.x), dev(u.dt), dev(u.A), dev(u.B), dev(u.C),
                         D=dev(u.D), dt_bias=dev(u.dt_bias), y=uy, status=status, stream=side)
        ssd.chunk_scan_gated_norm(d["x"], d["dt"], d["A"], d["B"], d["C"], zt, wt,
                                  cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size,
                                  group_size=gs, eps=n.eps, D=d["D"], dt_bias=d["dt_bias"],
                                  initial_states=d["initial_states"],
                                  has_initial_state=d["has_initial_state"], out=out,
                                  final_states=fs, status=status, stream=main)
        main.wait_stream(side)
        _, bits = ssd.read_status(status)
        assert bits == 0
        return out, fs, pool, uy

    out, fs, pool, uy = run(True)
    out2, fs2, pool2, uy2 = run(False)
    assert torch.equal(out, out2) and torch.equal(fs, fs2)
    assert torch.equal(pool, pool2) and torch.equal(uy, uy2)
    for grp in (0, 5):                                   # heads 16 grp .. 16 grp + 15
        heads = list(range(16 * grp, 16 * grp + 16))
        yr, fr = scan_oracle(s, heads=heads)
        cols = slice(gs * grp, gs * (grp + 1))
        outr = oracle.gated_rmsnorm(yr.reshape(T, gs), n.z.values[:, cols],
                                    n.weight.values[cols], group_size=gs, eps=n.eps)
        carried = norm_carried_rounding(yr.reshape(T, gs), n.z.values[:, cols],
                                        n.weight.values[cols], gs, n.eps)
        check_bf16(f"mixed group {grp} out", out[:, cols].float().cpu().numpy(), outr,
                   stored_bf16=True, carried=carried)
        check_bf16(f"mixed group {grp} final", fs[:, heads].cpu().numpy(), fr)
    ref_pool, yr_dec, st = oracle.state_update(u.pool.values, idx, u.x.values, u.dt.values,
                                               u.A.values, u.B.values, u.C.values,
                                               D=u.D.values, dt_bias=u.dt_bias.values)
    assert st == 0
    check_bf16("mixed decode y", uy.float().cpu().numpy(), yr_dec)
    check_bf16("mixed decode pool", pool.cpu().numpy(), ref_pool)


# The overlapped form: the scan (unsplit, 64-channel blocks) counts each finished 128-token
# chunk of each norm group in the workspace, and the norm, launched as a programmatic
# dependent, normalises those rows while the scan runs on.  Each case is checked to take
# that form (its workspace is the ready counters; the form needs at least 3072 tokens),
# then held bit for bit to the chained form of the same call, to the two plain calls and
# to the oracle.
OVERLAP_CASES = {
    # ragged varlen with empty and one-token sequences: one group of 4 heads
    "varlen_one_group_of_4_heads": (
        lambda: I.make_scan_inputs([700, 129, 1, 0, 300, 1000, 257, 128, 385, 1300], H=4,
                                   P=64, G=2, N=128, chunk_size=256, act="bf16", seed=211,
                                   init="all"), 256),
    # 16 heads in 4 groups of 4 heads, four groups per row
    "groups_of_4_heads": (
        lambda: I.make_scan_inputs([513, 64, 1300, 2300], H=16, P=64, G=2, N=128,
                                   chunk_size=128, act="bf16", seed=213, init=[1, 0, 1, 0]),
        256),
    # P = 128: a two-head CTA's two 64-channel head blocks lie in two different groups
    "p128_head_blocks_in_two_groups": (
        lambda: I.make_scan_inputs([400, 777, 3000], H=4, P=128, G=1, N=128, chunk_size=128,
                                   act="bf16", seed=215, init="all"), 256),
    # one group over all 1536 channels of the Mamba2-130M shape: 12 CTAs per group
    "mamba2_130m_one_group": (lambda: I.scan_workload("mamba2_130m"), 1536),
    # two longest sequences of equal length, neither first: the plain scan of the two-call
    # comparison runs its grid longest first, the overlapped form in batch order, and the
    # outputs agree bit for bit
    "tied_longest_not_first": (
        lambda: I.make_scan_inputs([513, 2300, 64, 2300, 0, 1], H=16, P=64, G=2, N=128,
                                   chunk_size=128, act="bf16", seed=219,
                                   init=[1, 0, 1, 1, 0, 1]), 256),
}


# heads per CTA of the scan (both take the overlapped form, in 64-channel blocks)
HB = [1, 2]


def _overlap_call(s, n, gs, *, workspace, want_y, z=True, status=None, head_block=2):
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    zt, wt = (dev(n.z) if z else None), dev(n.weight)
    y = _nan((T, H, P), d["x"].dtype) if want_y else None
    out = _nan((T, H * P), d["x"].dtype)
    fs = _nan((s.nseq, H, P, s.N), torch.float32)
    status = ssd.new_status() if status is None else status
    ssd.chunk_scan_gated_norm(d["x"], d["dt"], d["A"], d["B"], d["C"], zt, wt,
                              cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size,
                              group_size=gs, eps=n.eps, D=d["D"], dt_bias=d["dt_bias"],
                              initial_states=d["initial_states"],
                              has_initial_state=d["has_initial_state"], y=y, out=out,
                              final_states=fs, status=status, seg_chunks=-1,
                              head_block=head_block, p_block=64, workspace=workspace)
    _, bits = ssd.read_status(status)
    return out, y, fs, bits


def _queue_bytes(s, d_channels, gs):
    nid = -(-s.T // 128) + s.nseq
    return (nid * (d_channels // gs) * 4 + 16 + 255) // 256 * 256


def _takes_overlapped_form(s, n, gs, z=True, head_block=2):
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    out = torch.empty((T, H * P), dtype=d["x"].dtype, device="cuda")
    nws = ssd.chunk_scan_gated_norm_workspace_size(
        d["x"], d["B"], d["C"], dev(n.z) if z else None, dev(n.weight), out,
        cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size, group_size=gs, seg_chunks=-1,
        head_block=head_block, p_block=64)
    return nws == _queue_bytes(s, H * P, gs), nws


@pytest.mark.parametrize("case", sorted(OVERLAP_CASES))
@pytest.mark.parametrize("want_y", [True, False])
@pytest.mark.parametrize("hb", HB)
def test_overlapped_scan_gated_norm(case, want_y, hb):
    make, gs = OVERLAP_CASES[case]
    s = make()
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=217)
    ok, nws = _takes_overlapped_form(s, n, gs, head_block=hb)
    assert ok, f"not the overlapped form (workspace {nws})"
    out, y, fs, bits = _overlap_call(s, n, gs, workspace=None, want_y=want_y, head_block=hb)
    assert bits == 0
    chained = torch.empty(0, dtype=torch.uint8, device="cuda")   # too small: the chained form
    out_c, y_c, fs_c, bits_c = _overlap_call(s, n, gs, workspace=chained, want_y=want_y,
                                             head_block=hb)
    assert bits_c == 0
    out_sep, y_sep, fs_sep = _separate(s, n, gs, seg_chunks=-1, head_block=hb, p_block=64)
    assert torch.equal(out, out_c), "overlapped and chained forms differ"
    assert torch.equal(out, out_sep), "differs from the two plain calls"
    assert torch.equal(fs, fs_c) and torch.equal(fs, fs_sep)
    if want_y:
        assert torch.equal(y, y_c) and torch.equal(y, y_sep)
    yr, fr, outr = _oracle(s, n, gs)
    T = yr.shape[0]
    carried = norm_carried_rounding(yr.reshape(T, -1), n.z.values, n.weight.values, gs, n.eps)
    check_bf16(f"overlapped {case} out", out.float().cpu().numpy(), outr, stored_bf16=True,
               carried=carried)
    check_bf16(f"overlapped {case} final", fs.cpu().numpy(), fr)


def test_overlapped_no_gate_and_in_a_cuda_graph():
    """No gate, captured once and replayed twice from NaN outputs: the queue is zeroed by
    the call itself on every replay, and each replay equals the two plain calls."""
    make, gs = OVERLAP_CASES["groups_of_4_heads"]
    s = make()
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=219)
    assert _takes_overlapped_form(s, n, gs, z=False)[0]
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    wt = dev(n.weight)
    out = _nan((T, H * P), d["x"].dtype)
    fs = _nan((s.nseq, H, P, s.N), torch.float32)
    status = ssd.new_status()
    ws = torch.empty(_takes_overlapped_form(s, n, gs, z=False)[1], dtype=torch.uint8,
                     device="cuda")

    def call():
        ssd.chunk_scan_gated_norm(d["x"], d["dt"], d["A"], d["B"], d["C"], None, wt,
                                  cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size,
                                  group_size=gs, eps=n.eps, D=d["D"], dt_bias=d["dt_bias"],
                                  initial_states=d["initial_states"],
                                  has_initial_state=d["has_initial_state"], out=out,
                                  final_states=fs, status=status, seg_chunks=-1,
                                  head_block=2, workspace=ws)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    with torch.cuda.stream(s2):
        with torch.cuda.graph(g, stream=s2):
            call()
    torch.cuda.synchronize()
    out_sep, _, fs_sep = _separate(s, n, gs, seg_chunks=-1, z=False, head_block=2)
    for _ in range(2):
        out.fill_(float("nan"))
        fs.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_sep)
        assert torch.equal(fs, fs_sep)
    _, bits = ssd.read_status(status)
    assert bits == 0


@pytest.mark.parametrize("hb", HB)
def test_overlapped_heads_with_A_not_negative(hb):
    """Head pair 0 has both A >= 0 (its CTAs write zero rows and count every chunk at once),
    head 5 alone of its pair: the status bit is raised, the norm still receives every
    chunk, and the call equals its chained form bit for bit."""
    s = I.make_scan_inputs([600, 37, 900, 2600], H=8, P=64, G=2, N=128, chunk_size=128,
                           act="bf16", seed=221, init="all")
    A = s.A.values.copy()
    A[0], A[1], A[5] = 0.0, np.nan, 0.5
    s.A = I.Tensor(A, "f32")
    gs = 256
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=223)
    assert _takes_overlapped_form(s, n, gs, head_block=hb)[0]
    out, _, fs, bits = _overlap_call(s, n, gs, workspace=None, want_y=False, head_block=hb)
    assert bits & ssd.DEV_A_NOT_NEG
    out_c, _, fs_c, bits_c = _overlap_call(s, n, gs, workspace=torch.empty(0, dtype=torch.uint8,
                                                                            device="cuda"),
                                           want_y=False, head_block=hb)
    assert bits_c & ssd.DEV_A_NOT_NEG
    assert torch.equal(out, out_c)
    assert torch.equal(fs, fs_c)
    assert not torch.isnan(out).any()


# The overlapped form over a split scan: two heads per CTA, each segment of a sequence run
# from the state it enters with (state pass, fold, then the scan), so y is written once
# and counted for the norm.  The workspace is the split's, then the counters.  Held bit for
# bit to the chained form of the same split (the split's workspace only), to the two plain
# calls with the same split, and to the oracle.
SPLIT_OVERLAP_CASES = {
    "varlen_one_group_of_4_heads": ("varlen_one_group_of_4_heads", 2),
    "groups_of_4_heads": ("groups_of_4_heads", 3),
    "p128_head_blocks_in_two_groups": ("p128_head_blocks_in_two_groups", 4),
    "mamba2_130m_one_group": ("mamba2_130m_one_group", 4),
}


def _split_call(s, n, gs, seg, *, workspace, want_y):
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    y = _nan((T, H, P), d["x"].dtype) if want_y else None
    out = _nan((T, H * P), d["x"].dtype)
    fs = _nan((s.nseq, H, P, s.N), torch.float32)
    status = ssd.new_status()
    ssd.chunk_scan_gated_norm(d["x"], d["dt"], d["A"], d["B"], d["C"], dev(n.z), dev(n.weight),
                              cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size,
                              group_size=gs, eps=n.eps, D=d["D"], dt_bias=d["dt_bias"],
                              initial_states=d["initial_states"],
                              has_initial_state=d["has_initial_state"], y=y, out=out,
                              final_states=fs, status=status, seg_chunks=seg, head_block=2,
                              workspace=workspace)
    _, bits = ssd.read_status(status)
    return out, y, fs, bits


@pytest.mark.parametrize("case", sorted(SPLIT_OVERLAP_CASES))
@pytest.mark.parametrize("want_y", [True, False])
def test_overlapped_split_scan_gated_norm(case, want_y):
    name, seg = SPLIT_OVERLAP_CASES[case]
    make, gs = OVERLAP_CASES[name]
    s = make()
    n = I.make_norm_inputs(s.x.values.shape[0], s.H * s.P, gs, act="bf16", seed=225)
    d = _dev_inputs(s)
    T, H, P = d["x"].shape
    split = ssd.chunk_scan_workspace_size(d["x"], d["B"], d["C"], cu_seqlens=d["cu_seqlens"],
                                          chunk_size=s.chunk_size, seg_chunks=seg,
                                          head_block=2)
    out_t = torch.empty((T, H * P), dtype=d["x"].dtype, device="cuda")
    nws = ssd.chunk_scan_gated_norm_workspace_size(
        d["x"], d["B"], d["C"], dev(n.z), dev(n.weight), out_t, cu_seqlens=d["cu_seqlens"],
        chunk_size=s.chunk_size, group_size=gs, seg_chunks=seg, head_block=2)
    assert split > 0 and nws == split + _queue_bytes(s, H * P, gs), (split, nws)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    out, y, fs, bits = _split_call(s, n, gs, seg, workspace=ws, want_y=want_y)
    assert bits == 0
    ws_c = torch.empty(split, dtype=torch.uint8, device="cuda")   # the chained form
    out_c, y_c, fs_c, bits_c = _split_call(s, n, gs, seg, workspace=ws_c, want_y=want_y)
    assert bits_c == 0
    out_sep, y_sep, fs_sep = _separate(s, n, gs, seg_chunks=seg, head_block=2)
    assert torch.equal(out, out_c), "overlapped and chained forms differ"
    assert torch.equal(out, out_sep), "differs from the two plain calls"
    assert torch.equal(fs, fs_c) and torch.equal(fs, fs_sep)
    if want_y:
        assert torch.equal(y, y_c) and torch.equal(y, y_sep)
    yr, fr, outr = _oracle(s, n, gs)
    carried = norm_carried_rounding(yr.reshape(T, -1), n.z.values, n.weight.values, gs, n.eps)
    check_bf16(f"overlapped split {case} out", out.float().cpu().numpy(), outr,
               stored_bf16=True, carried=carried)
    check_bf16(f"overlapped split {case} final", fs.cpu().numpy(), fr)


@pytest.mark.parametrize("L", [1024, 4096, 16384, 65536])
def test_layer_single_sequence_full_size(L):
    """The single-sequence layer calls the benchmark times: one sequence of L tokens,
    H=128, P=64, G=8, N=128, an initial state, norm groups of 1024, through the form the
    library plans for it (chained at 1024 tokens, overlapped from 4096).  y and the final
    states of heads from four groups against the oracle; `out` on rows across the sequence
    against the oracle's gated norm of the call's own y (a property that holds at any
    size)."""
    from gpu_util import scan_oracle
    s = I.make_scan_inputs([L], H=128, P=64, G=8, N=128, chunk_size=128, act="bf16",
                           seed=231, init="all")
    T, gs = s.T, 1024
    n = I.make_norm_inputs(T, 128 * 64, gs, act="bf16", seed=233)
    d = _dev_inputs(s)
    nws = ssd.chunk_scan_gated_norm_workspace_size(
        d["x"], d["B"], d["C"], dev(n.z), dev(n.weight),
        torch.empty((T, 128 * 64), dtype=torch.bfloat16, device="cuda"),
        cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size, group_size=gs)
    overlapped = nws == _queue_bytes(s, 128 * 64, gs)
    assert overlapped == (L >= 4096), f"L={L}: workspace {nws}"
    del d
    out, y, fs, bits = _fused(s, n, gs, want_y=True)
    assert bits == 0
    heads = [0, 37, 64, 127]
    yr, fr = scan_oracle(s, heads=heads)
    yg = y.float().cpu().numpy()
    check_bf16(f"layer {L} y", yg[:, heads], yr, stored_bf16=True)
    check_bf16(f"layer {L} final", fs[:, heads].cpu().numpy(), fr)
    rows = np.arange(0, T, 997 if L > 4096 else 61)
    yrows = yg[rows].reshape(len(rows), -1)
    ref = oracle.gated_rmsnorm(yrows, n.z.values[rows], n.weight.values, group_size=gs,
                               eps=n.eps)
    check_bf16(f"layer {L} out rows", out.float().cpu().numpy()[rows], ref, stored_bf16=True)


def test_layer_nemotron_h_varlen_full_size():
    """The benchmark's headline call at full size: the 4 packed sequences (8192, 3000, 517,
    4675), H=128, G=8, initial states on sequences 0 and 2, norm groups of 1024, through the
    form the library plans (the overlapped one).  y and the final states of every head
    against the oracle, and `out` on rows of every sequence against the oracle's gated norm
    of the call's own y."""
    from gpu_util import scan_oracle
    s = I.scan_workload("nemotron_h_varlen")
    T, gs = s.T, 1024
    n = I.make_norm_inputs(T, 128 * 64, gs, act="bf16", seed=235)
    d = _dev_inputs(s)
    nws = ssd.chunk_scan_gated_norm_workspace_size(
        d["x"], d["B"], d["C"], dev(n.z), dev(n.weight),
        torch.empty((T, 128 * 64), dtype=torch.bfloat16, device="cuda"),
        cu_seqlens=d["cu_seqlens"], chunk_size=s.chunk_size, group_size=gs)
    assert nws == _queue_bytes(s, 128 * 64, gs), f"not the overlapped form (workspace {nws})"
    del d
    out, y, fs, bits = _fused(s, n, gs, want_y=True)
    assert bits == 0
    yr, fr = scan_oracle(s)
    yg = y.float().cpu().numpy()
    check_bf16("headline call y", yg, yr, stored_bf16=True)
    check_bf16("headline call final", fs.cpu().numpy(), fr)
    rows = np.concatenate([np.arange(a, b, 61) for a, b in zip(s.cu_seqlens[:-1], s.cu_seqlens[1:])])
    yrows = yg[rows].reshape(len(rows), -1)
    ref = oracle.gated_rmsnorm(yrows, n.z.values[rows], n.weight.values, group_size=gs,
                               eps=n.eps)
    check_bf16("headline call out rows", out.float().cpu().numpy()[rows], ref, stored_bf16=True)


def test_layer_mixed_64_prefills_full_size():
    """The mixed layer batch the benchmark times, at full size: 64 packed prefills of
    128..4096 tokens (133 547 tokens), H=128, P=64, G=8, N=128, initial states on every other
    sequence, norm groups of 1024, through the call as the library plans it (a grid of 28
    waves: the chained form).  Inputs are drawn on the device in the workloads'
    distributions (2 GB each of x and z: too slow to draw on the host in a test) and the
    oracle reads them back.  y and the final states of heads from four groups against the
    oracle, and `out` on rows of every sequence against the oracle's gated norm of the call's
    own y."""
    lens = np.random.default_rng(4243).integers(128, 4097, size=64)
    T, H, P, G, N, gs = int(lens.sum()), 128, 64, 8, 128, 1024
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(237)
    bf = torch.bfloat16

    def randn(*shape):
        return torch.randn(shape, generator=gen, device="cuda")

    x = randn(T, H, P).to(bf)
    dt = randn(T, H)
    A = -torch.exp(torch.rand(H, generator=gen, device="cuda") * math.log(16.0))
    u = torch.rand(H, generator=gen, device="cuda") * (0.1 - 1e-3) + 1e-3
    bias = torch.log(torch.expm1(u))
    Dp = randn(H)
    B = (randn(T, G, N) / math.sqrt(N)).to(bf)
    C = (randn(T, G, N) / math.sqrt(N)).to(bf)
    init = 0.1 * randn(64, H, P, N)
    hi = torch.tensor([1, 0] * 32, dtype=torch.uint8, device="cuda")
    z = randn(T, H * P).to(bf)
    w = (1 + 0.1 * randn(H * P)).to(bf)
    y = _nan((T, H, P), bf)
    out = _nan((T, H * P), bf)
    fs = _nan((64, H, P, N), torch.float32)
    status = ssd.new_status()
    ssd.chunk_scan_gated_norm(x, dt, A, B, C, z, w, cu_seqlens=torch.from_numpy(cu).cuda(),
                              chunk_size=128, group_size=gs, eps=1e-5, D=Dp, dt_bias=bias,
                              initial_states=init, has_initial_state=hi, y=y, out=out,
                              final_states=fs, status=status)
    _, bits = ssd.read_status(status)
    assert bits == 0
    heads = np.array([0, 37, 64, 127])
    g = heads // (H // G)
    th = torch.from_numpy(heads).cuda()
    tg = torch.from_numpy(g).cuda()
    host = lambda t: t.float().cpu().numpy()  # noqa: E731
    yr, fr = oracle.scan_seq(host(x[:, th]), host(dt[:, th]), host(A[th]), host(B[:, tg]),
                             host(C[:, tg]), D=host(Dp[th]), dt_bias=host(bias[th]),
                             initial_states=host(init[:, th]), has_initial_state=hi.cpu().numpy(),
                             cu_seqlens=cu)
    check_bf16("mixed 64 y", host(y[:, th]), yr, stored_bf16=True)
    check_bf16("mixed 64 final", host(fs[:, th]), fr)
    rows = torch.from_numpy(np.concatenate([np.arange(a, b, 211) for a, b in
                                            zip(cu[:-1], cu[1:])])).cuda()
    ref = oracle.gated_rmsnorm(host(y[rows]).reshape(len(rows), -1), host(z[rows]), host(w),
                               group_size=gs, eps=1e-5)
    check_bf16("mixed 64 out rows", host(out[rows]), ref, stored_bf16=True)
