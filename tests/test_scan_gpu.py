"""GPU parity of ssd_chunk_scan against the double-precision oracle.

fp32 inputs are held to rtol(K) (tolerance.py); bf16 inputs to rel-L2 <= 1e-2 and
max-abs <= 5e-2 on y and on the final states.  Shapes span several 128-token tiles,
ragged tails, one-token and empty sequences, and the full workload sizes (the large one
checked on a sample of heads computed by the oracle).
"""
import numpy as np
import pytest
import torch

import oracle

from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev, scan_gpu, scan_oracle
from tolerance import check_bf16, check_fp32, scan_K

pytestmark = pytest.mark.gpu


def _check_fp32_scan(name, s, y, fs):
    yr, fr, ya, fa = scan_oracle(s, with_abs=True)
    Ky, Kf = scan_K(s.cu_seqlens, s.H, s.P, s.N, s.has_initial_state)
    check_fp32(f"{name} y", y, yr, ya, Ky)
    check_fp32(f"{name} final", fs, fr, fa, Kf)


def test_tiny_fp32_layer():
    """64 tokens, H=4, P=16, G=1, N=16, chunk 16, fp32, zero initial state."""
    s = I.scan_workload("tiny_fp32")
    y, fs, bits = scan_gpu(s)
    assert bits == 0
    _check_fp32_scan("tiny_fp32", s, y, fs)


@pytest.mark.parametrize("N", [16, 48, 128])
def test_fp32_varlen_edges(N):
    s = I.make_scan_inputs([37, 1, 0, 16, 65, 3], H=4, P=16, G=2, N=N, chunk_size=16,
                           act="f32", seed=101, init=[1, 0, 1, 1, 0, 1])
    y, fs, bits = scan_gpu(s)
    assert bits == 0
    _check_fp32_scan(f"fp32 varlen N={N}", s, y, fs)
    # the empty sequence returns its initial state
    np.testing.assert_array_equal(fs[2], s.initial_states.values[2])


SEQS = [300, 129, 1, 64, 700, 0, 128, 127, 255]


# The tensor-core kernels: one head per CTA at channel blocks 16, 32 and 64, and the
# head-pair kernel (two heads of one group per CTA, 64 channels each).
TC_KERNELS = [(16, 1), (32, 1), (64, 1), (64, 2)]


@pytest.mark.parametrize("p_block,head_block", TC_KERNELS)
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_bf16_tensor_core_parity(p_block, head_block, chunk):
    s = I.make_scan_inputs(SEQS, H=4, P=64, G=2, N=128, chunk_size=chunk, act="bf16",
                           seed=103, init=[1, 0, 1, 1, 0, 1, 0, 1, 1])
    y, fs, bits = scan_gpu(s, impl="tc", p_block=p_block, head_block=head_block)
    assert bits == 0
    yr, fr = scan_oracle(s)
    tag = f"tc pb={p_block} hb={head_block} Q={chunk}"
    check_bf16(f"{tag} y", y, yr)
    check_bf16(f"{tag} final", fs, fr)


def test_bf16_simt_parity():
    s = I.make_scan_inputs([200, 1, 57], H=4, P=32, G=2, N=128, chunk_size=128, act="bf16",
                           seed=107, init=[1, 1, 0])
    y, fs, bits = scan_gpu(s, impl="simt")
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("simt bf16 y", y, yr)
    check_bf16("simt bf16 final", fs, fr)


def test_tc_without_D_and_final_states():
    s = I.make_scan_inputs([150, 90], H=2, P=32, G=1, N=128, chunk_size=128, act="bf16",
                           seed=109, init="all")
    y, fs, bits = scan_gpu(s, impl="tc", final=False, D=False)
    assert fs is None and bits == 0
    yr, _ = scan_oracle(s, D=False)
    check_bf16("tc no-D y", y, yr)


def test_tc_strided_projection_layout():
    """x, B and C read zero-copy as column slices of one packed projection buffer."""
    Ls, H, P, G, N = [333, 64], 4, 64, 2, 128
    s = I.make_scan_inputs(Ls, H=H, P=P, G=G, N=N, chunk_size=128, act="bf16", seed=113,
                           init=[1, 0])
    T = s.T
    W = H * P + 2 * G * N + 64          # pad so the token stride is not the dense size
    buf = torch.zeros((T, W), dtype=torch.bfloat16, device="cuda")
    buf[:, :H * P] = dev(s.x).view(T, H * P)
    buf[:, H * P:H * P + G * N] = dev(s.B).view(T, G * N)
    buf[:, H * P + G * N:H * P + 2 * G * N] = dev(s.C).view(T, G * N)
    x = buf[:, :H * P].view(T, H, P)
    B = buf[:, H * P:H * P + G * N].view(T, G, N)
    C = buf[:, H * P + G * N:H * P + 2 * G * N].view(T, G, N)
    yr, fr = scan_oracle(s)
    for impl in ("tc", "simt"):
        y, fs = ssd.chunk_scan(x, dev(s.dt), dev(s.A), B, C,
                               cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda(), chunk_size=128,
                               D=dev(s.D), dt_bias=dev(s.dt_bias),
                               initial_states=dev(s.initial_states),
                               has_initial_state=torch.from_numpy(s.has_initial_state).cuda(),
                               impl=impl)
        check_bf16(f"strided {impl} y", y.float().cpu().numpy(), yr)
        check_bf16(f"strided {impl} final", fs.cpu().numpy(), fr)


def test_tc_and_simt_agree():
    s = I.make_scan_inputs([513, 77], H=4, P=64, G=1, N=128, chunk_size=128, act="bf16",
                           seed=127, init=[1, 1])
    y1, f1, _ = scan_gpu(s, impl="tc")
    y2, f2, _ = scan_gpu(s, impl="simt")
    check_bf16("tc vs simt y", y1, y2)
    check_bf16("tc vs simt final", f1, f2)


# Split sequences: segments of k 128-token chunks, each scanned from zero, chained by the
# combine kernel and corrected by the fix-up kernel.  The lengths give sequences of 1 to
# 8 chunks with ragged tails, exact chunk multiples, one token and an empty one.
SEG_SEQS = [700, 129, 1, 0, 300, 1000, 257, 128, 385]
SEG_INIT = [1, 0, 1, 1, 0, 1, 1, 0, 1]


@pytest.mark.parametrize("p_block,head_block", TC_KERNELS)
@pytest.mark.parametrize("seg", [1, 2, 3])
def test_bf16_segmented_parity(p_block, head_block, seg):
    s = I.make_scan_inputs(SEG_SEQS, H=4, P=64, G=2, N=128, chunk_size=256, act="bf16",
                           seed=141, init=SEG_INIT)
    y, fs, bits = scan_gpu(s, impl="tc", p_block=p_block, seg_chunks=seg,
                           head_block=head_block)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16(f"seg={seg} pb={p_block} hb={head_block} y", y, yr)
    check_bf16(f"seg={seg} pb={p_block} hb={head_block} final", fs, fr)
    # the empty sequence still returns its initial state, untouched by the chaining
    np.testing.assert_array_equal(fs[3], s.initial_states.values[3])
    # and the split agrees with the unsplit chain
    y1, f1, _ = scan_gpu(s, impl="tc", p_block=p_block, seg_chunks=-1, head_block=head_block)
    check_bf16(f"seg={seg} vs unsplit y", y, y1)
    check_bf16(f"seg={seg} vs unsplit final", fs, f1)


def test_segmented_A_not_negative():
    s = I.make_scan_inputs([600, 200], H=3, P=32, G=1, N=128, chunk_size=128, act="bf16",
                           seed=143, init="all")
    A = s.A.values.copy()
    A[1] = 0.0
    s.A = I.Tensor(A, "f32")
    y, fs, bits = scan_gpu(s, impl="tc", seg_chunks=1)
    assert bits & ssd.DEV_A_NOT_NEG
    assert np.all(y[:, 1] == 0) and np.all(fs[:, 1] == 0)
    yr, fr = scan_oracle(s, heads=[0, 2])
    check_bf16("segmented good heads y", y[:, [0, 2]], yr)
    check_bf16("segmented good heads final", fs[:, [0, 2]], fr)


def test_segmented_needs_workspace():
    s = I.make_scan_inputs([600], H=2, P=32, G=1, N=128, chunk_size=128, act="bf16", seed=145)
    args = (dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C))
    kw = dict(cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda(), chunk_size=128, impl="tc",
              D=dev(s.D), dt_bias=dev(s.dt_bias))
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ssd.SsdError) as e:   # forced split, workspace too small
        ssd.chunk_scan(*args, seg_chunks=1, workspace=small, **kw)
    assert e.value.code == 1
    # with seg_chunks = 0 the same workspace just means "run unsplit"
    y, _ = ssd.chunk_scan(*args, workspace=small, **kw)
    yr, _ = scan_oracle(s)
    check_bf16("unsplit fallback y", y.float().cpu().numpy(), yr)


@pytest.mark.parametrize("seg", [-1, 1])
def test_pair_one_head_A_not_negative(seg):
    """A head pair whose second head fails the sign test: that head's y and final state
    are zero and the status bit is set, while its partner (same CTA, same C.B^T and the
    same batched products) still matches the oracle."""
    s = I.make_scan_inputs([600, 130], H=4, P=64, G=2, N=128, chunk_size=128, act="bf16",
                           seed=147, init="all")
    A = s.A.values.copy()
    A[1] = float("nan")
    A[2] = 0.0
    s.A = I.Tensor(A, "f32")
    y, fs, bits = scan_gpu(s, impl="tc", head_block=2, seg_chunks=seg)
    assert bits & ssd.DEV_A_NOT_NEG
    for h in (1, 2):
        assert np.all(y[:, h] == 0) and np.all(fs[:, h] == 0)
    yr, fr = scan_oracle(s, heads=[0, 3])
    check_bf16(f"pair bad heads seg={seg} y", y[:, [0, 3]], yr)
    check_bf16(f"pair bad heads seg={seg} final", fs[:, [0, 3]], fr)


def test_pair_headdim_128():
    """P = 128: each head pair runs as two CTAs, one per 64-channel block."""
    s = I.make_scan_inputs([300, 77, 513], H=4, P=128, G=1, N=128, chunk_size=128, act="bf16",
                           seed=149, init=[1, 0, 1])
    y, fs, bits = scan_gpu(s, impl="tc", head_block=2)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("pair P=128 y", y, yr)
    check_bf16("pair P=128 final", fs, fr)


@pytest.mark.parametrize("shape", [dict(H=3, G=1, P=64), dict(H=6, G=2, P=64),
                                   dict(H=4, G=2, P=32)])
def test_pair_unsupported_shapes(shape):
    """Two heads per CTA need H and H/G even and 64-channel blocks: other shapes are
    refused with SSD_ERR_UNSUPPORTED when the pair kernel is forced, and run one head per
    CTA when the library chooses."""
    s = I.make_scan_inputs([200], N=128, chunk_size=128, act="bf16", seed=151, init="all",
                           **shape)
    with pytest.raises(ssd.SsdError) as e:
        scan_gpu(s, impl="tc", head_block=2)
    assert e.value.code == 2
    y, fs, bits = scan_gpu(s, impl="tc")
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16(f"auto {shape} y", y, yr)


@pytest.mark.parametrize("impl", ["tc", "simt"])
def test_A_not_negative_sets_status(impl):
    s = I.make_scan_inputs([140], H=3, P=32, G=1, N=128, chunk_size=128, act="bf16", seed=131,
                           init="all")
    A = s.A.values.copy()
    A[1] = 0.0
    s.A = I.Tensor(A, "f32")
    y, fs, bits = scan_gpu(s, impl=impl)
    assert bits & ssd.DEV_A_NOT_NEG
    assert np.all(y[:, 1] == 0) and np.all(fs[:, 1] == 0)
    yr, fr = scan_oracle(s, heads=[0, 2])
    check_bf16(f"{impl} good heads y", y[:, [0, 2]], yr)


@pytest.mark.parametrize("impl", ["tc", "simt"])
def test_bad_cu_seqlens_sets_status(impl):
    s = I.make_scan_inputs([100, 50], H=2, P=32, G=1, N=128, chunk_size=128, act="bf16",
                           seed=137)
    cu = torch.tensor([0, 120, 100], dtype=torch.int32, device="cuda")  # decreasing
    status = ssd.new_status()
    ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C), cu_seqlens=cu,
                   chunk_size=128, status=status, impl=impl)
    rc, bits = ssd.read_status(status)
    assert bits & ssd.DEV_SEQ_META
    assert rc == 5


def test_host_validation_errors():
    s = I.make_scan_inputs([16], H=2, P=16, G=1, N=16, chunk_size=16, act="f32", seed=139)
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    with pytest.raises(ssd.SsdError) as e:
        ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C), cu_seqlens=cu,
                       chunk_size=0)
    assert e.value.code == 1
    with pytest.raises(ssd.SsdError) as e:   # fp32 has no tensor-core path
        ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C), cu_seqlens=cu,
                       chunk_size=16, impl="tc")
    assert e.value.code == 2


# ----------------------------------------------------------------------------- full sizes

@pytest.mark.parametrize("seg", [0, -1])
def test_mamba2_130m_layer_full(seg):
    """2 x 2048 tokens, H=24, P=64, G=1, N=128, chunk 256, initial states: whole output,
    as the library plans it (seg 0: split into segments) and as one chain per sequence."""
    s = I.scan_workload("mamba2_130m")
    y, fs, bits = scan_gpu(s, seg_chunks=seg)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16(f"mamba2_130m seg={seg} y", y, yr)
    check_bf16(f"mamba2_130m seg={seg} final", fs, fr)


def test_nemotron_h_varlen_all_heads():
    """4 packed sequences (8192, 3000, 517, 4675), H=128, G=8, as the library plans it
    (the launch the benchmark times): every head, every token, every final state."""
    s = I.scan_workload("nemotron_h_varlen")
    y, fs, bits = scan_gpu(s)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("nemotron_h y", y, yr)
    check_bf16("nemotron_h final", fs, fr)


@pytest.mark.parametrize("seg,head_block", [(4, 0), (-1, 1), (4, 1)])
def test_nemotron_h_varlen_sampled_heads(seg, head_block):
    """The same batch split into 4-chunk segments and with one head per CTA: heads from
    every group."""
    s = I.scan_workload("nemotron_h_varlen")
    y, fs, bits = scan_gpu(s, seg_chunks=seg, head_block=head_block)
    assert bits == 0
    heads = [0, 17, 38, 63, 64, 90, 111, 127]
    yr, fr = scan_oracle(s, heads=heads)
    check_bf16(f"nemotron_h seg={seg} hb={head_block} y", y[:, heads], yr)
    check_bf16(f"nemotron_h seg={seg} hb={head_block} final", fs[:, heads], fr)


def test_single_long_sequence_planned_split():
    """One 16384-token sequence on 24 heads: the planner splits it into segments (48 CTAs
    of 128 chunks would leave most SMs idle); sampled heads against the oracle, and the
    whole output against the unsplit chain."""
    s = I.scan_workload("mamba2_130m", seqlens=[16384])
    x = dev(s.x)
    assert ssd.chunk_scan_workspace_size(x, dev(s.B), dev(s.C),
                                         cu_seqlens=torch.from_numpy(s.cu_seqlens).cuda(),
                                         chunk_size=s.chunk_size) > 0
    y, fs, bits = scan_gpu(s)
    assert bits == 0
    heads = [0, 11, 23]
    yr, fr = scan_oracle(s, heads=heads)
    check_bf16("single 16384 split y", y[:, heads], yr)
    check_bf16("single 16384 split final", fs[:, heads], fr)
    y1, f1, _ = scan_gpu(s, seg_chunks=-1)
    check_bf16("single 16384 split vs unsplit y", y, y1)
    check_bf16("single 16384 split vs unsplit final", fs, f1)


# ----------------------------------------------------------------------- more edge shapes

def test_many_short_sequences_tc():
    """300 packed sequences of 0 to 40 tokens (a third of them empty or one token), mixed
    initial states: 300 chains of one partial chunk each."""
    rng = np.random.default_rng(501)
    lens = rng.integers(0, 41, 300)
    lens[::7] = 0
    lens[::11] = 1
    init = (rng.random(300) < 0.5).astype(int).tolist()
    s = I.make_scan_inputs(lens.tolist(), H=2, P=32, G=1, N=128, chunk_size=128, act="bf16",
                           seed=503, init=init)
    y, fs, bits = scan_gpu(s, impl="tc")
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("300 short seqs y", y, yr)
    check_bf16("300 short seqs final", fs, fr)
    empty = np.flatnonzero(lens == 0)
    np.testing.assert_array_equal(fs[empty], s.initial_states.values[empty])


@pytest.mark.parametrize("seg", [1, 2])
def test_split_many_sequences_segment_lookup(seg):
    """70 packed sequences (empty, one token, up to five chunks) split into segments of
    1 or 2 chunks: each CTA of the scan and of the fix-up finds its segment with one
    warp reading the lengths 32 sequences at a time, so the lookup crosses three groups
    of 32, with segment counts that differ from sequence to sequence."""
    rng = np.random.default_rng(509)
    lens = rng.choice([0, 1, 127, 128, 129, 300, 600], size=70)
    init = (rng.random(70) < 0.5).astype(int).tolist()
    s = I.make_scan_inputs(lens.tolist(), H=2, P=64, G=1, N=128, chunk_size=128, act="bf16",
                           seed=511, init=init)
    y, fs, bits = scan_gpu(s, impl="tc", seg_chunks=seg)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16(f"70 seqs seg {seg} y", y, yr)
    check_bf16(f"70 seqs seg {seg} final", fs, fr)
    empty = np.flatnonzero(lens == 0)
    np.testing.assert_array_equal(fs[empty], s.initial_states.values[empty])


def test_tc_headdim_128_group_per_head():
    """P = 128 (two 64-channel blocks per head), G = H: every head its own B and C."""
    s = I.make_scan_inputs([300, 77, 513], H=3, P=128, G=3, N=128, chunk_size=128, act="bf16",
                           seed=507, init=[1, 1, 0])
    for pb in (64, 32):
        y, fs, bits = scan_gpu(s, impl="tc", p_block=pb)
        assert bits == 0
        yr, fr = scan_oracle(s)
        check_bf16(f"P=128 pb={pb} y", y, yr)
        check_bf16(f"P=128 pb={pb} final", fs, fr)


def test_tc_plain_dt_no_D_all_initial():
    """dt used as given (no softplus, no bias: positive raw values), no D, initial states
    for every sequence with has_initial_state left NULL (all used)."""
    s = I.make_scan_inputs([250, 129, 1], H=4, P=64, G=2, N=128, chunk_size=128, act="bf16",
                           seed=509, init="all")
    s.dt = I.Tensor(np.abs(s.dt.values) * 0.05 + 0.01, "f32")
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    status = ssd.new_status()
    y, fs = ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C), cu_seqlens=cu,
                           chunk_size=128, dt_softplus=False,
                           initial_states=dev(s.initial_states), status=status, impl="tc")
    assert ssd.read_status(status)[1] == 0
    yr, fr = oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                             dt_softplus=False,
                             initial_states=s.initial_states.values, cu_seqlens=s.cu_seqlens)
    check_bf16("plain dt y", y.float().cpu().numpy(), yr)
    check_bf16("plain dt final", fs.cpu().numpy(), fr)


def test_split_instance_without_split_sequences():
    """A forced segment length longer than every sequence: the segmented kernel instance
    runs, but no sequence has a second segment, so no fix-up CTA has work."""
    s = I.make_scan_inputs([300, 5, 0, 250], H=2, P=64, G=1, N=128, chunk_size=256,
                           act="bf16", seed=511, init=[1, 0, 1, 1])
    y, fs, bits = scan_gpu(s, impl="tc", seg_chunks=8)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("no-split instance y", y, yr)
    check_bf16("no-split instance final", fs, fr)


# The decay mask is factorised per 8-token group (two multiplies per element) where the
# factors stay within range, and computed exactly per element where they do not.  With
# the workloads' dt every block takes the factorised form; these cases drive the exact
# form too.
MASK_KERNELS = [(64, 1), (0, 2)]


@pytest.mark.parametrize("p_block,head_block", MASK_KERNELS)
def test_strong_decay_takes_both_mask_forms(p_block, head_block):
    """Heads whose decay over 8 tokens exceeds the factor bound (A down to -4000: the exact
    form) beside heads far inside it, over ragged sequences."""
    s = I.make_scan_inputs([700, 129, 1, 300, 385], H=8, P=64, G=2, N=128, chunk_size=128,
                           act="bf16", seed=601, init="all")
    s.A = I.Tensor(np.array([-4000.0, -1.0, -300.0, -5.0, -60.0, -2.0, -900.0, -16.0],
                            dtype=np.float32), "f32")
    y, fs, bits = scan_gpu(s, impl="tc", p_block=p_block, head_block=head_block)
    assert bits == 0
    yr, fr = scan_oracle(s)
    assert np.isfinite(y).all() and np.isfinite(fs).all()
    check_bf16(f"strong decay hb={head_block} y", y, yr)
    check_bf16(f"strong decay hb={head_block} final", fs, fr)


@pytest.mark.parametrize("p_block,head_block", MASK_KERNELS)
def test_plain_dt_with_negative_steps(p_block, head_block):
    """dt used as given with some negative steps: the cumulative decay rises in places, so
    both the factorised form's range checks and the exact form see exp(cs_i - cs_j) > 1."""
    s = I.make_scan_inputs([520, 129, 7, 400], H=4, P=64, G=2, N=128, chunk_size=128,
                           act="bf16", seed=603, init="all")
    rng = np.random.default_rng(605)
    s.dt = I.Tensor((rng.uniform(-0.02, 0.06, size=s.dt.values.shape)).astype(np.float32), "f32")
    cu = torch.from_numpy(s.cu_seqlens).cuda()
    status = ssd.new_status()
    y, fs = ssd.chunk_scan(dev(s.x), dev(s.dt), dev(s.A), dev(s.B), dev(s.C), cu_seqlens=cu,
                           chunk_size=128, dt_softplus=False, D=dev(s.D),
                           initial_states=dev(s.initial_states), status=status, impl="tc",
                           p_block=p_block, head_block=head_block)
    assert ssd.read_status(status)[1] == 0
    yr, fr = oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                             D=s.D.values, dt_softplus=False,
                             initial_states=s.initial_states.values, cu_seqlens=s.cu_seqlens)
    check_bf16(f"negative dt hb={head_block} y", y.float().cpu().numpy(), yr)
    check_bf16(f"negative dt hb={head_block} final", fs.cpu().numpy(), fr)


@pytest.mark.parametrize("seg", [1, 2, 5])
def test_pair_split_headdim_128_groups(seg):
    """The two-head split at P = 128 (two 64-channel blocks per head pair: the state pass,
    the fold and the scan each run per block) and G = 2 (two head pairs per group), with
    sequences of whole segments, a partial last segment, one token and none."""
    s = I.make_scan_inputs([640, 77, 1, 0, 513, 1280], H=8, P=128, G=2, N=128, chunk_size=128,
                           act="bf16", seed=613, init=[1, 0, 1, 1, 0, 1])
    y, fs, bits = scan_gpu(s, impl="tc", head_block=2, seg_chunks=seg)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16(f"pair split P=128 seg={seg} y", y, yr)
    check_bf16(f"pair split P=128 seg={seg} final", fs, fr)
    np.testing.assert_array_equal(fs[3], s.initial_states.values[3])  # the empty sequence


def test_pair_split_without_D_and_final_states():
    """The two-head split with no D and no final states (the last segment writes nothing,
    the state pass and the fold still carry every later segment's entering state)."""
    s = I.make_scan_inputs([900, 300], H=4, P=64, G=1, N=128, chunk_size=256, act="bf16",
                           seed=617, init="all")
    y, fs, bits = scan_gpu(s, impl="tc", head_block=2, seg_chunks=2, final=False, D=False)
    assert bits == 0 and fs is None
    yr, _ = scan_oracle(s, D=False)
    check_bf16("pair split no D y", y, yr)


def test_pair_split_long_segments():
    """Segments of 12 chunks: the state pass's rings (3 TMA stages, 8 weight slots, 4 dt
    chunks) wrap several times within a segment; a 25-chunk sequence gives two whole
    segments and a one-chunk last one."""
    s = I.make_scan_inputs([3100, 200], H=4, P=64, G=2, N=128, chunk_size=128, act="bf16",
                           seed=619, init=[1, 1])
    y, fs, bits = scan_gpu(s, impl="tc", head_block=2, seg_chunks=12)
    assert bits == 0
    yr, fr = scan_oracle(s)
    check_bf16("pair split seg=12 y", y, yr)
    check_bf16("pair split seg=12 final", fs, fr)
    y1, f1, _ = scan_gpu(s, impl="tc", head_block=2, seg_chunks=-1)
    check_bf16("pair split seg=12 vs unsplit y", y, y1)
    check_bf16("pair split seg=12 vs unsplit final", fs, f1)


@pytest.mark.parametrize("p_block,head_block", [(64, 1), (64, 2)])
@pytest.mark.parametrize("nseq", [2, 31, 32, 33])
def test_longest_first_slot_order(p_block, head_block, nseq):
    """Packed sequences in ascending length, with runs of equal lengths and empty ones: an
    unsplit grid of up to 32 sequences runs them longest first, so every slot maps to another
    sequence and ties break by index; 33 sequences keep batch order."""
    rng = np.random.default_rng(521 + nseq)
    lens = np.sort(rng.choice([0, 1, 100, 128, 129, 256, 300, 513], size=nseq))
    init = (rng.random(nseq) < 0.5).astype(int).tolist()
    s = I.make_scan_inputs(lens.tolist(), H=2, P=64, G=1, N=128, chunk_size=128, act="bf16",
                           seed=523, init=init)
    y, fs, bits = scan_gpu(s, impl="tc", p_block=p_block, head_block=head_block, seg_chunks=0)
    assert bits == 0
    yr, fr = scan_oracle(s)
    tag = f"{nseq} ascending seqs pb={p_block} hb={head_block}"
    check_bf16(f"{tag} y", y, yr)
    check_bf16(f"{tag} final", fs, fr)
    empty = np.flatnonzero(lens == 0)
    np.testing.assert_array_equal(fs[empty], s.initial_states.values[empty])
