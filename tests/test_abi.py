"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every entry
point include/ssd.h declares, its argument structs have the C layout the binding
assumes, and host-side validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import subprocess

import pytest

from mamba2_ssd_state_gb300 import build as B
from mamba2_ssd_state_gb300 import ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ssd.load_library()


def test_exports_every_declared_entry_point(lib):
    names = ssd.header_functions()
    assert set(names) == {"ssd_chunk_scan", "ssd_chunk_scan_workspace_size",
                          "ssd_chunk_scan_static_ws", "ssd_chunk_scan_gated_norm",
                          "ssd_chunk_scan_gated_norm_workspace_size",
                          "ssd_state_update", "ssd_state_update_multi", "ssd_decode_layer_step",
                          "ssd_state_copy", "gated_rmsnorm", "ssd_read_status",
                          "ssd_status_string", "ssd_version"}
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing but the C ABI is exported
    assert exported == set(names)


def test_struct_layout_matches_c(tmp_path):
    fields = {"ssd_scan_args": ssd.ScanArgs, "ssd_update_args": ssd.UpdateArgs}
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "ssd.h"', "int main(void){"]
    for cname, cls in fields.items():
        src.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            src.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    src.append("return 0;}")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", f"-I{ROOT}/include", str(c), "-o", str(exe)], check=True)
    got = dict(ln.rsplit(" ", 1) for ln in subprocess.run([str(exe)], capture_output=True,
                                                          text=True, check=True).stdout.split("\n") if ln)
    for cname, cls in fields.items():
        assert int(got[cname]) == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(cls, f).offset, f


def _scan_args(**kw):
    a = ssd.ScanArgs()
    a.struct_size = ctypes.sizeof(ssd.ScanArgs)
    a.x = a.dt = a.A = a.B = a.C = a.cu_seqlens = a.y = 0x1000
    a.nseq, a.T, a.H, a.P, a.G, a.N, a.chunk_size = 1, 8, 4, 16, 2, 16, 16
    a.act_dtype = ssd.SSD_F32
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(struct_size=8), dict(A=None), dict(cu_seqlens=None), dict(x=None), dict(nseq=0),
    dict(H=3), dict(G=0), dict(P=0), dict(N=0), dict(chunk_size=0), dict(chunk_size=257),
    dict(act_dtype=7), dict(x_stride_t=10), dict(B_stride_t=5), dict(impl=9), dict(p_block=48),
    dict(seg_chunks=-2), dict(workspace_bytes=256), dict(head_block=3), dict(head_block=-1),
])
def test_scan_rejects_bad_arguments(lib, bad):
    a = _scan_args(**bad)
    assert lib.ssd_chunk_scan(ctypes.byref(a), None) == 1
    assert lib.ssd_chunk_scan(None, None) == 1


W = ctypes.c_void_p(0x9000)


def _scan_norm(lib, a, z=0x20000, w=W, wt=None, gs=16, eps=1e-5, out=0x40000):
    wt = ssd.SSD_F32 if wt is None else wt
    return lib.ssd_chunk_scan_gated_norm(ctypes.byref(a), ctypes.c_void_p(z), w, wt, gs,
                                         ctypes.c_float(eps), ctypes.c_void_p(out), None)


@pytest.mark.parametrize("bad", [
    dict(gs=0), dict(gs=7), dict(eps=-1.0), dict(eps=float("nan")), dict(w=None), dict(wt=5),
    dict(out=0), dict(z=0x1000),                   # z overlaps y
    dict(z=0x40000 + 4 * 8 * 64 - 4),              # z overlaps out by one element
])
def test_scan_gated_norm_rejects_bad_arguments(lib, bad):
    """Checked before any launch: the norm's parameters, and a z sharing bytes with y or
    out (the norm may read z while the scan is still writing)."""
    a = _scan_args()
    kw = dict(bad)
    if kw.get("out") == 0:
        a.y = None                                  # no y and no out: nothing to write to
    assert _scan_norm(lib, a, **kw) == 1
    assert lib.ssd_chunk_scan_gated_norm(None, None, W, ssd.SSD_F32, 16, ctypes.c_float(0.),
                                         None, None) == 1
    bad_scan = _scan_args(H=3)
    assert _scan_norm(lib, bad_scan) == 1


def test_scan_workspace_size(lib):
    """Host-side planning only: no kernel runs.  A forced split of k chunks per segment
    wants room for the bound nseq + (T + 127 nseq) // (128 k) on the segment count, each
    segment holding one fp32 [H, P, N] state, plus one fp32 decay per token and head."""
    kw = dict(act_dtype=ssd.SSD_BF16, nseq=2, T=4096, H=24, P=64, G=1, N=128, chunk_size=256)
    size = lambda **o: lib.ssd_chunk_scan_workspace_size(ctypes.byref(_scan_args(**{**kw, **o})))
    r256 = lambda b: (b + 255) // 256 * 256
    nseg = 2 + (4096 + 127 * 2) // (128 * 4)
    assert size(seg_chunks=4) == r256(nseg * 24 * 64 * 128 * 4 + 4096 * 24 * 4)
    # at most 64 segments per sequence: 1-chunk segments of a 16384-token batch become 2
    nseg = 2 + (16384 + 127 * 2) // (128 * 2)
    assert size(seg_chunks=1, T=16384) == r256(nseg * 24 * 64 * 128 * 4 + 16384 * 24 * 4)
    assert size(seg_chunks=-1) == 0                       # never split
    assert size(seg_chunks=4, impl=1) == 0                # SIMT path: no workspace
    assert size(seg_chunks=4, act_dtype=ssd.SSD_F32) == 0  # not a tensor-core shape
    # one head per CTA, the planner cuts two 2048-token sequences into 6-chunk segments
    # (channel block 64: 2 x 3 x 24 = 144 CTAs, one wave), keeps a Nemotron-H-shaped
    # batch whole, and splits one sequence of 16384 tokens
    assert size(head_block=1) == r256((2 + (4096 + 127 * 2) // (128 * 6)) * 24 * 64 * 128 * 4
                                      + 4096 * 24 * 4)
    assert size(nseq=4, T=16384, H=128, G=8, head_block=1) == 0
    auto = size(nseq=1, T=16384)
    assert auto > 0 and auto % 256 == 0
    # with head pairs allowed, the planner cuts the two 2048-token sequences into 3-chunk
    # segments of two heads per CTA (13 segments at most: 156 CTAs), keeps the
    # Nemotron-H-shaped varlen batch and single 16K-token Nemotron-H sequences whole (one
    # head per CTA there: 128 chains fill the GPU), and cuts a 64K-token one into 64-chunk
    # segments (9 at most) of two heads per CTA
    assert size() == r256(13 * 24 * 64 * 128 * 4 + 4096 * 24 * 4)
    assert size(nseq=4, T=16384, H=128, G=8) == 0
    assert size(nseq=1, T=16384, H=128, G=8) == 0
    assert size(nseq=1, T=65536, H=128, G=8) == r256(9 * 128 * 64 * 128 * 4 + 65536 * 128 * 4)
    assert lib.ssd_chunk_scan_workspace_size(None) == 0


def test_scan_gated_norm_workspace_size(lib):
    """Host-side planning only: no kernel runs.  The overlapped scan + norm (the
    tensor-core scan in 64-channel blocks, unsplit or split with two heads per CTA, bf16,
    groups of whole 64-channel head blocks, 16-byte aligned rows, at most two waves of
    CTAs) wants its ready counters: one int per chunk id (ceil(T/128) +
    nseq of them) and norm group, plus four ints, rounded up to 256 bytes (norm groups the vector norm takes: 8 x 32 x v channels, v
    <= 4, and multiples).  A two-head split within two waves comes first in the
    workspace; another split the planner would choose takes the workspace instead;
    anything the overlapped form cannot take (or fewer than 3072 tokens) wants none."""
    lib.ssd_chunk_scan_gated_norm_workspace_size.argtypes = [
        ctypes.POINTER(ssd.ScanArgs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p]
    lib.ssd_chunk_scan_gated_norm_workspace_size.restype = ctypes.c_size_t
    kw = dict(act_dtype=ssd.SSD_BF16, nseq=4, T=16384, H=128, P=64, G=8, N=128, chunk_size=128)
    r256 = lambda b: (b + 255) // 256 * 256
    queue = lambda T, nseq, ngroups: r256(((T + 127) // 128 + nseq) * ngroups * 4 + 16)

    def size(gs=1024, z=0x200000, w=0x300000, out=0x400000, y=0x100000, **o):
        a = _scan_args(**{**kw, **o})
        a.y = y
        return lib.ssd_chunk_scan_gated_norm_workspace_size(
            ctypes.byref(a), ctypes.c_void_p(z), ctypes.c_void_p(w), gs, ctypes.c_void_p(out))

    # the Nemotron-H-shaped varlen prefill: 256 pair CTAs, norm groups of 16 heads
    assert size() == queue(16384, 4, 8)
    assert size(head_block=2) == queue(16384, 4, 8)
    assert size(gs=256) == queue(16384, 4, 32)
    assert size(z=0) == queue(16384, 4, 8)              # no gate
    assert size(y=0) == queue(16384, 4, 8)              # y written into out
    assert size(gs=8192, H=128) == queue(16384, 4, 1)
    # anything else runs the norm after the scan and wants no queue
    assert size(gs=128) == 0                             # no vector norm for 16 vectors
    assert size(gs=96 * 8) == 0                          # group of 12.5 64-channel blocks
    assert size(z=0x200008) == 0                         # z rows not 16-byte aligned
    assert size(head_block=1) == 0                       # one head per CTA: 512 CTAs
    # a single 16K-token sequence: one head (128 CTAs) or two (64) per CTA both qualify
    # unsplit; told it may split, the two-head plan splits into two segments (192 CTAs
    # with the segment bound), which the overlapped form takes too: the split's workspace,
    # then the counters
    assert size(nseq=1, head_block=1) == queue(16384, 1, 8)
    assert size(nseq=1) == queue(16384, 1, 8)          # the planner's plan: one head
    assert size(nseq=1, head_block=2, seg_chunks=-1) == queue(16384, 1, 8)
    one = dict(kw, nseq=1, head_block=2)
    split1 = lib.ssd_chunk_scan_workspace_size(ctypes.byref(_scan_args(**one)))
    assert split1 > 0 and size(nseq=1, head_block=2) == split1 + queue(16384, 1, 8)
    assert size(nseq=1, head_block=1, p_block=32) == 0   # 32-channel blocks
    assert size(impl=1) == 0                             # SIMT scan
    assert size(act_dtype=ssd.SSD_F32) == 0              # fp32: no tensor-core scan
    assert size(nseq=8, T=32768) == 0                    # 512 CTAs: more than two waves
    assert size(T=0) == 0
    assert size(nseq=1, T=3071) == 0                     # short: the norm follows the scan
    assert size(nseq=1, T=3072) == queue(3072, 1, 8)
    assert size(gs=0) == 0 and size(gs=1000) == 0        # invalid group sizes
    # a split the planner is told to make takes the workspace (the norm then follows)
    split = lib.ssd_chunk_scan_workspace_size(ctypes.byref(_scan_args(**kw, seg_chunks=4)))
    assert split > 0 and size(seg_chunks=4) == split
    assert lib.ssd_chunk_scan_gated_norm_workspace_size(None, None, None, 1024, None) == 0


def test_update_rejects_bad_arguments(lib):
    a = ssd.UpdateArgs()
    a.struct_size = ctypes.sizeof(ssd.UpdateArgs)
    assert lib.ssd_state_update(ctypes.byref(a), None) == 1          # NULL pool
    a.state_pool = a.A = a.state_indices = a.x = a.dt = a.B = a.C = a.y = 0x1000
    a.num_slots, a.batch, a.H, a.P, a.G, a.N = 4, 2, 4, 16, 3, 16    # H % G != 0
    assert lib.ssd_state_update(ctypes.byref(a), None) == 1
    a.G = 2
    a.slot_stride = 5                                                 # smaller than a slot
    assert lib.ssd_state_update(ctypes.byref(a), None) == 1
    a.slot_stride, a.batch = 0, 70000                                 # beyond the grid limit
    assert lib.ssd_state_update(ctypes.byref(a), None) == 2


def test_norm_rejects_bad_arguments(lib):
    p = 0x1000
    assert lib.gated_rmsnorm(p, p, p, p, 4, 64, 48, 1e-5, 1, 1, None) == 1   # 64 % 48
    assert lib.gated_rmsnorm(p, p, None, p, 4, 64, 64, 1e-5, 1, 1, None) == 1
    assert lib.gated_rmsnorm(p, p, p, p, 4, 64, 64, -1.0, 1, 1, None) == 1
    assert lib.gated_rmsnorm(p, p, p, p, 4, 64, 64, 1e-5, 3, 1, None) == 1
    assert lib.ssd_read_status(None, 1, None, None) == 1


def test_decode_ops_reject_bad_arguments(lib):
    """Host-side validation of the decode-side entry points (nothing is launched)."""
    a = ssd.UpdateArgs()
    a.struct_size = ctypes.sizeof(ssd.UpdateArgs)
    a.state_pool = a.A = a.state_indices = a.x = a.dt = a.B = a.C = a.y = 0x1000
    a.num_slots, a.batch, a.H, a.P, a.G, a.N = 4, 2, 4, 16, 2, 16
    p = 0x1000
    assert lib.ssd_state_update_multi(ctypes.byref(a), 0, None, None) == 1        # ntok 0
    a.N = 48
    assert lib.ssd_state_update_multi(ctypes.byref(a), 2, None, None) == 2        # N 48
    a.N = 16
    # B or C not on a four-element boundary (8 bytes in bf16, 16 in fp32): refused
    # before anything is launched, since the kernel reads them four values at a time
    a.act_dtype = ssd.SSD_BF16
    for field, off in (("B", 2), ("C", 4), ("B", 6)):
        setattr(a, field, 0x1000 + off)
        assert lib.ssd_state_update_multi(ctypes.byref(a), 2, None, None) == 2
        setattr(a, field, 0x1000)
    a.act_dtype = ssd.SSD_F32
    a.C = 0x1008                                                                  # 8 of 16
    assert lib.ssd_state_update_multi(ctypes.byref(a), 2, None, None) == 2
    a.C = 0x1000
    for gs in (24, 8, 48):   # not a multiple of P, below P, not dividing H*P
        assert lib.ssd_decode_layer_step(ctypes.byref(a), p, p, 0, gs, 1e-5, p, None) == 1
    assert lib.ssd_decode_layer_step(ctypes.byref(a), p, None, 0, 32, 1e-5, p, None) == 1
    assert lib.ssd_decode_layer_step(ctypes.byref(a), p, p, 0, 32, -1.0, p, None) == 1
    # slot copy: sizes, alignment, grid limit
    assert lib.ssd_state_copy(p, 0, 2, p, p, 0, 2, p, -1, 64, None, None) == 1
    assert lib.ssd_state_copy(p, 0, 2, p, p, 0, 2, p, 0, 64, None, None) == 0     # nothing
    assert lib.ssd_state_copy(p, 32, 2, p, p, 0, 2, p, 1, 64, None, None) == 1    # stride
    assert lib.ssd_state_copy(p, 0, 2, p, p, 0, 2, p, 1, 6, None, None) == 2      # 6 % 4
    assert lib.ssd_state_copy(p + 4, 0, 2, p, p, 0, 2, p, 1, 64, None, None) == 2  # align
    assert lib.ssd_state_copy(p, 0, 2, p, p, 0, 2, p, 70000, 64, None, None) == 2


def test_status_strings_and_version(lib):
    assert lib.ssd_status_string(0) == b"SSD_OK"
    assert lib.ssd_status_string(3) == b"SSD_ERR_A_NOT_NEGATIVE"
    assert lib.ssd_version() >= 100


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(ssd, "_lib", None)
    with pytest.raises(RuntimeError):
        ssd.load_library(str(tmp_path / "nope.so"))
