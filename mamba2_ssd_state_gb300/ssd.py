"""Thin Python binding of libssd.so (C ABI in include/ssd.h).

Argument marshalling only: each function checks the torch tensors it is given (device,
dtype, shape, contiguity), fills the C argument struct with their device pointers and
the current CUDA stream, and calls the library.  Every step of the ops runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and a missing library
raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ssd.h")

SSD_F32, SSD_BF16 = 0, 1
IMPL = {"auto": 0, "simt": 1, "tc": 2}
DEV_A_NOT_NEG, DEV_INDEX_OOR, DEV_SEQ_META, DEV_TIMEOUT = 1, 2, 4, 8
STATUS_NAMES = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
                3: "SSD_ERR_A_NOT_NEGATIVE", 4: "SSD_ERR_INDEX", 5: "SSD_ERR_SEQ_META",
                6: "SSD_ERR_CUDA", 7: "SSD_ERR_TIMEOUT"}


class SsdError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


_vp, _i32, _i64, _u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32


class ScanArgs(ctypes.Structure):
    _fields_ = [("struct_size", _u32), ("x", _vp), ("x_stride_t", _i64), ("dt", _vp),
                ("dt_bias", _vp), ("dt_softplus", _i32), ("A", _vp), ("D", _vp), ("B", _vp),
                ("B_stride_t", _i64), ("C", _vp), ("C_stride_t", _i64),
                ("initial_states", _vp), ("has_initial_state", _vp), ("cu_seqlens", _vp),
                ("nseq", _i32), ("T", _i32), ("H", _i32), ("P", _i32), ("G", _i32),
                ("N", _i32), ("chunk_size", _i32), ("act_dtype", ctypes.c_int), ("y", _vp),
                ("final_states", _vp), ("d_status", _vp), ("impl", _i32), ("p_block", _i32),
                ("seg_chunks", _i32), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
                ("head_block", _i32)]


class UpdateArgs(ctypes.Structure):
    _fields_ = [("struct_size", _u32), ("state_pool", _vp), ("slot_stride", _i64),
                ("num_slots", _i32), ("state_indices", _vp), ("batch", _i32), ("x", _vp),
                ("dt", _vp), ("dt_bias", _vp), ("dt_softplus", _i32), ("A", _vp), ("B", _vp),
                ("C", _vp), ("D", _vp), ("y", _vp), ("H", _i32), ("P", _i32), ("G", _i32),
                ("N", _i32), ("act_dtype", ctypes.c_int), ("d_status", _vp)]


_lib = None


def load_library(path: str | None = None):
    """Load libssd.so once.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "mamba2_ssd_state_gb300.build.build() (needs nvcc)")
        lib = ctypes.CDLL(path)
        lib.ssd_chunk_scan.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.ssd_chunk_scan_workspace_size.argtypes = [ctypes.POINTER(ScanArgs)]
        lib.ssd_chunk_scan_workspace_size.restype = ctypes.c_size_t
        lib.ssd_chunk_scan_static_ws.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.ssd_chunk_scan_static_ws.restype = ctypes.c_int
        lib.ssd_chunk_scan_gated_norm.argtypes = [ctypes.POINTER(ScanArgs), _vp, _vp,
                                                  ctypes.c_int, _i32, ctypes.c_float, _vp, _vp]
        lib.ssd_chunk_scan_gated_norm.restype = ctypes.c_int
        lib.ssd_chunk_scan_gated_norm_workspace_size.argtypes = [ctypes.POINTER(ScanArgs), _vp,
                                                                 _vp, _i32, _vp]
        lib.ssd_chunk_scan_gated_norm_workspace_size.restype = ctypes.c_size_t
        lib.ssd_state_update_multi.argtypes = [ctypes.POINTER(UpdateArgs), _i32, _vp, _vp]
        lib.ssd_state_update_multi.restype = ctypes.c_int
        lib.ssd_decode_layer_step.argtypes = [ctypes.POINTER(UpdateArgs), _vp, _vp, ctypes.c_int,
                                              _i32, ctypes.c_float, _vp, _vp]
        lib.ssd_decode_layer_step.restype = ctypes.c_int
        lib.ssd_state_copy.argtypes = [_vp, _i64, _i32, _vp, _vp, _i64, _i32, _vp, _i32, _i64,
                                       _vp, _vp]
        lib.ssd_state_copy.restype = ctypes.c_int
        lib.ssd_state_update.argtypes = [ctypes.POINTER(UpdateArgs), _vp]
        lib.gated_rmsnorm.argtypes = [_vp, _vp, _vp, _vp, _i64, _i32, _i32, ctypes.c_float,
                                      ctypes.c_int, ctypes.c_int, _vp]
        lib.ssd_read_status.argtypes = [_vp, _i32, ctypes.POINTER(_u32), _vp]
        lib.ssd_status_string.argtypes = [ctypes.c_int]
        lib.ssd_status_string.restype = ctypes.c_char_p
        for f in (lib.ssd_chunk_scan, lib.ssd_state_update, lib.gated_rmsnorm,
                  lib.ssd_read_status, lib.ssd_version):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def header_functions(header: str = HEADER):
    """Names of the entry points that include/ssd.h declares."""
    txt = open(header).read()
    return sorted(set(re.findall(r"SSD_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)))


# ----------------------------------------------------------------------------- helpers

def _act(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise TypeError(f"activations must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t, name, dtype=None, shape=None, dev=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _token_stride(t, name, inner):
    """Token (first-dim) stride in elements; the inner dims must be dense."""
    if t.dim() < 2:
        raise ValueError(f"{name} must be at least 2-D")
    if t.numel() == 0:
        return int(inner)  # no element is addressed: any strides will do
    exp = 1
    for d in range(t.dim() - 1, 0, -1):
        if t.stride(d) != exp:
            raise ValueError(f"{name} must be dense in its trailing dims")
        exp *= t.shape[d]
    return int(t.stride(0)) if t.shape[0] > 1 else int(inner)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _raise(rc, where):
    if rc != 0:
        raise SsdError(rc, where)


# ----------------------------------------------------------------------------- ops

def chunk_scan(x, dt, A, B, C, *, cu_seqlens, chunk_size, D=None, dt_bias=None,
               dt_softplus=True, initial_states=None, has_initial_state=None, y=None,
               final_states=None, return_final_states=True, status=None, impl="auto",
               p_block=0, seg_chunks=0, workspace=None, stream=None, head_block=0):
    """Mamba2 chunked SSD scan over packed sequences (see ssd_chunk_scan in ssd.h).

    x [T,H,P], B/C [T,G,N] (bf16 or fp32, token stride may exceed the dense size);
    dt [T,H], A/D/dt_bias [H], initial_states [nseq,H,P,N] fp32; cu_seqlens int32
    [nseq+1] on the device.  seg_chunks: 0 = the library decides whether to split long
    sequences (it then gets a workspace from torch's allocator unless one is passed),
    -1 = never, k >= 1 = segments of k 128-token chunks.  head_block: heads per CTA of the
    tensor-core path (0 = the library decides, 1, or 2).  Returns (y, final_states)."""
    lib = load_library()
    a, y, final_states, _ws = _scan_args(
        lib, x, dt, A, B, C, cu_seqlens, chunk_size, D, dt_bias, dt_softplus, initial_states,
        has_initial_state, y, final_states, return_final_states, status, impl, p_block,
        seg_chunks, workspace, head_block)
    _raise(lib.ssd_chunk_scan(ctypes.byref(a), _stream(stream)), "ssd_chunk_scan")
    return y, final_states


def chunk_scan_gated_norm(x, dt, A, B, C, z, norm_weight, *, cu_seqlens, chunk_size,
                          group_size, eps=1e-5, D=None, dt_bias=None, dt_softplus=True,
                          initial_states=None, has_initial_state=None, y=None, out=None,
                          final_states=None, return_final_states=True, status=None,
                          impl="auto", p_block=0, seg_chunks=0, workspace=None, stream=None,
                          head_block=0):
    """The scan of chunk_scan followed by the gated RMSNorm of gated_rmsnorm over its
    output, in one call (ssd_chunk_scan_gated_norm in ssd.h).  z [T,H*P] (or None: no
    gate), norm_weight [H*P].  y (optional) receives the pre-norm output; without it the
    scan writes into out.  Returns (out [T,H*P], final_states)."""
    lib = load_library()
    T, H, P = x.shape
    dev = x.device
    _check(z, "z", x.dtype, (T, H * P), dev)
    _check(norm_weight, "norm_weight", None, (H * P,), dev)
    for t, nm in ((z, "z"), (norm_weight, "norm_weight")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if out is None:
        out = torch.empty((T, H * P), dtype=x.dtype, device=dev)
    _check(out, "out", x.dtype, (T, H * P), dev)
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    a, y, final_states, _ws = _scan_args(
        lib, x, dt, A, B, C, cu_seqlens, chunk_size, D, dt_bias, dt_softplus, initial_states,
        has_initial_state, y if y is not None else out.view(T, H, P), final_states,
        return_final_states, status, impl, p_block, seg_chunks, workspace, head_block,
        alloc_ws=False)
    if workspace is None:
        # the split of the scan, or the ready counters of the overlapped form
        nbytes = lib.ssd_chunk_scan_gated_norm_workspace_size(
            ctypes.byref(a), _ptr(z), _ptr(norm_weight), int(group_size), _ptr(out))
        if nbytes:
            _ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            a.workspace, a.workspace_bytes = _ptr(_ws), _ws.numel()
    _raise(lib.ssd_chunk_scan_gated_norm(ctypes.byref(a), _ptr(z), _ptr(norm_weight),
                                         _act(norm_weight), int(group_size), float(eps),
                                         _ptr(out), _stream(stream)),
           "ssd_chunk_scan_gated_norm")
    return out, final_states


def _scan_args(lib, x, dt, A, B, C, cu_seqlens, chunk_size, D, dt_bias, dt_softplus,
               initial_states, has_initial_state, y, final_states, return_final_states, status,
               impl, p_block, seg_chunks, workspace, head_block=0, alloc_ws=True):
    """ssd_scan_args for one scan call, with the outputs (and a workspace from torch's
    allocator, when the plan wants one and none was passed) made where missing."""
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    nseq = cu_seqlens.shape[0] - 1
    dev = x.device
    act = _act(x)
    _check(dt, "dt", torch.float32, (T, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(D, "D", torch.float32, (H,), dev)
    _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (T, G, N), dev)
    _check(C, "C", x.dtype, (T, G, N), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (nseq + 1,), dev)
    _check(initial_states, "initial_states", torch.float32, (nseq, H, P, N), dev)
    _check(has_initial_state, "has_initial_state", torch.uint8, (nseq,), dev)
    for t, nm in ((dt, "dt"), (A, "A"), (D, "D"), (dt_bias, "dt_bias"),
                  (cu_seqlens, "cu_seqlens"), (initial_states, "initial_states"),
                  (has_initial_state, "has_initial_state")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if y is None:
        y = torch.empty((T, H, P), dtype=x.dtype, device=dev)
    _check(y, "y", x.dtype, (T, H, P), dev)
    if not y.is_contiguous():
        raise ValueError("y must be contiguous")
    if final_states is None and return_final_states:
        final_states = torch.empty((nseq, H, P, N), dtype=torch.float32, device=dev)
    _check(final_states, "final_states", torch.float32, (nseq, H, P, N), dev)
    _check(status, "status", None, (1,), dev)
    a = ScanArgs()
    a.struct_size = ctypes.sizeof(ScanArgs)
    a.x, a.x_stride_t = _ptr(x), _token_stride(x, "x", H * P)
    a.dt, a.dt_bias, a.dt_softplus = _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus))
    a.A, a.D = _ptr(A), _ptr(D)
    a.B, a.B_stride_t = _ptr(B), _token_stride(B, "B", G * N)
    a.C, a.C_stride_t = _ptr(C), _token_stride(C, "C", G * N)
    a.initial_states, a.has_initial_state = _ptr(initial_states), _ptr(has_initial_state)
    a.cu_seqlens = _ptr(cu_seqlens)
    a.nseq, a.T, a.H, a.P, a.G, a.N, a.chunk_size = nseq, T, H, P, G, N, int(chunk_size)
    a.act_dtype = act
    a.y, a.final_states, a.d_status = _ptr(y), _ptr(final_states), _ptr(status)
    a.impl, a.p_block = IMPL[impl], int(p_block)
    a.seg_chunks, a.head_block = int(seg_chunks), int(head_block)
    if workspace is None and a.seg_chunks >= 0 and alloc_ws:
        nbytes = lib.ssd_chunk_scan_workspace_size(ctypes.byref(a))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _check(workspace, "workspace", torch.uint8, None, dev)
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
    return a, y, final_states, workspace


def chunk_scan_workspace_size(x, B, C, *, cu_seqlens, chunk_size, impl="auto", p_block=0,
                              seg_chunks=0, head_block=0):
    """Bytes of workspace chunk_scan would want for these shapes (0 = it would not split;
    ssd_chunk_scan_workspace_size in ssd.h).  y is taken as a dense aligned tensor."""
    lib = load_library()
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    a = ScanArgs()
    a.struct_size = ctypes.sizeof(ScanArgs)
    a.x, a.x_stride_t = _ptr(x), _token_stride(x, "x", H * P)
    a.B, a.B_stride_t = _ptr(B), _token_stride(B, "B", G * N)
    a.C, a.C_stride_t = _ptr(C), _token_stride(C, "C", G * N)
    a.dt = a.A = a.y = a.x
    a.cu_seqlens = _ptr(cu_seqlens)
    a.nseq, a.T, a.H, a.P, a.G, a.N = cu_seqlens.shape[0] - 1, T, H, P, G, N
    a.chunk_size, a.act_dtype = int(chunk_size), _act(x)
    a.impl, a.p_block, a.seg_chunks = IMPL[impl], int(p_block), int(seg_chunks)
    a.head_block = int(head_block)
    return int(lib.ssd_chunk_scan_workspace_size(ctypes.byref(a)))


def chunk_scan_gated_norm_workspace_size(x, B, C, z, norm_weight, out, *, cu_seqlens,
                                         chunk_size, group_size, y=None, impl="auto",
                                         p_block=0, seg_chunks=0, head_block=0):
    """Bytes of workspace chunk_scan_gated_norm wants for these tensors
    (ssd_chunk_scan_gated_norm_workspace_size in ssd.h): the split of the scan when its
    planner splits, else the ready counters of the overlapped form, else 0."""
    lib = load_library()
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    a = ScanArgs()
    a.struct_size = ctypes.sizeof(ScanArgs)
    a.x, a.x_stride_t = _ptr(x), _token_stride(x, "x", H * P)
    a.B, a.B_stride_t = _ptr(B), _token_stride(B, "B", G * N)
    a.C, a.C_stride_t = _ptr(C), _token_stride(C, "C", G * N)
    a.dt = a.A = a.x
    a.y = _ptr(y)
    a.cu_seqlens = _ptr(cu_seqlens)
    a.nseq, a.T, a.H, a.P, a.G, a.N = cu_seqlens.shape[0] - 1, T, H, P, G, N
    a.chunk_size, a.act_dtype = int(chunk_size), _act(x)
    a.impl, a.p_block, a.seg_chunks = IMPL[impl], int(p_block), int(seg_chunks)
    a.head_block = int(head_block)
    return int(lib.ssd_chunk_scan_gated_norm_workspace_size(
        ctypes.byref(a), _ptr(z), _ptr(norm_weight), int(group_size), _ptr(out)))


def _update_args(state_pool, state_indices, x, dt, A, B, C, D, dt_bias, dt_softplus, y,
                 status, tok_shape):
    """ssd_update_args for one decode call; tok_shape is () or (ntok,): the token axes
    between the request axis and the per-token dimensions of x, dt, B, C and y."""
    num_slots, H, P, N = state_pool.shape
    batch = state_indices.shape[0]
    G = B.shape[-2]
    dev = x.device
    bt = (batch, *tok_shape)
    _check(state_pool, "state_pool", torch.float32, None, dev)
    _check(state_indices, "state_indices", torch.int32, (batch,), dev)
    _check(x, "x", None, (*bt, H, P), dev)
    _check(dt, "dt", torch.float32, (*bt, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(D, "D", torch.float32, (H,), dev)
    _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (*bt, G, N), dev)
    _check(C, "C", x.dtype, (*bt, G, N), dev)
    _check(y, "y", x.dtype, (*bt, H, P), dev)
    for t, nm in ((x, "x"), (dt, "dt"), (B, "B"), (C, "C"), (state_indices, "state_indices"),
                  (y, "y")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if any(state_pool.stride(d) != s for d, s in ((3, 1), (2, N), (1, P * N))):
        raise ValueError("state_pool slots must be dense [H,P,N]")
    a = UpdateArgs()
    a.struct_size = ctypes.sizeof(UpdateArgs)
    a.state_pool, a.slot_stride, a.num_slots = _ptr(state_pool), int(state_pool.stride(0)), num_slots
    a.state_indices, a.batch = _ptr(state_indices), batch
    a.x, a.dt, a.dt_bias, a.dt_softplus = _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus))
    a.A, a.B, a.C, a.D, a.y = _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y)
    a.H, a.P, a.G, a.N = H, P, G, N
    a.act_dtype = _act(x)
    a.d_status = _ptr(status)
    return a


def state_update_multi(state_pool, state_indices, x, dt, A, B, C, *, D=None, dt_bias=None,
                       dt_softplus=True, y=None, inter_states=None, status=None, stream=None):
    """ntok decode tokens per request in one pass (ssd_state_update_multi in ssd.h).

    x [batch,ntok,H,P]; dt [batch,ntok,H]; B/C [batch,ntok,G,N].  inter_states: None, True
    (allocate) or an fp32 [batch,ntok,H,P,N] tensor receiving the state after each token.
    Returns (y [batch,ntok,H,P], inter_states)."""
    lib = load_library()
    batch, ntok, H, P = x.shape
    if y is None:
        y = torch.empty_like(x)
    if inter_states is True:
        inter_states = torch.empty((batch, ntok, H, P, state_pool.shape[3]), dtype=torch.float32,
                                   device=x.device)
    if inter_states is not None:
        _check(inter_states, "inter_states", torch.float32,
               (batch, ntok, H, P, state_pool.shape[3]), x.device)
        if not inter_states.is_contiguous():
            raise ValueError("inter_states must be contiguous")
    a = _update_args(state_pool, state_indices, x, dt, A, B, C, D, dt_bias, dt_softplus, y, status,
                     (ntok,))
    _raise(lib.ssd_state_update_multi(ctypes.byref(a), ntok, _ptr(inter_states), _stream(stream)),
           "ssd_state_update_multi")
    return y, inter_states


def decode_layer_step(state_pool, state_indices, x, dt, A, B, C, z, norm_weight, *, group_size,
                      eps=1e-5, D=None, dt_bias=None, dt_softplus=True, y=None, out=None,
                      status=None, stream=None):
    """State update + D skip + gated RMSNorm of one decode token, fused
    (ssd_decode_layer_step in ssd.h).  z [batch,H*P]; norm_weight [H*P].  y (optional)
    receives the pre-norm output.  Returns out [batch,H*P]."""
    lib = load_library()
    batch, H, P = x.shape
    dev = x.device
    _check(z, "z", x.dtype, (batch, H * P), dev)
    _check(norm_weight, "norm_weight", None, (H * P,), dev)
    for t, nm in ((z, "z"), (norm_weight, "norm_weight")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if out is None:
        out = torch.empty((batch, H * P), dtype=x.dtype, device=dev)
    _check(out, "out", x.dtype, (batch, H * P), dev)
    a = _update_args(state_pool, state_indices, x, dt, A, B, C, D, dt_bias, dt_softplus, y, status,
                     ())
    _raise(lib.ssd_decode_layer_step(ctypes.byref(a), _ptr(z), _ptr(norm_weight),
                                     _act(norm_weight), int(group_size), float(eps), _ptr(out),
                                     _stream(stream)), "ssd_decode_layer_step")
    return out


def state_copy(src_pool, src_idx, dst_pool, dst_idx, *, status=None, stream=None):
    """dst_pool[dst_idx[i]] = src_pool[src_idx[i]] for every pair without a -1
    (ssd_state_copy in ssd.h).  Pools fp32 [slots, ...] with dense slots."""
    lib = load_library()
    n = src_idx.shape[0]
    dev = src_pool.device
    _check(src_pool, "src_pool", torch.float32, None, dev)
    _check(dst_pool, "dst_pool", torch.float32, None, dev)
    _check(src_idx, "src_idx", torch.int32, (n,), dev)
    _check(dst_idx, "dst_idx", torch.int32, (n,), dev)
    slot = src_pool[0].numel()
    if dst_pool[0].numel() != slot:
        raise ValueError("source and destination slots differ in size")
    for t, nm in ((src_pool, "src_pool"), (dst_pool, "dst_pool")):
        if not t[0].is_contiguous():
            raise ValueError(f"{nm} slots must be dense")
    _raise(lib.ssd_state_copy(_ptr(src_pool), int(src_pool.stride(0)), src_pool.shape[0],
                              _ptr(src_idx), _ptr(dst_pool), int(dst_pool.stride(0)),
                              dst_pool.shape[0], _ptr(dst_idx), n, slot, _ptr(status),
                              _stream(stream)), "ssd_state_copy")
    return dst_pool


def state_update(state_pool, state_indices, x, dt, A, B, C, *, D=None, dt_bias=None,
                 dt_softplus=True, y=None, status=None, stream=None):
    """One decode token per request on the pooled state cache (ssd_state_update in ssd.h).

    state_pool [num_slots,H,P,N] fp32 (updated in place); state_indices int32 [batch]
    (-1 = padding row); x [batch,H,P]; dt [batch,H]; B/C [batch,G,N].  Returns y."""
    lib = load_library()
    num_slots, H, P, N = state_pool.shape
    batch = state_indices.shape[0]
    G = B.shape[1]
    dev = x.device
    _check(state_pool, "state_pool", torch.float32, None, dev)
    _check(state_indices, "state_indices", torch.int32, (batch,), dev)
    _check(x, "x", None, (batch, H, P), dev)
    _check(dt, "dt", torch.float32, (batch, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(D, "D", torch.float32, (H,), dev)
    _check(dt_bias, "dt_bias", torch.float32, (H,), dev)
    _check(B, "B", x.dtype, (batch, G, N), dev)
    _check(C, "C", x.dtype, (batch, G, N), dev)
    for t, nm in ((x, "x"), (dt, "dt"), (B, "B"), (C, "C"), (state_indices, "state_indices")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if any(state_pool.stride(d) != s for d, s in ((3, 1), (2, N), (1, P * N))):
        raise ValueError("state_pool slots must be dense [H,P,N]")
    if y is None:
        y = torch.empty((batch, H, P), dtype=x.dtype, device=dev)
    a = UpdateArgs()
    a.struct_size = ctypes.sizeof(UpdateArgs)
    a.state_pool, a.slot_stride, a.num_slots = _ptr(state_pool), int(state_pool.stride(0)), num_slots
    a.state_indices, a.batch = _ptr(state_indices), batch
    a.x, a.dt, a.dt_bias, a.dt_softplus = _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus))
    a.A, a.B, a.C, a.D, a.y = _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y)
    a.H, a.P, a.G, a.N = H, P, G, N
    a.act_dtype = _act(x)
    a.d_status = _ptr(status)
    _raise(lib.ssd_state_update(ctypes.byref(a), _stream(stream)), "ssd_state_update")
    return y


def gated_rmsnorm(x, z, weight, *, group_size, eps=1e-5, out=None, stream=None):
    """out = (x * silu(z)) / sqrt(mean_group((x * silu(z))^2) + eps) * weight."""
    lib = load_library()
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    dev = x.device
    _check(z, "z", x.dtype, tuple(x.shape), dev)
    _check(weight, "weight", None, (d,), dev)
    for t, nm in ((x, "x"), (z, "z"), (weight, "weight")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    if out is None:
        out = torch.empty_like(x)
    _raise(lib.gated_rmsnorm(_ptr(x), _ptr(z), _ptr(weight), _ptr(out), rows, d, int(group_size),
                             float(eps), _act(x), _act(weight), _stream(stream)), "gated_rmsnorm")
    return out


def read_status(status, clear=True, stream=None):
    """Synchronise, read (and optionally clear) the device status word: (code, bits)."""
    lib = load_library()
    bits = _u32(0)
    rc = lib.ssd_read_status(_ptr(status), int(bool(clear)), ctypes.byref(bits), _stream(stream))
    return rc, int(bits.value)


def new_status(device=None):
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")
