"""ctypes front end of the double-precision CPU oracle.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the product path (``mamba2_ssd_state_gb300``).
It shares no code with the CUDA library.

Every function takes numpy arrays in the library's layouts (see ``ssd_oracle.h``),
converts them to float64 (exact for the bf16/fp32 values the tests generate) and
returns float64 results.  ``SSD_ORACLE_LIB`` in the environment selects another build
of the same source (the mutation tests point it at a mutant build).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = os.environ.get("SSD_ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        up = ctypes.POINTER(ctypes.c_uint8)
        ci = ctypes.c_int
        lib.oracle_scan_seq.argtypes = [dp, dp, dp, ci, dp, dp, dp, dp, dp, up, ip, ci, ci, ci,
                                        ci, ci, ci, dp, dp, dp, dp]
        lib.oracle_scan_chunked.argtypes = [dp, dp, dp, ci, dp, dp, dp, dp, dp, up, ip, ci, ci,
                                            ci, ci, ci, ci, ci, dp, dp]
        lib.oracle_state_update.argtypes = [dp, ci, ip, ci, dp, dp, dp, ci, dp, dp, dp, dp, ci,
                                            ci, ci, ci, dp, ip]
        lib.oracle_gated_rmsnorm.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ci, ci,
                                             ctypes.c_double]
        for f in (lib.oracle_scan_seq, lib.oracle_scan_chunked, lib.oracle_state_update,
                  lib.oracle_gated_rmsnorm):
            f.restype = ci
        _lib = lib
    return _lib


def _d(a):
    """float64 C-contiguous copy (None stays None)."""
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _seq_inputs(x, dt, dt_bias, A, B, C, D, initial_states, has_initial_state, cu_seqlens):
    x, dt, dt_bias, A, B, C, D, init = map(_d, (x, dt, dt_bias, A, B, C, D, initial_states))
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    hi = None
    if has_initial_state is not None:
        hi = np.ascontiguousarray(np.asarray(has_initial_state, dtype=np.uint8))
    return x, dt, dt_bias, A, B, C, D, init, hi, cu, T, H, P, G, N


def scan_seq(x, dt, A, B, C, *, D=None, dt_bias=None, dt_softplus=True, initial_states=None,
             has_initial_state=None, cu_seqlens=None, with_abs=False):
    """Sequential recurrence in double.  Returns (y, final_states[, y_abs, final_abs])."""
    if cu_seqlens is None:
        cu_seqlens = [0, np.asarray(x).shape[0]]
    (x, dt, dt_bias, A, B, C, D, init, hi, cu, T, H, P, G, N) = _seq_inputs(
        x, dt, dt_bias, A, B, C, D, initial_states, has_initial_state, cu_seqlens)
    nseq = cu.shape[0] - 1
    y = np.empty((T, H, P))
    fs = np.empty((nseq, H, P, N))
    ya = np.empty((T, H, P)) if with_abs else None
    fa = np.empty((nseq, H, P, N)) if with_abs else None
    rc = _load().oracle_scan_seq(_ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)),
                                 _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                 _ptr(hi, ctypes.c_uint8), _ptr(cu, ctypes.c_int32), nseq, T, H,
                                 P, G, N, _ptr(y), _ptr(fs), _ptr(ya), _ptr(fa))
    if rc != 0:
        raise ValueError(f"oracle_scan_seq rejected its arguments (rc={rc})")
    return (y, fs, ya, fa) if with_abs else (y, fs)


def scan_chunked(x, dt, A, B, C, *, chunk_size, D=None, dt_bias=None, dt_softplus=True,
                 initial_states=None, has_initial_state=None, cu_seqlens=None):
    """Chunked restatement in double.  Returns (y, final_states)."""
    if cu_seqlens is None:
        cu_seqlens = [0, np.asarray(x).shape[0]]
    (x, dt, dt_bias, A, B, C, D, init, hi, cu, T, H, P, G, N) = _seq_inputs(
        x, dt, dt_bias, A, B, C, D, initial_states, has_initial_state, cu_seqlens)
    nseq = cu.shape[0] - 1
    y = np.empty((T, H, P))
    fs = np.empty((nseq, H, P, N))
    rc = _load().oracle_scan_chunked(_ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)),
                                     _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                     _ptr(hi, ctypes.c_uint8), _ptr(cu, ctypes.c_int32), nseq, T,
                                     H, P, G, N, int(chunk_size), _ptr(y), _ptr(fs))
    if rc != 0:
        raise ValueError(f"oracle_scan_chunked rejected its arguments (rc={rc})")
    return y, fs


def state_update(pool, state_indices, x, dt, A, B, C, *, D=None, dt_bias=None, dt_softplus=True):
    """One decode step.  Returns (new_pool, y, status_bits); the input pool is not modified."""
    pool = np.array(pool, dtype=np.float64, order="C", copy=True)
    x, dt, dt_bias, A, B, C, D = map(_d, (x, dt, dt_bias, A, B, C, D))
    idx = np.ascontiguousarray(np.asarray(state_indices, dtype=np.int32))
    num_slots, H, P, N = pool.shape
    batch = idx.shape[0]
    G = B.shape[1]
    y = np.empty((batch, H, P))
    st = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_state_update(_ptr(pool), num_slots, _ptr(idx, ctypes.c_int32), batch,
                                     _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)),
                                     _ptr(A), _ptr(B), _ptr(C), _ptr(D), H, P, G, N, _ptr(y),
                                     _ptr(st, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_state_update rejected its arguments (rc={rc})")
    return pool, y, int(st[0])


def gated_rmsnorm(x, z, weight, *, group_size, eps=1e-5):
    """Gate-then-norm with per-group variance, in double.  Returns out [rows, d]."""
    x, z, w = _d(x), _d(z), _d(weight)
    rows, d = x.shape
    out = np.empty((rows, d))
    rc = _load().oracle_gated_rmsnorm(_ptr(x), _ptr(z), _ptr(w), _ptr(out), rows, d,
                                      int(group_size), float(eps))
    if rc != 0:
        raise ValueError(f"oracle_gated_rmsnorm rejected its arguments (rc={rc})")
    return out


# ----------------------------------------------------------------- compositions
# The decode-side ops below are defined by the single-token update and the gated norm
# above (each pinned in tests/test_oracle_pins.py); here they are those definitions
# applied in order, with nothing fused or reordered.

def state_update_multi(pool, state_indices, x, dt, A, B, C, *, D=None, dt_bias=None,
                       dt_softplus=True):
    """ntok decode tokens per request: the single-token update applied token by token.
    x [batch, ntok, H, P] etc.  Returns (new_pool, y [batch, ntok, H, P], inter
    [batch, ntok, H, P, N] (state after each token, NaN where the row is skipped),
    status_bits)."""
    x, dt, B, C = (np.asarray(v) for v in (x, dt, B, C))
    batch, ntok = x.shape[:2]
    pool = np.array(pool, dtype=np.float64, order="C", copy=True)
    num_slots, H, P, N = pool.shape
    idx = np.asarray(state_indices, dtype=np.int32)
    y = np.empty((batch, ntok, H, P))
    inter = np.full((batch, ntok, H, P, N), np.nan)
    st = 0
    for t in range(ntok):
        pool, y[:, t], s_t = state_update(pool, idx, x[:, t], dt[:, t], A, B[:, t], C[:, t], D=D,
                                          dt_bias=dt_bias, dt_softplus=dt_softplus)
        st |= s_t
        for b in range(batch):
            if 0 <= idx[b] < num_slots:
                inter[b, t] = pool[idx[b]]
    return pool, y, inter, st


def decode_layer_step(pool, state_indices, x, dt, A, B, C, z, norm_weight, *, group_size,
                      eps=1e-5, D=None, dt_bias=None, dt_softplus=True):
    """The single-token update, then the gated norm of its output.  Returns
    (new_pool, y [batch, H, P], out [batch, H*P], status_bits)."""
    pool, y, st = state_update(pool, state_indices, x, dt, A, B, C, D=D, dt_bias=dt_bias,
                               dt_softplus=dt_softplus)
    batch, H, P = y.shape
    out = gated_rmsnorm(y.reshape(batch, H * P), z, norm_weight, group_size=group_size, eps=eps)
    return pool, y, out, st


def scan_gated_norm(x, dt, A, B, C, z, norm_weight, *, group_size, eps=1e-5, D=None,
                    dt_bias=None, dt_softplus=True, initial_states=None, has_initial_state=None,
                    cu_seqlens=None):
    """The prefill half of the layer in its order (scan with D skip, then the gated norm
    of the scan's output).  Returns (y [T, H, P], final_states, out [T, H*P])."""
    y, fs = scan_seq(x, dt, A, B, C, D=D, dt_bias=dt_bias, dt_softplus=dt_softplus,
                     initial_states=initial_states, has_initial_state=has_initial_state,
                     cu_seqlens=cu_seqlens)
    T, H, P = y.shape
    out = gated_rmsnorm(y.reshape(T, H * P), z, norm_weight, group_size=group_size, eps=eps)
    return y, fs, out


def state_copy(src_pool, src_idx, dst_pool, dst_idx):
    """Slot copy: for each pair with both indices >= 0, the destination slot becomes the
    source slot; a pair with an index outside [-1, slots) is skipped and raises the
    out-of-range bit (2).  Returns (new_dst, status_bits)."""
    src = np.asarray(src_pool)
    dst = np.array(dst_pool, copy=True)
    st = 0
    for s, d in zip(np.asarray(src_idx).tolist(), np.asarray(dst_idx).tolist()):
        if s < -1 or s >= src.shape[0] or d < -1 or d >= dst.shape[0]:
            st |= 2
            continue
        if s >= 0 and d >= 0:
            dst[d] = src[s]
    return dst, st
