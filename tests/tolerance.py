"""Comparison bars for the GPU path against the double-precision oracle.

fp32 paths use the bar of the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)" (section
"Evidence" and the #675 message): rtol(K) = 4 (K + 2) 2^-24 for an output produced by a
length-K recurrence / summation, applied here relative to the sum of the magnitudes of
every term that produced the output (the classical summation-error scale), plus the
smallest normal fp32 number.  Against an exact reference only the device's own
rounding counts (<= 2 ulp per expf, (K - 1) u summation).

bf16-input paths use relative L2 <= 1e-2 and max-abs <= 5e-2 per tensor.

Every comparison prints the fraction of its bar used, so a bar that stopped doing work
would show.
"""
import numpy as np

U = 2.0 ** -24
TINY = 2.0 ** -126


def rtol_K(K):
    return 4.0 * (np.asarray(K, dtype=np.float64) + 2.0) * U


def check_fp32(name, got, ref, scale, K):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bar = rtol_K(K) * np.asarray(scale, dtype=np.float64) + TINY
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    frac = float(np.max(err / bar)) if err.size else 0.0
    print(f"[bar] {name}: fp32 worst element used {100 * frac:.3f}% of rtol(K)")
    assert frac <= 1.0, f"{name}: error exceeds rtol(K) by {frac:.3f}x"
    return frac


def bf16_half_ulp(v):
    """Half the spacing of bf16 values at |v| (8 significand bits): the largest error
    rounding an exact value to bf16 can make.  0 at 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8.0), 0.0)


def norm_carried_rounding(y_ref, z, w, group_size, eps, dy=None):
    """Per-element bound (first order) on how far an error dy in y before the gated norm
    can move the norm's output.  With g = y silu(z) and r = (mean_group g^2 + eps)^-1/2,
    out_j = g_j r w_j, so a change dy moves out_j by silu(z_j) w_j r dy_j + out_j dr/r,
    and |dr/r| <= mean_group(|g| |silu(z)| |dy|) / (mean_group g^2 + eps).  By default
    |dy| is half a bf16 ulp of y (y stored in bf16), taken at 1.01 |y| so that a device
    value just above a power of two is covered.  z None = no gate."""
    y = np.asarray(y_ref, dtype=np.float64)
    rows, d = y.shape
    s = np.ones_like(y) if z is None else np.asarray(z, np.float64) / (
        1.0 + np.exp(-np.asarray(z, np.float64)))
    w = np.asarray(w, dtype=np.float64).reshape(1, d)
    dy = bf16_half_ulp(1.01 * np.abs(y)) if dy is None else np.abs(
        np.asarray(dy, dtype=np.float64)).reshape(rows, d)
    grp = lambda a: a.reshape(rows, d // group_size, group_size)  # noqa: E731
    g = grp(y * s)
    den = np.mean(g * g, axis=-1, keepdims=True) + eps
    r = 1.0 / np.sqrt(den)
    rel_r = np.mean(np.abs(g) * grp(np.abs(s) * dy), axis=-1, keepdims=True) / den
    out = g * r * grp(np.broadcast_to(w, y.shape))
    return (grp(np.abs(s * w) * dy) * r + np.abs(out) * rel_r).reshape(rows, d)


def check_bf16(name, got, ref, rel_l2_max=1e-2, max_abs_max=5e-2, stored_bf16=False,
               carried=None):
    """The bf16 bar: rel-L2 and max-abs against the double oracle.  With stored_bf16 the
    compared values were rounded to bf16 on output, and the max-abs bar is applied to the
    error beyond that rounding (half a bf16 ulp of the reference): above |v| = 16 the
    rounding alone can exceed 5e-2.  carried: a per-element allowance for bf16 roundings
    of stored intermediates carried to this output (norm_carried_rounding), taken off
    the error the same way."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if ref.size == 0:
        return 0.0, 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    err = np.abs(got - ref)
    if stored_bf16:
        err = np.maximum(err - bf16_half_ulp(ref), 0.0)
    if carried is not None:
        err = np.maximum(err - np.asarray(carried, dtype=np.float64).reshape(err.shape), 0.0)
    mx = float(np.max(err))
    print(f"[bar] {name}: rel-L2 {rel:.3e} ({100 * rel / rel_l2_max:.1f}% of bar), "
          f"max-abs {mx:.3e} ({100 * mx / max_abs_max:.1f}% of bar)")
    assert rel <= rel_l2_max, f"{name}: rel-L2 {rel:.3e} > {rel_l2_max}"
    assert mx <= max_abs_max, f"{name}: max-abs {mx:.3e} > {max_abs_max}"
    return rel, mx


def scan_K(cu_seqlens, H, P, N, has_init):
    """K of every y[t,h,p] (tokens since the sequence start, + 1 with an initial state,
    + N) and of every final state entry (sequence length + 1)."""
    cu = np.asarray(cu_seqlens)
    T = int(cu[-1])
    Ky = np.zeros((T, 1, 1))
    nseq = len(cu) - 1
    Kf = np.zeros((nseq, 1, 1, 1))
    for s in range(nseq):
        a, b = int(cu[s]), int(cu[s + 1])
        init = 1 if (has_init is not None and has_init[s]) else 0
        Ky[a:b, 0, 0] = np.arange(1, b - a + 1) + init + N
        Kf[s] = (b - a) + 1
    return Ky, Kf
