"""Seeded synthetic inputs for the SSD ops, shared by the tests and the benchmark.

This module only draws random numbers and rounds them to the storage type; it holds
none of the ops' arithmetic, and it imports neither the CUDA binding nor the oracle.
Draws use numpy's PCG64 generator (stable across library versions) in float32 and are
rounded to bfloat16 (round to nearest even) where a workload stores bfloat16, so every
consumer reads bit-identical values.

Distributions (Mamba2 / Nemotron-H style layers):
  x ~ N(0,1); dt_raw ~ N(0,1); dt_bias = log(expm1(U[1e-3, 0.1])) per head (so that
  softplus(dt_bias) is uniform on [1e-3, 0.1]); A = -exp(U[0, ln 16]) per head;
  B, C ~ N(0,1)/sqrt(N); D ~ N(0,1) per head; z ~ N(0,1); norm weight = 1 + 0.1 N(0,1);
  initial states ~ N(0, 0.1^2) (standard deviation 0.1) where present.
Seeds: the workload's base seed, plus a fixed offset per tensor.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------------
# bfloat16 storage helpers (bit manipulation only)
# ---------------------------------------------------------------------------------


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16, returned as float32."""
    return bf16_to_f32(bf16_bits(a))


@dataclass
class Tensor:
    """A host array plus the dtype it is stored in on the device ("f32" or "bf16").

    ``values`` is float32 holding exactly the stored values; ``bits`` is the uint16
    pattern for bf16 tensors."""
    values: np.ndarray
    dtype: str

    @property
    def bits(self) -> np.ndarray:
        assert self.dtype == "bf16"
        return bf16_bits(self.values)

    @property
    def shape(self):
        return self.values.shape


def _t(values: np.ndarray, dtype: str) -> Tensor:
    v = np.ascontiguousarray(values, dtype=np.float32)
    if dtype == "bf16":
        v = round_bf16(v)
    return Tensor(v, dtype)


# ---------------------------------------------------------------------------------
# Scan (prefill) inputs
# ---------------------------------------------------------------------------------


@dataclass
class ScanInputs:
    seqlens: list
    H: int
    P: int
    G: int
    N: int
    chunk_size: int
    act: str                       # "f32" or "bf16" for x, B, C (and y)
    x: Tensor = None
    dt: Tensor = None              # raw dt (before bias and softplus), f32 [T,H]
    dt_bias: Tensor = None         # f32 [H]
    A: Tensor = None               # f32 [H]
    B: Tensor = None
    C: Tensor = None
    D: Tensor = None               # f32 [H]
    initial_states: Tensor = None  # f32 [nseq,H,P,N] or None
    has_initial_state: np.ndarray = None  # uint8 [nseq] or None
    cu_seqlens: np.ndarray = field(default=None)

    @property
    def T(self):
        return int(sum(self.seqlens))

    @property
    def nseq(self):
        return len(self.seqlens)


def make_scan_inputs(seqlens, H, P, G, N, chunk_size, act="bf16", seed=1000,
                     init="none", dt_softplus_range=(1e-3, 0.1)) -> ScanInputs:
    """init: "none" (no initial states), "all" (every sequence), or a 0/1 list per sequence."""
    seqlens = [int(s) for s in seqlens]
    T = sum(seqlens)
    nseq = len(seqlens)
    rng = lambda k: np.random.default_rng(seed * 100 + k)  # noqa: E731
    inp = ScanInputs(seqlens, H, P, G, N, chunk_size, act)
    inp.x = _t(rng(1).standard_normal((T, H, P), dtype=np.float32), act)
    inp.dt = _t(rng(2).standard_normal((T, H), dtype=np.float32), "f32")
    lo, hi = dt_softplus_range
    u = rng(3).uniform(lo, hi, size=H)
    inp.dt_bias = _t(np.log(np.expm1(u)), "f32")
    inp.A = _t(-np.exp(rng(4).uniform(0.0, np.log(16.0), size=H)), "f32")
    inv = 1.0 / np.sqrt(N)
    inp.B = _t(rng(5).standard_normal((T, G, N), dtype=np.float32) * inv, act)
    inp.C = _t(rng(6).standard_normal((T, G, N), dtype=np.float32) * inv, act)
    inp.D = _t(rng(7).standard_normal(H, dtype=np.float32), "f32")
    if init == "none":
        inp.initial_states = None
        inp.has_initial_state = None
    else:
        mask = [1] * nseq if init == "all" else [int(v) for v in init]
        assert len(mask) == nseq
        st = rng(8).standard_normal((nseq, H, P, N), dtype=np.float32) * 0.1
        st[np.asarray(mask) == 0] = 0.0
        inp.initial_states = _t(st, "f32")
        inp.has_initial_state = np.asarray(mask, dtype=np.uint8)
    inp.cu_seqlens = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    return inp


# ---------------------------------------------------------------------------------
# Decode (state update) inputs
# ---------------------------------------------------------------------------------


@dataclass
class UpdateInputs:
    num_slots: int
    H: int
    P: int
    G: int
    N: int
    act: str
    pool: Tensor = None            # f32 [num_slots,H,P,N]
    state_indices: np.ndarray = None  # int32 [batch]
    x: Tensor = None
    dt: Tensor = None
    dt_bias: Tensor = None
    A: Tensor = None
    B: Tensor = None
    C: Tensor = None
    D: Tensor = None

    @property
    def batch(self):
        return int(self.state_indices.shape[0])


def padded_permutation(num_slots, batch, pad_frac=0.1, seed=3000):
    """The first `batch` entries of a seeded permutation of the slots, with
    round(pad_frac * batch) positions (chosen by a second permutation) set to -1."""
    r = np.random.default_rng(seed)
    idx = r.permutation(num_slots)[:batch].astype(np.int32)
    npad = int(round(pad_frac * batch))
    if npad:
        pos = np.random.default_rng(seed + 1).permutation(batch)[:npad]
        idx[pos] = -1
    return idx


def make_update_inputs(num_slots, state_indices, H, P, G, N, act="bf16", seed=3000,
                       pool_values=None, ntok=None) -> UpdateInputs:
    """Decode inputs for one token per request, or (ntok given) ntok tokens per request
    with a token axis after the request axis: x [batch, ntok, H, P] and so on."""
    idx = np.asarray(state_indices, dtype=np.int32)
    batch = idx.shape[0]
    bt = (batch,) if ntok is None else (batch, ntok)
    rng = lambda k: np.random.default_rng(seed * 100 + k)  # noqa: E731
    u = UpdateInputs(num_slots, H, P, G, N, act)
    if pool_values is None:
        pool_values = rng(9).standard_normal((num_slots, H, P, N), dtype=np.float32)
    u.pool = _t(pool_values, "f32")
    u.state_indices = idx
    u.x = _t(rng(1).standard_normal((*bt, H, P), dtype=np.float32), act)
    u.dt = _t(rng(2).standard_normal((*bt, H), dtype=np.float32), "f32")
    u.dt_bias = _t(np.log(np.expm1(rng(3).uniform(1e-3, 0.1, size=H))), "f32")
    u.A = _t(-np.exp(rng(4).uniform(0.0, np.log(16.0), size=H)), "f32")
    inv = 1.0 / np.sqrt(N)
    u.B = _t(rng(5).standard_normal((*bt, G, N), dtype=np.float32) * inv, act)
    u.C = _t(rng(6).standard_normal((*bt, G, N), dtype=np.float32) * inv, act)
    u.D = _t(rng(7).standard_normal(H, dtype=np.float32), "f32")
    return u


# ---------------------------------------------------------------------------------
# Gated norm inputs
# ---------------------------------------------------------------------------------


@dataclass
class NormInputs:
    rows: int
    d: int
    group_size: int
    eps: float
    act: str
    wdtype: str
    x: Tensor = None
    z: Tensor = None
    weight: Tensor = None


def make_norm_inputs(rows, d, group_size, act="bf16", wdtype=None, eps=1e-5, seed=4000,
                     x_values=None) -> NormInputs:
    wdtype = wdtype or act
    rng = lambda k: np.random.default_rng(seed * 100 + k)  # noqa: E731
    n = NormInputs(rows, d, group_size, eps, act, wdtype)
    if x_values is None:
        x_values = rng(1).standard_normal((rows, d), dtype=np.float32)
    n.x = _t(x_values, act)
    n.z = _t(rng(2).standard_normal((rows, d), dtype=np.float32), act)
    n.weight = _t(1.0 + 0.1 * rng(3).standard_normal(d, dtype=np.float32), wdtype)
    return n


# ---------------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------------

# Nemotron-H-shaped layer: H=128, P=64, G=8, N=128 (d_inner 8192, 8 norm groups of 1024)
NEMOTRON_H = dict(H=128, P=64, G=8, N=128)

WORKLOADS = {
    # tiny fp32 layer: one sequence of 64 tokens
    "tiny_fp32": dict(seqlens=[64], H=4, P=16, G=1, N=16, chunk_size=16, act="f32",
                      init="none", norm_group=64, seed=1000),
    # Mamba2-130M-shaped layer: 2 sequences of 2048, one norm group over d_inner=1536
    "mamba2_130m": dict(seqlens=[2048, 2048], H=24, P=64, G=1, N=128, chunk_size=256,
                        act="bf16", init="all", norm_group=1536, seed=1001),
    # Nemotron-H-shaped varlen prefill: 4 packed sequences, initial states on 0 and 2
    "nemotron_h_varlen": dict(seqlens=[8192, 3000, 517, 4675], chunk_size=128, act="bf16",
                              init=[1, 0, 1, 0], norm_group=1024, seed=1002, **NEMOTRON_H),
}


def scan_workload(name, **override) -> ScanInputs:
    w = dict(WORKLOADS[name])
    w.update(override)
    return make_scan_inputs(w["seqlens"], w["H"], w["P"], w["G"], w["N"], w["chunk_size"],
                            act=w["act"], seed=w["seed"], init=w["init"])
