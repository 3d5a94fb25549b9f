"""Pins for the CPU oracle: each checks it against something other than itself.

Every pin here is independent of the oracle's code: a brute-force quadratic form
evaluated in numpy with each decay recomputed from scratch, a closed form, an
invariance that exact arithmetic guarantees, or a library routine (torch's rms_norm,
silu).  The mutation tests (test_oracle_mutants.py) plant each of the pages' nine
mutations into the oracle and require this file to fail on every one of them.
"""
import math

import numpy as np
import pytest

from mamba2_ssd_state_gb300 import inputs as I


def _softplus(v):
    return np.logaddexp(0.0, v)  # library form of log(1 + e^v)


def _scan(oracle, s, chunked=None, with_abs=False, init=True, D=True):
    kw = dict(D=s.D.values if D else None, dt_bias=s.dt_bias.values,
              initial_states=s.initial_states.values if (init and s.initial_states) else None,
              has_initial_state=s.has_initial_state if init else None, cu_seqlens=s.cu_seqlens)
    if chunked:
        return oracle.scan_chunked(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                                   chunk_size=chunked, **kw)
    return oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                           with_abs=with_abs, **kw)


def _bruteforce(s):
    """Quadratic (attention-like) form of the SSD layer, every decay from scratch:
    y_t = sum_{u<=t} (C_t.B_u) exp(A sum_{r=u+1..t} dt_r) dt_u x_u
          + exp(A sum_{r=start..t} dt_r) C_t.h0 + D x_t."""
    x = s.x.values.astype(np.float64)
    B = s.B.values.astype(np.float64)
    C = s.C.values.astype(np.float64)
    A = s.A.values.astype(np.float64)
    Dv = s.D.values.astype(np.float64)
    dt = _softplus(s.dt.values.astype(np.float64) + s.dt_bias.values.astype(np.float64)[None, :])
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.zeros((T, H, P))
    fin = np.zeros((len(s.seqlens), H, P, N))
    for si in range(len(s.seqlens)):
        a0, a1 = int(s.cu_seqlens[si]), int(s.cu_seqlens[si + 1])
        for h in range(H):
            g = h // (H // G)
            h0 = np.zeros((P, N))
            if s.initial_states is not None and s.has_initial_state[si]:
                h0 = s.initial_states.values[si, h].astype(np.float64)
            for t in range(a0, a1):
                acc = np.zeros(P)
                for u in range(a0, t + 1):
                    decay = math.exp(A[h] * sum(dt[r, h] for r in range(u + 1, t + 1)))
                    acc += float(C[t, g] @ B[u, g]) * decay * dt[u, h] * x[u, h]
                dec0 = math.exp(A[h] * sum(dt[r, h] for r in range(a0, t + 1)))
                acc += dec0 * (h0 @ C[t, g])
                y[t, h] = acc + Dv[h] * x[t, h]
            f = math.exp(A[h] * sum(dt[r, h] for r in range(a0, a1))) * h0
            for u in range(a0, a1):
                decay = math.exp(A[h] * sum(dt[r, h] for r in range(u + 1, a1)))
                f = f + decay * dt[u, h] * np.outer(x[u, h], B[u, g])
            fin[si, h] = f
    return y, fin


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------------------------------
# scan: brute force, closed form, invariances
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("G", [1, 2])
def test_scan_seq_matches_bruteforce(oracle_mod, G):
    s = I.make_scan_inputs([17, 1, 9], H=4, P=3, G=G, N=5, chunk_size=4, act="f32",
                           seed=7, init=[1, 0, 1])
    y, fin = _scan(oracle_mod, s)
    yb, fb = _bruteforce(s)
    assert _rel(y, yb) < 1e-12
    assert _rel(fin, fb) < 1e-12


def test_scan_scalar_closed_form(oracle_mod):
    """H=P=N=G=1 with constant dt, A, B, C, x:
    h_t = a^(t+1) h0 + b (1 - a^(t+1)) / (1 - a), a = e^(dt A), b = dt B x;
    y_t = C h_t + D x.  dt enters through softplus(0 + log(expm1(dt)))."""
    L, dtv, Av, Bv, Cv, xv, Dv, h0 = 100, 0.05, -1.5, 0.7, -1.3, 0.9, 0.37, 2.5
    bias = math.log(math.expm1(dtv))
    y, fin = oracle_mod.scan_seq(np.full((L, 1, 1), xv), np.zeros((L, 1)), np.array([Av]),
                                 np.full((L, 1, 1), Bv), np.full((L, 1, 1), Cv), D=np.array([Dv]),
                                 dt_bias=np.array([bias]), initial_states=np.full((1, 1, 1, 1), h0))
    a = math.exp(dtv * Av)
    b = dtv * Bv * xv
    t = np.arange(L)
    h = a ** (t + 1) * h0 + b * (1 - a ** (t + 1)) / (1 - a)
    np.testing.assert_allclose(y[:, 0, 0], Cv * h + Dv * xv, rtol=1e-13)
    np.testing.assert_allclose(fin[0, 0, 0, 0], h[-1], rtol=1e-13)


def test_softplus_inverse_bias(oracle_mod):
    """softplus(0 + log(expm1(u))) = u: with dt_raw = 0 the step equals the drawn u,
    so one token from a zero state gives y = C dt B x + D x exactly."""
    for u in (1e-3, 0.02, 0.1, 3.0):
        y, _ = oracle_mod.scan_seq(np.ones((1, 1, 1)), np.zeros((1, 1)), np.array([-2.0]),
                                   np.ones((1, 1, 1)), np.ones((1, 1, 1)), D=np.array([0.0]),
                                   dt_bias=np.array([math.log(math.expm1(u))]))
        assert abs(y[0, 0, 0] - u) < 1e-15 * max(1.0, u) * 8


def test_softplus_off_uses_plain_sum(oracle_mod):
    y, _ = oracle_mod.scan_seq(np.ones((1, 1, 1)), np.full((1, 1), 0.25), np.array([-2.0]),
                               np.ones((1, 1, 1)), np.ones((1, 1, 1)), dt_bias=np.array([0.5]),
                               dt_softplus=False)
    assert y[0, 0, 0] == pytest.approx(0.75, rel=1e-15)


@pytest.mark.parametrize("Q", [1, 2, 3, 4, 16, 64, 1000])
def test_chunk_size_invariance(oracle_mod, Q):
    s = I.make_scan_inputs([70, 5, 33], H=4, P=4, G=2, N=6, chunk_size=Q, act="f32", seed=11,
                           init=[1, 1, 0])
    y, fin = _scan(oracle_mod, s)
    yc, fc = _scan(oracle_mod, s, chunked=Q)
    assert _rel(yc, y) < 1e-12
    assert _rel(fc, fin) < 1e-12


def test_split_sequence_equivalence(oracle_mod):
    """Scanning [0, L1) and feeding its final state as the initial state of [L1, L)
    equals one scan over [0, L) (the initial_states path carries the whole context)."""
    s = I.make_scan_inputs([64], H=3, P=4, G=1, N=5, chunk_size=8, act="f32", seed=13,
                           init="all")
    y, fin = _scan(oracle_mod, s)
    L1 = 23
    kw = dict(D=s.D.values, dt_bias=s.dt_bias.values)
    ya, fa = oracle_mod.scan_seq(s.x.values[:L1], s.dt.values[:L1], s.A.values,
                                 s.B.values[:L1], s.C.values[:L1],
                                 initial_states=s.initial_states.values, **kw)
    yb, fb = oracle_mod.scan_seq(s.x.values[L1:], s.dt.values[L1:], s.A.values,
                                 s.B.values[L1:], s.C.values[L1:], initial_states=fa, **kw)
    assert _rel(np.concatenate([ya, yb]), y) < 1e-12
    assert _rel(fb, fin) < 1e-12
    # and the chunked form with a chunk boundary that does not divide L1
    yc, fc = _scan(oracle_mod, s, chunked=8)
    assert _rel(yc, y) < 1e-12


def test_split_sequence_chunked(oracle_mod):
    s = I.make_scan_inputs([48], H=2, P=3, G=1, N=4, chunk_size=8, act="f32", seed=17,
                           init="all")
    kw = dict(D=s.D.values, dt_bias=s.dt_bias.values, chunk_size=8)
    y, fin = oracle_mod.scan_chunked(s.x.values, s.dt.values, s.A.values, s.B.values,
                                     s.C.values, initial_states=s.initial_states.values, **kw)
    L1 = 19
    ya, fa = oracle_mod.scan_chunked(s.x.values[:L1], s.dt.values[:L1], s.A.values,
                                     s.B.values[:L1], s.C.values[:L1],
                                     initial_states=s.initial_states.values, **kw)
    yb, fb = oracle_mod.scan_chunked(s.x.values[L1:], s.dt.values[L1:], s.A.values,
                                     s.B.values[L1:], s.C.values[L1:], initial_states=fa, **kw)
    assert _rel(np.concatenate([ya, yb]), y) < 1e-12
    assert _rel(fb, fin) < 1e-12


def test_abs_scale_bounds_output(oracle_mod):
    s = I.make_scan_inputs([30, 12], H=2, P=3, G=1, N=4, chunk_size=4, act="f32", seed=19,
                           init=[1, 0])
    y, fin, ya, fa = _scan(oracle_mod, s, with_abs=True)
    assert np.all(ya >= np.abs(y) * (1 - 1e-12))
    assert np.all(fa >= np.abs(fin) * (1 - 1e-12))


def test_empty_sequence_in_pack(oracle_mod):
    s = I.make_scan_inputs([5, 0, 4], H=2, P=2, G=1, N=3, chunk_size=2, act="f32", seed=23,
                           init=[1, 1, 1])
    y, fin = _scan(oracle_mod, s)
    # an empty sequence's final state is its initial state
    np.testing.assert_array_equal(fin[1], s.initial_states.values[1].astype(np.float64))
    yb, fb = _bruteforce(s)
    assert _rel(y, yb) < 1e-12


# ----------------------------------------------------------------------------------
# decode: continuity with prefill, pool bookkeeping, the A sign check
# ----------------------------------------------------------------------------------

def _prefill_then_decode(oracle_mod, s, slot, num_slots):
    """Run the prefill on tokens [0, L-1), put its final state in pool[slot], and decode
    token L-1 with state_indices = [slot]."""
    L = s.T
    kw = dict(D=s.D.values, dt_bias=s.dt_bias.values)
    ya, fa = oracle_mod.scan_seq(s.x.values[:L - 1], s.dt.values[:L - 1], s.A.values,
                                 s.B.values[:L - 1], s.C.values[:L - 1],
                                 initial_states=s.initial_states.values, **kw)
    H, P, N = s.H, s.P, s.N
    pool = np.random.default_rng(5).standard_normal((num_slots, H, P, N))
    pool[slot] = fa[0]
    newpool, yd, st = oracle_mod.state_update(pool, [slot], s.x.values[L - 1:], s.dt.values[L - 1:],
                                              s.A.values, s.B.values[L - 1:], s.C.values[L - 1:],
                                              **kw)
    return pool, newpool, yd, st


def test_decode_continues_prefill(oracle_mod):
    s = I.make_scan_inputs([21], H=4, P=3, G=2, N=5, chunk_size=4, act="f32", seed=29, init="all")
    y, fin = _scan(oracle_mod, s)
    pool, newpool, yd, st = _prefill_then_decode(oracle_mod, s, slot=2, num_slots=4)
    assert st == 0
    assert _rel(yd[0], y[-1]) < 1e-12
    assert _rel(newpool[2], fin[0]) < 1e-12
    for k in (0, 1, 3):
        np.testing.assert_array_equal(newpool[k], pool[k])


def test_decode_indices_and_null_rows(oracle_mod):
    """-1 rows touch no slot and give y = 0; the changed slots are exactly the active
    indices; each active row's result is one recurrence step on its own slot."""
    H, P, G, N, S = 4, 3, 2, 5, 6
    idx = np.array([3, -1, 0, 5, -1], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=31)
    newpool, y, st = oracle_mod.state_update(u.pool.values, idx, u.x.values, u.dt.values,
                                             u.A.values, u.B.values, u.C.values, D=u.D.values,
                                             dt_bias=u.dt_bias.values)
    assert st == 0
    pool = u.pool.values.astype(np.float64)
    changed = {k for k in range(S) if not np.array_equal(newpool[k], pool[k])}
    assert changed == {3, 0, 5}
    for b in (1, 4):
        assert np.all(y[b] == 0.0)
    # each active row equals a one-token scan from that slot's state
    for b, slot in enumerate(idx):
        if slot < 0:
            continue
        yb, fb = oracle_mod.scan_seq(u.x.values[b:b + 1], u.dt.values[b:b + 1], u.A.values,
                                     u.B.values[b:b + 1], u.C.values[b:b + 1], D=u.D.values,
                                     dt_bias=u.dt_bias.values,
                                     initial_states=pool[slot][None])
        assert _rel(y[b], yb[0]) < 1e-13
        assert _rel(newpool[slot], fb[0]) < 1e-13


def test_decode_out_of_range_index(oracle_mod):
    H, P, G, N, S = 2, 2, 1, 3, 3
    idx = np.array([1, 3, -2], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=37)
    newpool, y, st = oracle_mod.state_update(u.pool.values, idx, u.x.values, u.dt.values,
                                             u.A.values, u.B.values, u.C.values)
    assert st & 2
    pool = u.pool.values.astype(np.float64)
    np.testing.assert_array_equal(newpool[0], pool[0])
    np.testing.assert_array_equal(newpool[2], pool[2])
    assert not np.array_equal(newpool[1], pool[1])
    assert np.all(y[1] == 0) and np.all(y[2] == 0)


@pytest.mark.parametrize("bad", [0.0, -0.0, 1.0, float("nan")])
def test_decode_rejects_nonnegative_A(oracle_mod, bad):
    H, P, G, N, S = 3, 2, 1, 4, 2
    idx = np.array([1], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=41)
    A = u.A.values.astype(np.float64).copy()
    A[1] = bad
    newpool, y, st = oracle_mod.state_update(u.pool.values, idx, u.x.values, u.dt.values, A,
                                             u.B.values, u.C.values)
    assert st & 1
    pool = u.pool.values.astype(np.float64)
    np.testing.assert_array_equal(newpool[1, 1], pool[1, 1])   # the bad head's state is kept
    assert np.all(y[0, 1] == 0.0)
    assert not np.array_equal(newpool[1, 0], pool[1, 0])        # other heads still update


def test_decode_accepts_tiny_negative_A(oracle_mod):
    """The check is a sign test, not a magnitude floor: A = -1e-30 is accepted."""
    H, P, G, N, S = 1, 2, 1, 3, 1
    u = I.make_update_inputs(S, [0], H, P, G, N, act="f32", seed=43)
    newpool, y, st = oracle_mod.state_update(u.pool.values, [0], u.x.values, u.dt.values,
                                             np.array([-1e-30]), u.B.values, u.C.values)
    assert st == 0
    assert not np.array_equal(newpool[0], u.pool.values.astype(np.float64)[0])


# ----------------------------------------------------------------------------------
# gated RMSNorm
# ----------------------------------------------------------------------------------

def test_norm_matches_torch_rms_norm(oracle_mod):
    """Per-group gated norm equals torch's rms_norm over each group of x * silu(z)."""
    torch = pytest.importorskip("torch")
    rows, d, gs = 7, 48, 16
    n = I.make_norm_inputs(rows, d, gs, act="f32", seed=47)
    out = oracle_mod.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=gs,
                                   eps=1e-5)
    x = torch.tensor(n.x.values, dtype=torch.float64)
    z = torch.tensor(n.z.values, dtype=torch.float64)
    g = x * torch.nn.functional.silu(z)
    ref = torch.nn.functional.rms_norm(g.view(rows, d // gs, gs), (gs,), None, 1e-5)
    ref = ref.view(rows, d) * torch.tensor(n.weight.values, dtype=torch.float64)
    assert _rel(out, ref.numpy()) < 1e-13


def test_norm_constant_closed_form(oracle_mod):
    """x = c, z = z0 everywhere: out = w g / sqrt(g^2 + eps), g = c z0 / (1 + e^-z0)."""
    c, z0, eps = 0.8, 2.0, 1e-5
    d, gs = 32, 8
    w = np.linspace(0.5, 1.5, d)
    out = oracle_mod.gated_rmsnorm(np.full((2, d), c), np.full((2, d), z0), w, group_size=gs,
                                   eps=eps)
    g = c * z0 / (1 + math.exp(-z0))
    np.testing.assert_allclose(out, np.broadcast_to(w * g / math.sqrt(g * g + eps), (2, d)),
                               rtol=1e-14)


def test_norm_group_scale_invariance(oracle_mod):
    """Scaling one group's input by 10 leaves every other group's output unchanged and
    that group's output nearly unchanged (only through eps)."""
    rows, d, gs = 3, 64, 16
    n = I.make_norm_inputs(rows, d, gs, act="f32", seed=53)
    out = oracle_mod.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=gs)
    x2 = n.x.values.astype(np.float64).copy()
    x2[:, 16:32] *= 10.0
    out2 = oracle_mod.gated_rmsnorm(x2, n.z.values, n.weight.values, group_size=gs)
    np.testing.assert_array_equal(out2[:, :16], out[:, :16])
    np.testing.assert_array_equal(out2[:, 32:], out[:, 32:])
    np.testing.assert_allclose(out2[:, 16:32], out[:, 16:32], rtol=1e-3)


def test_norm_without_gate(oracle_mod):
    torch = pytest.importorskip("torch")
    rows, d = 4, 24
    n = I.make_norm_inputs(rows, d, d, act="f32", seed=59)
    out = oracle_mod.gated_rmsnorm(n.x.values, None, n.weight.values, group_size=d, eps=1e-6)
    ref = torch.nn.functional.rms_norm(torch.tensor(n.x.values, dtype=torch.float64), (d,),
                                       torch.tensor(n.weight.values, dtype=torch.float64), 1e-6)
    assert _rel(out, ref.numpy()) < 1e-13


# ------------------------------------------------------------- decode-side compositions

def test_multi_token_decode_equals_scan_from_the_slot(oracle_mod):
    """k decode tokens on a slot are the k-token scan started from that slot's state: the
    per-token update (applied k times) and the sequence scan are separate code paths of
    the oracle.  Every intermediate state is the final state of the scan's prefix."""
    H, P, G, N, S, k = 4, 3, 2, 5, 5, 6
    idx = np.array([4, -1, 1], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=61, ntok=k)
    pool0 = u.pool.values.astype(np.float64)
    newpool, y, inter, st = oracle_mod.state_update_multi(
        pool0, idx, u.x.values, u.dt.values, u.A.values, u.B.values, u.C.values, D=u.D.values,
        dt_bias=u.dt_bias.values)
    assert st == 0
    assert np.all(y[1] == 0.0) and np.all(np.isnan(inter[1]))
    for b, slot in ((0, 4), (2, 1)):
        ys, fs = oracle_mod.scan_seq(u.x.values[b], u.dt.values[b], u.A.values, u.B.values[b],
                                     u.C.values[b], D=u.D.values, dt_bias=u.dt_bias.values,
                                     initial_states=pool0[slot][None])
        assert _rel(y[b], ys) < 1e-12
        assert _rel(newpool[slot], fs[0]) < 1e-12
        for t in range(k):
            _, ft = oracle_mod.scan_seq(u.x.values[b, :t + 1], u.dt.values[b, :t + 1],
                                        u.A.values, u.B.values[b, :t + 1], u.C.values[b, :t + 1],
                                        D=u.D.values, dt_bias=u.dt_bias.values,
                                        initial_states=pool0[slot][None])
            assert _rel(inter[b, t], ft[0]) < 1e-12
    for slot in (0, 2, 3):
        np.testing.assert_array_equal(newpool[slot], pool0[slot])


def test_state_copy_invariants(oracle_mod):
    """Copy and copy back restores the pool; -1 on either side skips; an out-of-range
    index raises bit 2 and skips only its pair; slots not named stay identical."""
    rng = np.random.default_rng(67)
    src = rng.standard_normal((5, 2, 3, 4))
    dst = rng.standard_normal((4, 2, 3, 4))
    new, st = oracle_mod.state_copy(src, [3, -1, 0, 1], dst, [0, 2, -1, 3])
    assert st == 0
    np.testing.assert_array_equal(new[0], src[3])
    np.testing.assert_array_equal(new[3], src[1])
    for d in (1, 2):
        np.testing.assert_array_equal(new[d], dst[d])
    back, st = oracle_mod.state_copy(dst, [0, 3], new, [0, 3])
    np.testing.assert_array_equal(back, dst)
    new2, st = oracle_mod.state_copy(src, [5, 2], dst, [1, 1])
    assert st == 2
    np.testing.assert_array_equal(new2[1], src[2])
    new3, st = oracle_mod.state_copy(src, [0], dst, [-2])
    assert st == 2
    np.testing.assert_array_equal(new3, dst)


def test_decode_layer_output_has_unit_group_rms(oracle_mod):
    """The fused decode step's output divided by the norm weight has, per row and norm
    group, mean square mean(g^2) / (mean(g^2) + eps): 1 up to eps.  -1 rows give 0."""
    H, P, G, N, S, gs = 4, 8, 2, 6, 5, 16
    idx = np.array([2, -1, 0], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=71)
    n = I.make_norm_inputs(3, H * P, gs, act="f32", seed=73)
    eps = 1e-5
    pool, y, out, st = oracle_mod.decode_layer_step(
        u.pool.values, idx, u.x.values, u.dt.values, u.A.values, u.B.values, u.C.values,
        n.z.values, n.weight.values, group_size=gs, eps=eps, D=u.D.values,
        dt_bias=u.dt_bias.values)
    assert st == 0
    g = (y.reshape(3, H * P) * n.z.values / (1 + np.exp(-n.z.values.astype(np.float64))))
    r = out / n.weight.values.astype(np.float64)
    for b in (0, 2):
        for k in range(H * P // gs):
            sl = slice(k * gs, (k + 1) * gs)
            ms = np.mean(g[b, sl] ** 2)
            assert abs(np.mean(r[b, sl] ** 2) - ms / (ms + eps)) < 1e-12
    assert np.all(out[1] == 0.0)


def test_bf16_half_ulp_matches_rounding():
    """The bf16 half-ulp the tests allow on bf16-stored outputs is the largest error of
    rounding to bf16 (checked against torch's round-to-nearest-even conversion)."""
    torch = pytest.importorskip("torch")
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from tolerance import bf16_half_ulp
    v = (np.random.default_rng(79).standard_normal(20000) * np.exp2(
        np.random.default_rng(80).integers(-10, 10, 20000))).astype(np.float32)
    r = torch.tensor(v).to(torch.bfloat16).double().numpy()     # fp32 -> bf16, RNE
    v = v.astype(np.float64)
    assert np.all(np.abs(r - v) <= bf16_half_ulp(v))
    assert np.max(np.abs(r - v) / bf16_half_ulp(v)) > 0.99   # and it is tight
    assert bf16_half_ulp(16.3) == 2.0 ** -4


@pytest.mark.parametrize("gs", [1536, 128, 64])
def test_norm_carried_rounding_bounds_rounding_y(oracle_mod, gs):
    """The allowance the scan + norm test gives for y stored in bf16 between the two ops
    bounds what that rounding alone does to the norm's output (the oracle's norm of the
    exact y against its norm of y rounded to bf16), and stays small: its median is a
    small fraction of the 5e-2 max-abs bar."""
    torch = pytest.importorskip("torch")
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from tolerance import norm_carried_rounding
    rng = np.random.default_rng(97 + gs)
    rows, d = 48, 1536
    # heavy-tailed y (|y| up to about 40) and wide z, the hard case for the bound
    y = rng.standard_normal((rows, d)) * 3.0 * np.exp(0.7 * rng.standard_normal((rows, d)))
    bf = lambda a: torch.tensor(a.astype(np.float32)).to(torch.bfloat16).double().numpy()  # noqa
    z = bf(1.5 * rng.standard_normal((rows, d)))
    w = bf(1.0 + 0.1 * rng.standard_normal(d))
    exact = oracle_mod.gated_rmsnorm(y, z, w, group_size=gs, eps=1e-5)
    rounded = oracle_mod.gated_rmsnorm(bf(y), z, w, group_size=gs, eps=1e-5)
    allow = norm_carried_rounding(y, z, w, gs, 1e-5)
    diff = np.abs(exact - rounded)
    assert np.all(diff <= allow)
    assert np.max(diff / allow) > 0.3          # the bound is not loose by orders
    assert np.median(allow) < 2e-3

