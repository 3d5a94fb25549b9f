"""GPU parity of ssd_state_update (decode over the pooled state cache) against the oracle,
with bit-exact pool bookkeeping: slots not named by an active row stay bit-identical,
-1 rows touch nothing, and the set of changed slots is the set of active indices."""
import numpy as np
import pytest
import torch

import oracle
from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev, scan_gpu, scan_oracle
from tolerance import check_bf16, check_fp32

pytestmark = pytest.mark.gpu


def _update_gpu(u, pool, A=None):
    status = ssd.new_status()
    idx = torch.from_numpy(u.state_indices).cuda()
    y = ssd.state_update(pool, idx, dev(u.x), dev(u.dt), A if A is not None else dev(u.A),
                         dev(u.B), dev(u.C), D=dev(u.D), dt_bias=dev(u.dt_bias), status=status)
    rc, bits = ssd.read_status(status)
    return y, bits


def test_tiny_fp32_decode_after_prefill():
    """The 64-token fp32 layer is prefilled, its final state goes to slot 2 of a 4-slot
    pool (the other slots hold N(0,1) values), and the layer's next 8 tokens are decoded
    one at a time with state_indices=[2].  Decode must continue the prefill exactly: the
    8 outputs and the slot equal a 72-token scan of the oracle (K = tokens so far + N)."""
    w = dict(I.WORKLOADS["tiny_fp32"])
    full = I.make_scan_inputs([72], w["H"], w["P"], w["G"], w["N"], w["chunk_size"],
                              act="f32", seed=w["seed"], init="none")
    pre = I.make_scan_inputs([64], w["H"], w["P"], w["G"], w["N"], w["chunk_size"],
                             act="f32", seed=w["seed"], init="none")
    for name in ("x", "dt", "B", "C"):
        setattr(pre, name, I.Tensor(getattr(full, name).values[:64], "f32"))
    _, fs, _ = scan_gpu(pre)
    H, P, N = full.H, full.P, full.N
    pool0 = np.random.default_rng(2024).standard_normal((4, H, P, N)).astype(np.float32)
    pool0[2] = fs[0]
    pool = torch.from_numpy(pool0).cuda()
    yr, fr, ya, fa = scan_oracle(full, with_abs=True)
    idx = torch.tensor([2], dtype=torch.int32, device="cuda")
    for k in range(8):
        t = 64 + k
        before = pool.clone()
        status = ssd.new_status()
        y = ssd.state_update(pool, idx, dev(full.x)[t:t + 1], dev(full.dt)[t:t + 1],
                             dev(full.A), dev(full.B)[t:t + 1], dev(full.C)[t:t + 1],
                             D=dev(full.D), dt_bias=dev(full.dt_bias), status=status)
        assert ssd.read_status(status)[1] == 0
        check_fp32(f"decode step {k} y", y.cpu().numpy()[0], yr[t], ya[t], t + 1 + N)
        for slot in (0, 1, 3):
            assert torch.equal(pool[slot], before[slot])
    check_fp32("decode after 8 steps, slot 2", pool[2].cpu().numpy(), fr[0], fa[0], 72 + 1)


@pytest.mark.parametrize("N", [128, 64, 48])
def test_bf16_padded_batch(N):
    H, P, G, S = 8, 64, 2, 24
    idx = I.padded_permutation(S, 12, seed=77)
    assert (idx == -1).sum() == 1
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=211)
    pool = dev(u.pool)
    before = pool.clone()
    y, bits = _update_gpu(u, pool)
    assert bits == 0
    ref_pool, yr, st = oracle.state_update(u.pool.values, idx, u.x.values, u.dt.values,
                                           u.A.values, u.B.values, u.C.values, D=u.D.values,
                                           dt_bias=u.dt_bias.values)
    check_bf16(f"update N={N} y", y.float().cpu().numpy(), yr)
    active = sorted(int(v) for v in idx if v >= 0)
    check_bf16(f"update N={N} slots", pool[active].cpu().numpy(), ref_pool[active])
    changed = {k for k in range(S) if not torch.equal(pool[k], before[k])}
    assert changed == set(active)
    assert torch.all(y[torch.from_numpy(idx == -1).cuda()] == 0)


def test_null_row_never_touches_slot_0():
    H, P, G, N, S = 4, 32, 1, 128, 3
    idx = np.array([-1, 1, -1], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=223)
    pool = dev(u.pool)
    before = pool.clone()
    y, bits = _update_gpu(u, pool)
    assert bits == 0
    assert torch.equal(pool[0], before[0]) and torch.equal(pool[2], before[2])
    assert not torch.equal(pool[1], before[1])
    assert torch.all(y[0] == 0) and torch.all(y[2] == 0)


@pytest.mark.parametrize("bad", [0.0, -0.0, 1.0, float("nan")])
def test_A_check_on_decode(bad):
    H, P, G, N, S = 4, 32, 1, 128, 2
    u = I.make_update_inputs(S, [1], H, P, G, N, act="bf16", seed=227)
    A = dev(u.A)
    A[2] = bad
    pool = dev(u.pool)
    before = pool.clone()
    y, bits = _update_gpu(u, pool, A=A)
    assert bits & ssd.DEV_A_NOT_NEG
    assert torch.equal(pool[1, 2], before[1, 2])
    assert torch.all(y[0, 2] == 0)
    assert not torch.equal(pool[1, 0], before[1, 0])


def test_A_tiny_negative_accepted():
    H, P, G, N, S = 2, 16, 1, 128, 1
    u = I.make_update_inputs(S, [0], H, P, G, N, act="bf16", seed=229)
    A = torch.full((H,), -1e-30, dtype=torch.float32, device="cuda")
    pool = dev(u.pool)
    before = pool.clone()
    y, bits = _update_gpu(u, pool, A=A)
    assert bits == 0
    assert not torch.equal(pool[0], before[0])


def test_out_of_range_index():
    H, P, G, N, S = 2, 16, 1, 128, 3
    idx = np.array([5, 0, -3], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=233)
    pool = dev(u.pool)
    before = pool.clone()
    y, bits = _update_gpu(u, pool)
    assert bits & ssd.DEV_INDEX_OOR
    assert torch.equal(pool[1], before[1]) and torch.equal(pool[2], before[2])
    assert torch.all(y[0] == 0) and torch.all(y[2] == 0)


@pytest.mark.parametrize("batch", [1, 32, 128, 256])
def test_decode_pool_full_size(batch):
    """512-slot pool of [128, 64, 128] fp32 states (2 GiB), a seeded permutation with 10%
    of rows set to -1; every untouched slot bit-identical, active slots checked on a
    sample of heads against the oracle."""
    H, P, G, N, S = 128, 64, 8, 128, 512
    idx = I.padded_permutation(S, batch, seed=3000 + batch)
    u = I.make_update_inputs(1, idx, H, P, G, N, act="bf16", seed=3100 + batch,
                             pool_values=np.zeros((1, H, P, N), np.float32))
    gen = torch.Generator(device="cuda").manual_seed(99)
    pool = torch.randn((S, H, P, N), generator=gen, device="cuda", dtype=torch.float32)
    before = pool.clone()
    y, bits = _update_gpu(u, pool)
    torch.cuda.synchronize()
    assert bits == 0
    active = [int(v) for v in idx if v >= 0]
    untouched = torch.ones(S, dtype=torch.bool, device="cuda")
    untouched[active] = False
    assert torch.equal(pool[untouched], before[untouched])
    assert torch.all(y[torch.from_numpy(idx == -1).cuda()] == 0)
    heads = [0, 37, 64, 127]
    rows = [b for b, v in enumerate(idx) if v >= 0][:8]
    for b in rows:
        slot = int(idx[b])
        st0 = before[slot][heads].cpu().numpy()
        g = np.asarray(heads) // (H // G)
        yk, fk = oracle.scan_seq(u.x.values[b:b + 1][:, heads], u.dt.values[b:b + 1][:, heads],
                                 u.A.values[heads], u.B.values[b:b + 1][:, g],
                                 u.C.values[b:b + 1][:, g], D=u.D.values[heads],
                                 dt_bias=u.dt_bias.values[heads], initial_states=st0[None])
        check_bf16(f"pool b={batch} row {b} y", y[b, heads].float().cpu().numpy(), yk[0])
        check_bf16(f"pool b={batch} row {b} slot", pool[slot][heads].cpu().numpy(), fk[0])


def test_decode_pool_batch256_every_active_slot():
    """The batch-256 sweep point compared in full: every active row's y on all 128 heads
    and every active slot's new [128, 64, 128] state against the oracle; untouched slots
    bit-identical, -1 rows zero."""
    H, P, G, N, S, batch = 128, 64, 8, 128, 512, 256
    idx = I.padded_permutation(S, batch, seed=3000 + batch)
    u = I.make_update_inputs(1, idx, H, P, G, N, act="bf16", seed=3100 + batch,
                             pool_values=np.zeros((1, H, P, N), np.float32))
    gen = torch.Generator(device="cuda").manual_seed(101)
    pool = torch.randn((S, H, P, N), generator=gen, device="cuda", dtype=torch.float32)
    active = np.array([int(v) for v in idx if v >= 0])
    act_t = torch.from_numpy(active).long().cuda()
    before_active = pool[act_t].cpu().numpy()
    before = pool.clone()
    y, bits = _update_gpu(u, pool)
    torch.cuda.synchronize()
    assert bits == 0
    untouched = torch.ones(S, dtype=torch.bool, device="cuda")
    untouched[act_t] = False
    assert torch.equal(pool[untouched], before[untouched])
    del before
    # the oracle on a pool of the active slots only, rows re-indexed into it
    pos = {int(s): k for k, s in enumerate(active)}
    idx_o = np.array([pos.get(int(v), -1) for v in idx], dtype=np.int32)
    new_o, y_o, st = oracle.state_update(before_active, idx_o, u.x.values, u.dt.values,
                                         u.A.values, u.B.values, u.C.values, D=u.D.values,
                                         dt_bias=u.dt_bias.values)
    assert st == 0
    check_bf16("pool b=256 all rows y", y.float().cpu().numpy(), y_o)
    assert np.all(y_o[idx == -1] == 0)
    check_bf16("pool b=256 all active slots", pool[act_t].cpu().numpy(), new_o)
