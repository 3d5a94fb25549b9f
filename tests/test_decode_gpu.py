"""GPU parity of the decode-side ops against the oracle: the multi-token state update
(with its per-token states and a rollback through the slot copy), the slot copy itself
(bit-exact), and the fused decode layer step (state update + D + gated RMSNorm)."""
import numpy as np
import pytest
import torch

import oracle
from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev
from tolerance import check_bf16, check_fp32

pytestmark = pytest.mark.gpu


def _multi_gpu(u, pool, inter=True):
    status = ssd.new_status()
    idx = torch.from_numpy(u.state_indices).cuda()
    y, st = ssd.state_update_multi(pool, idx, dev(u.x), dev(u.dt), dev(u.A), dev(u.B), dev(u.C),
                                   D=dev(u.D), dt_bias=dev(u.dt_bias), inter_states=inter,
                                   status=status)
    return y, st, ssd.read_status(status)[1]


def _multi_oracle(u):
    return oracle.state_update_multi(u.pool.values, u.state_indices, u.x.values, u.dt.values,
                                     u.A.values, u.B.values, u.C.values, D=u.D.values,
                                     dt_bias=u.dt_bias.values)


@pytest.mark.parametrize("N,ntok", [(16, 1), (16, 5), (128, 4), (64, 3)])
def test_multi_token_fp32(N, ntok):
    """fp32 against the double oracle at rtol(K), K = tokens so far + N (a decode step's
    length-N sum on top of its state)."""
    H, P, G, S = 4, 32, 2, 6
    idx = np.array([5, -1, 0, 2], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=401, ntok=ntok)
    pool = dev(u.pool)
    before = pool.clone()
    y, inter, bits = _multi_gpu(u, pool)
    assert bits == 0
    ref_pool, yr, ir, st = _multi_oracle(u)
    # the summation-error scale: the same recurrence on absolute values (the decay factor
    # and dt are positive already)
    _, ya, ia, _ = oracle.state_update_multi(np.abs(u.pool.values), idx, np.abs(u.x.values),
                                             u.dt.values, u.A.values, np.abs(u.B.values),
                                             np.abs(u.C.values), D=np.abs(u.D.values),
                                             dt_bias=u.dt_bias.values)
    for b, slot in enumerate(idx):
        if slot < 0:
            assert torch.all(y[b] == 0)
            continue
        for t in range(ntok):
            check_fp32(f"multi N={N} y[{b},{t}]", y[b, t].cpu().numpy(), yr[b, t], ya[b, t],
                       t + 1 + N)
            check_fp32(f"multi N={N} state[{b},{t}]", inter[b, t].cpu().numpy(), ir[b, t],
                       ia[b, t], t + 2)
        np.testing.assert_array_equal(pool[slot].cpu().numpy(), inter[b, -1].cpu().numpy())
    for slot in (1, 3, 4):
        assert torch.equal(pool[slot], before[slot])


def test_multi_token_bf16_nemotron_shapes():
    """H=128, P=64, G=8, N=128 (the varlen workload's layer), 4 draft tokens, 16 requests
    on a 40-slot pool with 2 padding rows."""
    H, P, G, N, S, ntok = 128, 64, 8, 128, 40, 4
    idx = I.padded_permutation(S, 16, seed=409)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=411, ntok=ntok)
    pool = dev(u.pool)
    y, inter, bits = _multi_gpu(u, pool)
    assert bits == 0
    ref_pool, yr, ir, st = _multi_oracle(u)
    act = idx >= 0
    check_bf16("multi bf16 y", y.float().cpu().numpy()[act], yr[act])
    check_bf16("multi bf16 inter", inter.cpu().numpy()[act], ir[act])
    active = sorted(int(v) for v in idx if v >= 0)
    check_bf16("multi bf16 pool", pool[active].cpu().numpy(), ref_pool[active])


def test_rollback_restores_the_accepted_token():
    """Run 5 draft tokens, accept m of them per request (m = 0 restores the snapshot taken
    before the step), then restore slots from the per-token states with ssd_state_copy:
    the pool equals the oracle after m tokens, bit for bit what the kernel computed."""
    H, P, G, N, S, ntok = 8, 64, 2, 128, 12, 5
    idx = np.array([7, 2, 9, -1, 0], dtype=np.int32)
    accept = [3, 0, 5, 2, 1]
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=421, ntok=ntok)
    pool = dev(u.pool)
    snap = torch.empty((len(idx), H, P, N), device="cuda")          # snapshot pool
    ridx = torch.arange(len(idx), dtype=torch.int32, device="cuda")
    gidx = torch.from_numpy(idx).cuda()
    ssd.state_copy(pool, gidx, snap, torch.where(gidx >= 0, ridx, -1))
    before = pool.clone()
    y, inter, bits = _multi_gpu(u, pool)
    assert bits == 0
    # restore: from inter[b, m-1] (as a pool of batch*ntok slots) or from the snapshot
    src_i = [b * ntok + m - 1 if m > 0 else -1 for b, m in enumerate(accept)]
    dst_i = [int(s) if m > 0 else -1 for s, m in zip(idx, accept)]
    status = ssd.new_status()
    ssd.state_copy(inter.view(len(idx) * ntok, H, P, N), torch.tensor(src_i, dtype=torch.int32,
                   device="cuda"), pool, torch.tensor(dst_i, dtype=torch.int32, device="cuda"),
                   status=status)
    snap_src = [b if (m == 0 and idx[b] >= 0) else -1 for b, m in enumerate(accept)]
    snap_dst = [int(idx[b]) if s >= 0 else -1 for b, s in enumerate(snap_src)]
    ssd.state_copy(snap, torch.tensor(snap_src, dtype=torch.int32, device="cuda"), pool,
                   torch.tensor(snap_dst, dtype=torch.int32, device="cuda"), status=status)
    assert ssd.read_status(status)[1] == 0
    _, _, ir, _ = _multi_oracle(u)
    for b, (slot, m) in enumerate(zip(idx, accept)):
        if slot < 0:
            continue
        if m == 0:
            assert torch.equal(pool[slot], before[slot])
        else:
            assert torch.equal(pool[slot], inter[b, m - 1])
            check_bf16(f"rollback row {b} m={m}", pool[slot].cpu().numpy(), ir[b, m - 1])


def test_state_copy_bit_exact_with_skips_and_bounds():
    rng = np.random.default_rng(431)
    src = torch.from_numpy(rng.standard_normal((9, 4, 64, 128)).astype(np.float32)).cuda()
    dst0 = rng.standard_normal((6, 4, 64, 128)).astype(np.float32)
    dst = torch.from_numpy(dst0).cuda()
    si, di = [8, -1, 0, 3, 11, 5], [1, 0, -1, 4, 2, 5]      # pair 4: source out of range
    status = ssd.new_status()
    ssd.state_copy(src, torch.tensor(si, dtype=torch.int32, device="cuda"), dst,
                   torch.tensor(di, dtype=torch.int32, device="cuda"), status=status)
    assert ssd.read_status(status)[1] == ssd.DEV_INDEX_OOR
    ref, st = oracle.state_copy(src.cpu().numpy(), si, dst0, di)
    assert st == 2
    np.testing.assert_array_equal(dst.cpu().numpy(), ref)


def test_state_copy_within_one_pool():
    rng = np.random.default_rng(433)
    pool0 = rng.standard_normal((8, 2, 64, 16)).astype(np.float32)
    pool = torch.from_numpy(pool0).cuda()
    si, di = [0, 1, 2], [5, 6, 7]
    ssd.state_copy(pool, torch.tensor(si, dtype=torch.int32, device="cuda"), pool,
                   torch.tensor(di, dtype=torch.int32, device="cuda"))
    ref, _ = oracle.state_copy(pool0, si, pool0, di)
    np.testing.assert_array_equal(pool.cpu().numpy(), ref)


def _layer(u, n, gs, pool, wt=None, want_y=True):
    status = ssd.new_status()
    idx = torch.from_numpy(u.state_indices).cuda()
    batch = len(u.state_indices)
    y = torch.empty((batch, u.H, u.P), dtype=dev(u.x).dtype, device="cuda") if want_y else None
    out = ssd.decode_layer_step(pool, idx, dev(u.x), dev(u.dt), dev(u.A), dev(u.B), dev(u.C),
                                dev(n.z), wt if wt is not None else dev(n.weight), group_size=gs,
                                D=dev(u.D), dt_bias=dev(u.dt_bias), y=y, status=status)
    return out, y, ssd.read_status(status)[1]


@pytest.mark.parametrize("H,P,G,gs,batch", [(128, 64, 8, 1024, 32), (24, 64, 1, 1536, 8),
                                            (6, 64, 2, 192, 5), (4, 32, 2, 32, 3)])
def test_decode_layer_step_bf16(H, P, G, gs, batch):
    """Norm groups of 16, 24, 3 and 1 heads."""
    N, S = 128, batch + 7
    idx = I.padded_permutation(S, batch, seed=441 + batch)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="bf16", seed=443)
    n = I.make_norm_inputs(batch, H * P, gs, act="bf16", seed=445)
    pool = dev(u.pool)
    out, y, bits = _layer(u, n, gs, pool)
    assert bits == 0
    ref_pool, yr, outr, st = oracle.decode_layer_step(
        u.pool.values, idx, u.x.values, u.dt.values, u.A.values, u.B.values, u.C.values,
        n.z.values, n.weight.values, group_size=gs, D=u.D.values, dt_bias=u.dt_bias.values)
    # out is normalised: a channel can sit many group-RMS above the rest, where bf16's
    # own spacing passes 0.1; the max-abs bar counts the error beyond that rounding
    check_bf16(f"layer H={H} gs={gs} out", out.float().cpu().numpy(), outr, stored_bf16=True)
    check_bf16(f"layer H={H} gs={gs} y", y.float().cpu().numpy(), yr)
    active = sorted(int(v) for v in idx if v >= 0)
    check_bf16(f"layer H={H} gs={gs} pool", pool[active].cpu().numpy(), ref_pool[active])
    assert torch.all(out[torch.from_numpy(idx == -1).cuda()] == 0)


def test_decode_layer_step_fp32_and_unfused_agree():
    """fp32 activations with an fp32 weight, y not requested (the norm then runs in place
    on out); against the oracle and against ssd_state_update + gated_rmsnorm called
    separately."""
    H, P, G, N, S, gs, batch = 8, 16, 2, 32, 6, 64, 4
    idx = np.array([3, 0, -1, 5], dtype=np.int32)
    u = I.make_update_inputs(S, idx, H, P, G, N, act="f32", seed=451)
    n = I.make_norm_inputs(batch, H * P, gs, act="f32", seed=453)
    pool = dev(u.pool)
    pool2 = pool.clone()
    out, _, bits = _layer(u, n, gs, pool, want_y=False)
    assert bits == 0
    _, _, outr, _ = oracle.decode_layer_step(
        u.pool.values, idx, u.x.values, u.dt.values, u.A.values, u.B.values, u.C.values,
        n.z.values, n.weight.values, group_size=gs, D=u.D.values, dt_bias=u.dt_bias.values)
    np.testing.assert_allclose(out.cpu().numpy(), outr, rtol=2e-5, atol=2e-5)
    y2 = ssd.state_update(pool2, torch.from_numpy(idx).cuda(), dev(u.x), dev(u.dt), dev(u.A),
                          dev(u.B), dev(u.C), D=dev(u.D), dt_bias=dev(u.dt_bias))
    out2 = ssd.gated_rmsnorm(y2.view(batch, H * P), dev(n.z), dev(n.weight), group_size=gs)
    np.testing.assert_allclose(out.cpu().numpy(), out2.cpu().numpy(), rtol=2e-5, atol=2e-5)
    assert torch.equal(pool, pool2)


def test_decode_layer_step_rejects_bad_groups():
    H, P, G, N = 4, 32, 2, 16
    u = I.make_update_inputs(3, [0, 1], H, P, G, N, act="f32", seed=461)
    n = I.make_norm_inputs(2, H * P, 32, act="f32", seed=463)
    for gs in (48, 16, 96):   # not a multiple of P, smaller than P, not dividing H*P
        with pytest.raises(ssd.SsdError) as e:
            _layer(u, n, gs, dev(u.pool))
        assert e.value.code == 1
