"""GPU parity of gated_rmsnorm (gate first, per-group variance) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from mamba2_ssd_state_gb300 import inputs as I
from mamba2_ssd_state_gb300 import ssd
from gpu_util import dev
from tolerance import check_bf16, check_fp32

pytestmark = pytest.mark.gpu


def _run(n, z=True, out=None):
    return ssd.gated_rmsnorm(dev(n.x), dev(n.z) if z else None, dev(n.weight),
                             group_size=n.group_size, eps=n.eps, out=out)


def test_tiny_fp32_norm():
    n = I.make_norm_inputs(64, 64, 64, act="f32", seed=4000)
    out = _run(n).cpu().numpy()
    ref = oracle.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=64, eps=n.eps)
    check_fp32("norm tiny fp32", out, ref, np.abs(ref), 64)


@pytest.mark.parametrize("rows,d,gs,act,wt", [
    (37, 1536, 1536, "bf16", "bf16"),   # one group over the row (vector path, 6 per lane)
    (19, 8192, 1024, "bf16", "bf16"),   # 8 groups of 1024
    (11, 256, 16, "bf16", "f32"),       # many small groups (generic path)
    (9, 96, 32, "f32", "f32"),
    (5, 2048, 2048, "bf16", "f32"),
    (3, 640, 320, "bf16", "bf16"),      # group not a multiple of 256
])
def test_norm_shapes(rows, d, gs, act, wt):
    n = I.make_norm_inputs(rows, d, gs, act=act, wdtype=wt, seed=4100 + d)
    out = _run(n).float().cpu().numpy()
    ref = oracle.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=gs)
    if act == "bf16":
        check_bf16(f"norm {rows}x{d}/{gs}", out, ref)
    else:
        check_fp32(f"norm {rows}x{d}/{gs}", out, ref, np.abs(ref), gs)


def test_norm_without_gate_and_in_place():
    n = I.make_norm_inputs(8, 1024, 256, act="bf16", seed=4200)
    x = dev(n.x)
    out = ssd.gated_rmsnorm(x, None, dev(n.weight), group_size=256, eps=n.eps, out=x)
    assert out.data_ptr() == x.data_ptr()
    ref = oracle.gated_rmsnorm(n.x.values, None, n.weight.values, group_size=256)
    check_bf16("norm no gate in place", x.float().cpu().numpy(), ref)


def test_norm_per_group_not_whole_row():
    """Groups with very different scales: per-group variance keeps each group at unit RMS."""
    n = I.make_norm_inputs(4, 512, 128, act="bf16", seed=4300)
    xv = n.x.values.copy()
    xv[:, 128:256] *= 30.0
    n = I.make_norm_inputs(4, 512, 128, act="bf16", seed=4300, x_values=xv)
    out = _run(n).float().cpu().numpy()
    ref = oracle.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=128)
    check_bf16("norm per-group", out, ref)


def test_norm_full_size_sampled_rows():
    """16384 rows x d_inner 8192 in 8 groups of 1024 (bf16): sampled rows vs the oracle."""
    rows, d, gs = 16384, 8192, 1024
    gen = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn((rows, d), generator=gen, device="cuda").to(torch.bfloat16)
    z = torch.randn((rows, d), generator=gen, device="cuda").to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn((d,), generator=gen, device="cuda")).to(torch.bfloat16)
    out = ssd.gated_rmsnorm(x, z, w, group_size=gs, eps=1e-5)
    sel = np.random.default_rng(1).choice(rows, 64, replace=False)
    ref = oracle.gated_rmsnorm(x[sel].float().cpu().numpy(), z[sel].float().cpu().numpy(),
                               w.float().cpu().numpy(), group_size=gs)
    check_bf16("norm full sampled", out[sel].float().cpu().numpy(), ref)
