"""Golden fixtures (tests/golden/*.json, written by tests/golden/make_golden.py from the
oracle alone): the oracle must keep reproducing them, and the CUDA path must match them
within the fp32 bar."""
import json
import os

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def _a(v, dtype=np.float64):
    return np.asarray(v, dtype=dtype)


def test_oracle_reproduces_scan_fixture(oracle_mod):
    g = _load("scan_varlen_tiny.json")
    i = g["inputs"]
    y, fin = oracle_mod.scan_seq(_a(i["x"]), _a(i["dt"]), _a(i["A"]), _a(i["B"]), _a(i["C"]),
                                 D=_a(i["D"]), dt_bias=_a(i["dt_bias"]),
                                 initial_states=_a(i["initial_states"]),
                                 has_initial_state=i["has_initial_state"],
                                 cu_seqlens=i["cu_seqlens"])
    np.testing.assert_allclose(y, _a(g["outputs"]["y"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin, _a(g["outputs"]["final_states"]), rtol=1e-13, atol=1e-15)


def test_oracle_reproduces_update_fixture(oracle_mod):
    g = _load("state_update_tiny.json")
    i = g["inputs"]
    pool, y, st = oracle_mod.state_update(_a(i["pool"]), i["state_indices"], _a(i["x"]),
                                          _a(i["dt"]), _a(i["A"]), _a(i["B"]), _a(i["C"]),
                                          D=_a(i["D"]), dt_bias=_a(i["dt_bias"]))
    np.testing.assert_allclose(pool, _a(g["outputs"]["pool"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(y, _a(g["outputs"]["y"]), rtol=1e-13, atol=1e-15)
    assert st == g["outputs"]["status"]


def test_oracle_reproduces_norm_fixture(oracle_mod):
    g = _load("gated_norm_tiny.json")
    i = g["inputs"]
    out = oracle_mod.gated_rmsnorm(_a(i["x"]), _a(i["z"]), _a(i["weight"]),
                                   group_size=g["shape"]["group_size"], eps=g["shape"]["eps"])
    np.testing.assert_allclose(out, _a(g["outputs"]["out"]), rtol=1e-13, atol=1e-15)


@pytest.mark.gpu
def test_cuda_path_matches_golden_fixtures():
    import torch

    import oracle
    from mamba2_ssd_state_gb300 import ssd
    from tolerance import check_fp32, scan_K

    def t(v, dtype=torch.float32):
        return torch.tensor(np.asarray(v), dtype=dtype, device="cuda")

    g = _load("scan_varlen_tiny.json")
    i = g["inputs"]
    y, fin = ssd.chunk_scan(t(i["x"]), t(i["dt"]), t(i["A"]), t(i["B"]), t(i["C"]),
                            cu_seqlens=t(i["cu_seqlens"], torch.int32), chunk_size=4, D=t(i["D"]),
                            dt_bias=t(i["dt_bias"]), initial_states=t(i["initial_states"]),
                            has_initial_state=t(i["has_initial_state"], torch.uint8))
    sh = g["shape"]
    Ky, Kf = scan_K(i["cu_seqlens"], sh["H"], sh["P"], sh["N"], i["has_initial_state"])
    yr, fr = _a(g["outputs"]["y"]), _a(g["outputs"]["final_states"])
    _, _, ya, fa = oracle.scan_seq(_a(i["x"]), _a(i["dt"]), _a(i["A"]), _a(i["B"]), _a(i["C"]),
                                   D=_a(i["D"]), dt_bias=_a(i["dt_bias"]),
                                   initial_states=_a(i["initial_states"]),
                                   has_initial_state=i["has_initial_state"],
                                   cu_seqlens=i["cu_seqlens"], with_abs=True)
    check_fp32("golden scan y", y.cpu().numpy(), yr, ya, Ky)
    check_fp32("golden scan final", fin.cpu().numpy(), fr, fa, Kf)

    g = _load("state_update_tiny.json")
    i = g["inputs"]
    pool = t(i["pool"])
    y = ssd.state_update(pool, t(i["state_indices"], torch.int32), t(i["x"]), t(i["dt"]),
                         t(i["A"]), t(i["B"]), t(i["C"]), D=t(i["D"]), dt_bias=t(i["dt_bias"]))
    pr, yr = _a(g["outputs"]["pool"]), _a(g["outputs"]["y"])
    # error scale of each active row: its one-token recurrence evaluated on magnitudes
    pool0 = _a(i["pool"])
    for b, slot in enumerate(i["state_indices"]):
        if slot < 0:
            assert np.all(y.cpu().numpy()[b] == 0)
            continue
        _, _, ya, fa = oracle.scan_seq(_a(i["x"])[b:b + 1], _a(i["dt"])[b:b + 1], _a(i["A"]),
                                       _a(i["B"])[b:b + 1], _a(i["C"])[b:b + 1], D=_a(i["D"]),
                                       dt_bias=_a(i["dt_bias"]), initial_states=pool0[slot][None],
                                       with_abs=True)
        check_fp32(f"golden update y[{b}]", y.cpu().numpy()[b], yr[b], ya[0], 4 + 1)
        check_fp32(f"golden update slot {slot}", pool.cpu().numpy()[slot], pr[slot], fa[0], 4 + 1)
    np.testing.assert_array_equal(pool.cpu().numpy()[1], pool0[1].astype(np.float32))

    g = _load("gated_norm_tiny.json")
    i = g["inputs"]
    out = ssd.gated_rmsnorm(t(i["x"]), t(i["z"]), t(i["weight"]),
                            group_size=g["shape"]["group_size"], eps=g["shape"]["eps"])
    orf = _a(g["outputs"]["out"])
    check_fp32("golden norm", out.cpu().numpy(), orf, np.abs(orf), g["shape"]["group_size"])
