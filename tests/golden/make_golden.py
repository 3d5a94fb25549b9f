"""Write the golden fixtures in this directory from the CPU oracle (and only the oracle).

Each fixture is a small JSON text file holding seeded inputs and the oracle's outputs in
full double precision, with the source of the op it pins:
  scan_varlen_tiny.json   Mamba2 chunked SSD scan (vt::Mamba2ChunkScan of the vllm.cpp page
                          "W2 finish (KERNEL-SSM-MAMBA)"), 2 packed sequences, one with an
                          initial state; recurrence of Dao & Gu, "Transformers are SSMs".
  state_update_tiny.json  decode state update on a pool with a -1 row
                          (vt::Mamba2StateUpdate, same page, mutation rows M5, M6).
  gated_norm_tiny.json    gate-then-norm with per-group variance (vt::RmsNormGatedGroup,
                          same page, mutation rows M7, M8).
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mamba2_ssd_state_gb300 import inputs as I  # noqa: E402


def _l(a):
    return np.asarray(a, dtype=np.float64).tolist()


def scan_fixture():
    s = I.make_scan_inputs([7, 5], H=2, P=3, G=1, N=4, chunk_size=4, act="f32", seed=77,
                           init=[1, 0])
    y, fin = oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                             D=s.D.values, dt_bias=s.dt_bias.values,
                             initial_states=s.initial_states.values,
                             has_initial_state=s.has_initial_state, cu_seqlens=s.cu_seqlens)
    return {
        "source": "Mamba2 chunked SSD scan (vllm.cpp PR #566 'W2 finish (KERNEL-SSM-MAMBA)', "
                  "vt::Mamba2ChunkScan; recurrence of Dao & Gu 2024)",
        "shape": dict(seqlens=s.seqlens, H=2, P=3, G=1, N=4, chunk_size=4, dt_softplus=True),
        "inputs": dict(x=_l(s.x.values), dt=_l(s.dt.values), dt_bias=_l(s.dt_bias.values),
                       A=_l(s.A.values), B=_l(s.B.values), C=_l(s.C.values), D=_l(s.D.values),
                       initial_states=_l(s.initial_states.values),
                       has_initial_state=s.has_initial_state.tolist(),
                       cu_seqlens=s.cu_seqlens.tolist()),
        "outputs": dict(y=_l(y), final_states=_l(fin)),
    }


def update_fixture():
    idx = [2, -1, 0]
    u = I.make_update_inputs(3, idx, H=2, P=3, G=1, N=4, act="f32", seed=78)
    pool, y, st = oracle.state_update(u.pool.values, idx, u.x.values, u.dt.values, u.A.values,
                                      u.B.values, u.C.values, D=u.D.values,
                                      dt_bias=u.dt_bias.values)
    return {
        "source": "decode state update on a pooled state cache (vllm.cpp PR #566, "
                  "vt::Mamba2StateUpdate; mutation rows M5, M6)",
        "shape": dict(num_slots=3, H=2, P=3, G=1, N=4, dt_softplus=True),
        "inputs": dict(pool=_l(u.pool.values), state_indices=idx, x=_l(u.x.values),
                       dt=_l(u.dt.values), dt_bias=_l(u.dt_bias.values), A=_l(u.A.values),
                       B=_l(u.B.values), C=_l(u.C.values), D=_l(u.D.values)),
        "outputs": dict(pool=_l(pool), y=_l(y), status=st),
    }


def norm_fixture():
    n = I.make_norm_inputs(3, 16, 8, act="f32", seed=79)
    out = oracle.gated_rmsnorm(n.x.values, n.z.values, n.weight.values, group_size=8, eps=1e-5)
    return {
        "source": "silu-gated RMSNorm, per-group variance (vllm.cpp PR #566, "
                  "vt::RmsNormGatedGroup; mutation rows M7, M8)",
        "shape": dict(rows=3, d=16, group_size=8, eps=1e-5),
        "inputs": dict(x=_l(n.x.values), z=_l(n.z.values), weight=_l(n.weight.values)),
        "outputs": dict(out=_l(out)),
    }


def main():
    for name, fn in (("scan_varlen_tiny.json", scan_fixture),
                     ("state_update_tiny.json", update_fixture),
                     ("gated_norm_tiny.json", norm_fixture)):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=1)
        print("wrote", name)


if __name__ == "__main__":
    main()
