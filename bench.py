"""Benchmark of the Mamba2 SSD hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input shaped like a
Nemotron-H Mamba2 layer: 4 packed prefill sequences of [8192, 3000, 517, 4675] tokens
(16384 tokens, H=128, P=64, G=8, N=128, chunk 128, bf16 activations, fp32 initial states
on sequences 0 and 2) through the chunked scan with D skip and the silu-gated RMSNorm
(8 groups of 1024) in one call, then the next decode token of the same 4 requests through
the pooled state update.  `value` counts the prefill tokens only.
Inputs are resident in HBM; L2 (129 MB, smaller than the step's 0.9 GB of inputs and
outputs) is flushed between timed steps anyway (512 MB write, then a 512 MB read so no
dirty line is left to write back), outside the timed events.

Prints one JSON line (rank 0).  Also measured in the same run and reported as extra keys:
the Mamba2-130M-shaped layer step, the gated norm alone at the Nemotron-H shape, the
decode state update on a 512-slot [128, 64, 128] fp32 pool at batch 256 (HBM GB/s), the
decode layer step, the multi-token update beside the HBM write-only rate, the slot copy,
one long sequence on few heads, and the prefill layer path at Nemotron-H shapes (single
sequences of 1K..64K tokens, and a mixed batch with a concurrent decode).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (double precision, host cores) on a bounded sample
of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "nemotron_h_varlen"
METRIC = "Mamba2 SSD prefill tokens/s; decode state-update HBM GB/s vs peak"
KERNEL_CHUNK = 128  # tokens per chunk of the tensor-core scan kernels (their MMA tile)
SCAN_SRCS = ["scan_tc.cu", "scan_pair.cuh", "tc_ptx.cuh", "ssd_internal.cuh",
             "scan_segments.cuh", "scan_states.cuh"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def scan_sources_sha256():
    import hashlib

    h = hashlib.sha256()
    for f in SCAN_SRCS:
        h.update(open(os.path.join(ROOT, "mamba2_ssd_state_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def scan_traffic_from_profile(name):
    """DRAM bytes per launch of the scan from the committed ncu summary profiles/<name>,
    if the kernel sources still hash to what was profiled; else None."""
    import re

    try:
        txt = open(os.path.join(ROOT, "profiles", name)).read()
        digest = scan_sources_sha256()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", txt)
    m_traffic = re.search(r"traffic_bytes_per_launch\s*\|\s*(\d+)", txt)
    if not m_hash or not m_traffic or m_hash.group(1) != digest:
        return None
    return int(m_traffic.group(1))


def scan_bytes(T, H, P, G, N, nseq, n_init=None, final=True, act_bytes=2):
    """Algorithmic HBM bytes of one scan launch: x and y, B and C, dt, per-head params,
    the initial states that are read (n_init sequences; all when None) and the final
    states (intermediate chunk states are not counted)."""
    b = T * H * P * act_bytes * 2 + T * G * N * act_bytes * 2 + T * H * 4 + H * 4 * 3
    b += (nseq + 1) * 4
    b += (nseq if n_init is None else n_init) * H * P * N * 4
    if final:
        b += nseq * H * P * N * 4
    return b


def layer_bytes(T, H, P, G, N, nseq=0, n_init=0, final=False):
    """Algorithmic bytes of the prefill layer path (scan, D skip, gated norm) in bf16: x, z
    and out 2HP each, B and C 2GN each and dt 4H per token, plus the norm weight and, when
    asked, the initial states read and the final states written; y is an intermediate
    and not counted."""
    b = T * (6 * H * P + 4 * G * N + 4 * H) + 2 * H * P
    return b + (n_init + (nseq if final else 0)) * H * P * N * 4


def update_bytes(active, batch, H, P, G, N, act_bytes=2):
    """Algorithmic HBM bytes of one decode launch: each active slot's state read and
    written once, plus x, y, B, C, dt of every row and the per-head parameters."""
    return (active * H * P * N * 4 * 2 + batch * (2 * H * P * act_bytes + 2 * G * N * act_bytes
                                                  + H * 4 + 4) + H * 4 * 3)


def norm_bytes(rows, d, act_bytes=2, w_bytes=2):
    return rows * d * act_bytes * 3 + d * w_bytes


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


class L2Flush:
    """Between timed steps: write a 512 MB buffer (evicts the step's inputs from the
    129 MB L2), then read another 512 MB buffer, so the dirty lines of the write are
    written back before the next step starts and do not land inside its timing."""
    DESCRIPTION = ("flushed between steps: 512 MB write, then 512 MB read (clean L2), "
                   "outside the timed events")

    def __init__(self, torch, dev):
        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def flush(self):
        self.w.zero_()
        self.acc += self.r.sum()


def graph_of(torch, fn):
    """fn() captured in a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def timed_replays(torch, stream, l2, replay, n):
    """Device time (ms) of n replays, each after an L2 flush outside its events."""
    ts = []
    for _ in range(n):
        l2.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return ts


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch

    from mamba2_ssd_state_gb300 import build as lib_build
    from mamba2_ssd_state_gb300 import inputs as I
    from mamba2_ssd_state_gb300 import shard
    from mamba2_ssd_state_gb300 import ssd

    lib_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    hbm_peak, tc_peak, peak_kind = load_peaks()

    def T_(t):
        dtype = torch.bfloat16 if t.dtype == "bf16" else torch.float32
        return torch.from_numpy(np.ascontiguousarray(t.values)).to(dev, dtype)

    w = I.WORKLOADS[WORKLOAD]
    # data parallel: rank r processes its own batch of the workload, drawn with its own
    # seed; no collective on the data path
    s = I.scan_workload(WORKLOAD, seed=w["seed"] + 17 * rank)
    H, P, G, N, T, nseq = s.H, s.P, s.G, s.N, s.T, s.nseq
    d, group = H * P, w["norm_group"]
    x, dt, A, B, C, Dp, bias = (T_(s.x), T_(s.dt), T_(s.A), T_(s.B), T_(s.C), T_(s.D),
                                T_(s.dt_bias))
    init = T_(s.initial_states)
    hi = torch.from_numpy(s.has_initial_state).to(dev)
    n_init = int(np.sum(s.has_initial_state))
    cu = torch.from_numpy(s.cu_seqlens).to(dev)
    nrm = I.make_norm_inputs(T, d, group, act="bf16", seed=w["seed"] + 50)
    z, wt = T_(nrm.z), T_(nrm.weight)
    y = torch.empty((T, H, P), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((nseq, H, P, N), dtype=torch.float32, device=dev)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    # the next decode token of the nseq requests: their pool slots hold the final states
    # of the prefill after the first warm-up step
    pool = torch.zeros((nseq, H, P, N), dtype=torch.float32, device=dev)
    upd = I.make_update_inputs(nseq, list(range(nseq)), H, P, G, N, act="bf16",
                               seed=w["seed"] + 60)
    ux, udt, uB, uC = T_(upd.x), T_(upd.dt), T_(upd.B), T_(upd.C)
    uidx = torch.arange(nseq, dtype=torch.int32, device=dev)
    uy = torch.empty((nseq, H, P), dtype=torch.bfloat16, device=dev)
    status = ssd.new_status(dev)
    l2 = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()

    def scan_call():
        ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=s.chunk_size, D=Dp,
                       dt_bias=bias, initial_states=init, has_initial_state=hi, y=y,
                       final_states=fs, status=status)

    def norm_call():
        ssd.gated_rmsnorm(y.view(T, d), z, wt, group_size=group, eps=1e-5, out=out)

    def decode_call(st=None, inp=None):
        i = inp or dict(ux=ux, udt=udt, uB=uB, uC=uC)
        ssd.state_update(pool, uidx, i["ux"], i["udt"], A, i["uB"], i["uC"], D=Dp, dt_bias=bias,
                         y=uy, status=status, stream=st)

    # the call's workspace: the ready counters of its overlapped form (the norm normalises the
    # scan's finished chunks while the scan runs), or a split's, or none
    lws_bytes = ssd.chunk_scan_gated_norm_workspace_size(x, B, C, z, wt, out, cu_seqlens=cu,
                                                         chunk_size=s.chunk_size,
                                                         group_size=group)
    lws = torch.empty(max(lws_bytes, 1), dtype=torch.uint8, device=dev)
    scan_split_bytes = ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu,
                                                     chunk_size=s.chunk_size)
    norm_form = ("chained" if lws_bytes == 0 or lws_bytes == scan_split_bytes
                 else "overlapped")

    def layer_prefill(st=None, inp=None, out_=None):
        """The prefill half of the layer in one call: scan, D skip and gated norm, the norm
        a programmatic dependent of the scan that normalises in place in out."""
        i = inp or dict(x=x, dt=dt, B=B, C=C, init=init, z=z)
        ssd.chunk_scan_gated_norm(i["x"], i["dt"], A, i["B"], i["C"], i["z"], wt, cu_seqlens=cu,
                                  chunk_size=s.chunk_size, group_size=group, eps=1e-5, D=Dp,
                                  dt_bias=bias, initial_states=i["init"], has_initial_state=hi,
                                  out=out if out_ is None else out_, final_states=fs,
                                  status=status, stream=st, workspace=lws)

    # the scan is one launch, or two when the library splits the sequences into segments
    scan_split = ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu,
                                               chunk_size=s.chunk_size) > 0
    launches_per_step = (2 if scan_split else 1) + 2
    for i in range(max(args.warmup, 3)):
        l2.flush()
        scan_call()
        norm_call()
        decode_call()
        layer_prefill()
        if i == 0:
            torch.cuda.synchronize()
            pool.copy_(fs)   # the decode continues the requests just prefilled
    torch.cuda.synchronize()
    rc, bits = ssd.read_status(status)
    if bits:
        raise RuntimeError(f"device status bits {bits} after warm-up")

    # The timed step is one CUDA graph of its launches (the way a serving engine runs a
    # layer): no host work and no launch gaps.  The decode token follows the prefill on
    # the same stream: run beside it on a second stream it measured slower (422 against
    # 415 us), its blocks delaying the scan's first wave.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer_prefill()
        decode_call()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    # keep the GPU under the same load for a second first, so that the clock samples
    # (100 ms apart) cover the state it is timed in
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 1.0:
        for _ in range(10):
            l2.flush()
            graph.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for k in range(args.steps):
        l2.flush()             # outside the step's events
        evs[k][0].record(stream)
        graph.replay()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    ck = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = shard.max_over_ranks(sum(step_ms), dev)
    tokens_per_step = T       # prefill tokens; the decode tokens are not counted
    value = tokens_per_step * world * args.steps / (total_ms / 1e3)

    # per-op split of a step, each op graph-replayed alone after an L2 flush
    n_op = max(5, args.steps // 2)
    g_scan, g_norm, g_dec = graph_of(torch, scan_call), graph_of(torch, norm_call), \
        graph_of(torch, decode_call)
    g_layer = graph_of(torch, layer_prefill)
    scan_ms = timed_replays(torch, stream, l2, g_scan.replay, n_op)
    norm_ms = timed_replays(torch, stream, l2, g_norm.replay, n_op)
    dec_ms = timed_replays(torch, stream, l2, g_dec.replay, n_op)
    layer_ms = timed_replays(torch, stream, l2, g_layer.replay, n_op)
    med = lambda v: float(np.median(v))  # noqa: E731

    sbytes = scan_bytes(T, H, P, G, N, nseq, n_init=n_init)
    scan_avg = sum(scan_ms) / len(scan_ms)
    scan_kernels = ("scan_pair_kernel + scan_fixup_kernel" if scan_split
                    else "scan_pair_kernel (two heads of a group per CTA)")
    roof = {"bound": "hbm", "kernel": scan_kernels,
            "achieved": sbytes / (scan_avg / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
            "peak_kind": f"{peak_kind} hbm copy",
            "algorithmic_bytes_per_launch": sbytes, "avg_launch_us": scan_avg * 1e3,
            "traffic": scan_traffic_from_profile("scan_pair_nemotron_h_varlen.md"),
            "traffic_note": "ncu dram read+write of one scan launch at this workload "
                            "(profiles/scan_pair_nemotron_h_varlen.md), null if the kernel "
                            "sources changed since",
            "avg_launch_note": "one scan call replayed from a graph after an L2 flush, events "
                               "on the launching stream",
            "flops_per_launch": T * (G * (KERNEL_CHUNK + 1) * N + H * (KERNEL_CHUNK + 1) * P
                                     + 4 * H * P * N)}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["tflops"] = roof["flops_per_launch"] / (scan_avg / 1e3) / 1e12
    roof["frac_of_bf16_peak"] = roof["tflops"] / tc_peak
    nb = norm_bytes(T, d)
    norm_avg = sum(norm_ms) / len(norm_ms)
    lb = layer_bytes(T, H, P, G, N, nseq, n_init=n_init, final=True)
    layer_avg = sum(layer_ms) / len(layer_ms)

    extra = {}
    if rank == 0 and not args.no_extra:
        extra["mamba2_130m_layer"] = measure_130m(torch, I, ssd, dev, hbm_peak, peak_kind, l2)
        extra.update(measure_extra(torch, I, ssd, dev, hbm_peak, peak_kind))

    # end to end through the public API: every step copies its inputs from pinned host
    # memory and reads its result back.  Copies and compute run on three streams with two
    # sets of device buffers, so the copies of step k+1 and the read-back of step k-1
    # overlap the compute of step k (the copy engines and the SMs work at once).
    names = ("x", "dt", "B", "C", "init", "z", "ux", "udt", "uB", "uC")
    host_in = {k: v.detach().cpu().pin_memory() for k, v in
               zip(names, (x, dt, B, C, init, z, ux, udt, uB, uC))}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    sets = []
    for _ in range(2):
        sets.append(dict(inp={k: torch.empty_like(v, device=dev) for k, v in host_in.items()},
                         out=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
                         host_out=torch.empty((T, d), dtype=torch.bfloat16).pin_memory(),
                         ev={k: torch.cuda.Event() for k in ("h2d", "comp", "d2h")},
                         used=False))
    d2h = sets[0]["host_out"].numel() * sets[0]["host_out"].element_size()
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_step(k):
        st = sets[k % 2]
        ev = st["ev"]
        with torch.cuda.stream(s_h2d):
            if st["used"]:
                s_h2d.wait_event(ev["comp"])   # step k-2 finished reading this input set
            for k2, v in host_in.items():
                st["inp"][k2].copy_(v, non_blocking=True)
            ev["h2d"].record(s_h2d)
        stream.wait_event(ev["h2d"])
        if st["used"]:
            stream.wait_event(ev["d2h"])       # step k-2's result was read back
        di, o = st["inp"], st["out"]
        layer_prefill(stream, di, o)
        decode_call(stream, di)
        ev["comp"].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["comp"])
            st["host_out"].copy_(o, non_blocking=True)
            ev["d2h"].record(s_d2h)
        st["used"] = True

    for k in range(4):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    s_h2d.wait_event(e0)
    for k in range(args.steps):
        e2e_step(k)
    stream.wait_event(sets[(args.steps - 1) % 2]["ev"]["d2h"])
    stream.wait_event(sets[args.steps % 2]["ev"]["d2h"])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = shard.max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = tokens_per_step * world * args.steps / (e2e_ms / 1e3)

    rc, bits = ssd.read_status(status)
    if bits:
        raise RuntimeError(f"device status bits {bits} after the timed region")

    if rank != 0:
        return None
    cpu = None if args.no_cpu else cpu_baseline(s, nrm, w)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "Nemotron-H-shaped varlen prefill layer: 4 packed sequences "
                               "[8192, 3000, 517, 4675] (16384 tokens), H=128 P=64 G=8 N=128, "
                               "initial states on sequences 0 and 2; scan + D skip + gated "
                               "RMSNorm (8 groups of 1024) in one call, then the next decode "
                               "token of the 4 requests",
                   "seqlens": s.seqlens, "H": H, "P": P, "G": G, "N": N,
                   "chunk_size": s.chunk_size, "kernel_chunk": KERNEL_CHUNK,
                   "norm_group": group, "prefill_tokens_per_step": tokens_per_step,
                   "decode_tokens_per_step": nseq, "l2": L2Flush.DESCRIPTION,
                   "launch": "the step's kernels replayed as one CUDA graph on one stream: scan + "
                             "gated norm in one call (the norm a programmatic dependent of the "
                             "scan), then the decode token",
                   "norm_form": norm_form + (
                       ": the scan counts each finished 128-token chunk of each norm group "
                       "and the norm kernel normalises those rows while the scan "
                       "runs" if norm_form == "overlapped" else ": the norm follows the scan"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "breakdown_us": {"scan": 1e3 * med(scan_ms), "gated_rmsnorm": 1e3 * med(norm_ms),
                         "state_update_4_slots": 1e3 * med(dec_ms),
                         "scan_gated_norm_call": 1e3 * med(layer_ms),
                         "note": "each op replayed alone from a graph after an L2 flush"},
        "wall_s_timed_region": t_wall,
        "roofline": roof,
        "gated_rmsnorm_nemotron_h": {
            "workload": "16384 x 8192 bf16, 8 groups of 1024, gated (z), bf16 weight",
            "avg_launch_us": norm_avg * 1e3, "algorithmic_bytes_per_launch": nb,
            "achieved_gbs": nb / (norm_avg / 1e3) / 1e9,
            "frac": nb / (norm_avg / 1e3) / 1e9 / hbm_peak, "peak_kind": f"{peak_kind} hbm copy",
            "note": "replayed alone from a graph after an L2 flush"},
        "layer_call_nemotron_h": {
            "avg_launch_us": layer_avg * 1e3, "algorithmic_bytes_per_launch": lb,
            "achieved_gbs": lb / (layer_avg / 1e3) / 1e9,
            "frac": lb / (layer_avg / 1e3) / 1e9 / hbm_peak,
            "note": "scan + D + gated norm in one call (x, z, out, B, C, dt, states; y not "
                    "counted)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
        "cpu_baseline": cpu,
    }
    line.update(extra)
    return line


def measure_130m(torch, I, ssd, dev, hbm_peak, peak_kind, l2, iters=20):
    """The Mamba2-130M-shaped layer step: 2 x 2048 tokens (H=24, P=64, G=1, N=128, chunk
    256, initial states), scan + gated norm (d 1536, one group) in one call and one decode
    token of both requests on a second stream (the scan leaves SMs idle here, and beside
    it the decode measured faster than after it: 45 against 48 us), replayed as one graph
    after an L2 flush; plus the scan call alone against its roofline."""
    name = "mamba2_130m"
    w = I.WORKLOADS[name]
    s = I.scan_workload(name)

    def T_(t):
        dtype = torch.bfloat16 if t.dtype == "bf16" else torch.float32
        return torch.from_numpy(np.ascontiguousarray(t.values)).to(dev, dtype)

    H, P, G, N, T, nseq = s.H, s.P, s.G, s.N, s.T, s.nseq
    d = H * P
    x, dt, A, B, C, Dp, bias, init = (T_(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D,
                                                        s.dt_bias, s.initial_states))
    cu = torch.from_numpy(s.cu_seqlens).to(dev)
    nrm = I.make_norm_inputs(T, d, w["norm_group"], act="bf16", seed=w["seed"] + 50)
    z, wt = T_(nrm.z), T_(nrm.weight)
    y = torch.empty((T, H, P), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((nseq, H, P, N), dtype=torch.float32, device=dev)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    pool = 0.1 * torch.randn((nseq, H, P, N), dtype=torch.float32, device=dev)
    upd = I.make_update_inputs(nseq, list(range(nseq)), H, P, G, N, act="bf16",
                               seed=w["seed"] + 60)
    ux, udt, uB, uC = T_(upd.x), T_(upd.dt), T_(upd.B), T_(upd.C)
    uidx = torch.arange(nseq, dtype=torch.int32, device=dev)
    uy = torch.empty((nseq, H, P), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    nws = ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu, chunk_size=s.chunk_size)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)

    def scan_call():
        ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=s.chunk_size, D=Dp,
                       dt_bias=bias, initial_states=init, y=y, final_states=fs, workspace=ws)

    def layer():
        ssd.chunk_scan_gated_norm(x, dt, A, B, C, z, wt, cu_seqlens=cu, chunk_size=s.chunk_size,
                                  group_size=w["norm_group"], eps=1e-5, D=Dp, dt_bias=bias,
                                  initial_states=init, out=out, final_states=fs, workspace=ws)

    s_dec = torch.cuda.Stream(device=dev)
    for _ in range(3):
        scan_call()
        layer()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream()
        s_dec.wait_stream(cap)
        with torch.cuda.stream(s_dec):
            ssd.state_update(pool, uidx, ux, udt, A, uB, uC, D=Dp, dt_bias=bias, y=uy)
        layer()
        cap.wait_stream(s_dec)
    step = timed_replays(torch, stream, l2, g.replay, iters)
    g_scan = graph_of(torch, scan_call)
    sc = timed_replays(torch, stream, l2, g_scan.replay, iters)
    st_ms, sc_ms = float(np.median(step)), float(np.median(sc))
    sb = scan_bytes(T, H, P, G, N, nseq)
    return {"workload": "Mamba2-130M-shaped layer: 2 x 2048 tokens, H=24 P=64 G=1 N=128, chunk "
                        "256 (kernel chunk 128), scan + gated RMSNorm (d 1536) in one call + "
                        "decode of both requests on a second stream",
            "step_us": st_ms * 1e3, "prefill_tokens_per_s": T / (st_ms / 1e3),
            "scan_us": sc_ms * 1e3, "scan_split_into_segments": nws > 0,
            "scan_algorithmic_bytes": sb, "scan_achieved_gbs": sb / (sc_ms / 1e3) / 1e9,
            "scan_frac_hbm": sb / (sc_ms / 1e3) / 1e9 / hbm_peak,
            "scan_traffic": scan_traffic_from_profile("scan_split_mamba2_130m.md"),
            "peak_kind": f"{peak_kind} hbm copy",
            "note": "median of graph replays, each after an L2 flush"}


def measure_extra(torch, I, ssd, dev, hbm_peak, peak_kind, iters=20):
    """Decode at batch 256 on the 512-slot pool, the decode layer step, the multi-token
    update beside the HBM write-only rate, the slot copy, one long sequence on few heads
    (split into segments by the library's planner), and the Nemotron-H layer path."""
    res = {}
    stream = torch.cuda.current_stream()
    H, P, G, N, S, batch = 128, 64, 8, 128, 512, 256
    idx = I.padded_permutation(S, batch, seed=3000 + batch)
    u = I.make_update_inputs(1, idx, H, P, G, N, act="bf16", seed=3100 + batch,
                             pool_values=np.zeros((1, H, P, N), np.float32))

    def T_(t):
        dtype = torch.bfloat16 if t.dtype == "bf16" else torch.float32
        return torch.from_numpy(np.ascontiguousarray(t.values)).to(dev, dtype)

    pool = torch.randn((S, H, P, N), device=dev, dtype=torch.float32)
    args = (pool, torch.from_numpy(idx).to(dev), T_(u.x), T_(u.dt), T_(u.A), T_(u.B), T_(u.C))
    kw = dict(D=T_(u.D), dt_bias=T_(u.dt_bias))
    for _ in range(3):
        ssd.state_update(*args, **kw)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(iters):
        ssd.state_update(*args, **kw)
    ev1.record(stream)
    torch.cuda.synchronize()
    us = ev0.elapsed_time(ev1) * 1e3 / iters
    active = int((idx >= 0).sum())
    ub = update_bytes(active, batch, H, P, G, N)
    res["decode_state_update"] = {
        "workload": "512-slot pool of [128,64,128] fp32 states, batch 256, 10% rows -1 "
                    "(pool > L2)", "active_slots": active, "avg_launch_us": us,
        "algorithmic_bytes_per_launch": ub, "achieved_gbs": ub / (us / 1e6) / 1e9,
        "peak_gbs": hbm_peak, "frac": ub / (us / 1e6) / 1e9 / hbm_peak,
        "peak_kind": f"{peak_kind} hbm copy"}
    # the batch sweep of the decode workload (1, 32, 128 and 256 requests, 10 % of the rows
    # -1): one graph-replayed call after each L2 flush, so that small batches, whose states
    # would otherwise stay in L2 from one call to the next, read and write HBM
    l2 = L2Flush(torch, dev)
    sweep = {}
    for b in (1, 32, 128, 256):
        ib = I.padded_permutation(S, b, seed=3000 + b)
        ubi = I.make_update_inputs(1, ib, H, P, G, N, act="bf16", seed=3100 + b,
                                   pool_values=np.zeros((1, H, P, N), np.float32))
        ab = (pool, torch.from_numpy(ib).to(dev), T_(ubi.x), T_(ubi.dt), T_(ubi.A), T_(ubi.B),
              T_(ubi.C))
        kwb = dict(D=T_(ubi.D), dt_bias=T_(ubi.dt_bias))
        ssd.state_update(*ab, **kwb)
        g = graph_of(torch, lambda: ssd.state_update(*ab, **kwb))
        ts = []
        for _ in range(11):
            l2.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        usb = float(np.median(ts))
        act = int((ib >= 0).sum())
        byb = update_bytes(act, b, H, P, G, N)
        sweep[str(b)] = {"active_slots": act, "us": usb, "achieved_gbs": byb / (usb / 1e6) / 1e9,
                         "frac": byb / (usb / 1e6) / 1e9 / hbm_peak}
    res["decode_state_update_sweep"] = {
        "workload": "512-slot pool of [128,64,128] fp32 states, batch 1 / 32 / 128 / 256, 10% "
                    "rows -1; each call graph-replayed after an L2 flush (latency of one call, "
                    "launch included)", "by_batch": sweep, "peak_kind": f"{peak_kind} hbm copy"}
    # decode layer step (update + D + gated norm, 8 norm groups of 1024) on the same
    # pool and batch, against the two calls made separately
    z = torch.randn((batch, H * P), device=dev).to(torch.bfloat16)
    wn = (1 + 0.1 * torch.randn(H * P, device=dev)).to(torch.bfloat16)
    yb = torch.empty((batch, H, P), dtype=torch.bfloat16, device=dev)

    def timed(fn, n=iters):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) * 1e3 / n

    us_f = timed(lambda: ssd.decode_layer_step(*args, z, wn, group_size=1024, **kw))
    us_s = timed(lambda: ssd.gated_rmsnorm(ssd.state_update(*args, y=yb, **kw).view(batch, H * P),
                                           z, wn, group_size=1024))
    lb = ub + batch * H * P * 2 * 3 + H * P * 2  # + y read back, z in, out written
    res["decode_layer_step"] = {
        "workload": "update + D + gated RMSNorm (8 groups of 1024) in one call, batch 256 on "
                    "the 512-slot pool", "avg_launch_us": us_f, "separate_calls_us": us_s,
        "algorithmic_bytes_per_launch": lb, "achieved_gbs": lb / (us_f / 1e6) / 1e9,
        "frac": lb / (us_f / 1e6) / 1e9 / hbm_peak, "peak_kind": f"{peak_kind} hbm copy"}
    # multi-token update: 4 draft tokens for 64 requests, keeping every per-token state
    ntok, bm = 4, 64
    mi = I.padded_permutation(S, bm, seed=3200)
    mu = I.make_update_inputs(1, mi, H, P, G, N, act="bf16", seed=3210, ntok=ntok,
                              pool_values=np.zeros((1, H, P, N), np.float32))
    inter = torch.empty((bm, ntok, H, P, N), device=dev)
    margs = (pool, torch.from_numpy(mi).to(dev), T_(mu.x), T_(mu.dt), T_(mu.A), T_(mu.B),
             T_(mu.C))
    us_m = timed(lambda: ssd.state_update_multi(*margs, D=T_(mu.D), dt_bias=T_(mu.dt_bias),
                                                inter_states=inter))
    act_m = int((mi >= 0).sum())
    mb = act_m * H * P * N * 4 * (2 + ntok) + bm * ntok * (4 * H * P + 4 * G * N + 4 * H)
    mb_write = act_m * H * P * N * 4 * (1 + ntok) + bm * ntok * 2 * H * P
    # the HBM write-only rate on this GPU: a 1 GiB zero fill (torch's fill kernel), the
    # floor of a write-heavy kernel such as this one (5 of its 6 state passes are writes)
    wbuf = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    us_w = timed(lambda: wbuf.zero_())
    write_gbs = (1 << 30) / (us_w / 1e6) / 1e9
    del wbuf
    res["hbm_write_floor"] = {
        "workload": "1 GiB zero fill (write only), back to back", "avg_launch_us": us_w,
        "achieved_gbs": write_gbs, "frac_of_copy_peak": write_gbs / hbm_peak}
    res["state_update_multi"] = {
        "workload": "4 tokens per request, 64 requests (10% rows -1) on the 512-slot pool, "
                    "state after every token kept", "avg_launch_us": us_m,
        "algorithmic_bytes_per_launch": mb, "achieved_gbs": mb / (us_m / 1e6) / 1e9,
        "frac": mb / (us_m / 1e6) / 1e9 / hbm_peak, "peak_kind": f"{peak_kind} hbm copy",
        "written_bytes_per_launch": mb_write,
        "write_time_at_floor_us": mb_write / (write_gbs * 1e9) * 1e6,
        "frac_of_write_floor": (mb_write / (write_gbs * 1e9) * 1e6) / us_m}
    # slot copy: 64 states of 4 MiB into a snapshot pool
    snap = torch.empty((64, H, P, N), device=dev)
    ci = torch.from_numpy(I.padded_permutation(S, 64, seed=3300)).to(dev).abs()
    co = torch.arange(64, dtype=torch.int32, device=dev)
    us_c = timed(lambda: ssd.state_copy(pool, ci, snap, co))
    cb = 64 * H * P * N * 4 * 2
    res["state_copy"] = {
        "workload": "64 slots of [128,64,128] fp32 copied pool -> snapshot pool",
        "avg_launch_us": us_c, "algorithmic_bytes_per_launch": cb,
        "achieved_gbs": cb / (us_c / 1e6) / 1e9, "frac": cb / (us_c / 1e6) / 1e9 / hbm_peak,
        "peak_kind": f"{peak_kind} hbm copy"}
    del pool, args, inter, snap
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_scan(s, **kw):
        """Average device time of one chunk_scan call on workload s (inputs resident)."""
        tens = [T_(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D, s.dt_bias, s.initial_states)]
        x, dt, A, B, C, Dp, bias, init = tens
        hi = torch.from_numpy(s.has_initial_state).to(dev)
        cu = torch.from_numpy(s.cu_seqlens).to(dev)
        y = torch.empty_like(x)
        fs = torch.empty((s.nseq, s.H, s.P, s.N), dtype=torch.float32, device=dev)
        nws = ssd.chunk_scan_workspace_size(x, B, C, cu_seqlens=cu, chunk_size=s.chunk_size,
                                            seg_chunks=kw.get("seg_chunks", 0))
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)

        def run():
            ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=s.chunk_size, D=Dp,
                           dt_bias=bias, initial_states=init, has_initial_state=hi, y=y,
                           final_states=fs, workspace=ws, **kw)

        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(iters):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / iters, nws > 0

    # one long sequence on few heads: the case sequence splitting is for
    s = I.scan_workload("mamba2_130m", seqlens=[16384])
    us, split = time_scan(s)
    us1, _ = time_scan(s, seg_chunks=-1)
    sb = scan_bytes(s.T, s.H, s.P, s.G, s.N, s.nseq)
    res["scan_single_16384"] = {
        "workload": "one 16384-token sequence, H=24 P=64 G=1 N=128, chunk 256",
        "tokens_per_s": s.T / (us / 1e6), "avg_launch_us": us, "split_into_segments": split,
        "unsplit_us": us1, "achieved_gbs": sb / (us / 1e6) / 1e9,
        "frac_hbm": sb / (us / 1e6) / 1e9 / hbm_peak}
    res.update(measure_layer_nemotron_h(torch, ssd, dev, hbm_peak, peak_kind))
    return res


def measure_layer_nemotron_h(torch, ssd, dev, hbm_peak, peak_kind, iters=5):
    """The prefill layer path (ssd_chunk_scan_gated_norm: scan + D skip + gated RMSNorm in
    8 groups of 1024) at Nemotron-H shapes: single sequences of 1K..64K tokens, and a mixed
    batch of 64 packed prefills of 128..4096 tokens with the decode update of 256 pooled
    slots on a second stream.  Inputs are drawn on the device with torch's seeded generator
    in the layer's distributions (tens of GB of values: too slow to draw on the host)."""
    H, P, G, N = 128, 64, 8, 128
    d = H * P
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    l2 = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    res = {}

    def bf(t):
        return t.to(torch.bfloat16)

    def params():
        u = torch.rand(H, generator=gen, device=dev) * (0.1 - 1e-3) + 1e-3
        A = -torch.exp(torch.rand(H, generator=gen, device=dev) * math.log(16.0))
        return torch.log(torch.expm1(u)), A, torch.randn(H, generator=gen, device=dev)

    def inputs(T):
        return dict(x=bf(torch.randn((T, H, P), generator=gen, device=dev)),
                    dt=torch.randn((T, H), generator=gen, device=dev),
                    B=bf(torch.randn((T, G, N), generator=gen, device=dev) / math.sqrt(N)),
                    C=bf(torch.randn((T, G, N), generator=gen, device=dev) / math.sqrt(N)),
                    z=bf(torch.randn((T, d), generator=gen, device=dev)))

    bias, A, Dp = params()
    wn = bf(1 + 0.1 * torch.randn(d, generator=gen, device=dev))

    def layer_call(i, cu, nseq, out, fs, ws, st=None):
        ssd.chunk_scan_gated_norm(i["x"], i["dt"], A, i["B"], i["C"], i["z"], wn, cu_seqlens=cu,
                                  chunk_size=128, group_size=1024, eps=1e-5, D=Dp,
                                  dt_bias=bias, out=out, final_states=fs, workspace=ws,
                                  stream=st)

    def prepare(lens):
        T = int(sum(lens))
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
        i = inputs(T)
        out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        fs = torch.empty((len(lens), H, P, N), dtype=torch.float32, device=dev)
        # the call's workspace: the overlapped form's (its split's, if any, then the ready
        # counters), or the split of the chained form's scan, or none
        nws = ssd.chunk_scan_gated_norm_workspace_size(i["x"], i["B"], i["C"], i["z"], wn, out,
                                                       cu_seqlens=cu, chunk_size=128,
                                                       group_size=1024)
        split = ssd.chunk_scan_workspace_size(i["x"], i["B"], i["C"], cu_seqlens=cu,
                                              chunk_size=128)
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
        counters = (((T + 127) // 128 + len(lens)) * (d // 1024) * 4 + 16 + 255) // 256 * 256
        if nws > 0 and nws != split:
            form = "overlapped" if nws == counters else "overlapped, split"
        else:
            form = "chained, split" if split > 0 else "chained"
        return T, cu, i, out, fs, ws, form

    def timed_flushed(fn, n=iters):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(n):
            l2.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return float(np.median(ts))

    single = {}
    for L in (1024, 4096, 16384, 65536):
        T, cu, i, out, fs, ws, form = prepare([L])
        us = timed_flushed(lambda: layer_call(i, cu, 1, out, fs, ws))
        lb = layer_bytes(T, H, P, G, N, 1)
        single[str(L)] = {"us": us, "tokens_per_s": T / (us / 1e6), "form": form,
                          "achieved_gbs": lb / (us / 1e6) / 1e9,
                          "frac_hbm": lb / (us / 1e6) / 1e9 / hbm_peak}
        del i, out, fs, ws
    res["layer_nemotron_h_single_sequence"] = {
        "workload": "one sequence of L tokens, H=128 P=64 G=8 N=128, chunk 128: scan + D skip + "
                    "gated RMSNorm (8 groups of 1024) in one call, L2 flushed between calls",
        "algorithmic_bytes": "x, z, out 2HP + B, C 2GN + dt 4H per token (y not counted)",
        "peak_kind": f"{peak_kind} hbm copy", "by_L": single}

    # mixed: 64 packed prefills + a 256-slot decode update on a second stream
    lens = np.random.default_rng(4243).integers(128, 4097, size=64)
    T, cu, i, out, fs, ws, form = prepare(lens)
    S = 256
    pool = torch.randn((S, H, P, N), generator=gen, device=dev)
    idx = torch.randperm(S, generator=gen, device=dev).to(torch.int32)
    ux = bf(torch.randn((S, H, P), generator=gen, device=dev))
    udt = torch.randn((S, H), generator=gen, device=dev)
    uB = bf(torch.randn((S, G, N), generator=gen, device=dev) / math.sqrt(N))
    uC = bf(torch.randn((S, G, N), generator=gen, device=dev) / math.sqrt(N))
    uy = torch.empty((S, H, P), dtype=torch.bfloat16, device=dev)
    s_dec = torch.cuda.Stream(device=dev)

    def decode(st):
        ssd.state_update(pool, idx, ux, udt, A, uB, uC, D=Dp, dt_bias=bias, y=uy, stream=st)

    def mixed():
        s_dec.wait_stream(stream)
        decode(s_dec)
        layer_call(i, cu, len(lens), out, fs, ws, st=stream)
        stream.wait_stream(s_dec)

    us_mixed = timed_flushed(mixed)
    us_prefill = timed_flushed(lambda: layer_call(i, cu, len(lens), out, fs, ws))
    us_decode = timed_flushed(lambda: decode(stream))
    lb = layer_bytes(T, H, P, G, N, len(lens))
    ub = update_bytes(S, S, H, P, G, N)
    res["layer_nemotron_h_mixed"] = {
        "workload": f"64 packed prefills of 128..4096 tokens ({T} tokens), H=128 P=64 G=8 "
                    "N=128: scan + D skip + gated RMSNorm in one call, and the decode update "
                    "of 256 pooled slots (all active) on a second stream; L2 flushed between "
                    "iterations",
        "wall_us": us_mixed, "tokens_per_s": (T + S) / (us_mixed / 1e6),
        "prefill_alone_us": us_prefill, "decode_alone_us": us_decode,
        "form": form,
        "achieved_gbs": (lb + ub) / (us_mixed / 1e6) / 1e9,
        "frac_hbm": (lb + ub) / (us_mixed / 1e6) / 1e9 / hbm_peak,
        "peak_kind": f"{peak_kind} hbm copy"}
    del i, out, fs, ws, pool, l2
    return res


# ----------------------------------------------------------------------------- oracle

def oracle_step(s, nrm, upd, group, sl=None):
    """The oracle (as it stands) on the step's arithmetic, or on the sequences in slice sl
    of the batch: the scan, the gated norm of the scan's own output, and the decode token
    of those requests from the scan's final states."""
    import oracle

    cu = np.asarray(s.cu_seqlens)
    seqs = range(s.nseq) if sl is None else range(s.nseq)[sl]
    a, b = int(cu[seqs[0]]), int(cu[seqs[-1] + 1])
    lens = [int(cu[i + 1] - cu[i]) for i in seqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tok = slice(a, b)
    seq = slice(seqs[0], seqs[-1] + 1)
    y, fs = oracle.scan_seq(s.x.values[tok], s.dt.values[tok], s.A.values, s.B.values[tok],
                            s.C.values[tok], D=s.D.values, dt_bias=s.dt_bias.values,
                            initial_states=s.initial_states.values[seq],
                            has_initial_state=s.has_initial_state[seq], cu_seqlens=sub_cu)
    T = b - a
    oracle.gated_rmsnorm(y.reshape(T, s.H * s.P), nrm.z.values[tok], nrm.weight.values,
                         group_size=group)
    oracle.state_update(fs, np.arange(len(lens), dtype=np.int32), upd.x.values[seq],
                        upd.dt.values[seq], s.A.values, upd.B.values[seq], upd.C.values[seq],
                        D=s.D.values, dt_bias=s.dt_bias.values)
    return T


def cpu_baseline(s, nrm, w, budget_s=12.0):
    """The oracle as it stands, on the host cores: the same workload's whole step (scan,
    the gated norm of its output, the decode token), repeated while under the time budget
    (at least once)."""
    from mamba2_ssd_state_gb300 import inputs as I

    upd = I.make_update_inputs(s.nseq, list(range(s.nseq)), s.H, s.P, s.G, s.N, act="bf16",
                               seed=w["seed"] + 60)
    cores = os.cpu_count()
    t0 = time.perf_counter()
    reps, toks = 0, 0
    while True:
        toks += oracle_step(s, nrm, upd, w["norm_group"])
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 500:
            break
    el = time.perf_counter() - t0
    return {"value": toks / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} full step(s) of the same workload (scan of the 16384 packed "
                      f"tokens, gated norm of its output, decode of the 4 requests), double "
                      f"precision, OpenMP over (sequence, head)",
            "seconds": el}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from mamba2_ssd_state_gb300 import inputs as I
    from oracle import build as ob

    ob.build()
    w = I.WORKLOADS[WORKLOAD]
    s = I.scan_workload(WORKLOAD)
    nrm = I.make_norm_inputs(s.T, s.H * s.P, w["norm_group"], act="bf16", seed=w["seed"] + 50)
    upd = I.make_update_inputs(s.nseq, list(range(s.nseq)), s.H, s.P, s.G, s.N, act="bf16",
                               seed=w["seed"] + 60)
    # bounded sample per step: sequences 1 and 2 of the batch (3000 + 517 tokens, all 128
    # heads; sequence 2 with its initial state) through scan, gated norm and decode
    sl = slice(1, 3)

    def step():
        return oracle_step(s, nrm, upd, w["norm_group"], sl)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        toks += step()
    el = time.perf_counter() - t0
    v = toks / el
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Nemotron-H-shaped varlen prefill layer (sequences 1 and 2 "
                                   "of the [8192, 3000, 517, 4675] batch per step: 3517 tokens, "
                                   "H=128 P=64 G=8 N=128), scan + gated RMSNorm (8 groups of "
                                   "1024) + decode of those 2 requests"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "sequences 1 and 2 (3517 tokens) of the batch per step"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_only(args):
    """Launch one op on its benchmark workload warmup + steps times, nothing else."""
    import torch

    from mamba2_ssd_state_gb300 import build as lib_build
    from mamba2_ssd_state_gb300 import inputs as I
    from mamba2_ssd_state_gb300 import ssd

    lib_build.build()
    dev = torch.device("cuda", 0)

    def T_(t):
        dtype = torch.bfloat16 if t.dtype == "bf16" else torch.float32
        return torch.from_numpy(np.ascontiguousarray(t.values)).to(dev, dtype)

    if args.profile in ("scan", "scan_large", "scan_split", "norm", "norm_large", "layer_16k"):
        name = ("mamba2_130m" if args.profile in ("scan", "norm", "scan_split")
                else "nemotron_h_varlen")
        # scan_split: one 16384-token sequence, which the planner cuts into segments;
        # layer_16k: one Nemotron-H-shaped sequence of 16384 tokens through the scan + norm
        # call (the form the layer sweep times)
        if args.profile == "scan_split":
            s = I.scan_workload(name, seqlens=[16384])
        elif args.profile == "layer_16k":
            s = I.scan_workload(name, seqlens=[16384], init="all")
        else:
            s = I.scan_workload(name)
        x, dt, A, B, C, Dp, bias, init = (T_(t) for t in (s.x, s.dt, s.A, s.B, s.C, s.D,
                                                            s.dt_bias, s.initial_states))
        hi = torch.from_numpy(s.has_initial_state).to(dev)
        cu = torch.from_numpy(s.cu_seqlens).to(dev)
        y = torch.empty_like(x)
        fs = torch.empty((s.nseq, s.H, s.P, s.N), dtype=torch.float32, device=dev)
        if args.profile == "layer_16k":
            w = I.WORKLOADS[name]
            nrm = I.make_norm_inputs(s.T, s.H * s.P, w["norm_group"], act="bf16", seed=w["seed"] + 50)
            z, wt = T_(nrm.z), T_(nrm.weight)
            out = torch.empty((s.T, s.H * s.P), dtype=torch.bfloat16, device=dev)
            nws = ssd.chunk_scan_gated_norm_workspace_size(x, B, C, z, wt, out, cu_seqlens=cu,
                                                           chunk_size=s.chunk_size,
                                                           group_size=w["norm_group"])
            ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
            run = lambda: ssd.chunk_scan_gated_norm(  # noqa
                x, dt, A, B, C, z, wt, cu_seqlens=cu, chunk_size=s.chunk_size,
                group_size=w["norm_group"], D=Dp, dt_bias=bias, initial_states=init,
                has_initial_state=hi, final_states=fs, out=out, workspace=ws)
        elif args.profile in ("norm", "norm_large"):
            w = I.WORKLOADS[name]
            nrm = I.make_norm_inputs(s.T, s.H * s.P, w["norm_group"], act="bf16", seed=w["seed"] + 50)
            z, wt = T_(nrm.z), T_(nrm.weight)
            out = torch.empty((s.T, s.H * s.P), dtype=torch.bfloat16, device=dev)
            run = lambda: ssd.gated_rmsnorm(y.view(s.T, -1), z, wt, group_size=w["norm_group"],  # noqa
                                            out=out)
        else:
            run = lambda: ssd.chunk_scan(x, dt, A, B, C, cu_seqlens=cu, chunk_size=s.chunk_size,  # noqa
                                         D=Dp, dt_bias=bias, initial_states=init,
                                         has_initial_state=hi, y=y, final_states=fs)
    else:
        # a 96-slot pool (384 MiB, larger than L2) keeps a multi-pass capture small
        H, P, G, N, S, batch = 128, 64, 8, 128, 96, 96
        if args.profile == "multi":
            batch = 48
        idx = I.padded_permutation(S, batch, seed=3000 + batch)
        ntok = 4 if args.profile == "multi" else None
        u = I.make_update_inputs(1, idx, H, P, G, N, act="bf16", seed=3100 + batch,
                                 pool_values=np.zeros((1, H, P, N), np.float32), ntok=ntok)
        pool = torch.randn((S, H, P, N), device=dev, dtype=torch.float32)
        a = (pool, torch.from_numpy(idx).to(dev), T_(u.x), T_(u.dt), T_(u.A), T_(u.B), T_(u.C))
        if args.profile == "multi":   # 4 tokens per request, per-token states kept
            inter = torch.empty((batch, 4, H, P, N), device=dev)
            run = lambda: ssd.state_update_multi(*a, D=T_(u.D), dt_bias=T_(u.dt_bias),  # noqa
                                                 inter_states=inter)
        elif args.profile == "copy":  # 32 slots into a snapshot pool
            snap = torch.empty((32, H, P, N), device=dev)
            si = torch.arange(0, 64, 2, dtype=torch.int32, device=dev)
            di = torch.arange(32, dtype=torch.int32, device=dev)
            run = lambda: ssd.state_copy(pool, si, snap, di)  # noqa
        else:
            run = lambda: ssd.state_update(*a, D=T_(u.D), dt_bias=T_(u.dt_bias))  # noqa
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    print(f"profile {args.profile}: {args.warmup + args.steps} launches done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-extra", action="store_true", help="skip the decode / large-scan legs")
    ap.add_argument("--profile", choices=["scan", "scan_large", "scan_split", "norm", "norm_large",
                                          "layer_16k", "update", "multi", "copy"],
                    help="only launch this op's benchmark workload steps times (for ncu)")
    args = ap.parse_args()
    if args.profile:
        profile_only(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
