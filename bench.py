#!/usr/bin/env python3
"""Benchmark: GDN chunk forward on B4 T4096 H16 d128 C64, bf16, one GB300 per rank.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one gdn_chunk_fwd call over the whole workload.  That is the
whole hot path: gate prefix, beta-scaled masked K K^T, the UT solve, the WY
products, the serial state pass and the output.  The default (auto) path is
two launches per call: the per-chunk kernel over all SMs, then the state
kernel.
Inputs are seeded and synthetic, drawn by gated_delta_rule_gdn_gb300.workloads.

* value: tokens/s (B*T per step).  Inputs are resident in HBM and timed with
  CUDA events around each launch.  Before each timed step a 256 MiB device
  write flushes L2; the flush is outside the events.
* e2e: the same metric through the public API, from pinned host buffers.
  Every step copies the inputs host->device, runs the call, and copies o and
  the final state device->host.  Batched workloads pipeline the step per batch
  row (one call per row) on three streams: row b + 1 copies in while row b
  computes and row b - 1 copies out.
* roofline: algorithmic bytes of one call / the mean call time (all of the
  call's launches, on the launching stream), against the measured HBM copy
  bandwidth.  frac counts o in bf16, the survey's count: 1,032 B per
  token-head (q, k, v and o in bf16, g and beta in fp32; KDA 4 d_k more for
  its gate), plus the fp32 state read and write per sequence-head.  The call
  writes o in fp32 (bf16 rounding alone breaks the max-error bound), so
  frac_o_f32 is also given, on 1,288 B per token-head.
* cpu_baseline: the fp64 C oracle on the host cores (rank 0, N = 1).
* --impl reference: the oracle alone, timed as the reference arm.
Workloads 6 and 7 time the chunk backward (gdn_chunk_bwd) on the shapes of
workloads 1 and 3: one step is one backward call (three launches: the
per-chunk prep, the two state walks, the per-chunk gradients).  It is fp32 SIMT arithmetic, so its roofline is the fp32
FMA rate (152 SMs x 128 lanes x 2 flops x 2.07 GHz), against the algorithmic
flops of the chunkwise backward given in _bwd_flops.
Workload 0 (B1 T64 H1 d16 C16, fp32 inputs) runs on the generic fp32 kernel,
workload 8 (B4 T4096 H8 at head size 256) on the head-size-256 tensor-core pair;
their lines take the same form.
With N > 1 (torchrun), every rank runs its own replica: weak scaling, and no
collective on the data path.  A barrier and a max over ranks bracket the
timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunk-fwd tokens/s (B4·T4096·H16·d128 bf16) and % of roofline, 1×GB300"
UNIT = "tokens/s"
WORKLOAD = 1          # index of the workload in gated_delta_rule_gdn_gb300.workloads.CONFIGS (the default)
WORKLOAD_NAMES = {"gdn_prefill_b4_t4096_h16_d128_c64_bf16": 1}
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _metric(w) -> str:
    if WORKLOAD_NAMES.get(w.name) == 1:
        return METRIC
    return f"{w.kind.upper()} chunk-fwd tokens/s ({w.name}) and % of roofline, 1×GB300"


def _alg_bytes(w, o_bytes: int = 2) -> int:
    """Algorithmic HBM bytes of one chunk-forward call over workload w, o counted at o_bytes per element (2: the
    survey's count, o in bf16; 4: o as the call writes it, fp32)."""
    token_heads = w.B * w.T * w.H
    es = 2 if w.dtype == "bf16" else 4
    g_bytes = 4 * w.dk if w.kind == "kda" else 4
    per_token_head = es * (2 * w.dk + w.dv) + o_bytes * w.dv + g_bytes + 4   # q, k, v + o + g + beta
    N = w.n_seqs if w.n_seqs else w.B
    state = 2 * N * w.H * w.dk * w.dv * 4 if w.h0_std > 0 else N * w.H * w.dk * w.dv * 4
    return token_heads * per_token_head + state


# The kernel sources each recorded traffic figure depends on (the files that make the timed kernels' code).
TRAFFIC_SOURCES = {
    "chunk_gdn": ("chunk_gdn_tmem.cu", "chunk_gdn_common.cuh", "chunk_wy_common.cuh", "chunk_common.cuh",
                  "tc_common.cuh", "gate_act.cuh"),
    "chunk_gdn_d256": ("chunk_gdn_d256.cu", "chunk_gdn_common.cuh", "chunk_wy_common.cuh", "chunk_common.cuh",
                       "tc_common.cuh", "gate_act.cuh"),
    "chunk_kda": ("chunk_two_pass.cu", "chunk_wy_common.cuh", "chunk_common.cuh", "tc_common.cuh", "gate_act.cuh"),
    "decode": ("recurrent_step.cu", "gate_act.cuh"),
    "bwd": ("chunk_bwd.cu", "tc_common.cuh"),
    "chunk_generic": ("chunk_generic.cu",),
}


def _traffic_kind(workload: str) -> str:
    if "_f32" in workload:
        return "chunk_generic"
    if "_d256_" in workload:
        return "chunk_gdn_d256"
    if "_bwd_" in workload:
        return "bwd"
    if workload.startswith("decode") or "_decode_" in workload:
        return "decode"
    return "chunk_kda" if workload.startswith("kda") else "chunk_gdn"


def _code_only(src: str) -> str:
    """A CUDA source with its comments and blank lines removed (what a comment edit leaves unchanged)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def sources_sha256(kind: str = "chunk_gdn") -> str:
    """Hash of the kernel sources a recorded ncu traffic figure of this kind depends on (code only: an edit of
    the comments keeps the record)."""
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES[kind]:
        with open(os.path.join(ROOT, "gated_delta_rule_gdn_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def _traffic_for(workload: str):
    """ncu DRAM bytes per call (all launches of one step) for `workload`, if they were captured from the current
    kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[workload]
        ok = rec["sources_sha256"] == sources_sha256(_traffic_kind(workload))
        return int(rec["dram_bytes_per_call"]) if ok else None
    except Exception:
        return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons for one GPU in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 is None or t >= self.t0]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _init_pg(ws: int, backend: str):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Max of a scalar over the ranks of the default process group (identity for one rank)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _oracle_inputs(x, heads):
    import numpy as np
    import torch
    hs = torch.as_tensor(heads)
    arr = {k: np.ascontiguousarray(x[k].index_select(2, hs).to(torch.float64).numpy())
           for k in ("q", "k", "v", "g", "beta")}
    h0 = x["initial_state"]
    arr["h0"] = None if h0 is None else np.ascontiguousarray(h0.index_select(1, hs).to(torch.float64).numpy())
    return arr


def cpu_baseline(x, w, min_seconds=10.0, max_passes=60, heads=None):
    """Time the fp64 oracle on the host cores (bounded sample of the workload); returns a dict."""
    import oracle
    heads = list(range(w.H)) if heads is None else heads
    arr = _oracle_inputs(x, heads)
    oracle.load()
    passes, t_total = 0, 0.0
    while passes < max_passes and (passes == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        oracle.recurrence(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], x["scale"], arr["h0"],
                          x["cu_seqlens"], gate_per_channel=x["gate_per_channel"])
        t_total += time.perf_counter() - t0
        passes += 1
    frac = len(heads) / w.H
    tokens = w.B * w.T * frac * passes
    return {"value": tokens / t_total, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{w.B * len(heads)} (sequence, head) chains of {w.T} tokens ({len(heads)}/{w.H} heads), "
                      f"{passes} pass(es), {t_total:.1f} s; tokens/s scaled to all {w.H} heads"}


def _decode_sample(w, consts, step: int = 0):
    """fp64 oracle inputs of one decode step for every 16th (sequence, head) chain (512 of the 8192)."""
    from gated_delta_rule_gdn_gb300 import workloads as W
    import torch
    NH = w.N * w.H
    sample = torch.arange(0, NH, 16)
    x = W.decode_step_inputs(w, consts, step)
    h0 = consts["state"].reshape(NH, 1, w.dk, w.dv)[sample].to(torch.float64).numpy()
    q, k, v = (x[n].reshape(NH, 1, 1, -1)[sample].to(torch.float64).numpy() for n in ("q", "k", "v"))
    beta = x["beta"].reshape(NH, 1, 1)[sample].to(torch.float64).numpy()
    g = (x["g"].reshape(NH, 1, 1, -1) if w.kind == "kda" else x["g"].reshape(NH, 1, 1))[sample].to(torch.float64).numpy()
    return (q, k, v, g, beta, h0), len(sample), NH


def cpu_baseline_decode(w, consts, min_seconds=10.0, max_passes=2000):
    """Time the fp64 oracle on one decode step of a chain sample, repeated for about min_seconds; tokens/s scaled to
    all chains."""
    import oracle
    (q, k, v, g, beta, h0), n, NH = _decode_sample(w, consts)
    oracle.load()
    passes, t_total = 0, 0.0
    while passes < max_passes and (passes == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        oracle.recurrence(q, k, v, g, beta, w.scale, h0, gate_per_channel=w.kind == "kda")
        t_total += time.perf_counter() - t0
        passes += 1
    dt = t_total / passes * (NH / n)
    return {"value": w.N / dt, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"one decode step for {n} of {NH} (sequence, head) chains, {passes} pass(es), {t_total:.1f} s; "
                      f"time scaled to all chains"}


def run_reference_decode(args):
    """The oracle on a decode step: one token for a sample of the (sequence, head) chains, scaled to all of them."""
    from gated_delta_rule_gdn_gb300 import workloads as W
    import oracle
    import torch
    w = _decode_workload(args.workload)
    consts = W.decode_constants(w, seed=0)
    (q, k, v, g, beta, h0), n_sample, NH = _decode_sample(w, consts)
    sample = range(n_sample)
    oracle.load()
    run = lambda: oracle.recurrence(q, k, v, g, beta, w.scale, h0, gate_per_channel=w.kind == "kda")
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps * (NH / len(sample))
    value = w.N / dt
    line = {"impl": "reference", "metric": f"{w.kind.upper()} decode-step tokens/s ({w.name}) and % of HBM roofline, 1×GB300",
            "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": w.name, "N": w.N, "H": w.H, "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"per step one token for {len(sample)} of {NH} (sequence, head) chains; "
                                       f"time scaled to all chains"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


def run_reference(args):
    ws, rank, local = _dist()
    if ws > 1:
        if rank != 0:
            return 0
    if args.workload in DECODE:
        return run_reference_decode(args)
    from gated_delta_rule_gdn_gb300 import workloads as W
    import oracle
    w = _chunk_workload(args.workload)
    x = W.chunk_inputs(w, seed=0)
    heads = list(range(min(4, w.H)))     # one step = (up to) 4 heads of every sequence
    arr = _oracle_inputs(x, heads)
    oracle.load()
    run = lambda: oracle.recurrence(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], x["scale"], arr["h0"],
                                    x["cu_seqlens"], gate_per_channel=x["gate_per_channel"])
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = w.B * w.T * (len(heads) / w.H) / dt
    line = {"impl": "reference", "metric": _metric(w), "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                       "chunk_size": w.chunk_size},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"per step {w.B * len(heads)} (sequence, head) chains of {w.T} tokens "
                                       f"({len(heads)}/{w.H} heads); tokens/s scaled to all {w.H} heads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


BWD_OF = {6: 1, 7: 3}      # backward workload -> the forward workload it differentiates
DECODE = (4, 5)            # decode-step workloads
HEAD256 = 8                # GDN prefill at head size 256 (generic kernel)
ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def _bwd_name(w) -> str:
    return w.name.replace("_prefill", "").replace("_c64", "").replace(w.kind + "_", w.kind + "_bwd_", 1)


def _bwd_flops(w, C: int) -> int:
    """Algorithmic flops of one chunk-backward call (2 per multiply-add), per chunk of C rows and head:
    the recomputed forward (K K^T and Q K^T: C^2 d_k; Z: C d_k d_v; the solve: C^2 d_v / 2; the state update:
    C d_k d_v), and the backward (dDelta: C d_k d_v + C^2 d_v / 2; the back solve: C^2 d_v / 2; dP and dA: C^2 d_v;
    the state products h dO, h Y, dh Delta: 3 C d_k d_v; the four pair sums of dQ / dK: 2 C^2 d_k; the state
    gradient: 2 C d_k d_v).  Per-channel exponentials are not counted."""
    dk, dv = w.dk, w.dv
    macs = 3 * C * C * dk + 8 * C * dk * dv + 5 * C * C * dv // 2
    N = w.n_seqs if w.n_seqs else w.B
    chunks = N * math.ceil(w.T / C) if not w.n_seqs else math.ceil(w.T / C) + N
    return 2 * macs * chunks * w.H


def _bwd_chains_oracle(x, g, chains):
    """The (b, h) chains for the oracle's backward, stacked as a batch of single-head sequences (the oracle runs its
    chains in parallel over the host cores)."""
    import numpy as np
    sl = lambda t: np.ascontiguousarray(np.concatenate([t[b:b + 1, :, h:h + 1].double().numpy() for b, h in chains]))
    st = lambda t: None if t is None else np.ascontiguousarray(
        np.concatenate([t[b:b + 1, h:h + 1].double().numpy() for b, h in chains]))
    return (sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), sl(g["d_o"]), st(x["initial_state"]),
            st(g["d_final_state"]))


def _bwd_oracle_run(arrs, scale, per_channel):
    import oracle
    q, k, v, gg, beta, do, h0, dhT = arrs
    oracle.recurrence_backward(q, k, v, gg, beta, scale, do, h0, dhT, gate_per_channel=per_channel)


def _bwd_sample(w, n):
    """n (b, h) chains spread over the workload."""
    all_chains = [(b, h) for b in range(w.B) for h in range(w.H)]
    step = max(1, len(all_chains) // n)
    return all_chains[::step][:n]


def cpu_baseline_bwd(x, g, w, min_seconds=10.0, max_passes=60):
    import oracle
    oracle.load()
    chains = _bwd_sample(w, oracle.max_threads())
    arrs = _bwd_chains_oracle(x, g, chains)
    passes, t_total = 0, 0.0
    while passes < max_passes and (passes == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        _bwd_oracle_run(arrs, x["scale"], x["gate_per_channel"])
        t_total += time.perf_counter() - t0
        passes += 1
    tokens = w.T * len(chains) * passes / w.H
    return {"value": tokens / t_total, "unit": UNIT, "cores": min(oracle.max_threads(), len(chains)), "kind": "oracle",
            "sample": f"the oracle's backward on {len(chains)} (sequence, head) chains of {w.T} tokens in one call "
                      f"(one host thread per chain), {passes} pass(es), {t_total:.1f} s; tokens/s scaled to all "
                      f"{w.B * w.H} chains"}


def run_reference_bwd(args):
    """The oracle's backward: per step one chain per host thread, scaled to all chains."""
    from gated_delta_rule_gdn_gb300 import workloads as W
    import oracle
    w = W.config(BWD_OF[args.workload])
    x = W.chunk_inputs(w, seed=0)
    g = W.chunk_output_grads(x, seed=1, dhT_std=0.02)
    oracle.load()
    chains = _bwd_sample(w, oracle.max_threads())
    arrs = _bwd_chains_oracle(x, g, chains)
    for _ in range(args.warmup):
        _bwd_oracle_run(arrs, x["scale"], x["gate_per_channel"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _bwd_oracle_run(arrs, x["scale"], x["gate_per_channel"])
    dt = (time.perf_counter() - t0) / args.steps * (w.B * w.H) / len(chains)
    value = w.B * w.T / dt
    line = {"impl": "reference", "metric": f"{w.kind.upper()} chunk-bwd tokens/s ({_bwd_name(w)}), 1×GB300",
            "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": _bwd_name(w), "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(oracle.max_threads(), len(chains)),
                             "kind": "oracle",
                             "sample": f"per step {len(chains)} (sequence, head) chains of {w.T} tokens in one call, "
                                       f"one host thread each; time scaled to all {w.B * w.H} chains"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


def run_bwd(args):
    """One step = one chunk-backward call over the whole workload (inputs and upstream gradients resident)."""
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _init_pg(ws, "nccl")
    import gated_delta_rule_gdn_gb300 as gdn
    from gated_delta_rule_gdn_gb300 import build as libbuild, workloads as W
    if local == 0:
        libbuild.build()
    barrier(ws)
    gdn.load()
    w = W.config(BWD_OF[args.workload])
    x = W.chunk_inputs(w, seed=0)
    grads = W.chunk_output_grads(x, seed=1, dhT_std=0.02)
    x.update(grads)
    keys = [k for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens", "d_o", "d_final_state")
            if x[k] is not None]
    host = {k: x[k].pin_memory() for k in keys}
    d = {k: v.to(dev) for k, v in host.items()}
    per_channel = w.kind == "kda"
    n_seqs = 0 if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1
    C = 16     # the chunk the library takes by default for d_k <= 256
    ws_bytes = gdn.bwd_workspace_size(per_channel, w.B, w.T, w.H, w.dk, w.dv, C, n_seqs)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(dd):
        return gdn.chunk_bwd(per_channel, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["d_o"], scale=w.scale,
                             initial_state=dd.get("initial_state"), d_final_state=dd.get("d_final_state"),
                             cu_seqlens=dd.get("cu_seqlens"), chunk_size=C, stream=stream, workspace=workspace)

    for _ in range(args.warmup):
        flush.fill_(1)
        call(d)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(int(os.environ.get("GDN_BENCH_GPU_INDEX", local))) if rank == 0 else None
    if sampler:
        sampler.start()
        t_end = time.time() + 1.0
        while time.time() < t_end:
            call(d)
            torch.cuda.synchronize(dev)
        sampler.mark()
    barrier(ws)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record(stream)
        call(d)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs), ws, dev)
    clocks = sampler.stop() if sampler else None

    # end to end: inputs and upstream gradients host -> device, the call, the six gradients device -> host
    dd = {k: torch.empty_like(v) for k, v in d.items()}
    outs = call(d)
    outs_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs if t is not None]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_host)

    def e2e_step():
        for k in dd:
            dd[k].copy_(host[k], non_blocking=True)
        res = [t for t in call(dd) if t is not None]
        for hst, t in zip(outs_host, res):
            hst.copy_(t, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)

    tokens = w.B * w.T
    C_used = C
    flops = _bwd_flops(w, C_used)
    achieved = flops / (ms / 1e3) / 1e12
    line = {
        "metric": f"{w.kind.upper()} chunk-bwd tokens/s ({_bwd_name(w)}) and % of fp32 ALU roofline, 1×GB300",
        "value": tokens * ws / (ms / 1e3), "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; the forward recipe of the workload, dO N(0,1) bf16, dhT N(0,0.02))",
        "config": {"workload": _bwd_name(w), "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "chunk_size": C_used, "input_dtype": "bf16", "grad_dtype": "f32",
                   "l2": "flushed before each timed step (256 MiB device write, outside the events)",
                   "kernel": "chunk_bwd (prep, walks, gradients)", "launches_per_step": 3,
                   "timed_region_wall_ms": t_wall * 1e3},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": ALU_PEAK_TFLOPS, "unit": "TFLOP/s",
                     "frac": achieved / ALU_PEAK_TFLOPS, "traffic": _traffic_for(_bwd_name(w)),
                     "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz",
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": tokens * ws / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * 3,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(x, grads, w)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_ours(args):
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _init_pg(ws, "nccl")
    import gated_delta_rule_gdn_gb300 as gdn
    from gated_delta_rule_gdn_gb300 import build as libbuild, workloads as W
    if local == 0:
        libbuild.build()
    barrier(ws)
    gdn.load()
    w = _chunk_workload(args.workload)
    x = W.chunk_inputs(w, seed=0)
    keys = [k for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens") if x[k] is not None]
    host = {k: x[k].pin_memory() for k in keys}
    d = {k: v.to(dev) for k, v in host.items()}
    N = x["N"]
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.float32, device=dev)
    hT = torch.empty((N, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd = gdn.kda_chunk_fwd if w.kind == "kda" else gdn.gdn_chunk_fwd

    def call(dd, oo, hh):
        fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], scale=w.scale, initial_state=dd.get("initial_state"),
            output_final_state=True, cu_seqlens=dd.get("cu_seqlens"), chunk_size=w.chunk_size, algo=args.algo, o=oo,
            final_state=hh, stream=stream, o_dtype=torch.float32)

    for _ in range(args.warmup):
        flush.fill_(1)
        call(d, o, hT)
    torch.cuda.synchronize(dev)
    assert gdn.device_status() == 0

    sampler = ClockSampler(int(os.environ.get("GDN_BENCH_GPU_INDEX", local))) if rank == 0 else None
    if sampler:
        sampler.start()
        # keep the GPU busy (untimed) while the sampler starts, so clock samples reflect load
        t_end = time.time() + 1.0
        while time.time() < t_end:
            flush.fill_(1)
            call(d, o, hT)
            torch.cuda.synchronize(dev)
        sampler.mark()
    barrier(ws)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record(stream)
        call(d, o, hT)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    launch_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms = max_over_ranks(sum(launch_ms) / len(launch_ms), ws, dev)
    clocks = sampler.stop() if sampler else None
    assert gdn.device_status() == 0

    # end to end through the public API: pinned host -> device, call, device -> host, every step
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h_host = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size() + h_host.numel() * h_host.element_size()
    dd = {k: torch.empty_like(v) for k, v in d.items()}
    o2, h2 = torch.empty_like(o), torch.empty_like(hT)

    # Batched workloads pipeline the step per batch row on three streams (every (row, head) chain is independent):
    # row b + 1 copies in while row b computes and row b - 1 copies out.  Each row is one public-API call.
    rows = w.B if (w.B > 1 and x["cu_seqlens"] is None) else 1
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done_c = [None] * rows   # compute of row b finished (its inputs may be overwritten)
    done_o = [None] * rows   # copy-out of row b finished (its outputs may be overwritten)

    def e2e_step():
        if rows == 1:
            for k in dd:
                dd[k].copy_(host[k], non_blocking=True)
            call(dd, o2, h2)
            o_host.copy_(o2, non_blocking=True)
            h_host.copy_(h2, non_blocking=True)
            return
        for b in range(rows):
            sl = slice(b, b + 1)
            with torch.cuda.stream(s_in):
                if done_c[b] is not None:
                    s_in.wait_event(done_c[b])
                for k in dd:
                    dd[k][sl].copy_(host[k][sl], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            if done_o[b] is not None:
                stream.wait_event(done_o[b])
            call({k: v[sl] for k, v in dd.items()}, o2[sl], h2[sl])
            done_c[b] = torch.cuda.Event()
            done_c[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_c[b])
                o_host[sl].copy_(o2[sl], non_blocking=True)
                h_host[sl].copy_(h2[sl], non_blocking=True)
                done_o[b] = torch.cuda.Event()
                done_o[b].record(s_out)
        stream.wait_event(done_o[rows - 1])

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)

    tokens = w.B * w.T
    value = tokens * ws / (ms / 1e3)
    peak, peak_kind = _peaks()
    f32_in = w.dtype == "f32"
    alg = _alg_bytes(w, 4 if f32_in else 2)     # fp32 inputs: o is fp32 in the survey's count too
    alg32 = _alg_bytes(w, 4)
    achieved = alg / (ms / 1e3) / 1e9
    plan = gdn.chunk_plan(w.kind == "kda", w.B, w.T, w.H, w.dk, w.dv, w.chunk_size,
                          torch.float32 if f32_in else torch.bfloat16,
                          x["cu_seqlens"] is not None, args.algo)
    two_pass = "chunk_two_pass (chunk_intra_kernel, chunk_state_kernel)" if w.kind == "kda" else \
        "chunk_gdn_d256 (gdn_intra256_kernel, gdn_state256_kernel)" if w.dk == 256 else \
        "chunk_gdn_tmem (gdn_intra_kernel, gdn_state_kernel)"
    kernel, launches = {"two_pass": (two_pass, 2)}.get(plan, ("chunk_generic", 1))
    line = {
        "metric": _metric(w), "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32_in else "bf16",
        "data": "synthetic (seeded; q,k unit-norm N(0,1), v N(0,1), beta=sigmoid(N), log alpha=-A softplus(N+dt_bias))",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "chunk_size": w.chunk_size, "initial_state": x["initial_state"] is not None,
                   "output_final_state": True, "n_seqs": N,
                   "o_dtype": "f32",
                   "l2": "flushed before each timed step (256 MiB device write, outside the events)",
                   "kernel": kernel, "launches_per_step": launches, "timed_region_wall_ms": t_wall * 1e3},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _traffic_for(w.name), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6800 GB/s",
                     "algorithmic_bytes_per_launch": alg,
                     "o_bytes_counted": "f32 (fp32 inputs)" if f32_in else "bf16 (the survey's count)",
                     "frac_o_f32": alg32 / (ms / 1e3) / 1e9 / peak, "algorithmic_bytes_o_f32": alg32},
        "e2e": {"value": tokens * ws / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipeline": (f"per batch row ({rows} public-API calls), copies in / compute / copies out on three "
                             "streams") if rows > 1 else "one call; copies in, compute, copies out in order"},
        "gpu_launches": args.steps * launches,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, w)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _chunk_workload(which: int):
    """Chunk-forward workload `which`: 0-3 as listed in workloads.CONFIGS, 8 the head-size-256 prefill."""
    from gated_delta_rule_gdn_gb300 import workloads as W
    return W.HEAD256 if which == HEAD256 else W.config(which)


def _decode_workload(which: int):
    from gated_delta_rule_gdn_gb300 import workloads as W
    w4 = W.config(4)
    if which == 4:
        return w4
    return W.DecodeWorkload("kda_decode_n256_h32_d128", w4.N, w4.H, w4.dk, w4.dv, w4.steps, kind="kda")


def _decode_alg_bytes(w) -> int:
    """Algorithmic HBM bytes of one decode step: the fp32 state read and written, q, k, v (bf16), g, beta, o (fp32)."""
    nh = w.N * w.H
    g_bytes = 4 * w.dk if w.kind == "kda" else 4
    return nh * (2 * w.dk * w.dv * 4 + 2 * (2 * w.dk + w.dv) + g_bytes + 4 + 4 * w.dv)


def run_decode(args):
    """One step = one decode token for every (sequence, head): the state ([N, H, 128, 128] fp32) is read and written
    in place.  Inputs cycle through 8 pre-drawn steps; the 512 MiB state is larger than L2, so no flush is needed."""
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _init_pg(ws, "nccl")
    import gated_delta_rule_gdn_gb300 as gdn
    from gated_delta_rule_gdn_gb300 import build as libbuild, workloads as W
    if local == 0:
        libbuild.build()
    barrier(ws)
    gdn.load()
    w = _decode_workload(args.workload)
    consts = W.decode_constants(w, seed=0)
    state = consts["state"].to(dev)
    host = [W.decode_step_inputs(w, consts, s_) for s_ in range(8)]
    host = [{k: v.pin_memory() for k, v in x.items()} for x in host]
    dev_in = [{k: v.to(dev) for k, v in x.items()} for x in host]
    o = torch.empty((w.N, w.H, w.dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = gdn.kda_recurrent_step if w.kind == "kda" else gdn.gdn_recurrent_step

    def call(x, oo):
        step(x["q"], x["k"], x["v"], x["g"], x["beta"], state, scale=w.scale, o=oo, stream=stream)

    for i in range(args.warmup):
        call(dev_in[i % 8], o)
    torch.cuda.synchronize(dev)
    assert gdn.device_status() == 0
    sampler = ClockSampler(int(os.environ.get("GDN_BENCH_GPU_INDEX", local))) if rank == 0 else None
    if sampler:
        sampler.start()
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for i in range(8):
                call(dev_in[i], o)
            torch.cuda.synchronize(dev)
        sampler.mark()
    barrier(ws)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for i, (e0, e1) in enumerate(evs):
        e0.record(stream)
        call(dev_in[i % 8], o)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs), ws, dev)
    clocks = sampler.stop() if sampler else None
    assert gdn.device_status() == 0
    # end to end: each step's inputs host -> device, the call, o device -> host (the state stays resident)
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    dd = {k: torch.empty_like(v) for k, v in dev_in[0].items()}
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = o_host.numel() * o_host.element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        for k in dd:
            dd[k].copy_(host[i % 8][k], non_blocking=True)
        call(dd, o)
        o_host.copy_(o, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    tokens = w.N
    peak, peak_kind = _peaks()
    alg = _decode_alg_bytes(w)
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": f"{w.kind.upper()} decode-step tokens/s ({w.name}) and % of HBM roofline, 1×GB300",
        "value": tokens * ws / (ms / 1e3), "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k unit-norm, v N(0,1), beta=sigmoid(N), gates as the chunk recipes)",
        "config": {"workload": w.name, "N": w.N, "H": w.H, "dk": w.dk, "dv": w.dv, "o_dtype": "f32",
                   "l2": "not flushed: the 512 MiB state read and written every step is larger than L2",
                   "kernel": "recurrent_step", "timed_region_wall_ms": t_wall * 1e3},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _traffic_for(w.name), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6800 GB/s", "algorithmic_bytes_per_step": alg},
        "e2e": {"value": tokens * ws / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w, consts)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", choices=["auto", "generic", "two_pass"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", type=int, choices=[0, 1, 2, 3, 4, 5, 6, 7, 8], default=WORKLOAD,
                    help="0: GDN B1 T64 H1 d16 C16 fp32 (tiny), 1: GDN B4 T4096 H16 (the headline), 2: packed GDN 8 "
                         "seqs 65536 tokens H32, 3: KDA B2 T8192 H32, 4: GDN decode step 256 seqs H32, 5: KDA decode "
                         "step 256 seqs H32, 6: GDN chunk backward B4 T4096 H16, 7: KDA chunk backward B2 T8192 H32, "
                         "8: GDN B4 T4096 H8 at head size 256")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.workload in BWD_OF:
            ws, rank, _ = _dist()
            return 0 if ws > 1 and rank != 0 else run_reference_bwd(args)
        return run_reference(args)
    if args.workload in BWD_OF:
        return run_bwd(args)
    if args.workload in DECODE:
        return run_decode(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
