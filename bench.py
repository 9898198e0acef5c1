#!/usr/bin/env python3
"""Weight-stream benchmark of the groupwise-quantized small-T GEMV on GB300.

Workload: the per-token MLP + head weight stream of a 64-layer Qwen3.8-27B-
shaped model -- per layer a fused gate+up GEMV (4-bit, K=5120, N=34816) and a
down GEMV (K=17408, N=5120; 5-bit for layers 0-35, 4-bit for 36-63), then the
6-bit output head (K=5120, N=248320) -- run at T = 1, 4, 8 and 16 tokens.
Weights are seeded N(0, 0.02) draws encoded round-to-nearest on the device;
x is seeded N(0, 1) in bf16.  A step is one pass over the whole stack at each
T (4 x 129 GEMVs, 41.9 GB of packed weights), inputs resident in HBM.

The GEMVs of a pass are independent (no activation between them), so each
pass is grouped by tensor kind: the 64 gate+up GEMVs, the 36 5-bit and the 28
4-bit down GEMVs, the head; each group is one CUDA graph, and CUDA events
between the groups give the duration of each kind inside the timed region
(mean, median and minimum over the timed steps).

After timing, every graph is replayed once more per T and sampled rows of the
outputs it wrote (the last GEMV of the group) are compared with the CPU oracle
on the same weights and x; a mismatch fails the run.  The oracle is also timed
on the host cores (one core, and every core of the process's affinity mask).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (fp64)
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

# The CPU oracle runs one BLAS thread per process; fix it before numpy loads
# (spawned worker processes inherit the setting).
import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import multiprocessing
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HIDDEN, INTER, VOCAB, LAYERS, Q5_LAYERS = 5120, 17408, 248320, 64, 36
TS = (1, 4, 8, 16)
KINDS = ("gate_up", "down_q5", "down_q4", "head")
METRIC = "quantized GEMV weight-stream GB/s and % of GB300 HBM peak, T=1/8/16"
UNIT = "GB/s"


def stack_tensors():
    """(kind, layer, bits, K, N) of every GEMV of one pass."""
    out = []
    for l in range(LAYERS):
        out.append(("gate_up", l, 4, HIDDEN, 2 * INTER))
    for l in range(LAYERS):
        out.append(("down_q5" if l < Q5_LAYERS else "down_q4", l, 5 if l < Q5_LAYERS else 4,
                    INTER, HIDDEN))
    out.append(("head", 0, 6, HIDDEN, VOCAB))
    return out


def packed_bytes(bits, K, N):
    """Algorithmic bytes of one weight stream: packed codes + FP16 scales."""
    return N * K // 64 * (8 * bits + 2)


PASS_BYTES = sum(packed_bytes(b, K, N) for (_, _, b, K, N) in stack_tensors())
KIND_BYTES = {k: sum(packed_bytes(b, K, N) for (kk, _, b, K, N) in stack_tensors() if kk == k)
              for k in KINDS}
KIND_COUNT = {k: sum(1 for e in stack_tensors() if e[0] == k) for k in KINDS}
CONFIG = {
    "workload": "64-layer Qwen3.8-27B-shaped MLP+head weight stream: per layer gate+up Q4 "
                "5120x34816 and down 17408x5120 (Q5 layers 0-35, Q4 36-63), then the Q6 head "
                "5120x248320; T=1/4/8/16; group 64, FP16 scales",
    "T": list(TS),
    "weight_bytes_per_pass": PASS_BYTES,
    "l2": "inputs larger than L2 (10.49 GB of distinct packed weights per pass, L2 129 MB)",
    "launch": "one CUDA graph per tensor kind and T, programmatic dependent launch",
}
# Rows of the last tensor of each kind whose outputs are checked against the
# oracle (and on which the oracle is timed).
CHECK_ROWS = {"gate_up": 96, "down_q5": 24, "down_q4": 24, "head": 64}


def source_hash() -> str:
    """Hash of the kernel sources, to tell whether stored ncu counters still apply."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_weight_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def stored_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None if absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "gemv_gate_up_q4_T1_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_hash") != source_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ("active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        reasons = set()
        for _, _, flags in rows:
            for n, f in zip(names[1:], flags[1:]):
                if f.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ multi-rank helpers
def max_over_ranks(value: float, device=None) -> float:
    """The maximum of a per-rank float over the default process group; the
    value itself when no group is initialised (N = 1)."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, steps: int, bytes_per_step: int, ms: float) -> float:
    """Whole-job throughput: every rank streams ``bytes_per_step`` per step
    (replicas, weak scaling), divided by the slowest rank's time."""
    return world * steps * bytes_per_step / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ CPU oracle leg
SAMPLE_ROWS = {"gate_up": (4, HIDDEN, 96), "down": (5, INTER, 16), "head": (6, HIDDEN, 64)}


def oracle_sample(seconds: float, seed: int = 77):
    """Time the CPU oracle (fp64, this process, one BLAS thread) on sampled rows
    of the same workload: rows of the gate+up, down and head tensors at T = 1,
    4, 8, 16, in proportion to their bytes.  Returns (GB/s of packed-weight
    bytes, bytes, seconds, description)."""
    import oracle
    import synth
    prepared = []
    for i, (kind, (bits, K, n)) in enumerate(SAMPLE_ROWS.items()):
        rng = synth.generator(seed, 700 + i)
        w = synth.gauss_weights(rng, n, K)
        codes, sb = oracle.rtn_encode(w, bits)
        xs = {T: synth.gauss_x_bf16(rng, T, K) for T in TS}
        prepared.append((kind, bits, K, n, codes, sb, xs))
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        for (kind, bits, K, n, codes, sb, xs) in prepared:
            for T in TS:
                oracle.gemv(codes, sb, xs[T])
                done_bytes += packed_bytes(bits, K, n)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    desc = (f"oracle.gemv (fp64 numpy, one BLAS thread per process) on rounds of sampled rows "
            f"(gate+up 96 rows, down 16 rows, head 64 rows) at T=1,4,8,16")
    return done_bytes / el / 1e9, done_bytes, el, desc


def _oracle_worker(args):
    seconds, seed = args
    _, nbytes, el, _ = oracle_sample(seconds, seed)
    return nbytes, el


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pool():
    """One spawned worker process per core of the affinity mask (each with one
    BLAS thread); spawned, not forked, so a process that uses the GPU can
    start it."""
    n = host_cores()
    return multiprocessing.get_context("spawn").Pool(n), n


def oracle_all_cores(pool, n: int, seconds: float, seed: int = 77):
    """The sample on every worker at once, each timed over `seconds`.
    Returns (bytes summed over the workers, the slowest worker's seconds)."""
    res = pool.map(_oracle_worker, [(seconds, seed + i) for i in range(n)])
    return sum(b for b, _ in res), max(e for _, e in res)


def cpu_baseline(seconds: float):
    single, _, _, desc = oracle_sample(seconds)
    pool, n = oracle_pool()
    with pool:
        oracle_all_cores(pool, n, 0.2)                      # workers started and warm
        nbytes, el = oracle_all_cores(pool, n, seconds)
    return {"value": round(nbytes / el / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": desc + f"; {seconds:.1f} s on every core (one process each)",
            "single_core": {"value": round(single, 4), "cores": 1}}


def run_reference(args, rank):
    if rank != 0:
        return
    per_step = max(0.5, args.ref_step_seconds)
    pool, n = oracle_pool()
    with pool:
        for _ in range(args.warmup):
            oracle_all_cores(pool, n, per_step / 4)
        t0 = time.perf_counter()
        total_bytes = 0
        for _ in range(args.steps):
            nbytes, _ = oracle_all_cores(pool, n, per_step)
            total_bytes += nbytes
        el = time.perf_counter() - t0
    value = total_bytes / el / 1e9
    _, _, _, desc = oracle_sample(0.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": CONFIG,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": desc + f"; {per_step:.1f} s per step on every core "
                                          "(one process each)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg
def build_stack(torch, nqp, dev, seed):
    """Packed weights of every tensor, x arena (16 tokens per GEMV), y buffers;
    the fp32 rows of each kind's last tensor that the oracle check uses."""
    entries = []
    rng = np.random.default_rng(seed + 12345)
    last = {k: max(i for i, e in enumerate(stack_tensors()) if e[0] == k) for k in KINDS}
    for idx, (kind, layer, bits, K, N) in enumerate(stack_tensors()):
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1000003 + idx)
        w = torch.randn((N, K), generator=g, device=dev, dtype=torch.float32)
        w.mul_(0.02)
        qw = nqp.QuantizedWeight.from_fp32(w, bits)
        e = {"kind": kind, "layer": layer, "bits": bits, "K": K, "N": N, "qw": qw}
        if idx == last[kind]:
            rows = np.unique(np.concatenate([[0, 15, N - 1], rng.choice(N, CHECK_ROWS[kind], replace=False)]))
            e["check_rows"] = rows
            e["check_w"] = w[torch.from_numpy(rows).to(dev)].cpu().numpy()
        del w
        entries.append(e)
    torch.cuda.synchronize()
    rc = nqp.last_device_error()
    if rc != 0:
        raise RuntimeError(f"device status {rc} while preparing weights")
    # x arena: 16 tokens per GEMV, seeded N(0,1) rounded to bf16
    offs, tot = [], 0
    for e in entries:
        offs.append(tot)
        tot += 16 * e["K"]
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7919 + 1)
    x_arena = torch.randn(tot, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    for e, o in zip(entries, offs):
        e["x"] = x_arena[o:o + 16 * e["K"]].view(16, e["K"])
    ys = {k: torch.empty((16, n), dtype=torch.float32, device=dev)
          for k, n in (("gate_up", 2 * INTER), ("down_q5", HIDDEN), ("down_q4", HIDDEN),
                       ("head", VOCAB))}
    return entries, x_arena, ys


def capture(torch, nqp, entries, ys, T, kind, stream):
    sel = [e for e in entries if e["kind"] == kind]

    def run():
        for e in sel:
            nqp.gemv(e["qw"].packed, e["qw"].scales, e["x"][:T], ys[kind][:T], e["K"], e["N"], T,
                     e["bits"], stream=stream)
    with torch.cuda.stream(stream):
        run()                                     # plans cached, attributes set
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    return g, len(sel)


def check_outputs(torch, nqp, entries, ys, graphs, stream):
    """Replay every graph once per T and compare sampled rows of the output it
    wrote (its last GEMV) with the oracle on the same fp32 weights and x.
    Returns {kind_T: largest tolerance ratio} (<= 1 passes)."""
    import oracle
    out = {}
    for e in entries:
        if "check_rows" not in e:
            continue
        codes, sb = oracle.rtn_encode(e["check_w"], e["bits"])
        xb = e["x"].view(torch.int16).cpu().numpy().view(np.uint16)
        for T in TS:
            ys[e["kind"]].fill_(float("nan"))
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                graphs[(T, e["kind"])].replay()
            torch.cuda.synchronize()
            y = ys[e["kind"]][:T].cpu().numpy()[:, e["check_rows"]]
            y_ref, e_ref = oracle.gemv(codes, sb, xb[:T])
            out[f"{e['kind']}_T{T}"] = round(oracle.max_violation(y, y_ref, e_ref), 6)
    rc = nqp.last_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} in the output check")
    return out


def _graph_us(torch, stream, run, reps):
    """Average microseconds of `run` captured into one CUDA graph, replayed
    `reps` times back to back on `stream` (one warm replay first)."""
    with torch.cuda.stream(stream):
        run()                      # plans and kernel attributes set before capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def fused_head_times(torch, nqp, entries, stream, reps):
    """The output head through nq_gemv_head at every T (argmax, maximum and
    logsumexp per token, logits not stored), and through nq_gemv_head_topk
    with k = 8 and k = 32 (the same plus the top k per token; the merge
    kernel included), one CUDA graph per call kind and T: average
    microseconds per call and weight-stream GB/s."""
    e = next(x for x in entries if x["kind"] == "head")
    dev = e["x"].device
    ws = torch.empty(nqp.head_topk_workspace_bytes(), dtype=torch.uint8, device=dev)
    out = {}
    for T in (1, 2, 4, 8, 16):
        res = [torch.empty(T, dtype=dt, device=dev) for dt in (torch.int32, torch.float32, torch.float32)]
        tk_idx = torch.empty(T * 32, dtype=torch.int32, device=dev)    # [T, k] row-major
        tk_val = torch.empty(T * 32, dtype=torch.float32, device=dev)

        def head():
            nqp.gemv_head(e["qw"].packed, e["qw"].scales, e["x"][:T], e["K"], e["N"], T, e["bits"],
                          workspace=ws, argmax=res[0], maxval=res[1], lse=res[2], stream=stream)

        def topk(k):
            def run():
                nqp.gemv_head_topk(e["qw"].packed, e["qw"].scales, e["x"][:T], e["K"], e["N"], T,
                                   e["bits"], k, workspace=ws, topk_idx=tk_idx[:T * k].view(T, k),
                                   topk_val=tk_val[:T * k].view(T, k), argmax=res[0], maxval=res[1],
                                   lse=res[2], stream=stream)
            return run
        us = _graph_us(torch, stream, head, reps)
        out[f"T{T}"] = {"us_per_call": round(us, 2),
                        "gbs": round(KIND_BYTES["head"] / (us * 1e-6) / 1e9, 1)}
        for k in (8, 32):
            out[f"T{T}"][f"topk{k}_us_per_call"] = round(_graph_us(torch, stream, topk(k), reps), 2)
    rc = nqp.last_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} in the fused head")
    return out


def head_t2_time(torch, nqp, entries, ys, stream, reps):
    """The plain head GEMV at T = 2 (a verify batch the stack does not run),
    one launch per graph replay: microseconds and GB/s."""
    e = next(x for x in entries if x["kind"] == "head")

    def run():
        nqp.gemv(e["qw"].packed, e["qw"].scales, e["x"][:2], ys["head"][:2], e["K"], e["N"], 2,
                 e["bits"], stream=stream)
    us = _graph_us(torch, stream, run, reps)
    return {"us_per_launch": round(us, 2), "gbs": round(KIND_BYTES["head"] / (us * 1e-6) / 1e9, 1)}


def mlp_times(torch, nqp, entries, stream, reps):
    """The 64 decoder-layer MLPs through nq_mlp (gate+up with SwiGLU in the
    epilogue, its bf16 activations feeding the down projection) chained in
    one CUDA graph per T: the library's choice (two launches per layer) and,
    where it applies (T <= 8), the one-launch layer kernel; against the same
    128 GEMVs launched plainly (fp32 gate and up stored, independent x).  Per-layer microseconds and weight-stream
    GB/s.  (The stack's gate+up rows are not in the interleaved order a real
    layer uses; the work, and so the time, is the same.)"""
    gus = [e for e in entries if e["kind"] == "gate_up"]
    dns = [e for e in entries if e["kind"] in ("down_q5", "down_q4")]
    dev = gus[0]["x"].device
    nbytes = KIND_BYTES["gate_up"] + KIND_BYTES["down_q5"] + KIND_BYTES["down_q4"]
    act = torch.empty((16, INTER), dtype=torch.int16, device=dev)
    y1 = torch.empty((16, 2 * INTER), dtype=torch.float32, device=dev)
    y = torch.empty((16, HIDDEN), dtype=torch.float32, device=dev)
    out = {}
    for T in TS:
        def layers(launches):
            def run():
                for gu, dn in zip(gus, dns):
                    nqp.mlp(gu["qw"], dn["qw"], gu["x"][:T], act[:T], y[:T], T, launches=launches,
                            stream=stream)
            return run

        def plain():
            for gu, dn in zip(gus, dns):
                nqp.gemv(gu["qw"].packed, gu["qw"].scales, gu["x"][:T], y1[:T], gu["K"], gu["N"], T,
                         gu["bits"], stream=stream)
                nqp.gemv(dn["qw"].packed, dn["qw"].scales, dn["x"][:T], y[:T], dn["K"], dn["N"], T,
                         dn["bits"], stream=stream)
        res = {"mlp_us_per_layer": round(_graph_us(torch, stream, layers(0), reps) / LAYERS, 2)}
        if all(nqp.mlp_one_launch_ok(HIDDEN, INTER, HIDDEN, T, 4, b) for b in (5, 4)):
            res["one_launch_us_per_layer"] = round(_graph_us(torch, stream, layers(1), reps) / LAYERS, 2)
        res["two_gemv_us_per_layer"] = round(_graph_us(torch, stream, plain, reps) / LAYERS, 2)
        res["mlp_gbs"] = round(nbytes / LAYERS / (res["mlp_us_per_layer"] * 1e-6) / 1e9, 1)
        res["mlp_frac"] = round(res["mlp_gbs"] / measured_peaks()[0], 4)
        out[f"T{T}"] = res
    rc = nqp.last_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} in the MLP layers")
    return out


def encoder_times(torch, nqp, dev, reps=3):
    """Device round-to-nearest and searched encoders on one gate+up-sized
    fp32 matrix (K=5120, N=34816, 4-bit, synthetic imatrix), CUDA events; and
    the CPU oracle's searched encoder on a bounded sample of its groups."""
    import oracle
    import synth
    K, N, bits = HIDDEN, 2 * INTER, 4
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    w = torch.randn((N, K), generator=g, device=dev, dtype=torch.float32).mul_(0.02)
    imp = torch.from_numpy(synth.imatrix(synth.generator(4242, 1), K)).to(dev)
    codes = torch.empty((N, K), dtype=torch.int8, device=dev)
    scales = torch.empty((N, K // 64), dtype=torch.int16, device=dev)
    groups = N * K // 64
    out = {"shape": {"K": K, "N": N, "bits": bits, "groups": groups}}
    for name, fn in (("rtn", lambda: nqp.quantize_rtn(w, bits, codes=codes, scales=scales)),
                     ("search", lambda: nqp.quantize_search(w, bits, imp, codes=codes, scales=scales))):
        fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"ms": round(ms, 3), "mgroups_per_s": round(groups / ms / 1e3, 1)}
    rc = nqp.last_device_error()
    if rc != 0:
        raise RuntimeError(f"device status {rc} in the encoders")
    rows = 64                                   # bounded CPU sample: 64 rows = 5120 groups
    ws = w[:rows].cpu().numpy()
    t0 = time.perf_counter()
    oracle.search_encode(ws, bits, imp.cpu().numpy())
    el = time.perf_counter() - t0
    out["search_oracle_cpu"] = {"mgroups_per_s": round(rows * K / 64 / el / 1e6, 4), "cores": 1,
                                "sample": f"{rows} rows x {K} (fp64 numpy, one thread)"}
    del w, codes, scales
    return out


def _stats(vals):
    return {"mean": statistics.fmean(vals), "median": statistics.median(vals), "min": min(vals)}


def run_ours(args, rank, world, local_rank):
    import torch

    import quantized_weight_decode_gb300 as nqp
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    nqp.build()
    nqp.lib()
    dist = world > 1
    if dist:
        import torch.distributed as td

    def barrier():
        if dist:
            td.barrier()

    entries, x_arena, ys = build_stack(torch, nqp, dev, seed=args.seed + rank)
    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    launches_per_pass = 0
    for T in TS:
        for k in KINDS:
            graphs[(T, k)], n = capture(torch, nqp, entries, ys, T, k, stream)
            if T == TS[0]:
                launches_per_pass += n
    rc = nqp.last_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} after capture")

    def one_step(evs=None):
        for T in TS:
            for k in KINDS:
                graphs[(T, k)].replay()
                if evs is not None:
                    evs[(T, k)].append(torch.cuda.Event(enable_timing=True))
                    evs[(T, k)][-1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    stream.synchronize()

    # ---------------- timed region
    evs = {key: [] for key in graphs}
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            one_step(evs)
        end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    rc = nqp.last_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} in timed region")
    total_ms = max_over_ranks(start.elapsed_time(end), dev)

    # per-(T, kind) durations of every step, from consecutive events
    seg = {key: [] for key in graphs}
    prev = start
    for s in range(args.steps):
        for T in TS:
            for k in KINDS:
                e = evs[(T, k)][s]
                seg[(T, k)].append(prev.elapsed_time(e))
                prev = e

    # ---------------- outputs of the timed graphs against the oracle
    checks = check_outputs(torch, nqp, entries, ys, graphs, stream)
    checked = all(v <= 1.0 for v in checks.values())

    # ---------------- fused verify head (argmax, maximum, logsumexp per token)
    reps = max(10, min(args.steps, 50))
    head_fused = fused_head_times(torch, nqp, entries, stream, reps=reps)
    head_t2 = head_t2_time(torch, nqp, entries, ys, stream, reps=reps)

    # ---------------- the 64 decoder-layer MLPs: SwiGLU product then down (nq_mlp)
    mlp_layers = mlp_times(torch, nqp, entries, stream, reps=max(3, min(args.steps, 10)))

    # ---------------- offline encoders on one gate+up-sized matrix
    encoders = encoder_times(torch, nqp, dev) if rank == 0 else None

    # ---------------- end to end: x from pinned host, logits back to pinned host
    # Every step uploads its x arena and reads back its logits inside the timed
    # region.  Two buffer sets (x arena and outputs, each with its own graphs)
    # let step s + 1's upload and step s's read-back run on copy streams while
    # the GEMVs of the neighbouring step run, as a decode loop would pipeline
    # them; a set is reused only after its previous step's GEMVs and
    # read-backs have finished.
    x_host = torch.empty(x_arena.shape, dtype=x_arena.dtype, pin_memory=True)
    x_host.copy_(x_arena)
    y_host = {T: torch.empty((T, VOCAB), dtype=torch.float32, pin_memory=True) for T in TS}
    h2d = x_arena.numel() * x_arena.element_size()
    d2h = sum(T * VOCAB * 4 for T in TS)
    x_arena2 = x_arena.clone()
    entries2, off = [], 0
    for e in entries:
        entries2.append(dict(e, x=x_arena2[off:off + 16 * e["K"]].view(16, e["K"])))
        off += 16 * e["K"]
    ys2 = {k: torch.empty_like(v) for k, v in ys.items()}
    graphs2 = {(T, k): capture(torch, nqp, entries2, ys2, T, k, stream)[0] for T in TS for k in KINDS}
    sets = [(x_arena, ys, graphs), (x_arena2, ys2, graphs2)]
    up = torch.cuda.Stream(device=dev)     # host -> device
    down = torch.cuda.Stream(device=dev)   # device -> host

    def e2e_steps_run(nsteps, e_start=None, e_end=None):
        comp_done = [None, None]   # the set's last step: GEMVs finished (x no longer read)
        read_done = [None, None]   # the set's last step: logits read back (outputs free)
        first = torch.cuda.Event()
        first.record(stream)
        if e_start is not None:
            e_start.record(stream)
        up.wait_event(first)
        down.wait_event(first)
        for s_ in range(nsteps):
            xa, yb, gb = sets[s_ % 2]
            with torch.cuda.stream(up):
                if comp_done[s_ % 2] is not None:
                    up.wait_event(comp_done[s_ % 2])
                xa.copy_(x_host, non_blocking=True)
                x_ready = torch.cuda.Event()
                x_ready.record(up)
            with torch.cuda.stream(stream):
                stream.wait_event(x_ready)
                if read_done[s_ % 2] is not None:
                    stream.wait_event(read_done[s_ % 2])
                for T in TS:
                    for k in KINDS:
                        gb[(T, k)].replay()
                    head_done = torch.cuda.Event()
                    head_done.record(stream)
                    with torch.cuda.stream(down):
                        down.wait_event(head_done)
                        y_host[T].copy_(yb["head"][:T], non_blocking=True)
                comp_done[s_ % 2] = torch.cuda.Event()
                comp_done[s_ % 2].record(stream)
            read_done[s_ % 2] = torch.cuda.Event()
            read_done[s_ % 2].record(down)
        stream.wait_event(read_done[(nsteps - 1) % 2])
        if e_end is not None:
            e_end.record(stream)
        stream.synchronize()

    e2e_run_steps = max(3, min(args.steps, 50))
    e2e_run_steps += e2e_run_steps % 2           # both sets equally often
    e2e_steps_run(4)                             # warm-up: both sets' graphs uploaded
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e2e_steps_run(e2e_run_steps, e0, e1)
    e2e_steps = e2e_run_steps
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)

    if rank != 0:
        return
    if not checked:
        print(json.dumps({"error": "GPU outputs outside the oracle's tolerance", "checks": checks}),
              file=sys.stderr, flush=True)
        sys.exit(3)
    peak, peak_kind = measured_peaks()
    steps = args.steps
    value = whole_job_gbs(world, steps, len(TS) * PASS_BYTES, total_ms)
    e2e_value = whole_job_gbs(world, e2e_steps, len(TS) * PASS_BYTES, e2e_ms)
    per_t = {}
    for T in TS:
        ms = [sum(seg[(T, k)][s] for k in KINDS) for s in range(steps)]
        st = _stats(ms)
        gbs = PASS_BYTES / (st["mean"] * 1e-3) / 1e9
        per_t[str(T)] = {"us_per_pass": round(st["mean"] * 1e3, 2),
                         "us_per_pass_median": round(st["median"] * 1e3, 2),
                         "us_per_pass_min": round(st["min"] * 1e3, 2), "gbs": round(gbs, 1),
                         "frac_of_measured_hbm": round(gbs / peak, 4),
                         "frac_of_8tbs": round(gbs / 8000.0, 4)}
    kernels = {}
    for T in TS:
        for k in KINDS:
            n = KIND_COUNT[k]
            st = _stats([v * 1e3 / n for v in seg[(T, k)]])       # us per launch, per step
            gbs = KIND_BYTES[k] / n / (st["mean"] * 1e-6) / 1e9
            kernels[f"{k}_T{T}"] = {
                "us_per_launch": round(st["mean"], 2), "us_median": round(st["median"], 2),
                "us_min": round(st["min"], 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                "frac_of_min": round(KIND_BYTES[k] / n / (st["min"] * 1e-6) / 1e9 / peak, 4)}
    dom = kernels["gate_up_T1"]
    roofline = {"bound": "hbm", "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(dom["gbs"] / peak, 4), "traffic": stored_traffic(),
                "kernel": "nq_gemv_kernel<4,1,3> (4-bit, MMA route, x in registers) "
                          "gate+up Q4 K=5120 N=34816 at T=1",
                "bytes_per_launch": packed_bytes(4, HIDDEN, 2 * INTER),
                "peak_source": peak_kind,
                # the same product at every T of the step (T=16: nq_gemv_kernel<4,1,4>)
                "frac_by_T": {str(T): kernels[f"gate_up_T{T}"]["frac"] for T in TS}}
    # The single-shape configurations inside the stack (each kind's graph at T).
    configs = {
        "gate_up_q4_T1": kernels["gate_up_T1"]["frac"],
        "down_q5_T1": kernels["down_q5_T1"]["frac"], "down_q5_T8": kernels["down_q5_T8"]["frac"],
        "down_q5_T16": kernels["down_q5_T16"]["frac"],
        "head_q6_T1": kernels["head_T1"]["frac"], "head_q6_T2": round(head_t2["gbs"] / peak, 4),
        "head_q6_T4": kernels["head_T4"]["frac"], "head_q6_T8": kernels["head_T8"]["frac"],
        "head_q6_T16": kernels["head_T16"]["frac"],
    }
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(CONFIG, parallelism=f"replicas x{world}"),
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * len(TS) * launches_per_pass,
        "roofline": roofline,
        "cpu_baseline": cpu_baseline(args.cpu_seconds),
        "clocks": clocks,
        "checked": checked,
        "checks": checks,
        "per_T": per_t,
        "kernels": kernels,
        "configs_frac_of_measured": configs,
        "head_fused": head_fused,
        "head_T2": head_t2,
        "mlp_layers": mlp_layers,
        "encoders": encoders,
        "plans": {f"{k}_T{T}": nqp.plan(e["K"], e["N"], T, e["bits"])
                  for T in TS for k in KINDS
                  for e in [next(x for x in entries if x["kind"] == k)]},
        "source_hash": source_hash(),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ single shape
CONFIG_SHAPES = {
    "tiny_q4": (512, 256, 4, (1,)),
    "gate_up_q4": (HIDDEN, 2 * INTER, 4, (1,)),
    "down_q5": (INTER, HIDDEN, 5, (1, 8)),
    "head_q6": (HIDDEN, VOCAB, 6, (1, 2, 4, 8)),
}


def run_single(spec: str, reps: int, seed: int):
    """Time one GEMV shape "K,N,bits,T" (or a config name above, every T):
    `reps` launches over enough distinct packed copies (>= 3x L2) that no
    launch finds its weights in L2.  Prints one JSON line per (shape, T)."""
    import torch

    import quantized_weight_decode_gb300 as nqp
    torch.cuda.set_device(0)
    nqp.build()
    if spec in CONFIG_SHAPES:
        K, N, bits, Ts = CONFIG_SHAPES[spec]
    else:
        K, N, bits, T = (int(v) for v in spec.split(","))
        Ts = (T,)
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    w = torch.randn((N, K), generator=g, device=dev, dtype=torch.float32).mul_(0.02)
    qw = nqp.QuantizedWeight.from_fp32(w, bits)
    del w
    nbytes = packed_bytes(bits, K, N)
    copies = [qw] + [nqp.QuantizedWeight(qw.packed.clone(), qw.scales.clone(), K, N, bits)
                     for _ in range(max(0, (3 * 135_000_000) // nbytes))]
    for T in Ts:
        x = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((T, N), dtype=torch.float32, device=dev)
        for i in range(3):
            copies[i % len(copies)].gemv(x, y)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            copies[i % len(copies)].gemv(x, y)
        e1.record()
        torch.cuda.synchronize()
        rc = nqp.last_device_error()
        if rc != 0:
            raise RuntimeError(f"device status {rc}")
        us = e0.elapsed_time(e1) * 1e3 / reps
        peak, kind = measured_peaks()
        print(json.dumps({"shape": {"K": K, "N": N, "bits": bits, "T": T}, "us_per_launch": round(us, 2),
                          "gbs": round(nbytes / us / 1e3, 1), "frac_of_measured_hbm": round(nbytes / us / 1e3 / peak, 4),
                          "frac_of_8tbs": round(nbytes / us / 1e3 / 8000.0, 4), "weight_bytes": nbytes,
                          "copies": len(copies), "plan": nqp.plan(K, N, T, bits)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--single", default=None,
                    help='time one shape "K,N,bits,T" or a config name (%s)' % ", ".join(CONFIG_SHAPES))
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    if args.single:
        run_single(args.single, args.reps, args.seed)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as td
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        td.init_process_group(backend=backend)
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as td
        td.destroy_process_group()


if __name__ == "__main__":
    main()
