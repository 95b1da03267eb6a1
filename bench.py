"""Benchmark of the SSD prefill and the multi-step decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mamba2_2p7b|long_16k|hybrid_llama3_8b|tiny_f32|multistep_k8]

One step = one ssd_fwd call over the whole workload (every kernel of the
chunked algorithm) with inputs resident in HBM.  Default workload: one Mamba-2
2.7B SSD layer (batch 8, T 2048, 80 heads, P 64, N 128, chunk 256, bf16 I/O,
fp32 state), synthetic seeded inputs.  Metric: tokens x heads per second,
reported in M tok*heads/s, plus the fraction of the layer's roofline
(mandatory I/O over the measured HBM bandwidth).  The K timed steps are one
CUDA graph, replayed until at least one second of device time is measured;
ms_per_step is the median over the replays.  At N = 1 the default line also
carries the other four workloads (`workloads`), each measured the same way.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no exchange between (batch, head) pairs); rank 0 prints one
JSON line with the whole-job throughput over the max time across ranks.

--impl reference times the fp64 CPU oracle on bounded samples of the same
workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_model_09_b300 import synth  # noqa: E402

METRIC = "SSD fwd Mtok·heads/s at Mamba-2 2.7B shape; % of roofline (TC or HBM)"
UNIT = "Mtok·heads/s"
L2_BYTES = 126 * 1024 * 1024


# DRAM traffic per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) of
# the dominant kernels, with the sha1 of the kernel's source at capture time;
# the summaries are in profiles/.  A changed source reports null.
FUSED_SRCS = ("state_space_model_09_b300/csrc/ssd_fused_hb.cuh",
              "state_space_model_09_b300/csrc/ssd_scan.cuh",
              "state_space_model_09_b300/csrc/ssd_scan_hb.cuh",
              "state_space_model_09_b300/csrc/ssd_tc.cuh",
              "state_space_model_09_b300/csrc/ssd_device.cuh")
MS_SRCS = ("state_space_model_09_b300/csrc/ssd_kernels.cuh",
           "state_space_model_09_b300/csrc/ssd_device.cuh")
MEASURED_TRAFFIC = {
    # (kernel, workload): (DRAM bytes read + written per launch, the sources
    # the kernel is built from, sha1 of their concatenation when captured)
    ("chunk_fused_hb", "mamba2_2p7b"):
        (348_288_000, FUSED_SRCS,
         "bb867851599ddb933a8594dae51214315db77d83"),
    ("chunk_fused_hb", "hybrid_llama3_8b"):
        (406_779_776, FUSED_SRCS,
         "bb867851599ddb933a8594dae51214315db77d83"),
    ("multistep_kernel", "multistep_k8"):
        (68_785_152, MS_SRCS,
         "4503a261542508fe7c15bcd2eba12bf6d229c1cc"),
    ("multistep_kernel_verify", "multistep_k8"):
        (46_621_952, MS_SRCS,
         "4503a261542508fe7c15bcd2eba12bf6d229c1cc"),
    ("multistep_kernel_draft", "multistep_k8"):
        (44_964_480, MS_SRCS,
         "4503a261542508fe7c15bcd2eba12bf6d229c1cc"),
}


def measured_traffic(kernel: str, workload: str):
    """The ncu DRAM traffic of a kernel on a workload, or None when there is
    no capture or its sources changed since."""
    import hashlib
    ent = MEASURED_TRAFFIC.get((kernel, workload))
    if not ent:
        return None
    nbytes, srcs, sha = ent
    h = hashlib.sha1()
    try:
        for src in srcs:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return nbytes if h.hexdigest() == sha else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s nominal HBM3e figure quoted for the decode target


# ----------------------------------------------------------------------------- work model
def hb_fast_fraction(s: synth.FwdShape, inp) -> float:
    """Share of (batch, chunk, head) units whose in-chunk decay stays within the
    range of the head-pair form of the chunk scan (log2 of the chunk's total
    decay >= -192, with a shifted reference below -96); the rest are computed
    one by one.  Recomputed here in float64, for the report only."""
    dt = inp["dt"].astype(np.float64)
    sp = np.where(dt > 20.0, dt, np.log1p(np.exp(np.minimum(dt, 20.0))))
    dA = sp * inp["A"].astype(np.float64)[None, None, :] / math.log(2.0)
    b, T, H = dA.shape
    nc = math.ceil(T / s.chunk)
    pad = np.zeros((b, nc * s.chunk, H))
    pad[:, :T] = dA
    last = pad.reshape(b, nc, s.chunk, H).sum(axis=2)
    return float(np.mean(last >= -192.0))


def fwd_work(s: synth.FwdShape):
    """Algorithmic bytes / flops of the layer and of each stage (per call).

    Layer (mandatory I/O): x, y, B, C (io dtype), dt (f32), h0 if given,
    h_final (f32).  Flops count causal work only: P*Q(Q+1) (masked scores times
    x), 2QNP (chunk state), 2QNP (output from the initial state) per
    (b, chunk, head), plus N*Q(Q+1) per (b, chunk, distinct B/C group pair) for
    C B^T.

    Per stage: `mandatory` = the part of the layer's mandatory I/O the stage
    reads or writes (dt counts for the stages that read its per-token decays);
    `io` = everything the stage moves once, intermediates (chunk states, the
    decays) included; `flops` its causal tensor work."""
    io = 2 if s.io == synth.BF16 else 4
    b, T, H, P, N, Q = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.chunk
    nc = math.ceil(T / Q)
    x = b * T * H * P * io
    Bb = b * T * s.ngroups_b * N * io
    Cb = b * T * s.ngroups_c * N * io
    dt = b * T * H * 4
    st = b * H * N * P * 4
    h0 = st if s.h0 != "zero" else 0
    pairs = max(s.ngroups_b, s.ngroups_c)
    flops = b * nc * H * (P * Q * (Q + 1) + 4 * Q * N * P) + b * nc * pairs * N * Q * (Q + 1)
    layer_bytes = 2 * x + Bb + Cb + dt + h0 + st
    cs = b * H * nc * Q * 4
    S32 = b * nc * H * N * P * 4
    hin16 = b * nc * H * N * P * 2
    f_state = 2 * b * nc * H * Q * N * P
    f_scan = b * nc * H * (P * Q * (Q + 1) + 2 * Q * N * P) + b * nc * pairs * N * Q * (Q + 1)

    def stage(mandatory, io_bytes, fl):
        return dict(mandatory=mandatory, io=io_bytes, flops=fl)

    stages = {
        "dt_decay": stage(dt, 2 * dt, 0),
        "chunk_state_pass_tc": stage(x + Bb + dt + h0 + st, x + Bb + dt + h0 + hin16 + st, f_state),
        "chunk_scan_hl": stage(2 * x + Bb + Cb + dt, 2 * x + Bb + Cb + dt + hin16, f_scan),
        "state_fixup": stage(0, 2 * hin16 + st, 0),  # bound: every head split
        "dt_cumsum": stage(dt, dt + cs, 0),
        "chunk_state_simt": stage(x + Bb, x + Bb + cs + S32, f_state),
        "state_passing": stage(h0 + st, 2 * S32 + b * H * nc * 4 + h0 + st,
                               2 * b * nc * H * N * P),
        "chunk_scan_simt": stage(2 * x + Bb + Cb, 2 * x + Bb + Cb + cs + S32, f_scan),
    }
    # the head-pair kernels: the same inputs and outputs
    stages["chunk_scan_hb"] = stages["chunk_scan_hl"]
    stages["chunk_state_hb"] = stages["chunk_state_pass_tc"]
    # the one-pass kernel moves the layer's whole mandatory I/O (its prepass
    # re-reads x, B and dt of the split items' segments, and the flagged pass
    # the few long-decay (chunk, head) units: bounded above by these)
    stages["chunk_fused_hb"] = stage(layer_bytes, layer_bytes, flops)
    stages["chunk_fused_prepass"] = stage(0, x + Bb + dt, f_state)
    stages["chunk_scan_flagged"] = stage(0, 2 * x + Bb + Cb + dt + hin16, f_scan)
    return dict(layer_bytes=layer_bytes, flops=flops, stages=stages, tok_heads=b * T * H)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "--id=" + gpu_id, "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        with open(self.f.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(dev) -> str:
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        return str(dev)


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("SSD_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle timing
def time_oracle_fwd(shape, inp, pairs, threads=0):
    import oracle
    t0 = time.perf_counter()
    oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                   pairs=pairs, nthreads=threads)
    return time.perf_counter() - t0


def cpu_baseline(shape, inp, budget_s=20.0):
    """The oracle as it stands, on the host's cores, on a bounded sample of the
    workload: as many (b, h) pairs (whole sequences) as fit ~budget_s."""
    import oracle
    H = shape.nheads
    total = shape.batch * H
    cores = oracle.default_threads()
    probe = list(range(min(total, max(cores, 8))))
    tp = time_oracle_fwd(shape, inp, probe)
    per_pair = tp / len(probe)
    n = int(min(total, max(len(probe), budget_s / max(per_pair, 1e-9))))
    pairs = list(range(n))
    t = time_oracle_fwd(shape, inp, pairs)
    rate = n * shape.seqlen / t / 1e6
    return {"value": round(rate, 4), "unit": UNIT, "cores": min(cores, n), "kind": "oracle",
            "sample": "%d of %d (batch, head) pairs, whole %d-token sequences (%.1f s, fp64)"
                      % (n, total, shape.seqlen, t)}


def config_of(workload, shape, world):
    """The workload named by its sizes; identical in both arms."""
    if isinstance(shape, synth.MultistepShape):
        return {"workload": workload, "batch": shape.batch, "K": shape.K,
                "nheads": shape.nheads, "headdim": shape.headdim, "dstate": shape.dstate,
                "ngroups_b": shape.ngroups_b, "ngroups_c": shape.ngroups_c,
                "io": "bf16" if shape.io == synth.BF16 else "f32", "state": "f32",
                "chain": shape.steps, "parallelism": "replicas%d" % world}
    return {"workload": workload, "batch": shape.batch, "seq_len": shape.seqlen,
            "nheads": shape.nheads, "headdim": shape.headdim, "dstate": shape.dstate,
            "ngroups_b": shape.ngroups_b, "ngroups_c": shape.ngroups_c, "chunk": shape.chunk,
            "io": "bf16" if shape.io == synth.BF16 else "f32", "state": "f32",
            "h0": shape.h0, "parallelism": "replicas%d" % world}


def run_reference(args, shape, work):
    """--impl reference: the fp64 oracle on bounded samples of the workload."""
    inp = synth.make_fwd_inputs(shape, synth.WORKLOAD_SEEDS[args.workload])
    import oracle
    cores = oracle.default_threads()
    total = shape.batch * shape.nheads
    probe = list(range(min(total, cores)))
    per_pair = time_oracle_fwd(shape, inp, probe) / len(probe)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(total, budget / max(per_pair, 1e-9))))
    pairs = list(range(n))
    for _ in range(args.warmup):
        time_oracle_fwd(shape, inp, pairs)
    t = sum(time_oracle_fwd(shape, inp, pairs) for _ in range(args.steps))
    ms = t / args.steps * 1e3
    value = n * shape.seqlen / (t / args.steps) / 1e6
    sample = "%d of %d (batch, head) pairs per step, whole sequences" % (n, total)
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": config_of(args.workload, shape, args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": min(cores, n),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line, ensure_ascii=False))


def oracle_multistep_chain(calls: int, budget_s: float):
    """The fp64 oracle walking a multistep_k8 speculative chain (each call
    continues from the previous call's h_j) on a bounded sample of the
    (batch, head) pairs per call.  Returns (Mtok·heads/s, ms per call, cores,
    sample description)."""
    import oracle
    shape = synth.WORKLOADS["multistep_k8"]
    distinct = min(calls, 64)  # drafts drawn for 64 calls, reused cyclically (bounded memory)
    inp = synth.make_multistep_inputs(shape, synth.WORKLOAD_SEEDS["multistep_k8"], steps=distinct)
    b, H = shape.batch, shape.nheads
    total = b * H
    cores = oracle.default_threads()
    h = inp["h_cache"].copy()

    def call(i, pairs):
        i %= distinct
        _, hj, _ = oracle.ssd_multistep(inp["x"][i], inp["dt"][i], inp["A"], inp["B"][i],
                                        inp["C"][i], inp["D"], h, inp["j"][i], pairs=pairs)
        for q, pr in enumerate(pairs):  # the sampled pairs continue from h_j
            h[pr // H, pr % H] = hj[q]

    probe = list(range(min(total, max(cores, 8))))
    t0 = time.perf_counter()
    call(0, probe)
    per_pair = (time.perf_counter() - t0) / len(probe)
    h[:] = inp["h_cache"]
    n = int(max(1, min(total, budget_s / calls / max(per_pair, 1e-9))))
    pairs = list(range(n))
    warm = min(3, calls - 1)
    for i in range(warm):
        call(i, pairs)
    t0 = time.perf_counter()
    for i in range(warm, calls):
        call(i, pairs)
    t = (time.perf_counter() - t0) / (calls - warm)
    sample = ("%d of %d (batch, head) pairs per call, a %d-call chain from the cached state "
              "over %d distinct draft sets (fp64)" % (n, total, calls, distinct))
    return n * shape.K / t / 1e6, t * 1e3, min(cores, n), sample


MULTISTEP_METRIC = "SSD multistep decode Mtok·heads/s (K=8 verify, 1000-step speculative chain)"


def run_reference_multistep(args):
    """--impl reference on multistep_k8: the oracle chain, one call per step."""
    shape = synth.WORKLOADS["multistep_k8"]
    value, ms, cores, sample = oracle_multistep_chain(args.warmup + args.steps, 150.0)
    line = {"metric": MULTISTEP_METRIC,
            "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": config_of("multistep_k8", shape, args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line, ensure_ascii=False))


def n_copies(layer_bytes, dev=None):
    """Device copies of a prefill workload's inputs and outputs that the timed
    steps rotate over: enough to fill twice the L2 (one when a single copy
    already does)."""
    l2 = L2_BYTES
    if dev is not None:
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size or l2
    return 1 if layer_bytes >= 2 * l2 else -(-2 * l2 // layer_bytes)


def timed_replays(replay, steps, stream, min_s):
    """Replays `replay` (which enqueues `steps` steps on `stream`) until at
    least min_s of device time has been timed, each replay between two CUDA
    events on the stream.  Returns (median ms per step, repeats)."""
    import torch
    per = []
    total = 0.0
    while total < min_s * 1e3 or len(per) < 5:
        evs = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            replay()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        for e0, e1 in evs:
            t = e0.elapsed_time(e1)
            per.append(t / steps)
            total += t
    return statistics.median(per), len(per)


def roofline_of(name, st, seconds, pk, workload):
    """The roofline entry of one kernel: mandatory I/O (the layer's x, y, B, C,
    dt, h0, h_final that it moves) or causal tensor flops, per launch, over its
    event-timed duration."""
    t_hbm = st["mandatory"] / (pk["hbm"] * 1e9)
    t_tc = st["flops"] / (pk["bf16"] * 1e12)
    if t_tc > t_hbm:
        roof = {"bound": "tensor", "achieved": round(st["flops"] / seconds / 1e12, 2),
                "peak": pk["bf16"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(st["mandatory"] / seconds / 1e9, 1),
                "peak": pk["hbm"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = measured_traffic(name, workload)
    roof["kernel"] = name
    roof["algorithmic_bytes"] = st["mandatory"]
    roof["algorithmic_flops"] = st["flops"]
    roof["kernel_io_bytes"] = st["io"]
    roof["kernel_io_frac"] = round(st["io"] / seconds / 1e9 / pk["hbm"], 4)
    if roof["bound"] == "hbm":
        roof["frac_vs_nominal_8tbs"] = round(st["mandatory"] / seconds / 1e9 / NOMINAL_HBM_GBS, 4)
    roof["peak_source"] = pk["source"] + " (burst)"
    return roof


# ----------------------------------------------------------------------------- prefill
def measure_prefill(workload, shape, args, world, rank, dev, min_s, e2e=True, cpu_budget=20.0):
    """One prefill workload on this rank's GPU: the graph-replayed step, the
    per-kernel event times, the end-to-end call from host buffers and (rank 0
    at N = 1) the oracle on the host cores.  Returns the fields of its line."""
    import torch
    from state_space_model_09_b300 import ssd as S

    work = fwd_work(shape)
    inp = synth.make_fwd_inputs(shape, synth.WORKLOAD_SEEDS[workload] + 17 * rank)
    io_t = torch.bfloat16 if shape.io == synth.BF16 else torch.float32
    host = {}
    for k, v in inp.items():
        if v is None:
            host[k] = None
            continue
        t = torch.from_numpy(v)
        if k in ("x", "B", "C"):
            t = t.to(io_t)
        host[k] = t.pin_memory()
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    b, T, H, P = d["x"].shape
    N = d["B"].shape[3]
    y = torch.empty_like(d["x"])
    hf = torch.empty((b, H, N, P), dtype=torch.float32, device=dev)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    ws = S.workspace_for(dims, shape.chunk, dev)
    # a stream of our own (graphs cannot be captured on the legacy default
    # stream); every torch op below runs on it
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    names = [S.ssd_fwd_stage_name(dims, shape.chunk, i)
             for i in range(S.ssd_fwd_num_stages(dims, shape.chunk))]

    # Inputs smaller than twice the L2 are rotated over enough device copies
    # that every timed step reads data the previous steps have evicted.
    copies = n_copies(work["layer_bytes"], dev)
    sets = [(d, y, hf, ws)]
    for _ in range(copies - 1):
        sets.append(({k: (None if v is None else v.clone()) for k, v in d.items()},
                     torch.empty_like(y), torch.empty_like(hf), torch.empty_like(ws)))

    def step(i=0):
        dd, yy, hh_, ww = sets[i % copies]
        S.ssd_fwd(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["h0"], shape.chunk,
                  yy, hh_, ww, True, stream, dims)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    S.ssd_check_device_error(stream)
    # the timed steps replay as CUDA graphs of up to 500 steps (no host launch gaps)
    K = args.steps
    gsteps = min(K, max(500, copies))
    sizes = [gsteps] * (K // gsteps) + ([K % gsteps] if K % gsteps else [])
    graphs = {}
    for n in set(sizes):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        graphs[n] = g

    def replay():
        for n in sizes:
            graphs[n].replay()

    with torch.cuda.stream(stream):
        for i in range(copies):  # every copy once, so the first timed ones are out of L2
            step(i)
        replay()
    torch.cuda.synchronize()
    S.ssd_check_device_error(stream)

    # ---- timed region: the K-step block replayed until >= min_s, barrier +
    # synchronize on both sides; the median over the repeats
    clocks = ClockSampler(gpu_id_for(dev))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ms, reps = timed_replays(replay, K, stream, min_s)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    S.ssd_check_device_error(stream)
    ms = max_over_ranks(ms, world, dev)

    # ---- per-kernel durations (CUDA events on the launching stream); a
    # bounded device-side delay first lets the host queue every call, so no
    # stage waits on a launch
    nst = len(names)
    ks = max(20, min(K, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(ks)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(20_000_000)
    for i in range(ks):
        dd, yy, hh_, ww = sets[i % copies]
        S.ssd_fwd_profiled(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["h0"],
                           shape.chunk, yy, hh_, ww, evs[i], True, stream, dims)
    torch.cuda.synchronize()
    stage_ms = [statistics.median(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(ks))
                for k in range(nst)]

    out = {"ms": ms, "repeats": reps, "clocks": clk, "names": names, "stage_ms": stage_ms,
           "work": work, "launches": nst * K * reps}
    if e2e:
        out["e2e"] = e2e_prefill(S, shape, host, d, y, hf, ws, dims, stream, world, dev,
                                 max(3, min(K, 50)))
    if "chunk_scan_hb" in names:
        out["pair_form_share"] = round(hb_fast_fraction(shape, inp), 4)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and cpu_budget > 0:
        out["cpu_baseline"] = cpu_baseline(shape, inp, cpu_budget)
    return out


def e2e_prefill(S, shape, host, d, y, hf, ws, dims, stream, world, dev, ke):
    """End to end through the public API: every step copies its inputs in from
    pinned host memory, runs ssd_fwd and copies y and h_final back.  Two device
    sets of inputs and outputs let step i + 1's host-to-device copies (one
    stream) run while step i computes and step i - 1's results come back
    (another stream)."""
    import torch
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dsets = [(d, y, hf), ({k: (None if v is None else torch.empty_like(v)) for k, v in d.items()},
                          torch.empty_like(y), torch.empty_like(hf))]
    outs_h = [(torch.empty(y.shape, dtype=y.dtype, pin_memory=True),
               torch.empty(hf.shape, dtype=hf.dtype, pin_memory=True)) for _ in range(2)]
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "out", "done")}

    def e2e_step(i):
        k = i % 2
        dd, yy, hh = dsets[k]
        s_in.wait_event(ev["out"][k])  # step i - 2 has finished reading this input set
        with torch.cuda.stream(s_in):
            for name in ("x", "dt", "A", "B", "C", "D", "h0"):
                if host[name] is not None:
                    dd[name].copy_(host[name], non_blocking=True)
            ev["in"][k].record(s_in)
        stream.wait_event(ev["in"][k])
        stream.wait_event(ev["done"][k])  # step i - 2's results have left this output set
        S.ssd_fwd(dd["x"], dd["dt"], dd["A"], dd["B"], dd["C"], dd["D"], dd["h0"], shape.chunk,
                  yy, hh, ws, True, stream, dims)
        ev["out"][k].record(stream)
        s_out.wait_event(ev["out"][k])
        with torch.cuda.stream(s_out):
            outs_h[k][0].copy_(yy, non_blocking=True)
            outs_h[k][1].copy_(hh, non_blocking=True)
            ev["done"][k].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    s_in.wait_event(f0)
    for i in range(ke):
        e2e_step(i)
    for k in range(2):
        stream.wait_event(ev["done"][k])
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / ke, world, dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in host if host[k] is not None)
    d2h = y.numel() * y.element_size() + hf.numel() * hf.element_size()
    return {"ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def prefill_fields(workload, shape, m, world, pk):
    """The JSON fields of a measured prefill workload."""
    work = m["work"]
    ms = m["ms"]
    value = world * work["tok_heads"] / (ms * 1e-3) / 1e6
    names, stage_ms = m["names"], m["stage_ms"]
    dom = int(np.argmax(stage_ms))
    roof = roofline_of(names[dom], work["stages"][names[dom]], stage_ms[dom] * 1e-3, pk, workload)
    t_hbm = work["layer_bytes"] / (pk["hbm"] * 1e9)
    t_tc = work["flops"] / (pk["bf16"] * 1e12)
    f = {
        "value": round(value, 2), "ms_per_step": round(ms, 5), "repeats": m["repeats"],
        "roofline": roof,
        "layer_roofline": {"bytes": work["layer_bytes"], "flops": work["flops"],
                           "t_bound_us": round(max(t_hbm, t_tc) * 1e6, 2),
                           "bound": "hbm" if t_hbm >= t_tc else "tensor",
                           "frac": round(max(t_hbm, t_tc) / (ms * 1e-3), 4),
                           "frac_vs_nominal_8tbs": round(
                               work["layer_bytes"] / (NOMINAL_HBM_GBS * 1e9) / (ms * 1e-3), 4),
                           "peaks": "%s HBM %.1f GB/s, bf16 %.1f TFLOP/s"
                                    % (pk["source"], pk["hbm"], pk["bf16"])},
        "stages_ms": {n: round(t, 5) for n, t in zip(names, stage_ms)},
        "clocks": m["clocks"],
    }
    if "pair_form_share" in m:
        f["pair_form_share"] = m["pair_form_share"]
    if "e2e" in m:
        e = m["e2e"]
        f["e2e"] = {"value": round(world * work["tok_heads"] / (e["ms_per_step"] * 1e-3) / 1e6, 2),
                    "unit": UNIT, "h2d_bytes_per_step": e["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": e["d2h_bytes_per_step"],
                    "ms_per_step": round(e["ms_per_step"], 4)}
    if "cpu_baseline" in m:
        f["cpu_baseline"] = m["cpu_baseline"]
    return f


def timing_note(work, K, dev=None):
    lb = work["layer_bytes"]
    n = n_copies(lb, dev)
    l2 = ("no flush; inputs+outputs %.0f MB > 2 x 126 MB L2" % (lb / 1e6) if n == 1 else
          "no flush; steps rotate over %d copies of the %.1f MB inputs+outputs (%.0f MB > 2 x L2)"
          % (n, lb / 1e6, n * lb / 1e6))
    return {"l2": l2, "graph": "CUDA graph of the %d steps, replayed until >= 1 s; "
                              "ms_per_step = median over the replays" % K}


EXTRA_WORKLOADS = ("long_16k", "hybrid_llama3_8b", "tiny_f32", "multistep_k8")


def run_ours(args, shape, world, rank, local):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m = measure_prefill(args.workload, shape, args, world, rank, dev, args.min_seconds,
                        e2e=True, cpu_budget=20.0)
    # the other workloads of the layer, each measured the same way (N = 1 only)
    extra = {}
    if args.workload == "mamba2_2p7b" and world == 1 and not args.no_workloads:
        for wl in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            if wl == "multistep_k8":
                extra[wl] = multistep_summary(args, world, rank, local)
            else:
                s2 = synth.WORKLOADS[wl]
                m2 = measure_prefill(wl, s2, args, world, rank, dev, args.min_seconds,
                                     e2e=False, cpu_budget=6.0)
                extra[wl] = dict(config_of(wl, s2, world), **prefill_fields(wl, s2, m2, world, peaks()))
                extra[wl]["timing"] = timing_note(m2["work"], args.steps, dev)
    if rank != 0:
        return
    pk = peaks()
    f = prefill_fields(args.workload, shape, m, world, pk)
    line = {
        "metric": METRIC, "value": f.pop("value"), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": f.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.io == synth.BF16 else "f32", "data": "synthetic (seeded PCG64)",
        "config": config_of(args.workload, shape, world),
        "timing": timing_note(m["work"], args.steps, dev),
        "gpu_launches": m["launches"],
        "peaks_used": {"hbm_gbs": pk["hbm"], "bf16_tflops": pk["bf16"],
                       "bf16_tflops_sustained": pk["bf16_sus"], "source": pk["source"]},
    }
    line.update(f)
    if extra:
        line["workloads"] = extra
    print(json.dumps(line, ensure_ascii=False), flush=True)


# ----------------------------------------------------------------------------- multistep arm
def multistep_work(s: synth.MultistepShape, verify: bool = False, draft: bool = False):
    """Bytes of one multi-step call: h_cache in, h_j and h_K out (f32), x and y
    (io), B, C (io), dt (f32), j (int32).  A fused verify call moves two states
    (cache in, next cache out) and also reads the previous drafts' x, B, dt.  A
    draft-model step is a fused verify call with one new token (K = 1) after
    the K previous drafts."""
    io = 2 if s.io == synth.BF16 else 4
    st = s.batch * s.nheads * s.dstate * s.headdim * 4
    x = s.batch * s.K * s.nheads * s.headdim * io
    bc = s.batch * s.K * (s.ngroups_b + s.ngroups_c) * s.dstate * io
    dt = s.batch * s.K * s.nheads * 4
    if draft:
        x1, bc1, dt1 = x // s.K, bc // s.K, dt // s.K
        bp = s.batch * s.K * s.ngroups_b * s.dstate * io
        return dict(bytes=2 * st + x + bp + dt + 2 * x1 + bc1 + dt1 + s.batch * 4,
                    tok_heads=s.batch * s.nheads)
    if verify:
        bp = s.batch * s.K * s.ngroups_b * s.dstate * io
        return dict(bytes=2 * st + 3 * x + bc + bp + 2 * dt + s.batch * 4,
                    tok_heads=s.batch * s.K * s.nheads)
    return dict(bytes=3 * st + 2 * x + bc + dt + s.batch * 4,
                tok_heads=s.batch * s.K * s.nheads)


def run_sequential(args, shape, world, rank, local):
    """Prefill of the workload through ssd_fwd_sequential (windows of
    --window tokens chained through the state): one step = the whole
    sequence.  Reports the same throughput metric and the device workspace,
    which does not grow with the sequence length."""
    import torch
    from state_space_model_09_b300 import ssd as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = synth.make_fwd_inputs(shape, synth.WORKLOAD_SEEDS[args.workload] + 17 * rank)
    io_t = torch.bfloat16 if shape.io == synth.BF16 else torch.float32
    d = {}
    for k, v in inp.items():
        d[k] = None if v is None else (torch.from_numpy(v).to(io_t) if k in ("x", "B", "C")
                                       else torch.from_numpy(v)).to(dev)
    b, T, H, P = d["x"].shape
    y = torch.empty_like(d["x"])
    hf = torch.empty((b, H, d["B"].shape[3], P), dtype=torch.float32, device=dev)
    dims = S.dims_of(d["x"], d["B"], d["C"])
    nbytes = S.ssd_fwd_sequential_workspace_size(dims, shape.chunk, args.window)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        S.ssd_fwd_sequential(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                             shape.chunk, args.window, y, hf, ws, True, stream, dims)

    def block():
        for _ in range(args.steps):
            step()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    S.ssd_check_device_error(stream)
    clocks = ClockSampler(gpu_id_for(dev))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ms, reps = timed_replays(block, args.steps, stream, args.min_seconds)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world, dev)
    S.ssd_check_device_error(stream)
    if rank != 0:
        return
    print(json.dumps({
        "metric": "SSD sequential prefill Mtok·heads/s (windows chained through the state)",
        "value": round(world * shape.tok_heads / (ms * 1e-3) / 1e6, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "repeats": reps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.io == synth.BF16 else "f32", "data": "synthetic (seeded PCG64)",
        "config": dict(config_of(args.workload, shape, world), window=args.window,
                       workspace_bytes=nbytes,
                       whole_call_workspace_bytes=S.ssd_fwd_workspace_size(dims, shape.chunk)),
        "clocks": clk}), flush=True)


def run_cp(args, shape, world, rank, local):
    """Context parallelism's per-rank compute on one GPU (--cp R): the
    sequence cut into R contiguous segments on the chunk grid; each rank's
    phase 1 (ssd_fwd of its segment, rank 0 from h0, then
    ssd_cp_segment_decay) and phase 2 (ssd_cp_correct once every rank's decay
    and final state are gathered) are timed as CUDA-graph replays.  The
    gather itself is done here by device copies and not timed: with one GPU
    per call the exchange between GPUs is not measured.  The critical path of
    R concurrent ranks is max(phase 1) + exchange + max(phase 2)."""
    import torch
    from state_space_model_09_b300 import ssd as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    R = args.cp
    inp = synth.make_fwd_inputs(shape, synth.WORKLOAD_SEEDS[args.workload])
    io_t = torch.bfloat16 if shape.io == synth.BF16 else torch.float32
    T, Q = shape.seqlen, shape.chunk
    per = -(-T // R)
    per = -(-per // Q) * Q
    cuts = [min(T, r * per) for r in range(R + 1)]
    if any(cuts[r + 1] <= cuts[r] for r in range(R)):
        raise SystemExit("--cp %d leaves an empty segment of %d tokens" % (R, T))
    A = torch.from_numpy(inp["A"]).to(dev)
    D = None if inp["D"] is None else torch.from_numpy(inp["D"]).to(dev)
    h0 = None if inp["h0"] is None else torch.from_numpy(inp["h0"]).to(dev)
    b, H, P, N = shape.batch, shape.nheads, shape.headdim, shape.dstate
    stream = torch.cuda.Stream(dev)
    ranks = []
    for r in range(R):
        sl = slice(cuts[r], cuts[r + 1])
        seg = {k: torch.from_numpy(np.ascontiguousarray(inp[k][:, sl])) for k in ("x", "dt", "B", "C")}
        for k in ("x", "B", "C"):
            seg[k] = seg[k].to(io_t)
        seg = {k: v.to(dev) for k, v in seg.items()}
        dims = S.dims_of(seg["x"], seg["B"], seg["C"])
        ranks.append(dict(seg=seg, dims=dims, ws=S.workspace_for(dims, Q),
                          cws=torch.empty(S.ssd_cp_workspace_size(dims), dtype=torch.uint8,
                                          device=dev),
                          y=torch.empty_like(seg["x"]),
                          hl=torch.empty((b, H, N, P), dtype=torch.float32, device=dev),
                          hf=torch.empty((b, H, N, P), dtype=torch.float32, device=dev),
                          decay=torch.empty((b, H), dtype=torch.float32, device=dev)))
    decays = torch.empty((R, b, H), dtype=torch.float32, device=dev)
    finals = torch.empty((R, b, H, N, P), dtype=torch.float32, device=dev)

    def phase1(r):
        k = ranks[r]
        g = k["seg"]
        S.ssd_fwd(g["x"], g["dt"], A, g["B"], g["C"], D, h0 if r == 0 else None, Q, k["y"],
                  k["hl"], k["ws"], True, stream, k["dims"])
        S.ssd_cp_segment_decay(g["dt"], A, k["decay"], k["cws"], k["dims"], stream=stream)

    def gather():
        with torch.cuda.stream(stream):
            for r in range(R):
                decays[r].copy_(ranks[r]["decay"])
                finals[r].copy_(ranks[r]["hl"])

    def phase2(r):
        k = ranks[r]
        g = k["seg"]
        S.ssd_cp_correct(R, r, decays, finals, g["dt"], A, g["C"], k["y"], k["hf"], k["cws"],
                         k["dims"], stream=stream)

    with torch.cuda.stream(stream):
        for r in range(R):
            phase1(r)
        gather()
        for r in range(R):
            phase2(r)
    torch.cuda.synchronize()
    S.ssd_check_device_error(stream)
    reps = 10

    def timed(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        with torch.cuda.stream(stream):
            g.replay()
            ms, _ = timed_replays(g.replay, reps, stream, max(0.2, args.min_seconds / 4))
        torch.cuda.synchronize()
        return ms

    clocks = ClockSampler(gpu_id_for(dev))
    time.sleep(0.3)
    p1 = [timed(lambda r=r: phase1(r)) for r in range(R)]
    p2 = [timed(lambda r=r: phase2(r)) for r in range(R)]
    clk = clocks.stop()
    crit = max(p1) + max(p2)
    if rank != 0:
        return
    print(json.dumps({
        "metric": "SSD context-parallel prefill, per-rank compute on one GPU "
                  "(Mtok·heads/s if the R ranks ran concurrently, exchange excluded)",
        "value": round(shape.tok_heads / (crit * 1e-3) / 1e6, 2), "unit": UNIT, "n_gpus": 1,
        "ranks_emulated": R, "higher_is_better": True, "vs_baseline": None,
        "dtype": "bf16" if shape.io == synth.BF16 else "f32", "data": "synthetic (seeded PCG64)",
        "config": dict(config_of(args.workload, shape, 1), segments=cuts),
        "phase1_ms": [round(v, 5) for v in p1], "phase2_ms": [round(v, 5) for v in p2],
        "critical_path_ms": round(crit, 5),
        "exchange": "not measured: one GPU per call (per rank: decay [b,H] and final state "
                    "[b,H,N,P] float32, %d bytes)" % (4 * b * H * (1 + N * P)),
        "clocks": clk}), flush=True)


def measure_multistep(args, world, rank, dev, verify=False, chains=1, min_s=1.0, e2e=True,
                      draft=False):
    """The speculative chain: each call continues from the previous call's h_j
    (ssd_multistep) or from the next cache it stored (ssd_verify; with draft,
    the draft model's step: the previous call's K drafts, j of them accepted,
    folded into the cache and one new token decoded).  The
    1000-call chain is captured in a CUDA graph and replayed until >= min_s;
    ms per call = median replay time / calls.  With chains > 1, that many
    independent chains (own states, the same drafts) run interleaved, call i of
    every chain before call i + 1 of any: each call's cached state was then
    written (chains - 1) calls earlier, which at 128 MB a call is beyond the
    L2 for chains >= 3, so the states come from DRAM."""
    import torch
    from state_space_model_09_b300 import ssd as S

    shape = synth.WORKLOADS["multistep_k8"]
    verify = verify or draft
    work = multistep_work(shape, verify, draft)
    inp = synth.make_multistep_inputs(shape, synth.WORKLOAD_SEEDS["multistep_k8"] + 17 * rank)
    bf = torch.bfloat16
    X = torch.from_numpy(inp["x"]).to(bf).to(dev)
    DT = torch.from_numpy(inp["dt"]).to(dev)
    BB = torch.from_numpy(inp["B"]).to(bf).to(dev)
    CC = torch.from_numpy(inp["C"]).to(bf).to(dev)
    J = torch.from_numpy(inp["j"]).to(dev)
    A = torch.from_numpy(inp["A"]).to(dev)
    D = torch.from_numpy(inp["D"]).to(dev)
    h0 = torch.from_numpy(inp["h_cache"]).to(dev)
    st = [dict(bufs=[torch.empty_like(h0), torch.empty_like(h0)], hK=torch.empty_like(h0),
               Y=torch.empty_like(X[0])) for _ in range(chains)]
    dims = S.dims_of(X[0], BB[0], CC[0])
    steps = shape.steps
    stream = torch.cuda.Stream(dev)
    J0 = torch.zeros_like(J[0])
    if draft:  # the new token of each call: the first of its drafts, contiguous
        X1, DT1, BB1, CC1 = (t[:, :, :1].contiguous() for t in (X, DT, BB, CC))
        for c in st:
            c["Y"] = torch.empty_like(X1[0])

    def chain():
        cur = [h0] * chains
        for i in range(steps):
            for c in range(chains):
                nxt = st[c]["bufs"][i % 2]
                if verify:
                    # fused recompute + verify + cache: the cache is the state
                    # before the previous drafts, of which J[i-1] were accepted
                    p = i - 1 if i > 0 else 0
                    if draft:
                        S.ssd_verify(X[p], DT[p], BB[p], J[i - 1] if i > 0 else J0, X1[i],
                                     DT1[i], A, BB1[i], CC1[i], D, cur[c], st[c]["Y"], nxt,
                                     stream=stream)
                    else:
                        S.ssd_verify(X[p], DT[p], BB[p], J[i - 1] if i > 0 else J0, X[i], DT[i],
                                     A, BB[i], CC[i], D, cur[c], st[c]["Y"], nxt, stream=stream)
                else:
                    S.ssd_multistep(X[i], DT[i], A, BB[i], CC[i], D, cur[c], J[i], st[c]["Y"],
                                    nxt, st[c]["hK"], stream=stream, dims=dims)
                cur[c] = nxt

    with torch.cuda.stream(stream):
        chain()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // 3)):
            g.replay()
    torch.cuda.synchronize()
    S.ssd_check_device_error(stream)
    clocks = ClockSampler(gpu_id_for(dev))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ms_call, reps = timed_replays(g.replay, steps * chains, stream, min_s)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_call = max_over_ranks(ms_call, world, dev)
    S.ssd_check_device_error(stream)
    out = {"ms": ms_call, "repeats": reps, "clocks": clk, "work": work,
           "launches": steps * chains * reps}
    del g
    if e2e:
        out["e2e"] = e2e_multistep(S, inp, A, D, h0, dims, stream, world, dev, verify,
                                   100)
    return out


def e2e_multistep(S, inp, A, D, h0, dims, stream, world, dev, verify, ke):
    """End to end through the public API, as a decoder's serving loop runs it:
    each call's drafts (x, dt, B, C) and accepted count j are copied in from
    pinned host memory on one stream, the call runs on another and its y is
    read back to pinned host memory on a third; the recurrent state stays
    resident on the device, as a decoder's cache does.  The ke calls with all
    their copies are captured once in a CUDA graph (as a decoder captures its
    step) and the graph is replayed; ms per call = replay time / ke."""
    import torch
    bf = torch.bfloat16
    hx = {k: torch.from_numpy(inp[k][:ke]).pin_memory() for k in ("dt", "j")}
    for k in ("x", "B", "C"):
        hx[k] = torch.from_numpy(inp[k][:ke]).to(bf).pin_memory()
    # three device slots: a verify call also reads the previous call's drafts
    ns = 3
    dxs = [{k: torch.zeros_like(v[0], device=dev) for k, v in hx.items()} for _ in range(ns)]
    ys = [torch.empty(hx["x"][0].shape, dtype=bf, device=dev) for _ in range(2)]
    hys = [torch.empty(hx["x"][0].shape, dtype=bf, pin_memory=True) for _ in range(2)]
    bufs = [torch.empty_like(h0), torch.empty_like(h0)]
    hK = torch.empty_like(h0)
    J0 = torch.zeros(h0.shape[0], dtype=torch.int32, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    fork = torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in range(ns)]
    ev_used = [torch.cuda.Event() for _ in range(ns)]
    ev_y = [torch.cuda.Event() for _ in range(2)]
    ev_ydone = [torch.cuda.Event() for _ in range(2)]

    def chain():
        # every wait is on an event recorded earlier in the same chain (or
        # on the fork), so the chain can be captured
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        cur = h0
        for i in range(ke):
            k, kp = i % ns, (i - 1) % ns
            dx, dp = dxs[k], dxs[kp]
            if i >= ns:
                s_in.wait_event(ev_used[k])  # calls i - 3 and i - 2 are done with this slot
            with torch.cuda.stream(s_in):
                for name in ("x", "dt", "B", "C", "j"):
                    dx[name].copy_(hx[name][i], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_ydone[i % 2])  # y buffer read back
            yy, nxt = ys[i % 2], bufs[i % 2]
            if verify:
                S.ssd_verify(dp["x"], dp["dt"], dp["B"], dp["j"] if i > 0 else J0, dx["x"],
                             dx["dt"], A, dx["B"], dx["C"], D, cur, yy, nxt, stream=stream)
            else:
                S.ssd_multistep(dx["x"], dx["dt"], A, dx["B"], dx["C"], D, cur, dx["j"], yy,
                                nxt, hK, stream=stream, dims=dims)
            ev_used[k].record(stream)
            ev_used[kp].record(stream)  # a verify call read the previous call's slot too
            ev_y[i % 2].record(stream)
            s_out.wait_event(ev_y[i % 2])
            with torch.cuda.stream(s_out):
                hys[i % 2].copy_(yy, non_blocking=True)
                ev_ydone[i % 2].record(s_out)
            cur = nxt
        for k2 in range(2):
            stream.wait_event(ev_ydone[k2])

    with torch.cuda.stream(stream):
        chain()  # eager once: the library and the copies are warm
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(reps):
            g.replay()
        f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / (reps * ke), world, dev)
    h2d = sum(v[0].numel() * v[0].element_size() for v in hx.values())
    d2h = hys[0].numel() * hys[0].element_size()
    del g
    return {"ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def multistep_fields(m, world, pk, traffic):
    work = m["work"]
    gbs = work["bytes"] / (m["ms"] * 1e-3) / 1e9
    f = {"value": round(world * work["tok_heads"] / (m["ms"] * 1e-3) / 1e6, 2),
         "ms_per_step": round(m["ms"], 6), "repeats": m["repeats"],
         "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                      "frac": round(gbs / pk["hbm"], 4),
                      "frac_vs_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                      "traffic": traffic, "kernel": "multistep_kernel",
                      "algorithmic_bytes": work["bytes"],
                      "peak_source": pk["source"] + " (burst)"},
         "clocks": m["clocks"]}
    if traffic:
        f["roofline"]["dram_frac"] = round(traffic / (m["ms"] * 1e-3) / 1e9 / pk["hbm"], 4)
    if "e2e" in m:
        e = m["e2e"]
        f["e2e"] = {"value": round(world * work["tok_heads"] / (e["ms_per_step"] * 1e-3) / 1e6, 2),
                    "unit": UNIT, "h2d_bytes_per_step": e["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": e["d2h_bytes_per_step"],
                    "ms_per_step": round(e["ms_per_step"], 4)}
    return f


def multistep_summary(args, world, rank, local):
    """multistep_k8 inside the prefill line: the chain (states L2-warm), the
    same chain with cold states (four interleaved chains), and the fused
    verify chain, each with its own clocks; the oracle chain as CPU baseline."""
    import torch
    dev = torch.device("cuda", local)
    pk = peaks()
    shape = synth.WORKLOADS["multistep_k8"]
    m = measure_multistep(args, world, rank, dev, min_s=args.min_seconds)
    out = dict(config_of("multistep_k8", shape, world),
               **multistep_fields(m, world, pk, measured_traffic("multistep_kernel", "multistep_k8")))
    out["timing"] = ("CUDA graph of the 1000-call chain, replayed until >= 1 s; each call reads "
                     "the h_j the previous call wrote (L2-warm: states 3 x 42 MB per call)")
    torch.cuda.empty_cache()
    mc = measure_multistep(args, world, rank, dev, chains=4, min_s=args.min_seconds, e2e=False)
    out["cold_states"] = dict(multistep_fields(mc, world, pk, None),
                              timing="four independent chains interleaved: each call's cached "
                                     "state was written three calls (~385 MB) earlier")
    torch.cuda.empty_cache()
    mv = measure_multistep(args, world, rank, dev, verify=True, min_s=args.min_seconds, e2e=False)
    out["verify"] = dict(multistep_fields(mv, world, pk,
                                          measured_traffic("multistep_kernel_verify", "multistep_k8")),
                         call="ssd_verify")
    out["verify"]["roofline"]["kernel"] = "multistep_kernel (verify mode)"
    torch.cuda.empty_cache()
    md = measure_multistep(args, world, rank, dev, draft=True, min_s=args.min_seconds, e2e=False)
    out["draft"] = dict(multistep_fields(md, world, pk,
                                         measured_traffic("multistep_kernel_draft", "multistep_k8")),
                        call="ssd_verify, K = 1 after 8 previous drafts (draft-model step)")
    out["draft"]["roofline"]["kernel"] = "multistep_kernel (verify mode, K = 1)"
    if not args.no_cpu_baseline:
        value, _, cores, sample = oracle_multistep_chain(12, 6.0)
        out["cpu_baseline"] = {"value": round(value, 4), "unit": UNIT, "cores": cores,
                               "kind": "oracle", "sample": sample}
    return out


def run_multistep(args, world, rank, local):
    """--workload multistep_k8: one step = one call of the speculative chain."""
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = synth.WORKLOADS["multistep_k8"]
    m = measure_multistep(args, world, rank, dev, verify=args.verify, chains=args.chains,
                          min_s=args.min_seconds, draft=args.draft, e2e=not args.draft)
    if rank != 0:
        return
    pk = peaks()
    f = multistep_fields(m, world, pk, None if args.chains > 1 else measured_traffic(
        "multistep_kernel_draft" if args.draft else
        "multistep_kernel_verify" if args.verify else "multistep_kernel", "multistep_k8"))
    metric = ("SSD draft-model step Mtok·heads/s (8 previous drafts folded + 1 new token, "
              "1000-step chain)" if args.draft else
              "SSD fused verify decode Mtok·heads/s (recompute + K=8 verify + cache, "
              "1000-step speculative chain)" if args.verify else MULTISTEP_METRIC)
    line = {"metric": metric, "value": f.pop("value"), "unit": UNIT, "n_gpus": world,
            "steps": shape.steps * args.chains, "warmup": args.warmup,
            "ms_per_step": f.pop("ms_per_step"), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded PCG64)",
            "config": config_of("multistep_k8", shape, world),
            "timing": "CUDA graph of the chain (%d interleaved), replayed until >= 1 s; %s"
                      % (args.chains, "ssd_verify (K = 1)" if args.draft else
                         "ssd_verify" if args.verify else "ssd_multistep"),
            "gpu_launches": m["launches"]}
    line.update(f)
    if world == 1 and not args.no_cpu_baseline and not args.draft:
        value, _, cores, sample = oracle_multistep_chain(40, 20.0)
        line["cpu_baseline"] = {"value": round(value, 4), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line, ensure_ascii=False), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba2_2p7b", choices=list(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="the default workload's line without the other workloads")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="replay the timed block until this much device time is measured")
    ap.add_argument("--verify", action="store_true",
                    help="multistep_k8: time the chain of fused recompute + verify calls")
    ap.add_argument("--draft", action="store_true",
                    help="multistep_k8: time the draft-model step (fused verify call, K = 1)")
    ap.add_argument("--chains", type=int, default=1,
                    help="multistep_k8: independent chains interleaved (3+ keeps states cold)")
    ap.add_argument("--window", type=int, default=0,
                    help="prefill through ssd_fwd_sequential with windows of this many tokens")
    ap.add_argument("--cp", type=int, default=0,
                    help="prefill: context parallelism's per-rank compute for this many "
                         "ranks, emulated one after another on one GPU")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "multistep_k8":
        if args.impl == "reference":
            # the oracle is host code: rank 0 alone runs it, other ranks exit 0
            if int(os.environ.get("RANK", "0")) == 0:
                run_reference_multistep(args)
            return
        world, rank, local = dist_setup()
        run_multistep(args, world, rank, local)
        return
    shape = synth.WORKLOADS[args.workload]
    work = fwd_work(shape)
    if args.impl == "reference":
        # the oracle is host code: rank 0 alone runs it, other ranks exit 0
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args, shape, work)
        return
    world, rank, local = dist_setup()
    if args.window > 0:
        run_sequential(args, shape, world, rank, local)
        return
    if args.cp > 0:
        run_cp(args, shape, world, rank, local)
        return
    run_ours(args, shape, world, rank, local)


if __name__ == "__main__":
    main()
