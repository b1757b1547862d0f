"""Benchmark of the gated delta rule layer on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill (pre-pass, block kernel, varlen/tail handling) of one 4096-token
    sequence, Hk=16, Hv=32, dk=dv=128, bf16 I/O, fp32 state, chunk 64, zero
    initial state;
  * one decode step of 128 sequences with the same heads (fp32 state
    ~N(0, 0.02), in place).

`value` is the prefill throughput (Mtok/s); the decode step's time is under
"decode" (us/step). Both are timed with CUDA events on the stream the
kernels are launched on, L2 flushed (a 256 MiB write) before each timed
launch. `--impl reference` times the fp64 CPU oracle on the same workload
(a bounded sample) instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_PREFILL, HK, HV, DK, DV, CHUNK = 4096, 16, 32, 128, 128, 64
N_DECODE = 128
METRIC = "Gated-DeltaNet prefill Mtok/s & decode µs/step (1 GB300); % of roofline"
WORKLOAD = ("prefill B=1 T=4096 Hk=16 Hv=32 dk=dv=128 chunk=64 bf16, zero state; "
            "then decode step N=128 same heads, fp32 state")

# algorithmic bytes/flops (per token / per sequence)
IO_BYTES_PER_TOKEN = (HK * DK * 2 * 2) + (HV * DV * 2) * 2 + HV * 2 * 2  # q,k + v,out + g,b
STATE_BYTES = HV * DV * DK * 4
PREFILL_BYTES = T_PREFILL * IO_BYTES_PER_TOKEN + STATE_BYTES  # state written once (zero state in)
PREFILL_FLOPS_PER_TOKEN = HV * (5 * 2 * CHUNK * DK + 3 * 2 * DK * DV)  # chunk GEMMs (dk == dv)
DECODE_BYTES_PER_SEQ = 2 * STATE_BYTES + IO_BYTES_PER_TOKEN
# DRAM bytes per launch from the committed ncu captures (profiles/); None once a kernel
# has changed since its capture.
TRAFFIC = {"prefill": 129.6e6, "decode": 480.2e6, "scan": 488.7e6}
# nominal GB300 figures, reported beside the measured denominators
NOMINAL_HBM_GBS, NOMINAL_BF16_TFLOPS = 7900.0, 2250.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.t0 = time.time()
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        # wait for the first sample so that the timed region is covered
        deadline = time.time() + 5.0
        while time.time() < deadline and os.path.getsize(self.file.name) == 0:
            time.sleep(0.02)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, device):
    """Element-wise maximum over all ranks (the slowest replica sets the job's time)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world, units_per_rank, seconds):
    """Whole-job rate of `world` replicas that each process `units_per_rank` units, timed by
    the slowest: every rank runs its own copy of the workload (weak scaling, no exchange)."""
    return world * units_per_rank / seconds


def make_inputs(dev):
    from gated_deltanet_linear_delta_gb300 import inputs
    pb = inputs.prefill_4k(seed=0)
    q, k, v, g, b, st = inputs.make_decode_inputs(N_DECODE, seed=0)
    return pb, (q[0], k[0], v[0], g[0], b[0], st)


def run_ours(args, rank, world):
    import gated_deltanet_linear_delta_gb300 as gdn
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pb, dec = make_inputs(dev)
    d = pb.to(dev)
    out = torch.empty(T_PREFILL, HV, DV, dtype=torch.bfloat16, device=dev)
    st_out = torch.empty(1, HV, DV, DK, device=dev)
    qd, kd, vd, gd, bd = (x.to(dev) for x in dec[:5])
    state0 = dec[5].to(dev)
    dstate = state0.clone()
    dout = torch.empty(N_DECODE, HV, DV, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        gdn.gdn_prefill(d.q, d.k, d.v, d.g, d.b, None, st_out, out, None, B=1, chunk=CHUNK, stream=stream)

    def decode():
        gdn.gdn_decode_step(qd, kd, vd, gd, bd, dstate, dout, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        prefill()
        flush.fill_(2.0)
        decode()
    torch.cuda.synchronize()
    if gdn.gdn_get_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status reports an inconsistency")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(dev.index) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(1.0)
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            flush.fill_(2.0)
            ev[i][2].record(stream)
            decode()
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    pre_mean, dec_mean = sum(pre_ms) / len(pre_ms), sum(dec_ms) / len(dec_ms)
    step_ms = pre_mean + dec_mean
    if world > 1:
        pre_mean, dec_mean, step_ms = max_over_ranks([pre_mean, dec_mean, step_ms], dev)

    # decode batch sweep (same kernel, smaller batches), L2 flushed before each launch
    sweep = {}
    for n in (() if args.only_headline else (1, 8, 32, 128)):
        times = []
        for i in range(args.warmup + args.steps):
            flush.fill_(3.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gdn.gdn_decode_step(qd[:n], kd[:n], vd[:n], gd[:n], bd[:n], dstate[:n], dout[:n], stream=stream)
            e1.record(stream)
            if i >= args.warmup:
                times.append((e0, e1))
        torch.cuda.synchronize()
        us = 1e3 * sum(a.elapsed_time(b) for a, b in times) / len(times)
        sweep[str(n)] = round(us, 3)

    if args.only_headline:  # the timed step alone (for profiling runs)
        graph = other = copy_ref = multi = e2e = None
    else:
        graph = decode_graph_sweep(gdn, (qd, kd, vd, gd, bd), dstate, dout, stream)
        other = other_prefill_workloads(args, gdn, flush, stream, dev)
        copy_ref = copy_reference(args, flush, stream, dev)
        multi = multi_token_decode(args, gdn, flush, stream, dev)
        e2e = measure_e2e(args, gdn, pb, dec, dev, stream)
    hbm, bf16, src = peaks()
    pre_s = pre_mean / 1e3
    achieved_gbs = PREFILL_BYTES / pre_s / 1e9
    achieved_tfs = PREFILL_FLOPS_PER_TOKEN * T_PREFILL / pre_s / 1e12
    roof_time = max(PREFILL_BYTES / (hbm * 1e9), PREFILL_FLOPS_PER_TOKEN * T_PREFILL / (bf16 * 1e12))
    roof_nom = max(PREFILL_BYTES / (NOMINAL_HBM_GBS * 1e9),
                   PREFILL_FLOPS_PER_TOKEN * T_PREFILL / (NOMINAL_BF16_TFLOPS * 1e12))
    dec_bytes = N_DECODE * DECODE_BYTES_PER_SEQ
    dec_gbs = dec_bytes / (dec_mean / 1e3) / 1e9
    path = gdn.gdn_prefill_path(1, T_PREFILL, HK, HV, DK, DV, CHUNK, gdn.GDN_BF16)
    # the tensor-core path launches a planning kernel then the block kernel
    prefill_launches = 2 if path == 1 else 1
    clocks = clk.summary()
    value = job_throughput(world, T_PREFILL, pre_s) / 1e6
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "Mtok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, g=-softplus(N(0,1)), beta logits N(0,1))",
        "config": {"workload": WORKLOAD, "prefill_tokens": T_PREFILL, "decode_batch": N_DECODE,
                   "Hk": HK, "Hv": HV, "dk": DK, "dv": DV, "chunk": CHUNK,
                   "l2": "flushed: 256 MiB write before each timed launch",
                   "prefill_kernel": {1: "tcgen05 ring kernel (block preparation + state chains)",
                                      0: "CUDA-core block kernel"}.get(path, path),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "prefill": {"ms": round(pre_mean, 5), "Mtok_s": round(T_PREFILL / pre_s / 1e6, 3),
                    "GB_s": round(achieved_gbs, 1), "TFLOP_s": round(achieved_tfs, 2),
                    "roofline_ms": round(roof_time * 1e3, 5), "frac_of_roofline": round(roof_time / pre_s, 4),
                    "frac_of_nominal_roofline": round(roof_nom / pre_s, 4)},
        "decode": {"value": round(dec_mean * 1e3, 3), "unit": "us/step", "batch": N_DECODE,
                   "higher_is_better": False, "GB_s": round(dec_gbs, 1),
                   "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                                "frac": round(dec_gbs / hbm, 4), "traffic": TRAFFIC["decode"],
                                "peak_source": src, "frac_of_nominal": round(dec_gbs / NOMINAL_HBM_GBS, 4)},
                   "sweep_us": sweep, "graph": graph, "multi_token": multi, "copy_reference": copy_ref},
        "other_workloads": other,
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved_gbs / hbm, 4), "traffic": TRAFFIC["prefill"], "peak_source": src,
                     "kernel": "prefill", "frac_of_nominal": round(achieved_gbs / NOMINAL_HBM_GBS, 4)},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": (prefill_launches + 1) * args.steps,
        "wall_s_timed_region": round(wall, 4),
    }
    return line


def copy_reference(args, flush, stream, dev):
    """The decode step with its arithmetic removed: a device copy that reads and writes the same
    state bytes (128 sequences x 32 heads x 64 KiB), L2 flushed, CUDA events. This is what the
    decode kernel's memory traffic can reach on this GPU, measured in the same run."""
    src = torch.empty(N_DECODE * STATE_BYTES // 4, dtype=torch.float32, device=dev).normal_()
    dst = torch.empty_like(src)
    ev = []
    for i in range(args.warmup + min(args.steps, 50)):
        flush.fill_(6.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src)
        e1.record(stream)
        if i >= args.warmup:
            ev.append((e0, e1))
    torch.cuda.synchronize()
    us = 1e3 * sorted(a.elapsed_time(c) for a, c in ev)[len(ev) // 2]
    nbytes = 2 * N_DECODE * STATE_BYTES
    return {"us": round(us, 3), "GB_s": round(nbytes / us / 1e3, 1), "bytes": nbytes,
            "what": "torch copy of the decode state bytes (read + write), L2 flushed"}


def other_prefill_workloads(args, gdn, flush, stream, dev, reps=5):
    """The other prefill workloads (reported, not the headline): one 32768-token and one
    131072-token sequence with a seeded initial state, and 16 packed sequences of lengths
    U{256..16384} with their own states. L2 flushed before each launch; median of `reps`."""
    from gated_deltanet_linear_delta_gb300 import inputs
    hbm, bf16, src = peaks()
    cases = [("T=32768, seeded state", lambda: inputs.prefill_long(T=32768)),
             ("T=131072, seeded state", lambda: inputs.prefill_long(T=131072)),
             ("varlen 16 seqs U{256..16384}, seeded states", inputs.prefill_varlen)]
    res = {}
    for name, make in cases:
        b = make().to(dev)
        ntok = int(b.q.shape[0])
        out = torch.empty(b.v.shape, dtype=torch.bfloat16, device=dev)
        so = torch.empty(b.B, HV, DV, DK, device=dev)
        ev = []
        for i in range(2 + reps):
            flush.fill_(5.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gdn.gdn_prefill(b.q, b.k, b.v, b.g, b.b, b.state, so, out, b.cu_seqlens, B=b.B,
                            T=None if b.cu_seqlens is not None else b.T, chunk=CHUNK, stream=stream)
            e1.record(stream)
            if i >= 2:
                ev.append((e0, e1))
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(c) for a, c in ev)[len(ev) // 2]
        nbytes = ntok * IO_BYTES_PER_TOKEN + 2 * b.B * STATE_BYTES
        roof = max(nbytes / (hbm * 1e9), ntok * PREFILL_FLOPS_PER_TOKEN / (bf16 * 1e12))
        roof_nom = max(nbytes / (NOMINAL_HBM_GBS * 1e9), ntok * PREFILL_FLOPS_PER_TOKEN / (NOMINAL_BF16_TFLOPS * 1e12))
        res[name] = {"tokens": ntok, "ms": round(ms, 4), "Mtok_s": round(ntok / ms / 1e3, 3),
                     "GB_s": round(nbytes / ms / 1e6, 1), "roofline_ms": round(roof * 1e3, 4),
                     "frac_of_roofline": round(roof * 1e3 / ms, 4),
                     "frac_of_nominal_roofline": round(roof_nom * 1e3 / ms, 4)}
        if b.cu_seqlens is not None:  # then 128 decode steps on the sequences' final states
            res[name]["then_128_decode_steps"] = decode_after_prefill(gdn, so, stream, dev, steps=128)
        del b, out, so
    return res


def decode_after_prefill(gdn, states, stream, dev, steps=128):
    """`steps` decode steps on the states a prefill left (in place), captured once in a CUDA graph
    and replayed; fresh seeded token inputs per step; us per step and the rate of the
    bytes moved (each step reads and writes every state once)."""
    from gated_deltanet_linear_delta_gb300 import inputs
    n = states.shape[0]
    q, k, v, g, b, _ = inputs.make_decode_inputs(n, seed=7, steps=steps)
    q, k, v, g, b = (x.to(dev) for x in (q, k, v, g, b))
    out = torch.empty(steps, n, HV, DV, dtype=torch.bfloat16, device=dev)
    st = states.clone()

    def run():
        for t in range(steps):
            gdn.gdn_decode_step(q[t], k[t], v[t], g[t], b[t], st, out[t])
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        graph.replay()
        ev[0].record(stream)
        for _ in range(3):
            graph.replay()
        ev[1].record(stream)
    torch.cuda.synchronize()
    us = 1e3 * ev[0].elapsed_time(ev[1]) / (3 * steps)
    nbytes = n * DECODE_BYTES_PER_SEQ
    return {"sequences": n, "us_per_step": round(us, 3), "GB_s": round(nbytes / us / 1e3, 1),
            "l2": f"warm: the {n} states ({nbytes / 1e6:.0f} MB) stay in L2 between steps, so this is "
                  "not an HBM fraction"}


def multi_token_decode(args, gdn, flush, stream, dev, N=128, T=4):
    """N sequences x T tokens each (checking T speculated tokens) through gdn_prefill, which runs
    them as a token scan (one pass over each state), L2 flushed before each launch."""
    from gated_deltanet_linear_delta_gb300 import inputs
    hbm, _, src = peaks()
    b = inputs.make_batch(B=N, T=T, Hk=HK, Hv=HV, dk=DK, dv=DV, dtype="bf16", chunk=CHUNK, seed=0,
                          init_state=True).to(dev)
    out = torch.empty(b.v.shape, dtype=torch.bfloat16, device=dev)
    times = []
    for i in range(args.warmup + args.steps):
        flush.fill_(4.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gdn.gdn_prefill(b.q, b.k, b.v, b.g, b.b, b.state, b.state, out, None, B=N, T=T, chunk=CHUNK,
                        stream=stream)
        e1.record(stream)
        if i >= args.warmup:
            times.append((e0, e1))
    torch.cuda.synchronize()
    us = 1e3 * sum(a.elapsed_time(c) for a, c in times) / len(times)
    nbytes = N * (2 * STATE_BYTES + T * IO_BYTES_PER_TOKEN)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"sequences": N, "tokens_per_sequence": T, "us": round(us, 3),
            "kernel": {2: "token scan"}.get(gdn.gdn_prefill_path(N, T, HK, HV, DK, DV, CHUNK, gdn.GDN_BF16)),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "bytes": nbytes, "traffic": TRAFFIC["scan"],
                         "peak_source": src}}


def decode_graph_sweep(gdn, qkvgb, dstate, dout, stream, G=32, reps=20):
    """Decode steps back to back (the state updated in place, L2 warm): G launches issued eagerly
    against the same G launches captured once in a CUDA graph and replayed; us per step."""
    res = {"steps_per_graph": G, "l2": "warm (consecutive steps, no flush)"}
    for n in (1, 8, 32, 128):
        # views taken once, outside the timed loops: eager_us is the binding's call plus the launch
        qn, kn, vn, gn, bn, sn, on = (x[:n] for x in (*qkvgb, dstate, dout))

        def steps():
            for _ in range(G):
                gdn.gdn_decode_step(qn, kn, vn, gn, bn, sn, on)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            steps()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steps()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        with torch.cuda.stream(stream):
            for _ in range(3):
                steps()
                graph.replay()
            ev[0].record(stream)
            for _ in range(reps):
                steps()
            ev[1].record(stream)
            ev[2].record(stream)
            for _ in range(reps):
                graph.replay()
            ev[3].record(stream)
        torch.cuda.synchronize()
        res[str(n)] = {"eager_us": round(1e3 * ev[0].elapsed_time(ev[1]) / (reps * G), 3),
                       "graph_us": round(1e3 * ev[2].elapsed_time(ev[3]) / (reps * G), 3)}
        del graph
    res["host_us"] = host_call_cost(gdn, qkvgb, dstate, dout)
    return res


def host_call_cost(gdn, qkvgb, dstate, dout, calls=2000):
    """Host time per call (no GPU wait): a bare ctypes call into the library that does no CUDA
    work (gdn_prefill_path), the library's gdn_decode_step reached through ctypes with
    prepared integer arguments, and the Python binding's gdn_decode_step (argument
    marshalling included), for one sequence."""
    lib = gdn.library()
    n = 1
    qn, kn, vn, gn, bn, sn, on = (x[:n] for x in (*qkvgb, dstate, dout))
    hk, dk = qn.shape[1], qn.shape[2]
    hv, dv = vn.shape[1], vn.shape[2]
    raw = torch.cuda.current_stream().cuda_stream
    ptrs = [t.data_ptr() for t in (qn, kn, vn, gn, bn, sn, on)]

    def per_call(fn):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        dt = time.perf_counter() - t0
        torch.cuda.synchronize()
        return round(1e6 * dt / calls, 3)
    return {"bare_ctypes_us": per_call(lambda: lib.gdn_prefill_path(1, 64, hk, hv, dk, dv, 64, gdn.GDN_BF16)),
            "ctypes_decode_us": per_call(lambda: lib.gdn_decode_step(*ptrs, n, hk, hv, dk, dv, gdn.GDN_BF16, raw)),
            "binding_decode_us": per_call(lambda: gdn.gdn_decode_step(qn, kn, vn, gn, bn, sn, on)),
            "calls": calls}


E2E_FRAGMENT = 1024  # tokens per fragment of the host-to-host prefill


def measure_e2e(args, gdn, pb, dec, dev, stream):
    """The same prefill through the public host-memory entry point (gdn_prefill_from_host):
    inputs in pinned host memory are copied in, outputs and final state copied back, all inside
    the timed region; the library overlaps the copies with the computation fragment by fragment."""
    host = {n: getattr(pb, n).pin_memory() for n in ("q", "k", "v", "g", "b")}
    dbuf = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    dbuf["out"] = torch.empty(T_PREFILL, HV, DV, dtype=torch.bfloat16, device=dev)
    dbuf["state"] = torch.empty(HV, DV, DK, device=dev)
    h_out = torch.empty(dbuf["out"].shape, dtype=torch.bfloat16).pin_memory()
    h_st = torch.empty(HV, DV, DK).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = h_out.numel() * h_out.element_size() + h_st.numel() * h_st.element_size()
    times = []
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        gdn.gdn_prefill_from_host(host["q"], host["k"], host["v"], host["g"], host["b"], None, h_st, h_out, dbuf,
                                  chunk=CHUNK, fragment=E2E_FRAGMENT, stream=stream)
        stream.synchronize()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    mean = sum(times) / len(times)
    return {"value": round(T_PREFILL / mean / 1e6, 3), "unit": "Mtok/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(mean * 1e3, 4),
            "api": f"gdn_prefill_from_host, fragments of {E2E_FRAGMENT} tokens"}


def cpu_baseline_sample(threads=None, tokens=T_PREFILL, steps=1, warmup=0):
    """The fp64 oracle (token scan, as it stands), all 32 heads, on the first `tokens` tokens of
    the prefill prompt, one thread per (sequence, head) unit up to `threads`."""
    import oracle
    from gated_deltanet_linear_delta_gb300 import inputs
    pb = inputs.prefill_4k(seed=0)
    threads = threads or (os.cpu_count() or 1)
    sl = slice(0, tokens)
    args = [x[sl].double().numpy() for x in (pb.q, pb.k, pb.v, pb.g, pb.b)]
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        oracle.gdn_sequential(*args, None, None, B=1, threads=threads)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    dt = sum(times) / len(times)
    # one thread on a quarter of the sample (the per-core rate, next to the multi-core one)
    t1_tokens = max(tokens // 4, 1)
    s1 = slice(0, t1_tokens)
    t0 = time.perf_counter()
    oracle.gdn_sequential(*[x[s1] for x in args], None, None, B=1, threads=1)
    dt1 = time.perf_counter() - t0
    return {"value": round(tokens / dt / 1e6, 6), "unit": "Mtok/s", "cores": min(threads, HV), "kind": "oracle",
            "sample": f"{tokens} tokens of the 4096-token prompt, all 32 value heads, fp64 token scan",
            "seconds_per_pass": round(dt, 3), "cpu_model": cpu_model(),
            "single_thread": {"value": round(t1_tokens / dt1 / 1e6, 6), "unit": "Mtok/s",
                              "sample": f"{t1_tokens} tokens, all 32 value heads, one thread"}}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-headline", action="store_true",
                    help="time the prefill + decode step only (no other workloads, no e2e): for profiling")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the oracle on the host cores; rank 0 only
        if rank != 0:
            return
        base = cpu_baseline_sample(steps=args.steps, warmup=args.warmup)
        line = {"metric": METRIC, "value": base["value"], "unit": "Mtok/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "ms_per_step": round(1e3 * base["seconds_per_pass"], 3),
                "config": {"workload": WORKLOAD, "reference": "fp64 CPU oracle (token scan), bounded sample"},
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline_sample()
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
