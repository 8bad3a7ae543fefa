"""Benchmark of the quantized-KV decode path on GB300.

Workload (the headline configuration): GQA decode, batch 8, 32 query heads over 8 KV heads,
head dim 128, context 32768, bf16 K/V with Student-t(3) coordinates scaled to unit variance,
N(0,1) queries; schemes Plain-KV, TQ-KV, KQV and QKQV at n = 4 bits per coordinate.
One step = for each scheme: quantize-append one new token per (batch, KV head) at position
T-1 (the cache is pre-filled with T-1 tokens) and decode attention of every query head over the
T cached tokens.  Each scheme's cache (285-294 MB) is larger than L2 (129 MB) and the four are
visited in turn, so every step streams its caches from HBM.

Metric: cache-tokens/s = sum over schemes of B * H_kv * T / step time (one cache token = one
(batch, KV head, token) record with its K and V).  The roofline object reports the decode
kernels' algorithmic packed bytes / measured decode time against the measured HBM peak.

``--impl reference`` times the float64 CPU oracle on the host cores on a bounded sample of the
same workload (one slab per scheme per step).  Under torchrun every rank runs the full workload
on its own GPU (independent batches, no collective): weak scaling.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention cache-tokens/s and HBM GB/s (% peak); append tok/s"
UNIT = "cache-tokens/s"
WORKLOAD = ("GQA decode B=8 Hq=32 Hkv=8 d=128 T=32768, bf16 Student-t(3) K/V; "
            "Plain-KV, TQ-KV, KQV, QKQV at n=4; step = per scheme: append 1 token per slab + decode")
SCHEMES = [("plain", 4), ("tq", 4), ("kqv", 4), ("qkqv", 4)]

# DRAM bytes (read + write) per decode-kernel launch, from an ncu capture of this workload
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel sources whose
# digest is recorded here; any change to them reports traffic as null until recaptured.
DECODE_SOURCES = ["tq_decode_kernel.cuh", "tq_decode.cu", "tq_device.cuh", "tq_internal.h"]
DECODE_TRAFFIC = {
    "sources_sha256": "14efd43b28817c02554543f9005071bfac8766ab0ff2c0b21c755177770e1b12",
    "bytes_per_launch": {"plain4": 288946944, "tq4": 286169856, "kqv4": 290386432, "qkqv4": 294996992},
}


def decode_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "turboquant_quantized_kv_tq_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic(schemes):
    """Mean ncu DRAM bytes per decode launch over ``schemes``, or None when not captured for the
    current sources."""
    if DECODE_TRAFFIC["sources_sha256"] != decode_sources_digest():
        return None
    vals = [DECODE_TRAFFIC["bytes_per_launch"].get(f"{s}{n}") for s, n in schemes]
    if any(v is None for v in vals):
        return None
    return round(sum(vals) / len(vals))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, device=None):
    """The largest of every rank's ``value`` (the job's time is its slowest rank's); the value
    itself when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank_step, world, ms_per_step):
    """Units all ranks processed per second: every rank does the same work per step (weak
    scaling), and a step lasts as long as the slowest rank's."""
    return world * units_per_rank_step / (ms_per_step * 1e-3)


def record_bytes(scheme, n, d=128, m=128):
    """Packed bytes of one cache record (K and V of one token of one slab)."""
    from turboquant_quantized_kv_tq_gb300.binding import SCHEMES as S, tq_config, tq_config_from_scheme
    c = tq_config()
    tq_config_from_scheme(S[scheme], n, c)
    total = 0
    for cd in (c.k, c.v):
        total += d * cd.bits // 8 + 4
        if cd.qjl:
            total += m // 8 + 2
    return total


def step_launches(scheme, n):
    """Kernels one decode step launches for a scheme at head dim 128: the append (the sketch
    kernel for QJL sides, then the other side's encode if it has none), the query prep and the
    decode."""
    from turboquant_quantized_kv_tq_gb300.binding import SCHEMES as S, tq_config, tq_config_from_scheme
    c = tq_config()
    tq_config_from_scheme(S[scheme], n, c)
    nq = int(bool(c.k.qjl)) + int(bool(c.v.qjl))
    return (2 if nq == 1 else 1) + 2


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def build_caches(inp, device, T):
    """One QuantizedKVCache per scheme, pre-filled with T-1 tokens (untimed)."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    caches = []
    K = torch.from_numpy(inp.K.view(np.int16)).view(torch.bfloat16)
    V = torch.from_numpy(inp.V.view(np.int16)).view(torch.bfloat16)
    chunk = 4096
    for scheme, n in SCHEMES:
        kv = QuantizedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, T, scheme=scheme, n=n, seed=inp.seed, device=device)
        for s in range(0, T - 1, chunk):
            e = min(T - 1, s + chunk)
            kv.append(K[:, :, s:e].to(device), V[:, :, s:e].to(device), [s] * inp.B)
        caches.append(kv)
    torch.cuda.synchronize(device)
    return caches


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from workloads import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    inp = make_inputs("cfg2")
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    caches = build_caches(inp, device, T)
    # the token appended every step (position T-1) and the step's queries
    k_new = torch.from_numpy(inp.K[:, :, T - 1:T].view(np.int16)).view(torch.bfloat16).to(device)
    v_new = torch.from_numpy(inp.V[:, :, T - 1:T].view(np.int16)).view(torch.bfloat16).to(device)
    q = torch.from_numpy(inp.q).to(device)
    outs = [torch.empty_like(q) for _ in caches]
    seq = [T] * B
    start = [T - 1] * B
    for kv in caches:
        kv.workspace(T)
    stream = torch.cuda.current_stream(device)
    n_dec = len(caches)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_dec)]

    def step(timed_events=None):
        # per scheme: the append of the step's token, then the decode; as one library call (the
        # query preparation overlaps the append), or, to time the decode calls alone, as two
        for i, kv in enumerate(caches):
            if timed_events is None and not args.split_step:
                kv.append_decode(k_new, v_new, q, seq, out=outs[i])
                continue
            kv.append(k_new, v_new, start)
            if timed_events is not None:
                timed_events[i][0].record(stream)
            kv.decode(q, seq, out=outs[i])
            if timed_events is not None:
                timed_events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # per-scheme decode times (the roofline's denominators): eager steps with events around
    # every decode call
    dec_ms = [0.0] * n_dec
    n_ev = min(args.steps, 100)
    per_step_events = []
    for _ in range(n_ev):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_dec)]
        step(evs)
        per_step_events.append(evs)
    torch.cuda.synchronize(device)
    for evs in per_step_events:
        for i in range(n_dec):
            dec_ms[i] += evs[i][0].elapsed_time(evs[i][1])
    dec_ms = [x / n_ev for x in dec_ms]

    # the step as one CUDA graph (the same library calls, captured once): the timed loop replays
    # it, so host-side launch overhead does not gap the device work
    graph = None
    if not args.eager:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                step()
            torch.cuda.synchronize(device)
            graph = g
        except Exception as exc:  # fall back to eager steps, and say so
            print(f"graph capture failed, timing eager steps: {exc}", file=sys.stderr)
    run_step = graph.replay if graph is not None else step
    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        run_step()
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    total_ms = max_over_ranks(total_ms, device)
    ms_per_step = total_ms / args.steps
    tokens_per_step = n_dec * B * Hkv * T
    value = whole_job_value(tokens_per_step, world, ms_per_step)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, caches, inp, device, seq, start)

    # ---- append throughput on the prefill chunk of the long-context configuration
    append = run_prefill_append(args, device) if not args.skip_append else None

    # ---- several queries per sequence (G * nq = 8 query columns per KV head) on the first cache
    multi = run_multi_query(caches[0], SCHEMES[0], inp, device, T)

    # ---- chunked prefill over the same caches (dense tensor-core products)
    prefill = run_prefill(args, caches, inp, device, T) if not args.skip_prefill else None

    # ---- the second target configuration (128k context, G = 8), with its own roofline
    long_ctx = run_long_context(args, device) if not args.skip_long_context else None

    peak, peak_kind = measured_peak()
    rec = [record_bytes(s, n) for s, n in SCHEMES]
    dec_bytes = [B * Hkv * T * r for r in rec]
    achieved = sum(dec_bytes) / (sum(dec_ms) * 1e-3) / 1e9
    schemes = {f"{s}{n}": {"decode_us": round(dec_ms[i] * 1e3, 2),
                           "record_bytes": rec[i],
                           "GB_per_s": round(dec_bytes[i] / (dec_ms[i] * 1e-3) / 1e9, 1),
                           "cache_tokens_per_s": round(B * Hkv * T / (dec_ms[i] * 1e-3), 1)}
               for i, (s, n) in enumerate(SCHEMES)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded numpy PCG64; no public dataset)",
        "config": {"workload": WORKLOAD if len(SCHEMES) == 4 else WORKLOAD + " (scheme subset)",
                   "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": d,
                   "context": T, "schemes": [f"{s}-n{n}" for s, n in SCHEMES],
                   "l2": "inputs larger than L2: four caches of 285-294 MB visited per step",
                   "arith": "append fp32; decode scores/readout fp16 MMA operands, fp32 accumulation",
                   "parallelism": f"independent replicas x{world}",
                   "step_launch": "CUDA graph replay of the captured step" if graph is not None else "eager",
                   "step_calls": ("tq_quantize_append + tq_decode_attention per scheme" if args.split_step
                                  else "tq_append_decode_attention per scheme")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": decode_traffic(SCHEMES),
                     "kernel": "decode (query prep + fused split-K decode), all four schemes",
                     "peak_kind": peak_kind},
        "schemes": schemes,
        "e2e": e2e,
        "append": append,
        "multi_query": multi,
        "long_context": long_ctx,
        "prefill": prefill,
        "gpu_launches": args.steps * sum(step_launches(s, n) for s, n in SCHEMES),
        "clocks": clocks,
    }
    if rank == 0 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, caches, budget_s=args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, caches, inp, device, seq, start):
    """Same step through the public API, with the step's inputs copied from pinned host memory and
    the outputs read back to the host inside the timed region."""
    import torch
    B, T = inp.B, inp.T
    k_np = inp.K[:, :, T - 1:T].copy().view(np.int16)
    v_np = inp.V[:, :, T - 1:T].copy().view(np.int16)
    q_np = inp.q.astype(np.float32)
    # the step's inputs sit in one pinned buffer (new K, new V, q) and go over in one copy; each
    # scheme's output comes back in its own copy, overlapping the next scheme's decode
    nk, nv, nq = k_np.nbytes, v_np.nbytes, q_np.nbytes
    in_host = torch.empty(nk + nv + nq, dtype=torch.uint8).pin_memory()
    in_host[:nk].copy_(torch.from_numpy(k_np.reshape(-1).view(np.uint8)))
    in_host[nk:nk + nv].copy_(torch.from_numpy(v_np.reshape(-1).view(np.uint8)))
    in_host[nk + nv:].copy_(torch.from_numpy(q_np.reshape(-1).view(np.uint8)))
    in_dev = torch.empty_like(in_host, device=device)
    k_dev = in_dev[:nk].view(torch.bfloat16).view(k_np.shape)
    v_dev = in_dev[nk:nk + nv].view(torch.bfloat16).view(v_np.shape)
    q_dev = in_dev[nk + nv:].view(torch.float32).view(q_np.shape)
    out_host = torch.empty((len(caches),) + q_np.shape, dtype=torch.float32).pin_memory()
    outs = torch.empty(out_host.shape, dtype=torch.float32, device=device)

    stream = torch.cuda.current_stream(device)
    # each scheme's output goes back on a second stream while the next scheme decodes
    copy_stream = torch.cuda.Stream(device)
    done = [torch.cuda.Event() for _ in caches]

    def work():  # copy in, append + decode per scheme, copy out
        in_dev.copy_(in_host, non_blocking=True)
        for i, kv in enumerate(caches):
            if args.split_step:
                kv.append(k_dev, v_dev, start)
                kv.decode(q_dev, seq, out=outs[i])
            else:
                kv.append_decode(k_dev, v_dev, q_dev, seq, out=outs[i])
            done[i].record(stream)
            copy_stream.wait_event(done[i])
            with torch.cuda.stream(copy_stream):
                out_host[i].copy_(outs[i], non_blocking=True)
        stream.wait_stream(copy_stream)

    for _ in range(max(1, args.warmup)):
        work()
        stream.synchronize()
    # the same calls and copies captured once as a CUDA graph (the copies use the pinned host
    # buffers, so a caller refills them between replays); every timed step replays it and waits
    # for the outputs to reach the host
    run = work
    if not args.eager:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                work()
            stream.synchronize()
            run = g.replay
        except Exception as exc:
            print(f"e2e graph capture failed, timing eager steps: {exc}", file=sys.stderr)
    for _ in range(max(1, args.warmup)):
        run()
        stream.synchronize()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
        stream.synchronize()
    el = time.perf_counter() - t
    h2d = in_host.numel()
    d2h = out_host.numel() * 4
    value = len(caches) * B * inp.Hkv * T * args.steps / el
    return {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "step_launch": "CUDA graph replay, host waits every step" if run is not work else "eager, host waits every step"}


def run_multi_query(kv, scheme, inp, device, T):
    """Decode of nq = 8 / G queries per sequence in one pass (the chunk's last positions)."""
    import torch
    G = inp.Hq // inp.Hkv
    nq = max(1, 8 // G)
    rng = np.random.default_rng(7)
    q = torch.from_numpy(rng.standard_normal((inp.B, nq, inp.Hq, inp.d)).astype(np.float32)).to(device)
    out = torch.empty_like(q)
    seq = [T] * inp.B
    for _ in range(3):
        kv.decode_multi(q, seq, out=out)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record()
    for _ in range(reps):
        kv.decode_multi(q, seq, out=out)
    e1.record()
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) / reps * 1e3
    return {"scheme": f"{scheme[0]}{scheme[1]}", "nq": nq, "decode_us": round(us, 2),
            "query_cache_tokens_per_s": round(nq * inp.B * inp.Hkv * T / (us * 1e-6), 1)}


def run_prefill_append(args, device):
    """Quantize-append of a 4096-token prefill chunk (long-context configuration, KQV n=4)."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    B, Hkv, d, T, n_new = 1, 8, 128, 131072, 4096
    rng = np.random.default_rng(3)
    std = np.exp(rng.uniform(np.log(0.1), np.log(10.0), size=(2, Hkv, 1, d))).astype(np.float32)
    k = torch.from_numpy((std[0] * rng.standard_normal((B, Hkv, n_new, d))).astype(np.float32)).to(device).bfloat16()
    v = torch.from_numpy((std[1] * rng.standard_normal((B, Hkv, n_new, d))).astype(np.float32)).to(device).bfloat16()
    kv = QuantizedKVCache(d, 64, Hkv, B, T, scheme="kqv", n=4, seed=3, device=device)
    start = [T - n_new] * B
    for _ in range(3):
        kv.append(k, v, start)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        kv.append(k, v, start)
    e1.record()
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / reps
    vec = 2 * B * Hkv * n_new
    moved = vec * d * 2 + B * Hkv * n_new * record_bytes("kqv", 4)
    peak, peak_kind = measured_peak()
    gbs = moved / (ms * 1e-3) / 1e9
    return {"workload": "B=1 Hkv=8 d=128, 4096-token prefill chunk into a 131072-token KQV n=4 cache",
            "tok_per_s": round(B * n_new / (ms * 1e-3), 1), "vectors_per_s": round(vec / (ms * 1e-3), 1),
            "us": round(ms * 1e3, 2), "GB_per_s": round(gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None,
                         "algorithmic_bytes": int(moved),
                         "bytes": "bf16 K and V read (2 x 256 B per token and KV head) + the packed "
                                  "KQV n=4 record written (138 B)",
                         "kernel": "append (encode + QJL residual sketch), CUDA events over 10 calls",
                         "peak_kind": peak_kind}}


def measured_tensor_peak():
    """Dense bf16 tensor-core TFLOP/s of this machine's GPUs (burst: the prefill is timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def prefill_flops(scheme, n, B, Hq, nq, L, d=128, m=128):
    """Algorithmic FLOPs of a chunked prefill: per (query head, visible token) the score (d MACs,
    plus m for a QJL key sketch) and the readout (d MACs, plus m for a QJL value sketch)."""
    from turboquant_quantized_kv_tq_gb300.binding import SCHEMES as S, tq_config, tq_config_from_scheme
    c = tq_config()
    tq_config_from_scheme(S[scheme], n, c)
    macs = 2 * d + (m if c.k.qjl else 0) + (m if c.v.qjl else 0)
    visible = sum(max(0, L - nq + 1 + i) for i in range(nq))
    return 2.0 * macs * B * Hq * visible


def run_prefill(args, caches, inp, device, T, nq=512):
    """Chunked prefill over the headline caches: the last nq = 512 positions of each sequence as
    queries (G = 4 query heads per KV head: 2048 rows per KV head), each attending causally to its
    prefix of the T = 32768 stored tokens.  CUDA events over 5 calls per scheme."""
    import torch
    rng = np.random.default_rng(9)
    q = torch.from_numpy(rng.standard_normal((inp.B, nq, inp.Hq, inp.d)).astype(np.float32)).to(device)
    out = torch.empty_like(q)
    peak, peak_kind = measured_tensor_peak()
    res, tot_flops, tot_s = {}, 0.0, 0.0
    for (scheme, n), kv in zip(SCHEMES, caches):
        ws = torch.empty(kv.prefill_workspace_bytes(nq), dtype=torch.uint8, device=device)
        for _ in range(2):
            kv.prefill(q, [T] * inp.B, out=out, ws=ws)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record()
        for _ in range(reps):
            kv.prefill(q, [T] * inp.B, out=out, ws=ws)
        e1.record()
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / reps
        fl = prefill_flops(scheme, n, inp.B, inp.Hq, nq, T)
        tot_flops += fl
        tot_s += ms * 1e-3
        res[f"{scheme}{n}"] = {"ms": round(ms, 3), "query_tokens_per_s": round(inp.B * nq / (ms * 1e-3), 1),
                               "TFLOP_per_s": round(fl / (ms * 1e-3) / 1e12, 1),
                               "frac": round(fl / (ms * 1e-3) / 1e12 / peak, 4)}
        del ws
    achieved = tot_flops / tot_s / 1e12
    return {"workload": f"chunked prefill: B={inp.B} Hq={inp.Hq} Hkv={inp.Hkv} d={inp.d}, the last {nq} of "
                        f"{T} positions as queries (causal within the chunk), the headline caches",
            "timing": "CUDA events, 5 calls per scheme (query prep + prefill kernel)",
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "flops": "per (query head, visible token): 2 x (2 d + m per QJL side) -- the "
                                  "method's score and readout contractions, the fp16 lo terms not counted",
                         "kernel": "prefill (query prep + fused prefill kernel), all four schemes",
                         "peak_kind": peak_kind + " (bf16 dense, burst; fp16 MMAs run at the bf16 rate)"},
            "schemes": res}


def run_long_context(args, device):
    """The 128k-context configuration (B=1, Hq=64, Hkv=8, d=128, T=131072; KQV n=2/3/4): each
    scheme's cache filled by the library's append, then steps of three decode calls (one per
    scheme, so each decode's cache was last touched two caches -- 189-256 MB -- earlier, more
    than L2 holds), each call bracketed by CUDA events on the launching stream."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from workloads import CONFIGS, make_inputs
    c = CONFIGS["cfg4"]
    inp = make_inputs("cfg4")
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    to_t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    q = torch.from_numpy(inp.q).to(device)
    seq = [T] * B
    caches = []
    for scheme, n in c["schemes"]:
        kv = QuantizedKVCache(d, Hq, Hkv, B, T, scheme=scheme, n=n, seed=inp.seed, device=device)
        for s0 in range(0, T, 4096):
            e = min(T, s0 + 4096)
            kv.append(to_t(inp.K[:, :, s0:e]).to(device), to_t(inp.V[:, :, s0:e]).to(device), [s0] * B)
        kv.workspace(T)
        caches.append(kv)
    outs = [torch.empty_like(q) for _ in caches]
    stream = torch.cuda.current_stream(device)
    for _ in range(max(3, args.warmup)):
        for kv, o in zip(caches, outs):
            kv.decode(q, seq, out=o)
    torch.cuda.synchronize(device)
    reps = 50
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in caches]
           for _ in range(reps)]
    for r in range(reps):
        for i, (kv, o) in enumerate(zip(caches, outs)):
            evs[r][i][0].record(stream)
            kv.decode(q, seq, out=o)
            evs[r][i][1].record(stream)
    torch.cuda.synchronize(device)
    peak, peak_kind = measured_peak()
    res, tot_bytes, tot_s = {}, 0.0, 0.0
    for i, ((scheme, n), kv) in enumerate(zip(c["schemes"], caches)):
        us = sum(evs[r][i][0].elapsed_time(evs[r][i][1]) for r in range(reps)) / reps * 1e3
        rec = record_bytes(scheme, n)
        nbytes = B * Hkv * T * rec
        tot_bytes += nbytes
        tot_s += us * 1e-6
        res[f"{scheme}{n}"] = {"decode_us": round(us, 2), "record_bytes": rec,
                               "GB_per_s": round(nbytes / (us * 1e-6) / 1e9, 1),
                               "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
                               "cache_tokens_per_s": round(B * Hkv * T / (us * 1e-6), 1)}
    del caches
    torch.cuda.empty_cache()
    achieved = tot_bytes / tot_s / 1e9
    return {"workload": f"cfg4 long context: B={B} Hq={Hq} Hkv={Hkv} d={d} T={T}, KQV n=2/3/4, "
                        "Gaussian K/V with log-uniform per-channel std in [0.1, 10]",
            "timing": f"CUDA events per decode call (query prep + decode), {reps} steps of the three",
            "cache_tokens_per_s": round(len(res) * B * Hkv * T / tot_s, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": "decode (query prep + fused split-K decode), KQV n=2/3/4",
                         "peak_kind": peak_kind},
            "schemes": res}


def oracle_step(inp, bufs, ctxs, slabs, T):
    """The oracle decodes the given slabs of every scheme over T tokens."""
    done = 0
    for orc, buf in zip(ctxs, bufs):
        for (b, h) in slabs:
            orc.decode(buf, inp.q, [T] * inp.B, slabs=[(b, h)])
            done += T
    return done


def cpu_baseline(inp, caches, budget_s=20.0):
    """The float64 oracle on the host cores: decode of whole slabs of each scheme's cache (the
    cache bytes the GPU wrote), as many slabs as fit in about ``budget_s`` seconds."""
    from oracle.pipeline import OracleContext
    from oracle import codec as ocodec
    T = inp.T
    ctxs, bufs = [], []
    for (scheme, n), kv in zip(SCHEMES, caches):
        kc, vc = ocodec.scheme_codecs(scheme, n)
        ctxs.append(OracleContext(inp.d, inp.Hq, inp.Hkv, inp.B, T, kc, vc, inp.seed))
        bufs.append(kv.cache.cpu().numpy())
    slabs = [(b, h) for b in range(inp.B) for h in range(inp.Hkv)]
    done, t = 0, time.perf_counter()
    used = 0
    for s in slabs:
        done += oracle_step(inp, bufs, ctxs, [s], T)
        used += 1
        if time.perf_counter() - t > budget_s:
            break
    el = time.perf_counter() - t
    return {"value": round(done / el, 1), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{used} of {len(slabs)} (batch, KV head) slabs x 4 schemes, each decoded over "
                      f"{T} tokens for its {inp.Hq // inp.Hkv} query heads ({el:.1f} s)"}


def run_reference(args):
    """The oracle alone, on the host cores, timed per step on a bounded sample of the workload."""
    from oracle import codec as ocodec
    from oracle.pipeline import OracleContext
    from workloads import make_inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # one slab per scheme per step: inputs for batch 1, one KV head, full context
    inp = make_inputs("cfg2", B=1, Hkv=1, Hq=4)
    T = inp.T
    ctxs, bufs = [], []
    for scheme, n in SCHEMES:
        kc, vc = ocodec.scheme_codecs(scheme, n)
        orc = OracleContext(inp.d, inp.Hq, inp.Hkv, 1, T, kc, vc, inp.seed)
        buf = orc.new_cache()
        orc.append(buf, inp.k_f32()[:, :, :T].astype(np.float64), inp.v_f32()[:, :, :T].astype(np.float64), [0])
        ctxs.append(orc)
        bufs.append(buf)
    # each step decodes the first L tokens of the slab, L sized from the warm-up so that the K
    # timed steps take about args.ref_seconds in all (the oracle's cost is linear in L)
    t = time.perf_counter()
    for _ in range(args.warmup):
        oracle_step(inp, bufs, ctxs, [(0, 0)], T)
    per_full = (time.perf_counter() - t) / max(1, args.warmup)
    L = int(T * args.ref_seconds / (args.steps * per_full)) // 16 * 16
    L = max(16, min(T, L))
    t = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += oracle_step(inp, bufs, ctxs, [(0, 0)], L)
    el = time.perf_counter() - t
    value = done / el
    sample = (f"per step: one (batch, KV head) slab of each of the 4 schemes decoded over its first {L} "
              f"of {T} tokens (sized so {args.steps} steps take about {args.ref_seconds:.0f} s), 4 query heads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64; no public dataset)",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_workload(args):
    """Decode throughput of one of the other configurations at its full shape, per scheme: the
    cache filled by the library's append (4096-token chunks), then `reps` decode calls timed
    with CUDA events (query prep + decode).  One JSON line; not the headline contract line."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from workloads import CONFIGS, make_inputs
    name = args.workload
    device = torch.device("cuda", 0)
    inp = make_inputs(name)
    c = CONFIGS[name]
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    to_t = (lambda a: torch.from_numpy(a)) if inp.dtype == "f32" else \
        (lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16))
    q = torch.from_numpy(inp.q).to(device)
    out = torch.empty_like(q)
    seq = [T] * B
    peak, peak_kind = measured_peak()
    res = {}
    for scheme, n in c["schemes"]:
        if scheme == "headq":
            kv = QuantizedKVCache(d, Hq, Hkv, B, T, scheme=None, seed=inp.seed, k_codec=(n, 1, 0),
                                  v_codec=(4, 1, 0), headq_rank=c["headq_rank"], device=device)
            U = []
            for h in range(Hkv):  # calibration basis: top eigenvectors of the centred query covariance
                x = inp.extra["calib"][h].astype(np.float64)
                x = x - x.mean(axis=0, keepdims=True)
                w, vecs = np.linalg.eigh(x.T @ x)
                U.append(vecs[:, np.argsort(-w)[:c["headq_rank"]]])
            kv.set_headq_basis(torch.from_numpy(np.stack(U).astype(np.float32)).to(device))
        else:
            kv = QuantizedKVCache(d, Hq, Hkv, B, T, scheme=scheme, n=n, seed=inp.seed, device=device)
            if scheme == "squ":  # the regime's separate calibration sets for K and V
                from turboquant_quantized_kv_tq_gb300.calibration import spectral_tables
                for side, key in enumerate(("calib_k", "calib_v")):
                    E, sc, _ = spectral_tables(inp.extra[key])
                    kv.set_spectral_basis(side, torch.from_numpy(E).to(device), torch.from_numpy(sc).to(device))
        for s0 in range(0, T, 4096):
            e = min(T, s0 + 4096)
            kv.append(to_t(inp.K[:, :, s0:e]).to(device), to_t(inp.V[:, :, s0:e]).to(device), [s0] * B)
        kv.workspace(T)
        for _ in range(args.warmup):
            kv.decode(q, seq, out=out)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 50
        e0.record()
        for _ in range(reps):
            kv.decode(q, seq, out=out)
        e1.record()
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) / reps * 1e3
        rec = (kv.layout.k_block_bytes + kv.layout.v_block_bytes) / 16.0
        nbytes = B * Hkv * T * rec
        res[f"{scheme}{n}"] = {"decode_us": round(us, 2), "record_bytes": rec,
                               "GB_per_s": round(nbytes / (us * 1e-6) / 1e9, 1),
                               "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
                               "cache_tokens_per_s": round(B * Hkv * T / (us * 1e-6), 1)}
        del kv
        torch.cuda.empty_cache()
    print(json.dumps({"workload": f"{name}: B={B} Hq={Hq} Hkv={Hkv} d={d} T={T}", "unit": UNIT,
                      "peak_GBps": peak, "peak_kind": peak_kind, "timing": "CUDA events, 50 decode calls",
                      "schemes": res}), flush=True)


def run_paged(args):
    """The paged pool at the headline shape (B=8 Hq=32 Hkv=8 d=128 T=32768), per scheme: each
    sequence's 2048 blocks on shuffled pages, filled by the paged append (4096-token chunks, start
    positions on the device), then `reps` paged decode calls with device lengths, timed with CUDA
    events (query prep with the device work split + decode).  The same decode of a contiguous
    cache is timed beside it.  One JSON line; not the headline contract line."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import PagedKVCache, QuantizedKVCache
    from workloads import make_inputs
    device = torch.device("cuda", 0)
    inp = make_inputs("cfg2")
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    to_t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    mb = T // 16
    num_pages = B * mb + 64
    table = np.random.default_rng(11).permutation(num_pages)[:B * mb].reshape(B, mb).astype(np.int32)
    tdev = torch.from_numpy(table).to(device)
    q = torch.from_numpy(inp.q).to(device)
    out = torch.empty_like(q)
    seq_dev = torch.full((B,), T, dtype=torch.int32, device=device)
    peak, peak_kind = measured_peak()
    reps = 50

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps * 1e3

    res = {}
    for scheme, n in SCHEMES:
        pool = PagedKVCache(d, Hq, Hkv, B, num_pages, mb, scheme=scheme, n=n, seed=inp.seed, device=device)
        for s0 in range(0, T, 4096):
            start = torch.full((B,), s0, dtype=torch.int32, device=device)
            pool.append(to_t(inp.K[:, :, s0:s0 + 4096]).to(device), to_t(inp.V[:, :, s0:s0 + 4096]).to(device),
                        start, tdev)
        us_paged = timed(lambda: pool.decode(q, seq_dev, tdev, out=out))
        rec = (pool.layout.k_block_bytes + pool.layout.v_block_bytes) / 16.0
        del pool
        torch.cuda.empty_cache()
        kv = QuantizedKVCache(d, Hq, Hkv, B, T, scheme=scheme, n=n, seed=inp.seed, device=device)
        for s0 in range(0, T, 4096):
            kv.append(to_t(inp.K[:, :, s0:s0 + 4096]).to(device), to_t(inp.V[:, :, s0:s0 + 4096]).to(device),
                      [s0] * B)
        kv.workspace(T)
        us_contig = timed(lambda: kv.decode(q, [T] * B, out=out))
        del kv
        torch.cuda.empty_cache()
        nbytes = B * Hkv * T * rec
        res[f"{scheme}{n}"] = {"paged_decode_us": round(us_paged, 2), "contiguous_decode_us": round(us_contig, 2),
                               "record_bytes": rec, "GB_per_s": round(nbytes / (us_paged * 1e-6) / 1e9, 1),
                               "frac": round(nbytes / (us_paged * 1e-6) / 1e9 / peak, 4),
                               "cache_tokens_per_s": round(B * Hkv * T / (us_paged * 1e-6), 1)}
    print(json.dumps({"workload": f"paged: B={B} Hq={Hq} Hkv={Hkv} d={d} T={T}, {num_pages} pages of 16 "
                                  f"tokens x {Hkv} KV heads, block tables a random permutation",
                      "unit": UNIT, "peak_GBps": peak, "peak_kind": peak_kind,
                      "timing": f"CUDA events, {reps} decode calls", "schemes": res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: approximate time of the timed steps")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-append", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true", help="leave out the chunked-prefill leg")
    ap.add_argument("--skip-long-context", action="store_true",
                    help="leave out the 128k-context (cfg4) decode leg")
    ap.add_argument("--eager", action="store_true", help="time eager steps instead of a captured graph")
    ap.add_argument("--split-step", action="store_true",
                    help="append and decode as two library calls (no overlap of the query preparation "
                         "with the append)")
    ap.add_argument("--schemes", default=None,
                    help="comma-separated subset of plain4,tq4,kqv4,qkqv4 (default: all four)")
    ap.add_argument("--workload", default=None, choices=["cfg1", "cfg3", "cfg4", "cfg5", "sq", "paged", "append"],
                    help="decode throughput of another configuration at full size, of the paged pool "
                         "at the headline shape, or the prefill-chunk append alone (one JSON line)")
    args = ap.parse_args()
    if args.schemes:
        global SCHEMES
        known = {f"{s}{n}": (s, n) for s, n in SCHEMES}
        SCHEMES = [known[x.strip()] for x in args.schemes.split(",")]
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "paged":
        run_paged(args)
        return
    if args.workload == "append":
        import torch
        torch.cuda.set_device(0)
        print(json.dumps(run_prefill_append(args, torch.device("cuda", 0))), flush=True)
        return
    if args.workload:
        run_workload(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
