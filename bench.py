"""Batch-1 decode throughput of the 2.3B-class fp16 decoder on one GB300.

Workload: 25 layers, d_model 2560, 20 query heads x 128, 4 KV heads, SwiGLU 9728, tied
vocabulary 32000, fp16 weights ~N(0, 0.02) from a seed; a 512-token uniform-random prompt is
prefilled, then greedy decode steps run at contexts 513..1024 (a run longer than 512 steps
rewinds the cache to 512 and decodes the window again). One step = one decode step of the
whole model; the steps of a window run inside one persistent kernel launch.
--workload names another run: dense-2.3b-fp16-long-t0.7 (the same model after a 3,584-token
prompt, contexts 3585..4096, temperature 0.7 sampling with the seeded uniform stream),
dense-8b-bf16 (the 8B model, prompt 1024, contexts 1025..1280), moe-32x1408-top4-e4m3 (the MoE
model, prompt 256, contexts 257..768), dense-2.3b-e4m3 / dense-2.3b-nvfp4 (the 2.3B shape with e4m3
or NVFP4 layer matrices).
--batch N (N >= 2) measures N independent requests decoded together by the batched kernel
(value = tokens/s of all requests; the default, batch 1, is the benchmark's headline).
--prefill measures time to first token of the 3,584-token prompt through the tensor-core
prefill (adp_prefill_tc), beside the decode-kernel prefill.

Printed (one JSON line, rank 0):
  value      tokens/s, device-timed: the steps chained on the GPU (adp_generate_async), weights
             and KV resident in HBM, CUDA events around the timed region on the model's stream;
             three timed regions of exactly --steps steps, the median one reported;
  e2e        tokens/s through adp_decode_step with the token in and out of host memory every
             step (a 32-byte step state host->device, 8 bytes device->host, one sync per step);
  roofline   algorithmic bytes per launch (per step: every weight once + KV of the context + the
             new KV row; up to one window of steps per launch) / average launch duration, against
             the measured HBM copy bandwidth, the nominal 8 TB/s and a read-bandwidth probe run in
             the same process;
  cpu_baseline  the CPU oracle (plain fp32, all host cores) timed on a bounded sample.

--impl reference times the CPU oracle as the reference arm on the same workload.
Several GPUs (torchrun): independent replicas, one per GPU, no collective; value = all
tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tokens/s/request (2.3B fp16); achieved HBM GB/s vs GB300 peak"
WORKLOAD = "dense-2.3b-fp16"
# --workload: the benchmarked model and run.  The default is the 2.3B fp16 model at contexts
# 513..1024; the others are the long-context 2.3B run with temperature sampling, the 8B bf16 model,
# the top-4-of-32 MoE model with e4m3 experts, and the 2.3B shape with e4m3 or NVFP4 layer matrices
# (per-row fp32 scales; NVFP4 also an e4m3 scale per 16 elements; fp16 embedding and tied LM head).
# window: decode steps of one pass (contexts prompt + 1 .. prompt + window); temperature: 0 greedy,
# else sampling with the seeded uniform stream; cpu_steps: cap on the CPU oracle's timed steps.
WORKLOADS = {
    "dense-2.3b-fp16": {"metric": METRIC, "weights": "f16", "window": 512, "temperature": 0.0,
                        "data": "synthetic: seeded N(0,0.02) fp16 weights, 512 uniform-random prompt ids"},
    "dense-2.3b-e4m3": {"metric": "batch-1 decode tokens/s/request (2.3B, e4m3 layer weights); achieved HBM GB/s "
                                  "vs GB300 peak",
                        "weights": "e4m3 layer matrices with per-row f32 scales; f16 embedding, LM head, norms",
                        "window": 512, "temperature": 0.0,
                        "data": "synthetic: seeded N(0,0.02) weights quantised to e4m3 per row, 512 uniform-random "
                                "prompt ids"},
    "dense-2.3b-nvfp4": {"metric": "batch-1 decode tokens/s/request (2.3B, NVFP4 layer weights); achieved HBM GB/s "
                                   "vs GB300 peak",
                         "weights": "nvfp4 layer matrices (e2m1, e4m3 scale per 16 elements, f32 row scales); f16 "
                                    "embedding, LM head, norms",
                         "window": 512, "temperature": 0.0,
                         "data": "synthetic: seeded N(0,0.02) weights quantised to NVFP4 per row and 16-element "
                                 "block, 512 uniform-random prompt ids"},
    "dense-2.3b-fp16-long-t0.7": {
        "metric": "batch-1 decode tokens/s/request (2.3B fp16, contexts 3585..4096, T=0.7 sampling); achieved HBM "
                  "GB/s vs GB300 peak",
        "weights": "f16", "window": 512, "temperature": 0.7,
        "data": "synthetic: seeded N(0,0.02) fp16 weights, 3584 uniform-random prompt ids, seeded sampling uniforms"},
    "dense-8b-bf16": {"metric": "batch-1 decode tokens/s/request (8B bf16); achieved HBM GB/s vs GB300 peak",
                      "weights": "bf16 (untied LM head)", "window": 256, "temperature": 0.0, "cpu_steps": 16,
                      "data": "synthetic: seeded N(0,0.02) bf16 weights, 1024 uniform-random prompt ids"},
    "dense-8b-e4m3": {"metric": "batch-1 decode tokens/s/request (8B, e4m3 layer weights); achieved HBM GB/s vs "
                                "GB300 peak",
                      "weights": "e4m3 layer matrices with per-row f32 scales; bf16 embedding, untied LM head, norms",
                      "window": 256, "temperature": 0.0, "cpu_steps": 16,
                      "data": "synthetic: seeded N(0,0.02) weights quantised to e4m3 per row, 1024 uniform-random "
                              "prompt ids"},
    "dense-8b-nvfp4": {"metric": "batch-1 decode tokens/s/request (8B, NVFP4 layer weights); achieved HBM GB/s vs "
                                 "GB300 peak",
                       "weights": "nvfp4 layer matrices (e2m1, e4m3 scale per 16 elements, f32 row scales); bf16 "
                                  "embedding, untied LM head, norms",
                       "window": 256, "temperature": 0.0, "cpu_steps": 16,
                       "data": "synthetic: seeded N(0,0.02) weights quantised to NVFP4 per row and 16-element block, "
                               "1024 uniform-random prompt ids"},
    "moe-32x1408-top4-e4m3": {
        "metric": "batch-1 decode tokens/s/request (MoE, top-4 of 32 e4m3 experts); achieved HBM GB/s vs GB300 peak",
        "weights": "bf16 attention, embedding and tied LM head; f16 router; e4m3 experts with per-row f32 scales",
        "window": 512, "temperature": 0.0,
        "data": "synthetic: seeded N(0,0.02) weights (experts quantised to e4m3 per row), 256 uniform-random prompt "
                "ids"},
}
WINDOW = 512  # decode steps per pass (set from the workload in main)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = ("decode.cu", "decode_core.cuh", "device.cuh", "plan.h")  # the decode kernel's device code
BATCH_KERNEL_SOURCES = ("decode_batch.cu", "decode_core.cuh", "device.cuh", "plan.h")  # the batched kernel's


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    """sha256[:16] over a kernel's sources (host-only files do not change its traffic)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "autoregressive_decode_persistent_gb300", "csrc")
    for f in sources:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(src_hash: str, name: str | None = None):
    """DRAM bytes per decode step from the committed ncu summary, if it was taken on this kernel
    source (a launch of n chained steps moves n times as much)."""
    path = os.path.join(ROOT, "profiles", name or f"decode_kernel_{WORKLOAD}.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    m_hash = re.search(r"kernel source sha256\[:16\]:\s*`?([0-9a-f]{16})", text)
    m_tr = re.search(r"traffic bytes per step:\s*`?([0-9.e+]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != src_hash:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(cfg, W, seconds: float = 15.0, max_steps: int | None = None, warmup: int = 1):
    """The CPU oracle as it stands (plain mode) on a bounded sample of the workload: `warmup`
    untimed steps, then steps until `seconds` have passed or `max_steps` were taken."""
    import synth
    from oracle import PLAIN, OracleModel
    om = OracleModel(cfg, W)
    om.load_kv_prefix(*synth.kv_prefix(cfg, cfg["prompt_len"]))
    toks = synth.prompt(cfg, 64, seed=99)
    for i in range(max(1, warmup)):  # first calls: tables, page-in
        om.step(int(toks[i % len(toks)]), PLAIN)
    n, t0 = 0, time.perf_counter()
    while True:
        om.step(int(toks[(n + 1) % len(toks)]), PLAIN)
        n += 1
        el = time.perf_counter() - t0
        if (el >= seconds and n >= 2) or (max_steps and n >= max_steps):
            break
    cores = len(os.sched_getaffinity(0))
    return {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} plain-fp32 decode steps of the full {cfg['name']} model at contexts "
                      f"{cfg['prompt_len'] + max(1, warmup) + 1}..{cfg['prompt_len'] + max(1, warmup) + n} "
                      f"(synthetic {cfg['prompt_len']}-position KV prefix, {max(1, warmup)} untimed steps first), "
                      f"OpenMP over {cores} host threads, {el:.1f} s"}, n, el


def max_over_ranks(values, world: int) -> list[float]:
    """Element-wise maximum of per-rank timings over all ranks (every rank gets the result)."""
    vals = [float(v) for v in values]
    if world <= 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank: int, seconds_max: float, world: int) -> float:
    """Units all ranks processed (each the same number) per second of the slowest rank."""
    return world * units_per_rank / seconds_max


def launch_ablation(model, kv, tok0, P, dev, n):
    """The same device code as one launch per phase (plain stream, then a CUDA graph of those
    launches) against the persistent launch, each through adp_decode_step for n steps (host
    token in and out every step, as in e2e).  Gap per launch = extra time per step / extra launches."""
    import torch
    res = {}
    for mode, name in ((0, "persistent"), (1, "multikernel"), (2, "graph")):
        model.set_kernel_mode(mode)
        kv.truncate(P)
        t = tok0
        for _ in range(3):  # warm-up (and, in mode 2, the graph capture)
            t = kv.step(t)
        kv.truncate(P)
        t = tok0
        torch.cuda.synchronize(dev)
        h0 = time.perf_counter()
        for _ in range(n):
            t = kv.step(t)
        el = time.perf_counter() - h0
        res[name] = {"tokens_per_s": round(n / el, 2), "us_per_step": round(el / n * 1e6, 1),
                     "launches_per_step": model.launches_per_step}
    model.set_kernel_mode(0)
    extra = res["multikernel"]["launches_per_step"] - 1
    for name in ("multikernel", "graph"):
        gap = (res[name]["us_per_step"] - res["persistent"]["us_per_step"]) / max(extra, 1)
        res[name]["gap_us_per_extra_launch"] = round(gap, 3)
    res["steps"] = n
    return res


def workload_text(cfg) -> str:
    """The workload named by what it is: the model's shape, the prompt and the decode run."""
    c = cfg
    w = WORKLOADS[WORKLOAD]
    ffn = (f"{c['n_experts']} experts x ffn {c['d_expert']} top-{c['top_k']}" if c["n_experts"]
           else f"ffn {c['d_ff']}")
    P = c["prompt_len"]
    how = "greedy" if w["temperature"] <= 0 else f"T = {w['temperature']} sampling"
    return (f"{WORKLOAD}: {c['n_layers']} layers, d {c['d_model']}, {c['n_heads']}x{c['head_dim']} q heads, "
            f"{c['n_kv_heads']} kv heads, {ffn}, {'tied' if c['tied_embeddings'] else 'untied'} vocab {c['vocab']}; "
            f"batch 1, prompt {P}, {how} decode at contexts {P + 1}..{P + w['window']}")


def dtype_text(cfg) -> str:
    """The arithmetic of the path: stored weight and KV types, fp32 accumulation and activations."""
    c = cfg
    wt = {"f16": "f16", "bf16": "bf16", "e4m3": "e4m3 (per-row f32 scales)",
          "nvfp4": "nvfp4 (e4m3 block and f32 row scales)"}[c["weight_dtype"]]
    if c["n_experts"]:
        wt += f" attention, {c['expert_dtype']} experts"
    return f"{wt} weights, {c['kv_dtype']} KV cache, f32 accumulation and activations"


def read_probe(dev, nbytes=4 << 30, reps=5):
    """GB/s of the library's 16-byte read probe over a buffer larger than L2, in this process."""
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    stream = torch.cuda.current_stream(dev).cuda_stream
    gbs = adp.adp_measure_read_bandwidth(buf, nbytes, reps, stream)
    del buf
    torch.cuda.empty_cache()
    return gbs


def run_engine(args, rank: int, world: int):
    import torch

    import synth
    from autoregressive_decode_persistent_gb300 import bound, build
    from autoregressive_decode_persistent_gb300.model import DecodeModel

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    build.build()
    cfg = synth.get_config(WORKLOAD)
    if args.layers:
        cfg["n_layers"] = args.layers  # profiling only: a shorter model with the same layer shapes
    T = WORKLOADS[WORKLOAD]["temperature"]
    read_gbs = read_probe(dev)  # before the model: the probe's 4 GB buffer and the weights never coexist
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg)
    model = DecodeModel(cfg, W, device=dev)
    stream = torch.cuda.current_stream(dev)
    kv = model.new_kv()
    P = cfg["prompt_len"]
    tok0 = kv.prefill(prompt)
    out = torch.empty(WINDOW, dtype=torch.int32, device=dev)
    # sampling: the seeded uniform of each position of the window, resident on the device
    us = synth.sampling_uniforms(WINDOW, first=P) if T > 0 else None
    dev_u = torch.tensor(us, dtype=torch.float32, device=dev) if T > 0 else None

    def passes(n_steps):
        """Decode n_steps chained steps in windows of contexts P+1..P+WINDOW."""
        t = tok0
        left = n_steps
        while left > 0:
            k = min(left, WINDOW)
            kv.truncate(P)
            kv.generate_async(t, k, out, T, dev_u)
            left -= k

    # warm-up (untimed)
    passes(args.warmup)
    from autoregressive_decode_persistent_gb300 import adp
    adp.adp_sync(model.handle)
    torch.cuda.synchronize(dev)

    # three timed regions of exactly args.steps steps each (device events on the model's stream);
    # the reported one is the median
    runs = []
    with ClockSampler(local) as clocks:
        for _ in range(3):
            if world > 1:
                import torch.distributed as dist
                dist.barrier()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            passes(args.steps)
            e1.record(stream)
            e1.synchronize()
            adp.adp_sync(model.handle)
            runs.append(e0.elapsed_time(e1))
    ms = statistics.median(runs)

    # algorithmic bytes: contexts P+1 .. P+k in each window
    total_bytes = 0
    left = args.steps
    while left > 0:
        k = min(left, WINDOW)
        total_bytes += bound.mean_bytes_per_token(cfg, P + 1, k) * k
        left -= k
    n_launch = -(-args.steps // WINDOW)  # one launch per window of chained steps
    per_launch = total_bytes / n_launch
    launch_ms = ms / n_launch
    peak, peak_kind = _peaks()
    achieved = per_launch / (launch_ms * 1e-3) / 1e9

    # e2e through the public per-step call, host token in and out every step
    n_e2e = min(args.steps, 2 * WINDOW)
    kv.truncate(P)
    t = tok0
    torch.cuda.synchronize(dev)
    per_step = []
    h0 = time.perf_counter()
    for i in range(n_e2e):
        if i and i % WINDOW == 0:
            kv.truncate(P)
        s0 = time.perf_counter()
        t = kv.step(t, T, float(us[i % WINDOW]) if T > 0 else 0.0)
        per_step.append(time.perf_counter() - s0)
    h1 = time.perf_counter()
    per_step.sort()
    step_pct = {"p50_us": round(per_step[len(per_step) // 2] * 1e6, 1),
                "p99_us": round(per_step[min(len(per_step) - 1, int(len(per_step) * 0.99))] * 1e6, 1)}
    ms, e2e_s = max_over_ranks([ms, h1 - h0], world)
    e2e = whole_job_rate(n_e2e, e2e_s, world)

    ablation = launch_ablation(model, kv, tok0, P, dev, args.ablation_steps) if args.ablation_steps else None

    if args.timeline:
        write_timeline(args.timeline, model, kv, tok0, P, cfg)

    res = {
        "ms": ms, "runs_ms": runs, "steps": args.steps, "n_launch": n_launch, "step_pct": step_pct,
        "weight_bytes": bound.weight_bytes_per_token(cfg), "achieved_gbs": achieved, "per_launch_bytes": per_launch,
        "launch_ms": launch_ms, "peak": peak, "peak_kind": peak_kind, "read_gbs": read_gbs, "e2e": e2e,
        "n_e2e": n_e2e, "clocks": clocks.summary(), "ctas": model.num_ctas, "image_bytes": model.image_bytes,
        # one cooperative launch per window of chained steps (adp_generate_async)
        "launches": -(-args.steps // WINDOW) * model.launches_per_step, "ablation": ablation,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu"] = cpu_baseline(cfg, W, seconds=args.cpu_seconds,
                                  max_steps=WORKLOADS[WORKLOAD].get("cpu_steps"))[0]
    kv.close()
    model.close()
    return cfg, res


def run_engine_batch(args, rank: int, world: int):
    """The same workload as nb independent requests decoded together by the batched kernel: each
    request has its own 512-token prompt (prefilled alone) and cache; the timed region runs
    windows of chained batched steps (adp_generate_batch_async), every request at contexts
    513..1024."""
    import torch

    import synth
    from autoregressive_decode_persistent_gb300 import adp, bound, build
    from autoregressive_decode_persistent_gb300.model import DecodeModel

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    build.build()
    cfg = synth.get_config(WORKLOAD)
    if args.layers:
        cfg["n_layers"] = args.layers
    nb = args.batch
    W = synth.model_weights(cfg)
    model = DecodeModel(cfg, W, device=dev)
    if nb > model.max_batch:
        raise SystemExit(f"--batch {nb}: this model batches at most {model.max_batch} requests")
    stream = torch.cuda.current_stream(dev)
    P = cfg["prompt_len"]
    kvs = [model.new_kv() for _ in range(nb)]
    tok0 = [kvs[r].prefill(p) for r, p in enumerate(synth.batch_prompts(cfg, [P] * nb))]
    out = torch.empty((WINDOW, nb), dtype=torch.int32, device=dev)

    def passes(n_steps):
        left = n_steps
        while left > 0:
            k = min(left, WINDOW)
            for kv in kvs:
                kv.truncate(P)
            model.generate_batch_async(kvs, tok0, k, out)
            left -= k

    passes(args.warmup)
    adp.adp_sync(model.handle)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record(stream)
        passes(args.steps)
        e1.record(stream)
        e1.synchronize()
    adp.adp_sync(model.handle)
    ms = e0.elapsed_time(e1)
    total_bytes = 0
    left = args.steps
    while left > 0:
        k = min(left, WINDOW)
        total_bytes += bound.mean_batch_step_bytes(cfg, nb, P + 1, k) * k
        left -= k
    n_launch = -(-args.steps // WINDOW)
    per_launch = total_bytes / n_launch
    launch_ms = ms / n_launch
    peak, peak_kind = _peaks()
    achieved = per_launch / (launch_ms * 1e-3) / 1e9
    # e2e: adp_decode_batch per step, the nb tokens in and out of host memory every step
    n_e2e = min(args.steps, 2 * WINDOW)
    for kv in kvs:
        kv.truncate(P)
    t = list(tok0)
    torch.cuda.synchronize(dev)
    per_step = []
    h0 = time.perf_counter()
    for i in range(n_e2e):
        if i and i % WINDOW == 0:
            for kv in kvs:
                kv.truncate(P)
        s0 = time.perf_counter()
        t = model.step_batch(kvs, t)
        per_step.append(time.perf_counter() - s0)
    h1 = time.perf_counter()
    per_step.sort()
    step_pct = {"p50_us": round(per_step[len(per_step) // 2] * 1e6, 1),
                "p99_us": round(per_step[min(len(per_step) - 1, int(len(per_step) * 0.99))] * 1e6, 1)}
    ms, e2e_s = max_over_ranks([ms, h1 - h0], world)
    res = {
        "ms": ms, "steps": args.steps, "nb": nb, "n_launch": n_launch, "step_pct": step_pct,
        "weight_bytes": bound.weight_bytes_per_token(cfg), "achieved_gbs": achieved, "per_launch_bytes": per_launch,
        "launch_ms": launch_ms, "peak": peak, "peak_kind": peak_kind,
        "e2e": whole_job_rate(n_e2e * nb, e2e_s, world), "n_e2e": n_e2e, "clocks": clocks.summary(),
        "ctas": model.num_ctas, "launches": n_launch,
    }
    for kv in kvs:
        kv.close()
    model.close()
    return cfg, res


def emit_batch(args, cfg, res, world):
    nb = res["nb"]
    value = whole_job_rate(res["steps"] * nb, res["ms"] * 1e-3, world)
    src = kernel_source_hash(BATCH_KERNEL_SOURCES)
    prof = f"decode_batch_kernel_{WORKLOAD}-b{nb}.md"
    tr = profiled_traffic(src, prof)
    line = {
        "metric": f"batch-{nb} decode tokens/s, all requests (2.3B, {WORKLOADS[WORKLOAD]['weights'].split(';')[0]}); "
                  "achieved HBM GB/s vs GB300 peak",
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": res["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(res["ms"] / res["steps"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_text(cfg),
        "data": WORKLOADS[WORKLOAD]["data"] + f"; {nb} requests with their own prompts",
        "config": {
            "workload": f"{WORKLOAD} as {nb} independent requests decoded together: each prompt 512, greedy "
                        "decode at contexts 513..1024",
            "weights": WORKLOADS[WORKLOAD]["weights"], "kv_cache": "f16", "batch": nb, "prompt": cfg["prompt_len"],
            "per_request_tokens_per_s": round(value / nb, 2),
            "kernel": "batched persistent kernel: one cooperative launch per window of up to 512 chained "
                      "batched steps (e2e: one launch per step)",
            "ctas": res["ctas"],
            "l2": f"inputs larger than L2: every step streams {res['weight_bytes'] / 1e9:.2f} GB of weights",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "e2e": {"value": round(res["e2e"], 2), "unit": "tokens/s", "h2d_bytes_per_step": 192,
                "d2h_bytes_per_step": 4 * nb + 4, "steps": res["n_e2e"], "per_step": res["step_pct"],
                "path": "adp_decode_batch per step (host tokens in and out, stream sync)"},
        "roofline": {"bound": "hbm", "achieved": round(res["achieved_gbs"], 1), "peak": res["peak"],
                     "unit": "GB/s", "frac": round(res["achieved_gbs"] / res["peak"], 4),
                     "traffic": None if tr is None else round(tr * res["steps"] / res["n_launch"]),
                     "kernel": "adp::decode_batch_kernel", "bytes_per_launch": int(res["per_launch_bytes"]),
                     "launch_ms": round(res["launch_ms"], 5),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({res['peak_kind']}; read+write copy)"},
        "gpu_launches": res["launches"],
        **({"profiling_variant": f"{cfg['n_layers']} layers (not the workload)"} if args.layers else {}),
        "clocks": res["clocks"],
        "kernel_source": src,
    }
    print(json.dumps(line), flush=True)


def run_prefill(args, rank: int, world: int):
    """Time to first token of the long-prompt workload (3,584-token prompt on the 2.3B fp16 model):
    adp_prefill_tc (prompt contractions on the tensor cores, the last token through the decode
    kernel) against adp_prefill (every prompt token a decode step, the bit-exact path)."""
    import torch

    import synth
    from autoregressive_decode_persistent_gb300 import adp, build
    from autoregressive_decode_persistent_gb300.model import DecodeModel

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    build.build()
    cfg = synth.get_config("dense-2.3b-fp16-long-t0.7")
    if args.layers:
        cfg["n_layers"] = args.layers
    W = synth.model_weights(cfg)
    model = DecodeModel(cfg, W, device=dev)
    prompt = synth.prompt(cfg)
    P = len(prompt)
    kv = model.new_kv()
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):  # the first call also builds the tensor-core weight tiles
        kv.reset()
        kv.prefill_tc(prompt)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    times = []
    with ClockSampler(local) as clocks:
        for _ in range(args.steps):
            kv.reset()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            h0 = time.perf_counter()
            e0.record(stream)
            kv.prefill_tc(prompt)  # host tokens in, host token out (synchronises)
            e1.record(stream)
            e1.synchronize()
            times.append((e0.elapsed_time(e1), (time.perf_counter() - h0) * 1e3))
    dev_ms = statistics.median(t[0] for t in times)
    host_ms = statistics.median(t[1] for t in times)
    # the bit-exact path: P decode steps in one persistent launch
    kv.reset()
    torch.cuda.synchronize(dev)
    h0 = time.perf_counter()
    kv.prefill(prompt)
    step_ms = (time.perf_counter() - h0) * 1e3
    # the dominant kernel: the gate|up GEMM over the prompt's P - 1 tokens, timed alone
    M = P - 1
    N, K = 2 * cfg["d_ff"], cfg["d_model"]
    g_ms = adp.adp_debug_tc_gemm_time(model.handle, 2, M, 20)
    dev_ms, host_ms = max_over_ranks([dev_ms, host_ms], world)
    res = {"dev_ms": dev_ms, "host_ms": host_ms, "step_ms": step_ms, "P": P, "gemm_ms": g_ms,
           "gemm_flops": 2.0 * M * N * K, "gemm_shape": (M, N, K), "clocks": clocks.summary(),
           "ctas": model.num_ctas, "n_layers": cfg["n_layers"]}
    kv.close()
    model.close()
    return cfg, res


def emit_prefill(args, cfg, res, world):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    achieved = res["gemm_flops"] / (res["gemm_ms"] * 1e-3) / 1e12
    M, N, K = res["gemm_shape"]
    L = res["n_layers"]
    line = {
        "metric": f"time to first token, {res['P']}-token prompt (2.3B fp16, tensor-core prefill)",
        "value": round(res["dev_ms"], 3),
        "unit": "ms",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["dev_ms"], 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 GEMM operands, f32 accumulation and activations",
        "data": "synthetic: seeded N(0,0.02) fp16 weights, 3584 uniform-random prompt ids",
        "config": {
            "workload": "dense-2.3b-fp16-long-t0.7 prompt: 3584 tokens at positions 0..3583 into an empty cache, "
                        "then the first generated token (greedy)",
            "prefill_tokens_per_s": round(res["P"] / (res["dev_ms"] * 1e-3), 1),
            "decode_path_ttft_ms": round(res["step_ms"], 1),
            "speedup_over_decode_path": round(res["step_ms"] / res["dev_ms"], 2),
            "kernel": f"per layer 4 tcgen05 GEMMs (M {M}; RoPE and the KV write in the QKV epilogue, SwiGLU in "
                      "the gate|up epilogue), tcgen05 flash attention and 2 norm kernels; the last prompt token "
                      "through the persistent decode kernel",
            "ctas": res["ctas"],
            "l2": "inputs larger than L2: 4.69 GB of weight tiles and the growing KV cache per prefill",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "e2e": {"value": round(res["host_ms"], 3), "unit": "ms", "h2d_bytes_per_step": 4 * res["P"] + 32,
                "d2h_bytes_per_step": 8, "path": "adp_prefill_tc: host token ids in, next token out (synchronises)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": f"adp::tc_gemm_kernel (gate|up with the SwiGLU epilogue: M {M}, N {N}, K {K}), "
                               f"{res['gemm_ms'] * 1e3:.1f} us per launch, 20 launches timed alone",
                     "peak_source": f"MEASURED_PEAKS.json bf16_tflops ({peak_kind}, burst; f16 has the same nominal "
                                    "tensor rate as bf16)"},
        "gpu_launches": 1 + 7 * L + 1,  # embedding; per layer 2 norms, 4 GEMMs, attention; the last token
        **({"profiling_variant": f"{L} layers (not the workload)"} if args.layers else {}),
        "clocks": res["clocks"],
        "kernel_source": kernel_source_hash(("prefill.cu", "tc.cuh", "device.cuh", "plan.h")),
    }
    print(json.dumps(line), flush=True)


def write_timeline(path, model, kv, tok0, P, cfg):
    """Per-phase breakdown of one decode step from the kernel's %globaltimer stamps."""
    import numpy as np
    import torch
    from autoregressive_decode_persistent_gb300 import adp
    G, nph = adp.adp_debug_timeline_shape(model.handle)
    buf = torch.zeros(G * nph * 16, dtype=torch.int64, device=model.device)  # zero = no stamp
    adp.adp_debug_timeline(model.handle, buf)
    kv.truncate(P)
    t = tok0
    for _ in range(4):
        t = kv.step(t)
    adp.adp_debug_timeline(model.handle, None)
    tl = buf.view(G, nph, 16).cpu().numpy().astype(np.float64)
    np.save(os.path.splitext(path)[0] + "_raw.npy", tl)
    names = {0: "qkv", 1: "attn", 2: "wo", 3: "gate_up", 4: "down", 5: "router", 6: "expert_gate_up",
             7: "expert_down", 8: "lm_head", 9: "sample"}
    kinds = [names[k] for k in _phase_kinds(cfg)]
    origin = tl[:, 0, 0].min()
    per_kind = {}
    rows = []
    for ph in range(nph - 1):  # the sampling phase does not run at temperature 0
        s = tl[:, ph, :]
        pro = np.mean(s[:, 1] - s[:, 0]) / 1e3
        body = np.mean(s[:, 2] - s[:, 1]) / 1e3
        bar = np.mean(s[:, 3] - s[:, 2]) / 1e3
        span = (s[:, 3].max() - s[:, 0].min()) / 1e3
        k = kinds[ph]
        d = per_kind.setdefault(k, {"prologue_us": 0.0, "body_us": 0.0, "barrier_us": 0.0, "count": 0})
        d["prologue_us"] += pro
        d["body_us"] += body
        d["barrier_us"] += bar
        d["count"] += 1
        if k not in ("attn", "sample") and np.any(s[:, 4] > 0):
            d.setdefault("ring_full_us", 0.0)
            d["ring_full_us"] += float(np.mean(s[:, 7]) / 1e3)
            d.setdefault("issue_span_us", 0.0)
            d["issue_span_us"] += float(np.mean(s[:, 5] - s[:, 4]) / 1e3)
        if k == "attn":
            w = s[:, 4] > 0
            if w.any():
                d.setdefault("tma_us", 0.0)
                d["tma_us"] += float(np.mean(s[w, 4] - s[w, 1]) / 1e3)
                d.setdefault("compute_us", 0.0)
                d["compute_us"] += float(np.mean(s[w, 6] - s[w, 4]) / 1e3)
                d.setdefault("publish_us", 0.0)
                d["publish_us"] += float(np.mean(s[w, 5] - s[w, 6]) / 1e3)
            d.setdefault("merge_us_max", 0.0)
            d["merge_us_max"] += float(np.max(s[:, 2] - s[:, 7]) / 1e3)
            d.setdefault("items_end_us_max", 0.0)
            d["items_end_us_max"] += float(np.max(s[:, 7] - s[:, 1]) / 1e3)
        rows.append({"phase": ph, "kind": k, "start_us": (s[:, 0].min() - origin) / 1e3, "prologue_us": pro,
                     "body_us": body, "barrier_us": bar, "span_us": span,
                     "body_max_us": float(np.max(s[:, 2] - s[:, 1]) / 1e3)})
    step_us = (tl[:, nph - 2, 3].max() - origin) / 1e3
    out = {"step_us": step_us, "ctas": G, "phases": nph, "per_kind": per_kind, "per_phase": rows}
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(f"timeline: step {step_us:.1f} us", file=sys.stderr)
    for k, d in per_kind.items():
        extra = "  ".join(f"{n} {v:.1f}" for n, v in d.items() if n not in ("prologue_us", "body_us", "barrier_us",
                                                                                 "count"))
        print(f"  {k:16s} x{d['count']:3d}  prologue {d['prologue_us']:8.1f}  body {d['body_us']:8.1f}  "
              f"barrier {d['barrier_us']:8.1f} us  {extra}", file=sys.stderr)


def _phase_kinds(cfg):
    ks = []
    for _ in range(cfg["n_layers"]):
        ks += [0, 1, 2] + ([3, 4] if not cfg["n_experts"] else [5, 6, 7])
    return ks + [8, 9]


def emit_engine(args, cfg, res, world):
    value = whole_job_rate(res["steps"], res["ms"] * 1e-3, world)
    src = kernel_source_hash()
    line = {
        "metric": WORKLOADS[WORKLOAD]["metric"],
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": res["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(res["ms"] / res["steps"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_text(cfg),
        "data": WORKLOADS[WORKLOAD]["data"],
        "config": {
            "workload": workload_text(cfg),
            "weights": WORKLOADS[WORKLOAD]["weights"], "kv_cache": cfg["kv_dtype"], "batch": 1,
            "prompt": cfg["prompt_len"],
            "contexts": f"{cfg['prompt_len'] + 1}..{cfg['prompt_len'] + min(res['steps'], WINDOW)}",
            "temperature": WORKLOADS[WORKLOAD]["temperature"],
            "kernel": f"persistent: one cooperative launch per window of up to {WINDOW} chained decode steps "
                      "(e2e: one launch per step)",
            "ctas": res["ctas"],
            "l2": f"inputs larger than L2: every step streams {res['weight_bytes'] / 1e9:.2f} GB of weights "
                  "(L2 129 MB)",
            "timed_regions": "3 regions of exactly `steps` steps; value from the median region",
            "runs_tokens_per_s": [round(whole_job_rate(res["steps"], r * 1e-3, world), 2) for r in res["runs_ms"]],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "e2e": {"value": round(res["e2e"], 2), "unit": "tokens/s", "h2d_bytes_per_step": 32,
                "d2h_bytes_per_step": 8, "steps": res["n_e2e"], "per_step": res["step_pct"],
                "path": "adp_decode_step per token (host token in, host token out, stream sync)"},
        "roofline": {"bound": "hbm", "achieved": round(res["achieved_gbs"], 1), "peak": res["peak"],
                     "unit": "GB/s", "frac": round(res["achieved_gbs"] / res["peak"], 4),
                     "traffic": (None if profiled_traffic(src) is None
                                 else round(profiled_traffic(src) * res["steps"] / res["n_launch"])),
                     "kernel": "adp::decode_kernel",
                     "bytes_per_launch": int(res["per_launch_bytes"]),
                     "launch_ms": round(res["launch_ms"], 5),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({res['peak_kind']}; read+write copy)",
                     "frac_of_8000": round(res["achieved_gbs"] / 8000.0, 4),
                     "read_probe_gbs": round(res["read_gbs"], 1),
                     "frac_of_read_probe": round(res["achieved_gbs"] / res["read_gbs"], 4),
                     "read_probe": "same run: adp_measure_read_bandwidth, 16-byte loads over a 4 GiB buffer, "
                                   "5 launches timed with CUDA events"},
        "gpu_launches": res["launches"],
        **({"profiling_variant": f"{cfg['n_layers']} layers (not the workload)"} if args.layers else {}),
        "clocks": res["clocks"],
        "kernel_source": src,
    }
    if res.get("ablation"):
        line["launch_ablation"] = res["ablation"]
    if "cpu" in res:
        line["cpu_baseline"] = res["cpu"]
    print(json.dumps(line), flush=True)


def run_reference(args, rank: int, world: int):
    """Reference arm: the CPU oracle (plain fp32) on the same workload, bounded."""
    if rank != 0:
        return
    import synth
    cfg = synth.get_config(WORKLOAD)
    W = synth.model_weights(cfg)
    budget = max(10.0, min(120.0, args.cpu_seconds * 4))
    cpu, n, el = cpu_baseline(cfg, W, seconds=budget, max_steps=max(2, args.steps), warmup=args.warmup)
    value = cpu["value"]
    line = {
        "impl": "reference",
        "metric": WORKLOADS[WORKLOAD]["metric"],
        "value": round(value, 4),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": n,
        "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / n, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_text(cfg),
        "data": WORKLOADS[WORKLOAD]["data"],
        "config": {"workload": workload_text(cfg), "weights": WORKLOADS[WORKLOAD]["weights"], "batch": 1,
                   "prompt": cfg["prompt_len"]},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "reference": "CPU oracle (oracle/oracle.c, plain mode): the pages publish no code to install",
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["engine", "reference"], default="engine")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=WORKLOAD,
                    help="the benchmarked model (default: the 2.3B fp16 decoder)")
    ap.add_argument("--ablation-steps", type=int, default=64,
                    help="steps of the one-launch-per-phase ablation (0 = skip)")
    ap.add_argument("--timeline", default=None, help="write a per-phase breakdown of one step (JSON) here")
    ap.add_argument("--batch", type=int, default=1,
                    help="decode this many independent requests together (batched kernel; default 1: the "
                         "single-request benchmark)")
    ap.add_argument("--prefill", action="store_true",
                    help="time to first token of the 3584-token prompt through the tensor-core prefill")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: use this many layers of the workload's shape (the line says so)")
    args = ap.parse_args()
    globals()["WORKLOAD"] = args.workload
    globals()["WINDOW"] = WORKLOADS[args.workload]["window"]
    if (args.batch > 1 or args.prefill) and args.workload not in ("dense-2.3b-fp16", "dense-2.3b-e4m3",
                                                                  "dense-2.3b-nvfp4"):
        ap.error("--batch and --prefill measure the 2.3B model (--workload dense-2.3b-*)")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.batch < 1:
        ap.error("--batch must be >= 1")
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.prefill:
        cfg, res = run_prefill(args, rank, world)
        if rank == 0:
            emit_prefill(args, cfg, res, world)
    elif args.batch > 1:
        cfg, res = run_engine_batch(args, rank, world)
        if rank == 0:
            emit_batch(args, cfg, res, world)
    else:
        cfg, res = run_engine(args, rank, world)
        if rank == 0:
            emit_engine(args, cfg, res, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
