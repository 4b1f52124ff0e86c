"""Benchmark of the layer-streamed training step (one JSON line on stdout).

A step is one mt_train_step (every block streamed in from the pinned host arena,
forward, loss, backward, every gradient streamed back) followed by the host
Adam update (timed separately). Default workload: the 7B Llama-style model
(32 layers, hidden 4096, 32 heads, FFN 11008, vocab 32000, seq 4096, batch 2)
with synthetic seeded weights and uniform random tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 7b] [--impl reference]

--impl reference times the plain CPU oracle on the host cores (the reference
arm: a deliberately slow program, not an optimisation target).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIGS = {
    "tiny": dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, ffn=1024, vocab=1024, seq=128, batch=2),
    "1.3b": dict(n_layers=24, hidden=2048, n_heads=16, n_kv_heads=16, ffn=5504, vocab=32000, seq=2048, batch=4),
    "7b": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=4096, batch=2),
    "14b": dict(n_layers=48, hidden=5120, n_heads=40, n_kv_heads=8, ffn=13824, vocab=152064, seq=4096, batch=1),
    "7b_long": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=131072,
                    batch=1),
    # twice the long-context length: fp32 checkpoints stay in HBM (33 x 4.3 GB), the LM head
    # runs in 8 chunks of 32768 tokens, the host holds only the arena
    "7b_256k": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=262144,
                    batch=1),
}
NAMES = {"tiny": "tiny decoder (2L h256)", "1.3b": "1.3B Llama-style", "7b": "7B Llama-style",
         "14b": "14B GQA (48L h5120 40H/8KV)", "7b_long": "7B Llama-style, seq 131072",
         "7b_256k": "7B Llama-style, seq 262144"}
METRIC = "streamed train step TFLOPS & tokens/s at 7B/14B; % of per-layer roofline"


def model_flops(kw) -> float:
    """Model FLOPs of one training step: 6 P_nonemb T + 6 B s^2 h L (causal half) + 6 T h V (LM head)."""
    h, f, V, L, s, B = kw["hidden"], kw["ffn"], kw["vocab"], kw["n_layers"], kw["seq"], kw["batch"]
    hd = h // kw["n_heads"]
    qd, kvd = kw["n_heads"] * hd, kw["n_kv_heads"] * hd
    p_layer = qd * h + 2 * kvd * h + h * qd + 3 * f * h + 2 * h
    T = B * s
    return 6.0 * p_layer * L * T + 6.0 * B * s * s * h * L + 6.0 * T * h * V


def layer_params(kw) -> int:
    h, f = kw["hidden"], kw["ffn"]
    hd = h // kw["n_heads"]
    qd, kvd = kw["n_heads"] * hd, kw["n_kv_heads"] * hd
    return qd * h + 2 * kvd * h + h * qd + 3 * f * h + 2 * h


def per_layer_roofline_ms(kw, peak_tflops, h2d_gbs, d2h_gbs, offload=False) -> float:
    """Sum over block phases of max(FLOPs / peak, H2D bytes / H2D BW, D2H bytes / D2H BW).

    FLOPs are the method's work: per layer the forward (2 P T + the causal attention forward,
    two causal-half products of B s^2 h FLOPs each) and, in the backward phase, the recompute
    (the same again) plus the backward (4 P T + five causal-half products: S, dP, dV, dK, dQ).
    The kernels' own extra recomputation (the deterministic backward computes S and dP twice)
    is not counted as work."""
    h, V, L, s, B = kw["hidden"], kw["vocab"], kw["n_layers"], kw["seq"], kw["batch"]
    T = B * s
    P = layer_params(kw)
    attn_f = 2.0 * B * s * s * h
    pk = peak_tflops * 1e12
    hb, db = h2d_gbs * 1e9, d2h_gbs * 1e9
    ck = 4.0 * T * h if offload else 0.0
    t = 0.0
    # embedding block: the gather reads only the batch's rows of E from the arena and the
    # backward writes only the changed gradient rows (this batch's ids and zeros over the last
    # batch's): at most T rows in and 2 T rows out instead of the vocabulary
    e_in, e_out = 2.0 * min(T, V) * h, 2.0 * min(2 * T, V) * h
    t += e_in / hb  # embedding rows in
    for _ in range(L):  # forward
        t += max((2.0 * T * P + attn_f) / pk, 2.0 * P / hb, ck / db)
    head_f = 3 * 2.0 * T * h * V
    t += max(head_f / pk, 2.0 * (V * h + h) / hb, 2.0 * (V * h + h) / db)
    for _ in range(L):  # recompute (the forward's attention again) + backward (5 causal-half products)
        t += max((6.0 * T * P + 3.5 * attn_f) / pk, (2.0 * P + ck) / hb, 2.0 * P / db)
    t += e_out / db  # embedding gradient rows out
    return t * 1e3


# DRAM bytes per GEMM launch of the 7B step (read + write), from one ncu capture of a whole step
# (its launch list is summarised under profiles/); valid only for the GEMM source it was taken on.
GEMM_TRAFFIC = {"7b": (862.7e6, "9fe2aa5fb89dc33c")}


def gemm_traffic(config):
    """Measured DRAM bytes per GEMM launch for this workload, or None when there is no capture
    for it or the GEMM source has changed since the counters were taken."""
    import hashlib

    if config not in GEMM_TRAFFIC:
        return None
    bytes_, sha = GEMM_TRAFFIC[config]
    src = os.path.join(ROOT, "host_memory_streamed_stream_gb300", "csrc", "gemm.cu")
    return bytes_ if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == sha else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.idx = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def mem_available() -> int:
    """MemAvailable from /proc/meminfo in bytes (0 if unknown)."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def dist_setup(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist

    dist.init_process_group("gloo")
    return dist.get_rank(), dist.get_world_size(), dist


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(kw, budget_s=20.0, warmup=0):
    """Time the oracle as it stands, in its float32 instantiation (the plain fp32 CPU
    implementation of the step), on a bounded sample of the workload's shapes: one decoder
    layer plus the head, at the workload's hidden/FFN/vocab sizes, on one sequence of length
    min(seq, 512), after `warmup` untimed runs of the same sample. The rate is extrapolated to
    the whole step by model FLOPs. Returns (TFLOP/s, description, threads)."""
    import numpy as np

    import oracle
    import synth

    s = min(kw["seq"], 512)
    cfg = oracle.Config(n_layers=1, hidden=kw["hidden"], n_heads=kw["n_heads"], n_kv_heads=kw["n_kv_heads"],
                        ffn=kw["ffn"], vocab=kw["vocab"], seq=s, batch=1)
    W = oracle.init_params(cfg, synth, synth.WEIGHT_SEED)
    tok = synth.tokens(cfg.tokens, cfg.vocab)
    lab = synth.labels(cfg.tokens, cfg.vocab)
    sample_kw = dict(kw, n_layers=1, seq=s, batch=1)
    flops = model_flops(sample_kw)
    for _ in range(warmup):
        oracle.forward_backward(cfg, W, tok, lab, np.float32)
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.forward_backward(cfg, W, tok, lab, np.float32)
        runs += 1
        el = time.perf_counter() - t0
        if el > budget_s or el / runs * (runs + 1) > 2 * budget_s:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"oracle float32 forward+backward of 1 decoder layer + LM head at the workload's widths "
            f"(h {kw['hidden']}, ffn {kw['ffn']}, vocab {kw['vocab']}), 1 sequence of {s} tokens, {runs} run(s), "
            f"{el:.1f} s")
    return flops * runs / el / 1e12, desc, threads


def run_reference(args, kw):
    rank, world, dist = dist_setup(args.gpus)
    if rank != 0:
        return
    vals = []
    desc, threads = "", 1
    for i in range(max(1, args.steps)):
        # one untimed run ahead of the first timed sample warms the BLAS threads and the caches;
        # further warm-up runs would only lengthen the arm (each run is seconds)
        budget = max(min(3.0, args.ref_seconds), args.ref_seconds / max(1, args.steps))
        v, desc, threads = oracle_sample(kw, budget_s=budget, warmup=min(1, args.warmup) if i == 0 else 0)
        vals.append(v)
    value = statistics.median(vals)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,0.02) weights, uniform tokens)",
           "config": {"workload": NAMES[args.config], **kw, "sample": desc},
           "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------------------- GPU leg
def measure_link(torch, nbytes=1 << 30, reps=5):
    """Pinned host<->device copy bandwidth (GB/s) with CUDA events: H2D, D2H. The host buffer
    comes from the library's allocator, the same kind of memory as the arena."""
    import host_memory_streamed_stream_gb300 as mt

    buf = mt.HostArena(nbytes)
    h = torch.from_numpy(buf.array)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    res = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)), ("d2h", lambda: h.copy_(d, non_blocking=True))):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        res[name] = nbytes * reps / (a.elapsed_time(b) / 1e3) / 1e9
    del h, d
    buf.free()
    return res


def measure(args, name, kw, steps, warmup, kernel_steps, overlap_steps, link, peaks, dist, world, local):
    """Build one configuration's arena and trainer, run `warmup` untimed and `steps` timed steps
    (each: mt_train_step, then the host Adam), then the instrumented and overlapped extra steps;
    return the measured quantities. The arena is freed before returning."""
    import torch

    import host_memory_streamed_stream_gb300 as mt
    import synth

    flags = mt.FLAG_SINGLE_BUFFER if args.single_buffer else 0
    if args.fp32_master:
        flags |= mt.FLAG_FP32_MASTER
    if args.dense_embed:
        flags |= mt.FLAG_DENSE_EMBED
    if name == "7b_long":
        flags |= mt.FLAG_OFFLOAD_CKPT
    cfg = mt.ModelConfig(**kw, flags=flags)
    # the arena (and, with checkpoint offload, the checkpoints) are pinned host memory: refuse
    # to start rather than drive the host out of memory
    # (the allocator briefly holds 6 % more as spare pages)
    pinned = int(1.06 * mt.arena_bytes(cfg)) + (cfg.n_layers * cfg.tokens * cfg.hidden * 4
                                                if flags & mt.FLAG_OFFLOAD_CKPT else 0)
    avail = mem_available()
    if avail and avail < pinned + 8 * 2**30:
        return {"skipped": f"not enough host memory for {name}: {pinned / 2**30:.1f} GiB pinned + 8 GiB margin, "
                           f"{avail / 2**30:.1f} GiB available"}
    tok = synth.tokens(cfg.tokens, cfg.vocab)
    lab = synth.labels(cfg.tokens, cfg.vocab)
    t_setup = time.perf_counter()
    tr = mt.Trainer(cfg)
    arena_info = tr.arena.info()
    mt.fill_synthetic(cfg, tr.arena, synth, synth.WEIGHT_SEED)
    t_setup = time.perf_counter() - t_setup
    # the host Adam's memory roofline: a triad over the same threads, before the timed steps
    host_gbs, host_threads = mt.host_bandwidth(3 << 30, 5)

    step_no = 0

    def one_step():
        # public API: host tokens in, every block streamed, loss out (timed: `e2e`); then the
        # host Adam update, inside the timed region but timed separately (`adam_ms`)
        nonlocal step_no
        step_no += 1
        t0 = time.perf_counter()
        loss = tr.step(tok, lab)
        host_ms = (time.perf_counter() - t0) * 1e3
        st = tr.stats()
        tr.adam(step_no)
        st["adam_ms"] = tr.stats()["adam_ms"]
        return loss, host_ms, st

    losses = []
    for _ in range(warmup):
        losses.append(one_step()[0])
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0 = time.perf_counter()
    recs = []
    for _ in range(steps):
        loss, host_ms, st = one_step()
        losses.append(loss)
        recs.append((host_ms, st))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    # a second link probe right after the timed steps, next to the copy speed the steps achieved
    link_after = measure_link(torch)
    if dist is not None:
        dist.barrier()
    # per-kernel durations: CUDA events around every launch, in extra instrumented steps of
    # the same workload (the events cost the step a few percent, so `value` comes from the
    # un-instrumented steps above)
    tr.set_kernel_timing(True)
    krecs = []
    for _ in range(kernel_steps):
        _, _, st_k = one_step()
        krecs.append((st_k, tr.kernel_stats()))
    tr.set_kernel_timing(False)
    # the overlapped schedule: each block's host Adam update starts as soon as its gradients
    # land (mt_train_step_adam), timed as whole iterations
    ovl = []
    for _ in range(overlap_steps):
        step_no += 1
        t_a = time.perf_counter()
        tr.step_adam(tok, lab, step_no)
        ovl.append(((time.perf_counter() - t_a) * 1e3, tr.stats()["step_ms"]))

    step_ms = [r[1]["step_ms"] for r in recs]
    host_ms = [r[0] for r in recs]  # host wall time of the step call
    adam_ms = [r[1]["adam_ms"] for r in recs]
    dev_ms = max_over_ranks(dist, statistics.mean(step_ms))
    e2e_ms = max_over_ranks(dist, statistics.mean(host_ms))
    flops = model_flops(kw)
    ks = {}
    for _, k in krecs:
        for kname, d in k.items():
            a = ks.setdefault(kname, {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0})
            for f in a:
                a[f] += d[f]
    peak_sus = peaks["bf16_tflops_sustained"]
    roof_ms = per_layer_roofline_ms(kw, peak_sus, link["h2d"], link["d2h"], offload=bool(flags & mt.FLAG_OFFLOAD_CKPT))
    copy_busy = statistics.mean([r[1]["h2d_busy_ms"] + r[1]["d2h_busy_ms"] for r in recs])

    def phase_gbs(direction, phase):
        b = sum(r[1]["copy_bytes"][direction][phase] for r in recs)
        ms = sum(r[1]["copy_ms"][direction][phase] for r in recs)
        return round(b / (ms / 1e3) / 1e9, 1) if ms > 0 and b > 0 else None

    adam_floor_ms = 22.0 * cfg.params() / (host_gbs * 1e9) * 1e3 if host_gbs > 0 else None
    exposed = statistics.mean([r[1]["exposed_ms"] for r in recs])
    m = {
        "dev_ms": dev_ms, "e2e_ms": e2e_ms, "flops": flops, "tokens": cfg.tokens, "wall": wall, "clocks": clocks,
        "losses": losses, "last": recs[-1][1], "ks": ks, "ovl": ovl, "roof_ms": roof_ms, "t_setup": t_setup,
        "arena": arena_info,
        "value": flops * world / (dev_ms / 1e3) / 1e12, "e2e_value": flops * world / (e2e_ms / 1e3) / 1e12,
        "tokens_s": cfg.tokens * world / (dev_ms / 1e3),
        "kernels_per_step": statistics.mean([r[1]["kernel_launches"] for r in recs]),
        "host_ms": statistics.mean(host_ms), "adam_ms": statistics.mean(adam_ms),
        "adam_roofline": {"host_triad_gbs": round(host_gbs, 1), "threads": host_threads, "bytes_per_param": 22,
                          "floor_ms": round(adam_floor_ms, 1) if adam_floor_ms else None,
                          "frac": round(adam_floor_ms / statistics.mean(adam_ms), 4) if adam_floor_ms else None},
        "transfer": {"exposed_ms": round(exposed, 3), "copy_busy_ms": round(copy_busy, 3),
                     "hidden_frac": round(max(0.0, 1 - exposed / copy_busy), 4) if copy_busy > 0 else None,
                     "h2d_gbs_in_step": round(statistics.mean(
                         [r[1]["h2d_bytes"] / (r[1]["h2d_busy_ms"] / 1e3) / 1e9 for r in recs]), 1),
                     "d2h_gbs_in_step": round(statistics.mean(
                         [r[1]["d2h_bytes"] / (r[1]["d2h_busy_ms"] / 1e3) / 1e9 for r in recs]), 1),
                     "link_probe_after": {"h2d_gbs": round(link_after["h2d"], 1),
                                          "d2h_gbs": round(link_after["d2h"], 1)},
                     "fwd_ms": round(statistics.mean([r[1]["fwd_ms"] for r in recs]), 3),
                     "bwd_ms": round(statistics.mean([r[1]["bwd_ms"] for r in recs]), 3),
                     "h2d_gbs_fwd": phase_gbs(0, 0), "h2d_gbs_bwd": phase_gbs(0, 1),
                     "d2h_gbs_fwd": phase_gbs(1, 0), "d2h_gbs_bwd": phase_gbs(1, 1),
                     "first_copy_ms": round(statistics.mean([r[1]["first_copy_ms"] for r in recs]), 3),
                     "sparse_embed_steps": sum(int(r[1]["sparse_embed"]) for r in recs),
                     "embed_gather_gbs": round(statistics.mean([r[1]["embed_gather_gbs"] for r in recs]), 1)},
    }
    tr.close()  # frees the pinned arena before the next configuration or the oracle's CPU sample
    return m


def kernel_table(ks, kernel_steps):
    return {n: {"launches_per_step": d["launches"] / max(1, kernel_steps),
                "ms_per_step": round(d["ms"] / max(1, kernel_steps), 3),
                "tflops": round(d["flops"] / (d["ms"] / 1e3) / 1e12, 1) if d["ms"] > 0 and d["flops"] else None,
                "gbs": round(d["bytes"] / (d["ms"] / 1e3) / 1e9, 1) if d["ms"] > 0 and d["bytes"] else None}
            for n, d in ks.items()}


def host_warmup(nbytes: int, local: int) -> float:
    """Allocate, probe and release an arena-sized pinned buffer in a child process (seconds taken).

    Measured on this platform: host memory pinned for the first time in a process (after the box
    started, or after another process used and released it) can copy at 3-10 GB/s for the whole
    life of that process, although a probe right after allocating it read full speed; pinned
    again by a later process, the same memory copies at full speed. A short-lived child that
    pins as much as the run's largest arena first leaves the measured process normal memory."""
    t0 = time.perf_counter()
    code = ("import sys; sys.path.insert(0, %r); import torch; torch.cuda.set_device(%d); "
            "import host_memory_streamed_stream_gb300 as mt; a = mt.HostArena(%d); a.free()" % (ROOT, local, nbytes))
    subprocess.run([sys.executable, "-c", code], check=False, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
    return time.perf_counter() - t0


def run_gpu(args, kw):
    import torch

    rank, world, dist = dist_setup(args.gpus)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    warm_s = None
    if not args.no_host_warmup:
        import host_memory_streamed_stream_gb300 as mt

        # as large as the largest arena this run allocates (the main configuration or an 'also'
        # one), if the host has room for it next to the other ranks' (replicas share the host)
        names = [args.config] + [a for a in args.also.split(",") if a in CONFIGS]
        need = max(mt.arena_bytes(mt.ModelConfig(**CONFIGS[n])) for n in names)
        avail = mem_available()
        if avail and world > 1:
            need = min(need, avail // world - 8 * 2**30)
        if need > 0 and (not avail or 1.06 * need + 8 * 2**30 <= avail):
            warm_s = host_warmup(need, local)
    torch.cuda.set_device(local)
    peaks = load_peaks()
    link = measure_link(torch)
    m = measure(args, args.config, kw, args.steps, args.warmup, args.kernel_steps, args.overlap_steps, link, peaks,
                dist, world, local)
    if "skipped" in m:
        raise SystemExit(m["skipped"])
    # the other headline model size, measured after the main one in the same run with fewer steps
    also = {}
    for name in [a for a in args.also.split(",") if a and a != "none" and a != args.config]:
        a_steps = max(1, min(args.steps, 5))
        am = measure(args, name, CONFIGS[name], a_steps, 2, 1, 0, link, peaks, dist, world, local)
        if "skipped" in am:
            also[name] = {"skipped": am["skipped"]}
            continue
        a_roof = am["roof_ms"]
        ag = am["ks"].get("gemm", {"ms": 0.0, "flops": 0.0})
        also[name] = {
            "workload": NAMES[name], **CONFIGS[name], "steps": a_steps, "warmup": 2,
            "value": round(am["value"], 2), "unit": "TFLOPS", "ms_per_step": round(am["dev_ms"], 3),
            "tokens_per_s": round(am["tokens_s"], 1), "e2e_tflops": round(am["e2e_value"], 2),
            "per_layer_roofline": {"roofline_ms": round(a_roof, 3), "frac": round(a_roof / am["dev_ms"], 4)},
            "transfer": am["transfer"], "adam_ms": round(am["adam_ms"], 1), "adam_roofline": am["adam_roofline"],
            "gemm_tflops": round(ag["flops"] / (ag["ms"] / 1e3) / 1e12, 1) if ag["ms"] > 0 else None,
            "kernels": kernel_table(am["ks"], 1), "clocks": am["clocks"], "loss": [round(x, 5) for x in am["losses"]],
            "arena": am["arena"],
        }
    if rank != 0:
        return
    cpu_v, cpu_desc, cpu_threads = oracle_sample(kw, budget_s=args.cpu_budget) if not args.no_cpu else (None, "", 0)
    ks = m["ks"]
    g = ks.get("gemm", {"ms": 0.0, "flops": 0.0})  # no instrumented steps (--kernel-steps 0): no kernel rates
    gemm_alg_bytes = g.get("bytes", 0.0)
    gemm_tflops = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else 0.0
    peak_sus = peaks["bf16_tflops_sustained"]
    ovl = m["ovl"]
    out = {
        "metric": METRIC,
        "value": round(m["value"], 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(m["dev_ms"], 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights, unit gains, zero Adam state, uniform tokens/labels)",
        "config": {"workload": NAMES[args.config], **kw, "parallelism": f"replicas x{world}",
                   "state": "pinned host arena (bf16 W/G, fp32 Adam m/v), streamed per layer",
                   "l2": "inputs larger than L2: every step streams the whole arena's W/G sections",
                   "tflops_definition": "model FLOPs: 6 P_nonemb T + 6 B s^2 h L (causal) + 6 T h V",
                   "schedule": "single buffer (ablation)" if args.single_buffer else "double-buffered, 3 streams",
                   "master_weights": "fp32 (16 B/param)" if args.fp32_master else "none (12 B/param)"},
        "tokens_per_s": round(m["tokens_s"], 1),
        "per_layer_roofline": {"roofline_ms": round(m["roof_ms"], 3), "frac": round(m["roof_ms"] / m["dev_ms"], 4),
                               "peak_tflops": peak_sus, "h2d_gbs": round(link["h2d"], 1),
                               "d2h_gbs": round(link["d2h"], 1), "peak_source": peaks["source"] + " (sustained)"},
        "transfer": m["transfer"],
        "adam_ms": round(m["adam_ms"], 1),
        "adam_roofline": m["adam_roofline"],
        "iteration": {"ms_sequential": round(m["host_ms"] + m["adam_ms"], 1),
                      "ms_overlapped": round(statistics.mean([q[0] for q in ovl]), 1) if ovl else None,
                      "overlapped_step_ms": round(statistics.mean([q[1] for q in ovl]), 1) if ovl else None,
                      "note": "sequential: mt_train_step then mt_adam_step (the timed steps); overlapped: "
                              "mt_train_step_adam, each block's Adam update starting when its gradients land"},
        "loss": [round(x, 5) for x in m["losses"]],
        "roofline": {"bound": "tensor", "kernel": "tcgen05 GEMM (fwd/dgrad/wgrad)",
                     "achieved": round(gemm_tflops, 1), "peak": peak_sus, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / peak_sus, 4), "traffic": gemm_traffic(args.config),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
                     "algorithmic_bytes_per_launch": round(gemm_alg_bytes / max(1.0, g.get("launches", 0)))
                     if g.get("launches") else None,
                     "peak_source": peaks["source"] + " bf16 sustained",
                     "timing": f"CUDA events around each launch on the compute stream, {args.kernel_steps} "
                               "instrumented steps after the timed ones"},
        "kernels": kernel_table(ks, args.kernel_steps),
        "cpu_baseline": {"value": cpu_v, "unit": "TFLOPS", "cores": cpu_threads, "kind": "oracle",
                         "sample": cpu_desc},
        "e2e": {"value": round(m["e2e_value"], 2), "unit": "TFLOPS",
                "h2d_bytes_per_step": int(m["last"]["h2d_bytes"]), "d2h_bytes_per_step": int(m["last"]["d2h_bytes"]) + 8,
                "note": "host wall time of Trainer.step: host token arrays in, every block streamed, loss read back"},
        "gpu_launches": int(m["kernels_per_step"] * args.steps),
        "clocks": m["clocks"],
        "wall_s": round(m["wall"], 3),
        "setup_s": round(m["t_setup"], 1),
        "arena": m["arena"],
        "host_warmup_s": round(warm_s, 1) if warm_s is not None else None,
    }
    if also:
        out["also"] = also
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="7b", choices=list(CONFIGS))
    ap.add_argument("--impl", default="mt", choices=["mt", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: oracle time spread over the steps (at least min(3 s, this) each)")
    ap.add_argument("--kernel-steps", type=int, default=2)
    ap.add_argument("--overlap-steps", type=int, default=2)
    ap.add_argument("--single-buffer", action="store_true",
                    help="ablation: one device layer buffer, each block's copy then its compute")
    ap.add_argument("--fp32-master", action="store_true",
                    help="arena with an fp32 master copy of the weights (Adam updates it, W = bf16(P))")
    ap.add_argument("--dense-embed", action="store_true",
                    help="copy the embedding block whole instead of its batch rows through the mapped arena")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-host-warmup", action="store_true",
                    help="skip the child process that takes the first pinned allocation (see host_warmup)")
    ap.add_argument("--also", default="14b",
                    help="comma-separated further configurations measured after the main one with at most 5 timed "
                         "steps and reported under 'also' ('none': only the main one)")
    args = ap.parse_args()
    kw = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, kw)
    else:
        run_gpu(args, kw)


if __name__ == "__main__":
    main()
