"""Benchmark of the single-token decode step of one attention layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload full_b1_32k] [--replicas R] [--extra all|none|name,...]

One step = one pass of the whole decode path (input norm + QKV + norms + RoPE + KV append
-> flash-decode -> o_proj + residual) over one batch of the workload: one launch of the
persistent decode-step kernel.  Every timed step runs on a different layer replica (distinct
weights and caches in HBM, R replicas of ~179 MB for the 32K full-attention layer), so the
inputs of a step are never L2-resident: together they are far larger than the 129 MB L2.
The replicas are chained like the layers of a model (each step prefetches the next
replica's first weights during its own tail).

Printed (one JSON line, rank 0): steps/s for the whole job on the headline workload (the
32K full-attention layer at batch 1), ms per step, the roofline of the step kernel
(algorithmic bytes of the step -- Q8_0 weights, visible K/V rows, activations -- over its
CUDA-event duration, against the measured HBM copy bandwidth), the kernel's own duration
from its device timer stamps, the end-to-end rate through the host-buffer entry point, the
CPU oracle baseline, SM clocks sampled during the timed region, the launch count, and under
"workloads" the same figures for the other workloads (the tiny sliding layer, the
batch-16 sliding ring, the 128K batch-4 layer with softcap, the 16-token verify block, and
the layer's dense FFN half at batch 1 and 16).

The K timed steps are one CUDA graph whose first and last nodes record the timing events,
so the timed region is exactly the K steps on the device (no host launch latency).

--impl reference times the CPU oracle (the plain fp64 implementation the tests check the
library against) on the host cores, same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode steps/sec per layer at 1 GB300; achieved HBM GB/s as % of peak"
UNIT = "steps/s"
VERIFY_METRIC = "verify blocks/sec per layer (L tokens, bf16 weights)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
EXTRA = ("tiny_sliding", "sliding_b16_ring1024", "full_b4_128k_softcap", "verify_l16_8k",
         "global_hd512_32k", "verify_global_hd512_32k", "drafter_l16_8k", "ffn_b1", "ffn_b16", "tq8_full_b1_32k",
         "tq4_full_b1_32k", "tq8_global_hd512_32k")
# attention over a quantised (TurboQuant) KV cache: the attention shapes of the headline
# layer (batch 1, 32/8 heads, head dim 128) and of the global layer (16/2 heads, head dim
# 512), 32768 visible keys
# coded-cache attention workloads: bits, head dim, query heads, KV heads (batch 1, 32K keys)
TQ = {"tq8_full_b1_32k": (8, 128, 32, 8), "tq4_full_b1_32k": (4, 128, 32, 8),
      "tq8_global_hd512_32k": (8, 512, 16, 2)}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="full_b1_32k")
    p.add_argument("--replicas", type=int, default=8)
    p.add_argument("--extra", default="all",
                   help="other workloads measured in the same run: all, none, or names")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def cpu_info():
    """CPU model and logical core count of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        model = m.group(1).strip() if m else None
    except Exception:
        pass
    if not model and os.path.exists("/proc/cpuinfo"):
        m = re.search(r"model name\s*:\s*(.+)", open("/proc/cpuinfo").read())
        model = m.group(1).strip() if m else None
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count()}


def workload_bytes(w, pos):
    """Algorithmic bytes of one step: Q8_0 weights at 34/32 B per weight, the visible
    bf16 K and V rows, activations in and out, the appended K/V row."""
    H, nkv, hd = w.hidden, w.num_kv_heads, w.head_dim
    kv_proj = 1 if w.k_eq_v else 2  # k_eq_v layers have no V projection
    wbytes = (w.q_rows + kv_proj * w.kv_rows) * H * 34 // 32 + H * w.q_rows * 34 // 32
    kv = 0
    for P in pos:
        if w.ring:
            n = min(int(P) + 1, w.kv_capacity)
        elif w.layer_type == 0:
            n = int(P) - max(0, int(P) - w.window + 1) + 1
        else:
            n = int(P) + 1
        kv += n * nkv * hd * 2 * 2
    act = len(pos) * (H * 2 * 2 + nkv * hd * 2 * 2)
    return wbytes, kv, act


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def ncu_traffic(kernel_file, summary_name):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source it was
    taken on is the current one (its sha256 is recorded in the summary)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    src = os.path.join(ROOT, "quantized_attention_layer_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    text = open(path).read()
    m_sha = re.search(r"source sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram bytes per launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m_b.group(1)) if sha == m_sha.group(1) else None


def cpu_baseline(w, weights, x, pos, kv, budget_s=15.0):
    """The oracle on the host cores: all cores for ~2/3 of the budget, one core for the rest."""
    import oracle
    oracle.build()
    all_threads = oracle.num_threads()

    def rate(seconds):
        n, t0 = 0, time.perf_counter()
        while True:
            oracle.decode_step(w, weights, x, pos, kv["k_cache"], kv["v_cache"])
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
        return n, time.perf_counter() - t0

    n, dt = rate(budget_s * 2 / 3)
    oracle.set_num_threads(1)
    try:
        n1, dt1 = rate(budget_s / 3)
    finally:
        oracle.set_num_threads(all_threads)
    info = cpu_info()
    return {"value": n / dt, "unit": UNIT, "cores": all_threads, "kind": "oracle",
            "sample": f"{n} full oracle decode steps of {w.name} (batch {len(pos)}), fp64, "
                      f"{dt:.1f} s on {all_threads} threads; {n1} steps in {dt1:.1f} s on 1 thread",
            "single_thread": {"value": n1 / dt1, "unit": UNIT, "cores": 1},
            **info}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from quantized_attention_layer_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = wl.BY_NAME[args.workload]
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    if w.verify_len:  # the same operation as our arm: a verify block (after its context rows)
        S = wl.DRAFTER_CTX_ROWS if w.block_bidir else 0
        x_ctx = wl.bf16_normal((S, w.hidden), torch.Generator().manual_seed(w.seed + 5)) if S else None

        def step():
            kc, vc = kv["k_cache"], kv["v_cache"]
            if S:
                r = oracle.ctx_append(w, weights, x_ctx, w.base_pos - S, kc, vc)
                kc = torch.from_numpy(r["k_cache"].view(np.int16)).view(torch.bfloat16)
                vc = torch.from_numpy(r["v_cache"].view(np.int16)).view(torch.bfloat16)
            oracle.verify_block(w, weights, x, w.base_pos, kc, vc)
        metric, unit, what = VERIFY_METRIC, "blocks/s", "verify blocks"
        config = {"workload": w.name, "tokens": w.verify_len, "prior": w.base_pos}
    else:
        pos = wl.make_positions(w)

        def step():
            oracle.decode_step(w, weights, x, pos, kv["k_cache"], kv["v_cache"])
        metric, unit, what = METRIC, UNIT, "decode steps"
        config = {"workload": w.name, "batch": w.batch, "hidden": w.hidden,
                  "heads": f"{w.num_heads}/{w.num_kv_heads}", "head_dim": w.head_dim,
                  "context": int(pos.max()) + 1, "weights": "q8_0"}
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{args.steps} full oracle {what} of {w.name}",
                             **cpu_info()},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def timed_graph(stream, steps_fn, K):
    """A CUDA graph of K steps whose first and last nodes record timing events (events made
    with external=True become record nodes of the graph, replayed with it)."""
    ev0 = torch.cuda.Event(enable_timing=True, external=True)
    ev1 = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ev0.record(stream)
        steps_fn()
        ev1.record(stream)
    torch.cuda.synchronize()
    return g, ev0, ev1


def time_replays(graph, ev0, ev1, stream, world):
    """Replays the graph under load for ~0.5 s, then times one replay between a barrier and a
    synchronize on both sides; the sampler sees the same load.  Returns (ms, clocks)."""
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    per_replay_s = max(ev0.elapsed_time(ev1) * 1e-3, 1e-5)
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.5 / per_replay_s))):
                graph.replay()
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.2 / per_replay_s))):
                graph.replay()
        torch.cuda.synchronize()
        barrier(world)
    return max_over_ranks(ms, world), clk.summary()


def decode_workload(w, K, W, R, world, want_cpu=False):
    """Measures the decode step of workload `w`; returns the figures and the launch count."""
    from quantized_attention_layer_gb300 import hfa, workloads as wl
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    pos = wl.make_positions(w)
    kv = wl.make_kv_cache(w)
    B = len(pos)
    dev_w = hfa.weights_to_device(w, weights)
    stream = torch.cuda.Stream()
    layers, caches = [], []
    with torch.cuda.stream(stream):
        for _ in range(R):
            layers.append(hfa.Layer(hfa.desc_for(w), dev_w, stream=stream))
            caches.append((kv["k_cache"].cuda(), kv["v_cache"].cuda()))
    del dev_w
    if R >= 2:
        # replicas run one after another like the layers of a model: each step prefetches
        # the next replica's first weights into L2 during its own o_proj phase
        for r in range(R):
            layers[r].hfa_set_successor(layers[(r + 1) % R])
    xd = x.cuda()
    posd = torch.from_numpy(pos).cuda()
    out = torch.empty((B, w.hidden), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()

    def step(i):
        kc, vc = caches[i % R]
        layers[i % R].hfa_decode_step(xd, posd, pos, kc, vc, out, stream=stream)

    for i in range(max(3, W)):
        step(i)
    torch.cuda.synchronize()
    for L in layers:
        L.hfa_check_device_status(stream=stream)

    def steps():
        for i in range(K):
            step(i)

    graph, ev0, ev1 = timed_graph(stream, steps, K)
    ms, clocks = time_replays(graph, ev0, ev1, stream, world)
    ms_per_step = ms / K
    for L in layers:
        L.hfa_check_device_status(stream=stream)
    del graph

    # the kernel's own duration from its timer stamps (a separate, untimed replay)
    rows = layers[0].hfa_step_stamp_rows()
    stamps = torch.zeros((K, rows, 16), dtype=torch.int64, device="cuda")

    def stamped_steps():
        for i in range(K):
            L = layers[i % R]
            L.hfa_set_step_stamps(stamps[i])
            step(i)
            L.hfa_set_step_stamps(None)

    g2, e0, e1 = timed_graph(stream, stamped_steps, K)
    with torch.cuda.stream(stream):
        g2.replay()
        g2.replay()
    torch.cuda.synchronize()
    del g2
    s = stamps.cpu().numpy()
    spans = (s[:, :, 9].max(1) - s[:, :, 13].min(1)) / 1e3  # exit - dependency wait, us
    kernel_us = float(np.mean(spans[1:])) if K > 1 else float(spans[0])

    wbytes, kvbytes, actbytes = workload_bytes(w, pos)
    peak, peak_src = measured_peaks()
    step_bytes = wbytes + kvbytes + actbytes
    gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    res = {"ms_per_step": ms_per_step, "steps_per_s": world * 1e3 / ms_per_step,
           "step_bytes": step_bytes, "step_gbs": gbs, "frac": gbs / peak,
           "frac_of_nominal": gbs / NOMINAL_HBM_GBS, "peak": peak, "peak_source": peak_src,
           "kernel_us": kernel_us, "clocks": clocks, "launches": K, "batch": B,
           "context": int(pos.max()) + 1, "successor_prefetch": R >= 2, "replicas": R}

    # end to end: the host-buffer entry point (pinned input and output copies in every step)
    x_h = x.pin_memory()
    out_h = torch.empty((B, w.hidden), dtype=torch.bfloat16).pin_memory()
    for i in range(3):
        kc, vc = caches[i % R]
        layers[i % R].hfa_decode_step_host(x_h, pos, kc, vc, out_h, stream=stream)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(K):
        kc, vc = caches[i % R]
        layers[i % R].hfa_decode_step_host(x_h, pos, kc, vc, out_h, stream=stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    res["e2e"] = {"value": world * K / e2e_s, "unit": UNIT,
                  "h2d_bytes_per_step": B * w.hidden * 2 + B * 4, "d2h_bytes_per_step": B * w.hidden * 2}
    if want_cpu:
        res["cpu_inputs"] = (weights, x, pos, kv)
    for L in layers:
        L.hfa_check_device_status(stream=stream)
        L.hfa_set_successor(None)
    for L in layers:
        L.hfa_destroy()
    del caches
    torch.cuda.empty_cache()
    return res


def verify_workload(w, K, W, R, world):
    """The multi-token verify block (L tokens through one layer, bf16 weights): blocks/s,
    and the roofline of its QKV projection (tcgen05 GEMM).  A drafter workload (bidirectional
    block) first appends its context rows each step (K/V projections only)."""
    from quantized_attention_layer_gb300 import hfa, workloads as wl
    weights = wl.make_weights(w)
    x = wl.make_x(w)
    kv = wl.make_kv_cache(w)
    L, base = w.verify_len, w.base_pos
    S = wl.DRAFTER_CTX_ROWS if w.block_bidir else 0
    x_ctx = wl.bf16_normal((S, w.hidden), torch.Generator().manual_seed(w.seed + 5)).cuda() if S else None
    dev_w = hfa.weights_to_device(w, weights)
    stream = torch.cuda.Stream()
    layers, caches = [], []
    with torch.cuda.stream(stream):
        for _ in range(R):
            layers.append(hfa.Layer(hfa.desc_for(w), dev_w, stream=stream))
            caches.append((kv["k_cache"].cuda(), kv["v_cache"].cuda()))
    del dev_w
    xd = x.cuda()
    out = torch.empty((L, w.hidden), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()

    def step(i):
        kc, vc = caches[i % R]
        if S:
            layers[i % R].hfa_ctx_append(x_ctx, base - S, kc, vc, stream=stream)
        layers[i % R].hfa_verify_block(xd, base, kc, vc, out, stream=stream)

    for i in range(max(3, W)):
        step(i)
    torch.cuda.synchronize()

    def steps():
        for i in range(K):
            step(i)

    graph, ev0, ev1 = timed_graph(stream, steps, K)
    ms, clocks = time_replays(graph, ev0, ev1, stream, world)
    del graph
    for Lr in layers:
        Lr.hfa_check_device_status(stream=stream)
        Lr.hfa_set_kernel_timing(True)
        Lr.hfa_kernel_times()
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    kt = {}
    for Lr in layers:
        for name, (kms, cnt) in Lr.hfa_kernel_times().items():
            a = kt.setdefault(name, [0.0, 0])
            a[0] += kms
            a[1] += cnt
        Lr.hfa_set_kernel_timing(False)
    H, qr, kr = w.hidden, w.q_rows, w.kv_rows
    kv_proj = 1 if w.k_eq_v else 2  # k_eq_v layers have no V projection
    wqkv_bytes = (qr + kv_proj * kr) * H * 2
    wo_bytes = H * qr * 2
    kv_bytes = (base + L) * w.num_kv_heads * w.head_dim * 2 * 2
    step_bytes = wqkv_bytes + wo_bytes + kv_bytes + 2 * L * H * 2
    if S:  # the context rows: the K and V weight rows read again, their K/V rows written
        step_bytes += kv_proj * kr * H * 2 + S * H * 2 + S * 2 * kr * 2
    peak, src = measured_peaks()
    g = kt.get("verify_qkv_gemm", [float("nan"), 1])
    g_us = g[0] / max(g[1], 1) * 1e3
    flops = 2.0 * L * (qr + kv_proj * kr) * H
    ms_per_step = ms / K
    res = {"ms_per_step": ms_per_step, "blocks_per_s": world * 1e3 / ms_per_step,
           "step_bytes": step_bytes, "step_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
           "frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, "tokens": L, "prior": base,
           "qkv_gemm": {"avg_us": g_us, "gbs": wqkv_bytes / (g_us * 1e-6) / 1e9,
                        "frac": wqkv_bytes / (g_us * 1e-6) / 1e9 / peak,
                        "useful_tflops": flops / (g_us * 1e-6) / 1e12,
                        "traffic": ncu_traffic("k_verify.cu", f"verify_block_{w.name}.md")},
           "kernels": {k: {"avg_us": v[0] / max(v[1], 1) * 1e3, "launches": v[1],
                           "timing": "events around each host-launched kernel (no overlap)"}
                       for k, v in kt.items()},
           "clocks": clocks, "launches": (5 + (1 if w.post_norm else 0) + (2 if S else 0)) * K,
           "peak": peak,
           "peak_source": src, "context_rows": S}
    for Lr in layers:
        Lr.hfa_destroy()
    del caches
    torch.cuda.empty_cache()
    return res


def ffn_workload(f, K, W, R, world):
    """The dense FFN half (one persistent kernel per step): steps/s and its HBM roofline."""
    from quantized_attention_layer_gb300 import hfa, workloads as wl
    weights = wl.make_ffn_weights(f)
    h = wl.make_ffn_input(f).cuda()
    dev_w = hfa.ffn_weights_to_device(weights)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ffns = [hfa.Ffn(hfa.ffn_desc_for(f), dev_w, stream=stream) for _ in range(R)]
    del dev_w
    B, H, I = f.batch, f.hidden, f.intermediate
    out = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()

    def step(i):
        ffns[i % R].hfa_ffn_step(h, out, stream=stream)

    for i in range(max(3, W)):
        step(i)
    torch.cuda.synchronize()

    def steps():
        for i in range(K):
            step(i)

    graph, ev0, ev1 = timed_graph(stream, steps, K)
    ms, clocks = time_replays(graph, ev0, ev1, stream, world)
    del graph
    for F in ffns:
        F.hfa_ffn_check_status(stream=stream)
    wbytes = 3 * I * H // 32 * 34               # Q8_0 gate, up and down
    step_bytes = wbytes + 2 * B * H * 2 + 2 * H * 4 + (H if f.scalar_per_channel else 1) * 4
    peak, src = measured_peaks()
    ms_per_step = ms / K
    gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    res = {"unit": UNIT, "value": world * 1e3 / ms_per_step, "ms_per_step": ms_per_step,
           "step_bytes": step_bytes, "step_gbs": gbs, "frac": gbs / peak,
           "frac_of_nominal": gbs / NOMINAL_HBM_GBS, "peak_source": src, "batch": B,
           "shape": f"{H}->{I}->{H}", "replicas": R, "plan": ffns[0].hfa_ffn_plan_info(),
           "traffic": ncu_traffic("k_ffn.cu", f"ffn_step_{f.name}.md"), "clocks": clocks,
           "l2": f"inputs larger than L2: {R} replicas, {R * step_bytes / 1e9:.2f} GB"}
    for F in ffns:
        F.hfa_ffn_destroy()
    torch.cuda.empty_cache()
    return res


def tq_workload(spec, K, W, world, name):
    """Flash-decode over a coded KV cache (4- or 8-bit codes + f32 block norms for K and V;
    hfa_attention_decode_tq), and the bf16 attention of the same shape for comparison (head
    dims up to 256: the standalone bf16 attention has no 512 form)."""
    from quantized_attention_layer_gb300 import hfa, workloads as wl
    bits, hd, nh, nkv = spec
    B, C = 1, 32768
    w = wl.Workload(name="tq", hidden=256, num_heads=nh, num_kv_heads=nkv, head_dim=hd,
                    layer_type=wl.FULL, window=0, kv_capacity=C, ring=False, batch=B,
                    rope_theta=1e6, seed=11)
    desc = hfa.attn_desc_for(w)
    pos = np.full(B, C - 1, dtype=np.int32)
    posd = torch.from_numpy(pos).cuda()
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn((B, nh, hd), device="cuda", generator=g)
    o = torch.empty_like(q)
    fmt = hfa.TqFormat(hd, bits, wl.make_tq_signs(hd, 3))
    cb, nb = fmt.code_bytes, fmt.blocks
    step_bytes = B * nkv * C * (cb + nb * 4) * 2 + 2 * q.numel() * 4
    R = max(2, -(-300_000_000 // step_bytes))  # replicas: together larger than L2
    caches = []
    for _ in range(R):
        caches.append(tuple(
            torch.randint(0, 256, (B, nkv, C, cb), dtype=torch.uint8, device="cuda", generator=g)
            if k % 2 == 0 else torch.rand((B, nkv, C, nb), device="cuda", generator=g) + 0.5
            for k in range(4)))
    ws = torch.zeros(hfa.hfa_attention_tq_workspace_bytes(desc, B, C), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step(i):
        kc, kn, vc, vn = caches[i % R]
        fmt.hfa_attention_decode_tq(desc, q, posd, pos, kc, kn, None, vc, vn, ws, o, stream=stream)

    for i in range(max(3, W)):
        step(i)
    torch.cuda.synchronize()
    graph, ev0, ev1 = timed_graph(stream, lambda: [step(i) for i in range(K)], K)
    ms, clocks = time_replays(graph, ev0, ev1, stream, world)
    del graph, caches
    fmt.destroy()
    peak, src = measured_peaks()
    ms_per_step = ms / K
    gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    out = {"unit": "attention calls/s", "value": world * 1e3 / ms_per_step,
           "ms_per_step": ms_per_step, "step_bytes": step_bytes, "step_gbs": gbs,
           "frac": gbs / peak, "peak_source": src, "bits": bits,
           "shape": f"batch {B}, {nh}/{nkv} heads, hd {hd}, {C} keys", "replicas": R,
           "clocks": clocks, "traffic": ncu_traffic("k_tq_mma.cu", f"tq_attention_{name}.md"),
           "dense_bf16": None}
    if hd > 256:
        torch.cuda.empty_cache()
        return out
    # the same attention over a dense bf16 cache
    dense_bytes = B * nkv * C * hd * 2 * 2 + 2 * q.numel() * 4
    Rd = max(2, -(-300_000_000 // dense_bytes))
    kvs = [(torch.randn((B, nkv, C, hd), device="cuda", generator=g).to(torch.bfloat16),
            torch.randn((B, nkv, C, hd), device="cuda", generator=g).to(torch.bfloat16)) for _ in range(Rd)]
    wsd = torch.zeros(hfa.hfa_attention_workspace_bytes(desc, B), dtype=torch.uint8, device="cuda")

    def dstep(i):
        kc, vc = kvs[i % Rd]
        hfa.hfa_attention_decode(desc, q, posd, pos, kc, vc, wsd, o, stream=stream)

    for i in range(3):
        dstep(i)
    torch.cuda.synchronize()
    graph, ev0, ev1 = timed_graph(stream, lambda: [dstep(i) for i in range(K)], K)
    dms, _ = time_replays(graph, ev0, ev1, stream, world)
    del graph, kvs
    torch.cuda.empty_cache()
    dgbs = dense_bytes / (dms / K * 1e-3) / 1e9
    out["dense_bf16"] = {"ms_per_step": dms / K, "step_bytes": dense_bytes, "step_gbs": dgbs,
                         "frac": dgbs / peak}
    return out


def run_ours(args, rank, world, local):
    from quantized_attention_layer_gb300 import build, workloads as wl
    build.build()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    w = wl.BY_NAME[args.workload]
    K, W = args.steps, max(3, args.warmup)
    if w.verify_len:
        r = verify_workload(w, K, W, max(1, args.replicas), world)
        line = {"metric": VERIFY_METRIC, "value": r["blocks_per_s"],
                "unit": "blocks/s", "n_gpus": world, "steps": K, "warmup": W,
                "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": w.name, "tokens": w.verify_len, "prior": w.base_pos},
                **{k: v for k, v in r.items() if k not in ("ms_per_step", "blocks_per_s")}}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return

    R = max(1, args.replicas)
    main = decode_workload(w, K, W, R, world, want_cpu=rank == 0 and not args.no_cpu_baseline)
    cpu_inputs = main.pop("cpu_inputs", None)
    roofline = {"bound": "hbm", "achieved": main["step_gbs"], "peak": main["peak"], "unit": "GB/s",
                "frac": main["frac"], "frac_of_nominal_8tbs": main["frac_of_nominal"],
                "traffic": ncu_traffic("k_step.cuh", f"decode_step_{w.name}.md"),
                "kernel": "decode_step", "algorithmic_bytes_per_launch": main["step_bytes"],
                "peak_source": main["peak_source"],
                "duration": "CUDA events around the K steps on the device (first and last graph "
                            "nodes) / K launches"}
    line = {"metric": METRIC, "value": main["steps_per_s"], "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "batch": main["batch"], "hidden": w.hidden,
                       "heads": f"{w.num_heads}/{w.num_kv_heads}", "head_dim": w.head_dim,
                       "context": main["context"], "weights": "q8_0", "kv": "bf16",
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {R} layer replicas rotated, "
                             f"{R * main['step_bytes'] / 1e9:.2f} GB"},
            "timing": "one CUDA graph of the K steps, timing events recorded by its first and "
                      "last nodes; kernel duration from the kernel's own timer stamps",
            "successor_prefetch": main["successor_prefetch"],
            "step_gbs": main["step_gbs"], "step_frac_of_peak": main["frac"],
            "step_bytes": main["step_bytes"], "roofline": roofline,
            "kernels": {"decode_step": {"avg_us": main["kernel_us"], "launches": K,
                                        "source": "device timer stamps: last CTA end - "
                                                  "dependency wait, mean over the K steps"}},
            "e2e": main["e2e"], "clocks": main["clocks"]}
    extra = EXTRA if args.extra == "all" else (() if args.extra == "none" else
                                               tuple(n for n in args.extra.split(",") if n))
    wls = {}
    for name in extra:
        if name == w.name:
            continue
        if name in TQ:
            wls[name] = tq_workload(TQ[name], K, W, world, name)
            continue
        if name in wl.FFN_BY_NAME:
            wls[name] = ffn_workload(wl.FFN_BY_NAME[name], K, W, 8, world)
            continue
        we = wl.BY_NAME[name]
        if we.verify_len:
            r = verify_workload(we, K, W, 2, world)
            wls[name] = {"unit": "blocks/s", "value": r["blocks_per_s"], "ms_per_step": r["ms_per_step"],
                         "step_bytes": r["step_bytes"], "frac": r["frac"], "qkv_gemm": r["qkv_gemm"],
                         "kernels": r["kernels"], "clocks": r["clocks"]}
        else:
            Re = 2 if we.batch >= 4 else R  # the 128K batch-4 layer holds 2.2 GB of K/V per replica
            r = decode_workload(we, K, W, Re, world)
            wls[name] = {"unit": UNIT, "value": r["steps_per_s"], "ms_per_step": r["ms_per_step"],
                         "step_bytes": r["step_bytes"], "frac": r["frac"], "kernel_us": r["kernel_us"],
                         "e2e": r["e2e"], "replicas": Re, "clocks": r["clocks"]}
    if wls:
        line["workloads"] = wls
    line["gpu_launches"] = K  # one decode-step kernel per timed step
    if cpu_inputs is not None:
        weights, x, pos, kv = cpu_inputs
        line["cpu_baseline"] = cpu_baseline(w, weights, x, pos, kv)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
