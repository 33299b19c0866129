#!/usr/bin/env python3
"""Benchmark: one decode step of the Llama-3.1-8B GQA attention block.

Workload (default): B = 16 sequences at P = 1000 cached positions, T = 1 —
the decode point of "Llama 3.1 8B · Grouped-query attention" (1,001 keys
read, row 1000 written). A step is one call of the whole path (Q|K|V
projection with RoPE and cache append, split-K decode attention, output
projection) over the batch. Metric: seq-steps/s = B / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed steps, then exactly K steps bracketed by barrier +
synchronize, CUDA events on the launching stream. L2 (129 MB) is defeated by
rotating REPLICAS copies of weights + cache (each 150 MB) so every step
streams its bytes from HBM. Under torchrun (N > 1) every rank runs its own
replica of the step on its own GPU (no collective: batch rows are
independent); value = all ranks' sequences / max elapsed.

--impl reference times the CPU oracle (the plain fp64 definition of the
block) on rank 0: each step is one sequence of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

if "OMP_NUM_THREADS" not in os.environ:
    os.environ["OPENBLAS_NUM_THREADS"] = os.environ.get("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import gqa_inputs as I  # noqa: E402

METRIC = "GQA block decode seq-steps/s & HBM GB/s vs peak; prefill TFLOP/s vs peak"


def weight_bytes(kv_row: int = 1024) -> int:
    """Wq, Wk, Wv, Wo in bf16; kv_row = KV heads x 128 (1024, or 4096 for 32 KV heads)."""
    return (2 * 4096 + 2 * kv_row) * 4096 * 2
KERNELS = ("qkv_projection", "decode_attention", "o_projection")


def args_():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)  # ~0.25 s timed at B=16: several clock samples
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_b16_p1000")
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--graph-steps", type=int, default=0,
                    help="steps captured per CUDA graph (0: all timed steps, at most 64)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="headline only (by default its line also carries every other configuration)")
    ap.add_argument("--oracle-sample", type=float, default=None, help=argparse.SUPPRESS)  # internal: one-core leg
    ap.add_argument("--entry", choices=["block", "layer"], default="block",
                    help="block: delta = attention(x); layer: h = x + attention(RMSNorm(x)) (one more kernel)")
    ap.add_argument("--decode-kernels", choices=["fused", "three"], default="fused",
                    help="decode step as one persistent grid (default) or as three kernels")
    ap.add_argument("--attention-split", choices=["auto", "position", "head"], default="auto",
                    help="work split of the fused grid's attention (auto: chosen per call by the library)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def step_bytes(B: int, starts, kv_row: int = 1024) -> dict:
    """Algorithmic HBM bytes of one decode step, per kernel (see the design notes).
    A cache position is 2 * kv_row * 2 bytes of K and V (4,096 for 8 KV heads)."""
    pos_bytes = 4 * kv_row
    kv_read = sum((int(p) + 1) * pos_bytes for p in starts)
    wqkv = (4096 + 2 * kv_row) * 4096 * 2
    step = weight_bytes(kv_row) + kv_read + B * pos_bytes + 2 * B * 8192
    return {
        "qkv_projection": wqkv + B * 8192 + B * 8192 + B * pos_bytes,  # Wq|Wk|Wv, x, rotated q, new K/V rows
        "decode_attention": kv_read + B * 8192 + B * 8192,           # cache rows 0..P, q, o
        "o_projection": 33554432 + B * 8192 + B * 8192,              # Wo, o, delta
        "step": step,                                                # the roofline's byte count
        "decode_step": step,                                         # the fused kernel: the whole step
        "attention_norm": 2 * B * 8192 + 8192,                       # x in, normalised rows out, weight
    }


def step_flops(B: int, T: int, start: int, kv_row: int = 1024) -> dict:
    """Algorithmic FLOPs of one prefill call: projections 2*41,943,040 per
    token (8 KV heads), attention 16,384 per visible (query, key) pair (causal
    half only)."""
    pairs = B * sum(start + t + 1 for t in range(T))
    qkv = 2.0 * B * T * 4096 * (4096 + 2 * kv_row)
    return {
        "qkv_projection": qkv,
        "prefill_attention": 16384.0 * pairs,
        "o_projection": 2.0 * B * T * 4096 * 4096,
        "step": qkv + 2.0 * B * T * 4096 * 4096 + 16384.0 * pairs,
        "attention_norm": 3.0 * B * T * 4096,
    }


def load_peaks():
    """(hbm GB/s, bf16 TFLOP/s burst, kind)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_traffic(name: str, workload: str):
    """dram bytes per launch of kernel `name` at `workload` from the committed
    ncu summary, if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(f"{name}@{workload}")
    if not ent:
        return None
    srcs = ent["source"] if isinstance(ent["source"], list) else [ent["source"]]
    h = hashlib.sha256()
    for f in srcs:
        path = os.path.join(ROOT, "grouped_query_attention_gemv_gb300", "csrc", f)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return ent["bytes_per_launch"] if h.hexdigest()[:16] == ent.get("source_sha256_16") else None


class ClockSampler:
    """nvidia-smi samples (every 50 ms) while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        self.idx = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _stats(rows):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return (statistics.median(sm) if sm else None, max(smax) if smax else None, sorted(reasons))

    def summary(self, soak_replays=None):
        """sm_mhz and reasons from the samples inside the timed region, else
        (a region shorter than the sampling period) from the soak that replays
        the same graphs right after it; both sets are reported."""
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for t, r in self.rows if self.t0 and self.t1 and self.t0 <= t <= self.t1]
        soak = [r for t, r in self.rows if getattr(self, "s0", None) and self.s0 <= t <= getattr(self, "s1", 0)]
        use = inside or soak or [r for _, r in self.rows]
        sm, smax, reasons = self._stats(use)
        out = {"sm_mhz": sm, "sm_max_mhz": smax, "reasons": reasons, "samples": len(use),
               "samples_in_timed_region": len(inside),
               "source": "timed region" if inside else ("soak" if soak else "whole run")}
        if soak:
            s_sm, s_max, s_reasons = self._stats(soak)
            out["soak"] = {"sm_mhz": s_sm, "sm_max_mhz": s_max, "reasons": s_reasons, "samples": len(soak),
                           "replays": soak_replays}
        return out


def _oracle_inputs(w: I.Workload):
    """Seeded inputs of the workload for the oracle, in float64: (oracle module,
    weights, RoPE frequencies, per-sequence (x, cached K, cached V, start)).
    A workload whose cache would take over 256 MB of host memory keeps the
    caches of its first sequences only (at their own positions)."""
    from oracle import gqa as O
    gen, wt = I.draw_weights(w.dims, seed=w.seed)
    x = I.draw_x(gen, w.B, w.T)
    starts = w.start_positions().tolist()
    kv_row = w.n_kv_heads * 128
    nseq = w.B
    while nseq > 1 and nseq * w.cache_rows() * kv_row * 4 > (256 << 20):
        nseq //= 2
    ck, cv = I.draw_cache(nseq, w.cache_rows(), starts[:nseq], w.dims, seed=w.seed, device="cpu")
    W = {k: v.to(torch.float64).numpy() for k, v in wt.items()}
    r = I.LLAMA31_ROPE
    freqs = O.rope_frequencies(128, r.theta, r.scaled, r.factor, r.low_freq_factor, r.high_freq_factor,
                               r.original_context)
    per = [(x[b].to(torch.float64).numpy(), ck[b, :starts[b]].to(torch.float64).numpy(),
            cv[b, :starts[b]].to(torch.float64).numpy(), starts[b]) for b in range(nseq)]
    return O, W, freqs, per


def cpu_baseline(w: I.Workload, budget_s: float = 12.0, one_core: bool = True):
    """The oracle, as it stands, on a bounded sample: whole sequences of the
    workload (projections, attention, output) until the budget is spent. With
    ``one_core`` the same sample also runs in a child process whose BLAS is
    held to one thread (a shorter budget), reported as ``one_core_value``.
    Decode workloads report seq-steps/s, prefill workloads TFLOP/s (the
    algorithmic FLOPs of the sequences done). For a workload whose cache
    would not fit the sample's host memory budget (over 256 MB) the sample
    draws the cache of its first sequences only, at their own positions."""
    O, W, freqs, per = _oracle_inputs(w)
    nseq = len(per)
    kv_row = w.n_kv_heads * 128
    unit_step = _oracle_unit(w, O, W, freqs, per)
    n = 0
    t0 = time.perf_counter()
    while True:
        unit_step(n)
        n += 1
        el = time.perf_counter() - t0
        if el > budget_s or n >= 64 * w.B:
            break
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    if w.T > 1:
        flops = sum(step_flops(1, w.T, per[i % nseq][3], kv_row)["step"] for i in range(n))
        out = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} sequences of {w.name} ({w.T} tokens each: projections, causal attention, output "
                         f"projection), {el:.1f} s, numpy float64"}
    else:
        what = "layer steps (one sequence through one layer" if w.layers > 1 else "decode steps (whole sequences"
        out = {"value": n / el / w.layers, "unit": "seq-steps/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} single-sequence {what}: projections, attention over P+1 keys, output projection) "
                         f"of {w.name}, {el:.1f} s, numpy float64"
                         + (f"; value = that rate / {w.layers} layers" if w.layers > 1 else "")
                         + (f"; the caches of its first {nseq} sequences" if nseq < w.B else "")}
    if one_core:
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--workload", w.name, "--oracle-sample",
                            str(budget_s / 2)], env=env, capture_output=True, text=True, timeout=300)
        if r.returncode == 0 and r.stdout.strip():
            one = json.loads(r.stdout.strip().splitlines()[-1])
            out["one_core_value"] = one["value"]
            out["one_core_sample"] = one["sample"]
        else:
            out["one_core_value"] = None
    return out


def _oracle_unit(w: I.Workload, O, W, freqs, per):
    """One oracle unit of work: a sequence through the block (or, for a
    multi-layer workload, through one layer with its norm and residual)."""
    if w.layers > 1:
        g = I.draw_norm_weight(seed=w.seed).to(torch.float64).numpy()

        def unit(i):
            xb, kb, vb, sp = per[i % len(per)]
            O.layer_sequence_forward(xb, g, I.NORM_EPS, W["wq"], W["wk"], W["wv"], W["wo"], sp, kb, vb, freqs, 32, 8)
        return unit

    def unit(i):
        xb, kb, vb, sp = per[i % len(per)]
        O.sequence_forward(xb, W["wq"], W["wk"], W["wv"], W["wo"], sp, kb, vb, freqs, 32, w.n_kv_heads)
    return unit


def run_reference(a, w: I.Workload, rank: int, world: int):
    if rank != 0:
        return
    O, W, freqs, per = _oracle_inputs(w)
    starts = w.start_positions().tolist()

    unit = _oracle_unit(w, O, W, freqs, per)

    def step(i):   # one sequence through every layer
        for _ in range(w.layers):
            unit(i)

    for i in range(a.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(a.steps):
        step(i)
    el = time.perf_counter() - t0
    if w.T > 1:   # the arm's own metric: TFLOP/s of the sequences done
        kv_row = w.n_kv_heads * 128
        val = sum(step_flops(1, w.T, per[i % len(per)][3], kv_row)["step"] for i in range(a.steps)) / el / 1e12
        unit = "TFLOP/s"
    else:
        val = a.steps / el
        unit = "seq-steps/s"
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * el / a.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, a, starts), "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                                             "d2h_bytes_per_step": 0},
        "cpu_baseline": {"value": val, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"each step: one sequence of {w.name} through the CPU oracle "
                                   f"(numpy float64, whole sequence, {w.layers} layer(s))"},
    }))


def config_dict(w: I.Workload, a, starts, replicas=None):
    replicas = a.replicas if replicas is None else replicas
    c = {"workload": w.name, "B": w.B, "T": w.T, "s_max": w.cache_rows(), "d_model": 4096, "n_heads": 32,
         "n_kv_heads": w.n_kv_heads, "head_dim": 128,
         "l2": (f"inputs larger than L2: {replicas} rotating replicas of weights+cache+x, one per step"
                if replicas > 1 else "inputs larger than L2: the KV cache alone is several GB"),
         "parallelism": "replicas"}
    if w.layers > 1:
        c["layers"] = w.layers
        c["entry"] = "layer"
        c["l2"] = (f"inputs larger than L2: {w.layers} layers, each with its own weights and cache, "
                   "streamed back to back within a step")
    if w.T == 1:
        c["decode_kernels"] = a.decode_kernels
        if a.decode_kernels == "fused":
            c["attention_split"] = getattr(a, "attention_split", "auto")
    if getattr(a, "entry", "block") != "block":
        c["entry"] = a.entry
    if w.start_pos is not None:
        c["start_pos"] = w.start_pos
    else:
        c["start_pos_range"] = list(w.p_range)
        c["sum_keys"] = int(sum(int(p) + 1 for p in starts))
    return c


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world, dev):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# The other configurations of the benchmark, measured in the same run and
# attached to the headline line under "workloads": (name, step cap, replicas
# of weights + cache rotated between steps; one where the cache alone is far
# above L2)
SECONDARY = (("decode_b1_p15", 2000, 4), ("batched_decode_b64_p512_32768", 50, 1),
             ("long_decode_b8_p131071", 50, 1), ("prefill_b1_t2048", 200, 4), ("prefill_b4_t2048", 100, 2))
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, nominal
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 tensor, nominal
SOAK_S = 0.5                  # clock samples taken over graph replays after each timed region
GRAPH_STEPS_MAX = 64          # steps per captured graph by default
BACKLOG_CYCLES = 2_000_000    # ~1 ms device sleep before the start event


def measure(a, G, w, rank, world, local, dev, steps, warmup, replicas, full, shared_weights=None):
    """Time one workload: `steps` steps replayed from CUDA graphs (device
    time), a clock soak, per-kernel attribution and, with `full`, the
    end-to-end timings with host buffers. Returns the fields of its line."""
    decode = w.T == 1
    starts = w.start_positions().tolist()
    s_max = w.cache_rows()
    if shared_weights is not None:
        gen = torch.Generator().manual_seed(0)
        gen.set_state(shared_weights[1])
        wt_dev = shared_weights[0]
    else:
        gen, wt = I.draw_weights(w.dims, seed=w.seed)
        wt_dev = {k: v.to(dev) for k, v in wt.items()}
    x0 = I.draw_x(gen, w.B, w.T)
    ck0, cv0 = I.draw_cache(w.B, s_max, starts, w.dims, seed=w.seed)
    nkv = w.n_kv_heads
    kv_row = nkv * 128
    L = w.layers
    # a multi-layer step: one replica per layer (its own weights, cache and
    # workspace), chained; the working set (L x 150 MB) is far above L2
    R = L if L > 1 else max(1, replicas)
    max_start = max(starts)
    reps = []
    for r in range(R):
        wr = wt_dev if r == 0 else {k: v.clone() for k, v in wt_dev.items()}
        reps.append({**wr, "x": x0.to(dev), "ck": ck0.to(dev), "cv": cv0.to(dev),
                     "out": torch.empty_like(x0, device=dev),
                     "ws": G.make_workspace(w.B, w.T, max_start + w.T, dev)})
    del ck0, cv0
    sp = torch.tensor(starts, dtype=torch.int32, device=dev)
    rope = G.rope_table(s_max, device=dev)

    layer = a.entry == "layer" or L > 1
    if layer and nkv != 8:
        raise SystemExit("the layer entries take the 8-KV-head block only")
    norm_w = I.draw_norm_weight(seed=w.seed).to(dev)
    norms = [norm_w.clone() for _ in range(R)] if L > 1 else None

    def in_buf(i):
        return reps[0]["x"] if L > 1 else reps[i % R]["x"]

    def out_buf(i):
        return reps[-1]["out"] if L > 1 else reps[i % R]["out"]

    def step(i):
        # stream=None: the current stream (the capture stream while a graph is recorded)
        if L > 1:
            xin = reps[0]["x"]
            for li, r in enumerate(reps):
                G.layer_decode(xin, sp, max_start, norms[li], I.NORM_EPS, r["wq"], r["wk"], r["wv"], r["wo"], rope,
                               r["ck"], r["cv"], out=r["out"], workspace=r["ws"])
                xin = r["out"]
            return
        r = reps[i % R]
        if decode and layer:
            G.layer_decode(r["x"], sp, max_start, norm_w, I.NORM_EPS, r["wq"], r["wk"], r["wv"], r["wo"], rope,
                           r["ck"], r["cv"], out=r["out"], workspace=r["ws"])
        elif decode:
            G.decode(r["x"], sp, max_start, r["wq"], r["wk"], r["wv"], r["wo"], rope, r["ck"], r["cv"],
                     out=r["out"], workspace=r["ws"], n_kv_heads=nkv)
        elif layer:
            G.layer_forward(r["x"], starts[0], norm_w, I.NORM_EPS, r["wq"], r["wk"], r["wv"], r["wo"], rope,
                            r["ck"], r["cv"], out=r["out"], workspace=r["ws"])
        elif nkv != 8:
            G.block_forward(r["x"], starts[0], r["wq"], r["wk"], r["wv"], r["wo"], rope, r["ck"], r["cv"],
                            out=r["out"], workspace=r["ws"], n_kv_heads=nkv)
        else:
            G.prefill(r["x"], starts[0], r["wq"], r["wk"], r["wv"], r["wo"], rope, r["ck"], r["cv"],
                      out=r["out"], workspace=r["ws"])

    for i in range(max(warmup, R)):
        step(i)
    torch.cuda.synchronize()
    per_step_launches = G.last_launch_count() * L
    # a layer call adds the norm kernel, except where the fused decode grid folds it in
    launches_per_call = per_step_launches // L
    norm_kernel = layer and launches_per_call not in (1, 3)
    block_launches = launches_per_call - (1 if norm_kernel else 0)
    if decode:
        kernels = ("decode_step",) if block_launches == 1 else KERNELS
    else:
        kernels = ("qkv_projection", "prefill_attention", "o_projection")
    if norm_kernel:
        kernels = ("attention_norm",) + kernels
    for r in reps:
        assert G.device_status(r["ws"]) == 0, "device status set during warm-up"

    # the timed loop replays CUDA graphs holding GS consecutive steps (replicas
    # in turn), as a serving loop replays a captured multi-step decode, so the
    # device never waits for the host; a second graph holds the K % GS rest
    GS = a.graph_steps if a.graph_steps > 0 else min(steps, GRAPH_STEPS_MAX)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                step(i)
        return g
    g_full = capture(GS)
    g_rest = capture(steps % GS) if steps % GS else None
    g_full.replay()
    if g_rest is not None:
        g_rest.replay()
    torch.cuda.synchronize()

    # ---- timed region (device)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    # a device-side backlog before the start event (outside the timed region):
    # the host submits the timed graphs while it runs, so the region holds the
    # K steps' device time and no host submission latency
    torch.cuda._sleep(BACKLOG_CYCLES)
    e0.record(stream)
    for i in range(steps // GS):
        g_full.replay()
    if g_rest is not None:
        g_rest.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    _barrier(world)
    # ---- clock soak: the same graphs replayed for SOAK_S under the sampler
    # (a short timed region can fall between two samples)
    clocks.mark("s0")
    t_end = time.time() + SOAK_S
    soak_replays = 0
    while time.time() < t_end:
        for _ in range(16):
            g_full.replay()
        soak_replays += 16
        torch.cuda.synchronize()
    clocks.mark("s1")
    time.sleep(0.1)
    clocks.stop()
    ms = _max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms / steps
    launches = per_step_launches * steps
    for r in reps:
        assert G.device_status(r["ws"]) == 0, "device status set during the timed steps"

    # ---- per-kernel attribution: events recorded by the library around each
    # kernel, with a device-side backlog so host gaps do not enter the intervals
    ksteps = min(steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(ksteps)]
    for e4 in evs:          # torch only times events it has recorded once itself
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(3e8))
    for i in range(ksteps):
        G.set_profile_events(evs[i])
        step(i)
    G.set_profile_events(None)
    torch.cuda.synchronize()
    per_kernel = {k: statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs) for j, k in enumerate(kernels)}

    e2e = None
    if full:
        e2e = _end_to_end(a, G, w, step, in_buf, out_buf, x0, reps, R, L, layer, decode, sp, max_start, rope, nkv,
                          starts, dev, world, stream, steps)
    for r in reps:
        assert G.device_status(r["ws"]) == 0, "device status set during the end-to-end steps"

    hbm, tflops, peak_kind = load_peaks()
    dom = max(per_kernel, key=per_kernel.get)
    # the dominant kernel's duration: a one-kernel step takes its time per
    # step inside the replayed graphs (no longer than the step); a step of
    # several kernels takes the median of the events around the kernel
    one_kernel = len(kernels) == 1 and L == 1
    launch_ms = ms_step if one_kernel else per_kernel[dom]
    if decode:
        work = step_bytes(w.B, starts, kv_row)
        if layer:  # the norm's x in and rows out, the residual's x in
            work["step"] += 3 * w.B * 8192 + 8192
        work["step"] *= L   # per-kernel figures stay per launch (one layer)
        value = world * w.B * steps / (ms / 1e3)
        unit = "seq-steps/s"
        achieved = work[dom] / (launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": kernel_traffic(dom, w.name), "algorithmic_bytes_per_launch": work[dom],
                "launch_ms": launch_ms, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind}: copy, read + write)",
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS}
        step_rate = {"step_hbm_gbs": work["step"] / (ms_step / 1e3) / 1e9}
        step_rate["step_hbm_frac"] = step_rate["step_hbm_gbs"] / hbm
    else:
        work = step_flops(w.B, w.T, starts[0], kv_row)
        value = world * work["step"] * steps / (ms / 1e3) / 1e12
        unit = "TFLOP/s"
        achieved = work[dom] / (launch_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": kernel_traffic(dom, w.name), "algorithmic_flops_per_launch": work[dom],
                "launch_ms": launch_ms, "peak_source": f"MEASURED_PEAKS.json bf16_tflops ({peak_kind}: cuBLAS burst)",
                "nominal_peak": NOMINAL_BF16_TFLOPS, "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS}
        step_rate = {"step_tflops": work["step"] / (ms_step / 1e3) / 1e12}
        step_rate["step_tensor_frac"] = step_rate["step_tflops"] / tflops
    roof["launch_ms_source"] = ("time per step inside the replayed graphs (one kernel per step)" if one_kernel else
                                "median of events around the kernel's graph-free launches")
    if one_kernel:
        roof["launch_ms_graph_free"] = per_kernel[dom]
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) x and cache, N(0,1/4096) weights)",
        "config": config_dict(w, a, starts, R), **step_rate, "peak_kind": peak_kind,
        "roofline": roof,
        "kernels_ms": per_kernel,
        "gpu_launches": launches,
        "timing": f"device region replays CUDA graphs of {GS} consecutive steps (the same C-ABI call captured, "
                  f"replicas in turn), submitted behind a device-side sleep that precedes the start event; "
                  f"e2e calls the Python API per step",
        "clocks": clocks.summary(soak_replays=soak_replays),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if L > 1:
        line["timing"] += f"; a step chains {L} layer calls (one replica per layer), kernels_ms is one layer's launch"
    del reps
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def _end_to_end(a, G, w, step, in_buf, out_buf, x0, reps, R, L, layer, decode, sp, max_start, rope, nkv, starts, dev,
                world, stream, steps):
    """End to end with host buffers: pinned x in, delta out, copies inside the
    timed region. Two timings: serial through the device entry (torch copy
    in, step, torch copy out, one stream) and through the host-buffer entry."""
    xh = x0.pin_memory()
    oh = torch.empty_like(x0).pin_memory()
    for i in range(min(a.warmup, 5)):
        in_buf(i).copy_(xh, non_blocking=True)
        step(i)
        oh.copy_(out_buf(i), non_blocking=True)
    _barrier(world)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(steps):
        in_buf(i).copy_(xh, non_blocking=True)
        step(i)
        oh.copy_(out_buf(i), non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    ems_serial = _max_over_ranks(f0.elapsed_time(f1), world, dev)
    ems = ems_serial
    # the host-buffer C-ABI entry (x in, result out in host memory; the
    # library uploads the next step's input on its copy stream while a step
    # runs): one call per step, every copy inside the timed region
    host_entry = L == 1 and not layer
    if host_entry:
        stage = G.make_host_stage(w.B, w.T, dev)

        def host_step(i):
            r = reps[i % R]
            if decode:
                G.decode_host(xh, sp, max_start, r["wq"], r["wk"], r["wv"], r["wo"], rope, r["ck"], r["cv"],
                              out_host=oh, stage=stage, workspace=r["ws"], n_kv_heads=nkv)
            else:
                G.block_forward_host(xh, starts[0], r["wq"], r["wk"], r["wv"], r["wo"], rope, r["ck"], r["cv"],
                                     out_host=oh, stage=stage, workspace=r["ws"], n_kv_heads=nkv)
        for i in range(min(a.warmup, 5)):
            host_step(i)
        G.host_stage_wait(stage)
        _barrier(world)
        torch.cuda.synchronize()
        f0.record(stream)
        for i in range(steps):
            host_step(i)
        G.host_stage_wait(stage)   # the last read-backs are inside the region
        f1.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
        ems = _max_over_ranks(f0.elapsed_time(f1), world, dev)
        G.release_host_stage(stage)
    if decode:
        per = world * w.B * steps
        unit = "seq-steps/s"
        e2e_value, e2e_serial = per / (ems / 1e3), per / (ems_serial / 1e3)
    else:
        flops = world * step_flops(w.B, w.T, starts[0], w.n_kv_heads * 128)["step"] * steps
        unit = "TFLOP/s"
        e2e_value, e2e_serial = flops / (ems / 1e3) / 1e12, flops / (ems_serial / 1e3) / 1e12
    return {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": x0.numel() * 2,
            "d2h_bytes_per_step": x0.numel() * 2,
            "call": ("the host-buffer C-ABI entry per step (gqa_decode_host / gqa_block_forward_host: "
                     "uploads and read-backs on the library's copy streams, overlapping the neighbouring "
                     "steps; joined by gqa_host_stage_wait before the end event)") if host_entry
                    else "torch copies and the device entry per step, one stream",
            "serial_value": e2e_serial}


def main():
    a = args_()
    rank, world, local = dist_env()
    w = I.workload(a.workload)
    if a.oracle_sample is not None:   # the one-core leg of the CPU baseline (a child of cpu_baseline)
        print(json.dumps(cpu_baseline(w, a.oracle_sample, one_core=False)))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo" if a.impl == "reference" else "nccl")
    if a.impl == "reference":
        run_reference(a, w, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import grouped_query_attention_gemv_gb300 as G
    from grouped_query_attention_gemv_gb300 import build
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.set_decode_fusion(a.decode_kernels == "fused")
    G.set_decode_attention_split(a.attention_split)

    # the seeded weights, drawn once; workloads of the same model share them
    gen, wt = I.draw_weights(w.dims, seed=w.seed)
    shared = ({k: v.to(dev) for k, v in wt.items()}, gen.get_state())
    del wt
    line = measure(a, G, w, rank, world, local, dev, a.steps, a.warmup, a.replicas, True, shared)
    headline = w.name == args_default_workload() and a.entry == "block" and a.decode_kernels == "fused" \
        and a.attention_split == "auto" and not a.no_workloads
    if headline:
        line["workloads"] = {}
        for name, cap, reps in SECONDARY:
            ws_ = I.workload(name)
            n = min(a.steps, cap)
            sub = measure(a, G, ws_, rank, world, local, dev, n, min(a.warmup, 5), reps, False,
                          shared if ws_.dims == w.dims and ws_.seed == w.seed else None)
            keep = ("value", "unit", "ms_per_step", "steps", "warmup", "roofline", "clocks", "config", "gpu_launches",
                    "kernels_ms", "step_hbm_gbs", "step_hbm_frac", "step_tflops", "step_tensor_frac")
            line["workloads"][name] = {k: sub[k] for k in keep if k in sub}
            line["workloads"][name]["step_cap"] = cap
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if not a.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def args_default_workload() -> str:
    return "decode_b16_p1000"


if __name__ == "__main__":
    main()
