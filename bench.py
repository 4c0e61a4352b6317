"""Benchmark of the InfiniGen decode hot path on one GB300 (or N, one process per GPU).

A step is one decode step of every layer for the whole batch: layer 0 attends over its full
HBM-resident KV; each later layer is speculated from the previous layer's input, its selected
K/V rows are gathered from the pinned host pool on a side stream, and it attends over them;
every layer appends the new token.  The host-side counter pool manager runs once per step.

Workload (default): OPT-30B-shaped decode — 48 layers, 56 heads, head_dim 128, hidden 7168,
batch 16, prompt 1920 + up to 128 generated tokens, partial ratio 0.3, alpha 4, with 2 % of the
key rows planted at twice the norm so that attention is skewed; ~45 GB of fp16 KV sits in
pinned host memory.  Synthetic, seeded data (no trained weights or datasets).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_kv_cache_gb300 import synth  # noqa: E402

METRIC = "decode tokens/s"
UNIT = "tokens/s"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=4)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="opt-30b", choices=sorted(synth.WORKLOADS))
    p.add_argument("--alpha", type=float, default=None)
    p.add_argument("--gather-ctas", type=int, default=0)
    p.add_argument("--graph", type=int, default=1, help="1: replay each step from a CUDA graph")
    p.add_argument("--fused-select", type=int, default=1, help="1: fused score + select kernel (persistent, scores stay on chip)")
    p.add_argument("--policy", default="threshold", choices=["threshold", "head_avg", "normalized"],
                   help="selection policy (normalized: alpha in units of each head's score std)")
    p.add_argument("--pool-policy", default="counter", choices=["counter", "fifo", "lru"],
                   help="victim policy of a capacity-limited pool (workloads with pool_frac < 1)")
    p.add_argument("--batched-append", type=int, default=0,
                   help="1: all layers' new tokens appended in one launch after the step's fetches")
    p.add_argument("--append-on-fetch", type=int, default=0,
                   help="1: each layer's append runs on the fetch stream right after its gather")
    p.add_argument("--pool-fp8", type=int, default=0,
                   help="1: the host pool holds e4m3 codes (2d bytes per row, K then V; the row scales in HBM)")
    p.add_argument("--pool-int4", type=int, default=0,
                   help="1: the host pool holds signed 4-bit codes (d bytes per row, K then V; the row scales in HBM)")
    p.add_argument("--fused-fetch", type=int, default=-1,
                   help="1: layers 1.. attend straight from the pinned pool on the fetch stream (no staging); "
                        "0: stage the rows in HBM; -1 (default): fused for an int4 pool (measured faster there), "
                        "staged otherwise (measured equal for fp16 and fp8 pools)")
    p.add_argument("--sm-split", type=int, default=0,
                   help="N > 0: the fetch stream on N SMs of its own (green contexts), compute on the rest")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-layers", type=int, default=0, help="reference arm: layers of its oracle sample (0 = 2)")
    p.add_argument("--cpu-seqs", type=int, default=4, help="CPU baseline: sequences of the oracle's sample")
    p.add_argument("--oracle-layer-step", default=None, help=argparse.SUPPRESS)
    p.add_argument("--layers", type=int, default=0,
                   help="override the workload's layer count (small cases for profiling)")
    return p.parse_args(argv)


def workload_config(w: synth.Workload, alpha: float) -> dict:
    return {
        "workload": f"{w.name}-shaped decode: {w.layers} layers, {w.heads} heads, head_dim {w.head_dim}, "
                    f"hidden {w.hidden}, batch {w.batch}, prompt {w.prompt} + {w.gen} generated, "
                    f"partial ratio {w.ratio}, alpha {alpha}"
                    + (f", {int(w.planted_p * 100)}% planted key rows x{w.planted_gamma:g}" if w.planted_p else "")
                    + (f", RoPE theta {w.rope_theta:g}" if w.rope_theta else "")
                    + (f", pool {int(w.pool_frac * 100)}% of context" if w.pool_frac < 1 else ""),
        "layers": w.layers, "heads": w.heads, "head_dim": w.head_dim, "hidden": w.hidden,
        "batch": w.batch, "prompt": w.prompt, "gen": w.gen, "partial_k": w.k, "alpha": alpha,
        "kv_pool_gb": round(2 * w.layers * w.batch * w.heads * w.pool_cap * w.head_dim * 2 / 1e9, 2),
        "l2": "inputs larger than L2: each step reads every layer's partial-key cache "
              f"({w.layers * w.batch * w.heads * w.k * w.context * 2 / 1e9:.1f} GB in HBM) and "
              "layer 0's full KV, so no step finds the previous step's data in the 129 MB L2",
    }


# ---------------------------------------------------------------------------------------
# CPU oracle (the baseline and the reference arm)
# ---------------------------------------------------------------------------------------
def oracle_sample(w: synth.Workload, n_layers: int, alpha: float, batch: int = 1):
    """Inputs of one decode step for ``batch`` sequences and n_layers layers (same recipe)."""
    w1 = synth.scaled(w, batch=batch)
    Lcap = w1.lcap
    L = np.full(batch, min(w1.prompt, w1.pool_cap), dtype=np.int32)  # resident slots
    xs = synth.layer_inputs(w1, step=0, layers=n_layers + 1)
    layers = []
    for l in range(1, n_layers + 1):
        K, V = synth.pool_layer(w1, l, cap=Lcap)
        cols = synth.skewed_columns(w1, l)
        q, kn, vn = synth.token_inputs(w1, l, 0)
        if w1.rope_theta:  # RoPE models project with the full W_Q, rotate, then take A[:, S]
            g = np.random.default_rng(l)
            A = np.stack([np.linalg.qr(g.standard_normal((w1.head_dim, w1.head_dim)))[0] for _ in range(w1.heads)])
            W = (synth.normal_f16(synth.rng(w1.name, "Wq", l), (w1.hidden, w1.heads * w1.head_dim), w1.w_std), A)
        else:
            W = synth.skewed_partial_weight(w1, l)
        layers.append((xs[l - 1], W, K, V, cols, q, kn, vn))
    return w1, L, layers


def partial_caches(layers):
    """The partial key cache of each sampled layer (built by the prefill: not timed)."""
    from oracle import infinigen as ora

    return [ora.partial_key_cache(K, cols) for (_, _, K, _, cols, _, _, _) in layers]


def time_oracle(w1, L, layers, alpha, kparts=None) -> float:
    """The oracle's decode layer-steps over the sample: partial query, scores, selection, gather
    and attention (the partial key caches, the prefill's product, are built beforehand)."""
    from oracle import infinigen as ora

    scale = 1.0 / math.sqrt(w1.head_dim)
    kparts = kparts if kparts is not None else partial_caches(layers)
    t0 = time.perf_counter()
    for (x, W, K, V, cols, q, kn, vn), Kpart in zip(layers, kparts):
        if w1.rope_theta:
            qp = ora.partial_query_rope(x, W[0], W[1], cols, L, w1.rope_theta)
        else:
            qp = ora.partial_query(x, W, w1.heads, w1.k)
        s = ora.speculate(qp, Kpart, L, scale)
        idx, cnt, _ = ora.select(s, L, alpha)
        Kg, Vg = ora.gather(K, V, idx, K.shape[2])
        ora.attend(q, Kg, Vg, cnt, scale, kn, vn)
    return time.perf_counter() - t0


ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def oracle_layer_step_child(names, alpha) -> int:
    """(child process, BLAS pinned to one thread) one layer-step of each named workload, all its
    sequences: print {"name": seconds, ...}."""
    out = {}
    for name in names:
        w = synth.WORKLOADS[name]
        a = alpha if alpha in w.alphas else w.alphas[0]
        w1, L, layers = oracle_sample(w, 1, a, batch=w.batch)
        kp = partial_caches(layers)
        time_oracle(w1, L, layers, a, kp)  # warm
        out[name] = time_oracle(w1, L, layers, a, kp)
    print(json.dumps(out), flush=True)
    return 0


def oracle_one_thread(w: synth.Workload, alpha: float) -> dict | None:
    """One-thread oracle time of one layer-step (every sequence) of this workload and of the
    one-layer tiny workload, in a child process whose BLAS pool is held to one thread."""
    names = [w.name] + (["tiny"] if w.name != "tiny" else [])
    if w.name not in synth.WORKLOADS or synth.WORKLOADS[w.name] != w:
        return None  # a resized workload (--layers): its layer-step is the named one's
    env = dict(os.environ, **{k: "1" for k in ONE_THREAD_ENV})
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-layer-step", ",".join(names),
                            "--alpha", str(alpha)], env=env, capture_output=True, text=True, timeout=600)
        secs = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None
    return {name: {"layer_step_s": t, "sample": f"one decode layer-step of all {synth.WORKLOADS[name].batch} "
                                                f"sequences (layer 1), one BLAS thread"}
            for name, t in secs.items()}


def run_reference(args, w, alpha):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    n_layers = max(1, min(w.layers - 1, args.cpu_layers or 2))
    w1, L, layers = oracle_sample(w, n_layers, alpha)
    kp = partial_caches(layers)
    for _ in range(args.warmup):
        time_oracle(w1, L, layers, alpha, kp)
    times = [time_oracle(w1, L, layers, alpha, kp) for _ in range(args.steps)]
    total = sum(times)
    # tokens: one sequence through n_layers of the w.layers layers, per step
    tokens = args.steps * (n_layers / w.layers)
    value = tokens / total
    sample = f"1 of {w.batch} sequences x {n_layers} of {w.layers} layers per step (oracle layer-steps)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, alpha),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None
        # nvidia-smi's first query (its NVML start-up) is the costly one: let it finish before
        # the timed region opens, so that it does not land inside a timed step
        t_end = time.time() + 10.0
        while self.proc is not None and not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.05)
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start=None, t_end=None):
        """Median SM clock, its maximum and the throttle reasons seen, from the samples that arrived
        between t_start and t_end (host time; all samples when not given)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if (t_start is not None and t < t_start) or (t_end is not None and t > t_end):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def fetch_stream_summary(timelines, fused_fetch: bool) -> dict | None:
    """How busy the fetch stream was, from per-step timelines ([L, 6]: fetch, speculate+select,
    attend+append start/end in ms).  A gap before fetch l is charged to its selection when
    selection l ended after fetch l-1 did, else (staged fetch) to the gather buffer when the
    attention of layer l-2 that frees it ended after fetch l-1, else to launch latency."""
    if not timelines or timelines[0].shape[0] < 3:
        return None
    busy, span, gaps, by_sel, by_buf = 0.0, 0.0, [], 0, 0
    for T in timelines:
        L = T.shape[0]
        busy += float((T[1:, 1] - T[1:, 0]).sum())
        span += float(T[L - 1, 1] - T[1, 0])
        for l in range(2, L):
            prev_end = T[l - 1, 1]
            gaps.append(float(T[l, 0] - prev_end))
            if T[l, 3] > prev_end:
                by_sel += 1
            elif not fused_fetch and l >= 2 and T[l - 2, 5] > prev_end:
                by_buf += 1
    n = len(gaps)
    return {"busy_frac": busy / span if span > 0 else None, "gap_us_mean": 1e3 * sum(gaps) / n,
            "gated_by_select_frac": by_sel / n, "gated_by_buffer_frac": by_buf / n,
            "steps": len(timelines)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def gather_kernel_key(src: str) -> str:
    """The fp16 fetch kernel's source as the counters depend on it: the file's constants and macro
    defaults (code without comments) and the text of the k4_gather function itself, so that edits elsewhere in
    the file (the quantized fetch) do not void the counters."""
    start = src.index("k4_gather(")
    start = src.rfind("\n", 0, src.rfind("__global__", 0, start)) + 1
    end = src.index("\n}\n", start) + 3
    consts = [ln.split("//")[0].rstrip() for ln in src.splitlines()
              if ln.startswith("constexpr") or ln.startswith("#define")]
    return "\n".join(consts) + "\n" + src[start:end]


def gather_traffic_bytes():
    """DRAM bytes per launch of the fetch kernel from the committed ncu summary, or None when
    the kernel (gather_kernel_key) has changed since those counters were taken."""
    import hashlib

    prof = os.path.join(ROOT, "profiles", "k4_gather_opt30b_4layer.md")
    src = os.path.join(ROOT, "speculative_kv_cache_gb300", "csrc", "gather.cu")
    try:
        vals = dict(ln.split(":", 1) for ln in open(prof).read().splitlines() if ln.startswith("traffic_"))
        key = hashlib.sha1(gather_kernel_key(open(src).read()).encode()).hexdigest()
        if vals["traffic_kernel_sha1"].strip() != key:
            return None
        return float(vals["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def link_probes(torch, ig, device, reps: int = 5) -> dict:
    """The host link's read bandwidth three ways (GB/s, best of ``reps`` over 1 GiB each):
    a pinned host -> device copy (cudaMemcpyAsync), a zero-copy streaming read of mapped pinned
    memory, and a zero-copy gather of 256-byte rows at random positions (the fetch's pattern);
    the kernels at 1, 2 and 4 CTAs per SM.  The roofline takes the best of the three."""
    n = 1 << 30

    def best_ms(fn):
        best = 1e30
        for _ in range(reps + 1):  # the first run warms up
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    out = {}
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=device)
    out["copy"] = n / (best_ms(lambda: d.copy_(h, non_blocking=True)) * 1e-3) / 1e9
    del h
    # mapped pinned memory from the library's own pool allocator: one layer of 2^22 rows x 256 B
    rows = n // 256
    pool = ig.ig_pool_create(1, 1, 1, 128, rows)
    try:
        src, _ = ig.ig_pool_kv(pool, 0)
        sink = torch.zeros(4, dtype=torch.int32, device=device)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        idx = torch.randperm(rows, device=device, dtype=torch.int64).to(torch.int32)
        read, gather = 0.0, 0.0
        for per_sm in (1, 2, 4):
            ctas = per_sm * sms
            read = max(read, n / (best_ms(lambda: ig.ig_link_read(None, src, n, sink, ctas)) * 1e-3) / 1e9)
            gather = max(gather, n / (best_ms(lambda: ig.ig_link_gather(None, src, rows, 256, idx, rows, d, ctas))
                                      * 1e-3) / 1e9)
        ig.ig_check()
        out["zero_copy_read"] = read
        out["zero_copy_gather_256B"] = gather
    finally:
        torch.cuda.synchronize()
        ig.ig_pool_destroy(pool)
    del d
    out["best"] = max(out["copy"], out["zero_copy_read"], out["zero_copy_gather_256B"])
    out["best_of"] = max(("copy", "zero_copy_read", "zero_copy_gather_256B"), key=lambda k: out[k])
    return out


def oracle_on_bench_data(torch, w, alpha, device, n_seq: int) -> tuple[float, int]:
    """The oracle's time for one decode step (step 0) of every layer for the first ``n_seq``
    sequences of the benchmark's own inputs (drawn on the GPU, copied to the host; only the
    oracle's calls are timed): layer 0's dense attention, and for each later layer the partial
    query, the speculated scores, the selection, the gather and the attention."""
    from oracle import infinigen as ora

    scale = 1.0 / math.sqrt(w.head_dim)
    bs = list(range(n_seq))
    # resident tokens after the prompt: all of it, or the pool's capacity when the pool is
    # smaller (the decoder's positions default to the same count)
    n_res = min(w.prompt, w.pool_cap)
    L = np.full(n_seq, n_res, dtype=np.int32)
    x, q, kn, vn = (t[:, bs].cpu().numpy() for t in synth.torch_step_inputs(w, 0, device))
    total = 0.0
    for l in range(w.layers):
        t = synth.torch_layer(w, l, device)
        K, V = t["K"][bs].cpu().numpy(), t["V"][bs].cpu().numpy()
        cols = t["cols"].cpu().numpy()
        W = (t["Wq"].cpu().numpy(), t["A"].cpu().numpy()) if w.rope_theta else t["Wqp"].cpu().numpy()
        del t
        Kpart = ora.partial_key_cache(K, cols) if l else None  # built by the prefill: not timed
        t0 = time.perf_counter()
        if l == 0:
            ora.attend(q[0], K, V, np.full((n_seq, w.heads), n_res), scale, kn[0], vn[0])
        else:
            if w.rope_theta:
                qp = ora.partial_query_rope(x[l - 1], W[0], W[1], cols, L, w.rope_theta)
            else:
                qp = ora.partial_query(x[l - 1], W, w.heads, w.k)
            sc = ora.speculate(qp, Kpart, L, scale)
            idx, cnt, _ = ora.select(sc, L, alpha)
            Kg, Vg = ora.gather(K, V, idx, K.shape[2])
            ora.attend(q[l], Kg, Vg, cnt, scale, kn[l], vn[l])
        total += time.perf_counter() - t0
    return total, n_seq


def setup_decoder(torch, w, alpha, gather_ctas, device, steps_total, graph=False, fused_select=True,
                  fused_fetch=False, pool_policy=0, policy=0, pool_fp8=False, batched_append=False,
                  append_on_fetch=False, sm_split=0, pool_int4=False):
    from speculative_kv_cache_gb300.decoder import Decoder

    Lcap = w.lcap
    dec = Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=w.k, Lcap=Lcap,
                  pool_cap=w.pool_cap, alpha=alpha, rope_theta=w.rope_theta, gather_ctas=gather_ctas,
                  stage_timing=True, graph=bool(graph), fused_select=bool(fused_select),
                  fused_fetch=bool(fused_fetch), pool_policy=pool_policy, policy=policy,
                  pool_fp8=bool(pool_fp8), batched_append=bool(batched_append),
                  append_on_fetch=bool(append_on_fetch), sm_split=sm_split, pool_int4=bool(pool_int4),
                  device=device)
    for l in range(w.layers):
        t = synth.torch_layer(w, l, device)
        if w.rope_theta:
            A_cols = torch.stack([t["A"][h][:, t["cols"][h].long()] for h in range(w.heads)]).contiguous()
            dec.load_layer(l, t["K"], t["V"], t["cols"], Wq=t["Wq"], A_cols=A_cols)
        else:
            dec.load_layer(l, t["K"], t["V"], t["cols"], Wq_part=t["Wqp"])
        del t
    dec.prefill(w.prompt)
    # per-step inputs: layer inputs with cross-layer drift, queries, new keys/values
    xs, qs, kns, vns = [], [], [], []
    for s in range(steps_total):
        x, q, kn, vn = synth.torch_step_inputs(w, s, device)
        xs.append(x)
        qs.append(q)
        kns.append(kn)
        vns.append(vn)
    torch.cuda.synchronize()
    return dec, xs, qs, kns, vns


def reduce_over_ranks(torch, elapsed_ms: float, tokens: float, dist_on: bool):
    """Max of the elapsed time and sum of the tokens over all ranks (weak scaling)."""
    if not dist_on:
        return elapsed_ms, tokens
    import torch.distributed as dist

    t = torch.tensor([elapsed_ms], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    n = torch.tensor([tokens], dtype=torch.float64, device=t.device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def run_ours(args, w, alpha):
    # every warm-up, timed and end-to-end step generates one token; past the workload's 128
    # the generation simply runs longer (the context grows by the extra steps; config.gen says so)
    steps_needed = args.warmup + args.steps * (1 if args.no_e2e else 2)
    if steps_needed > w.gen:
        w = synth.scaled(w, gen=steps_needed)
    import torch

    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    device = f"cuda:{local}"
    torch.cuda.set_device(device)
    if dist_on:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device(device))

    def barrier():
        if dist_on:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()

    # CPU baseline: the oracle over every layer of one decode step of the benchmark's own data
    # for a sample of the sequences (about 10 s of NumPy float64 at the OPT-30B shape)
    # (on rank 0 of a one-GPU run only: with more ranks it would slow the others' setup)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_seq = max(1, min(w.batch, args.cpu_seqs))
        t_cpu, n_tok = oracle_on_bench_data(torch, w, alpha, device, n_seq)
        cpu = {"value": n_tok / t_cpu, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"one decode step (step 0, all {w.layers} layers) of {n_seq} of the {w.batch} "
                         f"sequences ({t_cpu:.1f} s of NumPy float64 on the host cores)"}
        one = oracle_one_thread(w, alpha)
        if one is not None:
            cpu["one_thread"] = one

    probes = link_probes(torch, ig, device)
    link = probes["best"]
    hbm_peak, hbm_src = measured_peaks()
    n_e2e = 0 if args.no_e2e else args.steps
    steps_total = args.warmup + args.steps + n_e2e
    fused_fetch = bool(args.pool_int4) if args.fused_fetch < 0 else bool(args.fused_fetch)
    pool_policy = {"counter": ig.IG_POOL_COUNTER, "fifo": ig.IG_POOL_FIFO, "lru": ig.IG_POOL_LRU}[args.pool_policy]
    policy = {"threshold": ig.IG_SEL_THRESHOLD, "head_avg": ig.IG_SEL_HEAD_AVG,
              "normalized": ig.IG_SEL_NORMALIZED}[args.policy]
    dec, xs, qs, kns, vns = setup_decoder(torch, w, alpha, args.gather_ctas, device, steps_total, args.graph,
                                          args.fused_select, fused_fetch, pool_policy, policy, args.pool_fp8,
                                          args.batched_append, args.append_on_fetch, args.sm_split,
                                          args.pool_int4)
    out = torch.empty((w.layers, w.batch, w.heads, w.head_dim), dtype=torch.float32, device=device)
    cnt_host = [torch.empty_like(dec.cnt, device="cpu").pin_memory() for _ in range(args.steps)]

    # the clock sampler starts (and takes its first, slow sample) before the warm-up, so that the
    # GPU is not left idle between the warm-up and the timed steps; only the samples that arrive
    # within the timed region are summarised
    clk = ClockSampler(local).__enter__()
    gc.collect()
    s = 0
    for _ in range(args.warmup):
        dec.step(xs[s], qs[s], kns[s], vns[s], out)
        s += 1
    dec.finish()
    ig.ig_check(dec.S)

    stage = [0.0, 0.0, 0.0, 0.0]
    stage_n = [0, 0, 0, 0]
    timelines = []
    # the host stays about one step ahead of the GPU (it reads each step's stage timeline one
    # step back), so a collector pause inside the timed region would idle the GPU: the collector
    # is held off until the timed steps are done
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # one event at the end of every step: the spread of the step times
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gc.disable()
    barrier()
    launches0 = ig.ig_launch_count()
    t_clock0 = time.time()
    t0.record(dec.S)
    for i in range(args.steps):
        dec.step(xs[s], qs[s], kns[s], vns[s], out)
        step_ev[i].record(dec.S)
        with torch.cuda.stream(dec.S):
            cnt_host[i].copy_(dec.cnt, non_blocking=True)
        if i > 0:  # the previous step's stage times, while this step is queued
            ms, n = dec.stage_ms(steps_back=1)
            for j in range(4):
                stage[j] += ms[j]
                stage_n[j] += n[j]
            timelines.append(dec.timeline(steps_back=1))
        s += 1
    t1.record(dec.S)
    t1.synchronize()
    ms, n = dec.stage_ms(steps_back=0)
    for j in range(4):
        stage[j] += ms[j]
        stage_n[j] += n[j]
    timelines.append(dec.timeline(steps_back=0))
    barrier()
    t_clock1 = time.time()
    gc.enable()
    launches = ig.ig_launch_count() - launches0
    elapsed = t0.elapsed_time(t1)
    step_ms = [t0.elapsed_time(step_ev[0])] + [step_ev[i - 1].elapsed_time(step_ev[i]) for i in range(1, args.steps)]
    dec.finish()
    ig.ig_check(dec.S)
    elapsed_max, tokens_all = reduce_over_ranks(torch, elapsed, float(w.batch * args.steps), dist_on)

    # selected counts -> algorithmic bytes
    cnts = np.stack([c.numpy() for c in cnt_host]).astype(np.int64)      # [steps, L, B, H]
    sel_rows = cnts[:, 1:].sum()                                          # layers 1.. gather
    ctx = np.array([w.prompt + args.warmup + i for i in range(args.steps)], dtype=np.float64)
    f = sel_rows / (args.steps * (w.layers - 1) * w.batch * w.heads * ctx.mean())
    # K + V bytes of a row over the link (a quantized row's codes; its scales are read from HBM)
    row_link = (2 * w.head_dim if args.pool_fp8 else w.head_dim if args.pool_int4 else 2 * w.head_dim * 2)
    G_total = sel_rows * row_link                                         # over the link
    gather_ms_per_launch = stage[0] / max(stage_n[0], 1)
    G_per_launch = G_total / max(stage_n[0], 1)
    achieved = G_per_launch / (gather_ms_per_launch * 1e-3) / 1e9
    # whole-step roofline: per layer the slower of HBM bytes at HBM peak and gathered bytes at
    # the link peak; layer 0 reads its full KV from HBM
    pk_bytes = w.batch * w.heads * w.k * ctx.mean() * 2
    # staged: the fetched rows are written to and read back from HBM once; fused: not at all
    hbm_l = pk_bytes + (0 if fused_fetch else cnts[:, 1:].sum(axis=(2, 3)).mean(axis=0) * 2 * w.head_dim * 2)
    link_l = cnts[:, 1:].sum(axis=(2, 3)).mean(axis=0) * row_link
    t_roof_s = float(np.maximum(hbm_l / (hbm_peak * 1e9), link_l / (link * 1e9)).sum())
    t_roof_s += w.batch * w.heads * ctx.mean() * w.head_dim * 2 * 2 / (hbm_peak * 1e9)
    ms_per_step = elapsed_max / args.steps
    hbm_gbs_alg = float(hbm_l.sum() + w.batch * w.heads * ctx.mean() * w.head_dim * 4) / (ms_per_step * 1e-3) / 1e9

    # end to end through host buffers (pinned): inputs up, outputs down, every step, through the
    # decoder's host-buffer call (its uploads and downloads overlap the neighbouring steps on two
    # copy streams)
    e2e = None
    if n_e2e:
        hx = [t.cpu().pin_memory() for t in xs[s:s + n_e2e]]
        hq = [t.cpu().pin_memory() for t in qs[s:s + n_e2e]]
        hk = [t.cpu().pin_memory() for t in kns[s:s + n_e2e]]
        hv = [t.cpu().pin_memory() for t in vns[s:s + n_e2e]]
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        gc.collect()
        # one untimed call sets up the copy stream and buffers and brings the GPU back from the
        # host-side preparation above
        dec.step_host(hx[0], hq[0], hk[0], hv[0], hout[0])
        dec.finish_host()
        hx, hq, hk, hv = hx[1:], hq[1:], hk[1:], hv[1:]
        n_e2e -= 1
        gc.disable()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        up, down = dec.host_streams()
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        e0.record(dec.S)
        up.wait_event(e0)
        for i in range(n_e2e):
            dec.step_host(hx[i], hq[i], hk[i], hv[i], hout[i % 2])
            e_ev[i].record(down)  # this step's output is in host memory
        e1.record(down)  # after the last step's output has come down
        e1.synchronize()
        barrier()
        gc.enable()
        dec.finish_host()
        e_each = [e0.elapsed_time(e_ev[0])] + [e_ev[i - 1].elapsed_time(e_ev[i]) for i in range(1, n_e2e)]
        e_ms, e_tok = reduce_over_ranks(torch, e0.elapsed_time(e1), float(w.batch * n_e2e), dist_on)
        bi = sum(t.numel() * t.element_size() for t in (hx[0], hq[0], hk[0], hv[0]))
        e2e = {"value": e_tok / (e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": out.numel() * out.element_size(),
               "api": "Decoder.step_host (pinned host inputs and output; transfers overlap the steps)",
               "step_ms_each": [round(x, 3) for x in e_each]}

    # the sampler runs on through the end-to-end steps (stopping nvidia-smi is not free either);
    # only the samples of the device-timed region are summarised
    t_clock2 = time.time()
    clk.__exit__(None, None, None)
    clocks = clk.summary(t_clock0, t_clock1)
    if not clocks["samples"]:  # a timed region shorter than the sampling period
        clocks = dict(clk.summary(t_clock0, t_clock2), window="the device-timed and end-to-end steps")

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_all / (elapsed_max * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16 storage, fp32 accumulate", "data": "synthetic (seeded, random-init weights)",
            "config": dict(workload_config(w, alpha), cuda_graph=bool(args.graph),
                           fused_select=bool(args.fused_select), fused_fetch=fused_fetch,
                           selection=args.policy, batched_append=bool(args.batched_append),
                           append_on_fetch=bool(args.append_on_fetch), pool_dtype=("fp8-e4m3 codes in the pinned pool, fp32 row scales in HBM" if args.pool_fp8 else
                                       "int4 codes in the pinned pool, fp32 row scales in HBM" if args.pool_int4
                                       else "fp16"),
                           pool_policy=args.pool_policy if w.pool_frac < 1 else None,
                           # the pinned pool as allocated: fp16 rows, or one record of codes per row
                           pinned_pool_gb=round(w.layers * w.batch * w.heads * w.pool_cap
                                                * (2 * w.head_dim if args.pool_fp8 else w.head_dim if args.pool_int4
                                                   else 4 * w.head_dim) / 1e9, 2),
                           sm_split=({"fetch_sms": dec.fetch_sms, "compute_sms": dec.compute_sms}
                                     if args.sm_split else None)),
            "step_ms": {"p50": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms),
                        "mean": statistics.fmean(step_ms), "each": [round(t, 3) for t in step_ms]},
            "us_per_layer_step": 1000 * ms_per_step / w.layers,
            "us_per_layer_step_p50": 1000 * statistics.median(step_ms) / w.layers,
            "selected_fraction": float(f),
            "link_gbs": G_total / args.steps / (ms_per_step * 1e-3) / 1e9,
            "hbm_alg_gbs": hbm_gbs_alg,
            "us_per_speculative_layer_step": 1000 * (ms_per_step - stage[3] / args.steps) / max(1, w.layers - 1),
            "layer0_ms_per_step": stage[3] / args.steps,
            "hbm_alg_frac": {"of_measured": hbm_gbs_alg / hbm_peak, "of_nominal_8000": hbm_gbs_alg / 8000.0},
            "fetch_stream": fetch_stream_summary(timelines, fused_fetch),
            "stage_ms_per_step": {("fetch_attend" if fused_fetch else "gather"): stage[0] / args.steps,
                                  "speculate_select": stage[1] / args.steps,
                                  ("combine_append" if fused_fetch else "attend_append"): stage[2] / args.steps},
            "e2e": e2e,
            "gpu_launches": int(launches),
            "roofline": {"kernel": ("k5_fetch_attend (fused zero-copy fetch + partial attention)" if fused_fetch
                                    else "k4_gather_q (zero-copy fetch and dequantization of the selected rows)"
                                    if (args.pool_fp8 or args.pool_int4)
                                    else "k4_gather (zero-copy fetch of the selected K/V rows)"),
                         "bound": "host-link", "achieved": achieved, "peak": link,
                         "unit": "GB/s", "frac": achieved / link,
                         "traffic": (None if (fused_fetch or args.pool_fp8 or args.pool_int4)
                                     else gather_traffic_bytes()),
                         "traffic_note": "DRAM read+write bytes per launch (ncu, same per-layer shape); "
                                         "the kernel's algorithmic bytes cross the host link, not DRAM",
                         "peak_source": f"measured in this run: best of three host-link probes "
                                        f"({probes['best_of']}; best of 5 x 1 GiB each)",
                         "algorithmic_bytes_per_launch": G_per_launch,
                         "launch_ms": gather_ms_per_launch},
            "path_roofline": {"t_roof_ms": 1000 * t_roof_s, "t_step_ms": ms_per_step,
                              "frac": 1000 * t_roof_s / ms_per_step, "hbm_peak_gbs": hbm_peak,
                              "hbm_peak_source": hbm_src, "link_peak_gbs": link},
            "link_probes_gbs": {k: v for k, v in probes.items() if k != "best"},
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if dist_on:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_layer_step:
        return oracle_layer_step_child(args.oracle_layer_step.split(","), args.alpha or 4.0)
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = synth.scaled(w, layers=args.layers)
    alpha =args.alpha if args.alpha is not None else (4.0 if 4.0 in w.alphas else w.alphas[0])
    if args.impl == "reference":
        return run_reference(args, w, alpha)
    return run_ours(args, w, alpha)


if __name__ == "__main__":
    sys.exit(main())
