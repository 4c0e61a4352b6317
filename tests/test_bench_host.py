"""Host-side logic of bench.py: the oracle reference arm and the cross-rank reduction.

The multi-rank reduction (max of the elapsed time, sum of the tokens) runs here as two gloo
ranks on CPU; the GPU path uses the same function over NCCL.
"""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, tok = bench.reduce_over_ranks(torch, elapsed_ms=10.0 * (rank + 1), tokens=16.0, dist_on=True)
    q.put((rank, ms, tok))
    dist.destroy_process_group()


def test_reduce_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 20.0, 32.0), (1, 20.0, 32.0)]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_one_thread_oracle_layer_step_runs_in_a_child():
    import bench
    from speculative_kv_cache_gb300 import synth

    got = bench.oracle_one_thread(synth.WORKLOADS["tiny"], 4.0)
    assert set(got) == {"tiny"}
    assert got["tiny"]["layer_step_s"] > 0 and "one BLAS thread" in got["tiny"]["sample"]
    # a resized workload has no layer-step of its own name
    assert bench.oracle_one_thread(synth.scaled(synth.WORKLOADS["tiny"], layers=3), 4.0) is None


def test_fetch_stream_summary_charges_gaps():
    import numpy as np

    import bench

    nan = float("nan")
    # 4 layers; fetch l runs [f0, f1], select [s0, s1], attend [a0, a1] (ms)
    T = np.array([[nan, nan, nan, nan, 0.0, 0.1],
                  [0.0, 1.0, 0.0, 0.2, 0.2, 0.3],   # fetch 1
                  [1.5, 2.5, 0.3, 1.4, 1.6, 1.7],   # fetch 2 waited for select 2 (ended 1.4 > 1.0)
                  [2.6, 3.6, 1.7, 1.9, 2.5, 2.6]],  # fetch 3: select ended at 1.9 < 2.5; att(1) ended 0.3
                 dtype=np.float32)
    got = bench.fetch_stream_summary([T], fused_fetch=False)
    assert abs(got["busy_frac"] - 3.0 / 3.6) < 1e-6
    assert abs(got["gap_us_mean"] - 1e3 * (0.5 + 0.1) / 2) < 1e-3
    assert got["gated_by_select_frac"] == 0.5 and got["gated_by_buffer_frac"] == 0.0
    assert bench.fetch_stream_summary([T[:2]], fused_fetch=False) is None


def test_gather_kernel_key_is_the_fp16_fetch_kernel():
    import bench

    src = open(os.path.join(ROOT, "speculative_kv_cache_gb300", "csrc", "gather.cu")).read()
    key = bench.gather_kernel_key(src)
    body = key[key.index("__global__"):]
    assert body.startswith("__global__ void __launch_bounds__(kGatherThreads, IG_G_MIN_CTAS) k4_gather(")
    assert "k4_gather_q" not in body and body.endswith("\n}\n")
    assert "constexpr int kUnroll = IG_G_UNROLL;" in key and "#define IG_G_UNROLL 4" in key
    # the rows in flight are part of the key
    assert bench.gather_kernel_key(src.replace("#define IG_G_UNROLL 4", "#define IG_G_UNROLL 8")) != key
    # an edit outside the kernel leaves the key unchanged; one inside changes it
    assert bench.gather_kernel_key(src.replace("k4_gather_q", "k4_gather_x")) == key
    assert bench.gather_kernel_key(src.replace("kv[q] = ld_nc_v4(Kp + src);", "kv[q] = ld_nc_v4(Kp + src + 0);")) != key


@pytest.mark.parametrize("name,over", [
    ("opt-30b", dict(layers=2, heads=2, hidden=256, batch=2, prompt=96, gen=8)),
    # a pool smaller than the prompt (the Llama-2-13B 60 % pool): the oracle sees the resident rows
    ("llama-2-13b", dict(layers=2, heads=2, hidden=256, batch=2, prompt=200, gen=20)),
])
def test_cpu_baseline_runs_on_small_copies_of_the_workloads(name, over):
    import bench
    from speculative_kv_cache_gb300 import synth

    w = synth.scaled(synth.WORKLOADS[name], **over)
    assert (w.pool_cap < w.prompt) == (name == "llama-2-13b")
    secs, n = bench.oracle_on_bench_data(torch, w, w.alphas[0], "cpu", 1)
    assert n == 1 and secs > 0


def test_clock_summary_reads_the_timed_window_and_the_throttle_reasons():
    import bench

    clk = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.5, 0x0, {hw}, Not Active, Not Active, {cap}"
    clk.lines = [(1.0, row.format(sm=1000, hw="Not Active", cap="Not Active")),  # before the window
                 (2.0, row.format(sm=2070, hw="Not Active", cap="Active")),
                 (2.5, row.format(sm=2040, hw="Not Active", cap="Not Active")),
                 (3.0, row.format(sm=2070, hw="Active", cap="Not Active")),
                 (9.0, "garbled line")]
    s = clk.summary(1.5, 3.5)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown", "sw_power_cap"], "samples": 3}
    assert clk.summary(4.0, 5.0)["samples"] == 0
