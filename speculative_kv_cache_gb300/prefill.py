"""Prefill of one layer through the library (``ig_prefill_layer``), and its timing.

``prefill_decoder_layer`` fills a ``Decoder`` layer from the prompt's attention input and the
skewed weights: K~ and V on the tensor cores, the column choice, the partial weight and partial
key cache, the pool rows -- the inputs the decode step reads, built by the library itself
(InfiniGen paper-graph summary, section 3.4, "Prefill Stage", Steps 1-3; models without RoPE).

    python -m speculative_kv_cache_gb300.prefill      # times one OPT-30B-shaped layer
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import ig, synth


def prefill_decoder_layer(dec, l: int, X, Wq_t, Wk_t, Wv_t, workspace=None):
    """Prefill layer l >= 1 of ``dec`` (fp16 pool) from X [B, N, D] and W~_Q^T, W~_K^T, W_V^T
    [H*d, D] (device fp16).  Call ``dec.prefill(N)`` once after every layer is filled."""
    B, N, D = X.shape
    if workspace is None:
        workspace = torch.empty(ig.ig_prefill_workspace_bytes(B, N, dec.H, dec.d), dtype=torch.uint8,
                                device=X.device)
    dec.S.wait_stream(torch.cuda.current_stream(X.device))
    with torch.cuda.stream(dec.S):
        dec.Kpart[l].zero_()
        ig.ig_prefill_layer(dec.S, dec.pool, l, B, N, D, dec.H, dec.d, dec.ks[l], dec.Lcap, X, Wq_t, Wk_t, Wv_t,
                            dec.cols[l], dec.Wq_part[l], dec.Kpart[l], workspace, workspace.numel())
    dec.S.synchronize()
    return workspace


def prefill_decoder_layer_rope(dec, l: int, X, Wq_skew_t, Wk_t, Wv_t, A, workspace=None):
    """As :func:`prefill_decoder_layer` for a RoPE decoder: W~_Q^T (skewed, column score only),
    W_K^T and W_V^T (unskewed) [H*d, D] fp16 and the skew A [H, d, d] fp32, all on the device."""
    B, N, D = X.shape
    if workspace is None:
        workspace = torch.empty(ig.ig_prefill_workspace_bytes(B, N, dec.H, dec.d), dtype=torch.uint8,
                                device=X.device)
    dec.S.wait_stream(torch.cuda.current_stream(X.device))
    with torch.cuda.stream(dec.S):
        dec.Kpart[l].zero_()
        ig.ig_prefill_layer_rope(dec.S, dec.pool, l, B, N, D, dec.H, dec.d, dec.ks[l], dec.Lcap, dec.cfg.rope_theta,
                                 X, Wq_skew_t, Wk_t, Wv_t, A, dec.cols[l], dec.A_cols[l], dec.Kpart[l], workspace,
                                 workspace.numel())
    dec.S.synchronize()
    return workspace


def time_layer(w: synth.Workload, reps: int = 3, device: str = "cuda:0") -> dict:
    """Device time of one layer's prefill at the workload's shape, and of its parts."""
    dev = torch.device(device)
    B, N, D, H, d, k = w.batch, w.prompt, w.hidden, w.heads, w.head_dim, w.k
    Lcap = (w.pool_cap + 7) // 8 * 8
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    X = torch.randn((B, N, D), generator=g, device=dev).half()
    Wq_t, Wk_t, Wv_t = ((torch.randn((H * d, D), generator=g, device=dev) * w.w_std).half() for _ in range(3))
    pool = ig.ig_pool_create(1, B, H, d, w.pool_cap)
    try:
        cols = torch.empty((H, k), dtype=torch.int32, device=dev)
        Wqp = torch.empty((H * k, D), dtype=torch.float16, device=dev)
        Kpart = torch.zeros((B, H, k, Lcap), dtype=torch.float16, device=dev)
        ws = torch.empty(ig.ig_prefill_workspace_bytes(B, N, H, d), dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream(dev)
        M, Nn = B * N, H * d
        C = torch.empty((M, Nn), dtype=torch.float16, device=dev)
        cp = torch.empty(((M + 127) // 128, Nn), dtype=torch.float32, device=dev)

        def timed(fn):
            fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for _ in range(reps):
                fn()
            b.record(st)
            b.synchronize()
            ig.ig_check(st)
            return a.elapsed_time(b) / reps

        t_layer = timed(lambda: ig.ig_prefill_layer(st, pool, 0, B, N, D, H, d, k, Lcap, X, Wq_t, Wk_t, Wv_t, cols,
                                                    Wqp, Kpart, ws, ws.numel()))
        t_gemm = timed(lambda: ig.ig_gemm_tn(st, M, Nn, D, X, Wk_t, C, cp))
        flops = 2.0 * M * Nn * D
        pool_bytes = 2 * B * H * min(N, w.pool_cap) * d * 2
        return dict(workload=w.name, B=B, N=N, D=D, H=H, d=d, k=k, layer_ms=t_layer, gemm_ms=t_gemm,
                    gemm_tflops=flops / (t_gemm * 1e-3) / 1e12, projections_tflop=2 * flops / 1e12,
                    pool_write_bytes=pool_bytes,
                    rest_ms=t_layer - 2 * t_gemm,
                    pool_gbs_if_rest=pool_bytes / ((t_layer - 2 * t_gemm) * 1e-3) / 1e9)
    finally:
        ig.ig_pool_destroy(pool)


def time_gemm(n: int = 8192, reps: int = 5, device: str = "cuda:0") -> dict:
    """The GEMM alone on an n^3 problem (for the tensor roofline)."""
    dev = torch.device(device)
    A = torch.randn((n, n), device=dev).half()
    Bt = torch.randn((n, n), device=dev).half()
    C = torch.empty((n, n), dtype=torch.float16, device=dev)
    st = torch.cuda.current_stream(dev)
    ig.ig_gemm_tn(st, n, n, n, A, Bt, C)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        ig.ig_gemm_tn(st, n, n, n, A, Bt, C)
    b.record(st)
    b.synchronize()
    ig.ig_check(st)
    ms = a.elapsed_time(b) / reps
    return dict(n=n, ms=ms, tflops=2.0 * n ** 3 / (ms * 1e-3) / 1e12)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", default="opt-30b")
    p.add_argument("--gemm-only", action="store_true", help="time the n^3 GEMM alone")
    p.add_argument("--n", type=int, default=8192)
    a = p.parse_args(argv)
    print(json.dumps(time_gemm(a.n)), flush=True)
    if not a.gemm_only:
        print(json.dumps(time_layer(synth.WORKLOADS[a.workload])), flush=True)


if __name__ == "__main__":
    main()
