"""Speculation fidelity: how well the set speculated at layer i-1 matches layer i's attention.

The study the InfiniGen paper-graph summary's critique asks for (section 3.4, "Decoding
Stage"; the skew ablation of Fig 13): for every decode step, layer i >= 1, sequence and head,

  * recall@c and weight recall (``ig_attention_recall``) of the speculated set -- selected by
    the library's ``ig_speculate`` + ``ig_select`` from the partial query and partial key
    cache -- against the layer's real logits q_i . K_t;
  * the captured dot-product fraction (``ig_captured_fraction``) of the partial columns;

each with the skew (A from ``ig_skew_weights``, the skewed columns) and without it (the
unskewed weights and keys, columns chosen by the same column score in the unskewed basis),
and with the speculation fed layer i-1's input (the method) or layer i's own input (which
isolates what the column truncation alone loses).

Synthetic model (no trained weights here): Q/K weights with a power-law singular spectrum in a
random basis shared by a head's Q and K (``synth.structured_qk_weights``), hidden states
X ~ N(0, 1), keys K = X W_K, layer inputs drifting across layers with cos ~ 0.93.

    python -m speculative_kv_cache_gb300.fidelity
"""
from __future__ import annotations

import argparse
import json
import math

import numpy as np
import torch

from . import ig, synth


def fidelity_workload(layers=4, batch=2, heads=8, hidden=4096, prompt=2048) -> synth.Workload:
    return synth.scaled(synth.WORKLOADS["llama-2-7b"], name="fidelity", layers=layers, batch=batch, heads=heads,
                        hidden=hidden, prompt=prompt, gen=0, rope_theta=0.0, alphas=(4.0,))


def _raw_columns(Wq, K, H, d, k):
    """Top-k columns per head of the column score (sum |W_Q| + sum |K|) in the unskewed basis."""
    cs = Wq.float().abs().sum(0).view(H, d) + K.float().abs().sum(dim=(0, 1)).view(H, d)
    return torch.sort(torch.topk(cs, k, dim=1).indices, dim=1).values.int().contiguous()


class _Basis:
    """One basis (skewed or not) of one layer: weights, keys and partial tensors on the GPU."""

    def __init__(self, Wq, K, cols, H, d, k, Lcap, dev):
        B, T = K.shape[0], K.shape[1]
        self.Wq = Wq                                                        # [D, H*d] fp16
        self.cols = cols                                                    # [H, k] int32
        ci = cols.long()
        idx = (torch.arange(H, device=dev)[:, None] * d + ci).reshape(-1)
        self.Wqp_t = Wq[:, idx].t().contiguous()                           # [H*k, D]
        Kh = K.view(B, T, H, d).permute(0, 2, 1, 3)                        # [B, H, T, d]
        self.K = torch.zeros((B, H, Lcap, d), dtype=torch.float16, device=dev)
        self.K[:, :, :T] = Kh
        part = torch.gather(Kh, 3, ci[None, :, None, :].expand(B, H, T, k))
        self.Kpart = torch.zeros((B, H, k, Lcap), dtype=torch.float16, device=dev)
        self.Kpart[..., :T] = part.transpose(-1, -2)


def run(w: synth.Workload, alpha: float = 4.0, steps: int = 4, decay=0.5, device: str = "cuda:0",
        energy: float | None = None) -> list:
    """Per layer >= 1: mean recall, weight recall, selected fraction and captured fraction for
    the three variants (skew / no skew, speculating from layer i-1's or layer i's input).

    ``decay``: the spectral decay of the synthetic weights, one value or one per layer.
    ``energy``: choose each layer's partial width from its skewed query's spectrum
    (``ig_skew_spectrum`` + ``ig_ratio_from_spectrum``) instead of the workload's ratio."""
    dev = torch.device(device)
    B, H, d, D, L, T = w.batch, w.heads, w.head_dim, w.hidden, w.layers, w.prompt
    decays = list(decay) if hasattr(decay, "__len__") else [decay] * L
    Lcap = (T + 7) // 8 * 8
    scale = 1.0 / math.sqrt(d)
    f32, i32, u8 = torch.float32, torch.int32, torch.uint8
    Lv = torch.full((B,), T, dtype=i32, device=dev)
    sc = torch.empty((B, H, Lcap), dtype=f32, device=dev)
    idx = torch.empty((B, H, Lcap), dtype=i32, device=dev)
    cnt = torch.empty((B, H), dtype=i32, device=dev)
    rec = torch.empty((B, H), dtype=f32, device=dev)
    wt = torch.empty((B, H), dtype=f32, device=dev)
    frac = torch.empty((B, H), dtype=f32, device=dev)
    ws = torch.empty(max(ig.ig_speculate_workspace_bytes(B, D, H, d), 256), dtype=u8, device=dev)
    sws = torch.empty(max(ig.ig_select_workspace_bytes(B, H), 256), dtype=u8, device=dev)
    st = torch.cuda.current_stream(dev)
    rows = []
    for l in range(1, L):
        Wq_np, Wk_np = synth.structured_qk_weights(w, l, decays[l])
        k = w.k
        if energy is not None:
            Xs0, _, _ = synth.skew_inputs(w, l)
            sig = np.zeros((H, d), np.float32)
            ig.ig_skew_spectrum(D, H, d, 0.0, Xs0, Xs0.shape[0], Wq_np, sig)
            k = ig.ig_ratio_from_spectrum(H, d, sig, energy)
        X = torch.from_numpy(synth.hidden_states(w, l, T)).to(dev)
        Wq, Wk = torch.from_numpy(Wq_np).to(dev), torch.from_numpy(Wk_np).to(dev)
        K = (X.float() @ Wk.float()).half()                                # [B, T, H*d] unskewed
        # the skew: A and the skewed columns from a sample forward pass and the prompt keys
        Xs, _, _ = synth.skew_inputs(w, l)
        A = np.zeros((H, d, d), np.float32)
        Wq_skew = np.zeros_like(Wq_np)
        cols_s = np.zeros((H, k), np.int32)
        Kp = K.view(B * T, H, d).cpu().numpy()
        Kp_skew = np.zeros_like(Kp)
        # ig_skew_weights forms Q_s = X_s W_Q from the sample input itself (float64)
        kk = ig.ig_skew_weights(D, H, d, k / d, 0.0, Xs, Xs.shape[0], Wq_np, Wk_np, Kp, B * T, A, Wq_skew, None,
                                Kp_skew, cols_s)
        assert kk == k
        skew = _Basis(torch.from_numpy(Wq_skew).to(dev), torch.from_numpy(Kp_skew).to(dev).view(B, T, H * d),
                      torch.from_numpy(cols_s).to(dev), H, d, k, Lcap, dev)
        raw = _Basis(Wq, K, _raw_columns(Wq, K, H, d, k), H, d, k, Lcap, dev)
        acc = {}
        for s in range(steps):
            x = torch.from_numpy(synth.layer_inputs(w, step=s)).to(dev)    # [L, B, D]
            for name, basis, xin in (("skew", skew, x[l - 1]), ("skew_same_layer", skew, x[l]),
                                     ("no_skew", raw, x[l - 1])):
                q = (x[l].float() @ basis.Wq.float()).half().view(B, H, d).contiguous()  # real query
                ig.ig_speculate(st, B, D, H, k, Lcap, xin, basis.Wqp_t, basis.Kpart, Lv, scale, sc, None, ws,
                                ws.numel())
                ig.ig_select(st, B, H, Lcap, sc, Lv, alpha, ig.IG_SEL_THRESHOLD, 1.0, idx, cnt, None, sws,
                             sws.numel())
                ig.ig_attention_recall(st, B, H, d, Lcap, scale, q, basis.K, Lv, idx, cnt, rec, wt)
                ig.ig_captured_fraction(st, B, H, d, k, Lcap, q, basis.K, Lv, basis.cols, frac)
                a = acc.setdefault(name, dict(recall=[], weight=[], selected=[], captured=[]))
                a["recall"].append(rec.cpu().numpy().copy())
                a["weight"].append(wt.cpu().numpy().copy())
                a["selected"].append(cnt.cpu().numpy() / T)
                a["captured"].append(frac.cpu().numpy().copy())
        ig.ig_check(st)
        row = dict(layer=l, k=k, decay=decays[l])
        for name, a in acc.items():
            row[name] = {m: float(np.mean(v)) for m, v in a.items()}
        rows.append(row)
    # device time of the two diagnostics on the last layer (they read every key once)
    reps = 20
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    timing = {}
    for name, fn in (("attention_recall", lambda: ig.ig_attention_recall(st, B, H, d, Lcap, scale, q, skew.K, Lv,
                                                                           idx, cnt, rec, wt)),
                     ("captured_fraction", lambda: ig.ig_captured_fraction(st, B, H, d, k, Lcap, q, skew.K, Lv,
                                                                             skew.cols, frac))):
        fn()
        t0.record(st)
        for _ in range(reps):
            fn()
        t1.record(st)
        t1.synchronize()
        us = t0.elapsed_time(t1) / reps * 1e3
        timing[name] = dict(us=us, key_gbs=B * H * T * d * 2 / (us * 1e-6) / 1e9)
    rows.append(dict(timing=timing, B=B, H=H, L=T, d=d))
    return rows


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--alpha", type=float, default=4.0)
    p.add_argument("--steps", type=int, default=4)
    p.add_argument("--decay", default="0.5", help="one value, or one per layer (comma-separated)")
    p.add_argument("--energy", type=float, default=None,
                   help="choose each layer's width from its spectrum (captured-energy target)")
    p.add_argument("--layers", type=int, default=4)
    p.add_argument("--batch", type=int, default=2)
    p.add_argument("--heads", type=int, default=8)
    p.add_argument("--hidden", type=int, default=4096)
    p.add_argument("--prompt", type=int, default=2048)
    a = p.parse_args(argv)
    w = fidelity_workload(a.layers, a.batch, a.heads, a.hidden, a.prompt)
    decay = [float(x) for x in a.decay.split(",")]
    decay = decay[0] if len(decay) == 1 else decay
    for row in run(w, a.alpha, a.steps, decay, energy=a.energy):
        print(json.dumps(row), flush=True)


if __name__ == "__main__":
    main()
