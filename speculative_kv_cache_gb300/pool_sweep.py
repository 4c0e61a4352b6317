"""Memory-limit sweep of the pool's victim policies, with eviction-miss diagnostics.

InfiniGen bounds host memory with a pool of slots and a victim policy (paper-graph summary,
section 3.4, "KV Cache Pool Management Under Memory Pressure"; Table 2 compares FIFO, LRU
and the counter policy at an 80 % limit).  This module runs the decode-time selection of a
synthetic model under a capacity limit and measures what the limit costs the selection:

  * per decode step and layer >= 1, selection runs twice through the library's kernels
    (``ig_speculate`` + ``ig_select``): over the pool's resident slots (the real selection,
    whose "used" flags drive the policy) and over every token seen so far, from a partial key
    cache that keeps them all (what an unlimited pool would select);
  * ``ig_eviction_misses`` counts the tokens of the second selection that the pool no longer
    holds, and the share of the selected softmax weight (exp(s - max)) that falls on them;
  * the pool itself is the library's slot manager (``ig_pool_create_ex`` without storage:
    no rows need to move for this), stepped with ``ig_pool_step`` as the decoder steps it.

Inputs are the seeded synthetic ones of ``synth``, not trained weights: keys with planted
high-norm rows (the OPT-30B recipe) and layer inputs that drift across decode steps as they
drift across layers (cos ~ 0.93 between neighbours), so that what a head attends to persists
from step to step.  The sweep reports selection misses, not perplexity.

    python -m speculative_kv_cache_gb300.pool_sweep --limits 0.3,0.5,0.8,1.0
"""
from __future__ import annotations

import argparse
import json
import math
import time

import numpy as np
import torch

from . import ig, synth

POLICY_NAMES = {ig.IG_POOL_COUNTER: "counter", ig.IG_POOL_FIFO: "fifo", ig.IG_POOL_LRU: "lru"}


def _r8(n: int) -> int:
    return (n + 7) // 8 * 8


def sweep_workload(layers=4, batch=4, heads=8, hidden=7168, prompt=1024, gen=256) -> synth.Workload:
    """The default sweep model: OPT-30B's distributions (planted rows) at a small width."""
    return synth.scaled(synth.WORKLOADS["opt-30b"], name="pool-sweep", layers=layers, batch=batch,
                        heads=heads, hidden=hidden, prompt=prompt, gen=gen)


class _Layer:
    def __init__(self, w, l, T, LcapT, LcapS, dev):
        K, _ = synth.pool_layer(w, l, cap=T)                       # [B, H, T, d], token order
        self.K = torch.from_numpy(K).to(dev)
        self.cols = torch.from_numpy(synth.skewed_columns(w, l)).to(dev)
        self.Wqp = torch.from_numpy(np.ascontiguousarray(synth.skewed_partial_weight(w, l).T)).to(dev)
        ci = self.cols.long()
        part = torch.stack([self.K[:, h][..., ci[h]] for h in range(w.heads)], dim=1)  # [B,H,T,k]
        self.Kpart_tok = torch.zeros((w.batch, w.heads, w.k, LcapT), dtype=torch.float16, device=dev)
        self.Kpart_tok[..., :T].copy_(part.transpose(-1, -2))
        self.Kpart_slot = torch.zeros((w.batch, w.heads, w.k, LcapS), dtype=torch.float16, device=dev)


def run(w: synth.Workload, limit: float, policy: int, alpha: float = 4.0, steps: int | None = None,
        device: str = "cuda:0", record: bool = False) -> dict:
    """Decode ``steps`` tokens of ``w`` with a pool of round(limit * (prompt + steps)) slots.

    Returns totals over steps, layers >= 1, sequences and heads: tokens selected by the
    unlimited selection, eviction misses, miss rate, mean miss mass, evictions; with
    ``record``, also each step's used flags and placed slots (for tests).
    """
    dev = torch.device(device)
    steps = w.gen if steps is None else steps
    B, H, d, k, D = w.batch, w.heads, w.head_dim, w.k, w.hidden
    T = w.prompt + steps
    cap = max(1, int(math.floor(limit * T + 0.5)))
    cap = min(cap, T)
    LcapT, LcapS = _r8(T), _r8(cap)
    scale = 1.0 / math.sqrt(d)
    L = w.layers
    lay = [None] + [_Layer(w, l, T, LcapT, LcapS, dev) for l in range(1, L)]
    pool = ig.ig_pool_create_ex(L, B, 0, 0, cap, policy, ig.IG_POOL_NO_STORAGE)
    try:
        # prefill: the prompt's partial keys at the slots the manager gives them
        slots_pf = np.zeros(max(w.prompt, 1), np.int32)
        ig.ig_pool_prefill(pool, w.prompt, slots_pf)
        tok = np.zeros(cap, np.int32)
        ig.ig_pool_slot_tokens(pool, 0, 0, tok)  # the same for every (layer, sequence)
        live = np.nonzero(tok >= 0)[0]
        for l in range(1, L):
            lay[l].Kpart_slot[..., torch.from_numpy(live).to(dev)] = \
                lay[l].Kpart_tok[..., torch.from_numpy(tok[live]).long().to(dev)]
        f32, i32, u8 = torch.float32, torch.int32, torch.uint8
        sc_s = torch.empty((B, H, LcapS), dtype=f32, device=dev)
        idx_s = torch.empty((B, H, LcapS), dtype=i32, device=dev)
        cnt_s = torch.empty((B, H), dtype=i32, device=dev)
        sc_t = torch.empty((B, H, LcapT), dtype=f32, device=dev)
        idx_t = torch.empty((B, H, LcapT), dtype=i32, device=dev)
        cnt_t = torch.empty((L, B, H), dtype=i32, device=dev)
        miss_n = torch.empty((L, B, H), dtype=i32, device=dev)
        miss_m = torch.empty((L, B, H), dtype=f32, device=dev)
        used = torch.zeros((L, B, LcapS), dtype=u8, device=dev)
        resident = torch.zeros((L, B, LcapT), dtype=u8, device=dev)
        ws = torch.empty(max(ig.ig_speculate_workspace_bytes(B, D, H, k), 256), dtype=u8, device=dev)
        sws = torch.empty(max(ig.ig_select_workspace_bytes(B, H), 256), dtype=u8, device=dev)
        Lv_s = torch.empty(B, dtype=i32, device=dev)
        Lv_t = torch.empty(B, dtype=i32, device=dev)
        slot_dev = torch.empty(B, dtype=i32, device=dev)
        st = torch.cuda.current_stream(dev)
        used_host = np.zeros((L, B, LcapS), np.uint8)
        res_host = np.zeros((L, B, LcapT), np.uint8)
        totals = dict(selected=0, misses=0, mass_sum=0.0, mass_n=0)
        hist = []
        prev_used = None
        xs = torch.from_numpy(synth.layer_inputs_over_steps(w, steps)).to(dev)
        for s in range(steps):
            n_tok = w.prompt + s
            filled = min(n_tok, cap)
            # residency while step s runs: the pool before this step's token is placed
            res_host[:] = 0
            for l in range(1, L):
                for b in range(B):
                    ig.ig_pool_slot_tokens(pool, l, b, tok)
                    res_host[l, b, tok[tok >= 0]] = 1
            resident.copy_(torch.from_numpy(res_host))
            Lv_s.fill_(filled)
            Lv_t.fill_(n_tok)
            x = xs[s]
            for l in range(1, L):
                ig.ig_speculate(st, B, D, H, k, LcapS, x[l - 1], lay[l].Wqp, lay[l].Kpart_slot, Lv_s, scale, sc_s,
                                None, ws, ws.numel())
                ig.ig_select(st, B, H, LcapS, sc_s, Lv_s, alpha, ig.IG_SEL_THRESHOLD, 1.0, idx_s, cnt_s, used[l],
                             sws, sws.numel())
                ig.ig_speculate(st, B, D, H, k, LcapT, x[l - 1], lay[l].Wqp, lay[l].Kpart_tok, Lv_t, scale, sc_t,
                                None, ws, ws.numel())
                ig.ig_select(st, B, H, LcapT, sc_t, Lv_t, alpha, ig.IG_SEL_THRESHOLD, 1.0, idx_t, cnt_t[l], None,
                             sws, sws.numel())
                ig.ig_eviction_misses(st, B, H, LcapT, sc_t, idx_t, cnt_t[l], resident[l], miss_n[l], miss_m[l])
            used_host[:] = used.cpu().numpy()
            ig.ig_check(st)
            c = cnt_t[1:].cpu().numpy()
            n = miss_n[1:].cpu().numpy()
            m = miss_m[1:].cpu().numpy()
            totals["selected"] += int(c.sum())
            totals["misses"] += int(n.sum())
            totals["mass_sum"] += float(m[c > 0].sum())
            totals["mass_n"] += int((c > 0).sum())
            # place this step's token (folding the previous step's use first) and append its
            # partial key at the end of the step, as the decoder does
            slots = np.zeros((L, B), np.int32)
            ig.ig_pool_step(pool, prev_used, LcapS, slots)
            for l in range(1, L):
                slot_dev.copy_(torch.from_numpy(slots[l]))
                k_new = lay[l].K[:, :, n_tok].contiguous()
                ig.ig_append_kv(st, None, l, B, H, d, k, LcapS, slot_dev, lay[l].cols, k_new, k_new,
                                lay[l].Kpart_slot)
            if record:
                hist.append(dict(used=prev_used.copy() if prev_used is not None else None, slots=slots.copy()))
            prev_used = used_host.copy()
        ev = sum(ig.ig_pool_evictions(pool, l, b) for l in range(1, L) for b in range(B))
        torch.cuda.synchronize(dev)
        ig.ig_check(st)
    finally:
        ig.ig_pool_destroy(pool)
    out = dict(policy=POLICY_NAMES[policy], limit=limit, cap=cap, tokens=T, steps=steps,
               selected=totals["selected"], misses=totals["misses"],
               miss_rate=totals["misses"] / max(1, totals["selected"]),
               miss_mass=totals["mass_sum"] / max(1, totals["mass_n"]), evictions=int(ev))
    if record:
        out["history"] = hist
    return out


def time_pool_step(policy: int, layers: int, B: int, cap: int, steps: int = 20, use_prob: float = 0.1) -> float:
    """Host microseconds per ig_pool_step (fold one step's use and place one token in every
    (layer, sequence) pool) on a full pool of ``cap`` slots."""
    pool = ig.ig_pool_create_ex(layers, B, 0, 0, cap, policy, ig.IG_POOL_NO_STORAGE)
    try:
        ig.ig_pool_prefill(pool, cap)
        g = np.random.default_rng(0)
        used = [(g.random((layers, B, cap)) < use_prob).astype(np.uint8) for _ in range(4)]
        slots = np.zeros((layers, B), np.int32)
        t0 = time.perf_counter()
        for i in range(steps):
            ig.ig_pool_step(pool, used[i % 4], cap, slots)
        return (time.perf_counter() - t0) / steps * 1e6
    finally:
        ig.ig_pool_destroy(pool)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--limits", default="0.3,0.5,0.7,0.8,0.9,1.0")
    p.add_argument("--policies", default="fifo,lru,counter")
    p.add_argument("--alpha", type=float, default=4.0)
    p.add_argument("--layers", type=int, default=4)
    p.add_argument("--batch", type=int, default=4)
    p.add_argument("--heads", type=int, default=8)
    p.add_argument("--hidden", type=int, default=7168)
    p.add_argument("--prompt", type=int, default=1024)
    p.add_argument("--gen", type=int, default=256)
    a = p.parse_args(argv)
    w = sweep_workload(a.layers, a.batch, a.heads, a.hidden, a.prompt, a.gen)
    names = {v: k for k, v in POLICY_NAMES.items()}
    for pol in a.policies.split(","):
        for lim in (float(x) for x in a.limits.split(",")):
            r = run(w, lim, names[pol], alpha=a.alpha)
            print(json.dumps(r), flush=True)
    # host cost of the policy (Llama-2-13B pool shape: 40 layers, B8, 2458 slots)
    for pol in a.policies.split(","):
        print(json.dumps({"policy": pol, "pool_step_us": time_pool_step(names[pol], 40, 8, 2458)}), flush=True)


if __name__ == "__main__":
    main()
