"""The benchmarked decode step at each workload's full size, every layer, against the oracle.

The decoder runs exactly as the benchmark runs it (CUDA-graph replay, fused score + select, the
fetch staged in HBM on a side stream, the fp16 pool in pinned host memory, stage timing on; and
the benchmark's INT4 variant: INT4 codes in the pool, fetch and attention fused), over the benchmark's own seeded inputs, for every generated token of
the workload (128 steps, appends and, for the capped Llama-2-13B pool, evictions included).
At the first and the last step the oracle replays every layer for the first and the last
sequence, all heads, from the same input bytes and its own copy of the pool (the seeded rows
plus the tokens appended at the slots its own counter pool chose): speculation, threshold
selection and attention, each as the InfiniGen summary's section 3.4 "Decoding Stage" states
it (Steps 1-5), plus the dense layer 0 (HBM-resident, fp16 either way); with the INT4 pool the
attention's rows are the oracle's own INT4 quantization of its pool rows, dequantized.  The decoder keeps every layer's index list
(``keep_indices``; the kernels and grids are those of the benchmark).

Tolerances (the stated ones): index sets equal except tokens whose oracle score lies within
1e-3 of the threshold; attention outputs within 2e-3 absolute.  Where a head's sets are equal
the GPU output is compared with the oracle's attention over the oracle's own set; where they
differ by exempt tokens, with the oracle's attention over the GPU's set.

The oracle's pool model is driven by the GPU's per-step use flags (the use flags themselves are
compared with the oracle's selection at the two checked steps); every placement the runtime
makes for the sampled sequences must equal the oracle pool's.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from speculative_kv_cache_gb300 import synth  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"
CASES = [("opt-30b", 4.0, "fp16"), ("opt-6.7b", 4.0, "fp16"), ("llama-2-7b", 2.0, "fp16"),
         ("llama-2-7b", 4.0, "fp16"), ("llama-2-7b", 6.0, "fp16"), ("llama-2-13b", 4.0, "fp16"),
         # the benchmark's INT4 variant: INT4 codes in the pool, fetch and attention fused
         ("opt-30b", 4.0, "int4")]


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import decoder, ig

    return ig, decoder


def _bench_decoder(decoder, w, alpha, pool):
    """The decoder with the benchmark's default options (for an INT4 pool: the fused fetch)."""
    int4 = pool == "int4"
    return decoder.Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=w.k,
                           Lcap=w.lcap, pool_cap=w.pool_cap, alpha=alpha, rope_theta=w.rope_theta,
                           gather_ctas=0, stage_timing=True, graph=True, fused_select=True,
                           fused_fetch=int4, pool_int4=int4, keep_indices=True, device=DEV)


def _pool_rows(Kg, Vg, cnt, pool):
    """The rows the attention sees: the pool's own (fp16), or the oracle's INT4 quantization of
    them, dequantized (row by row, so quantizing the gathered rows equals quantizing the pool;
    only the first cnt[b, h] rows of each head are used, and only they are quantized)."""
    if pool == "fp16":
        return Kg, Vg
    valid = np.arange(Kg.shape[2])[None, None, :] < np.asarray(cnt)[:, :, None]
    out = []
    for X in (Kg, Vg):
        Y = X.copy()
        Y[valid] = ora.int4_dequantize_rows(*ora.int4_quantize_rows(X[valid]))
        out.append(Y)
    return out[0], out[1]


def _load(dec, w):
    for l in range(w.layers):
        t = synth.torch_layer(w, l, DEV)
        if w.rope_theta:
            A_cols = torch.stack([t["A"][h][:, t["cols"][h].long()] for h in range(w.heads)]).contiguous()
            dec.load_layer(l, t["K"], t["V"], t["cols"], Wq=t["Wq"], A_cols=A_cols)
        else:
            dec.load_layer(l, t["K"], t["V"], t["cols"], Wq_part=t["Wqp"])
        del t
    dec.prefill(w.prompt)


def _oracle_layer_state(w, l, bs, appends):
    """The oracle's copy of layer l for sequences ``bs``: the seeded pool rows with every
    appended token written at its slot, plus the layer's columns and weights (host arrays)."""
    t = synth.torch_layer(w, l, DEV)
    K = t["K"][bs].cpu().numpy()
    V = t["V"][bs].cpu().numpy()
    for slots, kn, vn in appends:  # slots [L, nb], kn / vn [L, nb, H, d]
        for j in range(len(bs)):
            K[j, :, slots[l, j]] = kn[l, j]
            V[j, :, slots[l, j]] = vn[l, j]
    host = {"K": K, "V": V, "cols": t["cols"].cpu().numpy()}
    for name in ("Wqp", "Wq", "A"):
        if name in t:
            host[name] = t[name].cpu().numpy()
    return host


def _check_step(w, alpha, dec, s, x, q, kn, vn, out, used, L_now, bs, appends, pool):
    """Every layer of step s for sequences ``bs`` against the oracle; returns (exempt, selected)."""
    scale = np.float32(1.0 / math.sqrt(w.head_dim))
    nb = len(bs)
    Lv = np.full(nb, L_now, dtype=np.int32)
    pos = np.full(nb, L_now, dtype=np.int32)  # the decoder's default position: the resident count
    x_h = x[:, bs].cpu().numpy()
    q_h, kn_h, vn_h = (a[:, bs].cpu().numpy() for a in (q, kn, vn))
    o_gpu = out[:, bs].cpu().numpy()
    idx_gpu = dec.idx[:, bs].cpu().numpy()
    cnt_gpu = dec.cnt[:, bs].cpu().numpy()
    used_gpu = used[:, bs]
    exempt = selected = 0
    # layer 0: dense attention over every resident row and the current token
    st0 = _oracle_layer_state(w, 0, bs, appends)
    o0 = ora.attend(q_h[0], st0["K"], st0["V"], np.full((nb, w.heads), L_now), scale, kn_h[0], vn_h[0])
    assert np.abs(o_gpu[0] - o0).max() <= 2e-3, f"step {s} layer 0"
    for l in range(1, w.layers):
        st = _oracle_layer_state(w, l, bs, appends)
        if w.rope_theta:
            qp = ora.partial_query_rope(x_h[l - 1], st["Wq"], st["A"], st["cols"], pos, w.rope_theta)
        else:
            qp = ora.partial_query(x_h[l - 1], st["Wqp"], w.heads, w.k)
        sc = ora.speculate(qp, ora.partial_key_cache(st["K"], st["cols"]), Lv, scale)
        want, want_cnt, want_used = ora.select(sc, Lv, alpha)
        gpu_sets = [[idx_gpu[l, j, h, :cnt_gpu[l, j, h]] for h in range(w.heads)] for j in range(nb)]
        same = np.ones((nb, w.heads), dtype=bool)
        for j in range(nb):
            thr = sc[j].max(axis=1) - alpha
            for h in range(w.heads):
                g = gpu_sets[j][h]
                assert np.all(np.diff(g) > 0) and (g.size == 0 or (g[0] >= 0 and g[-1] < L_now)), \
                    f"step {s} layer {l} ({bs[j]},{h}): indices must ascend within the resident slots"
                diff = set(g.tolist()) ^ set(want[j][h].tolist())
                for t in diff:
                    assert abs(sc[j, h, t] - thr[h]) <= 1e-3, \
                        f"step {s} layer {l} ({bs[j]},{h}) token {t}: gap {sc[j, h, t] - thr[h]}"
                exempt += len(diff)
                same[j, h] = not diff
                selected += g.size
        # attention: over the oracle's own sets where they match, over the GPU's where they differ
        Kg, Vg = _pool_rows(*ora.gather(st["K"], st["V"], want, w.lcap), want_cnt, pool)
        o_own = ora.attend(q_h[l], Kg, Vg, want_cnt, scale, kn_h[l], vn_h[l])
        err = np.abs(o_gpu[l] - o_own).max(axis=2)
        assert err[same].max(initial=0.0) <= 2e-3, f"step {s} layer {l}: output error {err[same].max()}"
        if not same.all():
            Kg, Vg = _pool_rows(*ora.gather(st["K"], st["V"], gpu_sets, w.lcap), cnt_gpu[l], pool)
            o_gs = ora.attend(q_h[l], Kg, Vg, cnt_gpu[l], scale, kn_h[l], vn_h[l])
            assert np.abs(o_gpu[l] - o_gs)[~same].max() <= 2e-3
        # the per-slot use flags the pool manager reads: the union of the heads' sets
        want_flags = np.zeros((nb, w.lcap), dtype=np.uint8)
        for j in range(nb):
            for h in range(w.heads):
                want_flags[j, gpu_sets[j][h]] = 1
        assert np.array_equal(used_gpu[l, :, :L_now], want_flags[:, :L_now])
        if same.all():
            assert np.array_equal(used_gpu[l, :, :L_now], want_used[:, :L_now])
    return exempt, selected


@pytest.mark.parametrize("name,alpha,pool", CASES,
                         ids=[f"{n}-a{a:g}" + ("" if p == "fp16" else f"-{p}") for n, a, p in CASES])
def test_benched_step_at_full_size(mods, name, alpha, pool):
    ig, decoder = mods
    w = synth.WORKLOADS[name]
    assert alpha in w.alphas
    bs = [0, w.batch - 1]
    dec = _bench_decoder(decoder, w, alpha, pool)
    try:
        _load(dec, w)
        capped = w.pool_cap < w.context
        # the oracle's pool model for the sampled sequences, after the same prompt
        opools = [[ora.CounterPool(w.pool_cap) for _ in bs] for _ in range(w.layers)]
        for l in range(w.layers):
            for p in opools[l]:
                for _ in range(w.prompt):
                    p.insert()
        appends = []
        prev_used = None
        exempt = selected = 0
        out = torch.empty((w.layers, w.batch, w.heads, w.head_dim), dtype=torch.float32, device=DEV)
        for s in range(w.gen):
            x, q, kn, vn = synth.torch_step_inputs(w, s, DEV)
            L_now = dec.step(x, q, kn, vn, out)
            slots = dec.slot_host[s % 2].numpy().copy()
            dec.finish()
            ig.ig_check(dec.S)
            assert L_now == min(w.prompt + s, w.pool_cap)
            used = dec.used_host[s % 2].numpy().copy()
            want_slots = np.zeros((w.layers, len(bs)), dtype=np.int64)
            for l in range(w.layers):
                for j, b in enumerate(bs):
                    u = prev_used[l, b] if (prev_used is not None and l > 0) else None
                    want_slots[l, j] = opools[l][j].evict(u)
            assert np.array_equal(slots[:, bs], want_slots), f"step {s}: pool placement"
            if not capped:
                assert np.all(want_slots == w.prompt + s)
            if s in (0, w.gen - 1):
                e, n = _check_step(w, alpha, dec, s, x, q, kn, vn, out, used, L_now, bs, appends, pool)
                exempt += e
                selected += n
            appends.append((want_slots, kn[:, bs].cpu().numpy(), vn[:, bs].cpu().numpy()))
            prev_used = used
        assert selected > 0 and exempt <= 1e-3 * selected
    finally:
        dec.close()
