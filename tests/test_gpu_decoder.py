"""The pipelined multi-layer decode step (ig_decode_step via Decoder) against the oracle.

Several decode steps of small OPT-shaped and Llama-shaped models run through the native
runtime; the oracle replays every layer of every step on its own copy of the pool and partial
key caches.  The GPU's index sets must equal the oracle's except tokens whose oracle score lies
within 1e-3 of the threshold (the stated exemption); layer outputs must agree within 2e-3 with
the oracle's attention over the GPU's sets.  With a capped pool, the slots the runtime evicts
must be the ones the oracle's counter pool picks from the same use flags.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from speculative_kv_cache_gb300 import synth  # noqa: E402
from gpu_util import index_sets_ok  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import decoder, ig

    return ig, decoder


def _layer_data(w, l, cap, rope, ratio=None):
    if ratio is not None:  # this layer's own partial width
        w = synth.scaled(w, ratio=ratio)
    K, V = synth.pool_layer(w, l, cap=cap)
    cols = synth.skewed_columns(w, l)
    if rope:
        g = np.random.default_rng(1000 + l)
        A = np.stack([np.linalg.qr(g.standard_normal((w.head_dim, w.head_dim)))[0] for _ in range(w.heads)])
        Wq = synth.normal_f16(synth.rng(w.name, "Wq", l), (w.hidden, w.heads * w.head_dim), w.w_std)
        return dict(K=K, V=V, cols=cols, A=A.astype(np.float32), Wq=Wq)
    return dict(K=K, V=V, cols=cols, Wqp=synth.skewed_partial_weight(w, l))


def _run(mods, w, steps, rope=False, check_slots=False, fused_select=True, fused_fetch=False, graph=False,
         ratios=None, batched_append=False, append_on_fetch=False, sm_split=0):
    ig, decoder = mods
    dev = "cuda:0"
    Lcap = w.lcap
    cap = w.pool_cap
    scale = np.float32(1.0 / math.sqrt(w.head_dim))
    alpha = 4.0
    ks = [synth.scaled(w, ratio=r).k for r in ratios] if ratios else [w.k] * w.layers
    dec = decoder.Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=ks if ratios else w.k,
                          Lcap=Lcap, pool_cap=cap, alpha=alpha, rope_theta=w.rope_theta,
                          fused_select=fused_select, fused_fetch=fused_fetch, graph=graph,
                          batched_append=batched_append, append_on_fetch=append_on_fetch, sm_split=sm_split,
                          device=dev)
    try:
        data = [_layer_data(w, l, cap, rope, ratios[l] if ratios else None) for l in range(w.layers)]
        for l, dd in enumerate(data):
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
            if rope:
                A_cols = np.stack([dd["A"][h][:, dd["cols"][h]] for h in range(w.heads)])
                dec.load_layer(l, t(dd["K"]), t(dd["V"]), dd["cols"], Wq=t(dd["Wq"]), A_cols=t(A_cols))
            else:
                dec.load_layer(l, t(dd["K"]), t(dd["V"]), dd["cols"], Wq_part=t(dd["Wqp"]))
        n_prompt = w.prompt
        dec.prefill(n_prompt)
        # the oracle's own state: pool rows and partial caches per layer, counter pools
        oK = [dd["K"].copy() for dd in data]
        oV = [dd["V"].copy() for dd in data]
        opools = [[ora.CounterPool(cap) for _ in range(w.batch)] for _ in range(w.layers)]
        for l in range(w.layers):
            for b in range(w.batch):
                for _ in range(n_prompt):
                    opools[l][b].insert()
        skipped = checked = 0
        prev_used = None
        for s in range(steps):
            x = synth.layer_inputs(w, step=s)
            qkv = [synth.token_inputs(w, l, s) for l in range(w.layers)]
            q = np.stack([a[0] for a in qkv])
            kn = np.stack([a[1] for a in qkv])
            vn = np.stack([a[2] for a in qkv])
            out = torch.empty((w.layers, w.batch, w.heads, w.head_dim), dtype=torch.float32, device=dev)
            L_now = min(n_prompt + s, cap)
            # oracle placement of this step's token (fold the previous step's use first)
            want_slots = np.zeros((w.layers, w.batch), dtype=np.int32)
            for l in range(w.layers):
                for b in range(w.batch):
                    u = prev_used[l, b] if (prev_used is not None and l > 0) else None
                    want_slots[l, b] = opools[l][b].evict(u)
            pos = np.full(w.batch, n_prompt + s, dtype=np.int32)
            got_L = dec.step(*(torch.from_numpy(a).to(dev) for a in (x, q, kn, vn)), out, positions=pos)
            dec.finish()
            ig.ig_check(dec.S)
            assert got_L == L_now
            if check_slots:
                assert np.array_equal(dec.slot_host[s % 2].numpy(), want_slots)
            used = dec.used_host[s % 2].numpy().copy()
            cnt = dec.cnt.cpu().numpy()
            idx_buf = dec.idx.cpu().numpy()
            o = out.cpu().numpy()
            Lv = np.full(w.batch, L_now, dtype=np.int32)
            # layer 0: dense attention over the resident tokens plus the new one
            o0 = ora.attend(q[0], oK[0], oV[0], np.full((w.batch, w.heads), L_now), scale, kn[0], vn[0])
            assert np.abs(o[0] - o0).max() <= 2e-3
            for l in range(1, w.layers):
                dd = data[l]
                if rope:
                    qp = ora.partial_query_rope(x[l - 1], dd["Wq"], dd["A"], dd["cols"], pos, w.rope_theta)
                else:
                    qp = ora.partial_query(x[l - 1], dd["Wqp"], w.heads, ks[l])
                Kpart = ora.partial_key_cache(oK[l], dd["cols"])
                sc = ora.speculate(qp, Kpart, Lv, scale)
                # the GPU's own index sets (both gather buffers survive a step of <= 3 layers):
                # equal to the oracle's except tokens within 1e-3 of the threshold
                gi = idx_buf[l % 2]
                exempt = index_sets_ok(gi, cnt[l], sc, Lv, alpha)
                skipped += exempt
                sets = [[gi[b, h, :cnt[l, b, h]] for h in range(w.heads)] for b in range(w.batch)]
                checked += int(cnt[l].sum())
                Kg, Vg = ora.gather(oK[l], oV[l], sets, Lcap)
                ol = ora.attend(q[l], Kg, Vg, cnt[l], scale, kn[l], vn[l])
                assert np.abs(o[l] - ol).max() <= 2e-3
                want_used = np.zeros((w.batch, Lcap), dtype=np.uint8)
                for b in range(w.batch):
                    for h in range(w.heads):
                        want_used[b, sets[b][h]] = 1
                assert np.array_equal(used[l, :, :L_now], want_used[:, :L_now])
            # the oracle appends the new token at the slots the pool chose
            for l in range(w.layers):
                for b in range(w.batch):
                    sl = want_slots[l, b]
                    oK[l][b, :, sl] = kn[l, b]
                    oV[l][b, :, sl] = vn[l, b]
            prev_used = used
        assert checked > 0 and skipped <= 0.01 * checked
        # the device-side appends landed in the pinned pool and the partial caches
        for l in range(1, w.layers):
            Kp, Vp = ig.pool_layer_view(dec.pool, l, w.batch, w.heads, cap, w.head_dim)
            assert np.array_equal(Kp, oK[l]) and np.array_equal(Vp, oV[l])
            kpart = dec.Kpart[l].cpu().numpy()[..., :cap]
            assert np.array_equal(kpart, ora.partial_key_cache(oK[l], data[l]["cols"]))
    finally:
        dec.close()


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("fetch", ["staged", "fused"])
def test_decoder_opt_shaped_steps(mods, fused, fetch):
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-opt", layers=3, batch=3, heads=6, hidden=768,
                     prompt=300, gen=8)
    _run(mods, w, steps=3, fused_select=fused, fused_fetch=fetch == "fused")


@pytest.mark.parametrize("fetch", ["staged", "fused"])
@pytest.mark.parametrize("append", ["per-layer", "batched", "on-fetch"])
def test_decoder_capped_pool_evicts_like_the_oracle(mods, fetch, append):
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-cap", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=10, pool_frac=0.95)
    assert w.pool_cap < w.prompt + 10
    _run(mods, w, steps=8, check_slots=True, fused_fetch=fetch == "fused", batched_append=append == "batched",
         append_on_fetch=append == "on-fetch")


@pytest.mark.parametrize("fetch", ["staged", "fused"])
def test_decoder_rope_steps(mods, fetch):
    w = synth.scaled(synth.WORKLOADS["llama-2-7b"], name="dec-rope", layers=3, batch=2, heads=4,
                     hidden=512, prompt=260, gen=8)
    _run(mods, w, steps=2, rope=True, fused_fetch=fetch == "fused")


@pytest.mark.parametrize("rope", [False, True])
def test_decoder_per_layer_widths(mods, rope):
    """Each layer with its own partial width (the per-layer ratio), fused and plain paths."""
    base = synth.WORKLOADS["llama-2-7b"] if rope else synth.WORKLOADS["opt-30b"]
    w = synth.scaled(base, name="dec-ks", layers=4, batch=2, heads=4, hidden=512, prompt=220, gen=8)
    _run(mods, w, steps=2, rope=rope, ratios=[0.3, 0.125, 0.5, 0.25])


def test_decoder_fused_fetch_graph_replay(mods):
    """Fused fetch + attention under CUDA-graph replay, with eviction, against the oracle."""
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-ffg", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=10, pool_frac=0.95)
    _run(mods, w, steps=4, check_slots=True, fused_fetch=True, graph=True)


@pytest.mark.parametrize("fetch", ["staged", "fused"])
def test_decoder_on_an_sm_split(mods, fetch):
    """The step on two green contexts (fetch stream on 16 SMs of its own, compute on the rest),
    eager and under CUDA-graph replay, against the oracle."""
    ig, _ = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-split", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=10, pool_frac=0.95)
    _run(mods, w, steps=4, check_slots=True, fused_fetch=fetch == "fused", sm_split=16)
    _run(mods, w, steps=4, check_slots=True, fused_fetch=fetch == "fused", graph=True, sm_split=16)


def test_sm_split_sizes_and_errors(mods):
    ig, _ = mods
    n = torch.cuda.get_device_properties(0).multi_processor_count
    h, cs, fs, nc, nf = ig.ig_sm_split_create(0, 20)
    try:
        assert cs and fs and cs != fs
        assert nf >= 20 and nc >= 1 and nc + nf <= n
    finally:
        ig.ig_sm_split_destroy(h)
    with pytest.raises(ig.IGError) as e:
        ig.ig_sm_split_create(0, n)
    assert e.value.status == ig.IG_ERR_INVALID
    with pytest.raises(ig.IGError):
        ig.ig_sm_split_create(0, 0)


def test_decoder_llama13b_width_capped_pool(mods):
    """Llama-2-13B-shaped layers at full width and context (pool capped at 60 %, RoPE):
    eviction happens at every step."""
    w = synth.scaled(synth.WORKLOADS["llama-2-13b"], name="dec-13b", layers=3)
    assert w.pool_cap == 2458 and w.pool_cap < w.prompt
    _run(mods, w, steps=3, rope=True, check_slots=True)


def _check_timeline(T, L, fused_fetch, eps=2e-3):
    """The stage timeline honours the step's dependencies (ms; event resolution ~0.5 us)."""
    assert T.shape == (L, 6)
    assert np.isnan(T[0, :4]).all() and np.isfinite(T[0, 4:]).all() and np.isfinite(T[1:]).all()
    assert T[1, 2] == 0.0  # the reference point: layer 1's speculation starts the step
    for j in (0, 2, 4):
        ok = ~np.isnan(T[:, j])
        assert (T[ok, j] <= T[ok, j + 1] + eps).all()
    for l in range(1, L):
        assert T[l, 0] >= T[l, 3] - eps  # the fetch waits for its selection
        assert T[l, 4] >= T[l, 1] - eps  # attention (staged) / append (fused) waits for the fetch
        if l >= 2:
            assert T[l, 0] >= T[l - 1, 1] - eps  # one fetch stream: fetches in layer order


@pytest.mark.parametrize("fused_fetch", [False, True])
def test_graph_replay_matches_eager_step(mods, fused_fetch):
    """The CUDA-graph form of the step gives the same bytes as the eager step, step after step."""
    ig, decoder = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-graph", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=10, pool_frac=0.95)
    dev = "cuda:0"
    outs = {}
    for graph in (False, True):
        dec = decoder.Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=w.k,
                              Lcap=w.lcap, pool_cap=w.pool_cap, alpha=4.0, graph=graph, stage_timing=graph,
                              fused_fetch=fused_fetch, device=dev)
        try:
            for l in range(w.layers):
                dd = _layer_data(w, l, w.pool_cap, False)
                t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
                dec.load_layer(l, t(dd["K"]), t(dd["V"]), dd["cols"], Wq_part=t(dd["Wqp"]))
            dec.prefill(w.prompt)
            res = []
            for s in range(5):  # crosses the capture step and eviction (the pool is full)
                x = torch.from_numpy(synth.layer_inputs(w, step=s)).to(dev)
                qkv = [synth.token_inputs(w, l, s) for l in range(w.layers)]
                q, kn, vn = (torch.from_numpy(np.stack([a[i] for a in qkv])).to(dev) for i in range(3))
                out = torch.empty((w.layers, w.batch, w.heads, w.head_dim), dtype=torch.float32, device=dev)
                dec.step(x, q, kn, vn, out)
                dec.finish()
                ig.ig_check(dec.S)
                res.append((out.cpu().numpy(), dec.cnt.cpu().numpy(), dec.slot_host[s % 2].numpy().copy()))
                if graph and s >= 1:
                    ms, n = dec.stage_ms()
                    assert n[0] == w.layers - 1 and ms[0] > 0
                    _check_timeline(dec.timeline(), w.layers, fused_fetch)
            outs[graph] = res
        finally:
            dec.close()
    for (o0, c0, s0), (o1, c1, s1) in zip(outs[False], outs[True]):
        assert np.array_equal(s0, s1) and np.array_equal(c0, c1)
        assert np.array_equal(o0, o1)


@pytest.mark.parametrize("graph", [False, True])
def test_step_from_host_buffers_equals_device_step(mods, graph):
    """Decoder.step_host (pinned host inputs and output, transfers on a copy stream overlapping
    the neighbouring steps) gives the same bytes as Decoder.step on device tensors, step after
    step, across graph capture and eviction."""
    ig, decoder = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-host", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=10, pool_frac=0.95)
    dev = "cuda:0"
    decs = []
    for _ in range(2):
        dec = decoder.Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=w.k,
                              Lcap=w.lcap, pool_cap=w.pool_cap, alpha=4.0, graph=graph, device=dev)
        for l in range(w.layers):
            dd = _layer_data(w, l, w.pool_cap, False)
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
            dec.load_layer(l, t(dd["K"]), t(dd["V"]), dd["cols"], Wq_part=t(dd["Wqp"]))
        dec.prefill(w.prompt)
        decs.append(dec)
    try:
        shape = (w.layers, w.batch, w.heads, w.head_dim)
        hout = [torch.empty(shape, dtype=torch.float32).pin_memory() for _ in range(5)]
        ref = []
        for s in range(5):
            x = synth.layer_inputs(w, step=s)
            qkv = [synth.token_inputs(w, l, s) for l in range(w.layers)]
            q, kn, vn = (np.stack([a[i] for a in qkv]) for i in range(3))
            out = torch.empty(shape, dtype=torch.float32, device=dev)
            decs[0].step(*(torch.from_numpy(a).to(dev) for a in (x, q, kn, vn)), out)
            decs[0].finish()
            ref.append(out.cpu().numpy())
            decs[1].step_host(*(torch.from_numpy(a).pin_memory() for a in (x, q, kn, vn)), hout[s])
        decs[1].finish_host()
        ig.ig_check()
        for s in range(5):
            assert np.array_equal(hout[s].numpy(), ref[s]), f"step {s}"
    finally:
        for dec in decs:
            dec.close()
