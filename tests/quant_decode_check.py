"""A few decode steps of a decoder with a quantized pool against the oracle (shared by the FP8 and
INT4 pool tests).

The oracle keeps its own copy of every layer's pool (the seeded fp16 rows plus each step's
appended token at the slot the pool manager gives it, here the next free slot), runs its own
speculation and threshold selection from the fp16 keys (the partial key cache is fp16 whatever
the pool holds), quantizes its own pool rows with its own encoder and dequantizes them, and
attends over its own sets.  The GPU's sets must equal the oracle's except tokens within 1e-3 of
the threshold; the outputs must agree within 2e-3 where the sets are equal, and, where exempt
tokens make them differ, with the oracle's attention over the GPU's set (both are correct
selections).  Nothing the GPU wrote is an input of the oracle.
"""
import math

import numpy as np
import torch

from oracle import infinigen as ora
from speculative_kv_cache_gb300 import synth


def run(ig, decoder, w, quant, pool_flag, fused_fetch, steps=2, alpha=4.0):
    """quant: 'fp8' or 'int4'; pool_flag: the Decoder keyword ('pool_fp8' or 'pool_int4')."""
    devn = "cuda:0"
    cap = w.pool_cap
    assert w.prompt + steps <= cap, "the check assumes the pool does not fill"
    scale = np.float32(1.0 / math.sqrt(w.head_dim))

    def qdq(X):
        if quant == "fp8":
            return ora.fp8_dequantize_rows(*ora.fp8_quantize_rows(X))
        return ora.int4_dequantize_rows(*ora.int4_quantize_rows(X))

    dec = decoder.Decoder(layers=w.layers, B=w.batch, H=w.heads, d=w.head_dim, D=w.hidden, k=w.k, Lcap=w.lcap,
                          pool_cap=cap, alpha=alpha, fused_fetch=fused_fetch, device=devn, **{pool_flag: True})
    try:
        pools, cols_l, w_l = [], [], []
        for l in range(w.layers):
            K, V = synth.pool_layer(w, l, cap=cap)
            cols = synth.skewed_columns(w, l)
            Wqp = synth.skewed_partial_weight(w, l)
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(devn)  # noqa: E731
            dec.load_layer(l, t(K), t(V), cols, Wq_part=t(Wqp))
            pools.append([K.copy(), V.copy()])
            cols_l.append(cols)
            w_l.append(Wqp)
        dec.prefill(w.prompt)
        checked = 0
        for s in range(steps):
            x = synth.layer_inputs(w, step=s)
            qkv = [synth.token_inputs(w, l, s) for l in range(w.layers)]
            q, kn, vn = (np.stack([a[i] for a in qkv]) for i in range(3))
            out = torch.empty((w.layers, w.batch, w.heads, w.head_dim), dtype=torch.float32, device=devn)
            L_now = dec.step(*(torch.from_numpy(a).to(devn) for a in (x, q, kn, vn)), out)
            dec.finish()
            ig.ig_check(dec.S)
            assert L_now == w.prompt + s
            o, cnt, idx_buf = out.cpu().numpy(), dec.cnt.cpu().numpy(), dec.idx.cpu().numpy()
            Lv = np.full(w.batch, L_now, dtype=np.int32)
            for l in range(1, w.layers):
                K, V = pools[l]
                qp = ora.partial_query(x[l - 1], w_l[l], w.heads, w.k)
                sc = ora.speculate(qp, ora.partial_key_cache(K, cols_l[l]), Lv, scale)
                want, want_cnt, _ = ora.select(sc, Lv, alpha)
                gi = idx_buf[l % 2]  # two index lists reused by layer parity: layers 1, 2 here
                gpu_sets = [[gi[b, h, :cnt[l, b, h]] for h in range(w.heads)] for b in range(w.batch)]
                same = np.ones((w.batch, w.heads), dtype=bool)
                for b in range(w.batch):
                    thr = sc[b].max(axis=1) - alpha
                    for h in range(w.heads):
                        diff = set(gpu_sets[b][h].tolist()) ^ set(want[b][h].tolist())
                        for tok in diff:
                            assert abs(sc[b, h, tok] - thr[h]) <= 1e-3, f"layer {l} ({b},{h}) token {tok}"
                        same[b, h] = not diff
                # the oracle's own quantization of its own pool rows (the resident ones)
                Kq, Vq = K.copy(), V.copy()
                Kq[:, :, :L_now] = qdq(K[:, :, :L_now])
                Vq[:, :, :L_now] = qdq(V[:, :, :L_now])
                Kg, Vg = ora.gather(Kq, Vq, want, w.lcap)
                ol = ora.attend(q[l], Kg, Vg, want_cnt, scale, kn[l], vn[l])
                err = np.abs(o[l] - ol).max(axis=2)
                assert err[same].max(initial=0.0) <= 2e-3, f"step {s} layer {l}: {err[same].max()}"
                if not same.all():
                    Kg, Vg = ora.gather(Kq, Vq, gpu_sets, w.lcap)
                    og = ora.attend(q[l], Kg, Vg, cnt[l], scale, kn[l], vn[l])
                    assert np.abs(o[l] - og).max(axis=2)[~same].max() <= 2e-3
                assert want_cnt.sum() > 0
                checked += 1
            # the step's token goes to the next free slot of every layer (the pool is not full)
            for l in range(w.layers):
                pools[l][0][:, :, L_now] = kn[l]
                pools[l][1][:, :, L_now] = vn[l]
        assert checked == steps * (w.layers - 1)
    finally:
        dec.close()
