"""The INT4 pool (signed 4-bit rows + per-row scale) on the GPU against the oracle, bit for bit.

As for the fp8 pool: the packed codes and scales that ig_pool_write, ig_append_kv and
ig_append_kv_layers store, and the fp16 rows ig_gather_kv produces from them, must equal the
oracle's (int4_quantize_rows, int4_pack, int4_dequantize_rows); then a few decoder steps with an
int4 pool against the oracle's attention over the dequantized rows of the GPU's own index sets.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from speculative_kv_cache_gb300 import synth  # noqa: E402
from gpu_util import dev, host  # noqa: E402
import quant_decode_check  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import decoder, ig

    return ig, decoder


def _rows(seed, B, H, cap, d):
    g = np.random.default_rng(seed)
    K = (g.standard_normal((B, H, cap, d)) * g.uniform(0.01, 30, (B, H, cap, 1))).astype(np.float16)
    V = (g.standard_normal((B, H, cap, d)) * 2).astype(np.float16)
    K[0, 0, 3] = 0                      # a zero row: scale 0, codes 0
    K[0, 0, 4, :5] = -0.0               # negative zeros in a nonzero row
    V[-1, -1, -1, 7] = 60000            # a large value (the row's amax)
    K[0, 1, 5] = np.arange(d) % 15 - 7  # an integer row with amax 7: codes equal the values
    return K, V


def _packed(X):
    codes, scales = ora.int4_quantize_rows(X)
    return ora.int4_pack(codes), scales, codes


@pytest.mark.parametrize("d", [64, 128])
def test_int4_pool_write_gather_append_bit_exact(mods, d):
    ig, _ = mods
    B, H, cap, Lcap = 2, 3, 40, 48
    K, V = _rows(d + 1, B, H, cap, d)
    pool = ig.ig_pool_create_ex(2, B, H, d, cap, ig.IG_POOL_COUNTER, ig.IG_POOL_INT4)
    try:
        ig.ig_pool_write(pool, None, 1, dev(K), dev(V))
        torch.cuda.synchronize()
        K4, V4, Ks, Vs = ig.pool_layer_view_int4(pool, 1, B, H, cap, d)
        wk, wks, ck = _packed(K)
        wv, wvs, cv = _packed(V)
        assert np.array_equal(K4, wk) and np.array_equal(V4, wv)
        assert np.array_equal(Ks.view(np.uint32), wks.view(np.uint32))
        assert np.array_equal(Vs.view(np.uint32), wvs.view(np.uint32))
        # gather: ragged counts, every slot at least once across heads
        g = np.random.default_rng(1)
        cnt = g.integers(0, cap + 1, size=(B, H)).astype(np.int32)
        cnt[0, 0] = cap
        idx = np.zeros((B, H, Lcap), np.int32)
        for b in range(B):
            for h in range(H):
                idx[b, h, :cnt[b, h]] = np.sort(g.permutation(cap)[:cnt[b, h]])
        Kg = torch.zeros((B, H, Lcap, d), dtype=torch.float16, device="cuda")
        Vg = torch.zeros_like(Kg)
        ig.ig_gather_kv(None, pool, 1, B, H, d, Lcap, dev(idx), dev(cnt), Kg, Vg, 0)
        ig.ig_check()
        Kd, Vd = ora.int4_dequantize_rows(ck, wks), ora.int4_dequantize_rows(cv, wvs)
        Kh, Vh = host(Kg), host(Vg)
        for b in range(B):
            for h in range(H):
                n = cnt[b, h]
                assert Kh[b, h, :n].tobytes() == Kd[b, h, idx[b, h, :n]].tobytes()
                assert Vh[b, h, :n].tobytes() == Vd[b, h, idx[b, h, :n]].tobytes()
        assert np.array_equal(Kd[0, 1, 5], K[0, 1, 5])  # the integer row comes back exactly
        # append: the new rows are quantized into their slots; the partial key stays fp16
        k = 16
        kn = (g.standard_normal((B, H, d)) * 3).astype(np.float16)
        vn = (g.standard_normal((B, H, d)) * 3).astype(np.float16)
        slot = np.array([7, -1][:B], np.int32)
        cols = np.stack([np.sort(g.permutation(d)[:k]) for _ in range(H)]).astype(np.int32)
        Kpart = torch.zeros((B, H, k, Lcap), dtype=torch.float16, device="cuda")
        ig.ig_append_kv(None, pool, 1, B, H, d, k, Lcap, dev(slot), dev(cols), dev(kn), dev(vn), Kpart)
        torch.cuda.synchronize()
        ig.ig_check()
        K4, V4, Ks, Vs = ig.pool_layer_view_int4(pool, 1, B, H, cap, d)
        ak, aks, _ = _packed(kn[0])
        av, avs, _ = _packed(vn[0])
        assert np.array_equal(K4[0, :, 7], ak) and np.array_equal(V4[0, :, 7], av)
        assert np.array_equal(Ks[0, :, 7], aks) and np.array_equal(Vs[0, :, 7], avs)
        assert np.array_equal(K4[1], wk[1]) and np.array_equal(Ks[1], wks[1])  # slot -1: untouched
        kp = host(Kpart)
        for h in range(H):
            assert np.array_equal(kp[0, h, :, 7], kn[0, h, cols[h]])
        # the batched append of two layers quantizes the same way
        kn2 = np.stack([kn, -kn]).astype(np.float16)
        vn2 = np.stack([vn, vn * 2]).astype(np.float16)
        slot2 = np.array([[-1] * B, [9, 11][:B]], np.int32)
        ig.ig_append_kv_layers(None, pool, 2, B, H, d, [0, 0], Lcap, dev(slot2), [None, None], dev(kn2), dev(vn2),
                               None)
        torch.cuda.synchronize()
        ig.ig_check()
        K4, V4, Ks, Vs = ig.pool_layer_view_int4(pool, 1, B, H, cap, d)
        for b in range(B):
            bk, bks, _ = _packed(kn2[1, b])
            bv, bvs, _ = _packed(vn2[1, b])
            s_ = slot2[1, b]
            assert np.array_equal(K4[b, :, s_], bk) and np.array_equal(Ks[b, :, s_], bks)
            assert np.array_equal(V4[b, :, s_], bv) and np.array_equal(Vs[b, :, s_], bvs)
        # the fp16-only calls refuse an int4 pool; the two formats exclude each other
        with pytest.raises(ig.IGError):
            ig.ig_pool_kv(pool, 1)
        with pytest.raises(ig.IGError):
            ig.ig_pool_create_ex(1, B, H, d, cap, ig.IG_POOL_COUNTER, ig.IG_POOL_INT4 | ig.IG_POOL_FP8)
    finally:
        ig.ig_pool_destroy(pool)


@pytest.mark.parametrize("fused_fetch", [False, True])
def test_decoder_with_int4_pool(mods, fused_fetch):
    """Decode steps over an INT4 pool, staged (the fetch dequantizes into HBM) or fused (the
    fetch stream's attention dequantizes in registers), against the oracle's own selection and its
    attention over its own quantization of its own pool rows (tests/quant_decode_check.py)."""
    ig, decoder = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-int4", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=6)
    quant_decode_check.run(ig, decoder, w, "int4", "pool_int4", fused_fetch)



@pytest.mark.parametrize("fmt", ["fp8", "int4"])
@pytest.mark.parametrize("with_new", [False, True])
@pytest.mark.parametrize("d,grid", [(128, 0), (64, 0), (128, 1), (128, 7), (128, 256)])
def test_fused_fetch_attend_on_quantized_pools(mods, fmt, with_new, d, grid):
    """ig_gather_attend on a quantized pool (codes over the host link, scales from HBM,
    dequantized in registers) against the oracle: its own quantization of the same seeded rows,
    dequantized, then its attention over the same index sets.  The OPT-30B recipe (key scale,
    planted rows) at 2 sequences x 8 heads and head dimensions 128 and 64, so that the
    pure-Python e4m3 encoder finishes in seconds; quantization is row by row, so quantizing only
    the gathered rows equals quantizing the pool."""
    ig, _ = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], batch=2, heads=8, head_dim=d)
    B, H, cap, Lcap = w.batch, w.heads, 2048, 2048
    K, V = synth.pool_layer(w, 1, cap=cap)
    q, kn, vn = synth.token_inputs(w, 1, 0)
    g = np.random.default_rng(5)
    cnt = np.clip(np.round(np.exp(g.normal(np.log(120), 0.9, size=(B, H)))), 0, 1900).astype(np.int32)
    cnt[0, 0], cnt[0, 1], cnt[1, 2] = 0, 1900, 1
    idx = np.zeros((B, H, Lcap), np.int32)
    for b in range(B):
        for h in range(H):
            idx[b, h, :cnt[b, h]] = np.sort(g.permutation(cap)[:cnt[b, h]])
    flag = ig.IG_POOL_FP8 if fmt == "fp8" else ig.IG_POOL_INT4
    pool = ig.ig_pool_create_ex(1, B, H, d, cap, ig.IG_POOL_COUNTER, flag)
    try:
        ig.ig_pool_write(pool, None, 0, dev(K), dev(V))
        ws = torch.empty(ig.ig_gather_attend_workspace_bytes(B, H, d, Lcap), dtype=torch.uint8, device="cuda")
        out = torch.empty((B, H, d), dtype=torch.float32, device="cuda")
        scale = float(np.float32(1.0 / math.sqrt(d)))
        # grid 0: the library's default; 1, 7, 256: one CTA for every row, ragged CTA ranges that
        # split heads at odd rows, more CTAs than the small heads need
        ig.ig_gather_attend(None, pool, 0, B, H, d, Lcap, scale, dev(q), dev(idx), dev(cnt),
                            dev(kn) if with_new else None, dev(vn) if with_new else None, out, ws, ws.numel(), grid)
        ig.ig_check()
        sets = [[idx[b, h, :cnt[b, h]] for h in range(H)] for b in range(B)]
        Kg, Vg = ora.gather(K, V, sets, Lcap)
        if fmt == "fp8":
            Kg = ora.fp8_dequantize_rows(*ora.fp8_quantize_rows(Kg))
            Vg = ora.fp8_dequantize_rows(*ora.fp8_quantize_rows(Vg))
        else:
            Kg = ora.int4_dequantize_rows(*ora.int4_quantize_rows(Kg))
            Vg = ora.int4_dequantize_rows(*ora.int4_quantize_rows(Vg))
        want = ora.attend(q, Kg, Vg, cnt, scale, kn if with_new else None, vn if with_new else None)
        assert np.abs(host(out) - want).max() <= 2e-3
    finally:
        ig.ig_pool_destroy(pool)
