"""The FP8 pool (e4m3 rows + per-row scale) on the GPU against the oracle, bit for bit.

Quantization on the way in (ig_pool_write, ig_append_kv), dequantization on the way out
(ig_gather_kv): the stored codes and scales and the fp16 rows the gather produces must equal
the oracle's; the partial key cache stays fp16 (the appended partial key is the unquantized
key column).  Then a few decoder steps with an fp8 pool against the oracle's attention over the
dequantized rows of the GPU's own index sets.
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
    return K, V


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_pool_write_gather_append_bit_exact(mods, d):
    ig, _ = mods
    B, H, cap, Lcap = 2, 3, 40, 48
    K, V = _rows(d, B, H, cap, d)
    pool = ig.ig_pool_create_ex(2, B, H, d, cap, ig.IG_POOL_COUNTER, ig.IG_POOL_FP8)
    try:
        ig.ig_pool_write(pool, None, 1, dev(K), dev(V))
        torch.cuda.synchronize()
        K8, V8, Ks, Vs = ig.pool_layer_view_fp8(pool, 1, B, H, cap, d)
        wk, wks = ora.fp8_quantize_rows(K)
        wv, wvs = ora.fp8_quantize_rows(V)
        assert np.array_equal(K8, wk) and np.array_equal(V8, wv)
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
        Kd, Vd = ora.fp8_dequantize_rows(wk, wks), ora.fp8_dequantize_rows(wv, wvs)
        Kh, Vh = host(Kg), host(Vg)
        for b in range(B):
            for h in range(H):
                n = cnt[b, h]
                assert Kh[b, h, :n].tobytes() == Kd[b, h, idx[b, h, :n]].tobytes()
                assert Vh[b, h, :n].tobytes() == Vd[b, h, idx[b, h, :n]].tobytes()
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
        K8, V8, Ks, Vs = ig.pool_layer_view_fp8(pool, 1, B, H, cap, d)
        ak, aks = ora.fp8_quantize_rows(kn[0])
        av, avs = ora.fp8_quantize_rows(vn[0])
        assert np.array_equal(K8[0, :, 7], ak) and np.array_equal(V8[0, :, 7], av)
        assert np.array_equal(Ks[0, :, 7], aks) and np.array_equal(Vs[0, :, 7], avs)
        assert np.array_equal(K8[1], wk[1]) and np.array_equal(Ks[1], wks[1])  # slot -1: untouched
        kp = host(Kpart)
        for h in range(H):
            assert np.array_equal(kp[0, h, :, 7], kn[0, h, cols[h]])
        # the fp16-only calls refuse an fp8 pool
        with pytest.raises(ig.IGError):
            ig.ig_pool_kv(pool, 1)
    finally:
        ig.ig_pool_destroy(pool)


@pytest.mark.parametrize("fused_fetch", [False, True])
def test_decoder_with_fp8_pool(mods, fused_fetch):
    """Decode steps over an FP8 pool, staged (the fetch dequantizes into HBM) or fused (the
    fetch stream's attention dequantizes in registers), against the oracle's own selection and its
    attention over its own quantization of its own pool rows (tests/quant_decode_check.py)."""
    ig, decoder = mods
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="dec-fp8", layers=3, batch=2, heads=4, hidden=512,
                     prompt=200, gen=6)
    quant_decode_check.run(ig, decoder, w, "fp8", "pool_fp8", fused_fetch)
