"""The prefill stage on the GPU against the oracle.

* ``ig_gemm_tn`` (the tcgen05 GEMM): against the float64 product rounded to fp16, within the
  fp16 rounding (half an ulp, one ulp allowed) plus the fp32 accumulation bound, over ragged
  M, N and K; its per-tile column sums of |C| within 1e-3 relative (fp16 rounding flips).
* ``ig_prefill_layer``: keys and values within the same bound of the oracle's, the columns equal
  (except heads whose k-th and (k+1)-th column scores are within 1e-4 relative), the partial
  weight exactly the chosen rows, the pool rows and the partial key cache at the oracle's slots.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from speculative_kv_cache_gb300 import synth  # noqa: E402
from gpu_util import dev, empty, host, workspace  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig as mod

    return mod


def _ulp16(x):
    """Spacing of fp16 values at |x| (subnormal spacing near 0)."""
    a = np.maximum(np.abs(x), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - 10)


# the last two have more tiles than SMs: each persistent CTA takes several, alternating its
# two accumulators and reusing each (ragged M, N and K in the second)
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 288, 72), (1000, 512, 1000), (129, 32, 8), (4096, 768, 2048),
                                   (16384, 1024, 128), (20000, 288, 72)])
def test_gemm_matches_float64(ig, M, N, K):
    g = np.random.default_rng(M + N + K)
    A = g.standard_normal((M, K)).astype(np.float16)
    Bt = (g.standard_normal((N, K)) * 0.05).astype(np.float16)
    C = empty((M, N), torch.float16)
    mt = (M + 127) // 128
    cp = empty((mt, N), torch.float32)
    ig.ig_gemm_tn(None, M, N, K, dev(A), dev(Bt), C, cp)
    ig.ig_check()
    ref = A.astype(np.float64) @ Bt.astype(np.float64).T
    absprod = np.abs(A.astype(np.float64)) @ np.abs(Bt.astype(np.float64)).T
    got = host(C).astype(np.float64)
    bound = _ulp16(ref) + K * 2.0 ** -23 * absprod
    assert np.all(np.abs(got - ref) <= bound)
    ref16 = np.abs(ref.astype(np.float16).astype(np.float64))
    want = np.stack([ref16[t * 128:(t + 1) * 128].sum(0) for t in range(mt)])
    assert np.allclose(host(cp), want, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("d,cap", [(128, 256), (128, 320), (64, 300)])
def test_prefill_layer_matches_oracle(ig, d, cap):
    B, N, D, H, k = 2, 300, 512, 4, 38 if d == 128 else 16
    Lcap = (cap + 7) // 8 * 8
    g = np.random.default_rng(d + cap)
    X = g.standard_normal((B, N, D)).astype(np.float16)
    Wq, Wk, Wv = ((g.standard_normal((D, H * d)) * 0.02 * (1 + np.arange(H * d) % 7)).astype(np.float16)
                  for _ in range(3))
    pool = ig.ig_pool_create(1, B, H, d, cap)
    try:
        cols = empty((H, k), torch.int32)
        Wqp_t = empty((H * k, D), torch.float16)
        Kpart = torch.zeros((B, H, k, Lcap), dtype=torch.float16, device="cuda")
        ws = workspace(ig.ig_prefill_workspace_bytes(B, N, H, d))
        t = lambda a: dev(np.ascontiguousarray(a.T))  # noqa: E731
        ig.ig_prefill_layer(None, pool, 0, B, N, D, H, d, k, Lcap, dev(X), t(Wq), t(Wk), t(Wv), cols, Wqp_t, Kpart,
                            ws, ws.numel())
        ig.ig_check()
        o = ora.prefill_layer(X, Wq, Wk, Wv, H, d, k, cap)
        Kg = host(ws[: B * N * H * d * 2].view(torch.float16)).reshape(B, N, H, d).astype(np.float64)
        Kw = o["K"].astype(np.float64)
        # fp16 rounding plus the fp32 accumulation bound over the D-long dot products
        X64 = np.abs(X.astype(np.float64))
        bk = (_ulp16(Kw) + D * 2.0 ** -23 * (X64 @ np.abs(Wk.astype(np.float64))).reshape(B, N, H, d))
        bv = (_ulp16(o["V"].astype(np.float64)) + D * 2.0 ** -23 * (X64 @ np.abs(Wv.astype(np.float64))).reshape(B, N, H, d))
        assert np.all(np.abs(Kg - Kw) <= bk)
        got_cols = host(cols)
        sc = ora.colscores(Wq, o["K"], H, d)
        same = np.ones(H, bool)
        for h in range(H):
            s_sorted = np.sort(sc[h])[::-1]
            near = s_sorted[k - 1] - s_sorted[k] <= 1e-4 * s_sorted[k - 1]
            same[h] = np.array_equal(got_cols[h], o["cols"][h])
            assert same[h] or near, h
        Wp = host(Wqp_t)
        for h in range(H):
            assert np.array_equal(Wp[h * k:(h + 1) * k], Wq.T[h * d + got_cols[h]])
        Kp, Vp = ig.pool_layer_view(pool, 0, B, H, cap, d)
        first = max(0, N - cap)
        for tt in range(first, N):
            sl = tt % cap
            assert np.all(np.abs(Kp[:, :, sl].astype(np.float64) - Kw[:, tt]) <= bk[:, tt])
            Vw = o["V"][:, tt].astype(np.float64)
            assert np.all(np.abs(Vp[:, :, sl].astype(np.float64) - Vw) <= bv[:, tt])
            # the pool holds exactly the keys the GEMM produced
            assert np.array_equal(Kp[:, :, sl].astype(np.float64), Kg[:, tt])
        kp = host(Kpart)[..., :cap]
        for h in range(H):
            if not same[h]:
                continue
            # the partial key cache holds exactly the chosen columns of the keys the GEMM produced
            for tt in range(first, N):
                assert np.array_equal(kp[:, h, :, tt % cap].astype(np.float64), Kg[:, tt, h][:, got_cols[h]])
    finally:
        ig.ig_pool_destroy(pool)


def test_decoder_built_by_the_library_prefill(ig):
    """A decoder whose layers >= 1 are filled by ig_prefill_layer (the library builds its own
    decode inputs: pool rows, columns, partial weight, partial key cache), then one decode step:
    its outputs match the oracle's attention over the oracle's own prefilled keys and values,
    on the GPU's index sets."""
    import math

    from speculative_kv_cache_gb300 import decoder, prefill

    L, B, H, d, D, N, k = 3, 2, 4, 128, 512, 200, 38
    cap, Lcap = N + 8, N + 8
    g = np.random.default_rng(5)
    dec = decoder.Decoder(layers=L, B=B, H=H, d=d, D=D, k=k, Lcap=Lcap, pool_cap=cap, alpha=4.0, device="cuda:0")
    try:
        orc = {}
        for l in range(L):
            X = g.standard_normal((B, N, D)).astype(np.float16)
            Wq, Wk, Wv = ((g.standard_normal((D, H * d)) * 0.05 * (1 + np.arange(H * d) % 5)).astype(np.float16)
                          for _ in range(3))
            o = ora.prefill_layer(X, Wq, Wk, Wv, H, d, k, cap)
            orc[l] = o
            if l == 0:  # layer 0 attends densely over HBM rows: its K/V are loaded as they are
                Kb = np.zeros((B, H, cap, d), np.float16)
                Vb = np.zeros_like(Kb)
                Kb[:, :, :N] = o["K"].transpose(0, 2, 1, 3)
                Vb[:, :, :N] = o["V"].transpose(0, 2, 1, 3)
                dec.load_layer(0, dev(Kb), dev(Vb), o["cols"], Wq_part=dev(o["Wq_part"]))
            else:
                t = lambda a: dev(np.ascontiguousarray(a.T))  # noqa: E731
                prefill.prefill_decoder_layer(dec, l, dev(X), t(Wq), t(Wk), t(Wv))
        dec.prefill(N)
        x = g.standard_normal((L, B, D)).astype(np.float16)
        q, kn, vn = (g.standard_normal((L, B, H, d)).astype(np.float16) for _ in range(3))
        out = torch.empty((L, B, H, d), dtype=torch.float32, device="cuda")
        dec.step(dev(x), dev(q), dev(kn), dev(vn), out)
        dec.finish()
        ig.ig_check(dec.S)
        o_gpu, cnt, idx_buf = host(out), host(dec.cnt), host(dec.idx)
        scale = np.float32(1.0 / math.sqrt(d))
        for l in range(1, L):
            gi = idx_buf[l % 2]
            sets = [[gi[b, h, :cnt[l, b, h]] for h in range(H)] for b in range(B)]
            assert all(int(t) < N for r in sets for s_ in r for t in s_)
            Kg, Vg = ora.gather(orc[l]["K_pool"], orc[l]["V_pool"], sets, Lcap)
            want = ora.attend(q[l], Kg, Vg, cnt[l], scale, kn[l], vn[l])
            assert np.abs(o_gpu[l] - want).max() <= 2e-3
            assert cnt[l].sum() > 0
    finally:
        dec.close()


@pytest.mark.parametrize("d,cap", [(128, 320), (64, 250)])
def test_prefill_layer_rope_matches_oracle(ig, d, cap):
    """RoPE prefill: keys within one fp16 ulp plus the fp32 bound of the oracle's RoPE_t(X W_K) A,
    columns as the oracle's (but near ties), A_cols exactly A[:, cols], pool rows and partial
    keys exactly the kernel's own keys at the oracle's slots."""
    B, N, D, H, k, theta = 2, 300, 512, 4, 38 if d == 128 else 16, 10000.0
    Lcap = (cap + 7) // 8 * 8
    g = np.random.default_rng(7 + d)
    X = g.standard_normal((B, N, D)).astype(np.float16)
    Wq, Wk, Wv = ((g.standard_normal((D, H * d)) * 0.02 * (1 + np.arange(H * d) % 5)).astype(np.float16)
                  for _ in range(3))
    A = np.stack([np.linalg.qr(g.standard_normal((d, d)))[0] for _ in range(H)])
    Wq_s = np.zeros_like(Wq)
    for h in range(H):
        Wq_s[:, h * d:(h + 1) * d] = (Wq[:, h * d:(h + 1) * d].astype(np.float64) @ A[h]).astype(np.float16)
    pool = ig.ig_pool_create(1, B, H, d, cap)
    try:
        cols = empty((H, k), torch.int32)
        Ac = empty((H, d, k), torch.float32)
        Kpart = torch.zeros((B, H, k, Lcap), dtype=torch.float16, device="cuda")
        ws = workspace(ig.ig_prefill_workspace_bytes(B, N, H, d))
        t = lambda a: dev(np.ascontiguousarray(a.T))  # noqa: E731
        ig.ig_prefill_layer_rope(None, pool, 0, B, N, D, H, d, k, Lcap, theta, dev(X), t(Wq_s), t(Wk), t(Wv),
                                 dev(A.astype(np.float32)), cols, Ac, Kpart, ws, ws.numel())
        ig.ig_check()
        o = ora.prefill_layer_rope(X, Wq_s, Wk, Wv, A.astype(np.float32).astype(np.float64), theta, H, d, k, cap)
        Kg = host(ws[: B * N * H * d * 2].view(torch.float16)).reshape(B, N, H, d).astype(np.float64)
        Kw = o["K"].astype(np.float64)
        # the unskewed key is rounded to fp16 on both sides, then rotated and skewed; the
        # projection's fp32 accumulation can move that rounding by an ulp, which the skew spreads
        X64 = np.abs(X.astype(np.float64))
        pre = D * 2.0 ** -23 * (X64 @ np.abs(Wk.astype(np.float64))).reshape(B, N, H, d)
        Kraw = (X.astype(np.float64) @ Wk.astype(np.float64)).reshape(B, N, H, d)
        braw = _ulp16(Kraw) + pre
        brot = braw + np.roll(braw, d // 2, axis=-1)  # a rotation mixes each pair (j, j + d/2)
        spread = np.einsum("bnhi,hij->bnhj", brot, np.abs(A))
        assert np.all(np.abs(Kg - Kw) <= _ulp16(Kw) + spread + 1e-6 * np.abs(Kw).max())
        got_cols = host(cols)
        sc = ora.colscores(Wq_s, o["K"], H, d)
        for h in range(H):
            s_sorted = np.sort(sc[h])[::-1]
            near = s_sorted[k - 1] - s_sorted[k] <= 1e-3 * s_sorted[k - 1]
            assert np.array_equal(got_cols[h], o["cols"][h]) or near, h
            assert np.array_equal(host(Ac)[h], A[h].astype(np.float32)[:, got_cols[h]])
        Kp, _ = ig.pool_layer_view(pool, 0, B, H, cap, d)
        kp = host(Kpart)
        for tt in range(max(0, N - cap), N):
            assert np.array_equal(Kp[:, :, tt % cap].astype(np.float64), Kg[:, tt])
            for h in range(H):
                assert np.array_equal(kp[:, h, :, tt % cap].astype(np.float64), Kg[:, tt, h][:, got_cols[h]])
    finally:
        ig.ig_pool_destroy(pool)


def test_rope_decoder_built_by_the_library_prefill(ig):
    """A RoPE decoder whose layers >= 1 are filled by ig_prefill_layer_rope, then one decode
    step against the oracle's attention over its own prefilled rows, on the GPU's index sets."""
    import math

    from speculative_kv_cache_gb300 import decoder, prefill

    L, B, H, d, D, N, k, theta = 3, 2, 4, 128, 512, 200, 38, 10000.0
    cap = Lcap = N + 8
    g = np.random.default_rng(9)
    dec = decoder.Decoder(layers=L, B=B, H=H, d=d, D=D, k=k, Lcap=Lcap, pool_cap=cap, alpha=4.0, rope_theta=theta,
                          device="cuda:0")
    try:
        orc = {}
        for l in range(L):
            X = g.standard_normal((B, N, D)).astype(np.float16)
            Wq, Wk, Wv = ((g.standard_normal((D, H * d)) * 0.05 * (1 + np.arange(H * d) % 5)).astype(np.float16)
                          for _ in range(3))
            A = np.stack([np.linalg.qr(g.standard_normal((d, d)))[0] for _ in range(H)]).astype(np.float32)
            Wq_s = np.concatenate([(Wq[:, h * d:(h + 1) * d].astype(np.float64) @ A[h]).astype(np.float16)
                                   for h in range(H)], axis=1)
            o = ora.prefill_layer_rope(X, Wq_s, Wk, Wv, A.astype(np.float64), theta, H, d, k, cap)
            orc[l] = (o, Wq, A)
            if l == 0:
                Kb = np.zeros((B, H, cap, d), np.float16)
                Vb = np.zeros_like(Kb)
                Kb[:, :, :N] = o["K"].transpose(0, 2, 1, 3)
                Vb[:, :, :N] = o["V"].transpose(0, 2, 1, 3)
                dec.load_layer(0, dev(Kb), dev(Vb), o["cols"], Wq=dev(Wq), A_cols=dev(o["A_cols"].astype(np.float32)))
            else:
                t = lambda a: dev(np.ascontiguousarray(a.T))  # noqa: E731
                dec.Wq[l].copy_(dev(Wq).t())  # the decode stage projects with the unskewed W_Q
                prefill.prefill_decoder_layer_rope(dec, l, dev(X), t(Wq_s), t(Wk), t(Wv), dev(A))
        dec.prefill(N)
        x = g.standard_normal((L, B, D)).astype(np.float16)
        q, kn, vn = (g.standard_normal((L, B, H, d)).astype(np.float16) for _ in range(3))
        out = torch.empty((L, B, H, d), dtype=torch.float32, device="cuda")
        dec.step(dev(x), dev(q), dev(kn), dev(vn), out, positions=np.full(B, N, np.int32))
        dec.finish()
        ig.ig_check(dec.S)
        o_gpu, cnt, idx_buf = host(out), host(dec.cnt), host(dec.idx)
        scale = np.float32(1.0 / math.sqrt(d))
        for l in range(1, L):
            gi = idx_buf[l % 2]
            sets = [[gi[b, h, :cnt[l, b, h]] for h in range(H)] for b in range(B)]
            o = orc[l][0]
            Kg, Vg = ora.gather(o["K_pool"], o["V_pool"], sets, Lcap)
            want = ora.attend(q[l], Kg, Vg, cnt[l], scale, kn[l], vn[l])
            # the oracle attends over its own keys, which differ from the kernels' by the
            # projection's rounding twice over (before and after the rotation): a relative term
            assert np.abs(o_gpu[l] - want).max() <= 2e-3 + 5e-4 * np.abs(want).max()
            assert cnt[l].sum() > 0
    finally:
        dec.close()
