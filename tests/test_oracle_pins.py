"""Pins of the CPU oracle against what the InfiniGen pages and plain mathematics fix.

None of these tests needs a GPU.  Each one is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand) makes it fail.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

from oracle import infinigen as ora
from speculative_kv_cache_gb300 import synth


def _rand(seed, shape, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# --- P1: the skew is an orthogonal rotation, so rotated dot products are unchanged -------
@pytest.mark.parametrize("theta", [0.0, 10000.0])
def test_p1_skew_is_orthogonal_and_preserves_dot_products(theta):
    H, d, D, Ns = 3, 16, 48, 64
    Xs = _rand(1, (Ns, D)).astype(np.float16)
    Wq = _rand(2, (D, H * d), 0.02).astype(np.float16)
    Wk = _rand(3, (D, H * d), 0.02).astype(np.float16)
    A, _, _, _, _ = ora.skew(Xs, Wq, Wk, H, d, rope_theta=theta)
    for h in range(H):
        assert np.abs(A[h].T @ A[h] - np.eye(d)).max() < 1e-12
    # full-width rotated q.k equals unrotated q.k (float64, before any fp16 rounding)
    x = _rand(4, (5, D))
    y = _rand(5, (7, D))
    q = (x @ Wq.astype(np.float64)).reshape(5, H, d)
    kk = (y @ Wk.astype(np.float64)).reshape(7, H, d)
    if theta:
        q = ora.rope(q, np.arange(5)[:, None] + 100, theta)
        kk = ora.rope(kk, np.arange(7)[:, None], theta)
    for h in range(H):
        ref = q[:, h] @ kk[:, h].T
        rot = (q[:, h] @ A[h]) @ (kk[:, h] @ A[h]).T
        assert np.abs(rot - ref).max() <= 1e-5 * np.abs(ref).max()


# --- P2: Q A = U Sigma: columns orthogonal, norms are the singular values, descending -----
def test_p2_skewed_sample_queries_are_u_sigma():
    H, d, D, Ns = 2, 12, 40, 50
    Xs = _rand(11, (Ns, D)).astype(np.float16)
    Wq = _rand(12, (D, H * d), 0.02).astype(np.float16)
    A, sig, _, _, _ = ora.skew(Xs, Wq, Wq, H, d)
    Q = Xs.astype(np.float64) @ Wq.astype(np.float64)
    for h in range(H):
        Qh = Q[:, h * d:(h + 1) * d]
        QA = Qh @ A[h]
        G = QA.T @ QA
        # singular values from an independent route: eigenvalues of the Gram matrix
        ev = np.sort(scipy.linalg.eigvalsh(Qh.T @ Qh))[::-1]
        assert np.allclose(np.sqrt(np.diag(G)), np.sqrt(np.maximum(ev, 0)), rtol=1e-10, atol=1e-12)
        assert np.all(np.diff(np.diag(G)) <= 1e-9)
        off = G - np.diag(np.diag(G))
        assert np.abs(off).max() < 1e-9 * np.abs(G).max()
        assert np.allclose(sig[h], np.sqrt(np.maximum(ev, 0)), rtol=1e-10)


def test_p2_sign_canonicalisation():
    A = np.array([[0.6, -0.8], [-0.8, -0.6]])
    C = ora.canonical_signs(A)
    assert np.array_equal(C, np.array([[-0.6, 0.8], [0.8, 0.6]]))
    # ties go to the lowest row
    T = ora.canonical_signs(np.array([[-0.5, 0.5], [0.5, 0.5]]))
    assert T[0, 0] == 0.5 and T[1, 0] == -0.5


# --- P3: ratio 1 and alpha = inf reproduce dense attention ---------------------------------
@pytest.mark.parametrize("with_new", [False, True])
def test_p3_full_ratio_infinite_alpha_is_dense_attention(with_new):
    B, H, d, D, L, Ns = 2, 3, 8, 24, 20, 40
    Xs = _rand(21, (Ns, D)).astype(np.float16)
    Wq = _rand(22, (D, H * d), 0.05).astype(np.float16)
    A, _, Wq_s, _, _ = ora.skew(Xs, Wq, Wq, H, d)
    k = ora.partial_columns(1.0, d)
    assert k == d
    K = _rand(23, (B, H, L, d))
    V = _rand(24, (B, H, L, d))
    q = _rand(25, (B, H, d))
    kn = _rand(26, (B, H, d))
    vn = _rand(27, (B, H, d))
    Kt = np.einsum("bhtc,hcj->bhtj", K, A)
    qt = np.einsum("bhc,hcj->bhj", q, A)
    knt = np.einsum("bhc,hcj->bhj", kn, A)
    cols = ora.choose_columns(Wq_s, None, H, d, k)
    assert np.array_equal(cols, np.tile(np.arange(d), (H, 1)))
    Kpart = ora.partial_key_cache(Kt, cols)
    Wqp = ora.partial_weight(Wq_s, cols, H, d)
    x = _rand(28, (B, D)).astype(np.float16)
    scale = 1 / math.sqrt(d)
    r = ora.decode_layer_step(x, Wqp, Kpart, np.full(B, L), qt, Kt, V, H=H, k=k, scale=scale,
                              alpha=np.inf, k_new=knt if with_new else None,
                              v_new=vn if with_new else None)
    assert np.all(r["cnt"] == L)
    for b in range(B):
        for h in range(H):
            Kd, Vd = K[b, h], V[b, h]
            if with_new:
                Kd = np.vstack([Kd, kn[b, h]])
                Vd = np.vstack([Vd, vn[b, h]])
            w = scipy.special.softmax(np.float32(scale) * (Kd @ q[b, h]))
            assert np.allclose(r["out"][b, h], w @ Vd, rtol=0, atol=1e-12)


# --- P5: the page's worked number e^-5 ~ 0.0067 ~ 1/148.4 ----------------------------------
def test_p5_alpha_five_weight_ratio(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "softmax_alpha5.json")))
    d = 4
    scale = 1.0  # the gap is stated in logit units
    q = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    Kg = np.zeros((1, 1, 2, d))
    Kg[0, 0, 0, 0] = 10.0
    Kg[0, 0, 1, 0] = 10.0 - g["gap"]
    Vg = np.zeros((1, 1, 2, d))
    Vg[0, 0, 0, 1] = 1.0
    Vg[0, 0, 1, 2] = 1.0
    o = ora.attend(q, Kg, Vg, np.array([[2]]), scale)[0, 0]
    ratio = o[2] / o[1]
    assert round(ratio, g["weight_ratio_printed_digits"]) == g["weight_ratio"]
    assert round(1 / ratio, g["inverse_printed_digits"]) == g["inverse"]


# --- P6: partial weight / partial key cache fractions ---------------------------------------
def test_p6_memory_fractions(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "memory_fraction.json")))
    for s in g["shapes"]:
        k = ora.partial_columns(g["ratio"], s["head_dim"])
        kv_frac = 100.0 * k / (2 * s["head_dim"])          # k of 2d numbers per token and head
        w_frac = 100.0 * s["heads"] * k * s["hidden"] / (g["params_per_block_over_hidden_sq"] * s["hidden"] ** 2)
        assert abs(kv_frac - g["partial_key_cache_pct"]) <= g["printed_tolerance_pct"]
        assert abs(w_frac - g["partial_weight_pct"]) <= g["printed_tolerance_pct"]
    assert ora.partial_columns(0.3, 128) == 38
    assert ora.partial_columns(0.25, 64) == 16


# --- P7: cap rounding reproduces the page's 102 and 410 ------------------------------------
def test_p7_cap_rounding(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "transfer_cap.json")))
    for n, want in g["cases"]:
        assert ora.cap_count(g["cap_frac"], n) == want
    assert ora.cap_count(1.0, 77) == 77


# --- P8: alpha -> 0+ keeps only the maximum (and exact ties) -------------------------------
def test_p8_tiny_alpha_selects_argmax_and_ties():
    s = np.array([[[0.5, 2.0, -1.0, 2.0, 1.999]]])
    idx, cnt, used = ora.select(s, [5], 1e-30)
    assert list(idx[0][0]) == [1, 3] and cnt[0, 0] == 2
    assert list(used[0]) == [0, 1, 0, 1, 0]


# --- P9: flipping a column sign of A changes nothing downstream ----------------------------
def test_p9_sign_flip_invariance():
    B, H, d, D, L, Ns = 2, 2, 16, 32, 30, 48
    Xs = _rand(31, (Ns, D)).astype(np.float16)
    Wq = _rand(32, (D, H * d), 0.05).astype(np.float16)
    A, _, _, _, _ = ora.skew(Xs, Wq, Wq, H, d)
    K = _rand(33, (B, H, L, d))
    V = _rand(34, (B, H, L, d))
    q = _rand(35, (B, H, d))
    x = _rand(36, (B, D))
    k = ora.partial_columns(0.3, d)
    res = []
    for flip in [None, 3]:
        Af = A.copy()
        if flip is not None:
            Af[:, :, flip] *= -1
        Wq_s = np.concatenate([Wq.astype(np.float64)[:, h * d:(h + 1) * d] @ Af[h] for h in range(H)], 1)
        Kt = np.einsum("bhtc,hcj->bhtj", K, Af)
        qt = np.einsum("bhc,hcj->bhj", q, Af)
        cols = ora.choose_columns(Wq_s, np.transpose(Kt, (0, 2, 1, 3)), H, d, k)
        Kpart = ora.partial_key_cache(Kt, cols)
        r = ora.decode_layer_step(x, ora.partial_weight(Wq_s, cols, H, d), Kpart, np.full(B, L), qt, Kt, V,
                                  H=H, k=k, scale=1 / math.sqrt(d), alpha=2.0)
        res.append((cols, r))
    (c0, r0), (c1, r1) = res
    assert np.array_equal(c0, c1)
    assert np.allclose(r0["scores"], r1["scores"], atol=1e-12)
    assert all(np.array_equal(r0["idx"][b][h], r1["idx"][b][h]) for b in range(B) for h in range(H))
    assert np.allclose(r0["out"], r1["out"], atol=1e-12)


# --- P10: pool slot order is free ----------------------------------------------------------
def test_p10_slot_permutation():
    B, H, d, k, L = 2, 3, 8, 3, 25
    Kt = _rand(41, (B, H, L, d))
    V = _rand(42, (B, H, L, d))
    q = _rand(43, (B, H, d))
    qp = _rand(44, (B, H, k))
    cols = np.array([[0, 2, 5]] * H)
    perm = np.random.default_rng(45).permutation(L)
    outs, sets = [], []
    for P in [np.arange(L), perm]:
        Kp, Vp = Kt[:, :, P], V[:, :, P]
        Kpart = ora.partial_key_cache(Kp, cols)
        s = ora.speculate(qp, Kpart, np.full(B, L), 0.7)
        idx, cnt, _ = ora.select(s, np.full(B, L), 1.5)
        Kg, Vg = ora.gather(Kp, Vp, idx, L)
        outs.append(ora.attend(q, Kg, Vg, cnt, 0.35))
        sets.append([[set(P[np.asarray(idx[b][h])].tolist()) for h in range(H)] for b in range(B)])
    assert sets[0] == sets[1]
    assert np.allclose(outs[0], outs[1], atol=1e-12)


# --- P11: the selected count never drops as alpha grows ------------------------------------
def test_p11_count_monotone_in_alpha():
    s = _rand(51, (3, 4, 200))
    prev = None
    for a in [0.1, 0.5, 1, 2, 3, 4, 6, 9, np.inf]:
        _, cnt, _ = ora.select(s, [200, 150, 17], a)
        if prev is not None:
            assert np.all(cnt >= prev)
        prev = cnt
    assert np.array_equal(prev, np.array([[200] * 4, [150] * 4, [17] * 4]))


# --- P12: KV-cache bytes of the OPT-30B-shaped workload ------------------------------------
def test_p12_kv_bytes():
    w = synth.WORKLOADS["opt-30b"]
    b = ora.kv_bytes(w.layers, w.batch, w.context, w.hidden)
    assert b == 48 * 16 * 2048 * 7168 * 4
    assert abs(b / 1e9 - 45.1) < 0.05


# --- RoPE: reduces to complex rotation for d = 2; relative-position property -----------------
def test_rope_two_dims_is_complex_rotation():
    x = _rand(61, (7, 2))
    p = np.arange(7) * 3 + 1
    z = (x[:, 0] + 1j * x[:, 1]) * np.exp(1j * p)      # theta^0 = 1 for the only pair
    r = ora.rope(x, p, 10000.0)
    assert np.allclose(r[:, 0], z.real, atol=1e-13) and np.allclose(r[:, 1], z.imag, atol=1e-13)


def test_rope_relative_position_and_norm():
    d = 16
    q = _rand(62, d)
    kk = _rand(63, d)
    a = ora.rope(q, 40, 10000.0) @ ora.rope(kk, 13, 10000.0)
    b = ora.rope(q, 27, 10000.0) @ kk
    assert abs(a - b) < 1e-12
    assert abs(np.linalg.norm(ora.rope(q, 99, 500.0)) - np.linalg.norm(q)) < 1e-12
    assert np.allclose(ora.rope(q, 0, 10000.0), q)
    # pair j is (j, j + d/2), not (2j, 2j + 1): only dims 0 and 8 mix for the fastest pair
    e0 = np.zeros(d)
    e0[0] = 1.0
    r = ora.rope(e0, 1, 10000.0)
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2 and abs(r[8] - math.sin(1.0)) < 1e-15


def test_partial_query_rope_identity_skew_matches_rope_of_projection():
    B, H, d, D = 2, 2, 8, 16
    x = _rand(64, (B, D))
    Wq = _rand(65, (D, H * d), 0.1)
    A = np.stack([np.eye(d)] * H)
    cols = np.tile(np.arange(d), (H, 1))
    pos = np.array([5, 900])
    got = ora.partial_query_rope(x, Wq, A, cols, pos, 10000.0)
    q = (x @ Wq).reshape(B, H, d)
    for b in range(B):
        for h in range(H):
            want = ora.rope(q[b, h], pos[b], 10000.0)
            assert np.allclose(got[b, h], want, atol=1e-13)


# --- column choice: the combined score keeps both kinds of outlier column -------------------
def test_column_choice_combines_query_and_key_outliers(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "column_choice.json")))
    W = np.array(g["Wq_skew"])
    K = np.array(g["K_skew"])[:, None, :]
    assert list(ora.choose_columns(W, K, 1, g["head_dim"], g["k"])[0]) == g["expected_cols"]
    assert list(ora.choose_columns(W, None, 1, g["head_dim"], g["k"])[0]) == g["query_only_cols"]
    assert list(ora.choose_columns(np.zeros_like(W), K, 1, g["head_dim"], g["k"])[0]) == g["key_only_cols"]


# --- head averaging rounds half up, minimum one token ---------------------------------------
def test_head_avg_count_rounding():
    # counts per head 3, 5, 4, 6 -> mean 4.5 -> 5 tokens per head
    s = np.full((1, 4, 10), -100.0)
    for h, c in enumerate([3, 5, 4, 6]):
        s[0, h, :c] = 0.0
    s[0, :, 9] = -50.0
    idx, cnt, _ = ora.select(s, [10], 1.0, ora.SEL_HEAD_AVG)
    assert list(cnt[0]) == [5, 5, 5, 5]
    # head 0 has three tied at 0, then takes the best of the rest: -50 at t = 9, then t = 3
    assert list(idx[0][0]) == [0, 1, 2, 3, 9]
    # mean 0.25 rounds to 0 but the minimum is one
    s2 = np.zeros((1, 4, 6))
    s2[0, 0, 2] = 10.0
    s2[0, 1:, :] = np.nan
    idx2, cnt2, _ = ora.select(s2, [6], 1.0, ora.SEL_HEAD_AVG)
    assert list(cnt2[0]) == [1, 0, 0, 0] and list(idx2[0][0]) == [2]


# --- speculation fidelity diagnostics ----------------------------------------------------------
def test_recall_is_one_when_speculation_is_the_real_query_and_all_columns():
    """Ratio 1 (every column) and the real query as the speculation query: the speculated
    scores are the real ones, so the threshold set is a top set and recall is exactly 1."""
    g = np.random.default_rng(3)
    B, H, T, d = 2, 3, 50, 16
    q = g.standard_normal((B, H, d))
    K = g.standard_normal((B, H, T, d))
    L = np.array([50, 31])
    z = ora.real_scores(q, K, L, 0.25)
    idx, cnt, _ = ora.select(z, L, 1.0)
    rec, wt = ora.speculation_recall(z, idx, cnt, L)
    assert np.all(rec == 1.0)
    # weight recall: the softmax mass of the selected set, computed directly
    for b in range(B):
        for h in range(H):
            e = np.exp(z[b, h, :L[b]] - z[b, h, :L[b]].max())
            assert wt[b, h] == pytest.approx(e[list(idx[b][h])].sum() / e.sum(), rel=1e-12)
    # alpha = inf selects everything: all the weight
    idx, cnt, _ = ora.select(z, L, float("inf"))
    _, wt = ora.speculation_recall(z, idx, cnt, L)
    assert np.allclose(wt, 1.0, rtol=1e-14)


def test_recall_closed_form_and_ties():
    z = np.array([[[5.0, 4.0, 3.0, 2.0, 1.0]]])
    L = np.array([5])
    # speculated {0, 3}: top-2 real = {0, 1}; token 3 is not among them -> 1/2
    rec, _ = ora.speculation_recall(z, [[np.array([0, 3])]], np.array([[2]]), L)
    assert rec[0, 0] == 0.5
    # ties at the c-th score count as hits
    z2 = np.array([[[5.0, 4.0, 4.0, 1.0]]])
    rec, _ = ora.speculation_recall(z2, [[np.array([0, 2])]], np.array([[2]]), np.array([4]))
    assert rec[0, 0] == 1.0
    rec, wt = ora.speculation_recall(z2, [[np.array([], int)]], np.array([[0]]), np.array([4]))
    assert rec[0, 0] == 0.0 and wt[0, 0] == 0.0


def test_captured_fraction_closed_forms():
    q = np.array([[[1.0, -2.0, 3.0, 0.0]]])
    K = np.array([[[[1.0, 1.0, -1.0, 5.0], [2.0, 0.0, 1.0, 1.0]]]])
    L = np.array([2])
    # |q_c K_tc|: token 0 -> 1, 2, 3, 0; token 1 -> 2, 0, 3, 0; total 11
    assert ora.captured_fraction(q, K, L, np.array([[0, 2]]))[0, 0] == pytest.approx(9 / 11, rel=1e-15)
    assert ora.captured_fraction(q, K, L, np.array([[0, 1, 2, 3]]))[0, 0] == 1.0
    assert ora.captured_fraction(q, K, np.array([1]), np.array([[1]]))[0, 0] == pytest.approx(2 / 6, rel=1e-15)


# --- normalized threshold (alpha in units of the head's score spread) ----------------------------
def test_normalized_threshold_closed_form():
    s = np.array([[[0.0, 1.0, 2.0, 3.0]]])
    L = np.array([4])
    sigma = math.sqrt(1.25)  # population std of 0, 1, 2, 3
    for alpha, want in [(0.5, [3]), (1.0, [2, 3]), (2.0, [1, 2, 3]), (3.0, [0, 1, 2, 3])]:
        idx, cnt, _ = ora.select(s, L, alpha, ora.SEL_NORMALIZED)
        assert list(idx[0][0]) == want, (alpha, alpha * sigma)
    # the cap still applies
    idx, cnt, _ = ora.select(s, L, 3.0, ora.SEL_NORMALIZED, cap_frac=0.5)
    assert list(idx[0][0]) == [2, 3]


def test_normalized_threshold_is_scale_and_shift_invariant():
    g = np.random.default_rng(5)
    s = g.standard_normal((2, 3, 40))
    L = np.array([40, 17])
    base, _, _ = ora.select(s, L, 2.0, ora.SEL_NORMALIZED)
    for a, c in [(7.0, 0.0), (0.01, 3.0), (1.0, -50.0)]:
        got, _, _ = ora.select(a * s + c, L, 2.0, ora.SEL_NORMALIZED)
        for b in range(2):
            for h in range(3):
                assert list(got[b][h]) == list(base[b][h])
    # a plain threshold is not scale invariant: scaling the scores down selects more
    plain, _, _ = ora.select(0.01 * s, L, 2.0)
    assert sum(len(x) for r in plain for x in r) > sum(len(x) for r in base for x in r)


def test_normalized_threshold_zero_spread_keeps_all_ties():
    s = np.full((1, 1, 5), 2.5)
    idx, cnt, _ = ora.select(s, np.array([5]), 1.0, ora.SEL_NORMALIZED)
    assert cnt[0, 0] == 5


# --- prefill stage (Steps 1-3) -------------------------------------------------------------------
def test_prefill_keys_are_the_skewed_prompt_keys():
    """X (W_K A) is (X W_K) A: the prefill's keys from the skewed weight equal the skew's own
    rotation of the unskewed prompt keys, up to the two fp16 roundings."""
    w = synth.scaled(synth.WORKLOADS["tiny"], name="pf", heads=2, hidden=256, batch=2, prompt=24)
    H, d, k = w.heads, w.head_dim, w.k
    Xs, Wq, Wk = synth.skew_inputs(w)
    X = synth.hidden_states(w, 0, w.prompt)
    Kraw = (X.astype(np.float64) @ Wk.astype(np.float64)).astype(np.float16).reshape(-1, H, d)
    A, _, Wq_s, Wk_s, K_s = ora.skew(Xs, Wq, Wk, H, d, Kprompt=Kraw)
    Wv = synth.normal_f16(synth.rng(w.name, "Wv", 0), Wq.shape, w.w_std)
    out = ora.prefill_layer(X, Wq_s, Wk_s, Wv, H, d, k, cap=w.prompt)
    got = out["K"].reshape(-1, H, d).astype(np.float64)
    want = K_s.astype(np.float64)
    assert np.abs(got - want).max() <= 4e-3 * np.abs(want).max()
    # the columns come from W~_Q and these keys: the same as the oracle's column choice on the
    # skew's own keys unless the two roundings flip a near tie
    sc = ora.colscores(Wq_s, out["K"], H, d)
    for h in range(H):
        s_sorted = np.sort(sc[h])[::-1]
        if s_sorted[k - 1] - s_sorted[k] > 1e-3 * s_sorted[k - 1]:
            assert np.array_equal(out["cols"][h], ora.choose_columns(Wq_s, K_s, H, d, k)[h])


def test_prefill_pool_placement_is_the_counter_pool_prefill():
    g = np.random.default_rng(3)
    B, N, D, H, d, k, cap = 1, 11, 32, 2, 8, 3, 4
    X = g.standard_normal((B, N, D)).astype(np.float16)
    W = [(g.standard_normal((D, H * d)) * 0.1).astype(np.float16) for _ in range(3)]
    out = ora.prefill_layer(X, W[0], W[1], W[2], H, d, k, cap)
    pool = ora.CounterPool(cap)
    owner = {}
    for t in range(N):
        owner[pool.insert()] = t
    for s_, t in owner.items():
        assert np.array_equal(out["K_pool"][:, :, s_], out["K"][:, t])
        assert np.array_equal(out["V_pool"][:, :, s_], out["V"][:, t])
    assert np.array_equal(out["K_part"], ora.partial_key_cache(out["K_pool"], out["cols"]))


# --- per-layer partial width from the spectrum ---------------------------------------------------
def test_energy_k_closed_forms():
    flat = np.ones((3, 128))
    for e in (0.1, 0.3, 0.5, 0.9, 1.0):
        assert ora.energy_k(flat, e) == math.ceil(e * 128 - 1e-9)
    spike = np.zeros((2, 64))
    spike[:, 0] = 5.0
    assert ora.energy_k(spike, 0.99) == 1
    # sigma_i^2 = 2^-i: captured fraction after k is (1 - 2^-k) / (1 - 2^-d)
    geo = np.sqrt(2.0 ** -np.arange(32))[None, :]
    assert ora.energy_k(geo, 0.9) == 4 and ora.energy_k(geo, 0.99) == 7
    # non-decreasing in the energy target; the mean over heads
    g = np.random.default_rng(2)
    s = np.sort(g.random((4, 128)), axis=1)[:, ::-1]
    ks = [ora.energy_k(s, e) for e in np.linspace(0.05, 1.0, 20)]
    assert ks == sorted(ks)
    two = np.stack([np.ones(10), np.r_[1.0, np.zeros(9)]])  # head means 0.1 k and 1.0
    assert ora.energy_k(two, 0.6) == 2  # (0.2 + 1) / 2 = 0.6


def test_skew_spectrum_is_the_svd_of_the_sample_queries():
    w = synth.scaled(synth.WORKLOADS["tiny"], name="spec", heads=2, hidden=256)
    Xs, Wq, Wk = synth.skew_inputs(w)
    A, sig, _, _, _ = ora.skew(Xs, Wq, Wk, w.heads, w.head_dim)
    Q = Xs.astype(np.float64) @ Wq.astype(np.float64)
    for h in range(w.heads):
        Qh = Q[:, h * w.head_dim:(h + 1) * w.head_dim]
        # singular values: the column norms of Q_h A_h, descending
        assert np.allclose(np.linalg.norm(Qh @ A[h], axis=0), sig[h], rtol=1e-10)
        assert np.all(np.diff(sig[h]) <= 0)


def test_prefill_rope_keys_are_the_skews_rotated_prompt_keys():
    """RoPE prefill: RoPE_t(X W_K) A equals what the skew produces from the post-RoPE prompt
    keys (ora.skew with Kprompt), and the partial key of slot t scored with the partial RoPE
    query equals the full rotated dot product restricted to the columns (the identity the
    decode stage relies on)."""
    w = synth.scaled(synth.WORKLOADS["llama-2-7b"], name="pfr", heads=2, hidden=256, batch=1, prompt=40,
                     head_dim=64, sample_rows=256)
    H, d, k, th = w.heads, w.head_dim, w.k, w.rope_theta
    Xs, Wq, Wk = synth.skew_inputs(w)
    X = synth.hidden_states(w, 0, w.prompt)
    Kraw = (X.astype(np.float64) @ Wk.astype(np.float64)).astype(np.float16).reshape(1, -1, H, d)
    Kpost = ora.rope(Kraw.astype(np.float64), np.arange(w.prompt)[None, :, None], th).reshape(-1, H, d)
    A, _, Wq_s, _, K_s = ora.skew(Xs, Wq, Wk, H, d, rope_theta=th, Kprompt=Kpost)
    Wv = synth.normal_f16(synth.rng(w.name, "Wv", 0), Wq.shape, w.w_std)
    o = ora.prefill_layer_rope(X, Wq_s, Wk, Wv, A, th, H, d, k, cap=w.prompt)
    assert np.abs(o["K"].reshape(-1, H, d).astype(np.float64) - K_s.astype(np.float64)).max() <= \
        2e-3 * np.abs(K_s.astype(np.float64)).max()
    # decode identity: q A[:, S] . K~[:, S] with the rotated query
    x = synth.normal_f16(synth.rng(w.name, "xq", 0), (1, w.hidden), 1.0)
    pos = np.array([w.prompt])
    qp = ora.partial_query_rope(x, Wq, A, o["cols"], pos, th)  # [1, H, k]
    for h in range(H):
        kp = o["K_part"][0, h].astype(np.float64)  # [k, cap]
        assert np.allclose(qp[0, h] @ kp, qp[0, h] @ o["K"][0, :, h][:, o["cols"][h]].T.astype(np.float64))
        assert np.array_equal(o["A_cols"][h], A[h][:, o["cols"][h]])


# --- Prefill Step 3 (extract the partial weight): a hand-written two-head case -------------
def test_partial_weight_hand_written_two_heads():
    """W~_Q is 3 x 8 (D = 3, H = 2 heads of d = 4); head 0 keeps columns {1, 3}, head 1 keeps
    {0, 2}.  Entry (r, c) of W~_Q is 10 * r + c, so every column's origin can be read off its
    values.  Head 1's columns sit at offset h * d = 4 in W~_Q: columns 4 and 6, not 0 and 2."""
    W = np.array([[10 * r + c for c in range(8)] for r in range(3)], dtype=np.float16)
    cols = np.array([[1, 3], [0, 2]], dtype=np.int32)
    got = ora.partial_weight(W, cols, H=2, d=4)
    want = np.array([[1, 3, 4, 6],
                     [11, 13, 14, 16],
                     [21, 23, 24, 26]], dtype=np.float16)
    assert got.shape == (3, 4) and got.dtype == np.float16
    assert np.array_equal(got, want)
    # the partial query through it is x . W~_Q restricted to those columns, by hand
    x = np.array([[1.0, -2.0, 0.5]], dtype=np.float16)
    q = ora.partial_query(x, got, H=2, k=2)
    assert q.shape == (1, 2, 2)
    assert np.array_equal(q[0], [[1 - 22 + 10.5, 3 - 26 + 11.5], [4 - 28 + 12.0, 6 - 32 + 13.0]])


# --- Speculation fidelity: real logits of a two-token case --------------------------------
def test_real_scores_two_token_closed_form():
    """q = (1, 2), keys (3, 4) and (-1, 0.5), scale 0.5: logits 0.5 * 11 = 5.5 and
    0.5 * 0 = 0; the third slot is past L and must read -inf.  A second sequence with L = 1
    checks that L is taken per sequence."""
    q = np.array([[[1.0, 2.0]], [[2.0, 0.0]]])           # [B=2, H=1, d=2]
    K = np.array([[[[3.0, 4.0], [-1.0, 0.5], [7.0, 7.0]]],
                  [[[1.0, 9.0], [5.0, 5.0], [0.0, 0.0]]]])  # [B=2, H=1, T=3, d=2]
    z = ora.real_scores(q, K, np.array([2, 1]), 0.5)
    assert z.shape == (2, 1, 3)
    assert z[0, 0, 0] == 5.5 and z[0, 0, 1] == 0.0 and np.isneginf(z[0, 0, 2])
    assert z[1, 0, 0] == 1.0 and np.isneginf(z[1, 0, 1]) and np.isneginf(z[1, 0, 2])
