"""ig_skew_weights (host one-sided Jacobi SVD, rotation, column choice) against the oracle.

The library call runs on the host, but it is a compute call of the library, so these tests sit
with the GPU suite.  Comparisons: the skew matrices A (both sides fix column signs the same
way) within 1e-5; W~_Q, W~_K and the skewed prompt keys as fp16 bit patterns, allowing a few
one-ulp differences where the float64 products of the two sides straddle an fp16 rounding
boundary; the chosen columns exactly, except columns whose oracle score is within 1e-6
(relative) of the k-th best, where the choice is a near tie (parity unpinned there).
"""
import numpy as np
import pytest

from oracle import infinigen as ora
from speculative_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig():
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig as mod

    return mod


def _f16_close(a, b, max_frac=1e-3):
    a16, b16 = a.view(np.uint16).astype(np.int32), b.view(np.uint16).astype(np.int32)
    diff = a16 != b16
    if diff.any():
        # only one-ulp flips (same sign, neighbouring bit patterns)
        assert np.abs(a16[diff] - b16[diff]).max() == 1
    assert diff.mean() <= max_frac, diff.mean()


CASES = {
    "tiny": (synth.WORKLOADS["tiny"], 0.0, 256, 1),
    "tiny-rope": (synth.scaled(synth.WORKLOADS["tiny"], name="tiny-rope", rope_theta=10000.0), 10000.0, 256, 1),
    "opt-6.7b-layer": (synth.WORKLOADS["opt-6.7b"], 0.0, 96, 1),
    "llama-2-7b-layer": (synth.WORKLOADS["llama-2-7b"], 10000.0, 96, 1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_skew_matches_oracle(ig, name):
    w, theta, n_keys, batch = CASES[name]
    Xs, Wq, Wk = synth.skew_inputs(w, layer=1)
    Kp = synth.prompt_keys_unskewed(w, layer=1, tokens=n_keys)[:batch].reshape(-1, w.heads, w.head_dim)
    H, d, D = w.heads, w.head_dim, w.hidden
    k = ora.partial_columns(w.ratio, d)
    A = np.zeros((H, d, d), dtype=np.float32)
    Wq_s = np.zeros((D, H * d), dtype=np.float16)
    Wk_s = np.zeros((D, H * d), dtype=np.float16)
    Kp_s = np.zeros_like(Kp)
    cols = np.zeros((H, k), dtype=np.int32)
    got_k = ig.ig_skew_weights(D, H, d, w.ratio, theta, Xs, Xs.shape[0], Wq, Wk, Kp, Kp.shape[0], A, Wq_s, Wk_s,
                               Kp_s, cols)
    assert got_k == k
    A_o, _, Wq_o, Wk_o, Kp_o = ora.skew(Xs, Wq, Wk, H, d, rope_theta=theta, Kprompt=Kp)
    assert np.abs(A.astype(np.float64) - A_o).max() <= 1e-5
    _f16_close(Wq_s, Wq_o)
    _f16_close(Wk_s, Wk_o)
    _f16_close(Kp_s, Kp_o)
    cols_o = ora.choose_columns(Wq_o, Kp_o, H, d, k)
    score = ora.colscores(Wq_o, Kp_o, H, d)
    for h in range(H):
        kth = np.sort(score[h])[::-1][k - 1]
        tie = set(np.nonzero(np.abs(score[h] - kth) <= 1e-6 * kth)[0].tolist())
        assert set(cols[h].tolist()) - tie == set(cols_o[h].tolist()) - tie
        assert list(cols[h]) == sorted(cols[h])


def test_skew_rejects_bad_arguments(ig):
    z = np.zeros(64, dtype=np.float16)
    with pytest.raises(ig.IGError) as e:
        ig.ig_skew_weights(8, 1, 8, 1.5, 0.0, z, 8, z, z, None, 0, np.zeros(64, np.float32), None, None, None,
                           np.zeros(8, np.int32))
    assert e.value.status == ig.IG_ERR_INVALID
    with pytest.raises(ig.IGError):
        ig.ig_skew_weights(8, 1, 7, 0.5, 10000.0, z, 8, z, z, None, 0, np.zeros(64, np.float32), None, None,
                           None, np.zeros(8, np.int32))


def test_spectrum_and_energy_k_match_oracle():
    """ig_skew_spectrum equals the oracle's singular values; ig_ratio_from_spectrum equals the
    oracle's energy_k on the same spectrum, at several targets."""
    from oracle import infinigen as ora
    from speculative_kv_cache_gb300 import ig, synth

    w = synth.scaled(synth.WORKLOADS["tiny"], name="spec2", heads=3, hidden=256)
    H, d = w.heads, w.head_dim
    Xs, Wq, Wk = synth.skew_inputs(w)
    Wq_s, _ = synth.structured_qk_weights(w, 0, 0.7)
    for W in (Wq, Wq_s):
        sig = np.zeros((H, d), np.float32)
        ig.ig_skew_spectrum(w.hidden, H, d, 0.0, Xs, Xs.shape[0], W, sig)
        _, want, _, _, _ = ora.skew(Xs, W, Wk, H, d)
        assert np.allclose(sig, want, rtol=1e-5, atol=1e-6 * want.max())
        for e in (0.3, 0.5, 0.8, 0.95):
            assert ig.ig_ratio_from_spectrum(H, d, sig, e) == ora.energy_k(sig.astype(np.float64), e)
