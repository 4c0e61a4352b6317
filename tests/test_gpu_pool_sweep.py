"""Pool policies under real selection traffic, and the eviction-miss diagnostic, on the GPU.

* ``ig_eviction_misses`` against the oracle's count and mass on the same selections;
* the memory-limit sweep loop (``pool_sweep.run``): with no limit it misses nothing; under a
  limit, every placement the native manager makes from the GPU's own "used" flags equals the
  oracle pool model's for the same policy (counter, FIFO, LRU).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from gpu_util import dev, empty, host  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig, pool_sweep

    return ig, pool_sweep


@pytest.mark.parametrize("B,H,Lcap", [(1, 1, 8), (2, 3, 40), (4, 8, 1032)])
def test_eviction_misses_matches_oracle(mods, B, H, Lcap):
    ig, _ = mods
    g = np.random.default_rng(B * 100 + Lcap)
    # scores on a 1/64 grid (exact in fp32), selection by the oracle, random residency
    scores = (g.integers(-400, 400, size=(B, H, Lcap)) / 64.0).astype(np.float32)
    L = np.full(B, Lcap, np.int32)
    L[0] = max(1, Lcap // 3)
    oi, oc, _ = ora.select(scores, L, 2.0)
    oc = oc.astype(np.int32)
    oc[0, 0] = 0  # a head with nothing selected
    idx = np.zeros((B, H, Lcap), np.int32)
    for b in range(B):
        for h in range(H):
            idx[b, h, :oc[b, h]] = oi[b][h][:oc[b, h]]
    resident = (g.random((B, Lcap)) < 0.6).astype(np.uint8)
    resident[-1] = 1  # one sequence fully resident
    n = empty((B, H), torch.int32)
    m = empty((B, H), torch.float32)
    ig.ig_eviction_misses(None, B, H, Lcap, dev(scores), dev(idx), dev(oc), dev(resident), n, m)
    ig.ig_check()
    sel = [[idx[b, h, :oc[b, h]] for h in range(H)] for b in range(B)]
    wn, wm = ora.eviction_misses(scores, sel, oc, resident.astype(bool))
    assert np.array_equal(host(n), wn)
    assert np.allclose(host(m), wm, rtol=1e-5, atol=1e-7)
    assert np.all(host(n)[-1] == 0) and host(n)[0, 0] == 0 and host(m)[0, 0] == 0.0


def _tiny(pool_sweep):
    return pool_sweep.sweep_workload(layers=3, batch=2, heads=4, hidden=7168, prompt=96, gen=24)


def test_sweep_without_limit_misses_nothing(mods):
    ig, pool_sweep = mods
    r = pool_sweep.run(_tiny(pool_sweep), 1.0, ig.IG_POOL_COUNTER)
    assert r["misses"] == 0 and r["evictions"] == 0 and r["selected"] > 0 and r["miss_mass"] == 0.0


@pytest.mark.parametrize("policy", [0, 1, 2])
def test_sweep_placements_equal_the_oracle_policy(mods, policy):
    ig, pool_sweep = mods
    w = _tiny(pool_sweep)
    r = pool_sweep.run(w, 0.5, policy, record=True)
    T = w.prompt + w.gen
    cap = int(np.floor(0.5 * T + 0.5))
    assert r["cap"] == cap and r["evictions"] == (w.layers - 1) * w.batch * (T - cap)
    assert 0 <= r["misses"] <= r["selected"]
    models = [[ora.make_pool(cap, policy) for _ in range(w.batch)] for _ in range(w.layers)]
    for row in models:
        for m in row:
            for _ in range(w.prompt):
                m.insert()
    for step in r["history"]:
        used = step["used"]
        for l in range(1, w.layers):
            for b in range(w.batch):
                want = models[l][b].evict(used[l, b] if used is not None else None)
                assert step["slots"][l, b] == want
