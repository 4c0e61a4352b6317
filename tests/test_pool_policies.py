"""The native pool manager's three victim policies (counter, FIFO, LRU; section 3.4, pool
management, Table 2) against the oracle's pool models, slot for slot.

The manager is created without storage (IG_POOL_NO_STORAGE), so these tests need no GPU: the
victim choice is host code.  Every placement must equal the oracle's, and so must the slot ->
token map and the eviction count."""
import numpy as np
import pytest

from oracle import infinigen as ora


@pytest.fixture(scope="module")
def ig():
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig as mod

    return mod


POLICIES = {"counter": 0, "fifo": 1, "lru": 2}


@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("cap,prompt,use_prob", [(8, 5, 0.3), (8, 12, 0.2), (16, 30, 0.05), (5, 5, 0.9)])
def test_native_policy_matches_oracle_slot_for_slot(ig, policy, cap, prompt, use_prob):
    pol = POLICIES[policy]
    layers, B, steps = 2, 3, 120
    pool = ig.ig_pool_create_ex(layers, B, 0, 0, cap, pol, ig.IG_POOL_NO_STORAGE)
    try:
        models = [[ora.make_pool(cap, pol) for _ in range(B)] for _ in range(layers)]
        want = [m.insert() for row in models for m in row for _ in range(prompt)]
        got = np.zeros(prompt, np.int32)
        ig.ig_pool_prefill(pool, prompt, got)
        assert got.tolist() == want[:prompt]
        g = np.random.default_rng(cap * 100 + prompt)
        Lcap = cap + 3
        for t in range(steps):
            used = (g.random((layers, B, Lcap)) < use_prob).astype(np.uint8)
            slots = np.zeros((layers, B), np.int32)
            ig.ig_pool_step(pool, used if t else None, Lcap, slots)
            for l in range(layers):
                for b in range(B):
                    assert slots[l, b] == models[l][b].evict(used[l, b] if t else None), (t, l, b)
        for l in range(layers):
            for b in range(B):
                m = models[l][b]
                tok = np.zeros(cap, np.int32)
                ig.ig_pool_slot_tokens(pool, l, b, tok)
                assert tok.tolist() == m.seq.tolist()
                assert ig.ig_pool_evictions(pool, l, b) == max(0, prompt + steps - cap)
    finally:
        ig.ig_pool_destroy(pool)


@pytest.mark.parametrize("policy", list(POLICIES))
def test_update_then_evict_equals_step(ig, policy):
    """ig_pool_update + ig_pool_evict(NULL) is the same action as ig_pool_evict(used)."""
    pol, cap = POLICIES[policy], 6
    a = ig.ig_pool_create_ex(1, 1, 0, 0, cap, pol, ig.IG_POOL_NO_STORAGE)
    b = ig.ig_pool_create_ex(1, 1, 0, 0, cap, pol, ig.IG_POOL_NO_STORAGE)
    try:
        g = np.random.default_rng(4)
        for t in range(40):
            used = (g.random(cap) < 0.4).astype(np.uint8)
            sa, _ = ig.ig_pool_evict(a, 0, 0, used if t else None)
            if t:
                ig.ig_pool_update(b, 0, 0, used)
            sb, _ = ig.ig_pool_evict(b, 0, 0, None)
            assert sa == sb
    finally:
        ig.ig_pool_destroy(a)
        ig.ig_pool_destroy(b)


def test_free_slots_report_no_token_and_storage_calls_are_refused(ig):
    pool = ig.ig_pool_create_ex(1, 2, 0, 0, 4, ig.IG_POOL_LRU, ig.IG_POOL_NO_STORAGE)
    try:
        ig.ig_pool_evict(pool, 0, 1, None)
        tok = np.zeros(4, np.int32)
        ig.ig_pool_slot_tokens(pool, 0, 1, tok)
        assert tok.tolist() == [0, -1, -1, -1]
        with pytest.raises(ig.IGError) as e:
            ig.ig_pool_kv(pool, 0)
        assert e.value.status == ig.IG_ERR_INVALID and "storage" in str(e.value)
    finally:
        ig.ig_pool_destroy(pool)
    with pytest.raises(ig.IGError):
        ig.ig_pool_create_ex(1, 1, 0, 0, 4, 7, ig.IG_POOL_NO_STORAGE)
