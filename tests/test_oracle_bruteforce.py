"""P4 and P13: the oracle against scalar-loop brute force on tiny inputs, and the pool rules.

The brute-force versions below are written as explicit Python loops over single numbers,
independently of the vectorised oracle, on inputs small enough (L <= 16, d <= 8) to check
every entry.
"""
import math

import numpy as np
import pytest

from oracle import infinigen as ora


def _bf_scores(qp, Kpart, L, scale):
    B, H, k = qp.shape
    out = {}
    for b in range(B):
        for h in range(H):
            for t in range(L[b]):
                acc = 0.0
                for c in range(k):
                    acc += float(qp[b, h, c]) * float(Kpart[b, h, c, t])
                out[(b, h, t)] = float(np.float32(scale)) * acc
    return out


def _bf_threshold(vals, alpha):
    m = max(vals)
    return [t for t, v in enumerate(vals) if m - v < alpha]


def _bf_topn(vals, n):
    pairs = sorted([(-v, t) for t, v in enumerate(vals)])
    return sorted(t for _, t in pairs[:n])


def _bf_attend(q, rows_k, rows_v, scale):
    z = []
    for r in rows_k:
        acc = 0.0
        for c in range(len(q)):
            acc += float(q[c]) * float(r[c])
        z.append(float(np.float32(scale)) * acc)
    m = max(z)
    e = [math.exp(v - m) for v in z]
    tot = sum(e)
    out = [0.0] * len(rows_v[0])
    for w, r in zip(e, rows_v):
        for c in range(len(r)):
            out[c] += (w / tot) * float(r[c])
    return out


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("policy,cap", [(ora.SEL_THRESHOLD, 1.0), (ora.SEL_THRESHOLD, 0.25),
                                        (ora.SEL_HEAD_AVG, 1.0), (ora.SEL_HEAD_AVG, 0.3)])
def test_p4_layer_step_brute_force(seed, policy, cap):
    g = np.random.default_rng(seed)
    B, H, d, D, k = 2, 3, 8, 12, 3
    Lcap = 16
    L = np.array([16, int(g.integers(1, 16))])
    x = (g.standard_normal((B, D))).astype(np.float16)
    Wqp = (g.standard_normal((D, H * k)) * 0.5).astype(np.float16)
    Kpool = (g.standard_normal((B, H, Lcap, d))).astype(np.float16)
    Vpool = (g.standard_normal((B, H, Lcap, d))).astype(np.float16)
    cols = np.array([np.sort(g.permutation(d)[:k]) for _ in range(H)])
    Kpart = ora.partial_key_cache(Kpool, cols)
    q = (g.standard_normal((B, H, d))).astype(np.float16)
    kn = (g.standard_normal((B, H, d))).astype(np.float16)
    vn = (g.standard_normal((B, H, d))).astype(np.float16)
    scale, alpha = 0.6, 1.3
    r = ora.decode_layer_step(x, Wqp, Kpart, L, q, Kpool, Vpool, H=H, k=k, scale=scale, alpha=alpha,
                              policy=policy, cap_frac=cap, k_new=kn, v_new=vn)
    # partial query, scalar loops
    qp = np.zeros((B, H, k))
    for b in range(B):
        for j in range(H * k):
            acc = 0.0
            for i in range(D):
                acc += float(x[b, i]) * float(Wqp[i, j])
            qp[b, j // k, j % k] = acc
    assert np.allclose(r["q_part"], qp, rtol=1e-12, atol=1e-12)
    # partial key rows must be the chosen columns of the full keys
    for b in range(B):
        for h in range(H):
            for c in range(k):
                for t in range(Lcap):
                    assert Kpart[b, h, c, t] == Kpool[b, h, t, cols[h, c]]
    bs = _bf_scores(qp, Kpart, L, scale)
    for (b, h, t), v in bs.items():
        assert abs(r["scores"][b, h, t] - v) <= 1e-12 * max(1.0, abs(v))
    for b in range(B):
        assert np.all(np.isneginf(r["scores"][b, :, L[b]:]))
    # selection
    for b in range(B):
        capn = int(math.floor(float(np.float32(cap)) * L[b] + 0.5)) if cap < 1 else int(L[b])
        sel = {}
        for h in range(H):
            vals = [bs[(b, h, t)] for t in range(L[b])]
            s = _bf_threshold(vals, alpha)
            if policy == ora.SEL_THRESHOLD and len(s) > capn:
                s = _bf_topn(vals, capn)
            sel[h] = s
        if policy == ora.SEL_HEAD_AVG:
            mean = sum(len(v) for v in sel.values()) / H
            cbar = min(max(1, int(math.floor(mean + 0.5))), capn)
            for h in range(H):
                sel[h] = _bf_topn([bs[(b, h, t)] for t in range(L[b])], cbar)
        for h in range(H):
            assert list(r["idx"][b][h]) == sel[h]
            assert r["cnt"][b, h] == len(sel[h])
        for t in range(Lcap):
            assert r["used"][b, t] == int(any(t in sel[h] for h in range(H)))
        # attention over the selected rows plus the current token
        for h in range(H):
            rk = [Kpool[b, h, t] for t in sel[h]] + [kn[b, h]]
            rv = [Vpool[b, h, t] for t in sel[h]] + [vn[b, h]]
            o = _bf_attend(q[b, h], rk, rv, scale)
            assert np.allclose(r["out"][b, h], o, rtol=0, atol=1e-12)


def test_select_ignores_nan_and_handles_empty():
    s = np.array([[[np.nan, 1.0, 0.5, np.nan], [np.nan] * 4]])
    idx, cnt, used = ora.select(s, [4], 0.75)
    assert list(idx[0][0]) == [1, 2] and cnt[0, 1] == 0
    idx, cnt, used = ora.select(np.zeros((1, 2, 8)), [0], 4.0)
    assert cnt.sum() == 0 and used.sum() == 0


def test_gather_copies_rows_exactly():
    g = np.random.default_rng(3)
    Kp = g.standard_normal((2, 2, 9, 4)).astype(np.float16)
    Vp = g.standard_normal((2, 2, 9, 4)).astype(np.float16)
    idx = [[np.array([0, 8]), np.array([3])], [np.array([]), np.array([1, 2, 5])]]
    Kg, Vg = ora.gather(Kp, Vp, idx, 9)
    for b in range(2):
        for h in range(2):
            for j, t in enumerate(idx[b][h]):
                assert Kg[b, h, j].tobytes() == Kp[b, h, int(t)].tobytes()
                assert Vg[b, h, j].tobytes() == Vp[b, h, int(t)].tobytes()


# --- P13: pool rules -------------------------------------------------------------------------
def test_p13_pool_no_eviction_when_capacity_suffices():
    p = ora.CounterPool(10)
    assert [p.evict(None) for _ in range(10)] == list(range(10))


def test_p13_pool_zero_counters_is_fifo():
    p = ora.CounterPool(4)
    slots = [p.evict(None) for _ in range(11)]
    assert slots == [0, 1, 2, 3, 0, 1, 2, 3, 0, 1, 2]


def test_p13_pool_evicts_smallest_counter_then_oldest():
    p = ora.CounterPool(4)
    for _ in range(4):
        p.insert()
    # slot 2 used twice, slot 0 once, slots 1 and 3 never
    p.update([1, 0, 1, 0])
    p.update([0, 0, 1, 0])
    assert p.insert() == 1          # counters 1,0,2,0 -> smallest 0, oldest of {1, 3} is 1
    assert p.insert() == 3          # slot 1 is new (counter 0, newest) -> slot 3 is older
    assert p.counter.tolist() == [1, 0, 2, 0]


def test_p13_pool_halving_keeps_order():
    p = ora.CounterPool(3)
    for _ in range(3):
        p.insert()
    for i in range(255):
        p.update([1, 1 if i % 2 == 0 else 0, 0])
    # slot 0 reached 255 and everything was halved once
    assert p.counter.tolist() == [127, 64, 0]
    assert p.counter[0] > p.counter[1] > p.counter[2]
    assert p.insert() == 2


def test_p13_pool_brute_force_against_slot_history():
    g = np.random.default_rng(9)
    cap, steps = 6, 60
    p = ora.CounterPool(cap)
    owner = {}
    cnt = [0] * cap
    seqs = [0] * cap
    filled = 0
    nxt = 0
    for t in range(steps):
        used = (g.random(cap) < 0.3).astype(np.uint8)
        got = p.evict(used if t else None)
        # brute force of the same rules
        if t:
            for s in range(filled):
                if used[s]:
                    cnt[s] = min(255, cnt[s] + 1)
            if filled and max(cnt[:filled]) >= 255:
                cnt = [c >> 1 for c in cnt]
        if filled < cap:
            want = filled
            filled += 1
        else:
            want = min(range(cap), key=lambda s: (cnt[s], seqs[s], s))
        cnt[want] = 0
        seqs[want] = nxt
        nxt += 1
        owner[want] = t
        assert got == want


# --- pool policies of Table 2: FIFO and LRU ---------------------------------------------------
def test_fifo_pool_cycles_the_slots_and_keeps_the_newest():
    p = ora.FifoPool(5)
    slots = [p.evict(np.ones(5, np.uint8)) for _ in range(17)]
    # free slots in order, then the oldest entry: slot t mod 5 whatever the use
    assert slots == [t % 5 for t in range(17)]
    # the resident tokens are the last 5 inserted (token numbers 12..16)
    assert sorted(p.seq.tolist()) == list(range(12, 17))


def _lru_list_model(cap, steps, use_prob, seed):
    """Textbook LRU with an ordered list (least recent first): a use moves the entry to the
    most-recent end, an insertion appends there, the victim is the first entry.  Entries used
    in the same update move in insertion order, so the newest of them ends most recent."""
    g = np.random.default_rng(seed)
    order = []          # token numbers, least recent first
    slot_of = {}        # token -> slot
    free = list(range(cap))
    out = []
    for t in range(steps):
        used = (g.random(cap) < use_prob).astype(np.uint8)
        if t:
            tokens_used = sorted(tok for tok, s in slot_of.items() if used[s])
            for tok in tokens_used:
                order.remove(tok)
                order.append(tok)
        if free:
            s = free.pop(0)
        else:
            victim = order.pop(0)
            s = slot_of.pop(victim)
        slot_of[t] = s
        order.append(t)
        out.append((s, used if t else None))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("cap,use_prob", [(4, 0.3), (7, 0.1), (9, 0.6)])
def test_lru_pool_equals_the_textbook_list_lru(seed, cap, use_prob):
    hist = _lru_list_model(cap, 80, use_prob, seed)
    p = ora.LruPool(cap)
    for want, used in hist:
        assert p.evict(used) == want


def test_lru_keeps_a_hot_entry_that_fifo_drops():
    lru, fifo = ora.LruPool(3), ora.FifoPool(3)
    for _ in range(3):
        lru.insert(), fifo.insert()
    # slot 0 (the oldest token) is used at every step
    for _ in range(6):
        u = np.array([1, 0, 0], np.uint8)
        s_l, s_f = lru.evict(u), fifo.evict(u)
        assert s_l != 0
    assert 0 in lru.seq.tolist() and 0 not in fifo.seq.tolist()


def test_make_pool_dispatch():
    assert isinstance(ora.make_pool(3, ora.POOL_COUNTER), ora.CounterPool)
    assert isinstance(ora.make_pool(3, ora.POOL_FIFO), ora.FifoPool)
    assert isinstance(ora.make_pool(3, ora.POOL_LRU), ora.LruPool)


def test_eviction_misses_closed_form():
    # one head, tokens 0..3 selected with scores 0, -1, -2, -3; tokens 1 and 3 are gone
    scores = np.array([[[0.0, -1.0, -2.0, -3.0]]])
    idx = [[np.array([0, 1, 2, 3])]]
    cnt = np.array([[4]])
    resident = np.array([[1, 0, 1, 0]], bool)
    n, mass = ora.eviction_misses(scores, idx, cnt, resident)
    e = np.exp(-np.arange(4.0))
    assert n[0, 0] == 2
    assert mass[0, 0] == pytest.approx((e[1] + e[3]) / e.sum(), rel=1e-15)
    # nothing evicted, or nothing selected: no misses
    n, mass = ora.eviction_misses(scores, idx, cnt, np.ones((1, 4), bool))
    assert n[0, 0] == 0 and mass[0, 0] == 0.0
    n, mass = ora.eviction_misses(scores, idx, np.array([[0]]), resident)
    assert n[0, 0] == 0 and mass[0, 0] == 0.0


# --- FP8 (e4m3) pool rows -----------------------------------------------------------------------
def test_e4m3_known_codes_and_round_trip():
    assert ora.e4m3_encode(0.0) == 0x00 and ora.e4m3_encode(-0.0) == 0x80
    assert ora.e4m3_encode(1.0) == 0x38 and ora.e4m3_encode(-1.0) == 0xB8
    assert ora.e4m3_encode(448.0) == 0x7E and ora.e4m3_encode(1e6) == 0x7E and ora.e4m3_encode(-500) == 0xFE
    assert ora.e4m3_encode(2.0 ** -9) == 0x01           # smallest subnormal
    assert ora.e4m3_encode(2.0 ** -10) == 0x00          # halfway to 0: ties to even
    assert ora.e4m3_encode(3 * 2.0 ** -10) == 0x02      # halfway between 1 and 2 (x 2^-9): even
    assert ora.e4m3_encode(1.0625) == 0x38              # halfway between 1 and 1.125: even (1)
    assert ora.e4m3_encode(1.1875) == 0x3A              # halfway between 1.125 and 1.25: even (1.25)
    assert ora.e4m3_decode(0x7E) == 448.0 and math.isnan(ora.e4m3_decode(0x7F))
    # every finite code decodes and encodes back to itself (-0 to 0x80)
    for c in range(256):
        v = ora.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert ora.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_is_the_nearest_value():
    finite = sorted({ora.e4m3_decode(c) for c in range(256)} - {float("nan")})
    finite = [v for v in finite if not math.isnan(v)]
    g = np.random.default_rng(0)
    for x in np.concatenate([g.standard_normal(2000) * 30, g.standard_normal(500) * 0.01]):
        got = ora.e4m3_decode(ora.e4m3_encode(x))
        best = min(abs(v - x) for v in finite)
        assert abs(got - x) == best


def test_fp8_rows_scale_and_error_bound():
    g = np.random.default_rng(1)
    X = (g.standard_normal((3, 5, 64)) * 2).astype(np.float16)
    X[0, 0] = 0
    codes, scales = ora.fp8_quantize_rows(X)
    assert scales[0, 0] == 0 and not codes[0, 0].any()
    Y = ora.fp8_dequantize_rows(codes, scales)
    Xf, Yf = X.astype(np.float32), Y.astype(np.float32)
    amax = np.abs(Xf).max(-1, keepdims=True)
    # the largest element maps to +-448 exactly; e4m3 keeps 3 mantissa bits: relative error
    # <= 2^-4 for normal values, absolute <= 2^-10 * scale below the normal range
    assert np.all(np.abs(Yf - Xf) <= np.maximum(np.abs(Xf) * 2.0 ** -4, amax / 448 * 2.0 ** -9) + 1e-3 * amax + 1e-6)
    r = np.unravel_index(np.abs(Xf[1, 2]).argmax(), (64,))
    assert ora.e4m3_decode(codes[1, 2][r]) in (448.0, -448.0)


# --- INT4 pool rows -----------------------------------------------------------------------------
def test_int4_rows_exact_on_integer_rows_and_zero_rows():
    # amax = 7: the reciprocal 7/7 and the scale 7/7 are exactly 1, so integer rows in [-7, 7]
    # are their own codes and decode back exactly
    g = np.random.default_rng(2)
    X = g.integers(-7, 8, size=(4, 32)).astype(np.float16)
    X[:, 0] = 7
    X[3] = 0
    codes, scales = ora.int4_quantize_rows(X)
    assert np.array_equal(scales[:3], np.ones(3, np.float32)) and scales[3] == 0
    assert np.array_equal(codes[:3].astype(np.int64), X[:3].astype(np.int64)) and not codes[3].any()
    assert np.array_equal(ora.int4_dequantize_rows(codes, scales), X)


def test_int4_rows_rounding_symmetry_and_error_bound():
    g = np.random.default_rng(3)
    X = (g.standard_normal((6, 128)) * g.uniform(0.01, 50, (6, 1))).astype(np.float16)
    codes, scales = ora.int4_quantize_rows(X)
    codes_neg, scales_neg = ora.int4_quantize_rows(-X)
    assert np.array_equal(scales, scales_neg) and np.array_equal(codes_neg, -codes)  # ties to even: symmetric
    assert codes.min() >= -7 and codes.max() <= 7
    Xf = X.astype(np.float64)
    amax = np.abs(Xf).max(-1)
    for r in range(6):  # the largest element maps to +-7
        assert abs(int(codes[r, np.abs(Xf[r]).argmax()])) == 7
    # brute force: each code is the integer nearest x / scale (within the float32 rounding of
    # the reciprocal), so the reconstruction is within half a step
    step = amax / 7
    Y = ora.int4_dequantize_rows(codes, scales).astype(np.float64)
    assert np.all(np.abs(Y - Xf) <= step[:, None] * (0.5 + 1e-5) + np.abs(Y) * 2.0 ** -11)
    for r in range(6):
        for i in range(128):
            cand = [c for c in range(-7, 8)]
            dist = [abs(c * step[r] - Xf[r, i]) for c in cand]
            best = min(dist)
            assert abs(int(codes[r, i]) * step[r] - Xf[r, i]) <= best + 1e-6 * step[r]


def test_int4_packing_nibble_order():
    codes = np.array([[1, -1, 7, -7, 0, -8 + 1, 3, -2]], dtype=np.int8)
    packed = ora.int4_pack(codes)
    # written out by hand: byte j = (code[2j] & 15) | (code[2j+1] & 15) << 4
    want = []
    for j in range(4):
        a, b = int(codes[0, 2 * j]), int(codes[0, 2 * j + 1])
        want.append((a & 15) | ((b & 15) << 4))
    assert packed.tolist() == [want] == [[0xF1, 0x97, 0x90, 0xE3]]
    g = np.random.default_rng(4)
    c = g.integers(-7, 8, size=(5, 64)).astype(np.int8)
    assert np.array_equal(ora.int4_unpack(ora.int4_pack(c)), c)
