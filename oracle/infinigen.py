"""Plain CPU oracle for InfiniGen's per-layer decode-step speculation and sparse attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links this module;
only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.
It shares no code with the CUDA library: it is NumPy in float64, written step by step from
the method's description, with no blocking, fusion or reordering beyond what that
description states.

Source: "InfiniGen: Efficient Generative Inference of Large Language Models with Dynamic KV
Cache Management" (Lee, Lee, Seo, Sim; OSDI 2024, arXiv 2406.19707), as retold by the
paper-graph summary page of that paper, section 3.4 ("Detailed, Sentence-Based Technical
Breakdown").  Every function below names the part of that section it follows.

Readings taken where the page is silent or garbled (each is listed in the design notes):
  * score scale: speculated and real logits carry the 1/sqrt(d) factor, passed in as
    ``scale`` (the page writes softmax(QK^T)V without one);
  * the skew is per head: A_h is d x d (a full D x D rotation would mix heads);
  * k = floor(ratio * d + 0.5) columns per head; the same columns serve every sequence;
  * the column score sums the per-column absolute sums of W~_Q and K~ (the page's
    element-wise sum of two differently shaped matrices cannot be taken literally);
  * RoPE, when present, is applied before the skew: q~ = RoPE(q) A, k~ = RoPE(k) A;
  * the current token's own key/value always join the attended set;
  * the threshold test s_t > max - alpha is evaluated as max - s_t < alpha, so the maximum
    is kept for every alpha > 0 even where max - alpha rounds back to max;
  * multi-head averaging rounds the mean count half-up, with a minimum of one token;
  * the transfer cap and the averaged count keep the best tokens by (score desc, index asc);
  * pool counters are 8-bit, +1 per (layer, step) when any head selected the slot, halved
    for the whole (layer, sequence) pool when one of them reaches 255; the victim is the
    smallest counter, then the oldest insertion, then the lowest slot;
  * FIFO evicts the oldest insertion; LRU evicts the slot whose last selection (by any head)
    is oldest, where entering the pool counts as a selection at that moment, ties going to
    the oldest insertion;
  * an eviction miss is a token that selection over every token seen so far would pick but
    that the pool no longer holds;
  * the FP8 pool (follow-up work: selective prefetch of a quantized pool): every (token, head)
    row of keys and values is stored as e4m3 codes with one float32 scale, amax / 448, the
    codes being round-to-nearest-even e4m3 (saturating at 448) of x * (448 / amax) in float32;
    a row of zeros keeps scale 0; the partial key cache stays float16;
  * the INT4 pool: the same record idea with signed 4-bit codes in [-7, 7], scale amax / 7,
    codes the nearest integers (ties to even) of x * (7 / amax) in float32, two codes per byte
    (even element in the low nibble);
  * speculation fidelity: recall@c counts the speculated tokens whose real score is at least
    the c-th largest real score (c = the speculated count; ties at that score count as hits);
    the captured fraction is the share of sum_t sum_c |q_c k_tc| that the partial columns hold.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test (closed forms,
values the page prints, brute force on tiny inputs).  Two choices are consistency-checked
only ("parity unpinned"): the column choice on isotropic synthetic data (near ties), and the
RoPE placement reading.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEL_THRESHOLD = 0
SEL_HEAD_AVG = 1
SEL_NORMALIZED = 2


# ----------------------------------------------------------------------------------------
# Hyper-parameters and accounting
# ----------------------------------------------------------------------------------------
def partial_columns(ratio: float, d: int) -> int:
    """Number of partial columns per head, k = round(ratio * d) half-up.

    Section 3.4, "Skewed Partial Weights" (k = 0.3 x D) applied per head of width d.
    """
    return int(math.floor(float(ratio) * d + 0.5))


def cap_count(cap_frac: float, n_tokens: int) -> int:
    """Per-layer transfer cap in tokens: round(cap_frac * n) half-up; cap_frac >= 1 means none.

    Section 3.4, "Decoding Stage", Step 5 (up to 20 % of the KV cache).  The arithmetic is
    done in float64 on the float32 value of ``cap_frac`` (the library takes a C float).
    """
    cf = float(np.float32(cap_frac))
    if cf >= 1.0:
        return int(n_tokens)
    return int(math.floor(cf * float(n_tokens) + 0.5))


def kv_bytes(layers: int, batch: int, tokens: int, hidden: int, elem_bytes: int = 2) -> int:
    """Full KV cache size: keys and values of every token, layer and sequence (Fig 2 formula)."""
    return layers * batch * tokens * hidden * 2 * elem_bytes


# ----------------------------------------------------------------------------------------
# RoPE (the rotate-half form, pairs (j, j + d/2))
# ----------------------------------------------------------------------------------------
def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding of the last axis of ``x`` (length d, even).

    Pair j (j < d/2) is the plane (x_j, x_{j+d/2}), turned by the angle p * theta^(-2j/d).
    ``positions`` broadcasts against ``x.shape[:-1]``.  The page names only
    ``apply_rotary_pos_emb``/``rotate_half``; this is the standard half-split form.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * j / d)
    ang = np.asarray(positions, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, lo * s + hi * c], axis=-1)


# ----------------------------------------------------------------------------------------
# Offline skew (section 3.4, "Skewed Partial Weights": Q = U S V^T, A = V, W~ = W A)
# ----------------------------------------------------------------------------------------
def canonical_signs(A: np.ndarray) -> np.ndarray:
    """Flip each column of A so that its entry of largest magnitude is positive.

    Ties go to the lowest row.  Any column sign is a valid SVD; this fixes one.
    """
    A = np.array(A, dtype=np.float64, copy=True)
    for j in range(A.shape[1]):
        r = int(np.argmax(np.abs(A[:, j])))
        if A[r, j] < 0:
            A[:, j] = -A[:, j]
    return A


def sample_queries(Xs: np.ndarray, Wq: np.ndarray, H: int, d: int, rope_theta: float = 0.0):
    """Per-head sample query matrices Q_h = X_s W_Q,h (float64), post-RoPE at positions 0..Ns-1."""
    X = np.asarray(Xs, dtype=np.float64)
    W = np.asarray(Wq, dtype=np.float64)
    Q = (X @ W).reshape(X.shape[0], H, d)
    if rope_theta:
        Q = rope(Q, np.arange(X.shape[0])[:, None], rope_theta)
    return Q


def skew(Xs, Wq, Wk, H: int, d: int, rope_theta: float = 0.0, Kprompt=None):
    """Offline skewing controller.

    For each head h: Q_h = X_s W_Q,h; SVD Q_h = U S V^T; A_h = V (columns in descending
    singular value, signs canonical).  W~_Q,h = W_Q,h A_h and W~_K,h = W_K,h A_h, rounded once
    to fp16.  If ``Kprompt`` ([N, H, d], unskewed, post-RoPE for RoPE models) is given, the
    skewed prompt keys K~ = K A are returned too (rounded to fp16).

    Returns (A [H,d,d] float64, sigma [H,d], Wq_skew fp16 [D,H*d], Wk_skew fp16 [D,H*d],
    K_skew fp16 [N,H,d] or None).
    """
    Q = sample_queries(Xs, Wq, H, d, rope_theta)
    Wq64 = np.asarray(Wq, dtype=np.float64)
    Wk64 = np.asarray(Wk, dtype=np.float64)
    D = Wq64.shape[0]
    A = np.zeros((H, d, d))
    sig = np.zeros((H, d))
    Wq_s = np.zeros((D, H * d), dtype=np.float16)
    Wk_s = np.zeros((D, H * d), dtype=np.float16)
    for h in range(H):
        _, s, vt = np.linalg.svd(Q[:, h, :], full_matrices=False)
        A[h] = canonical_signs(vt.T)
        sig[h] = s
        Wq_s[:, h * d:(h + 1) * d] = (Wq64[:, h * d:(h + 1) * d] @ A[h]).astype(np.float16)
        Wk_s[:, h * d:(h + 1) * d] = (Wk64[:, h * d:(h + 1) * d] @ A[h]).astype(np.float16)
    Ks = None
    if Kprompt is not None:
        K64 = np.asarray(Kprompt, dtype=np.float64)
        Ks = np.einsum("nhc,hcj->nhj", K64, A).astype(np.float16)
    return A, sig, Wq_s, Wk_s, Ks


def energy_k(sigma, energy: float) -> int:
    """Per-layer partial width from the skewed query's spectrum (the per-layer ratio proposed
    as follow-up work): the smallest k in [1, d] whose captured energy, the mean over heads of
    sum_{i<k} sigma_i^2 / sum_i sigma_i^2 (singular values in descending order), reaches
    ``energy``; a head with no energy counts as fully captured."""
    sig = np.asarray(sigma, dtype=np.float64)
    H, d = sig.shape
    e2 = sig * sig
    tot = e2.sum(axis=1)
    frac = np.where(tot[:, None] > 0, np.cumsum(e2, axis=1) / np.where(tot > 0, tot, 1.0)[:, None], 1.0)
    mean = frac.mean(axis=0)
    for kk in range(1, d + 1):
        if mean[kk - 1] >= energy:
            return kk
    return d


def choose_columns(Wq_skew, K_skew, H: int, d: int, k: int) -> np.ndarray:
    """Partial weight index generation (section 3.4, "Prefill Stage", Step 2, Fig 9).

    colscore_h[c] = sum_r |W~_Q,h[r, c]| + sum_t |K~_h[t, c]| (t over every prompt key of every
    sequence); keep the k largest (ties to the lower column), stored ascending.
    ``K_skew`` is [..., H, d] (any leading token axes) or None.
    Returns int32 [H, k].
    """
    W = np.abs(np.asarray(Wq_skew, dtype=np.float64))
    cols = np.zeros((H, k), dtype=np.int32)
    for h in range(H):
        score = W[:, h * d:(h + 1) * d].sum(axis=0)
        if K_skew is not None:
            Kh = np.abs(np.asarray(K_skew, dtype=np.float64)[..., h, :]).reshape(-1, d)
            score = score + Kh.sum(axis=0)
        order = sorted(range(d), key=lambda c: (-score[c], c))
        cols[h] = np.sort(np.array(order[:k], dtype=np.int32))
    return cols


def colscores(Wq_skew, K_skew, H: int, d: int) -> np.ndarray:
    """The column scores used by :func:`choose_columns` ([H, d], float64)."""
    W = np.abs(np.asarray(Wq_skew, dtype=np.float64))
    out = np.zeros((H, d))
    for h in range(H):
        out[h] = W[:, h * d:(h + 1) * d].sum(axis=0)
        if K_skew is not None:
            out[h] += np.abs(np.asarray(K_skew, dtype=np.float64)[..., h, :]).reshape(-1, d).sum(axis=0)
    return out


def partial_weight(Wq_skew, cols, H: int, d: int) -> np.ndarray:
    """Step 3 of the prefill stage: W~_Q^partial = the selected columns, head-contiguous.

    Returns fp16 [D, H*k] whose column h*k + i is W~_Q[:, h*d + cols[h, i]].
    """
    k = cols.shape[1]
    W = np.asarray(Wq_skew)
    out = np.zeros((W.shape[0], H * k), dtype=W.dtype)
    for h in range(H):
        out[:, h * k:(h + 1) * k] = W[:, h * d + cols[h]]
    return out


def partial_key_cache(K_pool, cols) -> np.ndarray:
    """Step 3 of the prefill stage: the partial key cache, the selected columns of each key.

    K_pool [B, H, T, d] (skewed keys by slot) -> [B, H, k, T]: row c of head h holds
    K~[b, h, :, cols[h, c]], token axis last (the layout the score step reads).
    """
    K = np.asarray(K_pool)
    B, H, T, d = K.shape
    k = cols.shape[1]
    out = np.zeros((B, H, k, T), dtype=K.dtype)
    for h in range(H):
        for c in range(k):
            out[:, h, c, :] = K[:, h, :, cols[h, c]]
    return out


def prefill_layer(X, Wq_skew, Wk_skew, Wv, H: int, d: int, k: int, cap: int):
    """Prefill Stage, Steps 1-3, for one layer (no RoPE).

    Step 1: the prompt's skewed keys K~ = X W~_K and values V = X W_V (float64, rounded once to
    float16), stored in the pool: the pool places prompt tokens as the counter pool does
    (token t at slot t mod cap; with more tokens than slots the last cap stay).  Step 2: the
    columns, from W~_Q and the keys of every prompt token of every sequence.  Step 3: the
    partial query weight and the partial key cache of the resident slots.

    X [B, N, D] fp16; W~_Q, W~_K, W_V [D, H*d] fp16.  Returns a dict: K, V [B, N, H, d] fp16,
    cols [H, k], Wq_part [D, H*k] fp16, K_pool, V_pool [B, H, cap, d] fp16, K_part [B, H, k, cap].
    """
    X64 = np.asarray(X, dtype=np.float64)
    B, N, _ = X64.shape
    Kt = (X64 @ np.asarray(Wk_skew, dtype=np.float64)).astype(np.float16).reshape(B, N, H, d)
    Vt = (X64 @ np.asarray(Wv, dtype=np.float64)).astype(np.float16).reshape(B, N, H, d)
    cols = choose_columns(Wq_skew, Kt, H, d, k)
    Kp = np.zeros((B, H, cap, d), dtype=np.float16)
    Vp = np.zeros((B, H, cap, d), dtype=np.float16)
    for t in range(max(0, N - cap), N):
        Kp[:, :, t % cap] = Kt[:, t]
        Vp[:, :, t % cap] = Vt[:, t]
    return dict(K=Kt, V=Vt, cols=cols, Wq_part=partial_weight(Wq_skew, cols, H, d), K_pool=Kp, V_pool=Vp,
                K_part=partial_key_cache(Kp, cols))


def prefill_layer_rope(X, Wq_skew, Wk, Wv, A, theta: float, H: int, d: int, k: int, cap: int):
    """Prefill Stage, Steps 1-3, for one layer of a RoPE model.

    The keys are rotated before the skew, so the skew cannot live in W_K: K = X W_K (rounded
    once to float16, as a projection stores it), then K~_h = RoPE_t(K_h) A_h at the token's
    position t (float64, rounded once to float16).  V = X W_V.  The columns come from W~_Q =
    W_Q A and the keys; the decode stage of a RoPE model takes A_h[:, S_h] instead of a partial
    weight.  Pool placement and the partial key cache as in :func:`prefill_layer`.

    Returns a dict as :func:`prefill_layer` with A_cols [H, d, k] (float64) for Wq_part.
    """
    X64 = np.asarray(X, dtype=np.float64)
    B, N, _ = X64.shape
    Kraw = (X64 @ np.asarray(Wk, dtype=np.float64)).astype(np.float16).reshape(B, N, H, d)
    Kr = rope(Kraw.astype(np.float64), np.arange(N)[None, :, None], theta)
    A64 = np.asarray(A, dtype=np.float64)
    Kt = np.einsum("bnhi,hij->bnhj", Kr, A64).astype(np.float16)
    Vt = (X64 @ np.asarray(Wv, dtype=np.float64)).astype(np.float16).reshape(B, N, H, d)
    cols = choose_columns(Wq_skew, Kt, H, d, k)
    Kp = np.zeros((B, H, cap, d), dtype=np.float16)
    Vp = np.zeros((B, H, cap, d), dtype=np.float16)
    for t in range(max(0, N - cap), N):
        Kp[:, :, t % cap] = Kt[:, t]
        Vp[:, :, t % cap] = Vt[:, t]
    A_cols = np.stack([A64[h][:, cols[h]] for h in range(H)])
    return dict(K=Kt, V=Vt, cols=cols, A_cols=A_cols, K_pool=Kp, V_pool=Vp, K_part=partial_key_cache(Kp, cols))


# ----------------------------------------------------------------------------------------
# Decode stage (section 3.4, "Decoding Stage: Speculative KV Selection and Prefetching")
# ----------------------------------------------------------------------------------------
def partial_query(x, Wq_part, H: int, k: int) -> np.ndarray:
    """Step 1: q~p(i) = x_a(i-1) W~_Q^partial,(i).  x [B, D] fp16, W [D, H*k] -> [B, H, k] float64."""
    q = np.asarray(x, dtype=np.float64) @ np.asarray(Wq_part, dtype=np.float64)
    return q.reshape(q.shape[0], H, k)


def partial_query_rope(x, Wq, A, cols, positions, theta: float) -> np.ndarray:
    """Step 1 for RoPE models: q = x W_Q,h, rotated at the token's position, then q A_h[:, S_h].

    x [B, D]; Wq [D, H*d] (unskewed); A [H, d, d]; cols [H, k]; positions [B].
    Returns [B, H, k] float64.
    """
    H, d, _ = np.asarray(A).shape
    B = np.asarray(x).shape[0]
    q = (np.asarray(x, dtype=np.float64) @ np.asarray(Wq, dtype=np.float64)).reshape(B, H, d)
    q = rope(q, np.asarray(positions)[:, None], theta)
    k = cols.shape[1]
    out = np.zeros((B, H, k))
    for h in range(H):
        out[:, h, :] = q[:, h, :] @ np.asarray(A[h], dtype=np.float64)[:, cols[h]]
    return out


def speculate(q_part, K_part, L_valid, scale) -> np.ndarray:
    """Step 2: SpecScore = scale * q~p (K~p)^T over the resident tokens.

    q_part [B, H, k] float; K_part [B, H, k, Lcap] fp16 (column-major per head, token axis
    last); L_valid [B].  Slots t >= L_valid[b] get -inf.  ``scale`` is taken at float32
    precision (it is a C float in the library) and applied in float64.
    Returns [B, H, Lcap] float64.
    """
    q = np.asarray(q_part, dtype=np.float64)
    K = np.asarray(K_part, dtype=np.float64)
    B, H, k, Lcap = K.shape
    sc = float(np.float32(scale))
    s = np.full((B, H, Lcap), -np.inf)
    for b in range(B):
        L = int(L_valid[b])
        s[b, :, :L] = sc * np.einsum("hc,hct->ht", q[b], K[b, :, :, :L])
    return s


def _best_first(s: np.ndarray, n: int) -> np.ndarray:
    """Indices of the n best entries by (score desc, index asc), NaN never chosen, ascending."""
    ok = [t for t in range(len(s)) if not np.isnan(s[t])]
    ok.sort(key=lambda t: (-s[t], t))
    return np.array(sorted(ok[:n]), dtype=np.int64)


def select(scores, L_valid, alpha, policy: int = SEL_THRESHOLD, cap_frac: float = 1.0):
    """Steps 3-4 (and the Step 5 cap): which tokens each head prefetches.

    Threshold: I = {t : s_t > max(s) - alpha}, with max over the resident, non-NaN scores,
    evaluated as (max(s) - s_t) < alpha; NaN scores are never selected.  The comparison is made in the dtype of ``scores``
    (float64 end to end; float32 when the kernel's own scores are fed in), with
    ``alpha`` taken at float32 precision.
    Cap (cap_frac < 1): a head with more than cap_n = round(cap_frac * L) tokens keeps its
    cap_n best by (score desc, index asc).
    HEAD_AVG: cbar = max(1, round_half_up(mean_h |I_h|)), at most cap_n; every head then keeps
    its cbar best (same order), regardless of the threshold.
    NORMALIZED (the portable threshold alpha' = alpha / sigma proposed as follow-up work, read
    per head): I = {t : max - s_t < alpha * sigma} plus the ties of the maximum, sigma the
    population standard deviation of the head's resident, non-NaN scores; the cap as above.
    Returns (idx list-of-lists [B][H] of ascending int arrays, cnt int32 [B, H],
    used uint8 [B, Lcap] = 1 where any head of sequence b selected slot t).
    """
    s_all = np.asarray(scores)
    dt = s_all.dtype.type
    B, H, Lcap = s_all.shape
    a = dt(np.float32(alpha))
    idx = [[None] * H for _ in range(B)]
    cnt = np.zeros((B, H), dtype=np.int32)
    used = np.zeros((B, Lcap), dtype=np.uint8)
    for b in range(B):
        L = int(L_valid[b])
        capn = cap_count(cap_frac, L)
        for h in range(H):
            s = s_all[b, h, :L]
            finite = s[~np.isnan(s)]
            if finite.size == 0:
                idx[b][h] = np.zeros(0, dtype=np.int64)
                continue
            m = dt(finite.max())
            if policy == SEL_NORMALIZED:
                # alpha in units of the head's score spread; the maximum and its ties are
                # kept even when the spread is 0
                sigma = float(np.std(finite.astype(np.float64)))
                ah = dt(np.float32(alpha) * dt(sigma))
                sel = np.array([t for t in range(L) if not np.isnan(s[t])
                                and (dt(m - s[t]) < ah or dt(m - s[t]) == 0)], dtype=np.int64)
            else:
                # s_t > m - alpha, evaluated as the gap m - s_t < alpha so that the maximum
                # itself (gap exactly 0) is kept for every alpha > 0
                sel = np.array([t for t in range(L) if dt(m - s[t]) < a], dtype=np.int64)
            if policy in (SEL_THRESHOLD, SEL_NORMALIZED) and sel.size > capn:
                sel = _best_first(s, capn)
            idx[b][h] = sel
        if policy == SEL_HEAD_AVG:
            tot = sum(len(idx[b][h]) for h in range(H))
            cbar = max(1, (2 * tot + H) // (2 * H))
            cbar = min(cbar, capn)
            for h in range(H):
                idx[b][h] = _best_first(s_all[b, h, :L], cbar)
        for h in range(H):
            cnt[b, h] = len(idx[b][h])
            used[b, idx[b][h]] = 1
    return idx, cnt, used


def gather(K_pool, V_pool, idx, Lcap: int):
    """Step 5: copy the selected full key/value rows out of the pool.

    K_pool, V_pool: [B, H, Cap, d] (one layer).  Returns Kg, Vg [B, H, Lcap, d] with rows
    j < cnt[b, h] filled (idx[b][h][j]) and the rest zero.
    """
    Kp = np.asarray(K_pool)
    Vp = np.asarray(V_pool)
    B, H, _, d = Kp.shape
    Kg = np.zeros((B, H, Lcap, d), dtype=Kp.dtype)
    Vg = np.zeros((B, H, Lcap, d), dtype=Vp.dtype)
    for b in range(B):
        for h in range(H):
            ii = np.asarray(idx[b][h], dtype=np.int64)
            Kg[b, h, :len(ii)] = Kp[b, h, ii]
            Vg[b, h, :len(ii)] = Vp[b, h, ii]
    return Kg, Vg


def attend(q, Kg, Vg, cnt, scale, k_new=None, v_new=None) -> np.ndarray:
    """Inference controller: attention over the prefetched rows (plus the current token).

    z_j = scale * q . K_j over j < cnt[b, h] (and the current token's own key if given);
    w = softmax(z); o = sum_j w_j V_j, all in float64.  Returns [B, H, d] float64.
    """
    q64 = np.asarray(q, dtype=np.float64)
    K = np.asarray(Kg, dtype=np.float64)
    V = np.asarray(Vg, dtype=np.float64)
    B, H, _, d = K.shape
    sc = float(np.float32(scale))
    out = np.zeros((B, H, d))
    for b in range(B):
        for h in range(H):
            c = int(cnt[b, h])
            Ks, Vs = K[b, h, :c], V[b, h, :c]
            if k_new is not None:
                Ks = np.concatenate([Ks, np.asarray(k_new, dtype=np.float64)[b, h][None]], 0)
                Vs = np.concatenate([Vs, np.asarray(v_new, dtype=np.float64)[b, h][None]], 0)
            if Ks.shape[0] == 0:
                continue
            z = sc * (Ks @ q64[b, h])
            w = np.exp(z - z.max())
            w = w / w.sum()
            out[b, h] = w @ Vs
    return out


# ----------------------------------------------------------------------------------------
# KV cache pool (section 3.4, "KV Cache Pool Management Under Memory Pressure", Table 2)
# ----------------------------------------------------------------------------------------
@dataclass
class CounterPool:
    """One (layer, sequence) pool of ``cap`` slots with counter-based eviction.

    Counters are 8-bit: +1 per update when the slot was used (saturating at 255); when any
    counter reaches 255 every counter of the pool is halved.  Insertion fills free slots in
    order; once full, the victim is the slot with the smallest counter, then the oldest
    insertion, then the lowest index.  A new entry starts at counter 0.
    """
    cap: int
    counter: np.ndarray = field(default=None)
    seq: np.ndarray = field(default=None)
    filled: int = 0
    next_seq: int = 0

    def __post_init__(self):
        self.counter = np.zeros(self.cap, dtype=np.int64)
        self.seq = np.zeros(self.cap, dtype=np.int64)

    def update(self, used) -> None:
        used = np.asarray(used)[: self.cap]
        for s in range(self.filled):
            if used[s]:
                self.counter[s] = min(255, self.counter[s] + 1)
        if self.filled and self.counter[: self.filled].max() >= 255:
            self.counter[: self.filled] >>= 1

    def insert(self) -> int:
        if self.filled < self.cap:
            slot = self.filled
            self.filled += 1
        else:
            # smallest counter, then oldest insertion, then lowest slot (lexsort: last key first)
            slot = int(np.lexsort((np.arange(self.cap), self.seq, self.counter))[0])
        self.counter[slot] = 0
        self.seq[slot] = self.next_seq
        self.next_seq += 1
        return slot

    def evict(self, used) -> int:
        """One decode-step pool action: fold in this step's use, then place the new token."""
        if used is not None:
            self.update(used)
        return self.insert()


class FifoPool:
    """One (layer, sequence) pool with first-in-first-out eviction.

    Section 3.4, "KV Cache Pool Management Under Memory Pressure" (the FIFO policy of
    Table 2): the victim is the entry that has been in the pool longest.  Use does not
    matter, so ``update`` only checks its argument.
    """

    def __init__(self, cap: int):
        self.cap = cap
        self.seq = np.zeros(cap, dtype=np.int64)
        self.filled = 0
        self.next_seq = 0

    def update(self, used) -> None:
        np.asarray(used)

    def insert(self) -> int:
        if self.filled < self.cap:
            slot = self.filled
            self.filled += 1
        else:
            slot = int(np.argmin(self.seq))  # insertion numbers are unique
        self.seq[slot] = self.next_seq
        self.next_seq += 1
        return slot

    def evict(self, used) -> int:
        if used is not None:
            self.update(used)
        return self.insert()


class LruPool:
    """One (layer, sequence) pool with least-recently-used eviction.

    Section 3.4, "KV Cache Pool Management Under Memory Pressure" (the LRU policy of
    Table 2): the victim is the entry selected for prefetching least recently by any head.
    Time advances by one per update; a slot used in an update takes that time, a new entry
    takes the time of its insertion; the victim has the oldest time, then the oldest
    insertion, then the lowest slot.
    """

    def __init__(self, cap: int):
        self.cap = cap
        self.last = np.zeros(cap, dtype=np.int64)
        self.seq = np.zeros(cap, dtype=np.int64)
        self.clock = 0
        self.filled = 0
        self.next_seq = 0

    def update(self, used) -> None:
        used = np.asarray(used)[: self.cap]
        self.clock += 1
        for s in range(self.filled):
            if used[s]:
                self.last[s] = self.clock

    def insert(self) -> int:
        if self.filled < self.cap:
            slot = self.filled
            self.filled += 1
        else:
            slot = int(np.lexsort((np.arange(self.cap), self.seq, self.last))[0])
        self.last[slot] = self.clock
        self.seq[slot] = self.next_seq
        self.next_seq += 1
        return slot

    def evict(self, used) -> int:
        if used is not None:
            self.update(used)
        return self.insert()


POOL_COUNTER, POOL_FIFO, POOL_LRU = 0, 1, 2


def make_pool(cap: int, policy: int):
    """The pool model for one of the three victim policies of Table 2."""
    return {POOL_COUNTER: CounterPool, POOL_FIFO: FifoPool, POOL_LRU: LruPool}[policy](cap)


def eviction_misses(scores, idx, cnt, resident):
    """Selections of tokens the pool no longer holds (diagnostic, not a step of the method).

    ``scores`` [B, H, T] are speculated scores over every token seen so far (token index t),
    ``idx``/``cnt`` the selection over them, ``resident`` [B, T] whether token t is in the pool.
    Returns (miss count [B, H], miss mass [B, H]): the mass is the share of the selected
    tokens' softmax weight, exp(s_t - m) over the selected set, that falls on missed tokens.
    """
    scores = np.asarray(scores, dtype=np.float64)
    B, H = np.asarray(cnt).shape
    n_miss = np.zeros((B, H), dtype=np.int64)
    mass = np.zeros((B, H), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            sel = [int(t) for t in idx[b][h][: cnt[b][h]]]
            if not sel:
                continue
            m = max(scores[b, h, t] for t in sel)
            w = {t: math.exp(scores[b, h, t] - m) for t in sel}
            missed = [t for t in sel if not resident[b][t]]
            n_miss[b, h] = len(missed)
            mass[b, h] = sum(w[t] for t in missed) / sum(w.values())
    return n_miss, mass


# ----------------------------------------------------------------------------------------
# FP8 (e4m3) pool rows (a follow-up of the method: selective prefetch of a quantized pool)
# ----------------------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of an e4m3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (m/8 * 2^-6); S.1111.111 is NaN and there is no infinity."""
    sgn = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sgn * (m / 8.0) * 2.0 ** -6
    return sgn * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 byte to x (ties to the even mantissa), magnitudes above 448 saturating."""
    x = float(x)
    sign = 0x80 if (x < 0 or (x == 0 and math.copysign(1.0, x) < 0)) else 0
    a = abs(x)
    if a >= E4M3_MAX:
        return sign | 0x7E
    # spacing of the representable values around a: 2^-9 below the normal range, else 2^(e-3)
    e = -6 if a < 2.0 ** -6 else math.floor(math.log2(a))
    step = 2.0 ** (e - 3)
    q = float(np.rint(a / step)) * step          # round half to even on the quotient
    if q >= E4M3_MAX:
        return sign | 0x7E
    if q == 0:
        return sign
    if q < 2.0 ** -6:
        return sign | int(round(q / 2.0 ** -9))
    ee = math.floor(math.log2(q))
    mm = int(round((q / 2.0 ** ee - 1.0) * 8))
    return sign | ((ee + 7) << 3) | mm


def fp8_quantize_rows(X):
    """Rows (last axis) of float16 X -> (e4m3 codes uint8, float32 scales)."""
    X = np.asarray(X, dtype=np.float16).astype(np.float32)
    flat = X.reshape(-1, X.shape[-1])
    codes = np.zeros(flat.shape, dtype=np.uint8)
    scales = np.zeros(flat.shape[0], dtype=np.float32)
    for r in range(flat.shape[0]):
        amax = np.float32(np.abs(flat[r]).max())
        if amax == 0:
            continue
        inv = np.float32(np.float32(E4M3_MAX) / amax)
        scales[r] = np.float32(amax / np.float32(E4M3_MAX))
        for i in range(flat.shape[1]):
            codes[r, i] = e4m3_encode(float(np.float32(flat[r, i] * inv)))
    return codes.reshape(X.shape), scales.reshape(X.shape[:-1])


def fp8_dequantize_rows(codes, scales):
    """float16 rows: float32(e4m3 value) * scale, rounded to float16."""
    codes = np.asarray(codes)
    table = np.array([0.0 if (c & 0x7F) == 0x7F else e4m3_decode(c) for c in range(256)], dtype=np.float32)
    vals = table[codes] * np.asarray(scales, dtype=np.float32)[..., None]
    return vals.astype(np.float32).astype(np.float16)


# ----------------------------------------------------------------------------------------
# INT4 pool rows (the follow-up's own format: selective prefetch of a 4-bit pool)
# ----------------------------------------------------------------------------------------
INT4_MAX = 7


def int4_quantize_rows(X):
    """Rows (last axis) of float16 X -> (signed codes int8 in [-7, 7], float32 scales): the
    row's scale is amax / 7, its codes the nearest integers (ties to even) to x * (7 / amax)
    in float32; a row of zeros keeps scale 0 and zero codes."""
    X = np.asarray(X, dtype=np.float16).astype(np.float32)
    flat = X.reshape(-1, X.shape[-1])
    codes = np.zeros(flat.shape, dtype=np.int8)
    scales = np.zeros(flat.shape[0], dtype=np.float32)
    for r in range(flat.shape[0]):
        amax = np.float32(np.abs(flat[r]).max())
        if amax == 0:
            continue
        inv = np.float32(np.float32(INT4_MAX) / amax)
        scales[r] = np.float32(amax / np.float32(INT4_MAX))
        v = (flat[r] * inv).astype(np.float32)
        codes[r] = np.clip(np.rint(v), -INT4_MAX, INT4_MAX).astype(np.int8)
    return codes.reshape(X.shape), scales.reshape(X.shape[:-1])


def int4_pack(codes):
    """Signed 4-bit codes (last axis even) -> bytes: element 2j in the low nibble of byte j,
    element 2j + 1 in the high one, each as its two's-complement low four bits."""
    c = (np.asarray(codes).astype(np.int16) & 0xF).astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def int4_unpack(packed):
    """Inverse of int4_pack: bytes -> signed codes int8."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int8)
    hi = (p >> 4).astype(np.int8)
    lo = np.where(lo > 7, lo - 16, lo).astype(np.int8)
    hi = np.where(hi > 7, hi - 16, hi).astype(np.int8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def int4_dequantize_rows(codes, scales):
    """float16 rows: float32(code) * scale, rounded to float16."""
    vals = np.asarray(codes, dtype=np.float32) * np.asarray(scales, dtype=np.float32)[..., None]
    return vals.astype(np.float32).astype(np.float16)


# ----------------------------------------------------------------------------------------
# Speculation fidelity (diagnostics the summary's critique asks for; not steps of the method)
# ----------------------------------------------------------------------------------------
def real_scores(q, K, L_valid, scale):
    """Layer i's actual attention logits z[b,h,t] = scale * q[b,h] . K[b,h,t], t < L (else -inf)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    B, H, T, _ = K.shape
    z = np.full((B, H, T), -np.inf)
    for b in range(B):
        n = int(L_valid[b])
        z[b, :, :n] = float(scale) * np.einsum("hd,htd->ht", q[b], K[b, :, :n])
    return z


def speculation_recall(z, idx, cnt, L_valid):
    """How well a speculated set matches the real attention of its layer.

    For each (b, h) with c = cnt > 0 speculated tokens: recall = |{t in I : z_t >= z_(c)}| / c,
    z_(c) the c-th largest real score among the L resident tokens (ties at z_(c) are hits); and
    weight = sum_{t in I} softmax(z)_t over the resident tokens.  Heads with c = 0 give 0, 0.
    """
    z = np.asarray(z, dtype=np.float64)
    B, H = np.asarray(cnt).shape
    rec = np.zeros((B, H))
    wt = np.zeros((B, H))
    for b in range(B):
        n = int(L_valid[b])
        for h in range(H):
            c = int(cnt[b][h])
            if c == 0 or n == 0:
                continue
            zz = z[b, h, :n]
            thr = np.sort(zz)[::-1][min(c, n) - 1]
            sel = [int(t) for t in idx[b][h][:c]]
            rec[b, h] = sum(1 for t in sel if zz[t] >= thr) / c
            e = np.exp(zz - zz.max())
            wt[b, h] = e[sel].sum() / e.sum()
    return rec, wt


def captured_fraction(q, K, L_valid, cols):
    """Share of the dot-product magnitude that the partial columns hold, per (b, h):
    sum_t sum_{c in S_h} |q_c K_tc| / sum_t sum_c |q_c K_tc| over the resident tokens t < L."""
    q = np.abs(np.asarray(q, dtype=np.float64))
    K = np.abs(np.asarray(K, dtype=np.float64))
    cols = np.asarray(cols)
    B, H = q.shape[:2]
    out = np.zeros((B, H))
    for b in range(B):
        n = int(L_valid[b])
        for h in range(H):
            prod = q[b, h][None, :] * K[b, h, :n]
            tot = prod.sum()
            out[b, h] = prod[:, cols[h]].sum() / tot if tot > 0 else 0.0
    return out


# ----------------------------------------------------------------------------------------
# One layer-step, end to end
# ----------------------------------------------------------------------------------------
def decode_layer_step(x_prev, Wq_part, K_part, L_valid, q, K_pool, V_pool, *, H, k, scale,
                      alpha, policy=SEL_THRESHOLD, cap_frac=1.0, k_new=None, v_new=None):
    """Speculate layer i from layer i-1's input, select, gather, and attend at layer i.

    Returns a dict with q_part, scores, idx, cnt, used, out (float64).
    """
    Lcap = np.asarray(K_part).shape[-1]
    qp = partial_query(x_prev, Wq_part, H, k)
    s = speculate(qp, K_part, L_valid, scale)
    idx, cnt, used = select(s, L_valid, alpha, policy, cap_frac)
    Kg, Vg = gather(K_pool, V_pool, idx, Lcap)
    out = attend(q, Kg, Vg, cnt, scale, k_new, v_new)
    return dict(q_part=qp, scores=s, idx=idx, cnt=cnt, used=used, out=out)
